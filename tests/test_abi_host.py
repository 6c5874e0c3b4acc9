"""C-ABI checks that need no GPU: exports, host allocator / request map against the oracle,
host position map, and argument validation."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import dcp_workloads as W
import oracle as O
from decode_context_mla_gb300 import _native
from decode_context_mla_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from decode_context_mla_gb300.build import build
    build()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        with open(os.path.join(ROOT, "include", fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(dcpmla_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(_native.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_native.SIGNATURES), "binding signature table out of sync with header"


def test_status_strings_and_version():
    lib = _native.lib()
    assert lib.dcpmla_version() >= 1
    for st in (0, -1, -2, -3, -4, -5):
        assert lib.dcpmla_status_string(st)
    assert lib.dcpmla_status_string(-99) == b"unknown status"


@pytest.mark.parametrize("name", ["tiny", "dsv3", "long", "bimodal", "fp8"])
def test_page_tables_bit_exact_against_oracle(name):
    """The C++ allocator and request map give the oracle's page tables for every workload."""
    w = W.WORKLOADS[name]
    lens = w.seq_lens()
    pages = w.pages_per_request()
    order = W.free_list_order(w.seed, sum(pages))
    h = B.dcpmla_alloc_create(w.c, sum(pages) * w.P, w.P, order)
    m = B.dcpmla_reqmap_create(h, w.B, max(pages))
    alloc = O.SharedVirtualAllocator(w.c, sum(pages) * w.P, w.P, order.tolist())
    rmap = O.RequestTokenMap(alloc)
    for b, L in enumerate(lens):
        assert B.dcpmla_reqmap_extend(m, b, L) == 0
        rmap.extend(b, L)
    got, got_lens = B.dcpmla_reqmap_page_table(m, list(range(w.B)), max(pages))
    want = rmap.page_table(range(w.B), max(pages))
    assert np.array_equal(got.numpy(), want)
    assert got_lens.tolist() == lens
    assert B.dcpmla_alloc_free_count(h) == 0          # sized exactly
    with pytest.raises(B.DcpmlaError) as e:
        B.dcpmla_reqmap_extend(m, 0, w.P * w.c)
    assert e.value.status == B.ERR_CAPACITY
    B.dcpmla_reqmap_destroy(m)
    B.dcpmla_alloc_destroy(h)


@pytest.mark.parametrize("c,P,I", [(1, 16, 1), (3, 5, 1), (4, 16, 1), (8, 64, 1), (2, 16, 1), (16, 1, 1),
                                   (2, 64, 16), (4, 16, 4), (8, 16, 2), (3, 8, 8)])
def test_host_position_map_bit_exact(c, P, I):
    rng = np.random.default_rng(c * 100 + P)
    lens = rng.integers(1, 3000, size=5).tolist()
    pages = [-(-L // (P * c)) for L in lens]
    order = torch.from_numpy(rng.permutation(sum(pages)).astype(np.int32))
    h = B.dcpmla_alloc_create(c, sum(pages) * P, P, order)
    m = B.dcpmla_reqmap_create(h, len(lens), max(pages))
    alloc = O.SharedVirtualAllocator(c, sum(pages) * P, P, order.tolist())
    rmap = O.RequestTokenMap(alloc)
    for b, L in enumerate(lens):
        B.dcpmla_reqmap_extend(m, b, L)
        rmap.extend(b, L)
    pt, _ = B.dcpmla_reqmap_page_table(m, list(range(len(lens))), max(pages))
    req = np.concatenate([np.full(L, b) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    v, own, phys = B.dcpmla_map_positions(pt, c, P, torch.from_numpy(req), torch.from_numpy(pos),
                                          interleave=I)
    for b in range(len(lens)):
        sel = req == b
        wv, wo, wp = O.map_positions(rmap, b, pos[sel], I)
        assert np.array_equal(v.numpy()[sel], wv)
        assert np.array_equal(own.numpy()[sel], wo)
        assert np.array_equal(phys.numpy()[sel], wp)


def test_allocator_validation_and_all_or_nothing():
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_alloc_create(0, 64, 16)
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_alloc_create(2, 60, 16)                           # not whole pages
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_alloc_create(2, 64, 16, torch.tensor([0, 1, 1, 3], dtype=torch.int32))
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_alloc_create(65, 64, 16)                          # beyond the shard limit
    h = B.dcpmla_alloc_create(2, 64, 16, torch.tensor([2, 0, 3, 1], dtype=torch.int32))
    assert B.dcpmla_effective_page_size(h) == 32
    assert B.dcpmla_alloc_pages(h, 3).tolist() == [2, 0, 3]
    with pytest.raises(B.DcpmlaError) as e:
        B.dcpmla_alloc_pages(h, 2)
    assert e.value.status == B.ERR_CAPACITY
    assert B.dcpmla_alloc_free_count(h) == 1                       # nothing taken
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_free_pages(h, torch.tensor([0, 1], dtype=torch.int32))   # 1 is not allocated
    assert B.dcpmla_alloc_free_count(h) == 1                       # nothing freed
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_free_pages(h, torch.tensor([0, 0], dtype=torch.int32))   # twice
    B.dcpmla_free_pages(h, torch.tensor([0], dtype=torch.int32))
    assert B.dcpmla_alloc_pages(h, 2).tolist() == [1, 0]
    m = B.dcpmla_reqmap_create(h, 2, 4)
    with pytest.raises(B.DcpmlaError) as e:
        B.dcpmla_reqmap_extend(m, 0, 1)                            # no page left
    assert e.value.status == B.ERR_CAPACITY
    assert B.dcpmla_reqmap_length(m, 0) == 0                       # unchanged
    with pytest.raises(B.DcpmlaError):
        B.dcpmla_reqmap_extend(m, 2, 1)                            # no such request
    B.dcpmla_reqmap_destroy(m)
    B.dcpmla_alloc_destroy(h)


def test_request_map_release_returns_pages():
    h = B.dcpmla_alloc_create(4, 16 * 8, 16)
    m = B.dcpmla_reqmap_create(h, 3, 8)
    B.dcpmla_reqmap_extend(m, 0, 130)                              # 3 virtual pages of 64
    B.dcpmla_reqmap_extend(m, 1, 64)
    assert B.dcpmla_alloc_free_count(h) == 4
    B.dcpmla_reqmap_release(m, 0)
    assert B.dcpmla_alloc_free_count(h) == 7
    assert B.dcpmla_reqmap_length(m, 0) == 0
    pt, lens = B.dcpmla_reqmap_page_table(m, [0, 1], 4)
    assert pt.tolist() == [[-1, -1, -1, -1], [3, -1, -1, -1]] and lens.tolist() == [0, 64]
    with pytest.raises(B.DcpmlaError) as e:
        B.dcpmla_reqmap_page_table(m, [1], 0)
    B.dcpmla_reqmap_destroy(m)
    B.dcpmla_alloc_destroy(h)


def test_device_calls_reject_bad_arguments_before_launch():
    """Host-side checks fail before anything is enqueued (no GPU needed to reach them)."""
    lib = _native.lib()
    ws = ctypes.c_size_t()
    assert lib.dcpmla_decode_workspace_size(1, 0, 16, 16, 4, 4, 0, 4, ctypes.byref(ws)) == -1
    assert lib.dcpmla_decode_workspace_size(1, 1, 16, 16, 4, 4, 7, 4, ctypes.byref(ws)) == -2
    assert lib.dcpmla_decode_workspace_size(1, 17, 16, 16, 4, 4, 0, 4, ctypes.byref(ws)) == -2
    assert lib.dcpmla_lse_merge(None, None, 0, 4, 0, None, None, None, None) == -1
    assert lib.dcpmla_lse_merge(None, None, 2, 4, 3, None, None, None, None) == -1
    assert lib.dcpmla_lse_merge(None, None, 2, 4, 0, None, None, None, None) == -1
    assert lib.dcpmla_slot_map(None, 1, 4, 4, 0, 1, 16, None, None, 5, None, None, None, None,
                               None) == -1
    assert lib.dcpmla_slot_map(None, 1, 4, 4, 2, 3, 16, None, None, 5, None, None, None, None,
                               None) == -1                    # interleave must divide P
    assert lib.dcpmla_kv_append(None, None, 5, 10, 2, None, None, None, 576, None, 576, None, 1,
                                None, None) == -2
    # a zero-sized call is a no-op
    assert lib.dcpmla_lse_merge(None, None, 2, 0, 0, None, None, None, None) == 0
