"""Python binding of libdcpmla: the C entry points under the same names.

Argument marshalling only: torch tensors become device pointers and the
caller's current CUDA stream is passed through; every step runs in the
library's CUDA kernels.  Tensor checks here only guard the marshalling (a
host tensor must never be handed over as a device pointer).
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence

import torch

from ._native import lib

D_LATENT, D_ROPE, D_K = 512, 64, 576
MAX_SHARDS = 64
KV_BF16, KV_E4M3 = 0, 1
LSE_E, LSE_2 = 0, 1
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
DERR_PAGE, DERR_POSITION, DERR_SLOT, DERR_LENGTH, DERR_TIMEOUT = 1, 2, 4, 8, 16


class DcpmlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().dcpmla_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _check(status: int, where: str) -> None:
    if status != OK:
        raise DcpmlaError(status, where)


def _dev(t: Optional[torch.Tensor], name: str, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return C.c_void_p(t.data_ptr())


def _host_i32(t: torch.Tensor, name: str):
    if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host int32 tensor")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ptr_array(tensors: Sequence[torch.Tensor], name: str, dtype=None):
    arr = (C.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = _dev(t, f"{name}[{i}]", dtype).value
    return arr


# ---------------------------------------------------------------------------
# Host: shared virtual allocator and request -> token map
# ---------------------------------------------------------------------------
def dcpmla_alloc_create(c: int, phys_capacity_tokens: int, phys_page: int,
                        initial_order: Optional[torch.Tensor] = None) -> C.c_void_p:
    h = C.c_void_p()
    order = None if initial_order is None else _host_i32(initial_order, "initial_order")
    _check(lib().dcpmla_alloc_create(c, phys_capacity_tokens, phys_page, order, C.byref(h)),
           "dcpmla_alloc_create")
    return h


def dcpmla_alloc_destroy(h) -> None:
    _check(lib().dcpmla_alloc_destroy(h), "dcpmla_alloc_destroy")


def dcpmla_alloc_geometry(h) -> dict:
    c, P, vp = C.c_int32(), C.c_int32(), C.c_int32()
    n, cap = C.c_int64(), C.c_int64()
    _check(lib().dcpmla_alloc_geometry(h, C.byref(c), C.byref(P), C.byref(vp), C.byref(n),
                                       C.byref(cap)), "dcpmla_alloc_geometry")
    return dict(c=c.value, phys_page=P.value, virtual_page=vp.value, num_pages=n.value,
                virtual_capacity=cap.value)


def dcpmla_alloc_free_count(h) -> int:
    n = C.c_int64()
    _check(lib().dcpmla_alloc_free_count(h, C.byref(n)), "dcpmla_alloc_free_count")
    return n.value


def dcpmla_effective_page_size(h) -> int:
    out = C.c_int32()
    _check(lib().dcpmla_effective_page_size(h, C.byref(out)), "dcpmla_effective_page_size")
    return out.value


def dcpmla_alloc_pages(h, n: int) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.int32)
    _check(lib().dcpmla_alloc_pages(h, n, C.c_void_p(out.data_ptr())), "dcpmla_alloc_pages")
    return out


def dcpmla_free_pages(h, ids: torch.Tensor) -> None:
    _check(lib().dcpmla_free_pages(h, ids.numel(), _host_i32(ids, "ids")), "dcpmla_free_pages")


def dcpmla_reqmap_create(alloc, max_requests: int, max_pages_per_request: int) -> C.c_void_p:
    h = C.c_void_p()
    _check(lib().dcpmla_reqmap_create(alloc, max_requests, max_pages_per_request, C.byref(h)),
           "dcpmla_reqmap_create")
    return h


def dcpmla_reqmap_destroy(h) -> None:
    _check(lib().dcpmla_reqmap_destroy(h), "dcpmla_reqmap_destroy")


def dcpmla_reqmap_extend(h, req: int, n_new: int) -> int:
    first = C.c_int64()
    _check(lib().dcpmla_reqmap_extend(h, req, n_new, C.byref(first)), "dcpmla_reqmap_extend")
    return first.value


def dcpmla_reqmap_release(h, req: int) -> None:
    _check(lib().dcpmla_reqmap_release(h, req), "dcpmla_reqmap_release")


def dcpmla_reqmap_length(h, req: int) -> int:
    n = C.c_int64()
    _check(lib().dcpmla_reqmap_length(h, req, C.byref(n)), "dcpmla_reqmap_length")
    return n.value


def dcpmla_reqmap_page_table(h, reqs: Sequence[int], max_pages: int, pad: int = -1):
    r = torch.tensor(list(reqs), dtype=torch.int32)
    table = torch.empty((len(reqs), max_pages), dtype=torch.int32)
    lens = torch.empty(len(reqs), dtype=torch.int32)
    _check(lib().dcpmla_reqmap_page_table(h, C.c_void_p(r.data_ptr()), len(reqs), max_pages, pad,
                                          C.c_void_p(table.data_ptr()),
                                          C.c_void_p(lens.data_ptr())),
           "dcpmla_reqmap_page_table")
    return table, lens


def dcpmla_map_positions(page_table: torch.Tensor, c: int, P: int, req: torch.Tensor,
                         pos: torch.Tensor, interleave: int = 1):
    """Host arrays in, (vslot int64, owner int32, phys int64) out."""
    assert page_table.dtype == torch.int32 and page_table.dim() == 2 and not page_table.is_cuda
    req = req.to(torch.int32).contiguous()
    pos = pos.to(torch.int64).contiguous()
    n = pos.numel()
    v = torch.empty(n, dtype=torch.int64)
    o = torch.empty(n, dtype=torch.int32)
    s = torch.empty(n, dtype=torch.int64)
    pt = page_table.contiguous()
    _check(lib().dcpmla_map_positions(C.c_void_p(pt.data_ptr()), pt.shape[1], c, interleave, P,
                                      C.c_void_p(req.data_ptr()), C.c_void_p(pos.data_ptr()), n,
                                      C.c_void_p(v.data_ptr()), C.c_void_p(o.data_ptr()),
                                      C.c_void_p(s.data_ptr())), "dcpmla_map_positions")
    return v, o, s


# ---------------------------------------------------------------------------
# Device calls (asynchronous on the current stream)
# ---------------------------------------------------------------------------
def dcpmla_slot_map(page_table: torch.Tensor, num_pages: int, c: int, P: int, req: torch.Tensor,
                    pos: torch.Tensor, vslot: Optional[torch.Tensor], owner: Optional[torch.Tensor],
                    phys: Optional[torch.Tensor], err: Optional[torch.Tensor], stream=None,
                    interleave: int = 1) -> None:
    n = pos.numel()
    _check(lib().dcpmla_slot_map(
        _dev(page_table, "page_table", torch.int32), page_table.shape[0], page_table.shape[1],
        num_pages, c, interleave, P, _dev(req, "req", torch.int32), _dev(pos, "pos", torch.int64), n,
        _dev(vslot, "vslot", torch.int64, True), _dev(owner, "owner", torch.int32, True),
        _dev(phys, "phys", torch.int64, True), _dev(err, "err", torch.int32, True),
        _stream(stream)), "dcpmla_slot_map")


def dcpmla_kv_append(pools: Sequence[torch.Tensor], scale_pools: Optional[Sequence[torch.Tensor]],
                     kv_dtype: int, owner: torch.Tensor, phys: torch.Tensor, ckv: torch.Tensor,
                     krope: torch.Tensor, row_scales: Optional[torch.Tensor],
                     err: Optional[torch.Tensor], stream=None) -> None:
    c = len(pools)
    pool_rows = pools[0].shape[0]
    parr = _ptr_array(pools, "pools")
    sarr = None if scale_pools is None else _ptr_array(scale_pools, "scale_pools", torch.float32)
    n = owner.numel()
    if ckv.dim() != 2 or krope.dim() != 2 or ckv.stride(1) != 1 or krope.stride(1) != 1:
        raise ValueError("ckv / krope must be 2-D with unit inner stride")
    if not (ckv.is_cuda and krope.is_cuda):
        raise ValueError("ckv / krope must be CUDA tensors")
    _check(lib().dcpmla_kv_append(
        parr, sarr, kv_dtype, pool_rows, c, _dev(owner, "owner", torch.int32),
        _dev(phys, "phys", torch.int64), C.c_void_p(ckv.data_ptr()), ckv.stride(0),
        C.c_void_p(krope.data_ptr()), krope.stride(0),
        _dev(row_scales, "row_scales", torch.float32, True), n,
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_kv_append")


def dcpmla_decode_workspace_size(B: int, Tq: int, H: int, P: int, c: int, shard_count: int,
                                 kv_dtype: int, max_pages: int) -> int:
    out = C.c_size_t()
    _check(lib().dcpmla_decode_workspace_size(B, Tq, H, P, c, shard_count, kv_dtype, max_pages,
                                              C.byref(out)), "dcpmla_decode_workspace_size")
    return out.value


PATH_TC_FEWHEAD, PATH_TC_ROWS, PATH_CUDA_CORE = 1, 2, 3


def dcpmla_decode_path(B: int, Tq: int, H: int, P: int, c: int, shard_count: int,
                       kv_dtype: int, max_pages: int) -> tuple:
    """(path, kernel launches per dcpmla_decode call) for this shape on the current device."""
    path, n = C.c_int32(), C.c_int32()
    _check(lib().dcpmla_decode_path(B, Tq, H, P, c, shard_count, kv_dtype, max_pages,
                                    C.byref(path), C.byref(n)), "dcpmla_decode_path")
    return path.value, n.value


def dcpmla_decode(q: torch.Tensor, pools: Sequence[torch.Tensor],
                  scale_pools: Optional[Sequence[torch.Tensor]], kv_dtype: int,
                  page_table: torch.Tensor, seq_lens: torch.Tensor, P: int, c: int,
                  shard_begin: int, shard_count: int, sm_scale: float, lse_base: int,
                  o_part: torch.Tensor, lse_part: torch.Tensor, workspace: Optional[torch.Tensor],
                  err: Optional[torch.Tensor], stream=None, interleave: int = 1) -> None:
    """q: bf16 [B, Tq, H, 576]; pools: c tensors [pool_rows, 576]; page_table int32 [B, max_pages]."""
    B, Tq, H, _ = q.shape
    if len(pools) != c:
        raise ValueError("need one pool per shard")
    parr = _ptr_array(pools, "pools")
    sarr = None if scale_pools is None else _ptr_array(scale_pools, "scale_pools", torch.float32)
    ws = None if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().dcpmla_decode(
        _dev(q, "q", torch.bfloat16), parr, sarr, kv_dtype, pools[0].shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1],
        _dev(seq_lens, "seq_lens", torch.int32), B, Tq, H, P, c, interleave, shard_begin,
        shard_count, float(sm_scale), lse_base, _dev(o_part, "o_part", torch.float32),
        _dev(lse_part, "lse_part", torch.float32), ws, ws_bytes,
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_decode")


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def dcpmla_decode_noalloc(q: torch.Tensor, pools: Sequence[torch.Tensor],
                          scale_pools: Optional[Sequence[torch.Tensor]], kv_dtype: int,
                          page_table: torch.Tensor, seq_lens: torch.Tensor, P: int, c: int,
                          shard_begin: int, shard_count: int, sm_scale: float, lse_base: int,
                          o_part: torch.Tensor, lse_part: torch.Tensor,
                          err: Optional[torch.Tensor], stream=None) -> None:
    """dcpmla_decode without a caller workspace (scratch is the library's static device array)."""
    B_, Tq, H, _ = q.shape
    if len(pools) != c:
        raise ValueError("need one pool per shard")
    parr = _ptr_array(pools, "pools")
    sarr = None if scale_pools is None else _ptr_array(scale_pools, "scale_pools", torch.float32)
    _check(lib().dcpmla_decode_noalloc(
        _dev(q, "q", torch.bfloat16), parr, sarr, kv_dtype, pools[0].shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1],
        _dev(seq_lens, "seq_lens", torch.int32), B_, Tq, H, P, c, shard_begin, shard_count,
        float(sm_scale), lse_base, _dev(o_part, "o_part", torch.float32),
        _dev(lse_part, "lse_part", torch.float32), _dev(err, "err", torch.int32, True),
        _stream(stream)), "dcpmla_decode_noalloc")


def dcpmla_testing_set_wait_limit(cycles: int) -> None:
    """Testing only: pipeline-wait limit (clock64 cycles) of later decode launches; <= 0 restores
    the default of about one second."""
    _check(lib().dcpmla_testing_set_wait_limit(int(cycles)), "dcpmla_testing_set_wait_limit")


def dcpmla_lse_merge(o_part: torch.Tensor, lse_part: torch.Tensor, c: int, rows: int,
                     lse_base: int, o: torch.Tensor, lse: Optional[torch.Tensor],
                     err: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(lib().dcpmla_lse_merge(
        _dev(o_part, "o_part", torch.float32), _dev(lse_part, "lse_part", torch.float32), c, rows,
        lse_base, _dev(o, "o", torch.float32), _dev(lse, "lse", torch.float32, True),
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_lse_merge")


# ---------------------------------------------------------------------------
# Relayout, un-stripe gather, E4M3 quantising append, HiCache index filter
# ---------------------------------------------------------------------------
def dcpmla_relayout_dense_to_striped(dense: torch.Tensor, dense_scales: Optional[torch.Tensor],
                                     dense_page_table: torch.Tensor, pools: Sequence[torch.Tensor],
                                     scale_pools: Optional[Sequence[torch.Tensor]], kv_dtype: int,
                                     page_table: torch.Tensor, seq_lens: torch.Tensor, P: int, c: int,
                                     err: Optional[torch.Tensor], stream=None,
                                     interleave: int = 1) -> None:
    """dense: [dense_rows, 576] (bf16 or uint8 E4M3 codes); tables int32 [B, *]; pools: c tensors."""
    B_ = page_table.shape[0]
    parr = _ptr_array(pools, "pools")
    sarr = None if scale_pools is None else _ptr_array(scale_pools, "scale_pools", torch.float32)
    _check(lib().dcpmla_relayout_dense_to_striped(
        _dev(dense, "dense"), _dev(dense_scales, "dense_scales", torch.float32, True), dense.shape[0],
        _dev(dense_page_table, "dense_page_table", torch.int32), dense_page_table.shape[1], parr, sarr,
        kv_dtype, pools[0].shape[0], _dev(page_table, "page_table", torch.int32), page_table.shape[1],
        _dev(seq_lens, "seq_lens", torch.int32), B_, P, c, interleave,
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_relayout_dense_to_striped")


def dcpmla_gather_unstriped(pools: Sequence[torch.Tensor], scale_pools: Optional[Sequence[torch.Tensor]],
                            kv_dtype: int, page_table: torch.Tensor, seq_lens: torch.Tensor, P: int,
                            c: int, out: torch.Tensor, out_scales: Optional[torch.Tensor],
                            err: Optional[torch.Tensor], stream=None, interleave: int = 1) -> None:
    """out: [B, capacity, 576] (kv dtype); out_scales: fp32 [B, capacity] for E4M3."""
    parr = _ptr_array(pools, "pools")
    sarr = None if scale_pools is None else _ptr_array(scale_pools, "scale_pools", torch.float32)
    _check(lib().dcpmla_gather_unstriped(
        parr, sarr, kv_dtype, pools[0].shape[0], _dev(page_table, "page_table", torch.int32),
        page_table.shape[1], _dev(seq_lens, "seq_lens", torch.int32), page_table.shape[0], P, c,
        interleave, _dev(out, "out"), _dev(out_scales, "out_scales", torch.float32, True), out.shape[1],
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_gather_unstriped")


def dcpmla_kv_append_e4m3(pools: Sequence[torch.Tensor], scale_pools: Sequence[torch.Tensor],
                          owner: torch.Tensor, phys: torch.Tensor, ckv: torch.Tensor,
                          krope: torch.Tensor, err: Optional[torch.Tensor], stream=None) -> None:
    """ckv: bf16 [n, >=512], krope: bf16 [n, >=64] (rows may be strided)."""
    n = owner.numel()
    if ckv.dtype != torch.bfloat16 or krope.dtype != torch.bfloat16 or not ckv.is_cuda:
        raise ValueError("ckv / krope must be bf16 CUDA tensors")
    if ckv.stride(1) != 1 or krope.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    _check(lib().dcpmla_kv_append_e4m3(
        _ptr_array(pools, "pools", torch.uint8), _ptr_array(scale_pools, "scale_pools", torch.float32),
        pools[0].shape[0], len(pools), _dev(owner, "owner", torch.int32), _dev(phys, "phys", torch.int64),
        C.c_void_p(ckv.data_ptr()), ckv.stride(0), C.c_void_p(krope.data_ptr()), krope.stride(0), n,
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_kv_append_e4m3")


def dcpmla_hicache_filter_workspace_size(n: int) -> int:
    out = C.c_size_t()
    _check(lib().dcpmla_hicache_filter_workspace_size(n, C.byref(out)), "dcpmla_hicache_filter_workspace_size")
    return out.value


def dcpmla_hicache_filter(idx: torch.Tensor, c: int, rank: int, out: torch.Tensor, count: torch.Tensor,
                          workspace: Optional[torch.Tensor], err: Optional[torch.Tensor], stream=None,
                          interleave: int = 1) -> None:
    """idx: int64 [n] widened-page slots; out: int64 [n]; count: int64 [1] (device)."""
    n = idx.numel()
    ws = None if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().dcpmla_hicache_filter(
        _dev(idx, "idx", torch.int64), n, c, interleave, rank, _dev(out, "out", torch.int64),
        _dev(count, "count", torch.int64), ws, ws_bytes, _dev(err, "err", torch.int32, True),
        _stream(stream)), "dcpmla_hicache_filter")


# ---------------------------------------------------------------------------
# Fused decode + merge
# ---------------------------------------------------------------------------
def dcpmla_decode_merged_workspace_size(B: int, Tq: int, H: int, P: int, c: int, kv_dtype: int,
                                        max_pages: int) -> int:
    out = C.c_size_t()
    _check(lib().dcpmla_decode_merged_workspace_size(B, Tq, H, P, c, kv_dtype, max_pages, C.byref(out)),
           "dcpmla_decode_merged_workspace_size")
    return out.value


def dcpmla_decode_merged(q: torch.Tensor, pools: Sequence[torch.Tensor],
                         scale_pools: Optional[Sequence[torch.Tensor]], kv_dtype: int,
                         page_table: torch.Tensor, seq_lens: torch.Tensor, P: int, c: int, sm_scale: float,
                         lse_base: int, o: torch.Tensor, lse: torch.Tensor, workspace: Optional[torch.Tensor],
                         err: Optional[torch.Tensor], stream=None, interleave: int = 1) -> None:
    """All c shards decoded and merged: o fp32 [B, Tq, H, 512], lse fp32 [B, Tq, H]."""
    B_, Tq, H, _ = q.shape
    if len(pools) != c:
        raise ValueError("need one pool per shard")
    parr = _ptr_array(pools, "pools")
    sarr = None if scale_pools is None else _ptr_array(scale_pools, "scale_pools", torch.float32)
    ws = None if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().dcpmla_decode_merged(
        _dev(q, "q", torch.bfloat16), parr, sarr, kv_dtype, pools[0].shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1],
        _dev(seq_lens, "seq_lens", torch.int32), B_, Tq, H, P, c, interleave, float(sm_scale), lse_base,
        _dev(o, "o", torch.float32), _dev(lse, "lse", torch.float32), ws, ws_bytes,
        _dev(err, "err", torch.int32, True), _stream(stream)), "dcpmla_decode_merged")
