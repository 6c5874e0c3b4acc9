// C entry points of the shard-local decode: argument checks and dispatch.
//
// SGLang "Decode Context Parallelism" docs, MLA decode dataflow and DCP x
// speculative decoding: each shard's kernel gets the rank-local page table,
// cp_world (c), cp_rank (r) and the global KV length, and returns the
// rank-local (output, LSE).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "decode.cuh"

using namespace dcpmla;

namespace {

int fill_args(DecodeArgs& a, const void* d_q, void* const* pools, float* const* scale_pools,
              int32_t kv_dtype, int64_t pool_rows, const int32_t* d_page_table, int32_t max_pages,
              const int32_t* d_seq_lens, int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
              int32_t interleave, int32_t shard_begin, int32_t shard_count, float sm_scale,
              int32_t lse_base, float* d_o_part, float* d_lse_part, int32_t* d_err, bool check_ptrs) {
  if (B < 0 || Tq < 1 || H < 1 || P < 1 || c < 1 || c > DCPMLA_MAX_SHARDS || max_pages < 1 ||
      pool_rows < 0 || shard_begin < 0 || shard_count < 1 || shard_begin + shard_count > c)
    return DCPMLA_ERR_INVALID;
  if (interleave < 1 || P % interleave) return DCPMLA_ERR_INVALID;
  if (lse_base != DCPMLA_LSE_E && lse_base != DCPMLA_LSE_2) return DCPMLA_ERR_INVALID;
  if (kv_dtype != DCPMLA_KV_BF16 && kv_dtype != DCPMLA_KV_E4M3) return DCPMLA_ERR_UNSUPPORTED;
  if (Tq > 16 || (int64_t)Tq * H > 1024) return DCPMLA_ERR_UNSUPPORTED;
  if (!(sm_scale > 0.f) || !(sm_scale < 1e30f)) return DCPMLA_ERR_INVALID;
  a = DecodeArgs{};
  a.q = static_cast<const __nv_bfloat16*>(d_q);
  a.fp8 = kv_dtype == DCPMLA_KV_E4M3;
  a.pool_rows = pool_rows;
  a.num_pages = pool_rows / P;
  a.pt = d_page_table;
  a.max_pages = max_pages;
  a.seq_lens = d_seq_lens;
  a.B = B; a.Tq = Tq; a.H = H; a.R = Tq * H; a.P = P; a.c = c; a.I = interleave;
  a.shard_begin = shard_begin;
  a.shard_count = shard_count;
  a.sm_scale = sm_scale;
  a.base2 = lse_base == DCPMLA_LSE_2;
  a.o_part = d_o_part;
  a.lse_part = d_lse_part;
  a.err = d_err;
  if (!check_ptrs) return DCPMLA_OK;
  if (!d_q || !pools || !d_page_table || !d_seq_lens || !d_o_part || !d_lse_part)
    return DCPMLA_ERR_INVALID;
  if (!aligned16(d_q) || !aligned16(d_o_part)) return DCPMLA_ERR_INVALID;
  if (a.fp8 && !scale_pools) return DCPMLA_ERR_INVALID;
  for (int r = shard_begin; r < shard_begin + shard_count; ++r) {
    if (!pools[r] || !aligned16(pools[r])) return DCPMLA_ERR_INVALID;
    a.kv.pool[r] = pools[r];
    if (a.fp8) {
      if (!scale_pools[r]) return DCPMLA_ERR_INVALID;
      a.kv.scale[r] = scale_pools[r];
    }
  }
  return DCPMLA_OK;
}

}  // namespace

namespace dcpmla {

LaunchKey launch_key(const DecodeArgs& a, const void* ws, size_t ws_bytes, int tag) {
  LaunchKey k;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  auto u = [](const void* ptr) { return (uint64_t)reinterpret_cast<uintptr_t>(ptr); };
  k.add((uint64_t)(uint32_t)tag);
  k.add((uint64_t)(uint32_t)dev);
  k.add(u(ws));
  k.add((uint64_t)ws_bytes);
  k.add(u(a.q));
  for (int r = a.shard_begin; r < a.shard_begin + a.shard_count; ++r) {
    k.add(u(a.kv.pool[r]));
    k.add(u(a.kv.scale[r]));
  }
  k.add((uint64_t)a.fp8);
  k.add((uint64_t)a.pool_rows);
  k.add((uint64_t)a.num_pages);
  k.add(u(a.pt));
  k.add(u(a.seq_lens));
  k.add((uint64_t)(uint32_t)a.max_pages);
  k.add(((uint64_t)(uint32_t)a.B << 32) | (uint32_t)a.Tq);
  k.add(((uint64_t)(uint32_t)a.H << 32) | (uint32_t)a.R);
  k.add(((uint64_t)(uint32_t)a.P << 32) | (uint32_t)a.c);
  k.add(((uint64_t)(uint32_t)a.shard_begin << 32) | (uint32_t)a.shard_count);
  uint32_t sc = 0;
  memcpy(&sc, &a.sm_scale, 4);
  k.add(((uint64_t)(uint32_t)a.I << 32) | sc);
  k.add((uint64_t)a.base2);
  k.add(u(a.o_part));
  k.add(u(a.lse_part));
  k.add(u(a.err));
  return k;
}

namespace {
std::atomic<int32_t> g_wait_kcycles{kDefaultWaitKcycles};
}

int32_t pipeline_wait_kcycles() { return g_wait_kcycles.load(std::memory_order_relaxed); }

int ensure_smem_attr(const void* func, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;   // (function, device)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DCPMLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& d : done)
    if (d.first == func && d.second == dev) return DCPMLA_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return DCPMLA_ERR_CUDA;
  done.emplace_back(func, dev);
  return DCPMLA_OK;
}

}  // namespace dcpmla

namespace {

// Few query rows (<= 16, bf16 KV) run on the token-major tensor-core kernel;
// other shapes the tensor cores take run on the 128-row-tile kernel; the rest
// on the CUDA-core kernel.
size_t workspace_for(const DecodeArgs& a, int sm) {
  if (fh_supported(a, sm)) return fh_workspace_bytes(a, sm);
  return tc_supported(a) ? tc_workspace_bytes(a, sm) : fma_workspace_bytes(a, sm);
}

}  // namespace

extern "C" {

int dcpmla_testing_set_wait_limit(int64_t cycles) {
  // in units of 1024 cycles, rounded down (0: the first failed try gives up), capped at 2^31 units
  const int64_t k = cycles > 0 ? std::min<int64_t>(cycles >> 10, INT32_MAX) : (int64_t)kDefaultWaitKcycles;
  g_wait_kcycles.store((int32_t)k, std::memory_order_relaxed);
  return DCPMLA_OK;
}

int dcpmla_decode_workspace_size(int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
                                 int32_t shard_count, int32_t kv_dtype, int32_t max_pages,
                                 size_t* out) {
  if (!out) return DCPMLA_ERR_INVALID;
  DecodeArgs a;
  const int st = fill_args(a, nullptr, nullptr, nullptr, kv_dtype, 0, nullptr, max_pages, nullptr,
                           B, Tq, H, P, c, 1, 0, shard_count, 1.f, DCPMLA_LSE_E, nullptr, nullptr,
                           nullptr, false);
  if (st != DCPMLA_OK) return st;
  const int sm = device_sm_count();
  if (sm <= 0) return DCPMLA_ERR_CUDA;
  *out = workspace_for(a, sm);
  return DCPMLA_OK;
}

int dcpmla_decode_path(int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c, int32_t shard_count,
                       int32_t kv_dtype, int32_t max_pages, int32_t* path, int32_t* kernel_launches) {
  DecodeArgs a;
  const int st = fill_args(a, nullptr, nullptr, nullptr, kv_dtype, 0, nullptr, max_pages, nullptr,
                           B, Tq, H, P, c, 1, 0, shard_count, 1.f, DCPMLA_LSE_E, nullptr, nullptr,
                           nullptr, false);
  if (st != DCPMLA_OK) return st;
  const int sm = device_sm_count();
  if (sm <= 0) return DCPMLA_ERR_CUDA;
  int pth = DCPMLA_PATH_CUDA_CORE, n = 1;
  if (fh_supported(a, sm)) {
    pth = DCPMLA_PATH_TC_FEWHEAD;
    n = 2;   // decode + merge of split units
  } else if (tc_supported(a)) {
    pth = DCPMLA_PATH_TC_ROWS;
    n = tc_kernel_launches(a);
  }
  if (path) *path = pth;
  if (kernel_launches) *kernel_launches = B == 0 ? 0 : n;
  return DCPMLA_OK;
}

int dcpmla_decode(const void* d_q, void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                  int64_t pool_rows, const int32_t* d_page_table, int32_t max_pages,
                  const int32_t* d_seq_lens, int32_t B, int32_t Tq, int32_t H, int32_t P,
                  int32_t c, int32_t interleave, int32_t shard_begin, int32_t shard_count,
                  float sm_scale, int32_t lse_base, float* d_o_part, float* d_lse_part,
                  void* d_workspace, size_t ws_bytes, int32_t* d_err, void* stream) {
  DecodeArgs a;
  int st = fill_args(a, d_q, pools, scale_pools, kv_dtype, pool_rows, d_page_table, max_pages,
                     d_seq_lens, B, Tq, H, P, c, interleave, shard_begin, shard_count, sm_scale,
                     lse_base, d_o_part, d_lse_part, d_err, true);
  if (st != DCPMLA_OK) return st;
  if (B == 0) return DCPMLA_OK;
  const int sm = device_sm_count();
  if (sm <= 0) return DCPMLA_ERR_CUDA;
  if (fh_supported(a, sm)) return launch_decode_fh(a, d_workspace, ws_bytes, sm, (cudaStream_t)stream);
  if (tc_supported(a)) return launch_decode_tc(a, d_workspace, ws_bytes, sm, (cudaStream_t)stream);
  return launch_decode_fma(a, d_workspace, ws_bytes, sm, (cudaStream_t)stream);
}

// Fused decode + merge of all c shards.  The bf16 tensor-core kernels merge without
// per-shard outputs (token-major: a merge kernel over every unit of the request; 128-row
// tiles: a merge kernel over the persistent grid's partials, or the last CTA of a
// request's row tile); E4M3 on the tensor cores and the CUDA-core path decode into
// per-shard partials in the workspace and merge them with the LSE-merge kernel (for
// E4M3 that measured faster than merging in the decode's last CTAs: 6.49 against
// 6.73 ms on the FP8 verification batch).
namespace {
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool merge_in_decode(const DecodeArgs& a, int sm) {
  return fh_supported(a, sm) || (tc_supported(a) && !a.fp8);
}

size_t merged_ws(const DecodeArgs& a, int sm, size_t* part_off) {
  if (fh_supported(a, sm)) return fh_workspace_bytes(a, sm);
  if (tc_supported(a) && !a.fp8) return tc_workspace_bytes(a, sm, true);
  const size_t f = align256(tc_supported(a) ? tc_workspace_bytes(a, sm, false) : fma_workspace_bytes(a, sm));
  if (part_off) *part_off = f;
  const size_t rows = (size_t)a.shard_count * a.B * a.R;
  return f + align256(rows * kDL * 4) + rows * 4;
}
}  // namespace

int dcpmla_decode_merged_workspace_size(int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
                                        int32_t kv_dtype, int32_t max_pages, size_t* out) {
  if (!out) return DCPMLA_ERR_INVALID;
  DecodeArgs a;
  const int st = fill_args(a, nullptr, nullptr, nullptr, kv_dtype, 0, nullptr, max_pages, nullptr, B, Tq, H, P,
                           c, 1, 0, c, 1.f, DCPMLA_LSE_E, nullptr, nullptr, nullptr, false);
  if (st != DCPMLA_OK) return st;
  const int sm = device_sm_count();
  if (sm <= 0) return DCPMLA_ERR_CUDA;
  *out = merged_ws(a, sm, nullptr);
  return DCPMLA_OK;
}

int dcpmla_decode_merged(const void* d_q, void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                         int64_t pool_rows, const int32_t* d_page_table, int32_t max_pages,
                         const int32_t* d_seq_lens, int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
                         int32_t interleave, float sm_scale, int32_t lse_base, float* d_o, float* d_lse,
                         void* d_workspace, size_t ws_bytes, int32_t* d_err, void* stream) {
  DecodeArgs a;
  int st = fill_args(a, d_q, pools, scale_pools, kv_dtype, pool_rows, d_page_table, max_pages, d_seq_lens, B,
                     Tq, H, P, c, interleave, 0, c, sm_scale, lse_base, d_o, d_lse, d_err, true);
  if (st != DCPMLA_OK) return st;
  if (B == 0) return DCPMLA_OK;
  const int sm = device_sm_count();
  if (sm <= 0) return DCPMLA_ERR_CUDA;
  size_t part_off = 0;
  const size_t need = merged_ws(a, sm, &part_off);
  if (ws_bytes < need || (need && !d_workspace)) return DCPMLA_ERR_CAPACITY;
  cudaStream_t s = (cudaStream_t)stream;
  if (fh_supported(a, sm)) return launch_decode_fh(a, d_workspace, ws_bytes, sm, s, true);
  if (merge_in_decode(a, sm)) return launch_decode_tc(a, d_workspace, ws_bytes, sm, s, true);
  uint8_t* w = static_cast<uint8_t*>(d_workspace);
  const size_t rows = (size_t)c * B * a.R;
  float* o_part = reinterpret_cast<float*>(w + part_off);
  float* lse_part = reinterpret_cast<float*>(w + part_off + align256(rows * kDL * 4));
  DecodeArgs ap = a;
  ap.o_part = o_part;
  ap.lse_part = lse_part;
  st = tc_supported(ap) ? launch_decode_tc(ap, d_workspace, part_off, sm, s, false)
                        : launch_decode_fma(ap, d_workspace, part_off, sm, s);
  if (st != DCPMLA_OK) return st;
  return dcpmla_lse_merge(o_part, lse_part, c, (int64_t)B * a.R, lse_base, d_o, d_lse, d_err, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode.
//
// For callers that cannot hand the decode a workspace: the split-KV partials
// and arrival counters live in this file-scope device array instead.  Every
// GPU that loads the library reserves it (DCPMLA_NOALLOC_SCRATCH_BYTES) until
// the process exits.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol, so its device address is looked up once per
// device (with that device current) and cached; kernels get that address.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DCPMLA_NOALLOC_SCRATCH_BYTES];

int noalloc_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[256] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DCPMLA_ERR_CUDA;
  if (dev < 0 || dev >= 256) return DCPMLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DCPMLA_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return DCPMLA_OK;
}

}  // namespace

extern "C" int dcpmla_decode_noalloc(const void* d_q, void* const* pools,
                                     float* const* scale_pools, int32_t kv_dtype,
                                     int64_t pool_rows, const int32_t* d_page_table,
                                     int32_t max_pages, const int32_t* d_seq_lens, int32_t B,
                                     int32_t Tq, int32_t H, int32_t P, int32_t c,
                                     int32_t shard_begin, int32_t shard_count, float sm_scale,
                                     int32_t lse_base, float* d_o_part, float* d_lse_part,
                                     int32_t* d_err, void* stream) {
  DecodeArgs a;
  int st = fill_args(a, d_q, pools, scale_pools, kv_dtype, pool_rows, d_page_table, max_pages,
                     d_seq_lens, B, Tq, H, P, c, 1, shard_begin, shard_count, sm_scale, lse_base,
                     d_o_part, d_lse_part, d_err, true);
  if (st != DCPMLA_OK) return st;
  if (B == 0) return DCPMLA_OK;
  const int sm = device_sm_count();
  if (sm <= 0) return DCPMLA_ERR_CUDA;
  if (fma_workspace_bytes(a, sm) > (size_t)DCPMLA_NOALLOC_SCRATCH_BYTES) return DCPMLA_ERR_CAPACITY;
  void* scratch = nullptr;
  st = noalloc_scratch_address(&scratch);
  if (st != DCPMLA_OK) return st;
  return launch_decode_fma(a, scratch, (size_t)DCPMLA_NOALLOC_SCRATCH_BYTES, sm,
                           (cudaStream_t)stream);
}
