// Slot map, KV append (compacting write) and the exact LSE merge.
//
// SGLang "Decode Context Parallelism" docs:
//   Architecture > Virtual KV layout -- owner(v) = v mod c, physical(v) = floor(v/c);
//     a rank keeps only its own positions and compacts them into its pool.
//   MLA decode dataflow -- lse = logsumexp_r(lse_r), o = sum_r exp(lse_r - lse) o_r,
//     in the attention backend's LSE base (e or 2).
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace dcpmla {

int device_sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// ---------------------------------------------------------------------------
// Slot map: (request, position) -> (virtual slot, owner, physical slot)
// ---------------------------------------------------------------------------
__global__ void slot_map_kernel(const int32_t* __restrict__ pt, int32_t n_requests,
                                int32_t max_pages, int64_t num_pages, int32_t c, int32_t I, int32_t P,
                                const int32_t* __restrict__ req, const int64_t* __restrict__ pos,
                                int64_t n, int64_t* vslot, int32_t* owner, int64_t* phys,
                                int32_t* err) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t vp = (int64_t)P * c;
  const int32_t b = req[i];
  const int64_t p = pos[i];
  int64_t v = -1;
  int bad = 0;
  if (b < 0 || b >= n_requests || p < 0 || p / vp >= max_pages) {
    bad = DCPMLA_DERR_POSITION;
  } else {
    const int32_t g = pt[(int64_t)b * max_pages + p / vp];
    if (g < 0 || (int64_t)g >= num_pages)
      bad = DCPMLA_DERR_PAGE;
    else
      v = (int64_t)g * vp + p % vp;
  }
  if (bad) set_err(err, bad);
  if (vslot) vslot[i] = v;
  // runs of I consecutive slots per rank; I = 1 is owner = v mod c, phys = floor(v / c)
  if (owner) owner[i] = bad ? -1 : (int32_t)((v / I) % c);
  if (phys) phys[i] = bad ? -1 : (v / ((int64_t)I * c)) * I + v % I;
}

// ---------------------------------------------------------------------------
// KV append: copy each new row to its owner's pool at its physical slot.
// One thread per 16-byte chunk of a stored row.
// ---------------------------------------------------------------------------
__global__ void kv_append_kernel(ShardPtrs dst, int32_t esize, int64_t pool_rows, int32_t c,
                                 const int32_t* __restrict__ owner,
                                 const int64_t* __restrict__ phys, const uint8_t* __restrict__ ckv,
                                 int64_t ckv_stride_b, const uint8_t* __restrict__ krope,
                                 int64_t krope_stride_b, const float* __restrict__ row_scales,
                                 int64_t n, int32_t* err) {
  const int lat_chunks = kDL * esize / 16;
  const int rope_chunks = kDR * esize / 16;
  const int per_row = lat_chunks + rope_chunks;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * per_row) return;
  const int64_t i = t / per_row;
  const int k = (int)(t % per_row);
  const int32_t r = owner[i];
  if (r == -1) return;
  const int64_t s = phys[i];
  if (r < 0 || r >= c || s < 0 || s >= pool_rows) {
    if (k == 0) set_err(err, DCPMLA_DERR_SLOT);
    return;
  }
  uint8_t* row = (uint8_t*)dst.pool[r] + s * (int64_t)(kDK * esize);
  const uint4* src;
  if (k < lat_chunks)
    src = reinterpret_cast<const uint4*>(ckv + i * ckv_stride_b) + k;
  else
    src = reinterpret_cast<const uint4*>(krope + i * krope_stride_b) + (k - lat_chunks);
  reinterpret_cast<uint4*>(row)[k] = __ldg(src);
  if (k == 0 && row_scales) dst.scale[r][s] = row_scales[i];
}

// ---------------------------------------------------------------------------
// Exact LSE merge over c partials; one 128-thread block per row, 4 dims/thread.
// Base e uses expf/logf and base 2 exp2f/log2f directly, so c = 1 returns the
// input unchanged (weight exp(0) = 1, log(1) = 0).
// ---------------------------------------------------------------------------
template <bool kBase2>
__global__ void __launch_bounds__(128) lse_merge_kernel(const float* __restrict__ o_part,
                                                        const float* __restrict__ lse_part,
                                                        int32_t c, int64_t rows,
                                                        float* __restrict__ o,
                                                        float* __restrict__ lse_out) {
  const int64_t row = blockIdx.x;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int r = 0; r < c; ++r) m = fmaxf(m, __ldg(lse_part + (int64_t)r * rows + row));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (m != -INFINITY) {
    float sum = 0.f;
    for (int r = 0; r < c; ++r) {
      const float x = __ldg(lse_part + (int64_t)r * rows + row);
      sum += kBase2 ? exp2f(x - m) : expf(x - m);
    }
    lse = m + (kBase2 ? log2f(sum) : logf(sum));
    for (int r = 0; r < c; ++r) {
      const float x = __ldg(lse_part + (int64_t)r * rows + row);
      const float w = kBase2 ? exp2f(x - lse) : expf(x - lse);
      if (w == 0.f) continue;
      const float4 v =
          __ldg(reinterpret_cast<const float4*>(o_part + ((int64_t)r * rows + row) * kDL) +
                threadIdx.x);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  reinterpret_cast<float4*>(o + row * kDL)[threadIdx.x] = acc;
  if (lse_out && threadIdx.x == 0) lse_out[row] = lse;
}

}  // namespace dcpmla

using namespace dcpmla;

extern "C" {

int dcpmla_slot_map(const int32_t* d_page_table, int32_t n_requests, int32_t max_pages,
                    int64_t num_pages, int32_t c, int32_t interleave, int32_t P, const int32_t* d_req,
                    const int64_t* d_pos, int64_t n, int64_t* d_vslot, int32_t* d_owner,
                    int64_t* d_phys, int32_t* d_err, void* stream) {
  if (n < 0 || c < 1 || c > DCPMLA_MAX_SHARDS || P < 1 || max_pages < 1 || n_requests < 0 ||
      num_pages < 0)
    return DCPMLA_ERR_INVALID;
  if (interleave < 1 || P % interleave) return DCPMLA_ERR_INVALID;
  if (n == 0) return DCPMLA_OK;
  if (!d_page_table || !d_req || !d_pos) return DCPMLA_ERR_INVALID;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  if (blocks > INT32_MAX) return DCPMLA_ERR_UNSUPPORTED;
  slot_map_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      d_page_table, n_requests, max_pages, num_pages, c, interleave, P, d_req, d_pos, n, d_vslot,
      d_owner, d_phys, d_err);
  return launch_status();
}

int dcpmla_kv_append(void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                     int64_t pool_rows, int32_t c, const int32_t* d_owner, const int64_t* d_phys,
                     const void* d_ckv, int64_t ckv_stride, const void* d_krope,
                     int64_t krope_stride, const float* d_row_scales, int64_t n, int32_t* d_err,
                     void* stream) {
  if (c < 1 || c > DCPMLA_MAX_SHARDS || n < 0 || pool_rows < 0) return DCPMLA_ERR_INVALID;
  if (kv_dtype != DCPMLA_KV_BF16 && kv_dtype != DCPMLA_KV_E4M3) return DCPMLA_ERR_UNSUPPORTED;
  if (n == 0) return DCPMLA_OK;
  if (!pools || !d_owner || !d_phys || !d_ckv || !d_krope) return DCPMLA_ERR_INVALID;
  const int esize = kv_dtype == DCPMLA_KV_BF16 ? 2 : 1;
  const bool fp8 = kv_dtype == DCPMLA_KV_E4M3;
  if (fp8 && (!scale_pools || !d_row_scales)) return DCPMLA_ERR_INVALID;
  if (ckv_stride < kDL || krope_stride < kDR) return DCPMLA_ERR_INVALID;
  if ((ckv_stride * esize) % 16 || (krope_stride * esize) % 16 || !aligned16(d_ckv) ||
      !aligned16(d_krope))
    return DCPMLA_ERR_INVALID;
  ShardPtrs dst{};
  for (int r = 0; r < c; ++r) {
    if (!pools[r] || !aligned16(pools[r])) return DCPMLA_ERR_INVALID;
    dst.pool[r] = pools[r];
    if (fp8) {
      if (!scale_pools[r]) return DCPMLA_ERR_INVALID;
      dst.scale[r] = scale_pools[r];
    }
  }
  const int per_row = kDK * esize / 16;
  const int64_t total = n * per_row;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > INT32_MAX) return DCPMLA_ERR_UNSUPPORTED;
  kv_append_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      dst, esize, pool_rows, c, d_owner, d_phys, (const uint8_t*)d_ckv, ckv_stride * esize,
      (const uint8_t*)d_krope, krope_stride * esize, fp8 ? d_row_scales : nullptr, n, d_err);
  return launch_status();
}

int dcpmla_lse_merge(const float* d_o_part, const float* d_lse_part, int32_t c, int64_t rows,
                     int32_t lse_base, float* d_o, float* d_lse, int32_t* d_err, void* stream) {
  (void)d_err;
  if (c < 1 || rows < 0) return DCPMLA_ERR_INVALID;
  if (lse_base != DCPMLA_LSE_E && lse_base != DCPMLA_LSE_2) return DCPMLA_ERR_INVALID;
  if (rows == 0) return DCPMLA_OK;
  if (!d_o_part || !d_lse_part || !d_o) return DCPMLA_ERR_INVALID;
  if (!aligned16(d_o_part) || !aligned16(d_o)) return DCPMLA_ERR_INVALID;
  if (rows > INT32_MAX) return DCPMLA_ERR_UNSUPPORTED;
  if (lse_base == DCPMLA_LSE_2)
    lse_merge_kernel<true><<<(unsigned)rows, 128, 0, (cudaStream_t)stream>>>(d_o_part, d_lse_part,
                                                                            c, rows, d_o, d_lse);
  else
    lse_merge_kernel<false><<<(unsigned)rows, 128, 0, (cudaStream_t)stream>>>(
        d_o_part, d_lse_part, c, rows, d_o, d_lse);
  return launch_status();
}

}  // extern "C"
