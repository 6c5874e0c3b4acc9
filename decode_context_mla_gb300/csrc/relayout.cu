// Layout moves around the striped cache, and the quantising append.
//
//   relayout  SGLang "Decode Context Parallelism" docs, DCP x PD disaggregation:
//             a DCP-1 prefill cache (dense pages) is copied token by token into
//             the striped decode pools; the plan carries the exact token count, so
//             rows of a partial final page are not copied.
//   gather    same page, Communication backends (extend gathers the cached prefix
//             shards and restores token order); vLLM GLM-5.3 serving post, DCP
//             section (a temporary full-context copy): striped pools -> one
//             contiguous copy per request in token order.
//   HiCache   same page, DCP x HiCache L2: an index list in widened-page slot
//             space keeps the slots this rank owns, mapped to local slots.
//   E4M3 append  per-token amax / 448 scale, codes rounded to nearest-even,
//             written to the owner pool with the scale.
//
// All are HBM- or latency-bound; none uses the tensor cores.
#include <algorithm>

#include "decode.cuh"

using namespace dcpmla;

namespace {

// Where position p of request b lives in the striped pools (owner, physical slot),
// or owner -1 when the page-table entry is outside the pools.
struct Slot {
  int32_t owner;
  int64_t phys;
};
__device__ __forceinline__ Slot striped_slot(const int32_t* vpt_row, int64_t p, int32_t c, int32_t I, int32_t P,
                                             int64_t num_pages) {
  const int64_t vp = (int64_t)P * c;
  const int32_t g = __ldg(vpt_row + p / vp);
  Slot s;
  if (g < 0 || (int64_t)g >= num_pages) {
    s.owner = -1;
    s.phys = -1;
    return s;
  }
  const int64_t v = (int64_t)g * vp + p % vp;
  s.owner = (int32_t)((v / I) % c);
  s.phys = (v / ((int64_t)I * c)) * I + v % I;
  return s;
}

__device__ __forceinline__ int64_t dense_slot(const int32_t* dpt_row, int64_t p, int32_t P, int64_t dense_pages) {
  const int32_t g = __ldg(dpt_row + p / P);
  if (g < 0 || (int64_t)g >= dense_pages) return -1;
  return (int64_t)g * P + p % P;
}

// dir = 0: dense -> striped (relayout); dir = 1: striped -> contiguous (gather).
// Each warp moves kWarpTok tokens per iteration: lanes 0..kWarpTok-1 look up one
// token's source and destination rows, the addresses are broadcast with shuffles,
// and every lane issues all of its 16-byte loads before any store.
constexpr int kWarpTok = 4;

template <int kDir, int kChunks>
__global__ void __launch_bounds__(256) move_rows_kernel(
    const uint8_t* __restrict__ dense, const float* __restrict__ dense_scales, int64_t dense_rows,
    const int32_t* __restrict__ dense_pt, int32_t dense_max_pages, ShardPtrs pools, int64_t pool_rows,
    const int32_t* __restrict__ pt, int32_t max_pages, const int32_t* __restrict__ lens, int32_t P, int32_t c,
    int32_t I, bool fp8, uint8_t* __restrict__ out, float* __restrict__ out_scales, int64_t out_cap,
    int32_t* err) {
  constexpr int kRowBytes = kChunks * 16;
  constexpr int kPer = (kWarpTok * kChunks + 31) / 32;   // chunks per lane per iteration
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t L = __ldg(lens + b);
  const int64_t limit = kDir == 0 ? min((int64_t)dense_max_pages * P, (int64_t)max_pages * P * c)
                                  : min(out_cap, (int64_t)max_pages * P * c);
  if (L < 0 || L > limit) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_err(err, DCPMLA_DERR_LENGTH);
    return;
  }
  const int32_t* vpt_row = pt + (int64_t)b * max_pages;
  const int32_t* dpt_row = kDir == 0 ? dense_pt + (int64_t)b * dense_max_pages : nullptr;
  const int64_t num_pages = pool_rows / P, dense_pages = dense_rows / P;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kWarpTok; t0 < L;
       t0 += warps * kWarpTok) {
    // lane k < kWarpTok resolves token t0 + k: source and destination row pointers
    const uint8_t* src = nullptr;
    uint8_t* dst = nullptr;
    const float* ssrc = nullptr;
    float* sdst = nullptr;
    if (lane < kWarpTok && t0 + lane < L) {
      const int64_t p = t0 + lane;
      const Slot sl = striped_slot(vpt_row, p, c, I, P, num_pages);
      int64_t d = 0;
      if (kDir == 0) d = dense_slot(dpt_row, p, P, dense_pages);
      if (sl.owner < 0 || d < 0) {
        set_err(err, DCPMLA_DERR_PAGE);
      } else if (kDir == 0) {
        src = dense + d * kRowBytes;
        dst = static_cast<uint8_t*>(pools.pool[sl.owner]) + sl.phys * kRowBytes;
        if (fp8) {
          ssrc = dense_scales + d;
          sdst = pools.scale[sl.owner] + sl.phys;
        }
      } else {
        src = static_cast<const uint8_t*>(pools.pool[sl.owner]) + sl.phys * kRowBytes;
        dst = out + ((int64_t)b * out_cap + p) * kRowBytes;
        if (fp8) {
          ssrc = pools.scale[sl.owner] + sl.phys;
          sdst = out_scales + (int64_t)b * out_cap + p;
        }
      }
    }
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = k * 32 + lane;                      // (token, chunk) pair of this lane
      const int tk = e / kChunks, ch = e % kChunks;
      const uint8_t* s = reinterpret_cast<const uint8_t*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(src), tk < kWarpTok ? tk : 0));
      v[k] = (e < kWarpTok * kChunks && s) ? __ldcs(reinterpret_cast<const uint4*>(s) + ch) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = k * 32 + lane;
      const int tk = e / kChunks, ch = e % kChunks;
      uint8_t* d = reinterpret_cast<uint8_t*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), tk < kWarpTok ? tk : 0));
      if (e < kWarpTok * kChunks && d) reinterpret_cast<uint4*>(d)[ch] = v[k];
    }
    if (fp8 && lane < kWarpTok && ssrc) *sdst = __ldcs(ssrc);
  }
}

// ---------------------------------------------------------------------------
// E4M3 quantising append: one warp per new token row (576 bf16 values).
// Lane l holds latent values [16l, 16l + 16); lanes 0-3 also rope values
// [16l, 16l + 16).  In float32: amax = max |x|, scale = amax / 448 (IEEE
// division), code = E4M3(clamp(x / scale, +-448)) rounded to nearest-even; a row of
// zeros stores scale 0 and zero codes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unpack_bf16x8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Whether v lies within one binary32 step of a point where rounding to E4M3 changes direction
// (a midpoint between two E4M3 values): below 2^-6 E4M3 steps by 2^-9, from there on it keeps
// three fraction bits, and below 2^-10 everything rounds to zero.
__device__ __forceinline__ bool near_e4m3_midpoint(float v) {
  const uint32_t u = __float_as_uint(v) & 0x7FFFFFFFu;
  const int e = (int)(u >> 23) - 127;
  if (e < -10) return false;
  const int drop = e >= -6 ? 20 : 14 - e;                  // binary32 bits below the E4M3 step
  const uint32_t sig = (u & 0x7FFFFFu) | 0x800000u;
  const uint32_t low = sig & ((1u << drop) - 1u), half = 1u << (drop - 1);
  return low + 1u >= half && low <= half + 1u;
}

// x / scale for the E4M3 code, with the code of the correctly rounded quotient.  Markstein's
// correction of a reciprocal product (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34, 1990): with y = RN(1 / b), q = RN(a y)
// lies within two steps of a / b, and q + RN(a - b q) y (one FMA) within 2.5e-7 of a step, so
// its rounding is RN(a / b) or a neighbour.  Two neighbouring binary32 values round to
// different E4M3 codes only if one of them is an E4M3 midpoint, so where the result is within a
// step of one the IEEE division decides.  `fast` is false when the reciprocal of the scale
// would overflow (a subnormal scale); the IEEE division serves there too.
__device__ __forceinline__ float div_scale(float a, float b, float y, bool fast) {
  if (!fast) return __fdiv_rn(a, b);
  const float q = __fmul_rn(a, y);
  const float r = __fmaf_rn(-q, b, a);
  const float qc = __fmaf_rn(r, y, q);
  return near_e4m3_midpoint(qc) ? __fdiv_rn(a, b) : qc;
}

__global__ void __launch_bounds__(256) append_e4m3_kernel(
    ShardPtrs dst, int64_t pool_rows, int32_t c, const int32_t* __restrict__ owner,
    const int64_t* __restrict__ phys, const uint8_t* __restrict__ ckv, int64_t ckv_stride_b,
    const uint8_t* __restrict__ krope, int64_t krope_stride_b, int64_t n, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= n) return;
  // the row's values (16 latent and 2 rope dims a lane) and its destination, all in flight at once
  const uint4* src = reinterpret_cast<const uint4*>(ckv + row * ckv_stride_b) + 2 * lane;
  const uint4 l0 = __ldg(src), l1 = __ldg(src + 1);
  const uint32_t rp = __ldg(reinterpret_cast<const uint32_t*>(krope + row * krope_stride_b) + lane);
  const int32_t r = __ldg(owner + row);
  const int64_t s = __ldg(phys + row);
  if (r < 0 || r >= c || s < 0 || s >= pool_rows) {   // uniform across the warp
    if (lane == 0) set_err(err, DCPMLA_DERR_SLOT);
    return;
  }
  float lat[16];
  {
    float a[8], b[8];
    unpack_bf16x8(l0, a);
    unpack_bf16x8(l1, b);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lat[i] = a[i];
      lat[8 + i] = b[i];
    }
  }
  const float rope0 = __uint_as_float(rp << 16), rope1 = __uint_as_float(rp & 0xFFFF0000u);
  float amax = fmaxf(fabsf(rope0), fabsf(rope1));
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(lat[i]));
  // non-negative floats order like their bit patterns
  amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
  const float scale = __fdiv_rn(amax, 448.f);
  const bool fast = scale >= 1.17549435e-38f;   // a normal scale: its reciprocal is finite
  const float ys = fast ? __frcp_rn(scale) : 0.f;
  uint8_t* prow = static_cast<uint8_t*>(dst.pool[r]) + s * kDK;
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = 4 * k;
    if (scale > 0.f) {
      float y[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) y[m] = fminf(fmaxf(div_scale(lat[i + m], scale, ys, fast), -448.f), 448.f);
      w[k] = (uint32_t)e4m3x2(y[0], y[1]) | ((uint32_t)e4m3x2(y[2], y[3]) << 16);
    } else {
      w[k] = 0u;
    }
  }
  reinterpret_cast<uint4*>(prow)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
  uint16_t rw = 0;
  if (scale > 0.f)
    rw = e4m3x2(fminf(fmaxf(div_scale(rope0, scale, ys, fast), -448.f), 448.f),
                fminf(fmaxf(div_scale(rope1, scale, ys, fast), -448.f), 448.f));
  reinterpret_cast<uint16_t*>(prow + kDL)[lane] = rw;
  if (lane == 0) dst.scale[r][s] = scale;
}

// ---------------------------------------------------------------------------
// HiCache index filter: order-preserving compaction in one pass (a chained scan with
// decoupled look-back: Merrill and Garland, "Single-pass Parallel Prefix Scan with
// Decoupled Look-back", NVIDIA technical report NVR-2016-002).
// ---------------------------------------------------------------------------
constexpr int kFilterWarps = 8;
constexpr int kFilterRounds = 16;                                  // 32-index rounds per warp
constexpr int kFilterBlock = kFilterWarps * kFilterRounds * 32;    // 4096 indices per block
// A block's status word: flag in bits 62-63 (0 not yet, 1 its own count, 2 the inclusive
// count of every block up to it), the count in bits 0-61.
constexpr uint64_t kStatAgg = 1ull << 62, kStatInc = 2ull << 62, kStatVal = (1ull << 62) - 1;
constexpr long long kLookbackSpins = 1ll << 22;                     // per predecessor window

// owner and local slot of widened-page slot i (i >= 0); 32-bit division when i fits, and a
// shift and a mask when c is a power of two (cs = log2 c, else -1)
__device__ __forceinline__ void owner_local(int64_t i, int32_t c, int32_t cs, int32_t I, int32_t& own, int64_t& loc) {
  if ((uint64_t)i <= 0xFFFFFFFFull) {
    const uint32_t u = (uint32_t)i, q = I == 1 ? u : u / (uint32_t)I;
    const uint32_t w = cs >= 0 ? q >> cs : q / (uint32_t)c;
    own = (int32_t)(cs >= 0 ? q & (uint32_t)(c - 1) : q - w * (uint32_t)c);
    loc = (int64_t)w * I + (u - q * (uint32_t)I);
  } else {
    const int64_t q = i / I, w = q / c;
    own = (int32_t)(q - w * c);
    loc = w * I + (i - q * I);
  }
}
__device__ __forceinline__ bool owned(int64_t i, int32_t c, int32_t cs, int32_t I, int32_t rank) {
  if (i < 0) return false;
  int32_t o;
  int64_t l;
  owner_local(i, c, cs, I, o, l);
  return o == rank;
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}

// One pass over the list.  Blocks take tiles in the order they start (a ticket), so a block
// waits only for blocks already running.  Each warp takes 512 consecutive indices (16 rounds
// of 32, in order); the block publishes its count, then warp 0 looks back over the status
// words of the 32 tiles before it at a time, summing counts until a tile that already holds
// its inclusive prefix, publishes its own inclusive prefix and the block writes its kept
// slots there.  A look-back that waits past its limit sets DCPMLA_DERR_TIMEOUT (and the
// outputs are invalid); it never blocks for good.
__global__ void __launch_bounds__(kFilterWarps * 32, 4) filter_onepass_kernel(
    const int64_t* __restrict__ idx, int64_t n, int32_t c, int32_t cs, int32_t I, int32_t rank, uint64_t* status,
    unsigned int* ticket, int64_t* __restrict__ out, int64_t* count, int32_t* err) {
  __shared__ uint32_t warp_n[kFilterWarps];
  __shared__ uint64_t prefix_s;
  __shared__ int tile_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) tile_s = (int)atomicAdd(ticket, 1u);
  __syncthreads();
  const int tile = tile_s;
  const int64_t base = (int64_t)tile * kFilterBlock + warp * (kFilterRounds * 32);
  // the values are read again (from L1) for the kept entries once the prefix is known, so
  // none is held across the look-back
  int64_t v[kFilterRounds];
#pragma unroll
  for (int k = 0; k < kFilterRounds; ++k) {
    const int64_t i = base + k * 32 + lane;
    v[k] = i < n ? __ldg(idx + i) : -1;   // past the list: dropped, not reported
  }
  uint32_t keep = 0, mine = 0;   // bit k: round k's index is kept
  bool neg = false;
#pragma unroll
  for (int k = 0; k < kFilterRounds; ++k) {
    neg |= v[k] < 0 && base + k * 32 + lane < n;
    const bool kp = owned(v[k], c, cs, I, rank);
    keep |= kp ? 1u << k : 0u;
    mine += __popc(__ballot_sync(0xffffffffu, kp));
  }
  if (__any_sync(0xffffffffu, neg) && lane == 0) set_err(err, DCPMLA_DERR_POSITION);
  if (lane == 0) warp_n[warp] = mine;
  __syncthreads();
  if (warp == 0) {
    uint32_t total = 0;
#pragma unroll
    for (int w = 0; w < kFilterWarps; ++w) total += warp_n[w];
    uint64_t prefix = 0;
    if (tile == 0) {
      if (lane == 0) st_release_u64(status, kStatInc | total);
    } else {
      if (lane == 0) st_release_u64(status + tile, kStatAgg | total);
      // look back in windows of 32 predecessors (lane l: tile - 1 - l), nearest first
      int j = tile - 1;
      bool timed_out = false;
      while (j >= 0) {
        const int t = j - lane;
        uint64_t sw = t >= 0 ? ld_acquire_u64(status + t) : kStatInc;
        long long spins = 0;
        while (!__all_sync(0xffffffffu, (sw >> 62) != 0)) {
          if (++spins > kLookbackSpins) {
            timed_out = true;
            break;
          }
          if ((sw >> 62) == 0) sw = ld_acquire_u64(status + t);
        }
        if (timed_out) break;
        const uint32_t inc = __ballot_sync(0xffffffffu, (sw >> 62) == 2);
        const int first = inc ? __ffs(inc) - 1 : 32;            // the nearest inclusive tile
        uint64_t add = lane <= first ? (sw & kStatVal) : 0;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) add += __shfl_xor_sync(0xffffffffu, add, d);
        prefix += add;
        if (inc) break;
        j -= 32;
      }
      if (timed_out && lane == 0) set_err(err, DCPMLA_DERR_TIMEOUT);
      if (lane == 0) st_release_u64(status + tile, kStatInc | (prefix + total));
    }
    if (lane == 0) {
      prefix_s = prefix;
      if ((int64_t)(tile + 1) * kFilterBlock >= n) *count = (int64_t)(prefix + total);   // the last tile
    }
  }
  __syncthreads();
  uint64_t pos = prefix_s;
  for (int w = 0; w < warp; ++w) pos += warp_n[w];
#pragma unroll
  for (int k = 0; k < kFilterRounds; ++k) {
    const bool kp = (keep >> k) & 1u;
    const uint32_t bal = __ballot_sync(0xffffffffu, kp);
    if (kp) {
      int32_t o;
      int64_t l;
      owner_local(__ldg(idx + base + k * 32 + lane), c, cs, I, o, l);
      out[pos + __popc(bal & ((1u << lane) - 1u))] = l;
    }
    pos += __popc(bal);
  }
}

int check_pools(void* const* pools, float* const* scale_pools, int32_t c, bool fp8, ShardPtrs& sp) {
  sp = ShardPtrs{};
  for (int r = 0; r < c; ++r) {
    if (!pools[r] || !aligned16(pools[r])) return DCPMLA_ERR_INVALID;
    sp.pool[r] = pools[r];
    if (fp8) {
      if (!scale_pools || !scale_pools[r]) return DCPMLA_ERR_INVALID;
      sp.scale[r] = scale_pools[r];
    }
  }
  return DCPMLA_OK;
}

// Blocks per request: enough warps for the longest request, at most one wave of
// 8-warp blocks over the SMs for all requests together.
int move_grid_x(int32_t max_pages, int32_t P, int32_t c, int32_t B) {
  const int64_t tokens = (int64_t)max_pages * P * c;
  const int64_t blocks = (tokens + 8 * kWarpTok - 1) / (8 * kWarpTok);
  const int64_t wave = std::max<int64_t>(1, (int64_t)device_sm_count() * 8 / std::max(B, 1));
  return (int)std::min<int64_t>(std::max<int64_t>(blocks, 1), std::max<int64_t>(wave, 1));
}

}  // namespace

extern "C" {

int dcpmla_relayout_dense_to_striped(const void* d_dense, const float* d_dense_scales, int64_t dense_rows,
                                     const int32_t* d_dense_page_table, int32_t dense_max_pages,
                                     void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                                     int64_t pool_rows, const int32_t* d_page_table, int32_t max_pages,
                                     const int32_t* d_seq_lens, int32_t B, int32_t P, int32_t c,
                                     int32_t interleave, int32_t* d_err, void* stream) {
  if (B < 0 || P < 1 || c < 1 || c > DCPMLA_MAX_SHARDS || max_pages < 1 || dense_max_pages < 1 ||
      pool_rows < 0 || dense_rows < 0 || interleave < 1 || P % interleave)
    return DCPMLA_ERR_INVALID;
  if (kv_dtype != DCPMLA_KV_BF16 && kv_dtype != DCPMLA_KV_E4M3) return DCPMLA_ERR_UNSUPPORTED;
  if (B == 0) return DCPMLA_OK;
  const bool fp8 = kv_dtype == DCPMLA_KV_E4M3;
  if (!d_dense || !aligned16(d_dense) || !pools || !d_dense_page_table || !d_page_table || !d_seq_lens)
    return DCPMLA_ERR_INVALID;
  if (fp8 && !d_dense_scales) return DCPMLA_ERR_INVALID;
  ShardPtrs sp;
  const int rc = check_pools(pools, scale_pools, c, fp8, sp);
  if (rc != DCPMLA_OK) return rc;
  if (B > 65535) return DCPMLA_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)move_grid_x(max_pages, P, c, B), (unsigned)B);
  if (fp8)
    move_rows_kernel<0, kDK / 16><<<grid, 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(d_dense), d_dense_scales, dense_rows, d_dense_page_table, dense_max_pages, sp,
        pool_rows, d_page_table, max_pages, d_seq_lens, P, c, interleave, true, nullptr, nullptr, 0, d_err);
  else
    move_rows_kernel<0, 2 * kDK / 16><<<grid, 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(d_dense), nullptr, dense_rows, d_dense_page_table, dense_max_pages, sp,
        pool_rows, d_page_table, max_pages, d_seq_lens, P, c, interleave, false, nullptr, nullptr, 0, d_err);
  return launch_status();
}

int dcpmla_gather_unstriped(void* const* pools, float* const* scale_pools, int32_t kv_dtype, int64_t pool_rows,
                            const int32_t* d_page_table, int32_t max_pages, const int32_t* d_seq_lens, int32_t B,
                            int32_t P, int32_t c, int32_t interleave, void* d_out, float* d_out_scales,
                            int64_t out_capacity, int32_t* d_err, void* stream) {
  if (B < 0 || P < 1 || c < 1 || c > DCPMLA_MAX_SHARDS || max_pages < 1 || pool_rows < 0 || out_capacity < 0 ||
      interleave < 1 || P % interleave)
    return DCPMLA_ERR_INVALID;
  if (kv_dtype != DCPMLA_KV_BF16 && kv_dtype != DCPMLA_KV_E4M3) return DCPMLA_ERR_UNSUPPORTED;
  if (B == 0) return DCPMLA_OK;
  const bool fp8 = kv_dtype == DCPMLA_KV_E4M3;
  if (!d_out || !aligned16(d_out) || !pools || !d_page_table || !d_seq_lens) return DCPMLA_ERR_INVALID;
  if (fp8 && !d_out_scales) return DCPMLA_ERR_INVALID;
  ShardPtrs sp;
  const int rc = check_pools(pools, scale_pools, c, fp8, sp);
  if (rc != DCPMLA_OK) return rc;
  if (B > 65535) return DCPMLA_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)move_grid_x(max_pages, P, c, B), (unsigned)B);
  if (fp8)
    move_rows_kernel<1, kDK / 16><<<grid, 256, 0, (cudaStream_t)stream>>>(
        nullptr, nullptr, 0, nullptr, 1, sp, pool_rows, d_page_table, max_pages, d_seq_lens, P, c, interleave,
        true, static_cast<uint8_t*>(d_out), d_out_scales, out_capacity, d_err);
  else
    move_rows_kernel<1, 2 * kDK / 16><<<grid, 256, 0, (cudaStream_t)stream>>>(
        nullptr, nullptr, 0, nullptr, 1, sp, pool_rows, d_page_table, max_pages, d_seq_lens, P, c, interleave,
        false, static_cast<uint8_t*>(d_out), nullptr, out_capacity, d_err);
  return launch_status();
}

int dcpmla_kv_append_e4m3(void* const* pools, float* const* scale_pools, int64_t pool_rows, int32_t c,
                          const int32_t* d_owner, const int64_t* d_phys, const void* d_ckv, int64_t ckv_stride,
                          const void* d_krope, int64_t krope_stride, int64_t n, int32_t* d_err, void* stream) {
  if (c < 1 || c > DCPMLA_MAX_SHARDS || n < 0 || pool_rows < 0) return DCPMLA_ERR_INVALID;
  if (n == 0) return DCPMLA_OK;
  if (!pools || !scale_pools || !d_owner || !d_phys || !d_ckv || !d_krope) return DCPMLA_ERR_INVALID;
  if (!aligned16(d_ckv) || !aligned16(d_krope) || ckv_stride < kDL || krope_stride < kDR ||
      (ckv_stride * 2) % 16 || (krope_stride * 2) % 16)
    return DCPMLA_ERR_INVALID;
  ShardPtrs sp;
  const int rc = check_pools(pools, scale_pools, c, true, sp);
  if (rc != DCPMLA_OK) return rc;
  const int64_t blocks = (n * 32 + 255) / 256;
  if (blocks > INT32_MAX) return DCPMLA_ERR_UNSUPPORTED;
  append_e4m3_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      sp, pool_rows, c, d_owner, d_phys, static_cast<const uint8_t*>(d_ckv), ckv_stride * 2,
      static_cast<const uint8_t*>(d_krope), krope_stride * 2, n, d_err);
  return launch_status();
}

int dcpmla_hicache_filter_workspace_size(int64_t n, size_t* out) {
  if (n < 0 || !out) return DCPMLA_ERR_INVALID;
  *out = (size_t)((n + kFilterBlock - 1) / kFilterBlock + 1) * 8;   // status words and the ticket
  return DCPMLA_OK;
}

int dcpmla_hicache_filter(const int64_t* d_idx, int64_t n, int32_t c, int32_t interleave, int32_t rank,
                          int64_t* d_out, int64_t* d_count, void* d_workspace, size_t ws_bytes, int32_t* d_err,
                          void* stream) {
  if (n < 0 || c < 1 || interleave < 1 || rank < 0 || rank >= c || !d_count) return DCPMLA_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  if (n == 0) return cudaMemsetAsync(d_count, 0, sizeof(int64_t), st) == cudaSuccess ? DCPMLA_OK : DCPMLA_ERR_CUDA;
  if (!d_idx || !d_out) return DCPMLA_ERR_INVALID;
  const int64_t nb = (n + kFilterBlock - 1) / kFilterBlock;
  if ((size_t)(nb + 1) * 8 > ws_bytes || !d_workspace) return DCPMLA_ERR_CAPACITY;
  if (nb > INT32_MAX || n > (int64_t)UINT32_MAX) return DCPMLA_ERR_UNSUPPORTED;
  uint64_t* status = static_cast<uint64_t*>(d_workspace);
  unsigned int* ticket = reinterpret_cast<unsigned int*>(status + nb);
  if (cudaMemsetAsync(d_workspace, 0, (size_t)(nb + 1) * 8, st) != cudaSuccess) return DCPMLA_ERR_CUDA;
  const int32_t cs = (c & (c - 1)) == 0 ? __builtin_ctz((unsigned)c) : -1;
  filter_onepass_kernel<<<(unsigned)nb, kFilterWarps * 32, 0, st>>>(d_idx, n, c, cs, interleave, rank, status,
                                                                    ticket, d_out, d_count, d_err);
  return launch_status();
}

}  // extern "C"
