// Shard-local absorbed-MLA decode on the 5th-generation tensor cores
// (tcgen05 MMA with TMEM accumulators, TMA tile loads), for shapes whose
// query rows (heads x query tokens) form a real M dimension of 128.
//
// SGLang "Decode Context Parallelism" docs, MLA decode dataflow: each shard
// returns its locally normalised o_r and lse_r; DCP x speculative decoding:
// the causal test uses global positions (shard-local token j of shard r is
// position j*c + r).  vLLM GLM-5.3 serving post, footnote arithmetic: scores
// over the 576-d key, values over the 512-d latent.
//
// One CTA = (request b, shard r, KV split, 128 query rows, one half of the
// 512 value dims).  The two halves of a row tile are adjacent CTAs that read
// the same KV tiles (the second read hits L2); each computes the full scores
// (the 128 x 512 fp32 output accumulator alone would fill all of TMEM).
//
//   warp 0     TMA producer: Q dims 256..575 once, then 64-token KV tiles
//              (9 column chunks of 64 bf16, 128-byte swizzle) into 2 stages.
//   warp 1     allocates TMEM; one thread issues the MMAs:
//                S  = Q K^T   (M 128, N 64, K 576; Q dims 0..255 from TMEM)
//                O += P V     (M 128, N 256, K 64;  P from TMEM, V MN-major;
//                              P as a bf16 hi + lo pair, so two MMAs per k-step)
//   warps 2-5  softmax: one query row per thread; online softmax in base 2
//              with a lazily updated reference max (O is rescaled only when a
//              tile's max exceeds the reference by more than 8), P written
//              back to TMEM as bf16 hi/lo; epilogue normalises O and writes it.
//
// TMEM columns: O [0,256), S/P double buffer [256,384), Q dims 0..255 [384,512).
// Every mbarrier wait is bounded; a timeout sets DCPMLA_DERR_TIMEOUT, all
// roles drain, TMEM is freed and the CTA returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "decode.cuh"
#include "sm100.cuh"

namespace dcpmla {
namespace {

using namespace sm100;

constexpr int kMaxTcShards = 16;
constexpr int kRows = 128;
constexpr int kTileTok = 64;
constexpr int kChunks = 9;                           // 576 / 64
constexpr int kChunkBytes = kTileTok * 128;          // 64 tokens x 128 B
constexpr int kStageBytes = kChunks * kChunkBytes;   // 72 KB
constexpr int kStages = 2;
constexpr int kQLoChunks = 4;                        // Q dims 0..255 in TMEM
constexpr int kQHiChunks = kChunks - kQLoChunks;     // Q dims 256..575 in SMEM
constexpr int kQHiBytes = kQHiChunks * kRows * 128;  // 80 KB
constexpr int kThreads = 192;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384, kTmemCols = 512;
constexpr size_t kSmemBytes = 1024 + kQHiBytes + kStages * kStageBytes;
constexpr long long kWaitCycles = 2000000000LL;     // about one second

struct TcParams {
  CUtensorMap tm_q;                   // Q as [B*R, 576] bf16, box {64, 128}
  CUtensorMap tm_kv[kMaxTcShards];    // pool (shard_begin + i) as [pool_rows, 576], box {64, box_rows}
  DecodeArgs a;
  int32_t box_rows;                   // rows per TMA box: min(P, 64)
  int32_t num_splits, chunk, row_tiles;
  float* ws_o;
  float* ws_lse;
  uint32_t* ws_cnt;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half)
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ TcParams p) {
  const DecodeArgs& a = p.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kQHiBytes;
  __shared__ uint64_t bar_kv_full[kStages], bar_kv_empty[kStages], bar_s_full[2], bar_p_full[2];
  __shared__ uint64_t bar_q_full, bar_o, bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s, bad_s, last_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vh = blockIdx.x & 1, split = blockIdx.x >> 1, rt = blockIdx.y, bz = blockIdx.z;
  const int b = bz / a.shard_count, sr = bz % a.shard_count, r = a.shard_begin + sr;
  const int L = a.seq_lens[b];
  const int64_t R = a.R;
  const int32_t* pt_row = a.pt + (int64_t)b * a.max_pages;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bar_s_full[s]), 1);
      mbar_init(smem_u32(&bar_p_full[s]), 128);
    }
    mbar_init(smem_u32(&bar_q_full), 128 + 1);
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_s = 0;
    bad_s = 0;
    last_s = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  // Range of this split and validation of every page the request uses.
  int j0 = 0, j1 = 0;
  if (L < a.Tq || (int64_t)L > (int64_t)a.max_pages * a.P * a.c) {
    if (tid == 0) atomicOr(&bad_s, DCPMLA_DERR_LENGTH);
  } else {
    const int n = L > r ? (L - r + a.c - 1) / a.c : 0;
    j0 = min(split * p.chunk, n);
    j1 = min(n, j0 + p.chunk);
    const int npages = (int)(((int64_t)L + (int64_t)a.P * a.c - 1) / ((int64_t)a.P * a.c));
    for (int pg = tid; pg < npages; pg += kThreads) {
      const int32_t g = pt_row[pg];
      if (g < 0 || (int64_t)g >= a.num_pages) atomicOr(&bad_s, DCPMLA_DERR_PAGE);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (bad_s) {
    if (tid == 0) set_err(a.err, bad_s);
    j1 = j0;
  }
  const int ntiles = (j1 - j0 + kTileTok - 1) / kTileTok;
  volatile int* abort_flag = &abort_s;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0 && ntiles > 0) {
      const CUtensorMap* kvmap = &p.tm_kv[sr];
      prefetch_tmap(kvmap);
      const uint32_t qb = smem_u32(&bar_q_full);
      mbar_arrive_expect_tx(qb, kQHiBytes);
      for (int c = 0; c < kQHiChunks; ++c)
        tma_load_2d(smem_u32(sQ + c * kRows * 128), &p.tm_q, (kQLoChunks + c) * 64,
                    (int)(b * R + rt * kRows), qb);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i & 1;
        if (i >= kStages && !wait_bar(smem_u32(&bar_kv_empty[st]), ((i >> 1) - 1) & 1, abort_flag))
          break;
        const int t0 = j0 + i * kTileTok;
        const int ntok = min(kTileTok, j1 - t0);
        const int box = p.box_rows;
        const int nbox = box >= kTileTok ? 1 : (ntok + box - 1) / box;
        const uint32_t full = smem_u32(&bar_kv_full[st]);
        mbar_arrive_expect_tx(full, (uint32_t)(nbox * box * 128 * kChunks));
        for (int pb = 0; pb < nbox; ++pb) {
          const int tok = t0 + pb * box;
          const int64_t g = pt_row[tok / a.P];
          const int y = (int)(g * a.P + (tok % a.P));
          const uint32_t dst = smem_u32(sKV + st * kStageBytes + pb * box * 128);
          for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kChunkBytes, kvmap, c * 64, y, full);
        }
        issued = i + 1;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        for (int i = max(0, issued - kStages); i < issued; ++i) {
          const long long t0 = clock64();
          while (!mbar_try_wait(smem_u32(&bar_kv_full[i & 1]), (i >> 1) & 1) &&
                 clock64() - t0 < kWaitCycles / 8) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0 && ntiles > 0) {
      const uint32_t idesc_qk = idesc_bf16(kRows, kTileTok, false, false);
      const uint32_t idesc_pv = idesc_bf16(kRows, 256, false, true);
      const uint32_t sq = smem_u32(sQ), skv = smem_u32(sKV);
      bool ok = wait_bar(smem_u32(&bar_q_full), 0, abort_flag);
      tc_fence_after();
      for (int i = 0; ok && i <= ntiles; ++i) {
        if (i < ntiles) {
          const int st = i & 1, sb = i & 1;
          if (!wait_bar(smem_u32(&bar_kv_full[st]), (i >> 1) & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + sb * kTileTok;
          const uint32_t kbase = skv + st * kStageBytes;
          for (int c = 0; c < kChunks; ++c)
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = desc_sw128(kbase + c * kChunkBytes + k * 32, 16, 1024);
              const uint32_t acc = (c | k) != 0;
              if (c < kQLoChunks)
                mma_ts(d, tmem + kColQ + c * 32 + k * 8, bd, idesc_qk, acc);
              else
                mma_ss(d, desc_sw128(sq + (c - kQLoChunks) * kRows * 128 + k * 32, 16, 1024), bd,
                       idesc_qk, acc);
            }
          mma_commit(smem_u32(&bar_s_full[sb]));
        }
        if (i >= 1) {
          const int pi = i - 1, st = pi & 1, sb = pi & 1;
          if (!wait_bar(smem_u32(&bar_p_full[sb]), (pi >> 1) & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t vbase = skv + st * kStageBytes + vh * 4 * kChunkBytes;
          for (int k = 0; k < 8; ++k) {          // k < 4: P_hi, k >= 4: P_lo, same V rows
            const uint64_t bd = desc_sw128(vbase + (k & 3) * 2048, kChunkBytes, 1024);
            mma_ts(tmem + kColO, tmem + kColS + sb * kTileTok + k * 8, bd, idesc_pv,
                   (pi > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&bar_kv_empty[st]));
          mma_commit(smem_u32(&bar_o));
        }
      }
      // drain: every MMA issued above completes before TMEM is released
      mma_commit(smem_u32(&bar_drain));
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&bar_drain), 0) && clock64() - t0 < kWaitCycles) {
      }
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int64_t grow = (int64_t)rt * kRows + row;          // row within the request
    const int qpos = L - a.Tq + (int)(grow / a.H);
    const float qscale = a.sm_scale * kLog2e;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    if (ntiles > 0) {
      // Q dims 0..255 of this row into TMEM as packed bf16 pairs
      const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * R + grow) * kDK);
      for (int c16 = 0; c16 < 8; ++c16) {
        uint32_t rr[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 u = __ldg(qsrc + c16 * 4 + v);
          rr[v * 4 + 0] = u.x; rr[v * 4 + 1] = u.y; rr[v * 4 + 2] = u.z; rr[v * 4 + 3] = u.w;
        }
        tmem_st16(tmem + lane_off + kColQ + c16 * 16, rr);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_q_full));
    }
    for (int i = 0; i < ntiles; ++i) {
      const int sb = i & 1;
      const int t0 = j0 + i * kTileTok;
      const int ntok = min(kTileTok, j1 - t0);
      ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bar_s_full[sb]), (i >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float x[kTileTok];
      {
        uint32_t u[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tmem_ld16(tmem + lane_off + kColS + sb * kTileTok + q * 16, u);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) x[q * 16 + k] = __uint_as_float(u[k]);
        }
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int k = 0; k < kTileTok; ++k) {
        const bool vis = (k < ntok) && ((t0 + k) * a.c + r <= qpos);
        x[k] = vis ? x[k] * qscale : -INFINITY;
        tmax = fmaxf(tmax, x[k]);
      }
      // Lazy reference max: move it only when this tile's max exceeds it by more
      // than 8 (so every weight 2^(x - m_ref) stays <= 256).  Rows that move it
      // after O holds data rescale O; the TMEM traffic is done warp-wide.
      const bool move = tmax > m_ref + 8.f;
      const bool rescale_me = move && m_ref != -INFINITY;
      if (__any_sync(0xffffffffu, rescale_me)) {
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bar_o), (i - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const float alpha = rescale_me ? exp2f(m_ref - tmax) : 1.f;
        for (int q = 0; q < 16; ++q) {
          uint32_t u[16];
          tmem_ld16(tmem + lane_off + kColO + q * 16, u);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
          tmem_st16(tmem + lane_off + kColO + q * 16, u);
        }
        l *= alpha;
      }
      if (move) m_ref = tmax;
      const float mr = m_ref == -INFINITY ? 0.f : m_ref;    // every x is -inf then
      // P goes to the MMA as a bf16 pair P = hi + lo (hi = bf16(p), lo = bf16(p - hi)):
      // one bf16 rounding of the weights alone would cost ~1e-3 relative error in O.
      float ps = 0.f;
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int k = 0; k < kTileTok; k += 2) {
        const float p0 = exp2f(x[k] - mr);
        const float p1 = exp2f(x[k + 1] - mr);
        ps += p0 + p1;
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        const float2 hf = __bfloat1622float2(h);
        hi[k >> 1] = *reinterpret_cast<const uint32_t*>(&h);
        lo[k >> 1] = pack_bf16(p0 - hf.x, p1 - hf.y);
      }
      l += ps;
      const uint32_t pcol = tmem + lane_off + kColS + sb * kTileTok;
      tmem_st16(pcol, *reinterpret_cast<uint32_t(*)[16]>(&hi[0]));
      tmem_st16(pcol + 16, *reinterpret_cast<uint32_t(*)[16]>(&hi[16]));
      tmem_st16(pcol + 32, *reinterpret_cast<uint32_t(*)[16]>(&lo[0]));
      tmem_st16(pcol + 48, *reinterpret_cast<uint32_t(*)[16]>(&lo[16]));
      if (ntok < kTileTok) {
        // rows past the split's last token hold stale data: zero this half's V rows
        uint4* v = reinterpret_cast<uint4*>(sKV + sb * kStageBytes + vh * 4 * kChunkBytes);
        const int tail = kTileTok - ntok;
        for (int e = row; e < 4 * tail * 8; e += 128) {
          const int cch = e / (tail * 8), rem = e % (tail * 8);
          v[(cch * kChunkBytes + (ntok + rem / 8) * 128) / 16 + rem % 8] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p_full[sb]));
    }
    // ---- epilogue ----
    if (ok && ntiles > 0)
      ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bar_o), (ntiles - 1) & 1, abort_flag));
    tc_fence_after();
    const bool direct = p.num_splits == 1;
    float* dst = direct ? a.o_part + (((int64_t)sr * a.B + b) * R + grow) * kDL + vh * 256
                        : p.ws_o + (((int64_t)split * a.B * a.shard_count + bz) * R + grow) * kDL +
                              vh * 256;
    const bool read_o = ok && ntiles > 0;                   // uniform across the warp
    const bool live = read_o && l > 0.f;
    const float inv = live ? 1.f / l : 0.f;
    for (int q = 0; q < 16; ++q) {
      uint32_t u[16];
      if (read_o) {
        tmem_ld16(tmem + lane_off + kColO + q * 16, u);
        tmem_ld_wait();
      }
      float4* d4 = reinterpret_cast<float4*>(dst + q * 16);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        d4[v] = live ? make_float4(__uint_as_float(u[4 * v]) * inv, __uint_as_float(u[4 * v + 1]) * inv,
                                   __uint_as_float(u[4 * v + 2]) * inv, __uint_as_float(u[4 * v + 3]) * inv)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (vh == 0) {
      const float lse2 = live ? m_ref + log2f(l) : -INFINITY;
      if (direct)
        a.lse_part[((int64_t)sr * a.B + b) * R + grow] = a.base2 ? lse2 : lse2 * kLn2;
      else
        p.ws_lse[((int64_t)split * a.B * a.shard_count + bz) * R + grow] = lse2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (abort_s && tid == 0) set_err(a.err, DCPMLA_DERR_TIMEOUT);
  if (p.num_splits == 1) return;

  // ---- split combine: the last of the 2 * num_splits CTAs of (b, r, row tile) merges ----
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(p.ws_cnt + (int64_t)bz * p.row_tiles + rt, 1u);
    last_s = prev == (uint32_t)(2 * p.num_splits - 1);
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  const int64_t sstride = (int64_t)a.B * a.shard_count * R;
  for (int e = tid; e < kRows * (kDL / 4); e += kThreads) {
    const int rrow = e / (kDL / 4), d4 = e % (kDL / 4);
    const int64_t base = (int64_t)bz * R + (int64_t)rt * kRows + rrow;
    float m = -INFINITY;
    for (int s = 0; s < p.num_splits; ++s) m = fmaxf(m, __ldcg(p.ws_lse + s * sstride + base));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse2 = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int s = 0; s < p.num_splits; ++s) sum += exp2f(__ldcg(p.ws_lse + s * sstride + base) - m);
      lse2 = m + log2f(sum);
      for (int s = 0; s < p.num_splits; ++s) {
        const float w = exp2f(__ldcg(p.ws_lse + s * sstride + base) - lse2);
        if (w == 0.f) continue;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (s * sstride + base) * kDL) + d4);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    const int64_t orow = ((int64_t)sr * a.B + b) * R + (int64_t)rt * kRows + rrow;
    reinterpret_cast<float4*>(a.o_part + orow * kDL)[d4] = acc;
    if (d4 == 0) a.lse_part[orow] = a.base2 ? lse2 : lse2 * kLn2;
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

int encode_rows_576(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return DCPMLA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)kDK, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDK * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DCPMLA_OK : DCPMLA_ERR_CUDA;
}

struct TcPlan {
  int32_t splits, chunk, row_tiles;
  size_t cnt_off, lse_off, o_off, bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

TcPlan plan_tc(const DecodeArgs& a, int sm_count) {
  TcPlan p{};
  p.row_tiles = a.R / kRows;
  const int64_t units = (int64_t)a.B * a.shard_count * p.row_tiles;   // pairs of CTAs
  const int64_t n_max = (int64_t)a.max_pages * a.P;
  const int64_t want = std::max<int64_t>(1, (sm_count + units - 1) / std::max<int64_t>(units, 1));
  const int64_t max_splits = std::max<int64_t>(1, n_max / 256);
  const int64_t splits = std::min(want, max_splits);
  int64_t chunk = (n_max + splits - 1) / splits;
  chunk = (chunk + kTileTok - 1) / kTileTok * kTileTok;
  p.chunk = (int32_t)chunk;
  p.splits = (int32_t)((n_max + chunk - 1) / chunk);
  if (p.splits <= 1) {
    p.splits = 1;
    return p;
  }
  const int64_t rows_all = (int64_t)a.B * a.shard_count * a.R;
  p.cnt_off = 0;
  p.lse_off = align256((size_t)units * 4);
  p.o_off = p.lse_off + align256((size_t)p.splits * rows_all * 4);
  p.bytes = p.o_off + (size_t)p.splits * rows_all * kDL * 4;
  return p;
}

}  // namespace

bool tc_supported(const DecodeArgs& a) {
  if (a.fp8) return false;
  if (a.R % kRows != 0 || a.shard_count > kMaxTcShards) return false;
  if (!(a.P % kTileTok == 0 || (kTileTok % a.P == 0 && a.P % 8 == 0))) return false;
  if ((int64_t)a.B * a.R > INT32_MAX || a.pool_rows > INT32_MAX) return false;
  return true;
}

size_t tc_workspace_bytes(const DecodeArgs& a, int sm_count) { return plan_tc(a, sm_count).bytes; }

int launch_decode_tc(const DecodeArgs& a, void* ws, size_t ws_bytes, int sm_count, cudaStream_t st) {
  const TcPlan plan = plan_tc(a, sm_count);
  if (ws_bytes < plan.bytes || (plan.bytes && !ws)) return DCPMLA_ERR_CAPACITY;
  TcParams* tp = new (std::nothrow) TcParams();
  if (!tp) return DCPMLA_ERR_CAPACITY;
  TcParams& p = *tp;
  p.a = a;
  p.box_rows = std::min(a.P, kTileTok);
  p.num_splits = plan.splits;
  p.chunk = plan.chunk;
  p.row_tiles = plan.row_tiles;
  int rc = encode_rows_576(&p.tm_q, a.q, (uint64_t)a.B * a.R, kRows);
  for (int i = 0; rc == DCPMLA_OK && i < a.shard_count; ++i)
    rc = encode_rows_576(&p.tm_kv[i], a.kv.pool[a.shard_begin + i], (uint64_t)a.pool_rows,
                         (uint32_t)p.box_rows);
  if (rc == DCPMLA_OK && plan.splits > 1) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.ws_cnt = reinterpret_cast<uint32_t*>(w + plan.cnt_off);
    p.ws_lse = reinterpret_cast<float*>(w + plan.lse_off);
    p.ws_o = reinterpret_cast<float*>(w + plan.o_off);
    if (cudaMemsetAsync(p.ws_cnt, 0, (size_t)a.B * a.shard_count * plan.row_tiles * 4, st) != cudaSuccess)
      rc = DCPMLA_ERR_CUDA;
  }
  if (rc == DCPMLA_OK) {
    const int64_t z = (int64_t)a.B * a.shard_count;
    if (z > 65535 || plan.row_tiles > 65535 || 2LL * plan.splits > INT32_MAX) rc = DCPMLA_ERR_UNSUPPORTED;
  }
  if (rc == DCPMLA_OK &&
      cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes) != cudaSuccess)
    rc = DCPMLA_ERR_CUDA;
  if (rc == DCPMLA_OK) {
    const dim3 grid((unsigned)(2 * plan.splits), (unsigned)plan.row_tiles,
                    (unsigned)(a.B * a.shard_count));
    decode_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(p);
    rc = launch_status();
  }
  delete tp;
  return rc;
}

}  // namespace dcpmla
