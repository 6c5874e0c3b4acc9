// Shard-local absorbed-MLA decode on the 5th-generation tensor cores for few
// query rows (heads x query tokens <= 16), where the rows are too few to fill an
// MMA's M dimension but the KV tokens are not: the contractions run transposed.
//
// SGLang "Decode Context Parallelism" docs, MLA decode dataflow: each shard
// returns its locally normalised o_r and lse_r; DCP x speculative decoding:
// the causal test uses global positions (shard-local token j of shard r is
// position j*c + r).  vLLM GLM-5.3 serving post, footnote arithmetic: scores
// over the 576-d key, values over the 512-d latent.
//
//   S^T [64 tokens x 16 rows]    = K [64 x 576] Q^T           (M = tokens, N = rows)
//   O^T [512 dims x 16 rows]    += V^T [512 x 64] P^T          (M = dims,  N = rows)
//
// Every CTA works alone on 64-token tiles over all 576 key dims, so no partial score
// crosses between SMs.  The score MMA has M = 64: its rows land in TMEM lanes 0-15 of
// each 32-lane quarter (row r at lane 32 (r / 16) + r % 16).
//
// The grid is persistent: the 64-token tiles of all (request, shard) items form one
// sequence, and CTA k of G takes the contiguous share [T k / G, T (k + 1) / G), so
// every CTA streams the same amount of KV with as few item switches as possible.
// An item cut by a share boundary writes fp32 partials that a small second kernel
// merges.
//
//   warp 0     TMA producer: Q^T of the unit (one 16-row box per 64-dim chunk),
//              then 64-token KV tiles (one 4-D box per page box, all nine chunks)
//              into a 2-deep stage ring, and L2 prefetches of the tiles a few
//              places further on, so that the ring's loads mostly hit L2.
//   warp 1     issues the QK MMAs (one elected lane of the converged warp): M 64,
//              N 16.  QK may run ahead of PV: a score buffer is free once the softmax
//              has loaded it.
//   warps 2-9  softmax, two warpgroups of 8 query rows each; in each warp lanes 0-15
//              hold the quarter's 16 tokens: base-2 online softmax with a lazily moved
//              per-row reference max, P^T to shared memory, unit epilogue (one value
//              dim per lane).
//   warp 10    issues the PV MMAs (one elected lane): M 128 (V^T MN-major, four
//              value blocks), N 32 = P as a bf16 hi part (rows 0-15) and lo part
//              (rows 16-31).
//
// TMEM columns: S^T double buffer [0, 32), O^T double buffer (by unit) [64, 320):
// buffer o, value block m (128 dims): hi rows at 64 + 128o + 32m, lo rows 16 later.
// Every mbarrier wait is bounded; a timeout sets DCPMLA_DERR_TIMEOUT, all roles
// drain, TMEM is freed.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <numeric>

#include "decode.cuh"
#include "sm100.cuh"

namespace dcpmla {
namespace {

using namespace sm100;

constexpr int kMaxFhShards = 8;
constexpr int kTok = 64;                       // tokens per tile = MMA M of the score product
constexpr int kRp = 16;                        // query rows per tile (MMA N); rows >= R are padding
constexpr int kNck = 9;                        // 64-dim column chunks of a 576-dim key row
constexpr int kChunk = kTok * 128;             // one 64-dim column chunk of a tile: 8 KB
constexpr int kStage = kNck * kChunk;          // 72 KB
// A stage is row-group major: [8-token group g][chunk c][8 tokens x 128 B], each 1 KB piece a
// 128-byte-swizzle atom, so one 4-D TMA box lands all of a page box's chunks; for the MMAs the
// 8-token groups of a chunk are 9 KB apart and a chunk's groups start c KB in.
constexpr int kStages = 2;
constexpr int kLook = 3;                       // page-id lookahead (tiles); L2 prefetch kLook - 1 ahead
constexpr int kQChunk = kRp * 128;             // Q^T chunk [16 rows x 64 dims]
constexpr int kQBuf = kNck * kQChunk;
constexpr int kPBuf = kTok * 64;               // P^T of a tile: a 64-byte line (32 rows) per token
constexpr int kMaxItems = 2048;                // (request, shard) pairs per launch
constexpr int kMaxCtas = 160;                  // CTAs of the persistent grid
constexpr int kSoftmaxThreads = 256;
constexpr int kPvWarp = 10;
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr uint32_t kColS = 0, kColO = 64, kTmemCols = 512;

constexpr int kOffKV = 0;
constexpr int kOffQ = kOffKV + kStages * kStage;
constexpr int kOffP = kOffQ + 2 * kQBuf;
constexpr int kOffPre = kOffP + 2 * kPBuf;
constexpr size_t kSmemBytes = 1024 + kOffPre + (kMaxItems + 1) * 4;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kOffPre % 1024 == 0, "1 KB aligned buffers");

struct FhParams {
  CUtensorMap tm_kv[kMaxFhShards];   // pool as {64, 8, 9 chunks, rows / 8}, box {64, 8, 9, box_rows / 8}
  CUtensorMap tm_q;                  // Q as [B * R, 576] bf16, box {64, 16}
  DecodeArgs a;
  int32_t box_rows;                  // rows per TMA box: gcd(P, 16)
  float* ws_o;                       // [slots, R, 512]: slot item + CTA
  float* ws_lse;                     // [slots, R] (base 2)
  int32_t* ws_bad;                   // [slots]: the unit needed a page outside the pools
  int32_t* ws_pre;                   // [B * shard_count + 1]: first tile of each (request, shard)
  int32_t fused;                     // 1: every unit to the workspace, merged over shards into o, lse
  int32_t wait_kcycles;              // a pipeline wait gives up after 1024 x this many clock64 cycles
};
static_assert(sizeof(FhParams) <= 4096, "kernel parameter space");

// Tokens of request b on shard r (0 for a length the launch rejects).
__device__ __forceinline__ int shard_tokens(const DecodeArgs& a, int L, int r) {
  if (L < a.Tq || (int64_t)L > (int64_t)a.max_pages * a.P * a.c) return 0;
  return shard_len(L, r, a.c, a.I);
}

// Work split.  All (request, shard) items' 64-token tiles form one sequence of T
// tiles; CTA k of G takes tiles [T k / G, T (k + 1) / G), so every CTA streams
// the same amount of KV.  A unit is the part of one item inside a cluster's share: an
// item inside one share is written straight to the output, the others to workspace
// slot item + k (unique: a later cluster starts at the same or a later item) and a
// merge kernel combines them.
struct Unit {
  int item, b, sr, r, L;
  int j0, j1, ntiles;   // shard-local token range and its 64-token tiles
  int slot;             // workspace slot of its partial
  bool whole;           // every tile of the item: no merge
};

// Start of cluster k's share of the T-tile sequence: floor(T k / G), in 32 bits when T G
// fits (the common case; a 64-bit division costs several times more).
__device__ __forceinline__ int fh_bound(int T, int k, int G) {
  if ((uint32_t)T <= 0xFFFFFFFFu / (uint32_t)G) return (int)((uint32_t)T * (uint32_t)k / (uint32_t)G);
  return (int)((int64_t)T * k / G);
}

// The part of item `it` (tiles [pre[it], pre[it + 1]) of the sequence) in the share
// [t_lo, t_hi) of cluster cl; false if they do not meet.
__device__ __forceinline__ bool fh_unit(const DecodeArgs& a, const int* pre, int it, int t_lo, int t_hi, int cl,
                                        Unit& x) {
  const int s0 = pre[it], s1 = pre[it + 1];
  const int s = max(s0, t_lo), e = min(s1, t_hi);
  if (e <= s) return false;
  x.item = it;
  x.b = it / a.shard_count;
  x.sr = it % a.shard_count;
  x.r = a.shard_begin + x.sr;
  x.L = __ldg(a.seq_lens + x.b);
  const int n = shard_tokens(a, x.L, x.r);
  x.j0 = (s - s0) * kTok;
  x.j1 = min(n, (e - s0) * kTok);
  x.ntiles = e - s;
  x.slot = it + cl;
  x.whole = s == s0 && e == s1;
  return true;
}

// The cluster whose share holds tile t (T > 0).
__device__ __forceinline__ int fh_cluster_of(int T, int t, int G) {
  const int64_t k0 = (uint32_t)T <= 0xFFFFFFFFu / (uint32_t)G ? (int64_t)((uint32_t)t * (uint32_t)G / (uint32_t)T)
                                                             : (int64_t)t * G / T;
  int k = (int)(k0 < G - 1 ? k0 : G - 1);
  while (k + 1 < G && fh_bound(T, k + 1, G) <= t) ++k;
  while (k > 0 && fh_bound(T, k, G) > t) --k;
  return k;
}

// kRL: waits give up after the launch's wait_kcycles instead of the fixed limit (tests only)
template <bool kRL>
__global__ void __launch_bounds__(kThreads, 1) decode_fh_bf16_kernel(const __grid_constant__ FhParams p) {
  const DecodeArgs& a = p.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = smem + kOffKV;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sP = smem + kOffP;
  int* sPre = reinterpret_cast<int*>(smem + kOffPre);
  __shared__ uint64_t bar_kv_full[kStages], bar_kv_empty[kStages];
  __shared__ uint64_t bar_q_full[2], bar_q_free[2];
  __shared__ uint64_t bar_s_full[2], bar_s_free[2], bar_p_full[2], bar_p_free[2], bar_o_free[2], bar_o_full[2];
  __shared__ uint64_t bar_o, bar_drain;
  __shared__ __align__(16) float red_s[2][2][4][8];     // [tile parity][warpgroup][quarter][row]
  __shared__ __align__(16) float lsum_s[2][2][4][8];   // [unit parity][warpgroup][quarter][row]
  __shared__ int seg_s[kThreads];
  __shared__ uint32_t tmem_base_s;
  __shared__ int ubad_s[2][2], issued_s, q_issued_s;
  __shared__ WaitCtl wctl_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = (int)gridDim.x, cl = (int)blockIdx.x;
  const int nitems = a.B * a.shard_count;
  const int64_t R = a.R;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bar_q_full[s]), 1);
      mbar_init(smem_u32(&bar_q_free[s]), 1);
      mbar_init(smem_u32(&bar_s_full[s]), 1);
      mbar_init(smem_u32(&bar_s_free[s]), kSoftmaxThreads / 32);
      mbar_init(smem_u32(&bar_p_full[s]), kSoftmaxThreads);
      mbar_init(smem_u32(&bar_p_free[s]), 1);
      mbar_init(smem_u32(&bar_o_free[s]), kSoftmaxThreads);
      mbar_init(smem_u32(&bar_o_full[s]), 1);
    }
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_drain), 2);                  // both MMA issuers
    wctl_s.abort = 0;
    wctl_s.limit_kcycles = p.wait_kcycles;
    issued_s = 0;
    q_issued_s = 0;
    ubad_s[0][0] = ubad_s[0][1] = ubad_s[1][0] = ubad_s[1][1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();

  // ---- work split, computed identically by every CTA ----
  // tiles per item into sPre[item + 1], then the prefix sum (each thread a segment)
  const int seg = (nitems + kThreads - 1) / kThreads;
  const int s0 = min(nitems, tid * seg), s1 = min(nitems, s0 + seg);
  {
    int sum = 0;
    for (int it = s0; it < s1; ++it) {
      const int b = it / a.shard_count, r = a.shard_begin + it % a.shard_count;
      const int L = __ldg(a.seq_lens + b);
      if (blockIdx.x == 0 && (L < a.Tq || (int64_t)L > (int64_t)a.max_pages * a.P * a.c))
        set_err(a.err, DCPMLA_DERR_LENGTH);
      const int t = (shard_tokens(a, L, r) + kTok - 1) / kTok;
      sPre[it + 1] = t;
      sum += t;
    }
    seg_s[tid] = sum;
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int kPer = (kThreads + 31) / 32;   // segments per lane (the tail lanes hold zeros)
    int tot = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int q = lane * kPer + k;
      tot += q < kThreads ? seg_s[q] : 0;
    }
    int incl = tot;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - tot;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int q = lane * kPer + k;
      if (q < kThreads) {
        const int v = seg_s[q];
        seg_s[q] = run;
        run += v;
      }
    }
  }
  __syncthreads();
  {
    int run = seg_s[tid];
    if (tid == 0) sPre[0] = 0;
    for (int it = s0; it < s1; ++it) {
      run += sPre[it + 1];
      sPre[it + 1] = run;
    }
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int it = tid; it <= nitems; it += kThreads) p.ws_pre[it] = sPre[it];
  // this CTA's share of the tile sequence, and the items it meets
  const int T = sPre[nitems];
  const int t_lo = fh_bound(T, cl, G), t_hi = fh_bound(T, cl + 1, G);
  int it_lo = 0, it_hi = -1;
  if (t_hi > t_lo) {
    int lo = 0, hi = nitems;   // pre[lo] <= t_lo < pre[lo + 1] (the first item holding t_lo)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sPre[mid] <= t_lo) lo = mid;
      else hi = mid;
    }
    it_lo = lo;
    hi = nitems;               // the last item starting before t_hi
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sPre[mid] < t_hi) lo = mid;
      else hi = mid;
    }
    it_hi = lo;
  }
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile WaitCtl* abort_flag = &wctl_s;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      for (int i = 0; i < a.shard_count; ++i) prefetch_tmap(&p.tm_kv[i]);
    }
    bool ok = true;
    int gi = 0, kk = 0, issued = 0, q_issued = 0;
    const int box = p.box_rows;
    // Page ids run kLook tiles ahead of the loads (across unit boundaries) through a
    // per-lane FIFO: entry k holds, for lane l, box l of the tile k places ahead
    // (its raw page id, rows, offset in the page, and the tile's shard).  The tile
    // kLook - 1 places ahead is also prefetched into L2, so the ring's loads mostly
    // hit L2; no page-table read is waited on between a stage's release and its load.
    int pu = it_lo, pi = 0;   // lookahead cursor: item, tile within its unit
    Unit px{};
    auto skip_empty = [&]() {
      while (pu <= it_hi && !fh_unit(a, sPre, pu, t_lo, t_hi, cl, px)) ++pu;
    };
    auto lookup = [&](int& g_, int& rows_, int& off_, int& sr_) {
      g_ = 0;
      rows_ = 0;
      off_ = 0;
      sr_ = 0;
      if (pu > it_hi) return;
      const int pt0 = px.j0 + pi * kTok;
      const int nb = (min(kTok, px.j1 - pt0) + box - 1) / box;
      sr_ = px.sr;
      if (lane < nb) {
        const int tok = pt0 + lane * box;
        rows_ = min(box, px.j1 - tok);
        off_ = tok % a.P;
        g_ = __ldg(a.pt + (int64_t)px.b * a.max_pages + tok / a.P);
      }
      if (++pi >= px.ntiles) {
        pi = 0;
        ++pu;
        skip_empty();
      }
    };
    int fg[kLook], fr[kLook], fo[kLook], fs[kLook];
    skip_empty();
#pragma unroll
    for (int k = 0; k < kLook; ++k) lookup(fg[k], fr[k], fo[k], fs[k]);
    for (int it = it_lo; ok && it <= it_hi; ++it) {
      Unit x;
      if (!fh_unit(a, sPre, it, t_lo, t_hi, cl, x)) continue;
      const int qb = kk & 1;
      const CUtensorMap* kvmap = &p.tm_kv[x.sr];
      bool okq = true;
      if (lane == 0) {
        if (kk >= 2) okq = wait_bar<false, kRL>(smem_u32(&bar_q_free[qb]), ((kk >> 1) - 1) & 1, abort_flag);
        if (okq) {
          q_issued = kk + 1;
          const uint32_t qf = smem_u32(&bar_q_full[qb]);
          mbar_arrive_expect_tx(qf, (uint32_t)(kNck * kQChunk));
          for (int c = 0; c < kNck; ++c)
            tma_load_2d(smem_u32(sQ + qb * kQBuf + c * kQChunk), &p.tm_q, c * 64, (int)(x.b * R), qf);
        }
      }
      ok = __shfl_sync(0xffffffffu, (int)okq, 0) != 0;
      for (int i = 0; ok && i < x.ntiles; ++i, ++gi) {
        const int st = gi & 1;
        const int t0 = x.j0 + i * kTok;
        const int ntok = min(kTok, x.j1 - t0);
        const int nbox = (ntok + box - 1) / box;
        // page of each box (lane < nbox, from the FIFO's head); a bad page id is
        // reported and read as page 0
        int y = 0;
        if (lane < nbox) {
          int g = fg[0];
          if (g < 0 || (int64_t)g >= a.num_pages) {
            set_err(a.err, DCPMLA_DERR_PAGE);
            g = 0;
          }
          y = g * a.P + fo[0];
        }
        bool okw = true;
        if (lane == 0 && gi >= kStages)
          okw = wait_bar<false, kRL>(smem_u32(&bar_kv_empty[st]), ((gi >> 1) - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, (int)okw, 0) != 0;
        if (!ok) break;
        const uint32_t full = smem_u32(&bar_kv_full[st]);
        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(nbox * box * 128 * kNck));
        __syncwarp();
        if (lane < nbox) {
          // the box's rows (whole 8-token groups) and all nine chunks in one copy
          tma_load_4d(smem_u32(sKV + st * kStage + lane * (box >> 3) * kNck * 1024), kvmap, 0, 0, 0, y >> 3, full);
        }
        issued = gi + 1;
        // L2 prefetch of the tile kLook - 1 places ahead: a box's rows are contiguous
        // in the pool
        if (fr[kLook - 1] > 0) {
          int g = fg[kLook - 1];
          if (g < 0 || (int64_t)g >= a.num_pages) g = 0;   // reported when the tile is loaded
          const int64_t py = (int64_t)g * a.P + fo[kLook - 1];
          const uint8_t* src =
              static_cast<const uint8_t*>(a.kv.pool[a.shard_begin + fs[kLook - 1]]) + py * (kDK * 2);
          bulk_prefetch_l2(src, (uint32_t)fr[kLook - 1] * (kDK * 2));   // a multiple of 16 bytes
        }
#pragma unroll
        for (int k = 0; k + 1 < kLook; ++k) {
          fg[k] = fg[k + 1];
          fr[k] = fr[k + 1];
          fo[k] = fo[k + 1];
          fs[k] = fs[k + 1];
        }
        lookup(fg[kLook - 1], fr[kLook - 1], fo[kLook - 1], fs[kLook - 1]);
      }
      ++kk;
    }
    if (lane == 0) {                                   // drained at the teardown
      issued_s = issued;
      q_issued_s = q_issued;
    }
  } else if (warp == 1 || warp == kPvWarp) {
    // ---------------------------------------------------------------- MMA
    // Two issuing warps, each blocking on its own barriers: warp 1 issues the QK of
    // each tile once its KV landed and the softmax has loaded the scores two tiles
    // back (whose TMEM buffer it overwrites), so QK runs ahead of PV; warp kPvWarp
    // issues each tile's PV once its P is written, which frees the tile's stage for
    // the next load.  The whole warp runs the loop (waits, descriptors) and one
    // elected lane issues each MMA and commit, so the operands stay warp-uniform.  A
    // commit tracks the MMAs of the lane issuing it.
    constexpr uint32_t idesc_qk = idesc_bf16(kTok, kRp, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16(128, 2 * kRp, true, true);
    // Base descriptors; the start-address field is the low 14 bits (address >> 4),
    // so a constant byte offset is added as (offset >> 4) without carries.
    const uint64_t kA0 = desc_sw128(smem_u32(sKV), 16, kNck * 1024);      // keys, K-major
    const uint64_t vA0 = desc_sw128(smem_u32(sKV), 1024, kNck * 1024);    // values, MN-major
    const uint64_t qB0 = desc_sw128(smem_u32(sQ), 16, 1024);              // Q^T, K-major
    const uint64_t pB0 = desc_sw64(smem_u32(sP), 8192, 512);              // P^T, MN-major (32 rows per token)
    const bool qk_role = warp == 1;
    bool ok = true;
    int gt = 0, kk = 0;                  // tiles and units so far
    for (int it = it_lo; ok && it <= it_hi; ++it) {
      Unit x;
      if (!fh_unit(a, sPre, it, t_lo, t_hi, cl, x)) continue;
      const int ntiles = x.ntiles;
      const int qb = kk & 1, ob = kk & 1;
      if (qk_role) {
        ok = __all_sync(0xffffffffu, wait_bar<false, kRL>(smem_u32(&bar_q_full[qb]), (kk >> 1) & 1, abort_flag));
        for (int i = 0; ok && i < ntiles; ++i, ++gt) {
          const int sb = gt & 1;
          if (gt >= 2)
            ok = __all_sync(0xffffffffu,
                            wait_bar<false, kRL>(smem_u32(&bar_s_free[sb]), ((gt >> 1) - 1) & 1, abort_flag));
          if (ok) ok = __all_sync(0xffffffffu, wait_bar<false, kRL>(smem_u32(&bar_kv_full[sb]), (gt >> 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + (uint32_t)(sb * kRp);
#pragma unroll
          for (int c = 0; c < kNck; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss_warp(d, kA0 + (uint64_t)((sb * kStage + c * 1024 + k * 32) >> 4),
                          qB0 + (uint64_t)((qb * kQBuf + c * kQChunk + k * 32) >> 4), idesc_qk, (c | k) != 0);
          }
          mma_commit_warp(smem_u32(&bar_s_full[sb]));
        }
        if (ok) mma_commit_warp(smem_u32(&bar_q_free[qb]));   // the unit's Q buffer may be refilled
      } else {
        for (int i = 0; ok && i < ntiles; ++i, ++gt) {
          const int sb = gt & 1;
          ok = __all_sync(0xffffffffu, wait_bar<false, kRL>(smem_u32(&bar_p_full[sb]), (gt >> 1) & 1, abort_flag));
          if (ok && i == 0 && kk >= 2)
            ok = __all_sync(0xffffffffu,
                            wait_bar<false, kRL>(smem_u32(&bar_o_free[ob]), ((kk >> 1) - 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
            const uint32_t d = tmem + kColO + (uint32_t)(ob * 128 + mb * 32);
#pragma unroll
            for (int ks = 0; ks < kTok / 16; ++ks) {
              const uint64_t ad = vA0 + (uint64_t)((sb * kStage + 2 * mb * 1024 + ks * 2 * kNck * 1024) >> 4);
              const uint64_t bd = pB0 + (uint64_t)((sb * kPBuf + ks * 1024) >> 4);
              mma_ss_warp(d, ad, bd, idesc_pv, (i == 0 && ks == 0) ? 0u : 1u);
            }
          }
          mma_commit_warp(smem_u32(&bar_kv_empty[sb]));
          mma_commit_warp(smem_u32(&bar_p_free[sb]));
          mma_commit_warp(smem_u32(&bar_o));
          // the unit's O^T is complete: one phase of its buffer's barrier per unit
          if (i == ntiles - 1) mma_commit_warp(smem_u32(&bar_o_full[ob]));
        }
      }
      ++kk;
    }
    // drain: every MMA issued above completes before TMEM is released (one arrival per
    // issuing warp)
    mma_commit_warp(smem_u32(&bar_drain));
    const long long t0 = clock64();
    while (!mbar_try_wait(smem_u32(&bar_drain), 0) && clock64() - t0 < kDrainCycles) {
    }
  } else {
    // -------------------------------------------------------------- softmax
    // Warps 2..9: warpgroup g handles query rows [8g, 8g + 8).  For S^T (M = 64) lanes
    // 0-15 of warp quarter q hold tokens 16q + lane; for O^T (M = 128) every lane holds
    // value dim 32q + lane of each block.
    const int g = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const bool live = lane < 16;                             // a token lane of the score tile
    const int tok = quarter * 16 + (lane & 15);              // its token within the tile
    const int dl = quarter * 32 + lane;                      // its value dim within a block
    const int stid = g * 128 + dl;                           // 0..255
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float qscale = a.sm_scale * kLog2e;
    bool ok = true;
    int gi = 0, kk = 0, uc = 0;
    for (int it = it_lo; ok && it <= it_hi; ++it) {
      Unit x;
      if (!fh_unit(a, sPre, it, t_lo, t_hi, cl, x)) continue;
      const int ob = kk & 1;
      const int up = uc & 1;
      int qpos[8];
      bool rvalid[8];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int row = 8 * g + n;
        rvalid[n] = row < R;
        qpos[n] = x.L - a.Tq + (rvalid[n] ? row / a.H : 0);
      }
      const int qpos_min = x.L - a.Tq;
      const bool all_rows = R >= kRp;
      const int32_t* pt_row = a.pt + (int64_t)x.b * a.max_pages;
      bool bad = false;   // a page this thread's tokens need is outside the pools
      float m_ref[8], lt[8];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        m_ref[n] = -INFINITY;
        lt[n] = 0.f;
      }
      for (int i = 0; i < x.ntiles; ++i, ++gi) {   // left only together, at a barrier-OR
        const int sb = gi & 1;
        const int t0 = x.j0 + i * kTok;
        const int ntok = min(kTok, x.j1 - t0);
        const bool in_tile = live && tok < ntok;
        // this thread's page id, checked at the end of the tile (its load is in
        // flight meanwhile)
        const int gpg = in_tile ? __ldg(pt_row + (t0 + tok) / a.P) : 0;
        // A failed wait does not leave the loop at once: every warp of the warpgroup goes on
        // to the warpgroup's barrier-OR below, skipping the work of the failed steps.  A named
        // barrier has no time limit, so all of its threads must reach it: the softmax warps
        // leave their loops only where a barrier-OR over the warpgroup tells every warp the
        // same, and every named barrier here is one warpgroup's own.
        if (ok) ok = __all_sync(0xffffffffu, wait_bar<false, kRL>(smem_u32(&bar_s_full[sb]), (gi >> 1) & 1, abort_flag));
        uint32_t own[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (ok) {
          tc_fence_after();
          tmem_ld8(tmem + lane_off + kColS + (uint32_t)(sb * kRp + 8 * g), own);
          tmem_ld_wait();
          // the score buffer may take the QK two tiles ahead
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_s_free[sb]));
        }
        // causal / tail / padding-row mask, base-2 scaling
        // (a tile every row sees whole, the common case, skips the per-token position)
        const bool full_vis = all_rows && ntok == kTok && shard_pos(t0 + kTok - 1, x.r, a.c, a.I) <= qpos_min;
        float s[8];
        if (full_vis) {
#pragma unroll
          for (int n = 0; n < 8; ++n) s[n] = live ? __uint_as_float(own[n]) * qscale : -INFINITY;
        } else {
          const int64_t kpos = shard_pos(t0 + tok, x.r, a.c, a.I);
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            const bool vis = live && rvalid[n] && in_tile && kpos <= qpos[n];
            s[n] = vis ? __uint_as_float(own[n]) * qscale : -INFINITY;
          }
        }
        // Lazy reference max: a row moves it only when this tile's max exceeds it
        // by more than 8 (every weight 2^(s - m_ref) stays <= 256); rows that move
        // it after O holds data rescale their O^T columns and partial sums.  Whether
        // any row of the warpgroup moves (or any of its warps failed a wait) is one
        // barrier-OR; only then is the tile's exact per-row max formed (warp
        // reduction, then across the 4 warps).
        bool over = !ok;
#pragma unroll
        for (int n = 0; n < 8; ++n) over |= s[n] > m_ref[n] + 8.f;
        if (named_bar_or(1 + g, 128, over)) {
          // the warpgroup leaves the loop together if any of its warps failed a wait
          if (named_bar_or(1 + g, 128, !ok)) {
            ok = false;
            break;
          }
          float wm[8];
#pragma unroll
          for (int n = 0; n < 8; ++n) wm[n] = warp_max_f32(s[n]);
          if (lane == 0) {
            float4* dst = reinterpret_cast<float4*>(red_s[sb][g][quarter]);
            dst[0] = make_float4(wm[0], wm[1], wm[2], wm[3]);
            dst[1] = make_float4(wm[4], wm[5], wm[6], wm[7]);
          }
          named_bar_sync(1 + g, 128);
          float tmax[8];
#pragma unroll
          for (int n = 0; n < 8; ++n) tmax[n] = -INFINITY;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 m0 = reinterpret_cast<const float4*>(red_s[sb][g][q])[0];
            const float4 m1 = reinterpret_cast<const float4*>(red_s[sb][g][q])[1];
            tmax[0] = fmaxf(tmax[0], m0.x); tmax[1] = fmaxf(tmax[1], m0.y);
            tmax[2] = fmaxf(tmax[2], m0.z); tmax[3] = fmaxf(tmax[3], m0.w);
            tmax[4] = fmaxf(tmax[4], m1.x); tmax[5] = fmaxf(tmax[5], m1.y);
            tmax[6] = fmaxf(tmax[6], m1.z); tmax[7] = fmaxf(tmax[7], m1.w);
          }
          bool any_rescale = false;
          float alpha[8];
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            const bool mv = tmax[n] > m_ref[n] + 8.f;
            const bool rs = mv && m_ref[n] != -INFINITY;
            alpha[n] = rs ? ex2_approx(m_ref[n] - tmax[n]) : 1.f;
            any_rescale |= rs;
            if (mv) m_ref[n] = tmax[n];
          }
          if (any_rescale) {   // the same decision in every thread of the warpgroup
            // O^T holds every PV before this tile once PV(gi - 1) completes.  QK runs
            // ahead of PV, so PV(gi - 2) may still be in flight: wait for it first
            // (its P buffer's barrier), or the parity wait on bar_o could match the
            // phase before.
            if (ok && gi >= 2)
              ok = __all_sync(0xffffffffu,
                              wait_bar<false, kRL>(smem_u32(&bar_p_free[sb]), ((gi >> 1) - 1) & 1, abort_flag));
            if (ok) ok = __all_sync(0xffffffffu, wait_bar<false, kRL>(smem_u32(&bar_o), (gi - 1) & 1, abort_flag));
            // on a failed wait the rescale is skipped (the output is invalid then); the
            // warp leaves at the next decision barrier
            if (ok) {
              tc_fence_after();
#pragma unroll
              for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
                for (int part = 0; part < 2; ++part) {   // hi rows, then lo rows
                  const uint32_t col =
                      tmem + lane_off + kColO + (uint32_t)(ob * 128 + mb * 32 + part * 16 + 8 * g);
                  uint32_t v[8];
                  tmem_ld8(col, v);
                  tmem_ld_wait();
#pragma unroll
                  for (int n = 0; n < 8; ++n) v[n] = __float_as_uint(__uint_as_float(v[n]) * alpha[n]);
                  tmem_st8(col, v);
                }
              }
              tmem_st_wait();
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) lt[n] *= alpha[n];
          }
        }
        // P^T as bf16 hi (rows 0-15) + lo (rows 16-31); one bf16 rounding of the
        // weights alone would cost ~1e-3 relative error in O.  P buffer sb was last read
        // by PV(gi - 2), which had completed before this tile's KV load was issued (the
        // load waited for that PV's commit on the stage's empty barrier), and this
        // tile's scores come after that load: no wait is needed here.
        // P^T is MN-major with a 64-byte swizzle: a token's 32 rows (hi 0-15, lo 16-31) are
        // one 64-byte line, 8 tokens an atom; this thread's 8 hi and 8 lo rows are one
        // 16-byte unit each (unit u of line t sits at u ^ ((t % 8) / 2))
        uint32_t hp[4], lp[4];
#pragma unroll
        for (int n = 0; n < 8; n += 2) {
          const float mr0 = m_ref[n] == -INFINITY ? 0.f : m_ref[n];   // every s is -inf then
          const float mr1 = m_ref[n + 1] == -INFINITY ? 0.f : m_ref[n + 1];
          const float p0 = ex2_approx(s[n] - mr0), p1 = ex2_approx(s[n + 1] - mr1);
          lt[n] += p0;
          lt[n + 1] += p1;
          const __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
          const float2 hf = __bfloat1622float2(hh);
          hp[n >> 1] = *reinterpret_cast<const uint32_t*>(&hh);
          const __nv_bfloat162 ll = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
          lp[n >> 1] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        if (ok) {
          if (live) {
            uint8_t* line = sP + sb * kPBuf + (tok >> 3) * 512 + (tok & 7) * 64;
            const int sw = (tok & 7) >> 1;
            *reinterpret_cast<uint4*>(line + ((g ^ sw) << 4)) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
            *reinterpret_cast<uint4*>(line + (((2 + g) ^ sw) << 4)) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
          }
          if (ntok < kTok) {
            // rows past the unit's last token hold stale data: zero their value chunks
            uint4* v = reinterpret_cast<uint4*>(sKV + sb * kStage);
            const int tail = kTok - ntok;
            for (int e = stid; e < 8 * tail * 8; e += kSoftmaxThreads) {
              const int cch = e / (tail * 8), rem = e % (tail * 8), t = ntok + rem / 8;
              v[((t >> 3) * kNck * 1024 + cch * 1024 + (t & 7) * 128) / 16 + rem % 8] = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_p_full[sb]));
        }
        bad |= gpg < 0 || (int64_t)gpg >= a.num_pages;
      }
      // the warpgroup leaves together if any of its warps failed a wait (a failure after the
      // last tile's barrier-OR, in the rescale or the P buffer's wait, shows here)
      if (named_bar_or(1 + g, 128, !ok)) {
        ok = false;
        break;
      }
      // ---- unit epilogue: O^T / l, partial or final output ----
      if (ok && x.ntiles > 0) {
        // Not bar_o: when the last tile's softmax ends, the PV two tiles back may
        // still be running, and a parity wait on bar_o would then match an older
        // phase.  bar_o_full[ob] completes once per unit on this buffer.
        ok = __all_sync(0xffffffffu, wait_bar<false, kRL>(smem_u32(&bar_o_full[ob]), (kk >> 1) & 1, abort_flag));
        if (ok) tc_fence_after();   // else the output is invalid; the unit ends below
      }
      // a unit that needed a bad page is written as empty (its partial, for a split item)
      // (tagged with the unit's ordinal: a slot is rewritten only two units later,
      // after every thread has passed the next unit's barrier)
      // (each warpgroup checks every token of the tile, so its own flag is the unit's)
      if (bad) ubad_s[up][g] = uc + 1;
      named_bar_sync(1 + g, 128);
      const bool unit_bad = ubad_s[up][g] == uc + 1;
      // row sums over the token lanes: warp butterfly, then the 4 warps in order
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        float v = lt[n];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        lt[n] = v;
      }
      if (lane == 0) {
        float4* dst = reinterpret_cast<float4*>(lsum_s[up][g][quarter]);
        dst[0] = make_float4(lt[0], lt[1], lt[2], lt[3]);
        dst[1] = make_float4(lt[4], lt[5], lt[6], lt[7]);
      }
      named_bar_sync(1 + g, 128);
      float inv[8], ltot[8];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        ltot[n] = ((lsum_s[up][g][0][n] + lsum_s[up][g][1][n]) + lsum_s[up][g][2][n]) + lsum_s[up][g][3][n];
        inv[n] = ltot[n] > 0.f ? 1.f / ltot[n] : 0.f;
      }
      const bool direct = !p.fused && x.whole;
      const bool empty_out = direct && unit_bad;
      const int64_t orow0 = direct ? ((int64_t)x.sr * a.B + x.b) * R : (int64_t)x.slot * R;
      float* obase = direct ? a.o_part : p.ws_o;
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
        uint32_t hv[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (x.ntiles > 0 && ok) {
          const uint32_t col = tmem + lane_off + kColO + (uint32_t)(ob * 128 + mb * 32 + 8 * g);
          tmem_ld8(col, hv);
          tmem_ld8(col + 16, lv);
          tmem_ld_wait();
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int row = 8 * g + n;
          if (row >= R) continue;
          const float val =
              (x.ntiles > 0 && !empty_out) ? (__uint_as_float(hv[n]) + __uint_as_float(lv[n])) * inv[n] : 0.f;
          obase[(orow0 + row) * kDL + mb * 128 + dl] = val;
        }
      }
      if (quarter == 0 && lane == 0) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int row = 8 * g + n;
          if (row >= R) continue;
          const float lse2 = (ltot[n] > 0.f && !empty_out) ? m_ref[n] + log2f(ltot[n]) : -INFINITY;
          if (direct) a.lse_part[orow0 + row] = a.base2 ? lse2 : lse2 * kLn2;
          else p.ws_lse[orow0 + row] = lse2;
        }
      }
      if (x.ntiles > 0) {
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_o_free[ob]));
        ++kk;
      }
      // a split item's units are merged by the combine kernel; it also reads this flag
      if (!direct && stid == 0) p.ws_bad[x.slot] = unit_bad ? 1 : 0;
      ++uc;
      // the unit loop's condition must agree in every thread of the warpgroup
      if (named_bar_or(1 + g, 128, !ok)) ok = false;
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role has left its loop.  After an abort, the KV and Q loads issued before it may
  // still be in flight (their consumers gave up): they land before this CTA's shared memory
  // goes away.
  if (tid == 0 && wctl_s.abort) {
    drain_ring(bar_kv_full, kStages, issued_s);
    drain_ring(bar_q_full, 2, q_issued_s);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  __syncthreads();
  if (wctl_s.abort && tid == 0) set_err(a.err, DCPMLA_DERR_TIMEOUT);
}

// Merge of the (request, shard) items split between CTAs: one block per (item,
// query row), 128 threads x 4 value dims.  The exact LSE merge of the partials (base 2):
// lse = log2 sum_k 2^lse_k, o = sum_k 2^(lse_k - lse) o_k.  An item with no tiles (an
// empty shard or a rejected length) is written as empty, and so is one any partial of
// which needed a bad page; an item inside one cluster's share was written by the decode.
// `pre` is the tile prefix over items; clusters with an empty share (more clusters
// than tiles) hold no partial.
__global__ void __launch_bounds__(128) fh_combine_kernel(const DecodeArgs a, const int32_t* __restrict__ pre, int G,
                                                         const float* __restrict__ ws_o,
                                                         const float* __restrict__ ws_lse,
                                                         const int32_t* __restrict__ ws_bad) {
  const int item = blockIdx.x, row = blockIdx.y, t = threadIdx.x;
  const int nitems = a.B * a.shard_count;
  const int T = pre[nitems], s0 = pre[item], s1 = pre[item + 1];
  const int64_t R = a.R;
  int k0 = 0, k1 = -1;
  if (s1 > s0) {
    k0 = fh_cluster_of(T, s0, G);
    k1 = fh_cluster_of(T, s1 - 1, G);
    if (k0 == k1) return;
  }
  bool bad = false;
  float m = -INFINITY;
  for (int k = k0; k <= k1; ++k) {
    if (fh_bound(T, k, G) == fh_bound(T, k + 1, G)) continue;
    bad |= ws_bad[item + k] != 0;
    m = fmaxf(m, ws_lse[(int64_t)(item + k) * R + row]);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse2 = -INFINITY;
  if (!bad && m != -INFINITY) {
    float sum = 0.f;
    for (int k = k0; k <= k1; ++k)
      if (fh_bound(T, k, G) != fh_bound(T, k + 1, G)) sum += exp2f(ws_lse[(int64_t)(item + k) * R + row] - m);
    lse2 = m + log2f(sum);
    for (int k = k0; k <= k1; ++k) {
      if (fh_bound(T, k, G) == fh_bound(T, k + 1, G)) continue;
      const float w = exp2f(ws_lse[(int64_t)(item + k) * R + row] - lse2);
      const float4 v = __ldcs(reinterpret_cast<const float4*>(ws_o + ((int64_t)(item + k) * R + row) * kDL) + t);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  const int b = item / a.shard_count, sr = item % a.shard_count;
  const int64_t orow = ((int64_t)sr * a.B + b) * R + row;
  reinterpret_cast<float4*>(a.o_part + orow * kDL)[t] = acc;
  if (t == 0) a.lse_part[orow] = a.base2 ? lse2 : lse2 * kLn2;
}

// Fused decode + merge: block (b, row) merges the partials of every unit of every shard of
// request b for that query row (SGLang DCP docs, MLA decode dataflow: the exact LSE merge; the
// partials of a split shard merge the same way), in base 2, into o [B, R, 512] and lse [B, R]
// (base converted at the end).  Warp 0 gathers the partials, lane l those of shard l (its
// units' LSEs, then a warp max and sum); the block's 128 threads then form the weighted sums,
// 4 dims each.  A shard any unit of which needed a bad page is left out, as the unfused path
// writes it as empty (lse = -inf).
constexpr int kMergeParts = kMaxFhShards + kMaxCtas;  // shards + share boundaries in a request

__global__ void __launch_bounds__(128) fh_merge_all_kernel(const DecodeArgs a, const int32_t* __restrict__ pre,
                                                           int G, const float* __restrict__ ws_o,
                                                           const float* __restrict__ ws_lse,
                                                           const int32_t* __restrict__ ws_bad) {
  const int b = blockIdx.x, row = blockIdx.y, t = threadIdx.x, lane = t & 31;
  const int64_t R = a.R;
  __shared__ float w_s[kMergeParts];
  __shared__ int slot_s[kMergeParts];
  __shared__ int n_s;
  if (t < 32) {
    const int T = pre[a.B * a.shard_count];
    int k0 = 0, k1 = -1;
    bool use = false;
    const int item = b * a.shard_count + lane;
    if (lane < a.shard_count) {
      const int s0 = pre[item], s1 = pre[item + 1];
      if (s1 > s0) {
        k0 = fh_cluster_of(T, s0, G);
        k1 = fh_cluster_of(T, s1 - 1, G);
        bool bad = false;
        for (int k = k0; k <= k1; ++k)
          if (fh_bound(T, k, G) != fh_bound(T, k + 1, G)) bad |= ws_bad[item + k] != 0;
        use = !bad;
      }
    }
    auto live = [&](int k) { return fh_bound(T, k, G) != fh_bound(T, k + 1, G); };
    int cnt = 0;
    float m = -INFINITY;
    if (use)
      for (int k = k0; k <= k1; ++k)
        if (live(k)) {
          m = fmaxf(m, ws_lse[(int64_t)(item + k) * R + row]);
          ++cnt;
        }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    float sum = 0.f;
    if (use && m != -INFINITY)
      for (int k = k0; k <= k1; ++k)
        if (live(k)) sum += exp2f(ws_lse[(int64_t)(item + k) * R + row] - m);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    const float lse2 = sum > 0.f ? m + log2f(sum) : -INFINITY;
    int off = cnt;                                        // exclusive scan of the counts
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, off, d);
      if (lane >= d) off += v;
    }
    const int total = __shfl_sync(0xffffffffu, off, 31);
    off -= cnt;
    if (use)
      for (int k = k0; k <= k1; ++k)
        if (live(k)) {
          w_s[off] = lse2 == -INFINITY ? 0.f : exp2f(ws_lse[(int64_t)(item + k) * R + row] - lse2);
          slot_s[off++] = item + k;
        }
    if (lane == 0) {
      n_s = total;
      a.lse_part[(int64_t)b * R + row] = a.base2 ? lse2 : lse2 * kLn2;
    }
  }
  __syncthreads();
  const int n = n_s;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int j = 0;
  for (; j + 4 <= n; j += 4) {                            // four independent loads in flight
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = __ldcs(reinterpret_cast<const float4*>(ws_o + ((int64_t)slot_s[j + u] * R + row) * kDL) + t);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = w_s[j + u];
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
  }
  for (; j < n; ++j) {
    const float w = w_s[j];
    const float4 v = __ldcs(reinterpret_cast<const float4*>(ws_o + ((int64_t)slot_s[j] * R + row) * kDL) + t);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  reinterpret_cast<float4*>(a.o_part + ((int64_t)b * R + row) * kDL)[t] = acc;
}

struct FhPlan {
  int32_t ctas, slots;
  size_t pre_off, bad_off, lse_off, o_off, bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

FhPlan plan_fh(const DecodeArgs& a, int sm_count) {
  FhPlan p{};
  const int64_t items = (int64_t)a.B * a.shard_count;
  // one CTA per SM, but no more CTAs than tiles can exist: a shard holds at most
  // max_pages * P of a request's tokens (small problems then launch few CTAs and the
  // combine walks few shares)
  const int64_t tiles_max = items * (((int64_t)a.max_pages * a.P + kTok - 1) / kTok);
  p.ctas = (int32_t)std::max<int64_t>(1, std::min<int64_t>(std::min(sm_count, kMaxCtas), tiles_max));
  p.slots = (int32_t)(items + p.ctas);   // partial of item it in CTA k: slot it + k
  p.pre_off = 0;
  p.bad_off = align256((size_t)(items + 1) * 4);
  p.lse_off = p.bad_off + align256((size_t)p.slots * 4);
  p.o_off = p.lse_off + align256((size_t)p.slots * a.R * 4);
  p.bytes = p.o_off + (size_t)p.slots * a.R * kDL * 4;
  return p;
}

}  // namespace

bool fh_supported(const DecodeArgs& a, int sm_count) {
  if (a.fp8 || a.R > kRp || sm_count < 1) return false;
  if (a.shard_count > kMaxFhShards) return false;
  if (a.P % 8 != 0) return false;   // page boxes of gcd(P, 16) rows: whole 8-token groups
  if ((int64_t)a.B * a.shard_count > kMaxItems) return false;
  // the tile sequence of all items fits 32-bit tile indices
  if ((int64_t)a.B * a.shard_count * (((int64_t)a.max_pages * a.P + kTok - 1) / kTok) > INT32_MAX) return false;
  if ((int64_t)a.B * a.R < kRp || (int64_t)a.B * a.R > INT32_MAX) return false;   // Q box of 16 rows
  if (a.pool_rows > INT32_MAX || a.pool_rows % 8 != 0) return false;   // 8-row TMA groups
  return true;
}

size_t fh_workspace_bytes(const DecodeArgs& a, int sm_count) { return plan_fh(a, sm_count).bytes; }

int launch_decode_fh(const DecodeArgs& a, void* ws, size_t ws_bytes, int sm_count, cudaStream_t st, bool fused) {
  const FhPlan plan = plan_fh(a, sm_count);
  if (ws_bytes < plan.bytes || !ws) return DCPMLA_ERR_CAPACITY;
  static ParamCache<FhParams> cache;
  const LaunchKey key = launch_key(a, ws, ws_bytes, fused ? 5 : 4);
  std::lock_guard<std::mutex> lk(cache.mu);
  bool fresh = false;
  FhParams* fp = cache.get(key, fresh);
  if (!fp) return DCPMLA_ERR_CAPACITY;
  FhParams& p = *fp;
  int rc = DCPMLA_OK;
  if (fresh) {
    p.a = a;
    // a box never crosses a page or a tile; boxes of 16 rows (8 a tile) land sooner than
    // larger ones (64-token pages: 0.874 ms on the long workload against 0.900 with 64-row boxes)
    p.box_rows = std::gcd(a.P, 16);
    p.fused = fused ? 1 : 0;
    rc = tma_encode_bf16_2d(&p.tm_q, a.q, (uint64_t)kDK, (uint64_t)a.B * a.R, 64, kRp);
    for (int i = 0; rc == DCPMLA_OK && i < a.shard_count; ++i)
      rc = tma_encode_kv_rowgroups(&p.tm_kv[i], a.kv.pool[a.shard_begin + i], (uint64_t)a.pool_rows, (uint32_t)kNck,
                                   (uint32_t)p.box_rows / 8);
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.ws_pre = reinterpret_cast<int32_t*>(w + plan.pre_off);
    p.ws_bad = reinterpret_cast<int32_t*>(w + plan.bad_off);
    p.ws_lse = reinterpret_cast<float*>(w + plan.lse_off);
    p.ws_o = reinterpret_cast<float*>(w + plan.o_off);
    if (rc != DCPMLA_OK) {
      cache.drop(fp);
      return rc;
    }
  }
  p.wait_kcycles = pipeline_wait_kcycles();
  const auto kern = p.wait_kcycles == kDefaultWaitKcycles ? decode_fh_bf16_kernel<false> : decode_fh_bf16_kernel<true>;
  rc = ensure_smem_attr((const void*)kern, (int)kSmemBytes);
  if (rc == DCPMLA_OK) {
    kern<<<plan.ctas, kThreads, kSmemBytes, st>>>(p);
    rc = launch_status();
  }
  if (rc == DCPMLA_OK && fused) {
    fh_merge_all_kernel<<<dim3((unsigned)a.B, (unsigned)a.R), 128, 0, st>>>(a, p.ws_pre, plan.ctas, p.ws_o,
                                                                           p.ws_lse, p.ws_bad);
    rc = launch_status();
  } else if (rc == DCPMLA_OK) {
    const dim3 grid((unsigned)(a.B * a.shard_count), (unsigned)a.R);
    fh_combine_kernel<<<grid, 128, 0, st>>>(a, p.ws_pre, plan.ctas, p.ws_o, p.ws_lse, p.ws_bad);
    rc = launch_status();
  }
  return rc;
}

}  // namespace dcpmla
