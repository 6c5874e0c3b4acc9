// Shard-local absorbed-MLA decode on CUDA cores (FP32 FMA + warp shuffles).
//
// SGLang "Decode Context Parallelism" docs, MLA decode dataflow: shard r
// returns its locally normalised output o_r and lse_r; DCP x speculative
// decoding: the shard kernel gets cp_world, cp_rank and the global KV length
// so that the causal test uses global positions.  vLLM GLM-5.3 serving post,
// footnote arithmetic: scores over the 576-d key, values over the 512-d latent.
//
// One CTA = (request b, shard r, group of 16 query rows, one split of the
// shard's tokens).  512 threads.  Per tile of 32 shard tokens:
//   * cp.async streams the 32 stored rows (16-byte vectors) into a padded,
//     double-buffered shared-memory tile;
//   * QK: warp w owns query row w, lane l owns token l: a 576-long FP32 dot
//     product, then warp-shuffle max / sum for the online softmax (base 2,
//     the query pre-scaled by sm_scale * log2 e);
//   * PV: thread (half, k) owns latent dims 2k, 2k+1 for 8 of the 16 rows.
// Splits of one (b, r, row group) write partial (o, lse) to the workspace; the
// last split to finish (atomic arrival count, no waiting) merges them.
#include <algorithm>
#include <cmath>

#include "decode.cuh"

namespace dcpmla {
namespace {

constexpr int kRG = 16;          // query rows per CTA
constexpr int kTile = 32;        // shard tokens per tile
constexpr int kThreads = 512;
constexpr int kQStride = kDK + 4;          // floats per q row in SMEM (bank skew)
constexpr int kRowBf16 = kDK * 2 + 16;     // bytes per SMEM key row, bf16 (1168)
constexpr int kRowFp8 = kDK + 16;          // bytes per SMEM key row, e4m3 (592)

struct FmaParams {
  DecodeArgs a;
  int32_t num_splits;
  int32_t chunk;          // shard tokens per split (multiple of kTile)
  int32_t row_groups;
  float* ws_o;            // [splits, B*shard_count, R, 512]
  float* ws_lse;          // [splits, B*shard_count, R], base 2
  uint32_t* ws_cnt;       // [B*shard_count*row_groups]
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t w) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)w, __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// 8 key elements at byte offset `off` of a stored row, as floats.
template <bool kFp8>
__device__ __forceinline__ void load8(const uint8_t* row, int d, float (&k)[8]) {
  if constexpr (kFp8) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + d);
    float2 f;
    f = e4m3x2_to_f2((uint16_t)(u.x & 0xFFFF)); k[0] = f.x; k[1] = f.y;
    f = e4m3x2_to_f2((uint16_t)(u.x >> 16));    k[2] = f.x; k[3] = f.y;
    f = e4m3x2_to_f2((uint16_t)(u.y & 0xFFFF)); k[4] = f.x; k[5] = f.y;
    f = e4m3x2_to_f2((uint16_t)(u.y >> 16));    k[6] = f.x; k[7] = f.y;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(row + 2 * d);
    float2 f;
    f = bf16x2_to_f2(u.x); k[0] = f.x; k[1] = f.y;
    f = bf16x2_to_f2(u.y); k[2] = f.x; k[3] = f.y;
    f = bf16x2_to_f2(u.z); k[4] = f.x; k[5] = f.y;
    f = bf16x2_to_f2(u.w); k[6] = f.x; k[7] = f.y;
  }
}

template <bool kFp8>
__device__ __forceinline__ float2 load_v2(const uint8_t* row, int d) {
  if constexpr (kFp8) return e4m3x2_to_f2(*reinterpret_cast<const uint16_t*>(row + d));
  else return bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(row + 2 * d));
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) decode_fma_kernel(const FmaParams fp) {
  constexpr int kRow = kFp8 ? kRowFp8 : kRowBf16;
  constexpr int kChunks = kDK * (kFp8 ? 1 : 2) / 16;   // 16-byte chunks per stored row
  const DecodeArgs& a = fp.a;
  extern __shared__ __align__(16) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem);                        // [kRG][kQStride]
  uint8_t* k_s = smem + kRG * kQStride * 4;                           // [2][kTile][kRow]
  float* p_s = reinterpret_cast<float*>(k_s + 2 * kTile * kRow);      // [kTile][kRG]
  float* alpha_s = p_s + kTile * kRG;                                 // [kRG]
  float* scl_s = alpha_s + kRG;                                       // [2][kTile]
  float* m_s = scl_s + 2 * kTile;                                     // [kRG]
  float* l_s = m_s + kRG;                                             // [kRG]
  __shared__ int bad_s;
  __shared__ int last_s;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, grp = blockIdx.y;
  const int bz = blockIdx.z;
  const int b = bz / a.shard_count, sr = bz % a.shard_count;
  const int r = a.shard_begin + sr;
  const int row0 = grp * kRG;
  const int nrows = min(kRG, a.R - row0);
  const int L = a.seq_lens[b];
  const int32_t* pt_row = a.pt + (int64_t)b * a.max_pages;
  const uint8_t* pool = reinterpret_cast<const uint8_t*>(a.kv.pool[r]);
  const float* spool = a.kv.scale[r];

  if (tid == 0) { bad_s = 0; last_s = 0; }
  __syncthreads();
  int j0 = 0, j1 = 0;
  if (L < a.Tq || (int64_t)L > (int64_t)a.max_pages * a.P * a.c) {
    if (tid == 0) bad_s = DCPMLA_DERR_LENGTH;
  } else {
    const int n = shard_len(L, r, a.c, a.I);   // tokens of b on shard r
    j0 = min(split * fp.chunk, n);
    j1 = min(n, j0 + fp.chunk);
    // Every split checks all of the request's pages, so a bad entry empties the
    // whole (request, shard) result rather than one split of it.
    const int npages = (int)(((int64_t)L + (int64_t)a.P * a.c - 1) / ((int64_t)a.P * a.c));
    for (int pg = tid; pg < npages; pg += kThreads) {
      const int32_t g = pt_row[pg];
      if (g < 0 || (int64_t)g >= a.num_pages) atomicOr(&bad_s, DCPMLA_DERR_PAGE);
    }
  }
  __syncthreads();
  if (bad_s) {
    if (tid == 0) set_err(a.err, bad_s);
    j1 = j0;   // skip the work, emit an empty partial
  }

  // Query rows of this group, pre-scaled into base-2 score units.
  const float qscale = a.sm_scale * kLog2e;
  for (int e = tid; e < kRG * kDK; e += kThreads) {
    const int i = e / kDK, d = e % kDK;
    float v = 0.f;
    if (i < nrows) v = __bfloat162float(a.q[((int64_t)b * a.R + row0 + i) * kDK + d]) * qscale;
    q_s[i * kQStride + d] = v;
  }

  // QK role: warp = query row, lane = token.  PV role: half = row block, k = dim pair.
  const int qi = warp;
  const int qpos = (qi < nrows) ? L - a.Tq + (row0 + qi) / a.H : -1;
  float m_run = -INFINITY, l_run = 0.f;
  const int half = tid >> 8, dp = tid & 255;
  float acc[8][2];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = 0.f;

  auto load_tile = [&](int ts, int buf) {
    uint8_t* dst = k_s + buf * kTile * kRow;
    const int ntok = min(kTile, j1 - ts);
    for (int e = tid; e < ntok * kChunks; e += kThreads) {
      const int tt = e / kChunks, ch = e % kChunks;
      const int64_t slot = shard_slot(pt_row, ts + tt, a.P, a.num_pages);
      cp_async16(dst + tt * kRow + ch * 16, pool + slot * (kDK * (kFp8 ? 1 : 2)) + ch * 16);
    }
    if (kFp8 && tid < ntok) scl_s[buf * kTile + tid] = spool[shard_slot(pt_row, ts + tid, a.P, a.num_pages)];
    cp_async_commit();
  };

  const int ntiles = (j1 - j0 + kTile - 1) / kTile;
  if (ntiles > 0) load_tile(j0, 0);
  for (int it = 0; it < ntiles; ++it) {
    const int ts = j0 + it * kTile, buf = it & 1;
    if (it + 1 < ntiles) {
      load_tile(ts + kTile, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* kt = k_s + buf * kTile * kRow;
    const int ntok = min(kTile, j1 - ts);

    // ---- scores and online softmax (base 2) ----
    {
      float s = 0.f;
      const float* qrow = q_s + qi * kQStride;
      const uint8_t* krow = kt + lane * kRow;
#pragma unroll 4
      for (int d = 0; d < kDK; d += 8) {
        const float4 qa = *reinterpret_cast<const float4*>(qrow + d);
        const float4 qb = *reinterpret_cast<const float4*>(qrow + d + 4);
        float k[8];
        load8<kFp8>(krow, d, k);
        s = fmaf(qa.x, k[0], s); s = fmaf(qa.y, k[1], s);
        s = fmaf(qa.z, k[2], s); s = fmaf(qa.w, k[3], s);
        s = fmaf(qb.x, k[4], s); s = fmaf(qb.y, k[5], s);
        s = fmaf(qb.z, k[6], s); s = fmaf(qb.w, k[7], s);
      }
      const int j = ts + lane;
      const bool vis = (lane < ntok) && (shard_pos(j, r, a.c, a.I) <= qpos);
      float kscale = 1.f;
      if (kFp8 && lane < ntok) kscale = scl_s[buf * kTile + lane];
      s = vis ? s * kscale : -INFINITY;
      float mx = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run, mx);
      float alpha = 1.f, pj = 0.f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m_run - m_new);
        pj = exp2f(s - m_new);
      }
      float sum = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      p_s[lane * kRG + qi] = pj * kscale;     // e4m3: fold the token scale into P
      if (lane == 0) alpha_s[qi] = alpha;
    }
    __syncthreads();

    // ---- P V over the 512-d latent ----
    {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float al = alpha_s[half * 8 + i];
        acc[i][0] *= al;
        acc[i][1] *= al;
      }
      for (int tt = 0; tt < ntok; ++tt) {
        const float2 v = load_v2<kFp8>(kt + tt * kRow, 2 * dp);
        const float4 pa = *reinterpret_cast<const float4*>(p_s + tt * kRG + half * 8);
        const float4 pb = *reinterpret_cast<const float4*>(p_s + tt * kRG + half * 8 + 4);
        const float pr[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[i][0] = fmaf(pr[i], v.x, acc[i][0]);
          acc[i][1] = fmaf(pr[i], v.y, acc[i][1]);
        }
      }
    }
    __syncthreads();
  }

  if (lane == 0) { m_s[qi] = m_run; l_s[qi] = l_run; }
  __syncthreads();

  // ---- epilogue: normalise, write the partial or the shard result ----
  const int64_t R = a.R;
  const bool direct = fp.num_splits == 1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = half * 8 + i;
    if (row >= nrows) continue;
    const float l = l_s[row];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float2 o = make_float2(acc[i][0] * inv, acc[i][1] * inv);
    float* dst = direct ? a.o_part + (((int64_t)sr * a.B + b) * R + row0 + row) * kDL
                        : fp.ws_o + (((int64_t)split * a.B * a.shard_count + bz) * R + row0 + row) * kDL;
    reinterpret_cast<float2*>(dst)[dp] = o;
  }
  if (tid < nrows) {
    const float l = l_s[tid];
    const float lse2 = l > 0.f ? m_s[tid] + log2f(l) : -INFINITY;
    if (direct)
      a.lse_part[((int64_t)sr * a.B + b) * R + row0 + tid] = a.base2 ? lse2 : lse2 * kLn2;
    else
      fp.ws_lse[((int64_t)split * a.B * a.shard_count + bz) * R + row0 + tid] = lse2;
  }
  if (direct) return;

  // ---- split combine by the last CTA to arrive (no waiting) ----
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(fp.ws_cnt + (int64_t)bz * fp.row_groups + grp, 1u);
    last_s = (prev == (uint32_t)fp.num_splits - 1);
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  const int64_t sstride = (int64_t)a.B * a.shard_count * R;
  for (int row = 0; row < nrows; ++row) {
    const int64_t base = (int64_t)bz * R + row0 + row;
    float m = -INFINITY;
    for (int s = 0; s < fp.num_splits; ++s) m = fmaxf(m, __ldcg(fp.ws_lse + s * sstride + base));
    float lse2 = -INFINITY, acc_o = 0.f;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int s = 0; s < fp.num_splits; ++s) sum += exp2f(__ldcg(fp.ws_lse + s * sstride + base) - m);
      lse2 = m + log2f(sum);
      for (int s = 0; s < fp.num_splits; ++s) {
        const float w = exp2f(__ldcg(fp.ws_lse + s * sstride + base) - lse2);
        if (w != 0.f) acc_o = fmaf(w, __ldcg(fp.ws_o + (s * sstride + base) * kDL + tid), acc_o);
      }
    }
    a.o_part[(((int64_t)sr * a.B + b) * R + row0 + row) * kDL + tid] = acc_o;
    if (tid == 0) a.lse_part[((int64_t)sr * a.B + b) * R + row0 + row] = a.base2 ? lse2 : lse2 * kLn2;
  }
}

struct FmaPlan {
  int32_t splits, chunk, row_groups;
  size_t cnt_off, lse_off, o_off, bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

FmaPlan plan_fma(const DecodeArgs& a, int sm_count) {
  FmaPlan p{};
  p.row_groups = (a.R + kRG - 1) / kRG;
  const int64_t units = (int64_t)a.B * a.shard_count * p.row_groups;
  const int64_t n_max = (int64_t)a.max_pages * a.P;   // shard tokens bound
  const int64_t target = 8LL * std::max(sm_count, 1);
  int64_t chunk = (units * n_max + target - 1) / target;
  chunk = std::min<int64_t>(std::max<int64_t>(chunk, 64), 4096);
  chunk = (chunk + kTile - 1) / kTile * kTile;
  p.chunk = (int32_t)chunk;
  p.splits = (int32_t)std::max<int64_t>(1, (n_max + chunk - 1) / chunk);
  if (p.splits == 1) return p;
  const int64_t rows_all = (int64_t)a.B * a.shard_count * a.R;
  p.cnt_off = 0;
  p.lse_off = align256((size_t)units * 4);
  p.o_off = p.lse_off + align256((size_t)p.splits * rows_all * 4);
  p.bytes = p.o_off + (size_t)p.splits * rows_all * kDL * 4;
  return p;
}

size_t smem_bytes(bool fp8) {
  const int row = fp8 ? kRowFp8 : kRowBf16;
  return (size_t)kRG * kQStride * 4 + 2 * kTile * row + kTile * kRG * 4 + kRG * 4 + 2 * kTile * 4 +
         2 * kRG * 4;
}

}  // namespace

size_t fma_workspace_bytes(const DecodeArgs& a, int sm_count) { return plan_fma(a, sm_count).bytes; }

int launch_decode_fma(const DecodeArgs& a, void* ws, size_t ws_bytes, int sm_count, cudaStream_t st) {
  const FmaPlan plan = plan_fma(a, sm_count);
  if (ws_bytes < plan.bytes || (plan.bytes && !ws)) return DCPMLA_ERR_CAPACITY;
  // every refusal comes before the first enqueue: a refused call leaves the workspace alone
  const int64_t z = (int64_t)a.B * a.shard_count;
  if (z > 65535 || plan.row_groups > 65535) return DCPMLA_ERR_UNSUPPORTED;
  const size_t smem = smem_bytes(a.fp8);
  const auto kern = a.fp8 ? decode_fma_kernel<true> : decode_fma_kernel<false>;
  if (ensure_smem_attr((const void*)kern, (int)smem) != DCPMLA_OK) return DCPMLA_ERR_CUDA;
  FmaParams fp{};
  fp.a = a;
  fp.num_splits = plan.splits;
  fp.chunk = plan.chunk;
  fp.row_groups = plan.row_groups;
  if (plan.splits > 1) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    fp.ws_cnt = reinterpret_cast<uint32_t*>(w + plan.cnt_off);
    fp.ws_lse = reinterpret_cast<float*>(w + plan.lse_off);
    fp.ws_o = reinterpret_cast<float*>(w + plan.o_off);
    const size_t cnt_bytes = (size_t)a.B * a.shard_count * plan.row_groups * 4;
    if (cudaMemsetAsync(fp.ws_cnt, 0, cnt_bytes, st) != cudaSuccess) return DCPMLA_ERR_CUDA;
  }
  const dim3 grid((unsigned)plan.splits, (unsigned)plan.row_groups, (unsigned)z);
  kern<<<grid, kThreads, smem, st>>>(fp);
  return launch_status();
}

}  // namespace dcpmla
