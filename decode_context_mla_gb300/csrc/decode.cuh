// Arguments of one dcpmla_decode call after host-side validation, shared by
// the decode kernels.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace dcpmla {

struct DecodeArgs {
  const __nv_bfloat16* q;   // [B, Tq, H, 576]
  ShardPtrs kv;             // indexed by absolute shard id
  bool fp8;
  int64_t pool_rows;
  int64_t num_pages;        // pool_rows / P
  const int32_t* pt;        // [B, max_pages]
  int32_t max_pages;
  const int32_t* seq_lens;  // [B], global lengths
  int32_t B, Tq, H, R, P, c, shard_begin, shard_count;
  int32_t I;                // interleave size: tokens go to shards in runs of I
  float sm_scale;
  bool base2;
  float* o_part;            // [shard_count, B, R, 512]
  float* lse_part;          // [shard_count, B, R]
  int32_t* err;
};

// 2-D tensor map over a row-major bf16 matrix [rows, cols] with 128-byte swizzle.
int tma_encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                       uint32_t box_rows);
// A bf16 pool [rows, 576] viewed as {64 dims, 8 rows, 9 chunks of 64 dims, rows / 8 row
// groups}: one box {64, 8, chunks, groups} lands as [group][chunk][8 rows x 128 B]
// 128-byte-swizzle atoms (rows % 8 == 0).
int tma_encode_kv_rowgroups(CUtensorMap* m, const void* base, uint64_t rows, uint32_t chunks, uint32_t groups);

// Tensor-core path for few query rows (<= 16): KV tokens are the MMA's M dimension.
bool fh_supported(const DecodeArgs& a, int sm_count);
size_t fh_workspace_bytes(const DecodeArgs& a, int sm_count);
// fused: write every unit to the workspace and merge all shards into o = a.o_part
// [B, R, 512], lse = a.lse_part [B, R] (shard_count must be c).
int launch_decode_fh(const DecodeArgs& a, void* ws, size_t ws_bytes, int sm_count, cudaStream_t st,
                     bool fused = false);

// Tensor-core path (tcgen05 / TMEM / TMA): 128-row query tiles, bf16 or e4m3 KV.
bool tc_supported(const DecodeArgs& a);
size_t tc_workspace_bytes(const DecodeArgs& a, int sm_count, bool fused = false);
// kernel launches of one launch_decode_tc call (the persistent bf16 grid: prefix, decode, combine)
int tc_kernel_launches(const DecodeArgs& a, bool fused = false);
// fused: as for launch_decode_fh (every shard and split merged into o, lse).
int launch_decode_tc(const DecodeArgs& a, void* ws, size_t ws_bytes, int sm_count, cudaStream_t st,
                     bool fused = false);

// Generic CUDA-core path (any head count, bf16 or e4m3).
size_t fma_workspace_bytes(const DecodeArgs& a, int sm_count);
int launch_decode_fma(const DecodeArgs& a, void* ws, size_t ws_bytes, int sm_count,
                      cudaStream_t st);

}  // namespace dcpmla
