// Shared device/host helpers for the libdcpmla CUDA sources.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dcpmla.h"

namespace dcpmla {

constexpr int kDL = DCPMLA_D_LATENT;   // 512
constexpr int kDR = DCPMLA_D_ROPE;     // 64
constexpr int kDK = DCPMLA_D_K;        // 576
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct ShardPtrs {
  void* pool[DCPMLA_MAX_SHARDS];
  float* scale[DCPMLA_MAX_SHARDS];
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? DCPMLA_OK : DCPMLA_ERR_CUDA;
}

// SM count of the current device (cached per device id).
int device_sm_count();

// Tokens go to shards in runs of `I` consecutive positions, round-robin (vLLM DCP
// study page, configuration example: the KV interleave size; I = 1 is the SGLang
// layout owner = v mod c).  Global position of shard r's local token j:
// (j is a shard-local index, < 2^31; I = 1, the common layout, needs no division)
__host__ __device__ __forceinline__ int64_t shard_pos(int32_t j, int32_t r, int32_t c, int32_t I) {
  if (I == 1) return (int64_t)j * c + r;
  const int32_t q = j / I;
  return (int64_t)q * I * c + (int64_t)r * I + (j - q * I);
}
// Number of the first L positions that shard r holds (L < 2^31; 32-bit arithmetic,
// which also keeps a 64-bit division helper out of the decode kernels).
__host__ __device__ __forceinline__ int32_t shard_len(int32_t L, int32_t r, int32_t c, int32_t I) {
  const int32_t round = I * c, full = L / round;
  int32_t extra = L - full * round - r * I;
  extra = extra < 0 ? 0 : (extra > I ? I : extra);
  return full * I + extra;
}

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

// Shard-local token j of request b lives on shard r at this physical slot:
// virtual page j / P of the request (one widened page of P*c positions is one
// physical page of P slots per shard), offset j % P.  Returns -1 for a page
// entry outside [0, num_pages).
__device__ __forceinline__ int64_t shard_slot(const int32_t* pt_row, int32_t j, int32_t P,
                                              int64_t num_pages) {
  const int32_t g = __ldg(pt_row + j / P);
  if (g < 0 || (int64_t)g >= num_pages) return -1;
  return (int64_t)g * P + (j % P);
}

}  // namespace dcpmla
