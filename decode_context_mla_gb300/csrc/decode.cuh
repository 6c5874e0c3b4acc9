// Arguments of one dcpmla_decode call after host-side validation, shared by
// the decode kernels.
#pragma once
#include <cuda.h>

#include <mutex>
#include <new>

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

// ---------------------------------------------------------------------------
// Host-side reuse of prepared launches.  A decode call's kernel parameters (the
// encoded tensor maps among them) depend only on its arguments, so a call that
// repeats an earlier one (same pointers, shapes, workspace and device) reuses the
// block prepared then instead of encoding it again.
// ---------------------------------------------------------------------------
struct LaunchKey {
  uint64_t w[80];
  int n = 0;
  void add(uint64_t v) {
    if (n < 80) w[n] = v;
    ++n;
  }
  bool operator==(const LaunchKey& o) const {
    if (n != o.n || n > 80) return false;
    for (int i = 0; i < n; ++i)
      if (w[i] != o.w[i]) return false;
    return true;
  }
};

// Every argument the preparation reads, plus the workspace, a kernel tag and the device.
LaunchKey launch_key(const DecodeArgs& a, const void* ws, size_t ws_bytes, int tag);

// A few prepared parameter blocks of one kind, least recently used evicted.  The caller
// holds `mu` from get() until its launches have been enqueued.
template <class Params, int kSlots = 8>
struct ParamCache {
  std::mutex mu;
  struct Slot {
    LaunchKey key;
    Params* p = nullptr;
    uint64_t used = 0;
  };
  Slot slots[kSlots];
  uint64_t tick = 0;
  // The block for `key`; `fresh` is set when it was (re)zeroed and must be filled.
  // nullptr when no memory could be had.
  Params* get(const LaunchKey& key, bool& fresh) {
    if (key.n > 80) {
      fresh = true;
      return nullptr;
    }
    Slot* victim = &slots[0];
    for (Slot& s : slots) {
      if (s.p && s.key == key) {
        s.used = ++tick;
        fresh = false;
        return s.p;
      }
      if (!s.p || s.used < victim->used) victim = &s;
    }
    if (!victim->p) victim->p = new (std::nothrow) Params();
    if (!victim->p) return nullptr;
    *victim->p = Params{};
    victim->key = key;
    victim->used = ++tick;
    fresh = true;
    return victim->p;
  }
  // Forget a block whose preparation failed.
  void drop(const Params* p) {
    for (Slot& s : slots)
      if (s.p == p) s.key.n = -1;
  }
};

// Limit after which a decode pipeline wait gives up, in units of 1024 clock64 cycles: about
// one second unless a test has lowered it (dcpmla_testing_set_wait_limit).
constexpr int32_t kDefaultWaitKcycles = 2000000000 / 1024;
int32_t pipeline_wait_kcycles();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (function, device).
int ensure_smem_attr(const void* func, int bytes);

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
