/*
 * dcpmla.h -- C ABI of libdcpmla: striped absorbed-MLA decode with an exact
 * log-sum-exp merge (decode context parallelism, DCP), all shards on one GPU.
 *
 * The c "ranks" of a DCP group are c separate physical KV pools resident in
 * the same GPU's memory.  Position p of a request lives at virtual slot v; the
 * shard that owns v is v mod c and it keeps the row at physical slot
 * floor(v / c) of its own pool.  Each shard computes a locally normalised
 * partial output and its LSE over only its own tokens; the merge combines the
 * partials exactly.
 *
 * Conventions for every call
 *   - Return value: DCPMLA_OK (0) or a negative DCPMLA_ERR_* status.  No C++
 *     exception crosses this boundary.  dcpmla_status_string() names a status.
 *   - Host objects (allocator, request map) are owned by the library and
 *     freed by their *_destroy call.  Every device buffer is owned by the
 *     caller; the library never allocates or frees device memory.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  Host-side argument checks
 *     happen before anything is enqueued; a failing check enqueues nothing.
 *   - Problems that only the GPU can see (a page id outside the pool, a
 *     length beyond the page table) are OR'd into the caller's device word
 *     *d_err as DCPMLA_DERR_* bits; the affected work is skipped and its
 *     outputs are written as empty (o = 0, lse = -inf).  Kernels never trap.
 *     Read d_err after synchronising the stream.
 *   - Device pointers must be 16-byte aligned; rows are contiguous.
 *   - Dimensions: latent D_L = 512, rope D_R = 64, key D_K = 576.
 */
#ifndef DCPMLA_H
#define DCPMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCPMLA_D_LATENT 512
#define DCPMLA_D_ROPE 64
#define DCPMLA_D_K 576
#define DCPMLA_MAX_SHARDS 64

/* Status codes. */
#define DCPMLA_OK 0
#define DCPMLA_ERR_INVALID (-1)     /* bad argument: null/misaligned pointer, c < 1, P < 1, sizes */
#define DCPMLA_ERR_UNSUPPORTED (-2) /* valid but not implemented (dtype, shape)                  */
#define DCPMLA_ERR_CAPACITY (-3)    /* allocator exhausted / table too small / workspace short  */
#define DCPMLA_ERR_CUDA (-4)        /* a CUDA launch or runtime call failed                     */
#define DCPMLA_ERR_TIMEOUT (-5)     /* a bounded device wait gave up                            */

/* Device error bits (OR'd into *d_err). */
#define DCPMLA_DERR_PAGE 1      /* a page-table entry in use is outside [0, num_pages)        */
#define DCPMLA_DERR_POSITION 2  /* a position lies outside the request's pages                */
#define DCPMLA_DERR_SLOT 4      /* an owner / physical slot handed to kv_append is out of range */
#define DCPMLA_DERR_LENGTH 8    /* seq_len < Tq, or longer than max_pages * P * c             */
#define DCPMLA_DERR_TIMEOUT 16  /* a bounded wait inside a kernel gave up; outputs are invalid */

/* KV storage formats. */
#define DCPMLA_KV_BF16 0 /* row = 576 bf16 (512 latent then 64 rope), 1152 B                 */
#define DCPMLA_KV_E4M3 1 /* row = 576 OCP E4M3FN codes, 576 B, plus one fp32 scale per token  */

/* LSE bases. */
#define DCPMLA_LSE_E 0
#define DCPMLA_LSE_2 1

const char* dcpmla_status_string(int status);
int dcpmla_version(void);

/* ------------------------------------------------------------------------
 * Shared virtual allocator (host).
 * SGLang "Decode Context Parallelism" docs, Architecture > Virtual KV layout:
 * each rank has physical capacity C tokens in pages of P tokens; the DCP group
 * exposes one allocator with virtual capacity C*c and virtual page size P*c.
 * Page id g names virtual page g (virtual slots g*P*c .. g*P*c+P*c-1), which is
 * physical page g (slots g*P .. g*P+P-1) in every shard pool.
 *
 * dcpmla_alloc_create: c in [1, DCPMLA_MAX_SHARDS], P >= 1, C a multiple of P.
 *   initial_order: NULL (free list 0..C/P-1) or a host array of C/P page ids
 *   that must be a permutation; pages are taken from the front of the free
 *   list and returned to its back.  *out receives a handle owned by the
 *   library.  ERR_INVALID on bad geometry or a non-permutation.
 * dcpmla_alloc_pages: all-or-nothing; ERR_CAPACITY if fewer than n pages are
 *   free (nothing is taken).  out_ids: host array of n int32.
 * dcpmla_free_pages: ERR_INVALID if an id is not currently allocated (then
 *   nothing is freed).
 * ------------------------------------------------------------------------ */
typedef struct dcpmla_alloc dcpmla_alloc;
int dcpmla_alloc_create(int32_t c, int64_t phys_capacity_tokens, int32_t phys_page,
                        const int32_t* initial_order, dcpmla_alloc** out);
int dcpmla_alloc_destroy(dcpmla_alloc* a);
int dcpmla_alloc_geometry(const dcpmla_alloc* a, int32_t* c, int32_t* phys_page,
                          int32_t* virtual_page, int64_t* num_pages, int64_t* virtual_capacity);
int dcpmla_alloc_free_count(const dcpmla_alloc* a, int64_t* out);
int dcpmla_alloc_pages(dcpmla_alloc* a, int32_t n, int32_t* out_ids);
int dcpmla_free_pages(dcpmla_alloc* a, int32_t n, const int32_t* ids);

/* vLLM "Context Parallel Deployment", Decode Context Parallel: the effective
 * attention block size with DCP is the physical block times the DCP size
 * (DCP 4: a 16-token physical block stands for 64 tokens).  *out = P*c. */
int dcpmla_effective_page_size(const dcpmla_alloc* a, int32_t* out);

/* ------------------------------------------------------------------------
 * Request -> token map (host).
 * SGLang DCP docs, Virtual KV layout: every rank sees the same request-to-token
 * map.  Request b's positions 0..len-1 are laid out in order over its list of
 * virtual pages: position p is virtual slot pages[p / (P*c)]*(P*c) + p % (P*c).
 *
 * dcpmla_reqmap_create: requests are ids 0..max_requests-1, each with at most
 *   max_pages_per_request pages.  The map borrows `a` (which must outlive it).
 * dcpmla_reqmap_extend: grows request `req` by n_new >= 0 tokens, allocating
 *   virtual pages as needed; all-or-nothing (ERR_CAPACITY leaves the map and
 *   the allocator unchanged).  *out_first_position (may be NULL) receives the
 *   first new position.
 * dcpmla_reqmap_release: returns the request's pages to the allocator.
 * dcpmla_reqmap_page_table: writes a host row-major [n_reqs, max_pages] int32
 *   table (unused entries = pad) and, if out_seq_lens is not NULL, the lengths.
 *   ERR_CAPACITY if a request holds more than max_pages pages.
 * ------------------------------------------------------------------------ */
typedef struct dcpmla_reqmap dcpmla_reqmap;
int dcpmla_reqmap_create(dcpmla_alloc* a, int32_t max_requests, int32_t max_pages_per_request,
                         dcpmla_reqmap** out);
int dcpmla_reqmap_destroy(dcpmla_reqmap* m);
int dcpmla_reqmap_extend(dcpmla_reqmap* m, int32_t req, int64_t n_new, int64_t* out_first_position);
int dcpmla_reqmap_release(dcpmla_reqmap* m, int32_t req);
int dcpmla_reqmap_length(const dcpmla_reqmap* m, int32_t req, int64_t* out);
int dcpmla_reqmap_page_table(const dcpmla_reqmap* m, const int32_t* reqs, int32_t n_reqs,
                             int32_t max_pages, int32_t pad, int32_t* out_table,
                             int32_t* out_seq_lens);

/* Interleave size (vLLM DCP study page, configuration example: the DCP KV
 * interleave size, default 1 token): tokens go to ranks in runs of
 * `interleave` consecutive virtual slots, round-robin over the c ranks:
 *   owner(v) = floor(v / I) mod c,   physical(v) = floor(v / (I*c)) * I + v mod I,
 * which for I = 1 is the SGLang layout owner = v mod c, physical = floor(v / c).
 * I must divide P, so that a widened page of P*c slots is still one physical
 * page of P slots on every rank (page id g on every pool); a call with I < 1 or
 * P mod I != 0 returns DCPMLA_ERR_INVALID.  Shard r's local token j is then
 * global position floor(j / I) * I * c + r * I + j mod I. */

/* Host position map (same arithmetic as dcpmla_slot_map, on host arrays).
 * For i < n: request req[i] (a row of page_table [*, max_pages]), position
 * pos[i] -> vslot[i], owner[i] and phys[i] as above (I = interleave).
 * ERR_INVALID if a position's page entry is negative or beyond max_pages. */
int dcpmla_map_positions(const int32_t* page_table, int32_t max_pages, int32_t c,
                         int32_t interleave, int32_t P, const int32_t* req, const int64_t* pos,
                         int64_t n, int64_t* vslot, int32_t* owner, int64_t* phys);

/* ------------------------------------------------------------------------
 * Device slot map (SGLang DCP docs, Virtual KV layout: owner(v) = v mod c,
 * physical(v) = floor(v / c); with interleave I as stated above).
 * d_page_table: device int32 [n_requests, max_pages]; d_req, d_pos: device
 * arrays of n request indices / positions.  Writes d_vslot (int64), d_owner
 * (int32) and d_phys (int64), each of n entries; any output pointer may be
 * NULL.  A request index outside [0, n_requests), a page entry outside
 * [0, num_pages) or a position past max_pages*P*c sets DCPMLA_DERR_POSITION /
 * DCPMLA_DERR_PAGE and writes owner = -1, vslot = phys = -1 for that entry.
 * ------------------------------------------------------------------------ */
int dcpmla_slot_map(const int32_t* d_page_table, int32_t n_requests, int32_t max_pages,
                    int64_t num_pages, int32_t c, int32_t interleave, int32_t P, const int32_t* d_req,
                    const int64_t* d_pos, int64_t n, int64_t* d_vslot, int32_t* d_owner,
                    int64_t* d_phys, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * KV append: the compacting write (SGLang DCP docs, Virtual KV layout: on
 * write a rank keeps only its own positions and compacts them into its
 * physical pool).  Row i is written only to pool owner[i], at physical slot
 * phys[i]; an owner of -1 skips the row; any other out-of-range owner or slot
 * sets DCPMLA_DERR_SLOT and skips it.
 *
 * pools: HOST array of c device pointers; pool r holds pool_rows rows of 576
 *   elements in the storage format (bf16 or E4M3 codes).
 * scale_pools: HOST array of c device float pointers ([pool_rows] each) for
 *   E4M3, NULL for bf16.
 * d_ckv: n rows of the 512-d latent, row stride ckv_stride elements;
 * d_krope: n rows of the 64-d rope key, row stride krope_stride elements;
 *   both already in the storage format.  d_row_scales: n fp32 scales (E4M3).
 * The copy is bit-exact.  Strides must keep every row 16-byte aligned.
 * ------------------------------------------------------------------------ */
int dcpmla_kv_append(void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                     int64_t pool_rows, int32_t c, const int32_t* d_owner, const int64_t* d_phys,
                     const void* d_ckv, int64_t ckv_stride, const void* d_krope,
                     int64_t krope_stride, const float* d_row_scales, int64_t n, int32_t* d_err,
                     void* stream);

/* ------------------------------------------------------------------------
 * Shard-local absorbed-MLA decode (SGLang DCP docs, MLA decode dataflow and
 * DCP x speculative decoding; vLLM GLM-5.3 serving post, footnote arithmetic
 * for the 576-d scores and 512-d values).
 *
 * For every request b, query token t < Tq, head h and shard r in
 * [shard_begin, shard_begin + shard_count):
 *   shard-local token j of request b is global position p = j*c + r (with
 *   interleave I: floor(j/I)*I*c + r*I + j mod I), stored in pool r at
 *   physical slot page_table[b][j / P]*P + j % P; it is visible to
 *   query t iff p <= L_b - Tq + t (causality over global positions);
 *   s_j   = sm_scale * (q[b,t,h,:] . key_j)  over all 576 dims
 *           (E4M3: key_j = code_j * scale_j);
 *   o_r   = sum_j softmax(s)_j * key_j[0:512]   (normalised over shard r only);
 *   lse_r = ln sum_j e^{s_j}  (DCPMLA_LSE_E) or that / ln 2 (DCPMLA_LSE_2).
 * A shard with no visible token gives o_r = 0 and lse_r = -inf.
 *
 * d_q: bf16 [B, Tq, H, 576] (512 absorbed latent query then 64 rope query).
 * pools / scale_pools: as in dcpmla_kv_append (HOST arrays of c device
 *   pointers, indexed by absolute shard id).
 * d_page_table: int32 [B, max_pages]; d_seq_lens: int32 [B], the GLOBAL
 *   context length L_b (tokens attended, including the Tq query tokens).
 * d_o_part: fp32 [shard_count, B, Tq, H, 512]; d_lse_part: fp32
 *   [shard_count, B, Tq, H] (index 0 = shard_begin).
 * d_workspace: device scratch of at least dcpmla_decode_workspace_size()
 *   bytes for the same arguments (may be NULL when that size is 0); the call
 *   clears what it needs.  Calls sharing a workspace must not overlap.
 * Supported: Tq in [1, 16], H*Tq in [1, 1024], kv_dtype bf16 or E4M3.
 * Arithmetic: fp32 accumulation on every path.  bf16 KV: the output is within
 * 2e-3 (max over rows of |err|_inf / |o|_inf) of the exact result on N(0,1)
 * data.  E4M3 KV on the tensor cores: codes convert exactly to fp16, the query
 * is rounded to fp16, P to fp16 (pre-multiplied by the value scale), and the
 * two partial sums that make up the 576-d score (CTA pair halves) are each
 * rounded to fp16 at 2^-10 scale before they are added (partials beyond ~6.7e7
 * code units saturate): within 1e-2 of the result on the dequantised keys
 * (~2e-3 on N(0,1) data).
 * ------------------------------------------------------------------------ */
int dcpmla_decode(const void* d_q, void* const* pools, float* const* scale_pools,
                  int32_t kv_dtype, int64_t pool_rows, const int32_t* d_page_table,
                  int32_t max_pages, const int32_t* d_seq_lens, int32_t B, int32_t Tq, int32_t H,
                  int32_t P, int32_t c, int32_t interleave, int32_t shard_begin,
                  int32_t shard_count, float sm_scale, int32_t lse_base, float* d_o_part,
                  float* d_lse_part, void* d_workspace, size_t ws_bytes, int32_t* d_err,
                  void* stream);

/* Bytes of device workspace dcpmla_decode needs for the same B, Tq, H, P, c,
 * shard_count, kv_dtype and max_pages (every L_b is at most max_pages*P*c).
 * The answer depends on the current device's SM count. */
int dcpmla_decode_workspace_size(int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
                                 int32_t shard_count, int32_t kv_dtype, int32_t max_pages,
                                 size_t* out);

/* Which decode kernels dcpmla_decode runs for the same arguments as
 * dcpmla_decode_workspace_size, on the current device (host only, no launch):
 *   *path = DCPMLA_PATH_TC_FEWHEAD: tensor cores with the KV tokens as the MMA's
 *           M dimension (at most 16 query rows H*Tq, at least 16 in the batch,
 *           bf16 KV, at most 8 shards in the call, P a multiple of 8);
 *           DCPMLA_PATH_TC_ROWS: tensor cores on 128-row query tiles (at most 8
 *           shards in the call, P a multiple of 64 or a divisor of 64 that is a
 *           multiple of 8);
 *           DCPMLA_PATH_CUDA_CORE: CUDA-core kernel (other shapes);
 *   *kernel_launches = kernels one dcpmla_decode call enqueues (memsets excluded).
 * Either output pointer may be NULL. */
#define DCPMLA_PATH_TC_FEWHEAD 1
#define DCPMLA_PATH_TC_ROWS 2
#define DCPMLA_PATH_CUDA_CORE 3
int dcpmla_decode_path(int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c, int32_t shard_count,
                       int32_t kv_dtype, int32_t max_pages, int32_t* path, int32_t* kernel_launches);

/* ------------------------------------------------------------------------
 * Fused decode + merge (SGLang DCP docs, MLA decode dataflow: every shard's
 * locally normalised (o_r, lse_r) goes into the exact LSE merge).  Decodes all
 * c shards of every request as dcpmla_decode does and writes the merged result
 * directly: d_o fp32 [B, Tq, H, 512] = sum_r b^(lse_r - lse) o_r and d_lse fp32
 * [B, Tq, H] = log_b sum_r b^(lse_r), in lse_base; there is no per-shard output.
 * The bf16 tensor-core paths write no per-shard output (the token-major path and
 * the persistent 128-row grid end in one merge kernel over every partial of the
 * request, the non-persistent 128-row kernel merges in the last CTA of each
 * request's row tile); E4M3 on the tensor cores and the CUDA-core path decode
 * into per-shard partials in the workspace and then run the LSE merge.  A shard that needed a bad page id is
 * left out of the merge (DCPMLA_DERR_PAGE is set), like its empty partial in
 * the unfused path.  Arguments as in dcpmla_decode; d_workspace: at least
 * dcpmla_decode_merged_workspace_size() bytes for the same shape.
 * ------------------------------------------------------------------------ */
int dcpmla_decode_merged_workspace_size(int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
                                        int32_t kv_dtype, int32_t max_pages, size_t* out);
int dcpmla_decode_merged(const void* d_q, void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                         int64_t pool_rows, const int32_t* d_page_table, int32_t max_pages,
                         const int32_t* d_seq_lens, int32_t B, int32_t Tq, int32_t H, int32_t P, int32_t c,
                         int32_t interleave, float sm_scale, int32_t lse_base, float* d_o, float* d_lse,
                         void* d_workspace, size_t ws_bytes, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * Token relayout, DCP-1 prefill cache -> striped decode pools (SGLang DCP
 * docs, DCP x PD disaggregation: dense prefill pages are not copied straight
 * into striped storage; a DCP-1 prefill feeds DCP decode through a token
 * relayout whose plan carries the exact token count, so a partial final page
 * leaks no stale rows; page size and KV dtype match on both sides).
 *
 * For request b < B and each position p < d_seq_lens[b], the stored row at
 * dense slot d_dense_page_table[b][p / P] * P + p % P of d_dense is copied
 * byte for byte to pools[owner(p)] at physical(p), with owner and physical from
 * d_page_table (virtual pages of P*c) and the interleave size (as in
 * dcpmla_slot_map); for E4M3 the fp32 scale d_dense_scales[dense slot] goes to
 * scale_pools[owner][physical].  Nothing else is written.
 * d_dense: [dense_rows, 576] rows of kv_dtype (1152 B bf16, 576 B E4M3),
 *   16-byte aligned; d_dense_page_table: int32 [B, dense_max_pages];
 * pools / scale_pools: HOST arrays of c device pointers, as in
 *   dcpmla_kv_append; d_page_table: int32 [B, max_pages]; d_seq_lens: int32 [B].
 * Device errors: a length above dense_max_pages*P or max_pages*P*c sets
 * DCPMLA_DERR_LENGTH and skips the request; a page id outside either pool sets
 * DCPMLA_DERR_PAGE and skips that token.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
int dcpmla_relayout_dense_to_striped(const void* d_dense, const float* d_dense_scales, int64_t dense_rows,
                                     const int32_t* d_dense_page_table, int32_t dense_max_pages,
                                     void* const* pools, float* const* scale_pools, int32_t kv_dtype,
                                     int64_t pool_rows, const int32_t* d_page_table, int32_t max_pages,
                                     const int32_t* d_seq_lens, int32_t B, int32_t P, int32_t c,
                                     int32_t interleave, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * Un-stripe gather, striped pools -> one contiguous copy per request in token
 * order (SGLang DCP docs, Communication backends: extend gathers the cached
 * prefix shards and restores token order; vLLM GLM-5.3 serving post, DCP
 * section: a temporary full-context copy of the shards).
 *
 * d_out[b][p] (rows of kv_dtype, [B, out_capacity, 576], 16-byte aligned) =
 * pools[owner(p)][physical(p)] for p < d_seq_lens[b]; for E4M3 also
 * d_out_scales[b][p] ([B, out_capacity] fp32).  Rows at p >= d_seq_lens[b] are
 * not written.  Errors as for the relayout (a length above out_capacity or
 * max_pages*P*c sets DCPMLA_DERR_LENGTH).
 * ------------------------------------------------------------------------ */
int dcpmla_gather_unstriped(void* const* pools, float* const* scale_pools, int32_t kv_dtype, int64_t pool_rows,
                            const int32_t* d_page_table, int32_t max_pages, const int32_t* d_seq_lens, int32_t B,
                            int32_t P, int32_t c, int32_t interleave, void* d_out, float* d_out_scales,
                            int64_t out_capacity, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * E4M3 quantising append: like dcpmla_kv_append into E4M3 pools, but from bf16
 * rows, computing each token's scale (the FP8 cache with one fp32 scale per
 * token that the FP8 workload stores).  In float32: amax = max |x| over the 576
 * values, scale = amax / 448 (IEEE division), code = E4M3FN(clamp(x / scale,
 * -448, 448)) rounded to nearest-even (IEEE signed zero); a row of zeros gets
 * scale 0 and zero codes.  Codes go to pools[owner][phys], the scale to
 * scale_pools[owner][phys].
 * d_ckv: bf16 [n, ckv_stride] (first 512 used), d_krope: bf16 [n, krope_stride]
 * (first 64 used), both 16-byte aligned with strides in elements that keep
 * rows 16-byte aligned; d_owner / d_phys as from dcpmla_slot_map.  An entry
 * with owner outside [0, c) or phys outside [0, pool_rows) sets
 * DCPMLA_DERR_SLOT and is skipped.
 * ------------------------------------------------------------------------ */
int dcpmla_kv_append_e4m3(void* const* pools, float* const* scale_pools, int64_t pool_rows, int32_t c,
                          const int32_t* d_owner, const int64_t* d_phys, const void* d_ckv, int64_t ckv_stride,
                          const void* d_krope, int64_t krope_stride, int64_t n, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * HiCache index filter (SGLang DCP docs, DCP x HiCache L2: the controller
 * addresses P*c slots per widened page while each buffer stores its P local
 * rows; before a host<->device transfer both index lists keep the positions
 * this rank owns and map i to floor(i / c)).
 *
 * d_idx: int64 [n] slots in widened-page space.  Writes, in input order, the
 * local slot of every entry that `rank` owns (owner / physical with the
 * interleave size, floor(i / c) for interleave 1) to d_out (int64, room for n)
 * and their number to *d_count (device int64).  A negative index sets
 * DCPMLA_DERR_POSITION and is dropped.  d_workspace: at least
 * dcpmla_hicache_filter_workspace_size(n) bytes (ERR_CAPACITY otherwise); the
 * call clears it.  One pass: blocks wait (bounded) for their predecessors'
 * counts; a wait that runs out sets DCPMLA_DERR_TIMEOUT (outputs invalid).
 * ------------------------------------------------------------------------ */
int dcpmla_hicache_filter_workspace_size(int64_t n, size_t* out);
int dcpmla_hicache_filter(const int64_t* d_idx, int64_t n, int32_t c, int32_t interleave, int32_t rank,
                          int64_t* d_out, int64_t* d_count, void* d_workspace, size_t ws_bytes, int32_t* d_err,
                          void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free decode.  The pages have no counterpart to this call: it is
 * a library convenience.
 *
 * Some callers cannot allocate device memory where they run the decode: a
 * plugin whose host framework owns all device memory and forbids allocation
 * in its enqueue path, a process whose memory is already fully reserved by a
 * caching allocator, or a latency-critical loop in which cudaMalloc/cudaFree
 * would synchronise the device.  This call takes the same arguments as
 * dcpmla_decode minus the workspace and the interleave size (it serves the
 * plain striping, interleave 1) and computes the same result with the
 * CUDA-core decode kernel; its split-KV scratch is a static device array of
 * DCPMLA_NOALLOC_SCRATCH_BYTES that every GPU loading the library keeps until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *   - Shapes whose scratch need exceeds DCPMLA_NOALLOC_SCRATCH_BYTES are
 *     rejected with DCPMLA_ERR_CAPACITY before anything is enqueued (use
 *     dcpmla_decode with a caller workspace for those).
 *   - The first call on each device looks up the scratch array's device
 *     address (with that device current) and caches it; make that first call
 *     before any stream capture.
 *   - All calls share the one array; the call clears what must start at zero.
 *     Calls that overlap on the GPU (other streams, other threads) race on it:
 *     order them on one stream or synchronise between them.
 * ------------------------------------------------------------------------ */
#define DCPMLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int dcpmla_decode_noalloc(const void* d_q, void* const* pools, float* const* scale_pools,
                          int32_t kv_dtype, int64_t pool_rows, const int32_t* d_page_table,
                          int32_t max_pages, const int32_t* d_seq_lens, int32_t B, int32_t Tq,
                          int32_t H, int32_t P, int32_t c, int32_t shard_begin,
                          int32_t shard_count, float sm_scale, int32_t lse_base, float* d_o_part,
                          float* d_lse_part, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * Testing only: the limit of the tensor-core decode kernels' pipeline waits.
 * The pages have no counterpart to this call.
 *
 * Every wait inside the tensor-core decode kernels (a TMA tile landing, an MMA
 * completing, the peer CTA's partial scores arriving) gives up after a limit
 * of clock64 cycles, about one second by default.  A wait that gives up sets
 * DCPMLA_DERR_TIMEOUT in *d_err and aborts its CTA: every role leaves its
 * loop, the copies and MMAs already issued are waited for, TMEM is freed, and
 * the kernel returns; that call's outputs are invalid (some may be left
 * unwritten).  This call sets the limit for decode launches enqueued after it,
 * rounded down to a multiple of 1024 cycles (so cycles < 1024 makes every wait
 * that is not already satisfied give up at once; cycles <= 0 restores the
 * default); it exists so that tests can make the
 * waits run out on purpose and check that the error is reported and the
 * context stays usable.  Process-wide; not for production use.
 * ------------------------------------------------------------------------ */
int dcpmla_testing_set_wait_limit(int64_t cycles);

/* ------------------------------------------------------------------------
 * Exact LSE merge (SGLang DCP docs, MLA decode dataflow): for every row,
 *   lse = log_b sum_r b^{lse_r},   o = sum_r b^{lse_r - lse} * o_r,
 * with b = e or 2 (the decode's LSE base); the maximum is factored out so no
 * power overflows; an all -inf row gives o = 0, lse = -inf.
 * d_o_part: fp32 [c, rows, 512]; d_lse_part: fp32 [c, rows];
 * d_o: fp32 [rows, 512]; d_lse: fp32 [rows] (may be NULL).  With c = 1 the
 * output equals the input bit for bit.
 * ------------------------------------------------------------------------ */
int dcpmla_lse_merge(const float* d_o_part, const float* d_lse_part, int32_t c, int64_t rows,
                     int32_t lse_base, float* d_o, float* d_lse, int32_t* d_err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DCPMLA_H */
