/*
 * slora.h -- C ABI of the GB300 heterogeneous-batch LoRA library (libslora.so).
 *
 * The library implements the data-parallel hot path of S-LoRA ("S-LoRA:
 * Serving Thousands of Concurrent LoRA Adapters", MLSys 2024): for every
 * token i of one batch, with its own adapter a = a(i) of its own rank r_a,
 *
 *     y_i  +=  s * (x_i A_a) B_a
 *
 * where the rows of A_a and B_a are not contiguous tensors but sit on pages
 * of one unified pool that the adapters share with the KV cache.
 *   - Unified Paging: one pool of fixed-size pages holds adapter weights of
 *     different ranks and KV tensors of different lengths (nubint.ai review,
 *     abstract and method list; dongaigc.com summary, section 1).
 *   - Adapters live in host memory and are fetched to the GPU on demand,
 *     asynchronously (nubint.ai review, abstract; cmlonder.com newsletter,
 *     section "Iddia ve Gerceklik").
 *   - Heterogeneous batching: one pass computes the LoRA part for tokens of
 *     many adapters of different ranks directly on non-contiguous memory
 *     (dongaigc.com summary, section 2; nubint.ai review, method list).
 *   - The base model's batched GEMM is computed elsewhere; this library only
 *     adds the adapter part into its output y (nubint.ai review, method list:
 *     base computation batched, adapter computation separate).
 *
 * Conventions for every function below
 *   - Return value: SLORA_OK (0) or a negative SLORA_ERR_* code.  On error
 *     nothing observable changed (allocator state, page tables, device data)
 *     unless the description says otherwise; slora_last_error_string() then
 *     holds a one-line reason (thread-local, valid until the next call on
 *     the same thread).
 *   - "device pointer" = memory of the GPU current when the pool was
 *     created; "host pointer" = ordinary (preferably pinned) host memory.
 *   - Streams/events are cudaStream_t / cudaEvent_t passed as void*.  All
 *     device work of the pool is ordered on its compute stream, except
 *     adapter copies, which run on its copy stream.  No function blocks the
 *     host on the GPU unless it says so.
 *   - A pool is not thread-safe: the caller serialises calls on one pool.
 *   - 16-bit values are IEEE binary16 (SLORA_F16) or bfloat16 (SLORA_BF16);
 *     accumulation is fp32; y is rounded once, to nearest even.
 */
#ifndef SLORA_H
#define SLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define SLORA_OK 0
#define SLORA_ERR_INVALID (-1)      /* bad argument, size, alignment or id */
#define SLORA_ERR_OOM (-2)          /* not enough free pages; state unchanged */
#define SLORA_ERR_EXISTS (-3)       /* adapter id already resident */
#define SLORA_ERR_NOT_RESIDENT (-4) /* adapter id not resident */
#define SLORA_ERR_BUSY (-5)         /* reserved, never returned: an evict of an adapter still in use
                                       is ordered by events instead (see slora_adapter_evict) */
#define SLORA_ERR_CUDA (-6)         /* a CUDA runtime call failed (see error string) */
#define SLORA_ERR_DEVICE (-7)       /* a kernel reported bad input (see slora_device_status) */
#define SLORA_ERR_TIMEOUT (-8)      /* a kernel's bounded wait gave up (device status only) */
#define SLORA_ERR_DEVICE_ASSERT (-9) /* a bounds check of the SLORA_DEBUG build failed (device status only) */

/* ---- element types and apply modes -------------------------------------- */
#define SLORA_F16 0
#define SLORA_BF16 1

#define SLORA_MODE_AUTO 0    /* large batches: tcgen05 for long segments, CUDA cores for the rest; small batches: CUDA cores */
#define SLORA_MODE_DECODE 1  /* every segment on the CUDA-core gather kernels */
#define SLORA_MODE_PREFILL 2 /* every segment on the tcgen05 kernels (CUDA-core kernels when the page size is not a multiple of 64) */

/* Library limits (also checked at run time). */
#define SLORA_MAX_PROJ 128         /* projections per pool (e.g. 32 layers x q, k, v, o) */
#define SLORA_MAX_PROJ_PER_CALL 8  /* projections of one slora_lora_apply_multi call */
#define SLORA_MAX_RANK 256         /* largest adapter rank */
#define SLORA_MAX_ADAPTERS 32768   /* adapter ids 0 .. max_adapters-1 */

typedef struct slora_pool slora_pool; /* opaque, owned by the library */

/*
 * The token grouping of one batch (the "segments" of segmented gather
 * matrix-vector products, SGMV: cmlonder.com newsletter, section "Iddia ve
 * Gerceklik").  Tokens are stably sorted by adapter id, ascending; tokens
 * with id -1 carry no adapter and are left out, as are tokens that name an
 * adapter that is not resident or an id outside [-1, max_adapters) (those
 * are counted in counts[2] and raise the device status
 * SLORA_ERR_NOT_RESIDENT or SLORA_ERR_INVALID; the first such token seen
 * decides which).  All arrays are DEVICE memory
 * owned by the pool; they stay valid until the next slora_build_segments on
 * the same pool (or the next evict), which invalidates every earlier handle
 * (generation check).
 */
typedef struct slora_segments {
  int32_t T;                  /* tokens in the batch */
  int32_t max_segs;           /* capacity of seg_adapter / seg_start */
  const int32_t* perm;        /* [T] sorted position j -> token index; [0, counts[1]) valid */
  const int32_t* seg_start;   /* [max_segs + 1] first sorted position of each segment */
  const int32_t* seg_adapter; /* [max_segs] adapter id of each segment (ascending) */
  const int32_t* counts;      /* [16] {num_segs, n_sorted, bad_tokens, internal work totals...} */
  uint64_t generation;        /* must match the pool's current segment generation */
} slora_segments;

/*
 * Create a pool over a caller-owned device buffer.  The pool is the unified
 * memory pool of S-LoRA's Unified Paging (dongaigc.com summary, section 1
 * "Unified Paging": one pool of pages managed together for adapter weights
 * and KV-cache tensors; nubint.ai review, method list): pages of H elements,
 * the unit one token's K or V vector of one layer takes, so that adapter rows
 * of every rank and KV slots of every length are allocated from one free list
 * without fragmenting it.
 *   d_pool      device buffer of num_pages * page_elems 16-bit elements,
 *               16-byte aligned; caller-owned, must outlive the pool.  NULL
 *               creates a PLANNING pool: host allocator and page tables only,
 *               no CUDA call is ever made (loads only allocate; build/apply
 *               return SLORA_ERR_INVALID).
 *   num_pages   pages in the pool (> 0, < 2^31)
 *   page_elems  H = elements per page = the hidden size = one token's K (or
 *               V) vector for one layer, so one KV slot of one token and one
 *               layer is two pages; multiple of 8, <= 65536
 *   dtype       SLORA_F16 or SLORA_BF16 (pool, x and y share it)
 *   max_adapters, max_rank   adapter ids are 0..max_adapters-1, ranks 1..max_rank
 *   max_tokens  largest batch (T) accepted by slora_build_segments
 *   num_proj, proj_in, proj_out   the projections adapters carry (host
 *               arrays, copied); every dim a positive multiple of 8
 *   compute, copy   cudaStream_t for kernels / for adapter copies (may be
 *               equal; NULL = legacy default stream)
 * Allocates with cudaMalloc: the device page table (max_adapters * max_rank
 * * sum_q(ceil(in_q/H)+ceil(out_q/H)) int32), segment arrays, the fp32
 * shrink scratch (SLORA_MAX_PROJ_PER_CALL * max_tokens * max_rank floats) and one
 * adapter-sized staging buffer; pins an equally sized host page-table mirror.
 */
int slora_pool_create(slora_pool** out, void* d_pool, int64_t num_pages, int32_t page_elems,
                      int32_t dtype, int32_t max_adapters, int32_t max_rank, int32_t max_tokens,
                      int32_t num_proj, const int32_t* proj_in, const int32_t* proj_out,
                      void* compute_stream, void* copy_stream);

/* Synchronises both streams and frees everything the pool allocated (not d_pool). */
int slora_pool_destroy(slora_pool* pool);

/*
 * KV-slot pages (PagedAttention-style: taken on demand, returned when a
 * request ends; fatihsoysal.com page, section "vLLM'in PagedAttention
 * Mekanizmasi").  alloc writes the n lowest-numbered free pages, ascending,
 * to out_pages (host int32[n]); all or nothing (SLORA_ERR_OOM).  free
 * returns n KV pages (host int32[n]); every page must be a KV page and
 * listed once, else SLORA_ERR_INVALID and nothing is freed.  Pages released
 * by slora_adapter_evict may still be read by kernels already queued on the
 * compute stream: write reused pages on that stream or after it.
 */
int slora_pages_alloc(slora_pool* pool, int64_t n, int32_t* out_pages);
int slora_pages_free(slora_pool* pool, int64_t n, const int32_t* pages);

/* Free page count and page size; any pointer may be NULL. */
int slora_pool_info(const slora_pool* pool, int64_t* free_pages, int64_t* num_pages,
                    int32_t* page_elems, int64_t* pages_per_rank);

/*
 * Load adapter `adapter_id` of rank `rank` from host memory into pool pages
 * (the on-demand fetch of the nubint.ai review, abstract).  Allocates
 * rank * sum_q(ceil(in_q/H) + ceil(out_q/H)) pages, lowest-numbered first,
 * and lists them in this page-table order: for each projection q, the rank
 * rows of A (each ceil(in_q/H) page chunks), then the rank rows of B (each
 * ceil(out_q/H) chunks); the i-th lowest page holds the i-th chunk.  The tail
 * of a row's last page is zero-filled.
 *   h_A[q]  host, rank x in_q 16-bit row-major: row k is column k of the
 *           in_q x rank matrix A (A transposed)
 *   h_B[q]  host, rank x out_q 16-bit row-major: row k is row k of B
 *   done    optional out: a cudaEvent_t (owned by the pool, valid until the
 *           adapter is evicted) that completes when the pages are written
 * The copies are queued on the copy stream after all work queued so far on
 * the compute stream (so pages freed earlier are no longer being read; weight
 * blocks that follow each other in host memory in the order above move in one
 * copy) and
 * the host buffers must stay untouched until `done` completes.  Later
 * slora_build_segments calls make the compute stream wait for pending loads.
 * Errors: SLORA_ERR_INVALID (id/rank out of range, NULL buffer),
 * SLORA_ERR_EXISTS, SLORA_ERR_OOM (state unchanged), SLORA_ERR_CUDA (the
 * pages are released again, state as before the call).
 * On a planning pool h_A / h_B may be NULL and nothing is copied.
 */
int slora_adapter_load(slora_pool* pool, int32_t adapter_id, int32_t rank,
                       const void* const* h_A, const void* const* h_B, void** done);

/*
 * Evict a resident adapter: its pages return to the free list at once and
 * its device rank is cleared on the compute stream (work queued before the
 * evict still sees the adapter; if the adapter's load is still copying, work
 * queued on the compute stream after the evict waits for those copies).  The pages' "race conditions in the adapter
 * manager under dynamic loading" (cmlonder.com newsletter, section "Iddia ve
 * Gerceklik") are answered by stream order rather than by refusing the evict
 * with SLORA_ERR_BUSY: a later load into the freed pages is queued after all
 * work queued on the compute stream before it, so no kernel still reading the
 * old rows can see the new ones.  Every segment handle built before the
 * evict becomes stale (build the segments again).  SLORA_ERR_NOT_RESIDENT if
 * it is not loaded.
 */
int slora_adapter_evict(slora_pool* pool, int32_t adapter_id);

/*
 * Per-adapter scale s_a (LoRA's alpha / r): applies compute
 *     y += s * s_a * (x A_a) B_a
 * for tokens of adapter a.  A load sets s_a = 1; this call changes it for
 * applies queued on the compute stream after it (it waits for the adapter's
 * own pending load first).  Errors: SLORA_ERR_NOT_RESIDENT for an adapter
 * that is not loaded, SLORA_ERR_INVALID for a scale that is not finite, and
 * for a planning pool (no device state).
 */
int slora_adapter_set_scale(slora_pool* pool, int32_t adapter_id, float scale);

/*
 * *ready = 1 once adapter `adapter_id`'s load has finished on the copy
 * stream (always on a planning pool), 0 while its copies are still running;
 * never blocks.  A scheduler that admits a request only when its adapter is
 * ready keeps slora_build_segments from making the compute stream wait for
 * copies (it waits for every load still running).  SLORA_ERR_NOT_RESIDENT if
 * the adapter is not loaded.
 */
int slora_adapter_ready(slora_pool* pool, int32_t adapter_id, int32_t* ready);

/* Host copy of an adapter's page table (page-table order above); *n = entries. */
int slora_adapter_pages(const slora_pool* pool, int32_t adapter_id, int32_t* out_pages,
                        int64_t capacity, int64_t* n);

/*
 * Group the batch's tokens by adapter on the GPU (one kernel on the compute
 * stream).  d_token_adapter: device int32[T], ids in [-1, max_adapters);
 * 0 <= T <= max_tokens.  Fills *out with pool-owned device arrays (see
 * slora_segments) plus the internal work lists of the apply kernels.
 *
 * CUDA graphs: this call and the apply calls only enqueue work on the
 * compute stream, so a step (segments, then one apply per layer) can be
 * captured in a graph and replayed, as long as the compute stream is not
 * the legacy default stream and no load of an adapter the batch uses is
 * still copying when the capture is made (its wait would refer to a copy
 * outside the graph).  A replay rebuilds the segments from the token ids
 * then in the captured buffer.
 */
int slora_build_segments(slora_pool* pool, const int32_t* d_token_adapter, int32_t T,
                         slora_segments* out);

/*
 * The same, for a caller that also holds the batch's ids on the host (a
 * scheduler builds them there): h_token_adapter, host int32[T], must list the
 * same ids as d_token_adapter.  The compute stream then waits only for the
 * pending loads of the adapters the batch names, not for every pending load
 * -- a load started for a request that has not joined the batch yet does not
 * hold this batch back.  h_token_adapter NULL: as slora_build_segments.
 */
int slora_build_segments_for(slora_pool* pool, const int32_t* d_token_adapter, int32_t T,
                             const int32_t* h_token_adapter, slora_segments* out);

/*
 * The heterogeneous-batch LoRA delta (dongaigc.com summary, section 2
 * "Heterogeneous Batching": the adapter part of tokens that use different
 * adapters of different ranks computed in one pass by custom kernels that
 * read the weights directly from the non-contiguous pool; cmlonder.com
 * newsletter, section "Iddia ve Gerceklik": segmented gather kernels, SGMV):
 * y += s * (x A_a) B_a for one projection `proj` over every token of the
 * batch `seg` was built from (tokens left out of the segments are not
 * touched).  x: device, T rows of proj_in[proj] elements, row stride ldx
 * elements; y: device, T rows of proj_out[proj], stride ldy, updated in
 * place.  Strides multiples of 8, pointers 16-byte aligned, x and y must not
 * overlap.  mode: SLORA_MODE_*.  Kernels only; nothing is synchronised.
 */
int slora_lora_apply(slora_pool* pool, const slora_segments* seg, int32_t proj, const void* d_x,
                     int64_t ldx, void* d_y, int64_t ldy, float s, int32_t mode);

/* The same for n <= SLORA_MAX_PROJ_PER_CALL projections (e.g. one layer's
 * q, k, v, o) in one set of launches. */
int slora_lora_apply_multi(slora_pool* pool, const slora_segments* seg, int32_t n,
                           const int32_t* projs, const void* const* d_x, const int64_t* ldx,
                           void* const* d_y, const int64_t* ldy, float s, int32_t mode);

/*
 * Comparator: the same delta by the "traditional batched matmul" variant
 * that the pages compare S-LoRA with (dongaigc.com summary, section
 * "S-LoRA的性能评估": S-LoRA against its own variants, one without unified
 * memory, one with traditional batched matrix multiplication).  Every token's
 * adapter rows are gathered out of the pool into dense tensors padded to the
 * pool's max_rank (zeros past the adapter's rank), two cuBLAS strided-batched
 * GEMMs give (x_t A) B per token (fp32 accumulation, v kept in fp32), and
 * y_t += s * s_a * delta_t is rounded once.  Arguments and errors as
 * slora_lora_apply (one projection; no mode).  Scratch: on the first call
 * the pool allocates max_tokens * max_rank * (2 * max h_in + 4 * max h_out)
 * bytes and a little more (slora_bmm_scratch_bytes reports it), freed with
 * the pool; SLORA_ERR_OOM if it cannot.  cuBLAS is opened on the first call
 * (SLORA_ERR_CUDA when it is not installed); nothing else in the library
 * needs it.  For measurement and comparison, not for serving.
 */
int slora_lora_apply_bmm(slora_pool* pool, const slora_segments* seg, int32_t proj, const void* d_x,
                         int64_t ldx, void* d_y, int64_t ldy, float s);
/* Bytes of comparator scratch the pool holds (0 before the first call). */
int slora_bmm_scratch_bytes(const slora_pool* pool, size_t* bytes);

/*
 * Synchronises the compute stream, returns in *status the first error a
 * kernel reported since the last call (SLORA_OK, SLORA_ERR_NOT_RESIDENT for a
 * token naming an adapter that is not loaded, SLORA_ERR_INVALID for an id
 * out of range, SLORA_ERR_TIMEOUT when a pipeline wait gave up) and clears it.
 */
int slora_device_status(slora_pool* pool, int32_t* status);

/*
 * Serialise the host allocator state for bit-exact comparison: int64
 * num_pages, int64 free_pages, int32 max_adapters, int32 stride, then
 * int32 owner[num_pages] (-1 free, -2 KV, else adapter id), int32
 * rank[max_adapters], int32 page_table[max_adapters * stride] (-1 unused).
 * With buf NULL only *len is set; otherwise *len must be >= the size.
 */
int slora_pool_snapshot(const slora_pool* pool, void* buf, size_t* len);

/*
 * Per-kernel device timing (tracing).  When enabled, every kernel the pool
 * launches is bracketed by CUDA events on its stream.  slora_timing_read
 * synchronises, then writes for each kernel kind k < *n (at most capacity):
 * names[k] (static strings), total milliseconds ms[k] and launches[k], and
 * resets the totals.
 */
int slora_timing_enable(slora_pool* pool, int32_t enable);
int slora_timing_read(slora_pool* pool, int32_t capacity, const char** names, double* ms,
                      int64_t* launches, int32_t* n);

/*
 * SLORA_MODE_AUTO's split.  In a batch of at least `tc_min_batch` tokens
 * (default 2048), segments of at least `tc_threshold` tokens (default 8) run
 * on the tcgen05 kernels and the rest on the CUDA-core kernel; a smaller
 * batch runs wholly on the CUDA-core kernel.  The defaults come from
 * measurements on GB300: on the 7B prefill batch (8,561 tokens) AUTO then
 * matches PREFILL, while on decode batches of 256-512 tokens the few long
 * segments leave the tensor-core kernels bound by latency and the CUDA-core
 * kernel is 1.8x faster.  tc_threshold takes effect at the next
 * slora_build_segments; tc_min_batch at the next apply.
 */
int slora_set_tc_threshold(slora_pool* pool, int32_t min_tokens);
int slora_set_tc_min_batch(slora_pool* pool, int32_t min_tokens);

/*
 * Failure injection on the host, for tests of the error paths (the pages'
 * concern about the adapter manager under dynamic loading: cmlonder.com
 * newsletter, section "Iddia ve Gerceklik").  Arms one fault on this pool;
 * it fires once, on the nth (counted from 1) event of its kind from now on:
 *   SLORA_FAULT_PAGE_ALLOC  a call that takes pages (slora_pages_alloc,
 *                           slora_adapter_load) fails with SLORA_ERR_OOM as
 *                           if the pool were full; nothing changes;
 *   SLORA_FAULT_COPY        a copy or kernel that slora_adapter_load enqueues
 *                           fails as a CUDA error would: the load returns
 *                           SLORA_ERR_CUDA and, once the copy stream has
 *                           finished what the load queued before the failure,
 *                           its pages are released again, the host state
 *                           (slora_pool_snapshot) exactly as before the call.
 * SLORA_FAULT_NONE (or nth = 0) disarms.  The environment variable
 * SLORA_FAULT="alloc:N" or "copy:N" arms the same fault in every pool the
 * process creates.  Nothing here touches a GPU.
 */
#define SLORA_FAULT_NONE 0
#define SLORA_FAULT_PAGE_ALLOC 1
#define SLORA_FAULT_COPY 2
int slora_debug_set_fault(slora_pool* pool, int32_t kind, int64_t nth);

/*
 * The SLORA_DEBUG build (libslora_debug.so, compiled with -DSLORA_DEBUG;
 * the Python binding loads it when the environment has SLORA_DEBUG=1)
 * checks, in every kernel, each page index it reads from a page table
 * against the pool's page count and each token index it reads from the
 * token order against the batch size.  A violation is reported by
 * slora_device_status as SLORA_ERR_DEVICE_ASSERT (the index is replaced by
 * 0, so no access leaves its buffer and no kernel waits for a copy that
 * never comes); results of that call are then meaningless.  Other builds
 * compile no checks.
 *
 * slora_debug_poke_page_table writes `value` into entry `entry` of the
 * pool's device page table (entries of adapter a start at a * stride) and
 * returns the previous value in *old: a test plants a bad page index and
 * puts the old one back.  The host copy of the table is not changed.  Only
 * in the SLORA_DEBUG build; other builds return SLORA_ERR_INVALID.  Not for
 * serving: the next apply reads the planted value.
 */
int slora_debug_poke_page_table(slora_pool* pool, int64_t entry, int32_t value, int32_t* old);

/*
 * Polls that each of the CUDA-core apply kernel's waits on other warps
 * (stages, v rows, partial sums, the grid barrier) makes before it gives up
 * (0: the built-in limit, 2^24).  A kernel that gives up records
 * SLORA_ERR_TIMEOUT in the device status (slora_device_status), waits with
 * the built-in limit for its own copies still in flight, and returns; y may
 * be partly updated.  For tests of the time-out path.
 */
int slora_debug_set_wait_limit(slora_pool* pool, uint32_t polls);

const char* slora_last_error_string(void);

/*
 * slora_lora_apply_noalloc -- y += s * (x A_a) B_a for one projection,
 * allocating nothing.  The pages describe no counterpart of this entry point.
 *
 * For callers that cannot call cudaMalloc where they compute the delta: a
 * serving runtime that has handed all GPU memory to its own arena (page pool,
 * KV cache, activations) and may not grow its footprint, or code that must
 * not allocate at all while it serves.  Such a caller owns every buffer
 * already; this call needs no slora_pool and makes no cudaMalloc, cudaFree or
 * other allocating call.  Its scratch (token grouping and the fp32 shrink
 * result) is one static device array of SLORA_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until the process exits.
 *   d_pool, page_elems, dtype   the page pool (device, 16-byte aligned)
 *   d_page_table, pt_stride     device int32; adapter a's entries start at
 *                               a * pt_stride, in the page-table order of
 *                               slora_adapter_load (the layout a pool uses);
 *                               every entry read must name a page of d_pool
 *   d_rank, max_adapters        device int32[max_adapters]; 0 = not resident;
 *                               ranks outside [1, rmax] count as 0, where
 *                               rmax = min(SLORA_MAX_RANK, pt_stride / E) and
 *                               E = sum_q(ceil(in_q/H) + ceil(out_q/H)) is
 *                               the entries one unit of rank takes, so no
 *                               adapter's rows run into the next adapter's
 *                               stretch of the page table
 *   num_proj, proj_in, proj_out host arrays: every projection adapters carry
 *   proj                        the projection to apply
 *   d_token_adapter, T          device int32[T], ids in [-1, max_adapters);
 *                               T <= SLORA_NOALLOC_MAX_TOKENS (else
 *                               SLORA_ERR_INVALID); tokens with id -1 or a
 *                               non-resident adapter are left unchanged
 *   d_x, ldx, d_y, ldy, s       as in slora_lora_apply
 *   stream                      cudaStream_t (NULL = legacy default stream)
 *   status                      optional (NULL: not reported): one int32 in
 *                               device memory or pinned host memory that
 *                               receives this call's device status on
 *                               `stream` once its kernels are done --
 *                               SLORA_OK, SLORA_ERR_NOT_RESIDENT (a token's
 *                               adapter has rank 0), SLORA_ERR_INVALID (an id
 *                               other than -1 outside [0, max_adapters)) or
 *                               SLORA_ERR_TIMEOUT (a kernel's bounded wait
 *                               gave up; y may be partly updated).  Read it
 *                               after synchronising the stream.
 * The first call on a device sets that device up (it looks up the device
 * address of the scratch array and sizes the kernels' grids); make that first
 * call before any stream capture.  Every call shares the one scratch array
 * and leaves the last call's contents in it: calls that may overlap on the
 * GPU (other streams, other threads) race and must be serialised by the
 * caller.
 */
#define SLORA_NOALLOC_MAX_TOKENS 2048
#define SLORA_NOALLOC_SCRATCH_BYTES 2351360u /* 2.24 MiB: grouping of 2048 tokens, 32768 ranks, v */
int slora_lora_apply_noalloc(const void* d_pool, int32_t page_elems, int32_t dtype,
                             const int32_t* d_page_table, int64_t pt_stride, const int32_t* d_rank,
                             int32_t max_adapters, int32_t num_proj, const int32_t* proj_in,
                             const int32_t* proj_out, int32_t proj, const int32_t* d_token_adapter,
                             int32_t T, const void* d_x, int64_t ldx, void* d_y, int64_t ldy, float s,
                             void* stream, int32_t* status);

#ifdef __cplusplus
}
#endif
#endif /* SLORA_H */
