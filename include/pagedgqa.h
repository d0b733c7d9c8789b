/*
 * pagedgqa.h -- C ABI of the paged grouped-query decode attention library
 * (libpagedgqa.so, CUDA, sm_103a).
 *
 * The operation (one decode step, one query token per sequence):
 *
 *   for every sequence b < B and query head h < H, with G = H / Hkv and
 *   kv head j = floor(h / G):
 *     out[b,h,:] = softmax_t( scale * q[b,h,:] . K_b[t,:] ) V_b[t,:],
 *                  t = 0 .. cache_seqlens[b]-1
 *   where K_b[t] / V_b[t] is row t % bs of physical block
 *   block_table[b][t / bs], kv head j, of the shared K/V pool.
 *
 * Sources, by page and section:
 *   - "Paged Attention Kernel Architecture for BI-V100": section 1 (problem
 *     definition), section 2 (split-KV partitions holding a (max_score,
 *     exp_sum, weighted_v) state merged by a combine op; a separate merge
 *     kernel), section 4 (one CTA per kv head serves all G query heads),
 *     section 6 (phase 1 partitioned attention, phase 2 cross-partition
 *     reduction).
 *   - "Paged attention" (Hugging Face Transformers docs), decoding path:
 *     block_table of shape (batch, max_blocks_per_seq) of physical block
 *     ids with -1 for unallocated blocks; cache_seqlens is the key length;
 *     the cache is indexed and then updated in place.
 *   - "v10_triton_paged_gqa", Core Principle: block-table translation,
 *     valid-token mask, running max / exp-sum / accumulator recurrence;
 *     the captured launch is replayed while inputs change in place.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to dense, row-major memory the
 *     caller owns (pa_decode_host / pa_decode_multi_host also take host
 *     buffers; see there); the library allocates nothing and keeps no
 *     per-call state.  The one exception is pa_decode_noalloc, whose scratch
 *     is a static device array inside the library (see there).
 *   - Every device pointer must be 16-byte aligned.
 *   - Layouts (dt = fp16 or bf16, the same for q, k and v):
 *       q              [B, H, d]            dt
 *       k_cache        [P, bs, Hkv, d]      dt   (P = num_blocks)
 *       v_cache        [P, bs, Hkv, d]      dt
 *       block_table    [B, max_blocks_per_seq] int32, -1 = unallocated
 *       cache_seqlens  [B]                  int32
 *       out            [B, H, d]            float32
 *       k_new, v_new   [B, Hkv, d]          dt
 *   - Supported: d in {64, 128, 256}; bs in {16, 32, 64}; H % Hkv == 0 and
 *     G = H / Hkv <= 8; 0 <= B <= PA_MAX_BATCH (B == 0 is a no-op);
 *     max_blocks_per_seq * bs, B * max_blocks_per_seq and
 *     Hkv * (max_blocks_per_seq + 64) below 2^31 (else PA_ERR_SHAPE).
 *   - Work is enqueued on `stream` (NULL = legacy default stream).  No entry
 *     point allocates or picks a launch shape from device data, and none but
 *     pa_read_status and the synchronous host-buffer calls synchronises (the first
 *     pa_decode_noalloc call on a device also enqueues one memset on its
 *     stream), so pa_decode and
 *     pa_cache_append can be captured in a CUDA graph
 *     and replayed after the inputs are changed in place.  The first call on
 *     a device performs one-time host-side setup (kernel attributes,
 *     occupancy query); make it before beginning a stream capture.
 *   - Host-side errors are reported by the return code before anything is
 *     enqueued.  Data errors found on the device never trap and never wait:
 *     they set a bit in the status word kept at the start of the workspace
 *     (pa_decode_noalloc: the caller's status word, if given) and make the
 *     affected outputs NaN (see pa_read_status).
 */
#ifndef PAGEDGQA_H
#define PAGEDGQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* pa_stream_t;

#define PA_MAX_BATCH 8192

/* Return codes (host side). */
#define PA_OK 0
#define PA_ERR_NULL (-1)        /* a required pointer is NULL */
#define PA_ERR_SHAPE (-2)       /* unsupported or inconsistent shape / dtype */
#define PA_ERR_ALIGN (-3)       /* a pointer is not 16-byte aligned */
#define PA_ERR_WORKSPACE (-4)   /* workspace smaller than pa_workspace_size */
#define PA_ERR_CUDA (-5)        /* a CUDA runtime/driver call failed */
#define PA_ERR_OPTION (-6)      /* invalid pa_options value */
#define PA_ERR_SCRATCH_LIMIT (-7) /* pa_decode_noalloc: needs more scratch than
                                     PA_STATIC_SCRATCH_BYTES */
#define PA_ERR_STATE (-8)       /* block manager: invalid handle, sequence id,
                                   index or request; nothing was changed */
#define PA_ERR_NO_BLOCKS (-9)   /* block manager: the free list is too short;
                                   nothing was changed */

/* Device status bits (sticky in the workspace status word). */
#define PA_STATUS_BAD_BLOCK 0x1u   /* a table entry inside a sequence's length is
                                      -1 or >= num_blocks; that (b, kv head)'s
                                      output heads are NaN */
#define PA_STATUS_BAD_SEQLEN 0x2u  /* cache_seqlens[b] < 0 or > max_blocks_per_seq*bs;
                                      all of sequence b's outputs are NaN */
#define PA_STATUS_TIMEOUT 0x4u     /* a pipeline wait gave up (never expected);
                                      outputs of that step are unreliable */
#define PA_STATUS_NO_SLOT 0x8u     /* pa_cache_append: position cache_seqlens[b]
                                      has no table column or an unmapped entry;
                                      nothing was written for that sequence */

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

typedef enum {
  PA_COMPUTE_AUTO = 0, /* library choice (tensor-core mma) */
  PA_COMPUTE_SIMT = 1, /* fp32 FMA on CUDA cores */
  PA_COMPUTE_MMA = 2,  /* mma.sync m16n8k16 tensor-core products, fp32 accumulate */
  PA_COMPUTE_TC = 3    /* tcgen05 tensor cores, accumulators in tensor memory,
                          128-token tiles: head_dim 128 only (else
                          PA_ERR_OPTION); not with pa_decode_append */
} pa_compute;

typedef struct pa_shape {
  int32_t batch;              /* B: sequences, one query token each */
  int32_t num_heads;          /* H: query heads */
  int32_t num_kv_heads;       /* Hkv: kv heads, H % Hkv == 0 */
  int32_t head_dim;           /* d */
  int32_t block_size;         /* bs: tokens per physical block */
  int32_t max_blocks_per_seq; /* columns of block_table */
  int32_t num_blocks;         /* P: physical blocks in the pool */
  int32_t dtype;              /* pa_dtype of q, k_cache, v_cache, k_new, v_new */
} pa_shape;

typedef struct pa_options {
  /* Split-KV partition size in tokens.  0: balanced split chosen on the
   * device each step from the actual lengths (every CTA of the persistent
   * grid gets an equal share of the (sequence, kv head, block) work).
   * > 0: fixed partitions of this many tokens (a multiple of block_size),
   * e.g. 512 as in the BI-V100 design's PARTITION_SIZE. */
  int32_t partition_tokens;
  int32_t compute;   /* pa_compute */
  int32_t num_ctas;  /* persistent grid size; 0 = one full wave of resident
                        CTAs on the current device.  Setting it makes
                        pa_workspace_size independent of the device. */
  int32_t stages;    /* TMA ring slots per warp (16-token K/V stages,
                        1..8; more than fit in shared memory next to the
                        kernel's other buffers is PA_ERR_OPTION); with
                        PA_COMPUTE_TC the CTA's 128-token V slots (2..4);
                        0 = library choice */
  int32_t phase;     /* pa_decode / pa_decode_append / pa_decode_multi:
                        PA_PHASE_BOTH (0) runs both kernels; PA_PHASE_SPLIT
                        only phase 1, PA_PHASE_MERGE only phase 2 (which must
                        follow phase 1 of the same step on the same stream),
                        e.g. to time the kernels apart */
  int32_t wait_limit_us; /* the longest one pipeline wait of the split kernel
                        may take before the step gives up (sets
                        PA_STATUS_TIMEOUT, outputs of that step unreliable);
                        0 = 2 s.  Such a wait is never expected to run out:
                        copies complete in microseconds.  The copies a CTA
                        has in flight when it gives up are always waited for
                        before it exits.  Not used by PA_COMPUTE_TC, whose
                        waits keep 2 s. */
  int32_t stall_test; /* testing the timeout path, 0 in normal use.  1: warp 0
                        of every CTA of the split kernel that has work waits
                        for its first tile on a barrier that nothing
                        completes, so that wait runs out after
                        wait_limit_us; the step then reports
                        PA_STATUS_TIMEOUT and the next call on the same
                        workspace is unaffected.  PA_COMPUTE_TC: PA_ERR_OPTION. */
} pa_options;

#define PA_PHASE_BOTH 0
#define PA_PHASE_SPLIT 1
#define PA_PHASE_MERGE 2

/* Bytes of workspace pa_decode / pa_decode_split / pa_decode_merge /
 * pa_cache_append need for this shape and these options (NULL = defaults).
 * The workspace holds the status word, the per-step length prefix sums and
 * the split-KV partial states (m, l, weighted_v[d]) in float32.  The caller
 * allocates it once, zero-fills it once (the status word and the cluster
 * kernel's CTA count in the first 256 bytes must start at 0; every call
 * leaves them 0 again, status bits aside), and may reuse it for every later
 * call with the same shape and options.
 * Two calls in flight at the same time must not share a workspace.
 * Returns PA_OK and writes *bytes, or a negative code.  With
 * options->num_ctas == 0 the size depends on the current device's SM count. */
int pa_workspace_size(const pa_shape* shape, const pa_options* options, size_t* bytes);

/* One decode step: out = paged GQA decode attention (formula at the top).
 * Launches the split kernel (phase 1: each persistent CTA streams its share
 * of (sequence, kv head, block) work through a multi-stage TMA pipeline and
 * computes all G query heads of the kv head at once) and the merge kernel
 * (phase 2: combine op over the pieces of every sequence that was split
 * across CTAs) -- or, for a step with few segments, the one cluster kernel
 * (see pa_launch_plan).  Sequences with cache_seqlens[b] == 0 get out = 0.
 * scale multiplies q . k (typically 1/sqrt(d)).  Table entries at or beyond
 * ceil(cache_seqlens[b] / bs) are never read.
 * Errors: PA_ERR_* before any launch; device-side data errors as status
 * bits (PA_STATUS_BAD_BLOCK, PA_STATUS_BAD_SEQLEN). */
int pa_decode(const pa_shape* shape, const pa_options* options, const void* q,
              const void* k_cache, const void* v_cache, const int32_t* block_table,
              const int32_t* cache_seqlens, float scale, float* out, void* workspace,
              size_t workspace_bytes, pa_stream_t stream);

/* Which kernels a step with this shape and these options launches on the
 * current device (max_q = 0: pa_decode; > 0: pa_decode_multi with at most
 * max_q query tokens per sequence).  info[0] = kernels per step (1: the
 * cluster kernel does the whole step -- a step with few (sequence, kv head)
 * segments and at most 64 MB of K/V even with every table row full, one
 * query token per sequence, the mma path with the balanced split and the
 * library's grid: each segment gets one thread-block cluster whose CTAs
 * fold their partial states through distributed shared memory, so no
 * workspace round trip and no second kernel; 2: the persistent split
 * kernel and the merge kernel), info[1] = CTAs of the step's first kernel,
 * info[2] = CTAs per cluster (0 without clusters), info[3] = ring slots per
 * warp.  Chosen from the shape and options only (a captured graph stays
 * valid); pa_decode_split then runs the whole step and pa_decode_merge
 * nothing.  The host-buffer calls make the same choice; pa_decode_append
 * and pa_decode_multi always use the two kernels.  Returns PA_OK or PA_ERR_*. */
int pa_launch_plan(const pa_shape* shape, const pa_options* options, int32_t max_q,
                   int32_t* info);

/* Phase 1 of pa_decode alone (same arguments).  Writes the outputs of every
 * sequence handled whole by one CTA and the partial states of the others
 * (with the cluster kernel: the whole step). */
int pa_decode_split(const pa_shape* shape, const pa_options* options, const void* q,
                    const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, float scale, float* out, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/* Phase 2 of pa_decode alone (same arguments; q, k_cache and v_cache are not
 * read).  Must follow pa_decode_split of the same step on the same stream.
 * Launches nothing when the step runs on the cluster kernel. */
int pa_decode_merge(const pa_shape* shape, const pa_options* options, const void* q,
                    const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, float scale, float* out, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/* Fused append-and-attend (the decoding path of the Hugging Face "Paged
 * attention" page: the kernel indexes the cache through block_table and
 * updates it in place).  For every sequence b: k_new[b,:,:] and v_new[b,:,:]
 * are written to position cache_seqlens[b] exactly as pa_cache_append writes
 * them, and out[b] attends over the cache_seqlens[b] + 1 tokens including
 * the new one -- in one pass: the one tile that holds the new position takes
 * the new row from k_new/v_new while also storing it.  cache_seqlens is not
 * incremented (the caller does that).  Arguments as pa_decode, plus
 * k_new/v_new [B, Hkv, d] and the pools writable.  A new position past the
 * table (cache_seqlens[b] + 1 > max_blocks_per_seq * bs) sets
 * PA_STATUS_BAD_SEQLEN | PA_STATUS_NO_SLOT; an unmapped entry for it sets
 * PA_STATUS_BAD_BLOCK; in both cases sequence b's outputs are NaN and its row
 * is not written.  Same workspace as pa_decode. */
int pa_decode_append(const pa_shape* shape, const pa_options* options, const void* q,
                     const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int32_t* block_table, const int32_t* cache_seqlens, float scale,
                     float* out, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* Several query tokens per sequence over the paged cache (chunked decode,
 * e.g. verifying draft tokens).  Query rows are packed as in the varlen path
 * of the Hugging Face "Paged attention" page: sequence b owns rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q [total_q, H, d] (the page's
 * cu_seq_lens_q, a DEVICE int32 array [B+1]), and out [total_q, H, d] fp32
 * gets the same rows.  The keys are the cache_seqlens[b] tokens of the paged
 * cache (block_table as in pa_decode), the query tokens themselves included:
 * the n_q query tokens of a sequence are its last n_q key positions, so
 * query i (0-based within its sequence) sees
 *   causal != 0:  keys t < clamp(cache_seqlens[b] - n_q + i + 1, 0, cache_seqlens[b])
 *   causal == 0:  all cache_seqlens[b] keys
 * and a query that sees no key gets 0.
 *   max_q:   host bound on n_q (the page's max_length_q), 1..PA_MAX_QUERY_TOKENS;
 *            it fixes the launch shape, so a captured graph stays valid while
 *            the lengths change under it.
 *   total_q: rows of q and out (host); the library reads and writes no row
 *            at or beyond it.
 * A sequence whose span is not non-decreasing within [0, total_q], or holds
 * more than max_q tokens, is skipped (its rows are not written) and sets
 * PA_STATUS_BAD_SEQLEN; an invalid cache_seqlens[b] makes its rows NaN and
 * sets the same bit; bad table entries as in pa_decode.  Rows that belong
 * to no sequence are not written.  The workspace must hold
 * pa_workspace_size_multi(shape, options, max_q) bytes (zero-filled once, as
 * for pa_decode).  Tensor-core path only (options->compute SIMT is
 * PA_ERR_OPTION).  Up to 32 (token, head) pairs of one kv head share one pass
 * over its K/V (16 at d = 256, and with PA_COMPUTE_TC): a sequence with
 * n_q * G above that is read ceil(n_q * G / 32) times (16). */
#define PA_MAX_QUERY_TOKENS 4096
int pa_workspace_size_multi(const pa_shape* shape, const pa_options* options, int32_t max_q,
                            size_t* bytes);
int pa_decode_multi(const pa_shape* shape, const pa_options* options, const void* q,
                    const int32_t* cu_seqlens_q, int32_t total_q, int32_t max_q, int32_t causal,
                    const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, float scale, float* out, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * End to end from host buffers.
 *
 * pa_decode_host is pa_decode for a caller whose step inputs and result live
 * in host memory: q_host [B, H, d], block_table_host [B, max_blocks_per_seq]
 * and cache_seqlens_host [B] are copied into device staging inside the
 * workspace, both phases run on the staged copies, and out_host [B, H, d]
 * fp32 receives the result; the call then waits for `stream` and returns.
 * The pools stay on the device (k_cache, v_cache: device pointers, as in
 * pa_decode).  Host buffers need no alignment; page-locked ones
 * (cudaHostAlloc / cudaHostRegister, 16-byte aligned) are read and written
 * by the kernels directly, pageable ones are copied (cudaMemcpyAsync, staged
 * by the driver).  Memory of the current device is accepted too (used in
 * place, like page-locked memory).  The
 * workspace (device, 16-byte aligned, zero-filled once) must hold
 * pa_workspace_size_host bytes: pa_workspace_size's plus the staging.
 * status_host: if not NULL, receives this call's device status bits (0 when
 * all went well; the workspace's own status word is left untouched); if
 * NULL, the bits accumulate in the workspace's status word as for pa_decode
 * (read them with pa_read_status).  options->phase must be PA_PHASE_BOTH.
 * Returns PA_OK or PA_ERR_*; argument errors are found before anything is
 * enqueued.  Not capturable in a CUDA graph (it synchronises). */
int pa_workspace_size_host(const pa_shape* shape, const pa_options* options, size_t* bytes);
int pa_decode_host(const pa_shape* shape, const pa_options* options, const void* q_host,
                   const void* k_cache, const void* v_cache, const int32_t* block_table_host,
                   const int32_t* cache_seqlens_host, float scale, float* out_host,
                   uint32_t* status_host, void* workspace, size_t workspace_bytes,
                   pa_stream_t stream);

/* pa_decode_multi from host buffers, as pa_decode_host: q_host
 * [total_q, H, d], cu_seqlens_q_host [B + 1], block_table_host,
 * cache_seqlens_host in; out_host [total_q, H, d] fp32 back.  The workspace
 * must hold pa_workspace_size_multi_host(shape, options, max_q, M) bytes
 * for some M >= total_q (PA_ERR_WORKSPACE otherwise). */
int pa_workspace_size_multi_host(const pa_shape* shape, const pa_options* options, int32_t max_q,
                                 int32_t max_total_q, size_t* bytes);
int pa_decode_multi_host(const pa_shape* shape, const pa_options* options, const void* q_host,
                         const int32_t* cu_seqlens_q_host, int32_t total_q, int32_t max_q,
                         int32_t causal, const void* k_cache, const void* v_cache,
                         const int32_t* block_table_host, const int32_t* cache_seqlens_host,
                         float scale, float* out_host, uint32_t* status_host, void* workspace,
                         size_t workspace_bytes, pa_stream_t stream);

/* pa_decode_host / pa_decode_multi_host without the wait: the call enqueues
 * the same work on `stream` and returns.  A serving loop that issues step
 * i + 1 before step i has finished keeps the GPU busy through the host's
 * own time per call, and step i + 1's staging of its inputs runs while step
 * i's last kernel finishes: the staging kernel is a programmatic dependent
 * of the kernel before it on the stream, fills its staging area, and only
 * then waits for that kernel.  (The decoding path of the Hugging Face
 * "Paged attention" page reads the cache in place at every step; only the
 * step's q, table and lengths move.)
 *   slot: 0 or 1, which of the workspace's two staging areas this call uses
 *         (else PA_ERR_OPTION).  Consecutive calls on a stream must
 *         alternate slots: a call may still be reading its slot while the
 *         next call fills the other one.
 *   workspace: pa_workspace_size_host_async / pa_workspace_size_multi_host_async
 *         bytes (room for both slots), zero-filled once; the partial states
 *         are shared by both slots (the kernels of consecutive calls on one
 *         stream never overlap where they use them).
 *   Host buffers: page-locked (cudaHostAlloc / cudaHostRegister) or
 *         device memory, as for pa_decode_host.  Pageable buffers work but
 *         the driver's staged copies make the call wait for them.  The call's
 *         inputs must stay unchanged, and out_host / status_host unread,
 *         until the stream has passed the call (cudaStreamSynchronize, or an
 *         event recorded after it); give each slot its own buffers when the
 *         next step is issued before the previous one is read.
 *   status_host: as for pa_decode_host, written when the call's kernels run.
 * Everything else (arguments, results, status bits, errors before anything
 * is enqueued) is as for the synchronous calls, and the result bits are the
 * same. */
int pa_workspace_size_host_async(const pa_shape* shape, const pa_options* options,
                                 size_t* bytes);
int pa_decode_host_async(const pa_shape* shape, const pa_options* options, const void* q_host,
                         const void* k_cache, const void* v_cache,
                         const int32_t* block_table_host, const int32_t* cache_seqlens_host,
                         float scale, float* out_host, uint32_t* status_host, int32_t slot,
                         void* workspace, size_t workspace_bytes, pa_stream_t stream);
int pa_workspace_size_multi_host_async(const pa_shape* shape, const pa_options* options,
                                       int32_t max_q, int32_t max_total_q, size_t* bytes);
int pa_decode_multi_host_async(const pa_shape* shape, const pa_options* options,
                               const void* q_host, const int32_t* cu_seqlens_q_host,
                               int32_t total_q, int32_t max_q, int32_t causal,
                               const void* k_cache, const void* v_cache,
                               const int32_t* block_table_host,
                               const int32_t* cache_seqlens_host, float scale, float* out_host,
                               uint32_t* status_host, int32_t slot, void* workspace,
                               size_t workspace_bytes, pa_stream_t stream);

/* Append one new token per sequence to the paged cache, in place: for every
 * b and kv head j, k_new[b,j,:] and v_new[b,j,:] are copied bit for bit to
 * row (cache_seqlens[b] % bs) of physical block
 * block_table[b][cache_seqlens[b] / bs] (the Hugging Face decoding-path
 * example: the next token of a sequence goes into the block that holds
 * position cache_seqlens[b]).  cache_seqlens is NOT incremented: the caller
 * does that (in place, so a captured graph stays valid).  A sequence whose
 * position has no table column or an unmapped entry gets no write and sets
 * PA_STATUS_NO_SLOT.  The workspace only needs room for the status word
 * (any workspace sized for pa_decode works). */
int pa_cache_append(const pa_shape* shape, const void* k_new, const void* v_new,
                    void* k_cache, void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, void* workspace, size_t workspace_bytes,
                    pa_stream_t stream);

/* Copy the status word of `workspace` to *flags (host), then clear it.
 * Synchronises `stream`.  Returns PA_OK or PA_ERR_*. */
int pa_read_status(void* workspace, uint32_t* flags, pa_stream_t stream);

/* Text for a return code (negative) or a status bit set (positive). */
const char* pa_status_string(int code);

/* pa_decode without a workspace: nothing is allocated, by the caller or
 * by the library.  (No page describes this; it serves callers that cannot
 * allocate device memory where they run decode -- e.g. a plugin whose host
 * framework owns all device allocations, or a serving loop that fixes its
 * memory at start-up and may not call cudaMalloc on its hot path.)
 *
 * Same arguments and result as pa_decode, minus the workspace.  The scratch
 * the kernels need lives in one static device array of PA_STATIC_SCRATCH_BYTES
 * that every GPU loading this library holds until the process exits.  A
 * problem whose pa_workspace_size exceeds that size is rejected with
 * PA_ERR_SCRATCH_LIMIT before anything is enqueued.  The default balanced
 * split fits for B <= PA_MAX_BATCH, G <= 8, d <= 256 whenever the persistent
 * grid has at most 256 CTAs (a 152-SM GPU runs 152); large fixed partitions
 * may not fit.
 *   status: device pointer to a uint32 that receives the PA_STATUS_* bits
 *           (OR-ed in; the caller zeroes it), or NULL to drop them.
 *   options->phase must be PA_PHASE_BOTH (else PA_ERR_OPTION): both kernels
 *   always run, since the scratch is shared by every call.
 * The first call on each device looks up the array's device address and
 * zeroes the array's 256-byte header on `stream` (with that device
 * current); make that first call before any stream capture.  All calls
 * share the one array and it keeps the previous call's contents (each call
 * rewrites everything it reads), so two calls that may overlap on the GPU
 * -- on different streams, or from different threads -- race and give wrong
 * results: serialise them. */
#define PA_STATIC_SCRATCH_BYTES (8u << 20)
int pa_decode_noalloc(const pa_shape* shape, const pa_options* options, const void* q,
                      const void* k_cache, const void* v_cache, const int32_t* block_table,
                      const int32_t* cache_seqlens, float scale, float* out, uint32_t* status,
                      pa_stream_t stream);

/* Host replica of the device work split of pa_decode (one query token per
 * sequence; pa_decode_multi charges each segment a larger overhead in its
 * balanced split), for inspection and tests.  Given host lengths, lists the
 * pieces CTA `cta` of a grid of `num_ctas` processes:
 * pieces[5*i .. 5*i+4] = (b, kv_head, first_block, end_block, slot) where
 * slot is the workspace slot of its partial state, or -1 when the piece is a
 * whole sequence/kv-head whose output the CTA writes directly.  Returns the
 * number of pieces (at most max_pieces are written), or a negative code. */
int pa_plan_pieces(const pa_shape* shape, const pa_options* options,
                   const int32_t* cache_seqlens_host, int32_t num_ctas, int32_t cta,
                   int32_t* pieces, int32_t max_pieces);

/* Host replica of the merge kernel's piece discovery.  Merge index `seg`
 * (balanced split: 0 <= seg < num_ctas, the segment that begins in split CTA
 * seg and continues past it; fixed split: 0 <= seg < B * Hkv, segment
 * (seg / Hkv, seg % Hkv)) combines the pieces in slots[0..n-1], in this
 * order, into out[b_j[0], heads of kv head b_j[1], :].  Returns n (0 when that
 * index merges nothing; b_j is then (-1, -1)) or a negative code. */
int pa_plan_merge(const pa_shape* shape, const pa_options* options,
                  const int32_t* cache_seqlens_host, int32_t num_ctas, int32_t seg,
                  int32_t* b_j, int32_t* slots, int32_t max_slots);

/* ------------------------------------------------------------------------
 * Block manager (host side) and block copy (device side).
 *
 * The host allocator of the pool of physical blocks, as the block manager of
 * the "paged-attention-runtime" design page (sections "System component
 * flow" and "BlockManager") describes it: a free list of physical block ids,
 * a reference count per block, and for every sequence the ordered list of
 * the blocks that hold its tokens (its row of block_table).  Its operations
 * are that page's allocate_blocks / free_sequence / share_prefix / cow_block:
 *   - sharing a prefix puts the source's first n blocks into the target's
 *     list and raises each one's count by one;
 *   - copy-on-write of a block whose count is above one takes a fresh block
 *     from the free list for the writer (count 1), lowers the old block's
 *     count, and leaves the data move to the caller (pa_copy_blocks);
 *   - a block whose count falls to zero goes back to the free list.
 * The manager owns host memory only; it never touches the device.  Every
 * call is serialised by a mutex inside the handle, so one handle may be used
 * from several host threads.  All calls return PA_OK (or a count) on
 * success, PA_ERR_STATE for a NULL handle / out-of-range id / impossible
 * request and PA_ERR_NO_BLOCKS when the free list is too short; on an error
 * the manager is left exactly as it was.  The free list is a stack: a new
 * manager hands out ids 0, 1, 2, ... and a block freed later is the next one
 * handed out.
 * ------------------------------------------------------------------------ */
typedef struct pa_block_manager pa_block_manager;

/* A manager for physical blocks 0..num_blocks-1 of block_size tokens, for
 * sequence ids 0..max_seqs-1 of at most max_blocks_per_seq blocks each.
 * Returns NULL when an argument is < 1 or memory runs out. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t max_seqs,
                               int32_t max_blocks_per_seq);
void pa_bm_destroy(pa_block_manager* bm);

/* allocate_blocks(seq, n): append n fresh blocks (count 1) to seq's list. */
int pa_bm_allocate(pa_block_manager* bm, int32_t seq, int32_t n);

/* free_sequence(seq): lower the count of every block of seq, return those
 * that reach zero to the free list, and empty seq's list. */
int pa_bm_free_sequence(pa_block_manager* bm, int32_t seq);

/* share_prefix(src, dst, n): dst (which must own no blocks) gets src's first
 * n blocks, each block's count raised by one. */
int pa_bm_share_prefix(pa_block_manager* bm, int32_t src, int32_t dst, int32_t n);

/* cow_block(seq, index): make block `index` of seq private before a write.
 * *old_block = the block seq held there; *new_block = the block it holds
 * now.  They differ only when the old block was shared: then the caller must
 * copy old -> new on the device (pa_copy_blocks) before writing into it. */
int pa_bm_copy_on_write(pa_block_manager* bm, int32_t seq, int32_t index, int32_t* old_block,
                        int32_t* new_block);

/* Make position `pos` of seq writable, as a decode step needs before
 * appending token pos: pos / block_size == the number of blocks seq owns
 * appends one fresh block (*old_block == *new_block); an earlier index is
 * cow_block(seq, pos / block_size).  A larger index is PA_ERR_STATE. */
int pa_bm_reserve_slot(pa_block_manager* bm, int32_t seq, int32_t pos, int32_t* old_block,
                       int32_t* new_block);

/* Write the block_table rows of the sequences seq_ids[0..rows-1] into the
 * host array table[rows][cols] (int32, -1 past each sequence's blocks).
 * PA_ERR_STATE if a sequence owns more than cols blocks. */
int pa_bm_block_table(pa_block_manager* bm, const int32_t* seq_ids, int32_t rows, int32_t cols,
                      int32_t* table);

/* Counters: PA_BM_FREE_BLOCKS (arg unused), PA_BM_REF_COUNT (arg = block),
 * PA_BM_SEQ_BLOCKS (arg = sequence).  Returns the count or PA_ERR_STATE. */
#define PA_BM_FREE_BLOCKS 0
#define PA_BM_REF_COUNT 1
#define PA_BM_SEQ_BLOCKS 2
int pa_bm_query(pa_block_manager* bm, int32_t what, int32_t arg);

/* Device half of copy-on-write: for i < n_pairs, physical block
 * pairs[2i+1] of k_cache and of v_cache becomes a bit-for-bit copy of block
 * pairs[2i] (all bs rows, all kv heads).  `pairs` is a DEVICE int32 array
 * [n_pairs, 2] so a captured graph can replay with new pairs.  Only
 * num_kv_heads, head_dim, block_size and num_blocks of `shape` are used
 * (head_dim a multiple of 8).  A pair with an id outside [0, num_blocks)
 * copies nothing and ORs PA_STATUS_BAD_BLOCK into *status (device uint32,
 * may be NULL).  Destinations must be distinct and no destination may be
 * another pair's source (the copies run concurrently).  k_cache and v_cache
 * must be 16-byte aligned; 0 <= n_pairs <= 65535. */
int pa_copy_blocks(const pa_shape* shape, void* k_cache, void* v_cache, const int32_t* pairs,
                   int32_t n_pairs, uint32_t* status, pa_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDGQA_H */
