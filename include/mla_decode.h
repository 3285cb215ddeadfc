/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library
 * (libmla_decode.so).
 *
 * The operation is Multi-head Latent Attention decode over a paged latent KV
 * cache: the computation of FlashMLA's flash_mla_with_kvcache and
 * get_mla_metadata, as the PAI tutorial "云上玩转DeepSeek系列之五" calls them
 * from vLLM (section 2, FlashMLAImpl / FlashMLAMetadataBuilder) and
 * benchmarks them (section 4, compare_a: q[b, s_q, h_q, d],
 * blocked_k[num_blocks, 64, h_kv, d], block_table, cache_seqlens, dv, causal,
 * returning out and lse).  For sequence i, query position j and head h, with
 * g = h / (h_q / h_kv):
 *
 *   visible t:  t < L_i, and with causal also t <= L_i - s_q + j
 *   K_t = kcache[block_table[i][t/64]][t%64][g][0:576],  V_t = K_t[0:512]
 *   out[i,j,h,:] = sum_t softmax_t(softmax_scale * <q[i,j,h,:], K_t>) V_t
 *   lse[i,h,j]   = ln sum_t exp(softmax_scale * <q[i,j,h,:], K_t>)
 *
 * A row with no visible token gets out = 0 and lse = -inf.  The split of the
 * KV length across SMs and the merge of the pieces by their log-sum-exps is
 * Flash-Decoding's (Hacker News thread on the FlashMLA release).  A cache
 * entry may be padded: `stride` is the number of elements from one entry to
 * the next, 576 or the 256-byte aligned 640 of vLLM PR #12676 ("Mem align KV
 * caches for CUDA devices"); the padding is never read.
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers on the current CUDA device, owned
 *    by the caller.  The library allocates nothing and never synchronises; the
 *    calls only enqueue kernels on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and may be captured in a CUDA graph.  The host-buffer
 *    calls at the end of this file (mla_host_*, mla_decode_host) are the one
 *    exception, and say how.
 *  - bf16 arrays are passed as void* holding IEEE bfloat16 values.
 *  - Arguments that the host can check are checked before anything is
 *    enqueued; a failed check returns a negative mla_status_t and enqueues
 *    nothing.
 *  - Problems only the device can see (a page id outside [0, num_blocks), a
 *    negative sequence length, an internal wait that timed out) are written to
 *    the caller's int32 `status` word in device memory.  The library never
 *    clears it: set it to 0 before the calls and read it after synchronising.
 *    A kernel that reports an error still exits normally; its outputs are then
 *    unspecified.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mla_status_t;
enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,  /* a shape or size outside what the call accepts   */
  MLA_ERR_UNSUPPORTED = -2,  /* legal in principle, not built here (e.g. d != 576) */
  MLA_ERR_ALIGNMENT = -3,    /* a pointer or stride not 16-byte aligned          */
  MLA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed                */
  MLA_ERR_BAD_BLOCK_ID = -5, /* device: block_table entry outside the cache      */
  MLA_ERR_TIMEOUT = -6,      /* device: a pipeline wait gave up                  */
  MLA_ERR_BAD_SEQLEN = -7,   /* device: cache_seqlens entry < 0                  */
  MLA_ERR_SCRATCH_TOO_SMALL = -8 /* the shape needs more than the built-in scratch */
};

typedef struct CUstream_st *mla_stream_t; /* the same type as cudaStream_t */

/* Human-readable name of a status code (static storage, never NULL). */
const char *mla_status_string(mla_status_t status);

/*
 * Recommended number of scheduler parts for `device`: how many decode units
 * fit on the GPU at once, divided among the (row tile, KV head) grid
 * dimensions of this shape.  A unit is a 2-CTA cluster of the 128-row kernel,
 * or, when s_q x (h_q / h_kv) <= 16, one CTA of the 16-row kernel.  Returns a count >= 1, or a negative
 * mla_status_t.  The first call per device queries occupancy; later calls are
 * cheap.
 */
int mla_num_parts(int s_q, int h_q, int h_kv, int device);

/* Size of the metadata array in int32 elements: num_parts x 8. */
size_t mla_metadata_ints(int num_parts);

/*
 * Bytes of scratch the decode call needs for split partial results:
 * (b + num_parts) x s_q x h_q x 512 fp32 partial outputs, then
 * (b + num_parts) x s_q x h_q fp32 partial lse, each block 256-byte aligned.
 */
size_t mla_workspace_bytes(int b, int s_q, int h_q, int num_parts);

/*
 * Split-KV schedule (the role of FlashMLA's get_mla_metadata, called once per
 * decode step and shared by every layer).  Cuts the (sequence, page) order of
 * the batch into num_parts contiguous, cost-balanced parts; each part becomes
 * one decode unit per KV head (and row tile): a 2-CTA cluster of the 128-row
 * kernel, or one CTA of the 16-row kernel.
 *   cache_seqlens  int32[b]            tokens per sequence (device)
 *   b              1 .. 16384
 *   num_parts      >= 1 (normally mla_num_parts())
 *   metadata       int32[num_parts*8]  out: per part {first seq, first page,
 *                                       last seq, end page, first split index, 0,0,0}
 *   num_splits     int32[b+1]          out: exclusive prefix sum of the number
 *                                       of pieces each sequence is cut into
 *   status         int32[1]            device error word (see conventions)
 * One single-block kernel on `stream`; no host synchronisation.
 */
mla_status_t mla_get_metadata(const int32_t *cache_seqlens, int b, int num_parts,
                              int32_t *metadata, int32_t *num_splits, int32_t *status,
                              mla_stream_t stream);

/*
 * MLA decode over the paged latent cache (the role of flash_mla_with_kvcache).
 *   q             bf16[b, s_q, h_q, d], contiguous, 16-byte aligned
 *   d             must be 576 (512 latent + 64 rope)
 *   kcache        bf16, entry (page, slot, g) at
 *                 kcache + ((page*block_size + slot)*h_kv + g)*stride; 16-byte aligned
 *   num_blocks    pages in the cache (num_blocks*64 < 2^31)
 *   block_size    must be 64
 *   h_kv          KV heads; h_q % h_kv == 0 and h_q/h_kv <= 128
 *   stride        elements per entry, >= 576 and a multiple of 8 (576 or 640)
 *   block_table   int32[b, max_blocks_per_seq]; only the first ceil(L_i/64)
 *                 entries of row i are read
 *   cache_seqlens int32[b], 0 <= L_i <= max_blocks_per_seq*64
 *   dv            must be 512
 *   metadata, num_parts, num_splits: from mla_get_metadata on the same
 *                 cache_seqlens (and the same num_parts)
 *   softmax_scale finite and > 0 (FlashMLA's benchmark uses d**-0.5)
 *   causal        0 or 1; with 1, query j sees tokens t <= L_i - s_q + j
 *   out           bf16[b, s_q, h_q, 512], 16-byte aligned (written)
 *   lse           fp32[b, h_q, s_q], natural log (written)
 *   workspace     >= mla_workspace_bytes(b, s_q, h_q, num_parts) bytes,
 *                 16-byte aligned, contents need not be initialised
 *   status        int32[1] device error word
 * Enqueues the decode kernel and the combine kernel on `stream`.
 */
mla_status_t mla_decode_with_kvcache(const void *q, int b, int s_q, int h_q, int d,
                                     const void *kcache, int64_t num_blocks, int block_size,
                                     int h_kv, int stride, const int32_t *block_table,
                                     int max_blocks_per_seq, const int32_t *cache_seqlens,
                                     int dv, const int32_t *metadata, int num_parts,
                                     const int32_t *num_splits, float softmax_scale, int causal,
                                     void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t *status,
                                     mla_stream_t stream);

/*
 * The two halves of mla_decode_with_kvcache, for callers that time or
 * schedule them separately.  mla_decode_splitkv takes the same arguments and
 * runs only the decode kernel: sequences cut into one piece get their out and
 * lse written directly; the pieces of the others go to `workspace` as
 * normalised fp32 partial outputs and fp32 natural-log partial lse.
 * mla_combine_splits then merges those pieces by their log-sum-exps (the
 * Flash-Decoding merge) into out and lse, and writes out = 0, lse = -inf for
 * sequences of length 0.  It must run after mla_decode_splitkv on the same
 * workspace, b, s_q, h_q and num_parts; ordering on one stream suffices.
 * num_parts also sets the merge kernel's shape: with num_parts >= 2 b
 * (sequences in many pieces) each row gets four warps, otherwise one.
 *
 * Both kernels are launched with programmatic dependent launch: they may
 * start their set-up (shared and tensor memory only) while the kernel before
 * them on the stream is still running, and wait for that kernel to complete
 * before they read or write any global memory, so stream order keeps its
 * usual meaning for the caller.
 */
mla_status_t mla_decode_splitkv(const void *q, int b, int s_q, int h_q, int d,
                                const void *kcache, int64_t num_blocks, int block_size,
                                int h_kv, int stride, const int32_t *block_table,
                                int max_blocks_per_seq, const int32_t *cache_seqlens, int dv,
                                const int32_t *metadata, int num_parts,
                                const int32_t *num_splits, float softmax_scale, int causal,
                                void *out, float *lse, void *workspace, size_t workspace_bytes,
                                int32_t *status, mla_stream_t stream);

mla_status_t mla_combine_splits(const int32_t *num_splits, int b, int s_q, int h_q,
                                const void *workspace, int num_parts, void *out, float *lse,
                                mla_stream_t stream);

/*
 * Diagnostic of the decode kernels' failure detection (no counterpart on the
 * pages).  Same arguments and host-side checks as mla_decode_with_kvcache, but
 * the kernel's TMA producer first waits on a barrier that nothing ever
 * completes, before it issues any copy.  Every wait in the kernels is bounded
 * (about 2 s): that wait gives up, raises the CTA's abort flag, every other
 * warp role leaves its own wait, the CTAs exit (the 128-row kernel's after
 * freeing their tensor memory),
 * and MLA_ERR_TIMEOUT (-6) is written to *status.  out and lse are left
 * undefined.  The device stays usable: the next call decodes normally.  Lets a
 * caller check that a wait that can never end is reported, not hung on.
 */
mla_status_t mla_selftest_wait_timeout(const void *q, int b, int s_q, int h_q, int d,
                                       const void *kcache, int64_t num_blocks, int block_size,
                                       int h_kv, int stride, const int32_t *block_table,
                                       int max_blocks_per_seq, const int32_t *cache_seqlens,
                                       int dv, const int32_t *metadata, int num_parts,
                                       const int32_t *num_splits, float softmax_scale,
                                       int causal, void *out, float *lse, void *workspace,
                                       size_t workspace_bytes, int32_t *status,
                                       mla_stream_t stream);

/*
 * Cache maintenance next to the decode (MLA caches have one latent KV head).
 *
 * mla_write_cache puts new tokens into the paged cache the decode reads:
 * for each token t with s = slot_mapping[t] >= 0, entry
 * (page s / block_size, slot s % block_size) receives the 512 latent values
 * kv_c[t] followed by the 64 rope values k_pe[t].  Negative slot ids are
 * skipped (padding tokens); slot ids >= num_blocks*block_size are skipped
 * and reported as MLA_ERR_BAD_BLOCK_ID in `status`.  The pad of 640-element
 * entries is never written.
 *   kv_c          bf16 rows of 512, `kv_c_row_stride` elements apart (>= 512, multiple of 8)
 *   k_pe          bf16 rows of 64, `k_pe_row_stride` elements apart (>= 64, multiple of 8)
 *   slot_mapping  int64[num_tokens]
 *   kcache        as for mla_decode_with_kvcache with h_kv = 1
 * All device pointers 16-byte aligned.  One kernel on `stream`.
 *
 * mla_copy_blocks is copy_blocks_mla of vLLM PR #12676: for each of
 * `num_layers` caches (kcaches: a DEVICE array of num_layers device pointers,
 * each 16-byte aligned) and each pair (src, dst) of block_mapping (int64[num_pairs][2],
 * device), page dst becomes a copy of page src, pad included.  Sources and
 * destinations must be disjoint; ids outside [0, num_blocks) are skipped and
 * reported as MLA_ERR_BAD_BLOCK_ID.  One kernel on `stream`.
 */
mla_status_t mla_write_cache(const void *kv_c, int64_t kv_c_row_stride, const void *k_pe,
                             int64_t k_pe_row_stride, const int64_t *slot_mapping,
                             int64_t num_tokens, void *kcache, int64_t num_blocks, int block_size,
                             int stride, int32_t *status, mla_stream_t stream);

mla_status_t mla_copy_blocks(const uint64_t *kcaches, int num_layers, const int64_t *block_mapping,
                             int64_t num_pairs, int64_t num_blocks, int block_size, int stride,
                             int32_t *status, mla_stream_t stream);

/*
 * Bytes of the library's built-in split-KV scratch (64 MiB), used by
 * mla_decode_with_kvcache_static.
 */
#define MLA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)

/*
 * mla_decode_with_kvcache without the `workspace` arguments: the split-KV
 * scratch (partial outputs of sequences cut into several pieces) comes from a
 * buffer of MLA_STATIC_WORKSPACE_BYTES that the library itself holds in device
 * memory, so the call allocates nothing and needs nothing allocated for it
 * beyond its inputs and outputs.  The pages have no counterpart of this call.
 *
 * It exists for callers that have no way to obtain device memory of their
 * own at the point of the call: code loaded into a host program whose device
 * memory is entirely owned by that program's pool and which gives its
 * plug-ins no allocator, or a latency-critical serving loop that must not
 * call cudaMalloc, which can synchronise the whole device.
 *
 * Limits and behaviour:
 *  - Every process that loads the library keeps the 64 MiB buffer on each GPU
 *    where the library's kernels are loaded, until it exits.
 *  - Shapes whose mla_workspace_bytes(b, s_q, h_q, num_parts) exceeds
 *    MLA_STATIC_WORKSPACE_BYTES are rejected with MLA_ERR_SCRATCH_TOO_SMALL
 *    before anything is enqueued (b=128, s_q=1, h_q=128 with 76 parts needs
 *    about 54 MB and fits).
 *  - The first call on a device looks the buffer's device address up
 *    (cudaGetSymbolAddress) with that device current and keeps it for the
 *    life of the process.  The address belongs to the device's primary
 *    context: after cudaDeviceReset, or with another context current on that
 *    device, it is no longer valid and the call must not be used.
 *  - All calls share the one buffer: calls whose kernels may overlap on the
 *    GPU (different streams without ordering, or several host threads) race
 *    on it and give undefined results.  Calls ordered on one stream are safe.
 *    The buffer keeps the last call's contents; nothing in it needs to start
 *    at zero, because each call writes every scratch entry it later reads.
 * All other arguments, results and errors are those of mla_decode_with_kvcache.
 */
mla_status_t mla_decode_with_kvcache_static(const void *q, int b, int s_q, int h_q, int d,
                                            const void *kcache, int64_t num_blocks,
                                            int block_size, int h_kv, int stride,
                                            const int32_t *block_table, int max_blocks_per_seq,
                                            const int32_t *cache_seqlens, int dv,
                                            const int32_t *metadata, int num_parts,
                                            const int32_t *num_splits, float softmax_scale,
                                            int causal, void *out, float *lse, int32_t *status,
                                            mla_stream_t stream);

/*
 * Decode from HOST buffers, with the copies overlapped with the compute.
 * The pages' benchmark hands the decode device tensors; a serving process
 * whose query vectors and block tables are built on the CPU must also move
 * them over and read the results back.  This call does the whole round trip:
 * it cuts the batch into `chunks` runs of consecutive sequences balanced by
 * their page counts, copies the inputs of run k to the device while run k-1
 * decodes, and copies the outputs of run k back while run k+1 decodes.  Each
 * run is an independent, complete decode (its own schedule over all
 * num_parts parts), so the results equal those of mla_decode_with_kvcache
 * up to the rounding of a different split-KV cut (identical with chunks = 1).
 *
 * A pipeline object holds two CUDA streams (copies in, copies out) and the
 * events that order them against the caller's stream; it is the only object
 * in this library that allocates anything, and only when it is created:
 *   mla_host_pipeline_create   creates one on the current device (*pipeline
 *                              receives it; MLA_ERR_CUDA if a stream or event
 *                              could not be made, nothing is then leaked)
 *   mla_host_pipeline_destroy  synchronises its streams and frees it (NULL is
 *                              accepted and ignored)
 * One pipeline serves one host thread at a time.
 */
typedef struct mla_host_pipeline mla_host_pipeline;

#define MLA_HOST_MAX_CHUNKS 8

mla_status_t mla_host_pipeline_create(mla_host_pipeline **pipeline);
mla_status_t mla_host_pipeline_destroy(mla_host_pipeline *pipeline);

/*
 * The cut mla_decode_host makes (pure host code, no GPU needed): writes
 * n + 1 sequence indices 0 = bounds[0] < bounds[1] < ... < bounds[n] = b into
 * `bounds` (room for MLA_HOST_MAX_CHUNKS + 1) and returns n, or a negative
 * mla_status_t for b < 1 or NULL pointers.  Sequence i costs
 * ceil(max(L_i, 0) / 64) + 1 units.  The first and the last run take half the
 * share of a middle run (shares 1, 2, ..., 2, 1 in halves of a share; two runs
 * share evenly), because their copies in and out have no decode to overlap:
 * run k ends at the first sequence where the running cost reaches
 * (2k - 1) / (2n - 2) of the total (k / 2 with two runs), moved as needed so
 * that every run holds at least one sequence.  chunks >= 1 asks for that many runs
 * (capped at MLA_HOST_MAX_CHUNKS and at b); chunks <= 0 picks
 * n = total pages / 2800, rounded, clamped to [1, 3]: fewer, larger runs when the
 * batch is small, so that the fixed cost of a run (a schedule, a pipeline
 * fill, a merge) stays small against its pages.
 */
int mla_host_chunks(const int32_t *cache_seqlens, int b, int chunks, int32_t *bounds);

/*
 * Device scratch for mla_decode_host: staging of q, block_table,
 * cache_seqlens, out and lse for the whole batch, MLA_HOST_MAX_CHUNKS sets of
 * scheduler metadata and one split-KV workspace, each 256-byte aligned.
 */
size_t mla_host_scratch_bytes(int b, int s_q, int h_q, int max_blocks_per_seq, int num_parts);

/*
 * Arguments as for mla_decode_with_kvcache, except:
 *   q, block_table, cache_seqlens   HOST arrays (same shapes and types)
 *   out, lse                        HOST arrays, written
 *   num_parts                       parts per run (normally mla_num_parts());
 *                                   there are no metadata/num_splits arguments:
 *                                   each run's schedule is made on the device
 *   chunks                          as for mla_host_chunks
 *   scratch                         DEVICE memory, >= mla_host_scratch_bytes(...)
 *                                   bytes, 256-byte aligned, owned by the caller
 *   kcache, status                  DEVICE, as before
 * Host memory should be page-locked (cudaHostAlloc / pinned): pageable
 * buffers give the same results without the overlap.  cache_seqlens is read
 * by the host during the call (to make the cut) and again by a copy later.
 * The call returns once everything is enqueued: q, block_table and
 * cache_seqlens must stay unchanged, and out and lse must not be read, until
 * `stream` has reached the call's end (e.g. cudaStreamSynchronize(stream)).
 * All work is ordered after the work already on `stream` and everything
 * enqueued on `stream` later runs after all of the call's copies.  Calls on
 * one pipeline are ordered after one another whatever their streams; two
 * pipelines must not share one scratch buffer while their calls may overlap.
 * The argument checks of mla_decode_with_kvcache (on the device staging
 * pointers) run before anything is enqueued; MLA_ERR_INVALID_ARG also for
 * a NULL pipeline, a pipeline made on another device, a scratch too small or
 * not 256-byte aligned, b above 16384, and any cache_seqlens entry outside
 * [0, max_blocks_per_seq*64] (checked on the host, since the lengths are
 * there).  A CUDA call that fails part-way
 * returns MLA_ERR_CUDA with the runs before it already enqueued; the copies
 * already queued on the pipeline's own streams are still joined into `stream`
 * (as far as the failing CUDA state allows), so synchronising `stream` still
 * waits for every write into out and lse.  Not meant for stream capture.
 */
mla_status_t mla_decode_host(mla_host_pipeline *pipeline, const void *q, int b, int s_q, int h_q,
                             int d, const void *kcache, int64_t num_blocks, int block_size,
                             int h_kv, int stride, const int32_t *block_table,
                             int max_blocks_per_seq, const int32_t *cache_seqlens, int dv,
                             int num_parts, float softmax_scale, int causal, void *out,
                             float *lse, int chunks, void *scratch, size_t scratch_bytes,
                             int32_t *status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
