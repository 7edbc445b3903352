/*
 * pkv -- decode attention over a paged KV cache, for GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is either a host pointer (marked "host") or
 * device memory the caller owns (marked "device"); the library allocates
 * nothing and keeps no state between calls.  Each call that launches work is
 * asynchronous and stream-ordered on `stream` (a cudaStream_t passed as
 * void*), never synchronises the host, and may be captured into a CUDA graph:
 * lengths and segment layout are read from device memory when the kernels
 * run, so one capture serves every length the grid was sized for.
 *
 * Errors come back two ways.  Problems visible on the host (bad sizes, null
 * or misaligned pointers, an unsupported head_dim or dtype) return a negative
 * pkv_status before anything is launched.  Problems only the device sees (a
 * segment whose fields are out of range, a block id outside the pool, ...)
 * set PKV_ERR_* bits in the caller's `err_flags` word with an atomic OR and
 * zero that segment's output; no kernel traps or asserts, and every wait
 * inside a kernel is bounded.
 *
 * Sources, by page and section:
 *   [vllm-omni paged_decode.py]  "Paged KV cache for SenseNova-U1
 *       autoregressive decode" (vLLM-Omni): module constants BLOCK_SIZE,
 *       BUCKETS, TAIL_STEP and _bucket_for; PagedDecodeCache (layout,
 *       attend, grow, load_prefix, reusable_for, to_dynamic_cache);
 *       DecodeGraphRunner.
 *   [tiny-llm kv_cache.py]  causal_kwargs; SlotKVCache.end_step /
 *       advance_host; SlotLayerKV.update.
 *   [ExecuTorch #24072]  triton::sdpa_varlen over a seq_info segment table.
 *   [ExecuTorch #24073]  CudaBatchedSequenceCache: ring rows, scratch column.
 *   [ExecuTorch #24074]  batched-sequence manifest: ring slot formula,
 *       max_segments, per-call causal flag.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tokens per page ([vllm-omni paged_decode.py] BLOCK_SIZE). */
#define PKV_BLOCK_SIZE 16

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_EMPTY = 1,          /* nothing to do (an empty prefix); not an error */
    PKV_SAME_BUCKET = 2,    /* resize not needed: the length fits the current bucket */
    PKV_EINVAL = -1,        /* an argument is out of range, null or misaligned */
    PKV_EUNSUPPORTED = -2,  /* dtype or head_dim the kernels do not cover */
    PKV_ECUDA = -3,         /* a CUDA launch or copy failed to enqueue */
    PKV_ECAPACITY = -4,     /* the destination cannot hold the requested tokens */
    PKV_ESTALE = -5         /* descriptors that do not describe the same cache shape */
} pkv_status;

typedef enum pkv_dtype { PKV_BF16 = 0, PKV_F32 = 1 } pkv_dtype;

/* Device-side error bits, OR-ed into *err_flags. */
#define PKV_ERR_SEGMENT  (1u << 0)  /* q_start/q_len/col/kv_end out of range, or kv_end < q_len */
#define PKV_ERR_CAPACITY (1u << 1)  /* flat layout: kv_end > max_blocks_per_seq * 16 */
#define PKV_ERR_RING     (1u << 2)  /* ring layout: window <= 0 or window + q_len - 1 > ring_rows */
#define PKV_ERR_BLOCK    (1u << 3)  /* a block-table entry the segment needs is outside [0, num_blocks) */
#define PKV_ERR_QLEN     (1u << 4)  /* q_len above the max_q_len the launch was sized for */
#define PKV_ERR_OVERLAP  (1u << 5)  /* an output row lies in two segments (its value is then unspecified) */
#define PKV_ERR_TIMEOUT  (1u << 6)  /* a bounded wait for a K/V copy inside the kernel gave up; output zeroed */

/* Flags for the attention calls. */
#define PKV_FLAG_SIMT  (1u << 0)  /* bf16: use the CUDA-core kernels instead of the tensor-core ones */
#define PKV_FLAG_PDL   (1u << 1)  /* launch with programmatic dependent launch; see pkv_attend_varlen */
#define PKV_FLAG_PREFETCH_NEXT (1u << 2)  /* warm L2 with layer + 1's pages; see pkv_attend_varlen */
#define PKV_FLAG_MMA_SYNC (1u << 3)  /* bf16, head_dim 128, > 8 rows per kv head: mma.sync tile instead of tcgen05 */

/*
 * One paged K/V cache: per layer, a K pool and a V pool, each
 * (num_blocks, 16, kv_heads, head_dim) of `dtype`, row-major
 * ([vllm-omni paged_decode.py] PagedDecodeCache docstring), plus one block
 * table shared by all layers, int32 (max_seqs, max_blocks_per_seq), row
 * `col` listing the pages of sequence `col` in order.
 *
 * ring_rows = 0 means flat storage: position p lives at page p / 16, offset
 * p % 16 of the sequence's table row, so a sequence holds at most
 * max_blocks_per_seq * 16 tokens.  ring_rows = R > 0 (a multiple of 16, at
 * most max_blocks_per_seq * 16) means ring storage for sliding-window
 * attention: position p lives at slot p % R ([ExecuTorch #24074]), and a
 * window of W keys with steps of up to q_len rows needs
 * R >= W + q_len - 1 ([ExecuTorch #24073]).
 *
 * The descriptor is host memory owned by the caller; k and v are host arrays
 * of num_layers device pointers (16-byte aligned).  bucket is the token
 * capacity the buffers were sized for and generation counts reallocations
 * ([vllm-omni paged_decode.py] PagedDecodeCache.generation); the library
 * reads both and writes generation only in pkv_resize_bucket.
 *
 * first_valid (optional, NULL = no padding) is a device int32 array with one
 * entry per table row: the sequence's first valid position, for batches of
 * left-padded sequences ([tiny-llm kv_cache.py] SlotKVCache,
 * padded_causal_mask).  Every query row of that sequence then ignores the
 * keys before it, and a query row whose own position lies before it (a
 * padding row) attends to its own key alone, so no row is empty.  A
 * negative entry counts as 0.  Only the attention calls read it, before the
 * dependency wait like the block table, so the kernel launched just before
 * a PDL attention call must not write it.
 */
typedef struct pkv_cache {
    int32_t num_layers;
    int32_t kv_heads;
    int32_t head_dim;           /* multiple of 8, at most 256 */
    int32_t dtype;              /* pkv_dtype */
    int64_t num_blocks;
    int32_t max_seqs;
    int32_t max_blocks_per_seq;
    int32_t ring_rows;
    int32_t reserved0;
    void *const *k;             /* host array [num_layers] of device pointers */
    void *const *v;             /* host array [num_layers] of device pointers */
    const int32_t *block_table; /* device [max_seqs][max_blocks_per_seq] */
    int64_t bucket;
    int64_t generation;
    const int32_t *first_valid; /* device [max_seqs] or NULL; see above */
} pkv_cache;

/*
 * Growth schedule of the single-sequence decode cache
 * ([vllm-omni paged_decode.py] _bucket_for): the first of 512, 1024, 2048,
 * 4096, 8192 that holds `length`; past 8192, 8192 plus as many 2048-token
 * steps as cover the rest.  length <= 0 returns 512.  Host only.
 */
int64_t pkv_bucket_for(int64_t length);

/* Static string for a pkv_status value. */
const char *pkv_status_str(int status);

/*
 * Append this step's K/V rows ([vllm-omni paged_decode.py]
 * PagedDecodeCache.attend, which writes at length - 1 because the caller has
 * already advanced the length; [tiny-llm kv_cache.py] SlotLayerKV.update).
 *
 * seq_info: device int32 [num_segments][4] = (q_start, q_len, col, kv_end)
 * ([ExecuTorch #24072]).  kv_end counts the sequence's keys after this
 * append, so query row q_start + i (0 <= i < q_len) is the token at position
 * kv_end - q_len + i, and its K and V rows are copied bit for bit into that
 * position's slot of sequence `col`.
 * k_new, v_new: device [total_rows][kv_heads][head_dim] of the cache dtype.
 * window: the attention window the rows will be used with (checked against
 * ring_rows when the cache is a ring; ignored for flat storage).
 *
 * A segment is written only if it is valid as a whole: 0 <= q_start,
 * q_start + q_len <= total_rows, 0 <= col < max_seqs, q_len <= kv_end, the
 * capacity / ring rule above holds and every slot it writes maps to a block
 * id in [0, num_blocks).  Otherwise nothing of it is written and the matching
 * PKV_ERR_* bit is set.  Rows no segment covers are not written.  Two
 * segments that write the same slot race (unspecified result).
 * err_flags: device uint32, OR-ed, never cleared by the library.
 */
int pkv_append(const pkv_cache *cache, int32_t layer,
               const void *k_new, const void *v_new, int32_t total_rows,
               const int32_t *seq_info, int32_t num_segments, int32_t window,
               uint32_t *err_flags, void *stream);

/*
 * Decode attention over the paged cache ([ExecuTorch #24072]
 * triton::sdpa_varlen semantics over the paged layout of
 * [vllm-omni paged_decode.py]).
 *
 * q: device [total_rows][num_q_heads][head_dim] of the cache dtype; q head h
 * reads kv head h / (num_q_heads / kv_heads) (grouped-query attention; the
 * ratio must be a whole number).  For segment (q_start, q_len, col, kv_end),
 * row q_start + i sits at position p = kv_end - q_len + i and sees keys
 *   causal:     [lo, p + 1),        lo = max(0, p - window + 1) if window > 0 else 0
 *   non-causal: [lo, kv_end),       lo = max(0, kv_end - window) if window > 0 else 0
 * (bottom-right causal alignment, [tiny-llm kv_cache.py] causal_kwargs; for
 * q_len = 1 both are the same).  With cache->first_valid set and
 * f = max(first_valid[col], 0): a row with p < f sees key p alone, any other
 * row has lo raised to at least f.  out[row][h][:] = softmax(softmax_scale *
 * q.k) weighted sum of V, in fp32; lse[row][h] = natural-log sum of
 * exp(softmax_scale * q.k) (may be NULL).  Rows no segment covers, and rows of
 * invalid segments, get out = 0 and lse = -inf.  Keys at or past kv_end and
 * table entries past the keys a segment needs are never read, so they may
 * hold anything (NaN included).
 *
 * max_q_len bounds every segment's q_len and max_kv bounds every segment's
 * kv_end; both only size the launch, so a graph captured once serves every
 * length up to them.  num_splits (0..16) is the number of CTAs that share one
 * (segment, kv head) key range as a thread-block cluster; their partial
 * softmax results are merged by log-sum-exp through distributed shared
 * memory in the same launch, so no workspace is needed (workspace NULL,
 * workspace_bytes 0; see pkv_attend_workspace_bytes for the other mode).  0 picks the count
 * from the launch shape: a power of two aiming at about three waves of
 * resident CTAs (one wave for the tcgen05 tile of wide bf16 groups), the
 * largest cluster the device can co-schedule below it, and, for kernels
 * that fit once per SM with few (segment, kv head) ranges, the cluster size
 * that needs the fewest waves of clusters resident at once.  The tcgen05
 * tile also runs a range of at most 24 groups of 64 keys on one CTA of its
 * cluster, and with up to 64 segments takes the ranges longest first; the
 * results do not depend on either.  A larger count than the segment has
 * 16-token pages leaves CTAs idle.
 *
 * flags: PKV_FLAG_SIMT selects the CUDA-core kernels for bf16 (fp32 always
 * uses them): at most 8 query rows per kv head take the decode kernel's
 * variant with fp32 FMA products, wider groups the general CUDA-core tile.
 * PKV_FLAG_MMA_SYNC keeps wide bf16 groups at head_dim 128 (more than 8
 * rows per kv head) on the mma.sync tile instead of the tcgen05 one.  PKV_FLAG_PDL launches with programmatic dependent launch: the
 * kernel may start reading cache slots of positions below kv_end - q_len,
 * the block table and seq_info while the previous kernel on the stream is
 * still running, so set it only when that previous kernel writes none of
 * those; q, k_new, v_new, out, lse and err_flags are touched only after it
 * has finished.  PKV_FLAG_PREFETCH_NEXT (ignored for the last layer) also
 * brings into L2 the pages of layer + 1 that cover the same key ranges, for
 * a caller whose next call attends layer + 1 with the same block table and
 * segments (one decode step): a hint only, it changes no result.  The
 * prefetch is capped at about 48 MB per call.
 *
 * Device pointers must be 16-byte aligned (out and lse: 4-byte).
 */
int pkv_attend_varlen(const pkv_cache *cache, int32_t layer,
                      const void *q, int32_t num_q_heads, int32_t total_rows,
                      const int32_t *seq_info, int32_t num_segments,
                      int32_t max_q_len, int64_t max_kv, int32_t num_splits,
                      float softmax_scale, int32_t causal, int32_t window,
                      float *out, float *lse,
                      void *workspace, int64_t workspace_bytes,
                      uint32_t *err_flags, uint32_t flags, void *stream);

/*
 * pkv_append followed by pkv_attend_varlen in one launch: the rows of this
 * step are written into the cache and attended to from k_new / v_new
 * directly.  Same arguments and results as the two calls in sequence, with
 * one extra condition: no two segments of the call may name the same `col`
 * (the two-call sequence has no such limit).
 */
int pkv_append_attend(const pkv_cache *cache, int32_t layer,
                      const void *q, const void *k_new, const void *v_new,
                      int32_t num_q_heads, int32_t total_rows,
                      const int32_t *seq_info, int32_t num_segments,
                      int32_t max_q_len, int64_t max_kv, int32_t num_splits,
                      float softmax_scale, int32_t causal, int32_t window,
                      float *out, float *lse,
                      void *workspace, int64_t workspace_bytes,
                      uint32_t *err_flags, uint32_t flags, void *stream);

/*
 * Bytes of workspace the two calls above need for these launch bounds when
 * given one (0: the launch never uses it).  With a workspace, the decode
 * kernel (at most 8 query rows per segment and kv head: G * max_q_len <= 8,
 * bf16, tensor-core path) splits a key range over independent CTAs (up to 64
 * per range, num_splits 0..64) that merge through it: each writes its
 * partial rows, and the last to finish (counted with an atomic it resets)
 * merges them.  Without one (NULL), the splits form a thread-block cluster
 * and merge through distributed shared memory (num_splits 0..16).  The
 * workspace is device memory the caller owns, 16-byte aligned, zero-filled
 * before its first use and not touched by the caller between calls: its
 * first bytes are per-range arrival counters that every call leaves at zero,
 * the rest is scratch.  Used with larger launch bounds (more segments or kv
 * heads) than before, it must be zero-filled again.  Calls that may run
 * concurrently need their own.  A workspace smaller than this size is rejected with
 * PKV_EINVAL.  Returns a negative pkv_status for invalid bounds.
 */
int64_t pkv_attend_workspace_bytes(const pkv_cache *cache, int32_t num_q_heads,
                                   int32_t num_segments, int32_t max_q_len,
                                   int64_t max_kv, int32_t num_splits, uint32_t flags);

/*
 * pkv_append_attend with the split-merge workspace taken from a fixed 8 MiB
 * scratch array in the library's device memory instead of the caller: no
 * allocation, no workspace argument.  The pages have no counterpart of this
 * call.  It serves callers that may not allocate device memory at the point
 * of the call: an allocator-free runtime, a custom-op shim that owns no
 * memory pool, or code running while an allocator must not be touched.  The
 * scratch is a file-scope __device__ array (every device that loads the
 * library holds it until the process exits), zero at load; the arrival
 * counters live in an array of their own that every call leaves at zero.
 * Its device address is looked up with cudaGetSymbolAddress on every call
 * (a host-side query, so a new context after cudaDeviceReset is picked up);
 * the first call on a device also loads the library's module there, so make
 * it before any stream capture.  A launch whose merge would need more than
 * 8 MiB (see pkv_attend_workspace_bytes) or more than 4096 (segment, kv
 * head, row tile) ranges is rejected with PKV_ECAPACITY before anything
 * runs; a failed lookup returns PKV_ECUDA.  The scratch is shared by every
 * call on a device and keeps the last call's partials, so calls that overlap
 * on the GPU race: issue them on one stream, or serialise them.  Otherwise
 * the same arguments, results and errors as pkv_append_attend.
 */
int pkv_append_attend_noalloc(const pkv_cache *cache, int32_t layer,
                              const void *q, const void *k_new, const void *v_new,
                              int32_t num_q_heads, int32_t total_rows,
                              const int32_t *seq_info, int32_t num_segments,
                              int32_t max_q_len, int64_t max_kv, int32_t num_splits,
                              float softmax_scale, int32_t causal, int32_t window,
                              float *out, float *lse,
                              uint32_t *err_flags, uint32_t flags, void *stream);

/*
 * Build a segment table from the flash-attention argument form
 * ([vllm-omni paged_decode.py] PagedDecodeCache.attend passes cu_seqlens_q
 * and seqused_k): seq_info[s] = (cu_seqlens_q[s], cu_seqlens_q[s+1] -
 * cu_seqlens_q[s], s, seqused_k[s]) for s < num_seqs.  All device int32.
 */
int pkv_seqinfo_from_seqused(const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                             int32_t num_seqs, int32_t *seq_info_out, void *stream);

/*
 * seq_clone of the batched-sequence cache ([ExecuTorch #24073]
 * CudaBatchedSequenceCache: a device copy of the source prefix), over the
 * paged layout: in every layer, positions 0 .. n-1 of the sequence in
 * block-table row src_col are copied bit for bit (all kv heads) to the same
 * positions of row dst_col, each side mapped through its own table row.
 * With ring storage only the last min(n, ring_rows) positions exist and are
 * copied (slot position % ring_rows on both sides).  Typical use: admit a
 * request that shares a prefix, then set its segment's kv_end to n.
 * All or nothing per layer: if any page either side needs is outside
 * [0, num_blocks), that layer is not written and PKV_ERR_BLOCK is set.  The
 * two rows' pages must not overlap (other than being identical).  Host
 * errors: a column outside [0, max_seqs), n < 0, or (flat layout) n beyond
 * the table's capacity (PKV_ECAPACITY).  Launches one kernel per layer.
 */
int pkv_seq_clone(const pkv_cache *cache, int32_t src_col, int32_t dst_col, int64_t n,
                  uint32_t *err_flags, void *stream);

/*
 * rewind of the batched-sequence cache ([ExecuTorch #24073], bounded by the
 * ring floor), on the device: kv_end -= amount[s] for every segment s
 * (amount: device int32[num_segments]), e.g. the draft tokens a verify step
 * rejected; their slots are simply rewritten by the next append.  A segment
 * keeps its kv_end and sets PKV_ERR_SEGMENT when amount < 0 or
 * amount > kv_end, and PKV_ERR_RING when the cache is a ring of R rows and
 * amount > R - window + 1 (the next step's window would need positions the
 * ring no longer holds; window must be > 0 with rings).  The block table is
 * untouched: removing a sequence (seq_rm) is the caller releasing its table
 * row's pages, which needs no device work.
 */
int pkv_rewind(const pkv_cache *cache, int32_t *seq_info, int32_t num_segments,
               const int32_t *amount, int32_t window, uint32_t *err_flags, void *stream);

/*
 * Advance every segment to the next step on the device: kv_end += q_len
 * ([tiny-llm kv_cache.py] SlotKVCache.end_step does the same for slot
 * lengths inside a captured graph, so a replay needs no host write).
 */
int pkv_advance(int32_t *seq_info, int32_t num_segments, void *stream);

/*
 * Move a cache to a larger bucket, keeping the first old_len tokens
 * ([vllm-omni paged_decode.py] PagedDecodeCache.grow).  new_cache describes
 * buffers the caller has already allocated for the new bucket (same layers,
 * kv_heads, head_dim, dtype, ring_rows = 0, identity-ordered tables); the
 * first old_len flat rows of every layer's K and V are copied from old to
 * new.  Only after every copy has been enqueued is new_cache->generation set
 * to old_cache->generation + 1, so a failure leaves both descriptors as they
 * were and a graph keyed on the old generation is never paired with half-built
 * buffers.  Returns PKV_SAME_BUCKET, copying nothing, when
 * new_cache->bucket == old_cache->bucket; PKV_ESTALE when the shapes differ;
 * PKV_ECAPACITY when old_len exceeds either cache's rows.
 */
int pkv_resize_bucket(const pkv_cache *old_cache, pkv_cache *new_cache,
                      int64_t old_len, void *stream);

/*
 * Copy a prefill cache into the paged buffers ([vllm-omni paged_decode.py]
 * PagedDecodeCache.load_prefix): for every layer l, token s < n and kv head
 * h, keys[l] + s*stride_s + h*stride_h (elements; head_dim contiguous) goes
 * to flat row s of layer l's K pool, and likewise values.  keys / values are
 * host arrays of num_layers device pointers, so a [B, H, S, D] tensor's
 * batch-0 view is passed with stride_s = D, stride_h = S*D.  Rows past n are
 * left as they were.  Returns PKV_EMPTY (and copies nothing) when n == 0 or
 * keys is NULL.
 */
int pkv_load_prefix(const pkv_cache *cache, const void *const *keys,
                    const void *const *values, int64_t n,
                    int64_t stride_s, int64_t stride_h, void *stream);

/*
 * Write-back for a stage that reads an ordinary cache
 * ([vllm-omni paged_decode.py] PagedDecodeCache.to_dynamic_cache): copy the
 * first n flat rows of layer `layer` into keys_out / values_out laid out
 * [kv_heads][n][head_dim] (device, contiguous).
 */
int pkv_to_contiguous(const pkv_cache *cache, int32_t layer, int64_t n,
                      void *keys_out, void *values_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
