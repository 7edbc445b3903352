/*
 * Paged decode attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library.  The product path never does: it has its own CUDA
 * kernels and shares no code, header or constant with this file.
 *
 * Plain fp64 loops written from the definition of the operation: gather each
 * visible key through the block table, take softmax(scale * q.k) over them and
 * average V with those weights.  No blocking, splitting, fusion or reordering.
 *
 * Sources (page title, section):
 *   [vllm-omni paged_decode.py]  SenseNova-U1 paged decode, vLLM-Omni:
 *       BLOCK_SIZE / BUCKETS / TAIL_STEP constants and _bucket_for;
 *       PagedDecodeCache.__init__ (pool layout, identity block table);
 *       PagedDecodeCache.attend (append at length-1, attend over seqused,
 *       causal=False for one token).
 *   [tiny-llm kv_cache.py]  causal_kwargs (bottom-right causal alignment of
 *       several new queries on a non-empty cache); SlotLayerKV.update
 *       (write at the current length, then attend through it).
 *   [ExecuTorch #24072]  triton::sdpa_varlen: seq_info (q_start, q_len, col,
 *       kv_end), causal / non-causal, sliding window, ring storage, GQA,
 *       rows no segment covers are zeroed.
 *   [ExecuTorch #24074]  ring slot = position % rows.
 *   [ExecuTorch #24073]  ring layers hold window + max_write - 1 rows;
 *       CudaBatchedSequenceCache's BatchControl: seq_clone (device copy of
 *       the source prefix), rewind (bounded by the ring floor).
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes): q head h uses kv head h / (Hq / Hkv); the window covers W keys
 * ending at the query's own position (causal) or at kv_end - 1 (non-causal);
 * kv_end counts the keys after this step's append; an empty key range gives
 * out = 0 and lse = -inf; a ring needs window > 0 and
 * window + q_len - 1 <= ring_rows; a segment that fails validation writes
 * nothing and its rows read 0; an append is gated by the slots it writes, an
 * attention by every key it reads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_BLOCK 16

/* Growth schedule printed in vllm-omni paged_decode.py (module constants). */
static const int64_t kBuckets[5] = {512, 1024, 2048, 4096, 8192};
static const int64_t kTailStep = 2048;

/* _bucket_for: first listed bucket that holds `length`, else the last bucket
 * plus enough TAIL_STEP-sized steps to cover the excess. */
int64_t oracle_bucket_for(int64_t length)
{
    for (int i = 0; i < 5; ++i)
        if (length <= kBuckets[i]) return kBuckets[i];
    int64_t over = length - kBuckets[4];
    int64_t steps = (over + kTailStep - 1) / kTailStep;
    return kBuckets[4] + steps * kTailStep;
}

/* Validation status of one segment; 0 = valid.  The same rules gate the
 * append and the attention. */
enum {
    OR_OK = 0,
    OR_BAD_SEGMENT = 1,   /* q_start / q_len / col / kv_end out of range */
    OR_CAPACITY = 2,      /* flat layout: kv_end beyond the table's capacity */
    OR_RING = 3,          /* ring layout: window missing or too wide for the ring */
    OR_BLOCK = 4          /* a block id the segment needs is out of range */
};

typedef struct {
    int64_t num_blocks;
    int kv_heads, head_dim;
    const int32_t *block_table;
    int max_seqs, max_blocks_per_seq;
    int ring_rows;        /* 0 = flat */
} oracle_pool;

/* Logical key position -> (block id, in-block offset) through the table. */
static int locate(const oracle_pool *P, int col, int64_t pos, int64_t *blk, int *off)
{
    int64_t r = P->ring_rows ? pos % P->ring_rows : pos;
    int64_t page = r / ORACLE_BLOCK;
    if (page < 0 || page >= P->max_blocks_per_seq) return OR_CAPACITY;
    int64_t b = P->block_table[(int64_t)col * P->max_blocks_per_seq + page];
    if (b < 0 || b >= P->num_blocks) return OR_BLOCK;
    *blk = b;
    *off = (int)(r % ORACLE_BLOCK);
    return OR_OK;
}

/* Key range [lo, hi) that query row i of a segment sees.  `first` is the
 * sequence's first valid position (left padding of a batched prefill,
 * [tiny-llm kv_cache.py] SlotKVCache / padded_causal_mask): keys before it
 * are hidden, and a row that itself sits before it sees only its own key
 * (the diagonal is always kept). */
static void key_range(int64_t kend, int64_t qlen, int64_t i, int causal, int window, int64_t first,
                      int64_t *lo, int64_t *hi)
{
    int64_t p = kend - qlen + i;          /* this row's own position */
    *hi = causal ? p + 1 : kend;
    int64_t last = causal ? p : kend - 1;
    *lo = 0;
    if (window > 0 && last - window + 1 > 0) *lo = last - window + 1;
    if (p < first) {
        *lo = p;
        *hi = p + 1;
    } else if (*lo < first) {
        *lo = first;
    }
}

/* Segment validity.  The attention needs every key any row of the segment
 * reads to map to a valid block; the append only needs the slots it writes
 * (positions kv_end - q_len .. kv_end - 1), so `written_only` narrows the
 * block check to those. */
static int check_segment(const oracle_pool *P, const int32_t *seg, int total_rows,
                         int causal, int window, int64_t first, int written_only)
{
    int64_t q0 = seg[0], ql = seg[1], col = seg[2], kend = seg[3];
    if (q0 < 0 || ql < 0 || q0 + ql > total_rows) return OR_BAD_SEGMENT;
    if (col < 0 || col >= P->max_seqs) return OR_BAD_SEGMENT;
    if (kend < ql) return OR_BAD_SEGMENT;
    if (P->ring_rows) {
        if (window <= 0 || window + ql - 1 > P->ring_rows) return OR_RING;
    } else if (kend > (int64_t)P->max_blocks_per_seq * ORACLE_BLOCK) {
        return OR_CAPACITY;
    }
    if (ql == 0) return OR_OK;
    /* Every key any row may read, and every slot the append writes, must map
     * to a valid block.  Rows' ranges are nested at the top (all end at or
     * before kv_end) and the first row starts lowest. */
    int64_t lo0, hi0, lo_last, hi_last;
    key_range(kend, ql, 0, causal, window, first, &lo0, &hi0);
    key_range(kend, ql, ql - 1, causal, window, first, &lo_last, &hi_last);
    int64_t lo = lo0 < lo_last ? lo0 : lo_last;
    if (written_only) lo = kend - ql;
    for (int64_t j = lo; j < kend; ++j) {
        int64_t b; int o;
        int st = locate(P, (int)col, j, &b, &o);
        if (st) return st;
    }
    return OR_OK;
}

/* Append: each query row's new K/V row goes to the slot of its own position
 * kv_end - q_len + i, copied bit for bit.  Rows of an invalid segment, and
 * rows no segment covers, are not written.  Returns a bitmask of
 * (1 << status) over segments that failed. */
int oracle_append(uint8_t *k_pool, uint8_t *v_pool, int elem_size,
                  int64_t num_blocks, int kv_heads, int head_dim,
                  const int32_t *block_table, int max_seqs, int max_blocks_per_seq,
                  int ring_rows, int window, int causal,
                  const uint8_t *k_new, const uint8_t *v_new, int total_rows,
                  const int32_t *seq_info, int num_segments)
{
    oracle_pool P = {num_blocks, kv_heads, head_dim, block_table, max_seqs,
                     max_blocks_per_seq, ring_rows};
    int64_t row_bytes = (int64_t)kv_heads * head_dim * elem_size;
    int errs = 0;
    for (int s = 0; s < num_segments; ++s) {
        const int32_t *seg = seq_info + 4 * s;
        int st = check_segment(&P, seg, total_rows, causal, window, 0, 1);
        if (st) { errs |= 1 << st; continue; }
        for (int64_t i = 0; i < seg[1]; ++i) {
            int64_t t = seg[0] + i;
            int64_t pos = (int64_t)seg[3] - seg[1] + i;
            int64_t b; int o;
            locate(&P, seg[2], pos, &b, &o);
            int64_t dst = (b * ORACLE_BLOCK + o) * row_bytes;
            memcpy(k_pool + dst, k_new + t * row_bytes, (size_t)row_bytes);
            memcpy(v_pool + dst, v_new + t * row_bytes, (size_t)row_bytes);
        }
    }
    return errs;
}

/* Attention over the live keys.  Layouts (row-major, fp64):
 *   q   [total_rows][q_heads][head_dim]
 *   k/v [num_blocks][16][kv_heads][head_dim]
 *   out [total_rows][q_heads][head_dim], lse [total_rows][q_heads] (natural log)
 * `work` is caller scratch of at least max_keys doubles (scores of one row).
 * Returns the failed-segment bitmask as oracle_append does. */
int oracle_attend(const double *q, int q_heads, int total_rows,
                  const double *k_pool, const double *v_pool,
                  int64_t num_blocks, int kv_heads, int head_dim,
                  const int32_t *block_table, int max_seqs, int max_blocks_per_seq,
                  int ring_rows, const int32_t *seq_info, int num_segments,
                  double scale, int causal, int window, const int32_t *first_valid,
                  double *out, double *lse, double *work)
{
    oracle_pool P = {num_blocks, kv_heads, head_dim, block_table, max_seqs,
                     max_blocks_per_seq, ring_rows};
    const int group = q_heads / kv_heads;
    const int D = head_dim;
    int errs = 0;

    /* Rows start at zero output and lse = -inf; only valid segments fill theirs. */
    for (int64_t e = 0; e < (int64_t)total_rows * q_heads * D; ++e) out[e] = 0.0;
    for (int64_t e = 0; e < (int64_t)total_rows * q_heads; ++e) lse[e] = -INFINITY;

    for (int s = 0; s < num_segments; ++s) {
        const int32_t *seg = seq_info + 4 * s;
        /* first valid position of the sequence (0 without left padding) */
        int64_t first = 0;
        if (first_valid && seg[2] >= 0 && seg[2] < max_seqs && first_valid[seg[2]] > 0) first = first_valid[seg[2]];
        int st = check_segment(&P, seg, total_rows, causal, window, first, 0);
        if (st) { errs |= 1 << st; continue; }
        int64_t q0 = seg[0], ql = seg[1], col = seg[2], kend = seg[3];
        for (int64_t i = 0; i < ql; ++i) {
            int64_t t = q0 + i;
            int64_t lo, hi;
            key_range(kend, ql, i, causal, window, first, &lo, &hi);
            for (int h = 0; h < q_heads; ++h) {
                int g = h / group;
                const double *qv = q + (t * q_heads + h) * D;
                double *o = out + (t * q_heads + h) * D;
                if (hi <= lo) continue;   /* nothing visible: stays 0 / -inf */
                /* scores x_j = scale * <q, k_j> and their maximum */
                double m = -INFINITY;
                for (int64_t j = lo; j < hi; ++j) {
                    int64_t b; int off;
                    locate(&P, (int)col, j, &b, &off);
                    const double *kv = k_pool + ((b * ORACLE_BLOCK + off) * kv_heads + g) * D;
                    double x = 0.0;
                    for (int d = 0; d < D; ++d) x += qv[d] * kv[d];
                    x *= scale;
                    work[j - lo] = x;
                    if (x > m) m = x;
                }
                /* softmax weights and the weighted sum of V */
                double sum = 0.0;
                for (int64_t j = lo; j < hi; ++j) {
                    int64_t b; int off;
                    locate(&P, (int)col, j, &b, &off);
                    const double *vv = v_pool + ((b * ORACLE_BLOCK + off) * kv_heads + g) * D;
                    double w = exp(work[j - lo] - m);
                    sum += w;
                    for (int d = 0; d < D; ++d) o[d] += w * vv[d];
                }
                for (int d = 0; d < D; ++d) o[d] /= sum;
                lse[t * q_heads + h] = m + log(sum);
            }
        }
    }
    return errs;
}

/* seq_clone: positions 0 .. n-1 of sequence src_col are copied bit for bit to
 * the same positions of dst_col (one layer's pools).  With ring storage of R
 * rows only the last min(n, R) positions exist and are copied.  All or
 * nothing: if any slot either side needs maps outside the table or the pool,
 * nothing is written.  Returns 0 or 1 << status. */
int oracle_seq_clone(uint8_t *k_pool, uint8_t *v_pool, int elem_size,
                     int64_t num_blocks, int kv_heads, int head_dim,
                     const int32_t *block_table, int max_seqs, int max_blocks_per_seq,
                     int ring_rows, int src_col, int dst_col, int64_t n)
{
    oracle_pool P = {num_blocks, kv_heads, head_dim, block_table, max_seqs,
                     max_blocks_per_seq, ring_rows};
    if (src_col < 0 || src_col >= max_seqs || dst_col < 0 || dst_col >= max_seqs || n < 0)
        return 1 << OR_BAD_SEGMENT;
    if (!ring_rows && n > (int64_t)max_blocks_per_seq * ORACLE_BLOCK) return 1 << OR_CAPACITY;
    int64_t lo = (ring_rows && n > ring_rows) ? n - ring_rows : 0;
    for (int64_t p = lo; p < n; ++p) {
        int64_t b; int o;
        int st = locate(&P, src_col, p, &b, &o);
        if (!st) st = locate(&P, dst_col, p, &b, &o);
        if (st) return 1 << st;
    }
    int64_t row_bytes = (int64_t)kv_heads * head_dim * elem_size;
    for (int64_t p = lo; p < n; ++p) {
        int64_t bs, bd; int os, od;
        locate(&P, src_col, p, &bs, &os);
        locate(&P, dst_col, p, &bd, &od);
        memmove(k_pool + (bd * ORACLE_BLOCK + od) * row_bytes, k_pool + (bs * ORACLE_BLOCK + os) * row_bytes,
                (size_t)row_bytes);
        memmove(v_pool + (bd * ORACLE_BLOCK + od) * row_bytes, v_pool + (bs * ORACLE_BLOCK + os) * row_bytes,
                (size_t)row_bytes);
    }
    return 0;
}

/* rewind: segment s moves back amount[s] positions (kv_end -= amount[s]),
 * e.g. draft tokens a verify step rejected.  Allowed when
 * 0 <= amount <= kv_end and, with ring storage of R rows and window W, when
 * amount <= R - W + 1: the positions the next window reads (from the new
 * kv_end - W + 1 on) must still be held by the ring, which keeps the last R.
 * A segment that breaks a rule keeps its kv_end.  Returns a bitmask of
 * (1 << status) over such segments. */
int oracle_rewind(int32_t *seq_info, int num_segments, const int32_t *amount, int ring_rows, int window)
{
    int errs = 0;
    for (int s = 0; s < num_segments; ++s) {
        int64_t kend = seq_info[4 * s + 3], a = amount[s];
        if (a < 0 || a > kend) { errs |= 1 << OR_BAD_SEGMENT; continue; }
        if (ring_rows && (window <= 0 || a > (int64_t)ring_rows - window + 1)) { errs |= 1 << OR_RING; continue; }
        seq_info[4 * s + 3] = (int32_t)(kend - a);
    }
    return errs;
}
