// Append, copy and segment-table kernels.
#pragma once

#include "common.cuh"

namespace pkv {

// Append this step's K/V rows (vLLM-Omni SenseNova-U1 PagedDecodeCache.attend:
// the new token goes to slot length - 1 because the caller has already
// advanced the length; ExecuTorch #24074: the in-graph write lands at
// position % rows for ring storage).  One CTA per segment; a segment is
// written only if every slot it writes is valid.
static __global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendParams p) {
    const int s = blockIdx.x;
    const Segment sg = load_segment(p.seq_info, s);
    unsigned fault = segment_fault(sg, p.total_rows, p.max_seqs, p.mbps, p.ring_rows, p.window);
    const int *bt_row = p.block_table + (long long)(fault ? 0 : sg.col) * p.mbps;
    const long long new_start = (long long)sg.kend - sg.ql;
    bool ok = true;
    if (!fault) {
        for (int i = threadIdx.x; i < sg.ql; i += blockDim.x) {
            const long long pos = new_start + i;
            const long long rr = p.ring_rows ? pos % p.ring_rows : pos;
            const int b = bt_row[rr / kPage];
            ok &= b >= 0 && (long long)b < p.num_blocks;
        }
    }
    ok = __syncthreads_and(ok);
    if (!fault && !ok) fault = PKV_ERR_BLOCK;
    if (fault) {
        if (threadIdx.x == 0) atomicOr(p.err, fault);
        return;
    }
    const int chunks = p.row_bytes / 16;
    const long long total = (long long)sg.ql * chunks;
    for (long long c = threadIdx.x; c < 2 * total; c += blockDim.x) {
        const int kv = c >= total;
        const long long rem = c - kv * total;
        const long long i = rem / chunks;
        const int ch = (int)(rem - i * chunks);
        const long long pos = new_start + i;
        const long long rr = p.ring_rows ? pos % p.ring_rows : pos;
        const long long b = bt_row[rr / kPage];
        const char *src = reinterpret_cast<const char *>(kv ? p.v_new : p.k_new) +
                          ((long long)sg.q0 + i) * p.row_bytes + ch * 16;
        char *dst = reinterpret_cast<char *>(kv ? p.v_pool : p.k_pool) +
                    (b * kPage + rr % kPage) * p.row_bytes + ch * 16;
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
    }
}

// Copy n x H rows of `row_bytes` between two strided layouts, for two tensor
// pairs at once (K and V).  Strides are in bytes and multiples of 16.
struct CopyParams {
    const char *src0, *src1;
    char *dst0, *dst1;
    long long n;
    int H, row_chunks;
    long long src_s, src_h, dst_s, dst_h;
};

static __global__ void __launch_bounds__(256) strided_copy_kernel(const __grid_constant__ CopyParams p) {
    const long long total = p.n * p.H * p.row_chunks;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < 2 * total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int which = idx >= total;
        const long long e = idx - which * total;
        const long long row = e / p.row_chunks;
        const int ch = (int)(e - row * p.row_chunks);
        const long long s = row / p.H;
        const int h = (int)(row - s * p.H);
        const char *src = (which ? p.src1 : p.src0) + s * p.src_s + h * p.src_h + ch * 16;
        char *dst = (which ? p.dst1 : p.dst0) + s * p.dst_s + h * p.dst_h + ch * 16;
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
    }
}

// seq_info[s] = (cu[s], cu[s+1] - cu[s], s, seqused[s]): the flash-attention
// argument form used by PagedDecodeCache.attend, as a segment table.
static __global__ void seqinfo_from_seqused_kernel(const int *cu, const int *used, int n, int4 *out) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s < n) out[s] = make_int4(cu[s], cu[s + 1] - cu[s], s, used[s]);
}

// kv_end += q_len for every segment: the device half of a decode step's
// length advance (tiny-llm kv_cache.py, SlotKVCache.end_step).
static __global__ void advance_kernel(int4 *seq_info, int n) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s < n) {
        int4 v = seq_info[s];
        v.w += v.y;
        seq_info[s] = v;
    }
}

// ---------------------------------------------------------------- batched-sequence cache operations

// seq_clone of ExecuTorch #24073 (CudaBatchedSequenceCache: a device copy of
// the source prefix) over the paged layout: positions lo .. n-1 of sequence
// `src` are copied row by row (all kv heads) to the same positions of `dst`,
// each side mapped through its block-table row (ring: position % rows), in
// up to kCloneLayers layers per launch.  Every CTA first checks every page
// either side touches, so the copy is all or nothing; a bad page id sets
// PKV_ERR_BLOCK.
constexpr int kCloneLayers = 64;
struct CloneParams {
    char *k[kCloneLayers];      // the layers' pools (read and written)
    char *v[kCloneLayers];
    int layers;
    const int *block_table;
    unsigned *err;
    long long num_blocks;
    long long lo, n;            // positions lo .. n-1
    int row_chunks;             // 16-byte chunks per token row (Hkv * D * elem / 16)
    int mbps, ring_rows, src, dst;
};

static __global__ void __launch_bounds__(256) seq_clone_kernel(const __grid_constant__ CloneParams p) {
    const int *bs = p.block_table + (long long)p.src * p.mbps;
    const int *bd = p.block_table + (long long)p.dst * p.mbps;
    const long long pb0 = p.lo / kPage, pb1 = (p.n + kPage - 1) / kPage;
    bool ok = true;
    for (long long pb = pb0 + threadIdx.x; pb < pb1; pb += blockDim.x) {
        const int tp = table_page((int)pb, p.ring_rows);
        const int a = bs[tp], b = bd[tp];
        ok &= a >= 0 && (long long)a < p.num_blocks && b >= 0 && (long long)b < p.num_blocks;
    }
    if (!__syncthreads_and(ok)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, PKV_ERR_BLOCK);
        return;
    }
    // work items: (position, layer, K or V) rows, each row_chunks 16-byte chunks
    const long long rows = p.n - p.lo, per_pos = 2LL * p.layers * p.row_chunks;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < rows * per_pos; c += stride) {
        const long long i = c / per_pos;
        const int rem = (int)(c - i * per_pos);
        const int t = rem / p.row_chunks, ch = rem - t * p.row_chunks;  // t = 2 * layer + (V ? 1 : 0)
        const long long pos = p.lo + i;
        const long long r = p.ring_rows ? pos % p.ring_rows : pos;
        const int tp = table_page((int)(pos / kPage), p.ring_rows);
        const long long s_slot = (long long)bs[tp] * kPage + r % kPage;
        const long long d_slot = (long long)bd[tp] * kPage + r % kPage;
        uint4 *base = reinterpret_cast<uint4 *>((t & 1) ? p.v[t >> 1] : p.k[t >> 1]);
        base[d_slot * p.row_chunks + ch] = base[s_slot * p.row_chunks + ch];
    }
}

// rewind of ExecuTorch #24073 (bounded by the ring floor): kv_end -= amount
// per segment when 0 <= amount <= kv_end and, with ring storage of R rows
// and window W, amount <= R - W + 1 (the next window's keys are still in the
// ring).  A segment that breaks a rule keeps its kv_end and sets
// PKV_ERR_SEGMENT (amount out of range) or PKV_ERR_RING (ring floor).
static __global__ void rewind_kernel(int4 *seq_info, const int *amount, int n, int ring_rows, int window,
                                     unsigned *err) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= n) return;
    int4 v = seq_info[s];
    const int a = amount[s];
    if (a < 0 || a > v.w) {
        atomicOr(err, PKV_ERR_SEGMENT);
        return;
    }
    if (ring_rows && (window <= 0 || (long long)a > (long long)ring_rows - window + 1)) {
        atomicOr(err, PKV_ERR_RING);
        return;
    }
    v.w -= a;
    seq_info[s] = v;
}

}  // namespace pkv
