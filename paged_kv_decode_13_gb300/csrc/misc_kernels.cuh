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

}  // namespace pkv
