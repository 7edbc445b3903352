// Device helpers shared by the pkv kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kPage = PKV_BLOCK_SIZE;  // tokens per page

// ---------------------------------------------------------------- element types

template <typename T> struct Elem;
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    __device__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
};
template <> struct Elem<float> {
    static constexpr int kBytes = 4;
    __device__ static float to_f32(float x) { return x; }
};

// ---------------------------------------------------------------- shared memory, mbarriers, TMA

__device__ __forceinline__ unsigned smem_u32(const void *p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async proxy (TMA completion).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// One bounded-time probe of a barrier phase (the hardware may suspend the
// thread for a short while before returning false).
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// 4-D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1, int c2,
                                            int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

// 5-D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1, int c2,
                                            int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
        : "memory");
}

// Bring one 5-D tiled box into L2 without writing shared memory.
__device__ __forceinline__ void tma_prefetch_l2_5d(const CUtensorMap *map, int c0, int c1, int c2, int c3, int c4) {
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
                 : "memory");
}

// Bring `bytes` contiguous bytes (16-byte aligned, a multiple of 16) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

// Bring one 4-D tiled box into L2 without writing shared memory.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// Byte offset of 16-byte chunk `chunk` of row `row` inside a page tile
// loaded with 128-byte swizzling: the tile is a run of 2 KB boxes (16 rows x
// 128 B), and inside each 1 KB half the chunk index is XOR-ed with row % 8.
__device__ __forceinline__ unsigned swz(int row, int chunk) {
    return (unsigned)((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------- programmatic dependent launch

// Wait until the grid this launch depends on has completed and its writes are
// visible (a no-op when the launch did not use programmatic serialisation).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Allow the next grid on the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ---------------------------------------------------------------- tensor-core fragments

__device__ __forceinline__ void ldmatrix_x4(unsigned (&r)[4], const void *smem) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
__device__ __forceinline__ void ldmatrix_x4_trans(unsigned (&r)[4], const void *smem) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const unsigned (&a)[4], unsigned b0,
                                               unsigned b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&v);
}

// Named barrier over `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- launch parameters

struct Segment {
    int q0, ql, col, kend;
};

// Everything one attention launch reads; passed by value as a grid constant.
struct AttendParams {
    CUtensorMap tmap_k;     // 4-D view (D, Hkv, 16, num_blocks) of this layer's K pool
    CUtensorMap tmap_v;
    const void *q;          // [rows][Hq][D]
    const void *k_new;      // fused append: [rows][Hkv][D], else null
    const void *v_new;
    void *k_pool_w;         // fused append: the pools, written at this step's slots
    void *v_pool_w;
    const int *block_table; // [max_seqs][mbps]
    const int4 *seq_info;   // [S]
    const int *first_valid; // [max_seqs] first non-padding position, or null (no padding)
    float *out;             // [rows][Hq][D]
    float *lse;             // [rows][Hq] or null
    unsigned *err;
    long long num_blocks;
    int Hq, Hkv, D, G;      // G = Hq / Hkv
    int total_rows, S;
    int max_seqs, mbps, ring_rows;
    int max_q_len;
    int row_tiles;          // CTAs along the rows of one (segment, kv head)
    int causal, window;
    float scale_log2;       // softmax_scale * log2(e)
    // 1: the four maps are the 5-D page view (64, 16, D / 64, Hkv, num_blocks)
    // that brings one kv head's page tile in one box; 0: the 4-D view
    // (D, Hkv, 16, num_blocks) with 64-element boxes.
    int page_box;
    // Optional L2 warm-up of the next layer's pages of the same key ranges
    // (the next call reads the same table and segments): the next layer's
    // pools, and how many pages of each CTA's range to warm (0 = off).
    const void *k_next;
    const void *v_next;
    int pf_next;
    // Split-K merge through global memory instead of the cluster (decode
    // kernel with a workspace): per (segment, kv head) unit the partial rows,
    // their (max, sum), flags and an arrival counter; all null = cluster merge.
    float *ws_part;         // [units][ncta][8][DP]
    float2 *ws_stat;        // [units][ncta][8]
    int *ws_flag;           // [units][ncta]
    int *ws_count;          // [units], zero between calls
};

struct AppendParams {
    const void *k_new, *v_new;  // [rows][Hkv][D]
    void *k_pool, *v_pool;
    const int *block_table;
    const int4 *seq_info;
    unsigned *err;
    long long num_blocks;
    int row_bytes;              // Hkv * D * elem
    int total_rows, S, max_seqs, mbps, ring_rows, window;
};

// ---------------------------------------------------------------- segment rules

// Field and capacity checks shared by append and attention; returns PKV_ERR_* or 0.
__device__ __forceinline__ unsigned segment_fault(const Segment &s, int total_rows, int max_seqs,
                                                  int mbps, int ring_rows, int window) {
    if (s.q0 < 0 || s.ql < 0 || (long long)s.q0 + s.ql > total_rows) return PKV_ERR_SEGMENT;
    if (s.col < 0 || s.col >= max_seqs) return PKV_ERR_SEGMENT;
    if (s.kend < s.ql || s.kend > 0x7fffffff - 2 * kPage) return PKV_ERR_SEGMENT;
    if (ring_rows) {
        if (window <= 0 || (long long)window + s.ql - 1 > ring_rows) return PKV_ERR_RING;
    } else if ((long long)s.kend > (long long)mbps * kPage) {
        return PKV_ERR_CAPACITY;
    }
    return 0;
}

// Page index in the sequence's table row for logical position-block `pb`
// (positions pb*16 .. pb*16+15).  Ring rows are a multiple of 16, so a page
// of positions never straddles the wrap.
__device__ __forceinline__ int table_page(int pb, int ring_rows) {
    return ring_rows ? pb % (ring_rows >> 4) : pb;
}

__device__ __forceinline__ Segment load_segment(const int4 *seq_info, int s) {
    int4 v = seq_info[s];
    return Segment{v.x, v.y, v.z, v.w};
}

// ---------------------------------------------------------------- key ranges

// Left padding ([tiny-llm kv_cache.py] SlotKVCache, padded_causal_mask):
// keys before a sequence's first valid position are hidden from every row,
// and a row that is itself padding sees only its own key (the diagonal is
// always kept, so no row is fully masked).
__device__ __forceinline__ int first_valid_of(const int *first_valid, int col) {
    return first_valid ? max(first_valid[col], 0) : 0;
}

// Keys [lo, hi) of the row at position `pos` of a segment ending at kv_end:
// causal rows end at their own position, a window of W keeps the last W keys
// up to the row's newest key, padding as above.
__device__ __forceinline__ void row_key_bounds(int pos, int kend, int causal, int window, int first,
                                               int &lo, int &hi) {
    const int newest = causal ? pos : kend - 1;
    hi = causal ? pos + 1 : kend;
    lo = window > 0 ? max(0, newest - window + 1) : 0;
    if (pos < first) {
        lo = pos;
        hi = pos + 1;
    } else {
        lo = max(lo, first);
    }
}

// Lowest key any row of the segment reads.  Bounds are non-decreasing in
// the row's position, so it is the first row's: with padded rows that is
// the step's first position (a padded row reads its own key; the others
// start at `first`, which is past it).
__device__ __forceinline__ int segment_key_lo(int new_start, int kend, int causal, int window, int first) {
    int lo, hi;
    row_key_bounds(new_start, kend, causal, window, first, lo, hi);
    return lo;
}

}  // namespace pkv
