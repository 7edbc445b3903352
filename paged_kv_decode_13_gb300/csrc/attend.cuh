// Split-K decode attention over a paged KV cache (sm_103a).
//
// Grid (C, kv_heads x row tiles, segments); the C CTAs along x form one
// thread-block cluster and split one (segment, kv head) key range between
// them.  A CTA holds the query rows of one kv head's GQA group (G heads x
// q_len rows, zero-padded to 16-row tiles) and streams its K/V pages through
// shared memory: TMA (cp.async.bulk.tensor, 128-byte swizzle) brings one page
// of one kv head (16 tokens) per stage into a ring of stages tracked by
// mbarriers, one elected thread per ring issuing the copies.  Warps are MT row
// tiles x KW key groups; each key group owns a ring and takes every KW-th
// page, keeping its own online-softmax state.  At the end the key groups merge
// in shared memory and the C partial results merge across the cluster through
// distributed shared memory, each CTA producing a slice of the output.
//
// Semantics follow the segment-table attention of ExecuTorch PR #24072
// (triton::sdpa_varlen) over the (num_blocks, 16, kv_heads, head_dim) paged
// layout of vLLM-Omni's SenseNova-U1 PagedDecodeCache: causal rows are aligned
// to kv_end (tiny-llm kv_cache.py, causal_kwargs), the window ends at the
// row's own position, ring storage maps position p to slot p % ring_rows
// (ExecuTorch #24074), rows no segment covers read zero.
#pragma once

#include <cooperative_groups.h>
#include <math_constants.h>

#include "common.cuh"

namespace pkv {

// Bound on the probes of one barrier phase; past it the kernel records
// PKV_ERR_TIMEOUT, zeroes the affected output and carries on.
constexpr int kWaitProbes = 1 << 20;

template <typename T_, int DP_, int MT_, int KW_, int NST_, bool MMA_>
struct AttnCfg {
    using T = T_;
    static constexpr int DP = DP_;      // head_dim rounded up to 64 / 128 / 256
    static constexpr int MT = MT_;      // 16-row tiles per CTA
    static constexpr int KW = KW_;      // key groups (pages interleaved across them)
    static constexpr int NST = NST_;    // pipeline stages per key group
    static constexpr bool MMA = MMA_;
    static constexpr int kWarps = MT * KW;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kRows = MT * 16;
    static constexpr int kElem = (int)sizeof(T);
    static constexpr int kEpc = 16 / kElem;               // elements per 16-byte chunk
    static constexpr int kChunks = DP / kEpc;             // 16-byte chunks per row
    static constexpr int kBoxEl = 128 / kElem;            // elements per 128-byte swizzle box row
    static constexpr int kBoxes = DP / kBoxEl;            // boxes per page tile
    static constexpr unsigned kTileBytes = kPage * DP * kElem;  // one K or V page of one kv head
    static constexpr unsigned kStageBytes = 2 * kTileBytes;
    static constexpr int kQLd = MMA ? DP + 8 : DP + 4;    // padded query row (elements of T / fp32)
    static constexpr size_t kPipeBytes = (size_t)KW * NST * kStageBytes;
    static constexpr size_t kMergeBytes = (size_t)KW * kRows * DP * 4 + (size_t)2 * KW * kRows * 4;
    static constexpr size_t kBodyBytes =
        ((kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes) + 1023) & ~size_t(1023);
    static constexpr size_t kQBytes = MMA ? (size_t)kRows * kQLd * 2 : (size_t)kRows * kQLd * 4;
    // per row: pm, pl, lo, hi, lse, and the cluster merge's gathered maxima / sums (16 CTAs each)
    static constexpr size_t kRowBytes = (size_t)kRows * (2 + 2 + 1 + 16 + 16) * 4;
    static constexpr size_t kBarBytes = (size_t)KW * NST * 8;
    static constexpr size_t kSimtBytes = MMA ? 0 : (size_t)kWarps * (16 * 16 + 16) * 4;
    static constexpr size_t kFlagBytes = 32 * 4;  // this CTA's poison flags, then the cluster's
    static constexpr size_t kCovBytes = (size_t)kThreads * 4;  // coverage flags of the first rows
    static constexpr size_t kBaseBytes =
        1024 + kBodyBytes + kQBytes + kRowBytes + kBarBytes + kSimtBytes + kFlagBytes + kCovBytes + 16;
    // Partial outputs pushed by the other CTAs of the cluster (one slice each);
    // without room for it the merge pulls them instead.
    static constexpr size_t kRecvNeed = ((size_t)kRows * DP + 16) * 4;
    static constexpr bool kPush = kBaseBytes + kRecvNeed <= 232448;
    static constexpr size_t kSmemBytes = kBaseBytes + (kPush ? kRecvNeed : 0);
    // L2 warm-up before the dependency wait: each key group prefetches up to
    // kL2Pages pages past its stages, about 512 KB per SM over the CTAs that
    // fit on one (at most 32 pages: the page-id window of a warp).
    static constexpr int kCtasPerSm = (int)(232448 / (kSmemBytes + 1024)) > 0 ? (int)(232448 / (kSmemBytes + 1024)) : 1;
    static constexpr int kL2PagesRaw = (int)(524288 / ((size_t)kCtasPerSm * KW * kStageBytes));
    static constexpr int kL2Pages = kL2PagesRaw < 1 ? 1 : kL2PagesRaw > 32 - NST ? 32 - NST : kL2PagesRaw;
    static_assert(DP % kBoxEl == 0, "page rows are whole 128-byte boxes");
    static_assert(kQBytes % 16 == 0, "smem sections stay 16-byte aligned");
    static_assert(!MMA || sizeof(T) == 2, "tensor-core path is bf16");
    static_assert(kRows <= kThreads, "one thread per row in the cluster merge");
};

// ---------------------------------------------------------------- small vector loads

template <typename T, int N>
__device__ __forceinline__ void load_f32(float (&o)[N], const T *src);

template <>
__device__ __forceinline__ void load_f32<float, 2>(float (&o)[2], const float *s) {
    float2 v = *reinterpret_cast<const float2 *>(s);
    o[0] = v.x; o[1] = v.y;
}
template <>
__device__ __forceinline__ void load_f32<float, 4>(float (&o)[4], const float *s) {
    float4 v = *reinterpret_cast<const float4 *>(s);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void bf2_to_f32(float *o, unsigned u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    float2 f = __bfloat1622float2(v);
    o[0] = f.x; o[1] = f.y;
}
template <>
__device__ __forceinline__ void load_f32<__nv_bfloat16, 2>(float (&o)[2], const __nv_bfloat16 *s) {
    bf2_to_f32(o, *reinterpret_cast<const unsigned *>(s));
}
template <>
__device__ __forceinline__ void load_f32<__nv_bfloat16, 4>(float (&o)[4], const __nv_bfloat16 *s) {
    uint2 v = *reinterpret_cast<const uint2 *>(s);
    bf2_to_f32(o, v.x); bf2_to_f32(o + 2, v.y);
}
template <>
__device__ __forceinline__ void load_f32<__nv_bfloat16, 8>(float (&o)[8], const __nv_bfloat16 *s) {
    uint4 v = *reinterpret_cast<const uint4 *>(s);
    bf2_to_f32(o, v.x); bf2_to_f32(o + 2, v.y); bf2_to_f32(o + 4, v.z); bf2_to_f32(o + 6, v.w);
}

// N consecutive elements starting at element `col` of row `row` in a
// swizzled page tile, widened to fp32 (N * sizeof(T) <= 16 and aligned).
template <typename T, int N>
__device__ __forceinline__ void tile_load(float (&o)[N], const unsigned char *tile, int row, int col) {
    constexpr int kEpc = 16 / (int)sizeof(T);
    const int chunk = col / kEpc, within = col - chunk * kEpc;
    load_f32<T, N>(o, reinterpret_cast<const T *>(tile + swz(row, chunk)) + within);
}

// ---------------------------------------------------------------- per-warp compute states

// Tensor-core state of one warp: a 16-row tile, fp32 accumulators in the
// mma.m16n8k16 C layout (thread holds rows lane/4 and lane/4 + 8).
template <class C>
struct MmaWarp {
    static constexpr int DP = C::DP, LD = C::kQLd;
    float m[2], l[2];
    float acc[DP / 8][4];
    unsigned qf[DP <= 128 ? DP / 16 : 1][4];

    __device__ void init(const __nv_bfloat16 *sQ, int mt, int lane) {
        m[0] = m[1] = -CUDART_INF_F;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int n = 0; n < DP / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        if constexpr (DP <= 128) {
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk)
                ldmatrix_x4(qf[kk], sQ + (mt * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
        }
    }

    // NP pages (16 keys each) in one pass: their Q.K^T and P.V products are
    // independent MMA chains, so two pages cost little more latency than one.
    template <int NP>
    __device__ void consume(const __nv_bfloat16 *sQ, const unsigned char *const *sK,
                            const unsigned char *const *sV, const int *pos0, const int *sLo, const int *sHi,
                            int mt, int lane, float scale_log2) {
        constexpr int NT = 2 * NP;  // 8-key column tiles of S
        float sc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        const int krow = (lane & 7) + ((lane >> 4) << 3);
        const int kchk = (lane >> 3) & 1;
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
            unsigned a[4];
            if constexpr (DP <= 128) {
                a[0] = qf[kk][0]; a[1] = qf[kk][1]; a[2] = qf[kk][2]; a[3] = qf[kk][3];
            } else {
                ldmatrix_x4(a, sQ + (mt * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
            }
#pragma unroll
            for (int pg = 0; pg < NP; ++pg) {
                unsigned b[4];
                ldmatrix_x4(b, sK[pg] + swz(krow, 2 * kk + kchk));
                mma_bf16_16816(sc[2 * pg], a, b[0], b[1]);
                mma_bf16_16816(sc[2 * pg + 1], a, b[2], b[3]);
            }
        }
        // Mask, online softmax (base 2).
        const int t4 = lane & 3;
        float mx[2], alpha[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = mt * 16 + (lane >> 2) + 8 * e;
            const int lo = sLo[r], hi = sHi[r];
            float best = -CUDART_INF_F;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int pos = pos0[n >> 1] + (n & 1) * 8 + 2 * t4 + c;
                    float v = sc[n][2 * e + c] * scale_log2;
                    v = (pos >= lo && pos < hi) ? v : -CUDART_INF_F;
                    sc[n][2 * e + c] = v;
                    best = fmaxf(best, v);
                }
            best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 1));
            best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 2));
            const float mnew = fmaxf(m[e], best);
            const float muse = mnew == -CUDART_INF_F ? 0.f : mnew;
            alpha[e] = exp2f(m[e] - muse);
            m[e] = mnew;
            mx[e] = muse;
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float pr = exp2f(sc[n][c] - mx[c >> 1]);
                sc[n][c] = pr;
                rs[c >> 1] += pr;
            }
        l[0] = l[0] * alpha[0] + rs[0];
        l[1] = l[1] * alpha[1] + rs[1];
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int n = 0; n < DP / 8; ++n) {
                acc[n][0] *= alpha[0]; acc[n][1] *= alpha[0];
                acc[n][2] *= alpha[1]; acc[n][3] *= alpha[1];
            }
        }
        // P (bf16, A layout straight from the S accumulators) times V.
        unsigned pa[NP][4];
#pragma unroll
        for (int pg = 0; pg < NP; ++pg) {
            pa[pg][0] = pack_bf16x2(sc[2 * pg][0], sc[2 * pg][1]);
            pa[pg][1] = pack_bf16x2(sc[2 * pg][2], sc[2 * pg][3]);
            pa[pg][2] = pack_bf16x2(sc[2 * pg + 1][0], sc[2 * pg + 1][1]);
            pa[pg][3] = pack_bf16x2(sc[2 * pg + 1][2], sc[2 * pg + 1][3]);
        }
        const int vrow = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int vchk = lane >> 4;
#pragma unroll
        for (int dn = 0; dn < DP / 16; ++dn) {
#pragma unroll
            for (int pg = 0; pg < NP; ++pg) {
                unsigned b[4];
                ldmatrix_x4_trans(b, sV[pg] + swz(vrow, 2 * dn + vchk));
                mma_bf16_16816(acc[2 * dn], pa[pg], b[0], b[1]);
                mma_bf16_16816(acc[2 * dn + 1], pa[pg], b[2], b[3]);
            }
        }
    }

    __device__ void store(float *sMo, float *sMm, float *sMl, int kw, int mt, int lane) {
        constexpr int R = C::kRows;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float ls = l[e];
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            const int r = mt * 16 + (lane >> 2) + 8 * e;
            if ((lane & 3) == 0) {
                sMm[kw * R + r] = m[e];
                sMl[kw * R + r] = ls;
            }
            float *row = sMo + ((size_t)kw * R + r) * DP;
#pragma unroll
            for (int n = 0; n < DP / 8; ++n) {
                *reinterpret_cast<float2 *>(row + n * 8 + 2 * (lane & 3)) =
                    make_float2(acc[n][2 * e], acc[n][2 * e + 1]);
            }
        }
    }
};

// CUDA-core state of one warp: 16 rows; for QK^T lane = key (lane % 16) x
// half of head_dim (lane / 16); for PV lane = head_dim / 32 columns.
template <class C>
struct SimtWarp {
    using T = typename C::T;
    static constexpr int DP = C::DP, EPC = C::kEpc, DPL = DP / 32;
    static constexpr int HCH = C::kChunks / 2;   // chunks per half row
    static constexpr int VL = DPL * C::kElem > 16 ? 16 / C::kElem : DPL;  // elements per V load
    float m[16], l[16];
    float acc[16][DPL];

    __device__ void init() {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            m[r] = -CUDART_INF_F;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[r][e] = 0.f;
        }
    }

    __device__ void consume(const float *sQf, const unsigned char *sK, const unsigned char *sV, long long pos0,
                            const int *sLo, const int *sHi, int mt, int lane, int nrw, float scale_log2,
                            float *sPw) {
        const int kq = lane & 15, hf = lane >> 4;
        float dot[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) dot[r] = 0.f;
#pragma unroll
        for (int c = 0; c < HCH; ++c) {
            const int col = (hf * HCH + c) * EPC;
            float kf[EPC];
            tile_load<T, EPC>(kf, sK, kq, col);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                if (r < nrw) {
                    const float *qr = sQf + (mt * 16 + r) * C::kQLd + col;
#pragma unroll
                    for (int e = 0; e < EPC; e += 4) {
                        float4 qv = *reinterpret_cast<const float4 *>(qr + e);
                        dot[r] = fmaf(qv.x, kf[e], dot[r]);
                        dot[r] = fmaf(qv.y, kf[e + 1], dot[r]);
                        dot[r] = fmaf(qv.z, kf[e + 2], dot[r]);
                        dot[r] = fmaf(qv.w, kf[e + 3], dot[r]);
                    }
                }
            }
        }
        const long long pos = pos0 + kq;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            if (r < nrw) {
                float d = dot[r] + __shfl_xor_sync(0xffffffffu, dot[r], 16);
                const int rr = mt * 16 + r;
                float sv = (pos >= sLo[rr] && pos < sHi[rr]) ? d * scale_log2 : -CUDART_INF_F;
                float best = sv;
                best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 1));
                best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 2));
                best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 4));
                best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 8));
                const float mnew = fmaxf(m[r], best);
                const float muse = mnew == -CUDART_INF_F ? 0.f : mnew;
                const float alpha = exp2f(m[r] - muse);
                const float pr = exp2f(sv - muse);
                m[r] = mnew;
                l[r] = l[r] * alpha + pr;
                if (hf == 0) sPw[r * 16 + kq] = pr;
                if (lane == 0) sPw[256 + r] = alpha;
            }
        }
        __syncwarp();
        const int d0 = lane * DPL;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            if (r < nrw) {
                const float a = sPw[256 + r];
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[r][e] *= a;
            }
        }
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
            float vf[DPL];
#pragma unroll
            for (int part = 0; part < DPL / VL; ++part) {
                float tmp[VL];
                tile_load<T, VL>(tmp, sV, k, d0 + part * VL);
#pragma unroll
                for (int e = 0; e < VL; ++e) vf[part * VL + e] = tmp[e];
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                if (r < nrw) {
                    const float pr = sPw[r * 16 + k];
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[r][e] = fmaf(pr, vf[e], acc[r][e]);
                }
            }
        }
        __syncwarp();
    }

    __device__ void store(float *sMo, float *sMm, float *sMl, int kw, int mt, int lane, int nrw) {
        constexpr int R = C::kRows;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float ls = l[r];
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            ls += __shfl_xor_sync(0xffffffffu, ls, 4);
            ls += __shfl_xor_sync(0xffffffffu, ls, 8);
            const int rr = mt * 16 + r;
            if (lane == 0) {
                sMm[kw * R + rr] = r < nrw ? m[r] : -CUDART_INF_F;
                sMl[kw * R + rr] = r < nrw ? ls : 0.f;
            }
            float *row = sMo + ((size_t)kw * R + rr) * DP + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) row[e] = r < nrw ? acc[r][e] : 0.f;
        }
    }
};

// ---------------------------------------------------------------- rows no segment covers

// Output rows are checked in slices of one CTA's thread count: slice k
// belongs to the CTA of linear index k (and k + grid size, k + 2 * grid
// size, ...), so the work spreads over the grid.  Segments with a negative
// q_start or non-positive q_len cover nothing.
__device__ __forceinline__ long long grid_cta_index() {
    return (long long)blockIdx.x + (long long)gridDim.x * ((long long)blockIdx.y + (long long)gridDim.y * blockIdx.z);
}
__device__ __forceinline__ long long grid_cta_count() {
    return (long long)gridDim.x * gridDim.y * gridDim.z;
}
__device__ __forceinline__ int coverage_slices(const AttendParams &p, int nthreads) {
    return (p.total_rows + nthreads - 1) / nthreads;
}

// Count, for each row of the slice starting at `base`, the segments that
// cover it: the threads take the segments in turn (one segment table read
// per thread and pass, whatever the row count) and add one per covered row
// of the slice in shared memory.  Leaves sCov[t] = 1 (no segment) | 2 (more
// than one) for row base + t and returns whether any flag is set.  Every
// thread of the CTA calls it.
static __device__ __noinline__ int coverage_scan(const AttendParams &p, int *sCov, int base, int nthreads) {
    const int tid = threadIdx.x;
    sCov[tid] = 0;
    __syncthreads();
    const long long hi_row = min((long long)base + nthreads, (long long)p.total_rows);
    #pragma unroll 1
    for (int s = tid; s < p.S; s += nthreads) {
        const Segment g = load_segment(p.seq_info, s);
        if (g.q0 < 0 || g.ql <= 0) continue;
        const long long a = max((long long)g.q0, (long long)base);
        const long long b = min((long long)g.q0 + g.ql, hi_row);
        #pragma unroll 1
        for (long long r = a; r < b; ++r) atomicAdd(sCov + (r - base), 1);
    }
    __syncthreads();
    const int cnt = sCov[tid];
    const int f = (long long)base + tid < hi_row ? ((cnt == 0 ? 1 : 0) | (cnt > 1 ? 2 : 0)) : 0;
    __syncthreads();
    sCov[tid] = f;
    return __syncthreads_or(f != 0);
}

// After the dependency wait: zero the rows of the slice at `base` that no
// segment covers (out = 0, lse = -inf) and report rows two segments claim.
static __device__ __noinline__ void coverage_fix(const AttendParams &p, const int *sCov, int base, int nthreads) {
    const int tid = threadIdx.x;
    const int n = min(nthreads, p.total_rows - base), per_row = p.Hq * p.D;
    if (tid < n && (sCov[tid] & 2)) atomicOr(p.err, PKV_ERR_OVERLAP);
    #pragma unroll 1
    for (int r = 0; r < n; ++r) {
        if (!(sCov[r] & 1)) continue;
        const long long t = (long long)base + r;
        #pragma unroll 1
        for (int e = tid; e < per_row; e += nthreads) p.out[t * per_row + e] = 0.f;
        if (p.lse)
            #pragma unroll 1
            for (int e = tid; e < p.Hq; e += nthreads) p.lse[t * p.Hq + e] = -CUDART_INF_F;
    }
}

// Before the dependency wait (the segment table is not written by the
// previous kernel): a CTA that owns a slice scans its first one.  Returns
// whether that slice needs fixing.
static __device__ __forceinline__ int coverage_begin(const AttendParams &p, int *sCov, bool cov_cta, int nthreads) {
    return cov_cta ? coverage_scan(p, sCov, (int)(grid_cta_index() * nthreads), nthreads) : 0;
}

// After the dependency wait, every thread of a CTA that owns a slice: fix
// the first slice, then scan and fix any further ones (grids with fewer CTAs
// than slices).
static __device__ __noinline__ void apply_coverage(const AttendParams &p, int *sCov, int cov_any, int nthreads) {
    const long long lin = grid_cta_index(), nct = grid_cta_count();
    const int slices = coverage_slices(p, nthreads);
    if (lin >= slices) return;
    if (cov_any) coverage_fix(p, sCov, (int)(lin * nthreads), nthreads);
    #pragma unroll 1
    for (long long k = lin + nct; k < slices; k += nct) {
        const int base = (int)(k * nthreads);
        __syncthreads();  // the previous slice's flags are no longer read
        if (coverage_scan(p, sCov, base, nthreads)) coverage_fix(p, sCov, base, nthreads);
    }
}

// Zero the rows of kv head g's group for a segment that failed validation.
static __device__ __noinline__ void zero_segment_rows(const AttendParams &p, const Segment &sg, int g, int nthreads) {
    if (sg.ql <= 0) return;
    const long long a = max(sg.q0, 0);
    const long long b = min((long long)sg.q0 + sg.ql, (long long)p.total_rows);
    const int per = p.G * p.D;
    #pragma unroll 1
    for (long long t = a; t < b; ++t) {
        float *o = p.out + (t * p.Hq + (long long)g * p.G) * p.D;
        #pragma unroll 1
        for (int e = threadIdx.x; e < per; e += nthreads) o[e] = 0.f;
        if (p.lse)
            #pragma unroll 1
            for (int e = threadIdx.x; e < p.G; e += nthreads) p.lse[t * p.Hq + g * p.G + e] = -CUDART_INF_F;
    }
}

// First CTA, after the dependency wait: zero the rows the pre-wait scan found
// uncovered among the first `nthreads` rows, flag double coverage, then scan
// and zero any rows past them.
// ---------------------------------------------------------------- merge of a CTA's partial rows

// Merge the key groups' partial rows of this CTA (sMo [KW][R][DP] fp32,
// base-2 (max, sum) in sMm / sMl [KW][R]) and, across the cluster of ncta
// CTAs that split the key range, the CTAs' partials; write out / lse for the
// rows_here rows starting at row0 of the (segment, kv head) group.  In push
// mode each CTA hands every element to the CTA that finishes it (the caller
// arrived on the cluster barrier at the start); in pull mode each CTA reads
// its slice from its peers.  A poisoned CTA (flags) zeroes the rows.  Every
// thread of the CTA calls it.
template <int DP, int KW, int R, int NT, bool kPush>
static __device__ __forceinline__ void merge_rows(const AttendParams &p, const Segment &sg, int g, int row0,
                                                  int rows_here, int flags, int rank, int ncta, float *sMo,
                                                  float *sMm, float *sMl, float *sPm, float *sPl, float *sLse,
                                                  float *sAllM, float *sAllL, int *sAllF, int *sFlag,
                                                  float *sRecv) {
    namespace cg = cooperative_groups;
    const int tid = threadIdx.x;
    constexpr float kLn2 = 0.6931471805599453f;
    auto out_row = [&](int r) {
        const int ur = row0 + r, i = ur / p.G, jh = ur - i * p.G;
        return ((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh;
    };
    cg::cluster_group cluster = cg::this_cluster();
    const int E = rows_here * DP;
    const int per = (E + ncta - 1) / ncta;  // output elements each CTA of the cluster finishes
    // Row statistics of the key-group merge, one thread per row: the max and
    // sum, and each key group's weight 2^(m_k - M), left in sMm for the
    // element pass.  A CTA alone in its cluster also keeps 1/L and the lse.
    if (tid < rows_here) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < KW; ++k) M = fmaxf(M, sMm[k * R + tid]);
        float L = 0.f;
#pragma unroll
        for (int k = 0; k < KW; ++k) {
            const float w = M == -CUDART_INF_F ? 0.f : exp2f(sMm[k * R + tid] - M);
            L = fmaf(w, sMl[k * R + tid], L);
            sMm[k * R + tid] = w;
        }
        sPm[tid] = M;
        if (ncta == 1) {
            const bool zero = flags || L <= 0.f;
            sPl[tid] = zero ? 0.f : 1.f / L;
            sLse[tid] = zero ? -CUDART_INF_F : (M + log2f(L)) * kLn2;
        } else {
            sPl[tid] = L;
        }
    }
    __syncthreads();
    // Owner of output element idx in the cluster: idx / per without an
    // integer division in the loop.
    const float inv_per = 1.f / (float)per;
    auto owner = [&](int idx) {
        int k = __float2int_rz((float)idx * inv_per);
        k -= k * per > idx;
        k += (k + 1) * per <= idx;
        return k;
    };
    if (kPush && ncta > 1) {
        // Every CTA of the cluster has started (the arrive at the top), so
        // peers' shared memory may be written from here on.
        asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
        if (tid < ncta) *cluster.map_shared_rank(sAllF + rank, tid) = flags;
#pragma unroll 1
        for (int idx = tid; idx < rows_here * ncta; idx += NT) {
            const int r = idx / ncta, c = idx - r * ncta;
            *cluster.map_shared_rank(sAllM + r * 16 + rank, c) = sPm[r];
            *cluster.map_shared_rank(sAllL + r * 16 + rank, c) = sPl[r];
        }
    }
    // Merge the key groups element by element; finish each element here when
    // the CTA is alone, otherwise hand it to the CTA that finishes it.
#pragma unroll 4
    for (int idx = tid; idx < E; idx += NT) {
        const int r = idx / DP, d = idx - r * DP;
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < KW; ++k) {
            // a key group with no visible key has weight 0 and a zero accumulator
            o = fmaf(sMm[k * R + r], sMo[((size_t)k * R + r) * DP + d], o);
        }
        if (ncta == 1) {
            const long long orow = out_row(r);
            if (d < p.D) p.out[orow * p.D + d] = flags ? 0.f : o * sPl[r];
            if (d == 0 && p.lse) p.lse[orow] = sLse[r];
        } else if constexpr (kPush) {
            const int k = owner(idx);
            *cluster.map_shared_rank(sRecv + rank * per + (idx - k * per), k) = o;
        } else {
            sMo[(size_t)r * DP + d] = o;  // element owned by this thread alone: merged in place
        }
    }
    if (ncta == 1) return;

    // ---- merge the cluster's partials (distributed shared memory)
    if constexpr (kPush) {
        cluster.sync();  // publishes every CTA's pushed partials
    } else {
        cluster.sync();
#pragma unroll 1
        for (int idx = tid; idx < rows_here * ncta; idx += NT) {
            const int r = idx / ncta, c = idx - r * ncta;
            sAllM[r * 16 + c] = *cluster.map_shared_rank(sPm + r, c);
            sAllL[r * 16 + c] = *cluster.map_shared_rank(sPl + r, c);
        }
        if (tid < ncta) sAllF[tid] = *cluster.map_shared_rank(sFlag, tid);
        __syncthreads();
    }
    int poison = 0;
#pragma unroll
    for (int c = 0; c < 16; ++c) poison |= c < ncta ? sAllF[c] : 0;
    const int e0 = rank * per, e1 = min(E, e0 + per);
#pragma unroll 1
    for (int idx = e0 + tid; idx < e1; idx += NT) {
        const int r = idx / DP, d = idx - r * DP;
        float m[16], l[16], v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            m[c] = c < ncta ? sAllM[r * 16 + c] : -CUDART_INF_F;
            l[c] = c < ncta ? sAllL[r * 16 + c] : 0.f;
            if constexpr (kPush)
                v[c] = c < ncta ? sRecv[c * per + (idx - e0)] : 0.f;
            else
                v[c] = c < ncta ? *cluster.map_shared_rank(sMo + (size_t)r * DP + d, c) : 0.f;
        }
        float M = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 16; ++c) M = fmaxf(M, m[c]);
        float W = 0.f, o = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            // A zero weight must not touch its partial: a poisoned one may hold NaN.
            const float w = (M == -CUDART_INF_F || m[c] == -CUDART_INF_F) ? 0.f : exp2f(m[c] - M);
            W = fmaf(w, l[c], W);
            o += w != 0.f ? w * v[c] : 0.f;
        }
        const bool zero = poison || W <= 0.f;
        const long long orow = out_row(r);
        if (d < p.D) p.out[orow * p.D + d] = zero ? 0.f : o / W;
        if (d == 0 && p.lse) p.lse[orow] = zero ? -CUDART_INF_F : (M + log2f(W)) * kLn2;
    }
    if constexpr (!kPush) cluster.sync();  // partials stay readable until every CTA has merged its slice
}

// ---------------------------------------------------------------- the kernel

template <class C>
__global__ void __launch_bounds__(C::kThreads) attend_kernel(const __grid_constant__ AttendParams p) {
    using T = typename C::T;
    namespace cg = cooperative_groups;
    constexpr int DP = C::DP, MT = C::MT, KW = C::KW, NST = C::NST;
    constexpr int EPC = C::kEpc, R = C::kRows, NT = C::kThreads;
    constexpr int GT = MT * 32;  // threads per key group
    // Each key group's last warp issues its copies: a tile with fewer rows
    // than the CTA holds leaves its last warps without rows to compute, and
    // the copies then cost the computing warps nothing.
    constexpr int kIssuer = MT - 1;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *body = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sMo = reinterpret_cast<float *>(body);          // [KW][R][DP], aliases the stages
    float *sMm = sMo + (size_t)KW * R * DP;                 // [KW][R]
    float *sMl = sMm + KW * R;                              // [KW][R]
    unsigned char *qarea = body + C::kBodyBytes;
    float *sPm = reinterpret_cast<float *>(qarea + C::kQBytes);  // [R] this CTA's merged max
    float *sPl = sPm + R;                                   // [R] and sum
    int *sLo = reinterpret_cast<int *>(sPl + R);            // [R] key bounds per row
    int *sHi = sLo + R;
    float *sLse = reinterpret_cast<float *>(sHi + R);       // [R] merged log-sum-exp
    float *sAllM = sLse + R;                                // [R][16] cluster maxima, then merge weights
    float *sAllL = sAllM + R * 16;                          // [R][16] cluster sums
    uint64_t *bars = reinterpret_cast<uint64_t *>(sAllL + R * 16);  // [KW][NST]
    float *sSimt = reinterpret_cast<float *>(bars + KW * NST);
    int *sFlag = reinterpret_cast<int *>(sSimt + (C::kSimtBytes / 4));  // [1] own flags: 1 bad page, 2 timeout
    int *sAllF = sFlag + 1;                                 // [16] flags of the cluster
    int *sCov = sFlag + 32;                                 // [NT] coverage flags of the first rows
    float *sRecv = reinterpret_cast<float *>(sCov + NT);    // pushed partial outputs (kPush)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = warp % MT, kw = warp / MT;
    const int gtid = tid - kw * GT;  // thread index inside the key group
    const int rank = blockIdx.x, ncta = gridDim.x;
    const int g = blockIdx.y / p.row_tiles, rt = blockIdx.y - g * p.row_tiles;
    const int s = blockIdx.z;
    // CTAs that own a slice of output rows for the coverage check.
    const bool cov_cta = grid_cta_index() < coverage_slices(p, NT);

    // Rows no segment covers: counted before the dependency wait (the
    // segment table is not written by the previous kernel), zeroed after it.
    const int cov_any = coverage_begin(p, sCov, cov_cta, NT);
    if (p.S == 0) {  // nothing but rows no segment covers
        pdl_wait();
        pdl_trigger();
        if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
        return;
    }

    // ---- segment and its key range (reads allowed before the dependency wait)
    const Segment sg = load_segment(p.seq_info, s);
    unsigned fault = segment_fault(sg, p.total_rows, p.max_seqs, p.mbps, p.ring_rows, p.window);
    if (!fault && sg.ql > p.max_q_len) fault = PKV_ERR_QLEN;
    const int rows_unit = fault ? 0 : sg.ql * p.G;
    const int row0 = rt * R;
    if (fault || row0 >= rows_unit) {  // uniform across the cluster: same segment and row tile
        pdl_wait();
        pdl_trigger();
        if (fault && rank == 0 && rt == 0) {
            if (tid == 0) atomicOr(p.err, fault);
            zero_segment_rows(p, sg, g, NT);
        }
        if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
        return;
    }
    if (C::kPush && ncta > 1)  // announce this CTA to the cluster; waited on before any remote store
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
    const int rows_here = min(R, rows_unit - row0);
    // Positions fit in 32 bits: kv_end <= 2^31 - 33 is part of segment validity.
    const int kend = sg.kend;
    const int new_start = kend - sg.ql;  // first position appended this step
    const int first = first_valid_of(p.first_valid, sg.col);
    const int lo_u = segment_key_lo(new_start, kend, p.causal, p.window, first);
    const int pb_begin = lo_u / kPage;
    const int pb_end = (kend + kPage - 1) / kPage;
    const int nblk = pb_end - pb_begin;
    const int bps = (nblk + ncta - 1) / ncta;
    const int active = (nblk + bps - 1) / bps;
    const int cb0 = pb_begin + rank * bps;
    const int nb = rank < active ? min(cb0 + bps, pb_end) - cb0 : 0;
    const int n_mine = nb > kw ? (nb - kw + KW - 1) / KW : 0;

    const T *knew = reinterpret_cast<const T *>(p.k_new);
    const T *vnew = reinterpret_cast<const T *>(p.v_new);
    const bool fused = knew != nullptr;
    const int dchunks = p.D / EPC;  // real 16-byte chunks per row
    const int *bt_row = p.block_table + (long long)sg.col * p.mbps;
    uint64_t *gbars = bars + kw * NST;
    unsigned char *gstage = body + (size_t)kw * NST * C::kStageBytes;
    const int lo_pos = cb0 * kPage, hi_pos = (cb0 + nb) * kPage;
    // This CTA's pages hold some of the step's own positions (fused call).
    const bool has_new = fused && rt == 0 && nb > 0 && new_start < hi_pos && kend > lo_pos;

    if (gtid == 0) {
        #pragma unroll 1
        for (int i = 0; i < NST; ++i) mbar_init(gbars + i, 1);
        fence_barrier_init();
    }
    if (tid == 0) sFlag[0] = 0;
    __syncthreads();

    // Fused append: written only if every slot of the segment's new rows maps
    // to a valid page (checked here, before the dependency wait: the block
    // table is not written by the previous kernel).
    bool app_ok = false;
    if (has_new) {
        bool ok = true;
        #pragma unroll 1
        for (int i = tid; i < sg.ql; i += NT) {
            const int pos = new_start + i;
            const int rr = p.ring_rows ? pos % p.ring_rows : pos;
            const int b = bt_row[rr / kPage];
            ok &= b >= 0 && (long long)b < p.num_blocks;
        }
        app_ok = __syncthreads_and(ok);
    }

    // Page ids of this group's pages, 32 at a time, held by the group's
    // issuing warp: lane l holds the id of the group's page (window + l).
    int id_reg = -1, id_window = -1;
    bool bad = false, timed_out = false;
    auto load_ids = [&](int j) {
        id_window = j & ~31;
        const int li = kw + (id_window + lane) * KW;
        id_reg = -1;
        if (li < nb) id_reg = bt_row[table_page(cb0 + li, p.ring_rows)];
    };
    // Warm L2 with page `bid` of this kv head (K and V).
    auto prefetch_page = [&](int bid) {
        if (p.page_box) {
            tma_prefetch_l2_5d(&p.tmap_k, 0, 0, 0, g, bid);
            tma_prefetch_l2_5d(&p.tmap_v, 0, 0, 0, g, bid);
        } else {
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b) {
                tma_prefetch_l2_4d(&p.tmap_k, b * C::kBoxEl, g, 0, bid);
                tma_prefetch_l2_4d(&p.tmap_v, b * C::kBoxEl, g, 0, bid);
            }
        }
    };
    // Issue the TMA copies of the group's j-th page (called by the group's
    // issuing warp).
    auto issue = [&](int j) {
        if ((j & ~31) != id_window) load_ids(j);
        const int bid = __shfl_sync(0xffffffffu, id_reg, j & 31);
        const bool ok = bid >= 0 && (long long)bid < p.num_blocks;
        bad |= !ok;
        if (lane == 0) {
            uint64_t *bar = gbars + (j % NST);
            unsigned char *st = gstage + (size_t)(j % NST) * C::kStageBytes;
            if (ok) {
                fence_proxy_async();
                mbar_expect_tx(bar, C::kStageBytes);
                if (p.page_box) {
                    tma_load_5d(st, &p.tmap_k, bar, 0, 0, 0, g, bid);
                    tma_load_5d(st + C::kTileBytes, &p.tmap_v, bar, 0, 0, 0, g, bid);
                } else {
#pragma unroll
                    for (int b = 0; b < C::kBoxes; ++b) {
                        tma_load_4d(st + b * 2048, &p.tmap_k, bar, b * C::kBoxEl, g, 0, bid);
                        tma_load_4d(st + C::kTileBytes + b * 2048, &p.tmap_v, bar, b * C::kBoxEl, g, 0, bid);
                    }
                }
            } else {
                mbar_arrive(bar);  // nothing to fetch: complete the phase, the result is discarded
            }
        }
    };
    // Pages wholly below new_start hold keys written before this step, so they
    // may be fetched before the dependency wait.  In the fused call every page
    // may: the step's own rows are replaced from k_new / v_new after the wait.
    auto early_ok = [&](int j) { return fused || (cb0 + kw + j * KW + 1) * kPage <= new_start; };
    // Bounded wait for the j-th page of the group; warp-uniform result.
    auto wait_page = [&](int j) {
        if (timed_out) return;
        bool done = false;
        if (lane == 0) {
            #pragma unroll 1
            for (int it = 0; it < kWaitProbes && !done; ++it) done = mbar_try_wait(gbars + (j % NST), (j / NST) & 1);
        }
        done = __shfl_sync(0xffffffffu, done, 0);
        if (!done) timed_out = true;
    };

    // Warm L2 with the rows read right after the wait: this tile's queries and,
    // in the fused call, this step's K/V rows.  A prefetch returns nothing, so
    // issuing it before the dependency wait cannot observe stale data.
    {
        const int lines = (p.D * C::kElem + 127) / 128;
        const int nq = rows_here * lines;
#pragma unroll 1
        for (int c = tid; c < nq; c += NT) {
            const int r = c / lines, ln = c - r * lines, ur = row0 + r, i = ur / p.G, jh = ur - i * p.G;
            const T *src = reinterpret_cast<const T *>(p.q) + (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D;
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + ln * 128));
        }
        if (has_new) {
            const int a = max(new_start, lo_pos), e = min(kend, hi_pos);
            const int n = (e - a) * 2 * lines;
#pragma unroll 1
            for (int c = tid; c < n; c += NT) {
                const int row = c / (2 * lines), rem = c - row * 2 * lines, kv = rem / lines, ln = rem - kv * lines;
                const T *src = (kv ? vnew : knew) + (((long long)sg.q0 + (a + row - new_start)) * p.Hkv + g) * p.D;
                asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + ln * 128));
            }
        }
    }

    // ---- prologue: start the first stages before waiting on the previous kernel
    int issued = 0;
    if (mt == kIssuer) {
        load_ids(0);
        #pragma unroll 1
        for (; issued < NST && issued < n_mine; ++issued) {
            if (!early_ok(issued)) break;
            issue(issued);
        }
    }
    // Pages past the shared-memory stages are prefetched into L2 now, so
    // their HBM traffic overlaps the previous kernel's tail and the later TMA
    // copies hit L2.  Lane l of the issuing warp holds page l's id.
    if (mt == kIssuer) {
        const int bid = id_reg;
        if (lane >= issued && lane < min(n_mine, NST + C::kL2Pages) && bid >= 0 && (long long)bid < p.num_blocks)
            prefetch_page(bid);
    }
    pdl_wait();
    pdl_trigger();

    // This step's rows that fall in the CTA's last page (decode: the one new
    // row) are loaded now, next to the query loads, by the key group that
    // consumes that page; the page fix-up stores them.
    const int last_li = nb - 1, last_pos0 = (cb0 + last_li) * kPage;
    const int pre_a = max(new_start, last_pos0), pre_n = has_new ? max(0, kend - pre_a) : 0;
    const bool pre_mine = pre_n > 0 && kw == last_li % KW;
    uint4 pre[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        pre[it] = make_uint4(0u, 0u, 0u, 0u);
        const int c = gtid + it * GT;
        if (pre_mine && c < 2 * pre_n * dchunks) {
            const int kv = c / (pre_n * dchunks), rem = c - kv * pre_n * dchunks;
            const int row = rem / dchunks, ch = rem - row * dchunks;
            pre[it] = *reinterpret_cast<const uint4 *>((kv ? vnew : knew) +
                                                       (((long long)sg.q0 + (pre_a + row - new_start)) * p.Hkv + g) * p.D +
                                                       ch * EPC);
        }
    }

    if (cov_cta) apply_coverage(p, sCov, cov_any, NT);

    // Query rows of this tile (all loads issued before any store) and their key bounds.
    {
        constexpr int kQIt = (R * C::kChunks + NT - 1) / NT;
        uint4 qv[kQIt];
#pragma unroll
        for (int it = 0; it < kQIt; ++it) {
            const int c = tid + it * NT;
            const int r = c / C::kChunks, ch = c - r * C::kChunks, ur = row0 + r;
            qv[it] = make_uint4(0u, 0u, 0u, 0u);
            if (c < R * C::kChunks && ur < rows_unit && ch < dchunks) {
                const int i = ur / p.G, jh = ur - i * p.G;
                qv[it] = *reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const T *>(p.q) +
                    (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D + ch * EPC);
            }
        }
#pragma unroll
        for (int it = 0; it < kQIt; ++it) {
            const int c = tid + it * NT;
            if (c >= R * C::kChunks) continue;
            const int r = c / C::kChunks, ch = c - r * C::kChunks;
            if constexpr (C::MMA) {
                *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(qarea) + r * C::kQLd + ch * EPC) = qv[it];
            } else {
                float f[EPC];
                load_f32<T, EPC>(f, reinterpret_cast<const T *>(&qv[it]));
                float *dst = reinterpret_cast<float *>(qarea) + r * C::kQLd + ch * EPC;
#pragma unroll
                for (int e = 0; e < EPC; ++e) dst[e] = f[e];
            }
        }
    }
#pragma unroll 1
    for (int r = tid; r < R; r += NT) {
        const int ur = row0 + r;
        int lo = 0, hi = 0;
        if (ur < rows_unit) row_key_bounds(new_start + ur / p.G, kend, p.causal, p.window, first, lo, hi);
        sLo[r] = lo;
        sHi[r] = hi;
    }
    if (mt == kIssuer) {
        #pragma unroll 1
        for (; issued < NST && issued < n_mine; ++issued) issue(issued);
    }
    __syncthreads();

    // ---- main loop over this group's pages
    const int nrw = max(0, min(16, rows_here - mt * 16));
    MmaWarp<C> mw;
    SimtWarp<C> sw;
    if constexpr (C::MMA) mw.init(reinterpret_cast<const T *>(qarea), mt, lane);
    else sw.init();
    float *sPw = sSimt + warp * (16 * 16 + 16);
    auto group_sync = [&]() {
        if constexpr (MT == 1) __syncwarp(); else named_barrier(1 + kw, GT);
    };

    // Rows outside [lo_u, kend) may hold anything (NaN included): zero them.
    // This step's own rows come from k_new / v_new in the fused call, and
    // the CTA that owns them also writes them into the cache here.
    auto fix_page = [&](int j, unsigned char *st, int pos0) {
        const int zlo = min(max(lo_u - pos0, 0), kPage);          // rows [0, zlo) precede the window
        const int zhi = min(max(kend - pos0, 0), kPage);          // rows [zhi, 16) are past kv_end
        const int na = fused ? min(max(new_start - pos0, 0), kPage) : zhi;  // rows [na, zhi) are new
        if (!(zlo > 0 || zhi < kPage || na < zhi)) return;
        const int nz = (zlo + kPage - zhi) * C::kChunks;
#pragma unroll 1
        for (int c = gtid; c < 2 * nz; c += GT) {
            const int kv = c >= nz, rem = c - kv * nz, o0 = rem / C::kChunks, ch = rem - o0 * C::kChunks;
            const int o = o0 < zlo ? o0 : zhi + (o0 - zlo);
            *reinterpret_cast<uint4 *>(st + kv * C::kTileBytes + swz(o, ch)) = make_uint4(0u, 0u, 0u, 0u);
        }
        const int nn = (zhi - na) * C::kChunks;
        if (nn > 0) {
            const bool to_pool = app_ok;
            const long long bpage = to_pool ? (long long)bt_row[table_page(pos0 / kPage, p.ring_rows)] : 0;
            const int ring_base = p.ring_rows ? pos0 % p.ring_rows : pos0;  // slot of the page's first row
            const bool preloaded = pre_mine && j == last_li / KW && pos0 + na == pre_a;
#pragma unroll 1
            for (int c = gtid; c < 2 * nn; c += GT) {
                const int kv = c >= nn, rem = c - kv * nn, r0 = rem / C::kChunks, ch = rem - r0 * C::kChunks;
                const int o = na + r0;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (ch < dchunks) {
                    // the preload enumerated (kv, row, real chunk); map this chunk onto it
                    const int pc = kv * pre_n * dchunks + r0 * dchunks + ch;
                    const int q = pc - gtid;
                    if (preloaded && q >= 0 && q % GT == 0 && q / GT < 2)
                        v = q == 0 ? pre[0] : pre[1];
                    else
                        v = *reinterpret_cast<const uint4 *>(
                            (kv ? vnew : knew) + (((long long)sg.q0 + (pos0 + o - new_start)) * p.Hkv + g) * p.D +
                            ch * EPC);
                    if (to_pool) {
                        const long long slot = bpage * kPage + (ring_base + o) % kPage;
                        *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(kv ? p.v_pool_w : p.k_pool_w) +
                                                   (slot * p.Hkv + g) * p.D + ch * EPC) = v;
                    }
                }
                *reinterpret_cast<uint4 *>(st + kv * C::kTileBytes + swz(o, ch)) = v;
            }
        }
        // The stage is rewritten by TMA only if it is refilled.
        if (j + NST < n_mine) fence_proxy_async();
        group_sync();
    };

    // Several pages per pass where the ring holds them (independent MMA
    // chains): four with eight stages, else two.
    constexpr int kPair = C::MMA && NST >= 8 ? 4 : C::MMA && NST >= 2 ? 2 : 1;
#pragma unroll 1
    for (int j = 0; j < n_mine; j += kPair) {
        const int np = min(kPair, n_mine - j);
        unsigned char *st[4];
        int pos0[4];
#pragma unroll
        for (int u = 0; u < kPair; ++u) {
            const int jj = j + min(u, np - 1);
            st[u] = gstage + (size_t)(jj % NST) * C::kStageBytes;
            pos0[u] = (cb0 + kw + jj * KW) * kPage;
        }
#pragma unroll
        for (int u = 0; u < kPair; ++u) {
            if (u < np) {
                wait_page(j + u);
                fix_page(j + u, st[u], pos0[u]);
            }
        }
        if (nrw > 0) {
            if constexpr (C::MMA) {
                const unsigned char *ks[4], *vs[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    ks[u] = st[min(u, kPair - 1)];
                    vs[u] = st[min(u, kPair - 1)] + C::kTileBytes;
                }
                if (np == 4)
                    mw.template consume<4>(reinterpret_cast<const T *>(qarea), ks, vs, pos0, sLo, sHi, mt, lane,
                                           p.scale_log2);
                else if (np == 3)
                    mw.template consume<3>(reinterpret_cast<const T *>(qarea), ks, vs, pos0, sLo, sHi, mt, lane,
                                           p.scale_log2);
                else if (np == 2)
                    mw.template consume<2>(reinterpret_cast<const T *>(qarea), ks, vs, pos0, sLo, sHi, mt, lane,
                                           p.scale_log2);
                else
                    mw.template consume<1>(reinterpret_cast<const T *>(qarea), ks, vs, pos0, sLo, sHi, mt, lane,
                                           p.scale_log2);
            } else {
                sw.consume(reinterpret_cast<const float *>(qarea), st[0], st[0] + C::kTileBytes, pos0[0], sLo, sHi,
                           mt, lane, nrw, p.scale_log2, sPw);
            }
        }
        group_sync();  // every warp of the group is done with these stages
        if (mt == kIssuer) {
#pragma unroll
            for (int u = 0; u < kPair; ++u)
                if (u < np && j + u + NST < n_mine) issue(j + u + NST);
        }
    }
    if (timed_out && lane == 0 && mt == kIssuer) {
        // Give the copies still in flight a bounded chance to land before the
        // stage memory is reused.
        #pragma unroll 1
        for (int j = max(0, n_mine - NST); j < n_mine; ++j)
            #pragma unroll 1
            for (int it = 0; it < kWaitProbes && !mbar_try_wait(gbars + (j % NST), (j / NST) & 1); ++it) {
            }
    }
    if ((bad || timed_out) && lane == 0) atomicOr(sFlag, (bad ? 1 : 0) | (timed_out ? 2 : 0));
    __syncthreads();  // stages are free, flags are final

    // ---- merge the key groups of this CTA
    const int flags = sFlag[0];
    if (nrw > 0 || !C::MMA) {
        if constexpr (C::MMA) mw.store(sMo, sMm, sMl, kw, mt, lane);
        else sw.store(sMo, sMm, sMl, kw, mt, lane, nrw);
    }
    if (tid == 0 && flags) atomicOr(p.err, ((flags & 1) ? PKV_ERR_BLOCK : 0u) | ((flags & 2) ? PKV_ERR_TIMEOUT : 0u));
    __syncthreads();

    merge_rows<DP, KW, R, NT, C::kPush>(p, sg, g, row0, rows_here, flags, rank, ncta, sMo, sMm, sMl, sPm, sPl, sLse,
                                        sAllM, sAllL, sAllF, sFlag, sRecv);
}

}  // namespace pkv
