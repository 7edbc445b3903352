// Split-K decode attention for narrow query groups (sm_103a).
//
// Same semantics and launch shape as attend_kernel (grid (C, kv_heads,
// segments), the C CTAs of a (segment, kv head) forming one cluster), for the
// decode case where a kv head's query group has at most 8 rows (G * q_len <=
// 8: one token of a GQA group, or a few tokens of a narrow group).  Such a
// group is too narrow for the 16-row side of an MMA tile, so the products are
// taken transposed, with the query rows as the 8-wide N side:
//
//   S^T (16 keys x 8 rows)   = K (16 keys x D) . Q^T        keys as M
//   O^T (D x 8 rows)        += V^T (D x 16 keys) . P^T      head_dim as M
//
// Q^T stays in registers as B fragments for the whole key range; P^T comes
// from the S^T accumulators through one in-register 8x8 transpose
// (movmatrix) per half page.  Every MMA row is a real key or a real head_dim
// column, where a 16-row query tile would leave 12 of its 16 rows empty for
// the common 4-head group.
//
// Each warp is a key group with its own ring of NST page stages (TMA,
// 128-byte swizzle, one mbarrier per stage) and takes every KW-th page of the
// CTA's range.  At the end the warps merge in shared memory (each writes its
// partial over its own, now idle, stages) and the CTAs merge through
// distributed shared memory: every CTA pushes its merged partial for each
// output slice straight into the shared memory of the CTA that owns that
// slice, one cluster barrier later the owner finishes its slice.
//
// Semantics follow the segment-table attention of ExecuTorch PR #24072
// (triton::sdpa_varlen) over the paged layout of vLLM-Omni's SenseNova-U1
// PagedDecodeCache, exactly as attend_kernel.
#pragma once

#include "attend.cuh"

namespace pkv {

// Key ranges of at most this many pages per compute warp run on one CTA.
constexpr int kSoloPages = 3;
// Lazy rescaling threshold of the online softmax (base-2 exponent): weights
// stay at most 2^8, well inside fp32 and with bf16's relative precision.
constexpr float kLazyLog2 = 8.f;

template <int DP_, int KW_, int NST_, bool SIMT_ = false>
struct DecCfg {
    using T = __nv_bfloat16;
    static constexpr int DP = DP_;      // head_dim rounded up to 64 / 128 / 256
    static constexpr bool SIMT = SIMT_; // dot products on the CUDA cores (fp32 FMA) instead of mma.sync
    static constexpr int KW = KW_;      // warps = key groups
    static constexpr int NST = NST_;    // page stages per warp
    static constexpr int kThreads = KW * 32;
    static constexpr int kRows = 8;                      // query rows per CTA (the MMA N side)
    static constexpr int kKT = DP / 16;                  // 16-wide steps over head_dim
    static constexpr int kEpc = 8;                       // bf16 elements per 16-byte chunk
    static constexpr int kChunks = DP / kEpc;
    static constexpr int kBoxEl = 64;                    // elements per 128-byte swizzle box row
    static constexpr int kBoxes = DP / kBoxEl;
    static constexpr unsigned kTileBytes = kPage * DP * 2;
    static constexpr unsigned kStageBytes = 2 * kTileBytes;
    static constexpr size_t kPipeBytes = (size_t)KW * NST * kStageBytes;
    static constexpr int kPartLd = DP + 4;               // padded row of a warp's partial (bank spread)
    static constexpr size_t kPartBytes = (size_t)kRows * kPartLd * 4 + 2 * kRows * 4;
    // Pushed by the cluster: C CTAs x 8 rows x per columns (per = the power
    // of two >= DP / C, so C * per < 2 * DP); then (max, sum) per CTA and row.
    static constexpr int kRecvLd = 2 * DP;
    static constexpr size_t kRecvBytes = (size_t)kRows * kRecvLd * 4;
    static constexpr size_t kWnBytes = (size_t)kRows * 16 * 4 + kRows * 4;  // merge weights, lse per row
    static constexpr size_t kStatBytes = (size_t)16 * kRows * 8;
    static constexpr size_t kBarBytes = (size_t)KW * NST * 8;
    static constexpr size_t kFlagBytes = 32 * 4;
    static constexpr size_t kCovBytes = (size_t)kThreads * 4;
    // CUDA-core variant: each lane owns kE consecutive head_dim columns; a
    // warp's page weights P go through shared memory, [row][token] with rows
    // padded to kPLd floats (conflict-free stores, 16-byte aligned rows).
    static constexpr int kE = DP / 32;
    static constexpr int kPLd = kPage + 4;
    static constexpr size_t kPBytes = SIMT ? 16 + (size_t)KW * kRows * kPLd * 4 : 0;
    static constexpr size_t kSmemBytes =
        1024 + kPipeBytes + kRecvBytes + kStatBytes + kBarBytes + kFlagBytes + kCovBytes + kWnBytes + kPBytes;
    // L2 warm-up before the dependency wait: each warp prefetches up to
    // kL2Pages pages past its stages, about 512 KB per SM over the CTAs that
    // fit on one (at most 32 pages: the page-id window of a warp).
    static constexpr int kCtasPerSm = (int)(232448 / (kSmemBytes + 1024)) > 0 ? (int)(232448 / (kSmemBytes + 1024)) : 1;
    static constexpr int kL2PagesRaw = (int)(524288 / ((size_t)kCtasPerSm * KW * kStageBytes));
    static constexpr int kL2Pages = kL2PagesRaw < 1 ? 1 : kL2PagesRaw > 32 - NST ? 32 - NST : kL2PagesRaw;
    static_assert(kThreads >= 128, "the merges map 8 rows x 16 onto the first 128 threads");
    static_assert(kPartBytes <= NST * kStageBytes, "a warp's partial fits over its own stages");
    static_assert(DP % kBoxEl == 0, "page rows are whole 128-byte boxes");
};

// Transpose of the 8x8 bf16 matrix whose row lane/4, columns 2*(lane%4) and
// 2*(lane%4)+1 this thread holds.
__device__ __forceinline__ unsigned movmatrix_trans(unsigned x) {
    unsigned y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// One halving step of a reduce-scatter across lanes: the lane whose bit `m`
// is set keeps the upper HALF values, the other the lower, each adding its
// partner's copy.  Returns the offset of the kept half.
template <int HALF>
__device__ __forceinline__ int rs_halve(float (&x)[16], int lane_bits, int m) {
    const bool upper = (lane_bits & m) != 0;
#pragma unroll
    for (int e = 0; e < HALF; ++e) {
        const float send = upper ? x[e] : x[e + HALF];
        const float keep = upper ? x[e + HALF] : x[e];
        x[e] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    return upper ? HALF : 0;
}

// Register budget for the CTAs that fit on one SM by shared memory (two at
// head_dim 64 / 128, one at 256).
template <class C>
__global__ void __launch_bounds__(C::kThreads, C::kCtasPerSm) decode_kernel(const __grid_constant__ AttendParams p) {
    using T = __nv_bfloat16;
    namespace cg = cooperative_groups;
    constexpr int DP = C::DP, KW = C::KW, NST = C::NST, NT = C::kThreads, KT = C::kKT, LD = C::kPartLd;
    constexpr int EPC = C::kEpc;
    constexpr float kLn2 = 0.6931471805599453f;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *pipe = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sRecv = reinterpret_cast<float *>(pipe + C::kPipeBytes);      // [ncta][8][per]
    float2 *sStat = reinterpret_cast<float2 *>(sRecv + C::kRows * C::kRecvLd);  // [16][8] (max, sum)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sStat + 16 * C::kRows);  // [KW][NST]
    int *sFlag = reinterpret_cast<int *>(bars + KW * NST);  // [0] own flags: 1 bad page, 2 timeout
    int *sAllF = sFlag + 1;                                 // [16] flags of the cluster
    int *sCov = sFlag + 32;                                 // [NT] coverage flags of the first rows
    float *sWn = reinterpret_cast<float *>(sCov + NT);      // [8][16] normalised cluster merge weights
    // CUDA-core variant: this warp's page weights, [8 rows][kPLd]
    float *sP = reinterpret_cast<float *>(
                    (reinterpret_cast<uintptr_t>(sWn + C::kRows * 16 + C::kRows) + 15) & ~uintptr_t(15)) +
                (threadIdx.x >> 5) * C::kRows * C::kPLd;

    const int tid = threadIdx.x, kw = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;  // MMA fragment coordinates
    const int rank = blockIdx.x, ncta = gridDim.x;
    const int g = blockIdx.y;  // one CTA row per kv head: the whole group fits the 8 rows
    const int s = blockIdx.z;
    // CTAs that own a slice of output rows for the coverage check.
    const bool cov_cta = grid_cta_index() < coverage_slices(p, NT);

    // Rows no segment covers: counted before the dependency wait, zeroed after.
    const int cov_any = coverage_begin(p, sCov, cov_cta, NT);
    if (p.S == 0) {
        pdl_wait();
        pdl_trigger();
        if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
        return;
    }

    // ---- segment and its key range (reads allowed before the dependency wait)
    const Segment sg = load_segment(p.seq_info, s);
    unsigned fault = segment_fault(sg, p.total_rows, p.max_seqs, p.mbps, p.ring_rows, p.window);
    if (!fault && sg.ql > p.max_q_len) fault = PKV_ERR_QLEN;
    const int rows_unit = fault ? 0 : sg.ql * p.G;  // <= 8: max_q_len * G <= 8 selects this kernel
    if (fault || rows_unit == 0) {  // uniform across the cluster
        pdl_wait();
        pdl_trigger();
        if (fault && rank == 0) {
            if (tid == 0) atomicOr(p.err, fault);
            zero_segment_rows(p, sg, g, NT);
        }
        if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
        return;
    }
    const int kend = sg.kend;
    const int new_start = kend - sg.ql;
    const int first = first_valid_of(p.first_valid, sg.col);
    const int lo_u = segment_key_lo(new_start, kend, p.causal, p.window, first);
    const int pb_begin = lo_u / kPage;
    const int pb_end = (kend + kPage - 1) / kPage;
    const int nblk = pb_end - pb_begin;
    // A short range (a few pages per warp) is cheaper on one CTA than split
    // and merged across the cluster: the first CTA then takes it alone and
    // the cluster's merge is skipped (uniformly: it depends on kv_end only).
    const bool solo = nblk <= kSoloPages * KW;
    const int ncl = solo ? 1 : ncta;  // CTAs that share the range
    const bool gm = p.ws_count != nullptr;  // partials merged through global memory, no cluster
    const int bps = solo ? nblk : (nblk + ncta - 1) / ncta;
    const int active = bps > 0 ? (nblk + bps - 1) / bps : 0;
    const int cb0 = pb_begin + rank * bps;
    const int nb = rank < active ? min(cb0 + bps, pb_end) - cb0 : 0;
    const int n_mine = nb > kw ? (nb - kw + KW - 1) / KW : 0;
    // A CTA with nothing to read or write (a solo range's other ranks; with
    // the global merge, ranks past the active ones) only does its share of
    // the coverage check.
    if ((solo && rank > 0) || (gm && rank >= active)) {
        if (cov_cta) {
            pdl_wait();
            pdl_trigger();
            apply_coverage(p, sCov, cov_any, NT);
        }
        return;
    }
    if (ncl > 1 && !gm)  // announce this CTA to the cluster; waited on before any remote store
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");

    const T *knew = reinterpret_cast<const T *>(p.k_new);
    const T *vnew = reinterpret_cast<const T *>(p.v_new);
    const bool fused = knew != nullptr;
    const int dchunks = p.D / EPC;
    const int *bt_row = p.block_table + (long long)sg.col * p.mbps;
    uint64_t *wbars = bars + kw * NST;
    unsigned char *wstage = pipe + (size_t)kw * NST * C::kStageBytes;
    const int lo_pos = cb0 * kPage, hi_pos = (cb0 + nb) * kPage;
    const bool has_new = fused && nb > 0 && new_start < hi_pos && kend > lo_pos;

    if (lane == 0) {
        #pragma unroll 1
        for (int i = 0; i < NST; ++i) mbar_init(wbars + i, 1);
        fence_barrier_init();
    }
    if (tid == 0) sFlag[0] = 0;
    __syncthreads();

    // ---- page ids and TMA issue (lane l of the warp holds the id of its page window + l)
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
    // Issue the TMA copies of the warp's j-th page.
    auto issue = [&](int j) {
        if ((j & ~31) != id_window) load_ids(j);
        const int bid = __shfl_sync(0xffffffffu, id_reg, j & 31);
        const bool ok = bid >= 0 && (long long)bid < p.num_blocks;
        bad |= !ok;
        if (lane == 0) {
            uint64_t *bar = wbars + (j % NST);
            unsigned char *st = wstage + (size_t)(j % NST) * C::kStageBytes;
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
    // Pages wholly below new_start were written before this step and may be
    // fetched before the dependency wait; in the fused call every page may
    // (the step's own rows are replaced from k_new / v_new after it).
    auto early_ok = [&](int j) { return fused || (cb0 + kw + j * KW + 1) * kPage <= new_start; };
    // Bounded wait for the warp's j-th page; every lane observes the phase.
    auto wait_page = [&](int j) {
        if (timed_out) return;
        bool done = false;
        #pragma unroll 1
        for (int it = 0; it < kWaitProbes && !done; ++it) done = mbar_try_wait(wbars + (j % NST), (j / NST) & 1);
        if (!__all_sync(0xffffffffu, done)) timed_out = true;
    };

    // A whole page of the next layer (every kv head, K and V: one contiguous
    // block each), one bulk prefetch per tensor.
    const unsigned page_bytes = (unsigned)(kPage * p.Hkv * p.D * (int)sizeof(T));
    auto warm_next = [&](int bid) {
        bulk_prefetch_l2(reinterpret_cast<const char *>(p.k_next) + (size_t)bid * page_bytes, page_bytes);
        bulk_prefetch_l2(reinterpret_cast<const char *>(p.v_next) + (size_t)bid * page_bytes, page_bytes);
    };

    int issued = 0;
    load_ids(0);
    #pragma unroll 1
    for (; issued < NST && issued < n_mine; ++issued) {
        if (!early_ok(issued)) break;
        issue(issued);
    }
    // V rows outside [lo_u, kend) may hold anything (NaN included) and are
    // zeroed in shared memory (their scores are masked).
    auto zero_stale = [&](unsigned char *st, int zlo, int zhi) {
        const int nz = (zlo + kPage - zhi) * C::kChunks;
        #pragma unroll 1
        for (int c = lane; c < nz; c += 32) {
            const int o0 = c / C::kChunks, ch = c - o0 * C::kChunks;
            const int o = o0 < zlo ? o0 : zhi + (o0 - zlo);
            *reinterpret_cast<uint4 *>(st + C::kTileBytes + swz(o, ch)) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // Edge pages already in flight (the last page past kv_end, the first
    // before the window) are zeroed now, while the previous kernel runs.
    unsigned prezero = 0;
    #pragma unroll 1
    for (int j = 0; j < issued; ++j) {
        const int pos0 = (cb0 + kw + j * KW) * kPage;
        const int zlo = min(max(lo_u - pos0, 0), kPage), zhi = min(max(kend - pos0, 0), kPage);
        if (zlo > 0 || zhi < kPage) {
            wait_page(j);
            if (!timed_out) {
                zero_stale(wstage + (size_t)(j % NST) * C::kStageBytes, zlo, zhi);
                prezero |= 1u << j;
            }
        }
    }
    // The warp's pages past its stages go to L2 now, so their HBM traffic
    // overlaps the previous kernel's tail.  Lane l holds the id of the warp's
    // page kw + l * KW.
    {
        const int bid = id_reg;
        if (lane >= issued && lane < min(n_mine, NST + C::kL2Pages) && bid >= 0 && (long long)bid < p.num_blocks)
            prefetch_page(bid);
    }
    // The next layer's first pages of the same range (same table and
    // segments: the pages its CTAs copy into their stages as they start), so
    // a CTA of the next layer that starts late finds them in L2; its later
    // pages it warms itself.  Whole pages, warmed by the CTAs of the same
    // cluster rank in turn (page li by kv head li % Hkv).
    if (p.pf_next > 0) {
        const int li = kw + lane * KW, bid = id_reg;
        if (li < min(min(nb, p.pf_next), KW * NST) && li % p.Hkv == g && bid >= 0 && (long long)bid < p.num_blocks)
            warm_next(bid);
    }
    // The step's rows in the CTA's last page (decode: the one new row) are
    // handled by the warp that computes that page.
    const int last_li = nb - 1, last_pos0 = (cb0 + last_li) * kPage;
    const int pre_a = max(new_start, last_pos0), pre_n = has_new ? max(0, kend - pre_a) : 0;
    const bool pre_mine = pre_n > 0 && kw == last_li % KW;
    // Append validity (all-or-nothing over the segment's new rows): the block
    // table is not written by the previous kernel.  One new row lives in the
    // last page, whose id this warp already holds; more rows are looked up.
    bool app_ok = false;
    if (has_new && sg.ql == 1 && last_li / KW < 32) {
        const int bid = __shfl_sync(0xffffffffu, id_reg, last_li / KW);
        app_ok = bid >= 0 && (long long)bid < p.num_blocks;
    } else if (has_new) {
        bool ok = true;
        #pragma unroll 1
        for (int i = lane; i < sg.ql; i += 32) {
            const int pos = new_start + i;
            const int rr = p.ring_rows ? pos % p.ring_rows : pos;
            const int b = bt_row[rr / kPage];
            ok &= b >= 0 && (long long)b < p.num_blocks;
        }
        app_ok = __all_sync(0xffffffffu, ok);
    }
    // Warm L2 with what is read right after the wait: the group's query rows
    // and this step's K/V rows.
    if (kw == 0) {
        const int lines = (p.D * 2 + 127) / 128;
        #pragma unroll 1
        for (int c = lane; c < rows_unit * lines; c += 32) {
            const int r = c / lines, ln = c - r * lines, i = r / p.G, jh = r - i * p.G;
            const T *src = reinterpret_cast<const T *>(p.q) + (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D;
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + ln * 128));
        }
    }
    if (has_new && kw == 1 % KW) {
        const int lines = (p.D * 2 + 127) / 128;
        const int a = max(new_start, lo_pos), e = min(kend, hi_pos);
        #pragma unroll 1
        for (int c = lane; c < (e - a) * 2 * lines; c += 32) {
            const int row = c / (2 * lines), rem = c - row * 2 * lines, kv = rem / lines, ln = rem - kv * lines;
            const T *src = (kv ? vnew : knew) + (((long long)sg.q0 + (a + row - new_start)) * p.Hkv + g) * p.D;
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + ln * 128));
        }
    }

    pdl_wait();
    pdl_trigger();

    // ---- after the wait: Q^T fragments (CUDA-core variant: this lane's
    // columns of every row in fp32), this step's new rows, row bounds
    constexpr bool SIMT = C::SIMT;
    constexpr int E = C::kE;
    unsigned qb[KT][2];
    float qs[SIMT ? C::kRows : 1][E];
    if constexpr (SIMT) {
#pragma unroll
        for (int n = 0; n < C::kRows; ++n) {
            const int i = n / p.G, jh = n - i * p.G, col = lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) qs[n][e] = 0.f;
            if (n < rows_unit && col < p.D)
                load_f32<T, E>(qs[n], reinterpret_cast<const T *>(p.q) +
                                          (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D + col);
        }
    } else {
        const bool real = gq < rows_unit;
        const int i = gq / p.G, jh = gq - i * p.G;
        const T *qrow = reinterpret_cast<const T *>(p.q) +
                        (((long long)sg.q0 + (real ? i : 0)) * p.Hq + (long long)g * p.G + (real ? jh : 0)) * p.D;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            const int d0 = kk * 16 + 2 * tq, d1 = d0 + 8;
            qb[kk][0] = real && d0 < p.D ? *reinterpret_cast<const unsigned *>(qrow + d0) : 0u;
            qb[kk][1] = real && d1 < p.D ? *reinterpret_cast<const unsigned *>(qrow + d1) : 0u;
        }
    }
    // This step's rows in the CTA's last page, loaded beside the queries; the
    // page fix-up stores them.
    uint4 pre[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        pre[it] = make_uint4(0u, 0u, 0u, 0u);
        const int c = lane + it * 32;
        if (pre_mine && c < 2 * pre_n * dchunks) {
            const int kv = c / (pre_n * dchunks), rem = c - kv * pre_n * dchunks;
            const int row = rem / dchunks, ch = rem - row * dchunks;
            pre[it] = *reinterpret_cast<const uint4 *>((kv ? vnew : knew) +
                                                       (((long long)sg.q0 + (pre_a + row - new_start)) * p.Hkv + g) * p.D +
                                                       ch * EPC);
        }
    }
    // Key bounds of the two rows this thread's fragments hold (2tq, 2tq+1);
    // padding rows see no key.
    int lo_r[2], hi_r[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int n = 2 * tq + e;
        lo_r[e] = 0;
        hi_r[e] = 0;
        if (n < rows_unit)
            row_key_bounds(new_start + n / p.G, kend, p.causal, p.window, first, lo_r[e], hi_r[e]);
    }
    // CUDA-core variant: a lane's scores are those of row lane / 4.
    const int rs = lane >> 2;
    int lo_s = 0, hi_s = 0;
    if (SIMT && rs < rows_unit) row_key_bounds(new_start + rs / p.G, kend, p.causal, p.window, first, lo_s, hi_s);
    if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
    #pragma unroll 1
    for (; issued < NST && issued < n_mine; ++issued) issue(issued);

    // ---- main loop over the warp's pages
    float acc[KT][4];
#pragma unroll
    for (int dt = 0; dt < KT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
    float m_r[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_r[2] = {0.f, 0.f};
    // CUDA-core variant: O rows x this lane's columns; (max, sum) of row rs
    float acs[SIMT ? C::kRows : 1][E];
#pragma unroll
    for (int n = 0; n < (SIMT ? C::kRows : 1); ++n)
#pragma unroll
        for (int e = 0; e < E; ++e) acs[n][e] = 0.f;
    float m_s = -CUDART_INF_F, l_s = 0.f;
    const int krow = (lane & 7) + (((lane >> 3) & 1) << 3), kchk = lane >> 4;
    const int vrow = (lane & 7) + ((lane >> 4) << 3), vchk = (lane >> 3) & 1;

    // Edge pages: stale V rows zeroed (unless done before the wait).  This
    // step's own rows come from k_new / v_new in the fused call, and the warp
    // that holds them also writes them into the cache.
    auto fix_page = [&](int j, unsigned char *st, int pos0) {
        const int zlo = min(max(lo_u - pos0, 0), kPage);
        const int zhi = min(max(kend - pos0, 0), kPage);
        const int na = fused ? min(max(new_start - pos0, 0), kPage) : zhi;
        if (!(zlo > 0 || zhi < kPage || na < zhi)) return;
        if (!(j < 32 && ((prezero >> j) & 1u))) zero_stale(st, zlo, zhi);
        const int nnr = zhi - na;  // new rows in this page
        if (nnr > 0) {
            const long long bpage = app_ok ? (long long)bt_row[table_page(pos0 / kPage, p.ring_rows)] : 0;
            const int ring_base = p.ring_rows ? pos0 % p.ring_rows : pos0;
            const bool preloaded = pre_mine && j == last_li / KW && pos0 + na == pre_a;
            const int nn = nnr * dchunks;
            #pragma unroll 1
            for (int it = 0; it * 32 < 2 * nn; ++it) {
                const int c = lane + it * 32;
                if (c < 2 * nn) {
                    const int kv = c / nn, rem = c - kv * nn, r0 = rem / dchunks, ch = rem - r0 * dchunks;
                    const int o = na + r0;
                    uint4 v;
                    if (preloaded && it < 2)
                        v = it == 0 ? pre[0] : pre[1];
                    else
                        v = *reinterpret_cast<const uint4 *>(
                            (kv ? vnew : knew) + (((long long)sg.q0 + (pos0 + o - new_start)) * p.Hkv + g) * p.D +
                            ch * EPC);
                    if (app_ok) {
                        const long long slot = bpage * kPage + (ring_base + o) % kPage;
                        *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(kv ? p.v_pool_w : p.k_pool_w) +
                                                   (slot * p.Hkv + g) * p.D + ch * EPC) = v;
                    }
                    *reinterpret_cast<uint4 *>(st + kv * C::kTileBytes + swz(o, ch)) = v;
                }
            }
        }
        if (j + NST < n_mine) fence_proxy_async();  // the stage is rewritten by TMA only if refilled
        __syncwarp();
    };

    #pragma unroll 1
    for (int j = 0; j < n_mine; ++j) {
        unsigned char *st = wstage + (size_t)(j % NST) * C::kStageBytes;
        const int pos0 = (cb0 + kw + j * KW) * kPage;
        wait_page(j);
        fix_page(j, st, pos0);
        if constexpr (SIMT) {
            // Scores of 4 keys at a time: each lane sums its columns for
            // every (row, key) slot, then a reduce-scatter across the warp
            // leaves slot `lane` = (row lane / 4, key lane % 4) with lane.
            float sc[4];
#pragma unroll
            for (int tg = 0; tg < 4; ++tg) {
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = 0.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float kf[E];
                    tile_load<T, E>(kf, st, tg * 4 + u, lane * E);
#pragma unroll
                    for (int n = 0; n < C::kRows; ++n)
#pragma unroll
                        for (int e = 0; e < E; ++e) x[n * 4 + u] = fmaf(qs[n][e], kf[e], x[n * 4 + u]);
                }
#pragma unroll
                for (int h = 16; h >= 1; h >>= 1) {
                    const bool upper = (lane & h) != 0;
#pragma unroll
                    for (int e = 0; e < h; ++e) {
                        const float send = upper ? x[e] : x[e + h];
                        const float keep = upper ? x[e + h] : x[e];
                        x[e] = keep + __shfl_xor_sync(0xffffffffu, send, h);
                    }
                }
                const int pos = pos0 + tg * 4 + (lane & 3);
                sc[tg] = (pos >= lo_s && pos < hi_s) ? x[0] * p.scale_log2 : -CUDART_INF_F;
            }
            // Lazy running maximum of row rs (its 4 lanes), as in the tensor-core path.
            float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            if (__any_sync(0xffffffffu, mx > m_s + kLazyLog2)) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(m_s, mx);
                const float al = mn == -CUDART_INF_F ? 1.f : exp2f(m_s - mn);
                m_s = mn;
                l_s *= al;
#pragma unroll
                for (int n = 0; n < C::kRows; ++n) {
                    const float a = __shfl_sync(0xffffffffu, al, n * 4);
#pragma unroll
                    for (int e = 0; e < E; ++e) acs[n][e] *= a;
                }
            }
            const float mu = m_s == -CUDART_INF_F ? 0.f : m_s;
#pragma unroll
            for (int tg = 0; tg < 4; ++tg) {
                const float pw = exp2f(sc[tg] - mu);
                l_s += pw;
                sP[rs * C::kPLd + tg * 4 + (lane & 3)] = pw;
            }
            __syncwarp();
            // O += P V over this lane's columns.
            const unsigned char *sv = st + C::kTileBytes;
#pragma unroll
            for (int tg = 0; tg < 4; ++tg) {
                float4 pr[C::kRows];
#pragma unroll
                for (int n = 0; n < C::kRows; ++n)
                    pr[n] = *reinterpret_cast<const float4 *>(sP + n * C::kPLd + tg * 4);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float vf[E];
                    tile_load<T, E>(vf, sv, tg * 4 + u, lane * E);
#pragma unroll
                    for (int n = 0; n < C::kRows; ++n) {
                        const float pw = u == 0 ? pr[n].x : u == 1 ? pr[n].y : u == 2 ? pr[n].z : pr[n].w;
#pragma unroll
                        for (int e = 0; e < E; ++e) acs[n][e] = fmaf(pw, vf[e], acs[n][e]);
                    }
                }
            }
        } else {
            // S^T = K . Q^T, two accumulation chains over head_dim.
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    #pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                unsigned a[4];
                ldmatrix_x4(a, st + swz(krow, 2 * kk + kchk));
                if (kk & 1) mma_bf16_16816(sb, a, qb[kk][0], qb[kk][1]);
                else mma_bf16_16816(sa, a, qb[kk][0], qb[kk][1]);
            }
            // This thread holds keys gq, gq + 8 of rows 2tq, 2tq + 1: mask, online softmax (base 2).
            const int p0 = pos0 + gq, p1 = p0 + 8;
            float v[4];
            v[0] = (p0 >= lo_r[0] && p0 < hi_r[0]) ? (sa[0] + sb[0]) * p.scale_log2 : -CUDART_INF_F;
            v[1] = (p0 >= lo_r[1] && p0 < hi_r[1]) ? (sa[1] + sb[1]) * p.scale_log2 : -CUDART_INF_F;
            v[2] = (p1 >= lo_r[0] && p1 < hi_r[0]) ? (sa[2] + sb[2]) * p.scale_log2 : -CUDART_INF_F;
            v[3] = (p1 >= lo_r[1] && p1 < hi_r[1]) ? (sa[3] + sb[3]) * p.scale_log2 : -CUDART_INF_F;
            // Lazy running maximum: a row's reference max moves only when a score
            // exceeds it by more than kLazyLog2, so the weights stay below
            // 2^kLazyLog2 and the common page needs no cross-lane reduction and
            // no rescale.  (m, l, acc) stay consistent with whatever reference
            // the row holds, which is all the merges need.
            float mx0 = fmaxf(v[0], v[2]), mx1 = fmaxf(v[1], v[3]);
            if (__any_sync(0xffffffffu, mx0 > m_r[0] + kLazyLog2 || mx1 > m_r[1] + kLazyLog2)) {
    #pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);
                const float al0 = mn0 == -CUDART_INF_F ? 1.f : exp2f(m_r[0] - mn0);
                const float al1 = mn1 == -CUDART_INF_F ? 1.f : exp2f(m_r[1] - mn1);
                m_r[0] = mn0;
                m_r[1] = mn1;
                l_r[0] *= al0;
                l_r[1] *= al1;
    #pragma unroll
                for (int dt = 0; dt < KT; ++dt) {
                    acc[dt][0] *= al0; acc[dt][1] *= al1;
                    acc[dt][2] *= al0; acc[dt][3] *= al1;
                }
            }
            const float mu0 = m_r[0] == -CUDART_INF_F ? 0.f : m_r[0], mu1 = m_r[1] == -CUDART_INF_F ? 0.f : m_r[1];
            const float p00 = exp2f(v[0] - mu0), p01 = exp2f(v[1] - mu1);
            const float p10 = exp2f(v[2] - mu0), p11 = exp2f(v[3] - mu1);
            l_r[0] += p00 + p10;
            l_r[1] += p01 + p11;
            // P^T as B fragments: transpose the (key x row) halves in registers.
            const unsigned b0 = movmatrix_trans(pack_bf16x2(p00, p01));
            const unsigned b1 = movmatrix_trans(pack_bf16x2(p10, p11));
            // O^T += V^T . P^T, one independent MMA per 16 columns of head_dim.
            const unsigned char *sv = st + C::kTileBytes;
    #pragma unroll
            for (int dt = 0; dt < KT; ++dt) {
                unsigned a[4];
                ldmatrix_x4_trans(a, sv + swz(vrow, 2 * dt + vchk));
                mma_bf16_16816(acc[dt], a, b0, b1);
            }
        }
        __syncwarp();  // every lane is done with the stage
        if (j + NST < n_mine) issue(j + NST);
    }
    if (timed_out && lane == 0) {
        // Give copies still in flight a bounded chance to land before the
        // stage memory is reused.
        #pragma unroll 1
        for (int j = max(0, n_mine - NST); j < n_mine; ++j)
            #pragma unroll 1
            for (int it = 0; it < kWaitProbes && !mbar_try_wait(wbars + (j % NST), (j / NST) & 1); ++it) {
            }
    }
    if ((bad || timed_out) && lane == 0) atomicOr(sFlag, (bad ? 1 : 0) | (timed_out ? 2 : 0));

    // ---- the warp's partial, written over its own stages: O^T as [row][col], max and sum per row
    if constexpr (SIMT) {
        l_s += __shfl_xor_sync(0xffffffffu, l_s, 1);
        l_s += __shfl_xor_sync(0xffffffffu, l_s, 2);
        float *part = reinterpret_cast<float *>(wstage);
        float *pm = part + C::kRows * LD, *pl = pm + C::kRows;
#pragma unroll
        for (int n = 0; n < C::kRows; ++n)
#pragma unroll
            for (int e = 0; e < E; ++e) part[n * LD + lane * E + e] = acs[n][e];
        if ((lane & 3) == 0) {
            pm[rs] = m_s;
            pl[rs] = l_s;
        }
    } else {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], o);
            l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], o);
        }
        float *part = reinterpret_cast<float *>(wstage);
        float *pm = part + C::kRows * LD, *pl = pm + C::kRows;
#pragma unroll
        for (int dt = 0; dt < KT; ++dt) {
            const int d = dt * 16 + gq;
            part[(2 * tq) * LD + d] = acc[dt][0];
            part[(2 * tq + 1) * LD + d] = acc[dt][1];
            part[(2 * tq) * LD + d + 8] = acc[dt][2];
            part[(2 * tq + 1) * LD + d + 8] = acc[dt][3];
        }
        if (gq == 0) {
            pm[2 * tq] = m_r[0];
            pm[2 * tq + 1] = m_r[1];
            pl[2 * tq] = l_r[0];
            pl[2 * tq + 1] = l_r[1];
        }
    }
    __syncthreads();
    const int flags = sFlag[0];
    if (tid == 0 && flags) atomicOr(p.err, ((flags & 1) ? PKV_ERR_BLOCK : 0u) | ((flags & 2) ? PKV_ERR_TIMEOUT : 0u));

    auto out_row = [&](int n) {
        const int i = n / p.G, jh = n - i * p.G;
        return ((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh;
    };
    auto part_of = [&](int k) { return reinterpret_cast<const float *>(pipe + (size_t)k * NST * C::kStageBytes); };

    cg::cluster_group cluster = cg::this_cluster();
    // Output columns each CTA of the cluster finishes: a power of two, so the
    // last CTAs may get none.
    int lg = 0;
    while ((1 << lg) * ncl < DP) ++lg;
    const int per = 1 << lg;
    const int unit = blockIdx.z * gridDim.y + blockIdx.y;
    if (ncl > 1 && !gm) {
        // Every CTA of the cluster has started (the arrive at the top), so
        // peers' shared memory may be written from here on.
        asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
        if (tid < ncl) *cluster.map_shared_rank(sAllF + rank, tid) = flags;
    }
    // ---- merge the warps: thread = (row n, block of CB columns); the
    // block goes whole to the CTA that finishes those columns (per >= CB).
    constexpr int CB = DP / 16;
    {
        const int n = tid >> 4, cq = tid & 15, d0 = cq * CB;
        if (n < rows_unit) {
            float mk[KW], M = -CUDART_INF_F;
#pragma unroll
            for (int k = 0; k < KW; ++k) {
                mk[k] = part_of(k)[C::kRows * LD + n];
                M = fmaxf(M, mk[k]);
            }
            float w[KW], L = 0.f;
#pragma unroll
            for (int k = 0; k < KW; ++k) {
                // a warp with no visible key has weight 0 and a zero accumulator
                w[k] = (M == -CUDART_INF_F || mk[k] == -CUDART_INF_F) ? 0.f : exp2f(mk[k] - M);
                L = fmaf(w[k], part_of(k)[C::kRows * LD + C::kRows + n], L);
            }
            float o[CB];
#pragma unroll
            for (int e = 0; e < CB; ++e) o[e] = 0.f;
#pragma unroll
            for (int k = 0; k < KW; ++k) {
#pragma unroll
                for (int e = 0; e < CB; e += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(part_of(k) + n * LD + d0 + e);
                    o[e] = fmaf(w[k], v.x, o[e]);
                    o[e + 1] = fmaf(w[k], v.y, o[e + 1]);
                    o[e + 2] = fmaf(w[k], v.z, o[e + 2]);
                    o[e + 3] = fmaf(w[k], v.w, o[e + 3]);
                }
            }
            if (ncl == 1) {
                const long long orow = out_row(n);
                const bool zero = flags || !(L > 0.f);
                const float inv = zero ? 0.f : 1.f / L;
#pragma unroll
                for (int e = 0; e < CB; ++e)
                    if (d0 + e < p.D) p.out[orow * p.D + d0 + e] = zero ? 0.f : o[e] * inv;  // o may be NaN when poisoned
                if (cq == 0 && p.lse) p.lse[orow] = zero ? -CUDART_INF_F : (M + log2f(L)) * kLn2;
            } else if (gm) {
                float *dst = p.ws_part + (((size_t)unit * ncta + rank) * C::kRows + n) * DP + d0;
#pragma unroll
                for (int e = 0; e < CB; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                if (cq == 0) p.ws_stat[((size_t)unit * ncta + rank) * C::kRows + n] = make_float2(M, L);
            } else {
                float *dst = cluster.map_shared_rank(sRecv + ((rank * C::kRows + n) << lg) + (d0 & (per - 1)), d0 >> lg);
#pragma unroll
                for (int e = 0; e < CB; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                if (cq < ncl) *cluster.map_shared_rank(sStat + rank * C::kRows + n, cq) = make_float2(M, L);
            }
        }
    }
    if (ncl == 1) return;

    if (gm) {
        // ---- the last of the range's CTAs to arrive merges every partial
        if (tid == 0) p.ws_flag[(size_t)unit * ncta + rank] = flags;
        __threadfence();  // this CTA's partial is visible before its arrival is counted
        __syncthreads();
        if (tid == 0) sFlag[20] = atomicAdd(p.ws_count + unit, 1) == active - 1;
        __syncthreads();
        if (!sFlag[20]) return;
        __threadfence();
        const float *wp = p.ws_part + (size_t)unit * ncta * C::kRows * DP;
        const float2 *wst = p.ws_stat + (size_t)unit * ncta * C::kRows;
        // Issue every global read at once: the statistics, the flags and the
        // async copies staging the partials' rows in shared memory (the idle
        // stages, as many partials per batch as fit).
        const int n = tid >> 4, c16 = tid & 15;  // thread = (row n, sources c16, c16 + 16, ...)
        float2 st[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = c16 + 16 * i;
            st[i] = (c < active && n < rows_unit) ? __ldcg(wst + (size_t)c * C::kRows + n)
                                                  : make_float2(-CUDART_INF_F, 0.f);
        }
        const int fl = tid < active ? __ldcg(p.ws_flag + (size_t)unit * ncta + tid) : 0;
        float *stg = reinterpret_cast<float *>(pipe);
        const int q4 = DP / 4, per_c = rows_unit * q4;  // 16-byte chunks per partial
        const int cap = (int)(C::kPipeBytes / ((size_t)rows_unit * DP * 4));
        auto stage_batch = [&](int c0, int nc) {
            #pragma unroll 1
            for (int x = tid; x < nc * per_c; x += NT) {
                const int c = x / per_c, r = x - c * per_c, nn = r / q4, ch = r - nn * q4;
                const unsigned dst = smem_u32(stg + ((size_t)c * rows_unit + nn) * DP + ch * 4);
                const float *src = wp + ((size_t)(c0 + c) * C::kRows + nn) * DP + ch * 4;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
            }
            asm volatile("cp.async.commit_group;\n" ::: "memory");
        };
        int c0 = 0, nc = min(cap, active);
        stage_batch(0, nc);
        const int poison = __syncthreads_or(fl != 0);
        float *sWg = sRecv;  // [8][64] normalised weights (the cluster's receive buffer is unused here)
        {   // max and sum by 16-lane shuffles
            float M = -CUDART_INF_F;
#pragma unroll
            for (int i = 0; i < 4; ++i) M = fmaxf(M, st[i].x);
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float w[4], W = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // A zero weight must not touch its partial: a poisoned one may hold NaN.
                w[i] = (M == -CUDART_INF_F || st[i].x == -CUDART_INF_F) ? 0.f : exp2f(st[i].x - M);
                W = fmaf(w[i], st[i].y, W);
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
            const bool zero = poison || !(W > 0.f);
            const float inv = zero ? 0.f : 1.f / W;
            if (n < C::kRows)
#pragma unroll
                for (int i = 0; i < 4; ++i) sWg[n * 64 + c16 + 16 * i] = zero ? 0.f : w[i] * inv;  // w may be NaN when poisoned
            if (c16 == 0 && n < rows_unit && p.lse) p.lse[out_row(n)] = zero ? -CUDART_INF_F : (M + log2f(W)) * kLn2;
        }
        constexpr int EPT = (C::kRows * DP + NT - 1) / NT;  // elements per thread at most
        float acc[EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) acc[i] = 0.f;
        #pragma unroll 1
        for (;;) {
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
            __syncthreads();  // the batch and the weights are in shared memory
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int e = tid + i * NT;
                if (e < rows_unit * DP) {
                    const int nn = e / DP, d = e - nn * DP;
                    float o = acc[i];
                    #pragma unroll 4
                    for (int c = 0; c < nc; ++c) {
                        const float w = sWg[nn * 64 + c0 + c];
                        o += w != 0.f ? w * stg[((size_t)c * rows_unit + nn) * DP + d] : 0.f;
                    }
                    acc[i] = o;
                }
            }
            c0 += nc;
            if (c0 >= active) break;
            nc = min(cap, active - c0);
            __syncthreads();  // the batch is consumed
            stage_batch(c0, nc);
        }
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            const int e = tid + i * NT;
            if (e < rows_unit * DP) {
                const int nn = e / DP, d = e - nn * DP;
                if (d < p.D) p.out[out_row(nn) * p.D + d] = acc[i];
            }
        }
        if (tid == 0) p.ws_count[unit] = 0;  // ready for the next call
        return;
    }

    // ---- merge the cluster's partials of this CTA's columns
    cluster.sync();  // publishes every CTA's pushed partials
    int poison = 0;
#pragma unroll
    for (int c = 0; c < 16; ++c) poison |= c < ncl ? sAllF[c] : 0;
    // thread = (row n, source CTA c): normalised weight by 16-lane shuffles
    const int n = tid >> 4, c = tid & 15;
    float wn;
    {
        const float2 st = (c < ncl && n < rows_unit) ? sStat[c * C::kRows + n] : make_float2(-CUDART_INF_F, 0.f);
        float M = st.x;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        // A zero weight must not touch its partial: a poisoned one may hold NaN.
        const float w = (M == -CUDART_INF_F || st.x == -CUDART_INF_F) ? 0.f : exp2f(st.x - M);
        float W = w * st.y;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
        const bool zero = poison || !(W > 0.f);
        wn = zero ? 0.f : w / W;
        if (c == 0 && n < rows_unit && rank == 0 && p.lse)
            p.lse[out_row(n)] = zero ? -CUDART_INF_F : (M + log2f(W)) * kLn2;
    }
    const int d_base = rank << lg;
    if (per == 8 || per == 16) {
        // Each thread weighs its source's slice; a reduce-scatter over the
        // 16 sources leaves each lane one column's sum.
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = 0.f;
        if (c < ncl && n < rows_unit && wn != 0.f && d_base < DP) {
            const float *src = sRecv + ((c * C::kRows + n) << lg);
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                if (e < per) {
                    const float4 v = *reinterpret_cast<const float4 *>(src + e);
                    x[e] = wn * v.x; x[e + 1] = wn * v.y; x[e + 2] = wn * v.z; x[e + 3] = wn * v.w;
                }
            }
        }
        // halving steps over lane bits 8, 4, 2 (and 1 for 16 columns): keep the
        // half this lane's bit selects, add the partner's copy of it
        int idx = 0;
        if (per == 16) {
            idx += rs_halve<8>(x, c, 8);
            idx += rs_halve<4>(x, c, 4);
            idx += rs_halve<2>(x, c, 2);
            idx += rs_halve<1>(x, c, 1);
        } else {
            idx += rs_halve<4>(x, c, 8);
            idx += rs_halve<2>(x, c, 4);
            idx += rs_halve<1>(x, c, 2);
            x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
        }
        const int d = d_base + idx;
        if (n < rows_unit && (per == 16 || (c & 1) == 0) && d < p.D) p.out[out_row(n) * p.D + d] = x[0];
        return;
    }
    // wider slices (small clusters): weights through shared memory
    if (tid < C::kRows * 16) sWn[n * 16 + c] = wn;
    __syncthreads();
    #pragma unroll 1
    for (int e = tid; e < (rows_unit << lg); e += NT) {
        const int nn = e >> lg, dl = e & (per - 1), d = d_base + dl;
        if (d >= DP) continue;
        float o = 0.f;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
            if (cc < ncl) {
                const float w = sWn[nn * 16 + cc];
                const float v = sRecv[((cc * C::kRows + nn) << lg) + dl];
                o += w != 0.f ? w * v : 0.f;
            }
        }
        if (d < p.D) p.out[out_row(nn) * p.D + d] = o;
    }
}

}  // namespace pkv
