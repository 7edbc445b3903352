// Tensor-core (tcgen05) attention tile for wide query groups (sm_103a).
//
// The row class of speculative verify and chunked steps: one (segment, kv
// head) carries G * q_len query rows, up to 128 (GQA 64:8 with 16 draft
// tokens), so the products Q K^T and P V are real contractions.  They run on
// the 5th-generation tensor cores: one thread issues tcgen05.mma (bf16 in,
// fp32 accumulate) with both operands in shared memory, S and O live in
// tensor memory (TMEM), and the softmax threads move S out of and P into
// shared memory.  Same launch shape, key split and semantics as attend_kernel
// (grid (C, kv_heads, segments); the C CTAs of a range are one cluster and
// merge through distributed shared memory with merge_rows).
//
// Per CTA (192 threads):
//   warps 0-3   softmax: thread t owns query row t (TMEM lane t); after the
//               loop the epilogue reads O back and hands it to the merge;
//   warp 4      TMA issue: K and V of 4 pages (64 keys) per stage, each page
//               as two 64-column boxes so a stage is a K-major tile of 64
//               keys (128-byte swizzle) for Q K^T and an MN-major tile for
//               P V;
//   warp 5      MMA: waits for a stage, fixes its edge pages (stale rows
//               zeroed, this step's rows taken from k_new / v_new and
//               appended to the cache), issues S(j) = Q K_j^T (M = 128, N =
//               64, 8 steps over head_dim) and, once P(j-1) is written,
//               O += P(j-1) V(j-1) (M = 128, N = 128, 4 steps of 16 keys);
//               also owns the TMEM allocation.
// TMEM: S double-buffered in columns 0-63 / 64-127, O in 128-255.
//
// The online softmax keeps one row per thread (no cross-lane reduction) and
// raises a row's reference maximum lazily: only when a score exceeds it by
// more than 2^8, and then O is rescaled in TMEM after the previous P V has
// landed.  Every wait is bounded; a timeout poisons the CTA's output
// (PKV_ERR_TIMEOUT), drains what is in flight and frees TMEM.
//
// Semantics follow the segment-table attention of ExecuTorch PR #24072
// (triton::sdpa_varlen) over the paged layout of vLLM-Omni's SenseNova-U1
// PagedDecodeCache, exactly as attend_kernel.
#pragma once

#include "attend.cuh"

namespace pkv {

template <int NS_>
struct VfyCfg {
    using T = __nv_bfloat16;
    static constexpr int DP = 128;                  // head_dim (this tile needs exactly 128)
    static constexpr int NS = NS_;                  // stages of 4 pages
    static constexpr int kRows = 128;               // query rows per CTA = TMEM lanes
    static constexpr int kThreads = 192;
    static constexpr int kPages = 4;                // pages per stage (N = 64 keys)
    static constexpr unsigned kQBytes = kRows * DP * 2;            // two 64-column halves
    static constexpr unsigned kHalf = kPages * kPage * 128;        // 64 keys x 128 B
    static constexpr unsigned kStageBytes = 4 * kHalf;             // K halves, then V halves
    static constexpr unsigned kPBytes = kRows * 128;               // 128 rows x 64 keys bf16
    static constexpr size_t kLoopBytes = (size_t)NS * kStageBytes + 2 * kPBytes;
    // after the loop the stages and P buffers hold the partial rows and their (max, sum)
    static constexpr size_t kMergeBytes = (size_t)kRows * DP * 4 + 2 * kRows * 4;
    static constexpr size_t kBodyBytes = kLoopBytes > kMergeBytes ? kLoopBytes : kMergeBytes;
    // per row: pm, pl, lse, the cluster merge's gathered maxima / sums (16 CTAs each)
    static constexpr size_t kRowBytes = (size_t)kRows * (3 + 16 + 16) * 4;
    static constexpr int kBars = 2 * NS + 9;  // full, empty [NS]; s_full, s_free, p_full, pv_done [2]; drain
    static constexpr size_t kMiscBytes = (size_t)kBars * 8 + 16 + 32 * 4 + (size_t)kThreads * 4;
    static constexpr size_t kSmemBytes = 1024 + kQBytes + kBodyBytes + kRowBytes + kMiscBytes;
    static constexpr int kTmemCols = 256;
    static_assert(kSmemBytes <= 232448, "exceeds the per-CTA shared memory limit");
    static_assert(kQBytes % 1024 == 0 && kStageBytes % 1024 == 0 && kPBytes % 1024 == 0,
                  "operand tiles start on 1024-byte swizzle atoms");
};

// ---------------------------------------------------------------- tcgen05 helpers

// Shared-memory matrix descriptor: 128-byte swizzle, start / leading /
// stride byte offsets in 16-byte units, descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, A K-major, B
// K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(unsigned d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(unsigned taddr, float (&v)[32]) {
    unsigned r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(unsigned taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Nanoseconds since an arbitrary origin (the global timer).
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
    return t;
}
// Wall-clock bound of one wait in this kernel: a wait that runs past it
// poisons the CTA (PKV_ERR_TIMEOUT) instead of hanging the launch.
constexpr unsigned long long kWaitNs = 20ull * 1000 * 1000;

// Time-bounded wait for a barrier phase (one thread; no abort check).
__device__ __forceinline__ bool mbar_wait_ns(uint64_t *bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    #pragma unroll 1
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}

// Offset of 16-byte chunk `c` (0..7) of row `r` in a tile of 128-byte rows
// loaded with 128-byte swizzling (rows grouped in 1024-byte atoms).
__device__ __forceinline__ unsigned swz_row(int r, int c) { return (unsigned)(r * 128 + ((c ^ (r & 7)) << 4)); }

// ---------------------------------------------------------------- the kernel

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1) verify_kernel(const __grid_constant__ AttendParams p) {
    using T = __nv_bfloat16;
    constexpr int DP = C::DP, NS = C::NS, R = C::kRows, NT = C::kThreads, PG = C::kPages;
    constexpr int EPC = 8;  // bf16 per 16-byte chunk

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sQ = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *body = sQ + C::kQBytes;                  // stages, then the two P buffers
    unsigned char *sP = body + (size_t)NS * C::kStageBytes;
    float *sMo = reinterpret_cast<float *>(body);           // after the loop: [R][DP] partial rows
    float *sMm = sMo + (size_t)R * DP;                      // [R] base-2 max
    float *sMl = sMm + R;                                   // [R] sum
    float *rows = reinterpret_cast<float *>(body + C::kBodyBytes);
    float *sPm = rows, *sPl = sPm + R, *sLse = sPl + R;
    float *sAllM = sLse + R, *sAllL = sAllM + R * 16;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sAllL + R * 16);
    uint64_t *full = bars, *empty = bars + NS;              // [NS] each
    uint64_t *s_full = bars + 2 * NS, *s_free = s_full + 2, *p_full = s_free + 2, *pv_done = p_full + 2;
    uint64_t *drain = pv_done + 2;
    unsigned *tslot = reinterpret_cast<unsigned *>(bars + C::kBars);
    volatile int *sAbort = reinterpret_cast<volatile int *>(tslot + 1);
    int *sFlag = reinterpret_cast<int *>(tslot + 4);        // [0] own flags: 1 bad page, 2 timeout
    int *sAllF = sFlag + 1;                                 // [16] flags of the cluster
    int *sCov = sFlag + 32;                                 // [NT] coverage flags

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = blockIdx.x, ncta = gridDim.x;
    const int g = blockIdx.y / p.row_tiles, rt = blockIdx.y - g * p.row_tiles;
    const int s = blockIdx.z;
    const bool cov_cta = grid_cta_index() < coverage_slices(p, NT);
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
    const int rows_unit = fault ? 0 : sg.ql * p.G;
    const int row0 = rt * R;
    if (fault || row0 >= rows_unit) {  // uniform across the cluster
        pdl_wait();
        pdl_trigger();
        if (fault && rank == 0 && rt == 0) {
            if (tid == 0) atomicOr(p.err, fault);
            zero_segment_rows(p, sg, g, NT);
        }
        if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
        return;
    }
    const int rows_here = min(R, rows_unit - row0);
    const int kend = sg.kend;
    const int new_start = kend - sg.ql;
    const int first = first_valid_of(p.first_valid, sg.col);
    const int lo_u = segment_key_lo(new_start, kend, p.causal, p.window, first);
    const int pb_begin = lo_u / kPage;
    const int pb_end = (kend + kPage - 1) / kPage;
    const int nblk = pb_end - pb_begin;
    const int bps = (nblk + ncta - 1) / ncta;
    const int active = (nblk + bps - 1) / bps;
    const int cb0 = pb_begin + rank * bps;
    const int nb = rank < active ? min(cb0 + bps, pb_end) - cb0 : 0;
    const int ngr = (nb + PG - 1) / PG;                     // stages (groups of 4 pages) of this CTA
    const int lo_pos = cb0 * kPage, hi_pos = (cb0 + nb) * kPage;

    const T *knew = reinterpret_cast<const T *>(p.k_new);
    const T *vnew = reinterpret_cast<const T *>(p.v_new);
    const bool fused = knew != nullptr;
    const int dchunks = p.D / EPC;
    const int *bt_row = p.block_table + (long long)sg.col * p.mbps;
    const bool has_new = fused && rt == 0 && nb > 0 && new_start < hi_pos && kend > lo_pos;

    if (tid == 0) {
        #pragma unroll 1
        for (int i = 0; i < C::kBars; ++i) mbar_init(bars + i, (i >= 2 * NS + 2 && i < 2 * NS + 6) ? 4 : 1);
        fence_barrier_init();
        sFlag[0] = 0;
        *sAbort = 0;
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tmem = *tslot;

    // Append validity, all or nothing over the segment's new rows (the block
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

    // Bounded wait of a whole warp on one phase (every lane observes it); gives
    // up at once when another role has already timed out.  Warp-uniform:
    // false on a timeout (which raises the abort for the other roles).
    auto wait_bar = [&](uint64_t *bar, unsigned parity) -> bool {
        bool ok = mbar_try_wait(bar, parity);
        if (!ok) {
            const unsigned long long t0 = global_ns();
            #pragma unroll 1
            while (!ok) {
                ok = mbar_try_wait(bar, parity);
                if (!ok && (*sAbort || global_ns() - t0 > kWaitNs)) break;
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) *sAbort = 1;
        return ok;
    };

    // ---- TMA issue (warp 4): group j = pages cb0 + 4j .. cb0 + 4j + 3
    int id_reg = -1, id_window = -1, issued = 0;
    bool bad = false;
    auto load_ids = [&](int li0) {
        id_window = li0 & ~31;
        const int li = id_window + lane;
        id_reg = li < nb ? bt_row[table_page(cb0 + li, p.ring_rows)] : -1;
    };
    auto issue = [&](int j) {
        const int st = j % NS;
        unsigned char *stage = body + (size_t)st * C::kStageBytes;
        int ok_pages = 0;
        unsigned okmask = 0;
#pragma unroll
        for (int u = 0; u < PG; ++u) {
            const int li = j * PG + u;
            if (li < nb) {
                if ((li & ~31) != id_window) load_ids(li);
                const int bid = __shfl_sync(0xffffffffu, id_reg, li & 31);
                const bool ok = bid >= 0 && (long long)bid < p.num_blocks;
                bad |= !ok;
                if (ok) { okmask |= 1u << u; ++ok_pages; }
            }
        }
        if (lane == 0) {
            uint64_t *bar = full + st;
            fence_proxy_async();
            if (ok_pages) {
                mbar_expect_tx(bar, (unsigned)ok_pages * 4u * 2048u);
            } else {
                mbar_arrive(bar);
            }
        }
#pragma unroll
        for (int u = 0; u < PG; ++u) {
            const int li = j * PG + u;
            const int bid = li < nb ? __shfl_sync(0xffffffffu, id_reg, li & 31) : -1;
            if (lane == 0 && ((okmask >> u) & 1u)) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tma_load_4d(stage + h * C::kHalf + u * 2048, &p.tmap_k, full + st, h * 64, g, 0, bid);
                    tma_load_4d(stage + 2 * C::kHalf + h * C::kHalf + u * 2048, &p.tmap_v, full + st, h * 64, g, 0,
                                bid);
                }
            }
        }
    };
    // Pages wholly below new_start may be fetched before the dependency wait;
    // in the fused call every page may (this step's rows are replaced after it).
    auto early_ok = [&](int j) { return fused || (cb0 + min(j * PG + PG, nb)) * kPage <= new_start; };

    if (warp == 4) {
        load_ids(0);
        #pragma unroll 1
        for (; issued < NS && issued < ngr; ++issued) {
            if (!early_ok(issued)) break;
            issue(issued);
        }
        // The first 32 pages that are not in flight go to L2 now, so their
        // HBM traffic overlaps the previous kernel's tail: lane l holds the
        // id of page l.
        if (id_window == 0 && lane >= issued * PG && lane < nb && id_reg >= 0 && (long long)id_reg < p.num_blocks) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tma_prefetch_l2_4d(&p.tmap_k, h * 64, g, 0, id_reg);
                tma_prefetch_l2_4d(&p.tmap_v, h * 64, g, 0, id_reg);
            }
        }
    }
    // Warm L2 with the rows read right after the wait: this tile's queries
    // and, in the fused call, this step's K/V rows.
    {
        const int nq = rows_here * 2;
        #pragma unroll 1
        for (int c = tid; c < nq; c += NT) {
            const int r = c >> 1, ur = row0 + r, i = ur / p.G, jh = ur - i * p.G;
            const T *src = reinterpret_cast<const T *>(p.q) + (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D;
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + (c & 1) * 128));
        }
        if (has_new) {
            const int a = max(new_start, lo_pos), e = min(kend, hi_pos);
            #pragma unroll 1
            for (int c = tid; c < (e - a) * 4; c += NT) {
                const int row = c >> 2, kv = (c >> 1) & 1;
                const T *src = (kv ? vnew : knew) + (((long long)sg.q0 + (a + row - new_start)) * p.Hkv + g) * p.D;
                asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + (c & 1) * 128));
            }
        }
    }

    pdl_wait();
    pdl_trigger();

    // ---- queries: 128 rows x 128 columns, K-major, 128-byte swizzle, two
    // 64-column halves; rows past the group are zero.
    {
        constexpr int kIt = (R * 16 + NT - 1) / NT;
        uint4 qv[kIt];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int c = tid + it * NT, r = c >> 4, ch = c & 15, ur = row0 + r;
            qv[it] = make_uint4(0u, 0u, 0u, 0u);
            if (c < R * 16 && r < rows_here && ch < dchunks) {
                const int i = ur / p.G, jh = ur - i * p.G;
                qv[it] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.q) +
                                                          (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D +
                                                          ch * EPC);
            }
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int c = tid + it * NT, r = c >> 4, ch = c & 15;
            if (c < R * 16)
                *reinterpret_cast<uint4 *>(sQ + (ch >> 3) * (R * 128) + swz_row(r, ch & 7)) = qv[it];
        }
    }
    fence_proxy_async();
    if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
    if (warp == 4) {
        #pragma unroll 1
        for (; issued < NS && issued < ngr; ++issued) issue(issued);
    }
    __syncthreads();  // queries staged

    bool timed_out = false;
    const unsigned lane_off = (unsigned)(32 * (warp & 3)) << 16;

    if (warp == 4) {
        // ---------------- TMA issue: refill each stage once its P V has completed
        #pragma unroll 1
        for (int j = issued; j < ngr; ++j) {
            if (!wait_bar(empty + (j % NS), ((j / NS) - 1) & 1)) { timed_out = true; break; }
            issue(j);
            issued = j + 1;
        }
        // Drain: every issued stage has landed before its memory is reused or freed.
        if (lane == 0) {
            #pragma unroll 1
            for (int j = max(0, issued - NS); j < issued; ++j)
                if (!mbar_wait_ns(full + (j % NS), (j / NS) & 1)) break;
        }
    } else if (warp == 5) {
        // ---------------- edge-page fix-up and MMA issue
        const uint32_t id_s = umma_idesc_bf16(128, 64, 0), id_o = umma_idesc_bf16(128, 128, 1);
        const unsigned q_addr = smem_u32(sQ);
        // Stale rows zeroed, this step's rows written into the stage (and the cache).
        auto fix_group = [&](int j, unsigned char *stage) {
            bool any = false;
#pragma unroll 1
            for (int u = 0; u < PG; ++u) {
                const int li = j * PG + u;
                const int pos0 = (cb0 + li) * kPage;
                int zlo, zhi, na;
                if (li < nb) {
                    zlo = min(max(lo_u - pos0, 0), kPage);
                    zhi = min(max(kend - pos0, 0), kPage);
                    na = fused ? min(max(new_start - pos0, 0), kPage) : zhi;
                } else {
                    zlo = kPage; zhi = kPage; na = kPage;  // no page: all 16 rows zeroed
                }
                if (!(zlo > 0 || zhi < kPage || na < zhi)) continue;
                any = true;
                const int nz = (zlo + kPage - zhi) * 16;  // (row, chunk) pairs of stale rows, K and V
                #pragma unroll 1
                for (int c = lane; c < 2 * nz; c += 32) {
                    const int kv = c >= nz, rem = c - kv * nz, o0 = rem >> 4, ch = rem & 15;
                    const int o = o0 < zlo ? o0 : zhi + (o0 - zlo);
                    *reinterpret_cast<uint4 *>(stage + kv * 2 * C::kHalf + (ch >> 3) * C::kHalf + u * 2048 +
                                               swz_row(o, ch & 7)) = make_uint4(0u, 0u, 0u, 0u);
                }
                const int nn = (zhi - na) * 16;
                if (nn > 0) {
                    const long long bpage = app_ok ? (long long)bt_row[table_page(pos0 / kPage, p.ring_rows)] : 0;
                    const int ring_base = p.ring_rows ? pos0 % p.ring_rows : pos0;
                    #pragma unroll 1
                    for (int c = lane; c < 2 * nn; c += 32) {
                        const int kv = c >= nn, rem = c - kv * nn, r0 = rem >> 4, ch = rem & 15;
                        const int o = na + r0;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (ch < dchunks) {
                            v = *reinterpret_cast<const uint4 *>(
                                (kv ? vnew : knew) + (((long long)sg.q0 + (pos0 + o - new_start)) * p.Hkv + g) * p.D +
                                ch * EPC);
                            if (app_ok) {
                                const long long slot = bpage * kPage + (ring_base + o) % kPage;
                                *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(kv ? p.v_pool_w : p.k_pool_w) +
                                                           (slot * p.Hkv + g) * p.D + ch * EPC) = v;
                            }
                        }
                        *reinterpret_cast<uint4 *>(stage + kv * 2 * C::kHalf + (ch >> 3) * C::kHalf + u * 2048 +
                                                   swz_row(o, ch & 7)) = v;
                    }
                }
            }
            if (any) fence_proxy_async();  // generic writes before the tensor core reads the stage
            __syncwarp();
        };
        auto issue_pv = [&](int i) {
            const int b = i & 1, st = i % NS;
            if (!wait_bar(p_full + b, (i >> 1) & 1)) return false;
            tc_fence_after();
            if (lane == 0) {
                const unsigned p_addr = smem_u32(sP + b * C::kPBytes);
                const unsigned v_addr = smem_u32(body + (size_t)st * C::kStageBytes + 2 * C::kHalf);
#pragma unroll
                for (int u = 0; u < PG; ++u)
                    umma_bf16(tmem + 128, umma_desc(p_addr + u * 32, 16, 1024),
                              umma_desc(v_addr + u * 2048, C::kHalf, 1024), id_o, (i > 0 || u > 0) ? 1 : 0);
                umma_commit(empty + st);
                umma_commit(pv_done + b);
            }
            __syncwarp();
            return true;
        };
        #pragma unroll 1
        for (int j = 0; j < ngr && !timed_out; ++j) {
            const int st = j % NS, b = j & 1;
            unsigned char *stage = body + (size_t)st * C::kStageBytes;
            if (!wait_bar(full + st, (j / NS) & 1)) { timed_out = true; break; }
            fix_group(j, stage);
            if (j >= 2 && !wait_bar(s_free + b, ((j - 2) >> 1) & 1)) { timed_out = true; break; }
            tc_fence_after();
            if (lane == 0) {
                const unsigned k_addr = smem_u32(stage);
#pragma unroll
                for (int k = 0; k < DP / 16; ++k)
                    umma_bf16(tmem + b * 64, umma_desc(q_addr + (k >> 2) * (R * 128) + (k & 3) * 32, 16, 1024),
                              umma_desc(k_addr + (k >> 2) * C::kHalf + (k & 3) * 32, 16, 1024), id_s, k > 0 ? 1 : 0);
                umma_commit(s_full + b);
            }
            __syncwarp();
            if (j >= 1 && !issue_pv(j - 1)) { timed_out = true; break; }
        }
        if (!timed_out && ngr > 0 && !issue_pv(ngr - 1)) timed_out = true;
        // Drain: every MMA this thread issued has completed before TMEM or the
        // stages are released.
        if (lane == 0) {
            umma_commit(drain);
            mbar_wait_ns(drain, 0);
        }
        __syncwarp();
    } else {
        // ---------------- softmax: thread = query row
        const int r = tid;
        int lo_r = 0, hi_r = 0;
        if (r < rows_here) row_key_bounds(new_start + (row0 + r) / p.G, kend, p.causal, p.window, first, lo_r, hi_r);
        hi_r = min(hi_r, hi_pos);
        float m = -CUDART_INF_F, l = 0.f;
        #pragma unroll 1
        for (int j = 0; j < ngr; ++j) {
            const int b = j & 1;
            if (!wait_bar(s_full + b, (j >> 1) & 1)) { timed_out = true; break; }
            tc_fence_after();
            float x[64];
            {
                float t0[32], t1[32];
                tmem_ld32(tmem + lane_off + b * 64, t0);
                tmem_ld32(tmem + lane_off + b * 64 + 32, t1);
#pragma unroll
                for (int k = 0; k < 32; ++k) { x[k] = t0[k]; x[32 + k] = t1[k]; }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free + b);
            const int pos0 = lo_pos + j * PG * kPage;
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const int pos = pos0 + k;
                x[k] = (pos >= lo_r && pos < hi_r) ? x[k] * p.scale_log2 : -CUDART_INF_F;
                mx = fmaxf(mx, x[k]);
            }
            // Lazy reference maximum: raised only when a score passes it by 2^8.
            const bool grow = mx > m + 8.f;
            if (__any_sync(0xffffffffu, grow)) {
                const float m_new = grow ? mx : m;
                const float alpha = (!grow || m == -CUDART_INF_F) ? (grow ? 0.f : 1.f) : exp2f(m - m_new);
                if (j > 0 && __any_sync(0xffffffffu, grow && m != -CUDART_INF_F)) {
                    // O holds P V up to group j - 1 against the old reference:
                    // wait for that product, then rescale in TMEM.
                    if (!wait_bar(pv_done + ((j - 1) & 1), ((j - 1) >> 1) & 1)) { timed_out = true; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < DP; c0 += 32) {
                        float o[32];
                        tmem_ld32(tmem + lane_off + 128 + c0, o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] *= alpha;
                        tmem_st32(tmem + lane_off + 128 + c0, o);
                    }
                    tc_fence_before();
                }
                l *= alpha;
                m = m_new;
            }
            const float mu = m == -CUDART_INF_F ? 0.f : m;
            // P(j) goes to buffer b once P V(j - 2) has read it.
            if (j >= 2 && !wait_bar(pv_done + b, ((j - 2) >> 1) & 1)) { timed_out = true; break; }
            unsigned char *prow = sP + b * C::kPBytes;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float e[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    e[k] = exp2f(x[c * 8 + k] - mu);
                    l += e[k];
                }
                uint4 v;
                v.x = pack_bf16x2(e[0], e[1]);
                v.y = pack_bf16x2(e[2], e[3]);
                v.z = pack_bf16x2(e[4], e[5]);
                v.w = pack_bf16x2(e[6], e[7]);
                *reinterpret_cast<uint4 *>(prow + swz_row(r, c)) = v;
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + b);
        }
        // ---------------- epilogue: this row's partial O, base-2 max and sum
        if (!timed_out && ngr > 0 && !wait_bar(pv_done + ((ngr - 1) & 1), ((ngr - 1) >> 1) & 1)) timed_out = true;
        timed_out = __any_sync(0xffffffffu, timed_out);
        if (!timed_out && ngr > 0) {
            tc_fence_after();
            // The stages are idle once the last product has landed; the
            // partial rows overwrite them (after the barrier below).
            float o[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(tmem + lane_off + 128 + q * 32, o[q]);
            tc_fence_before();
            named_barrier(1, 128);  // every softmax warp has read its O rows: stages may be overwritten
            float *dst = sMo + (size_t)r * DP;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4 *>(dst + q * 32 + k) = make_float4(o[q][k], o[q][k + 1], o[q][k + 2], o[q][k + 3]);
        } else {
            named_barrier(1, 128);
            float *dst = sMo + (size_t)r * DP;
#pragma unroll 4
            for (int k = 0; k < DP; k += 4) *reinterpret_cast<float4 *>(dst + k) = make_float4(0.f, 0.f, 0.f, 0.f);
            m = -CUDART_INF_F;
            l = 0.f;
        }
        sMm[r] = m;
        sMl[r] = l;
    }
    if (timed_out && lane == 0) atomicOr(sFlag, 2);
    if (bad && lane == 0) atomicOr(sFlag, 1);
    tc_fence_before();
    __syncthreads();  // partial rows written, every tcgen05 access done
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
    const int flags = sFlag[0];
    if (tid == 0 && flags) atomicOr(p.err, ((flags & 1) ? PKV_ERR_BLOCK : 0u) | ((flags & 2) ? PKV_ERR_TIMEOUT : 0u));
    merge_rows<DP, 1, R, NT, false>(p, sg, g, row0, rows_here, flags, rank, ncta, sMo, sMm, sMl, sPm, sPl, sLse,
                                    sAllM, sAllL, sAllF, sFlag, nullptr);
}

}  // namespace pkv
