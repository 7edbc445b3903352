// Tensor-core (tcgen05) attention tile for wide query groups (sm_103a).
//
// The row class of speculative verify and chunked steps: one (segment, kv
// head) carries G * q_len query rows, up to 128 (GQA 64:8 with 16 draft
// tokens), so the products Q K^T and P V are real contractions.  They run on
// the 5th-generation tensor cores: two issuing threads (one for S, one for
// P V) run tcgen05.mma (bf16 in, fp32 accumulate) with Q, K and V in shared
// memory and S, P and O in tensor memory (TMEM); the softmax threads read S
// from TMEM and write P back over it.  Same semantics and key split as
// attend_kernel (grid (C, kv_heads, segments); the C CTAs of a range are one
// cluster and merge through distributed shared memory, each CTA pushing rows
// into the stage area of the CTA that finishes them).
//
// Per CTA (448 threads):
//   warps 0-7   softmax: row t of the tile (TMEM lane t) belongs to warps
//               t / 32 and t / 32 + 4, each taking 32 of a stage's 64 keys
//               with a running maximum and sum of its own and its own O
//               accumulator (O_0 for keys 0-31 of every stage, O_1 for
//               32-63), so the halves never wait for each other inside the
//               loop; they are combined once, in the epilogue.  The warps
//               also stage Q in shared memory, write P over the S columns
//               they have read, and after the loop write their rows out (one
//               CTA per range) or push them to the CTA of the cluster that
//               merges those rows;
//   warps 8, 11 K loads, alternate stages: 4 pages (64 keys) per stage,
//               each page as two 64-column TMA boxes, so a stage is one
//               K-major tile of 64 keys (128-byte swizzle) for Q K^T; a stage
//               is released as soon as its S product has completed;
//   warps 10, 12 V loads, alternate stages: 4 pages per stage, one TMA box
//               per page (two 64-column parts), an MN-major tile of 16 keys
//               for each step of P V; released when its P V has completed;
//   warp 9      S products: fixes this step's K rows into the stage (taken
//               from k_new, appended to the cache), issues S(j) = Q K_j^T
//               (M = 128, N = 64, A = Q from shared memory, 8 steps over
//               head_dim) once P V(j - NB) has freed its TMEM buffer; also
//               owns the TMEM allocation;
//   warp 13     P V products: fixes edge V pages (stale rows zeroed, this
//               step's rows from v_new, appended), and once P(j) is in TMEM
//               issues O_0 += P(j) V(j) over keys 0-31 and O_1 += ... over
//               keys 32-63 (M = 128, N = 128, A = P from TMEM, 2 steps of 16
//               keys each).
// One thread issuing every copy, or every product, was the limit: a warp's
// later instructions wait behind its tensor-core and TMA issues, so two
// loaders per stream and separate S and P V issuers keep each queue short.
// TMEM (512 columns allocated): S / P in NB = 3 buffers of 64 columns from
// column 0 (each half's P as bf16 pairs in the first 16 of its own 32 S
// columns), then O_0 and O_1 (128 columns each).  Q sits in shared memory
// (K-major, 128-byte swizzle): a product whose A operand comes from TMEM
// issues at 117 cycles against 67 from shared memory (N <= 128).  Shared
// memory holds Q (32 KB) and the K and V stages: 11 stages (176 KB) of loads
// in flight.
//
// Scheduling: a CTA's fixed cost (first page loads, cluster merge) is worth
// about 15 groups of 64 keys, so with few segments the CTAs take ranges
// longest first, a range of at most kSoloGroups groups runs on one CTA
// without a merge, and the planner aims at one wave of CTAs.
//
// The online softmax keeps each half row in one thread (no cross-lane
// reduction) and raises its reference maximum lazily: only when a score
// exceeds it by more than 2^8, and then its O is rescaled in TMEM after the
// previous P V has landed.  Every wait is bounded; a timeout poisons the
// CTA's output (PKV_ERR_TIMEOUT), drains what is in flight and frees TMEM.
//
// Semantics follow the segment-table attention of ExecuTorch PR #24072
// (triton::sdpa_varlen) over the paged layout of vLLM-Omni's SenseNova-U1
// PagedDecodeCache, exactly as attend_kernel.
#pragma once

#include "attend.cuh"

namespace pkv {

template <int NK_, int NV_>
struct VfyCfg {
    using T = __nv_bfloat16;
    static constexpr int DP = 128;                  // head_dim (this tile needs exactly 128)
    static constexpr int NK = NK_;                  // K stages of 4 pages
    static constexpr int NV = NV_;                  // V stages of 4 pages
    static constexpr int kRows = 128;               // query rows per CTA = TMEM lanes
    static constexpr int kThreads = 448;            // 8 softmax warps, 2 K loaders, 2 V loaders, S and P V issuers
    static constexpr int kLoaders = 2;              // loader warps per stream (alternate stages)
    static constexpr int kPages = 4;                // pages per stage (N = 64 keys)
    static constexpr unsigned kHalf = kPages * kPage * 128;        // 64 keys x 128 B
    static constexpr unsigned kKStage = 2 * kHalf;                 // K: two 64-column halves
    static constexpr unsigned kVStage = kPages * 4096;             // V: one 4 KB box per page
    static constexpr size_t kLoopBytes = (size_t)NK * kKStage + (size_t)NV * kVStage;
    // After the loop the stage area receives the rows pushed by the cluster:
    // (max, sum) per source and row, then the rows, 16 sources at most.
    static constexpr size_t kRecvStat = (size_t)16 * kRows * 8;
    static constexpr size_t kRecvBytes = kRecvStat + ((size_t)kRows + 16) * DP * 4;
    static constexpr size_t kBodyBytes = kLoopBytes > kRecvBytes ? kLoopBytes : kRecvBytes;
    // Q: two K-major halves of 128 rows x 64 columns, 128-byte swizzle
    static constexpr size_t kQHalf = (size_t)kRows * 128;
    static constexpr size_t kQBytes = 2 * kQHalf;
    // merge weights [16][rows], cluster flags [16], per-half row maxima and sums [2][rows] each
    static constexpr size_t kWnBytes = (size_t)16 * kRows * 4 + 16 * 4 + 2 * kRows * 4 + 2 * kRows * 4;
    static constexpr int NB = 3;                    // S / P buffers in TMEM
    // K, V full / empty; s_full, p_full, pv_done [NB]; drain
    static constexpr int kBars = 2 * NK + 2 * NV + 3 * NB + 1;
    static constexpr size_t kMiscBytes = (size_t)kBars * 8 + 16 + 32 * 4 + (size_t)kThreads * 4;
    static constexpr size_t kSmemBytes = 1024 + kBodyBytes + kQBytes + kWnBytes + kMiscBytes;
    static constexpr int kTmemCols = 512;
    static constexpr int kSoloGroups = 24;          // a range of at most this many groups runs on one CTA
    static constexpr int kRankSegs = 64;            // up to this many segments launch longest range first
    static_assert(kSmemBytes <= 232448, "exceeds the per-CTA shared memory limit");
    static_assert(kKStage % 1024 == 0 && kVStage % 1024 == 0 && kBodyBytes % 1024 == 0,
                  "operand tiles start on 1024-byte swizzle atoms");
    // A loader waits on the release of its stage's previous use; with at
    // least as many stages as loaders that use is never two phases back.
    static_assert(NK >= kLoaders && NV >= kLoaders, "ring shorter than its loaders");
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
// As umma_bf16 with A (M x 16, bf16 pairs per 32-bit column, row = lane) read from TMEM.
__device__ __forceinline__ void umma_bf16_ts(unsigned d_tmem, unsigned a_tmem, uint64_t b, uint32_t idesc,
                                             int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
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

// 16 32-bit columns into this thread's TMEM lane (warp-collective; waits for completion).
__device__ __forceinline__ void tmem_st16(unsigned taddr, const unsigned (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Offset of 16-byte chunk `c` (0..7) of row `r` in a tile of 128-byte rows
// loaded with 128-byte swizzling (rows grouped in 1024-byte atoms).
__device__ __forceinline__ unsigned swz_row(int r, int c) { return (unsigned)(r * 128 + ((c ^ (r & 7)) << 4)); }

// ---------------------------------------------------------------- the kernel

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1) verify_kernel(const __grid_constant__ AttendParams p) {
    using T = __nv_bfloat16;
    namespace cg = cooperative_groups;
    constexpr int DP = C::DP, NK = C::NK, NV = C::NV, R = C::kRows, NT = C::kThreads, PG = C::kPages;
    constexpr int EPC = 8;  // bf16 per 16-byte chunk
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10, kWarpK2 = 11, kWarpV2 = 12, kWarpPv = 13;
    constexpr int NL = C::kLoaders;
    constexpr int NB = C::NB;
    constexpr unsigned kColO = 64 * NB;  // O_h at kColO + 128 h

    extern __shared__ unsigned char smem_raw[];
    unsigned char *body = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sK = body;                                      // NK K stages
    unsigned char *sV = sK + (size_t)NK * C::kKStage;              // NV V stages
    unsigned char *sQ = body + C::kBodyBytes;                      // Q, two K-major halves
    float *sWn = reinterpret_cast<float *>(sQ + C::kQBytes);       // [16][R] merge weights
    int *sCf = reinterpret_cast<int *>(sWn + 16 * R);              // [16] flags pushed by the cluster
    float *sXm = reinterpret_cast<float *>(sCf + 16);              // [2][R] row maxima of each half
    float *sXl = sXm + 2 * R;                                      // [2][R] row sums of each half
    uint64_t *bars = reinterpret_cast<uint64_t *>(sXl + 2 * R);
    uint64_t *k_full = bars, *k_empty = bars + NK, *v_full = bars + 2 * NK, *v_empty = v_full + NV;
    uint64_t *s_full = v_empty + NV, *p_full = s_full + NB, *pv_done = p_full + NB;
    uint64_t *drain = pv_done + NB;
    unsigned *tslot = reinterpret_cast<unsigned *>(bars + C::kBars);
    volatile int *sAbort = reinterpret_cast<volatile int *>(tslot + 1);
    int *sAppOk = reinterpret_cast<int *>(tslot + 2);
    int *sFlag = reinterpret_cast<int *>(tslot + 4);            // [0] own flags: 1 bad page, 2 timeout
    int *sCov = sFlag + 32;                                     // [NT] coverage flags

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool softmax = warp < 8;
    const int quad = warp & 3, half = (warp >> 2) & 1;          // softmax: TMEM lane quadrant, key / column half
    const int r = quad * 32 + lane;                             // softmax: this thread's row of the tile
    const int rank = blockIdx.x, ncta = gridDim.x;
    const int g = blockIdx.y / p.row_tiles, rt = blockIdx.y - g * p.row_tiles;
    const bool cov_cta = grid_cta_index() < coverage_slices(p, NT);
    const int cov_any = coverage_begin(p, sCov, cov_cta, NT);
    if (p.S == 0) {
        pdl_wait();
        pdl_trigger();
        if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
        return;
    }
    // Longest ranges first: with few segments every CTA ranks them by their
    // key count (ties by index) and takes the blockIdx.z-th, so the longest
    // ranges start in the first wave and the short ones fill the tail.  Any
    // order is correct; this only schedules.  (The merge weights' space is
    // idle until the epilogue.)
    int s = blockIdx.z;
    if (p.S <= C::kRankSegs) {
        int *sLen = reinterpret_cast<int *>(sWn), *sPick = sLen + C::kRankSegs;
        if (tid < p.S) {
            const Segment t = load_segment(p.seq_info, tid);
            const int lo = p.window > 0 ? max(0, t.kend - t.ql - p.window + 1) : 0;
            sLen[tid] = max(0, t.kend - lo);
        }
        __syncthreads();
        if (tid < p.S) {
            int k = 0;
            for (int u = 0; u < p.S; ++u) k += (sLen[u] > sLen[tid]) || (sLen[u] == sLen[tid] && u < tid);
            if (k == (int)blockIdx.z) *sPick = tid;
        }
        __syncthreads();
        s = *sPick;
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
    // A short range runs on the cluster's first CTA alone, without a merge;
    // the others leave at once (uniform: every CTA of the cluster sees the
    // same range, so no cluster barrier is ever half attended).
    const bool solo = ncta > 1 && (nblk + PG - 1) / PG <= C::kSoloGroups;
    const int ncl = solo ? 1 : ncta;  // CTAs sharing the range
    if (solo && rank > 0) {
        if (cov_cta) {
            pdl_wait();
            pdl_trigger();
            apply_coverage(p, sCov, cov_any, NT);
        }
        return;
    }
    const int bps = (nblk + ncl - 1) / ncl;
    const int active = (nblk + bps - 1) / bps;
    const int cb0 = pb_begin + rank * bps;
    const int nb = rank < active ? min(cb0 + bps, pb_end) - cb0 : 0;
    const int ngr = (nb + PG - 1) / PG;                     // groups of 4 pages of this CTA
    const int lo_pos = cb0 * kPage, hi_pos = (cb0 + nb) * kPage;

    const T *knew = reinterpret_cast<const T *>(p.k_new);
    const T *vnew = reinterpret_cast<const T *>(p.v_new);
    const bool fused = knew != nullptr;
    const int dchunks = p.D / EPC;
    const int *bt_row = p.block_table + (long long)sg.col * p.mbps;
    const bool has_new = fused && rt == 0 && nb > 0 && new_start < hi_pos && kend > lo_pos;

    if (tid == 0) {
        #pragma unroll 1
        for (int i = 0; i < C::kBars; ++i) {
            const bool eight = i >= 2 * NK + 2 * NV + NB && i < 2 * NK + 2 * NV + 2 * NB;  // p_full: every softmax warp
            mbar_init(bars + i, eight ? 8 : 1);
        }
        fence_barrier_init();
        sFlag[0] = 0;
        *sAbort = 0;
        *sAppOk = 0;
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tmem = *tslot;
    const unsigned lane_off = (unsigned)(32 * quad) << 16;

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

    // ---- TMA loads (warps 8, 11: K; 10, 12: V): group j = pages cb0 + 4j .. + 3,
    // loader lidx of a stream issuing the groups j = lidx (mod 2)
    const bool loader = warp == kWarpK || warp == kWarpV || warp == kWarpK2 || warp == kWarpV2;
    const bool is_v = warp == kWarpV || warp == kWarpV2;
    const int lidx = (warp == kWarpK2 || warp == kWarpV2) ? 1 : 0;
    int id_reg = -1, id_window = -1, issued = lidx;
    bool bad = false;
    auto load_ids = [&](int li0) {
        id_window = li0 & ~31;
        const int li = id_window + lane;
        id_reg = li < nb ? bt_row[table_page(cb0 + li, p.ring_rows)] : -1;
    };
    // K comes in 2 KB TMA boxes (16 keys x 64 columns) into two 64-column
    // halves of the stage, so the stage is one K-major tile of 64 keys; V in
    // 4 KB boxes, one per page (16 keys x two 64-column parts).
    auto issue = [&](int j) {
        uint64_t *bar = (is_v ? v_full + j % NV : k_full + j % NK);
        unsigned char *stage = is_v ? sV + (size_t)(j % NV) * C::kVStage : sK + (size_t)(j % NK) * C::kKStage;
        int ok_pages = 0;
        unsigned okmask = 0;
        int bids[PG];
#pragma unroll
        for (int u = 0; u < PG; ++u) {
            const int li = j * PG + u;
            bids[u] = -1;
            if (li < nb) {
                if ((li & ~31) != id_window) load_ids(li);
                bids[u] = __shfl_sync(0xffffffffu, id_reg, li & 31);
                const bool ok = bids[u] >= 0 && (long long)bids[u] < p.num_blocks;
                bad |= !ok;
                if (ok) { okmask |= 1u << u; ++ok_pages; }
            }
        }
        if (lane == 0) {
            fence_proxy_async();
            if (ok_pages) mbar_expect_tx(bar, (unsigned)ok_pages * 4096u);
            else mbar_arrive(bar);
#pragma unroll
            for (int u = 0; u < PG; ++u) {
                if (!((okmask >> u) & 1u)) continue;
                if (is_v) {
                    tma_load_5d(stage + u * 4096, &p.tmap_v, bar, 0, 0, 0, g, bids[u]);
                } else {
                    tma_load_4d(stage + u * 2048, &p.tmap_k, bar, 0, g, 0, bids[u]);
                    tma_load_4d(stage + C::kHalf + u * 2048, &p.tmap_k, bar, 64, g, 0, bids[u]);
                }
            }
        }
    };
    // Pages wholly below new_start may be fetched before the dependency wait;
    // in the fused call every page may (this step's rows are replaced after it).
    auto early_ok = [&](int j) { return fused || (cb0 + min(j * PG + PG, nb)) * kPage <= new_start; };
    const int NSt = is_v ? NV : NK;

    if (loader) {
        load_ids(0);
        #pragma unroll 1
        for (; issued < NSt && issued < ngr; issued += NL) {
            if (!early_ok(issued)) break;
            issue(issued);
        }
    }
    // Append validity, all or nothing over the segment's new rows (the block
    // table is not written by the previous kernel); kept for the MMA warp.
    if (has_new && softmax) {
        bool ok = true;
        #pragma unroll 1
        for (int i = tid; i < sg.ql; i += 256) {
            const int pos = new_start + i;
            const int rr = p.ring_rows ? pos % p.ring_rows : pos;
            const int b = bt_row[rr / kPage];
            ok &= b >= 0 && (long long)b < p.num_blocks;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0 && !ok) atomicOr(sAppOk, 1);
    }
    // Warm L2 with the rows read right after the wait: this tile's queries
    // and, in the fused call, this step's K/V rows.
    if (softmax) {
        if (r < rows_here) {
            const int ur = row0 + r, i = ur / p.G, jh = ur - i * p.G;
            const T *src = reinterpret_cast<const T *>(p.q) + (((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh) * p.D;
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + half * 128));
        }
        if (has_new) {
            const int a = max(new_start, lo_pos), e = min(kend, hi_pos);
            #pragma unroll 1
            for (int c = tid; c < (e - a) * 4; c += 256) {
                const int row = c >> 2, kv = (c >> 1) & 1;
                const T *src = (kv ? vnew : knew) + (((long long)sg.q0 + (a + row - new_start)) * p.Hkv + g) * p.D;
                asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char *>(src) + (c & 1) * 128));
            }
        }
    }

    pdl_wait();
    pdl_trigger();

    // ---- queries into shared memory: each softmax thread its row's half
    // (64 columns = one swizzled 128-byte row of that half's tile); rows
    // past the group are zero.
    if (softmax) {
        uint4 qv[8];
        const int ur = row0 + r, i = ur / p.G, jh = ur - i * p.G;
        const T *src = reinterpret_cast<const T *>(p.q) + (((long long)sg.q0 + (r < rows_here ? i : 0)) * p.Hq +
                                                            (long long)g * p.G + (r < rows_here ? jh : 0)) * p.D;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            qv[c] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows_here && half * 8 + c < dchunks) qv[c] = *reinterpret_cast<const uint4 *>(src + (half * 8 + c) * EPC);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(sQ + half * C::kQHalf + swz_row(r, c)) = qv[c];
        fence_proxy_async();  // the tensor core reads Q through the async proxy
    }
    if (cov_cta) apply_coverage(p, sCov, cov_any, NT);
    if (loader) {
        #pragma unroll 1
        for (; issued < NSt && issued < ngr; issued += NL) issue(issued);
    }
    tc_fence_before();
    __syncthreads();  // queries in shared memory, append validity known
    tc_fence_after();
    const bool app_ok = has_new && *sAppOk == 0;

    bool timed_out = false;
    float m = -CUDART_INF_F, l = 0.f;  // softmax: this row's reference max and this half's sum

    if (loader) {
        // ---------------- refill each stage once its product has completed
        uint64_t *emp = is_v ? v_empty : k_empty;
        #pragma unroll 1
        for (int j = issued; j < ngr; j += NL) {
            if (!wait_bar(emp + (j % NSt), ((j / NSt) - 1) & 1)) { timed_out = true; break; }
            issue(j);
            issued = j + NL;
        }
        // Drain: every issued stage has landed before its memory is reused or
        // freed.  The first loader of the stream waits on each stage's last
        // use, whichever loader issued it (an earlier use's phase may have
        // been overtaken).
        if (lane == 0 && lidx == 0) {
            uint64_t *fb = is_v ? v_full : k_full;
            #pragma unroll 1
            for (int j = max(0, ngr - NSt); j < ngr; ++j)
                if (!mbar_wait_ns(fb + (j % NSt), (j / NSt) & 1)) break;
        }
    } else if (warp == kWarpMma || warp == kWarpPv) {
        // ---------------- edge-page fix-up and MMA issue (S: warp 9, P V: warp 13)
        const uint32_t id_s = umma_idesc_bf16(128, 64, 0), id_o = umma_idesc_bf16(128, 128, 1);
        // Rows of page u of group j: stale ones [0, zlo) and [zhi, 16) (V
        // zeroed), this step's ones [na, zhi) (K or V from k_new / v_new, also
        // appended to the cache).  A page past the range is all stale.
        auto page_rows = [&](int j, int u, int &zlo, int &zhi, int &na) {
            const int li = j * PG + u, pos0 = (cb0 + li) * kPage;
            if (li < nb) {
                zlo = min(max(lo_u - pos0, 0), kPage);
                zhi = min(max(kend - pos0, 0), kPage);
                na = fused ? min(max(new_start - pos0, 0), kPage) : zhi;
            } else {
                zlo = kPage; zhi = kPage; na = kPage;
            }
        };
        // this step's rows [na, zhi) of page u into the stage (and the cache)
        auto put_new = [&](int kv, unsigned char *stage, int j, int u, int na, int zhi) {
            const int pos0 = (cb0 + j * PG + u) * kPage, nn = (zhi - na) * 16;
            const long long bpage = app_ok ? (long long)bt_row[table_page(pos0 / kPage, p.ring_rows)] : 0;
            const int ring_base = p.ring_rows ? pos0 % p.ring_rows : pos0;
            #pragma unroll 1
            for (int c = lane; c < nn; c += 32) {
                const int o = na + (c >> 4), ch = c & 15;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (ch < dchunks) {
                    v = *reinterpret_cast<const uint4 *>((kv ? vnew : knew) +
                                                         (((long long)sg.q0 + (pos0 + o - new_start)) * p.Hkv + g) * p.D +
                                                         ch * EPC);
                    if (app_ok) {
                        const long long slot = bpage * kPage + (ring_base + o) % kPage;
                        *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(kv ? p.v_pool_w : p.k_pool_w) +
                                                   (slot * p.Hkv + g) * p.D + ch * EPC) = v;
                    }
                }
                const unsigned off = kv ? u * 4096 + (ch >> 3) * 2048 + swz_row(o, ch & 7)
                                        : (ch >> 3) * C::kHalf + u * 2048 + swz_row(o, ch & 7);
                *reinterpret_cast<uint4 *>(stage + off) = v;
            }
        };
        // A group wholly inside the CTA's range and below this step's rows
        // (and, for V, at or above the first visible key) needs no fix-up;
        // deciding that up front keeps the per-page checks off the issuing
        // warps' critical path (they measured 0.6 us per group).
        const int clean_hi = fused ? new_start : kend;
        auto interior = [&](int j, bool v) {
            const int g0 = (cb0 + j * PG) * kPage, g1 = g0 + PG * kPage;
            return j * PG + PG <= nb && g1 <= clean_hi && (!v || g0 >= lo_u);
        };
        // K: only this step's rows (stale keys are masked out of S).
        auto fix_k = [&](int j, unsigned char *stage) {
            if (interior(j, false)) return;
            bool any = false;
#pragma unroll 1
            for (int u = 0; u < PG; ++u) {
                int zlo, zhi, na;
                page_rows(j, u, zlo, zhi, na);
                if (na < zhi) { any = true; put_new(0, stage, j, u, na, zhi); }
            }
            if (any) fence_proxy_async();  // generic writes before the tensor core reads the stage
            __syncwarp();
        };
        // V: stale rows zeroed (P is zero there, but 0 x NaN is not), this step's rows.
        auto fix_v = [&](int j, unsigned char *stage) {
            if (interior(j, true)) return;
            bool any = false;
#pragma unroll 1
            for (int u = 0; u < PG; ++u) {
                int zlo, zhi, na;
                page_rows(j, u, zlo, zhi, na);
                if (zlo > 0 || zhi < kPage) {
                    any = true;
                    const int nz = (zlo + kPage - zhi) * 16;
                    #pragma unroll 1
                    for (int c = lane; c < nz; c += 32) {
                        const int o0 = c >> 4, ch = c & 15;
                        const int o = o0 < zlo ? o0 : zhi + (o0 - zlo);
                        *reinterpret_cast<uint4 *>(stage + u * 4096 + (ch >> 3) * 2048 + swz_row(o, ch & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (na < zhi) { any = true; put_new(1, stage, j, u, na, zhi); }
            }
            if (any) fence_proxy_async();
            __syncwarp();
        };
        auto issue_pv = [&](int i) {
            const int b = i % NB, vs = i % NV;
            unsigned char *stage = sV + (size_t)vs * C::kVStage;
            if (!wait_bar(v_full + vs, (i / NV) & 1)) return false;
            fix_v(i, stage);
            if (!wait_bar(p_full + b, (i / NB) & 1)) return false;
            tc_fence_after();
            if (lane == 0) {
                const unsigned v_addr = smem_u32(stage);
#pragma unroll
                for (int u = 0; u < PG; ++u) {
                    const int h = u >> 1;  // keys 0-31 -> O_0 (P of half 0), 32-63 -> O_1 (P of half 1)
                    umma_bf16_ts(tmem + kColO + h * 128, tmem + b * 64 + h * 32 + (u & 1) * 8,
                                 umma_desc(v_addr + u * 4096, 2048, 1024), id_o, (i > 0 || (u & 1)) ? 1 : 0);
                }
                umma_commit(v_empty + vs);
                umma_commit(pv_done + b);
            }
            __syncwarp();
            return true;
        };
        if (warp == kWarpMma) {
        #pragma unroll 1
        for (int j = 0; j < ngr && !timed_out; ++j) {
            const int ks = j % NK, b = j % NB;
            unsigned char *stage = sK + (size_t)ks * C::kKStage;
            if (!wait_bar(k_full + ks, (j / NK) & 1)) { timed_out = true; break; }
            fix_k(j, stage);
            // S(j) overwrites buffer b, which P V(j - NB) reads P(j - NB) from.
            if (j >= NB && !wait_bar(pv_done + b, ((j - NB) / NB) & 1)) { timed_out = true; break; }
            tc_fence_after();
            if (lane == 0) {
                const unsigned k_addr = smem_u32(stage), q_addr = smem_u32(sQ);
#pragma unroll
                for (int k = 0; k < DP / 16; ++k)
                    umma_bf16(tmem + b * 64, umma_desc(q_addr + (k >> 2) * (unsigned)C::kQHalf + (k & 3) * 32, 16, 1024),
                              umma_desc(k_addr + (k >> 2) * C::kHalf + (k & 3) * 32, 16, 1024), id_s, k > 0 ? 1 : 0);
                umma_commit(s_full + b);
                umma_commit(k_empty + ks);
            }
            __syncwarp();
        }
        // Drain: every MMA this thread issued has completed before TMEM or the
        // stages are released.
        if (lane == 0) {
            umma_commit(drain);
            mbar_wait_ns(drain, 0);
        }
        __syncwarp();
        } else {
        int last = -1;
        #pragma unroll 1
        for (int i = 0; i < ngr && !timed_out; ++i) {
            if (!issue_pv(i)) { timed_out = true; break; }
            last = i;
        }
        // Drain: the last commit completes after every product this thread issued.
        if (lane == 0 && last >= 0) mbar_wait_ns(pv_done + (last % NB), (last / NB) & 1);
        __syncwarp();
        }
    } else if (softmax) {
        // ---------------- softmax: this thread = (row r, 32 keys of each stage)
        int lo_r = 0, hi_r = 0;
        if (r < rows_here) row_key_bounds(new_start + (row0 + r) / p.G, kend, p.causal, p.window, first, lo_r, hi_r);
        hi_r = min(hi_r, hi_pos);
        #pragma unroll 1
        for (int j = 0; j < ngr; ++j) {
            const int b = j % NB;  // S / P buffer
            if (!wait_bar(s_full + b, (j / NB) & 1)) { timed_out = true; break; }
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + lane_off + b * 64 + half * 32, x);
            const int pos0 = lo_pos + j * PG * kPage + half * 32;
            // Key bounds per score only where some real row of the warp
            // does not see all 32 keys (padding rows are never written out).
            if (__all_sync(0xffffffffu, r >= rows_here || (pos0 >= lo_r && pos0 + 32 <= hi_r))) {
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] *= p.scale_log2;
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int pos = pos0 + k;
                    x[k] = (pos >= lo_r && pos < hi_r) ? x[k] * p.scale_log2 : -CUDART_INF_F;
                }
            }
            float mx;
            {   // row maximum of the 32 scores as a tree (depth 5, not a 32-long chain)
                float t[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) t[k] = fmaxf(x[k], x[k + 16]);
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int k = 0; k < w; ++k) t[k] = fmaxf(t[k], t[k + w]);
                mx = t[0];
            }
            // Lazy reference maximum: raised only when a score passes it by 2^8.
            const bool grow = mx > m + 8.f;
            if (__any_sync(0xffffffffu, grow)) {
                const float m_new = grow ? mx : m;
                const float alpha = (!grow || m == -CUDART_INF_F) ? (grow ? 0.f : 1.f) : exp2f(m - m_new);
                if (j > 0 && __any_sync(0xffffffffu, grow && m != -CUDART_INF_F)) {
                    // O_half holds P V up to group j - 1 against the old
                    // reference: wait for that product, then rescale it.
                    if (!wait_bar(pv_done + ((j - 1) % NB), ((j - 1) / NB) & 1)) { timed_out = true; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        float o[32];
                        tmem_ld32(tmem + lane_off + kColO + half * 128 + c0, o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] *= alpha;
                        tmem_st32(tmem + lane_off + kColO + half * 128 + c0, o);
                    }
                }
                l *= alpha;
                m = m_new;
            }
            const float mu = m == -CUDART_INF_F ? 0.f : m;
            unsigned pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float e0 = exp2f(x[2 * k] - mu), e1 = exp2f(x[2 * k + 1] - mu);
                l += e0 + e1;
                pk[k] = pack_bf16x2(e0, e1);
            }
            // P(j) as bf16 pairs over the first 16 of this half's S columns (read above)
            tmem_st16(tmem + lane_off + b * 64 + half * 32, pk);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + b);
        }
        // the last product has landed before O is read back
        if (!timed_out && ngr > 0 && !wait_bar(pv_done + ((ngr - 1) % NB), ((ngr - 1) / NB) & 1)) timed_out = true;
        timed_out = __any_sync(0xffffffffu, timed_out);
        sXm[half * R + r] = m;
        sXl[half * R + r] = timed_out ? 0.f : l;
    }
    if (timed_out && lane == 0) atomicOr(sFlag, 2);
    if (bad && lane == 0) atomicOr(sFlag, 1);
    tc_fence_before();
    __syncthreads();  // every role is done; the stage area is idle
    tc_fence_after();
    const int flags = sFlag[0];
    if (tid == 0 && flags) atomicOr(p.err, ((flags & 1) ? PKV_ERR_BLOCK : 0u) | ((flags & 2) ? PKV_ERR_TIMEOUT : 0u));
    const bool has_o = ngr > 0 && !(flags & 2);  // O_0, O_1 in TMEM hold this CTA's product
    // The row's two halves against one reference: weights w_h = 2^(m_h - m)
    // (a half that saw no key has weight 0 and is never multiplied in).
    float w0 = 0.f, w1 = 0.f;
    if (softmax) {
        const float m0 = sXm[r], m1 = sXm[R + r];
        m = fmaxf(m0, m1);
        w0 = (m == -CUDART_INF_F || m0 == -CUDART_INF_F) ? 0.f : exp2f(m0 - m);
        w1 = (m == -CUDART_INF_F || m1 == -CUDART_INF_F) ? 0.f : exp2f(m1 - m);
        l = w0 * sXl[r] + w1 * sXl[R + r];
        if (!has_o) { m = -CUDART_INF_F; l = 0.f; }
    }
    // This thread's 32 columns c0.. of the row's combined (unnormalised) O.
    auto o_cols = [&](int c0, float (&o)[32]) {
        if (!has_o) {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0.f;
            return;
        }
        float o1[32];
        tmem_ld32(tmem + lane_off + kColO + half * 64 + c0, o);
        tmem_ld32(tmem + lane_off + kColO + 128 + half * 64 + c0, o1);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = (w0 != 0.f ? w0 * o[e] : 0.f) + (w1 != 0.f ? w1 * o1[e] : 0.f);
    };

    // ---- epilogue: rows of O straight from TMEM
    auto out_row = [&](int rr) {
        const int ur = row0 + rr, i = ur / p.G, jh = ur - i * p.G;
        return ((long long)sg.q0 + i) * p.Hq + (long long)g * p.G + jh;
    };
    // out is only required to be 4-byte aligned: vector stores when it is 16.
    const bool out16 = (reinterpret_cast<uintptr_t>(p.out) & 15u) == 0;
    auto store4 = [&](float *dst, float4 v) {
        if (out16) {
            *reinterpret_cast<float4 *>(dst) = v;
        } else {
            dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
        }
    };
    if (ncl == 1) {
        if (softmax) {
            const bool zero = flags || !(l > 0.f);
            const float inv = zero ? 0.f : 1.f / l;
            float *dst = p.out + out_row(min(r, rows_here - 1)) * p.D + half * 64;
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float o[32];
                o_cols(c0, o);
                if (r < rows_here) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        store4(dst + c0 + k, zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                                                  : make_float4(o[k] * inv, o[k + 1] * inv, o[k + 2] * inv,
                                                                o[k + 3] * inv));
                }
            }
            if (half == 0 && r < rows_here && p.lse)
                p.lse[out_row(r)] = zero ? -CUDART_INF_F : (m + log2f(l)) * kLn2;
        }
    } else {
        // Rows are merged by owner: CTA k of the cluster finishes rows
        // [k * per, (k + 1) * per).  Every CTA pushes each row's (max, sum)
        // and partial O into the owner's (idle) stage area.
        cg::cluster_group cluster = cg::this_cluster();
        const int per = (rows_here + ncta - 1) / ncta;
        float2 *rStat = reinterpret_cast<float2 *>(body);                       // [16][per]
        float *rRows = reinterpret_cast<float *>(body + C::kRecvStat);         // [16][per][DP]
        cluster.sync();  // every CTA is past its loop: its stage area may be written
        if (tid < ncta) *cluster.map_shared_rank(sCf + rank, tid) = flags;
        if (softmax) {
            const int k = min(r / per, ncta - 1), rr = r - k * per;
            if (half == 0 && r < rows_here) *cluster.map_shared_rank(rStat + rank * per + rr, k) = make_float2(m, l);
            float *dst = r < rows_here ? cluster.map_shared_rank(rRows + ((size_t)rank * per + rr) * DP + half * 64, k)
                                       : nullptr;
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float o[32];
                o_cols(c0, o);
                if (r < rows_here)
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
            }
        }
        cluster.sync();  // publishes the pushed rows
        int poison = 0;
#pragma unroll
        for (int c = 0; c < 16; ++c) poison |= c < ncta ? sCf[c] : 0;
        const int r0 = rank * per, nr = max(0, min(per, rows_here - r0));
        // per owned row: normalised weight of each source, and the lse
        if (tid < nr) {
            float M = -CUDART_INF_F;
#pragma unroll 1
            for (int c = 0; c < ncta; ++c) M = fmaxf(M, rStat[c * per + tid].x);
            float W = 0.f;
#pragma unroll 1
            for (int c = 0; c < ncta; ++c) {
                const float2 st = rStat[c * per + tid];
                // a zero weight must not touch its partial: a poisoned one may hold NaN
                const float w = (M == -CUDART_INF_F || st.x == -CUDART_INF_F) ? 0.f : exp2f(st.x - M);
                sWn[c * R + tid] = w;
                W = fmaf(w, st.y, W);
            }
            const bool zero = poison || !(W > 0.f);
            const float inv = zero ? 0.f : 1.f / W;
#pragma unroll 1
            for (int c = 0; c < ncta; ++c) sWn[c * R + tid] = zero ? 0.f : sWn[c * R + tid] * inv;
            if (p.lse) p.lse[out_row(r0 + tid)] = zero ? -CUDART_INF_F : (M + log2f(W)) * kLn2;
        }
        __syncthreads();
#pragma unroll 1
        for (int e = tid * 4; e < nr * DP; e += NT * 4) {
            const int rr = e / DP, d = e - rr * DP;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
            for (int c = 0; c < ncta; ++c) {
                const float w = sWn[c * R + rr];
                if (w != 0.f) {
                    const float4 v = *reinterpret_cast<const float4 *>(rRows + ((size_t)c * per + rr) * DP + d);
                    o.x = fmaf(w, v.x, o.x); o.y = fmaf(w, v.y, o.y); o.z = fmaf(w, v.z, o.z); o.w = fmaf(w, v.w, o.w);
                }
            }
            store4(p.out + out_row(r0 + rr) * p.D + d, o);
        }
    }
    tc_fence_before();
    __syncthreads();  // every TMEM read is done
    if (warp == kWarpMma) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

}  // namespace pkv
