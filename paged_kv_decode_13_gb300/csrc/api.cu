// C-ABI entry points of libpkv: argument checks, launch planning and launches.
// Every entry point validates on the host first and returns a negative
// pkv_status before launching anything; nothing here allocates memory,
// synchronises the host or keeps state beyond per-process kernel attributes.
#include <cuda_runtime.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "launch.h"
#include "misc_kernels.cuh"

using namespace pkv;

namespace {

constexpr int kDefaultSms = 152;       // GB300, used when no device is visible
constexpr int kTargetWaves = 3;        // split count: about this many waves of resident CTAs
constexpr int kMaxCluster = 16;        // largest thread-block cluster (non-portable size)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(int dtype) { return dtype == PKV_BF16 ? 2 : dtype == PKV_F32 ? 4 : 0; }

int check_cache(const pkv_cache *c) {
    if (!c) return PKV_EINVAL;
    if (c->dtype != PKV_BF16 && c->dtype != PKV_F32) return PKV_EUNSUPPORTED;
    // vLLM-Omni paged_decode_supported: head_dim a multiple of 8, at most 256.
    if (c->head_dim <= 0 || c->head_dim % 8 != 0 || c->head_dim > 256) return PKV_EUNSUPPORTED;
    if (c->num_layers <= 0 || c->kv_heads <= 0 || c->num_blocks <= 0) return PKV_EINVAL;
    if (c->num_blocks > INT32_MAX || c->kv_heads > 65535) return PKV_EINVAL;
    if (c->max_seqs <= 0 || c->max_blocks_per_seq <= 0) return PKV_EINVAL;
    if (!c->k || !c->v || !c->block_table) return PKV_EINVAL;
    if ((reinterpret_cast<uintptr_t>(c->block_table) & 3u) != 0) return PKV_EINVAL;
    if ((reinterpret_cast<uintptr_t>(c->first_valid) & 3u) != 0) return PKV_EINVAL;
    if (c->ring_rows < 0 || c->ring_rows % PKV_BLOCK_SIZE != 0) return PKV_EINVAL;
    if ((long long)c->ring_rows > (long long)c->max_blocks_per_seq * PKV_BLOCK_SIZE) return PKV_EINVAL;
    return PKV_OK;
}

int check_layer(const pkv_cache *c, int layer) {
    if (layer < 0 || layer >= c->num_layers) return PKV_EINVAL;
    if (!c->k[layer] || !c->v[layer] || !aligned16(c->k[layer]) || !aligned16(c->v[layer])) return PKV_EINVAL;
    return PKV_OK;
}

// Launch plan of one attention call.
struct Plan {
    AttnKernel k;
    int G, rows_max, row_tiles, units, ncta;
    bool gm;  // decode kernel merging its splits through a global workspace (no cluster)
};

constexpr int kMaxSplitsGm = 64;  // splits per key range when merging through global memory

// SMs of the current device (GB300's count when no device answers).
int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return kDefaultSms;
    }
    return n > 0 ? n : kDefaultSms;
}

// Workspace layout of the global merge: partial rows, (max, sum), flags,
// counters, each region 256-byte aligned.
struct WsLayout {
    size_t part, stat, flag, count, total;
};
// The counters come first, at a place that depends only on the unit count.
WsLayout ws_layout(long long units, int ncta, int dp) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    WsLayout w;
    w.count = 0;
    w.part = al((size_t)units * 4);
    w.stat = al(w.part + (size_t)units * ncta * 8 * dp * 4);
    w.flag = al(w.stat + (size_t)units * ncta * 8 * 8);
    w.total = al(w.flag + (size_t)units * ncta * 4);
    return w;
}

AttnKernel pick(int variant, int dp, int rc) {
    switch (variant * 1000 + dp) {
        case 64: return pick_0_64(rc);
        case 128: return pick_0_128(rc);
        case 256: return pick_0_256(rc);
        case 1064: return pick_1_64(rc);
        case 1128: return pick_1_128(rc);
        case 1256: return pick_1_256(rc);
        case 2064: return pick_2_64(rc);
        case 2128: return pick_2_128(rc);
        case 2256: return pick_2_256(rc);
    }
    return AttnKernel{nullptr, 0, 0, 0, 0, false, false};
}

// Clusters of c CTAs of this kernel that the device holds at once (c = 1:
// resident CTAs); cached per kernel and size, 0 when none fits or no device
// answers the query.
int active_clusters(const AttnKernel &k, int c) {
    static std::mutex mu;
    static const void *fns[64];
    static int count[64][kMaxCluster + 1];
    static int n = 0;
    if (c < 1 || c > kMaxCluster) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < n; ++i)
        if (fns[i] == k.fn) slot = i;
    if (slot < 0 && n < 64) {
        slot = n++;
        fns[slot] = k.fn;
        for (int i = 0; i <= kMaxCluster; ++i) count[slot][i] = -1;
    }
    if (slot >= 0 && count[slot][c] >= 0) return count[slot][c];
    int clusters = 0;
    if (c == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, k.threads, k.smem) != cudaSuccess) {
            cudaGetLastError();
            per_sm = 0;
        }
        clusters = per_sm * device_sms();
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)c, 1, 1);
        cfg.blockDim = dim3((unsigned)k.threads);
        cfg.dynamicSmemBytes = k.smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)c;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, k.fn, &cfg) != cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
        }
    }
    clusters = std::max(clusters, 0);
    if (slot >= 0) count[slot][c] = clusters;
    return clusters;
}

// Largest cluster size <= want that the device can schedule for this kernel
// (1 when no device answers the query).
int schedulable_cluster(const AttnKernel &k, int want) {
    for (int c = want; c > 1; --c)
        if (active_clusters(k, c) > 0) return c;
    return 1;
}

// Automatic split count of a kernel that fits once per SM.  A key range's
// CTAs form one cluster, and clusters only start where a GPC has that many
// free SMs, so a large cluster size can leave part of the units for a second
// or third wave (16-CTA clusters: seven at a time on GB300's 152 SMs).  The
// time of a launch goes about as waves / cluster size, waves = units over the
// clusters held at once; take the size at or below `want` that minimises it,
// and of equal ones the size with fewer waves (each wave repeats the ramp-up
// and the merge).  The waves run in lock step only when there are few units
// (at most half the resident CTAs), each split across many CTAs; with more
// units of uneven length the split balances the long ranges instead, so
// those launches keep `want`.  Kernels that fit twice per SM keep it too:
// there the second slot holds the next layer's CTAs (programmatic launch),
// which the wave count does not see.
int wave_cluster(const AttnKernel &k, long long units, int want) {
    const int resident = active_clusters(k, 1);
    if (want <= 1 || units <= 0 || resident > device_sms() || 2 * units > resident) return want;
    auto waves = [&](int c) {
        const long long a = active_clusters(k, c);
        return a > 0 ? (units + a - 1) / a : (long long)1 << 40;
    };
    int best = want;
    long long best_w = waves(want);
    for (int c = want - 1; c >= 1; --c) {
        const long long w = waves(c);
        // w / c against best_w / best, exactly
        const long long lhs = w * best, rhs = best_w * c;
        if (lhs < rhs || (lhs == rhs && w < best_w)) {
            best = c;
            best_w = w;
        }
    }
    return best;
}

int make_plan(const pkv_cache *c, int Hq, int S, int max_q_len, long long max_kv, int num_splits,
              unsigned flags, bool want_gm, Plan *pl) {
    int st = check_cache(c);
    if (st) return st;
    if (Hq <= 0 || Hq % c->kv_heads != 0) return PKV_EINVAL;
    if (S < 0 || S > 65535 || max_q_len <= 0 || max_kv <= 0 || num_splits < 0 || num_splits > kMaxSplitsGm)
        return PKV_EINVAL;
    const int D = c->head_dim;
    const int dp = D <= 64 ? 64 : D <= 128 ? 128 : 256;
    const int variant = c->dtype == PKV_F32 ? kSimtF32 : (flags & PKV_FLAG_SIMT) ? kSimtBf16 : kMmaBf16;
    pl->G = Hq / c->kv_heads;
    const long long rows_max = (long long)pl->G * max_q_len;
    if (rows_max > (1 << 20)) return PKV_EINVAL;
    pl->rows_max = (int)rows_max;
    // bf16 groups of at most 8 rows take the decode kernel (rows as the MMA's
    // N side; with PKV_FLAG_SIMT its CUDA-core variant).  Long buckets take
    // the decode configuration with more warps (class 5).
    const long long max_pages0 = (max_kv + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE + 1;
    // Wider bf16 groups with head_dim 128 take the tcgen05 tile (class 6)
    // unless the caller asks for the mma.sync one.
    const bool tc = variant == kMmaBf16 && rows_max > 8 && D == 128 && !(flags & PKV_FLAG_MMA_SYNC);
    const int rc = (variant != kSimtF32 && rows_max <= 8) ? (max_pages0 > 256 ? 5 : 4)
                   : tc ? 6
                   : rows_max <= 16 ? 0 : rows_max <= 32 ? 1 : rows_max <= 64 ? 2 : 3;
    pl->k = pick(variant, dp, rc);
    if (!pl->k.fn) return PKV_EUNSUPPORTED;
    pl->gm = want_gm && (rc == 4 || rc == 5);
    if (!pl->gm && num_splits > kMaxCluster) return PKV_EINVAL;
    pl->row_tiles = (int)((rows_max + pl->k.rows - 1) / pl->k.rows);
    if ((long long)c->kv_heads * pl->row_tiles > 65535) return PKV_EINVAL;
    const long long units = (long long)std::max(S, 1) * c->kv_heads * pl->row_tiles;
    pl->units = (int)units;
    const long long max_pages = (max_kv + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE + 1;
    long long n = num_splits;
    if (pl->gm) {
        // independent CTAs: one per SM across the launch (the next layer's
        // CTAs take the second slot of each SM), at least 4 pages each
        if (n == 0) n = std::min<long long>({(device_sms() + units - 1) / units, std::max<long long>(1, max_pages / 4),
                                             (long long)kMaxSplitsGm});
        pl->ncta = (int)std::max<long long>(1, std::min<long long>(n, max_pages));
        return PKV_OK;
    }
    if (n == 0) {
        // CTAs of this kernel that fit on one SM by shared memory.  The
        // tcgen05 tile aims at one wave: its fixed cost per CTA (first page
        // loads, cluster merge) is worth about 15 groups of 64 keys, and it
        // orders ranges longest first and runs short ones alone instead.
        const long long per_sm = std::max<long long>(1, 232448 / ((long long)pl->k.smem + 1024));
        const long long target = (long long)(pl->k.tc ? 1 : kTargetWaves) * device_sms() * per_sm;
        const long long want = (target + units - 1) / units;
        n = 1;
        while (n < want && n < kMaxCluster) n *= 2;
    }
    if ((rc == 4 || rc == 5) && num_splits == 0) {
        // decode kernel: no more CTAs than keep each of their warps two pages
        long long cap = 1;
        while (cap * 2 <= max_pages / 8 && cap * 2 <= kMaxCluster) cap *= 2;
        n = std::min(n, cap);
    }
    n = std::max<long long>(1, std::min<long long>(n, max_pages));
    pl->ncta = (int)n;
    return PKV_OK;
}

// Opt a kernel into its dynamic shared memory size and cluster sizes once per process.
int prepare_kernel(const AttnKernel &k) {
    static std::mutex mu;
    static const void *done[64];
    static int ndone = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ndone; ++i)
        if (done[i] == k.fn) return PKV_OK;
    // Ask for the largest shared-memory carveout so two CTAs fit on an SM:
    // with programmatic dependent launch the next layer's CTAs can then start
    // streaming their pages beside this layer's.
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess ||
        cudaFuncSetAttribute(k.fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(k.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ECUDA;
    }
    if (ndone < 64) done[ndone++] = k.fn;
    return PKV_OK;
}

int launch_status(cudaError_t e) {
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ECUDA;
    }
    return PKV_OK;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 4-D view (head_dim, kv_heads, 16, num_blocks) of one pool; a box is 128
// bytes of one row of one kv head across the 16 tokens of a page, loaded with
// 128-byte swizzling.
int encode_pool(CUtensorMap *map, const void *pool, const pkv_cache *c) {
    auto fn = encode_fn();
    if (!fn) return PKV_ECUDA;
    const int eb = elem_bytes(c->dtype);
    const cuuint64_t D = (cuuint64_t)c->head_dim, H = (cuuint64_t)c->kv_heads;
    cuuint64_t dims[4] = {D, H, (cuuint64_t)PKV_BLOCK_SIZE, (cuuint64_t)c->num_blocks};
    cuuint64_t strides[3] = {D * eb, H * D * eb, (cuuint64_t)PKV_BLOCK_SIZE * H * D * eb};
    cuuint32_t box[4] = {(cuuint32_t)(128 / eb), 1, (cuuint32_t)PKV_BLOCK_SIZE, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, c->dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    4, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ECUDA;
}

// 5-D view (64, 16, D / 64, kv_heads, num_blocks) of one pool, head_dim
// split into 64-element halves (or quarters) ordered after the 16 tokens: one
// box is a whole page tile of one kv head, laid out in shared memory exactly
// as the 4-D view's D / 64 boxes back to back (128-byte swizzle).  Needs
// head_dim a multiple of 64 (no partial last part).
int encode_pool_pages(CUtensorMap *map, const void *pool, const pkv_cache *c) {
    auto fn = encode_fn();
    if (!fn) return PKV_ECUDA;
    const int eb = elem_bytes(c->dtype);
    const cuuint64_t D = (cuuint64_t)c->head_dim, H = (cuuint64_t)c->kv_heads;
    const cuuint64_t part = 128 / eb;
    cuuint64_t dims[5] = {part, (cuuint64_t)PKV_BLOCK_SIZE, D / part, H, (cuuint64_t)c->num_blocks};
    cuuint64_t strides[4] = {H * D * eb, part * eb, D * eb, (cuuint64_t)PKV_BLOCK_SIZE * H * D * eb};
    cuuint32_t box[5] = {(cuuint32_t)part, (cuuint32_t)PKV_BLOCK_SIZE, (cuuint32_t)(D / part), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, c->dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    5, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ECUDA;
}

int attend_common(const pkv_cache *c, int layer, const void *q, const void *k_new, const void *v_new,
                  int Hq, int total_rows, const int *seq_info, int S, int max_q_len, long long max_kv,
                  int num_splits, float scale, int causal, int window, float *out, float *lse,
                  void *workspace, long long workspace_bytes, unsigned *err, unsigned flags, void *stream,
                  int *counters = nullptr) {
    Plan pl;
    int st = make_plan(c, Hq, S, max_q_len, max_kv, num_splits, flags, workspace != nullptr, &pl);
    if (st) return st;
    if (workspace && (!aligned16(workspace) || workspace_bytes < 0)) return PKV_EINVAL;
    if ((st = check_layer(c, layer))) return st;
    if (total_rows < 0 || window < 0 || (causal != 0 && causal != 1)) return PKV_EINVAL;
    if (!err || !out || (total_rows > 0 && (!q || !aligned16(q)))) return PKV_EINVAL;
    if (S > 0 && (!seq_info || !aligned16(seq_info))) return PKV_EINVAL;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return PKV_EINVAL;
    if (k_new && (!v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_EINVAL;
    if (S == 0 && total_rows == 0) return PKV_OK;
    const bool gm = pl.gm && S > 0 && pl.ncta > 1;
    const WsLayout wl = ws_layout((long long)S * c->kv_heads * pl.row_tiles, pl.ncta, pl.k.dp);
    if (gm && workspace_bytes < (long long)wl.total) return PKV_EINVAL;
    if ((st = prepare_kernel(pl.k))) return st;
    int ncta = S == 0 ? 1 : pl.gm ? pl.ncta : schedulable_cluster(pl.k, pl.ncta);
    if (S > 0 && !pl.gm && num_splits == 0) ncta = wave_cluster(pl.k, pl.units, ncta);

    AttendParams p;
    // bf16 page tiles come in one box when head_dim fills its padded width
    // exactly (128 or 256); otherwise, and for fp32, the 4-D view.
    const bool page_box = c->dtype == PKV_BF16 && c->head_dim == pl.k.dp && c->head_dim > 64 && !pl.k.tc;
    auto encode = [&](CUtensorMap *m, const void *pool) {
        return page_box ? encode_pool_pages(m, pool, c) : encode_pool(m, pool, c);
    };
    p.page_box = page_box ? 1 : 0;
    if (pl.k.tc) {
        // tcgen05 tile: K in 64-column boxes (one K-major tile per 4 pages), V in page boxes
        if ((st = encode_pool(&p.tmap_k, c->k[layer], c)) || (st = encode_pool_pages(&p.tmap_v, c->v[layer], c)))
            return st;
    } else if ((st = encode(&p.tmap_k, c->k[layer])) || (st = encode(&p.tmap_v, c->v[layer]))) {
        return st;
    }
    p.q = q;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_pool_w = c->k[layer];
    p.v_pool_w = c->v[layer];
    p.block_table = c->block_table;
    p.seq_info = reinterpret_cast<const int4 *>(seq_info);
    p.first_valid = c->first_valid;
    p.out = out;
    p.lse = lse;
    p.err = err;
    p.num_blocks = c->num_blocks;
    p.Hq = Hq;
    p.Hkv = c->kv_heads;
    p.D = c->head_dim;
    p.G = pl.G;
    p.total_rows = total_rows;
    p.S = S;
    p.max_seqs = c->max_seqs;
    p.mbps = c->max_blocks_per_seq;
    p.ring_rows = c->ring_rows;
    p.max_q_len = max_q_len;
    p.row_tiles = pl.row_tiles;
    p.causal = causal;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.ws_part = nullptr;
    p.ws_stat = nullptr;
    p.ws_flag = nullptr;
    p.ws_count = nullptr;
    if (gm) {
        char *base = reinterpret_cast<char *>(workspace);
        p.ws_part = reinterpret_cast<float *>(base + wl.part);
        p.ws_stat = reinterpret_cast<float2 *>(base + wl.stat);
        p.ws_flag = reinterpret_cast<int *>(base + wl.flag);
        p.ws_count = counters ? counters : reinterpret_cast<int *>(base + wl.count);
    }
    p.k_next = p.v_next = nullptr;
    p.pf_next = 0;
    if ((flags & PKV_FLAG_PREFETCH_NEXT) && layer + 1 < c->num_layers && S > 0 && !check_layer(c, layer + 1)) {
        p.k_next = c->k[layer + 1];
        p.v_next = c->v[layer + 1];
        // L2 budget: ~48 MB; a page is warmed once for all kv heads (K and V).
        const long long page = 2LL * PKV_BLOCK_SIZE * c->kv_heads * c->head_dim * elem_bytes(c->dtype);
        p.pf_next = (int)std::max<long long>(0, std::min<long long>(1 << 20, (48LL << 20) / ((long long)ncta * S * page)));
    }

    cudaLaunchConfig_t cfg = {};
    if (S == 0)
        cfg.gridDim = dim3(1, 1, 1);
    else
        cfg.gridDim = dim3((unsigned)ncta, (unsigned)(c->kv_heads * pl.row_tiles), (unsigned)S);
    cfg.blockDim = dim3((unsigned)pl.k.threads);
    cfg.dynamicSmemBytes = pl.k.smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (ncta > 1 && !gm) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)ncta;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (flags & PKV_FLAG_PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = (unsigned)na;
    void *args[] = {&p};
    return launch_status(cudaLaunchKernelExC(&cfg, pl.k.fn, args));
}

int copy_rows(const void *s0, const void *s1, void *d0, void *d1, long long n, int H, int row_bytes,
              long long ss, long long sh, long long ds, long long dh, void *stream) {
    if (n <= 0) return PKV_OK;
    CopyParams p{reinterpret_cast<const char *>(s0), reinterpret_cast<const char *>(s1),
                 reinterpret_cast<char *>(d0), reinterpret_cast<char *>(d1), n, H, row_bytes / 16,
                 ss, sh, ds, dh};
    const long long total = 2 * n * H * (row_bytes / 16);
    const long long blocks = std::min<long long>((total + 255) / 256, (long long)kDefaultSms * 8);
    strided_copy_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return launch_status(cudaSuccess);
}

// Fixed split-merge scratch of pkv_append_attend_noalloc: file-scope device
// memory (zero at module load; every call leaves its counters at zero), so
// that entry point never allocates.
// The arrival counters live in an array of their own, so they are zero at
// every call whatever shape the previous call had.
constexpr long long kStaticScratchBytes = 8ll << 20;
constexpr int kStaticUnits = 4096;
static __device__ __align__(256) unsigned char g_split_scratch[kStaticScratchBytes];
static __device__ __align__(256) int g_split_counters[kStaticUnits];

// Device addresses of g_split_scratch and g_split_counters in the current
// context.  Looked up on every call: the lookup is a host-side query, and an
// address cached from an earlier context (before a cudaDeviceReset, say)
// would be stale.  The first lookup on a device loads the library's module.
bool static_scratch(void **scratch, int **counters) {
    void *a = nullptr, *b = nullptr;
    if (cudaGetSymbolAddress(&a, g_split_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&b, g_split_counters) != cudaSuccess || !a || !b) {
        cudaGetLastError();
        return false;
    }
    *scratch = a;
    *counters = reinterpret_cast<int *>(b);
    return true;
}

}  // namespace

extern "C" {

int64_t pkv_bucket_for(int64_t length) {
    // vLLM-Omni paged_decode.py: BUCKETS then TAIL_STEP-sized growth.
    static const int64_t buckets[] = {512, 1024, 2048, 4096, 8192};
    for (int64_t b : buckets)
        if (length <= b) return b;
    const int64_t tail = 2048;
    return 8192 + ((length - 8192 + tail - 1) / tail) * tail;
}

const char *pkv_status_str(int s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_EMPTY: return "empty: nothing to copy";
        case PKV_SAME_BUCKET: return "same bucket: no resize needed";
        case PKV_EINVAL: return "invalid argument";
        case PKV_EUNSUPPORTED: return "unsupported dtype or head_dim";
        case PKV_ECUDA: return "CUDA launch or copy failed";
        case PKV_ECAPACITY: return "capacity exceeded";
        case PKV_ESTALE: return "caches describe different shapes";
    }
    return "unknown status";
}

int pkv_append(const pkv_cache *c, int32_t layer, const void *k_new, const void *v_new, int32_t total_rows,
               const int32_t *seq_info, int32_t S, int32_t window, uint32_t *err, void *stream) {
    int st = check_cache(c);
    if (st) return st;
    if ((st = check_layer(c, layer))) return st;
    if (S < 0 || total_rows < 0 || window < 0 || !err) return PKV_EINVAL;
    if (S == 0) return PKV_OK;
    if (!seq_info || !aligned16(seq_info)) return PKV_EINVAL;
    if (total_rows > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_EINVAL;
    AppendParams p;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_pool = c->k[layer];
    p.v_pool = c->v[layer];
    p.block_table = c->block_table;
    p.seq_info = reinterpret_cast<const int4 *>(seq_info);
    p.err = err;
    p.num_blocks = c->num_blocks;
    p.row_bytes = c->kv_heads * c->head_dim * elem_bytes(c->dtype);
    p.total_rows = total_rows;
    p.S = S;
    p.max_seqs = c->max_seqs;
    p.mbps = c->max_blocks_per_seq;
    p.ring_rows = c->ring_rows;
    p.window = window;
    append_kernel<<<(unsigned)S, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return launch_status(cudaSuccess);
}

int pkv_attend_varlen(const pkv_cache *c, int32_t layer, const void *q, int32_t Hq, int32_t total_rows,
                      const int32_t *seq_info, int32_t S, int32_t max_q_len, int64_t max_kv, int32_t num_splits,
                      float scale, int32_t causal, int32_t window, float *out, float *lse, void *workspace,
                      int64_t workspace_bytes, uint32_t *err, uint32_t flags, void *stream) {
    return attend_common(c, layer, q, nullptr, nullptr, Hq, total_rows, seq_info, S, max_q_len, max_kv,
                         num_splits, scale, causal, window, out, lse, workspace, workspace_bytes, err, flags,
                         stream);
}

int pkv_append_attend(const pkv_cache *c, int32_t layer, const void *q, const void *k_new, const void *v_new,
                      int32_t Hq, int32_t total_rows, const int32_t *seq_info, int32_t S, int32_t max_q_len,
                      int64_t max_kv, int32_t num_splits, float scale, int32_t causal, int32_t window,
                      float *out, float *lse, void *workspace, int64_t workspace_bytes, uint32_t *err,
                      uint32_t flags, void *stream) {
    if (total_rows > 0 && (!k_new || !v_new)) return PKV_EINVAL;
    return attend_common(c, layer, q, total_rows > 0 ? k_new : nullptr, total_rows > 0 ? v_new : nullptr, Hq,
                         total_rows, seq_info, S, max_q_len, max_kv, num_splits, scale, causal, window, out, lse,
                         workspace, workspace_bytes, err, flags, stream);
}

int pkv_append_attend_noalloc(const pkv_cache *c, int32_t layer, const void *q, const void *k_new,
                              const void *v_new, int32_t Hq, int32_t total_rows, const int32_t *seq_info, int32_t S,
                              int32_t max_q_len, int64_t max_kv, int32_t num_splits, float scale, int32_t causal,
                              int32_t window, float *out, float *lse, uint32_t *err, uint32_t flags, void *stream) {
    const int64_t need = pkv_attend_workspace_bytes(c, Hq, S, max_q_len, max_kv, num_splits, flags);
    if (need < 0) return (int)need;
    if (need > 0) {
        // One arrival counter per (segment, kv head, row tile) range: the
        // same count the kernel indexes them by.
        Plan pl;
        const int st = make_plan(c, Hq, S, max_q_len, max_kv, num_splits, flags, true, &pl);
        if (st) return st;
        if (need > kStaticScratchBytes || (long long)S * c->kv_heads * pl.row_tiles > kStaticUnits)
            return PKV_ECAPACITY;  // rejected before any launch
    }
    void *ws = nullptr;
    int *counters = nullptr;
    if (need > 0 && !static_scratch(&ws, &counters)) return PKV_ECUDA;
    if (total_rows > 0 && (!k_new || !v_new)) return PKV_EINVAL;
    return attend_common(c, layer, q, total_rows > 0 ? k_new : nullptr, total_rows > 0 ? v_new : nullptr, Hq,
                         total_rows, seq_info, S, max_q_len, max_kv, num_splits, scale, causal, window, out, lse, ws,
                         need > 0 ? kStaticScratchBytes : 0, err, flags, stream, counters);
}

int64_t pkv_attend_workspace_bytes(const pkv_cache *c, int32_t Hq, int32_t S, int32_t max_q_len, int64_t max_kv,
                                   int32_t num_splits, uint32_t flags) {
    Plan pl;
    const int st = make_plan(c, Hq, S, max_q_len, max_kv, num_splits, flags, true, &pl);
    if (st) return st;
    if (!pl.gm || S == 0 || pl.ncta <= 1) return 0;
    return (int64_t)ws_layout((long long)S * c->kv_heads * pl.row_tiles, pl.ncta, pl.k.dp).total;
}

int pkv_seq_clone(const pkv_cache *c, int32_t src_col, int32_t dst_col, int64_t n, uint32_t *err, void *stream) {
    int st = check_cache(c);
    if (st) return st;
    if (!err || n < 0 || src_col < 0 || src_col >= c->max_seqs || dst_col < 0 || dst_col >= c->max_seqs)
        return PKV_EINVAL;
    if (!c->ring_rows && n > (long long)c->max_blocks_per_seq * PKV_BLOCK_SIZE) return PKV_ECAPACITY;
    if (n > INT32_MAX - PKV_BLOCK_SIZE) return PKV_EINVAL;
    for (int l = 0; l < c->num_layers; ++l)
        if ((st = check_layer(c, l))) return st;
    if (n == 0 || src_col == dst_col) return PKV_OK;
    const long long lo = (c->ring_rows && n > c->ring_rows) ? n - c->ring_rows : 0;
    const int row_chunks = c->kv_heads * c->head_dim * elem_bytes(c->dtype) / 16;
    for (int l0 = 0; l0 < c->num_layers; l0 += kCloneLayers) {
        CloneParams p = {};
        p.layers = std::min(kCloneLayers, c->num_layers - l0);
        for (int i = 0; i < p.layers; ++i) {
            p.k[i] = reinterpret_cast<char *>(c->k[l0 + i]);
            p.v[i] = reinterpret_cast<char *>(c->v[l0 + i]);
        }
        p.block_table = c->block_table;
        p.err = err;
        p.num_blocks = c->num_blocks;
        p.lo = lo;
        p.n = n;
        p.row_chunks = row_chunks;
        p.mbps = c->max_blocks_per_seq;
        p.ring_rows = c->ring_rows;
        p.src = src_col;
        p.dst = dst_col;
        const long long total = 2LL * p.layers * (n - lo) * row_chunks;
        const long long blocks = std::max<long long>(1, std::min<long long>((total + 255) / 256, (long long)device_sms() * 8));
        seq_clone_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
        if ((st = launch_status(cudaSuccess))) return st;
    }
    return PKV_OK;
}

int pkv_rewind(const pkv_cache *c, int32_t *seq_info, int32_t n, const int32_t *amount, int32_t window,
               uint32_t *err, void *stream) {
    int st = check_cache(c);
    if (st) return st;
    if (n < 0 || window < 0 || !err) return PKV_EINVAL;
    if (n == 0) return PKV_OK;
    if (!seq_info || !aligned16(seq_info) || !amount || (reinterpret_cast<uintptr_t>(amount) & 3u)) return PKV_EINVAL;
    rewind_kernel<<<(unsigned)((n + 127) / 128), 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<int4 *>(seq_info), amount, n, c->ring_rows, window, err);
    return launch_status(cudaSuccess);
}

int pkv_seqinfo_from_seqused(const int32_t *cu, const int32_t *used, int32_t n, int32_t *out, void *stream) {
    if (n < 0) return PKV_EINVAL;
    if (n == 0) return PKV_OK;
    if (!cu || !used || !out || !aligned16(out)) return PKV_EINVAL;
    seqinfo_from_seqused_kernel<<<(unsigned)((n + 127) / 128), 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        cu, used, n, reinterpret_cast<int4 *>(out));
    return launch_status(cudaSuccess);
}

int pkv_advance(int32_t *seq_info, int32_t n, void *stream) {
    if (n < 0) return PKV_EINVAL;
    if (n == 0) return PKV_OK;
    if (!seq_info || !aligned16(seq_info)) return PKV_EINVAL;
    advance_kernel<<<(unsigned)((n + 127) / 128), 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<int4 *>(seq_info), n);
    return launch_status(cudaSuccess);
}

int pkv_resize_bucket(const pkv_cache *o, pkv_cache *n, int64_t old_len, void *stream) {
    int st = check_cache(o);
    if (st) return st;
    if ((st = check_cache(n))) return st;
    if (o->num_layers != n->num_layers || o->kv_heads != n->kv_heads || o->head_dim != n->head_dim ||
        o->dtype != n->dtype)
        return PKV_ESTALE;
    if (o->ring_rows || n->ring_rows) return PKV_EINVAL;
    if (old_len < 0) return PKV_EINVAL;
    if (n->bucket == o->bucket) return PKV_SAME_BUCKET;
    if (old_len > o->num_blocks * PKV_BLOCK_SIZE || old_len > n->num_blocks * PKV_BLOCK_SIZE) return PKV_ECAPACITY;
    const int row = o->head_dim * elem_bytes(o->dtype);
    const long long tok = (long long)o->kv_heads * row;
    for (int l = 0; l < o->num_layers; ++l) {
        if (check_layer(o, l) || check_layer(n, l)) return PKV_EINVAL;
    }
    for (int l = 0; l < o->num_layers; ++l) {
        st = copy_rows(o->k[l], o->v[l], n->k[l], n->v[l], old_len, o->kv_heads, row, tok, row, tok, row, stream);
        if (st) return st;
    }
    n->generation = o->generation + 1;
    return PKV_OK;
}

int pkv_load_prefix(const pkv_cache *c, const void *const *keys, const void *const *values, int64_t n,
                    int64_t stride_s, int64_t stride_h, void *stream) {
    int st = check_cache(c);
    if (st) return st;
    if (n == 0 || !keys) return PKV_EMPTY;
    if (n < 0 || !values) return PKV_EINVAL;
    if (n > c->num_blocks * PKV_BLOCK_SIZE) return PKV_ECAPACITY;
    const int eb = elem_bytes(c->dtype);
    const int row = c->head_dim * eb;
    if (stride_s < 0 || stride_h < 0 || (stride_s * eb) % 16 || (stride_h * eb) % 16) return PKV_EINVAL;
    for (int l = 0; l < c->num_layers; ++l) {
        if (check_layer(c, l) || !keys[l] || !values[l] || !aligned16(keys[l]) || !aligned16(values[l]))
            return PKV_EINVAL;
    }
    const long long tok = (long long)c->kv_heads * row;
    for (int l = 0; l < c->num_layers; ++l) {
        st = copy_rows(keys[l], values[l], c->k[l], c->v[l], n, c->kv_heads, row, stride_s * eb, stride_h * eb,
                       tok, row, stream);
        if (st) return st;
    }
    return PKV_OK;
}

int pkv_to_contiguous(const pkv_cache *c, int32_t layer, int64_t n, void *keys_out, void *values_out,
                      void *stream) {
    int st = check_cache(c);
    if (st) return st;
    if ((st = check_layer(c, layer))) return st;
    if (n < 0 || n > c->num_blocks * PKV_BLOCK_SIZE) return PKV_ECAPACITY;
    if (n == 0) return PKV_OK;
    if (!keys_out || !values_out || !aligned16(keys_out) || !aligned16(values_out)) return PKV_EINVAL;
    const int row = c->head_dim * elem_bytes(c->dtype);
    const long long tok = (long long)c->kv_heads * row;
    return copy_rows(c->k[layer], c->v[layer], keys_out, values_out, n, c->kv_heads, row, tok, row, row,
                     n * row, stream);
}

}  // extern "C"
