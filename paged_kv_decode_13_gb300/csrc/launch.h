// Host-side view of the compiled attention kernels.
#pragma once

#include <stddef.h>

namespace pkv {

// One compiled attention configuration.
struct AttnKernel {
    const void *fn;   // __global__ attend_kernel<...>
    int threads;
    size_t smem;      // dynamic shared memory bytes
    int rows;         // query rows per CTA (16 * row tiles)
    int dp;           // padded head_dim
    bool mma;
    bool tc;          // tcgen05 tile (verify_kernel): reads pages through the 4-D view
};

// Compute variants.
enum Variant { kMmaBf16 = 0, kSimtBf16 = 1, kSimtF32 = 2 };

// Row class: 0 for <= 16 query rows per (segment, kv head), 1 for <= 32,
// 2 for <= 64, 3 for more (128 per CTA, extra CTAs along the rows beyond);
// 4 for <= 8 bf16 rows (decode_kernel, tensor-core or CUDA-core variant), 5
// the same for buckets over 256 pages; 6 for more than 8 rows on the tcgen05 tile
// (verify_kernel, bf16 with head_dim 128: 128 rows per CTA).
#define PKV_DECLARE_PICK(V, DP) AttnKernel pick_##V##_##DP(int row_class);
PKV_DECLARE_PICK(0, 64)
PKV_DECLARE_PICK(0, 128)
PKV_DECLARE_PICK(0, 256)
PKV_DECLARE_PICK(1, 64)
PKV_DECLARE_PICK(1, 128)
PKV_DECLARE_PICK(1, 256)
PKV_DECLARE_PICK(2, 64)
PKV_DECLARE_PICK(2, 128)
PKV_DECLARE_PICK(2, 256)
#undef PKV_DECLARE_PICK

}  // namespace pkv
