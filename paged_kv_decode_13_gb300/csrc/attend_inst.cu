// Instantiates the attention kernel for one (variant, padded head_dim) pair.
// Built once per pair with -DPKV_INST_VARIANT=<0|1|2> -DPKV_INST_DP=<64|128|256>
// so the configurations compile in parallel.
//
// Per row class the tuple is (row tiles MT, key groups KW, stages NST): stage
// counts keep a CTA near 100-135 KB of shared memory where the page size
// allows (two CTAs per SM), and fp32 / wide heads drop to fewer key groups or
// a 64-row cap to stay inside the 227 KB limit.  The 128-row tensor-core
// class takes eight stages: its ring aliases the key-group merge buffer,
// which is at least as large, so the deeper ring costs no shared memory.
#include "attend.cuh"
#include "decode.cuh"
#include "launch.h"
#include "verify.cuh"

#ifndef PKV_INST_VARIANT
#error "PKV_INST_VARIANT not set"
#endif
#ifndef PKV_INST_DP
#error "PKV_INST_DP not set"
#endif

namespace pkv {

template <class C>
static AttnKernel info() {
    static_assert(C::kSmemBytes <= 232448, "exceeds the per-CTA shared memory limit");
    return AttnKernel{reinterpret_cast<const void *>(&attend_kernel<C>), C::kThreads, C::kSmemBytes,
                      C::kRows, C::DP, C::MMA};
}

// Decode kernel for groups of at most 8 query rows (row class 4; class 5 for
// long buckets, with more warps where head_dim 128 allows).  The CUDA-core
// variant keeps the tensor-core one's warps and stages.
template <class C>
static AttnKernel dinfo() {
    static_assert(C::kSmemBytes <= 232448, "exceeds the per-CTA shared memory limit");
    return AttnKernel{reinterpret_cast<const void *>(&decode_kernel<C>), C::kThreads, C::kSmemBytes,
                      C::kRows, C::DP, !C::SIMT};
}

// tcgen05 tile for wide bf16 groups with head_dim 128 (row class 6).
template <class C>
static AttnKernel vinfo() {
    static_assert(C::kSmemBytes <= 232448, "exceeds the per-CTA shared memory limit");
    return AttnKernel{reinterpret_cast<const void *>(&verify_kernel<C>), C::kThreads, C::kSmemBytes,
                      C::kRows, C::DP, true, true};
}

using B16 = __nv_bfloat16;
#define CFG(T, MT, KW, NST, MMA) info<AttnCfg<T, PKV_INST_DP, MT, KW, NST, MMA>>()

#define PICK_NAME2(V, DP) pick_##V##_##DP
#define PICK_NAME(V, DP) PICK_NAME2(V, DP)

AttnKernel PICK_NAME(PKV_INST_VARIANT, PKV_INST_DP)(int rc) {
#if PKV_INST_VARIANT == 0
#if PKV_INST_DP == 64
    {
        if (rc >= 4) return dinfo<DecCfg<64, 4, 6>>();
        if (rc == 0) return CFG(B16, 1, 4, 4, true);
        if (rc == 1) return CFG(B16, 2, 2, 4, true);
        if (rc == 2) return CFG(B16, 4, 1, 4, true);
        return CFG(B16, 8, 1, 8, true);
    }
#elif PKV_INST_DP == 128
    {
        if (rc == 6) return vinfo<VfyCfg<5, 6>>();
        if (rc == 5) return dinfo<DecCfg<128, 6, 2>>();
        if (rc == 4) return dinfo<DecCfg<128, 4, 3>>();
        if (rc == 0) return CFG(B16, 1, 4, 3, true);
        if (rc == 1) return CFG(B16, 2, 2, 4, true);
        if (rc == 2) return CFG(B16, 4, 1, 4, true);
        return CFG(B16, 8, 1, 8, true);
    }
#else
    {
        // one CTA per SM at this width whatever the split: six warps of two
        // stages (192 KB in flight) spread the per-page MMA latency over
        // more warps than four of three (long ranges: 327 against 332 us)
        if (rc >= 4) return dinfo<DecCfg<256, 6, 2>>();
        if (rc == 0) return CFG(B16, 1, 4, 2, true);
        if (rc == 1) return CFG(B16, 2, 2, 3, true);
        if (rc == 2) return CFG(B16, 4, 1, 4, true);
        return CFG(B16, 8, 1, 8, true);
    }
#endif
#elif PKV_INST_VARIANT == 1
#if PKV_INST_DP == 64
    {
        if (rc >= 4) return dinfo<DecCfg<64, 4, 6, true>>();
        if (rc == 0) return CFG(B16, 1, 4, 4, false);
        if (rc == 1) return CFG(B16, 2, 2, 4, false);
        if (rc == 2) return CFG(B16, 4, 1, 4, false);
        return CFG(B16, 8, 1, 4, false);
    }
#elif PKV_INST_DP == 128
    {
        if (rc == 5) return dinfo<DecCfg<128, 6, 2, true>>();
        if (rc == 4) return dinfo<DecCfg<128, 4, 3, true>>();
        if (rc == 0) return CFG(B16, 1, 4, 3, false);
        if (rc == 1) return CFG(B16, 2, 2, 4, false);
        if (rc == 2) return CFG(B16, 4, 1, 4, false);
        return CFG(B16, 8, 1, 4, false);
    }
#else
    {
        if (rc >= 4) return dinfo<DecCfg<256, 6, 2, true>>();
        if (rc == 0) return CFG(B16, 1, 4, 2, false);
        if (rc == 1) return CFG(B16, 2, 2, 3, false);
        return CFG(B16, 4, 1, 4, false);
    }
#endif
#else
#if PKV_INST_DP == 64
    {
        if (rc == 0) return CFG(float, 1, 4, 3, false);
        if (rc == 1) return CFG(float, 2, 2, 4, false);
        if (rc == 2) return CFG(float, 4, 1, 4, false);
        return CFG(float, 8, 1, 4, false);
    }
#elif PKV_INST_DP == 128
    {
        if (rc == 0) return CFG(float, 1, 4, 2, false);
        if (rc == 1) return CFG(float, 2, 2, 3, false);
        if (rc == 2) return CFG(float, 4, 1, 4, false);
        return CFG(float, 8, 1, 4, false);
    }
#else
    {
        if (rc == 0) return CFG(float, 1, 2, 2, false);
        if (rc == 1) return CFG(float, 2, 2, 2, false);
        return CFG(float, 4, 1, 2, false);
    }
#endif
#endif
}

}  // namespace pkv
