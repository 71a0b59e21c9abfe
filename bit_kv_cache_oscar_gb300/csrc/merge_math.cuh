// The merge's own 2^x, shared by oscar_merge and the decode launch that merges in its last
// cluster, so that both give the same bits.
#pragma once

#include "oscar_internal.cuh"

namespace oscar {

// 2^x by Cody–Waite range reduction and a degree-7 Taylor polynomial:
// n = rint(x), f = x - n in [-1/2, 1/2], 2^f = sum_k (f ln2)^k / k! by Horner,
// 2^x = 2^f * 2^n.  Coefficients: binary32 roundings of (ln 2)^k / k!.
// x < -125 (and -inf) gives 0.
__device__ __forceinline__ float exp2_taylor(float x) {
    if (!(x >= -125.0f)) return 0.0f;
    if (x > 127.0f) return INFINITY;
    const float n = rintf(x);
    const float f = __fsub_rn(x, n);
    float p = 0x1.ffcbfcp-17f;                 // (ln2)^7 / 7!
    p = __fmaf_rn(p, f, 0x1.430912p-13f);      // (ln2)^6 / 6!
    p = __fmaf_rn(p, f, 0x1.5d87fep-10f);      // (ln2)^5 / 5!
    p = __fmaf_rn(p, f, 0x1.3b2ab6p-7f);       // (ln2)^4 / 4!
    p = __fmaf_rn(p, f, 0x1.c6b08ep-5f);       // (ln2)^3 / 3!
    p = __fmaf_rn(p, f, 0x1.ebfbe0p-3f);       // (ln2)^2 / 2!
    p = __fmaf_rn(p, f, 0x1.62e430p-1f);       // ln2
    p = __fmaf_rn(p, f, 1.0f);
    const float two_n = __uint_as_float((uint32_t)((int)n + 127) << 23);
    return __fmul_rn(p, two_n);
}

}  // namespace oscar
