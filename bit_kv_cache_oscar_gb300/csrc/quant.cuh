// The INT2 quantizer of one 128-channel row, shared by every kernel that writes the pool.
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — rotate,
// clip, quantize, pack (4 x 2-bit per byte); estelledc notes "案例 2" — clip ratios.
// Per group of g channels: lo = c*min, hi = c*max (min/max read a signed zero as +0),
// zero = bf16(lo), scale = bf16((hi - lo)/3), code = clamp(rint((y - zero)/scale), 0, 3)
// with the stored bf16 zero and scale, code 0 when scale = 0; code i of the row sits at
// bits 2*(i mod 4) of byte i/4.  Explicit round-to-nearest intrinsics fix every rounding.
// With a non-uniform codebook lv (cb = true; OSCAR news article, closing paragraph on the
// Lloyd-Max codebook) the zero and scale are the same and the code is the number of fp32
// midpoints (lv[k] + lv[k+1]) * 0.5 at or below u = (y - zero)/scale (code 0 for NaN or scale 0).
#pragma once

#include "oscar_internal.cuh"

namespace oscar {

// One channel per thread: j = this thread's channel (0..127) within a group of 128 threads
// that are 4 whole warps (warp j/32 of them); sync() synchronizes exactly those 128 threads
// (it is called only when group > 32).  red: 8 floats of shared scratch for the group.
template <typename Sync>
__device__ __forceinline__ void quantize_row_store(float y, float clip, int group, bool store, uint8_t *codes_row,
                                                   uint16_t *scale_row, uint16_t *zero_row, float *red, int j,
                                                   Sync sync, bool cb = false, float4 lv = float4{}) {
    const int lane = j & 31, warp = j >> 5;
    float mn = y, mx = y;
#pragma unroll
    for (int o = 16; o; o >>= 1) {               // a warp is one group at g = 32, part of one above
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (group > 32) {
        sync();
        if (lane == 0) {
            red[warp] = mn;
            red[4 + warp] = mx;
        }
        sync();
        const int wpg = group >> 5;              // warps per group
        const int w0 = (warp / wpg) * wpg;
        mn = red[w0];
        mx = red[4 + w0];
        for (int w = w0 + 1; w < w0 + wpg; ++w) {
            mn = fminf(mn, red[w]);
            mx = fmaxf(mx, red[4 + w]);
        }
    }
    mn = __fadd_rn(mn, 0.0f);                    // a signed zero is read as +0
    mx = __fadd_rn(mx, 0.0f);
    const float lo = __fmul_rn(clip, mn);        // clipped range c*[min, max]
    const float hi = __fmul_rn(clip, mx);
    const float step = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    const uint16_t zb = f32_to_bf16_rn(lo);
    const uint16_t sb = f32_to_bf16_rn(step);
    const float z = bf16_to_f32(zb), s = bf16_to_f32(sb);
    int c = 0;
    if (s != 0.0f) {
        const float u = __fdiv_rn(__fsub_rn(y, z), s);
        if (cb) {
            const float t0 = __fmul_rn(__fadd_rn(lv.x, lv.y), 0.5f), t1 = __fmul_rn(__fadd_rn(lv.y, lv.z), 0.5f);
            const float t2 = __fmul_rn(__fadd_rn(lv.z, lv.w), 0.5f);
            c = (u >= t0) + (u >= t1) + (u >= t2);
        } else {
            const float r = rintf(u);
            c = r >= 3.0f ? 3 : (r >= 0.0f ? (int)r : 0);
        }
    }
    uint32_t v = (uint32_t)c << (2 * (lane & 3));
    v |= __shfl_xor_sync(0xffffffffu, v, 1);
    v |= __shfl_xor_sync(0xffffffffu, v, 2);
    if (store) {
        if ((lane & 3) == 0) codes_row[j >> 2] = (uint8_t)v;
        if ((j % group) == 0) {
            scale_row[j / group] = sb;
            zero_row[j / group] = zb;
        }
    }
}

}  // namespace oscar
