// Internal declarations of liboscar.so: device helpers and the launch functions
// that api.cu calls after validating arguments.  Not installed, not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "oscar.h"

namespace oscar {

constexpr int kHeadDim = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ void flag_status(int32_t *status, int32_t bit) {
    if (status) atomicOr(status, bit);
}

// Page-aligned split of the history [sink, h_end) of one request: split s of S
// covers logical pages [first + s*per, first + (s+1)*per) clipped to the history.
struct SplitRange {
    int lo, hi;   // token range [lo, hi), empty if lo >= hi
};

__device__ __forceinline__ SplitRange history_split(int sink, int h_end, int page_size, int S, int s) {
    int first = sink / page_size;
    int last = (h_end + page_size - 1) / page_size;
    int n = last - first;
    SplitRange r{0, 0};
    if (n <= 0) return r;
    int per = (n + S - 1) / S;
    int a = (first + s * per) * page_size;
    int b = (first + (s + 1) * per) * page_size;
    r.lo = a > sink ? a : sink;
    r.hi = b < h_end ? b : h_end;
    if (r.lo >= r.hi) r.lo = r.hi = 0;
    return r;
}

// Same rule over [0, T) for the all-BF16 comparison kernel.
__device__ __forceinline__ SplitRange full_split(int T, int page_size, int S, int s) {
    int n = (T + page_size - 1) / page_size;
    SplitRange r{0, 0};
    if (n <= 0) return r;
    int per = (n + S - 1) / S;
    r.lo = s * per * page_size;
    int b = (s + 1) * per * page_size;
    r.hi = b < T ? b : T;
    if (r.lo >= r.hi) r.lo = r.hi = 0;
    return r;
}

// Clamp the per-request lengths the way every kernel reads them; flags bad input.
__device__ __forceinline__ void read_lengths(const int32_t *seq_len, const int32_t *hist_end, int b, int sink,
                                             int max_tokens, int32_t *status, int &T, int &h) {
    T = seq_len[b];
    h = hist_end ? hist_end[b] : 0;
    bool bad = false;
    if (T < 0) { T = 0; bad = true; }
    if (T > max_tokens) { T = max_tokens; bad = true; }
    int lo = sink < T ? sink : T;
    if (hist_end) {
        if (h < lo) { h = lo; bad = bad || (T >= sink); }
        if (h > T) { h = T; bad = true; }
    }
    if (bad && threadIdx.x == 0) flag_status(status, OSCAR_DEV_BAD_LENGTH);
}

// Record the one-line reason returned by oscar_last_error_string() and return `code`.
oscar_status_t set_last_error(oscar_status_t code, const char *msg);

// ---------------------------------------------------------------- launches --

struct Int2PoolView {
    const uint8_t *codes_k, *codes_v;
    const uint16_t *scale_k, *zero_k, *scale_v, *zero_v;
    int n_pages;
};

struct Bf16PoolView {
    const uint16_t *k, *v;
    int n_pages;
};

struct PartialsView {
    float *m, *l, *acc;
    int S;
};

cudaError_t launch_demote(const oscar_layout_t &L, Bf16PoolView src, const int32_t *bf16_pt,
                          const oscar_int2_pool_t &dst, const int32_t *int2_pt, int max_pages, int batch,
                          const int32_t *req_idx, const int32_t *pos, int n, const float *RK,
                          const float *RV, float cK, float cV, float *rot_out, int32_t *status,
                          cudaStream_t st);

cudaError_t launch_quantize_rotated(const oscar_layout_t &L, const float *x, int n, float clip, uint8_t *codes,
                                    uint16_t *scale, uint16_t *zero, cudaStream_t st);

cudaError_t launch_rotate_q(const oscar_layout_t &L, const uint16_t *q, const float *RK, int batch,
                            float *q_rot, cudaStream_t st);

cudaError_t launch_int2_attention(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool,
                                  const int32_t *pt, int max_pages, const int32_t *seq_len,
                                  const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                  int32_t *status, cudaStream_t st);

// mode 0: sink + recent of each request into slot S; mode 1: all of [0, T) split S ways.
cudaError_t launch_bf16_attention(const oscar_layout_t &L, const uint16_t *q, Bf16PoolView pool,
                                  const int32_t *pt, int max_pages, const int32_t *seq_len,
                                  const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                  int mode, int32_t *status, cudaStream_t st);

cudaError_t launch_merge(const oscar_layout_t &L, PartialsView p, const float *RV, int batch, uint16_t *out,
                         float *out_f32, float *lse, cudaStream_t st);

}  // namespace oscar
