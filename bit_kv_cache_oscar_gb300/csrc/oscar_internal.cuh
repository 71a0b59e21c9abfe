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

constexpr int kTileTokens = 16;   // split granularity: 16-token tiles at absolute positions 16i..16i+15

// Balanced split of [lo_tok, hi_tok) into S parts of whole tiles: with first = lo_tok/16 and
// n = ceil(hi_tok/16) - first tiles, part s covers tiles [first + floor(s*n/S), first +
// floor((s+1)*n/S)), clipped to [lo_tok, hi_tok).  lo_tok must be a multiple of 16.
struct SplitRange {
    int lo, hi;   // token range [lo, hi), empty if lo >= hi
    int tile_lo, tile_hi;
};

__device__ __forceinline__ SplitRange tile_split(int lo_tok, int hi_tok, int S, int s) {
    SplitRange r{0, 0, 0, 0};
    const int first = lo_tok / kTileTokens;
    const int n = (hi_tok + kTileTokens - 1) / kTileTokens - first;
    if (n <= 0) return r;
    const int a = first + (int)(((long long)s * n) / S);
    const int b = first + (int)(((long long)(s + 1) * n) / S);
    r.lo = a * kTileTokens > lo_tok ? a * kTileTokens : lo_tok;
    r.hi = b * kTileTokens < hi_tok ? b * kTileTokens : hi_tok;
    r.tile_lo = a;
    r.tile_hi = b;
    if (r.lo >= r.hi) r.lo = r.hi = r.tile_lo = r.tile_hi = 0;
    return r;
}

// History split s of S of one request: [sink, h_end) (sink is a multiple of 16).
__device__ __forceinline__ SplitRange history_split(int sink, int h_end, int S, int s) {
    return tile_split(sink, h_end, S, s);
}

// Same rule over [0, T) for the all-BF16 comparison kernel.
__device__ __forceinline__ SplitRange full_split(int T, int S, int s) { return tile_split(0, T, S, s); }

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

// Raise (never lower) a kernel's dynamic shared-memory limit on the current device to `smem`.
// One kernel serves layouts of different sizes, and a lower setting would make an earlier,
// larger launch configuration fail; process-wide, safe across host threads.
cudaError_t ensure_dyn_smem(const void *kern, int smem);

// Process-wide launch-overlap switch (programmatic dependent launch); see oscar.h.
bool launch_overlap();

// Launch configuration with the programmatic-serialization attribute when overlap is on.
// `attrs` must have room for the attribute and outlive the launch call.
inline void add_overlap_attr(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attrs) {
    if (!launch_overlap()) return;
    cudaLaunchAttribute &at = attrs[cfg.numAttrs++];
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
}

// ---------------------------------------------------------------- launches --

struct Int2PoolView {
    const uint8_t *codes_k, *codes_v;
    const uint16_t *scale_k, *zero_k, *scale_v, *zero_v;
    int n_pages;
};

// The same pool, writable (the demotion's destination).
struct Int2PoolMut {
    uint8_t *codes_k, *codes_v;
    uint16_t *scale_k, *zero_k, *scale_v, *zero_v;
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

// Tensor-core bulk demotion of position ranges (demote_tc.cu).
bool demote_range_supported(const oscar_layout_t &L);
cudaError_t launch_demote_range(const oscar_layout_t &L, Bf16PoolView src, const int32_t *bf16_pt,
                                const oscar_int2_pool_t &dst, const int32_t *int2_pt, int max_pages, int batch,
                                const int32_t *pos_begin, const int32_t *pos_end, const float *RK, const float *RV,
                                float cK, float cV, float *rot_out, int32_t *status, cudaStream_t st);

cudaError_t launch_quantize_rotated(const oscar_layout_t &L, const float *x, int n, float clip, uint8_t *codes,
                                    uint16_t *scale, uint16_t *zero, cudaStream_t st);

cudaError_t launch_rotate_q(const oscar_layout_t &L, const uint16_t *q, const float *RK, int batch,
                            float *q_rot, cudaStream_t st);

cudaError_t launch_int2_attention(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool,
                                  const int32_t *pt, int max_pages, const int32_t *seq_len,
                                  const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                  int32_t *status, cudaStream_t st);

// Tensor-core INT2 kernel (n_kv_heads in {1, 2, 4, 8}); launch_int2_attention dispatches to it.
bool int2_mma_supported(const oscar_layout_t &L);

// The layout's codebooks: all levels zero = uniform (levels 0, 1, 2, 3).
inline bool uniform_codebook(const oscar_layout_t &L) {
    for (int k = 0; k < 4; ++k)
        if (L.levels_k[k] != 0.0f || L.levels_v[k] != 0.0f) return false;
    return true;
}
// The levels a kernel uses (0, 1, 2, 3 for the uniform codebook).
inline float4 codebook_levels(const oscar_layout_t &L, bool values) {
    if (uniform_codebook(L)) return make_float4(0.f, 1.f, 2.f, 3.f);
    const float *l = values ? L.levels_v : L.levels_k;
    return make_float4(l[0], l[1], l[2], l[3]);
}
// Window clusters (the BF16 sink/recent part) per request of the tensor-core INT2 kernel: two for
// a single request with 8 kv heads (four heads each: a window CTA's rows then fit its buffers in
// one round trip), else one (with more requests the history clusters need the CTA slots).
int int2_mma_window_clusters(const oscar_layout_t &L, int batch);
// CTAs per cluster the tensor-core INT2 kernel will use for this layout (8 if no device is
// visible); *active (optional) gets how many such clusters are resident at once (0 if unknown).
int int2_mma_cluster_size(const oscar_layout_t &L, int *active = nullptr);
// The tensor-core INT2 history splits (history) and/or the BF16 sink/recent window
// (window) in one launch; the window CTAs write partial slot S.  With RK non-null the history
// CTAs compute q_rot = q . R_K themselves (q_rot is not read).
cudaError_t launch_decode_mma(const oscar_layout_t &L, const float *q_rot, const float *RK, Int2PoolView pool,
                              const int32_t *pt, const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt,
                              int max_pages, const int32_t *seq_len, const int32_t *hist_end, int batch,
                              float sm_scale, PartialsView out, int32_t *status, bool history, bool window,
                              cudaStream_t st);

// Per-step demotion folded into the window CTAs of launch_decode_mma: request b demotes
// position dem_pos[b] (>= hist_end[b], or -1 for none) of every kv head, K and V, from the BF16
// pool into dst (the INT2 pool).  Set on the launch through this descriptor.
struct FusedDemotion {
    const int32_t *dem_pos;     // NULL: no demotion
    const float *RV;
    float cK, cV;
    Int2PoolMut dst;
};
cudaError_t launch_decode_mma_demote(const oscar_layout_t &L, const float *RK, Int2PoolView pool, const int32_t *pt,
                                     const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt, int max_pages,
                                     const int32_t *seq_len, const int32_t *hist_end, int batch, float sm_scale,
                                     PartialsView out, int32_t *status, const FusedDemotion &dem,
                                     int32_t *arrivals, int *clusters, int32_t *sched, cudaStream_t st);
// (arrivals: NULL, or int32 [batch] to which each cluster of request b adds 1 once its partial
// slot is written; *clusters gets the count per request that the merge then waits for.
// sched: NULL (fixed history splits) or int32 [2][batch], zero and left zero: the history CTAs
// take 64-token units from a shared per-request counter)
// The history after a shared prefix and the BF16 window, one launch: history [max(hist_lo, sink),
// hist_end) in partial slots slot0 .. S - 1 (slots below slot0 belong to the prefix launch),
// window in slot S; q_rot from oscar_rotate_q.
cudaError_t launch_decode_mma_suffix(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool, const int32_t *pt,
                                     const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt, int max_pages,
                                     const int32_t *seq_len, const int32_t *hist_end, int batch, float sm_scale,
                                     PartialsView out, int32_t *status, int hist_lo, int slot0, int32_t *sched,
                                     cudaStream_t st);
// Shared-prefix history partials on the 5th-generation tensor cores: every request of the batch
// reads the INT2 pages of positions [sink, prefix_end) through the page table row `prefix_pt`; the
// prefix is cut into `splits` token splits written to partial slots 0 .. splits - 1 of every
// (request, query head).  Group 128 only.
cudaError_t launch_prefix_attention(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool,
                                    const int32_t *prefix_pt, int prefix_end, int batch, int splits, float sm_scale,
                                    PartialsView out, int32_t *status, cudaStream_t st);

// Tensor-core BF16 kernel (mode 0 any n_kv_heads; mode 1 n_kv_heads in {1, 2, 4, 8}).
bool bf16_mma_supported(const oscar_layout_t &L, int mode);
cudaError_t launch_bf16_attention_mma(const oscar_layout_t &L, const uint16_t *q, Bf16PoolView pool,
                                      const int32_t *pt, int max_pages, const int32_t *seq_len,
                                      const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                      int mode, int32_t *status, cudaStream_t st);

// mode 0: sink + recent of each request into slot S; mode 1: all of [0, T) split S ways.
cudaError_t launch_bf16_attention(const oscar_layout_t &L, const uint16_t *q, Bf16PoolView pool,
                                  const int32_t *pt, int max_pages, const int32_t *seq_len,
                                  const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                  int mode, int32_t *status, cudaStream_t st);

// counters NULL: the merge waits for the previous kernel (programmatic dependent launch).  Else
// int32 [2][batch], zero before the call and left zero: each request's merge starts once
// counters[b] reaches `expected` (the decode launch's arrivals); counters[batch + b] counts the
// merge CTAs of b that have seen it, and the last one resets both.
cudaError_t launch_merge(const oscar_layout_t &L, PartialsView p, const float *RV, int batch, uint16_t *out,
                         float *out_f32, float *lse, cudaStream_t st, int32_t *counters = nullptr,
                         int expected = 0, int32_t *status = nullptr);

}  // namespace oscar
