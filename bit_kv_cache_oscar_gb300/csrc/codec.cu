// Demotion (rotate -> clip -> quantize -> pack), the quantizer alone, and the
// query rotation.
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — the
// oldest recent token is rotated, clipped, quantized and packed (4 x 2-bit per
// byte) into the INT2 history; "Together AI 開源 OSCAR" (news.chathome.org),
// "OSCAR 的不同之處" — R = U·H_Had·P_br fixed per layer and kv head;
// estelledc notes "案例 2" — clip ratios c_K ~ 0.96, c_V ~ 0.92.
//
// Arithmetic contract (shared with nothing else in this library; the tests hold
// the reference): rotation y_j = fma-chain over i = 0..127 of x_i * R[i][j] in
// fp32; quantizer on the fp32 row with explicit round-to-nearest intrinsics, so
// that given equal fp32 rows the codes, scale and zero are bit-identical to the
// definition.  One CTA of 128 threads owns one 128-channel row at a time
// (thread j = channel j).

#include "oscar_internal.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace oscar {
namespace {

constexpr int kThreads = 128;
constexpr int kTokPerPass = 8;       // rows rotated together (R element reused 8x)
constexpr int kTokPerCta = 256;      // rows per CTA before the grid grows

// Quantize one row held one channel per thread (thread j = channel j of a 128-thread CTA).
__device__ __forceinline__ void quantize_row_store(float y, float clip, int group, bool store,
                                                   uint8_t *codes_row, uint16_t *scale_row,
                                                   uint16_t *zero_row, float *red, bool cb, float4 lv) {
    oscar::quantize_row_store(y, clip, group, store, codes_row, scale_row, zero_row, red, (int)threadIdx.x,
                              [] { __syncthreads(); }, cb, lv);
}

struct DemoteArgs {
    Bf16PoolView src;
    const int32_t *bf16_pt, *int2_pt;
    uint8_t *codes_k, *codes_v;
    uint16_t *scale_k, *zero_k, *scale_v, *zero_v;
    int int2_pages;
    int max_pages, batch, page_size, n_kv, group;
    const int32_t *req_idx, *pos;
    int n;
    const float *RK, *RV;
    float cK, cV;
    bool cb;                 // non-uniform codebooks lk (keys), lv (values)
    float4 lk, lv;
    float *rot_out;
    int32_t *status;
};

// grid.x = 2 * n_kv (kv head, K or V), grid.y = ceil(n / kTokPerCta).
// Dynamic smem: R (128 x 128 fp32) + kTokPerPass rows + small scratch.
__global__ void __launch_bounds__(kThreads) demote_kernel(DemoteArgs a) {
    extern __shared__ __align__(16) float smem[];
    __shared__ __align__(8) uint64_t rbar;              // R landed (expect-tx)
    float *Rs = smem;                                   // [128][128]
    float *xs = Rs + kHeadDim * kHeadDim;               // [kTokPerPass][128]
    float *red = xs + kTokPerPass * kHeadDim;           // [8]
    int *dst_row = reinterpret_cast<int *>(red + 8);    // [kTokPerPass]

    const int h = blockIdx.x >> 1, which = blockIdx.x & 1;
    const int j = threadIdx.x;
    const float *Rb = which ? a.RV : a.RK;               // NULL R_V: values stored as they are
    const float *R = Rb ? Rb + (size_t)h * kHeadDim * kHeadDim : nullptr;
    const float clip = which ? a.cV : a.cK;
    const uint16_t *src = which ? a.src.v : a.src.k;
    uint8_t *codes = which ? a.codes_v : a.codes_k;
    uint16_t *scale = which ? a.scale_v : a.scale_k;
    uint16_t *zero = which ? a.zero_v : a.zero_k;
    const int gpr = kHeadDim / a.group;                 // groups per row

    // R (64 KB) in one bulk copy: a loop of vector loads waits for each batch in turn
    if (R && j == 0) {
        mbar_init(saddr(&rbar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(saddr(&rbar), kHeadDim * kHeadDim * 4);
        tma_load_1d(saddr(Rs), R, kHeadDim * kHeadDim * 4, saddr(&rbar));
    }
    __syncthreads();
    if (R && !mbar_wait(saddr(&rbar), 0) && j == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);

    const int i0 = blockIdx.y * kTokPerCta;
    const int i1 = min(a.n, i0 + kTokPerCta);
    for (int base = i0; base < i1; base += kTokPerPass) {
        const int cnt = min(kTokPerPass, i1 - base);
        __syncthreads();
        for (int t = 0; t < kTokPerPass; ++t) {
            float x = 0.0f;
            int drow = -1;
            if (t < cnt) {
                const int b = a.req_idx[base + t], p = a.pos[base + t];
                const int lp = p / a.page_size, slot = p % a.page_size;
                bool ok = p >= 0 && lp < a.max_pages && b >= 0 && b < a.batch;
                if (!ok && j == 0) flag_status(a.status, OSCAR_DEV_BAD_LENGTH);
                if (ok) {
                    const int sp = a.bf16_pt[(size_t)b * a.max_pages + lp];
                    const int dp = a.int2_pt[(size_t)b * a.max_pages + lp];
                    if (sp < 0 || sp >= a.src.n_pages) {
                        if (j == 0) flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
                    } else if (dp < 0 || dp >= a.int2_pages) {
                        if (j == 0) flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
                    } else {
                        x = bf16_to_f32(src[(((size_t)sp * a.page_size + slot) * a.n_kv + h) * kHeadDim + j]);
                        drow = (dp * a.page_size + slot) * a.n_kv + h;
                    }
                }
            }
            xs[t * kHeadDim + j] = x;
            if (j == 0) dst_row[t] = drow;
        }
        __syncthreads();

        float acc[kTokPerPass];
#pragma unroll
        for (int t = 0; t < kTokPerPass; ++t) acc[t] = R ? 0.0f : xs[t * kHeadDim + j];
#pragma unroll 4
        for (int i = 0; i < (R ? kHeadDim : 0); i += 4) {
            const float r0 = Rs[(i + 0) * kHeadDim + j], r1 = Rs[(i + 1) * kHeadDim + j];
            const float r2 = Rs[(i + 2) * kHeadDim + j], r3 = Rs[(i + 3) * kHeadDim + j];
#pragma unroll
            for (int t = 0; t < kTokPerPass; ++t) {
                const float4 xv = reinterpret_cast<const float4 *>(xs + t * kHeadDim)[i >> 2];
                acc[t] = __fmaf_rn(xv.x, r0, acc[t]);
                acc[t] = __fmaf_rn(xv.y, r1, acc[t]);
                acc[t] = __fmaf_rn(xv.z, r2, acc[t]);
                acc[t] = __fmaf_rn(xv.w, r3, acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < kTokPerPass; ++t) {
            if (t >= cnt) break;                          // cnt is uniform across the CTA
            const int drow = dst_row[t];
            if (a.rot_out) a.rot_out[(((size_t)(base + t) * 2 + which) * a.n_kv + h) * kHeadDim + j] = acc[t];
            const size_t r = drow < 0 ? 0 : (size_t)drow;
            quantize_row_store(acc[t], clip, a.group, drow >= 0, codes + r * (kHeadDim / 4),
                               scale + r * gpr, zero + r * gpr, red, a.cb, which ? a.lv : a.lk);
        }
    }
}

__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const float *x, int n, float clip, int group,
                                                                 uint8_t *codes, uint16_t *scale, uint16_t *zero,
                                                                 bool cb, float4 lv) {
    __shared__ float red[8];
    const int r = blockIdx.x;
    if (r >= n) return;
    const int gpr = kHeadDim / group;
    const float y = x[(size_t)r * kHeadDim + threadIdx.x];
    quantize_row_store(y, clip, group, true, codes + (size_t)r * (kHeadDim / 4), scale + (size_t)r * gpr,
                       zero + (size_t)r * gpr, red, cb, lv);
}

// grid.x = batch * n_kv * 4 (a quarter of the 128 output channels per CTA), 32*G threads;
// thread (g, j) computes q_rot[g][c] = fma-chain_i q[g][i] * R[i][c] for c = 32*quarter + j.
// The CTA first stages its 128 x 32 block of R in shared memory with independent vector loads.
template <int G>
__global__ void __launch_bounds__(32 * G) rotate_q_kernel(const uint16_t *q, const float *RK, int n_kv,
                                                         float *q_rot) {
    __shared__ float qs[G][kHeadDim];
    __shared__ __align__(16) float Rs[kHeadDim][32];
    const int quarter = blockIdx.x & 3, bh = blockIdx.x >> 2;
    const int b = bh / n_kv, h = bh % n_kv;
    const int tid = threadIdx.x, g = tid >> 5, j = tid & 31;
    const size_t row0 = ((size_t)b * n_kv + h) * G;        // first query row of this kv head
    const float *R = RK + (size_t)h * kHeadDim * kHeadDim + quarter * 32;
    for (int e = tid; e < kHeadDim * 8; e += 32 * G) {       // 128 rows x 8 float4
        const int i = e >> 3, c4 = e & 7;
        reinterpret_cast<float4 *>(&Rs[i][0])[c4] = __ldg(reinterpret_cast<const float4 *>(R + i * kHeadDim) + c4);
    }
    pdl_wait();                                             // q and q_rot belong to the previous kernel
    for (int e = tid; e < G * kHeadDim; e += 32 * G) qs[e / kHeadDim][e % kHeadDim] = bf16_to_f32(q[row0 * kHeadDim + e]);
    __syncthreads();
    float acc = 0.0f;
#pragma unroll 16
    for (int i = 0; i < kHeadDim; ++i) acc = __fmaf_rn(qs[g][i], Rs[i][j], acc);
    // The attention kernel that follows may launch only now: launched earlier, its CTAs take
    // SM slots piecemeal while this and the previous kernels still hold some, and its clusters
    // end up placed worse than on an idle GPU.
    pdl_trigger();
    q_rot[(row0 + g) * kHeadDim + quarter * 32 + j] = acc;
}

}  // namespace

cudaError_t launch_demote(const oscar_layout_t &L, Bf16PoolView src, const int32_t *bf16_pt,
                          const oscar_int2_pool_t &dst, const int32_t *int2_pt, int max_pages, int batch,
                          const int32_t *req_idx, const int32_t *pos, int n, const float *RK,
                          const float *RV, float cK, float cV, float *rot_out, int32_t *status,
                          cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    DemoteArgs a;
    a.src = src;
    a.bf16_pt = bf16_pt;
    a.int2_pt = int2_pt;
    a.codes_k = dst.codes_k;
    a.codes_v = dst.codes_v;
    a.scale_k = dst.scale_k;
    a.zero_k = dst.zero_k;
    a.scale_v = dst.scale_v;
    a.zero_v = dst.zero_v;
    a.int2_pages = dst.n_pages;
    a.max_pages = max_pages;
    a.batch = batch;
    a.page_size = L.page_size;
    a.n_kv = L.n_kv_heads;
    a.group = L.group;
    a.req_idx = req_idx;
    a.pos = pos;
    a.n = n;
    a.RK = RK;
    a.RV = RV;
    a.cK = cK;
    a.cV = cV;
    a.cb = !uniform_codebook(L);
    a.lk = codebook_levels(L, false);
    a.lv = codebook_levels(L, true);
    a.rot_out = rot_out;
    a.status = status;
    const size_t smem = sizeof(float) * (kHeadDim * kHeadDim + kTokPerPass * kHeadDim + 8) + sizeof(int) * kTokPerPass;
    if (cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(demote_kernel), (int)smem)) return e;
    dim3 grid(2 * L.n_kv_heads, (n + kTokPerCta - 1) / kTokPerCta);
    demote_kernel<<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rotated(const oscar_layout_t &L, const float *x, int n, float clip, uint8_t *codes,
                                    uint16_t *scale, uint16_t *zero, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    quantize_rows_kernel<<<n, kThreads, 0, st>>>(x, n, clip, L.group, codes, scale, zero, !uniform_codebook(L),
                                                 codebook_levels(L, false));
    return cudaGetLastError();
}

cudaError_t launch_rotate_q(const oscar_layout_t &L, const uint16_t *q, const float *RK, int batch,
                            float *q_rot, cudaStream_t st) {
    if (batch <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(batch * L.n_kv_heads * 4);
    cfg.blockDim = dim3(32 * L.gqa);
    cfg.stream = st;
    cfg.attrs = attrs;
    add_overlap_attr(cfg, attrs);
    switch (L.gqa) {
        case 1: return cudaLaunchKernelEx(&cfg, rotate_q_kernel<1>, q, RK, L.n_kv_heads, q_rot);
        case 2: return cudaLaunchKernelEx(&cfg, rotate_q_kernel<2>, q, RK, L.n_kv_heads, q_rot);
        case 4: return cudaLaunchKernelEx(&cfg, rotate_q_kernel<4>, q, RK, L.n_kv_heads, q_rot);
        case 8: return cudaLaunchKernelEx(&cfg, rotate_q_kernel<8>, q, RK, L.n_kv_heads, q_rot);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace oscar
