// Online-softmax merge of the history splits and the BF16 partial, with the
// history accumulator rotated back by R_V^T.
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — the
// BF16 and INT2 partial results are combined by an online softmax merge;
// "Together AI 開源 OSCAR" (news.chathome.org), "OSCAR 的不同之處" — values are
// stored rotated by R_V = U_S·H·P_br, so the history part of the output is
// brought back with R_V^T.
//
// The fold is an ordered fp32 sequence with explicit round-to-nearest
// intrinsics and its own 2^x, so that equal partials give equal output bits:
//   M' = max(M, m_i); a = 2^(M - M'); b = 2^(m_i - M');
//   L = fma(L, a, l_i*b); A_d = fma(A_d, a, acc_i,d*b)
// history slots 0..S-1 in ascending order, then A'_j = fma-chain_i A_i*R_V[j][i],
// then the BF16 slot S, then o = A'/L (IEEE division), rounded to bf16.

#include "oscar_internal.cuh"

namespace oscar {
namespace {

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

constexpr int kPad = kHeadDim + 1;   // R_V rows padded: thread j reads row j conflict-free

// grid = (n_kv, batch); 128 threads, thread j owns output channel j.
__global__ void __launch_bounds__(128) merge_kernel(PartialsView p, const float *RV, int n_kv, int gqa,
                                                    uint16_t *out, float *out_f32, float *lse) {
    extern __shared__ __align__(16) float smem[];
    float *Rs = smem;                                  // [128][129] if RV
    float *As = smem + (RV ? kHeadDim * kPad : 0);     // [128]
    const int kvh = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
    const int S = p.S, n_q_heads = n_kv * gqa;
    if (RV) {
        const float *R = RV + (size_t)kvh * kHeadDim * kHeadDim;
        for (int i = 0; i < kHeadDim; ++i) Rs[i * kPad + j] = __ldg(R + i * kHeadDim + j);
    }
    for (int g = 0; g < gqa; ++g) {
        const size_t row0 = ((size_t)b * n_q_heads + kvh * gqa + g) * (S + 1);
        float M = -INFINITY, L = 0.0f, A = 0.0f;
        for (int i = 0; i < S; ++i) {
            const float li = p.l[row0 + i];
            if (!(li > 0.0f)) continue;
            const float mi = p.m[row0 + i];
            const float Mn = mi > M ? mi : M;
            const float a = exp2_taylor(__fsub_rn(M, Mn));
            const float bb = exp2_taylor(__fsub_rn(mi, Mn));
            L = __fmaf_rn(L, a, __fmul_rn(li, bb));
            A = __fmaf_rn(A, a, __fmul_rn(p.acc[(row0 + i) * kHeadDim + j], bb));
            M = Mn;
        }
        float Ar = A;
        if (RV) {
            __syncthreads();
            As[j] = A;
            __syncthreads();
            float r = 0.0f;
#pragma unroll 8
            for (int i = 0; i < kHeadDim; ++i) r = __fmaf_rn(As[i], Rs[j * kPad + i], r);
            Ar = r;
        }
        const float lS = p.l[row0 + S];
        if (lS > 0.0f) {
            const float mS = p.m[row0 + S];
            const float Mn = mS > M ? mS : M;
            const float a = exp2_taylor(__fsub_rn(M, Mn));
            const float bb = exp2_taylor(__fsub_rn(mS, Mn));
            L = __fmaf_rn(L, a, __fmul_rn(lS, bb));
            Ar = __fmaf_rn(Ar, a, __fmul_rn(p.acc[(row0 + S) * kHeadDim + j], bb));
            M = Mn;
        }
        const float o = L > 0.0f ? __fdiv_rn(Ar, L) : 0.0f;
        const size_t orow = (size_t)b * n_q_heads + kvh * gqa + g;
        if (out) out[orow * kHeadDim + j] = f32_to_bf16_rn(o);
        if (out_f32) out_f32[orow * kHeadDim + j] = o;
        if (lse && j == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_merge(const oscar_layout_t &L, PartialsView p, const float *RV, int batch, uint16_t *out,
                         float *out_f32, float *lse, cudaStream_t st) {
    if (batch <= 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((RV ? kHeadDim * kPad : 0) + kHeadDim);
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(sizeof(float) * (kHeadDim * kPad + kHeadDim)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    merge_kernel<<<dim3(L.n_kv_heads, batch), 128, smem, st>>>(p, RV, L.n_kv_heads, L.gqa, out, out_f32, lse);
    return cudaGetLastError();
}

}  // namespace oscar
