// Online-softmax merge of the history splits and the BF16 partial, with the
// history accumulator rotated back by R_V^T.
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — the
// BF16 and INT2 partial results are combined by an online softmax merge;
// "Together AI 開源 OSCAR" (news.chathome.org), "OSCAR 的不同之處" — values are
// stored rotated by R_V = U_S·H·P_br, so the history part of the output is
// brought back with R_V^T.
//
// The combination is an ordered fp32 computation with explicit round-to-nearest
// intrinsics and its own 2^x, so that equal partials give equal output bits:
//   M = max of m_i over the non-empty partials (history and BF16), w_i = 2^(m_i - M);
//   L = fma(l_i, w_i, L), A_d = fma(acc_i,d, w_i, A_d) over history slots 0..S-1 ascending;
//   A'_j = fma-chain_i A_i * R_V[j][i]; then the BF16 slot S with its weight;
//   o = A'/L (IEEE division), rounded to bf16.
// Taking the global maximum first (rather than a running one) keeps the weights
// independent, so they are computed in parallel and the sums are plain FMA chains.

#include "oscar_internal.cuh"
#include "ptx.cuh"
#include "merge_math.cuh"

namespace oscar {
namespace {

constexpr int kPad = kHeadDim + 1;   // R_V rows padded: thread j reads row j conflict-free
constexpr int kQuarter = kHeadDim / 4;
constexpr int kChunk = 48;                                // history slots staged in shared memory at a time
constexpr int kV4 = kChunk * kHeadDim / 4 / 128;          // float4 loads per thread and chunk

// grid = (Hq, batch, 4 with R_V / 1 without); 128 threads.  Every CTA merges the history
// slots of one query head for all 128 channels (thread j owns channel j); with R_V, CTA z
// then rotates back output channels [32 z, 32 z + 32) (thread j < 32 owns channel 32 z + j)
// from the 32 rows of R_V that it staged before waiting for the partials' producer.
// The accumulator rows of up to kChunk slots at a time are brought into shared memory by all
// threads with 16-byte loads, all in flight at once (the first chunk's together with m and l).
// Dynamic smem: [R_V 32 x 129 if RV] [A 128] [X kChunk x 128] [w S+1] [l S+1] [red 8].
__global__ void __launch_bounds__(128) merge_kernel(PartialsView p, const float *RV, int n_q_heads, int gqa,
                                                    uint16_t *out, float *out_f32, float *lse, int32_t *counters,
                                                    int expected, int batch, int32_t *status) {
    extern __shared__ __align__(16) float smem[];
    const int hq = blockIdx.x, b = blockIdx.y, z = blockIdx.z, j = threadIdx.x;
    const int S = p.S;
    float *Rs = smem;
    float *As = smem + (RV ? kQuarter * kPad : 0);
    float *Xs = As + kHeadDim;
    float *ws = Xs + kChunk * kHeadDim;
    float *ls = ws + (S + 1);
    float *red = ls + (S + 1);
    const size_t row0 = ((size_t)b * n_q_heads + hq) * (S + 1);

    if (RV) {
        // rows 32 z .. 32 z + 31 of this head's R_V (32 rows x 32 float4)
        const float4 *R = reinterpret_cast<const float4 *>(RV + ((size_t)(hq / gqa) * kHeadDim + z * kQuarter) * kHeadDim);
#pragma unroll
        for (int e = j; e < kQuarter * kHeadDim / 4; e += 128) {
            const float4 v = __ldg(R + e);
            float *dst = Rs + (e >> 5) * kPad + (e & 31) * 4;
            dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
        }
    }
    if (!counters) {
        pdl_wait();                              // the partials come from the previous kernels
    } else {
        // Request b's partials are complete once its clusters have all counted (each counts after
        // its slot writes, with release): wait for that rather than for the whole decode grid.
        // This grid launched only after every decode CTA had passed its loop, so all of them are
        // running and the count arrives; the wait is bounded all the same.
        if (j == 0) {
            int32_t n = 0;
            for (long i = 0; i < kSpinLimit; ++i) {
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(n) : "l"(counters + b) : "memory");
                if (n >= expected) break;
                __nanosleep(32);
            }
            if (n < expected) flag_status(status, OSCAR_DEV_WAIT_TIMEOUT);
            // the last of b's merge CTAs to get here resets both counts for the next launch
            const int per_req = gridDim.x * gridDim.z;
            if (atomicAdd(counters + batch + b, 1) == per_req - 1) {
                counters[b] = 0;
                counters[batch + b] = 0;
                __threadfence();
            }
        }
        __syncthreads();
    }

    // slots [c0, c0 + kChunk) of the accumulator rows (contiguous, 512 bytes each) -> Xs
    const float4 *acc4 = reinterpret_cast<const float4 *>(p.acc + row0 * kHeadDim);
    float4 xv[kV4];
    auto load_chunk = [&](int c0) {
        const int n4 = min(kChunk, S - c0) * (kHeadDim / 4);
#pragma unroll
        for (int u = 0; u < kV4; ++u)
            if (j + 128 * u < n4) xv[u] = acc4[(size_t)c0 * (kHeadDim / 4) + j + 128 * u];
    };
    auto store_chunk = [&](int c0) {
        const int n4 = min(kChunk, S - c0) * (kHeadDim / 4);
#pragma unroll
        for (int u = 0; u < kV4; ++u)
            if (j + 128 * u < n4) reinterpret_cast<float4 *>(Xs)[j + 128 * u] = xv[u];
    };
    load_chunk(0);
    const int c = RV ? z * kQuarter + (j & (kQuarter - 1)) : j;   // output channel (threads j < 32 with R_V)
    const float xS = p.acc[(row0 + S) * kHeadDim + c];

    float mloc = -INFINITY;
    for (int i = j; i <= S; i += 128) {
        const float li = p.l[row0 + i], mi = p.m[row0 + i];
        ls[i] = li;
        ws[i] = mi;
        if (li > 0.0f && mi > mloc) mloc = mi;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if ((j & 31) == 0) red[j >> 5] = mloc;
    store_chunk(0);
    __syncthreads();
    const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    for (int i = j; i <= S; i += 128) ws[i] = ls[i] > 0.0f ? exp2_taylor(__fsub_rn(ws[i], M)) : 0.0f;
    __syncthreads();

    // empty slots are skipped by select: L = fma(l_i, w_i, L), A = fma(acc_i, w_i, A), i ascending
    float L = 0.0f, A = 0.0f;
    for (int c0 = 0; c0 < S; c0 += kChunk) {
        if (c0 > 0) {
            __syncthreads();                     // the previous chunk is consumed
            load_chunk(c0);
            store_chunk(c0);
            __syncthreads();
        }
        const int n = min(kChunk, S - c0);
#pragma unroll 8
        for (int i = 0; i < n; ++i) {
            const float li = ls[c0 + i], w = ws[c0 + i];
            const bool on = li > 0.0f;
            L = on ? __fmaf_rn(li, w, L) : L;
            A = on ? __fmaf_rn(Xs[i * kHeadDim + j], w, A) : A;
        }
    }
    float Ar = A;
    if (RV) {
        As[j] = A;
        __syncthreads();
        if (j >= kQuarter) return;
        float r = 0.0f;
#pragma unroll 8
        for (int i = 0; i < kHeadDim; ++i) r = __fmaf_rn(As[i], Rs[j * kPad + i], r);
        Ar = r;
    }
    if (ls[S] > 0.0f) {
        const float w = ws[S];
        L = __fmaf_rn(ls[S], w, L);
        Ar = __fmaf_rn(xS, w, Ar);
    }
    // The next kernel may launch only now: launched right after the wait above, the following
    // layer's decode CTAs start beside this grid's and the step was measured 18 % slower.
    pdl_trigger();
    const float o = L > 0.0f ? __fdiv_rn(Ar, L) : 0.0f;
    const size_t orow = (size_t)b * n_q_heads + hq;
    if (out) out[orow * kHeadDim + c] = f32_to_bf16_rn(o);
    if (out_f32) out_f32[orow * kHeadDim + c] = o;
    if (lse && z == 0 && j == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const oscar_layout_t &L, PartialsView p, const float *RV, int batch, uint16_t *out,
                         float *out_f32, float *lse, cudaStream_t st, int32_t *counters, int expected,
                         int32_t *status) {
    if (batch <= 0) return cudaSuccess;
    const int hq = L.n_kv_heads * L.gqa;
    const size_t smem = sizeof(float) * ((RV ? kQuarter * kPad : 0) + kHeadDim + kChunk * kHeadDim + 2 * (p.S + 1) + 8);
    if (cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(merge_kernel), (int)smem)) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(hq, batch, RV ? 4 : 1);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attrs;
    add_overlap_attr(cfg, attrs);
    return cudaLaunchKernelEx(&cfg, merge_kernel, p, RV, hq, L.gqa, out, out_f32, lse, counters, expected, batch,
                              status);
}

}  // namespace oscar
