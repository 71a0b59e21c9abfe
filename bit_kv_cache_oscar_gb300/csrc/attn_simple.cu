// Decode-attention partials on CUDA cores: INT2 history splits and BF16
// sink/recent (or all-BF16) splits.
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — the
// INT2 kernel unpacks codes, restores scale/zero and accumulates in floating
// point; the BF16 kernel handles sink/recent; partial results are merged by an
// online softmax.  "Together AI 開源 OSCAR" (news.chathome.org), "服務系統" —
// 64 sink + 256 recent tokens in BF16, paged.
//
// One CTA = (request, kv head, split), 4 warps; each warp walks every 4th
// token of the split, each lane owns 4 consecutive channels (one byte of
// codes), logits are reduced with warp shuffles, and the G query heads of the
// kv head share every key/value read (GQA packing).  Partials are in the
// base-2 domain: t = sm_scale * logit * log2(e).

#include "oscar_internal.cuh"

namespace oscar {
namespace {

constexpr int kWarps = 4;

template <int G>
struct WarpState {
    float m[G], l[G], acc[G][4];
    __device__ void init() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[h][c] = 0.0f;
        }
    }
    // Fold one token: per-lane partial dot products -> logits, then update.
    __device__ void fold(float (&part)[G], const float (&val)[4], float scale2) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = part[h];
#pragma unroll
            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const float t = s * scale2;
            const float mn = fmaxf(m[h], t);
            const float a = exp2f(m[h] - mn);
            const float p = exp2f(t - mn);
            l[h] = l[h] * a + p;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[h][c] = acc[h][c] * a + p * val[c];
            m[h] = mn;
        }
    }
};

// Combine the kWarps warp states in shared memory and write one partial slot
// for the G query heads of kv head `kvh`.
template <int G>
__device__ void combine_and_store(WarpState<G> &st, int b, int kvh, int n_q_heads, int S1, int slot,
                                  PartialsView out) {
    __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
    __shared__ float sm_acc[kWarps][G][kHeadDim];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            sm_m[warp][h] = st.m[h];
            sm_l[warp][h] = st.l[h];
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) sm_acc[warp][h][lane * 4 + c] = st.acc[h][c];
    __syncthreads();
    const int d = threadIdx.x;   // 128 threads: one channel each
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][h]);
        float L = 0.0f, A = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(sm_m[w][h] - M);
                L += sm_l[w][h] * f;
                A += sm_acc[w][h][d] * f;
            }
        }
        const size_t row = ((size_t)b * n_q_heads + kvh * G + h) * S1 + slot;
        out.acc[row * kHeadDim + d] = A;
        if (d == 0) {
            out.m[row] = M;
            out.l[row] = L;
        }
    }
}

struct Int2Args {
    const float *q_rot;
    Int2PoolView pool;
    const int32_t *pt;
    int max_pages, page_size, n_kv, group, sink;
    const int32_t *seq_len, *hist_end;
    float scale2;
    PartialsView out;
    int32_t *status;
    float4 lk, lv;           // codebook levels of keys and values (0, 1, 2, 3: uniform)
};

// level of a 2-bit code
__device__ __forceinline__ float code_level(const float4 &l, uint32_t c) {
    return (c & 2u) ? ((c & 1u) ? l.w : l.z) : ((c & 1u) ? l.y : l.x);
}

template <int G>
__global__ void __launch_bounds__(128) int2_split_kernel(Int2Args a) {
    const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_q_heads = a.n_kv * G, S = a.out.S;
    int T, he;
    read_lengths(a.seq_len, a.hist_end, b, a.sink, a.max_pages * a.page_size, a.status, T, he);
    const SplitRange r = history_split(a.sink, he, S, s);

    float q[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float4 v = reinterpret_cast<const float4 *>(
            a.q_rot + ((size_t)b * n_q_heads + kvh * G + h) * kHeadDim)[lane];
        q[h][0] = v.x; q[h][1] = v.y; q[h][2] = v.z; q[h][3] = v.w;
    }
    const int gpr = kHeadDim / a.group;
    const int grp = (lane * 4) / a.group;

    WarpState<G> st;
    st.init();
    for (int p = r.lo + warp; p < r.hi; p += kWarps) {
        const int page = a.pt[(size_t)b * a.max_pages + p / a.page_size];
        if (page < 0 || page >= a.pool.n_pages) {
            if (lane == 0) flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
            continue;
        }
        const size_t row = ((size_t)page * a.page_size + p % a.page_size) * a.n_kv + kvh;
        const uint32_t ck = a.pool.codes_k[row * (kHeadDim / 4) + lane];
        const uint32_t cv = a.pool.codes_v[row * (kHeadDim / 4) + lane];
        const float zk = bf16_to_f32(a.pool.zero_k[row * gpr + grp]);
        const float sk = bf16_to_f32(a.pool.scale_k[row * gpr + grp]);
        const float zv = bf16_to_f32(a.pool.zero_v[row * gpr + grp]);
        const float sv = bf16_to_f32(a.pool.scale_v[row * gpr + grp]);
        float kh[4], vh[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            kh[c] = fmaf(code_level(a.lk, (ck >> (2 * c)) & 3u), sk, zk);
            vh[c] = fmaf(code_level(a.lv, (cv >> (2 * c)) & 3u), sv, zv);
        }
        float part[G];
#pragma unroll
        for (int h = 0; h < G; ++h) part[h] = q[h][0] * kh[0] + q[h][1] * kh[1] + q[h][2] * kh[2] + q[h][3] * kh[3];
        st.fold(part, vh, a.scale2);
    }
    combine_and_store<G>(st, b, kvh, n_q_heads, S + 1, s, a.out);
}

struct Bf16Args {
    const uint16_t *q;
    Bf16PoolView pool;
    const int32_t *pt;
    int max_pages, page_size, n_kv, sink;
    const int32_t *seq_len, *hist_end;
    float scale2;
    PartialsView out;
    int mode;      // 0: sink + recent -> slot S; 1: split s of [0, T) -> slot s, slot S empty
    int32_t *status;
};

template <int G>
__global__ void __launch_bounds__(128) bf16_split_kernel(Bf16Args a) {
    const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_q_heads = a.n_kv * G, S = a.out.S;
    int T, he;
    read_lengths(a.seq_len, a.mode == 0 ? a.hist_end : nullptr, b, a.sink, a.max_pages * a.page_size, a.status,
                 T, he);
    int lo0, hi0, lo1, hi1;
    if (a.mode == 0) {
        lo0 = 0; hi0 = min(a.sink, T);
        lo1 = max(he, hi0); hi1 = T;
    } else {
        const SplitRange r = full_split(T, S, s);
        lo0 = r.lo; hi0 = r.hi; lo1 = hi1 = 0;
    }
    float q[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint2 v = reinterpret_cast<const uint2 *>(a.q + ((size_t)b * n_q_heads + kvh * G + h) * kHeadDim)[lane];
        q[h][0] = __uint_as_float(v.x << 16); q[h][1] = __uint_as_float(v.x & 0xffff0000u);
        q[h][2] = __uint_as_float(v.y << 16); q[h][3] = __uint_as_float(v.y & 0xffff0000u);
    }
    WarpState<G> st;
    st.init();
    const int n0 = hi0 - lo0, n1 = hi1 - lo1;
    for (int i = warp; i < n0 + n1; i += kWarps) {
        const int p = i < n0 ? lo0 + i : lo1 + (i - n0);
        const int page = a.pt[(size_t)b * a.max_pages + p / a.page_size];
        if (page < 0 || page >= a.pool.n_pages) {
            if (lane == 0) flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
            continue;
        }
        const size_t row = ((size_t)page * a.page_size + p % a.page_size) * a.n_kv + kvh;
        const uint2 kk = reinterpret_cast<const uint2 *>(a.pool.k + row * kHeadDim)[lane];
        const uint2 vv = reinterpret_cast<const uint2 *>(a.pool.v + row * kHeadDim)[lane];
        const float k4[4] = {__uint_as_float(kk.x << 16), __uint_as_float(kk.x & 0xffff0000u),
                             __uint_as_float(kk.y << 16), __uint_as_float(kk.y & 0xffff0000u)};
        const float v4[4] = {__uint_as_float(vv.x << 16), __uint_as_float(vv.x & 0xffff0000u),
                             __uint_as_float(vv.y << 16), __uint_as_float(vv.y & 0xffff0000u)};
        float part[G];
#pragma unroll
        for (int h = 0; h < G; ++h) part[h] = q[h][0] * k4[0] + q[h][1] * k4[1] + q[h][2] * k4[2] + q[h][3] * k4[3];
        st.fold(part, v4, a.scale2);
    }
    combine_and_store<G>(st, b, kvh, n_q_heads, S + 1, a.mode == 0 ? S : s, a.out);
    if (a.mode == 1 && s == 0) {
        // slot S is empty for an all-BF16 cache
        for (int h = 0; h < G; ++h) {
            const size_t row = ((size_t)b * n_q_heads + kvh * G + h) * (S + 1) + S;
            a.out.acc[row * kHeadDim + threadIdx.x] = 0.0f;
            if (threadIdx.x == 0) {
                a.out.m[row] = -INFINITY;
                a.out.l[row] = 0.0f;
            }
        }
    }
}

template <template <int> class K, typename Args>
cudaError_t launch_g(int gqa, dim3 grid, Args a, cudaStream_t st) {
    switch (gqa) {
        case 1: K<1>::run(grid, a, st); break;
        case 2: K<2>::run(grid, a, st); break;
        case 4: K<4>::run(grid, a, st); break;
        case 8: K<8>::run(grid, a, st); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int G>
struct Int2Launcher {
    static void run(dim3 grid, Int2Args a, cudaStream_t st) { int2_split_kernel<G><<<grid, 128, 0, st>>>(a); }
};
template <int G>
struct Bf16Launcher {
    static void run(dim3 grid, Bf16Args a, cudaStream_t st) { bf16_split_kernel<G><<<grid, 128, 0, st>>>(a); }
};

}  // namespace

cudaError_t launch_int2_attention(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool,
                                  const int32_t *pt, int max_pages, const int32_t *seq_len,
                                  const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                  int32_t *status, cudaStream_t st) {
    if (batch <= 0) return cudaSuccess;
    if (int2_mma_supported(L))
        return launch_decode_mma(L, q_rot, nullptr, pool, pt, nullptr, Bf16PoolView{nullptr, nullptr, 0}, nullptr,
                                 max_pages, seq_len, hist_end, batch, sm_scale, out, status, true, false, st);
    Int2Args a{q_rot, pool, pt, max_pages, L.page_size, L.n_kv_heads, L.group, L.sink, seq_len, hist_end,
               sm_scale * kLog2e, out, status, codebook_levels(L, false), codebook_levels(L, true)};
    return launch_g<Int2Launcher>(L.gqa, dim3(out.S, L.n_kv_heads, batch), a, st);
}

cudaError_t launch_bf16_attention(const oscar_layout_t &L, const uint16_t *q, Bf16PoolView pool,
                                  const int32_t *pt, int max_pages, const int32_t *seq_len,
                                  const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                  int mode, int32_t *status, cudaStream_t st) {
    if (batch <= 0) return cudaSuccess;
    if (mode == 0 && int2_mma_supported(L))   // the window CTAs of the tensor-core INT2 kernel
        return launch_decode_mma(L, nullptr, nullptr, Int2PoolView{}, nullptr, q, pool, pt, max_pages, seq_len,
                                 hist_end, batch, sm_scale, out, status, false, true, st);
    if (bf16_mma_supported(L, mode))
        return launch_bf16_attention_mma(L, q, pool, pt, max_pages, seq_len, hist_end, batch, sm_scale, out, mode,
                                         status, st);
    Bf16Args a{q, pool, pt, max_pages, L.page_size, L.n_kv_heads, L.sink, seq_len, hist_end,
               sm_scale * kLog2e, out, mode, status};
    return launch_g<Bf16Launcher>(L.gqa, dim3(mode == 0 ? 1 : out.S, L.n_kv_heads, batch), a, st);
}

}  // namespace oscar
