// INT2-history decode-attention partials on the tensor cores (sm_103a).
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — the
// INT2 kernel unpacks the 2-bit codes, restores scale/zero and accumulates in
// floating point; "Together AI 開源 OSCAR" (news.chathome.org), "OSCAR 的不同之處"
// — queries meet the rotated keys as q·R_K, values stay rotated until the merge.
//
// Design (one CTA = one history split of one request, all kv heads <= 8):
//  * a producer warp copies 16-token tiles (codes for all heads + bf16
//    scale/zero) into a ring of shared-memory stages with cp.async, head-major
//    ([head][token][32 B]), and signals an mbarrier per stage; 8 consumer warps
//    each own one kv head (and a share of the tiles when there are fewer heads);
//  * q·k_hat = scale * (q_rot · code) + zero * sum(q_rot) per group, and
//    sum_t p_t v_hat_t = sum_t p_t zero_t + sum_t (p_t scale_t) code_t: both
//    contractions run on mma.sync m16n8k16 (f16 in, fp32 accumulate) with the
//    code matrix as the A operand;
//  * a 2-bit code c placed in a f16 mantissa with no exponent bits is the
//    subnormal c * 2^(2k) * 2^-24 (k = its position), so unpacking is a
//    byte permute plus an AND; the power-of-two factors are folded into the
//    other operand or the output;
//  * the other operand (q_rot, and p*scale) is split into f16 hi + lo parts
//    that fill the 8 MMA columns (4 query heads x {hi, lo}), giving ~22-bit
//    operands at no extra MMA cost for GQA 4;
//  * online softmax in the base-2 domain; the per-tile P operand is moved
//    from the QK accumulator layout to the PV operand layout through a small
//    per-warp shared buffer; each warp takes two 16-token tiles per pass.
// Every wait is bounded: a wait that gives up sets OSCAR_DEV_WAIT_TIMEOUT.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstring>

#include "oscar_internal.cuh"
#include "ptx.cuh"
#include "quant.cuh"
#include "merge_math.cuh"
#include "tma.cuh"

namespace oscar {
namespace {

constexpr int kCW = 8;                       // consumer warps
constexpr int kThreads = (kCW + 1) * 32;     // + producer warp
constexpr int kTilesPerStage = 4;
constexpr int kStageTok = kTileTokens * kTilesPerStage;
constexpr int kMaxStages = 4;

constexpr uint32_t kM0 = 0x00030003u, kM1 = 0x000C000Cu, kM2 = 0x00300030u, kM3 = 0x00C000C0u,
                   kM4 = 0x03000300u;
constexpr float kTwo24 = 16777216.0f;

__device__ __forceinline__ uint32_t pack2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// f16 hi part (part == 0) or lo part (part == 1) of v.
__device__ __forceinline__ __half split_part(float v, int part) {
    const __half h = __float2half_rn(v);
    return part ? __float2half_rn(v - __half2float(h)) : h;
}

// QK operand: register r (0..7) of one token's 16-channel word w (channels 16W + r in the low
// half, 16W + 8 + r in the high half), value code * kQF[r] * 2^-24.
__device__ __forceinline__ uint32_t qk_reg(uint32_t w, uint32_t wb, int r) {
    switch (r) {
        case 0: return w & kM0;
        case 1: return w & kM1;
        case 2: return w & kM2;
        case 3: return w & kM3;
        case 4: return w & kM4;
        case 5: return wb & kM1;
        case 6: return wb & kM2;
        default: return wb & kM3;
    }
}
// factors of registers 0..7: 1, 4, 16, 64, 256, 4, 16, 64
__device__ __host__ constexpr float qk_factor(int r) { return r == 4 ? 256.f : (float)(1 << (2 * (r & 3))); }

// Group-pure QK mapping (groups of 32 or 64 channels): in MMA m = 2 Gb + j a thread with lane
// parity odd uses registers qk_rsel(j, 0, odd) (A k-columns 2t, 2t+1) and qk_rsel(j, 1, odd)
// (2t+8, 2t+9) of its word W = 2 Gb + (t >> 1): even lanes registers 0, 1 / 4, 5, odd lanes 2, 3 /
// 6, 7, so the two lanes that share a word take disjoint halves of it.
__device__ __host__ __forceinline__ int qk_rsel(int j, int e, int odd) { return 4 * j + 2 * odd + e; }

// PV operand: register i (0..15) of the pair (token x, token y) for channel 16W + i, from the
// byte permutes P1..P4 of their words; value code * pv_factor(i) * 2^-24.
__device__ __forceinline__ uint32_t pv_reg(uint32_t P1, uint32_t P2, uint32_t P3, uint32_t P4, int i) {
    switch (i) {
        case 0: return P1 & kM0;
        case 1: return P1 & kM1;
        case 2: return P1 & kM2;
        case 3: return P1 & kM3;
        case 4: return P1 & kM4;
        case 5: return P2 & kM1;
        case 6: return P2 & kM2;
        case 7: return P2 & kM3;
        case 8: return P2 & kM4;
        case 9: return P3 & kM1;
        case 10: return P3 & kM2;
        case 11: return P3 & kM3;
        case 12: return P3 & kM4;
        case 13: return P4 & kM1;
        case 14: return P4 & kM2;
        default: return P4 & kM3;
    }
}
// factors of registers 0..15: 1, 4, 16, 64, 256, 4, 16, 64, 256, 4, 16, 64, 256, 4, 16, 64
__device__ __host__ constexpr float pv_factor(int i) {
    return i == 0 ? 1.f : (i % 4 == 0 ? 256.f : (float)(1 << (2 * (i % 4))));
}

struct MmaArgs {
    const float *q_rot;
    Int2PoolView pool;
    const int32_t *pt;
    int max_pages, page_size, n_kv, sink;
    const int32_t *seq_len, *hist_end;
    float scale2;
    PartialsView out;
    int32_t *status;
    int stages, stage_bytes, off_v, off_s, arr_bytes, ws_bytes, stage_off;
    int csize;        // CTAs per cluster; each cluster writes one partial slot
    int res_off;      // byte offset (from the first stage) of the per-CTA result area
    int hist_ctas;    // CTAs of grid.x that take the history (after the window CTAs)
    int hist_lo;      // the history this launch takes starts at max(hist_lo, sink) (a tile boundary)
    int slot0;        // its splits write partial slots slot0 .. S - 1 (slots below: another launch's)
    int win_ctas;     // CTAs [0, win_ctas) of grid.x take the BF16 window (whole clusters)
    int win_heads;    // kv heads per window cluster
    const float *RK;            // non-null: history CTAs rotate q themselves (q_rot unused)
    int rot_off;                // byte offset (from the aligned base) of the rotated-query rows [Hq][128]
    int wbuf_tok;               // window CTAs: tokens per row buffer (two buffers from the first stage)
    int wbuf_bytes;             // window CTAs: bytes available for the two buffers
    int rk_chunk;               // bytes of R staged per step in the stage area by the window CTAs' demotion
    const uint16_t *q;          // raw bf16 queries (window CTAs, and the rotation when RK is set)
    FusedDemotion dem;          // per-step demotion done by the window CTAs (dem.dem_pos NULL: none)
    int group;
    // per-request arrival counts for the merge launch (NULL: the merge waits for the whole grid)
    int32_t *arrivals;          // [batch]: +1 per cluster once its partial slot is written
    // dynamic tile scheduling (NULL: fixed splits): [batch] units taken, [batch] CTAs done
    int32_t *sched;
    int pf_units;               // dynamic units: the taker of unit u brings unit u + pf_units into L2 (0: none)
    Bf16PoolView bpool;         // BF16 sink/recent pool and its page table (window CTAs)
    const int32_t *bpt;
};

// Per-CTA result area: m [Hq], l [Hq], then acc [Hq][128] from float res_acc(Hq) on, a multiple
// of 4 floats so that the accumulator rows take 16-byte vector stores for any Hq.  The cluster
// combine's receive area follows it: one record per (source CTA, query head), kRec floats each.
__host__ __device__ constexpr int res_acc(int Hq) { return (2 * Hq + 3) & ~3; }
__host__ __device__ constexpr int res_floats(int Hq) { return res_acc(Hq) + Hq * kHeadDim; }
constexpr int kRec = kHeadDim + 4;   // acc [128], m, l, 2 unused
// bytes of the receive area for n query heads (clusters of at most 8 CTAs: at most n + 7 records)
// and, after it, one record's room for the combine's weights (J (C + 1) <= 96 floats)
__host__ __device__ constexpr int recv_bytes(int n) { return (n + 8) * kRec * 4; }

// Cluster reduction: every CTA of a cluster holds (m, l, acc) for each query head of its
// sub-split in `res`; CTA `rank` combines query heads hq0 + rank, hq0 + rank + C, ... (of the nhq
// heads from hq0 on) over the C CTAs in rank order and writes partial slot `slot`.  Each CTA first
// pushes its results to the owning CTAs (16-byte remote stores into their receive areas, right
// after `res`), so that the owners combine from their own shared memory.  Every thread calls this.
__device__ __forceinline__ void cluster_combine(const MmaArgs &a, const float *res, int Hq, int b, int slot,
                                                int hq0 = 0, int nhq = -1) {
    const int C = a.csize;
    if (nhq < 0) nhq = Hq;
    const int J = (nhq + C - 1) / C;                     // query heads per owning CTA
    float *recv = const_cast<float *>(res) + res_floats(Hq);   // [C sources][J][kRec]
    cluster_sync_all();                 // every CTA of the cluster has its result and a free receive area
    const int rank = (int)cluster_ctarank();
    constexpr int kQ = kRec / 4;                         // float4 per record
    for (int e = threadIdx.x; e < nhq * kQ; e += blockDim.x) {
        const int i = e / kQ, p = e % kQ, hq = hq0 + i;
        const float4 v = p < kHeadDim / 4 ? *reinterpret_cast<const float4 *>(res + res_acc(Hq) + hq * kHeadDim + 4 * p)
                                          : make_float4(res[hq], res[Hq + hq], 0.f, 0.f);
        float *dst = recv + (size_t)(rank * J + i / C) * kRec + 4 * p;
        st_dsmem_f32x4(saddr(dst), (uint32_t)(i % C), v);
    }
    cluster_sync_all();                 // every record is in place (no CTA reads another's memory after this)
    const size_t S1 = (size_t)a.out.S + 1;
    const int mine = (nhq - rank + C - 1) / C;
    // per owned head j: the maximum M_j of the C sources and their weights 2^(m - M_j), once
    // (wt[j][0] = M_j, wt[j][1 + q] = weight of source q), after the receive area
    float *wt = recv + (size_t)(Hq + 7) * kRec;
    for (int e = threadIdx.x; e < mine * C; e += blockDim.x) {
        const int j = e / C, q = e % C;
        float M = -INFINITY;
        for (int q2 = 0; q2 < C; ++q2) M = fmaxf(M, recv[(q2 * J + j) * kRec + kHeadDim]);
        if (q == 0) wt[j * (C + 1)] = M;
        wt[j * (C + 1) + 1 + q] = M != -INFINITY ? exp2f(recv[(q * J + j) * kRec + kHeadDim] - M) : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < mine * kHeadDim; e += blockDim.x) {
        const int j = e / kHeadDim, d = e % kHeadDim, hq = hq0 + rank + j * C;
        const float *w = wt + j * (C + 1);
        const float M = w[0];
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int q = 0; q < C; ++q) {
                const float *r = recv + (q * J + j) * kRec;
                const float f = w[1 + q];
                if (d == 0) L = fmaf(r[kHeadDim + 1], f, L);
                A = fmaf(r[d], f, A);
            }
        }
        const size_t row = ((size_t)b * Hq + hq) * S1 + slot;
        a.out.acc[row * kHeadDim + d] = A;
        if (d == 0) {
            a.out.m[row] = M;
            a.out.l[row] = L;
        }
    }
}


// Fold U tokens (K/V rows kk, vv: lane l holds channels 4l..4l+3; ok[u] = token present) into
// the online softmax (base 2) of the warp's G query heads.  The U*G per-lane partial dot
// products are summed across the warp by a reduce-scatter (each step halves the values a lane
// keeps), so a sum costs about one shuffle instead of five; the sums are then broadcast and
// every lane updates m, l and its accumulator channels for all heads.
template <int G, int U>
__device__ __forceinline__ void window_fold(const float (&q)[G][4], const uint2 (&kk)[U], const uint2 (&vv)[U],
                                            const bool (&ok)[U], float scale2, float (&m)[G], float (&l)[G],
                                            float (&acc)[G][4], int lane) {
    constexpr int V = U * G;                           // value index u * G + hh
    static_assert((V & (V - 1)) == 0 && V <= 32, "U * G must be a power of two up to 32");
    constexpr int LOGV = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : 5;
    float v[V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float k0 = __uint_as_float(kk[u].x << 16), k1 = __uint_as_float(kk[u].x & 0xffff0000u);
        const float k2 = __uint_as_float(kk[u].y << 16), k3 = __uint_as_float(kk[u].y & 0xffff0000u);
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
            v[u * G + hh] = fmaf(q[hh][3], k3, fmaf(q[hh][2], k2, fmaf(q[hh][1], k1, q[hh][0] * k0)));
    }
    // reduce-scatter: at distance D = 16 >> k a lane keeps the upper half of its n values when
    // lane & D, the lower half otherwise; after LOGV steps v[0] is value idx(lane), then plain sums
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int D = 16 >> k;
        const int n = V >> k;
        if (n > 1) {
            const bool up = (lane & D) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = up ? v[i] : v[i + n / 2];
                const float keep = up ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, D);
            }
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], D);
        }
    }
    float t[V];                                        // every lane: all U x G logits (base 2)
#pragma unroll
    for (int j = 0; j < V; ++j) {
        int src = 0;                                   // the lane holding value j
#pragma unroll
        for (int k = 0; k < LOGV; ++k) src |= ((j >> (LOGV - 1 - k)) & 1) * (16 >> k);
        t[j] = __shfl_sync(0xffffffffu, v[0], src) * scale2;
    }
    float vf[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        vf[u][0] = __uint_as_float(vv[u].x << 16); vf[u][1] = __uint_as_float(vv[u].x & 0xffff0000u);
        vf[u][2] = __uint_as_float(vv[u].y << 16); vf[u][3] = __uint_as_float(vv[u].y & 0xffff0000u);
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float mx = m[hh];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (ok[u]) mx = fmaxf(mx, t[u * G + hh]);
        if (mx == -INFINITY) continue;                  // nothing folded yet for this head
        const float al = ex2_approx(m[hh] - mx);
        float ls = 0.f, a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float pr = ok[u] ? ex2_approx(t[u * G + hh] - mx) : 0.f;
            ls += pr;
#pragma unroll
            for (int c = 0; c < 4; ++c) a4[c] = fmaf(pr, vf[u][c], a4[c]);
        }
        l[hh] = fmaf(l[hh], al, ls);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[hh][c] = fmaf(acc[hh][c], al, a4[c]);
        m[hh] = mx;
    }
}

// ---- BF16 sink/recent window, on CUDA cores, in the window clusters (first in the grid).
// Window positions of request b, in order: [0, n0) then [lo1, T), n0 = min(sink, T),
// lo1 = max(h_end, n0).  Window cluster k takes kv heads [k nh, (k + 1) nh) (nh = win_heads);
// its CTA of rank r takes positions [r n / C, (r + 1) n / C).  Warp w takes kv head k nh + w % nh
// and every (8 / nh)-th group of positions of that range; lane l owns channels 4l..4l+3.  Each
// token is folded into a per-warp online softmax (base 2), the warps of a kv head are combined in
// a fixed order, and the CTA's result goes to the cluster combine or straight to partial slot S.
// The K and V rows come through shared memory: the copy warp fills chunks of up to 32 tokens (this
// cluster's heads of each token: one bulk copy per token for K and one for V) in two buffers, so
// that up to two chunks are in flight at once.  `area` is the CTA's stage area; after the fold it
// holds the warp results and the CTA result.  Every thread of the CTA calls this.
template <int G>
__device__ void window_cta(const MmaArgs &a, uint8_t *area, uint64_t *wbar, int T, int he, int b, int wr) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = a.n_kv, Hq = Hkv * G, S = a.out.S;
    const int C = a.csize, nh = a.win_heads;
    const int h0 = (wr / C) * nh, rk = wr % C;
    const int n0 = min(a.sink, T), lo1 = max(he, n0);
    const int n = n0 + (T - lo1);
    const int i_lo = (int)((long long)rk * n / C), i_hi = (int)((long long)(rk + 1) * n / C);
    float m[G], l[G], acc[G][4];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[hh][c] = 0.f;
    }
    const int hl = warp % nh, h = h0 + hl, sub = warp / nh, nsub = kCW / nh;
    float q[G][4];
    if (warp < kCW) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const uint2 v = reinterpret_cast<const uint2 *>(a.q + ((size_t)b * Hq + h * G + hh) * kHeadDim)[lane];
            q[hh][0] = __uint_as_float(v.x << 16); q[hh][1] = __uint_as_float(v.x & 0xffff0000u);
            q[hh][2] = __uint_as_float(v.y << 16); q[hh][3] = __uint_as_float(v.y & 0xffff0000u);
        }
    }
    constexpr int U = 4;
    if (a.wbuf_tok >= U) {
        const int CH = a.wbuf_tok, nt = i_hi - i_lo, nch = (nt + CH - 1) / CH;
        const int rowb = nh * kHeadDim * 2;                   // this cluster's heads of one token's K (or V) row
        uint32_t *valid = reinterpret_cast<uint32_t *>(wbar + 2);   // per buffer: bit j = token j's page is valid
        auto fill = [&](int k) {                              // the copy warp; lane j copies token j of the chunk
            const int buf = k & 1, j0 = k * CH, cnt = min(CH, nt - j0);
            uint8_t *dk = area + (size_t)buf * 2 * CH * rowb, *dv = dk + (size_t)CH * rowb;
            size_t row = 0;
            bool ok = false;
            if (lane < cnt) {
                const int i = i_lo + j0 + lane;
                const int p = i < n0 ? i : lo1 + (i - n0);
                const int page = p / a.page_size < a.max_pages ? a.bpt[(size_t)b * a.max_pages + p / a.page_size] : -1;
                ok = page >= 0 && page < a.bpool.n_pages;
                if (ok) row = ((size_t)page * a.page_size + p % a.page_size) * Hkv + h0;
                else flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
            }
            const uint32_t vbits = __ballot_sync(0xffffffffu, ok);
            fence_proxy_async_smem();                         // the warps' reads of this buffer came first
            if (lane == 0) {
                valid[buf] = vbits;
                mbar_arrive_expect_tx(saddr(&wbar[buf]), 2u * (uint32_t)__popc(vbits) * rowb);
            }
            __syncwarp();
            if (ok) {
                // (the window rows are read once per step: evict-first in L2)
                const uint64_t pol = l2_evict_first_policy();
                tma_load_1d(saddr(dk + (size_t)lane * rowb), a.bpool.k + row * kHeadDim, rowb, saddr(&wbar[buf]), pol);
                tma_load_1d(saddr(dv + (size_t)lane * rowb), a.bpool.v + row * kHeadDim, rowb, saddr(&wbar[buf]), pol);
            }
        };
        if (threadIdx.x == 0) {
            mbar_init(saddr(&wbar[0]), 1);
            mbar_init(saddr(&wbar[1]), 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (warp == kCW)
            for (int k = 0; k < 2 && k < nch; ++k) fill(k);
        for (int k = 0; k < nch; ++k) {
            const int buf = k & 1, cnt = min(CH, nt - k * CH);
            if (warp < kCW) {
                if (!mbar_wait(saddr(&wbar[buf]), (k >> 1) & 1) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                const uint32_t vb = valid[buf];
                const uint8_t *dk = area + (size_t)buf * 2 * CH * rowb, *dv = dk + (size_t)CH * rowb;
                for (int j0 = sub * U; j0 < cnt; j0 += U * nsub) {
                    uint2 kk[U], vv[U];
                    bool ok[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int j = j0 + u;
                        ok[u] = j < cnt && ((vb >> j) & 1);
                        const size_t off = (size_t)(ok[u] ? j : 0) * rowb + hl * kHeadDim * 2;
                        kk[u] = reinterpret_cast<const uint2 *>(dk + off)[lane];
                        vv[u] = reinterpret_cast<const uint2 *>(dv + off)[lane];
                    }
                    window_fold<G, U>(q, kk, vv, ok, a.scale2, m, l, acc, lane);
                }
            }
            __syncthreads();                                  // buffer `buf` is consumed
            if (warp == kCW && k + 2 < nch) fill(k + 2);
        }
        // (the consumer warps waited for every fill; after a wait that gave up, the copy warp makes
        // sure that no copy is still landing before the buffers are reused and the CTA leaves)
        if (warp == kCW)
            for (int k = nch > 2 ? nch - 2 : 0; k < nch; ++k)
                if (!mbar_wait(saddr(&wbar[k & 1]), (k >> 1) & 1) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
    } else if (warp < kCW) {
        // (buffers too small for the layout) Tokens in chunks of 64 per warp: the chunk's page ids
        // are read once (two per lane), then U tokens' K/V rows are loaded together and folded.
        for (int c0 = i_lo + sub; c0 < i_hi; c0 += 64 * nsub) {
          int pg[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
              const int i = c0 + (lane + 32 * r) * nsub;
              pg[r] = -1;
              if (i < i_hi) {
                  const int p = i < n0 ? i : lo1 + (i - n0);
                  pg[r] = a.bpt[(size_t)b * a.max_pages + p / a.page_size];
              }
          }
          for (int k0 = 0; k0 < 64 && c0 + k0 * nsub < i_hi; k0 += U) {
            const int pgr = k0 < 32 ? pg[0] : pg[1];
            uint2 kk[U], vv[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = c0 + (k0 + u) * nsub;
                const int page = __shfl_sync(0xffffffffu, pgr, (k0 & 31) + u);
                ok[u] = false;
                kk[u] = vv[u] = make_uint2(0u, 0u);
                if (i < i_hi) {
                    const int p = i < n0 ? i : lo1 + (i - n0);
                    if (page >= 0 && page < a.bpool.n_pages) {
                        const size_t row = ((size_t)page * a.page_size + p % a.page_size) * Hkv + h;
                        kk[u] = __ldg(reinterpret_cast<const uint2 *>(a.bpool.k + row * kHeadDim) + lane);
                        vv[u] = __ldg(reinterpret_cast<const uint2 *>(a.bpool.v + row * kHeadDim) + lane);
                        ok[u] = true;
                    } else if (lane == 0) {
                        flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
                    }
                }
            }
            window_fold<G, U>(q, kk, vv, ok, a.scale2, m, l, acc, lane);
          }
        }
    }
    __syncthreads();                                          // (the row buffers are consumed)
    // warp results: wsm = [warp][G] m, [warp][G] l, [warp][G][128] acc; the CTA result after them
    float *wsm = reinterpret_cast<float *>(area);
    float *res = wsm + kCW * G * (2 + kHeadDim);
    if (warp < kCW) {
        float *wm = wsm, *wl = wsm + kCW * G, *wa = wsm + 2 * kCW * G;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            if (lane == 0) {
                wm[warp * G + hh] = m[hh];
                wl[warp * G + hh] = l[hh];
            }
            *reinterpret_cast<float4 *>(wa + (warp * G + hh) * kHeadDim + 4 * lane) =
                make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
        }
    }
    pdl_trigger();
    __syncthreads();
    const bool to_res = C > 1;
    const float *wm = wsm, *wl = wsm + kCW * G, *wa = wsm + 2 * kCW * G;
    for (int e = threadIdx.x; e < nh * G * kHeadDim; e += blockDim.x) {
        const int hq = h0 * G + e / kHeadDim, d = e % kHeadDim, hv = hq / G - h0, hh = hq % G;
        float M = -INFINITY;
        for (int w = hv; w < kCW; w += nh) M = fmaxf(M, wm[w * G + hh]);
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int w = hv; w < kCW; w += nh) {
                const float f = exp2f(wm[w * G + hh] - M);
                L = fmaf(wl[w * G + hh], f, L);
                A = fmaf(wa[(w * G + hh) * kHeadDim + d], f, A);
            }
        }
        if (to_res) {
            res[res_acc(Hq) + hq * kHeadDim + d] = A;
            if (d == 0) {
                res[hq] = M;
                res[Hq + hq] = L;
            }
        } else {
            const size_t row = ((size_t)b * Hq + hq) * (S + 1) + S;
            a.out.acc[row * kHeadDim + d] = A;
            if (d == 0) {
                a.out.m[row] = M;
                a.out.l[row] = L;
            }
        }
    }
    if (to_res) cluster_combine(a, res, Hq, b, S, h0 * G, nh * G);
}

// ---- Per-step demotion by the window CTAs: request b's position dem_pos[b] (one that left the
// recent window; this launch still reads it from BF16) is rotated by R_K / R_V, clipped,
// quantized and packed into the INT2 pool for kv heads wr, wr + wc, ...  The arithmetic is
// oscar_demote's: y_j = fma-chain_i x_i * R[i][j] (i ascending, fp32), or y = x for values when
// R_V is NULL, then the shared quantizer.  R is staged through the stage area a chunk at a time.
// All threads call this.
__device__ void window_demote(const MmaArgs &a, float *small, uint8_t *area, int T, int he, int b, int wr, int wc) {
    const int tid = threadIdx.x;
    const int Hkv = a.n_kv, ps = a.page_size;
    const int p = a.dem.dem_pos[b];
    if (p < 0) return;
    int sp = -1, dp = -1;
    const bool in_range = p >= he && p < T && p / ps < a.max_pages;
    if (in_range) {
        sp = a.bpt[(size_t)b * a.max_pages + p / ps];
        dp = a.pt[(size_t)b * a.max_pages + p / ps];
    }
    if (!in_range || sp < 0 || sp >= a.bpool.n_pages || dp < 0 || dp >= a.dem.dst.n_pages) {
        if (tid == 0)
            flag_status(a.status, !in_range ? OSCAR_DEV_BAD_LENGTH
                                            : (sp < 0 || sp >= a.bpool.n_pages) ? OSCAR_DEV_BAD_BF16_PAGE
                                                                                : OSCAR_DEV_BAD_INT2_PAGE);
        return;
    }
    float *xs = small;                           // [128] the source row
    float *red = small + kHeadDim;               // [8]
    uint64_t *bar = reinterpret_cast<uint64_t *>(small + kHeadDim + 8);   // R chunk landed (expect-tx)
    float *Rs = reinterpret_cast<float *>(area);
    const int rpc = a.rk_chunk / (kHeadDim * 4), nch = kHeadDim / rpc;
    const int gpr = kHeadDim / a.group;
    const size_t srow = ((size_t)sp * ps + p % ps) * Hkv, drow = ((size_t)dp * ps + p % ps) * Hkv;
    if (tid == 0) {
        mbar_init(saddr(bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    int n = 0;                                   // bulk copies so far (phase parity)
    for (int hk = wr; hk < Hkv; hk += wc) {
        for (int which = 0; which < 2; ++which) {
            const float *Rb = which ? a.dem.RV : a.RK;       // NULL R_V: values stored as they are
            const float *R = Rb ? Rb + (size_t)hk * kHeadDim * kHeadDim : nullptr;
            __syncthreads();                     // the previous row's xs and Rs are consumed
            if (tid < kHeadDim) xs[tid] = bf16_to_f32((which ? a.bpool.v : a.bpool.k)[(srow + hk) * kHeadDim + tid]);
            float y = 0.f;
            if (!R) {
                __syncthreads();
                if (tid < kHeadDim) y = xs[tid];
            }
            for (int c = 0; c < (R ? nch : 0); ++c, ++n) {
                if (c > 0) __syncthreads();
                if (tid == 0) {                  // one bulk copy of the chunk (rows c*rpc ...)
                    fence_proxy_async_smem();    // the area held the window's generic stores
                    mbar_arrive_expect_tx(saddr(bar), a.rk_chunk);
                    tma_load_1d(saddr(Rs), R + (size_t)c * rpc * kHeadDim, a.rk_chunk, saddr(bar));
                }
                if (!mbar_wait(saddr(bar), n & 1) && tid == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                __syncthreads();
                if (tid < kHeadDim) {
#pragma unroll 8
                    for (int i = 0; i < rpc; ++i) y = __fmaf_rn(xs[c * rpc + i], Rs[i * kHeadDim + tid], y);
                }
            }
            if (tid < kHeadDim) {                // warps 0..3: one channel each
                uint8_t *codes = which ? a.dem.dst.codes_v : a.dem.dst.codes_k;
                uint16_t *scale = which ? a.dem.dst.scale_v : a.dem.dst.scale_k;
                uint16_t *zero = which ? a.dem.dst.zero_v : a.dem.dst.zero_k;
                const size_t r = drow + hk;
                quantize_row_store(y, which ? a.dem.cV : a.dem.cK, a.group, true, codes + r * (kHeadDim / 4),
                                   scale + r * gpr, zero + r * gpr, red, tid,
                                   [] { asm volatile("bar.sync 2, 128;" ::: "memory"); });
            }
        }
    }
}

// ---- The same per-step demotion of kv head hk (K for which = 0, V for 1, from w0 to w1 - 1), done
// by the consumer warps 0..3 of a history CTA before its main loop (with dynamic history units,
// whose sharing absorbs the delay).  R is read from global memory (L2: every request's demotion
// reads it); the stage area holds the KV stream.  xs: 136 floats of free shared memory.  Threads
// 0..127 call this.
__device__ void history_demote(const MmaArgs &a, float *xs, int T, int he, int b, int hk, int w0, int w1) {
    const int tid = threadIdx.x;
    const int Hkv = a.n_kv, ps = a.page_size;
    const int p = a.dem.dem_pos[b];
    if (p < 0) return;
    int sp = -1, dp = -1;
    const bool in_range = p >= he && p < T && p / ps < a.max_pages;
    if (in_range) {
        sp = a.bpt[(size_t)b * a.max_pages + p / ps];
        dp = a.pt[(size_t)b * a.max_pages + p / ps];
    }
    if (!in_range || sp < 0 || sp >= a.bpool.n_pages || dp < 0 || dp >= a.dem.dst.n_pages) {
        if (tid == 0)
            flag_status(a.status, !in_range ? OSCAR_DEV_BAD_LENGTH
                                            : (sp < 0 || sp >= a.bpool.n_pages) ? OSCAR_DEV_BAD_BF16_PAGE
                                                                                : OSCAR_DEV_BAD_INT2_PAGE);
        return;
    }
    float *red = xs + kHeadDim;
    const int gpr = kHeadDim / a.group;
    const size_t srow = ((size_t)sp * ps + p % ps) * Hkv + hk, drow = ((size_t)dp * ps + p % ps) * Hkv + hk;
    auto sync128 = [] { asm volatile("bar.sync 2, 128;" ::: "memory"); };
    for (int which = w0; which < w1; ++which) {
        const float *Rb = which ? a.dem.RV : a.RK;       // NULL R_V: values stored as they are
        sync128();                                       // the previous row's xs is consumed
        xs[tid] = bf16_to_f32((which ? a.bpool.v : a.bpool.k)[srow * kHeadDim + tid]);
        sync128();
        float y = 0.f;
        if (!Rb) {
            y = xs[tid];
        } else {
            const float *R = Rb + (size_t)hk * kHeadDim * kHeadDim + tid;
            for (int i0 = 0; i0 < kHeadDim; i0 += 16) {
                float rv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) rv[u] = __ldg(R + (size_t)(i0 + u) * kHeadDim);
#pragma unroll
                for (int u = 0; u < 16; ++u) y = __fmaf_rn(xs[i0 + u], rv[u], y);
            }
        }
        uint8_t *codes = which ? a.dem.dst.codes_v : a.dem.dst.codes_k;
        uint16_t *scale = which ? a.dem.dst.scale_v : a.dem.dst.scale_k;
        uint16_t *zero = which ? a.dem.dst.zero_v : a.dem.dst.zero_k;
        quantize_row_store(y, which ? a.dem.cV : a.dem.cK, a.group, true, codes + drow * (kHeadDim / 4),
                           scale + drow * gpr, zero + drow * gpr, red, tid, sync128);
    }
}

// ---- Arrival count for the merge launch: once every CTA of the cluster has written its part of
// the cluster's partial slot, one thread adds 1 to arrivals[b].  The fence orders each thread's
// slot writes before the cluster barrier, and the barrier before the count (release at gpu
// scope), so a merge CTA that reads the full count with acquire sees every slot.  Every thread
// of the CTA calls this.
__device__ __forceinline__ void arrive_count(const MmaArgs &a, int b) {
    const int C = a.csize;
    __threadfence();
    if (C > 1) cluster_sync_all(); else __syncthreads();
    if ((C > 1 ? cluster_ctarank() : 0) == 0 && threadIdx.x == 0) {
        __threadfence();
        atomicAdd(a.arrivals + b, 1);
    }
}

constexpr float kLazy = 8.0f;   // log2 headroom before the running maximum is raised
// The running maximum before any finite logit: far below every logit, so that 2^(logit - it) and
// 2^(it - first maximum) underflow to 0 and the first finite maximum always raises it (no test for
// "no maximum yet" per token); masked tokens (-inf) still give 0.
constexpr float kNoMax = -0x1p100f;
// rotated-query rows in shared memory: element d of a row at d + 4 (d / 32) (row stride 144), so
// that the operand reads of a warp (4 heads x 4 column groups) spread over the banks and every
// run of 4 columns stays 16-byte aligned (the cluster's CTAs push the rows 4 columns at a time)
constexpr int kQS = kHeadDim + kHeadDim / 8;
__device__ __forceinline__ int qs_col(int d) { return d + 4 * (d >> 5); }
constexpr int kWsWords = 20;    // words per P-operand column: 2 tiles x 8 + 4 (bank spread)


// (v0, v1) -> f16x2 of the round-to-nearest values (hi) and f16x2 of their residuals (lo)
__device__ __forceinline__ void split2(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(v0, v1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// TMA: 8 kv heads.  The copy warp moves a stage's codes with 3-D tensor-map boxes of whole
// 256-byte rows (128-byte swizzle; one box per array for a unit inside one page, else one per tile)
// and its scale/zero rows with 1-D bulk copies; otherwise (1, 2 or 4 kv heads) it scatters
// 16-byte cp.async chunks head-major.
template <int G, int NGRP, bool TMA>
__global__ void __launch_bounds__(kThreads, (G == 8 ? 1 : 2))
    int2_mma_kernel(MmaArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tmk1, const __grid_constant__ CUtensorMap tmv1) {
    constexpr int NT = (G == 8) ? 2 : 1;      // n-tiles of 8 columns: 4 heads x {hi, lo} each
    constexpr int NCOL = 8 * NT;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // swizzled boxes land on 1024-byte boundaries: the carve-up starts at an aligned address
    uint8_t *smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);   // full[0..3], empty[4..7]
    int *masks = reinterpret_cast<int *>(smem + 64);        // per stage: bit j = tile j holds data
    uint8_t *stage0 = smem + a.stage_off;

    // grid.x: the window cluster first (so that it starts at once and its work hides behind the
    // history), then the history CTAs; s = this CTA's index among the history CTAs.
    const int s = (int)blockIdx.x - a.win_ctas, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // With 8 kv heads (the tensor-map path) the stage layout is compile-time: addresses fold.
    const int Hkv = TMA ? 8 : a.n_kv, Hq = Hkv * G, S = a.out.S;
    constexpr int kCodesTma = kTilesPerStage * 4096;     // one array's codes of a stage (8 kv heads)
    const int off_v = TMA ? kCodesTma : a.off_v, off_s = TMA ? 2 * kCodesTma : a.off_s;
    const int arr_bytes = TMA ? kStageTok * 8 * NGRP * 2 : a.arr_bytes;
    const int stage_bytes = TMA ? ((2 * kCodesTma + 4 * kStageTok * 8 * NGRP * 2 + 127) & ~127) : a.stage_bytes;
    int T, he;
    read_lengths(a.seq_len, a.hist_end, b, a.sink, a.max_pages * a.page_size, a.status, T, he);
    if (s < 0) {                               // a BF16 window CTA (uniform over the cluster)
        pdl_wait();                            // q and the partials belong to the previous kernels
        window_cta<G>(a, stage0, reinterpret_cast<uint64_t *>(smem + 112), T, he, b, (int)blockIdx.x);
        // (after the cluster's last barrier: the stage area is free again)
        if (a.dem.dem_pos && !(a.sched && a.hist_ctas >= Hkv))
            window_demote(a, reinterpret_cast<float *>(smem + 128), stage0, T, he, b, (int)blockIdx.x, a.win_ctas);
        if (a.arrivals) arrive_count(a, b);
        return;
    }
    // this launch's history: [hl, he) (hist_lo above the sink: a shared prefix another launch takes)
    const int hl = min(max(a.hist_lo, a.sink), he);
    const SplitRange r = history_split(hl, he, a.hist_ctas, s);       // C sub-splits per slot
    // Dynamic scheduling: the copy warps of all of b's history CTAs take units of kTilesPerStage
    // tiles of the whole history [sink, he) from a shared counter, so that CTAs that run faster
    // (an SM to themselves) take more; each stage carries its first tile (or -1: no more).
    const bool dyn = a.sched != nullptr;
    const int hist_first = hl / kTileTokens;       // the history starts on a tile boundary
    const int hist_tile_hi = (he + kTileTokens - 1) / kTileTokens;
    const int dyn_units = hist_tile_hi > hist_first ? (hist_tile_hi - hist_first + kTilesPerStage - 1) / kTilesPerStage : 0;
    const int tok_hi = dyn ? he : r.hi, tile_hi = dyn ? hist_tile_hi : r.tile_hi;
    int *stage_tile = reinterpret_cast<int *>(smem + 80);     // per stage: first tile, -1 = the end

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(saddr(&bars[i]), TMA ? 1 : 33);   // TMA: the expect-tx arrival; else 32 cp.async + mask
            mbar_init(saddr(&bars[4 + i]), kCW);
        }
        if (a.RK && a.csize > 1) mbar_init(saddr(smem + 104), 1);   // the peers' rotated-query rows landed
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // With the fused rotation each CTA of a cluster rotates the queries of some kv heads and sends
    // the rows to its peers with bulk copies that complete on their smem + 104 barrier: every CTA
    // initialises that barrier before any peer may copy into it (the cluster barrier below), and
    // expects the bytes of the rows it does not compute itself.
    const bool rot_phase = a.RK && a.csize > 1;
    if (rot_phase) {
        cluster_sync_all();
        if (threadIdx.x == 0) {
            const int C = a.csize, rank = (int)cluster_ctarank();
            const int own = rank < Hkv ? (Hkv - 1 - rank) / C + 1 : 0;
            mbar_arrive_expect_tx(saddr(smem + 104), (uint32_t)((Hkv - own) * G * kQS * 4));
        }
    }

    // ------------------------------------------------------------ producer --
    if (warp == kCW) {
        // The KV copies start at the launch, while the consumer warps load R_K and q and rotate (with
        // the unit-sized copies this measured faster than holding them until R_K and q had landed:
        // 35.8 against 36.4 us per layer at 100K tokens, 25.2 against 25.7 at 32K).
        const int lgH = Hkv == 1 ? 0 : Hkv == 2 ? 1 : Hkv == 4 ? 2 : 3;
        // Page ids of 32 consecutive logical pages, lane i holding page pg_base + i: one load
        // serves 32 pages (128 tiles at 64-token pages), so the copies never wait on the table.
        const int tpp = a.page_size / kTileTokens;           // tiles per page
        const int tile_bytes = 2 * kTileTokens * 8 * 32 + 4 * kTileTokens * 8 * NGRP * 2;   // TMA path (8 heads)
        const int32_t *prow = a.pt + (size_t)b * a.max_pages;
        int pg_base = (dyn ? hist_first : r.tile_lo) / tpp;
        int pg_reg = (pg_base + lane < a.max_pages) ? prow[pg_base + lane] : -1;
        // dynamic units: the next unit and its tiles' page ids (lane j < kTilesPerStage: tile
        // t0 + j) are taken one stage ahead, so that the count and the table loads overlap the wait
        // Units are handed out in order, so unit u + pf_units is taken about pf_units / (history CTAs)
        // stages later: its taker-to-be finds it in L2 if the taker of u asks for it now (lanes
        // kTilesPerStage .. 2 kTilesPerStage - 1 load its tiles' page ids and issue the L2 prefetches).
        // This keeps more of the history in flight than the shared-memory stages hold.
        auto take_unit = [&](int &nt0, int &npg) {
            int u = 0;
            if (lane == 0) u = atomicAdd(a.sched + b, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            nt0 = u < dyn_units ? hist_first + u * kTilesPerStage : -1;
            const int pu = u + a.pf_units, j = lane - kTilesPerStage;
            const bool pf = a.pf_units > 0 && j >= 0 && j < kTilesPerStage && pu < dyn_units;
            const int tile = pf ? hist_first + pu * kTilesPerStage + j : nt0 + lane;
            const bool ld = pf || (nt0 >= 0 && lane < kTilesPerStage);
            npg = (ld && tile < tile_hi) ? prow[tile / tpp] : -1;
            if (pf && npg >= 0 && npg < a.pool.n_pages) {
                const size_t row0 = (size_t)npg * a.page_size + (tile * kTileTokens) % a.page_size;
                const uint32_t cb = kTileTokens * Hkv * 32, sbt = kTileTokens * Hkv * NGRP * 2;
                prefetch_l2(a.pool.codes_k + row0 * Hkv * 32, cb);
                prefetch_l2(a.pool.codes_v + row0 * Hkv * 32, cb);
                const size_t so = row0 * Hkv * NGRP;
                prefetch_l2(a.pool.scale_k + so, sbt);
                prefetch_l2(a.pool.zero_k + so, sbt);
                prefetch_l2(a.pool.scale_v + so, sbt);
                prefetch_l2(a.pool.zero_v + so, sbt);
            }
        };
        int nxt_t0 = -1, nxt_pg = -1;
        if (dyn) take_unit(nxt_t0, nxt_pg);
        int fix_t0 = r.tile_lo;                                // fixed splits: the next stage's first tile
        bool ok = true;
        int armed = 0;                                         // stage fills started (expect-tx armed)
        for (int it = 0; ok; ++it) {
            const int st = it % a.stages;
            if (it >= a.stages && !mbar_wait(saddr(&bars[4 + st]), ((it / a.stages) - 1) & 1)) {
                if (lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                ok = false;
                break;
            }
            armed = it + 1;
            int t0, unit_pg = -1;                              // this stage's first tile, -1: no more
            // (with dynamic units the next unit is taken after this stage's copies are issued: the
            // count's round trip and the page-table load then overlap the wait for the next stage)
            if (dyn) {
                t0 = nxt_t0;
                unit_pg = nxt_pg;
            } else {
                t0 = fix_t0 < r.tile_hi ? fix_t0 : -1;
            }
            if (lane == 0) stage_tile[st] = t0;
            if (t0 < 0) {                                      // an empty stage marks the end
                if constexpr (TMA) {
                    if (lane == 0) {
                        masks[st] = 0;
                        mbar_arrive_expect_tx(saddr(&bars[st]), 0);
                    }
                } else {
                    if (lane == 0) masks[st] = 0;
                    cp_async_arrive(saddr(&bars[st]));
                    if (lane == 0) mbar_arrive(saddr(&bars[st]));
                }
                break;
            }
            // the stage takes tiles [t0, t_stop): up to the next unit boundary counted from the first
            // history tile (a fixed split's first stage may be partial; every later one is whole)
            const int t_stop = min(tile_hi, t0 + kTilesPerStage - ((t0 - hist_first) & (kTilesPerStage - 1)));
            fix_t0 = t_stop;
            uint8_t *sb = stage0 + st * stage_bytes;
            int mask = 0;
            if constexpr (TMA) {
                // A unit whose tiles lie in one page moves with six copies, lanes 0..5: one 64-row box
                // per code array and the unit's rows of each scale/zero array.  Otherwise tile j moves
                // with lanes 8 j + op: op 0, 1 a 16-row box of the K, V codes, op 2..5 the tile's
                // scale/zero rows.  (Per copy the engine pays a fixed cost: few large copies move the
                // stage at a higher rate than a copy per tile, array and half row.)
                const bool one_page = (t0 % tpp) + kTilesPerStage <= tpp;
                const int jl = one_page ? 0 : lane >> 3, op = one_page ? lane : lane & 7;
                int row0 = 0;
                for (int j = 0; j < kTilesPerStage; ++j) {
                    const int tile = t0 + j;
                    if (tile >= t_stop) break;
                    const int lp = tile / tpp;
                    if (!dyn && lp - pg_base >= 32) {
                        pg_base = lp;
                        pg_reg = (pg_base + lane < a.max_pages) ? prow[pg_base + lane] : -1;
                    }
                    const int page = dyn ? __shfl_sync(0xffffffffu, unit_pg, j)
                                         : __shfl_sync(0xffffffffu, pg_reg, lp - pg_base);
                    if (page < 0 || page >= a.pool.n_pages) {
                        if (lane == 0) flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
                        continue;
                    }
                    mask |= 1 << j;
                    if (j == jl) row0 = page * a.page_size + (tile * kTileTokens) % a.page_size;
                }
                // (one page: the whole unit lands, also the rows past the range, which the mask hides)
                const uint32_t full = saddr(&bars[st]);
                const int nsb = kTileTokens * 8 * NGRP * 2;          // bytes of one tile's scale/zero rows
                if (lane == 0) {
                    masks[st] = mask;
                    mbar_arrive_expect_tx(full, one_page ? (mask ? kTilesPerStage * tile_bytes : 0) : __popc(mask) * tile_bytes);
                }
                __syncwarp();
                if (((mask >> jl) & 1) && op < 6) {
                    // the KV stream is read once per step: evict-first in L2, so that the lines read again
                    // (code, R_K, queries, partials) stay
                    const uint64_t pol = l2_evict_first_policy();
                    const uint32_t d = saddr(sb) + jl * 4096;
                    if (op < 2) {
                        tma_load_3d(d + op * off_v, one_page ? (op ? &tmv : &tmk) : (op ? &tmv1 : &tmk1), 0, 0, row0, full,
                                    pol);
                    } else {
                        const int arr = op - 2;
                        const uint16_t *src = arr == 0 ? a.pool.scale_k : arr == 1 ? a.pool.zero_k
                                            : arr == 2 ? a.pool.scale_v : a.pool.zero_v;
                        tma_load_1d(saddr(sb + off_s) + arr * arr_bytes + jl * nsb, src + (size_t)row0 * 8 * NGRP,
                                    one_page ? kTilesPerStage * nsb : nsb, full, pol);
                    }
                }
                if (dyn) take_unit(nxt_t0, nxt_pg);
                continue;
            }
            for (int j = 0; j < kTilesPerStage; ++j) {
                const int tile = t0 + j;
                if (tile >= t_stop) break;
                const int pos0 = tile * kTileTokens;
                const int lp = tile / tpp;
                if (!dyn && lp - pg_base >= 32) {              // warp-uniform refill of the page window
                    pg_base = lp;
                    pg_reg = (pg_base + lane < a.max_pages) ? prow[pg_base + lane] : -1;
                }
                const int page = dyn ? __shfl_sync(0xffffffffu, unit_pg, j)
                                     : __shfl_sync(0xffffffffu, pg_reg, lp - pg_base);
                if (page < 0 || page >= a.pool.n_pages) {
                    if (lane == 0) flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
                    continue;
                }
                mask |= 1 << j;
                const size_t row0 = (size_t)page * a.page_size + (pos0 % a.page_size);
                const uint8_t *srck = a.pool.codes_k + row0 * Hkv * 32;
                const uint8_t *srcv = a.pool.codes_v + row0 * Hkv * 32;
                const int nck = 32 << lgH;              // 16-byte chunks: [slot][head][2 halves]
                const uint32_t tile_dst = saddr(sb) + j * kTileTokens * 32;
                for (int c = lane; c < nck; c += 32) {
                    const int slot = c >> (lgH + 1), head = (c >> 1) & (Hkv - 1), half = c & 1;
                    const uint32_t dst = tile_dst + head * (kStageTok * 32) + slot * 32 + half * 16;
                    cp_async16(dst, srck + c * 16);
                    cp_async16(dst + off_v, srcv + c * 16);
                }
                const int nsc = (2 * NGRP) << lgH;      // 16-byte chunks of one scale/zero array
                const size_t soff = row0 * Hkv * NGRP;
                const uint32_t sdst = saddr(sb + off_s) + j * nsc * 16;
                for (int c = lane; c < nsc; c += 32) {
                    cp_async16(sdst + c * 16, reinterpret_cast<const uint8_t *>(a.pool.scale_k + soff) + c * 16);
                    cp_async16(sdst + arr_bytes + c * 16, reinterpret_cast<const uint8_t *>(a.pool.zero_k + soff) + c * 16);
                    cp_async16(sdst + 2 * arr_bytes + c * 16,
                               reinterpret_cast<const uint8_t *>(a.pool.scale_v + soff) + c * 16);
                    cp_async16(sdst + 3 * arr_bytes + c * 16,
                               reinterpret_cast<const uint8_t *>(a.pool.zero_v + soff) + c * 16);
                }
            }
            if (lane == 0) masks[st] = mask;
            cp_async_arrive(saddr(&bars[st]));
            if (lane == 0) mbar_arrive(saddr(&bars[st]));
            if (dyn) take_unit(nxt_t0, nxt_pg);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if constexpr (TMA) {
            // No copy may still be landing when the CTA leaves: after a wait that gave up, the stages'
            // last fills may be outstanding, so wait (bounded) for each of them (no wait otherwise).
            for (int k = armed > a.stages ? armed - a.stages : 0; k < armed; ++k)
                if (!mbar_wait(saddr(&bars[k % a.stages]), (k / a.stages) & 1) && lane == 0)
                    flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
        }
        // the last of b's history CTAs to stop taking units resets b's counters for the next launch
        if (dyn && lane == 0 && atomicAdd(a.sched + gridDim.y + b, 1) == a.hist_ctas - 1) {
            a.sched[b] = 0;
            a.sched[gridDim.y + b] = 0;
            __threadfence();
        }
        if (a.csize > 1) cluster_combine(a, reinterpret_cast<const float *>(stage0 + a.res_off), Hq, b, a.slot0 + s / a.csize);
        if (a.arrivals) arrive_count(a, b);
        return;
    }

    // ----------------------------------------------------------- consumers --
    // The copies above read only the pool, the page table and the lengths (and R_K below is as
    // fixed as they are); q, q_rot and the partials belong to the previous kernels in the stream.
    const int h = warp % Hkv, sub = warp / Hkv, nsub = kCW / Hkv;
    const int gid = lane >> 2, t = lane & 3;
    const int C = a.csize, rank = C > 1 ? (int)cluster_ctarank() : 0;
    float *qrot_s = reinterpret_cast<float *>(smem + a.rot_off);     // [Hq][kQS] rotated queries of the request
    if (!a.RK) {
        pdl_wait();
    } else {
        // q_rot = q . R_K for kv heads rank, rank + C, ... of this CTA, with R_K read straight from
        // global memory (it stays in L2), so that the stages fill with KV pages meanwhile.  Consumer
        // warp w sums rows [16 w, 16 w + 16) of R_K for columns 4 l .. 4 l + 3 (lane l) of every
        // query head of the kv head, as fp32 FMA chains in ascending row order; q_rot is the sum of
        // the eight partial sums in warp order, and it is written into every CTA of the cluster.
        float *part = reinterpret_cast<float *>(smem + 128);          // [kCW][G][128] partial sums
        float *qsl = part + warp * G * kHeadDim;   // this warp's rows of q ([G][16]), in its own partial area
        float4 r[16];
        auto load_r = [&](int hk) {
            const float4 *R4 = reinterpret_cast<const float4 *>(a.RK + ((size_t)hk * kHeadDim + 16 * warp) * kHeadDim) + lane;
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = __ldg(R4 + k * (kHeadDim / 4));
        };
        auto load_q = [&](int hk) {
            if (lane < 2 * G) {
                const int g = lane >> 1, hf = lane & 1;
                const uint4 v = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * Hq + hk * G + g) * kHeadDim + 16 * warp)[hf];
                float4 *d = reinterpret_cast<float4 *>(qsl + g * 16 + hf * 8);
                d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                   __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
                d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                                   __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
            }
            __syncwarp();
        };
        // R_K (read once from L2 by every cluster) and q, while the copy warp fills the stages
        if (rank < Hkv) load_r(rank);
        pdl_wait();                                                  // q may come from the previous kernel
        if (rank < Hkv) load_q(rank);
        __syncwarp();
        for (int hk = rank; hk < Hkv; hk += C) {
            if (hk != rank) {
                load_r(hk);
                load_q(hk);
            }
            float4 acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float qv = qsl[g * 16 + k];
                    acc[g].x = __fmaf_rn(qv, r[k].x, acc[g].x);
                    acc[g].y = __fmaf_rn(qv, r[k].y, acc[g].y);
                    acc[g].z = __fmaf_rn(qv, r[k].z, acc[g].z);
                    acc[g].w = __fmaf_rn(qv, r[k].w, acc[g].w);
                }
            }
            __syncwarp();                                            // (the sums overwrite this warp's q rows)
#pragma unroll
            for (int g = 0; g < G; ++g) *reinterpret_cast<float4 *>(part + (warp * G + g) * kHeadDim + 4 * lane) = acc[g];
            consumer_sync();
            // q_rot columns j .. j + 3 of query head g: the partial sums in warp order, pushed to every CTA
            for (int e = threadIdx.x; e < G * kHeadDim / 4; e += kCW * 32) {
                const int g = e / (kHeadDim / 4), j = (e % (kHeadDim / 4)) * 4;
                float4 v = *reinterpret_cast<const float4 *>(part + g * kHeadDim + j);
#pragma unroll
                for (int w2 = 1; w2 < kCW; ++w2) {
                    const float4 u = *reinterpret_cast<const float4 *>(part + (w2 * G + g) * kHeadDim + j);
                    v.x = __fadd_rn(v.x, u.x);
                    v.y = __fadd_rn(v.y, u.y);
                    v.z = __fadd_rn(v.z, u.z);
                    v.w = __fadd_rn(v.w, u.w);
                }
                *reinterpret_cast<float4 *>(qrot_s + (hk * G + g) * kQS + qs_col(j)) = v;
            }
            consumer_sync();                                         // the rows are complete, the sums consumed
            if (C > 1 && threadIdx.x < C && threadIdx.x != rank) {   // one bulk copy of the rows per peer
                fence_proxy_async_smem();
                const uint32_t rows = saddr(qrot_s + hk * G * kQS);
                dsmem_bulk_copy(rows, rows, (uint32_t)(G * kQS * 4), saddr(smem + 104), (uint32_t)threadIdx.x);
            }
        }
        if (C > 1 && !mbar_wait(saddr(smem + 104), 0) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
    }
    // with dynamic history units the per-step demotion is done here: K and V of kv head s by history
    // CTA s, or, with at least 2 Hkv history CTAs, K of head s by CTA s and V by CTA Hkv + s (half
    // the delay each)
    if (a.dem.dem_pos && a.sched && a.hist_ctas >= Hkv && threadIdx.x < kHeadDim) {
        const bool split = a.hist_ctas >= 2 * Hkv;
        if (s < (split ? 2 * Hkv : Hkv))
            history_demote(a, reinterpret_cast<float *>(smem + 128), T, he, b, s % Hkv,
                           split ? s / Hkv : 0, split ? s / Hkv + 1 : 2);
    }
    // rotated query element (hq, d): the previous kernel's q_rot, or this CTA's copy of the rows
    auto qrot = [&](int hq, int d) -> float {
        return a.RK ? qrot_s[hq * kQS + qs_col(d)] : a.q_rot[((size_t)b * Hq + hq) * kHeadDim + d];
    };

    // Power-of-two prescale of the warp's queries: the largest |q_rot| of the kv head's query
    // heads is brought into [2^14, 2^15), so that q_rot / factor (factors 1 .. 256) uses the f16
    // range of the split operand whatever the queries' magnitude; 2^e goes into the logit scale.
    float qsc = 1.f, cscq;
    {
        float qmax = 0.f;
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int c = 0; c < 4; ++c) qmax = fmaxf(qmax, fabsf(qrot(h * G + hh, 4 * lane + c)));
#pragma unroll
        for (int o = 16; o; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
        // qmax in [2^(eb-127), 2^(eb-126)): scale 2^(141-eb), undone by 2^(eb-141)
        const int eb = min(max((int)((__float_as_uint(qmax) >> 23) & 0xffu), 15), 254);
        float qinv = 1.f;
        if (qmax > 0.f && qmax < INFINITY) {
            qsc = __uint_as_float((uint32_t)(268 - eb) << 23);
            qinv = __uint_as_float((uint32_t)(eb - 14) << 23);
        }
        cscq = a.scale2 * kTwo24 * qinv;
    }
    // B operand of QK: q_rot * qsc split into f16 hi/lo, divided by the code factor of its k-row.
    uint32_t bq[NT][8][2];
    float qz[NT][NGRP];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hh = nt * 4 + (gid >> 1), part = gid & 1;
        const bool valid = hh < G;
        const int hq = h * G + (valid ? hh : 0);
        if constexpr (NGRP == 1) {
#pragma unroll
            for (int kap = 0; kap < 2; ++kap)
#pragma unroll
                for (int sg = 0; sg < 4; ++sg)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int rr = 2 * sg + e, W = 2 * t + kap;
                        const float inv = qsc / qk_factor(rr);
                        const float v0 = valid ? qrot(hq, 16 * W + rr) * inv : 0.f;
                        const float v1 = valid ? qrot(hq, 16 * W + 8 + rr) * inv : 0.f;
                        bq[nt][kap * 4 + sg][e] = pack2(split_part(v0, part), split_part(v1, part));
                    }
        } else {
            // group-pure MMAs: MMA m = 2 Gb + j covers 32-channel block Gb; this thread's k-rows are
            // channels 16 W + r (+ 8) of word W = 2 Gb + (t >> 1), registers r = qk_rsel(j, e, t & 1)
#pragma unroll
            for (int Gb = 0; Gb < 4; ++Gb)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int rr = qk_rsel(j, e, t & 1), W = 2 * Gb + (t >> 1);
                        const float inv = qsc / qk_factor(rr);
                        const float v0 = valid ? qrot(hq, 16 * W + rr) * inv : 0.f;
                        const float v1 = valid ? qrot(hq, 16 * W + 8 + rr) * inv : 0.f;
                        bq[nt][2 * Gb + j][e] = pack2(split_part(v0, part), split_part(v1, part));
                    }
        }
    }
    // per-group sums of q_rot for the zero-point term, for the head this thread owns (nt*4 + t)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jg = 0; jg < NGRP; ++jg) qz[nt][jg] = 0.f;
    for (int hh = 0; hh < G; ++hh) {
        const int hq = h * G + hh;
        const float sum4 = (qrot(hq, 4 * lane) + qrot(hq, 4 * lane + 1)) + (qrot(hq, 4 * lane + 2) + qrot(hq, 4 * lane + 3));
        const int lg = (4 * lane) * NGRP / kHeadDim;
#pragma unroll
        for (int jg = 0; jg < NGRP; ++jg) {
            float x = lg == jg ? sum4 : 0.f;
#pragma unroll
            for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                if (hh == nt * 4 + t) qz[nt][jg] = x * a.scale2;
        }
    }
    // Byte offsets of this thread's code words inside a tile (rows gid / gid+8 for K; rows t,
    // t+8, t+4, t+12 for V), and the tile base of head h.  TMA tiles are [16 rows][2 halves][128 B]
    // with 16-byte chunk c of row r, half f stored at chunk c ^ ((2 r + f) & 7); cp.async tiles are
    // [head][row][32 B].  Rows 8 or 4 apart share the swizzle: kofs1 and the V rows are kofs0 and
    // vofs0 plus constants (kVrow rows of kRowB bytes).
    constexpr int kRowB = TMA ? 256 : 32;
    constexpr int kVrow[4] = {0, 8, 4, 12};
    int kofs0, kofs1, vofs0;
    if constexpr (TMA) {
        const int hh = h & 3, hf = h >> 2, ck = 2 * hh + (t >> 1), cv = 2 * hh + (gid >> 2);
        kofs0 = gid * 256 + hf * 128 + ((ck ^ ((2 * gid + hf) & 7)) << 4) + (t & 1) * 8;
        vofs0 = t * 256 + hf * 128 + ((cv ^ ((2 * t + hf) & 7)) << 4) + (gid & 3) * 4;
    } else {
        kofs0 = gid * 32 + 8 * t;
        vofs0 = t * 32 + 4 * gid;
    }
    kofs1 = kofs0 + 8 * kRowB;
    // group-pure mapping (NGRP > 1): word 2 Gb + (t >> 1) of K rows gid, gid + 8 and word
    // 2 Gb + (gid >> 2) of V rows t, t + 8, t + 4, t + 12, for 32-channel blocks Gb = 0..3
    int kofg[4], vofg[4][4];
    if constexpr (NGRP > 1) {
        const int vrow[4] = {t, t + 8, t + 4, t + 12};
#pragma unroll
        for (int Gb = 0; Gb < 4; ++Gb) {
            const int wk = 2 * Gb + (t >> 1), wv = 2 * Gb + (gid >> 2);
            if constexpr (TMA) {
                const int hh = h & 3, hf = h >> 2;
                kofg[Gb] = gid * 256 + hf * 128 + (((2 * hh + (wk >> 2)) ^ ((2 * gid + hf) & 7)) << 4) + (wk & 3) * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    vofg[Gb][i] = vrow[i] * 256 + hf * 128 + (((2 * hh + (wv >> 2)) ^ ((2 * vrow[i] + hf) & 7)) << 4) +
                                  (wv & 3) * 4;
            } else {
                kofg[Gb] = gid * 32 + 4 * wk;
#pragma unroll
                for (int i = 0; i < 4; ++i) vofg[Gb][i] = vrow[i] * 32 + 4 * wv;
            }
        }
    }
    auto tile_base = [&](const uint8_t *arr, int j) -> const uint8_t * {
        return TMA ? arr + j * 4096 : arr + h * (kStageTok * 32) + j * (kTileTokens * 32);
    };
    const float csc = cscq;                     // logit scale of the MMA dot products
    const int rs = Hkv * NGRP;                  // scale/zero elements per token row in a stage
    const int arr_el = arr_bytes / 2;
    uint32_t *Ws = reinterpret_cast<uint32_t *>(smem + 128 + warp * a.ws_bytes);   // [NGRP][NCOL][kWsWords]

    float m_run[NT], m_true[NT], l_run[NT], zs[NT][NGRP];
    float oacc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt] = kNoMax;
        m_true[nt] = -INFINITY;
        l_run[nt] = 0.f;
#pragma unroll
        for (int jg = 0; jg < NGRP; ++jg) zs[nt][jg] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) oacc[nt][mt][c] = 0.f;
    }

    // Value-scale normalisation (both loops): vlim is a power of two above every value scale seen so
    // far (raised with a stage's maximum; the accumulators rescale by the ratio) and vmul = 128 / vlim,
    // so that w = p * scale_v * vmul < 2^8 * 2^7 stays inside the f16 range of the split PV operand
    // whatever the scales' magnitude; vlim / 128 goes into the output.
    float vlim = 0.f, vmul = 0.f;
    // raise the bound to cover vm (warp-uniform); returns the factor for the accumulators
    auto raise_vlim = [&](float vm) -> float {
        if (!(vm > vlim)) return 1.f;
        // vm in [2^(eb-127), 2^(eb-126)): vlim = 2^(eb-126), vmul = 2^7 / vlim
        const int eb = min(max((int)((__float_as_uint(vm) >> 23) & 0xffu), 7), 252);
        const float nl = __uint_as_float((uint32_t)(eb + 1) << 23);
        const float r = __fdiv_rn(vlim, nl);
        vlim = nl;
        vmul = __uint_as_float((uint32_t)(260 - eb) << 23);
        return r;
    };
    float vout = 1.f;                            // output factor of the value-scale normalisation
    if constexpr (TMA && NGRP == 1) {
        // ---- 8 kv heads, one group per head: a warp takes its kv head's four tiles of a stage in
        // one pass (64 tokens: one running-maximum update and one rescale vote per stage).
        //  1. lane l converts the stage's scale/zero of tokens l and l + 32 to fp32 once:
        //     Sw[tok] = (scale_k * cscq, zero_k, scale_v * vmul, zero_v), zero for tokens outside
        //     the range (vmul from the value-scale bound, raised with the stage's maximum).
        //  2. QK MMAs of the four tiles, interleaved (four independent accumulator chains).
        //  3. logits, stage maximum, lazy rescale, P * scale_v -> per-warp P buffer (hi, lo).
        //  4. PV MMAs of the four tiles.
        constexpr int kWs4 = kTilesPerStage * 8 + 4;        // words per P-buffer column (bank spread)
        uint32_t *Wp = reinterpret_cast<uint32_t *>(smem + 128 + warp * a.ws_bytes);   // [NCOL][kWs4]
        float4 *Sw = reinterpret_cast<float4 *>(Wp + NCOL * kWs4);                    // [64] per token
        int st = 0, ph = 0;
        for (;; st = (st + 1 == a.stages) ? 0 : st + 1, ph ^= (st == 0)) {
            if (!mbar_wait(saddr(&bars[st]), ph)) {
                if (lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                break;
            }
            const int t0 = stage_tile[st];
            if (t0 < 0) break;                        // the copy warp has no more tiles
            const uint8_t *sb = stage0 + st * stage_bytes;
            const int mask = masks[st];
            const int lim = tok_hi - t0 * kTileTokens;   // stage tokens [0, lim) lie inside the range
            const bool whole = mask == (1 << kTilesPerStage) - 1 && lim >= kStageTok;

            // 1. per-token fp32 scale/zero of kv head h
            float vres;
            {
                const uint16_t *s16 = reinterpret_cast<const uint16_t *>(sb + off_s) + h;
                constexpr int kRows = (kStageTok + 31) / 32;   // tokens per lane
                float4 e[kRows];
                float vm = 0.f;
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const int tok = lane + 32 * r;
                    const bool ok = ((mask >> (tok >> 4)) & 1) && tok < lim;
                    const int o = tok * 8;
                    e[r] = ok ? make_float4(bf16_to_f32(s16[o]), bf16_to_f32(s16[arr_el + o]),
                                            bf16_to_f32(s16[2 * arr_el + o]), bf16_to_f32(s16[3 * arr_el + o]))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                    vm = fmaxf(vm, e[r].z);
                }
                // (value scales are >= 0, +0 for tokens outside the range: their bit patterns order as
                // the values do, so one integer reduction gives the warp's maximum)
                vm = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(vm)));
                vres = raise_vlim(vm);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    e[r].x *= cscq;
                    e[r].z *= vmul;
                    Sw[lane + 32 * r] = e[r];
                }
                __syncwarp();
            }

            // 2. S = K_codes . q_rot for the four tiles (rows tokens gid, gid + 8; columns 4 heads x hi/lo)
            float sacc[kTilesPerStage][NT][4];
#pragma unroll
            for (int u = 0; u < kTilesPerStage; ++u)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sacc[u][nt][c] = 0.f;
            {
                uint2 kw0[kTilesPerStage], kw1[kTilesPerStage];
#pragma unroll
                for (int u = 0; u < kTilesPerStage; ++u) {
                    const uint8_t *Kc = sb + u * 4096;
                    kw0[u] = *reinterpret_cast<const uint2 *>(Kc + kofs0);
                    kw1[u] = *reinterpret_cast<const uint2 *>(Kc + kofs1);
                }
#pragma unroll
                for (int kap = 0; kap < 2; ++kap) {
                    uint32_t w0[kTilesPerStage], w1[kTilesPerStage], w0b[kTilesPerStage], w1b[kTilesPerStage];
#pragma unroll
                    for (int u = 0; u < kTilesPerStage; ++u) {
                        w0[u] = kap ? kw0[u].y : kw0[u].x;
                        w1[u] = kap ? kw1[u].y : kw1[u].x;
                        w0b[u] = __byte_perm(w0[u], 0, 0x3321);
                        w1b[u] = __byte_perm(w1[u], 0, 0x3321);
                    }
#pragma unroll
                    for (int sg = 0; sg < 4; ++sg)
#pragma unroll
                        for (int u = 0; u < kTilesPerStage; ++u) {
                            const uint32_t a0 = qk_reg(w0[u], w0b[u], 2 * sg), a1 = qk_reg(w1[u], w1b[u], 2 * sg);
                            const uint32_t a2 = qk_reg(w0[u], w0b[u], 2 * sg + 1), a3 = qk_reg(w1[u], w1b[u], 2 * sg + 1);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816_nv(sacc[u][nt], a0, a1, a2, a3, bq[nt][kap * 4 + sg][0], bq[nt][kap * 4 + sg][1]);
                        }
                }
            }

            // 3. logits (base 2) of tokens 16 u + gid (+ 8) for head nt * 4 + t; online softmax
            float alpha[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float tv[kTilesPerStage][2];
#pragma unroll
                for (int u = 0; u < kTilesPerStage; ++u)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float2 sz = *reinterpret_cast<const float2 *>(Sw + 16 * u + gid + 8 * e);
                        tv[u][e] = fmaf(sz.x, sacc[u][nt][2 * e] + sacc[u][nt][2 * e + 1], sz.y * qz[nt][0]);
                    }
                if (!whole) {                             // (uniform) tokens outside the range
#pragma unroll
                    for (int u = 0; u < kTilesPerStage; ++u)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            if (!((mask >> u) & 1) || 16 * u + gid + 8 * e >= lim) tv[u][e] = -INFINITY;
                }
                float mx = tv[0][0];
#pragma unroll
                for (int u = 0; u < kTilesPerStage; ++u)
#pragma unroll
                    for (int e = 0; e < 2; ++e) mx = fmaxf(mx, tv[u][e]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                m_true[nt] = fmaxf(m_true[nt], mx);
                float mn = m_run[nt], al = 1.f;
                if (mx > mn + kLazy) {                    // also the first finite maximum (mn = kNoMax)
                    al = ex2_approx(mn - mx);
                    mn = mx;
                }
                m_run[nt] = mn;
                alpha[nt] = al;
                float ls = 0.f, zadd = 0.f;
                const int c_hi = nt * 8 + 2 * t;
#pragma unroll
                for (int u = 0; u < kTilesPerStage; ++u) {
                    float w[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = ex2_approx(tv[u][e] - mn);
                        const float2 vz = *reinterpret_cast<const float2 *>(reinterpret_cast<const float *>(Sw + 16 * u + gid + 8 * e) + 2);
                        ls += pv;
                        w[e] = pv * vz.x;
                        zadd = fmaf(pv, vz.y, zadd);
                    }
                    // tokens gid, gid + 8 of tile u are PV k-columns 2 gid, 2 gid + 1: one word
                    uint32_t hi, lo;
                    split2(w[0], w[1], hi, lo);
                    Wp[c_hi * kWs4 + u * 8 + gid] = hi;
                    Wp[(c_hi + 1) * kWs4 + u * 8 + gid] = lo;
                }
                l_run[nt] = fmaf(l_run[nt], al, ls);
                zs[nt][0] = fmaf(zs[nt][0], al, zadd);
            }
            bool any = vres != 1.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) any |= alpha[nt] != 1.f;
            if (__any_sync(0xffffffffu, any)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float f = alpha[nt] * vres;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) oacc[nt][mt][c] *= f;
                }
            }
            __syncwarp();

            // 4. O += V_codes^T . (P * scale_v); m-tile mt row gid / gid + 8 = channel 16 gid + 2 mt / + 1
#pragma unroll
            for (int u = 0; u < kTilesPerStage; ++u) {
                const uint8_t *Vc = sb + off_v + u * 4096;
                uint32_t bw[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t *col = Wp + (nt * 8 + gid) * kWs4 + u * 8;
                    bw[nt][0] = col[t];
                    bw[nt][1] = col[t + 4];
                }
                // k-columns 2t, 2t+1 <- tokens t, t+8; 2t+8, 2t+9 <- tokens t+4, t+12
                const uint32_t X = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[0] * kRowB);
                const uint32_t Y = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[1] * kRowB);
                const uint32_t X2 = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[2] * kRowB);
                const uint32_t Y2 = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[3] * kRowB);
                const uint32_t P1 = __byte_perm(X, Y, 0x5410), P2 = __byte_perm(X, Y, 0x6521);
                const uint32_t P3 = __byte_perm(X, Y, 0x7632), P4 = __byte_perm(X, Y, 0x7733);
                const uint32_t Q1 = __byte_perm(X2, Y2, 0x5410), Q2 = __byte_perm(X2, Y2, 0x6521);
                const uint32_t Q3 = __byte_perm(X2, Y2, 0x7632), Q4 = __byte_perm(X2, Y2, 0x7733);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const uint32_t a0 = pv_reg(P1, P2, P3, P4, 2 * mt), a1 = pv_reg(P1, P2, P3, P4, 2 * mt + 1);
                    const uint32_t a2 = pv_reg(Q1, Q2, Q3, Q4, 2 * mt), a3 = pv_reg(Q1, Q2, Q3, Q4, 2 * mt + 1);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816_nv(oacc[nt][mt], a0, a1, a2, a3, bw[nt][0], bw[nt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(saddr(&bars[4 + st]));
        }
    } else {
    int st = 0, ph = 0;                          // stage and its phase parity, stepped (no division)
    for (;; st = (st + 1 == a.stages) ? 0 : st + 1, ph ^= (st == 0)) {
        if (!mbar_wait(saddr(&bars[st]), ph)) {
            if (lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
            break;
        }
        const int t0 = stage_tile[st];
        if (t0 < 0) break;                        // the copy warp has no more tiles
        const uint8_t *sb = stage0 + st * stage_bytes;
        const int mask = masks[st];
        {
            // value-scale bound over this warp's tiles of the stage (valid tokens only; lane l reads
            // token l % 16 of a tile, groups l / 16, l / 16 + 2, ...)
            float vm = 0.f;
            for (int j = sub; j < kTilesPerStage; j += nsub) {
                const int tok = lane & 15;
                if (((mask >> j) & 1) && tok < tok_hi - (t0 + j) * kTileTokens) {
                    const uint16_t *svp = reinterpret_cast<const uint16_t *>(sb + off_s) + 2 * arr_el +
                                          (j * kTileTokens + tok) * rs + h * NGRP;
                    for (int jg = lane >> 4; jg < NGRP; jg += 2) vm = fmaxf(vm, bf16_to_f32(svp[jg]));
                }
            }
            vm = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(vm)));
            const float vres = raise_vlim(vm);
            if (vres != 1.f) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) oacc[nt][mt][c] *= vres;
            }
        }
        // this warp's tiles of the stage: sub, sub + nsub, ...; taken two at a time (32 tokens)
        for (int ja = sub; ja < kTilesPerStage; ja += 2 * nsub) {
            const int jb_raw = ja + nsub;
            const bool ua = (mask >> ja) & 1;
            const bool ub = jb_raw < kTilesPerStage && ((mask >> jb_raw) & 1);
            if (!ua && !ub) continue;
            const int jt[2] = {ja, jb_raw < kTilesPerStage ? jb_raw : ja};
            const bool uok[2] = {ua, ub};

            // ---- NGRP > 1: group-pure MMAs, each group's dot products folded into the logits at once:
            // tq[u][nt][e] = sum over groups (ascending) of scale*csc*dot + zero*qz (tokens gid, gid+8)
            float tq[2][NT][2];
            if constexpr (NGRP > 1) {
                constexpr int kBpg = 4 / NGRP;             // 32-channel blocks per group
                const bool odd = t & 1;
                const uint32_t mA0 = odd ? kM2 : kM0, mB0 = odd ? kM3 : kM1, mA1 = odd ? kM2 : kM4;
                const uint32_t mB1 = odd ? kM3 : kM1;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint8_t *Kc = tile_base(sb, jt[u]);
                    const uint16_t *sk = reinterpret_cast<const uint16_t *>(sb + off_s) + jt[u] * kTileTokens * rs + h * NGRP;
                    float sg[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) tq[u][nt][0] = tq[u][nt][1] = 0.f;
#pragma unroll
                    for (int Gb = 0; Gb < 4; ++Gb) {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(Kc + kofg[Gb]);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(Kc + kofg[Gb] + (TMA ? 8 * 256 : 8 * 32));
                        const uint32_t w0b = __byte_perm(w0, 0, 0x3321), w1b = __byte_perm(w1, 0, 0x3321);
                        const uint32_t w0s = odd ? w0b : w0, w1s = odd ? w1b : w1;
                        if (Gb % kBpg == 0) {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int c = 0; c < 4; ++c) sg[nt][c] = 0.f;
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t a0 = j ? (w0s & mA1) : (w0 & mA0), a1 = j ? (w1s & mA1) : (w1 & mA0);
                            const uint32_t a2 = j ? (w0b & mB1) : (w0 & mB0), a3 = j ? (w1b & mB1) : (w1 & mB0);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816(sg[nt], a0, a1, a2, a3, bq[nt][2 * Gb + j][0], bq[nt][2 * Gb + j][1]);
                        }
                        if (Gb % kBpg == kBpg - 1) {
                            const int jg = Gb / kBpg;
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int tok = gid + 8 * e;
                                const float sc = bf16_to_f32(sk[tok * rs + jg]), zc = bf16_to_f32(sk[arr_el + tok * rs + jg]);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    tq[u][nt][e] += fmaf(sc * csc, sg[nt][2 * e] + sg[nt][2 * e + 1], zc * qz[nt][jg]);
                            }
                        }
                    }
                }
            }

            // ---- S = K_codes . q_rot for both tiles (rows = tokens gid, gid+8; cols = 4 heads x hi/lo)
            float sacc[2][NT][4];                        // (NGRP == 1)
            if constexpr (NGRP == 1) {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sacc[u][nt][c] = 0.f;
                uint2 kw0[2], kw1[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint8_t *Kc = tile_base(sb, jt[u]);
                    kw0[u] = *reinterpret_cast<const uint2 *>(Kc + kofs0);
                    kw1[u] = *reinterpret_cast<const uint2 *>(Kc + kofs1);
                }
#pragma unroll
                for (int kap = 0; kap < 2; ++kap) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t w0 = kap ? kw0[u].y : kw0[u].x, w1 = kap ? kw1[u].y : kw1[u].x;
                        const uint32_t w0b = __byte_perm(w0, 0, 0x3321), w1b = __byte_perm(w1, 0, 0x3321);
#pragma unroll
                        for (int sg = 0; sg < 4; ++sg) {
                            const uint32_t a0 = qk_reg(w0, w0b, 2 * sg), a1 = qk_reg(w1, w1b, 2 * sg);
                            const uint32_t a2 = qk_reg(w0, w0b, 2 * sg + 1), a3 = qk_reg(w1, w1b, 2 * sg + 1);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816(sacc[u][nt], a0, a1, a2, a3, bq[nt][kap * 4 + sg][0], bq[nt][kap * 4 + sg][1]);
                        }
                    }
                }
            }

            // ---- logits of 4 tokens per thread, online softmax over the 32 tokens, P*scale -> Ws.
            // Tiles start inside the range (its start is a tile boundary), so a token is valid when
            // its tile holds data and it lies below the range's end.  The running maximum is raised only when the
            // pass's maximum exceeds it by more than kLazy (so P <= 2^kLazy and most passes skip the
            // rescale); the true maximum is tracked alongside and restored at the end.
            float alpha[NT];
            int lim[2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
                lim[u] = uok[u] ? tok_hi - (t0 + jt[u]) * kTileTokens : 0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float tv[2][2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint16_t *sk = reinterpret_cast<const uint16_t *>(sb + off_s) +
                                         jt[u] * kTileTokens * rs + h * NGRP;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = gid + 8 * e;
                        float tt = 0.f;
                        if constexpr (NGRP == 1) {
                            const float sc = bf16_to_f32(sk[tok * rs]), zc = bf16_to_f32(sk[arr_el + tok * rs]);
                            tt += fmaf(sc * csc, sacc[u][nt][2 * e] + sacc[u][nt][2 * e + 1], zc * qz[nt][0]);
                        } else {
                            tt = tq[u][nt][e];
                        }
                        tv[u][e] = tok < lim[u] ? tt : -INFINITY;
                    }
                }
                float mx = fmaxf(fmaxf(tv[0][0], tv[0][1]), fmaxf(tv[1][0], tv[1][1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                m_true[nt] = fmaxf(m_true[nt], mx);
                float mn = m_run[nt], al = 1.f;
                if (mx > mn + kLazy) {                 // also the first finite maximum (mn = kNoMax)
                    al = ex2_approx(mn - mx);
                    mn = mx;
                }
                float pv[2][2];
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int e = 0; e < 2; ++e) pv[u][e] = ex2_approx(tv[u][e] - mn);
                alpha[nt] = al;
                m_run[nt] = mn;
                l_run[nt] = fmaf(l_run[nt], al, (pv[0][0] + pv[0][1]) + (pv[1][0] + pv[1][1]));
#pragma unroll
                for (int jg = 0; jg < NGRP; ++jg) {
                    float zadd = 0.f;
                    uint32_t *Wg = Ws + jg * NCOL * kWsWords;
                    const int c_hi = nt * 8 + 2 * t;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint16_t *sk = reinterpret_cast<const uint16_t *>(sb + off_s) +
                                             jt[u] * kTileTokens * rs + h * NGRP;
                        float w[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = gid + 8 * e;
                            const float svv = bf16_to_f32(sk[2 * arr_el + tok * rs + jg]);
                            const float zvv = bf16_to_f32(sk[3 * arr_el + tok * rs + jg]);
                            // rows past the valid range hold arbitrary bits (NaN included): select, never multiply
                            const bool ok = tok < lim[u];
                            w[e] = ok ? pv[u][e] * (svv * vmul) : 0.f;
                            zadd = ok ? fmaf(pv[u][e], zvv, zadd) : zadd;
                        }
                        // tokens gid, gid + 8 are PV k-columns 2 gid, 2 gid + 1 of tile u: one word
                        uint32_t hi, lo;
                        split2(w[0], w[1], hi, lo);
                        Wg[c_hi * kWsWords + u * 8 + gid] = hi;
                        Wg[(c_hi + 1) * kWsWords + u * 8 + gid] = lo;
                    }
                    zs[nt][jg] = fmaf(zs[nt][jg], al, zadd);
                }
            }
            bool any = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) any |= alpha[nt] != 1.f;
            if (__any_sync(0xffffffffu, any)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) oacc[nt][mt][c] *= alpha[nt];
            }
            __syncwarp();

            // ---- O += V_codes^T . (P*scale)  (k = tokens, cols = heads x hi/lo).  Rows: with one group,
            // m-tile mt row gid / gid + 8 = channel 16 gid + 2 mt / + 1; with NGRP > 1 (group-pure
            // m-tiles, one group's P*scale each), m-tile 2 Gb + j row gid / gid + 8 = channel
            // 32 Gb + 4 gid + 2 j / + 1 (byte 8 Gb + gid of the row)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint8_t *Vc = tile_base(sb + off_v, jt[u]);
                uint32_t bw[NGRP][NT][2];
#pragma unroll
                for (int jg = 0; jg < NGRP; ++jg)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint32_t *col = Ws + jg * NCOL * kWsWords + (nt * 8 + gid) * kWsWords + u * 8;
                        bw[jg][nt][0] = col[t];
                        bw[jg][nt][1] = col[t + 4];
                    }
                if constexpr (NGRP == 1) {
                    // k-columns 2t, 2t+1 <- tokens t, t+8; 2t+8, 2t+9 <- tokens t+4, t+12
                    const uint32_t X = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[0] * kRowB);
                    const uint32_t Y = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[1] * kRowB);
                    const uint32_t X2 = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[2] * kRowB);
                    const uint32_t Y2 = *reinterpret_cast<const uint32_t *>(Vc + vofs0 + kVrow[3] * kRowB);
                    const uint32_t P1 = __byte_perm(X, Y, 0x5410), P2 = __byte_perm(X, Y, 0x6521);
                    const uint32_t P3 = __byte_perm(X, Y, 0x7632), P4 = __byte_perm(X, Y, 0x7733);
                    const uint32_t Q1 = __byte_perm(X2, Y2, 0x5410), Q2 = __byte_perm(X2, Y2, 0x6521);
                    const uint32_t Q3 = __byte_perm(X2, Y2, 0x7632), Q4 = __byte_perm(X2, Y2, 0x7733);
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const uint32_t a0 = pv_reg(P1, P2, P3, P4, 2 * mt), a1 = pv_reg(P1, P2, P3, P4, 2 * mt + 1);
                        const uint32_t a2 = pv_reg(Q1, Q2, Q3, Q4, 2 * mt), a3 = pv_reg(Q1, Q2, Q3, Q4, 2 * mt + 1);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma16816(oacc[nt][mt], a0, a1, a2, a3, bw[0][nt][0], bw[0][nt][1]);
                    }
                } else {
                    // byte gid & 3 of the word of token t (t + 4) low, of token t + 8 (t + 12) high
                    const uint32_t selv = (uint32_t)(gid & 3) | ((uint32_t)(4 + (gid & 3)) << 8);
#pragma unroll
                    for (int Gb = 0; Gb < 4; ++Gb) {
                        const uint32_t X = *reinterpret_cast<const uint32_t *>(Vc + vofg[Gb][0]);
                        const uint32_t Y = *reinterpret_cast<const uint32_t *>(Vc + vofg[Gb][1]);
                        const uint32_t X2 = *reinterpret_cast<const uint32_t *>(Vc + vofg[Gb][2]);
                        const uint32_t Y2 = *reinterpret_cast<const uint32_t *>(Vc + vofg[Gb][3]);
                        const uint32_t P = __byte_perm(X, Y, selv), Q = __byte_perm(X2, Y2, selv);
                        const int jg = Gb * NGRP / 4;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t mlo = j ? kM2 : kM0, mhi = j ? kM3 : kM1;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816(oacc[nt][2 * Gb + j], P & mlo, P & mhi, Q & mlo, Q & mhi, bw[jg][nt][0],
                                         bw[jg][nt][1]);
                        }
                    }
                }
            }
            __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(saddr(&bars[4 + st]));
    }
    }

    vout = vlim * (1.f / 128.f);
    // The next kernel in the stream may launch once every CTA's consumers are past their loop
    // (only they trigger: the copy warp finishes its loop stages ahead of them).
    pdl_trigger();
    // ---- finish: reduce the per-thread sums over the 8 lanes of a column, scale the outputs
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], o);
#pragma unroll
            for (int jg = 0; jg < NGRP; ++jg) zs[nt][jg] += __shfl_xor_sync(0xffffffffu, zs[nt][jg], o);
        }
    }
    // output element i of this thread: channel and code factor (see the PV mapping above)
    auto out_ch = [&](int i) { return NGRP == 1 ? 16 * gid + i : 32 * (i >> 2) + 4 * gid + (i & 3); };
    // back to the split's true maximum: l, the zero-point sum and the accumulators scale by 2^(m_run - m_true)
    float fix[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        fix[nt] = m_true[nt] == -INFINITY ? 1.f : ex2_approx(m_run[nt] - m_true[nt]);
        l_run[nt] *= fix[nt];
        m_run[nt] = m_true[nt];
    }
    float outv[NT][16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        if constexpr (NGRP == 1) {
            const float z = zs[nt][0];
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                outv[nt][2 * mt] = fmaf(oacc[nt][mt][0] + oacc[nt][mt][1], kTwo24 / pv_factor(2 * mt) * vout, z) * fix[nt];
                outv[nt][2 * mt + 1] =
                    fmaf(oacc[nt][mt][2] + oacc[nt][mt][3], kTwo24 / pv_factor(2 * mt + 1) * vout, z) * fix[nt];
            }
        } else {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const float z = zs[nt][(mt >> 1) * NGRP / 4];
                const float f0 = kTwo24 / (float)(1 << (2 * ((2 * mt) & 3))) * vout;
                const float f1 = kTwo24 / (float)(1 << (2 * ((2 * mt + 1) & 3))) * vout;
                outv[nt][2 * mt] = fmaf(oacc[nt][mt][0] + oacc[nt][mt][1], f0, z) * fix[nt];
                outv[nt][2 * mt + 1] = fmaf(oacc[nt][mt][2] + oacc[nt][mt][3], f1, z) * fix[nt];
            }
        }
    }

    const size_t S1 = (size_t)S + 1;
    // destination of this CTA's result: the partial slot (no cluster) or the shared result area
    float *res = reinterpret_cast<float *>(stage0 + a.res_off);   // [Hq] m, [Hq] l, [Hq][128] acc
    const bool to_res = a.csize > 1;
    if (nsub == 1) {
        if (to_res) consumer_sync();            // the result area overlaps the stages
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = nt * 4 + t;
            if (hh < G) {
                const int hq = h * G + hh;
                const size_t row = ((size_t)b * Hq + hq) * S1 + a.slot0 + s;
                float *dst = to_res ? res + res_acc(Hq) + hq * kHeadDim : a.out.acc + row * kHeadDim;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<float4 *>(dst + out_ch(4 * q4)) =
                        make_float4(outv[nt][4 * q4], outv[nt][4 * q4 + 1], outv[nt][4 * q4 + 2], outv[nt][4 * q4 + 3]);
                if (gid == 0) {
                    (to_res ? res + hq : a.out.m + row)[0] = m_run[nt];
                    (to_res ? res + Hq + hq : a.out.l + row)[0] = l_run[nt];
                }
            }
        }
        if (to_res) cluster_combine(a, res, Hq, b, a.slot0 + s / a.csize);
        if (a.arrivals) arrive_count(a, b);
        return;
    }

    // several warps share a kv head: combine them in a fixed order (sub 0, 1, ...)
    consumer_sync();                            // every consumer is done with the stages
    float *cm = reinterpret_cast<float *>(stage0);               // [warp][NT*4] m
    float *cl = cm + kCW * NT * 4;                               // [warp][NT*4] l
    float *ca = cl + kCW * NT * 4;                               // [warp][NT*4][128] acc
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        if (gid == 0) {
            cm[warp * NT * 4 + nt * 4 + t] = m_run[nt];
            cl[warp * NT * 4 + nt * 4 + t] = l_run[nt];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) ca[(warp * NT * 4 + nt * 4 + t) * kHeadDim + out_ch(i)] = outv[nt][i];
    }
    consumer_sync();
    if (sub == 0) {
        // this warp (kv head h) combines warps h, h + Hkv, h + 2 Hkv, ...; lane = (head slot, channel block)
        for (int e = lane; e < NT * 4 * kHeadDim / 4; e += 32) {
            const int slot = e / (kHeadDim / 4), c4 = (e % (kHeadDim / 4)) * 4;
            const int nt = slot / 4, hh = slot % 4 + nt * 4;
            if (hh >= G) continue;
            float M = -INFINITY;
            for (int w = h; w < kCW; w += Hkv) M = fmaxf(M, cm[w * NT * 4 + slot]);
            float L = 0.f, A0 = 0.f, A1 = 0.f, A2 = 0.f, A3 = 0.f;
            if (M != -INFINITY) {
                for (int w = h; w < kCW; w += Hkv) {
                    const float f = exp2f(cm[w * NT * 4 + slot] - M);
                    const float *src = ca + (w * NT * 4 + slot) * kHeadDim + c4;
                    L = fmaf(cl[w * NT * 4 + slot], f, L);
                    A0 = fmaf(src[0], f, A0);
                    A1 = fmaf(src[1], f, A1);
                    A2 = fmaf(src[2], f, A2);
                    A3 = fmaf(src[3], f, A3);
                }
            }
            const int hq = h * G + hh;
            const size_t row = ((size_t)b * Hq + hq) * S1 + a.slot0 + s;
            *reinterpret_cast<float4 *>(to_res ? res + res_acc(Hq) + hq * kHeadDim + c4 : a.out.acc + row * kHeadDim + c4) =
                make_float4(A0, A1, A2, A3);
            if (c4 == 0) {
                (to_res ? res + hq : a.out.m + row)[0] = M;
                (to_res ? res + Hq + hq : a.out.l + row)[0] = L;
            }
        }
    }
    if (to_res) cluster_combine(a, res, Hq, b, a.slot0 + s / a.csize);
    if (a.arrivals) arrive_count(a, b);
}

// Largest cluster size C in {8, 4, 2} whose co-resident clusters still occupy at least 90% of
// the CTA slots of the GPU (clusters must fit inside one GPC); 1 if none does.  *active gets
// the number of clusters (or CTAs when C = 1) that are resident at once.  Cached per kernel.
int int2_cluster_size(const void *kern, int smem, int threads, int *active = nullptr) {
    struct Entry { const void *k; int smem, dev, c, active; };
    static thread_local Entry cache[32];
    static thread_local int n_cache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    for (int i = 0; i < n_cache; ++i)
        if (cache[i].k == kern && cache[i].smem == smem && cache[i].dev == dev) {
            if (active) *active = cache[i].active;
            return cache[i].c;
        }
    int best = 1, best_active = 1;
    if (ensure_dyn_smem(kern, smem) == cudaSuccess) {
        int sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
        best_active = per_sm * sms > 0 ? per_sm * sms : 1;
        for (int c = 8; c >= 2 && best == 1; c /= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(c * 64);
            cfg.blockDim = dim3(threads);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int ncl = 0;
            if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) == cudaSuccess && 10 * ncl * c >= 9 * per_sm * sms) {
                best = c;
                best_active = ncl;
            }
        }
        cudaGetLastError();
    }
    if (n_cache < 32) cache[n_cache++] = {kern, smem, dev, best, best_active};
    if (active) *active = best_active;
    return best;
}

// Shared-memory carve-up of the kernel for a layout; returns the dynamic smem bytes.
template <int G, int NGRP>
int mma_smem_plan(const oscar_layout_t &L, MmaArgs &a) {
    constexpr int NT = (G == 8) ? 2 : 1;
    const int Hkv = L.n_kv_heads, Hq = Hkv * G;
    a.off_v = Hkv * kStageTok * 32;
    a.arr_bytes = kStageTok * Hkv * NGRP * 2;
    a.off_s = 2 * a.off_v;
    a.stage_bytes = (a.off_s + 4 * a.arr_bytes + 127) & ~127;
    // per consumer warp: the P operand buffer (and, on the 8-kv-head single-group path, the
    // stage's per-token fp32 scale/zero); the same area first holds the rotation's partial sums
    if (Hkv == 8 && NGRP == 1)
        a.ws_bytes = 8 * NT * (kTilesPerStage * 8 + 4) * 4 + kStageTok * 16;
    else
        a.ws_bytes = NGRP * 8 * NT * kWsWords * 4;
    const int pre = kCW * a.ws_bytes > kCW * G * kHeadDim * 4 ? kCW * a.ws_bytes : kCW * G * kHeadDim * 4;
    a.stage_off = (128 + pre + 1023) & ~1023;   // stages start 1024-byte aligned
    const int budget = (G == 8 ? 200 : 110) * 1024;    // two CTAs per SM below G = 8
    const int rot_bytes = Hq * kQS * 4;                 // rotated queries (fused rotation)
    int stages = kMaxStages;
    while (stages > 2 && a.stage_off + stages * a.stage_bytes + rot_bytes > budget) --stages;
    a.stages = stages;
    const int combine = (kCW / Hkv > 1) ? kCW * NT * 4 * (2 + kHeadDim) * 4 : 0;
    a.res_off = combine;
    const int res_bytes = res_floats(Hq) * 4;
    // window CTAs: their warp results, their CTA result and its receive area, from the first stage on
    const int win_tail = kCW * G * (2 + kHeadDim) * 4 + res_bytes + recv_bytes(Hq);
    int tail = a.res_off + res_bytes + recv_bytes(Hq);
    if (win_tail > tail) tail = win_tail;
    const int area = stages * a.stage_bytes;             // (the window CTAs' demotion stages R here)
    a.rk_chunk = area >= 65536 ? 65536 : area >= 32768 ? 32768 : 16384;
    a.rot_off = a.stage_off + (area > tail ? area : tail);
    // the window CTAs use everything from the first stage to the end (neither the stages nor the
    // rotated-query rows) for two row buffers; set_window() sizes them for the launch's batch
    a.wbuf_bytes = a.rot_off + rot_bytes - a.stage_off;
    // + 1024: the kernel rounds the dynamic shared memory base up to a 1024-byte boundary
    return 1024 + a.rot_off + rot_bytes;
}

template <int G, int NGRP>
int mma_cluster_size(const oscar_layout_t &L, int *active) {
    MmaArgs a{};
    const int smem = mma_smem_plan<G, NGRP>(L, a);
    const void *kern = L.n_kv_heads == 8 ? reinterpret_cast<const void *>(int2_mma_kernel<G, NGRP, true>)
                                         : reinterpret_cast<const void *>(int2_mma_kernel<G, NGRP, false>);
    return int2_cluster_size(kern, smem, kThreads, active);
}

// An INT2 codes array of 8 kv heads, [rows = n_pages * page_size][256 bytes], as a 3-D uint8 tensor
// map [rows][2 halves][128 bytes] whose box is box_rows rows (both halves) with 128-byte swizzle:
// in shared memory row r's half f (4 heads) sits at r * 256 + f * 128, its 16-byte chunk c at
// chunk c ^ ((2 r + f) & 7).
bool codes_tensor_map(CUtensorMap *tm, const uint8_t *base, long long rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    const cuuint64_t dims[3] = {128, 2, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {128, 256};
    const cuuint32_t box[3] = {128, 2, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Window clusters per request and the window CTAs' row buffers (tokens of this cluster's kv heads
// per buffer, at most 32).
void set_window(const oscar_layout_t &L, int batch, MmaArgs &a) {
    a.win_heads = L.n_kv_heads / int2_mma_window_clusters(L, batch);
    a.wbuf_tok = a.wbuf_bytes / (2 * 2 * a.win_heads * kHeadDim * 2);
    if (a.wbuf_tok > 32) a.wbuf_tok = 32;
}

template <int G, int NGRP>
cudaError_t launch_mma(const oscar_layout_t &L, MmaArgs a, int batch, bool history, bool window, cudaStream_t st,
                       int *clusters) {
    const int smem = mma_smem_plan<G, NGRP>(L, a);
    set_window(L, batch, a);
    // the carve-up's invariants: vector and bulk-copy targets 16-byte aligned, tensor-map boxes
    // 1024-byte aligned, R_K chunks inside the stage area
    if (((a.stage_off | a.stage_bytes | a.off_v | a.off_s | a.arr_bytes | a.res_off | a.rot_off) & 15) ||
        (a.stage_off & 1023) || (a.stage_bytes & 1023 && L.n_kv_heads == 8) ||
        (a.RK && a.stages * a.stage_bytes < a.rk_chunk))
        return cudaErrorInvalidValue;
    const bool tma = L.n_kv_heads == 8;
    // the tensor-map kernel folds these for 8 kv heads
    if (tma && (a.off_v != kTilesPerStage * 4096 || a.off_s != 2 * kTilesPerStage * 4096 ||
                a.arr_bytes != kStageTok * 8 * NGRP * 2 ||
                a.stage_bytes != ((2 * kTilesPerStage * 4096 + 4 * kStageTok * 8 * NGRP * 2 + 127) & ~127)))
        return cudaErrorInvalidValue;
    auto kern = tma ? int2_mma_kernel<G, NGRP, true> : int2_mma_kernel<G, NGRP, false>;
    // codes: boxes of a whole unit (64 rows) and of one tile (16 rows)
    CUtensorMap tmk, tmv, tmk1, tmv1;
    memset(&tmk, 0, sizeof(tmk));
    memset(&tmv, 0, sizeof(tmv));
    memset(&tmk1, 0, sizeof(tmk1));
    memset(&tmv1, 0, sizeof(tmv1));
    if (tma && history) {
        const long long rows = (long long)a.pool.n_pages * L.page_size;
        if (!codes_tensor_map(&tmk, a.pool.codes_k, rows, kStageTok) ||
            !codes_tensor_map(&tmv, a.pool.codes_v, rows, kStageTok) ||
            !codes_tensor_map(&tmk1, a.pool.codes_k, rows, kTileTokens) ||
            !codes_tensor_map(&tmv1, a.pool.codes_v, rows, kTileTokens))
            return cudaErrorInvalidValue;
    }
    a.csize = int2_cluster_size(reinterpret_cast<const void *>(kern), smem, kThreads);
    if (cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(kern), smem)) return e;
    a.hist_ctas = history ? (a.out.S - a.slot0) * a.csize : 0;
    a.pf_units = 0;      // (measured slower at one, a half and two rounds of units ahead: kept off)
    a.win_ctas = window ? (L.n_kv_heads / a.win_heads) * a.csize : 0;
    if (clusters) *clusters = (a.hist_ctas + a.win_ctas) / a.csize;   // arrivals per request
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.win_ctas + a.hist_ctas, batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    add_overlap_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, kern, a, tmk, tmv, tmk1, tmv1);
}

}  // namespace

int int2_mma_cluster_size(const oscar_layout_t &L, int *active) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
        cudaGetLastError();
        if (active) *active = 0;
        return 8;
    }
    const int ngrp = kHeadDim / L.group;
#define OSCAR_CL_CASE(GG, NN) \
    if (L.gqa == GG && ngrp == NN) return mma_cluster_size<GG, NN>(L, active);
    OSCAR_CL_CASE(1, 1) OSCAR_CL_CASE(2, 1) OSCAR_CL_CASE(4, 1) OSCAR_CL_CASE(8, 1)
    OSCAR_CL_CASE(1, 2) OSCAR_CL_CASE(2, 2) OSCAR_CL_CASE(4, 2) OSCAR_CL_CASE(8, 2)
    OSCAR_CL_CASE(1, 4) OSCAR_CL_CASE(2, 4) OSCAR_CL_CASE(4, 4) OSCAR_CL_CASE(8, 4)
#undef OSCAR_CL_CASE
    return 1;
}

int int2_mma_window_clusters(const oscar_layout_t &L, int batch) { return L.n_kv_heads == 8 && batch == 1 ? 2 : 1; }

bool int2_mma_supported(const oscar_layout_t &L) {
    const int H = L.n_kv_heads;
    // (the code-as-f16-subnormal operands hold the uniform levels only)
    return (H == 1 || H == 2 || H == 4 || H == 8) && L.head_dim == kHeadDim && uniform_codebook(L);
}

static cudaError_t decode_mma_impl(const oscar_layout_t &L, const float *RK, Int2PoolView pool, const int32_t *pt,
                                   const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt, int max_pages,
                                   const int32_t *seq_len, const int32_t *hist_end, int batch, float sm_scale,
                                   PartialsView out, int32_t *status, const FusedDemotion &dem, cudaStream_t st,
                                   const float *q_rot, bool history, bool window, int32_t *arrivals,
                                   int *clusters, int32_t *sched, int hist_lo = 0, int slot0 = 0);

cudaError_t launch_decode_mma(const oscar_layout_t &L, const float *q_rot, const float *RK, Int2PoolView pool,
                              const int32_t *pt, const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt,
                              int max_pages, const int32_t *seq_len, const int32_t *hist_end, int batch,
                              float sm_scale, PartialsView out, int32_t *status, bool history, bool window,
                              cudaStream_t st) {
    FusedDemotion none{};
    return decode_mma_impl(L, RK, pool, pt, q, bpool, bpt, max_pages, seq_len, hist_end, batch, sm_scale, out, status,
                           none, st, q_rot, history, window, nullptr, nullptr, nullptr);
}

cudaError_t launch_decode_mma_suffix(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool, const int32_t *pt,
                                     const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt, int max_pages,
                                     const int32_t *seq_len, const int32_t *hist_end, int batch, float sm_scale,
                                     PartialsView out, int32_t *status, int hist_lo, int slot0, int32_t *sched,
                                     cudaStream_t st) {
    FusedDemotion none{};
    return decode_mma_impl(L, nullptr, pool, pt, q, bpool, bpt, max_pages, seq_len, hist_end, batch, sm_scale, out,
                           status, none, st, q_rot, true, true, nullptr, nullptr, sched, hist_lo, slot0);
}

cudaError_t launch_decode_mma_demote(const oscar_layout_t &L, const float *RK, Int2PoolView pool, const int32_t *pt,
                                     const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt, int max_pages,
                                     const int32_t *seq_len, const int32_t *hist_end, int batch, float sm_scale,
                                     PartialsView out, int32_t *status, const FusedDemotion &dem,
                                     int32_t *arrivals, int *clusters, int32_t *sched, cudaStream_t st) {
    return decode_mma_impl(L, RK, pool, pt, q, bpool, bpt, max_pages, seq_len, hist_end, batch, sm_scale, out, status,
                           dem, st, nullptr, true, true, arrivals, clusters, sched);
}

static cudaError_t decode_mma_impl(const oscar_layout_t &L, const float *RK, Int2PoolView pool, const int32_t *pt,
                                   const uint16_t *q, Bf16PoolView bpool, const int32_t *bpt, int max_pages,
                                   const int32_t *seq_len, const int32_t *hist_end, int batch, float sm_scale,
                                   PartialsView out, int32_t *status, const FusedDemotion &dem, cudaStream_t st,
                                   const float *q_rot, bool history, bool window, int32_t *arrivals,
                                   int *clusters, int32_t *sched, int hist_lo, int slot0) {
    if (clusters) *clusters = 0;
    if (batch <= 0 || (!history && !window)) return cudaSuccess;
    if (slot0 < 0 || slot0 >= out.S) return cudaErrorInvalidValue;
    MmaArgs a{};
    a.hist_lo = hist_lo;
    a.slot0 = slot0;
    if (history && window) a.arrivals = arrivals;
    if (history) a.sched = sched;
    a.RK = RK;
    a.dem = dem;
    a.group = L.group;
    a.q = q;
    a.bpool = bpool;
    a.bpt = bpt;
    a.q_rot = q_rot;
    a.pool = pool;
    a.pt = pt;
    a.max_pages = max_pages;
    a.page_size = L.page_size;
    a.n_kv = L.n_kv_heads;
    a.sink = L.sink;
    a.seq_len = seq_len;
    a.hist_end = hist_end;
    a.scale2 = sm_scale * kLog2e;
    a.out = out;
    a.status = status;
    const int ngrp = kHeadDim / L.group;
#define OSCAR_MMA_CASE(GG, NN) \
    if (L.gqa == GG && ngrp == NN) return launch_mma<GG, NN>(L, a, batch, history, window, st, clusters);
    OSCAR_MMA_CASE(1, 1) OSCAR_MMA_CASE(2, 1) OSCAR_MMA_CASE(4, 1) OSCAR_MMA_CASE(8, 1)
    OSCAR_MMA_CASE(1, 2) OSCAR_MMA_CASE(2, 2) OSCAR_MMA_CASE(4, 2) OSCAR_MMA_CASE(8, 2)
    OSCAR_MMA_CASE(1, 4) OSCAR_MMA_CASE(2, 4) OSCAR_MMA_CASE(4, 4) OSCAR_MMA_CASE(8, 4)
#undef OSCAR_MMA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace oscar
