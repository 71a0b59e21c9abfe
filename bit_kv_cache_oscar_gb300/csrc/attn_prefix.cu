// Shared-prefix (cascade) INT2 attention on the 5th-generation tensor cores.
//
// Requests whose page tables share the INT2 pages of a prefix (a radix prefix cache: "Together AI
// 開源 OSCAR", section 服務系統, paged and prefix-cache compatible; OSCAR news article, paragraphs
// on prefix-cache hits) read that prefix once per kv head for all of them: for one kv head all
// R*G query rows (<= 128) of R requests meet the same keys, so per 128-token tile
//   S[m][t]  = sum_k Q'[m][k] . Kc[t][k]            tcgen05 M128 N128 K16 x 8, Q' = Q_hi + Q_lo (f16)
//   logit    = csc * sk[t] * S[m][t] + zk[t] * qz[m]  (base 2)
//   O[m][n] += sum_t P'[m][t] . Vc[t][n]              tcgen05 M128 N128 K16 x 8, P' = (p * sv)_hi + _lo
// with the 2-bit codes as f16 subnormals c * f * 2^-24 (f a power of 4 set by the code's bit
// position); Q' is divided by f, O is multiplied by 2^24 / f at the end.  Kc is stored token-major
// ([t][k'], K-major B of QK, channels in the pair order k' = 16W + 2i + e -> channel 16W + i + 8e);
// Vc is stored channel-major ([n][t], K-major B of PV), two tokens per 32-bit word.  The logits'
// zero-point term needs one group per row (group 128).  One CTA per (token split, kv head, group
// of 128 / G requests); the phases of a tile run one after another.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include <cstring>

#include "oscar_internal.cuh"
#include "ptx.cuh"
#include "tma.cuh"

namespace oscar {
namespace {

constexpr int kPT = 128;                                 // tokens per tile
constexpr int kRows = 128;                               // query rows (MMA M)
constexpr int kOpBytes = kRows * kHeadDim * 2;           // a 128 x 128 f16 operand (32 KB)
constexpr int kHalf = kOpBytes / 2;                      // one 64-column half of it
constexpr int kOffQh = 0, kOffQl = kOpBytes, kOffK = 2 * kOpBytes, kOffV = 3 * kOpBytes;
constexpr int kOffPh = 4 * kOpBytes, kOffPl = 5 * kOpBytes;
constexpr int kStageB = 2 * kPT * 32;                    // one tile's codes: K [128][32 B], V [128][32 B]
constexpr int kOffStage = 6 * kOpBytes;                  // the stage of the next tile's codes
constexpr int kOffSzb = kOffStage + kStageB;             // tensor-map path: bf16 [4 arrays][128][8 heads]
constexpr int kOffSzf = kOffSzb + 4 * kPT * 16;          // fp32 [128][4]: sk * csc, zk, sv, zv
constexpr int kOffRed = kOffSzf + kPT * 16;              // [2 halves][128 rows] exchange of row values
constexpr int kOffPages = kOffRed + 2 * kRows * 4;       // the prefix's page ids (up to kMaxPages)
constexpr int kMaxPages = 1536;
constexpr int kOffBar = kOffPages + kMaxPages * 4;       // MMA mbarrier, TMEM address, copy mbarrier, piece mask
constexpr int kSmemP = kOffBar + 64 + 1024;
constexpr float kNoMaxP = -0x1p100f;                     // running maximum before any logit
constexpr int kThreadsP = 256;
constexpr uint32_t kTmemColsP = 256;                     // S: columns 0..127, O: 128..255
// tcgen05.mma kind::f16 instruction descriptor: fp32 D, f16 A and B (both K-major), M128 N128
constexpr uint32_t kIdescF16 = (1u << 4) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

constexpr uint32_t kM0 = 0x00030003u, kM1 = 0x000C000Cu, kM2 = 0x00300030u, kM3 = 0x00C000C0u,
                   kM4 = 0x03000300u;
constexpr float kTwo24 = 16777216.0f;

// factor of pair register i (0..7) of a 16-channel word: 1, 4, 16, 64, 256, 4, 16, 64
__device__ __host__ constexpr float pair_factor(int i) { return i == 4 ? 256.f : (float)(1 << (2 * (i & 3))); }

// byte offset of the 16-byte chunk holding elements (row n, columns k .. k + 7) of a 128-row K-major
// f16 operand in the 128-byte swizzle layout (k % 8 == 0)
__device__ __forceinline__ uint32_t sw_off(int n, int k) {
    return (uint32_t)((k >> 6) * kHalf + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

struct PrefixArgs {
    const float *q_rot;          // [B][Hq][128]
    int tma;                     // 8 kv heads, page size 32 / 64: tiles land by tensor-map copies
    int batch, G, n_kv;
    Int2PoolView pool;
    const int32_t *pages;        // logical page -> physical page of the shared positions
    int n_logical, page_size;
    int lo, hi;                  // positions [lo, hi)
    int splits;                  // token splits (grid.x) = partial slots 0 .. splits - 1
    float scale2;                // sm_scale * log2(e)
    PartialsView out;            // m, l [B][Hq][S + 1], acc [B][Hq][S + 1][128]
    int32_t *status;
};

// tmaps: codes K, codes V ([rows][8 heads][32 B], box 32 B x 1 head x page rows), scale K, zero K,
// scale V, zero V ([rows][8 heads] bf16, box 8 heads x page rows); unused when a.tma == 0.
struct PrefixMaps {
    CUtensorMap m[6];
};

__global__ void __launch_bounds__(kThreadsP, 1) prefix_attn_kernel(PrefixArgs a, const __grid_constant__ PrefixMaps tm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = saddr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, h = blockIdx.y;
    // this CTA's requests: b0 .. b0 + R - 1 (query row m = (b - b0) G + g)
    const int G = a.G, Hq = a.n_kv * G, b0 = blockIdx.z * (kRows / G);
    const int R = min(kRows / G, a.batch - b0), rows = R * G;
    const uint32_t bar = sb + kOffBar;
    const float csc = a.scale2 * kTwo24;

    // this split's 128-token tiles (absolute positions) that meet [lo, hi), balanced over the splits
    const int t_first = a.lo / kPT, nt = (a.hi + kPT - 1) / kPT - t_first;
    const int ta = t_first + (int)((long long)s * nt / a.splits);
    const int tb = t_first + (int)((long long)(s + 1) * nt / a.splits);

    if (warp == 0) {
        tmem_alloc(bar + 8, kTmemColsP);
        tmem_relinquish();
    }
    const uint32_t tbar = bar + 16;              // the tile's tensor-map copies (expect-tx)
    int *piece_ok = reinterpret_cast<int *>(sm + kOffBar + 24);    // pieces of the tile that were copied
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(tbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the prefix's page ids, read once (the copies of every tile index them)
    int *pages_s = reinterpret_cast<int *>(sm + kOffPages);
    const bool pages_in_smem = a.n_logical <= kMaxPages;
    if (pages_in_smem)
        for (int i = tid; i < a.n_logical; i += kThreadsP) pages_s[i] = a.pages[i];
    // Q' hi / lo, row m = r G + g (request r, query head g of kv head h), column k' = 16 W + 2 i + e
    for (int it = tid; it < kRows * 16; it += kThreadsP) {
        const int m = it & (kRows - 1), kc = (it >> 7) * 8;
        const bool valid = m < rows;
        const float *qrow = a.q_rot + (valid ? ((size_t)(b0 + m / G) * Hq + h * G + m % G) * kHeadDim : 0);
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int kp = kc + 2 * u, W = kp >> 4, i = (kp & 15) >> 1;
            const float inv = 1.0f / pair_factor(i);
            const float v0 = valid ? qrow[16 * W + i] * inv : 0.f;
            const float v1 = valid ? qrow[16 * W + 8 + i] * inv : 0.f;
            const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
            hv[u] = pack_h2(h0, h1);
            lv[u] = pack_h2(__float2half_rn(v0 - __half2float(h0)), __float2half_rn(v1 - __half2float(h1)));
        }
        *reinterpret_cast<uint4 *>(sm + kOffQh + sw_off(m, kc)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(sm + kOffQl + sw_off(m, kc)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
    // This thread's query row is m = 32 (warp & 3) + lane, the TMEM lane its warp reads; the two
    // warps of a lane quarter take the columns [64 hc, 64 hc + 64) of S, O and P' (hc = warp / 4).
    const int m = 32 * (warp & 3) + lane, hc = warp >> 2;
    float qz = 0.f;                              // scale2 * sum of the row's rotated query (zero-point term)
    if (m < rows) {
        const float *qrow = a.q_rot + ((size_t)(b0 + m / G) * Hq + h * G + m % G) * kHeadDim;
        for (int k = 0; k < kHeadDim; ++k) qz += qrow[k];
        qz *= a.scale2;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + kOffBar + 8);
    const uint32_t tS = tmem, tO = tmem + 128;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;     // this warp's TMEM lane quarter
    float *red = reinterpret_cast<float *>(sm + kOffRed);              // [2][128]

    // Tile t's codes into the stage buffer and this thread's two scale/zero values (array c / 128,
    // token c % 128 for c = tid, tid + 256) into sv: per-thread cp.async copies and loads.
    auto load_tile = [&](int t, uint16_t (&sv)[2]) {
        const int p0 = t * kPT;
        const int v_lo = max(a.lo, p0) - p0, v_hi = min(a.hi, p0 + kPT) - p0;
        const uint32_t stg = sb + kOffStage;
        for (int c = tid; c < kPT * 2; c += kThreadsP) {
            const int tk = c >> 1, p = p0 + tk, lp = p / a.page_size;
            const bool in = tk >= v_lo && tk < v_hi && lp < a.n_logical;
            const int pg = in ? (pages_in_smem ? pages_s[lp] : a.pages[lp]) : -1;
            if (pg >= 0 && pg < a.pool.n_pages) {
                const size_t row = ((size_t)pg * a.page_size + p % a.page_size) * a.n_kv + h;
                cp_async16(stg + tk * 32 + (c & 1) * 16, a.pool.codes_k + row * 32 + (c & 1) * 16);
                cp_async16(stg + kPT * 32 + tk * 32 + (c & 1) * 16, a.pool.codes_v + row * 32 + (c & 1) * 16);
            } else if (in && (c & 1) == 0) {
                flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int c = tid + kThreadsP * k, arr = c >> 7, tk = c & (kPT - 1), p = p0 + tk, lp = p / a.page_size;
            sv[k] = 0;
            if (tk >= v_lo && tk < v_hi && lp < a.n_logical) {
                const int pg = pages_in_smem ? pages_s[lp] : a.pages[lp];
                if (pg >= 0 && pg < a.pool.n_pages) {
                    const size_t row = ((size_t)pg * a.page_size + p % a.page_size) * a.n_kv + h;
                    const uint16_t *src = arr == 0 ? a.pool.scale_k : arr == 1 ? a.pool.zero_k
                                        : arr == 2 ? a.pool.scale_v : a.pool.zero_v;
                    sv[k] = src[row];
                }
            }
        }
    };
    auto store_sz = [&](const uint16_t (&sv)[2]) {
        float *dst = reinterpret_cast<float *>(sm + kOffSzf);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int c = tid + kThreadsP * k, arr = c >> 7, tk = c & (kPT - 1);
            const float f = bf16_to_f32(sv[k]);
            dst[tk * 4 + arr] = arr == 0 ? f * csc : f;
        }
    };
    // The tensor-map path (warp 0): the tile's page pieces (pr rows each) that meet [lo, hi), six
    // copies per piece (lane 6 k + o: piece k, o = codes K, codes V, scale K, zero K, scale V,
    // zero V) completing on tbar; the mask of copied pieces goes to piece_ok.
    const int pr = a.page_size < kPT ? a.page_size : kPT, npc = kPT / pr;
    auto issue_tma = [&](int t) {
        const int p0 = t * kPT;
        int pg = -1;
        if (lane < npc) {
            const int p = p0 + lane * pr, lp = p / a.page_size;
            if (p + pr > a.lo && p < a.hi && lp < a.n_logical) {
                pg = pages_in_smem ? pages_s[lp] : a.pages[lp];
                if (pg < 0 || pg >= a.pool.n_pages) {
                    flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
                    pg = -1;
                }
            }
        }
        const unsigned ok = __ballot_sync(0xffffffffu, pg >= 0);
        const int k = lane / 6, o = lane % 6;
        const int pgk = __shfl_sync(0xffffffffu, pg, k < npc ? k : 0);
        if (lane == 0) {
            *piece_ok = (int)ok;
            mbar_arrive_expect_tx(tbar, (uint32_t)(__popc(ok) * pr * 128));
        }
        __syncwarp();
        if (k < npc && ((ok >> k) & 1)) {
            const int row0 = pgk * a.page_size;
            if (o < 2)
                tma_load_3d(sb + kOffStage + o * kPT * 32 + k * pr * 32, &tm.m[o], 0, h, row0, tbar);
            else
                tma_load_2d(sb + kOffSzb + (o - 2) * kPT * 16 + k * pr * 16, &tm.m[o], 0, row0, tbar);
        }
    };

    float m_run = kNoMaxP, l_run = 0.f, z_run = 0.f;    // l and zero sums: this half's columns
    if (ta < tb) {
        if (a.tma) {
            if (warp == 0) issue_tma(ta);
        } else {
            uint16_t sv[2];
            load_tile(ta, sv);
            store_sz(sv);
        }
    }
    uint32_t r0[32], r1[32];
    for (int t = ta; t < tb; ++t) {
        const bool first = t == ta, more = t + 1 < tb;
        const int p0 = t * kPT;
        const int v_lo = max(a.lo, p0) - p0, v_hi = min(a.hi, p0 + kPT) - p0;   // valid tokens of the tile
        if (a.tma) {
            if (!mbar_wait(tbar, (t - ta) & 1) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
            // this head's scale/zero of the tile to fp32 (zero where nothing was copied or out of range)
            const int okm = *piece_ok;
            const uint16_t *szb = reinterpret_cast<const uint16_t *>(sm + kOffSzb);
            float *dst = reinterpret_cast<float *>(sm + kOffSzf);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = tid + kThreadsP * k, arr = c >> 7, tk = c & (kPT - 1);
                const bool in = tk >= v_lo && tk < v_hi && ((okm >> (tk / pr)) & 1);
                const float f = in ? bf16_to_f32(szb[(arr * kPT + tk) * 8 + h]) : 0.f;
                dst[tk * 4 + arr] = arr == 0 ? f * csc : f;
            }
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();                         // tile t's codes and scale/zero are in place
        const uint8_t *stg = sm + kOffStage;
        // 1. K codes -> Kc [t][k'] (8 f16 pairs per code word); warp task = (32 tokens, word W)
        for (int task = warp; task < 4 * 8; task += kThreadsP / 32) {
            const int tk = (task >> 3) * 32 + lane, W = task & 7;
            const uint32_t w = *reinterpret_cast<const uint32_t *>(stg + tk * 32 + W * 4);
            const uint32_t wb = __byte_perm(w, 0, 0x3321);
            *reinterpret_cast<uint4 *>(sm + kOffK + sw_off(tk, 16 * W)) = make_uint4(w & kM0, w & kM1, w & kM2, w & kM3);
            *reinterpret_cast<uint4 *>(sm + kOffK + sw_off(tk, 16 * W + 8)) =
                make_uint4(w & kM4, wb & kM1, wb & kM2, wb & kM3);
        }
        //    V codes -> Vc [n][t], tokens (t0, t0 + 1) in one word; warp task = (64 tokens, word W)
        for (int task = warp; task < 2 * 8; task += kThreadsP / 32) {
            const int t0 = (task >> 3) * 64 + 2 * lane, W = task & 7;
            const uint8_t *vs = stg + kPT * 32;
            const uint32_t x = *reinterpret_cast<const uint32_t *>(vs + t0 * 32 + W * 4);
            const uint32_t y = *reinterpret_cast<const uint32_t *>(vs + (t0 + 1) * 32 + W * 4);
            const uint32_t P = __byte_perm(x, y, 0x5410), Pb = __byte_perm(x, y, 0x6521);
            const uint32_t Q = __byte_perm(x, y, 0x7632), Qb = __byte_perm(x, y, 0x7733);
            const uint32_t v[16] = {P & kM0, P & kM1, P & kM2, P & kM3, P & kM4, Pb & kM1, Pb & kM2, Pb & kM3,
                                    Q & kM0, Q & kM1, Q & kM2, Q & kM3, Q & kM4, Qb & kM1, Qb & kM2, Qb & kM3};
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<uint32_t *>(sm + kOffV + sw_off(16 * W + i, t0 & ~7) + (t0 & 7) * 2) = v[i];
        }
        // 2. tile t + 1's copies start once every thread is done with the stage, and land under this tile
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        uint16_t nv[2];
        if (more) {
            if (!a.tma) load_tile(t + 1, nv);
            else if (warp == 0) issue_tma(t + 1);
        }
        // 3. S = Q' . Kc^T (Q_hi then Q_lo, 8 K16 steps each)
        if (warp == 4 && lane == 0) {
            tc_fence_after();
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    tc_mma_bf16(tS, sw128_kmajor_desc(sb + (hl ? kOffQl : kOffQh) + koff),
                                sw128_kmajor_desc(sb + kOffK + koff), kIdescF16, (hl | kk) != 0);
                }
            tc_commit(bar);
        }
        // 4. softmax of the row over the tile: logits of this half's 64 columns, the row maximum
        //    through the exchange, O rescaled when it rises, p = 2^(logit - m), P' = p * sv (f16 hi/lo)
        if (!mbar_wait(bar, 0) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
        tc_fence_after();
        const float *szf = reinterpret_cast<const float *>(sm + kOffSzf);
        tmem_ld32(tS + lane_base + 64 * hc, r0);
        tmem_ld32(tS + lane_base + 64 * hc + 32, r1);
        tmem_ld_wait();
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // (four chains)
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            const int tk = 64 * hc + j;
            const float4 f = *reinterpret_cast<const float4 *>(szf + tk * 4);
            const float lg = fmaf(f.x, __uint_as_float(j < 32 ? r0[j] : r1[j - 32]), f.y * qz);
            const float lv = tk >= v_lo && tk < v_hi ? lg : -INFINITY;
            if (j < 32) r0[j] = __float_as_uint(lv); else r1[j - 32] = __float_as_uint(lv);
            mx4[j & 3] = fmaxf(mx4[j & 3], lv);
        }
        red[hc * kRows + m] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        __syncthreads();
        const float m_new = fmaxf(m_run, fmaxf(red[m], red[kRows + m]));
        const float alpha = ex2_approx(m_run - m_new);   // 0 on the first tile
        if (!first && __any_sync(0xffffffffu, m_new > m_run)) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t (&r)[32] = c ? r1 : r0;
                tmem_ld32(tO + lane_base + 64 * hc + 32 * c, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                tmem_st32(tO + lane_base + 64 * hc + 32 * c, r);
            }
            tmem_st_wait();
            // (the logits were overwritten: read S again)
            tmem_ld32(tS + lane_base + 64 * hc, r0);
            tmem_ld32(tS + lane_base + 64 * hc + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const int tk = 64 * hc + j;
                const float4 f = *reinterpret_cast<const float4 *>(szf + tk * 4);
                const float lg = fmaf(f.x, __uint_as_float(j < 32 ? r0[j] : r1[j - 32]), f.y * qz);
                const float lv = tk >= v_lo && tk < v_hi ? lg : -INFINITY;
                if (j < 32) r0[j] = __float_as_uint(lv); else r1[j - 32] = __float_as_uint(lv);
            }
        }
        l_run *= alpha;
        z_run *= alpha;
        m_run = m_new;
        float l4[4] = {0.f, 0.f, 0.f, 0.f}, z4[4] = {0.f, 0.f, 0.f, 0.f};   // (four chains each)
#pragma unroll
        for (int j0 = 0; j0 < 64; j0 += 8) {
            uint32_t hv[4], lw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float pp[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = j0 + 2 * u + e, tk = 64 * hc + j;
                    const float4 f = *reinterpret_cast<const float4 *>(szf + tk * 4);
                    const float p = ex2_approx(__uint_as_float(j < 32 ? r0[j] : r1[j - 32]) - m_run);
                    l4[j & 3] += p;
                    z4[j & 3] = fmaf(p, f.w, z4[j & 3]);
                    pp[e] = p * f.z;
                }
                const __half h0 = __float2half_rn(pp[0]), h1 = __float2half_rn(pp[1]);
                hv[u] = pack_h2(h0, h1);
                lw[u] = pack_h2(__float2half_rn(pp[0] - __half2float(h0)), __float2half_rn(pp[1] - __half2float(h1)));
            }
            const int k = 64 * hc + j0;
            *reinterpret_cast<uint4 *>(sm + kOffPh + sw_off(m, k)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4 *>(sm + kOffPl + sw_off(m, k)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        z_run += (z4[0] + z4[1]) + (z4[2] + z4[3]);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // 5. O (+)= P' . Vc^T (P_hi then P_lo); the first tile overwrites O
        if (warp == 4 && lane == 0) {
            tc_fence_after();
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    tc_mma_bf16(tO, sw128_kmajor_desc(sb + (hl ? kOffPl : kOffPh) + koff),
                                sw128_kmajor_desc(sb + kOffV + koff), kIdescF16, !(first && hl == 0 && kk == 0));
                }
            tc_commit(bar);
        }
        // 6. the operands are rewritten by the next tile only once PV has read them; tile t + 1's
        //    scale/zero (cp.async path) replace this tile's, whose softmax is done
        if (more && !a.tma) store_sz(nv);
        if (!mbar_wait(bar, 1) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
        tc_fence_after();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");   // (no copy is outstanding: every tile was waited on)
    // epilogue: the row's l and zero sums over both halves; acc = O * 2^24 / factor(n) + z
    red[hc * kRows + m] = l_run;
    __syncthreads();
    const float l_tot = red[m] + red[kRows + m];
    __syncthreads();
    red[hc * kRows + m] = z_run;
    __syncthreads();
    const float z_tot = red[m] + red[kRows + m];
    {
        const int r = b0 + m / G, g = m % G;
        const bool out = m < rows;
        const size_t idx = out ? ((size_t)r * Hq + h * G + g) * (size_t)(a.out.S + 1) + s : 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t (&rr)[32] = c ? r1 : r0;
            if (ta < tb) {
                tmem_ld32(tO + lane_base + 64 * hc + 32 * c, rr);
                tmem_ld_wait();
            }
            if (out) {
                float *dst = a.out.acc + idx * kHeadDim + 64 * hc + 32 * c;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = 64 * hc + 32 * c + j;
                    dst[j] = ta < tb ? fmaf(__uint_as_float(rr[j]), kTwo24 / pair_factor(n & 7), z_tot) : 0.f;
                }
            }
        }
        if (out && hc == 0) {
            a.out.m[idx] = l_tot > 0.f ? m_run : -INFINITY;
            a.out.l[idx] = l_tot;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemColsP);
    }
}

}  // namespace

cudaError_t launch_prefix_attention(const oscar_layout_t &L, const float *q_rot, Int2PoolView pool,
                                    const int32_t *prefix_pt, int prefix_end, int batch, int splits, float sm_scale,
                                    PartialsView out, int32_t *status, cudaStream_t st) {
    if (batch <= 0 || prefix_end <= L.sink) return cudaSuccess;
    if (L.group != kHeadDim || splits < 1 || splits > out.S || L.gqa > kRows) return cudaErrorInvalidValue;
    PrefixArgs a;
    a.q_rot = q_rot;
    a.batch = batch;
    a.G = L.gqa;
    a.n_kv = L.n_kv_heads;
    a.pool = pool;
    a.pages = prefix_pt;
    a.n_logical = (prefix_end + L.page_size - 1) / L.page_size;
    a.page_size = L.page_size;
    a.lo = L.sink;
    a.hi = prefix_end;
    a.splits = splits;
    a.scale2 = sm_scale * kLog2e;
    a.out = out;
    a.status = status;
    PrefixMaps tm;
    memset(&tm, 0, sizeof(tm));
    a.tma = L.n_kv_heads == 8 && L.page_size >= 32;
    if (a.tma) {
        EncodeTiledFn fn = encode_fn();
        const cuuint64_t rows = (cuuint64_t)pool.n_pages * L.page_size;
        const cuuint32_t pr = (cuuint32_t)(L.page_size < kPT ? L.page_size : kPT);
        const cuuint32_t e3[3] = {1, 1, 1}, e2[2] = {1, 1};
        const cuuint64_t cdims[3] = {32, 8, rows}, cstr[2] = {32, 256};
        const cuuint32_t cbox[3] = {32, 1, pr};
        const cuuint64_t sdims[2] = {8, rows}, sstr[1] = {16};
        const cuuint32_t sbox[2] = {8, pr};
        const void *cbase[2] = {pool.codes_k, pool.codes_v};
        const void *sbase[4] = {pool.scale_k, pool.zero_k, pool.scale_v, pool.zero_v};
        bool ok = fn != nullptr;
        for (int i = 0; ok && i < 2; ++i)
            ok = fn(&tm.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(cbase[i]), cdims, cstr, cbox, e3,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        for (int i = 0; ok && i < 4; ++i)
            ok = fn(&tm.m[2 + i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(sbase[i]), sdims, sstr, sbox,
                    e2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        if (!ok) return cudaErrorInvalidValue;
    }
    if (cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(prefix_attn_kernel), kSmemP)) return e;
    const int groups = (batch + kRows / L.gqa - 1) / (kRows / L.gqa);
    prefix_attn_kernel<<<dim3(splits, L.n_kv_heads, groups), kThreadsP, kSmemP, st>>>(a, tm);
    return cudaGetLastError();
}

}  // namespace oscar
