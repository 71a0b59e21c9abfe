// Bulk demotion on the 5th-generation tensor cores (tcgen05): every position of a range of each
// request, every kv head, K and V, rotated (x . R), clipped, quantized and packed into the INT2 pool.
// This is how a whole prompt's history [sink, T - recent) enters the INT2 cache after prefill.
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph (rotate / clip /
// quantize / pack, 4 x 2-bit codes per byte); "Together AI 開源 OSCAR", section
// "OSCAR 的不同之處" (R_K, R_V); estelledc notes "核心要点" item 3 (the history is kept in INT2).
//
// Design.  The rotation of n rows is an [n x 128] . [128 x 128] GEMM per (K or V, kv head).  Each
// CTA (one per SM) is bound to one such pair and keeps its R in shared memory for the whole launch,
// as two bf16 halves R = R_hi + R_lo (R_lo = bf16(R - R_hi)) in the 128-byte-swizzled K-major layout
// that tcgen05.mma reads; the bf16 row x is exact, so x . R_hi + x . R_lo carries R to about 16
// significant bits and the rotated rows stay within 2^-14 ||x||_2 of the exact product.
// A tile is 128 consecutive positions of one request.
//   warp 0       TMA producer: the tile's 128 bf16 rows (256 bytes each, one per position, at the
//                pool's token stride) in page pieces, 4-stage ring, expect-tx mbarriers
//   warp 1       allocates the TMEM; one thread issues 16 MMAs M128 N128 K16 per tile
//                (x . R_hi then x . R_lo) into one of three TMEM accumulators, then tcgen05.commit
//   warps 2..13  three epilogue groups of 4 warps, one per accumulator: each thread owns a row
//                and reads it twice (tcgen05.ld 32x32b, 32 columns at a time): the groups' minima
//                and maxima, then the codes.
// The quantizer is the one of every other demotion path (per group of g channels: lo = c min,
// hi = c max, zero = bf16(lo), scale = bf16((hi - lo)/3), code = clamp(rint((y - zero)/scale), 0, 3)),
// computed bit for bit; the quotient is taken as (y - zero) * (1/scale) unless that product lies
// within 2^-18 of a half-integer, where the correctly rounded quotients decide (the product's
// error is below 2^-21 there, so both give the same code).
#include <cuda.h>
#include <cuda_bf16.h>

#include "oscar_internal.cuh"
#include "ptx.cuh"
#include "tma.cuh"

namespace oscar {
namespace {

constexpr int kTileRows = 128;                       // positions per tile (the MMA's M)
constexpr int kHalfBytes = kTileRows * 128;          // one 64-channel half of 128 bf16 rows
constexpr int kStageBytes = 2 * kHalfBytes;          // a tile (32 KB)
constexpr int kStagesTC = 4;
constexpr int kRBytes = 4 * kHalfBytes;              // R^T: hi and lo, two channel halves each (64 KB)
constexpr int kEpiGroups = 3;                        // (measured faster than 2 or 4)
constexpr int kBulkThreads = 64 + 128 * kEpiGroups;  // producer warp, MMA warp, epilogue groups
constexpr uint32_t kTmemCols = 512;                  // a power of two >= 128 per group's accumulator
constexpr uint32_t kIdesc = tc_idesc_bf16(128, 128);
constexpr int kOffR = 0;
constexpr int kOffA = kRBytes;
constexpr int kOffBar = kOffA + kStagesTC * kStageBytes;
constexpr int kBulkSmem = kOffBar + 256 + 1024;      // + slack to align the base to 1024 bytes
// |q - rint(q)| at or above this: q lies within 2^-18 of a half-integer
constexpr float kFastMargin = 0.5f - 0x1p-18f;

struct BulkArgs {
    int n_kv, page_size, group, max_pages, batch, bf16_pages, ctas_per_pair;
    const int32_t *bf16_pt, *int2_pt, *pos_begin, *pos_end;
    const float *RK, *RV;
    float cK, cV;
    Int2PoolMut dst;
    float *rot_out;
    int32_t *status;
};

// The tiles of one (K/V, kv head) pair in a fixed order: request by request, the 128-position
// tiles [128t, 128t + 128) that meet [pos_begin[b], pos_end[b]).  find() takes increasing i.
struct TileWalk {
    int b = 0, base = 0;
    __device__ __forceinline__ bool find(const BulkArgs &a, int i, int &rb, int &t, int &lo, int &hi) {
        for (; b < a.batch; ++b) {
            const int l = a.pos_begin[b], h = a.pos_end[b];
            const bool ok = l >= 0 && h > l && (long long)h <= (long long)a.max_pages * a.page_size;
            const int cnt = ok ? (h - 1) / kTileRows - l / kTileRows + 1 : 0;
            if (i < base + cnt) {
                rb = b;
                t = l / kTileRows + (i - base);
                lo = l;
                hi = h;
                return true;
            }
            base += cnt;
        }
        return false;
    }
};

// Packed fp32 pairs (sm_100 family: add / sub / mul .f32x2, each half rounded to nearest as
// the scalar instruction would): two elements per instruction where the quantizer's steps allow.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// min / max of three (the three-input forms of the sm_100 family)
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// The quantizer's codes of 32 channels y (one chunk of a row, inside one group of zero z, scale
// s != 0 and inv = 1/s rounded) as two 32-bit words, code i at bits 2i.
// Per element: q' = clamp((y - z) * inv, 0, 3), rounded to an integer (ties to even) by adding
// 1.5 * 2^23, whose low bits are then the code.  That is clamp(rint(q), 0, 3) of the correctly
// rounded quotient q whenever q' lies more than 2^-18 from a half-integer (|q' - q| < 2^-21 there).
// Returns the largest distance of a q' to its integer: at kFastMargin or above, the caller takes
// the chunk again through codes_chunk_exact.  The subtractions, the product and the rounding
// steps run on element pairs (the same roundings as one element at a time).
__device__ __forceinline__ float codes_chunk(const uint32_t (&v)[32], float z, float inv, uint32_t &w0,
                                             uint32_t &w1) {
    constexpr float kMagic = 12582912.0f;               // 1.5 * 2^23: y = kMagic + code, bits 0x4B400000 + code
    // sum over the 16 codes of a word of bits(y) * 4^i carries 0x4B400000 * (4^16 - 1) / 3 (mod 2^32)
    // besides the codes' own sum of code * 4^i; one subtraction per word removes it
    constexpr uint32_t kBias = 0x4B400000u * 0x55555555u;
    const uint64_t z2 = f2_pack(__float_as_uint(z), __float_as_uint(z));
    const uint64_t inv2 = f2_pack(__float_as_uint(inv), __float_as_uint(inv));
    const uint64_t mg2 = f2_pack(__float_as_uint(kMagic), __float_as_uint(kMagic));
    uint32_t w[2] = {0u, 0u};
    float e4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        float q0, q1;
        f2_unpack(f2_mul(f2_sub(f2_pack(v[i], v[i + 1]), z2), inv2), q0, q1);
        const float c0 = fminf(fmaxf(q0, 0.0f), 3.0f), c1 = fminf(fmaxf(q1, 0.0f), 3.0f);
        const uint64_t c2 = f2_pack(__float_as_uint(c0), __float_as_uint(c1));
        const uint64_t y2 = f2_add(c2, mg2);
        float y0, y1, d0, d1;
        f2_unpack(y2, y0, y1);
        f2_unpack(f2_sub(c2, f2_sub(y2, mg2)), d0, d1);
        e4[i & 3] = fmaxf(e4[i & 3], fabsf(d0));
        e4[(i + 1) & 3] = fmaxf(e4[(i + 1) & 3], fabsf(d1));
        w[i >> 4] += __float_as_uint(y0) * (1u << (2 * (i & 15))) + __float_as_uint(y1) * (1u << (2 * ((i + 1) & 15)));
    }
    w0 = w[0] - kBias;
    w1 = w[1] - kBias;
    return fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]));
}

// The same codes from the correctly rounded quotients, the chunk read again from TMEM at taddr
// (the whole warp calls it).  Kept out of line: it is rarely taken and long.
__device__ __noinline__ void codes_chunk_exact(uint32_t taddr, float z, float s, uint32_t &w0, uint32_t &w1) {
    __syncwarp();
    uint32_t v[32];
    tmem_ld32(taddr, v);
    tmem_ld_wait();
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float r = rintf(__fdiv_rn(__fsub_rn(__uint_as_float(v[i]), z), s));
        const uint32_t c = r >= 3.0f ? 3u : (r >= 0.0f ? (uint32_t)r : 0u);
        w[i >> 4] |= c << (2 * (i & 15));
    }
    w0 = w[0];
    w1 = w[1];
}

template <int GROUP>
__global__ void __launch_bounds__(kBulkThreads, 1)
    bulk_demote_kernel(BulkArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = saddr(sm);
    const uint32_t bars = sbase + kOffBar;
    // mbarriers: full[s] = bars + 8s, empty[s] = bars + 32 + 8s, acc_full[e] = bars + 64 + 8e,
    // acc_empty[e] = bars + 96 + 8e, done = bars + 128; the TMEM address at bars + 136
    const uint32_t bar_full = bars, bar_empty = bars + 32, bar_accf = bars + 64, bar_acce = bars + 96;
    const uint32_t bar_done = bars + 128, tmem_slot = bars + 136;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pairs = 2 * a.n_kv;
    const int pair = blockIdx.x % pairs, cta = blockIdx.x / pairs;
    const int kind = pair / a.n_kv, head = pair % a.n_kv;   // kind 0 = K, 1 = V
    const float *Rb = kind ? a.RV : a.RK;                   // NULL R_V: values stored as they are (R = I)
    const float *R = Rb ? Rb + (size_t)head * kHeadDim * kHeadDim : nullptr;
    const CUtensorMap *tm = kind ? &tmv : &tmk;
    const int cpp = a.ctas_per_pair;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesTC; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int e = 0; e < kEpiGroups; ++e) {
            mbar_init(bar_accf + 8 * e, 1);
            mbar_init(bar_acce + 8 * e, 128);
        }
        mbar_init(bar_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (blockIdx.x == 0)
            for (int b = 0; b < a.batch; ++b) {
                const int l = a.pos_begin[b], h = a.pos_end[b];
                if (l < 0 || h < l || (long long)h > (long long)a.max_pages * a.page_size)
                    flag_status(a.status, OSCAR_DEV_BAD_LENGTH);
            }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // R^T as bf16 hi / lo: operand row n = output channel n, K = input channel k; each work item
    // writes one 16-byte chunk (8 input channels) of one row of both, at its swizzled place
    for (int it = threadIdx.x; it < kHeadDim * 16; it += blockDim.x) {
        const int n = it & 127, k = (it >> 7) * 8;
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
            const float r0 = R ? R[(k + u) * kHeadDim + n] : (k + u == n ? 1.0f : 0.0f);
            const float r1 = R ? R[(k + u + 1) * kHeadDim + n] : (k + u + 1 == n ? 1.0f : 0.0f);
            const uint16_t h0 = f32_to_bf16_rn(r0), h1 = f32_to_bf16_rn(r1);
            const uint16_t l0 = f32_to_bf16_rn(__fsub_rn(r0, bf16_to_f32(h0)));
            const uint16_t l1 = f32_to_bf16_rn(__fsub_rn(r1, bf16_to_f32(h1)));
            hv[u >> 1] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            lv[u >> 1] = (uint32_t)l0 | ((uint32_t)l1 << 16);
        }
        const int off = (k >> 6) * kHalfBytes + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4);
        *reinterpret_cast<uint4 *>(sm + kOffR + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(sm + kOffR + 2 * kHalfBytes + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
    fence_proxy_async_smem();          // the tensor cores (async proxy) read what these stores wrote
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + kOffBar + 136);

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // Lane j copies piece j of the tile (rows of one page, or 128 rows); the page ids of the
        // next tile are loaded while this one waits for its stage.
        const int ps = a.page_size;
        const int rpl = ps < kTileRows ? ps : kTileRows;        // rows per copy: one page, or 128
        const int np = kTileRows / rpl;
        // this lane's piece of tile t of request b: its tensor-map row, or -1 (none or outside the range)
        auto piece_row = [&](int b, int t, int lo, int hi) -> int {
            const int p0 = t * kTileRows + lane * rpl;
            if (lane >= np || p0 + rpl <= lo || p0 >= hi) return -1;
            const int pg = a.bf16_pt[(size_t)b * a.max_pages + p0 / ps];
            if (pg < 0 || pg >= a.bf16_pages) {
                flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
                return -1;
            }
            return pg * ps + p0 % ps;
        };
        TileWalk wk;
        int b, t, lo, hi;
        int i = cta;
        bool have = wk.find(a, i, b, t, lo, hi);
        int z = have ? piece_row(b, t, lo, hi) : -1;
        int issued = 0;                            // stage fills armed
        for (int n = 0; have; ++n) {
            int b2 = 0, t2 = 0, lo2 = 0, hi2 = 0;
            const bool have2 = wk.find(a, i + cpp, b2, t2, lo2, hi2);
            const int z2 = have2 ? piece_row(b2, t2, lo2, hi2) : -1;
            const int s = n % kStagesTC;
            if (!mbar_wait(bar_empty + 8 * s, ((n / kStagesTC) & 1) ^ 1) && lane == 0)
                flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
            const unsigned valid = __ballot_sync(0xffffffffu, z >= 0);
            if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * s, (uint32_t)__popc(valid) * 2 * rpl * 128);
            issued = n + 1;
            __syncwarp();
            if (z >= 0) {
                const uint32_t dst = sbase + kOffA + s * kStageBytes + lane * rpl * 128;
                tma_load_3d(dst, tm, 0, head, z, bar_full + 8 * s);
                tma_load_3d(dst + kHalfBytes, tm, 64, head, z, bar_full + 8 * s);
            }
            i += cpp;
            have = have2;
            b = b2;
            t = t2;
            lo = lo2;
            hi = hi2;
            z = z2;
        }
        // No copy may still be landing when the CTA leaves: the MMA warp waited for every fill, but
        // after a wait that gave up the last fills may be outstanding; wait (bounded) for each of them.
        for (int k = issued > kStagesTC ? issued - kStagesTC : 0; k < issued; ++k)
            if (!mbar_wait(bar_full + 8 * (k % kStagesTC), (k / kStagesTC) & 1) && lane == 0)
                flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            TileWalk wk;
            int b, t, lo, hi;
            int n = 0;
            for (int i = cta; wk.find(a, i, b, t, lo, hi); i += cpp, ++n) {
                const int s = n % kStagesTC, e = n % kEpiGroups;
                if (!mbar_wait(bar_acce + 8 * e, ((n / kEpiGroups) & 1) ^ 1))
                    flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                if (!mbar_wait(bar_full + 8 * s, (n / kStagesTC) & 1)) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)e * 128;
                const uint32_t abase = sbase + kOffA + s * kStageBytes;
#pragma unroll
                for (int h = 0; h < 2; ++h)          // x . R_hi, then x . R_lo
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                        tc_mma_bf16(d, sw128_kmajor_desc(abase + koff),
                                    sw128_kmajor_desc(sbase + kOffR + h * 2 * kHalfBytes + koff), kIdesc,
                                    (h | kk) != 0);
                    }
                tc_commit(bar_empty + 8 * s);       // the stage is free once these MMAs have read it
                tc_commit(bar_accf + 8 * e);        // the accumulator is ready
            }
            tc_commit(bar_done);
            if (!mbar_wait(bar_done, 0)) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        // Each thread owns one row of the tile and reads it from TMEM twice, 32 columns at a time:
        // first for the groups' minima and maxima, then to quantize.
        constexpr int kGroups = kHeadDim / GROUP;
        const int eg = (warp - 2) >> 2;            // group = accumulator
        const int q = warp & 3;                    // the TMEM lane quarter this warp may read
        const int r = 32 * q + lane;               // this thread's row of the tile
        const float clip = kind ? a.cV : a.cK;
        uint8_t *codes = kind ? a.dst.codes_v : a.dst.codes_k;
        uint16_t *scale = kind ? a.dst.scale_v : a.dst.scale_k;
        uint16_t *zero = kind ? a.dst.zero_v : a.dst.zero_k;
        const int ps = a.page_size;
        TileWalk wk;
        int b, t, lo, hi;
        int n = 0;
        for (int i = cta + eg * cpp; wk.find(a, i, b, t, lo, hi); i += kEpiGroups * cpp, ++n) {
            // where this row goes (all threads still take part in the warp-wide TMEM loads): the page
            // ids are loaded now, for a position inside the range, and looked at after the passes
            const int p = t * kTileRows + r;
            const bool in_range = p >= lo && p < hi;
            const int lp = (in_range ? p : lo) / ps, slot = p % ps;
            const int sp = a.bf16_pt[(size_t)b * a.max_pages + lp];
            const int dp = a.int2_pt[(size_t)b * a.max_pages + lp];
            auto row_ok = [&]() {                  // (a bad BF16 page is flagged by the producer)
                return in_range && sp >= 0 && sp < a.bf16_pages && dp >= 0 && dp < a.dst.n_pages;
            };
            const size_t slot_row = (size_t)(dp < 0 ? 0 : dp) * ps + slot;
            if (!mbar_wait(bar_accf + 8 * eg, n & 1) && lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
            __syncwarp();
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)eg * 128;
            uint32_t v[32];
            float gmn[kGroups], gmx[kGroups];
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                gmn[g] = INFINITY;
                gmx[g] = -INFINITY;
            }
            // (the chunk loops are not unrolled: unrolled, the epilogue outgrew the instruction cache)
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                tmem_ld32(ta + 32 * c, v);
                tmem_ld_wait();
                // two chains of three-input minima / maxima (a signed zero's sign is dropped below)
                float mn2[2], mx2[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) mn2[u] = mx2[u] = __uint_as_float(v[u]);
#pragma unroll
                for (int k = 2; k < 32; k += 2) {
                    mn2[(k >> 1) & 1] = fmin3(mn2[(k >> 1) & 1], __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
                    mx2[(k >> 1) & 1] = fmax3(mx2[(k >> 1) & 1], __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
                }
                const float cmn = fminf(mn2[0], mn2[1]);
                const float cmx = fmaxf(mx2[0], mx2[1]);
#pragma unroll
                for (int g = 0; g < kGroups; ++g)
                    if (g == (32 * c) / GROUP) {
                        gmn[g] = fminf(gmn[g], cmn);
                        gmx[g] = fmaxf(gmx[g], cmx);
                    }
                if (a.rot_out && row_ok()) {
                    float4 *o = reinterpret_cast<float4 *>(a.rot_out + ((slot_row * 2 + kind) * a.n_kv + head) * kHeadDim) + 8 * c;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        o[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                           __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
                }
            }
            uint16_t zb[kGroups], sb[kGroups];
            float zf[kGroups], sf[kGroups], inv[kGroups];
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                const float mn = __fadd_rn(gmn[g], 0.0f);        // a signed zero is read as +0
                const float mx = __fadd_rn(gmx[g], 0.0f);
                const float glo = __fmul_rn(clip, mn);           // clipped range c*[min, max]
                const float ghi = __fmul_rn(clip, mx);
                zb[g] = f32_to_bf16_rn(glo);
                sb[g] = f32_to_bf16_rn(__fdiv_rn(__fsub_rn(ghi, glo), 3.0f));
                zf[g] = bf16_to_f32(zb[g]);
                sf[g] = bf16_to_f32(sb[g]);
                inv[g] = __frcp_rn(sf[g]);
            }
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = 0u;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float z = zf[0], sc = sf[0], iv = inv[0];
#pragma unroll
                for (int g = 1; g < kGroups; ++g)
                    if (g == (32 * c) / GROUP) {
                        z = zf[g];
                        sc = sf[g];
                        iv = inv[g];
                    }
                tmem_ld32(ta + 32 * c, v);
                tmem_ld_wait();
                uint32_t w0 = 0u, w1 = 0u;                       // a degenerate group (scale 0): code 0
                float e = 0.0f;
                if (sc != 0.0f) e = codes_chunk(v, z, iv, w0, w1);
                if (__any_sync(0xffffffffu, e >= kFastMargin)) {   // rare: exact quotients (whole warp)
                    uint32_t x0, x1;
                    codes_chunk_exact(ta + 32 * c, z, sc != 0.0f ? sc : 1.0f, x0, x1);
                    if (e >= kFastMargin) {
                        w0 = x0;
                        w1 = x1;
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (k == c) {
                        w[2 * k] = w0;
                        w[2 * k + 1] = w1;
                    }
            }
            tc_fence_before();
            mbar_arrive(bar_acce + 8 * eg);        // the MMA may overwrite the accumulator
            if (in_range && sp >= 0 && sp < a.bf16_pages && (dp < 0 || dp >= a.dst.n_pages))
                flag_status(a.status, OSCAR_DEV_BAD_INT2_PAGE);
            if (!row_ok()) continue;
            const size_t row = slot_row * a.n_kv + head;
            uint4 *cdst = reinterpret_cast<uint4 *>(codes + row * (kHeadDim / 4));
            cdst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            cdst[1] = make_uint4(w[4], w[5], w[6], w[7]);
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                scale[row * kGroups + g] = sb[g];
                zero[row * kGroups + g] = zb[g];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The BF16 pool [pages * page_size][n_kv][128] as a 3-D bf16 tensor map (channel, kv head, token
// slot) whose box is 64 channels (128 bytes, swizzled) x 1 head x rpl slots.
bool pool_tensor_map(CUtensorMap *tm, const uint16_t *base, int n_kv, long long slots, int rpl) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_kv, (cuuint64_t)slots};
    const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)n_kv * kHeadDim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)rpl};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool demote_range_supported(const oscar_layout_t &L) {
    const int ps = L.page_size;
    return ps >= 16 && (ps % kTileRows == 0 || kTileRows % ps == 0);
}

cudaError_t launch_demote_range(const oscar_layout_t &L, Bf16PoolView src, const int32_t *bf16_pt,
                                const oscar_int2_pool_t &dst, const int32_t *int2_pt, int max_pages, int batch,
                                const int32_t *pos_begin, const int32_t *pos_end, const float *RK, const float *RV,
                                float cK, float cV, float *rot_out, int32_t *status, cudaStream_t st) {
    if (batch <= 0) return cudaSuccess;
    if (!demote_range_supported(L)) return cudaErrorInvalidValue;
    const int rpl = L.page_size < kTileRows ? L.page_size : kTileRows;
    const long long slots = (long long)src.n_pages * L.page_size;
    CUtensorMap tmk, tmv;
    if (!pool_tensor_map(&tmk, src.k, L.n_kv_heads, slots, rpl) ||
        !pool_tensor_map(&tmv, src.v, L.n_kv_heads, slots, rpl))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) return e;
    BulkArgs a{};
    a.n_kv = L.n_kv_heads;
    a.page_size = L.page_size;
    a.group = L.group;
    a.max_pages = max_pages;
    a.batch = batch;
    a.bf16_pages = src.n_pages;
    const int pairs = 2 * L.n_kv_heads;
    a.ctas_per_pair = sms / pairs > 0 ? sms / pairs : 1;
    a.bf16_pt = bf16_pt;
    a.int2_pt = int2_pt;
    a.pos_begin = pos_begin;
    a.pos_end = pos_end;
    a.RK = RK;
    a.RV = RV;
    a.cK = cK;
    a.cV = cV;
    a.dst = Int2PoolMut{dst.codes_k, dst.codes_v, dst.scale_k, dst.zero_k, dst.scale_v, dst.zero_v, dst.n_pages};
    a.rot_out = rot_out;
    a.status = status;
    const void *kern;
    switch (L.group) {
        case 32: kern = reinterpret_cast<const void *>(bulk_demote_kernel<32>); break;
        case 64: kern = reinterpret_cast<const void *>(bulk_demote_kernel<64>); break;
        case 128: kern = reinterpret_cast<const void *>(bulk_demote_kernel<128>); break;
        default: return cudaErrorInvalidValue;
    }
    if (cudaError_t e = ensure_dyn_smem(kern, kBulkSmem)) return e;
    const dim3 grid(pairs * a.ctas_per_pair);
    switch (L.group) {
        case 32: bulk_demote_kernel<32><<<grid, kBulkThreads, kBulkSmem, st>>>(a, tmk, tmv); break;
        case 64: bulk_demote_kernel<64><<<grid, kBulkThreads, kBulkSmem, st>>>(a, tmk, tmv); break;
        default: bulk_demote_kernel<128><<<grid, kBulkThreads, kBulkSmem, st>>>(a, tmk, tmv); break;
    }
    return cudaGetLastError();
}

}  // namespace oscar
