// BF16 decode-attention partials on the tensor cores: the sink + recent windows of
// every request (one partial per request and query head, slot S), and the all-BF16
// cache used as the comparison kernel (splits of [0, T), slots 0..S-1).
//
// Method: OSCAR news article (m.kljzs.com mirror), online-path paragraph — a BF16
// kernel handles sink/recent and its partial is merged with the INT2 ones;
// "Together AI 開源 OSCAR" (news.chathome.org), "服務系統" — 64 sink + 256 recent
// tokens stay BF16 and unrotated, so they meet the unrotated query.
//
// Structure (same pipeline as the INT2 kernel): a producer warp stages (kv head,
// 16-token tile) units of K and V rows into shared memory and signals an mbarrier
// per stage; 8 consumer warps take one unit each per stage.  With 8 kv heads and the
// whole cache (the comparison kernel) a stage is one tile of all 8 heads, moved by
// 32 tensor-map boxes of 16 rows x 64 channels (128-byte swizzle: 16-byte chunk c of
// row r at c ^ (r & 7)); otherwise by 16-byte cp.async chunks under the same swizzle
// of 256-byte rows.  Either way the ldmatrix reads are conflict-free.  q and K are
// both bf16, so S = K q^T runs on mma.sync bf16 with exact products; P V takes
// V^T through ldmatrix.trans and P split into bf16 hi + lo parts (4 query heads x
// {hi, lo} fill the 8 MMA columns).  Online softmax in the base-2 domain.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstring>

#include "oscar_internal.cuh"
#include "ptx.cuh"
#include "tma.cuh"

namespace oscar {
namespace {

constexpr int kCW = 8;
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kUnitBytes = 2 * kTileTokens * kHeadDim * 2;   // K then V rows of one (head, tile): 8 KB
constexpr int kStageBytes = kCW * kUnitBytes;                // one unit per consumer warp
constexpr int kStages = 3;

struct BfArgs {
    const uint16_t *q;
    Bf16PoolView pool;
    const int32_t *pt;
    int max_pages, page_size, n_kv, sink;
    const int32_t *seq_len, *hist_end;
    float scale2;
    PartialsView out;
    int mode;
    int32_t *status;
    int ws_bytes, stage_off;
};

__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

__device__ __forceinline__ __nv_bfloat16 split_bf16(float v, int part) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    return part ? __float2bfloat16_rn(v - __bfloat162float(h)) : h;
}

// The tiles one CTA visits.  mode 1: tiles of split s of [0, T).  mode 0: the sink
// tiles [0, ceil(min(sink, T)/16)) then the recent tiles from floor(h/16) to ceil(T/16).
struct Tiles {
    int n, first, n_sink, rec0;
    __device__ int tile(int k) const { return n_sink ? (k < n_sink ? k : rec0 + (k - n_sink)) : first + k; }
};

// TMA: mode 1 with 8 kv heads (a stage = one tile of every head, tensor-map boxes); tmk / tmv map
// the BF16 pool's K / V as [rows][8 heads][128 channels] bf16.
template <int G, bool TMA>
__global__ void __launch_bounds__(kThreads, 1)
    bf16_mma_kernel(BfArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    constexpr int NT = (G == 8) ? 2 : 1;
    constexpr int NCOL = 8 * NT;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // tensor-map boxes land on 1024-byte boundaries: the carve-up starts at an aligned address
    uint8_t *smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *stage0 = smem + a.stage_off;

    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = a.n_kv, Hq = Hkv * G, S = a.out.S;
    int T, he;
    read_lengths(a.seq_len, a.mode == 0 ? a.hist_end : nullptr, b, a.sink, a.max_pages * a.page_size, a.status,
                 T, he);
    // heads of this CTA: mode 0 one kv head (blockIdx.x), mode 1 all of them
    const int Hc = a.mode == 0 ? 1 : Hkv;
    const int h0 = a.mode == 0 ? blockIdx.x : 0;
    const int tps = kCW / Hc;                     // tiles per stage
    Tiles tl{0, 0, 0, 0};
    int lo0, hi0, lo1, hi1;                       // valid positions [lo0, hi0) U [lo1, hi1)
    if (a.mode == 0) {
        hi0 = min(a.sink, T);
        lo0 = 0;
        lo1 = max(he, hi0);
        hi1 = T;
        tl.n_sink = (hi0 + kTileTokens - 1) / kTileTokens;
        tl.rec0 = lo1 / kTileTokens;
        const int rec_n = lo1 < hi1 ? (hi1 + kTileTokens - 1) / kTileTokens - tl.rec0 : 0;
        tl.n = tl.n_sink + rec_n;
        if (tl.n_sink == 0) {                     // no sink tiles: list the recent ones directly
            tl.first = tl.rec0;
        }
    } else {
        const SplitRange r = full_split(T, S, blockIdx.x);
        lo0 = r.lo;
        hi0 = r.hi;
        lo1 = hi1 = 0;
        tl.first = r.tile_lo;
        tl.n = r.tile_hi - r.tile_lo;
    }
    const int n_iters = (tl.n + tps - 1) / tps;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(saddr(&bars[i]), TMA ? 1 : 32);   // TMA: the expect-tx arrival; else 32 cp.async
            mbar_init(saddr(&bars[4 + i]), kCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ------------------------------------------------------------ producer --
    if (warp == kCW) {
        int armed = 0;
        for (int it = 0; it < n_iters; ++it) {
            const int st = it % kStages;
            if (it >= kStages && !mbar_wait(saddr(&bars[4 + st]), ((it / kStages) - 1) & 1)) {
                if (lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
                break;
            }
            const uint32_t sb = saddr(stage0 + st * kStageBytes);
            if constexpr (TMA) {
                // one tile of all 8 heads: lane = 16 kind + 2 head + half (kind 0 K, 1 V) copies the box
                // of 16 rows x 64 channels of that head and half, to (kind, head, half) x 2 KB
                const int pos0 = tl.tile(it) * kTileTokens;
                const int page = a.pt[(size_t)b * a.max_pages + pos0 / a.page_size];
                const bool ok = page >= 0 && page < a.pool.n_pages;
                if (lane == 0) {
                    if (!ok) flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
                    mbar_arrive_expect_tx(saddr(&bars[st]), ok ? (uint32_t)kStageBytes : 0u);
                }
                armed = it + 1;
                __syncwarp();
                if (ok) {
                    const int row0 = page * a.page_size + pos0 % a.page_size;
                    const int kind = lane >> 4, head = (lane >> 1) & 7, half = lane & 1;
                    tma_load_3d(sb + lane * 2048, kind ? &tmv : &tmk, half * 64, head, row0, saddr(&bars[st]));
                }
                continue;
            }
            for (int u = 0; u < kCW; ++u) {
                const int k = it * tps + u / Hc;
                if (k >= tl.n) break;
                const int head = h0 + u % Hc;
                const int pos0 = tl.tile(k) * kTileTokens;
                const int page = a.pt[(size_t)b * a.max_pages + pos0 / a.page_size];
                if (page < 0 || page >= a.pool.n_pages) {
                    if (lane == 0 && u % Hc == 0) flag_status(a.status, OSCAR_DEV_BAD_BF16_PAGE);
                    continue;
                }
                const size_t row0 = (size_t)page * a.page_size + (pos0 % a.page_size);
                const uint8_t *srck = reinterpret_cast<const uint8_t *>(a.pool.k) + (row0 * Hkv + head) * 256;
                const uint8_t *srcv = reinterpret_cast<const uint8_t *>(a.pool.v) + (row0 * Hkv + head) * 256;
                const uint32_t dst = sb + u * kUnitBytes;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int c = lane + 32 * m, r = c >> 4, ch = c & 15;
                    const size_t so = (size_t)r * Hkv * 256 + ch * 16;
                    const uint32_t d = dst + r * 256 + ((ch ^ (r & 7)) << 4);
                    cp_async16(d, srck + so);
                    cp_async16(d + 4096, srcv + so);
                }
            }
            cp_async_arrive(saddr(&bars[st]));
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if constexpr (TMA) {
            // no copy may still be landing when the CTA leaves (see the INT2 kernel's copy warp)
            for (int k = armed > kStages ? armed - kStages : 0; k < armed; ++k)
                if (!mbar_wait(saddr(&bars[k % kStages]), (k / kStages) & 1) && lane == 0)
                    flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
        }
        return;
    }

    // ----------------------------------------------------------- consumers --
    const int hl = warp % Hc, sub = warp / Hc, nsub = kCW / Hc;
    const int h = h0 + hl;
    const int gid = lane >> 2, t = lane & 3;

    // B operand of S = K q^T: column 2j = query head j of the n-tile, column 2j+1 = 0.
    uint32_t bq[NT][8][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hh = nt * 4 + (gid >> 1);
        const bool valid = (gid & 1) == 0 && hh < G;
        const uint32_t *qr = reinterpret_cast<const uint32_t *>(a.q + ((size_t)b * Hq + h * G + (valid ? hh : 0)) * kHeadDim);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            bq[nt][ks][0] = valid ? qr[ks * 8 + t] : 0u;
            bq[nt][ks][1] = valid ? qr[ks * 8 + 4 + t] : 0u;
        }
    }
    __nv_bfloat16 *Ws = reinterpret_cast<__nv_bfloat16 *>(smem + 128 + warp * a.ws_bytes);

    float m_run[NT], l_run[NT];
    float oacc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt] = -INFINITY;
        l_run[nt] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) oacc[nt][mt][c] = 0.f;
    }
    // ldmatrix lane roles: QK A (rows = tokens), PV A = V^T (trans)
    const int qk_row = (lane & 7) + ((lane >> 3) & 1) * 8, qk_half = lane >> 4;
    const int pv_row = (lane & 7) + (lane >> 4) * 8, pv_half = (lane >> 3) & 1;

    for (int it = 0; it < n_iters; ++it) {
        const int st = it % kStages;
        if (!mbar_wait(saddr(&bars[st]), (it / kStages) & 1)) {
            if (lane == 0) flag_status(a.status, OSCAR_DEV_WAIT_TIMEOUT);
            break;
        }
        const int k = it * tps + sub;
        if (k < tl.n) {
            const int pos0 = tl.tile(k) * kTileTokens;
            const int page = a.pt[(size_t)b * a.max_pages + pos0 / a.page_size];
            if (page >= 0 && page < a.pool.n_pages) {
                // TMA: head h's boxes at (h * 2 + half) x 2 KB (K) and 32 KB further (V), rows of 128 bytes;
                // cp.async: this warp's unit, K rows of 256 bytes then V rows 4 KB further
                const uint32_t Kb = TMA ? saddr(stage0 + st * kStageBytes + h * 4096)
                                        : saddr(stage0 + st * kStageBytes + warp * kUnitBytes);
                const uint32_t Vb = Kb + (TMA ? 32768 : 4096);
                // 16-byte chunk ch (0..15) of row r: its address under either layout
                auto chunk_addr = [&](uint32_t base, int r, int ch) -> uint32_t {
                    return TMA ? base + (ch >> 3) * 2048 + r * 128 + (((ch & 7) ^ (r & 7)) << 4)
                               : base + r * 256 + ((ch ^ (r & 7)) << 4);
                };
                float sacc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sacc[nt][c] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    const int ch = 2 * ks + qk_half;
                    ldmatrix_x4(chunk_addr(Kb, qk_row, ch), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816_bf16(sacc[nt], a0, a1, a2, a3, bq[nt][ks][0], bq[nt][ks][1]);
                }
                const int p0 = pos0 + gid, p1 = pos0 + gid + 8;
                const bool v0 = (p0 >= lo0 && p0 < hi0) || (p0 >= lo1 && p0 < hi1);
                const bool v1 = (p1 >= lo0 && p1 < hi0) || (p1 >= lo1 && p1 < hi1);
                float alpha[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float t0 = v0 ? sacc[nt][0] * a.scale2 : -INFINITY;
                    const float t1 = v1 ? sacc[nt][2] * a.scale2 : -INFINITY;
                    float mx = fmaxf(t0, t1);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float mn = fmaxf(m_run[nt], mx);
                    float q0 = 0.f, q1 = 0.f, al = 1.f;
                    if (mn != -INFINITY) {
                        al = exp2f(m_run[nt] - mn);
                        q0 = exp2f(t0 - mn);
                        q1 = exp2f(t1 - mn);
                    }
                    alpha[nt] = al;
                    m_run[nt] = mn;
                    l_run[nt] = fmaf(l_run[nt], al, q0 + q1);
                    const int c_hi = nt * 8 + 2 * t;
                    Ws[c_hi * 16 + gid] = split_bf16(q0, 0);
                    Ws[(c_hi + 1) * 16 + gid] = split_bf16(q0, 1);
                    Ws[c_hi * 16 + gid + 8] = split_bf16(q1, 0);
                    Ws[(c_hi + 1) * 16 + gid + 8] = split_bf16(q1, 1);
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
                uint32_t bw[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const __nv_bfloat16 *col = Ws + (nt * 8 + gid) * 16;
                    bw[nt][0] = *reinterpret_cast<const uint32_t *>(col + 2 * t);
                    bw[nt][1] = *reinterpret_cast<const uint32_t *>(col + 2 * t + 8);
                }
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    const int ch = 2 * mt + pv_half;
                    ldmatrix_x4_trans(chunk_addr(Vb, pv_row, ch), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816_bf16(oacc[nt][mt], a0, a1, a2, a3, bw[nt][0], bw[nt][1]);
                }
                __syncwarp();
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(saddr(&bars[4 + st]));
    }

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], o);

    // output channels of thread (gid, t): 16*mt + gid (c0 + c1) and 16*mt + 8 + gid (c2 + c3)
    const int slot = a.mode == 0 ? S : blockIdx.x;
    const size_t S1 = (size_t)S + 1;
    if (nsub == 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = nt * 4 + t;
            if (hh < G) {
                const size_t row = ((size_t)b * Hq + h * G + hh) * S1 + slot;
                float *dst = a.out.acc + row * kHeadDim;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    dst[16 * mt + gid] = oacc[nt][mt][0] + oacc[nt][mt][1];
                    dst[16 * mt + 8 + gid] = oacc[nt][mt][2] + oacc[nt][mt][3];
                }
                if (gid == 0) {
                    a.out.m[row] = m_run[nt];
                    a.out.l[row] = l_run[nt];
                }
            }
        }
    } else {
        consumer_sync();
        float *cm = reinterpret_cast<float *>(stage0);
        float *cl = cm + kCW * NT * 4;
        float *ca = cl + kCW * NT * 4;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int e = warp * NT * 4 + nt * 4 + t;
            if (gid == 0) {
                cm[e] = m_run[nt];
                cl[e] = l_run[nt];
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                ca[e * kHeadDim + 16 * mt + gid] = oacc[nt][mt][0] + oacc[nt][mt][1];
                ca[e * kHeadDim + 16 * mt + 8 + gid] = oacc[nt][mt][2] + oacc[nt][mt][3];
            }
        }
        consumer_sync();
        if (sub == 0) {
            for (int e = lane; e < NT * 4 * kHeadDim / 4; e += 32) {
                const int sl = e / (kHeadDim / 4), c4 = (e % (kHeadDim / 4)) * 4;
                const int hh = sl;
                if (hh >= G) continue;
                float M = -INFINITY;
                for (int w = hl; w < kCW; w += Hc) M = fmaxf(M, cm[w * NT * 4 + sl]);
                float L = 0.f, A0 = 0.f, A1 = 0.f, A2 = 0.f, A3 = 0.f;
                if (M != -INFINITY) {
                    for (int w = hl; w < kCW; w += Hc) {
                        const float f = exp2f(cm[w * NT * 4 + sl] - M);
                        const float *src = ca + (w * NT * 4 + sl) * kHeadDim + c4;
                        L = fmaf(cl[w * NT * 4 + sl], f, L);
                        A0 = fmaf(src[0], f, A0);
                        A1 = fmaf(src[1], f, A1);
                        A2 = fmaf(src[2], f, A2);
                        A3 = fmaf(src[3], f, A3);
                    }
                }
                const size_t row = ((size_t)b * Hq + h * G + hh) * S1 + slot;
                *reinterpret_cast<float4 *>(a.out.acc + row * kHeadDim + c4) = make_float4(A0, A1, A2, A3);
                if (c4 == 0) {
                    a.out.m[row] = M;
                    a.out.l[row] = L;
                }
            }
        }
    }
    if (a.mode == 1 && blockIdx.x == 0) {
        // an all-BF16 cache has no history partial: slot S is empty
        for (int e = threadIdx.x; e < Hq * kHeadDim; e += kCW * 32) {
            const size_t row = ((size_t)b * Hq + e / kHeadDim) * S1 + S;
            a.out.acc[row * kHeadDim + e % kHeadDim] = 0.f;
            if (e % kHeadDim == 0) {
                a.out.m[row] = -INFINITY;
                a.out.l[row] = 0.f;
            }
        }
    }
}

// The BF16 pool's K or V, [rows = n_pages * page_size][8 heads][128 channels] bf16, as a 3-D tensor
// map whose box is 64 channels x 1 head x 16 rows (128-byte rows, 128-byte swizzle).
bool pool_tensor_map(CUtensorMap *tm, const uint16_t *base, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    const cuuint64_t dims[3] = {128, 8, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {256, 2048};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTileTokens};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_bf(BfArgs a, dim3 grid, cudaStream_t st) {
    constexpr int NT = (G == 8) ? 2 : 1;
    a.ws_bytes = 8 * NT * 16 * 2;
    // stages start 1024-byte aligned (tensor-map boxes with 128-byte swizzle); the kernel rounds the
    // dynamic shared memory base up to 1024 bytes
    a.stage_off = (128 + kCW * a.ws_bytes + 1023) & ~1023;
    const int combine = kCW * NT * 4 * (2 + kHeadDim) * 4;
    const int smem = 1024 + a.stage_off + (kStages * kStageBytes > combine ? kStages * kStageBytes : combine);
    const bool tma = a.mode == 1 && a.n_kv == 8;
    CUtensorMap tmk, tmv;
    memset(&tmk, 0, sizeof(tmk));
    memset(&tmv, 0, sizeof(tmv));
    if (tma) {
        const long long rows = (long long)a.pool.n_pages * a.page_size;
        if (!pool_tensor_map(&tmk, a.pool.k, rows) || !pool_tensor_map(&tmv, a.pool.v, rows)) return cudaErrorInvalidValue;
    }
    auto kern = tma ? bf16_mma_kernel<G, true> : bf16_mma_kernel<G, false>;
    if (cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(kern), smem)) return e;
    kern<<<grid, kThreads, smem, st>>>(a, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace

bool bf16_mma_supported(const oscar_layout_t &L, int mode) {
    const int H = L.n_kv_heads;
    return mode == 0 || H == 1 || H == 2 || H == 4 || H == 8;
}

cudaError_t launch_bf16_attention_mma(const oscar_layout_t &L, const uint16_t *q, Bf16PoolView pool,
                                      const int32_t *pt, int max_pages, const int32_t *seq_len,
                                      const int32_t *hist_end, int batch, float sm_scale, PartialsView out,
                                      int mode, int32_t *status, cudaStream_t st) {
    if (batch <= 0) return cudaSuccess;
    BfArgs a{};
    a.q = q;
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
    a.mode = mode;
    a.status = status;
    const dim3 grid(mode == 0 ? L.n_kv_heads : out.S, batch);
    switch (L.gqa) {
        case 1: return launch_bf<1>(a, grid, st);
        case 2: return launch_bf<2>(a, grid, st);
        case 4: return launch_bf<4>(a, grid, st);
        case 8: return launch_bf<8>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace oscar
