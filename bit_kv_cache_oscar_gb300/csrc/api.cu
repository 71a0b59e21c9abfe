// C ABI of liboscar.so: argument validation, the device status word, dispatch
// to the kernels.  Declarations and contracts: include/oscar.h.

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "oscar_internal.cuh"

namespace {

thread_local std::string g_last_error = "no error";

oscar_status_t fail(oscar_status_t code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
oscar_status_t fail(oscar_status_t code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

oscar_status_t cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return OSCAR_OK;
    return fail(OSCAR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device status word (one per device that loads the library); kernels get its address.
__device__ int32_t g_device_status;

constexpr int kMaxDevices = 64;
int32_t *g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_status_mu;

int32_t *status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int32_t *>(p);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

oscar_status_t check_layout(const oscar_layout_t *L) {
    if (!L) return fail(OSCAR_ERR_INVALID_ARG, "layout is NULL");
    if (L->head_dim != 128) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d: only 128 is supported", L->head_dim);
    if (L->n_kv_heads < 1 || L->n_kv_heads > 64)
        return fail(OSCAR_ERR_UNSUPPORTED, "n_kv_heads %d outside 1..64", L->n_kv_heads);
    if (L->gqa != 1 && L->gqa != 2 && L->gqa != 4 && L->gqa != 8)
        return fail(OSCAR_ERR_UNSUPPORTED, "gqa %d: supported 1, 2, 4, 8", L->gqa);
    if (L->page_size != 16 && L->page_size != 32 && L->page_size != 64)
        return fail(OSCAR_ERR_UNSUPPORTED, "page_size %d: supported 16, 32, 64", L->page_size);
    if (L->group != 32 && L->group != 64 && L->group != 128)
        return fail(OSCAR_ERR_UNSUPPORTED, "group %d: supported 32, 64, 128", L->group);
    if (L->sink < 0 || L->sink % L->page_size != 0)
        return fail(OSCAR_ERR_INVALID_ARG, "sink %d must be >= 0 and a multiple of page_size %d", L->sink,
                    L->page_size);
    if (L->recent < 0) return fail(OSCAR_ERR_INVALID_ARG, "recent %d < 0", L->recent);
    if (!oscar::uniform_codebook(*L)) {
        for (const float *lv : {L->levels_k, L->levels_v})
            for (int k = 0; k < 4; ++k)
                if (!std::isfinite(lv[k]) || (k > 0 && !(lv[k] > lv[k - 1])))
                    return fail(OSCAR_ERR_INVALID_ARG, "codebook levels must be finite and strictly increasing");
    }
    return OSCAR_OK;
}

oscar_status_t check_int2_pool(const oscar_int2_pool_t *p) {
    if (!p) return fail(OSCAR_ERR_INVALID_ARG, "INT2 pool is NULL");
    const void *ptrs[6] = {p->codes_k, p->codes_v, p->scale_k, p->zero_k, p->scale_v, p->zero_v};
    for (const void *q : ptrs) {
        if (!q) return fail(OSCAR_ERR_INVALID_ARG, "INT2 pool has a NULL array");
        if (!aligned16(q)) return fail(OSCAR_ERR_INVALID_ARG, "INT2 pool array not 16-byte aligned");
    }
    if (p->n_pages < 1) return fail(OSCAR_ERR_INVALID_ARG, "INT2 pool n_pages %d < 1", p->n_pages);
    return OSCAR_OK;
}

oscar_status_t check_bf16_pool(const oscar_bf16_pool_t *p) {
    if (!p) return fail(OSCAR_ERR_INVALID_ARG, "BF16 pool is NULL");
    if (!p->k || !p->v) return fail(OSCAR_ERR_INVALID_ARG, "BF16 pool has a NULL array");
    if (!aligned16(p->k) || !aligned16(p->v)) return fail(OSCAR_ERR_INVALID_ARG, "BF16 pool not 16-byte aligned");
    if (p->n_pages < 1) return fail(OSCAR_ERR_INVALID_ARG, "BF16 pool n_pages %d < 1", p->n_pages);
    return OSCAR_OK;
}

oscar_status_t check_partials(const oscar_partials_t *p) {
    if (!p) return fail(OSCAR_ERR_INVALID_ARG, "partials is NULL");
    if (!p->m || !p->l || !p->acc) return fail(OSCAR_ERR_INVALID_ARG, "partials has a NULL array");
    if (!aligned16(p->acc)) return fail(OSCAR_ERR_INVALID_ARG, "partials acc not 16-byte aligned");
    if (p->n_splits < 1 || p->n_splits > 1024)
        return fail(OSCAR_ERR_INVALID_ARG, "n_splits %d outside 1..1024", p->n_splits);
    return OSCAR_OK;
}

#define TRY(x)                                \
    do {                                      \
        oscar_status_t s_ = (x);              \
        if (s_ != OSCAR_OK) return s_;        \
    } while (0)

oscar::Int2PoolView int2_view(const oscar_int2_pool_t *p) {
    return {p->codes_k, p->codes_v, p->scale_k, p->zero_k, p->scale_v, p->zero_v, p->n_pages};
}
oscar::Bf16PoolView bf16_view(const oscar_bf16_pool_t *p) { return {p->k, p->v, p->n_pages}; }
oscar::PartialsView part_view(const oscar_partials_t *p) { return {p->m, p->l, p->acc, p->n_splits}; }

}  // namespace

oscar_status_t oscar::set_last_error(oscar_status_t code, const char *msg) { return fail(code, "%s", msg); }

namespace {
std::atomic<int> g_overlap{0};
}  // namespace

bool oscar::launch_overlap() { return g_overlap.load(std::memory_order_relaxed) != 0; }

namespace {
struct SmemLimit {
    const void *kern;
    int dev, bytes;
};
std::mutex g_smem_mu;
SmemLimit g_smem[256];
int g_n_smem = 0;
}  // namespace

cudaError_t oscar::ensure_dyn_smem(const void *kern, int smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_smem_mu);
    int k = 0;
    while (k < g_n_smem && !(g_smem[k].kern == kern && g_smem[k].dev == dev)) ++k;
    if (k < g_n_smem && g_smem[k].bytes >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (k == g_n_smem) {
        if (g_n_smem == 256) return cudaSuccess;        // untracked: set again next time
        g_smem[g_n_smem++] = {kern, dev, smem};
    } else {
        g_smem[k].bytes = smem;
    }
    return cudaSuccess;
}

extern "C" {

size_t oscar_partials_ml_floats(const oscar_layout_t *L, int32_t batch, int32_t n_splits) {
    if (!L || batch < 0 || n_splits < 0) return 0;
    return (size_t)batch * L->n_kv_heads * L->gqa * (size_t)(n_splits + 1);
}

size_t oscar_partials_acc_floats(const oscar_layout_t *L, int32_t batch, int32_t n_splits) {
    return oscar_partials_ml_floats(L, batch, n_splits) * (L ? (size_t)L->head_dim : 0);
}

int32_t oscar_suggest_splits(const oscar_layout_t *L, int32_t batch, int32_t max_hist_tokens, int32_t sm_count) {
    if (!L || L->page_size <= 0 || batch <= 0 || sm_count <= 0) return 1;
    const int tiles = (max_hist_tokens + 15) / 16;
    long want;
    int active = 0;
    if (oscar::int2_mma_supported(*L)) {
        // one split = a cluster of C CTAs (all kv heads each): as many splits as clusters fit at once
        // (one or two more clusters per request take the BF16 window).  When the batch's clusters
        // cannot run in one wave anyway, about four waves of clusters: the requests' lengths may
        // differ, and small clusters queued behind the first wave even out the SMs' finishing times.
        const int c = oscar::int2_mma_cluster_size(*L, &active);
        if (active <= 0) active = (2 * sm_count) / c;
        const int win = oscar::int2_mma_window_clusters(*L, batch);
        want = (long)batch * (1 + win) > active ? (4L * active) / batch - win : active / batch - win;
    } else {
        // one 4-warp CTA per (split, kv head): about sixteen CTAs per SM (their warps take one
        // token at a time and need many warps in flight; 100K tokens, 8 kv heads: 1152, 641 and
        // 484 us per layer at 38, 152 and 304 splits)
        want = (16L * sm_count + (long)batch * L->n_kv_heads - 1) / ((long)batch * L->n_kv_heads);
    }
    if (want > tiles) want = tiles;
    if (want < 1) want = 1;
    if (want > 1024) want = 1024;
    return (int32_t)want;
}

oscar_status_t oscar_demote(const oscar_layout_t *layout, const oscar_bf16_pool_t *src,
                            const int32_t *bf16_page_table, const oscar_int2_pool_t *dst,
                            const int32_t *int2_page_table, int32_t max_pages_per_req, int32_t batch,
                            const int32_t *req_idx,
                            const int32_t *positions, int32_t n, const float *R_K, const float *R_V, float c_K,
                            float c_V, float *rotated_out, void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(src));
    TRY(check_int2_pool(dst));
    if (n < 0 || n > 65535 * 256) return fail(OSCAR_ERR_INVALID_ARG, "n %d outside 0..%d", n, 65535 * 256);
    if (n == 0) return OSCAR_OK;
    if (!bf16_page_table || !int2_page_table || !req_idx || !positions || !R_K)
        return fail(OSCAR_ERR_INVALID_ARG, "NULL page table, index or R_K");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    if (batch < 1) return fail(OSCAR_ERR_INVALID_ARG, "batch %d < 1", batch);
    if (!aligned16(R_K) || !aligned16(R_V)) return fail(OSCAR_ERR_INVALID_ARG, "R_K/R_V not 16-byte aligned");
    if (!(c_K > 0.0f) || !(c_V > 0.0f)) return fail(OSCAR_ERR_INVALID_ARG, "clip ratios must be > 0");
    return cuda_status(oscar::launch_demote(*layout, bf16_view(src), bf16_page_table, *dst, int2_page_table,
                                            max_pages_per_req, batch, req_idx, positions, n, R_K, R_V, c_K, c_V,
                                            rotated_out, status_ptr(), (cudaStream_t)stream),
                       "oscar_demote launch");
}

oscar_status_t oscar_demote_range(const oscar_layout_t *layout, const oscar_bf16_pool_t *src,
                                  const int32_t *bf16_page_table, const oscar_int2_pool_t *dst,
                                  const int32_t *int2_page_table, int32_t max_pages_per_req, int32_t batch,
                                  const int32_t *pos_begin, const int32_t *pos_end, const float *R_K,
                                  const float *R_V, float c_K, float c_V, float *rotated_out, void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(src));
    TRY(check_int2_pool(dst));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!bf16_page_table || !int2_page_table || !pos_begin || !pos_end || !R_K)
        return fail(OSCAR_ERR_INVALID_ARG, "NULL page table, range or R_K");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    if (!(c_K > 0.0f) || !(c_V > 0.0f)) return fail(OSCAR_ERR_INVALID_ARG, "clip ratios must be > 0");
    if (!aligned16(src->k) || !aligned16(src->v) || !aligned16(dst->codes_k) || !aligned16(dst->codes_v) ||
        !aligned16(rotated_out))
        return fail(OSCAR_ERR_INVALID_ARG, "pool arrays and rotated_out must be 16-byte aligned");
    if (!oscar::demote_range_supported(*layout))
        return fail(OSCAR_ERR_UNSUPPORTED, "page_size %d neither divides nor is a multiple of 128",
                    layout->page_size);
    if (!oscar::uniform_codebook(*layout))
        return fail(OSCAR_ERR_UNSUPPORTED, "the tensor-core bulk demotion quantizes to the uniform levels only; "
                                           "use oscar_demote");
    return cuda_status(oscar::launch_demote_range(*layout, bf16_view(src), bf16_page_table, *dst, int2_page_table,
                                                  max_pages_per_req, batch, pos_begin, pos_end, R_K, R_V, c_K, c_V,
                                                  rotated_out, status_ptr(), (cudaStream_t)stream),
                       "oscar_demote_range launch");
}

oscar_status_t oscar_quantize_rotated(const oscar_layout_t *layout, const float *x_rot, int32_t n, float clip,
                                      uint8_t *codes, uint16_t *scale, uint16_t *zero, void *stream) {
    TRY(check_layout(layout));
    if (n < 0 || n > 2147483647 / 128) return fail(OSCAR_ERR_INVALID_ARG, "n %d out of range", n);
    if (n == 0) return OSCAR_OK;
    if (!x_rot || !codes || !scale || !zero) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (!(clip > 0.0f)) return fail(OSCAR_ERR_INVALID_ARG, "clip must be > 0");
    return cuda_status(oscar::launch_quantize_rotated(*layout, x_rot, n, clip, codes, scale, zero,
                                                      (cudaStream_t)stream),
                       "oscar_quantize_rotated launch");
}

oscar_status_t oscar_rotate_q(const oscar_layout_t *layout, const uint16_t *q, const float *R_K, int32_t batch,
                              float *q_rot, void *stream) {
    TRY(check_layout(layout));
    if (batch < 0) return fail(OSCAR_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q || !R_K || !q_rot) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    return cuda_status(oscar::launch_rotate_q(*layout, q, R_K, batch, q_rot, (cudaStream_t)stream),
                       "oscar_rotate_q launch");
}

oscar_status_t oscar_decode_attention(const oscar_layout_t *layout, const uint16_t *q, const float *q_rot,
                                      const oscar_bf16_pool_t *bf16_pool, const int32_t *bf16_page_table,
                                      const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
                                      int32_t max_pages_per_req, const int32_t *seq_len, const int32_t *hist_end,
                                      int32_t batch, float sm_scale, const oscar_partials_t *partials,
                                      void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(bf16_pool));
    TRY(check_int2_pool(int2_pool));
    TRY(check_partials(partials));
    if (batch < 0) return fail(OSCAR_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q || !q_rot || !bf16_page_table || !int2_page_table || !seq_len || !hist_end)
        return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (!aligned16(q_rot) || !aligned16(q)) return fail(OSCAR_ERR_INVALID_ARG, "q/q_rot not 16-byte aligned");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    if (batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d > 65535", batch);
    int32_t *st = status_ptr();
    cudaStream_t s = (cudaStream_t)stream;
    if (oscar::int2_mma_supported(*layout))   // history splits and window in one launch
        return cuda_status(oscar::launch_decode_mma(*layout, q_rot, nullptr, int2_view(int2_pool), int2_page_table, q,
                                                    bf16_view(bf16_pool), bf16_page_table, max_pages_per_req,
                                                    seq_len, hist_end, batch, sm_scale, part_view(partials), st,
                                                    true, true, s),
                           "decode attention launch");
    cudaError_t e = oscar::launch_int2_attention(*layout, q_rot, int2_view(int2_pool), int2_page_table,
                                                 max_pages_per_req, seq_len, hist_end, batch, sm_scale,
                                                 part_view(partials), st, s);
    if (e != cudaSuccess) return cuda_status(e, "INT2 attention launch");
    e = oscar::launch_bf16_attention(*layout, q, bf16_view(bf16_pool), bf16_page_table, max_pages_per_req,
                                     seq_len, hist_end, batch, sm_scale, part_view(partials), 0, st, s);
    return cuda_status(e, "BF16 sink/recent attention launch");
}

oscar_status_t oscar_decode_attention_shared_prefix(
    const oscar_layout_t *layout, const uint16_t *q, const float *q_rot, const oscar_bf16_pool_t *bf16_pool,
    const int32_t *bf16_page_table, const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
    int32_t max_pages_per_req, const int32_t *seq_len, const int32_t *hist_end, int32_t batch, float sm_scale,
    int32_t prefix_end, int32_t prefix_splits, const oscar_partials_t *partials, int32_t *tile_counters,
    void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(bf16_pool));
    TRY(check_int2_pool(int2_pool));
    TRY(check_partials(partials));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q || !q_rot || !bf16_page_table || !int2_page_table || !seq_len || !hist_end)
        return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (!aligned16(q_rot) || !aligned16(q)) return fail(OSCAR_ERR_INVALID_ARG, "q/q_rot not 16-byte aligned");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    if (!oscar::int2_mma_supported(*layout) || layout->group != 128)
        return fail(OSCAR_ERR_UNSUPPORTED, "the shared-prefix path needs 1, 2, 4 or 8 kv heads, the uniform "
                                           "codebook and group 128");
    if (prefix_end % 16 != 0 || prefix_end <= layout->sink ||
        (long long)prefix_end > (long long)max_pages_per_req * layout->page_size)
        return fail(OSCAR_ERR_INVALID_ARG, "prefix_end %d: a multiple of 16 in (sink, max_pages_per_req*page_size]",
                    prefix_end);
    if (prefix_splits < 1 || prefix_splits >= partials->n_splits)
        return fail(OSCAR_ERR_INVALID_ARG, "prefix_splits %d outside 1..n_splits-1 (%d)", prefix_splits,
                    partials->n_splits - 1);
    int32_t *st = status_ptr();
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = oscar::launch_prefix_attention(*layout, q_rot, int2_view(int2_pool), int2_page_table, prefix_end,
                                                   batch, prefix_splits, sm_scale, part_view(partials), st, s);
    if (e != cudaSuccess) return cuda_status(e, "shared-prefix attention launch");
    return cuda_status(oscar::launch_decode_mma_suffix(*layout, q_rot, int2_view(int2_pool), int2_page_table, q,
                                                       bf16_view(bf16_pool), bf16_page_table, max_pages_per_req,
                                                       seq_len, hist_end, batch, sm_scale, part_view(partials), st,
                                                       prefix_end, prefix_splits, tile_counters, s),
                       "suffix attention launch");
}

oscar_status_t oscar_decode_attention_fused(const oscar_layout_t *layout, const uint16_t *q, const float *R_K,
                                            const oscar_bf16_pool_t *bf16_pool, const int32_t *bf16_page_table,
                                            const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
                                            int32_t max_pages_per_req, const int32_t *seq_len,
                                            const int32_t *hist_end, int32_t batch, float sm_scale,
                                            const oscar_partials_t *partials, const int32_t *demote_pos,
                                            const float *R_V, float c_K, float c_V, uint16_t *out,
                                            float *out_f32, float *lse, int32_t *merge_counters,
                                            int32_t *tile_counters, void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(bf16_pool));
    TRY(check_int2_pool(int2_pool));
    TRY(check_partials(partials));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q || !R_K || !bf16_page_table || !int2_page_table || !seq_len || !hist_end)
        return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (!aligned16(q) || !aligned16(R_K)) return fail(OSCAR_ERR_INVALID_ARG, "q/R_K not 16-byte aligned");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    if (!oscar::int2_mma_supported(*layout))
        return fail(OSCAR_ERR_UNSUPPORTED, "fused rotation needs 1, 2, 4 or 8 kv heads and the uniform codebook; "
                                           "use oscar_rotate_q + "
                                           "oscar_decode_attention");
    oscar::FusedDemotion dem{};
    if (!aligned16(R_V)) return fail(OSCAR_ERR_INVALID_ARG, "R_V not 16-byte aligned");
    if (demote_pos) {
        dem.dem_pos = demote_pos;
        dem.RV = R_V;
        dem.cK = c_K;
        dem.cV = c_V;
        dem.dst = {int2_pool->codes_k, int2_pool->codes_v, int2_pool->scale_k, int2_pool->zero_k,
                   int2_pool->scale_v, int2_pool->zero_v, int2_pool->n_pages};
    }
    const bool merge = out || out_f32;
    int32_t *arrivals = merge && merge_counters ? merge_counters : nullptr;
    int clusters = 0;
    cudaError_t e = oscar::launch_decode_mma_demote(*layout, R_K, int2_view(int2_pool), int2_page_table, q,
                                                    bf16_view(bf16_pool), bf16_page_table, max_pages_per_req,
                                                    seq_len, hist_end, batch, sm_scale, part_view(partials),
                                                    status_ptr(), dem, arrivals, &clusters, tile_counters,
                                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e, "fused decode attention launch");
    if (merge)
        return cuda_status(oscar::launch_merge(*layout, part_view(partials), R_V, batch, out, out_f32, lse,
                                               (cudaStream_t)stream, arrivals, clusters, status_ptr()),
                           "oscar_merge launch");
    return OSCAR_OK;
}

oscar_status_t oscar_decode_attention_history(const oscar_layout_t *layout, const float *q_rot,
                                              const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
                                              int32_t max_pages_per_req, const int32_t *seq_len,
                                              const int32_t *hist_end, int32_t batch, float sm_scale,
                                              const oscar_partials_t *partials, void *stream) {
    TRY(check_layout(layout));
    TRY(check_int2_pool(int2_pool));
    TRY(check_partials(partials));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q_rot || !int2_page_table || !seq_len || !hist_end) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (!aligned16(q_rot)) return fail(OSCAR_ERR_INVALID_ARG, "q_rot not 16-byte aligned");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    return cuda_status(oscar::launch_int2_attention(*layout, q_rot, int2_view(int2_pool), int2_page_table,
                                                    max_pages_per_req, seq_len, hist_end, batch, sm_scale,
                                                    part_view(partials), status_ptr(), (cudaStream_t)stream),
                       "INT2 attention launch");
}

oscar_status_t oscar_decode_attention_window(const oscar_layout_t *layout, const uint16_t *q,
                                             const oscar_bf16_pool_t *bf16_pool, const int32_t *bf16_page_table,
                                             int32_t max_pages_per_req, const int32_t *seq_len,
                                             const int32_t *hist_end, int32_t batch, float sm_scale,
                                             const oscar_partials_t *partials, void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(bf16_pool));
    TRY(check_partials(partials));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q || !bf16_page_table || !seq_len || !hist_end) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    return cuda_status(oscar::launch_bf16_attention(*layout, q, bf16_view(bf16_pool), bf16_page_table,
                                                    max_pages_per_req, seq_len, hist_end, batch, sm_scale,
                                                    part_view(partials), 0, status_ptr(), (cudaStream_t)stream),
                       "BF16 sink/recent attention launch");
}

oscar_status_t oscar_merge(const oscar_layout_t *layout, const oscar_partials_t *partials, const float *R_V,
                           int32_t batch, uint16_t *out, float *out_f32, float *lse, void *stream) {
    TRY(check_layout(layout));
    TRY(check_partials(partials));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!out && !out_f32) return fail(OSCAR_ERR_INVALID_ARG, "out and out_f32 are both NULL");
    return cuda_status(oscar::launch_merge(*layout, part_view(partials), R_V, batch, out, out_f32, lse,
                                           (cudaStream_t)stream),
                       "oscar_merge launch");
}

oscar_status_t oscar_bf16_decode_attention(const oscar_layout_t *layout, const uint16_t *q,
                                           const oscar_bf16_pool_t *pool, const int32_t *page_table,
                                           int32_t max_pages_per_req, const int32_t *seq_len, int32_t batch,
                                           float sm_scale, const oscar_partials_t *partials, void *stream) {
    TRY(check_layout(layout));
    TRY(check_bf16_pool(pool));
    TRY(check_partials(partials));
    if (batch < 0 || batch > 65535) return fail(OSCAR_ERR_INVALID_ARG, "batch %d outside 0..65535", batch);
    if (batch == 0) return OSCAR_OK;
    if (!q || !page_table || !seq_len) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (max_pages_per_req < 1) return fail(OSCAR_ERR_INVALID_ARG, "max_pages_per_req %d < 1", max_pages_per_req);
    return cuda_status(oscar::launch_bf16_attention(*layout, q, bf16_view(pool), page_table, max_pages_per_req,
                                                    seq_len, nullptr, batch, sm_scale, part_view(partials), 1,
                                                    status_ptr(), (cudaStream_t)stream),
                       "BF16 attention launch");
}

oscar_status_t oscar_get_device_status(int32_t *status_bits, void *stream) {
    if (!status_bits) return fail(OSCAR_ERR_INVALID_ARG, "status_bits is NULL");
    int32_t *p = status_ptr();
    if (!p) return fail(OSCAR_ERR_CUDA, "device status word unavailable");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(status_bits, p, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e, "reading device status");
}

const char *oscar_last_error_string(void) { return g_last_error.c_str(); }

const char *oscar_version(void) { return "0.1.0"; }

oscar_status_t oscar_set_launch_overlap(int32_t enabled) {
    g_overlap.store(enabled ? 1 : 0, std::memory_order_relaxed);
    return OSCAR_OK;
}

int32_t oscar_get_launch_overlap(void) { return g_overlap.load(std::memory_order_relaxed); }

}  // extern "C"
