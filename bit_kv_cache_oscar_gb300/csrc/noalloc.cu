// Decode attention + merge in one call, for callers that cannot allocate
// device memory.
//
// oscar_decode_attention needs a caller-allocated partials buffer (scratch
// between the split kernels and the merge).  Some callers cannot provide one:
// code running inside a host framework that owns every device allocation and
// hands out no workspace, or a latency-critical loop that must never enter the
// allocator.  This entry point keeps the partials in a fixed device array that
// lives in this library instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds OSCAR_NOALLOC_SCRATCH_BYTES of it until the process exits
// (CUDA may load the library's device code, and reserve the array, when a
// device first uses it).  Host code cannot use the variable's name as a device
// address, so every call looks the address up on the current device with
// cudaGetSymbolAddress (a host-side query, no allocation once the code is
// loaded; looking it up each time also survives a device reset).  All calls
// share the array, so calls whose work overlaps on the GPU (different streams,
// or different host threads on one stream order) race on it and must be
// serialised by the caller.

#include "oscar_internal.cuh"

namespace {

constexpr size_t kScratchFloats = OSCAR_NOALLOC_SCRATCH_BYTES / sizeof(float);

__device__ __align__(256) float g_noalloc_partials[kScratchFloats];

// Device address of g_noalloc_partials on the current device.
oscar_status_t scratch_address(float **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_partials);
    if (e != cudaSuccess || !p)
        return oscar::set_last_error(OSCAR_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
    *out = static_cast<float *>(p);
    return OSCAR_OK;
}

}  // namespace

extern "C" oscar_status_t oscar_decode_attention_noalloc(
    const oscar_layout_t *layout, const uint16_t *q, const float *q_rot, const oscar_bf16_pool_t *bf16_pool,
    const int32_t *bf16_page_table, const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
    int32_t max_pages_per_req, const int32_t *seq_len, const int32_t *hist_end, int32_t batch, float sm_scale,
    int32_t n_splits, const float *R_V, uint16_t *out, float *out_f32, float *lse, void *stream) {
    if (!layout) return oscar::set_last_error(OSCAR_ERR_INVALID_ARG, "layout is NULL");
    if (batch < 0 || n_splits < 1 || n_splits > 1024)
        return oscar::set_last_error(OSCAR_ERR_INVALID_ARG, "batch < 0 or n_splits outside 1..1024");
    if (batch == 0) return OSCAR_OK;
    const size_t ml = oscar_partials_ml_floats(layout, batch, n_splits);
    const size_t acc = oscar_partials_acc_floats(layout, batch, n_splits);
    // m and l each padded to 64 floats (256 bytes) so that acc starts 256-byte aligned.
    const size_t ml_pad = (ml + 63) / 64 * 64;
    if (2 * ml_pad + acc > kScratchFloats)
        return oscar::set_last_error(
            OSCAR_ERR_INVALID_ARG,
            "batch x query heads x (n_splits + 1) too large for the no-alloc scratch "
            "(needs (2*ceil64(B*Hq*(S+1)) + B*Hq*(S+1)*head_dim) floats <= OSCAR_NOALLOC_SCRATCH_BYTES/4)");
    float *base = nullptr;
    oscar_status_t st = scratch_address(&base);
    if (st != OSCAR_OK) return st;
    oscar_partials_t part;
    part.m = base;
    part.l = base + ml_pad;
    part.acc = base + 2 * ml_pad;
    part.n_splits = n_splits;
    st = oscar_decode_attention(layout, q, q_rot, bf16_pool, bf16_page_table, int2_pool, int2_page_table,
                                max_pages_per_req, seq_len, hist_end, batch, sm_scale, &part, stream);
    if (st != OSCAR_OK) return st;
    return oscar_merge(layout, &part, R_V, batch, out, out_f32, lse, stream);
}
