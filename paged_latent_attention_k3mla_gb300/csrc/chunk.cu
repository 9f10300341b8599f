// chunk.cu -- many new tokens per slot per call (chunked prefill).
//
// pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode": the PR's
// follow-up list queues chunked prefill, which replaces the token-by-token loop
// over a prompt.  A chunk of n_b new tokens of slot b occupies positions
// pos0[b] .. pos0[b] + n_b - 1.  Two calls serve it:
//   * k3mla_append_latent_rows writes all the chunk's latent rows into their
//     mapped pages (the M1 commit's indexed row write, one row per token);
//   * k3mla_chunk_views gives every query token j of the chunk its own view of
//     the slot: the slot's block table row and a context of pos0[b] + j + 1
//     tokens.  That context IS the causal mask within the chunk: query j sees the
//     rows before the chunk and the chunk's rows 0..j, never the later ones.  The
//     paged decode then runs over the views unchanged (one view per query), its
//     result for view (b, j) the attention output of token pos0[b] + j.
// Rows of a slot are packed: slot b's rows are rows row_start[b] ..
// row_start[b + 1] - 1 of the c_kv / k_rope inputs and of the views.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int AR_ROWS = 8;       // rows per CTA of the row append
constexpr int AR_THREADS = 96;   // a row is 288 32-bit words: three per thread

// grid (B, ceil(max_rows / AR_ROWS)); block AR_THREADS.
__global__ void __launch_bounds__(AR_THREADS) k3mla_append_rows_kernel(
    uint16_t* __restrict__ slab, int n_pages, int n_layers, int layer, const int32_t* __restrict__ table,
    int max_pages, const int32_t* __restrict__ pos0, const int32_t* __restrict__ row_start,
    const uint16_t* __restrict__ c_kv, int64_t c_stride, const uint16_t* __restrict__ k_rope, int64_t r_stride,
    int32_t* dev_err)
{
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x;
    const int r0 = row_start[b], n = row_start[b + 1] - r0, p0 = pos0[b];
    for (int k = 0; k < AR_ROWS; ++k) {
        const int j = blockIdx.y * AR_ROWS + k;
        if (j >= n) break;
        const int p = p0 + j;
        const int lp = p / PAGE;
        const int32_t id = (p >= 0 && lp < max_pages) ? table[(size_t)b * max_pages + lp] : -1;
        if (id < 0 || id >= n_pages) {
            if (threadIdx.x == 0 && dev_err) atomicOr(dev_err, (int)K3MLA_DEV_UNMAPPED);
            continue;
        }
        const size_t row = ((size_t)id * (size_t)n_layers + (size_t)layer) * PAGE + (size_t)(p % PAGE);
        uint32_t* dst = reinterpret_cast<uint32_t*>(slab + row * ROW);
        const uint32_t* src_c = reinterpret_cast<const uint32_t*>(c_kv + (size_t)(r0 + j) * c_stride);
        const uint32_t* src_r = reinterpret_cast<const uint32_t*>(k_rope + (size_t)(r0 + j) * r_stride);
        for (int i = threadIdx.x; i < ROW / 2; i += AR_THREADS)
            dst[i] = (i < LORA / 2) ? src_c[i] : src_r[i - LORA / 2];
    }
}

// grid (R); block 128.  View r belongs to the slot b with row_start[b] <= r < row_start[b + 1].
__global__ void __launch_bounds__(128) k3mla_chunk_views_kernel(const int32_t* __restrict__ table, int B,
                                                               int max_pages, const int32_t* __restrict__ pos0,
                                                               const int32_t* __restrict__ row_start,
                                                               int32_t* __restrict__ vtable, int32_t* __restrict__ vctx)
{
    griddep_wait();
    griddep_launch_dependents();
    const int r = blockIdx.x;
    int lo = 0, hi = B;  // the last b with row_start[b] <= r (row_start is non-decreasing)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (row_start[mid] <= r) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    const bool inside = r >= row_start[b] && r < row_start[b + 1];
    if (threadIdx.x == 0) vctx[r] = inside ? pos0[b] + (r - row_start[b]) + 1 : 0;
    for (int i = threadIdx.x; i < max_pages; i += blockDim.x)
        vtable[(size_t)r * max_pages + i] = inside ? table[(size_t)b * max_pages + i] : -1;
}

}  // namespace k3

using namespace k3;

extern "C" int k3mla_append_latent_rows(uint16_t* slab, int n_pages, int n_layers, int layer,
                                        const int32_t* block_table, int max_pages_per_slot, const int32_t* pos0,
                                        const int32_t* row_start, const uint16_t* c_kv, int64_t c_stride,
                                        const uint16_t* k_rope, int64_t r_stride, int B, int max_rows,
                                        int32_t* dev_err, void* stream)
{
    if (B < 0 || max_rows < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers ||
        max_pages_per_slot <= 0 || c_stride < LORA || r_stride < ROPE || (c_stride & 1) || (r_stride & 1)) {
        set_error("k3mla_append_latent_rows: invalid sizes or strides");
        return K3MLA_E_INVALID;
    }
    if (B == 0 || max_rows == 0) return K3MLA_OK;
    if (!slab || !block_table || !pos0 || !row_start || !c_kv || !k_rope || !aligned(slab, 4) ||
        !aligned(c_kv, 4) || !aligned(k_rope, 4)) {
        set_error("k3mla_append_latent_rows: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    const int gy = (max_rows + AR_ROWS - 1) / AR_ROWS;
    if (gy > 65535) {
        set_error("k3mla_append_latent_rows: max_rows too large");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    return launch_pdl(k3mla_append_rows_kernel, dim3(B, gy), dim3(AR_THREADS), 0,
                      reinterpret_cast<cudaStream_t>(stream), "k3mla_append_rows_kernel", slab, n_pages, n_layers,
                      layer, block_table, max_pages_per_slot, pos0, row_start, c_kv, c_stride, k_rope, r_stride,
                      dev_err);
}

extern "C" int k3mla_chunk_views(const int32_t* block_table, int B, int max_pages_per_slot, const int32_t* pos0,
                                 const int32_t* row_start, int R, int32_t* view_table, int32_t* view_ctx,
                                 void* stream)
{
    if (B <= 0 || R < 0 || max_pages_per_slot <= 0) {
        set_error("k3mla_chunk_views: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if (R == 0) return K3MLA_OK;
    if (!block_table || !pos0 || !row_start || !view_table || !view_ctx) {
        set_error("k3mla_chunk_views: null pointer");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    return launch_pdl(k3mla_chunk_views_kernel, dim3(R), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                      "k3mla_chunk_views_kernel", block_table, B, max_pages_per_slot, pos0, row_start, view_table,
                      view_ctx);
}
