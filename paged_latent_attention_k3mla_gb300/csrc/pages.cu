// pages.cu -- whole-page copies between page-first slabs.
//
// pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M1 commit: a
// prefilled sequence is adopted into a decode slot by copying its pages whole.
// In the page-first slab [page][layer][64][576] bf16 a page is one contiguous
// block of n_layers * 64 * 576 elements (every layer's rows of those 64 tokens),
// so adopting a page, or un-sharing a page that two slots map (copy on write),
// is one contiguous block copy.  The copy is HBM-bound (read + write of
// n_layers * 73,728 bytes per page); each CTA moves 16-byte vectors, eight in
// flight per thread, over one page of one (src, dst) pair.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int CP_THREADS = 256;
constexpr int CP_VEC = 8;  // 16-byte vectors in flight per thread

// grid (chunks of a page, pairs); block CP_THREADS.  A pair with an id outside its slab is skipped
// and flagged (K3MLA_DEV_BAD_PAGE, once per pair by the first CTA of the pair).
__global__ void __launch_bounds__(CP_THREADS) k3mla_copy_pages_kernel(uint16_t* __restrict__ dst_slab, int dst_n_pages,
                                                                      const uint16_t* __restrict__ src_slab,
                                                                      int src_n_pages, const int32_t* __restrict__ src_ids,
                                                                      const int32_t* __restrict__ dst_ids,
                                                                      size_t page_vecs, int32_t* dev_err)
{
    griddep_wait();
    griddep_launch_dependents();
    const int pair = blockIdx.y;
    const int32_t s = src_ids[pair], d = dst_ids[pair];
    if (s < 0 || s >= src_n_pages || d < 0 || d >= dst_n_pages) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && dev_err) atomicOr(dev_err, (int)K3MLA_DEV_BAD_PAGE);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(src_slab) + (size_t)s * page_vecs;
    uint4* dst = reinterpret_cast<uint4*>(dst_slab) + (size_t)d * page_vecs;
    const size_t step = (size_t)gridDim.x * CP_THREADS * CP_VEC;
    for (size_t base = (size_t)blockIdx.x * CP_THREADS * CP_VEC + threadIdx.x; base < page_vecs; base += step) {
        uint4 v[CP_VEC];
#pragma unroll
        for (int k = 0; k < CP_VEC; ++k) {
            const size_t i = base + (size_t)k * CP_THREADS;
            if (i < page_vecs) v[k] = src[i];
        }
#pragma unroll
        for (int k = 0; k < CP_VEC; ++k) {
            const size_t i = base + (size_t)k * CP_THREADS;
            if (i < page_vecs) dst[i] = v[k];
        }
    }
}

}  // namespace k3

using namespace k3;

extern "C" int k3mla_copy_pages(uint16_t* dst_slab, int dst_n_pages, const uint16_t* src_slab, int src_n_pages,
                                int n_layers, const int32_t* src_ids, const int32_t* dst_ids, int n,
                                int32_t* dev_err, void* stream)
{
    if (n < 0 || n_layers <= 0 || dst_n_pages <= 0 || src_n_pages <= 0 || n > 65535) {
        set_error("k3mla_copy_pages: invalid sizes (n must be in [0, 65535])");
        return K3MLA_E_INVALID;
    }
    if (n == 0) return K3MLA_OK;
    if (!dst_slab || !src_slab || !src_ids || !dst_ids || !aligned(dst_slab, 16) || !aligned(src_slab, 16)) {
        set_error("k3mla_copy_pages: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    const size_t page_vecs = (size_t)n_layers * PAGE * ROW * 2 / 16;  // 4,608 16-byte vectors per layer
    const size_t per_cta = (size_t)CP_THREADS * CP_VEC;
    size_t chunks = (page_vecs + per_cta - 1) / per_cta;
    if (chunks > 1024) chunks = 1024;  // a grid-stride loop covers the rest of a very deep page
    return launch_pdl(k3mla_copy_pages_kernel, dim3((unsigned)chunks, (unsigned)n), dim3(CP_THREADS), 0,
                      reinterpret_cast<cudaStream_t>(stream), "k3mla_copy_pages_kernel", dst_slab, dst_n_pages,
                      src_slab, src_n_pages, src_ids, dst_ids, page_vecs, dev_err);
}
