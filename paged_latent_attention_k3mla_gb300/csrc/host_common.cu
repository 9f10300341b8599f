// host_common.cu -- error text, launch checks, device check and TMA descriptor
// creation for libk3mla.
#include <cstdarg>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace k3 {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

int check_launch(const char* what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s: %s", what, cudaGetErrorString(e));
        return K3MLA_E_CUDA;
    }
    return K3MLA_OK;
}

bool device_ok()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        set_error("no CUDA device");
        return false;
    }
    static int cached[64];
    static std::once_flag once[64];
    if (dev < 0 || dev >= 64) return false;
    std::call_once(once[dev], [dev]() {
        int maj = 0, min = 0;
        cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
        cached[dev] = maj * 10 + min;
    });
    if (cached[dev] != 103) {
        set_error("libk3mla is built for sm_103a; current device is sm_%d", cached[dev]);
        return false;
    }
    return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled unavailable");
        return K3MLA_E_CUDA;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
        return K3MLA_E_CUDA;
    }
    return K3MLA_OK;
}

int make_tmap_slab_3d(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems, uint32_t n_chunks,
                      uint32_t box_rows, uint32_t box_chunks)
{
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled unavailable");
        return K3MLA_E_CUDA;
    }
    cuuint64_t dims[3] = {64, rows, n_chunks};
    cuuint64_t strides[2] = {(cuuint64_t)row_elems * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (3-D slab view) failed (%d)", (int)r);
        return K3MLA_E_CUDA;
    }
    return K3MLA_OK;
}

int make_tmap_store(CUtensorMap* map, bool f32, uint32_t rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box, bool swizzle128)
{
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled unavailable");
        return K3MLA_E_CUDA;
    }
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], estr[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                    const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (store view) failed (%d)", (int)r);
        return K3MLA_E_CUDA;
    }
    return K3MLA_OK;
}

}  // namespace k3

extern "C" const char* k3mla_last_error(void) { return k3::g_err; }
