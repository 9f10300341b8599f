// expanded.cu -- the expanded-cache design that the absorbed decode replaces, as an A/B baseline.
//
// pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M2 commit: before the absorbed
// kernel, every token's latent was expanded by kv_b into per-head K (192 = 128 nope + the 64-wide
// rope key) and V (128) rows -- about 1.47 MB per token over 24 MLA layers against 27.6 KB for the
// latent row -- and decode ran ordinary attention over them.  This file builds that cache for one
// layer from the latent slab and decodes over it, so that the two designs can be timed on the same
// GPU and workload.
//
//   expanded cache   [n_pages][64 tokens][96 heads][320] bf16 for one layer: K nope (128), K rope (64),
//                    V (128) of head h for the token at that page position (the same block tables
//                    address it as the latent slab).
//   build            per (head, part, group of pages) a CTA stages W_UK[h] or W_UV[h] (128 KB, TMA) and,
//                    page by page, the page's latent (64 KB, TMA), and runs OUT^T[128 x 64 tokens] =
//                    W[h] [128 x 512] . C^T [512 x 64] on tcgen05 (32 MMAs, M = 128, N = 64), landing bf16.
//   decode           one warp per (slot, head): lane l holds q[6l .. 6l + 5] and V dims 4l .. 4l + 3; per
//                    token the 192-wide dot is a warp reduction, the score lands as the absorbed chain
//                    lands it (bf16(bf16(dot) * scale)), and an online softmax accumulates p V in f32.
//                    Bandwidth-bound (640 bytes per token and head), so CUDA cores, not tensor cores.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int XR = NOPE + ROPE + VH;           // 320: one head's expanded row
constexpr int XB_THREADS = 128;                // build: four warps read the accumulator back
constexpr int XB_A = 8 * 128 * 128;            // W part: [8 chunks][128 rows][128 B]
constexpr int XB_B = 8 * PAGE * 128;           // page latent: [8 chunks][64 rows][128 B]
constexpr uint64_t XB_WAIT_NS = 1000000000ull; // bounded waits: 1 s
constexpr int XD_WARPS = 4;                    // decode: heads (warps) per CTA
constexpr int XD_TOK = 4;                      // decode: tokens whose loads are in flight together

__device__ __forceinline__ bool xb_wait(uint64_t* bar, uint32_t parity, int32_t* dev_err)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_test_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity)) {
        if (globaltimer() - t0 > XB_WAIT_NS) {
            if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// grid (96 heads, 2 parts: 0 = W_UK -> K nope, 1 = W_UV -> V, page groups); block 128.
__global__ void __launch_bounds__(XB_THREADS, 1)
    k3mla_expand_cache_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_c,
                              const uint16_t* __restrict__ slab, int n_pages, int n_layers, int layer,
                              uint16_t* __restrict__ xcache, int32_t* dev_err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sb = sa + XB_A;
    __shared__ uint64_t w_full, c_full, d_full;
    __shared__ uint32_t tmem_slot;
    const int h = blockIdx.x, part = blockIdx.y;
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    if (threadIdx.x == 0) {
        mbar_init(&w_full, 1);
        mbar_init(&c_full, 1);
        mbar_init(&d_full, 1);
        fence_mbarrier_init_cluster();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    griddep_wait();
    griddep_launch_dependents();
    bool ok = true;
    if (threadIdx.x == 0) {  // W_UK[h] (rows h * 256 ..) or W_UV[h] (rows h * 256 + 128 ..), 512 columns
        mbar_arrive_expect_tx(&w_full, XB_A);
        for (int c = 0; c < 8; ++c)
            tma_load_3d(sa + c * (128 * 128), &tmap_w, 0, h * WROWS_PER_HEAD + part * NOPE, c, &w_full);
        ok = xb_wait(&w_full, 0, dev_err);
    }
    const uint64_t ad = make_sdesc(smem_u32(sa), 16, 1024);
    const uint64_t bd = make_sdesc(smem_u32(sb), 16, 1024);
    const uint32_t idesc = make_idesc_bf16(128, PAGE, 0, 0);
    const int off = part == 0 ? 0 : NOPE + ROPE;
    uint32_t ph = 0;
    for (int pg = blockIdx.z; pg < n_pages; pg += gridDim.z, ph ^= 1u) {
        if (threadIdx.x == 0) {
            if (ok) {  // the page's 64 latent rows at this layer
                mbar_arrive_expect_tx(&c_full, XB_B);
                tma_load_3d(sb, &tmap_c, 0, (pg * n_layers + layer) * PAGE, 0, &c_full);
                ok = xb_wait(&c_full, ph, dev_err);
            }
            if (ok) {
                tc_fence_after();
                for (int ks = 0; ks < LORA / 16; ++ks) {
                    const int c = ks >> 2, kk = ks & 3;
                    umma_ss(tbase, ad + (uint64_t)((c * (128 * 128) + kk * 32) >> 4),
                            bd + (uint64_t)((c * (PAGE * 128) + kk * 32) >> 4), idesc, ks > 0 ? 1u : 0u);
                }
            }
            umma_commit(&d_full);
        }
        const bool done = xb_wait(&d_full, ph, dev_err);
        tc_fence_after();
        // lane quarter `warp` holds rows 32 warp .. 32 warp + 31 (dims of K nope or V), columns = tokens
        if (__all_sync(0xFFFFFFFFu, done)) {
            const int d = 32 * (int)warp + (int)lane;
            uint16_t* dst = xcache + ((size_t)pg * PAGE * H + h) * XR + off + d;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                tmem_ld32(tbase + ((32u * warp) << 16) + 32u * (uint32_t)half, r);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    dst[(size_t)(32 * half + t) * H * XR] = (uint16_t)(pack_bf16x2(__uint_as_float(r[t]), 0.f) & 0xFFFFu);
            }
            if (part == 0)  // the rope key: the same 64 values for every head
                for (int i = (int)threadIdx.x; i < PAGE * (ROPE / 8); i += XB_THREADS) {
                    const int t = i / (ROPE / 8), u = i % (ROPE / 8);
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        slab + (((size_t)pg * n_layers + layer) * PAGE + t) * ROW + LORA + 8 * u);
                    *reinterpret_cast<uint4*>(xcache + (((size_t)pg * PAGE + t) * H + h) * XR + NOPE + 8 * u) = v;
                }
        }
        tc_fence_before();
        __syncthreads();  // the accumulator and the page buffer are free for the next page
    }
    if (!ok && threadIdx.x == 0) {  // a wait gave up: let issued copies land before the CTA exits
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
    }
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, 64);
}

// grid (B, 96 / XD_WARPS); block 32 * XD_WARPS: warp = head.
__global__ void __launch_bounds__(32 * XD_WARPS, 12)  // 12 CTAs an SM: 64 slots x 96 heads in one wave
    k3mla_expanded_decode_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ xcache, int n_pages,
                                 const int32_t* __restrict__ table, int max_pages, const int32_t* __restrict__ ctx_len,
                                 int max_ctx, uint32_t scale2, uint16_t* __restrict__ out, int32_t* dev_err)
{
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x;
    const int h = blockIdx.y * XD_WARPS + (int)(threadIdx.x >> 5);
    const int l = (int)lane_id();
    int n = ctx_len[b];
    const int cap = min(max_ctx, max_pages * PAGE);
    if (n > cap) {
        if (l == 0 && h == 0 && dev_err) atomicOr(dev_err, (int)K3MLA_DEV_CTX);
        n = cap;
    }
    n = max(n, 0);
    // this lane's six q values (dims 6l .. 6l + 5 of nope | rope)
    float qv[6];
    {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(q + ((size_t)b * H + h) * QDIM + 6 * l);
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const uint32_t w = qw[i];
            qv[2 * i] = __uint_as_float(w << 16);
            qv[2 * i + 1] = __uint_as_float(w & 0xFFFF0000u);
        }
    }
    const float LOG2E = 1.4426950408889634f;
    float m = -INFINITY, lsum = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int t0 = 0; t0 < n; t0 += XD_TOK) {
        uint32_t kw[XD_TOK][3];
        uint2 vw[XD_TOK];
#pragma unroll
        for (int u = 0; u < XD_TOK; ++u) {  // every load of the batch first
            const int t = t0 + u;
            kw[u][0] = kw[u][1] = kw[u][2] = 0u;
            vw[u] = make_uint2(0u, 0u);
            if (t < n) {
                const int32_t id = table[(size_t)b * max_pages + t / PAGE];
                if (id >= 0 && id < n_pages) {
                    const uint16_t* row = xcache + (((size_t)id * PAGE + t % PAGE) * H + h) * XR;
                    const uint32_t* kr = reinterpret_cast<const uint32_t*>(row + 6 * l);
                    kw[u][0] = kr[0];
                    kw[u][1] = kr[1];
                    kw[u][2] = kr[2];
                    vw[u] = *reinterpret_cast<const uint2*>(row + NOPE + ROPE + 4 * l);
                } else if (id != -1 && l == 0 && dev_err) {
                    atomicOr(dev_err, (int)K3MLA_DEV_BAD_PAGE);  // read as a zero row, like -1
                }
            }
        }
#pragma unroll
        for (int u = 0; u < XD_TOK; ++u) {
            if (t0 + u >= n) break;
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                part = fmaf(qv[2 * i], __uint_as_float(kw[u][i] << 16), part);
                part = fmaf(qv[2 * i + 1], __uint_as_float(kw[u][i] & 0xFFFF0000u), part);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
            // the score lands as the absorbed chain lands it: bf16(dot), then bf16(. * scale)
            const float s = bf16lo_to_f32(mul_bf16x2(pack_bf16x2(part, part), scale2));
            if (s > m) {
                const float a = ex2_approx((m - s) * LOG2E);  // 0 for the first token (m = -inf)
                lsum *= a;
#pragma unroll
                for (int d = 0; d < 4; ++d) o[d] *= a;
                m = s;
            }
            const float p = ex2_approx((s - m) * LOG2E);
            lsum += p;
            o[0] = fmaf(p, __uint_as_float(vw[u].x << 16), o[0]);
            o[1] = fmaf(p, __uint_as_float(vw[u].x & 0xFFFF0000u), o[1]);
            o[2] = fmaf(p, __uint_as_float(vw[u].y << 16), o[2]);
            o[3] = fmaf(p, __uint_as_float(vw[u].y & 0xFFFF0000u), o[3]);
        }
    }
    const float rl = n > 0 ? 1.f / lsum : 0.f;
    uint2 res;
    res.x = pack_bf16x2(o[0] * rl, o[1] * rl);
    res.y = pack_bf16x2(o[2] * rl, o[3] * rl);
    *reinterpret_cast<uint2*>(out + ((size_t)b * H + h) * VH + 4 * l) = res;
}

}  // namespace k3

using namespace k3;

extern "C" size_t k3mla_expanded_cache_bytes(int n_pages)
{
    return n_pages <= 0 ? 0 : (size_t)n_pages * PAGE * H * XR * 2;
}

extern "C" int k3mla_expand_latent_cache(const uint16_t* slab, int n_pages, int n_layers, int layer,
                                         const uint16_t* w_kv_b, uint16_t* xcache, int32_t* dev_err, void* stream)
{
    if (n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers) {
        set_error("k3mla_expand_latent_cache: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if ((long long)n_pages * n_layers * PAGE > 0x7FFFFFFFll) {
        set_error("k3mla_expand_latent_cache: slab rows exceed the 2^31 TMA row range");
        return K3MLA_E_INVALID;
    }
    if (!slab || !w_kv_b || !xcache || !aligned(slab, 16) || !aligned(w_kv_b, 16) || !aligned(xcache, 16)) {
        set_error("k3mla_expand_latent_cache: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    CUtensorMap tm_w, tm_c;
    int rc = make_tmap_slab_3d(&tm_w, w_kv_b, (uint64_t)H * WROWS_PER_HEAD, LORA, 8, 128, 1);
    if (rc) return rc;
    rc = make_tmap_slab_3d(&tm_c, slab, (uint64_t)n_pages * n_layers * PAGE, ROW, 9, PAGE, 8);
    if (rc) return rc;
    const int smem = XB_A + XB_B + 1024;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaFuncSetAttribute(k3mla_expand_cache_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const int groups = n_pages < 8 ? n_pages : 8;
    return launch_pdl(k3mla_expand_cache_kernel, dim3(H, 2, groups), dim3(XB_THREADS), smem,
                      reinterpret_cast<cudaStream_t>(stream), "k3mla_expand_cache_kernel", tm_w, tm_c, slab,
                      n_pages, n_layers, layer, xcache, dev_err);
}

extern "C" int k3mla_expanded_decode(const uint16_t* q, const uint16_t* xcache, int n_pages, const int32_t* block_table,
                                     int max_pages_per_slot, const int32_t* ctx_len, uint16_t scale_bf16, uint16_t* out,
                                     int B, int max_ctx, int32_t* dev_err, void* stream)
{
    if (B < 0 || n_pages <= 0 || max_pages_per_slot <= 0 || max_ctx <= 0) {
        set_error("k3mla_expanded_decode: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if (!q || !xcache || !block_table || !ctx_len || !out || !aligned(q, 4) || !aligned(xcache, 16) ||
        !aligned(out, 8)) {
        set_error("k3mla_expanded_decode: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    if (B > 65535) {
        set_error("k3mla_expanded_decode: grid too large");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    const uint32_t scale2 = ((uint32_t)scale_bf16 << 16) | (uint32_t)scale_bf16;
    return launch_pdl(k3mla_expanded_decode_kernel, dim3(B, H / XD_WARPS), dim3(32 * XD_WARPS), 0,
                      reinterpret_cast<cudaStream_t>(stream), "k3mla_expanded_decode_kernel", q, xcache, n_pages,
                      block_table, max_pages_per_slot, ctx_len, max_ctx, scale2, out, dev_err);
}
