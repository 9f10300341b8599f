// merge_expand.cu -- merge of a slot's split partials and the W_UV expansion.
//
// For each (slot b, head h), the splits of the context are merged in ascending
// split order with the usual max-rescaled sum (m = max_i m_i; l = sum_i l_i
// e^(m_i - m); o = sum_i o_i e^(m_i - m)), o_lat lands in bf16 as o / l (pegainfer
// PR #869, "K3: paged latent MLA KV + absorbed decode", M2 commit: "f32 latent
// accumulation over ascending t landing bf16"), and out[b][h] = bf16(W_UV[h]
// o_lat) with W_UV read in place from w_kv_b ("f32 W_UV expansion landing bf16").
// Per head the expansion is a [B x 512] x [512 x 128] product: one CTA per
// (half of v, head) keeps its 64 KB of W_UV in shared memory and runs it on
// tensor cores with mma.sync, so W_UV is read from HBM once per layer.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace k3 {

__device__ __forceinline__ uint32_t mx_smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t mx_pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ int mx_ctx_effective(const int32_t* ctx_len, int b, int max_ctx, int max_pages)
{
    int n = ctx_len[b];
    int cap = min(max_ctx, max_pages * PAGE);
    n = n > cap ? cap : n;
    return n < 0 ? 0 : n;
}


constexpr int MX_THREADS = 256;
constexpr int W_PITCH = LORA + 8;   // bf16 elements per smem row (16-byte pad)


__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// grid (2 halves of v, 96 heads); each CTA keeps W_UV[h][64 v][512] in shared memory.
__global__ void __launch_bounds__(MX_THREADS) k3mla_merge_expand_kernel(const MergeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint16_t* sw = reinterpret_cast<uint16_t*>(smem_raw);   // [64][W_PITCH]
    uint16_t* so = sw + 64 * W_PITCH;                         // [16][W_PITCH]
    const int vh = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // W_UV[h] rows vh*64 .. vh*64+63 (w_kv_b rows h*256 + 128 + v)
    const uint16_t* wsrc = p.w_kv_b + ((size_t)h * WROWS_PER_HEAD + NOPE + vh * 64) * LORA;
    for (int q = tid; q < 64 * (LORA / 8); q += MX_THREADS) {
        const int r = q / (LORA / 8), c8 = q % (LORA / 8);
        *reinterpret_cast<uint4*>(sw + r * W_PITCH + c8 * 8) =
            __ldg(reinterpret_cast<const uint4*>(wsrc + (size_t)r * LORA) + c8);
    }

    for (int m0 = 0; m0 < p.B; m0 += 16) {
        __syncthreads();
        {   // merge: thread -> (row r, dims 32*jc .. 32*jc+31)
            const int r = tid >> 4, jc = tid & 15;
            const int b = m0 + r;
            float o[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0.f;
            float l = 1.f;
            if (b < p.B) {
                const int ctx = mx_ctx_effective(p.ctx_len, b, p.max_ctx, p.max_pages);
                const int ns = (ctx + p.split - 1) / p.split;
                if (ns > 0) {
                    const float* ml = p.ws_ml + ((size_t)b * p.nsplit * H + h) * 4;
                    float m = -INFINITY;
                    for (int i = 0; i < ns; ++i) m = fmaxf(m, ml[(size_t)i * H * 4]);
                    l = 0.f;
                    float best = -INFINITY;
                    int best_t = -1;
                    for (int i = 0; i < ns; ++i) {
                        const float* mi = ml + (size_t)i * H * 4;
                        const float wgt = expf(mi[0] - m);
                        l += wgt * mi[1];
                        const float* oi = p.ws_o + (((size_t)b * p.nsplit + i) * H + h) * LORA + 32 * jc;
#pragma unroll
                        for (int k = 0; k < 32; k += 4) {
                            const float4 v = *reinterpret_cast<const float4*>(oi + k);
                            o[k + 0] += wgt * v.x;
                            o[k + 1] += wgt * v.y;
                            o[k + 2] += wgt * v.z;
                            o[k + 3] += wgt * v.w;
                        }
                        if (mi[2] > best) {
                            best = mi[2];
                            best_t = __float_as_int(mi[3]);
                        }
                    }
                    if (p.argmax && vh == 0 && jc == 0) p.argmax[(size_t)b * H + h] = best_t;
                } else if (p.argmax && vh == 0 && jc == 0) {
                    p.argmax[(size_t)b * H + h] = -1;
                }
            }
            const float inv_l_div = l;  // divide each element by l (IEEE quotient)
            uint32_t* dst = reinterpret_cast<uint32_t*>(so + r * W_PITCH + 32 * jc);
#pragma unroll
            for (int k = 0; k < 32; k += 2) dst[k >> 1] = mx_pack_bf16x2(o[k] / inv_l_div, o[k + 1] / inv_l_div);
        }
        __syncthreads();
        // out[16 x 64] = o_lat[16 x 512] . W_UV^T ; warp w -> v columns 8w .. 8w+7
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t a_base = mx_smem_u32(so) + ((lane & 15) * W_PITCH + (lane >> 4) * 8) * 2;
        const uint32_t b_base = mx_smem_u32(sw) + ((8 * warp + (lane & 7)) * W_PITCH + ((lane >> 3) & 1) * 8) * 2;
#pragma unroll 4
        for (int ks = 0; ks < LORA / 16; ++ks) {
            uint32_t a0, a1, a2, a3, b0, b1;
            ldsm_x4(a_base + ks * 32, a0, a1, a2, a3);
            ldsm_x2(b_base + ks * 32, b0, b1);
            mma_bf16_16816(acc, a0, a1, a2, a3, b0, b1);
        }
        const int g = lane >> 2, t4 = lane & 3;
        const int v = vh * 64 + 8 * warp + 2 * t4;
        if (m0 + g < p.B)
            *reinterpret_cast<uint32_t*>(p.out + ((size_t)(m0 + g) * H + h) * VH + v) = mx_pack_bf16x2(acc[0], acc[1]);
        if (m0 + g + 8 < p.B)
            *reinterpret_cast<uint32_t*>(p.out + ((size_t)(m0 + g + 8) * H + h) * VH + v) =
                mx_pack_bf16x2(acc[2], acc[3]);
    }
}


int launch_merge_expand(const MergeParams& mp, cudaStream_t st)
{
    static bool attr_set[64] = {};
    const int smem = (64 + 16) * W_PITCH * 2;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaFuncSetAttribute(k3mla_merge_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    k3mla_merge_expand_kernel<<<dim3(2, H), dim3(MX_THREADS), smem, st>>>(mp);
    return check_launch("k3mla_merge_expand_kernel");
}

}  // namespace k3
