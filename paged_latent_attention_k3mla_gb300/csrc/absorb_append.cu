// absorb_append.cu -- q absorption and the latent-row append.
//
// q absorption (pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode",
// M2 commit: "q_abs = W_UK^T q_nope is precomputed" and "q absorption lands
// bf16"): q_abs[b][h][j] = bf16(sum_d W_UK[h][d][j] q_nope[b][h][d]) for j < 512,
// then q_rope is copied to q_abs[b][h][512:576].  Per head this is a small
// [B x 128] x [128 x 512] product whose cost is reading W_UK (12.6 MB per layer);
// it runs on tensor cores with mma.sync (f32 accumulation), one CTA per
// (head, 128 output columns), W_UK staged once in shared memory.
//
// Append (same PR, M1 commit): the new token's 512-wide latent and 64-wide rope
// key land in row ((page * L + layer) * 64 + pos % 64) of the page-first slab,
// page = block_table[b][pos / 64]; the element index is size_t (the slab passes
// 2^31 elements).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace k3 {

constexpr int AB_THREADS = 256;
constexpr int AB_NCOLS = 128;             // output columns per CTA
constexpr int AB_PITCH = AB_NCOLS + 8;    // W tile pitch (elements), 16-byte pad
constexpr int AQ_PITCH = NOPE + 8;        // q tile pitch (elements)

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// grid (512 / 128 column blocks, 96 heads)
__global__ void __launch_bounds__(AB_THREADS) k3mla_absorb_kernel(const uint16_t* __restrict__ q,
                                                                    const uint16_t* __restrict__ w,
                                                                    uint16_t* __restrict__ q_abs, int B)
{
    __shared__ __align__(16) uint16_t sw[NOPE * AB_PITCH];   // W_UK[h][d][nb*128 + n]
    __shared__ __align__(16) uint16_t sq[16 * AQ_PITCH];     // q_nope rows of 16 slots
    const int nb = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const uint16_t* wsrc = w + (size_t)h * WROWS_PER_HEAD * LORA + nb * AB_NCOLS;
    for (int i = tid; i < NOPE * (AB_NCOLS / 8); i += AB_THREADS) {
        const int d = i / (AB_NCOLS / 8), c8 = i % (AB_NCOLS / 8);
        *reinterpret_cast<uint4*>(sw + d * AB_PITCH + c8 * 8) =
            __ldg(reinterpret_cast<const uint4*>(wsrc + (size_t)d * LORA) + c8);
    }
    if (nb == 0) {  // rope half copied through
        for (int i = tid; i < B * (ROPE / 8); i += AB_THREADS) {
            const int b = i / (ROPE / 8), c8 = i % (ROPE / 8);
            *reinterpret_cast<uint4*>(q_abs + ((size_t)b * H + h) * ROW + LORA + c8 * 8) =
                __ldg(reinterpret_cast<const uint4*>(q + ((size_t)b * H + h) * QDIM + NOPE) + c8);
        }
    }
    // warp -> output columns 16*warp .. 16*warp+15 (two n8 tiles)
    const uint32_t a_base = smem_addr(sq) + ((lane & 15) * AQ_PITCH + (lane >> 4) * 8) * 2;
    // x4.trans over W[k][n]: lane -> k row (lane & 7) + 8*((lane>>3)&1), n block 8*(lane>>4)
    const uint32_t b_base =
        smem_addr(sw) + (((lane & 7) + 8 * ((lane >> 3) & 1)) * AB_PITCH + 16 * warp + 8 * (lane >> 4)) * 2;
    for (int m0 = 0; m0 < B; m0 += 16) {
        __syncthreads();
        {
            const int r = tid >> 4, c8 = tid & 15;  // 16 rows x 16 chunks of 8
            const int b = m0 + r;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (b < B) v = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)b * H + h) * QDIM) + c8);
            *reinterpret_cast<uint4*>(sq + r * AQ_PITCH + c8 * 8) = v;
        }
        __syncthreads();
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < NOPE / 16; ++ks) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(a_base + ks * 32));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                         : "r"(b_base + ks * 16 * AB_PITCH * 2));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(acc[0][0]), "+f"(acc[0][1]), "+f"(acc[0][2]), "+f"(acc[0][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(acc[1][0]), "+f"(acc[1][1]), "+f"(acc[1][2]), "+f"(acc[1][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b2), "r"(b3));
        }
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = nb * AB_NCOLS + 16 * warp + 8 * nt + 2 * t4;
            if (m0 + g < B)
                *reinterpret_cast<uint32_t*>(q_abs + ((size_t)(m0 + g) * H + h) * ROW + col) =
                    pack2(acc[nt][0], acc[nt][1]);
            if (m0 + g + 8 < B)
                *reinterpret_cast<uint32_t*>(q_abs + ((size_t)(m0 + g + 8) * H + h) * ROW + col) =
                    pack2(acc[nt][2], acc[nt][3]);
        }
    }
}

// one CTA of 96 threads per slot; each thread moves three 32-bit words
__global__ void __launch_bounds__(96) k3mla_append_kernel(uint16_t* __restrict__ slab, int n_pages, int n_layers,
                                                            int layer, const int32_t* __restrict__ table,
                                                            int max_pages, const int32_t* __restrict__ pos,
                                                            const uint16_t* __restrict__ c_kv, int64_t c_stride,
                                                            const uint16_t* __restrict__ k_rope, int64_t r_stride,
                                                            int32_t* dev_err)
{
    const int b = blockIdx.x;
    const int p = pos[b];
    if (p < 0) return;
    const int lp = p / PAGE;
    int32_t id = -1;
    if (lp < max_pages) id = table[(size_t)b * max_pages + lp];
    if (id < 0 || id >= n_pages) {
        if (threadIdx.x == 0 && dev_err) atomicOr(dev_err, (int)K3MLA_DEV_UNMAPPED);
        return;
    }
    const size_t row = ((size_t)id * (size_t)n_layers + (size_t)layer) * PAGE + (size_t)(p % PAGE);
    uint32_t* dst = reinterpret_cast<uint32_t*>(slab + row * ROW);
    const uint32_t* src_c = reinterpret_cast<const uint32_t*>(c_kv + (size_t)b * c_stride);
    const uint32_t* src_r = reinterpret_cast<const uint32_t*>(k_rope + (size_t)b * r_stride);
    for (int i = threadIdx.x; i < ROW / 2; i += 96)
        dst[i] = (i < LORA / 2) ? src_c[i] : src_r[i - LORA / 2];
}

}  // namespace k3

using namespace k3;

extern "C" int k3mla_absorb_q(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, int B, void* stream)
{
    if (B < 0) {
        set_error("k3mla_absorb_q: B < 0");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if (!q || !w_kv_b || !q_abs || !aligned(q, 16) || !aligned(w_kv_b, 16) || !aligned(q_abs, 16)) {
        set_error("k3mla_absorb_q: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    k3mla_absorb_kernel<<<dim3(LORA / AB_NCOLS, H), AB_THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        q, w_kv_b, q_abs, B);
    return check_launch("k3mla_absorb_kernel");
}

extern "C" int k3mla_append_latent(uint16_t* slab, int n_pages, int n_layers, int layer,
                                   const int32_t* block_table, int max_pages_per_slot, const int32_t* pos,
                                   const uint16_t* c_kv, int64_t c_stride, const uint16_t* k_rope,
                                   int64_t r_stride, int B, int32_t* dev_err, void* stream)
{
    if (B < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers || max_pages_per_slot <= 0 ||
        c_stride < LORA || r_stride < ROPE || (c_stride & 1) || (r_stride & 1)) {
        set_error("k3mla_append_latent: invalid sizes or strides");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if (!slab || !block_table || !pos || !c_kv || !k_rope || !aligned(slab, 4) || !aligned(c_kv, 4) ||
        !aligned(k_rope, 4)) {
        set_error("k3mla_append_latent: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    k3mla_append_kernel<<<B, 96, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, pos, c_kv, c_stride, k_rope, r_stride,
        dev_err);
    return check_launch("k3mla_append_kernel");
}
