// exact.cu -- the rounding chain, landing for landing, on the GPU.
//
// pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M2 commit: the
// certified chain is (1) q absorption lands bf16, (2) an f32 score dot over the 576
// row entries in ascending order lands bf16, (3) times the bf16 scale, landed bf16,
// (4) f32 max and f32 sum of exp in a fixed order, (5) probabilities land bf16
// after normalising, (6) f32 latent accumulation over ascending t lands bf16,
// (7) f32 W_UV expansion lands bf16.  The page's own kernel kept that chain with
// three sweeps over the context; the one-pass kernel of decode.cu trades it for a
// single read of the cache (tensor-core summation order, online softmax).
//
// This mode keeps it.  Every sum is one thread's sequential loop in the chain's
// index order (products of two bf16 values are exact in f32, so a fused
// multiply-add rounds exactly as the multiply-then-add of the chain), exp is the
// double-precision exp rounded once to f32, normalisation is the IEEE quotient.
// Fixed orders rule out the tensor cores, so these are CUDA-core kernels:
//   E0 absorption   thread per (slot, head, j): sum over d = 0..127
//   E1 scores       CTA per (slot, 8 pages): Q and each page staged in shared
//                   memory; thread per (4 tokens, 3 heads): sums over k = 0..575
//   E2 softmax      CTA per (slot, head): max and exps across the block, the sum
//                   of exp thread 0's loop over t ascending, p_t = bf16(e_t / l),
//                   argmax (lowest t with the largest p)
//   E3 latent sum   CTA per (slot, 64 dims): thread per (4 dims, 6 heads), sums
//                   over t ascending, pages staged in shared memory
//   E4 expansion    CTA per (head, 16 slots): W_UV[h] staged; thread per v:
//                   sixteen sums over j = 0..511
// Interpretation where the pages are silent (the same as the CPU oracle's): a -1
// table entry is an all-zero row that takes part in the softmax; positions >=
// ctx_len are never read; ctx_len == 0 gives zeros and argmax -1.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

__device__ __forceinline__ float ex_bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint16_t ex_land(float f)  // round to nearest even, f32 -> bf16
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(f));
    return (uint16_t)(r & 0xFFFFu);
}

__device__ __forceinline__ int ex_ctx(const int32_t* ctx_len, int b, int max_ctx, int max_pages)
{
    int n = ctx_len[b];
    const int cap = min(max_ctx, max_pages * PAGE);
    n = n > cap ? cap : n;
    return n < 0 ? 0 : n;
}

// Row pointer of logical token t of slot b, or null for a zero row (-1, or a bad id: flagged).
__device__ __forceinline__ const uint16_t* ex_row(const uint16_t* slab, int n_pages, int n_layers, int layer,
                                                  const int32_t* table, int max_pages, int b, int t,
                                                  int32_t* dev_err)
{
    const int32_t id = table[(size_t)b * max_pages + t / PAGE];
    if (id == -1) return nullptr;
    if (id < -1 || id >= n_pages) {
        if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_BAD_PAGE);
        return nullptr;
    }
    return slab + (((size_t)id * n_layers + layer) * PAGE + (size_t)(t % PAGE)) * ROW;
}

// ---- E0: absorption ------------------------------------------------------------------------
// grid (B, 96); block 512 (j).  q_abs[b][h][j] = bf16(sum_{d ascending} W_UK[h][d][j] q_nope[d]).
__global__ void __launch_bounds__(LORA) ex_absorb_kernel(const uint16_t* __restrict__ q,
                                                        const uint16_t* __restrict__ w_kv_b,
                                                        uint16_t* __restrict__ q_abs)
{
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x, h = blockIdx.y, j = threadIdx.x;
    __shared__ float qn[NOPE];
    const uint16_t* qb = q + ((size_t)b * H + h) * QDIM;
    if (j < NOPE) qn[j] = ex_bf(qb[j]);
    __syncthreads();
    const uint16_t* w = w_kv_b + (size_t)h * WROWS_PER_HEAD * LORA + j;
    float acc = 0.f;
    for (int d = 0; d < NOPE; ++d) acc = __fadd_rn(acc, __fmul_rn(ex_bf(w[(size_t)d * LORA]), qn[d]));
    uint16_t* qa = q_abs + ((size_t)b * H + h) * ROW;
    qa[j] = ex_land(acc);
    if (j < ROPE) qa[LORA + j] = qb[NOPE + j];
}

// ---- E1: scores ----------------------------------------------------------------------------
constexpr int E1_PAGES = 8;              // pages per CTA (Q is staged once for them)
constexpr int E1_THREADS = 512;
constexpr int E1_QP = ROW + 2;           // padded row pitch (elements): rows start in distinct banks
constexpr int E1_SMEM = (H + PAGE) * E1_QP * 2;
constexpr int E1_TOK = 4, E1_HEADS = 3;  // register tile of one thread: 4 tokens x 3 heads

// grid (B, ceil(max_ctx / (64 * E1_PAGES))); block 512.  s[b][h][t] = bf16(bf16(dot) * scale).
// Thread (warp w, lane l): tokens g, g + 16, g + 32, g + 48 of the page (g = l % 16) and heads
// 3 (2 w + l / 16) .. + 2; each of its 12 dots is one sequential sum over k = 0..575 ascending (a fused
// multiply-add of two bf16 values rounds as the chain's multiply-then-add: the product is exact).
__global__ void __launch_bounds__(E1_THREADS) ex_scores_kernel(
    const uint16_t* __restrict__ q_abs, const uint16_t* __restrict__ slab, int n_pages, int n_layers, int layer,
    const int32_t* __restrict__ table, int max_pages, const int32_t* __restrict__ ctx_len, int max_ctx,
    uint16_t scale_bf16, uint16_t* __restrict__ s_out, int s_pitch, int32_t* dev_err)
{
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ uint16_t ex_smem[];
    uint16_t* Qs = ex_smem;                  // [96][E1_QP]
    uint16_t* Rs = ex_smem + H * E1_QP;      // [64][E1_QP]
    const int b = blockIdx.x;
    const int n = ex_ctx(ctx_len, b, max_ctx, max_pages);
    const int t_begin = blockIdx.y * E1_PAGES * PAGE;
    if (t_begin >= n) return;
    const int t_end = min(n, t_begin + E1_PAGES * PAGE);
    const float scale = ex_bf(scale_bf16);
    for (int i = threadIdx.x; i < H * (ROW / 2); i += E1_THREADS) {
        const int h = i / (ROW / 2), k2 = i % (ROW / 2);
        reinterpret_cast<uint32_t*>(Qs + h * E1_QP)[k2] =
            reinterpret_cast<const uint32_t*>(q_abs + ((size_t)b * H + h) * ROW)[k2];
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane & 15, h0 = E1_HEADS * (2 * warp + (lane >> 4));
    for (int t0 = t_begin; t0 < t_end; t0 += PAGE) {
        __syncthreads();  // Q staged / the previous page's rows no longer read
        for (int i = threadIdx.x; i < PAGE * (ROW / 2); i += E1_THREADS) {
            const int r = i / (ROW / 2), k2 = i % (ROW / 2);
            const int t = t0 + r;
            uint32_t v = 0u;
            if (t < t_end) {
                const uint16_t* row = ex_row(slab, n_pages, n_layers, layer, table, max_pages, b, t,
                                             k2 == 0 ? dev_err : nullptr);
                if (row) v = reinterpret_cast<const uint32_t*>(row)[k2];
            }
            reinterpret_cast<uint32_t*>(Rs + r * E1_QP)[k2] = v;
        }
        __syncthreads();
        float acc[E1_TOK][E1_HEADS];
#pragma unroll
        for (int a = 0; a < E1_TOK; ++a)
#pragma unroll
            for (int c = 0; c < E1_HEADS; ++c) acc[a][c] = 0.f;
        const uint32_t* rw[E1_TOK];
#pragma unroll
        for (int a = 0; a < E1_TOK; ++a) rw[a] = reinterpret_cast<const uint32_t*>(Rs + (g + 16 * a) * E1_QP);
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(Qs + h0 * E1_QP);
#pragma unroll 2
        for (int k2 = 0; k2 < ROW / 2; ++k2) {  // k = 2 k2, then 2 k2 + 1: ascending
            float rlo[E1_TOK], rhi[E1_TOK];
#pragma unroll
            for (int a = 0; a < E1_TOK; ++a) {
                const uint32_t rv = rw[a][k2];
                rlo[a] = __uint_as_float(rv << 16);
                rhi[a] = __uint_as_float(rv & 0xFFFF0000u);
            }
#pragma unroll
            for (int c = 0; c < E1_HEADS; ++c) {
                const uint32_t qv = qw[c * (E1_QP / 2) + k2];
                const float qlo = __uint_as_float(qv << 16), qhi = __uint_as_float(qv & 0xFFFF0000u);
#pragma unroll
                for (int a = 0; a < E1_TOK; ++a) {
                    acc[a][c] = __fmaf_rn(qlo, rlo[a], acc[a][c]);
                    acc[a][c] = __fmaf_rn(qhi, rhi[a], acc[a][c]);
                }
            }
        }
#pragma unroll
        for (int a = 0; a < E1_TOK; ++a) {
            const int t = t0 + g + 16 * a;
            if (t < t_end)
#pragma unroll
                for (int c = 0; c < E1_HEADS; ++c)
                    s_out[((size_t)b * H + h0 + c) * s_pitch + t] = ex_land(__fmul_rn(ex_bf(ex_land(acc[a][c])), scale));
        }
    }
}

// ---- E2: softmax -----------------------------------------------------------------------------
// grid (B * 96); block E2_THREADS; dynamic smem: e_t for the row (max_ctx f32).  The max, the exps
// and the landings are independent per token and run across the block; the sum of exp is thread
// 0's loop over t ascending.  Overwrites s with bf16 p; argmax = lowest t with the largest p.
constexpr int E2_THREADS = 256;
constexpr int E2_MAX_SMEM = 200 * 1024;  // e_t of one row: max_ctx <= 51,200

__global__ void __launch_bounds__(E2_THREADS) ex_softmax_kernel(const int32_t* __restrict__ ctx_len, int max_ctx,
                                                               int max_pages, uint16_t* __restrict__ sp, int s_pitch,
                                                               int32_t* __restrict__ argmax)
{
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ float ex_e[];
    __shared__ float red_f[E2_THREADS / 32];
    __shared__ int red_i[E2_THREADS / 32];
    __shared__ float l_sh;
    const int i = blockIdx.x, b = i / H;
    const int n = ex_ctx(ctx_len, b, max_ctx, max_pages);
    uint16_t* row = sp + (size_t)i * s_pitch;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (n == 0) {
        if (argmax && threadIdx.x == 0) argmax[i] = -1;
        return;
    }
    float m = -INFINITY;  // the max does not depend on the order it is taken in
    for (int t = threadIdx.x; t < n; t += E2_THREADS) m = fmaxf(m, ex_bf(row[t]));
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red_f[warp] = m;
    __syncthreads();
    m = red_f[0];
    for (int w = 1; w < E2_THREADS / 32; ++w) m = fmaxf(m, red_f[w]);
    for (int t = threadIdx.x; t < n; t += E2_THREADS) ex_e[t] = (float)exp((double)__fsub_rn(ex_bf(row[t]), m));
    __syncthreads();
    if (threadIdx.x == 0) {  // l = sum of e_t over t ascending, one rounding per addition
        float l = 0.f;
        for (int t = 0; t < n; ++t) l = __fadd_rn(l, ex_e[t]);
        l_sh = l;
    }
    __syncthreads();
    const float l = l_sh;
    float best = -1.f;
    int bt = n;
    for (int t = threadIdx.x; t < n; t += E2_THREADS) {
        const uint16_t pb = ex_land(__fdiv_rn(ex_e[t], l));
        const float p = ex_bf(pb);
        row[t] = pb;
        if (p > best) {  // t grows within a thread: the first t attaining its best
            best = p;
            bt = t;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {  // largest p, then lowest t
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int ot = __shfl_xor_sync(0xFFFFFFFFu, bt, o);
        if (ob > best || (ob == best && ot < bt)) {
            best = ob;
            bt = ot;
        }
    }
    __syncthreads();  // red_f is reused
    if (lane == 0) {
        red_f[warp] = best;
        red_i[warp] = bt;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < E2_THREADS / 32; ++w)
            if (red_f[w] > best || (red_f[w] == best && red_i[w] < bt)) {
                best = red_f[w];
                bt = red_i[w];
            }
        if (argmax) argmax[i] = bt;
    }
}

// ---- E3: latent sum --------------------------------------------------------------------------
constexpr int E3_THREADS = 256;          // (16 groups of 4 dims) x (16 groups of 6 heads)
constexpr int E3_DIMS = 64;              // latent dims per CTA
constexpr int E3_PP = 100;               // ps row pitch (floats): 8-byte aligned 6-head groups
constexpr int E3_SMEM = PAGE * E3_DIMS * 4 + PAGE * E3_PP * 4;  // c slice [64][64] f32 + p [64][100] f32

// grid (B, 512 / 64); o_lat[h][b][j] = bf16(sum_{t ascending} p_t c_t[j]).  Thread (warp w, lane l),
// i = 32 w + l: dims 4 (i % 16) .. + 3 of the block and heads 6 (i / 16) .. + 5, each of its 24 sums one
// sequential loop over t ascending (fused multiply-add of two bf16 values: the product is exact).
__global__ void __launch_bounds__(E3_THREADS) ex_latent_kernel(
    const uint16_t* __restrict__ slab, int n_pages, int n_layers, int layer, const int32_t* __restrict__ table,
    int max_pages, const int32_t* __restrict__ ctx_len, int B, int max_ctx, const uint16_t* __restrict__ p,
    int s_pitch, uint16_t* __restrict__ olat)
{
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ float ex_f[];
    float* cs = ex_f;                   // [64 tokens][64 dims]
    float* ps = ex_f + PAGE * E3_DIMS;  // [64 tokens][E3_PP] (heads 0..95)
    const int b = blockIdx.x, jb = blockIdx.y * E3_DIMS;
    const int n = ex_ctx(ctx_len, b, max_ctx, max_pages);
    const int dg = threadIdx.x & 15, hg = 6 * (threadIdx.x >> 4);
    float acc[6][4];
#pragma unroll
    for (int u = 0; u < 6; ++u)
#pragma unroll
        for (int d = 0; d < 4; ++d) acc[u][d] = 0.f;
    for (int t0 = 0; t0 < n; t0 += PAGE) {
        const int cnt = min(PAGE, n - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < PAGE * (E3_DIMS / 8); i += E3_THREADS) {  // 16 bytes = 8 dims each
            const int r = i >> 3, u = i & 7;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < cnt) {
                const uint16_t* row = ex_row(slab, n_pages, n_layers, layer, table, max_pages, b, t0 + r, nullptr);
                if (row) v = *reinterpret_cast<const uint4*>(row + jb + 8 * u);
            }
            float4* dst = reinterpret_cast<float4*>(cs + r * E3_DIMS + 8 * u);
            dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                 __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
            dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                                 __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
        }
        for (int i = threadIdx.x; i < H * (PAGE / 8); i += E3_THREADS) {  // 8 tokens of one head each
            const int h = i >> 3, r0 = 8 * (i & 7);
            const uint16_t* src = p + ((size_t)b * H + h) * s_pitch + t0 + r0;
#pragma unroll
            for (int e = 0; e < 8; ++e) ps[(r0 + e) * E3_PP + h] = (r0 + e < cnt) ? ex_bf(src[e]) : 0.f;
        }
        __syncthreads();
        for (int r = 0; r < cnt; ++r) {
            const float4 c = *reinterpret_cast<const float4*>(cs + r * E3_DIMS + 4 * dg);
            const float2* pr = reinterpret_cast<const float2*>(ps + r * E3_PP + hg);
#pragma unroll
            for (int q2 = 0; q2 < 3; ++q2) {
                const float2 pv = pr[q2];
                const float pp[2] = {pv.x, pv.y};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float* a = acc[2 * q2 + e];
                    a[0] = __fmaf_rn(pp[e], c.x, a[0]);
                    a[1] = __fmaf_rn(pp[e], c.y, a[1]);
                    a[2] = __fmaf_rn(pp[e], c.z, a[2]);
                    a[3] = __fmaf_rn(pp[e], c.w, a[3]);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 6; ++u) {
        const uint32_t lo = (uint32_t)ex_land(acc[u][0]) | ((uint32_t)ex_land(acc[u][1]) << 16);
        const uint32_t hi = (uint32_t)ex_land(acc[u][2]) | ((uint32_t)ex_land(acc[u][3]) << 16);
        *reinterpret_cast<uint2*>(olat + ((size_t)(hg + u) * B + b) * LORA + jb + 4 * dg) = make_uint2(lo, hi);
    }
}

// ---- E4: expansion ---------------------------------------------------------------------------
constexpr int E4_SLOTS = 16;             // slots per CTA (W_UV[h] is staged once for them)
constexpr int E4_WP = LORA + 2;          // padded W_UV row pitch (elements): rows start in distinct banks
constexpr int E4_SMEM = VH * E4_WP * 2 + E4_SLOTS * LORA * 4;

// grid (96, ceil(B / 16)); block 128 (v).  out[b][h][v] = bf16(sum_{j ascending} W_UV[h][v][j] o_lat[j]),
// sixteen slots' sums side by side in each thread.
__global__ void __launch_bounds__(VH) ex_expand_kernel(const uint16_t* __restrict__ olat, int B,
                                                      const uint16_t* __restrict__ w_kv_b,
                                                      uint16_t* __restrict__ out)
{
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ uint16_t ex_w[];
    float* ol = reinterpret_cast<float*>(ex_w + VH * E4_WP);  // [16][512]
    const int h = blockIdx.x, b0 = blockIdx.y * E4_SLOTS, v = threadIdx.x;
    const uint16_t* wsrc = w_kv_b + ((size_t)h * WROWS_PER_HEAD + NOPE) * LORA;
    for (int k = threadIdx.x; k < VH * (LORA / 2); k += VH) {
        const int r = k / (LORA / 2), c2 = k % (LORA / 2);
        reinterpret_cast<uint32_t*>(ex_w + r * E4_WP)[c2] = reinterpret_cast<const uint32_t*>(wsrc + (size_t)r * LORA)[c2];
    }
    for (int k = threadIdx.x; k < E4_SLOTS * LORA; k += VH) {
        const int s = k / LORA, j = k % LORA;
        ol[k] = (b0 + s < B) ? ex_bf(olat[((size_t)h * B + b0 + s) * LORA + j]) : 0.f;
    }
    __syncthreads();
    float acc[E4_SLOTS];
#pragma unroll
    for (int s = 0; s < E4_SLOTS; ++s) acc[s] = 0.f;
    const uint16_t* wr = ex_w + v * E4_WP;
    for (int j = 0; j < LORA; ++j) {
        const float w = ex_bf(wr[j]);
#pragma unroll
        for (int s = 0; s < E4_SLOTS; ++s) acc[s] = __fadd_rn(acc[s], __fmul_rn(w, ol[s * LORA + j]));
    }
#pragma unroll
    for (int s = 0; s < E4_SLOTS; ++s)
        if (b0 + s < B) out[((size_t)(b0 + s) * H + h) * VH + v] = ex_land(acc[s]);
}

}  // namespace k3

using namespace k3;

static size_t ex_pitch(int max_ctx) { return ((size_t)max_ctx + 7) / 8 * 8; }

extern "C" size_t k3mla_decode_exact_workspace_bytes(int B, int max_ctx)
{
    if (B <= 0 || max_ctx <= 0) return 0;
    const size_t sp = ((size_t)B * H * ex_pitch(max_ctx) * 2 + 255) & ~size_t(255);
    const size_t qa = ((size_t)B * H * ROW * 2 + 255) & ~size_t(255);
    return sp + qa + (size_t)B * H * LORA * 2;
}

extern "C" int k3mla_decode_exact(const uint16_t* q, const uint16_t* slab, int n_pages, int n_layers, int layer,
                                  const int32_t* block_table, int max_pages_per_slot, const int32_t* ctx_len,
                                  const uint16_t* w_kv_b, uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t,
                                  void* workspace, size_t ws_bytes, int B, int max_ctx, int32_t* dev_err,
                                  void* stream)
{
    if (B < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers || max_pages_per_slot <= 0 ||
        max_ctx <= 0) {
        set_error("k3mla_decode_exact: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if (!q || !slab || !block_table || !ctx_len || !w_kv_b || !out || !workspace || !aligned(q, 4) ||
        !aligned(slab, 16) || !aligned(out, 2) || !aligned(workspace, 256)) {
        set_error("k3mla_decode_exact: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    const size_t need = k3mla_decode_exact_workspace_bytes(B, max_ctx);
    if (ws_bytes < need) {
        set_error("k3mla_decode_exact: workspace %zu < %zu bytes", ws_bytes, need);
        return K3MLA_E_WORKSPACE;
    }
    const int nchunk = (max_ctx + E1_PAGES * PAGE - 1) / (E1_PAGES * PAGE);
    if ((size_t)max_ctx * 4 > (size_t)E2_MAX_SMEM) {
        set_error("k3mla_decode_exact: max_ctx above %d", E2_MAX_SMEM / 4);
        return K3MLA_E_INVALID;
    }
    if ((long long)B * H > 0x7FFFFFFFll || B > 65535 || nchunk > 65535) {
        set_error("k3mla_decode_exact: grid too large");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaFuncSetAttribute(ex_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, E1_SMEM);
        cudaFuncSetAttribute(ex_latent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, E3_SMEM);
        cudaFuncSetAttribute(ex_softmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, E2_MAX_SMEM);
        cudaFuncSetAttribute(ex_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, E4_SMEM);
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const int pitch = (int)ex_pitch(max_ctx);
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    uint16_t* sp = reinterpret_cast<uint16_t*>(ws);
    const size_t sp_bytes = ((size_t)B * H * pitch * 2 + 255) & ~size_t(255);
    uint16_t* q_abs = reinterpret_cast<uint16_t*>(ws + sp_bytes);
    const size_t qa_bytes = ((size_t)B * H * ROW * 2 + 255) & ~size_t(255);
    uint16_t* olat = reinterpret_cast<uint16_t*>(ws + sp_bytes + qa_bytes);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = launch_pdl(ex_absorb_kernel, dim3(B, H), dim3(LORA), 0, st, "ex_absorb_kernel", q, w_kv_b, q_abs);
    if (rc) return rc;
    rc = launch_pdl(ex_scores_kernel, dim3(B, nchunk), dim3(E1_THREADS), (size_t)E1_SMEM, st, "ex_scores_kernel",
                    q_abs, slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, ctx_len, max_ctx,
                    scale_bf16, sp, pitch, dev_err);
    if (rc) return rc;
    rc = launch_pdl(ex_softmax_kernel, dim3(B * H), dim3(E2_THREADS), (size_t)max_ctx * 4, st, "ex_softmax_kernel",
                    ctx_len, max_ctx, max_pages_per_slot, sp, pitch, argmax_t);
    if (rc) return rc;
    rc = launch_pdl(ex_latent_kernel, dim3(B, LORA / E3_DIMS), dim3(E3_THREADS), (size_t)E3_SMEM, st,
                    "ex_latent_kernel", slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, ctx_len, B,
                    max_ctx, sp, pitch, olat);
    if (rc) return rc;
    return launch_pdl(ex_expand_kernel, dim3(H, (B + E4_SLOTS - 1) / E4_SLOTS), dim3(VH), (size_t)E4_SMEM, st,
                      "ex_expand_kernel", olat, B, w_kv_b, out);
}
