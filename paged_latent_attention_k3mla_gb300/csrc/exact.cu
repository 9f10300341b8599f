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
//   E1 scores       CTA per (slot, 128 tokens): Q and the rows staged in shared
//                   memory by 32-dim chunks; thread per (8 tokens, 8 heads): sums
//                   over k = 0..575
//   E2 softmax      CTA per (slot, head): max and exps across the block, the sum
//                   of exp thread 0's loop over t ascending, p_t = bf16(e_t / l),
//                   argmax (lowest t with the largest p)
//   E3 latent sum   CTA per (slot, 64 dims): thread per (8 dims, 6 heads), sums
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
constexpr int E1_TB = 2 * PAGE;          // tokens per CTA
constexpr int E1_KC = 32;                // dims per staged chunk (576 = 18 chunks)
constexpr int E1_NKC = ROW / E1_KC;
constexpr int E1_TT = 8, E1_HT = 8;      // register tile of one thread: 8 tokens x 8 heads
constexpr int E1_THREADS = (E1_TB / E1_TT) * (H / E1_HT);  // 16 token groups x 12 head groups = 192
constexpr int E1_RP = E1_TB + 4;         // Rs row pitch (floats): 16-byte rows, rows 4 banks apart
constexpr int E1_BUF = E1_KC * (E1_RP + H);  // one stage: Rs [KC][RP] + Qs [KC][96], f32
constexpr int E1_SMEM = 2 * E1_BUF * 4;
constexpr int E1_RPIECES = E1_TB * E1_KC / 8;  // 512 pieces of 8 dims of a row per chunk
constexpr int E1_QPIECES = H * E1_KC / 8;      // 384 pieces of 8 dims of Q per chunk
static_assert(E1_THREADS == 192 && E1_QPIECES == 2 * E1_THREADS && E1_RPIECES <= 3 * E1_THREADS, "staging split");
static_assert(H * E1_TB * 2 <= E1_SMEM, "the bf16 score tile fits in the staging buffers");

// grid (B, ceil(max_ctx / 128)); block 192.  s[b][h][t] = bf16(bf16(dot) * scale).  Q and the 128
// tokens' rows are staged in chunks of 32 dims as f32, transposed ([k][token], [k][head]) and
// double-buffered (the next chunk's loads are in flight while this one is used).  Thread (warp w,
// lane l): tokens 8 tg .. 8 tg + 7 with tg = 8 (w & 1) + (l & 7), heads 8 hg .. 8 hg + 7 with hg =
// 4 (w >> 1) + (l >> 3); each of its 64 dots is one sequential sum over k = 0..575 ascending (a fused
// multiply-add of two bf16 values rounds as the chain's multiply-then-add: the product is exact).
__global__ void __launch_bounds__(E1_THREADS) ex_scores_kernel(
    const uint16_t* __restrict__ q_abs, const uint16_t* __restrict__ slab, int n_pages, int n_layers, int layer,
    const int32_t* __restrict__ table, int max_pages, const int32_t* __restrict__ ctx_len, int max_ctx,
    uint16_t scale_bf16, uint16_t* __restrict__ s_out, int s_pitch, int32_t* dev_err)
{
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ float ex_sf[];
    const int b = blockIdx.x;
    const int n = ex_ctx(ctx_len, b, max_ctx, max_pages);
    const int t_begin = blockIdx.y * E1_TB;
    if (t_begin >= n) return;
    const int t_end = min(n, t_begin + E1_TB);
    const int tid = (int)threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tg = 8 * (warp & 1) + (lane & 7), hg = 4 * (warp >> 1) + (lane >> 3);
    // staging roles: row piece i = tid + 192 e (e < 3, i < 512): token i % 128, dims 8 (i / 128) .. + 7;
    // Q piece i = tid + 192 e (e < 2): head i / 4, dims 8 (i % 4) .. + 7
    const uint16_t* srow[3];
#pragma unroll
    for (int e = 0; e < 3; ++e) {
        const int i = tid + E1_THREADS * e, t = t_begin + (i & (E1_TB - 1));
        srow[e] = (i < E1_RPIECES && t < t_end) ? ex_row(slab, n_pages, n_layers, layer, table, max_pages, b, t, dev_err)
                                                : nullptr;
    }
    const uint16_t* qrow = q_abs + (size_t)b * H * ROW;
    uint4 rv[3], qv[2];
    auto load = [&](int kc) {
        const int k0 = kc * E1_KC;
#pragma unroll
        for (int e = 0; e < 3; ++e) {
            const int i = tid + E1_THREADS * e;
            rv[e] = srow[e] ? *reinterpret_cast<const uint4*>(srow[e] + k0 + 8 * (i >> 7)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = tid + E1_THREADS * e;
            qv[e] = *reinterpret_cast<const uint4*>(qrow + (size_t)(i >> 2) * ROW + k0 + 8 * (i & 3));
        }
    };
    auto store = [&](int buf) {
        float* Rs = ex_sf + buf * E1_BUF;
        float* Qs = Rs + E1_KC * E1_RP;
#pragma unroll
        for (int e = 0; e < 3; ++e) {
            const int i = tid + E1_THREADS * e;
            if (i < E1_RPIECES) {
                const uint32_t w[4] = {rv[e].x, rv[e].y, rv[e].z, rv[e].w};
                const int t = i & (E1_TB - 1), kb = 8 * (i >> 7);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    Rs[(kb + 2 * u) * E1_RP + t] = __uint_as_float(w[u] << 16);
                    Rs[(kb + 2 * u + 1) * E1_RP + t] = __uint_as_float(w[u] & 0xFFFF0000u);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = tid + E1_THREADS * e;
            const uint32_t w[4] = {qv[e].x, qv[e].y, qv[e].z, qv[e].w};
            const int h = i >> 2, kb = 8 * (i & 3);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                Qs[(kb + 2 * u) * H + h] = __uint_as_float(w[u] << 16);
                Qs[(kb + 2 * u + 1) * H + h] = __uint_as_float(w[u] & 0xFFFF0000u);
            }
        }
    };
    float acc[E1_TT][E1_HT];
#pragma unroll
    for (int a = 0; a < E1_TT; ++a)
#pragma unroll
        for (int c = 0; c < E1_HT; ++c) acc[a][c] = 0.f;
    load(0);
    store(0);
    __syncthreads();
#pragma unroll 1
    for (int kc = 0; kc < E1_NKC; ++kc) {
        if (kc + 1 < E1_NKC) load(kc + 1);  // in flight while chunk kc is used
        const float* Rs = ex_sf + (kc & 1) * E1_BUF;
        const float* Qs = Rs + E1_KC * E1_RP;
#pragma unroll 4
        for (int k = 0; k < E1_KC; ++k) {
            const float4 r0 = *reinterpret_cast<const float4*>(Rs + k * E1_RP + 8 * tg);
            const float4 r1 = *reinterpret_cast<const float4*>(Rs + k * E1_RP + 8 * tg + 4);
            const float4 q0 = *reinterpret_cast<const float4*>(Qs + k * H + 8 * hg);
            const float4 q1 = *reinterpret_cast<const float4*>(Qs + k * H + 8 * hg + 4);
            const float r[E1_TT] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            const float q[E1_HT] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
            for (int a = 0; a < E1_TT; ++a)
#pragma unroll
                for (int c = 0; c < E1_HT; ++c) acc[a][c] = __fmaf_rn(q[c], r[a], acc[a][c]);
        }
        if (kc + 1 < E1_NKC) store((kc + 1) & 1);
        __syncthreads();
    }
    // the landed scores through shared memory ([96 heads][128 tokens] bf16), then row by row
    const float scale = ex_bf(scale_bf16);
    uint16_t* S = reinterpret_cast<uint16_t*>(ex_sf);
#pragma unroll
    for (int a = 0; a < E1_TT; ++a)
#pragma unroll
        for (int c = 0; c < E1_HT; ++c)
            S[(8 * hg + c) * E1_TB + 8 * tg + a] = ex_land(__fmul_rn(ex_bf(ex_land(acc[a][c])), scale));
    __syncthreads();
    const int cnt = t_end - t_begin;
    for (int i = tid; i < H * (E1_TB / 8); i += E1_THREADS) {
        const int h = i / (E1_TB / 8), j = 8 * (i % (E1_TB / 8));
        uint16_t* dst = s_out + ((size_t)b * H + h) * s_pitch + t_begin + j;
        const uint16_t* src = S + h * E1_TB + j;
        if (j + 8 <= cnt) {
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
        } else {
            for (int e = 0; j + e < cnt; ++e) dst[e] = src[e];
        }
    }
}

// ---- the chain's exp: f32 of the exact exponential --------------------------------------------
// The chain takes e_t as the double exponential rounded once to f32, which is the f32 nearest to
// e^x unless e^x lies within a double rounding error of a point halfway between two f32 values.
// FP64 runs at a small fraction of the FP32 rate here, so the exp is first evaluated in f32 pairs
// (an unevaluated sum hi + lo; Knuth's and Dekker's error-free sums, the exact product from the fused
// multiply-add), by table-driven argument reduction (Tang, 1989) with a Cody-Waite split constant:
//   x = k ln2 / 32 + r, |r| <= ln2 / 64, with ln2 / 32 split as L1 + L2 + L3 (L1, L2 short enough that
//   k L1 and k L2 are exact for |k| < 2^12, so x - k L1 is exact);
//   e^r = 1 + r + r^2 / 2 + tail, tail = r^3 / 6 + r^4 / 24 + r^5 / 120 in plain f32 (|tail| < 2.2e-7;
//   the truncation r^6 / 720 < 2^-48);
//   e^x = 2^(k >> 5) * 2^((k & 31) / 32) * e^r, the 32 values 2^(j/32) as f32 pairs (X_TH, X_TL, each
//   the f32 nearest to 2^(j/32) and to the remainder).
// The pair's error is below 2^-43 of e^x over the whole range used (measured over every f32 in
// [-87, 0] against a long-double reference).  When the pair lies farther than 2^-40 e^x from every
// rounding boundary of the f32 grid, its rounding is the rounding of e^x, and is returned; otherwise
// (a few in 10^5 arguments), and for x outside [-87, 0], the double exponential decides.
__device__ __constant__ float X_TH[32] = {
    0x1.000000p+0f, 0x1.059b0ep+0f, 0x1.0b5586p+0f, 0x1.11301ep+0f, 0x1.172b84p+0f, 0x1.1d4874p+0f, 0x1.2387a6p+0f,
    0x1.29e9e0p+0f, 0x1.306fe0p+0f, 0x1.371a74p+0f, 0x1.3dea64p+0f, 0x1.44e086p+0f, 0x1.4bfdaep+0f, 0x1.5342b6p+0f,
    0x1.5ab07ep+0f, 0x1.6247ecp+0f, 0x1.6a09e6p+0f, 0x1.71f75ep+0f, 0x1.7a1148p+0f, 0x1.82589ap+0f, 0x1.8ace54p+0f,
    0x1.93737cp+0f, 0x1.9c4918p+0f, 0x1.a5503cp+0f, 0x1.ae89fap+0f, 0x1.b7f770p+0f, 0x1.c199bep+0f, 0x1.cb720ep+0f,
    0x1.d5818ep+0f, 0x1.dfc974p+0f, 0x1.ea4afap+0f, 0x1.f50766p+0f};
__device__ __constant__ float X_TL[32] = {
    0.0f, -0x1.9d4f52p-25f, 0x1.9f3122p-25f, -0x1.fdb496p-25f, -0x1.c15742p-27f, -0x1.d2e8cap-25f, 0x1.ceac48p-25f,
    -0x1.5c0424p-25f, 0x1.4636e2p-25f, -0x1.18aac6p-25f, 0x1.824684p-25f, 0x1.8624b4p-30f, -0x1.593abcp-25f,
    -0x1.2c5610p-25f, -0x1.5bd5ecp-27f, -0x1.f8b550p-25f, 0x1.9fcef4p-26f, 0x1.1d8beep-25f, -0x1.829fd0p-25f,
    -0x1.accc7cp-26f, 0x1.15506ep-27f, -0x1.e64744p-25f, 0x1.51f848p-27f, -0x1.b83b54p-25f, -0x1.a94b14p-26f,
    -0x1.a09438p-25f, -0x1.3d56b2p-27f, -0x1.8837ccp-27f, -0x1.822dbcp-27f, -0x1.908c94p-25f, 0x1.52486cp-27f,
    -0x1.246eb0p-26f};

// Error-free transformations: a + b = s + e exactly (any order of magnitude; Knuth), and the same when
// |a| >= |b| (Dekker).
__device__ __forceinline__ void x_two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void x_fast_two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// f32 of e^x as the chain defines it; `tl` / `th`: the 2^(j/32) pairs (shared or constant memory).
// *fast (optional) tells whether the f32 pair decided.
__device__ __forceinline__ float ex_exp(float x, const float* th, const float* tl, bool* fast = nullptr)
{
    if (x >= -87.0f && x <= 0.0f) {
        const float kf = rintf(__fmul_rn(x, 0x1.715476p+5f));  // 32 / ln2
        const int k = (int)kf;
        const float rhi = __fsub_rn(x, __fmul_rn(kf, 0x1.62ep-6f));  // exact
        float rh, rl;
        x_two_sum(rhi, -__fmul_rn(kf, 0x1.0cp-20f), rh, rl);
        rl = __fmaf_rn(-kf, -0x1.05c61p-34f, rl);
        x_fast_two_sum(rh, rl, rh, rl);  // |rl| <= ulp(rh) / 2
        const float a = __fmul_rn(rh, rh);
        const float ae = __fmaf_rn(rh, rh, -a);  // rh^2 = a + ae
        float t = __fmaf_rn(rh, 1.0f / 120.0f, 1.0f / 24.0f);
        t = __fmaf_rn(rh, t, 1.0f / 6.0f);
        const float tail = __fmul_rn(__fmul_rn(a, rh), t);
        float s, se, s2, se2;
        x_two_sum(1.0f, rh, s, se);
        x_two_sum(s, __fmul_rn(0.5f, a), s2, se2);
        const float lo = __fadd_rn(
            __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(se, se2), __fmul_rn(0.5f, ae)), tail), rl), __fmul_rn(rh, rl));
        float eh, el;
        x_fast_two_sum(s2, lo, eh, el);
        const int j = k & 31, m = k >> 5;
        const float ph = __fmul_rn(eh, th[j]);
        const float pe = __fmaf_rn(eh, th[j], -ph);
        const float q = __fadd_rn(__fadd_rn(pe, __fmul_rn(eh, tl[j])), __fmul_rn(el, th[j]));
        float yh, yl;
        x_fast_two_sum(ph, q, yh, yl);
        const uint32_t bits = __float_as_uint(yh);
        const float ulp = __uint_as_float((((bits >> 23) & 0xFFu) - 23u) << 23);
        const float h = (yl < 0.0f && (bits & 0x7FFFFFu) == 0u) ? 0.25f * ulp : 0.5f * ulp;
        if (__fadd_rn(fabsf(yl), __fmul_rn(0x1p-40f, yh)) < h) {
            if (fast) *fast = true;
            return __fmul_rn(yh, __uint_as_float((uint32_t)(m + 127) << 23));  // exact: a normal f32
        }
    }
    if (fast) *fast = false;
    return (float)exp((double)x);
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
    __shared__ float x_th[32], x_tl[32];  // indexed per thread: shared, not constant, memory
    if (threadIdx.x < 32) {
        x_th[threadIdx.x] = X_TH[threadIdx.x];
        x_tl[threadIdx.x] = X_TL[threadIdx.x];
    }
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
    for (int t = threadIdx.x; t < n; t += E2_THREADS) ex_e[t] = ex_exp(__fsub_rn(ex_bf(row[t]), m), x_th, x_tl);
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

// Diagnostic: the chain's exp on n arguments; fast[i] = 1 where the f32 pair decided.
__global__ void ex_exp_diag_kernel(const float* __restrict__ x, float* __restrict__ y, int32_t* __restrict__ fast,
                                   int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    bool f = false;
    y[i] = ex_exp(x[i], X_TH, X_TL, &f);
    if (fast) fast[i] = f ? 1 : 0;
}

// ---- E3: latent sum --------------------------------------------------------------------------
constexpr int E3_THREADS = 128;          // (8 groups of 8 dims) x (16 groups of 6 heads)
constexpr int E3_DIMS = 64;              // latent dims per CTA
constexpr int E3_PP = 100;               // ps row pitch (floats): 8-byte aligned 6-head groups
constexpr int E3_SMEM = PAGE * E3_DIMS * 4 + PAGE * E3_PP * 4;  // c slice [64][64] f32 + p [64][100] f32
constexpr int E3_CV = PAGE * E3_DIMS / 8 / E3_THREADS;           // 16-byte c pieces per thread and page (4)
constexpr int E3_PV = H * PAGE / 8 / E3_THREADS;                 // 16-byte p pieces per thread and page (6)
static_assert(E3_CV * 8 * E3_THREADS == PAGE * E3_DIMS && E3_PV * 8 * E3_THREADS == H * PAGE, "staging split");

// grid (B, 512 / 64); o_lat[h][b][j] = bf16(sum_{t ascending} p_t c_t[j]).  Thread i: dims 8 (i % 8) ..
// + 7 of the block and heads 6 (i / 8) .. + 5, each of its 48 sums one sequential loop over t ascending
// (fused multiply-add of two bf16 values: the product is exact).  A page's c slice and probabilities
// are staged in shared memory as f32; the next page's are loaded into registers while this one is used.
__global__ void __launch_bounds__(E3_THREADS, 4) ex_latent_kernel(
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
    const int tid = (int)threadIdx.x;
    const int dg = tid & 7, hg = 6 * (tid >> 3);
    const uint16_t* prow = p + (size_t)b * H * s_pitch;
    uint4 cv[E3_CV], pv[E3_PV];
    // c piece m: token (tid + 128 m) / 8, dims 8 ((tid + 128 m) % 8); p piece m: head (tid + 128 m) % 96,
    // tokens 8 ((tid + 128 m) / 96) .. + 7 (a warp's lanes take 32 heads of one token group)
    auto load = [&](int t0) {
        const int cnt = min(PAGE, n - t0);
#pragma unroll
        for (int m = 0; m < E3_CV; ++m) {
            const int i = tid + E3_THREADS * m, r = i >> 3, u = i & 7;
            const uint16_t* row = r < cnt ? ex_row(slab, n_pages, n_layers, layer, table, max_pages, b, t0 + r, nullptr)
                                          : nullptr;
            cv[m] = row ? *reinterpret_cast<const uint4*>(row + jb + 8 * u) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < E3_PV; ++m) {
            const int i = tid + E3_THREADS * m, h = i % H, r0 = 8 * (i / H);
            if (r0 + 8 <= cnt) {
                pv[m] = *reinterpret_cast<const uint4*>(prow + (size_t)h * s_pitch + t0 + r0);
            } else {  // the last, partial group of the context: zeros past it
                uint16_t e[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) e[k] = r0 + k < cnt ? prow[(size_t)h * s_pitch + t0 + r0 + k] : (uint16_t)0;
                pv[m] = make_uint4((uint32_t)e[0] | ((uint32_t)e[1] << 16), (uint32_t)e[2] | ((uint32_t)e[3] << 16),
                                   (uint32_t)e[4] | ((uint32_t)e[5] << 16), (uint32_t)e[6] | ((uint32_t)e[7] << 16));
            }
        }
    };
    auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
    auto hi = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
    float acc[6][8];
#pragma unroll
    for (int u = 0; u < 6; ++u)
#pragma unroll
        for (int d = 0; d < 8; ++d) acc[u][d] = 0.f;
    if (n > 0) load(0);
    for (int t0 = 0; t0 < n; t0 += PAGE) {
        const int cnt = min(PAGE, n - t0);
        __syncthreads();  // the previous page is no longer read
#pragma unroll
        for (int m = 0; m < E3_CV; ++m) {
            const int i = tid + E3_THREADS * m, r = i >> 3, u = i & 7;
            float4* dst = reinterpret_cast<float4*>(cs + r * E3_DIMS + 8 * u);
            dst[0] = make_float4(lo(cv[m].x), hi(cv[m].x), lo(cv[m].y), hi(cv[m].y));
            dst[1] = make_float4(lo(cv[m].z), hi(cv[m].z), lo(cv[m].w), hi(cv[m].w));
        }
#pragma unroll
        for (int m = 0; m < E3_PV; ++m) {
            const int i = tid + E3_THREADS * m, h = i % H, r0 = 8 * (i / H);
            const uint32_t w[4] = {pv[m].x, pv[m].y, pv[m].z, pv[m].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ps[(r0 + 2 * k) * E3_PP + h] = lo(w[k]);
                ps[(r0 + 2 * k + 1) * E3_PP + h] = hi(w[k]);
            }
        }
        __syncthreads();
        if (t0 + PAGE < n) load(t0 + PAGE);  // in flight while this page is used
        // operands of token r + 1 are loaded while token r's 48 fmas run (shared-memory latency); the
        // staged rows past cnt are zeros, so the load one past the last token stays in the tile
        float4 c0 = *reinterpret_cast<const float4*>(cs + 8 * dg);
        float4 c1 = *reinterpret_cast<const float4*>(cs + 8 * dg + 4);
        float2 p0 = *reinterpret_cast<const float2*>(ps + hg);
        float2 p1 = *reinterpret_cast<const float2*>(ps + hg + 2);
        float2 p2 = *reinterpret_cast<const float2*>(ps + hg + 4);
#pragma unroll 2
        for (int r = 0; r < cnt; ++r) {
            const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            const float pp[6] = {p0.x, p0.y, p1.x, p1.y, p2.x, p2.y};
            const int rn = r + 1 < PAGE ? r + 1 : r;
            c0 = *reinterpret_cast<const float4*>(cs + rn * E3_DIMS + 8 * dg);
            c1 = *reinterpret_cast<const float4*>(cs + rn * E3_DIMS + 8 * dg + 4);
            p0 = *reinterpret_cast<const float2*>(ps + rn * E3_PP + hg);
            p1 = *reinterpret_cast<const float2*>(ps + rn * E3_PP + hg + 2);
            p2 = *reinterpret_cast<const float2*>(ps + rn * E3_PP + hg + 4);
#pragma unroll
            for (int u = 0; u < 6; ++u)
#pragma unroll
                for (int d = 0; d < 8; ++d) acc[u][d] = __fmaf_rn(pp[u], c[d], acc[u][d]);
        }
    }
#pragma unroll
    for (int u = 0; u < 6; ++u) {
        uint4 o;
        o.x = (uint32_t)ex_land(acc[u][0]) | ((uint32_t)ex_land(acc[u][1]) << 16);
        o.y = (uint32_t)ex_land(acc[u][2]) | ((uint32_t)ex_land(acc[u][3]) << 16);
        o.z = (uint32_t)ex_land(acc[u][4]) | ((uint32_t)ex_land(acc[u][5]) << 16);
        o.w = (uint32_t)ex_land(acc[u][6]) | ((uint32_t)ex_land(acc[u][7]) << 16);
        *reinterpret_cast<uint4*>(olat + ((size_t)(hg + u) * B + b) * LORA + jb + 8 * dg) = o;
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
    const int nchunk = (max_ctx + E1_TB - 1) / E1_TB;
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

extern "C" int k3mla_diag_exact_exp(const float* x, float* y, int32_t* fast, int n, void* stream)
{
    if (n < 0 || (n > 0 && (!x || !y || !aligned(x, 4) || !aligned(y, 4)))) {
        set_error("k3mla_diag_exact_exp: invalid arguments");
        return K3MLA_E_INVALID;
    }
    if (n == 0) return K3MLA_OK;
    if (!device_ok()) return K3MLA_E_DEVICE;
    return launch_pdl(ex_exp_diag_kernel, dim3((n + 255) / 256), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                      "ex_exp_diag_kernel", x, y, fast, n);
}
