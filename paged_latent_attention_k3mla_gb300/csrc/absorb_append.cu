// absorb_append.cu -- q absorption and the latent-row append.
//
// q absorption (pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode",
// M2 commit: "q_abs = W_UK^T q_nope is precomputed" and "q absorption lands
// bf16"): q_abs[b][h][j] = bf16(sum_d W_UK[h][d][j] q_nope[b][h][d]) for j < 512,
// then q_rope is copied to q_abs[b][h][512:576].  Per head this is a dense
// product across slots, Q_abs_h^T [512 x B] = W_UK[h]^T [512 x 128] . Q_nope_h^T
// [128 x B], whose cost is reading W_UK (12.6 MB per layer).  It runs on the
// 5th-generation tensor cores, one CTA per (head, tile of NB slots): W_UK[h] lands
// as the MN-major A operand ([8 chunks of 64 j][128 d][128 B], 128-byte swizzle) in
// eight TMA boxes, sixteen warps write the q_nope tile as the K-major B operand
// ([2 chunks of 64 d][NB slots][128 B]), and 32 MMAs (4 blocks of 128 j x 8 K
// steps) fill four 128 x NB f32 TMEM accumulators that the warps read back.  NB is
// 64 for batches of up to 64 slots and 128 above: one CTA per head then covers up to
// 128 slots (one wave on the GPU, W_UK read once) where 64-slot tiles would take
// two waves and read every W_UK[h] twice.
//
// Append (same PR, M1 commit): the new token's 512-wide latent and 64-wide rope
// key land in row ((page * L + layer) * 64 + pos % 64) of the page-first slab,
// page = block_table[b][pos / 64]; the element index is size_t (the slab passes
// 2^31 elements).  The append runs as its own kernel (k3mla_append_latent) or
// inside the absorption's grid (k3mla_absorb_q_append): the decode step does the
// two back to back and neither reads what the other writes, so one launch serves
// both and leaves one launch's latency off the chain into the decode.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int AB_WARPS = 16;
constexpr int AB_THREADS = 32 * AB_WARPS;
constexpr int AB_ROWS_PER_PASS = AB_THREADS / 8;  // slots staged / written per pass (8 threads a slot)
constexpr int AB_A_BYTES = 8 * NOPE * 128;        // W_UK[h]: 8 j-chunks x 128 d rows x 128 B
constexpr uint64_t AB_WAIT_NS = 1000000000ull;

// Slots per CTA (the MMA's N): the q_nope tile (2 d-chunks x NB slots x 128 B), the instruction
// descriptor (A MN-major, B K-major) and the TMEM of the four 128 x NB accumulators.
template <int NB>
struct AbTile {
    static_assert(NB == 64 || NB == 128, "64 or 128 slots per CTA");
    static constexpr int B_BYTES = 2 * NB * 128;
    static constexpr uint32_t IDESC = make_idesc_bf16(128, NB, 1, 0);
    static constexpr uint32_t TMEM = 4 * NB;
    static_assert(NB * LORA * 2 <= AB_A_BYTES, "the bf16 result tile fits over the W_UK buffer");
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Bounded mbarrier wait: false (and K3MLA_DEV_TIMEOUT when dev_err is given) after 1 s.
__device__ __noinline__ bool ab_wait(uint64_t* bar, uint32_t parity, int32_t* dev_err)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_test_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity)) {
        if (globaltimer() - t0 > AB_WAIT_NS) {
            if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// The append of one layer-call, carried by the absorption's launch (k3mla_absorb_q_append); B == 0
// when there is none.
struct AppendJob {
    uint16_t* slab;
    const int32_t* table;
    const int32_t* pos;
    const uint16_t* c_kv;
    const uint16_t* k_rope;
    int32_t* dev_err;
    int64_t c_stride, r_stride;
    int n_pages, n_layers, layer, max_pages, B;
    int pos_is_ctx;  // `pos` holds context lengths: the write position is pos[b] - 1
};
constexpr int AP_THREADS = 96;  // a row is 288 32-bit words: three per thread

// One slot's row: the slab row index (or -1 when the slot writes nothing) and this thread's three
// words of it (words w = at, at + 96, at + 192; latent below 256, rope from 256).
__device__ __forceinline__ int64_t append_fetch(const AppendJob& ap, int b, int at, uint32_t (&v)[3])
{
    const uint32_t* src_c = reinterpret_cast<const uint32_t*>(ap.c_kv + (size_t)b * ap.c_stride);
    const uint32_t* src_r = reinterpret_cast<const uint32_t*>(ap.k_rope + (size_t)b * ap.r_stride);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int w = at + AP_THREADS * k;
        v[k] = (w < LORA / 2) ? src_c[w] : src_r[w - LORA / 2];
    }
    const int p = ap.pos[b] - (ap.pos_is_ctx ? 1 : 0);
    if (p < 0) return -1;
    const int lp = p / PAGE;
    const int32_t id = (lp < ap.max_pages) ? ap.table[(size_t)b * ap.max_pages + lp] : -1;
    if (id < 0 || id >= ap.n_pages) {
        if (at == 0 && ap.dev_err) atomicOr(ap.dev_err, (int)K3MLA_DEV_UNMAPPED);
        return -1;
    }
    return ((int64_t)id * ap.n_layers + ap.layer) * PAGE + p % PAGE;
}

__device__ __forceinline__ void append_store(const AppendJob& ap, int64_t row, int at, const uint32_t (&v)[3])
{
    if (row < 0) return;
    uint32_t* dst = reinterpret_cast<uint32_t*>(ap.slab + (size_t)row * ROW);
#pragma unroll
    for (int k = 0; k < 3; ++k) dst[at + AP_THREADS * k] = v[k];
}

// grid (96 heads, ceil(B / NB) slot tiles); block AB_THREADS; thread 0 also issues the loads and MMAs.
template <int NB>
__global__ void __launch_bounds__(AB_THREADS, 1)
    k3mla_absorb_kernel(const __grid_constant__ CUtensorMap tmap_w, const uint16_t* __restrict__ q,
                        uint16_t* __restrict__ q_abs, int B, const AppendJob ap)
{
    using T = AbTile<NB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sb = sa + AB_A_BYTES;
    __shared__ uint64_t w_full, b_ready, d_full;
    __shared__ uint32_t tmem_slot;
    const int h = blockIdx.x;
    const int b0 = blockIdx.y * NB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&w_full, 1);
        mbar_init(&b_ready, AB_THREADS);
        mbar_init(&d_full, 1);
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, T::TMEM);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    if (threadIdx.x == 0) {  // W_UK[h] = w_kv_b rows h*256 .. h*256 + 127 ([d][j]), one box per 64 j
        mbar_arrive_expect_tx(&w_full, AB_A_BYTES);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            tma_load_3d_hint(sa + c * (NOPE * 128), &tmap_w, 0, h * WROWS_PER_HEAD, c, &w_full,
                             policy_evict_first());  // read once per layer
    }
    // the set-up and the weight load above overlap the previous kernel in the stream (the weights
    // are not written by it: see k3mla_absorb_q); q, q_abs and the append's buffers wait for it
    griddep_wait();
    griddep_launch_dependents();

    // The append (when this launch carries one): CTA `lin` writes the rows of slots lin, lin + ncta,
    // ... (one slot per CTA unless B exceeds the grid's CTAs) with its last AP_THREADS threads, once
    // their share of the B operand is written: the row's position and page id are two dependent
    // loads, which would hold the B operand (and the MMAs) back if they came first.
    const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x);
    const int ncta = (int)(gridDim.x * gridDim.y);
    const int at = (int)threadIdx.x - (AB_THREADS - AP_THREADS);
    const bool app_thread = lin < ap.B && at >= 0;

    {   // q_nope of the tile -> B operand; q_rope -> q_abs[..][512:576].  thread -> (slot r, segment seg)
        const int seg = threadIdx.x & 7;
#pragma unroll
        for (int r = threadIdx.x >> 3; r < NB; r += AB_ROWS_PER_PASS) {
            const int b = b0 + r;
            const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)b * H + h) * QDIM);
#pragma unroll
            for (int e = 0; e < 2; ++e) {  // 16-byte unit u = 2 seg + e: dims 8u .. 8u+7
                const int u = 2 * seg + e;
                const uint4 v = (b < B) ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
                const int c = u >> 3, uu = u & 7;
                *reinterpret_cast<uint4*>(sb + c * (NB * 128) + r * 128 + ((uu ^ (r & 7)) << 4)) = v;
            }
            if (b < B)
                reinterpret_cast<uint4*>(q_abs + ((size_t)b * H + h) * ROW + LORA)[seg] =
                    __ldg(src + NOPE / 8 + seg);
        }
        fence_proxy_async_cta();  // generic-proxy stores -> visible to the tensor core
        mbar_arrive(&b_ready);
    }
    if (app_thread) {
        for (int sl = lin; sl < ap.B; sl += ncta) {  // more than one slot only when B exceeds the grid's CTAs
            uint32_t av[3];
            const int64_t arow = append_fetch(ap, sl, at, av);
            append_store(ap, arow, at, av);
        }
    }
    if (threadIdx.x == 0) {
        const bool ok = ab_wait(&w_full, 0, nullptr) && ab_wait(&b_ready, 0, nullptr);
        if (ok) {
            tc_fence_after();
            const uint64_t ad = make_sdesc(smem_u32(sa), NOPE * 128, 1024);  // LBO: next 64-j chunk
            const uint64_t bd = make_sdesc(smem_u32(sb), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < NOPE / 16; ++ks)
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)  // four independent accumulators in turn
                    umma_ss(tbase + (uint32_t)(NB * mt),
                            ad + (uint64_t)((mt * 2 * NOPE * 128 + ks * 16 * 128) >> 4),
                            bd + (uint64_t)(((ks >> 2) * (NB * 128) + (ks & 3) * 32) >> 4), T::IDESC,
                            ks > 0 ? 1u : 0u);
        } else {
            const uint64_t t0 = globaltimer();  // let an in-flight TMA land before the CTA can exit
            while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
        }
        umma_commit(&d_full);
    }
    {   // epilogue: warp (quarter q, block mt) reads j = 128 mt + 32 q + lane for 32 of the tile's slots at
        // a time and lands bf16 values in a [NB slots][512] tile over the (now idle) W_UK buffer; once
        // those 32 slots are staged, the CTA writes their 1 KB rows of q_abs with 16-byte stores (measured
        // faster here than one thread's bulk tensor stores of the same tile) while the next 32 are staged
        const int qq = warp & 3, mt = warp >> 2;
        const bool got = __all_sync(0xFFFFFFFFu, ab_wait(&d_full, 0, nullptr));
        uint16_t* tile = reinterpret_cast<uint16_t*>(sa);
        if (got) tc_fence_after();
        const int j = 128 * mt + 32 * qq + lane;
        const int seg = threadIdx.x & 15;  // thread -> (slot 32 piece + tid / 16, 16-byte units 16k + seg)
#pragma unroll
        for (int piece = 0; piece < NB / 32; ++piece) {
            if (got) {
                uint32_t acc[32];
                tmem_ld32(tbase + ((uint32_t)(32 * qq) << 16) + (uint32_t)(NB * mt + 32 * piece), acc);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    tile[(32 * piece + k) * LORA + j] = (uint16_t)(pack2(__uint_as_float(acc[k]), 0.f) & 0xFFFFu);
            }
            __syncthreads();
            static_assert(AB_THREADS == 16 * 32, "16 threads a slot row, 32 rows a piece");
            const int r = 32 * piece + (threadIdx.x >> 4);
            if (b0 + r < B) {
                const uint4* srow = reinterpret_cast<const uint4*>(tile + r * LORA);
                uint4* drow = reinterpret_cast<uint4*>(q_abs + ((size_t)(b0 + r) * H + h) * ROW);
#pragma unroll
                for (int k = 0; k < 4; ++k) drow[seg + 16 * k] = srow[seg + 16 * k];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, T::TMEM);
}

// one CTA of 96 threads per slot; each thread moves three 32-bit words
__global__ void __launch_bounds__(96) k3mla_append_kernel(uint16_t* __restrict__ slab, int n_pages, int n_layers,
                                                            int layer, const int32_t* __restrict__ table,
                                                            int max_pages, const int32_t* __restrict__ pos,
                                                            const uint16_t* __restrict__ c_kv, int64_t c_stride,
                                                            const uint16_t* __restrict__ k_rope, int64_t r_stride,
                                                            int32_t* dev_err)
{
    griddep_wait();
    griddep_launch_dependents();
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

static int check_absorb(const char* who, const uint16_t* q, const uint16_t* w_kv_b, const uint16_t* q_abs, int B)
{
    if (B < 0) {
        set_error("%s: B < 0", who);
        return K3MLA_E_INVALID;
    }
    if (B > 0 && (!q || !w_kv_b || !q_abs || !aligned(q, 16) || !aligned(w_kv_b, 16) || !aligned(q_abs, 16))) {
        set_error("%s: null or misaligned pointer", who);
        return K3MLA_E_INVALID;
    }
    return K3MLA_OK;
}

static int check_append(const char* who, const uint16_t* slab, int n_pages, int n_layers, int layer,
                        const int32_t* block_table, int max_pages_per_slot, const int32_t* pos,
                        const uint16_t* c_kv, int64_t c_stride, const uint16_t* k_rope, int64_t r_stride, int B)
{
    if (B < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers || max_pages_per_slot <= 0 ||
        c_stride < LORA || r_stride < ROPE || (c_stride & 1) || (r_stride & 1)) {
        set_error("%s: invalid sizes or strides", who);
        return K3MLA_E_INVALID;
    }
    if (B > 0 && (!slab || !block_table || !pos || !c_kv || !k_rope || !aligned(slab, 4) || !aligned(c_kv, 4) ||
                  !aligned(k_rope, 4))) {
        set_error("%s: null or misaligned pointer", who);
        return K3MLA_E_INVALID;
    }
    return K3MLA_OK;
}

static int launch_absorb(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, int B, const AppendJob& ap,
                         void* stream)
{
    if (!device_ok()) return K3MLA_E_DEVICE;
    static bool attr_set[2][64] = {};
    const bool wide = B > 64;  // 128 slots per CTA: one CTA per head up to 128 slots
    const int nb = wide ? 128 : 64;
    const int smem = AB_A_BYTES + (wide ? AbTile<128>::B_BYTES : AbTile<64>::B_BYTES) + 1024;
    const void* fn = wide ? reinterpret_cast<const void*>(k3mla_absorb_kernel<128>)
                          : reinterpret_cast<const void*>(k3mla_absorb_kernel<64>);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[wide][dev]) {
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (dev >= 0 && dev < 64) attr_set[wide][dev] = true;
    }
    // w_kv_b viewed as (64 elements, 24576 rows of 512, 8 chunks): one box = 64 columns of W_UK[h]
    CUtensorMap tmap_w;
    const int rc = make_tmap_slab_3d(&tmap_w, w_kv_b, (uint64_t)H * WROWS_PER_HEAD, LORA, 8, NOPE, 1);
    if (rc) return rc;
    const dim3 grid(H, (B + nb - 1) / nb);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (wide)
        return launch_pdl(k3mla_absorb_kernel<128>, grid, dim3(AB_THREADS), smem, st, "k3mla_absorb_kernel", tmap_w,
                          q, q_abs, B, ap);
    return launch_pdl(k3mla_absorb_kernel<64>, grid, dim3(AB_THREADS), smem, st, "k3mla_absorb_kernel", tmap_w, q,
                      q_abs, B, ap);
}

extern "C" int k3mla_absorb_q(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, int B, void* stream)
{
    const int rc = check_absorb("k3mla_absorb_q", q, w_kv_b, q_abs, B);
    if (rc || B == 0) return rc;
    AppendJob none{};
    return launch_absorb(q, w_kv_b, q_abs, B, none, stream);  // none.B == 0: no append
}

extern "C" int k3mla_absorb_q_append(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, uint16_t* slab,
                                     int n_pages, int n_layers, int layer, const int32_t* block_table,
                                     int max_pages_per_slot, const int32_t* pos, const uint16_t* c_kv,
                                     int64_t c_stride, const uint16_t* k_rope, int64_t r_stride, int B,
                                     int32_t* dev_err, void* stream)
{
    int rc = check_absorb("k3mla_absorb_q_append", q, w_kv_b, q_abs, B);
    if (!rc)
        rc = check_append("k3mla_absorb_q_append", slab, n_pages, n_layers, layer, block_table, max_pages_per_slot,
                          pos, c_kv, c_stride, k_rope, r_stride, B);
    if (rc || B == 0) return rc;
    AppendJob ap;
    ap.slab = slab;
    ap.table = block_table;
    ap.pos = pos;
    ap.c_kv = c_kv;
    ap.k_rope = k_rope;
    ap.dev_err = dev_err;
    ap.c_stride = c_stride;
    ap.r_stride = r_stride;
    ap.n_pages = n_pages;
    ap.n_layers = n_layers;
    ap.layer = layer;
    ap.max_pages = max_pages_per_slot;
    ap.B = B;
    ap.pos_is_ctx = 0;
    return launch_absorb(q, w_kv_b, q_abs, B, ap, stream);
}

namespace k3 {
int launch_absorb_append_at_ctx(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, uint16_t* slab,
                                int n_pages, int n_layers, int layer, const int32_t* block_table,
                                int max_pages_per_slot, const int32_t* ctx_len, const uint16_t* c_kv,
                                int64_t c_stride, const uint16_t* k_rope, int64_t r_stride, int B, int32_t* dev_err,
                                cudaStream_t stream)
{
    AppendJob ap;
    ap.slab = slab;
    ap.table = block_table;
    ap.pos = ctx_len;
    ap.c_kv = c_kv;
    ap.k_rope = k_rope;
    ap.dev_err = dev_err;
    ap.c_stride = c_stride;
    ap.r_stride = r_stride;
    ap.n_pages = n_pages;
    ap.n_layers = n_layers;
    ap.layer = layer;
    ap.max_pages = max_pages_per_slot;
    ap.B = B;
    ap.pos_is_ctx = 1;
    return launch_absorb(q, w_kv_b, q_abs, B, ap, stream);
}
}  // namespace k3

extern "C" int k3mla_append_latent(uint16_t* slab, int n_pages, int n_layers, int layer,
                                   const int32_t* block_table, int max_pages_per_slot, const int32_t* pos,
                                   const uint16_t* c_kv, int64_t c_stride, const uint16_t* k_rope,
                                   int64_t r_stride, int B, int32_t* dev_err, void* stream)
{
    const int rc = check_append("k3mla_append_latent", slab, n_pages, n_layers, layer, block_table,
                                max_pages_per_slot, pos, c_kv, c_stride, k_rope, r_stride, B);
    if (rc || B == 0) return rc;
    if (!device_ok()) return K3MLA_E_DEVICE;
    return launch_pdl(k3mla_append_kernel, dim3(B), dim3(96), 0, reinterpret_cast<cudaStream_t>(stream),
                      "k3mla_append_kernel", slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, pos,
                      c_kv, c_stride, k_rope, r_stride, dev_err);
}
