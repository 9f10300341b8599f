// merge_expand.cu -- merge of a slot's split partials and the W_UV expansion.
//
// For each (slot b, head h), the splits of the context are merged in ascending
// split order with the usual max-rescaled sum (m = max_i m_i; l = sum_i l_i
// e^(m_i - m); o = sum_i o_i e^(m_i - m)), o_lat lands in bf16 as o / l (pegainfer
// PR #869, "K3: paged latent MLA KV + absorbed decode", M2 commit: "f32 latent
// accumulation over ascending t landing bf16"), and out[b][h] = bf16(W_UV[h]
// o_lat) with W_UV read in place from w_kv_b ("f32 W_UV expansion landing bf16").
//
// Per head the expansion is a dense product across slots,
//     OUT_h^T [128 v x B] = W_UV[h] [128 v x 512] . O_lat_h^T [512 x B],
// run on the 5th-generation tensor cores.  One CTA per (head, tile of slots):
//   * one elected thread stages W_UV[h] (128 KB) with eight 3-D TMA boxes, one per
//     64-column chunk (several boxes in flight load faster than one large box),
//     landing as the K-major A operand ([8 chunks][128 rows][128 B], 128-byte
//     swizzle), while
//   * the B operand (bf16 o_lat of the tile's slots, [8 chunks][tile rows][128 B],
//     same swizzle) is put together: a slot whose context had at most one split
//     already has its final o_lat in the workspace (the split kernel landed it:
//     the one partial's weight would be exp(0) = 1), and a slot with several
//     splits is merged here by one warp (four split groups, eight threads each
//     owning a 64-dim slice) and written straight into shared memory;
//   * the elected thread then issues 32 MMAs (M = 128 v, N = the tile, K = 16) into
//     a 128 x tile f32 TMEM accumulator, and the warps read it back (lane = v,
//     column = slot) and store bf16 out.
// When no slot of the launch can have more than one split, tiles are 64 slots and
// the elected thread TMA-loads the tile's o_lat rows ([96][B][512] bf16) as the B
// operand; otherwise tiles are 16 slots (one warp each).  W_UV is read from HBM
// once per layer and from L2 by the other tiles; the f32 partials are read once,
// from L2 where the split kernel just wrote them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int MX_SLOTS = 64;                   // slots per CTA (the MMA's N)
constexpr int MX_MERGE_WARPS = 16;             // merge + epilogue warps
constexpr int MX_THREADS = 32 * MX_MERGE_WARPS;  // thread 0 also issues the TMA loads and the MMAs
constexpr int MX_A_BYTES = 8 * VH * 128;       // W_UV[h]: 8 chunks x 128 rows x 128 B
constexpr int MX_B_BYTES = 8 * MX_SLOTS * 128; // o_lat tile: 8 chunks x 64 rows x 128 B
constexpr uint64_t MX_WAIT_NS = 1000000000ull;  // bounded waits: 1 s
constexpr int MX_G = 4;                        // split groups of a slot with several splits
constexpr int MX_MERGE_TILE = MX_THREADS / (8 * MX_G);  // 16 slots per CTA when merging
static_assert(8 * MX_G == 32, "one warp per slot: the group tree is a warp shuffle");
static_assert(MX_MERGE_TILE == 16, "the launch's merge tile");

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

// Bounded mbarrier wait: false (and K3MLA_DEV_TIMEOUT) after 1 s.
__device__ __noinline__ bool mx_wait(uint64_t* bar, uint32_t parity, int32_t* dev_err)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_test_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity)) {
        if (globaltimer() - t0 > MX_WAIT_NS) {
            if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// OUT_h^T [128 v x tile slots] = W_UV[h] . O_lat_h^T: 32 MMAs (K = 512) into one accumulator; the
// B operand holds `tile` rows per 64-dim chunk.
__device__ __forceinline__ void issue_expand(uint32_t tbase, const uint8_t* sa, const uint8_t* sb, int tile)
{
    const uint64_t ad = make_sdesc(smem_u32(sa), 16, 1024);
    const uint64_t bd = make_sdesc(smem_u32(sb), 16, 1024);
    const uint32_t idesc = make_idesc_bf16(128, (uint32_t)tile, 0, 0);
#pragma unroll
    for (int ks = 0; ks < LORA / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        umma_ss(tbase, ad + (uint64_t)((c * (VH * 128) + kk * 32) >> 4),
                bd + (uint64_t)((c * (tile * 128) + kk * 32) >> 4), idesc, ks > 0 ? 1u : 0u);
    }
}

// grid (96 heads, ceil(B / tile) slot tiles); block MX_THREADS.
__global__ void __launch_bounds__(MX_THREADS, 1)
    k3mla_merge_expand_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_o,
                              const MergeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sb = sa + MX_A_BYTES;
    __shared__ uint64_t w_full, b_ready, d_full, o_full;
    __shared__ uint32_t tmem_slot;
    const int h = blockIdx.x;
    const int b0 = blockIdx.y * p.tile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&w_full, 1);
        mbar_init(&b_ready, 32 * MX_MERGE_WARPS);
        mbar_init(&d_full, 1);
        mbar_init(&o_full, 1);
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tmap_w);
        if (p.nsplit == 1) tma_prefetch_desc(&tmap_o);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, MX_SLOTS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;

    if (threadIdx.x == 0) {
        // W_UV[h] = w_kv_b rows h*256 + 128 .. h*256 + 255, all 512 columns
        mbar_arrive_expect_tx(&w_full, MX_A_BYTES);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            tma_load_3d_hint(sa + c * (VH * 128), &tmap_w, 0, h * WROWS_PER_HEAD + NOPE, c, &w_full,
                             policy_evict_first());  // read once per layer
    }
    // W_UV is a layer weight no kernel of this library writes, so its load above overlaps the split
    // kernel, and so does the merge's read of the context lengths (the split kernel, which runs just
    // before in the stream, only reads them); the split results and the outputs wait for it
    if (p.nsplit == 1) {
        griddep_wait();
        griddep_launch_dependents();
        // ---- every slot has at most one split: the split kernel wrote final bf16 o_lat ([96][B][512]);
        // rows h B + b0 .. h B + b0 + 63 are the B operand as they stand (rows past the batch belong to
        // the next head or lie past the array, read as zeros: either way their columns are not stored)
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&o_full, MX_B_BYTES);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                tma_load_3d(sb + c * (MX_SLOTS * 128), &tmap_o, 0, h * p.B + b0, c, &o_full);
        }
        if (p.argmax && threadIdx.x < MX_SLOTS && b0 + (int)threadIdx.x < p.B) {
            const int b = b0 + (int)threadIdx.x;
            const int ctx = mx_ctx_effective(p.ctx_len, b, p.max_ctx, p.max_pages);
            p.argmax[(size_t)b * H + h] = ctx > 0 ? __float_as_int(p.ws_ml[((size_t)b * H + h) * 4 + 3]) : -1;
        }
        if (threadIdx.x == 0) {
            const bool ok = mx_wait(&w_full, 0, p.dev_err) && mx_wait(&o_full, 0, p.dev_err);
            if (ok) {
                tc_fence_after();
                issue_expand(tbase, sa, sb, p.tile);
            } else {
                const uint64_t t0 = globaltimer();  // let in-flight TMA copies land before the CTA exits
                while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
            }
            umma_commit(&d_full);
        }
    } else {
        // ---- tiles of 16 slots, one warp a slot: thread -> (slot r, split group g, segment seg).  A slot
        // whose context has at most one split (the same rule as the split kernel: its own ctx_len and
        // split_tokens) has its final o_lat in the workspace already, and its warp copies that row into
        // the B operand.  A slot with several splits is merged by MX_G = 4 split groups, group g walking
        // splits g, g + 4, ... in ascending order with a running max: a split's record (m_i, l_i, best
        // score, its token) is loaded with its partial, so the splits arrive in ceil(ns / 4) round trips
        // and no pass over the records comes first.  A fixed shuffle tree then brings the groups to
        // their common max and adds them: ((g0 + g1) + (g2 + g3)).  A group without splits adds exactly
        // nothing.  The grouping is the same for every slot and launch, so a slot's result depends on
        // its own splits only.  The row's 512 dims are 128 float4; float4 f belongs to segment f % 8.
        const int r = (int)threadIdx.x >> 5, g = ((int)threadIdx.x >> 3) & (MX_G - 1), seg = threadIdx.x & 7;
        const int b = b0 + r;
        int n = 0, ns = 0;
        if (b < p.B) {
            n = mx_ctx_effective(p.ctx_len, b, p.max_ctx, p.max_pages);
            ns = slot_nsplit(n, slot_split(n, p.split_tokens));
        }
        griddep_wait();
        griddep_launch_dependents();
        const float* ml = p.ws_ml + ((size_t)b * p.nsplit * H + h) * 4;
        if (ns <= 1) {  // warp-uniform: one warp per slot
            const int l32 = (int)threadIdx.x & 31;
            const uint4* src = reinterpret_cast<const uint4*>(p.ws_olat + ((size_t)h * p.B + b) * LORA);
#pragma unroll
            for (int k = 0; k < 2; ++k) {  // 16-byte unit u of the row: dims 8u .. 8u+7, chunk u / 8
                const int u = 2 * l32 + k, c = u >> 3, uu = u & 7;
                const uint4 v = b < p.B ? src[u] : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sb + c * (p.tile * 128) + r * 128 + ((uu ^ (r & 7)) << 4)) = v;
            }
            if (p.argmax && b < p.B && l32 == 0) p.argmax[(size_t)b * H + h] = n > 0 ? __float_as_int(ml[3]) : -1;
        } else {
            float m = -INFINITY, best = -INFINITY, l = 0.f;
            int best_t = -1;
            float acc[64];
#pragma unroll
            for (int k = 0; k < 64; ++k) acc[k] = 0.f;
            for (int i = g; i < ns; i += MX_G) {
                const float4 rec = *reinterpret_cast<const float4*>(ml + (size_t)i * H * 4);
                const float4* oi =
                    reinterpret_cast<const float4*>(p.ws_o + (((size_t)b * p.nsplit + i) * H + h) * LORA);
                const float mn = fmaxf(m, rec.x);
                const float a = expf(m - mn);      // 0 before the group's first split (m = -inf)
                const float wgt = expf(rec.x - mn);
                l = l * a + wgt * rec.y;
                if (rec.z > best) {  // ascending splits: the lowest t wins ties
                    best = rec.z;
                    best_t = __float_as_int(rec.w);
                }
                m = mn;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float4 v = oi[seg + 8 * k];
                    acc[4 * k + 0] = acc[4 * k + 0] * a + wgt * v.x;
                    acc[4 * k + 1] = acc[4 * k + 1] * a + wgt * v.y;
                    acc[4 * k + 2] = acc[4 * k + 2] * a + wgt * v.z;
                    acc[4 * k + 3] = acc[4 * k + 3] * a + wgt * v.w;
                }
            }
#pragma unroll
            for (int o = 8; o < 8 * MX_G; o <<= 1) {  // the groups of one slot are lanes 8 g + seg of its warp
                const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o);
                const float bo = __shfl_xor_sync(0xFFFFFFFFu, best, o);
                const int to = __shfl_xor_sync(0xFFFFFFFFu, best_t, o);
                const float mn = fmaxf(m, mo);
                const float a = (m == mn) ? 1.f : expf(m - mn);  // a group without splits keeps m = -inf
                l *= a;
                l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
#pragma unroll
                for (int k = 0; k < 64; ++k) {
                    acc[k] *= a;
                    acc[k] += __shfl_xor_sync(0xFFFFFFFFu, acc[k], o);
                }
                if (bo > best || (bo == best && to < best_t && to >= 0)) {  // the lower token on a tie
                    best = bo;
                    best_t = to;
                }
                m = mn;
            }
            if (p.argmax && g == 0 && seg == 0) p.argmax[(size_t)b * H + h] = best_t;
            if (g == 0) {
                const float rl = 1.f / l;  // o_lat = bf16(o * (1 / l)): one division per thread
                // dims d = 32 k + 4 seg + (0..3): chunk d / 64, 16-byte unit (d % 64) / 8
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int c = k >> 1;
                    const int u = 4 * (k & 1) + (seg >> 1);
                    const uint2 v = make_uint2(mx_pack_bf16x2(acc[4 * k + 0] * rl, acc[4 * k + 1] * rl),
                                               mx_pack_bf16x2(acc[4 * k + 2] * rl, acc[4 * k + 3] * rl));
                    *reinterpret_cast<uint2*>(sb + c * (p.tile * 128) + r * 128 + ((u ^ (r & 7)) << 4) +
                                              8 * (seg & 1)) = v;
                }
            }
        }
        fence_proxy_async_cta();  // generic-proxy stores -> visible to the tensor core
        mbar_arrive(&b_ready);
        if (threadIdx.x == 0) {  // the MMAs, once W_UV[h] has landed and every row of o_lat is written
            const bool ok = mx_wait(&w_full, 0, p.dev_err) && mx_wait(&b_ready, 0, p.dev_err);
            if (ok) {
                tc_fence_after();
                issue_expand(tbase, sa, sb, p.tile);
            } else {
                // a wait gave up: let an in-flight TMA land before the CTA can exit
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
            }
            umma_commit(&d_full);  // arrives once every MMA above is complete (at once if none)
        }
    }
    {
        // ---- epilogue: warp (quarter q, group cg) reads v rows 32q .. 32q+31, slots 16cg .. 16cg+15, and
        // lands bf16 out in a [tile slots][128 v] tile over the (now idle) W_UV buffer; the CTA then writes
        // each slot's 256-byte row of out with 16-byte stores
        const int q = warp & 3, cg = warp >> 2;
        const bool got = __all_sync(0xFFFFFFFFu, mx_wait(&d_full, 0, p.dev_err));
        uint16_t* tile = reinterpret_cast<uint16_t*>(sa);
        if (got && 16 * cg < p.tile) {
            tc_fence_after();
            uint32_t acc16[16];
            tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * cg), acc16);
            tmem_wait_ld();
            const int v = 32 * q + lane;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                tile[(16 * cg + j) * VH + v] = (uint16_t)(mx_pack_bf16x2(__uint_as_float(acc16[j]), 0.f) & 0xFFFFu);
        }
        __syncthreads();
        if (got)
            for (int u = (int)threadIdx.x; u < p.tile * (VH / 8); u += MX_THREADS) {
                const int r = u / (VH / 8), k = u % (VH / 8), bb = b0 + r;
                if (bb < p.B)
                    reinterpret_cast<uint4*>(p.out + ((size_t)bb * H + h) * VH)[k] =
                        reinterpret_cast<const uint4*>(tile + r * VH)[k];
            }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, MX_SLOTS);
}



// Every slot with at most one split and more than one 64-slot tile (a batch of token rows, say): one
// CTA a head loads W_UV[h] once and takes the tiles in turn.  A tile's o_lat is TMA-loaded as soon as
// the MMAs of the tile before have read the B buffer, while that tile's outputs are written: its
// epilogue stages them beside W_UV (the last tile's over W_UV, which no MMA reads any more).
constexpr int MX_O_BYTES = MX_SLOTS * VH * 2;  // a tile's bf16 outputs, staged for 16-byte stores

__global__ void __launch_bounds__(MX_THREADS, 1)
    k3mla_expand_tiles_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_o,
                              const MergeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sb = sa + MX_A_BYTES;
    uint16_t* so_next = reinterpret_cast<uint16_t*>(sb + MX_B_BYTES);
    __shared__ uint64_t w_full, d_full, o_full;
    __shared__ uint32_t tmem_slot;
    __shared__ int gave_up;  // a wait ran out: the remaining tiles are skipped
    const int h = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = (p.B + MX_SLOTS - 1) / MX_SLOTS;

    if (threadIdx.x == 0) {
        gave_up = 0;
        mbar_init(&w_full, 1);
        mbar_init(&d_full, 1);
        mbar_init(&o_full, 1);
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_o);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, MX_SLOTS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    if (threadIdx.x == 0) {  // W_UV[h], as in k3mla_merge_expand_kernel: a weight, loaded before the grid wait
        mbar_arrive_expect_tx(&w_full, MX_A_BYTES);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            tma_load_3d_hint(sa + c * (VH * 128), &tmap_w, 0, h * WROWS_PER_HEAD + NOPE, c, &w_full,
                             policy_evict_first());
    }
    griddep_wait();
    griddep_launch_dependents();
    auto load_tile = [&](int t) {  // o_lat rows h B + 64 t .. as the B operand (rows past the batch unused)
        mbar_arrive_expect_tx(&o_full, MX_B_BYTES);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            tma_load_3d(sb + c * (MX_SLOTS * 128), &tmap_o, 0, h * p.B + t * MX_SLOTS, c, &o_full);
    };
    if (threadIdx.x == 0) load_tile(0);
    for (int t = 0; t < ntiles; ++t) {
        const int b0 = t * MX_SLOTS;
        const bool last = t + 1 == ntiles;
        const uint32_t par = (uint32_t)t & 1u;
        if (p.argmax && threadIdx.x < MX_SLOTS && b0 + (int)threadIdx.x < p.B) {
            const int b = b0 + (int)threadIdx.x;
            const int ctx = mx_ctx_effective(p.ctx_len, b, p.max_ctx, p.max_pages);
            p.argmax[(size_t)b * H + h] = ctx > 0 ? __float_as_int(p.ws_ml[((size_t)b * H + h) * 4 + 3]) : -1;
        }
        if (threadIdx.x == 0) {
            const bool ok = mx_wait(&w_full, 0, p.dev_err) && mx_wait(&o_full, par, p.dev_err);
            if (ok) {
                tc_fence_after();
                issue_expand(tbase, sa, sb, MX_SLOTS);
            } else {
                gave_up = 1;
                const uint64_t t0 = globaltimer();  // let in-flight TMA copies land before the CTA exits
                while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
            }
            umma_commit(&d_full);
            if (ok && !last && mx_wait(&d_full, par, p.dev_err)) load_tile(t + 1);  // the MMAs read sb
        }
        // epilogue: warp (quarter q, group cg) reads v rows 32q .. 32q+31, slots 16cg .. 16cg+15
        uint16_t* so = last ? reinterpret_cast<uint16_t*>(sa) : so_next;
        const int q = warp & 3, cg = warp >> 2;
        const bool got = __all_sync(0xFFFFFFFFu, mx_wait(&d_full, par, p.dev_err));
        if (got) {
            tc_fence_after();
            uint32_t acc16[16];
            tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * cg), acc16);
            tmem_wait_ld();
            const int v = 32 * q + lane;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                so[(16 * cg + j) * VH + v] = (uint16_t)(mx_pack_bf16x2(__uint_as_float(acc16[j]), 0.f) & 0xFFFFu);
        }
        tc_fence_before();  // the TMEM loads before the next tile's MMAs
        __syncthreads();
        if (got)
            for (int u = (int)threadIdx.x; u < MX_SLOTS * (VH / 8); u += MX_THREADS) {
                const int r = u / (VH / 8), k = u % (VH / 8), bb = b0 + r;
                if (bb < p.B)
                    reinterpret_cast<uint4*>(p.out + ((size_t)bb * H + h) * VH)[k] =
                        reinterpret_cast<const uint4*>(so + r * VH)[k];
            }
        __syncthreads();  // the staging buffer is free again; gave_up is seen by every thread
        tc_fence_after();
        if (*reinterpret_cast<volatile int*>(&gave_up)) break;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, MX_SLOTS);
}

int launch_merge_expand(const MergeParams& mp, cudaStream_t st)
{
    static bool attr_set[64] = {};
    const int smem = MX_A_BYTES + MX_B_BYTES + 1024;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaFuncSetAttribute(k3mla_merge_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    // w_kv_b viewed as (64 elements, 24576 rows of 512, 8 chunks): one box = one chunk of W_UV[h]
    CUtensorMap tmap_w, tmap_o;
    int rc = make_tmap_slab_3d(&tmap_w, mp.w_kv_b, (uint64_t)H * WROWS_PER_HEAD, LORA, 8, VH, 1);
    if (rc) return rc;
    // final o_lat viewed as (64 elements, 96 B rows of 512, 8 chunks): one box = 64 slots of a chunk
    std::memset(&tmap_o, 0, sizeof(tmap_o));
    if (mp.nsplit == 1) {
        rc = make_tmap_slab_3d(&tmap_o, mp.ws_olat, (uint64_t)H * mp.B, LORA, 8, MX_SLOTS, 1);
        if (rc) return rc;
    }
    if (mp.nsplit == 1 && mp.B > MX_SLOTS) {  // several tiles of final o_lat: one CTA a head takes them all
        static bool tiles_attr_set[64] = {};
        const int smem_t = MX_A_BYTES + MX_B_BYTES + MX_O_BYTES + 1024;
        if (dev < 0 || dev >= 64 || !tiles_attr_set[dev]) {
            cudaFuncSetAttribute(k3mla_expand_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_t);
            if (dev >= 0 && dev < 64) tiles_attr_set[dev] = true;
        }
        return launch_pdl(k3mla_expand_tiles_kernel, dim3(H), dim3(MX_THREADS), smem_t, st,
                          "k3mla_expand_tiles_kernel", tmap_w, tmap_o, mp);
    }
    const dim3 grid(H, (mp.B + mp.tile - 1) / mp.tile);
    return launch_pdl(k3mla_merge_expand_kernel, grid, dim3(MX_THREADS), smem, st, "k3mla_merge_expand_kernel",
                      tmap_w, tmap_o, mp);
}

}  // namespace k3
