// decode.cu -- paged absorbed-MLA decode for sm_103a.
//
// Math (pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M2
// commit): for slot b, head h and logical token t with cache row r_t (a -1 block
// table entry is an all-zero row),
//     s_t   = bf16( bf16( q_abs[h] . r_t ) * scale )          (dot over 576)
//     p     = softmax(s)
//     o_lat = bf16( sum_t p_t r_t[0:512] )
//     out   = bf16( W_UV[h] o_lat )
// q_abs comes from k3mla_absorb_q; W_UV is read in place from w_kv_b.
//
// Structure (GB300-first; the page's own 3-sweep kernel is prior art only):
//   * The context of a slot is cut into fixed splits of `split` logical tokens
//     (a multiple of the 128-token tile).  Each split is one unit of work for a
//     CLUSTER OF TWO CTAs, and each 64-token page is read once for all 96 heads:
//       - CTA rank 0 ("score CTA") holds q_abs for the slot in TMEM (lanes =
//         heads, 96 of 128 used) and streams 128-token tiles through a TMA ring
//         of 16 KB chunks [128 tokens x 64 dims].  One tcgen05 MMA chain per
//         tile computes S^T[heads x 128 tokens] = Q . C^T (K = 576, A from TMEM,
//         B from shared memory) into TMEM.  Its four softmax warps (thread =
//         head) land the scores to bf16 exactly as the chain does, keep a lazily
//         rescaled running max per head, and write bf16 p_t straight into the
//         partner CTA's shared memory (distributed shared memory) as the K-major
//         B operand of the second contraction.
//       - CTA rank 1 ("PV CTA") streams the same tiles (dims 0..511, 32 KB
//         pair-slots [2 x 64 dims][128 tokens]) and accumulates
//         O^T[512 dims x 96 heads] += C^T . P^T in TMEM (four M = 128 blocks,
//         N = 96, K = 128 tokens per tile; A is the MN-major latent tile).  Its
//         four epilogue warps rescale O when the score CTA moves a head's
//         reference max, zero rows past the context in the final tile (stale
//         rows must not meet p = 0 as 0 * NaN), and write the split's f32
//         partial.
//     TMEM holds Q (288 columns) + S (128) in rank 0 and O (384) in rank 1,
//     which is why the two contractions live in different CTAs.
//   * A second kernel merges the splits of each (slot, head) in ascending split
//     order, lands o_lat in bf16 and expands it with W_UV[h] on tensor cores
//     (mma.sync; W_UV is read once per head).
// Split boundaries depend only on the logical position and ctx_len, and no
// physical page id enters the arithmetic, so a slot's result is bitwise
// independent of the batch, of padding and of page placement.
//
// Departures from the chain, all inside the stated tolerance: the tensor cores
// add the 576 products of a score and the tokens of o_lat in their own order;
// probabilities are landed in bf16 before normalisation (p~_t = bf16(exp(s_t -
// m_ref)), normalised by sum p~ at the end); the reference max m_ref of a head
// moves only when the tile max exceeds it by more than TAU (else exp(s - m_ref)
// <= e^TAU, far inside f32 / bf16 range); exp is the hardware ex2.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int NS0 = 13;                // score-CTA ring slots
constexpr int NS1 = 5;                 // PV-CTA ring pair-slots
constexpr int SLOT0 = 16384;           // [128 tokens][64 dims] bf16, two 8 KB TMA boxes
constexpr int SLOT1 = 32768;           // [2][128 tokens][64 dims] bf16, four boxes
constexpr int PT_ATOM = H * 128;       // 96 rows x 128 B = one K-atom of P^T
constexpr int PT_BYTES = 2 * PT_ATOM;  // P^T for a 128-token tile
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;          // score CTA: S^T [128 lanes x 128 cols f32]
constexpr uint32_t Q_COL = 128;        // score CTA: Q   [128 lanes x 288 cols (576 bf16)]
constexpr float TAU = 8.0f;            // max growth (natural log) before a rescale
constexpr uint64_t WAIT_NS = 1000000000ull;  // bounded waits: 1 s
constexpr uint32_t IDESC_S = make_idesc_bf16(128, 128, 0, 0);   // S^T = Q . C^T
constexpr uint32_t IDESC_PV = make_idesc_bf16(128, 96, 1, 0);   // O^T = C^T . P^T (A MN-major)
constexpr int THREADS = 192;

struct __align__(1024) Smem {
    union {
        uint8_t ring0[NS0][SLOT0];
        struct {
            uint8_t ring1[NS1][SLOT1];
            uint8_t pt[2][PT_BYTES];
        } c1;
    } u;
    float alpha[2][H];        // PV CTA: per-head rescale factors (written by the score CTA)
    uint32_t rflag[2][4];     // PV CTA: per-warp "some head rescaled" flags
    uint64_t full[16];
    uint64_t empty[16];
    uint64_t s_full, s_empty, q_ready;
    uint64_t p_full[2], p_empty[2];
    uint64_t o_done, epi_req, epi_done;
    uint32_t tmem_base;
    uint32_t epi_cmd, epi_slot, epi_stage, epi_vrows;
    int32_t abort_flag;
};
static_assert(sizeof(Smem::u) == NS0 * SLOT0, "ring layouts");
static_assert(NS1 * SLOT1 + 2 * PT_BYTES == NS0 * SLOT0, "ring layouts");

struct DecodeParams {
    const uint16_t* q_abs;
    const int32_t* table;
    const int32_t* ctx_len;
    float* ws_o;    // [B][nsplit][96][512]
    float* ws_ml;   // [B][nsplit][96][4]: m_ref, l, best score, best t (int bits)
    int32_t* dev_err;
    int max_pages, n_pages, n_layers, layer;
    int B, max_ctx, split, nsplit;
    float scale;
};

__device__ __forceinline__ int ctx_effective(const int32_t* ctx_len, int b, int max_ctx, int max_pages,
                                             int32_t* dev_err, bool report)
{
    int n = ctx_len[b];
    int cap = min(max_ctx, max_pages * PAGE);
    if (n > cap) {
        if (report && dev_err) atomicOr(dev_err, (int)K3MLA_DEV_CTX);
        n = cap;
    }
    return n < 0 ? 0 : n;
}

// Bounded mbarrier wait: gives up after WAIT_NS or when this CTA aborted.
__device__ __noinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Smem& sm, int32_t* dev_err,
                                      bool cluster_scope = false)
{
    const uint32_t a = smem_u32(bar);
    if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
        if ((n & 127u) == 0) {
            if (*reinterpret_cast<volatile int32_t*>(&sm.abort_flag)) return false;
            if (globaltimer() - t0 > WAIT_NS) {
                *reinterpret_cast<volatile int32_t*>(&sm.abort_flag) = 1;
                if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// After an abort: let this thread's in-flight TMA copies / MMAs land (bounded, ~2 ms).
__device__ __noinline__ void drain_inflight()
{
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
}

// TMA row coordinate of logical page lp of slot b, or an out-of-range row (zero fill).
__device__ __forceinline__ int32_t page_row(const DecodeParams& p, int b, int lp, int n_lp, int32_t oob_row)
{
    if (lp >= n_lp) return oob_row;
    int32_t id = p.table[(size_t)b * p.max_pages + lp];
    if (id == -1) return oob_row;
    if (id < -1 || id >= p.n_pages) {
        if (p.dev_err) atomicOr(p.dev_err, (int)K3MLA_DEV_BAD_PAGE);
        return oob_row;
    }
    return (id * p.n_layers + p.layer) * PAGE;
}

// ---- shared building blocks (also used by the diagnostic kernel) ---------------

// Score CTA: rows 0..95 of Q (one row per thread h = 0..127, rows >= 96 zero)
// into TMEM columns [Q_COL, Q_COL+288) of lane h.  Called by warps 0..3.
__device__ __forceinline__ void load_q_tmem(uint32_t tbase, const uint16_t* qrow_or_null)
{
    const uint32_t w = threadIdx.x >> 5;
    const uint32_t taddr = tbase + ((32u * w) << 16) + Q_COL;
#pragma unroll 1
    for (int c = 0; c < 9; ++c) {
        uint32_t r[32];
        if (qrow_or_null) {
            const uint4* src = reinterpret_cast<const uint4*>(qrow_or_null + c * 64);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint4 v = __ldg(src + k);
                r[4 * k + 0] = v.x;
                r[4 * k + 1] = v.y;
                r[4 * k + 2] = v.z;
                r[4 * k + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        tmem_st32(taddr + c * 32, r);
    }
    tmem_wait_st();
}

// Score CTA: the MMAs of one 576-wide chunk c (4 K-steps of 16) of a tile.
__device__ __forceinline__ void issue_score_chunk(uint32_t tbase, uint32_t slot_addr, int c)
{
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        const uint32_t a = tbase + Q_COL + (uint32_t)(4 * c + ks) * 8u;
        const uint64_t bd = make_sdesc(slot_addr + ks * 32, 16, 1024);
        umma_ts(tbase + S_COL, a, bd, IDESC_S, (c | ks) != 0);
    }
}

// PV CTA: O^T block j (dims 128j..128j+127) += C^T . P^T over one 128-token tile.
__device__ __forceinline__ void issue_pv_block(uint32_t tbase, uint32_t pair_addr, uint32_t pt_addr, int j,
                                               bool accumulate_first)
{
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = make_sdesc(pair_addr + ks * 2048, SLOT1 / 2, 1024);
        const uint64_t bd = make_sdesc(pt_addr + (ks >> 2) * PT_ATOM + (ks & 3) * 32, 16, 1024);
        umma_ss(tbase + 96u * j, ad, bd, IDESC_PV, (accumulate_first || ks > 0) ? 1u : 0u);
    }
}

// Byte offset, inside a P^T buffer, of the 16-byte chunk holding tokens
// 64a + 8j .. 64a + 8j + 7 of head h (K-major, 128-byte swizzle).
__device__ __forceinline__ uint32_t pt_chunk_off(int h, int a, int j)
{
    return (uint32_t)(a * PT_ATOM + h * 128 + ((j ^ (h & 7)) << 4));
}

// ---- the split decode kernel ---------------------------------------------------

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k3mla_decode_split_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t rank = cluster_ctarank();
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();

    const int unit = blockIdx.x >> 1;
    const int b = unit / p.nsplit;
    const int s = unit % p.nsplit;
    const int ctx = ctx_effective(p.ctx_len, b, p.max_ctx, p.max_pages, p.dev_err,
                                  rank == 0 && threadIdx.x == 0 && s == 0);
    const int start = s * p.split;
    if (start >= ctx) return;  // empty split: both CTAs leave, nothing was shared
    const int ntok = min(ctx, start + p.split) - start;
    const int ntiles = (ntok + TILE - 1) / TILE;
    const int n_lp = (ctx + PAGE - 1) / PAGE;
    const int32_t oob_row = p.n_pages * p.n_layers * PAGE;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 16; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_empty, 3);
        mbar_init(&sm.q_ready, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.p_full[i], H);
            mbar_init(&sm.p_empty[i], 1);
        }
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.epi_req, 1);
        mbar_init(&sm.epi_done, 4);
        sm.abort_flag = 0;
        fence_mbarrier_init_cluster();
    }
    if (warp == 5) {
        tmem_alloc(&sm.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) tma_prefetch_desc(&tmap);
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;

    if (rank == 0) {
        // =========================== score CTA ===========================
        if (warp == 4) {
            if (lane == 0) {
                const uint64_t pol = policy_evict_first();
                int slot = 0;
                uint32_t ph = 0;
                bool ok = true;
                for (int i = 0; i < ntiles && ok; ++i) {
                    const int lp0 = start / PAGE + 2 * i;
                    const int32_t ya = page_row(p, b, lp0, n_lp, oob_row);
                    const int32_t yb = page_row(p, b, lp0 + 1, n_lp, oob_row);
                    for (int c = 0; c < 9; ++c) {
                        if (!wait_bar(&sm.empty[slot], ph ^ 1u, sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&sm.full[slot], SLOT0);
                        tma_load_2d(sm.u.ring0[slot], &tmap, 64 * c, ya, &sm.full[slot], pol);
                        tma_load_2d(sm.u.ring0[slot] + SLOT0 / 2, &tmap, 64 * c, yb, &sm.full[slot], pol);
                        if (++slot == NS0) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                }
                if (!ok) drain_inflight();
            }
        } else if (warp == 5) {
            if (lane == 0) {
                bool ok = wait_bar(&sm.q_ready, 0, sm, p.dev_err);
                tc_fence_after();
                int slot = 0;
                uint32_t ph = 0;
                for (int i = 0; i < ntiles && ok; ++i) {
                    if (!wait_bar(&sm.s_empty, (uint32_t)(i & 1) ^ 1u, sm, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int c = 0; c < 9; ++c) {
                        if (!wait_bar(&sm.full[slot], ph, sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_score_chunk(tbase, smem_u32(sm.u.ring0[slot]), c);
                        umma_commit(&sm.empty[slot]);
                        if (++slot == NS0) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                    if (ok) umma_commit(&sm.s_full);
                }
                if (!ok) drain_inflight();
            }
        } else {
            // softmax warps 0..3: thread h owns head h (h < 96)
            const int h = (int)threadIdx.x;
            load_q_tmem(tbase, h < H ? p.q_abs + ((size_t)b * H + h) * ROW : nullptr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.q_ready);
            if (warp < 3) {
                const uint32_t t_lane = tbase + ((32u * warp) << 16);
                const float scale = p.scale;
                const float LOG2E = 1.4426950408889634f;
                float m_ref = -INFINITY, l = 0.f, best_s = -INFINITY;
                int best_t = -1;
                bool ok = true;
                const uint32_t pt_remote0 = mapa(smem_u32(sm.u.c1.pt[0]), 1);
                const uint32_t pt_remote1 = mapa(smem_u32(sm.u.c1.pt[1]), 1);
                for (int i = 0; i < ntiles; ++i) {
                    const bool got = wait_bar(&sm.s_full, (uint32_t)(i & 1), sm, p.dev_err);
                    __syncwarp();
                    if (!__all_sync(0xFFFFFFFFu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nvalid = min(TILE, ntok - TILE * i);
                    uint32_t sp[64];  // bf16 scores, two per word (token 2k low, 2k+1 high)
                    float tmax = -INFINITY;
#pragma unroll
                    for (int piece = 0; piece < 4; ++piece) {
                        uint32_t r[32];
                        tmem_ld32(t_lane + S_COL + 32 * piece, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            const int t = 32 * piece + k;
                            // land the dot in bf16, multiply by the bf16 scale, land again
                            const uint32_t d2 = pack_bf16x2(__uint_as_float(r[k]), __uint_as_float(r[k + 1]));
                            float s0 = bf16lo_to_f32(d2) * scale;
                            float s1 = bf16hi_to_f32(d2) * scale;
                            uint32_t s2 = pack_bf16x2(s0, s1);
                            if (t >= nvalid) s2 = (s2 & 0xFFFF0000u) | 0xFF80u;            // -inf
                            if (t + 1 >= nvalid) s2 = (s2 & 0x0000FFFFu) | 0xFF800000u;
                            sp[t >> 1] = s2;
                            tmax = fmaxf(tmax, fmaxf(bf16lo_to_f32(s2), bf16hi_to_f32(s2)));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.s_empty);

                    if (tmax > best_s) {  // lowest logical t attaining the best score
                        best_s = tmax;
                        int first = 0;
                        for (int k = 63; k >= 0; --k) {
                            if (bf16hi_to_f32(sp[k]) == tmax) first = 2 * k + 1;
                            if (bf16lo_to_f32(sp[k]) == tmax) first = 2 * k;
                        }
                        best_t = start + TILE * i + first;
                    }
                    float alpha = 1.f;
                    bool resc = false;
                    if (i == 0) {
                        m_ref = tmax;
                    } else if (tmax > m_ref + TAU) {
                        alpha = ex2_approx((m_ref - tmax) * LOG2E);
                        l *= alpha;
                        m_ref = tmax;
                        resc = true;
                    }
                    const float mb = m_ref * LOG2E;
                    uint32_t pp[64];
#pragma unroll
                    for (int k = 0; k < 64; ++k) {
                        const float e0 = ex2_approx(fmaf(bf16lo_to_f32(sp[k]), LOG2E, -mb));
                        const float e1 = ex2_approx(fmaf(bf16hi_to_f32(sp[k]), LOG2E, -mb));
                        const uint32_t q2 = pack_bf16x2(e0, e1);
                        l += bf16lo_to_f32(q2);
                        l += bf16hi_to_f32(q2);
                        pp[k] = q2;
                    }
                    const int stage = i & 1;
                    const bool freed = wait_bar(&sm.p_empty[stage], (uint32_t)((i >> 1) & 1) ^ 1u, sm, p.dev_err);
                    if (!__all_sync(0xFFFFFFFFu, freed)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = stage ? pt_remote1 : pt_remote0;
#pragma unroll
                    for (int a = 0; a < 2; ++a)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int k = 32 * a + 4 * j;
                            st_cluster_v4(dst + pt_chunk_off(h, a, j), make_uint4(pp[k], pp[k + 1], pp[k + 2], pp[k + 3]));
                        }
                    st_cluster_u32(mapa(smem_u32(&sm.alpha[stage][h]), 1), __float_as_uint(alpha));
                    const uint32_t any = __ballot_sync(0xFFFFFFFFu, resc);
                    if (lane == 0) st_cluster_u32(mapa(smem_u32(&sm.rflag[stage][warp]), 1), any ? 1u : 0u);
                    fence_proxy_async_cluster();
                    mbar_arrive_remote(mapa(smem_u32(&sm.p_full[stage]), 1));
                }
                if (ok) {
                    float* ml = p.ws_ml + (((size_t)b * p.nsplit + s) * H + h) * 4;
                    ml[0] = m_ref;
                    ml[1] = l;
                    ml[2] = best_s;
                    ml[3] = __int_as_float(best_t);
                    // the PV CTA's last releases of the P buffers land here before exit
                    for (int i = max(0, ntiles - 2); i < ntiles && ok; ++i)
                        ok = wait_bar(&sm.p_empty[i & 1], (uint32_t)(((i >> 1) & 1)), sm, p.dev_err);
                }
            }
        }
    } else {
        // ============================ PV CTA ============================
        if (warp == 4) {
            if (lane == 0) {
                const uint64_t pol = policy_evict_first();
                int slot = 0;
                uint32_t ph = 0;
                bool ok = true;
                for (int i = 0; i < ntiles && ok; ++i) {
                    const int lp0 = start / PAGE + 2 * i;
                    const int32_t ya = page_row(p, b, lp0, n_lp, oob_row);
                    const int32_t yb = page_row(p, b, lp0 + 1, n_lp, oob_row);
                    for (int j = 0; j < 4; ++j) {
                        if (!wait_bar(&sm.empty[slot], ph ^ 1u, sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        uint8_t* dst = sm.u.c1.ring1[slot];
                        mbar_arrive_expect_tx(&sm.full[slot], SLOT1);
                        tma_load_2d(dst, &tmap, 128 * j, ya, &sm.full[slot], pol);
                        tma_load_2d(dst + 8192, &tmap, 128 * j, yb, &sm.full[slot], pol);
                        tma_load_2d(dst + 16384, &tmap, 128 * j + 64, ya, &sm.full[slot], pol);
                        tma_load_2d(dst + 24576, &tmap, 128 * j + 64, yb, &sm.full[slot], pol);
                        if (++slot == NS1) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                }
                if (!ok) drain_inflight();
            }
        } else if (warp == 5) {
            if (lane == 0) {
                int slot = 0;
                uint32_t ph = 0;
                uint32_t epi_k = 0;
                bool ok = true;
                for (int i = 0; i < ntiles && ok; ++i) {
                    const int stage = i & 1;
                    if (!wait_bar(&sm.p_full[stage], (uint32_t)((i >> 1) & 1), sm, p.dev_err, true)) {
                        ok = false;
                        break;
                    }
                    const volatile uint32_t* rf = sm.rflag[stage];
                    const bool resc = (i > 0) && ((rf[0] | rf[1] | rf[2]) != 0u);
                    const int nvalid = min(TILE, ntok - TILE * i);
                    const bool tail = nvalid < TILE;
                    if (tail) {  // the epilogue zeroes stale rows once the tile has landed
                        int sl = slot;
                        uint32_t pf = ph;
                        for (int j = 0; j < 4 && ok; ++j) {
                            ok = wait_bar(&sm.full[sl], pf, sm, p.dev_err);
                            if (++sl == NS1) {
                                sl = 0;
                                pf ^= 1u;
                            }
                        }
                        if (!ok) break;
                    }
                    if (resc || tail) {
                        if (resc) umma_commit(&sm.o_done);
                        sm.epi_cmd = (resc ? 1u : 0u) | (tail ? 2u : 0u);
                        sm.epi_slot = (uint32_t)slot;
                        sm.epi_stage = (uint32_t)stage;
                        sm.epi_vrows = (uint32_t)nvalid;
                        mbar_arrive(&sm.epi_req);
                        if (!wait_bar(&sm.epi_done, epi_k & 1u, sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        ++epi_k;
                    }
                    const uint32_t pt = smem_u32(sm.u.c1.pt[stage]);
                    for (int j = 0; j < 4; ++j) {
                        if (!tail && !wait_bar(&sm.full[slot], ph, sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv_block(tbase, smem_u32(sm.u.c1.ring1[slot]), pt, j, i > 0);
                        umma_commit(&sm.empty[slot]);
                        if (++slot == NS1) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                    if (ok) umma_commit_mc(&sm.p_empty[stage], (uint16_t)0x1);
                }
                if (ok) {
                    umma_commit(&sm.o_done);
                    sm.epi_cmd = 4u;
                    mbar_arrive(&sm.epi_req);
                } else {
                    drain_inflight();
                    *reinterpret_cast<volatile int32_t*>(&sm.abort_flag) = 1;
                }
            }
        } else {
            // epilogue warps 0..3: thread owns TMEM lane 32*warp + lane (a latent dim per block)
            const uint32_t t_lane = tbase + ((32u * warp) << 16);
            uint32_t k = 0, od = 0;
            for (;;) {
                const bool got = wait_bar(&sm.epi_req, k & 1u, sm, p.dev_err);
                if (!__all_sync(0xFFFFFFFFu, got)) break;
                ++k;
                const uint32_t cmd = *reinterpret_cast<volatile uint32_t*>(&sm.epi_cmd);
                if (cmd & 1u) {  // rescale O^T columns by alpha[head]
                    const bool got = wait_bar(&sm.o_done, od & 1u, sm, p.dev_err);
                    if (!__all_sync(0xFFFFFFFFu, got)) break;
                    ++od;
                    tc_fence_after();
                    const float* al = sm.alpha[sm.epi_stage];
                    for (int j = 0; j < 4; ++j)
                        for (int piece = 0; piece < 3; ++piece) {
                            uint32_t r[32];
                            const uint32_t ta = t_lane + 96u * j + 32u * piece;
                            tmem_ld32(ta, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                r[c] = __float_as_uint(__uint_as_float(r[c]) * al[32 * piece + c]);
                            tmem_st32(ta, r);
                        }
                    tmem_wait_st();
                    tc_fence_before();
                }
                if (cmd & 2u) {  // zero rows >= vrows of the tile's four pair-slots
                    const int vr = (int)sm.epi_vrows;
                    const int rows = TILE - vr;
                    const int per_half = rows * 8;  // 16-byte chunks
                    const int total = 4 * 2 * per_half;
                    for (int q = (int)threadIdx.x; q < total; q += 128) {
                        const int sl_off = q / (2 * per_half);
                        const int rem = q % (2 * per_half);
                        const int half = rem / per_half;
                        const int c16 = rem % per_half;
                        const int row = vr + c16 / 8;
                        const int sl = ((int)sm.epi_slot + sl_off) % NS1;
                        uint4* d = reinterpret_cast<uint4*>(sm.u.c1.ring1[sl] + half * (SLOT1 / 2) + row * 128 +
                                                            (c16 % 8) * 16);
                        *d = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_cta();
                }
                if (cmd & 4u) {  // final: write the split's f32 partial O
                    const bool got = wait_bar(&sm.o_done, od & 1u, sm, p.dev_err);
                    if (!__all_sync(0xFFFFFFFFu, got)) break;
                    ++od;
                    tc_fence_after();
                    float* o = p.ws_o + (((size_t)b * p.nsplit + s) * H) * LORA;
                    for (int j = 0; j < 4; ++j) {
                        const int d = 128 * j + 32 * (int)warp + (int)lane;
                        for (int piece = 0; piece < 3; ++piece) {
                            uint32_t r[32];
                            tmem_ld32(t_lane + 96u * j + 32u * piece, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                o[(size_t)(32 * piece + c) * LORA + d] = __uint_as_float(r[c]);
                        }
                    }
                    break;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.epi_done);
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tbase, TMEM_COLS);
}

// ---- merge of the splits + W_UV expansion ------------------------------------------

constexpr int MX_THREADS = 256;
constexpr int W_PITCH = LORA + 8;   // bf16 elements per smem row (16-byte pad)

struct MergeParams {
    const float* ws_o;
    const float* ws_ml;
    const int32_t* ctx_len;
    const uint16_t* w_kv_b;
    uint16_t* out;
    int32_t* argmax;
    int B, max_ctx, max_pages, split, nsplit;
};

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
                const int ctx = ctx_effective(p.ctx_len, b, p.max_ctx, p.max_pages, nullptr, false);
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
            for (int k = 0; k < 32; k += 2) dst[k >> 1] = pack_bf16x2(o[k] / inv_l_div, o[k + 1] / inv_l_div);
        }
        __syncthreads();
        // out[16 x 64] = o_lat[16 x 512] . W_UV^T ; warp w -> v columns 8w .. 8w+7
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t a_base = smem_u32(so) + ((lane & 15) * W_PITCH + (lane >> 4) * 8) * 2;
        const uint32_t b_base = smem_u32(sw) + ((8 * warp + (lane & 7)) * W_PITCH + ((lane >> 3) & 1) * 8) * 2;
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
            *reinterpret_cast<uint32_t*>(p.out + ((size_t)(m0 + g) * H + h) * VH + v) = pack_bf16x2(acc[0], acc[1]);
        if (m0 + g + 8 < p.B)
            *reinterpret_cast<uint32_t*>(p.out + ((size_t)(m0 + g + 8) * H + h) * VH + v) =
                pack_bf16x2(acc[2], acc[3]);
    }
}

// ---- diagnostic: one tile of each contraction ----------------------------------------

__global__ void __launch_bounds__(128, 1)
    k3mla_diag_kernel(const __grid_constant__ CUtensorMap tmap, int mode, const uint16_t* a, float* d)
{
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    if (threadIdx.x == 0) {
        mbar_init(&sm.full[0], 1);
        mbar_init(&sm.o_done, 1);
        sm.abort_flag = 0;
        fence_mbarrier_init_cluster();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    const uint32_t t_lane = tbase + ((32u * warp) << 16);
    const int h = (int)threadIdx.x;
    const uint64_t pol = policy_evict_first();
    bool ok = true;
    if (mode == 0) {
        load_q_tmem(tbase, h < H ? a + (size_t)h * ROW : nullptr);
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&sm.full[0], 9 * SLOT0);
            for (int c = 0; c < 9; ++c) {
                tma_load_2d(sm.u.ring0[c], &tmap, 64 * c, 0, &sm.full[0], pol);
                tma_load_2d(sm.u.ring0[c] + SLOT0 / 2, &tmap, 64 * c, 64, &sm.full[0], pol);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            ok = wait_bar(&sm.full[0], 0, sm, nullptr);
            tc_fence_after();
            if (ok) {
                for (int c = 0; c < 9; ++c) issue_score_chunk(tbase, smem_u32(sm.u.ring0[c]), c);
                umma_commit(&sm.o_done);
            }
        }
        __syncthreads();
        ok = __all_sync(0xFFFFFFFFu, wait_bar(&sm.o_done, 0, sm, nullptr));
        tc_fence_after();
        if (ok)
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t r[32];
                tmem_ld32(t_lane + S_COL + 32 * piece, r);
                tmem_wait_ld();
                for (int c = 0; c < 32; ++c) d[(size_t)h * 128 + 32 * piece + c] = __uint_as_float(r[c]);
            }
    } else {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&sm.full[0], 4 * SLOT1);
            for (int j = 0; j < 4; ++j) {
                uint8_t* dst = sm.u.c1.ring1[j];
                tma_load_2d(dst, &tmap, 128 * j, 0, &sm.full[0], pol);
                tma_load_2d(dst + 8192, &tmap, 128 * j, 64, &sm.full[0], pol);
                tma_load_2d(dst + 16384, &tmap, 128 * j + 64, 0, &sm.full[0], pol);
                tma_load_2d(dst + 24576, &tmap, 128 * j + 64, 64, &sm.full[0], pol);
            }
        }
        if (h < H) {  // P^T row h from a[h][0..127]
            for (int aa = 0; aa < 2; ++aa)
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4*>(a + (size_t)h * 128 + 64 * aa + 8 * j);
                    *reinterpret_cast<uint4*>(sm.u.c1.pt[0] + pt_chunk_off(h, aa, j)) = v;
                }
        }
        fence_proxy_async_cta();
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            ok = wait_bar(&sm.full[0], 0, sm, nullptr);
            tc_fence_after();
            if (ok) {
                for (int j = 0; j < 4; ++j)
                    issue_pv_block(tbase, smem_u32(sm.u.c1.ring1[j]), smem_u32(sm.u.c1.pt[0]), j, false);
                umma_commit(&sm.o_done);
            }
        }
        __syncthreads();
        ok = __all_sync(0xFFFFFFFFu, wait_bar(&sm.o_done, 0, sm, nullptr));
        tc_fence_after();
        if (ok)
            for (int j = 0; j < 4; ++j)
                for (int piece = 0; piece < 3; ++piece) {
                    uint32_t r[32];
                    tmem_ld32(t_lane + 96u * j + 32u * piece, r);
                    tmem_wait_ld();
                    for (int c = 0; c < 32; ++c)
                        d[(size_t)(128 * j + 32 * warp + lane) * H + 32 * piece + c] = __uint_as_float(r[c]);
                }
    }
    if (!ok) drain_inflight();
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

static size_t smem_bytes() { return sizeof(Smem) + 1024; }

static int num_splits(int max_ctx, int split) { return (max_ctx + split - 1) / split; }

}  // namespace k3

using namespace k3;

extern "C" size_t k3mla_decode_workspace_bytes(int B, int max_ctx, int split_tokens)
{
    if (B <= 0 || max_ctx <= 0 || split_tokens <= 0) return 0;
    const size_t ns = (size_t)num_splits(max_ctx, split_tokens);
    const size_t o = (size_t)B * ns * H * LORA * sizeof(float);
    const size_t ml = (size_t)B * ns * H * 4 * sizeof(float);
    return ((o + 255) & ~size_t(255)) + ml;
}

extern "C" int k3mla_default_split_tokens(int B, int max_ctx)
{
    if (B <= 0 || max_ctx <= 0) return TILE;
    int clusters = 0;
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    clusters = sms / 2;
    int per_slot = clusters / B;
    if (per_slot < 1) per_slot = 1;
    int split = (max_ctx + per_slot - 1) / per_slot;
    split = (split + TILE - 1) / TILE * TILE;
    return split < TILE ? TILE : split;
}

extern "C" int k3mla_paged_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers,
                                  int layer, const int32_t* block_table, int max_pages_per_slot,
                                  const int32_t* ctx_len, const uint16_t* w_kv_b, uint16_t scale_bf16,
                                  uint16_t* out, int32_t* argmax_t, void* workspace, size_t ws_bytes, int B,
                                  int max_ctx, int split_tokens, int32_t* dev_err, void* stream)
{
    if (B < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers || max_pages_per_slot <= 0 ||
        max_ctx <= 0 || split_tokens <= 0 || split_tokens % TILE != 0) {
        set_error("k3mla_paged_decode: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if ((long long)n_pages * n_layers * PAGE + PAGE > 0x7FFFFFFFll) {
        set_error("k3mla_paged_decode: slab rows exceed the 2^31 TMA row range");
        return K3MLA_E_INVALID;
    }
    if (!q_abs || !slab || !block_table || !ctx_len || !w_kv_b || !out || !workspace ||
        !aligned(q_abs, 16) || !aligned(slab, 16) || !aligned(w_kv_b, 16) || !aligned(out, 4) ||
        !aligned(workspace, 256)) {
        set_error("k3mla_paged_decode: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    const size_t need = k3mla_decode_workspace_bytes(B, max_ctx, split_tokens);
    if (ws_bytes < need) {
        set_error("k3mla_paged_decode: workspace %zu < %zu bytes", ws_bytes, need);
        return K3MLA_E_WORKSPACE;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    const int ns = num_splits(max_ctx, split_tokens);
    if ((long long)B * ns * 2 > 0x7FFFFFFFll) {
        set_error("k3mla_paged_decode: grid too large");
        return K3MLA_E_INVALID;
    }
    CUtensorMap tmap;
    int rc = make_tmap_bf16_2d(&tmap, slab, ROW, (uint64_t)n_pages * n_layers * PAGE, 64, 64);
    if (rc) return rc;

    static bool attr_set[64] = {};
    const size_t smem = smem_bytes();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaFuncSetAttribute(k3mla_decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(k3mla_merge_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((64 + 16) * W_PITCH * 2));
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    DecodeParams dp;
    dp.q_abs = q_abs;
    dp.table = block_table;
    dp.ctx_len = ctx_len;
    float* ws_o = reinterpret_cast<float*>(workspace);
    const size_t o_bytes = ((size_t)B * ns * H * LORA * sizeof(float) + 255) & ~size_t(255);
    float* ws_ml = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + o_bytes);
    dp.ws_o = ws_o;
    dp.ws_ml = ws_ml;
    dp.dev_err = dev_err;
    dp.max_pages = max_pages_per_slot;
    dp.n_pages = n_pages;
    dp.n_layers = n_layers;
    dp.layer = layer;
    dp.B = B;
    dp.max_ctx = max_ctx;
    dp.split = split_tokens;
    dp.nsplit = ns;
    {
        uint32_t u = (uint32_t)scale_bf16 << 16;
        float f;
        memcpy(&f, &u, 4);
        dp.scale = f;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    k3mla_decode_split_kernel<<<dim3(2 * B * ns), dim3(THREADS), smem, st>>>(tmap, dp);
    rc = check_launch("k3mla_decode_split_kernel");
    if (rc) return rc;

    MergeParams mp;
    mp.ws_o = ws_o;
    mp.ws_ml = ws_ml;
    mp.ctx_len = ctx_len;
    mp.w_kv_b = w_kv_b;
    mp.out = out;
    mp.argmax = argmax_t;
    mp.B = B;
    mp.max_ctx = max_ctx;
    mp.max_pages = max_pages_per_slot;
    mp.split = split_tokens;
    mp.nsplit = ns;
    k3mla_merge_expand_kernel<<<dim3(2, H), dim3(MX_THREADS), (64 + 16) * W_PITCH * 2, st>>>(mp);
    return check_launch("k3mla_merge_expand_kernel");
}

extern "C" int k3mla_diag_umma(int mode, const uint16_t* a, const uint16_t* b, float* d, void* stream)
{
    if ((mode != 0 && mode != 1) || !a || !b || !d || !aligned(a, 16) || !aligned(b, 16)) {
        set_error("k3mla_diag_umma: invalid arguments");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    CUtensorMap tmap;
    int rc = make_tmap_bf16_2d(&tmap, b, ROW, 128, 64, 64);
    if (rc) return rc;
    const size_t smem = smem_bytes();
    cudaFuncSetAttribute(k3mla_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k3mla_diag_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(tmap, mode, a, d);
    return check_launch("k3mla_diag_kernel");
}
