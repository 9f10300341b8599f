// decode.cu -- paged absorbed-MLA decode for sm_103a: the split kernel.
//
// Math (pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M2
// commit): for slot b, head h and logical token t with cache row r_t (a -1 block
// table entry is an all-zero row),
//     s_t   = bf16( bf16( q_abs[h] . r_t ) * scale )          (dot over 576)
//     p     = softmax(s)
//     o_lat = bf16( sum_t p_t r_t[0:512] )
//     out   = bf16( W_UV[h] o_lat )
// q_abs comes from k3mla_absorb_q; the merge of splits and the W_UV expansion
// are in merge_expand.cu.
//
// Structure (GB300-first; the page's own 3-sweep kernel is prior art only).
// The context of a slot is cut into splits (slot_split: a fixed length, or by
// default ceil(n / 4096) equal splits of the slot's own n tokens); each split
// is one unit of work for a CLUSTER OF TWO CTAs, and the unit of the
// pipeline is one 64-token page, held whole in shared memory.
//   * rank 0, the score CTA, holds q_abs of the slot in TMEM (24 heads in each
//     32-lane quarter so that all four SM sub-partitions run softmax; 288
//     columns).  Pages stream in thirds ([3 chunks][64 rows][128 B], one 24 KB
//     3-D TMA box each) through a ring of eight units; third t of every page has
//     its own producer thread, and page i its MMA issuer thread i mod 3 (one
//     thread alone cannot issue M=128 x N=64 MMAs as fast as the tensor core
//     retires them).  The MMAs (A = Q from TMEM, B = the page, K-major, 128-byte
//     swizzle) write S^T[heads x 64 tokens] into one of three TMEM buffers.  Eight
//     softmax warps (thread = head; the pages of one parity per warp) land the
//     scores to bf16 exactly as the chain does -- bf16(dot), then bf16(. * scale)
//     with packed bf16x2 instructions -- keep a lazily moved reference max per
//     head, and copy bf16 p to the partner CTA's shared memory with one bulk
//     smem-to-DSMEM copy per warp and page (completion counted in bytes on the
//     partner's mbarrier), laid out as the K-major A operand of the second
//     contraction.
//   * rank 1, the PV CTA, streams the same pages (chunks 0..7 as two 32 KB
//     half-page boxes into a ring of five half-page slots, one producer each;
//     these reads mostly hit L2 right after the score CTA's; one of its warps
//     prefetches pages into L2 ahead of the score CTA, whose DRAM ingest is
//     bound by the 2.67 pages its ring holds in flight) and accumulates
//     O[heads x 512 dims] += P . C in TMEM (M = 128 rows, the 96 heads first;
//     two N = 256 halves; K = 64 tokens per page; B is the MN-major latent
//     page), so that a thread reading its TMEM lane holds one head's O row.  Its
//     epilogue warps rescale O when the score CTA moved a head's reference max
//     and zero rows past the context in the final page (stale rows must never
//     meet p = 0 as 0 * NaN); at the end six warps write O out -- the split's f32
//     partial, or, for a slot with a single split, final bf16 o_lat = bf16(O *
//     (1 / l)) -- in swizzled boxes that bulk tensor stores copy out.
// TMEM holds Q (288 columns) + S (3 x 64) in rank 0 and O (512) in rank 1, which
// is why the two contractions live in different CTAs.
//
// Split boundaries depend only on the logical position, the slot's own ctx_len
// and the split_tokens argument; whether a slot lands o_lat itself (one split)
// or leaves partials for the merge depends on the same; no physical page id
// enters the arithmetic.  So a slot's result is bitwise independent of the
// batch, of padding and of page placement.
//
// Departures from the chain, all inside the stated tolerance: the tensor cores
// add the 576 products of a score and the tokens of o_lat in their own order;
// probabilities are landed in bf16 before normalisation (p~_t = bf16(exp(s_t -
// m_ref)), normalised by the f32 sum of exp at the end); the reference max m_ref
// of a head moves only when a page max exceeds it by more than TAU (else
// exp(s - m_ref) <= e^TAU, far inside f32 / bf16 range); exp is the hardware ex2.
//
// Every wait is bounded: after WAIT_NS (1 s; shorter only through the diagnostic
// entry that tests this path) a wait sets K3MLA_DEV_TIMEOUT in the device error
// word, lets in-flight copies land and returns (no trap, no hang).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace k3 {

constexpr int NSLOT = 3;                       // score CTA: page slots (one producer + one issuer each)
constexpr int SLOT0 = 9 * PAGE * 128;          // 73728 B: [9 chunks][64 rows][128 B]
constexpr int CHUNK = PAGE * 128;              // 8192 B per chunk of a page slot
constexpr int HALF = 32;                       // PV CTA: tokens per half-page box
constexpr int THIRD = 3 * 8192;  // score CTA: a third of a page (3 chunks), one TMA box
constexpr int NHSLOT = 5;                      // PV CTA: half-page slots (one producer each)
constexpr int SLOT1 = 8 * HALF * 128;          // 32768 B: [8 chunks][32 rows][128 B], chunks 0..7 only
constexpr int HCHUNK = HALF * 128;             // 4096 B per chunk of a half-page slot

// The rows of a unit of work, one per TMEM lane of the score and PV contractions.  Decode: the 96 heads
// of one slot, 24 in each 32-lane quarter (lanes 24..31 idle), so that all four SM sub-partitions run
// softmax.  Multi-query (a prefill chunk): 32 heads of up to four consecutive tokens of one slot's chunk,
// one token per quarter, every lane a row; its larger Q and P tiles take a ring unit and a P buffer.
template <bool MQ> struct Cfg {
    static constexpr int RPQ = MQ ? 32 : 24;            // rows per 32-lane quarter
    static constexpr int ROWS = 4 * RPQ;                 // rows of the unit: 96 or 128
    static constexpr int NUNIT = MQ ? 7 : 8;             // score CTA: ring of third-page units
    static constexpr int Q_UNIT0 = MQ ? 2 : 4;           // score CTA: q_abs lands in ring units Q_UNIT0..
                                                         // (and the P staging area after them) until it is
                                                         // in TMEM, so the units before take pages meanwhile
    static constexpr int NPBUF = MQ ? 3 : 4;             // PV CTA: P buffers
    static constexpr int PSTAGE = RPQ * 128;             // score CTA: one softmax warp's P rows (x 64 tokens)
    static constexpr int QCHUNK = ROWS * 128;            // one 64-column chunk of Q, [rows][128 B]
    static constexpr int QBYTES = 9 * QCHUNK;            // q_abs of a unit (110592 B for decode)
    static constexpr int PT_BYTES = ROWS * 128;          // P^T [rows][64 tokens] bf16, K-major SW128
    static constexpr int META_ALPHA = PT_BYTES;          // f32 alpha[rows]
    static constexpr int META_FLAGS = PT_BYTES + 4 * ROWS;  // u32 flags[4]: "some row of quarter w rescaled"
    static constexpr int PCOPY = PT_BYTES + 4 * ROWS + 16;  // bytes stored per page (12688 for decode)
    static constexpr int PBUF = (PCOPY + 1023) / 1024 * 1024;  // buffer pitch: every P^T 1024-byte aligned
    static constexpr int WO_WARPS = MQ ? 8 : 6;          // PV CTA: warps writing O out
};
using CD = Cfg<false>;
constexpr int HPW = CD::RPQ;  // heads per softmax warp of the decode layout (lanes 0..23 of each quarter)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;                  // score CTA: S^T buffers r = 0..2 at 64 r
constexpr uint32_t Q_COL = 192;                // score CTA: Q, 288 columns (576 bf16)
constexpr float TAU = 16.0f;                   // max growth (natural log) before a rescale: p~ <= e^16,
                                               // l <= n e^16 stays far inside f32 for any context here
constexpr uint64_t WAIT_NS = 1000000000ull;    // bounded waits: 1 s
constexpr int PF_PAGES = 8;                    // PV CTA: L2 prefetch distance, pages past the latest P (measured
                                               // best of 4..9)
constexpr uint32_t IDESC_S = make_idesc_bf16(128, PAGE, 0, 0);  // S^T page = Q . C^T
constexpr uint32_t IDESC_PV = make_idesc_bf16(128, 256, 0, 1);  // O half = P . C (B MN-major)
// rank 0: warps 0-7 softmax, 8-10 producers, 11-13 MMA issuers; rank 1: warps 0-3
// epilogue, 4-8 producers, 9 MMA issuer, 10 L2 prefetch (decode), 11-13 idle.  Warp 8 allocates TMEM
// in both.
constexpr int THREADS = 448;
constexpr int W_PROD0 = 8, W_MMA0 = 11, W_ALLOC = 8;
// named barriers of the score CTA (0 is __syncthreads): the decision hand-off between the two
// softmax warps of a quarter (2 per quarter) and their final combine
constexpr uint32_t HAND_BAR0 = 1, FIN_BAR0 = 9;
// named barrier of the PV CTA's write-out (its six writing warps)
constexpr uint32_t WO_BAR = 13;
// 14 warps put four on some SM sub-partitions (16K registers each): at most 128 registers per thread.

template <bool MQ> struct __align__(1024) SmemT {
    using C = Cfg<MQ>;
    union {
        struct {
            uint8_t ring[C::NUNIT][THIRD];  // page thirds; q_abs is staged in units Q_UNIT0.. until in TMEM
            uint8_t pstage[8][C::PSTAGE];   // each softmax warp's P rows, copied to the PV CTA in bulk
        } c0;
        struct {
            uint8_t ring[NHSLOT][SLOT1];
            uint8_t recv[C::NPBUF][C::PBUF];
        } c1;
    } u;
    uint64_t full[9], empty[9];  // score CTA: one pair per third of a page slot; PV CTA: per half-slot
    uint64_t s_full[NSLOT], s_empty[NSLOT];
    uint64_t q_land, q_ready;
    uint64_t p_full[C::NPBUF], p_empty[C::NPBUF];
    uint64_t o_done, epi_req, epi_done;
    uint64_t l_full;         // PV CTA: 1 / l of every row has arrived (single-split launches)
    int32_t fin_ready;       // PV CTA: epilogue warps that saw O complete (4: write it out)
    int32_t p_seen;          // PV CTA: pages whose P has arrived (a count, read by the prefetch warp)
    float rl[C::ROWS];       // ... 1 / l by row, stored by the score CTA
    float xm[2][4][32];      // score CTA: reference max after a page, by page parity / quarter / lane
    float xa[2][4][32];      // ... and that page's rescale factor (1 when it kept the reference)
    float fin_l[4][32];      // ... the odd-page warp's sum of exp, best score and its token
    float fin_s[4][32];
    int32_t fin_t[4][32];
    // score CTA: the uses of a third-page unit go to different producer and issuer threads; a use
    // is handled only after the previous use of the unit has passed the same barrier, so a
    // barrier is never waited on two phases ahead (where its parity would repeat)
    int32_t unit_loaded[C::NUNIT];  // uses of the unit whose load has been issued
    int32_t unit_taken[C::NUNIT];   // uses of the unit whose MMAs have been issued
    uint32_t tmem_base;
    uint32_t epi_cmd, epi_slot0, epi_slot1, epi_stage, epi_vrows;
    int32_t abort_flag;
    int32_t early_n[NHSLOT];  // producer q: leading uses of its ring units loaded before the grid wait
    uint64_t wait_ns;  // the limit of every bounded wait of this CTA
    // multi-query: the token row of quarter w (-1: none) and its context length
    int32_t mq_row[4], mq_ntok[4];
};
template <bool MQ> constexpr bool smem_fits()
{
    using C = Cfg<MQ>;
    using S = SmemT<MQ>;
    static_assert(SLOT0 % 1024 == 0 && SLOT1 % 1024 == 0 && C::PBUF % 1024 == 0, "1024-byte aligned operand tiles");
    static_assert(NHSLOT <= 9 && 3 * NSLOT <= 9, "barrier arrays");
    static_assert(C::QBYTES <= (C::NUNIT - C::Q_UNIT0) * THIRD + 8 * C::PSTAGE,
                  "q_abs staging fits in units Q_UNIT0.. and the P staging area that follows them");
    static_assert((C::Q_UNIT0 * THIRD) % 1024 == 0 && C::PSTAGE % 128 == 0, "TMA and bulk-copy alignment");
    static_assert(C::PCOPY <= C::PBUF, "P buffer");
    static_assert(MQ || H * LORA * 4 <= NHSLOT * SLOT1 + C::NPBUF * C::PBUF,
                  "the final [96][512] f32 tile fits in the PV CTA's page ring and P buffers");
    static_assert((C::ROWS * 128) % 1024 == 0, "store boxes start 1024-byte aligned (128-byte swizzle)");
    static_assert((MQ ? 8 : 16) * C::ROWS * 128 <= NHSLOT * SLOT1 + C::NPBUF * C::PBUF,
                  "the write-out boxes fit in the ring and P buffers");
    static_assert(NHSLOT * SLOT1 + (C::NPBUF - 1) * C::PBUF + 128 * 128 <= sizeof(S::u),
                  "all 128 rows of the last P buffer, read as the A operand, lie in this CTA's tile area");
    static_assert(sizeof(S) + 1024 <= 227 * 1024, "shared memory of one CTA (with 1024-byte alignment slack)");
    return true;
}
static_assert(smem_fits<false>() && smem_fits<true>(), "shared-memory layouts");
using Smem = SmemT<false>;

struct DecodeParams {
    const int32_t* table;
    const int32_t* ctx_len;
    float* ws_o;    // [B][nsplit][96][512] f32 partials of slots with several splits (null if nsplit == 1)
    float* ws_ml;   // [B][nsplit][96][4]: m_ref, l, best score, best t (int bits)
    uint16_t* ws_olat;  // [96][B][512] bf16: final o_lat of every slot with at most one split
    int32_t* dev_err;
    int max_pages, n_pages, n_layers, layer;
    int B, max_ctx, split_tokens, nsplit;  // split_tokens 0: the default per-slot rule; nsplit: the grid's
    uint32_t scale2;  // the bf16 scale in both halves
    uint64_t wait_ns;  // bounded-wait limit: WAIT_NS, shorter only from the diagnostic entry
    int32_t withhold;  // diagnostic only, 0 otherwise: page k - 1's first third is never loaded
    int32_t early;     // 1 only from k3mla_decode_layer: see early_loads
    // multi-query units (a prefill chunk) only
    const int4* mq_groups;   // per group of up to four token rows: slot, first row, rows (0: no group)
    const int32_t* mq_ctx;   // per token row: its context length, clamped to the table
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

template <class S> __device__ __forceinline__ bool aborted(const S& sm)
{
    return *reinterpret_cast<const volatile int32_t*>(&sm.abort_flag) != 0;
}

// Bounded mbarrier wait, slow path: gives up after the CTA's wait limit or when this CTA aborted.
template <class S>
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, S& sm, int32_t* dev_err,
                                           bool cluster_scope)
{
    const uint32_t a = smem_u32(bar);
    if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
        if ((n & 127u) == 0) {
            if (aborted(sm)) return false;
            if (globaltimer() - t0 > sm.wait_ns) {
                *reinterpret_cast<volatile int32_t*>(&sm.abort_flag) = 1;
                if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded mbarrier wait: an inline non-blocking test first (most waits are already
// satisfied when they are reached), then the suspending slow path.
template <class S>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, S& sm, int32_t* dev_err,
                                         bool cluster_scope = false)
{
    const uint32_t a = smem_u32(bar);
    if (cluster_scope ? mbar_test_wait_cluster(a, parity) : mbar_test_wait(a, parity)) return true;
    return wait_bar_slow(bar, parity, sm, dev_err, cluster_scope);
}

// Bounded wait until a shared counter of this CTA reaches `target` (written by another thread of
// the CTA with a plain store); false when this CTA aborted or the wait timed out.
template <class S>
__device__ __noinline__ bool wait_count(const int32_t* counter, int32_t target, S& sm, int32_t* dev_err)
{
    const volatile int32_t* v = counter;
    if (*v >= target) return true;
    const uint64_t t0 = globaltimer();
    while (*v < target) {
        if (aborted(sm)) return false;
        if (globaltimer() - t0 > sm.wait_ns) {
            *reinterpret_cast<volatile int32_t*>(&sm.abort_flag) = 1;
            if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
    return true;
}

// After an abort: let this thread's in-flight TMA copies / MMAs land (bounded, ~2 ms).
__device__ __noinline__ void drain_inflight()
{
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
}

// First slab row of logical page lp of slot b at this layer, or a row past the
// end of the slab (the TMA box then reads zeros) for -1, for pages past the
// context, and for ids outside [-1, n_pages) (flagged).
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

// An empty context's final o_lat (single-split launches): zero rows [h][b][0:512] for every head.
__device__ __noinline__ void zero_olat(uint16_t* olat, int B, int b)
{
    for (int i = (int)threadIdx.x; i < H * LORA / 8; i += (int)blockDim.x)
        *reinterpret_cast<uint4*>(olat + ((size_t)(i / (LORA / 8)) * B + b) * LORA + 8 * (i % (LORA / 8))) =
            make_uint4(0u, 0u, 0u, 0u);
}

// ---- building blocks shared with the diagnostic kernel -----------------------------

// Score CTA, warps 0..3: copy Q (smem, [9 chunks][rows][128 B], 128-byte swizzle, as the TMA boxes
// land it) into TMEM columns [Q_COL, Q_COL + 288): lane 32w + l <- row RPQ w + l (l < RPQ), other
// lanes zero.
template <bool MQ> __device__ __forceinline__ void q_smem_to_tmem(uint32_t tbase, const uint8_t* qs)
{
    using C = Cfg<MQ>;
    const int w = (int)(threadIdx.x >> 5), l = (int)(threadIdx.x & 31);
    const int h = C::RPQ * w + l;
    const uint32_t taddr = tbase + ((32u * w) << 16) + Q_COL;
#pragma unroll 1
    for (int c = 0; c < 9; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (l < C::RPQ) v = *reinterpret_cast<const uint4*>(qs + c * C::QCHUNK + h * 128 + ((j ^ (h & 7)) << 4));
            r[4 * j + 0] = v.x;
            r[4 * j + 1] = v.y;
            r[4 * j + 2] = v.z;
            r[4 * j + 3] = v.w;
        }
        tmem_st32(taddr + c * 32, r);
    }
    tmem_wait_st();
}

// Score CTA: S^T[:, 64 tokens] = Q . C^T for one page slot (36 MMAs, K = 576).
// Descriptors advance by additions only, so the issuing thread spends its time
// issuing (chunk c is 8192 B = 512 descriptor units; a K step is 32 B = 2 units).
__device__ __forceinline__ void issue_score_page(uint32_t tbase, uint32_t d_col, uint32_t slot_addr)
{
    uint64_t bd = make_sdesc(slot_addr, 16, 1024);
    uint32_t a = tbase + Q_COL;
    const uint32_t d = tbase + d_col;
#pragma unroll 1
    for (int c = 0; c < 9; ++c) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_ts(d, a + 8u * ks, bd + 2u * ks, IDESC_S, (c | ks) != 0);
        a += 32u;
        bd += (uint64_t)(CHUNK >> 4);
    }
}

// Score CTA: the 12 K steps of third t (chunks 3t .. 3t+2, at third_addr) of the same product.
__device__ __forceinline__ void issue_score_third(uint32_t tbase, uint32_t d_col, uint32_t third_addr, int t)
{
    uint64_t bd = make_sdesc(third_addr, 16, 1024);
    uint32_t a = tbase + Q_COL + 96u * (uint32_t)t;
    const uint32_t d = tbase + d_col;
#pragma unroll
    for (int c = 0; c < 3; ++c) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_ts(d, a + 8u * ks, bd + 2u * ks, IDESC_S, (t | c | ks) != 0);
        a += 32u;
        bd += (uint64_t)(CHUNK >> 4);
    }
}

// PV CTA: O[128 rows = heads (rows 96.. unused) x 512 dims] (+)= P . C over one 64-token page held as
// two half-page slots ([8 chunks][32 rows][128 B] each).  A = P, K-major (the P buffer's rows are heads,
// 64 tokens each; rows 96..127 read whatever follows the buffer in this CTA's shared memory and only
// land in TMEM lanes nobody reads); B = C, MN-major (dims contiguous).  Two N = 256 halves of the dims
// x 4 K-steps of 16 tokens.
// Half hh of the page (tokens 32 hh .. 32 hh + 31, held in one slot): 4 MMAs.
__device__ __forceinline__ void issue_pv_half(uint32_t tbase, uint32_t half_addr, uint32_t pt_addr, int hh,
                                              bool accumulate_first)
{
    const uint64_t a0 = make_sdesc(pt_addr, 16, 1024);
    const uint64_t b0 = make_sdesc(half_addr, HCHUNK, 1024);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const uint64_t ad = a0 + (uint64_t)((uint32_t)((2 * hh + ks) * 32) >> 4);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const uint64_t bd = b0 + (uint64_t)((uint32_t)(4 * n * HCHUNK + ks * 2048) >> 4);
            umma_ss(tbase + 256u * n, ad, bd, IDESC_PV, (accumulate_first || hh > 0 || ks > 0) ? 1u : 0u);
        }
    }
}

__device__ __forceinline__ void issue_pv_page(uint32_t tbase, uint32_t half0_addr, uint32_t half1_addr,
                                              uint32_t pt_addr, bool accumulate_first)
{
    issue_pv_half(tbase, half0_addr, pt_addr, 0, accumulate_first);
    issue_pv_half(tbase, half1_addr, pt_addr, 1, accumulate_first);
}

// Byte offset in a P^T buffer of the 16-byte chunk with tokens 8j .. 8j+7 of head h.
__device__ __forceinline__ uint32_t pt_chunk_off(int h, int j) { return (uint32_t)(h * 128 + ((j ^ (h & 7)) << 4)); }

// PV CTA, after its roles: O [rows x 512 dims] f32 leaves TMEM through the (now idle) page ring and P
// buffers, laid out there as the 128-byte-swizzled boxes of bulk tensor stores: [rows][64 dims] bf16
// boxes of final o_lat = bf16(O * (1 / l)) when the unit is the row's only split, else [96 heads][32
// dims] f32 boxes of the split's partial as it stands (decode only: a multi-query unit always holds
// whole contexts).  Thread = row (TMEM lane); warps 0-2 (multi-query: 0-3) write the dims 0..255 and
// warps 4-6 (4-7) the dims 256..511, 64 dims (two TMEM loads, one wait) at a time, 16 bytes per store;
// whenever both halves have written theirs, thread 0 stores those boxes while the warps go on.  At the
// end it waits until the stores have read the tile (the writes reach global memory before the grid
// counts as complete, which is what the merge kernel waits for).  Kept out of line so that it does not
// weigh on the register allocation of the pipeline.  b: the slot; hb: a multi-query unit's head block.
template <bool MQ>
__device__ __noinline__ void pv_write_out(SmemT<MQ>& sm, const CUtensorMap* tm_olat, const CUtensorMap* tm_part,
                                          bool single, int nsplit, uint32_t tbase, int b, int s, int hb)
{
    using C = Cfg<MQ>;
    constexpr int BOX = C::ROWS * 128;  // one box of every row of the unit
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    uint8_t* tile = sm.u.c1.ring[0];
    if (warp < 8 && (MQ || (warp & 3u) < 3u)) {
        tc_fence_after();
        const int h = 32 * (int)(warp & 3u) + (int)lane, half = (int)(warp >> 2);
        const uint32_t ta = tbase + ((32u * (warp & 3u)) << 16) + 256u * (uint32_t)half;
        const float r = single ? sm.rl[h] : 1.f;
        const uint32_t sw = (uint32_t)(h & 7);
#pragma unroll 1
        for (int k2 = 0; k2 < 4; ++k2) {  // dims 256 half + 64 k2 .. + 63: two loads, one wait
            uint32_t rr[2][32];
            tmem_ld32(ta + 64u * (uint32_t)k2, rr[0]);
            tmem_ld32(ta + 64u * (uint32_t)k2 + 32u, rr[1]);
            tmem_wait_ld();
            if (MQ || single) {  // box 4 half + k2 (64 dims): the eight 16-byte chunks of row h
                uint8_t* row = tile + (4 * half + k2) * BOX + h * 128;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t* v = rr[i >> 2] + 8 * (i & 3);
                    *reinterpret_cast<uint4*>(row + (((uint32_t)i ^ sw) << 4)) =
                        make_uint4(pack_bf16x2(__uint_as_float(v[0]) * r, __uint_as_float(v[1]) * r),
                                   pack_bf16x2(__uint_as_float(v[2]) * r, __uint_as_float(v[3]) * r),
                                   pack_bf16x2(__uint_as_float(v[4]) * r, __uint_as_float(v[5]) * r),
                                   pack_bf16x2(__uint_as_float(v[6]) * r, __uint_as_float(v[7]) * r));
                }
            } else if constexpr (!MQ) {  // boxes 8 half + 2 k2 and + 1 (32 dims each): all chunks of row h
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint8_t* row = tile + (8 * half + 2 * k2 + e) * BOX + h * 128;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<uint4*>(row + (((uint32_t)i ^ sw) << 4)) =
                            make_uint4(rr[e][4 * i], rr[e][4 * i + 1], rr[e][4 * i + 2], rr[e][4 * i + 3]);
                }
            }
            fence_proxy_async_cta();  // the boxes are read by bulk tensor stores (async proxy)
            named_bar(WO_BAR, C::WO_WARPS * 32);
            if (threadIdx.x == 0) {
                if constexpr (MQ) {  // o_lat [96][R][512] as (512 dims, 96 heads, R rows): a full group's
                    // four rows in one box (64, 32, 4), else each row in its own (the rows after a short
                    // group belong to other units)
                    if (sm.mq_row[3] >= 0) {
                        tma_store_3d(tm_olat, tile + k2 * BOX, 64 * k2, 32 * hb, sm.mq_row[0]);
                        tma_store_3d(tm_olat, tile + (4 + k2) * BOX, 256 + 64 * k2, 32 * hb, sm.mq_row[0]);
                    } else {
                        for (int w = 0; w < 4; ++w) {
                            const int row = sm.mq_row[w];
                            if (row < 0) continue;
                            tma_store_3d(tm_part, tile + k2 * BOX + 32 * w * 128, 64 * k2, 32 * hb, row);
                            tma_store_3d(tm_part, tile + (4 + k2) * BOX + 32 * w * 128, 256 + 64 * k2, 32 * hb, row);
                        }
                    }
                } else if (single) {  // o_lat [96][B][512] as (512 dims, B slots, 96 heads), box (64, 1, 96)
                    tma_store_3d(tm_olat, tile + k2 * (H * 128), 64 * k2, b, 0);
                    tma_store_3d(tm_olat, tile + (4 + k2) * (H * 128), 256 + 64 * k2, b, 0);
                } else {  // partials [B][nsplit][96][512] as (512 dims, rows), box (32, 96)
                    const int row0 = (b * nsplit + s) * H;
                    for (int e = 0; e < 2; ++e) {
                        tma_store_2d(tm_part, tile + (2 * k2 + e) * (H * 128), 64 * k2 + 32 * e, row0);
                        tma_store_2d(tm_part, tile + (8 + 2 * k2 + e) * (H * 128), 256 + 64 * k2 + 32 * e, row0);
                    }
                }
                bulk_commit();
            }
        }
        if (threadIdx.x == 0) bulk_wait_read<0>();
    }
}

// ---- one split: geometry, barriers -------------------------------------------------------

// Where split s of slot b lies: set from the slot's (clamped) context; false for an empty split.
struct SplitGeom {
    int b, s, start, ntok, npg, n_lp, lp0;
    int hb;           // a multi-query unit's head block (heads 32 hb .. 32 hb + 31)
    bool single;      // the slot has at most one split: the PV CTA lands final o_lat itself
    int32_t oob_row;  // a slab row past the end (a TMA box there reads zeros)
};

__device__ __forceinline__ bool split_geom(SplitGeom& g, int ctx, const DecodeParams& p)
{
    const int split = slot_split(ctx, p.split_tokens);
    g.single = slot_nsplit(ctx, split) <= 1;
    g.start = g.s * split;
    if (g.start >= ctx) return false;
    g.ntok = min(ctx, g.start + split) - g.start;
    g.npg = (g.ntok + PAGE - 1) / PAGE;
    g.n_lp = (ctx + PAGE - 1) / PAGE;
    g.lp0 = g.start / PAGE;
    g.oob_row = p.n_pages * p.n_layers * PAGE;
    return true;
}

// Score CTA: where q_abs is staged (ring units Q_UNIT0.. and the P staging area after them).
template <bool MQ> __device__ __forceinline__ uint8_t* q_stage(SmemT<MQ>& sm)
{
    return reinterpret_cast<uint8_t*>(&sm.u) + Cfg<MQ>::Q_UNIT0 * THIRD;
}

// Thread 0: the mbarriers and counters of one split (the caller fences them for the cluster).
template <bool MQ>
__device__ __forceinline__ void init_decode_barriers(SmemT<MQ>& sm, uint32_t rank, bool single, uint64_t wait_ns)
{
    using C = Cfg<MQ>;
    sm.wait_ns = wait_ns;
    for (int i = 0; i < 9; ++i) {
        mbar_init(&sm.full[i], 1);
        mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < NSLOT; ++i) {
        mbar_init(&sm.s_full[i], 1);
        mbar_init(&sm.s_empty[i], 4);
    }
    for (int i = 0; i < C::NPBUF; ++i) {
        mbar_init(&sm.p_full[i], 1);
        mbar_init(&sm.p_empty[i], 1);
    }
    mbar_init(&sm.q_land, 1);
    mbar_init(&sm.q_ready, 4);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.epi_req, 1);
    mbar_init(&sm.epi_done, 4);
    mbar_init(&sm.l_full, 1);
    sm.abort_flag = 0;
    sm.fin_ready = 0;
    sm.p_seen = 0;
    for (int i = 0; i < NHSLOT; ++i) sm.early_n[i] = 0;
    for (int i = 0; i < C::NUNIT; ++i) {
        sm.unit_loaded[i] = 0;
        sm.unit_taken[i] = 0;
    }
    if (rank == 1) {  // the P buffers of pages 0 .. NPBUF-1 are expected before anything is sent
        for (int i = 0; i < C::NPBUF; ++i) mbar_arrive_expect_tx(&sm.p_full[i], C::PCOPY);
        if (single) mbar_arrive_expect_tx(&sm.l_full, 4 * C::ROWS);
    }
}

// The roles of both CTAs for one split: q_abs into TMEM, the page ring, the two contractions, the softmax,
// and the PV CTA's write-out of O.  Inlined into the kernel: the parameters it reads in its loops stay
// constant-bank operands (an out-of-line copy, reaching them through a pointer, ran some 50 % slower).
// A multi-query unit (MQ) runs the same roles over its rows: quarter w holds heads 32 hb .. 32 hb + 31 of
// token row mq_row[w], whose context is the first mq_ntok[w] tokens of the unit's pages.
template <bool MQ>
__device__ __forceinline__ void decode_roles(SmemT<MQ>& sm, const CUtensorMap& tmap_page, const CUtensorMap& tmap_page8,
                                             const CUtensorMap& tmap_q, const CUtensorMap& tmap_olat,
                                             const CUtensorMap& tmap_part, const DecodeParams& p, const SplitGeom& sg,
                                             uint32_t tbase, uint32_t rank, uint32_t warp, uint32_t lane)
{
    using C = Cfg<MQ>;
    const int b = sg.b, s = sg.s, start = sg.start, ntok = sg.ntok, npg = sg.npg, n_lp = sg.n_lp, lp0 = sg.lp0;
    const bool single = sg.single;
    const int32_t oob_row = sg.oob_row;
    if (rank == 0 && threadIdx.x == 0) {  // q_abs of the unit, staged in ring units Q_UNIT0.. until in TMEM
        if constexpr (MQ) {  // per chunk one box: heads 32 hb .. of four consecutive token rows, row w of the
            // group at row 32 w of the chunk (rows past the group are loaded too, or read as zeros past
            // the last token row, and land in lanes nobody reads)
            mbar_arrive_expect_tx(&sm.q_land, C::QBYTES);
            for (int c = 0; c < 9; ++c)
                tma_load_4d(q_stage(sm) + c * C::QCHUNK, &tmap_q, 0, 32 * sg.hb, sm.mq_row[0], c, &sm.q_land);
        } else {
            mbar_arrive_expect_tx(&sm.q_land, C::QBYTES);
            for (int c = 0; c < 9; ++c) tma_load_3d(q_stage(sm) + c * C::QCHUNK, &tmap_q, 0, b * H, c, &sm.q_land);
        }
    }

    if (rank == 0) {
        // =========================== score CTA ===========================
        if (warp >= W_PROD0 && warp < W_PROD0 + NSLOT) {
            if (lane == 0) {  // producer t streams third t (chunks 3t .. 3t+2) of every page
                // third g = 3i + t of the split lives in unit g % NUNIT; a unit's uses are strictly
                // ordered (a use is loaded only after the MMAs of the previous use released it)
                const int t = (int)warp - W_PROD0;
                bool ok = true, q_in_tmem = false;
                for (int i = sm.early_n[t]; i < npg && ok; ++i) {
                    const int g = 3 * i + t, u = g % C::NUNIT, k = g / C::NUNIT;
                    if (!q_in_tmem && g >= C::Q_UNIT0) {  // units Q_UNIT0.. hold q_abs until it is in TMEM
                        ok = wait_bar(&sm.q_ready, 0, sm, p.dev_err);
                        q_in_tmem = true;
                    }
                    if (!ok || (t == 0 && i + 1 == p.withhold)) break;  // (diagnostic: a load never issued)
                    const int32_t y = page_row(p, b, lp0 + i, n_lp, oob_row);
                    if (!wait_count(&sm.unit_loaded[u], k, sm, p.dev_err) ||
                        !wait_bar(&sm.empty[u], (uint32_t)(k & 1) ^ 1u, sm, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    *reinterpret_cast<volatile int32_t*>(&sm.unit_loaded[u]) = k + 1;
                    mbar_arrive_expect_tx(&sm.full[u], THIRD);
                    tma_load_3d(sm.u.c0.ring[u], &tmap_page, 0, y, 3 * t, &sm.full[u]);
                }
                if (!ok) drain_inflight();
            }
        } else if (warp >= W_MMA0 && warp < W_MMA0 + NSLOT) {
            if (lane == 0) {  // MMA issuer r: scores of the pages i = r (mod 3) into S buffer r
                const int r = (int)warp - W_MMA0;
                bool ok = wait_bar(&sm.q_ready, 0, sm, p.dev_err);
                tc_fence_after();
                for (int i = r; i < npg && ok; i += NSLOT) {
                    const int k = i / NSLOT;
                    if (!wait_bar(&sm.s_empty[r], (uint32_t)(k & 1) ^ 1u, sm, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    for (int t = 0; t < 3 && ok; ++t) {
                        const int g = 3 * i + t, u = g % C::NUNIT, ku = g / C::NUNIT;
                        if (!wait_count(&sm.unit_taken[u], ku, sm, p.dev_err) ||
                            !wait_bar(&sm.full[u], (uint32_t)(ku & 1), sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        *reinterpret_cast<volatile int32_t*>(&sm.unit_taken[u]) = ku + 1;
                        tc_fence_after();
                        issue_score_third(tbase, S_COL + 64u * r, smem_u32(sm.u.c0.ring[u]), t);
                        umma_commit(&sm.empty[u]);
                    }
                    if (ok) umma_commit(&sm.s_full[r]);
                }
                if (!ok) drain_inflight();
            }
        } else if (warp < 8) {
            // softmax warps 0..7: warp (qd = warp % 4, par = warp / 4) owns rows RPQ qd .. RPQ qd + RPQ-1
            // (thread l < RPQ -> row RPQ qd + l; decode: head 24 qd + l) for all 64 tokens of the pages
            // of parity par.  The
            // reference max is a chain through the pages: each warp hands its page's decision (new
            // reference max, rescale factor) to the other warp of its quarter through shared memory
            // and a named barrier, and takes the previous page's decision from it; everything else
            // (scores, max, argmax, exp, the P store) of the two pages runs in parallel.
            const int qd = (int)(warp & 3u), par = (int)(warp >> 2), l = (int)lane;
            const int h = C::RPQ * qd + l;  // the row (decode: the head)
            const bool has_head = l < C::RPQ;
            const int ntok_q = MQ ? sm.mq_ntok[qd] : ntok;  // the row's tokens in this split
            const uint32_t bar_in = HAND_BAR0 + 2u * (uint32_t)qd + (uint32_t)(par ^ 1);
            const uint32_t bar_out = HAND_BAR0 + 2u * (uint32_t)qd + (uint32_t)par;
            if (par == 0) {
                const bool qok = wait_bar(&sm.q_land, 0, sm, p.dev_err);
                if (__all_sync(0xFFFFFFFFu, qok)) q_smem_to_tmem<MQ>(tbase, q_stage(sm));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.q_ready);
            }
            const uint32_t t_lane = tbase + ((32u * qd) << 16) + S_COL;
            const float LOG2E = 1.4426950408889634f;
            float m_ref = -INFINITY, lsum = 0.f, best_s = -INFINITY;
            int best_t = -1;
            const uint32_t recv0 = mapa(smem_u32(sm.u.c1.recv[0]), 1);
            const uint32_t pfull0 = mapa(smem_u32(&sm.p_full[0]), 1);
            bool ok = true;
            for (int i = par; i < npg; i += 2) {
                const int r = i % NSLOT, k = i / NSLOT;
                if (ok) ok = __all_sync(0xFFFFFFFFu, wait_bar(&sm.s_full[r], (uint32_t)(k & 1), sm, p.dev_err));
                const int nvalid = min(PAGE, ntok_q - PAGE * i);
                uint32_t sp[32];  // bf16 scores: token 2q in the low half, 2q+1 in the high half
                if (ok) {
                    tc_fence_after();
                    uint32_t ra[32], rb[32];  // the page's 64 f32 scores of this thread's head
                    tmem_ld32(t_lane + 64u * r, ra);
                    tmem_ld32(t_lane + 64u * r + 32u, rb);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.s_empty[r]);  // the S buffer is free for page i + 3
#pragma unroll
                    for (int q = 0; q < 16; ++q) {  // bf16(dot), then bf16(bf16(dot) * scale)
                        sp[q] = mul_bf16x2(pack_bf16x2(__uint_as_float(ra[2 * q]), __uint_as_float(ra[2 * q + 1])),
                                           p.scale2);
                        sp[16 + q] = mul_bf16x2(
                            pack_bf16x2(__uint_as_float(rb[2 * q]), __uint_as_float(rb[2 * q + 1])), p.scale2);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) sp[q] = 0xFF80FF80u;
                }
                if (nvalid < PAGE) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        if (2 * q >= nvalid) sp[q] = (sp[q] & 0xFFFF0000u) | 0xFF80u;  // -inf
                        if (2 * q + 1 >= nvalid) sp[q] = (sp[q] & 0x0000FFFFu) | 0xFF800000u;
                    }
                }
                uint32_t g[8];  // max of each group of 8 tokens (packed: even tokens low, odd high)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    g[j] = max_bf16x2(max_bf16x2(sp[4 * j], sp[4 * j + 1]), max_bf16x2(sp[4 * j + 2], sp[4 * j + 3]));
                const uint32_t g4 = max_bf16x2(max_bf16x2(max_bf16x2(g[0], g[1]), max_bf16x2(g[2], g[3])),
                                               max_bf16x2(max_bf16x2(g[4], g[5]), max_bf16x2(g[6], g[7])));
                const float pmax = fmaxf(bf16lo_to_f32(g4), bf16hi_to_f32(g4));
                if (pmax > best_s) {  // lowest logical t attaining the best score
                    best_s = pmax;
                    int jg = 7;  // first group holding the max ...
#pragma unroll
                    for (int j = 6; j >= 0; --j)
                        if (fmaxf(bf16lo_to_f32(g[j]), bf16hi_to_f32(g[j])) == pmax) jg = j;
                    uint32_t w[4] = {sp[0], sp[1], sp[2], sp[3]};
#pragma unroll
                    for (int j = 1; j < 8; ++j)
                        if (jg == j) {
                            w[0] = sp[4 * j];
                            w[1] = sp[4 * j + 1];
                            w[2] = sp[4 * j + 2];
                            w[3] = sp[4 * j + 3];
                        }
                    int tq = 7;  // ... and the first token in it
#pragma unroll
                    for (int q = 3; q >= 0; --q) {
                        if (bf16hi_to_f32(w[q]) == pmax) tq = 2 * q + 1;
                        if (bf16lo_to_f32(w[q]) == pmax) tq = 2 * q;
                    }
                    best_t = start + PAGE * i + 8 * jg + tq;
                }
                // the decision of page i - 1, from the other warp
                float m_prev = -INFINITY;
                if (i > 0) {
                    named_bar(bar_in, 64);
                    m_prev = sm.xm[(i - 1) & 1][qd][l];
                    lsum *= sm.xa[(i - 1) & 1][qd][l];
                }
                float alpha = 1.f;
                bool resc = false;
                if (i == 0) {
                    m_ref = pmax;
                } else if (pmax > m_prev + TAU) {
                    alpha = ex2_approx((m_prev - pmax) * LOG2E);
                    lsum *= alpha;
                    m_ref = pmax;
                    resc = true;
                } else {
                    m_ref = m_prev;
                }
                sm.xm[i & 1][qd][l] = m_ref;  // hand this page's decision on
                sm.xa[i & 1][qd][l] = alpha;
                named_bar_arrive(bar_out, 64);
                // (multi-query: a row with no token yet keeps m_ref = -inf, and its p~ = exp(-inf) = 0)
                const float mb = (MQ && m_ref == -INFINITY) ? 0.f : m_ref * LOG2E;
                float part[8];  // independent partial sums, combined in a fixed order below
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // tokens 8j .. 8j+7: p~ = bf16(exp(s - m_ref)), in place of s
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t s2 = sp[4 * j + q];
                        const float e0 = ex2_approx(fmaf(bf16lo_to_f32(s2), LOG2E, -mb));
                        const float e1 = ex2_approx(fmaf(bf16hi_to_f32(s2), LOG2E, -mb));
                        acc += e0 + e1;
                        sp[4 * j + q] = pack_bf16x2(e0, e1);
                    }
                    part[j] = acc;
                }
                lsum += ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
                const int st = i % C::NPBUF;
                // this warp's P rows, laid out as they land (rows 24 qd .. 24 qd + 23 of the P^T
                // buffer), once the bulk copy of its previous page has read the staging rows
                uint8_t* stage = sm.u.c0.pstage[warp];
                if (lane == 0 && i >= 2) bulk_wait_read<0>();
                __syncwarp();
                if (has_head) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(stage + pt_chunk_off(h, j) - qd * C::PSTAGE) =
                            make_uint4(sp[4 * j], sp[4 * j + 1], sp[4 * j + 2], sp[4 * j + 3]);
                }
                fence_proxy_async_cta();  // the bulk copy reads the rows through the async proxy
                __syncwarp();
                // the PV CTA has finished with its buffer from page i - NPBUF
                bool freed = false;
                if (ok) freed = wait_bar(&sm.p_empty[st], (uint32_t)((i / C::NPBUF) & 1) ^ 1u, sm, p.dev_err);
                const uint32_t dst = recv0 + (uint32_t)(st * C::PBUF);
                const uint32_t bar = pfull0 + (uint32_t)(st * sizeof(uint64_t));
                if (freed && lane == 0) {
                    bulk_copy_to_cluster(dst + (uint32_t)(qd * C::PSTAGE), stage, C::PSTAGE, bar);
                    bulk_commit();
                }
                if (freed && has_head) st_async_b32(dst + C::META_ALPHA + 4 * h, __float_as_uint(alpha), bar);
                const uint32_t any = __ballot_sync(0xFFFFFFFFu, resc && has_head);
                if (freed && lane == 0) st_async_b32(dst + C::META_FLAGS + 4 * qd, any ? 1u : 0u, bar);
            }
            // the other warp's decision on the last page, when that page was not this warp's
            const int last = npg - 1;
            if ((last & 1) != par) {
                named_bar(bar_in, 64);
                m_ref = sm.xm[last & 1][qd][l];
                lsum *= sm.xa[last & 1][qd][l];
            }
            // l = (sum over even pages) + (sum over odd pages); best = the larger score, the lower t on ties
            if (par == 1) {
                sm.fin_l[qd][l] = lsum;
                sm.fin_s[qd][l] = best_s;
                sm.fin_t[qd][l] = best_t;
            }
            named_bar(FIN_BAR0 + (uint32_t)qd, 64);
            if (par == 0 && has_head && ok && !aborted(sm)) {
                const float s1 = sm.fin_s[qd][l];
                const int t1 = sm.fin_t[qd][l];
                if (s1 > best_s || (s1 == best_s && t1 < best_t && t1 >= 0)) {
                    best_s = s1;
                    best_t = t1;
                }
                const float ltot = lsum + sm.fin_l[qd][l];
                // multi-query: row (token row mq_row[qd], head 32 hb + l); a quarter without a token row
                // writes no record, and a row without tokens lands zeros (1 / l taken as 0)
                const int row = MQ ? sm.mq_row[qd] : b;
                if (!MQ || row >= 0) {
                    float* ml = MQ ? p.ws_ml + ((size_t)row * H + 32 * sg.hb + l) * 4
                                   : p.ws_ml + (((size_t)b * p.nsplit + s) * H + h) * 4;
                    ml[0] = m_ref;
                    ml[1] = ltot;
                    ml[2] = best_s;
                    ml[3] = __int_as_float(best_t);
                }
                // a single split is final: the PV CTA lands o_lat = bf16(O * (1 / l)) itself
                if (single)
                    st_async_b32(mapa(smem_u32(&sm.rl[h]), 1),
                                 __float_as_uint((MQ && !(ltot > 0.f)) ? 0.f : 1.f / ltot),
                                 mapa(smem_u32(&sm.l_full), 1));
            }
            // this warp's bulk copies are complete (their bytes have landed in the PV CTA), and the PV
            // CTA's last releases of its P buffers land here, before exit
            if (lane == 0) {
                bulk_wait<0>();
                for (int i = max(0, npg - C::NPBUF); i < npg && !aborted(sm); ++i)
                    wait_bar(&sm.p_empty[i % C::NPBUF], (uint32_t)((i / C::NPBUF) & 1), sm, p.dev_err);
            }
        }
    } else {
        // ============================ PV CTA ============================
        if (warp >= 4 && warp <= 8) {
            if (lane == 0) {  // producer q streams the half pages u = q (mod 5) into half-slot q
                const uint64_t pol = policy_evict_first();  // last reader of the latent
                const int q = (int)warp - 4;
                bool ok = true;
                for (int u = q + NHSLOT * sm.early_n[q]; u < 2 * npg && ok; u += NHSLOT) {
                    const int k = u / NHSLOT;
                    const int32_t y = page_row(p, b, lp0 + u / 2, n_lp, oob_row) + HALF * (u & 1);
                    if (!wait_bar(&sm.empty[q], (uint32_t)(k & 1) ^ 1u, sm, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.full[q], SLOT1);
                    tma_load_3d_hint(sm.u.c1.ring[q], &tmap_page8, 0, y, 0, &sm.full[q], pol);
                }
                if (!ok) drain_inflight();
            }
        } else if (warp == 9) {
            if (lane == 0) {
                uint32_t epi_k = 0;
                bool ok = true;
                for (int i = 0; i < npg && ok; ++i) {
                    const int st = i % C::NPBUF;
                    if (!wait_bar(&sm.p_full[st], (uint32_t)((i / C::NPBUF) & 1), sm, p.dev_err, true)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_cta();  // the P tile arrived through st.async; the MMA reads it
                    if constexpr (!MQ) *reinterpret_cast<volatile int32_t*>(&sm.p_seen) = i + 1;
                    const volatile uint32_t* rf =
                        reinterpret_cast<const volatile uint32_t*>(sm.u.c1.recv[st] + C::META_FLAGS);
                    const bool resc = (i > 0) && ((rf[0] | rf[1] | rf[2] | rf[3]) != 0u);
                    const int nvalid = min(PAGE, ntok - PAGE * i);
                    const bool tail = nvalid < PAGE;
                    const int u0 = 2 * i, q0 = u0 % NHSLOT, q1 = (u0 + 1) % NHSLOT;
                    if (!wait_bar(&sm.full[q0], (uint32_t)((u0 / NHSLOT) & 1), sm, p.dev_err) ||
                        !wait_bar(&sm.full[q1], (uint32_t)(((u0 + 1) / NHSLOT) & 1), sm, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    if (resc || tail) {
                        if (resc) umma_commit(&sm.o_done);
                        sm.epi_cmd = (resc ? 1u : 0u) | (tail ? 2u : 0u);
                        sm.epi_slot0 = (uint32_t)q0;
                        sm.epi_slot1 = (uint32_t)q1;
                        sm.epi_stage = (uint32_t)st;
                        sm.epi_vrows = (uint32_t)nvalid;
                        mbar_arrive(&sm.epi_req);
                        if (!wait_bar(&sm.epi_done, epi_k & 1u, sm, p.dev_err)) {
                            ok = false;
                            break;
                        }
                        ++epi_k;
                    }
                    tc_fence_after();
                    // each half-page slot goes back to its producer once the four MMAs that read it are done
                    issue_pv_half(tbase, smem_u32(sm.u.c1.ring[q0]), smem_u32(sm.u.c1.recv[st]), 0, i > 0);
                    umma_commit(&sm.empty[q0]);
                    issue_pv_half(tbase, smem_u32(sm.u.c1.ring[q1]), smem_u32(sm.u.c1.recv[st]), 1, i > 0);
                    umma_commit(&sm.empty[q1]);
                    umma_commit_mc(&sm.p_empty[st], (uint16_t)0x1);
                    if (i + C::NPBUF < npg) mbar_arrive_expect_tx(&sm.p_full[st], C::PCOPY);
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
        } else if (!MQ && warp == 10) {
            if (lane == 0) {  // once the P of page i has arrived, page i + PF_PAGES is prefetched into L2 for
                              // the score CTA.  The warp follows the PV issuer's count of pages (a barrier's
                              // parity would repeat if it fell behind) and skips the pages it fell behind on.
                for (int i = 0; i + PF_PAGES < npg; ++i) {
                    if (!wait_count(&sm.p_seen, i + 1, sm, p.dev_err)) break;
                    i = max(i, *reinterpret_cast<volatile int32_t*>(&sm.p_seen) - 1);
                    if (i + PF_PAGES >= npg) break;
                    const int32_t y = page_row(p, b, lp0 + i + PF_PAGES, n_lp, oob_row);
                    if (y != oob_row)
                        for (int t = 0; t < 3; ++t) tma_prefetch_3d(&tmap_page, 0, y, 3 * t);
                }
            }
        } else if (warp < 4) {
            // epilogue warps 0..3: thread owns TMEM lane 32*warp + lane, the O row of that head (lanes
            // 96.. are not heads)
            const uint32_t t_lane = tbase + ((32u * warp) << 16);
            uint32_t k = 0, od = 0;
            for (;;) {
                const bool got = wait_bar(&sm.epi_req, k & 1u, sm, p.dev_err);
                if (!__all_sync(0xFFFFFFFFu, got)) break;
                ++k;
                const uint32_t cmd = *reinterpret_cast<volatile uint32_t*>(&sm.epi_cmd);
                if (cmd & 1u) {  // rescale each head's O row by its alpha
                    const bool got2 = wait_bar(&sm.o_done, od & 1u, sm, p.dev_err);
                    if (!__all_sync(0xFFFFFFFFu, got2)) break;
                    ++od;
                    tc_fence_after();
                    const float* al = reinterpret_cast<const float*>(sm.u.c1.recv[sm.epi_stage] + C::META_ALPHA);
                    const float a = (MQ || warp < 3) ? al[32 * warp + lane] : 1.f;
                    if (__any_sync(0xFFFFFFFFu, a != 1.f)) {  // some head of this warp moved its reference
#pragma unroll 1
                        for (int cb = 0; cb < LORA / 32; ++cb) {
                            uint32_t rr[32];
                            tmem_ld32(t_lane + 32u * cb, rr);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c) rr[c] = __float_as_uint(__uint_as_float(rr[c]) * a);
                            tmem_st32(t_lane + 32u * cb, rr);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                }
                if (cmd & 2u) {  // zero rows >= vrows of chunks 0..7 of the final page (two half slots)
                    const int vr = (int)sm.epi_vrows;
                    const int per_chunk = (PAGE - vr) * 8;  // 16-byte pieces
                    for (int q = (int)threadIdx.x; q < 8 * per_chunk; q += 128) {
                        const int c = q / per_chunk, rem = q % per_chunk;
                        const int row = vr + rem / 8;  // page row
                        uint8_t* half = sm.u.c1.ring[row < HALF ? sm.epi_slot0 : sm.epi_slot1];
                        *reinterpret_cast<uint4*>(half + c * HCHUNK + (row % HALF) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_cta();
                }
                if (cmd & 4u) {  // final: O is complete (and, single split, 1 / l has arrived)
                    bool got2 = wait_bar(&sm.o_done, od & 1u, sm, p.dev_err);
                    if (single) got2 = got2 && wait_bar(&sm.l_full, 0, sm, p.dev_err, true);
                    if (__all_sync(0xFFFFFFFFu, got2) && lane == 0) atomicAdd(&sm.fin_ready, 1);
                    break;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.epi_done);
            }
        }
        __syncthreads();  // every role is done: the final write-out takes all warps
        if (*reinterpret_cast<volatile int32_t*>(&sm.fin_ready) == 4)
            pv_write_out<MQ>(sm, &tmap_olat, &tmap_part, single, p.nsplit, tbase, b, s, sg.hb);
    }

}

// The first uses of both page rings, issued before the grid wait when the kernel before in the stream
// is this library's absorption-append launch of the same layer-call (k3mla_decode_layer).  That
// launch writes only q_abs and the step's row of each slot, which lies in the slot's last logical
// page, so every other page is loaded here: the loads overlap the absorption.  Nothing else writes
// the slab or the block table meanwhile: the absorption-append grid lets this kernel start only
// after each of its CTAs has waited for the kernel before it to complete.  Producer lanes only.
__device__ __forceinline__ void early_loads(Smem& sm, const CUtensorMap& tmap_page, const CUtensorMap& tmap_page8,
                                            const DecodeParams& p, const SplitGeom& sg, uint32_t rank,
                                            uint32_t warp, uint32_t lane)
{
    if (lane != 0) return;
    if (rank == 0 && warp >= W_PROD0 && warp < W_PROD0 + NSLOT) {
        // producer t: third t of pages 0, 1, ... while they fall in the units q_abs leaves free
        const int t = (int)warp - W_PROD0;
        int i = 0;
        for (; 3 * i + t < CD::Q_UNIT0 && i < sg.npg && sg.lp0 + i < sg.n_lp - 1; ++i) {
            const int u = 3 * i + t;  // the unit's first use
            *reinterpret_cast<volatile int32_t*>(&sm.unit_loaded[u]) = 1;
            mbar_arrive_expect_tx(&sm.full[u], THIRD);
            tma_load_3d(sm.u.c0.ring[u], &tmap_page, 0, page_row(p, sg.b, sg.lp0 + i, sg.n_lp, sg.oob_row), 3 * t,
                        &sm.full[u]);
        }
        sm.early_n[t] = i;
    } else if (rank == 1 && warp >= 4 && warp <= 8) {
        // producer q: half page q into half-slot q (its first use)
        const int q = (int)warp - 4;
        if (q < 2 * sg.npg && sg.lp0 + q / 2 < sg.n_lp - 1) {
            mbar_arrive_expect_tx(&sm.full[q], SLOT1);
            tma_load_3d_hint(sm.u.c1.ring[q], &tmap_page8, 0,
                             page_row(p, sg.b, sg.lp0 + q / 2, sg.n_lp, sg.oob_row) + HALF * (q & 1), 0, &sm.full[q],
                             policy_evict_first());
            sm.early_n[q] = 1;
        }
    }
}

// ---- the split decode kernel ---------------------------------------------------------

// MQ: the multi-query form of a prefill chunk.  Unit u is head block u % 3 of group u / 3 (up to four
// consecutive token rows of one slot's chunk); the unit streams the slot's pages up to the longest
// context among its rows, each row masking the tokens past its own, in a single split.
template <bool MQ>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(128)
    k3mla_decode_split_kernel(const __grid_constant__ CUtensorMap tmap_page,
                              const __grid_constant__ CUtensorMap tmap_page8,
                              const __grid_constant__ CUtensorMap tmap_q,
                              const __grid_constant__ CUtensorMap tmap_olat,
                              const __grid_constant__ CUtensorMap tmap_part, const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    SmemT<MQ>& sm =
        *reinterpret_cast<SmemT<MQ>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t rank = cluster_ctarank();
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();

    const int unit = blockIdx.x >> 1;
    SplitGeom sg;
    sg.hb = 0;
    int mq_row[4] = {-1, -1, -1, -1}, mq_ntok[4] = {0, 0, 0, 0};
    if constexpr (MQ) {
        griddep_wait();  // the groups and row contexts come from the launch just before
        const int4 gr = p.mq_groups[unit / 3];  // (slot, first token row, rows, -)
        if (gr.z <= 0) return;                  // past the chunk's groups
        sg.b = gr.x;
        sg.s = 0;
        sg.hb = unit % 3;
        int ctx = 0;
        for (int w = 0; w < 4 && w < gr.z; ++w) {
            mq_row[w] = gr.y + w;
            mq_ntok[w] = p.mq_ctx[gr.y + w];
            ctx = max(ctx, mq_ntok[w]);
        }
        if (ctx <= 0) return;  // no row has a token: the launch before zeroed their o_lat
        sg.single = true;
        sg.start = 0;
        sg.ntok = ctx;
        sg.npg = (ctx + PAGE - 1) / PAGE;
        sg.n_lp = sg.npg;
        sg.lp0 = 0;
        sg.oob_row = p.n_pages * p.n_layers * PAGE;
    } else {
        sg.b = unit / p.nsplit;
        sg.s = unit % p.nsplit;
        const int ctx = ctx_effective(p.ctx_len, sg.b, p.max_ctx, p.max_pages, p.dev_err,
                                      rank == 0 && threadIdx.x == 0 && sg.s == 0);
        if (!split_geom(sg, ctx, p)) {  // empty split: both CTAs leave, nothing was shared
            if (sg.s == 0 && rank == 1) {  // an empty context: its o_lat is zero (the workspace is written
                griddep_wait();            // only after the kernel before has completed: it may still read it)
                zero_olat(p.ws_olat, p.B, sg.b);
            }
            return;
        }
    }

    if (threadIdx.x == 0) {
        init_decode_barriers(sm, rank, sg.single, p.wait_ns);
        if constexpr (MQ)
            for (int w = 0; w < 4; ++w) {
                sm.mq_row[w] = mq_row[w];
                sm.mq_ntok[w] = mq_ntok[w];
            }
        fence_mbarrier_init_cluster();
        if (rank == 0) tma_prefetch_desc(&tmap_q);
    }
    if (warp == W_ALLOC) {
        tmem_alloc(&sm.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmap_page);
        tma_prefetch_desc(&tmap_page8);
        if (rank == 1) tma_prefetch_desc(sg.single ? &tmap_olat : &tmap_part);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    // everything above overlaps the previous kernel in the stream (which must not write ctx_len, read
    // at the top to size the split); q_abs, the slab and the block table are read after it completed,
    // but for the early page loads of a layer-call
    if constexpr (!MQ)
        if (p.early) early_loads(sm, tmap_page, tmap_page8, p, sg, rank, warp, lane);
    griddep_wait();
    griddep_launch_dependents();
    decode_roles<MQ>(sm, tmap_page, tmap_page8, tmap_q, tmap_olat, tmap_part, p, sg, tbase, rank, warp, lane);

    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == W_ALLOC) tmem_dealloc(tbase, TMEM_COLS);
}

// ---- diagnostic: one page of each contraction --------------------------------------

__global__ void __launch_bounds__(128, 1)
    k3mla_diag_kernel(const __grid_constant__ CUtensorMap tmap_page, const __grid_constant__ CUtensorMap tmap_page8,
                      const __grid_constant__ CUtensorMap tmap_q, int mode, const uint16_t* a, float* d)
{
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    if (threadIdx.x == 0) {
        mbar_init(&sm.full[0], 1);
        mbar_init(&sm.q_land, 1);
        mbar_init(&sm.o_done, 1);
        sm.abort_flag = 0;
        sm.wait_ns = WAIT_NS;
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
    bool ok = true;
    if (mode == 0) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&sm.q_land, CD::QBYTES);
            for (int c = 0; c < 9; ++c) tma_load_3d(sm.u.c0.ring[3] + c * CD::QCHUNK, &tmap_q, 0, 0, c, &sm.q_land);
            mbar_arrive_expect_tx(&sm.full[0], SLOT0);
            for (int t = 0; t < 3; ++t) tma_load_3d(sm.u.c0.ring[0] + t * THIRD, &tmap_page, 0, 0, 3 * t, &sm.full[0]);
        }
        ok = __all_sync(0xFFFFFFFFu, wait_bar(&sm.q_land, 0, sm, nullptr));
        if (ok) q_smem_to_tmem<false>(tbase, sm.u.c0.ring[3]);
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            ok = wait_bar(&sm.full[0], 0, sm, nullptr);
            tc_fence_after();
            if (ok) {
                issue_score_page(tbase, S_COL, smem_u32(sm.u.c0.ring[0]));
                umma_commit(&sm.o_done);
            }
        }
        __syncthreads();
        ok = __all_sync(0xFFFFFFFFu, wait_bar(&sm.o_done, 0, sm, nullptr));
        tc_fence_after();
        if (ok)
            for (int piece = 0; piece < 2; ++piece) {  // row = head, through the lane map
                uint32_t r[32];
                tmem_ld32(t_lane + S_COL + 32 * piece, r);
                tmem_wait_ld();
                if (lane < HPW)
                    for (int c = 0; c < 32; ++c)
                        d[(size_t)(HPW * warp + lane) * 64 + 32 * piece + c] = __uint_as_float(r[c]);
            }
    } else {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&sm.full[0], 2 * SLOT1);
            tma_load_3d(sm.u.c1.ring[0], &tmap_page8, 0, 0, 0, &sm.full[0]);
            tma_load_3d(sm.u.c1.ring[1], &tmap_page8, 0, HALF, 0, &sm.full[0]);
        }
        const int h = (int)threadIdx.x;
        if (h < H)  // P^T row h from a[h][0..63]
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(sm.u.c1.recv[0] + pt_chunk_off(h, j)) =
                    *reinterpret_cast<const uint4*>(a + (size_t)h * 64 + 8 * j);
        fence_proxy_async_cta();
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            ok = wait_bar(&sm.full[0], 0, sm, nullptr);
            tc_fence_after();
            if (ok) {
                issue_pv_page(tbase, smem_u32(sm.u.c1.ring[0]), smem_u32(sm.u.c1.ring[1]), smem_u32(sm.u.c1.recv[0]),
                              false);
                umma_commit(&sm.o_done);
            }
        }
        __syncthreads();
        ok = __all_sync(0xFFFFFFFFu, wait_bar(&sm.o_done, 0, sm, nullptr));
        tc_fence_after();
        if (ok)  // TMEM lane = head (warps 0..2), column = dim; d is [512 dims][96 heads]
            for (int cb = 0; cb < LORA / 32; ++cb) {
                uint32_t r[32];
                tmem_ld32(t_lane + 32u * cb, r);
                tmem_wait_ld();
                if (warp < 3)
                    for (int c = 0; c < 32; ++c) d[(size_t)(32 * cb + c) * H + 32 * warp + lane] = __uint_as_float(r[c]);
            }
    }
    if (!ok) drain_inflight();
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

// ---- multi-query decode of a prefill chunk: its groups of token rows -------------------

// Upper bound of the groups of a chunk of R token rows over B slots: sum over slots of ceil(n_b / 4).
static inline int mq_max_groups(int B, int R) { return (R + 3 * B) / 4 + 1; }

// One CTA.  Token rows row_start[b] .. row_start[b+1]-1 (within [0, R)) belong to slot b, row j of
// them at position pos0[b] + j: its context is pos0[b] + j + 1 tokens (clamped to cap, flagged when
// it is larger).  Groups are up to four consecutive rows of one slot, slot by slot; the entries past
// the last group are empty.  A row without tokens gets zero o_lat here (no unit writes it).
__global__ void __launch_bounds__(1024) k3mla_mq_prep_kernel(const int32_t* __restrict__ pos0,
                                                             const int32_t* __restrict__ row_start, int B, int R,
                                                             int cap, int4* __restrict__ groups, int g_max,
                                                             int32_t* __restrict__ rctx, uint16_t* __restrict__ olat,
                                                             int32_t* dev_err)
{
    griddep_wait();
    __shared__ int off[1024];
    __shared__ int total;
    const int tid = (int)threadIdx.x;
    if (tid == 0) total = 0;
    __syncthreads();
    for (int b0 = 0; b0 < B; b0 += 1024) {
        const int b = b0 + tid;
        int lo = 0, n = 0;
        if (b < B) {
            lo = max(0, row_start[b]);
            n = max(0, min(R, row_start[b + 1]) - lo);
        }
        off[tid] = (n + 3) / 4;
        __syncthreads();
        if (tid == 0) {  // exclusive prefix of the group counts, after those of the slots before
            int acc = total;
            for (int i = 0; i < 1024 && b0 + i < B; ++i) {
                const int c = off[i];
                off[i] = acc;
                acc += c;
            }
            total = acc;
        }
        __syncthreads();
        for (int j = 0; 4 * j < n; ++j)
            if (off[tid] + j < g_max) groups[off[tid] + j] = make_int4(b, lo + 4 * j, min(4, n - 4 * j), 0);
        __syncthreads();
    }
    for (int g = total + tid; g < g_max; g += (int)blockDim.x) groups[g] = make_int4(0, 0, 0, 0);
    for (int r = tid; r < R; r += (int)blockDim.x) {
        int lo = 0, hi = B;  // the last slot b with row_start[b] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (row_start[mid] <= r) lo = mid;
            else hi = mid;
        }
        int c = 0;
        if (B > 0 && r >= row_start[lo] && r < row_start[lo + 1]) {
            c = pos0[lo] + (r - row_start[lo]) + 1;
            if (c > cap) {
                if (dev_err) atomicOr(dev_err, (int)K3MLA_DEV_CTX);
                c = cap;
            }
            c = max(c, 0);
        }
        rctx[r] = c;
        if (c == 0)  // o_lat [96][R][512]: this row's 96 rows of 1 KB
            for (int hh = 0; hh < H; ++hh) {
                uint4* dst = reinterpret_cast<uint4*>(olat + ((size_t)hh * R + r) * LORA);
                for (int k = 0; k < LORA / 8; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
            }
    }
    griddep_launch_dependents();
}

template <bool MQ> static size_t smem_bytes() { return sizeof(SmemT<MQ>) + 1024; }


static int make_maps(const void* slab, uint64_t rows, const void* q, uint64_t q_rows, CUtensorMap* page,
                     CUtensorMap* page8, CUtensorMap* qmap)
{
    int rc = make_tmap_slab_3d(page, slab, rows, ROW, 9, PAGE, 3);  // a third of a page
    if (rc) return rc;
    rc = make_tmap_slab_3d(page8, slab, rows, ROW, 9, HALF, 8);
    if (rc) return rc;
    return make_tmap_slab_3d(qmap, q, q_rows, ROW, 9, H, 1);  // one 64-column chunk per box
}

static void set_smem_attr(const void* fn, size_t bytes, bool* done)
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !done[dev]) {
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (dev >= 0 && dev < 64) done[dev] = true;
    }
}

}  // namespace k3

using namespace k3;

extern "C" size_t k3mla_decode_workspace_bytes(int B, int max_ctx, int split_tokens)
{
    if (B <= 0 || max_ctx <= 0 || split_tokens < 0) return 0;
    return ws_layout(B, launch_nsplit(max_ctx, split_tokens)).total;
}

extern "C" int k3mla_slot_split_tokens(int ctx, int split_tokens)
{
    if (split_tokens < 0) {
        set_error("k3mla_slot_split_tokens: split_tokens < 0");
        return K3MLA_E_INVALID;
    }
    return slot_split(ctx < 0 ? 0 : ctx, split_tokens);
}

static int paged_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers, int layer,
                        const int32_t* block_table, int max_pages_per_slot, const int32_t* ctx_len,
                        const uint16_t* w_kv_b, uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t,
                        void* workspace, size_t ws_bytes, int B, int max_ctx, int split_tokens, int32_t* dev_err,
                        void* stream, uint64_t wait_ns, int withhold, int early)
{
    if (B < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers || max_pages_per_slot <= 0 ||
        max_ctx <= 0 || split_tokens < 0 || split_tokens % TILE != 0) {
        set_error("k3mla_paged_decode: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if ((long long)n_pages * n_layers * PAGE + PAGE > 0x7FFFFFFFll || (long long)B * H > 0x7FFFFFFFll) {
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
    const int ns = launch_nsplit(max_ctx, split_tokens);
    if ((long long)B * ns * H > 0x7FFFFFFFll) {  // grid and partial-row coordinates
        set_error("k3mla_paged_decode: grid too large");
        return K3MLA_E_INVALID;
    }
    CUtensorMap tm_page, tm_page8, tm_q;
    int rc = make_maps(slab, (uint64_t)n_pages * n_layers * PAGE, q_abs, (uint64_t)B * H, &tm_page, &tm_page8, &tm_q);
    if (rc) return rc;
    static bool attr_done[64] = {};
    const size_t smem = smem_bytes<false>();
    set_smem_attr(reinterpret_cast<const void*>(k3mla_decode_split_kernel<false>), smem, attr_done);

    const WsLayout wl = ws_layout(B, ns);
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    DecodeParams dp;
    dp.table = block_table;
    dp.ctx_len = ctx_len;
    // every slot with at most one split lands final bf16 o_lat ([96][B][512]) in the split kernel; the
    // f32 partials exist only when some slot of the launch can have several splits
    dp.ws_olat = reinterpret_cast<uint16_t*>(ws + wl.olat);
    dp.ws_o = ns > 1 ? reinterpret_cast<float*>(ws + wl.o) : nullptr;
    dp.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
    dp.dev_err = dev_err;
    dp.max_pages = max_pages_per_slot;
    dp.n_pages = n_pages;
    dp.n_layers = n_layers;
    dp.layer = layer;
    dp.B = B;
    dp.max_ctx = max_ctx;
    dp.split_tokens = split_tokens;
    dp.nsplit = ns;
    dp.scale2 = ((uint32_t)scale_bf16 << 16) | (uint32_t)scale_bf16;
    dp.wait_ns = wait_ns;
    dp.withhold = withhold;
    dp.early = early;
    dp.mq_groups = nullptr;
    dp.mq_ctx = nullptr;
    // the PV CTAs' stores: o_lat [96][B][512] bf16 as (512 dims, B slots, 96 heads), and the f32 partials
    // [B][ns][96][512] as (512 dims, B ns 96 rows)
    CUtensorMap tm_olat, tm_part;
    {
        const uint64_t dims[3] = {LORA, (uint64_t)B, H};
        const uint64_t strides[2] = {LORA * 2, (uint64_t)B * LORA * 2};
        const uint32_t box[3] = {64, 1, H};
        rc = make_tmap_store(&tm_olat, false, 3, dp.ws_olat, dims, strides, box, true);
        if (rc) return rc;
    }
    if (ns > 1) {
        const uint64_t dims[2] = {LORA, (uint64_t)B * ns * H};
        const uint64_t strides[1] = {LORA * 4};
        const uint32_t box[2] = {32, H};
        rc = make_tmap_store(&tm_part, true, 2, dp.ws_o, dims, strides, box, true);
        if (rc) return rc;
    } else {
        tm_part = tm_olat;  // not used: no slot of this launch has several splits
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    rc = launch_pdl(k3mla_decode_split_kernel<false>, dim3(2 * B * ns), dim3(THREADS), smem, st, "k3mla_decode_split_kernel",
                    tm_page, tm_page8, tm_q, tm_olat, tm_part, dp);
    if (rc) return rc;

    MergeParams mp;
    mp.ws_o = dp.ws_o;
    mp.ws_ml = dp.ws_ml;
    mp.ws_olat = dp.ws_olat;
    mp.ctx_len = ctx_len;
    mp.w_kv_b = w_kv_b;
    mp.out = out;
    mp.argmax = argmax_t;
    mp.dev_err = dev_err;
    mp.B = B;
    mp.max_ctx = max_ctx;
    mp.max_pages = max_pages_per_slot;
    mp.split_tokens = split_tokens;
    mp.nsplit = ns;
    mp.tile = ns == 1 ? 64 : 16;  // every o_lat landed: TMA-loaded in 64-slot tiles; else merged, 16 a CTA
    return launch_merge_expand(mp, st);
}

extern "C" int k3mla_paged_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers,
                                  int layer, const int32_t* block_table, int max_pages_per_slot,
                                  const int32_t* ctx_len, const uint16_t* w_kv_b, uint16_t scale_bf16,
                                  uint16_t* out, int32_t* argmax_t, void* workspace, size_t ws_bytes, int B,
                                  int max_ctx, int split_tokens, int32_t* dev_err, void* stream)
{
    return paged_decode(q_abs, slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, ctx_len, w_kv_b,
                        scale_bf16, out, argmax_t, workspace, ws_bytes, B, max_ctx, split_tokens, dev_err, stream,
                        WAIT_NS, 0, 0);
}

extern "C" int k3mla_diag_decode_timeout(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers,
                                         int layer, const int32_t* block_table, int max_pages_per_slot,
                                         const int32_t* ctx_len, const uint16_t* w_kv_b, uint16_t scale_bf16,
                                         uint16_t* out, int32_t* argmax_t, void* workspace, size_t ws_bytes, int B,
                                         int max_ctx, int split_tokens, int withhold_page, uint32_t wait_us,
                                         int32_t* dev_err, void* stream)
{
    if (withhold_page < 1 || wait_us < 100 || wait_us > 100000) {
        set_error("k3mla_diag_decode_timeout: withhold_page >= 1 and 100 <= wait_us <= 100000");
        return K3MLA_E_INVALID;
    }
    return paged_decode(q_abs, slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, ctx_len, w_kv_b,
                        scale_bf16, out, argmax_t, workspace, ws_bytes, B, max_ctx, split_tokens, dev_err, stream,
                        (uint64_t)wait_us * 1000ull, withhold_page + 1, 0);
}

// ---- multi-query decode of a prefill chunk ---------------------------------------------

extern "C" size_t k3mla_chunk_decode_workspace_bytes(int B, int R, int max_ctx)
{
    if (B <= 0 || R <= 0 || max_ctx <= 0) return 0;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return ws_layout(R, 1).total + up((size_t)mq_max_groups(B, R) * sizeof(int4)) + up((size_t)R * 4);
}

extern "C" int k3mla_chunk_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers, int layer,
                                  const int32_t* block_table, int max_pages_per_slot, const int32_t* pos0,
                                  const int32_t* row_start, int B, int R, const uint16_t* w_kv_b,
                                  uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t, void* workspace,
                                  size_t ws_bytes, int max_ctx, int32_t* dev_err, void* stream)
{
    if (B <= 0 || R < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers ||
        max_pages_per_slot <= 0 || max_ctx <= 0) {
        set_error("k3mla_chunk_decode: invalid sizes");
        return K3MLA_E_INVALID;
    }
    if (R == 0) return K3MLA_OK;
    if ((long long)n_pages * n_layers * PAGE + PAGE > 0x7FFFFFFFll || (long long)R * H > 0x7FFFFFFFll ||
        6ll * mq_max_groups(B, R) > 0x7FFFFFFFll) {
        set_error("k3mla_chunk_decode: sizes exceed the 2^31 TMA row or grid range");
        return K3MLA_E_INVALID;
    }
    if (!q_abs || !slab || !block_table || !pos0 || !row_start || !w_kv_b || !out || !workspace ||
        !aligned(q_abs, 16) || !aligned(slab, 16) || !aligned(w_kv_b, 16) || !aligned(out, 4) ||
        !aligned(workspace, 256)) {
        set_error("k3mla_chunk_decode: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    const size_t need = k3mla_chunk_decode_workspace_bytes(B, R, max_ctx);
    if (ws_bytes < need) {
        set_error("k3mla_chunk_decode: workspace %zu < %zu bytes", ws_bytes, need);
        return K3MLA_E_WORKSPACE;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    const int G = mq_max_groups(B, R);
    const int cap = (int)std::min<long long>(max_ctx, (long long)max_pages_per_slot * PAGE);
    const int whole = (cap + TILE - 1) / TILE * TILE;  // one split holds any row's context
    const WsLayout wl = ws_layout(R, 1);
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    int4* groups = reinterpret_cast<int4*>(ws + wl.total);
    int32_t* rctx = reinterpret_cast<int32_t*>(ws + wl.total + ((G * sizeof(int4) + 255) & ~size_t(255)));
    uint16_t* olat = reinterpret_cast<uint16_t*>(ws + wl.olat);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = launch_pdl(k3mla_mq_prep_kernel, dim3(1), dim3(1024), 0, st, "k3mla_mq_prep_kernel", pos0, row_start, B,
                        R, cap, groups, G, rctx, olat, dev_err);
    if (rc) return rc;

    CUtensorMap tm_page, tm_page8, tm_q, tm_olat, tm_orow;
    rc = make_tmap_slab_3d(&tm_page, slab, (uint64_t)n_pages * n_layers * PAGE, ROW, 9, PAGE, 3);
    if (rc) return rc;
    rc = make_tmap_slab_3d(&tm_page8, slab, (uint64_t)n_pages * n_layers * PAGE, ROW, 9, HALF, 8);
    if (rc) return rc;
    {   // q_abs [R][96][576] as (64 elements, 96 heads, R rows, 9 chunks): one box = a chunk of 32 heads
        // of four consecutive token rows
        const uint64_t dims[4] = {64, H, (uint64_t)R, 9};
        const uint64_t strides[3] = {ROW * 2, (uint64_t)H * ROW * 2, 128};
        const uint32_t box[4] = {64, 32, 4, 1};
        rc = make_tmap_store(&tm_q, false, 4, q_abs, dims, strides, box, true);
        if (rc) return rc;
    }
    {   // o_lat [96][R][512] bf16 as (512 dims, 96 heads, R rows): boxes of 32 heads x 4 rows, or x 1 row
        const uint64_t dims[3] = {LORA, H, (uint64_t)R};
        const uint64_t strides[2] = {(uint64_t)R * LORA * 2, LORA * 2};
        const uint32_t box4[3] = {64, 32, 4}, box1[3] = {64, 32, 1};
        rc = make_tmap_store(&tm_olat, false, 3, olat, dims, strides, box4, true);
        if (!rc) rc = make_tmap_store(&tm_orow, false, 3, olat, dims, strides, box1, true);
        if (rc) return rc;
    }
    DecodeParams dp;
    std::memset(&dp, 0, sizeof(dp));
    dp.table = block_table;
    dp.ctx_len = rctx;
    dp.ws_olat = olat;
    dp.ws_o = nullptr;
    dp.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
    dp.dev_err = dev_err;
    dp.max_pages = max_pages_per_slot;
    dp.n_pages = n_pages;
    dp.n_layers = n_layers;
    dp.layer = layer;
    dp.B = R;
    dp.max_ctx = cap;
    dp.split_tokens = whole;
    dp.nsplit = 1;
    dp.scale2 = ((uint32_t)scale_bf16 << 16) | (uint32_t)scale_bf16;
    dp.wait_ns = WAIT_NS;
    dp.mq_groups = groups;
    dp.mq_ctx = rctx;
    static bool attr_done[64] = {};
    const size_t smem = smem_bytes<true>();
    set_smem_attr(reinterpret_cast<const void*>(k3mla_decode_split_kernel<true>), smem, attr_done);
    rc = launch_pdl(k3mla_decode_split_kernel<true>, dim3(2 * 3 * G), dim3(THREADS), smem, st,
                    "k3mla_decode_split_kernel<MQ>", tm_page, tm_page8, tm_q, tm_olat, tm_orow, dp);
    if (rc) return rc;

    MergeParams mp;
    mp.ws_o = nullptr;
    mp.ws_ml = dp.ws_ml;
    mp.ws_olat = olat;
    mp.ctx_len = rctx;
    mp.w_kv_b = w_kv_b;
    mp.out = out;
    mp.argmax = argmax_t;
    mp.dev_err = dev_err;
    mp.B = R;
    mp.max_ctx = cap;
    mp.max_pages = max_pages_per_slot;
    mp.split_tokens = whole;
    mp.nsplit = 1;
    mp.tile = 64;
    return launch_merge_expand(mp, st);
}

// ---- one decode step of one layer ------------------------------------------------------

static size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

extern "C" size_t k3mla_decode_layer_workspace_bytes(int B, int max_ctx)
{
    if (B <= 0 || max_ctx <= 0) return 0;
    return up256((size_t)B * H * ROW * 2) + ws_layout(B, launch_nsplit(max_ctx, 0)).total;
}

extern "C" int k3mla_decode_layer(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* slab, int n_pages,
                                  int n_layers, int layer, const int32_t* block_table, int max_pages_per_slot,
                                  const int32_t* ctx_len, const uint16_t* c_kv, int64_t c_stride,
                                  const uint16_t* k_rope, int64_t r_stride, uint16_t scale_bf16, uint16_t* out,
                                  int32_t* argmax_t, void* workspace, size_t ws_bytes, int B, int max_ctx,
                                  int32_t* dev_err, void* stream)
{
    if (B < 0 || n_pages <= 0 || n_layers <= 0 || layer < 0 || layer >= n_layers || max_pages_per_slot <= 0 ||
        max_ctx <= 0 || c_stride < LORA || r_stride < ROPE || (c_stride & 1) || (r_stride & 1)) {
        set_error("k3mla_decode_layer: invalid sizes or strides");
        return K3MLA_E_INVALID;
    }
    if (B == 0) return K3MLA_OK;
    if (!q || !w_kv_b || !slab || !block_table || !ctx_len || !c_kv || !k_rope || !out || !workspace ||
        !aligned(q, 16) || !aligned(w_kv_b, 16) || !aligned(slab, 16) || !aligned(out, 4) || !aligned(c_kv, 4) ||
        !aligned(k_rope, 4) || !aligned(workspace, 256)) {
        set_error("k3mla_decode_layer: null or misaligned pointer");
        return K3MLA_E_INVALID;
    }
    const size_t need = k3mla_decode_layer_workspace_bytes(B, max_ctx);
    if (ws_bytes < need) {
        set_error("k3mla_decode_layer: workspace %zu < %zu bytes", ws_bytes, need);
        return K3MLA_E_WORKSPACE;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    uint16_t* q_abs = reinterpret_cast<uint16_t*>(ws);
    uint8_t* dws = ws + up256((size_t)B * H * ROW * 2);
    const size_t dws_bytes = ws_bytes - (size_t)(dws - ws);
    const int rc = launch_absorb_append_at_ctx(q, w_kv_b, q_abs, slab, n_pages, n_layers, layer, block_table,
                                               max_pages_per_slot, ctx_len, c_kv, c_stride, k_rope, r_stride, B,
                                               dev_err, reinterpret_cast<cudaStream_t>(stream));
    if (rc) return rc;
    // the split kernel loads pages before the absorption-append launch has completed (early_loads): all
    // but the page each slot's row goes into
    return paged_decode(q_abs, slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, ctx_len, w_kv_b,
                        scale_bf16, out, argmax_t, dws, dws_bytes, B, max_ctx, K3MLA_SPLIT_AUTO, dev_err, stream,
                        WAIT_NS, 0, 1);
}

// ---- decode with built-in scratch ----------------------------------------------------
// For callers that cannot allocate device memory when they decode (a server that reserves
// all device memory for its own pool at start-up, a plugin that is handed only input and
// output pointers): the split results live in this fixed array instead of a caller's
// workspace.  Every device that loads the library holds it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[K3MLA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current CUDA context, looked up with that context's
// device current (in host code the array's name is only a host-side handle).  The address is cached
// per device together with the context it belongs to: a new context of the device (after
// cudaDeviceReset, say) loads the module again, possibly elsewhere, so the lookup is repeated.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
static CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

static int noalloc_scratch(void** out)
{
    static std::mutex mu;
    static void* addr[64] = {};
    static CUcontext owner[64] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        set_error("k3mla_paged_decode_noalloc: no usable current device (%s)", cudaGetErrorString(e));
        return K3MLA_E_CUDA;
    }
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) {
        set_error("k3mla_paged_decode_noalloc: cuCtxGetCurrent unavailable");
        return K3MLA_E_CUDA;
    }
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;  // none yet: the lookup below makes the primary one current
    std::lock_guard<std::mutex> lock(mu);
    if (!ctx || !addr[dev] || owner[dev] != ctx) {
        void* a = nullptr;
        e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
        if (e != cudaSuccess || !a) {
            set_error("k3mla_paged_decode_noalloc: cudaGetSymbolAddress failed on device %d: %s", dev,
                      cudaGetErrorString(e));
            return K3MLA_E_CUDA;
        }
        if (get(&ctx) != CUDA_SUCCESS || !ctx) {
            set_error("k3mla_paged_decode_noalloc: no current CUDA context on device %d", dev);
            return K3MLA_E_CUDA;
        }
        addr[dev] = a;
        owner[dev] = ctx;
    }
    *out = addr[dev];
    return K3MLA_OK;
}

extern "C" int k3mla_paged_decode_noalloc(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers,
                                          int layer, const int32_t* block_table, int max_pages_per_slot,
                                          const int32_t* ctx_len, const uint16_t* w_kv_b, uint16_t scale_bf16,
                                          uint16_t* out, int32_t* argmax_t, int B, int max_ctx, int split_tokens,
                                          int32_t* dev_err, void* stream)
{
    if (B > 0 && max_ctx > 0 && split_tokens >= 0) {
        const size_t need = k3mla_decode_workspace_bytes(B, max_ctx, split_tokens);
        if (need > (size_t)K3MLA_NOALLOC_SCRATCH_BYTES) {
            set_error("k3mla_paged_decode_noalloc: B=%d, max_ctx=%d, split_tokens=%d need %zu bytes of scratch; "
                      "the built-in scratch holds %zu",
                      B, max_ctx, split_tokens, need, (size_t)K3MLA_NOALLOC_SCRATCH_BYTES);
            return K3MLA_E_WORKSPACE;
        }
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    void* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return k3mla_paged_decode(q_abs, slab, n_pages, n_layers, layer, block_table, max_pages_per_slot, ctx_len,
                              w_kv_b, scale_bf16, out, argmax_t, scratch, (size_t)K3MLA_NOALLOC_SCRATCH_BYTES, B,
                              max_ctx, split_tokens, dev_err, stream);
}

extern "C" int k3mla_diag_umma(int mode, const uint16_t* a, const uint16_t* b, float* d, void* stream)
{
    if ((mode != 0 && mode != 1) || !a || !b || !d || !aligned(a, 16) || !aligned(b, 16)) {
        set_error("k3mla_diag_umma: invalid arguments");
        return K3MLA_E_INVALID;
    }
    if (!device_ok()) return K3MLA_E_DEVICE;
    CUtensorMap tm_page, tm_page8, tm_q;
    int rc = make_maps(b, PAGE, a, H, &tm_page, &tm_page8, &tm_q);
    if (rc) return rc;
    static bool attr_done[64] = {};
    const size_t smem = smem_bytes<false>();
    set_smem_attr(reinterpret_cast<const void*>(k3mla_diag_kernel), smem, attr_done);
    k3mla_diag_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(tm_page, tm_page8, tm_q, mode, a, d);
    return check_launch("k3mla_diag_kernel");
}
