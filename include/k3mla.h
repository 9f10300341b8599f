/*
 * k3mla.h -- C ABI of libk3mla.so: paged absorbed multi-head latent attention
 * (MLA) decode for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one pegainfer PR #869, "K3: paged latent MLA KV +
 * absorbed decode", describes:
 *   - M1 commit: a page-first latent slab [page][mla_layer][64 tokens][576]
 *     bf16 (512-wide kv latent c_t, then the 64-wide shared rope key), a per-slot
 *     int32 block table in which -1 reads as an all-zero latent, a free-list
 *     page allocator (claim on a 64-token boundary, release-all on slot reset),
 *     and the new token's row written into the mapped page with a size_t
 *     element index;
 *   - M2 commit: one absorbed kernel per MLA layer,
 *       score(t) = (W_UK[h]^T q_nope)^T c_t + q_rope^T k_rope_t,
 *       o[h]     = W_UV[h] (sum_t softmax(scale * score)_t c_t),
 *     with W_UK and W_UV read in place from w_kv_b (no expansion GEMM, no
 *     per-head K/V), and a runtime-length block-table walk.
 *
 * Geometry is fixed: 96 heads, q_nope 128, q_rope 64, v_head 128, kv_lora 512,
 * page 64 tokens, cache row 576 bf16.  w_kv_b is one layer's [96*256][512]
 * bf16 matrix; rows h*256 .. h*256+127 are W_UK[h] ([d][j]) and rows
 * h*256+128 .. h*256+255 are W_UV[h] ([v][j]).
 *
 * Conventions for every call below:
 *   - bf16 values travel as uint16_t bit patterns; every array is dense,
 *     row-major, in the layout its comment gives.
 *   - "device" pointers are CUDA device memory owned by the caller; the library
 *     never allocates, frees or synchronises device memory, so every device
 *     call other than k3mla_paged_decode_noalloc can be captured into a CUDA
 *     graph (nothing is stated here for that one).  `stream` is a cudaStream_t
 *     (NULL = the legacy default stream).
 *   - Return value: K3MLA_OK (0) or a negative K3MLA_E_* code.  Argument errors
 *     are detected on the host before anything is launched.  A launch failure
 *     returns K3MLA_E_CUDA (the CUDA error text is in k3mla_last_error()).
 *   - Problems only the device can see (a table id outside [-1, n_pages), an
 *     unmapped append position, a context longer than the table or max_ctx) never
 *     fault or trap: the kernel ORs a K3MLA_DEV_* bit into *dev_err (when the
 *     pointer is non-NULL), treats the entry as an all-zero latent or skips the
 *     write, and carries on.  Bounded device waits that run out set
 *     K3MLA_DEV_TIMEOUT and return.
 */
#ifndef K3MLA_H_
#define K3MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3MLA_HEADS 96
#define K3MLA_QK_NOPE 128
#define K3MLA_QK_ROPE 64
#define K3MLA_V_HEAD 128
#define K3MLA_KV_LORA 512
#define K3MLA_PAGE 64
#define K3MLA_ROW 576
#define K3MLA_TILE 128 /* tokens per decode tile; split_tokens must be a multiple */
#define K3MLA_SPLIT_AUTO 0     /* split_tokens: the default per-slot rule (see k3mla_paged_decode) */
#define K3MLA_SPLIT_MAX 4096   /* longest split of the default rule, in tokens */

#define K3MLA_OK 0
#define K3MLA_E_INVALID (-1)   /* bad pointer, size or alignment */
#define K3MLA_E_NO_PAGES (-2)  /* pool exhausted */
#define K3MLA_E_SLOT (-3)      /* slot index out of range */
#define K3MLA_E_CTX (-4)       /* context beyond the pool's max_ctx */
#define K3MLA_E_CUDA (-5)      /* a CUDA call failed */
#define K3MLA_E_WORKSPACE (-6) /* workspace too small */
#define K3MLA_E_DEVICE (-7)    /* the current device is not sm_103 */

#define K3MLA_DEV_BAD_PAGE 1u   /* table id outside [-1, n_pages): read as zero */
#define K3MLA_DEV_UNMAPPED 2u   /* append position unmapped or past the table: skipped */
#define K3MLA_DEV_CTX 4u        /* ctx_len > max_ctx or > table capacity: clamped */
#define K3MLA_DEV_TIMEOUT 8u    /* a bounded device wait ran out; outputs invalid */

/* Text of the last host-side error in this thread (never NULL). */
const char* k3mla_last_error(void);

/* ---- q absorption (PR #869, M2 commit: "q absorption lands bf16") ----------
 * q_abs[b][h][0:512]   = bf16( W_UK[h]^T q[b][h][0:128] )  (f32 accumulation)
 * q_abs[b][h][512:576] = q[b][h][128:192]                   (q_rope, copied)
 * q      device [B][96][192] bf16 (q_nope | q_rope)
 * w_kv_b device [24576][512] bf16, one layer
 * q_abs  device [B][96][576] bf16, written
 * B >= 0 (B == 0 launches nothing).  Pointers 16-byte aligned.
 * The kernel may start while the kernel before it in `stream` is still running
 * (programmatic dependent launch); it waits for that kernel before it reads q or
 * writes q_abs, but it starts loading w_kv_b at once, so w_kv_b must not be
 * written by the kernel immediately before this call in the stream. */
int k3mla_absorb_q(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, int B,
                   void* stream);

/* ---- append: the new token's latent row into its mapped page ---------------
 * (PR #869, M1 commit: "two indexed writes through the per-layer row shift";
 *  the element index is size_t because the slab passes 2^31 elements.)
 * For every b with pos[b] >= 0:
 *   page = block_table[b][pos[b] / 64]
 *   row  = ((size_t)page * n_layers + layer) * 64 + pos[b] % 64
 *   slab[row][0:512] = c_kv[b][0:512];  slab[row][512:576] = k_rope[b][0:64]
 * slab        device [n_pages][n_layers][64][576] bf16 (written in place)
 * block_table device [B][max_pages_per_slot] int32
 * pos         device [B] int32 write position (< 0: no write for that slot)
 * c_kv        device bf16, row b at c_kv + b * c_stride (elements)
 * k_rope      device bf16, row b at k_rope + b * r_stride (elements)
 * dev_err     device int32 or NULL: K3MLA_DEV_UNMAPPED for a -1 / out-of-range
 *             page or a position past the table (that row is skipped).
 * All bf16 pointers and strides 4-byte aligned (strides even). */
int k3mla_append_latent(uint16_t* slab, int n_pages, int n_layers, int layer,
                        const int32_t* block_table, int max_pages_per_slot,
                        const int32_t* pos, const uint16_t* c_kv, int64_t c_stride,
                        const uint16_t* k_rope, int64_t r_stride, int B,
                        int32_t* dev_err, void* stream);

/* ---- q absorption and append in one launch ------------------------------------
 * The two calls above, k3mla_absorb_q(q, w_kv_b, q_abs, B) and
 * k3mla_append_latent(slab, ..., B, dev_err), as one kernel launch: every
 * argument means what it means there, and so do the results, the alignment
 * rules and the error codes.  The page's decode step runs the append and the
 * absorption of a layer back to back and neither reads what the other writes;
 * carrying both in one grid takes one launch (and its latency) off the chain
 * that ends in the decode.  The append waits for the kernel before it in
 * `stream` (like the absorption's q); w_kv_b is read at once, as in
 * k3mla_absorb_q.  (The page has no single call for the pair: this one is a
 * launch-level fusion of its two steps.) */
int k3mla_absorb_q_append(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs,
                          uint16_t* slab, int n_pages, int n_layers, int layer,
                          const int32_t* block_table, int max_pages_per_slot,
                          const int32_t* pos, const uint16_t* c_kv, int64_t c_stride,
                          const uint16_t* k_rope, int64_t r_stride, int B,
                          int32_t* dev_err, void* stream);

/* ---- exact-chain decode (PR #869, M2 commit: the certified rounding chain) ----
 * The same result as k3mla_absorb_q + k3mla_paged_decode, computed landing for
 * landing as the chain states it: q absorption summed over d ascending, score
 * dots over the 576 entries ascending, f32 max and sum of exp over t ascending
 * (exp in double, rounded once to f32), p_t = bf16(e_t / l) with the IEEE
 * quotient, the latent sum over t ascending, the W_UV expansion over j ascending,
 * every landing round-to-nearest-even to bf16.  Each sum is one thread's
 * sequential loop, so the result does not depend on the GPU, the batch or the
 * page placement, and it matches a CPU run of the same chain bit for bit.  The
 * fixed orders rule out the tensor cores: this is a CUDA-core path, tens of
 * times slower than k3mla_paged_decode, meant as a reference mode.
 * q          device [B][96][192] bf16 (q_nope | q_rope), not q_abs
 * max_ctx    1 .. 51,200 (one row's exps are held in shared memory)
 * others     as for k3mla_paged_decode (no split; argmax_t may be NULL)
 * workspace  device, >= k3mla_decode_exact_workspace_bytes(B, max_ctx) bytes,
 *            256-byte aligned: bf16 scores then probabilities [B][96][max_ctx
 *            rounded up to 8], q_abs [B][96][576], o_lat [96][B][512]
 * Five kernels on `stream`, each reading nothing before the kernel ahead of it
 * has completed. */
size_t k3mla_decode_exact_workspace_bytes(int B, int max_ctx);
int k3mla_decode_exact(const uint16_t* q, const uint16_t* slab, int n_pages, int n_layers, int layer,
                       const int32_t* block_table, int max_pages_per_slot, const int32_t* ctx_len,
                       const uint16_t* w_kv_b, uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t,
                       void* workspace, size_t ws_bytes, int B, int max_ctx, int32_t* dev_err,
                       void* stream);

/* ---- chunked prefill: many new tokens per slot (PR #869 description,
 * follow-ups: chunked prefill in place of the token loop) --------------------
 * A chunk of n_b = row_start[b + 1] - row_start[b] new tokens of slot b sits at
 * positions pos0[b] .. pos0[b] + n_b - 1 (their pages already mapped, e.g. by
 * k3mla_pool_ensure(pool, b, pos0[b] + n_b)); the chunk's inputs are rows
 * row_start[b] .. row_start[b + 1] - 1 of the packed per-token arrays.
 *
 * k3mla_append_latent_rows: k3mla_append_latent for every token of every chunk
 * (row r of c_kv / k_rope lands in the mapped row of its position, size_t
 * index).  max_rows >= every n_b (sets the grid; rows past n_b are not read).
 * K3MLA_DEV_UNMAPPED in *dev_err for a row whose page is -1 / out of range or
 * whose position is negative or past the table (that row is skipped).
 *
 * k3mla_chunk_views: for every row r < R of the packed chunk (token j of slot b),
 * view_table[r][:] = block_table[b][:] and view_ctx[r] = pos0[b] + j + 1, so that
 * k3mla_paged_decode over the R views (with q_abs of the R tokens, B = R) gives
 * each token the causal attention of the chunk: token j sees the slot's rows
 * before the chunk and the chunk's rows 0..j.  Rows r >= row_start[B] get an
 * empty view (ctx 0, table -1).
 * block_table [B][max_pages_per_slot], pos0 [B], row_start [B + 1] (non-
 * decreasing), view_table [R][max_pages_per_slot], view_ctx [R]: device int32.
 * The decode reads its ctx_len when it starts, so call k3mla_chunk_views before
 * the absorption (k3mla_absorb_q), not immediately before k3mla_paged_decode. */
int k3mla_append_latent_rows(uint16_t* slab, int n_pages, int n_layers, int layer,
                             const int32_t* block_table, int max_pages_per_slot,
                             const int32_t* pos0, const int32_t* row_start,
                             const uint16_t* c_kv, int64_t c_stride,
                             const uint16_t* k_rope, int64_t r_stride, int B, int max_rows,
                             int32_t* dev_err, void* stream);
int k3mla_chunk_views(const int32_t* block_table, int B, int max_pages_per_slot,
                      const int32_t* pos0, const int32_t* row_start, int R,
                      int32_t* view_table, int32_t* view_ctx, void* stream);

/* k3mla_chunk_decode: the same causal attention of every token of the chunks
 * (row j of slot b over the slot's first pos0[b] + j + 1 tokens) in multi-query
 * form: up to four consecutive rows of one slot share each page load, one row
 * per 32-lane quarter of the contractions, 32 heads of each (all 128 rows of
 * an M = 128 MMA used), so a slot's pages are streamed ceil(n_b / 4) x 3 times
 * instead of n_b times, and no view table is needed.  Each row's context is
 * one split (the whole context: the split kernel's unit streams the pages up
 * to its longest row), and every row's result equals k3mla_paged_decode of
 * that row's view with a split_tokens at least the context, bit for bit.
 * q_abs      device [R][96][576] bf16: k3mla_absorb_q of the R token rows
 * block_table, pos0 [B], row_start [B + 1] (non-decreasing): as for
 *            k3mla_chunk_views; rows outside every slot's range, or whose
 *            context pos0[b] + j + 1 is < 1, get zero output (argmax -1)
 * out        device [R][96][128] bf16; argmax_t [R][96] int32 or NULL
 * max_ctx    >= every row's context (a longer one is clamped and flagged
 *            K3MLA_DEV_CTX, like ctx_len in k3mla_paged_decode)
 * workspace  device, >= k3mla_chunk_decode_workspace_bytes(B, R, max_ctx)
 *            bytes, 256-byte aligned: o_lat [96][R][512], the rows' records,
 *            the groups of rows and the rows' context lengths
 * Three kernels on `stream` (groups, split kernel, merge / expansion), each
 * reading nothing the one before writes until it has completed. */
size_t k3mla_chunk_decode_workspace_bytes(int B, int R, int max_ctx);
int k3mla_chunk_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers, int layer,
                       const int32_t* block_table, int max_pages_per_slot, const int32_t* pos0,
                       const int32_t* row_start, int B, int R, const uint16_t* w_kv_b,
                       uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t, void* workspace,
                       size_t ws_bytes, int max_ctx, int32_t* dev_err, void* stream);

/* ---- paged absorbed decode ---------------------------------------------------
 * For each slot b < B and head h, with n = ctx_len[b] tokens (logical token t
 * lives in page block_table[b][t / 64], row t % 64; a -1 entry is an all-zero
 * row that still takes part in the softmax):
 *   s_t   = bf16( bf16( q_abs[b][h] . row_t ) * scale )       (576-wide dot)
 *   p_t   = softmax_t(s)
 *   o_lat = bf16( sum_t p_t row_t[0:512] )
 *   out[b][h] = bf16( W_UV[h] o_lat )
 * (PR #869, M2 commit.)  Rows at positions >= n are never used, whatever they
 * hold.  n == 0 gives out = 0 and argmax -1.
 *
 * Splits.  The context of each slot is cut into splits; each split is reduced on
 * its own and a slot's splits are merged in a fixed order.  How a slot is cut is
 * a function of its own n and of split_tokens only:
 *   - split_tokens == K3MLA_SPLIT_AUTO (0), the default: ceil(n / K3MLA_SPLIT_MAX)
 *     splits of equal length, rounded up to a multiple of K3MLA_TILE
 *     (k3mla_slot_split_tokens gives the length);
 *   - split_tokens > 0 (a multiple of K3MLA_TILE): a split every split_tokens
 *     tokens.
 * A slot with one split (or none) lands its o_lat directly.  A slot with several
 * is merged by four split groups -- group g sums splits g, g + 4, g + 8, ... in
 * ascending order with a running max -- and the groups are then brought to their
 * common max and added as ((g0 + g1) + (g2 + g3)).  Neither the cut nor the merge
 * depends on B, max_ctx, the other slots, the page ids or the GPU, so for a given
 * split_tokens a slot's result is bitwise independent of the batch it is in, of
 * padding slots and of which physical pages hold it.
 *
 * q_abs       device [B][96][576] bf16 (from k3mla_absorb_q)
 * slab        device [n_pages][n_layers][64][576] bf16; n_pages*n_layers*64 < 2^31
 * block_table device [B][max_pages_per_slot] int32
 * ctx_len     device [B] int32 (clamped to min(max_ctx, 64*max_pages_per_slot),
 *             setting K3MLA_DEV_CTX when it had to be)
 * w_kv_b      device [24576][512] bf16, the layer's weights
 * scale_bf16  the softmax scale as a bf16 bit pattern (bf16(1/sqrt(192)) = 0x3D94)
 * out         device [B][96][128] bf16, written
 * argmax_t    device [B][96] int32 or NULL: per head, the lowest logical t with
 *             the largest bf16 score (-1 for an empty context)
 * workspace   device, >= k3mla_decode_workspace_bytes(B, max_ctx, split_tokens)
 *             bytes, 256-byte aligned; scratch, contents need no initialisation
 * max_ctx     upper bound of ctx_len, sets the grid (1 <= max_ctx)
 * dev_err     device int32 or NULL (K3MLA_DEV_* bits are ORed in)
 * Runs as two kernels on `stream`: the split decode, then the merge + W_UV
 * expansion.  Both may start while the kernel before them is still running
 * (programmatic dependent launch).  Before that kernel has completed, the split
 * kernel reads ctx_len (to cut each slot), so the kernel immediately before
 * this call in `stream` must not write ctx_len; q_abs, the slab, the block table
 * and the workspace are read or written only after the wait.  The merge kernel
 * loads w_kv_b and reads ctx_len early, while the split kernel (which writes
 * neither) still runs. */
size_t k3mla_decode_workspace_bytes(int B, int max_ctx, int split_tokens);
int k3mla_paged_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers,
                       int layer, const int32_t* block_table, int max_pages_per_slot,
                       const int32_t* ctx_len, const uint16_t* w_kv_b, uint16_t scale_bf16,
                       uint16_t* out, int32_t* argmax_t, void* workspace, size_t ws_bytes,
                       int B, int max_ctx, int split_tokens, int32_t* dev_err, void* stream);

/* ---- one decode step of one layer: append + absorption + paged decode -----------
 * (PR #869, M1 and M2 commits: the new token's row written into its mapped page,
 * q absorbed, then the absorbed attention over the slot's pages.)
 * Exactly k3mla_absorb_q_append with each slot's write position ctx_len[b] - 1
 * (no write for ctx_len[b] <= 0), followed by k3mla_paged_decode with
 * split_tokens = K3MLA_SPLIT_AUTO on the q_abs it produced: the same outputs, bit
 * for bit, and the same error behaviour, in three kernel launches on `stream`
 * (absorption with the append, split decode, merge / expansion).  ctx_len counts
 * this step's token.  The call a decode step makes once per MLA layer.
 * q, w_kv_b, slab, block_table, ctx_len, scale_bf16, out, argmax_t, B, max_ctx,
 *             dev_err: as for k3mla_absorb_q / k3mla_paged_decode
 * c_kv, c_stride, k_rope, r_stride: this step's rows, as for k3mla_append_latent
 * workspace   device, >= k3mla_decode_layer_workspace_bytes(B, max_ctx) bytes,
 *             256-byte aligned, scratch (q_abs, then the decode workspace); no
 *             initialisation needed.
 * As for k3mla_paged_decode, the kernel immediately before this call in `stream`
 * must not write ctx_len (the split kernel reads it when it starts); the first
 * kernel of the call reads q, the rows and the tables only after the kernel ahead
 * of it has completed, and w_kv_b at once.  Within the call the split kernel starts
 * loading each slot's pages, all but the one the step's row goes into, before the
 * append has finished: a page that receives a row must not be read by another slot
 * of the same call (the pool's copy on write keeps a slot's last page its own). */
size_t k3mla_decode_layer_workspace_bytes(int B, int max_ctx);
int k3mla_decode_layer(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* slab, int n_pages, int n_layers,
                       int layer, const int32_t* block_table, int max_pages_per_slot, const int32_t* ctx_len,
                       const uint16_t* c_kv, int64_t c_stride, const uint16_t* k_rope, int64_t r_stride,
                       uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t, void* workspace, size_t ws_bytes,
                       int B, int max_ctx, int32_t* dev_err, void* stream);

/* The split length a slot of context ctx gets from k3mla_paged_decode:
 * split_tokens when it is positive, else the default rule's length (at most
 * K3MLA_SPLIT_MAX; K3MLA_TILE for ctx <= 0).  The slot then has
 * ceil(ctx / length) splits.  A host-side helper: it touches no GPU. */
int k3mla_slot_split_tokens(int ctx, int split_tokens);

/* OPT-IN, BATCH-DEPENDENT NUMERICS.  A fixed split length for a whole batch whose
 * contexts the caller knows on the host, chosen for throughput: the shortest
 * multiple of K3MLA_TILE whose splits that hold tokens, sum_b ceil(ctx_b / split),
 * fit one wave of SM pairs of the current device (or max_ctx rounded up to
 * K3MLA_TILE when that already gives every slot one split or no length fits).
 * pegainfer PR #869 (M2 commit) reduces a context in splits merged in a fixed
 * order; on a ragged batch with few slots this length keeps more SM pairs busy
 * than the default rule.  The price: the length depends on every slot's context
 * and on the SM count, so passing it as split_tokens makes a slot's output bits
 * depend on the rest of the batch, on padding rows and on the GPU.  Callers that
 * need batch or padding invariance use K3MLA_SPLIT_AUTO instead.
 * ctx_host[b] for b < B is clamped to [0, max_ctx].  B <= 0 or max_ctx <= 0 gives
 * K3MLA_TILE; a NULL ctx_host with B > 0 gives K3MLA_E_INVALID. */
int k3mla_batch_planned_split_tokens(const int32_t* ctx_host, int B, int max_ctx);

/* ---- host page pool: free-list allocator (PR #869, M1 commit) ---------------
 * n_pages == 0 sizes the pool for full coverage: n_slots * ceil(max_ctx / 64)
 * pages, so every slot can reach max_ctx.  The free list holds page ids
 * 0 .. n_pages-1; shuffle_seed != 0 shuffles it (splitmix64-driven
 * Fisher-Yates) so that slots claim scattered ids.  The pool owns a host block
 * table [n_slots][max_pages] (max_pages = ceil(max_ctx / 64)), -1 = unmapped;
 * the caller copies it to the device.  Nothing here touches a GPU. */
typedef struct k3mla_pool k3mla_pool;
int k3mla_pool_create(int n_pages, int n_slots, int max_ctx, uint64_t shuffle_seed,
                      k3mla_pool** out);
/* Claims pages (one per 64-token boundary crossed) so that tokens
 * [0, new_len) of `slot` are mapped.  All-or-nothing: on K3MLA_E_NO_PAGES no
 * page is claimed.  new_len > max_ctx gives K3MLA_E_CTX. */
int k3mla_pool_ensure(k3mla_pool* pool, int slot, int new_len);
/* k3mla_pool_ensure for slots 0 .. n-1 in order, new_len[b] for slot b (host
 * array), in one call: a decode step's claims for the whole batch.  Stops at
 * the first slot that fails and returns its status (the slots before it keep
 * their pages; the failing slot is all-or-nothing as above); K3MLA_E_INVALID
 * for n < 0 or n > n_slots. */
int k3mla_pool_ensure_all(k3mla_pool* pool, const int32_t* new_len, int n);
/* Returns every page of `slot` to the free list and unmaps its table row. */
int k3mla_pool_release_slot(k3mla_pool* pool, int slot);
const int32_t* k3mla_pool_host_table(const k3mla_pool* pool);
int k3mla_pool_max_pages(const k3mla_pool* pool);
int k3mla_pool_n_pages(const k3mla_pool* pool);
/* Pool capacity and pages in use (PR #869 review: expose total / allocated).
 * A page mapped by several slots counts once. */
int k3mla_pool_stats(const k3mla_pool* pool, int* total, int* used);
void k3mla_pool_destroy(k3mla_pool* pool);

/* ---- page sharing (PR #869 description, follow-ups: block-pool reuse of cached
 * prefixes) -------------------------------------------------------------------
 * Every page carries a reference count: the number of slots that map it (0 =
 * free).  k3mla_pool_ensure claims pages with count 1; k3mla_pool_release_slot
 * decrements the counts of the slot's pages and returns a page to the free list
 * only when its count reaches 0.
 *
 * k3mla_pool_share_prefix maps the first ceil(n_tokens / 64) pages of src_slot
 * into the (empty) dst_slot -- the same physical ids, counts incremented -- so
 * the two slots share that prefix of the cache with no copy.  K3MLA_E_SLOT for
 * a slot out of range, K3MLA_E_CTX for n_tokens > max_ctx, K3MLA_E_INVALID when
 * dst_slot == src_slot, dst_slot maps any page, or src_slot maps fewer pages.
 *
 * Before writing token `pos` of `slot` (whose page must be mapped, else
 * K3MLA_E_CTX), call k3mla_pool_cow: 0 means the slot owns that page alone and
 * may write it in place; 1 means the page was shared, so the slot now maps a
 * fresh page (count 1, the old page's count decremented) and *src_page ->
 * *dst_page names the whole-page copy the caller must run (k3mla_copy_pages)
 * before the write; K3MLA_E_NO_PAGES leaves everything unchanged.
 * k3mla_pool_page_refs returns a page's count (K3MLA_E_INVALID for a bad id). */
int k3mla_pool_share_prefix(k3mla_pool* pool, int dst_slot, int src_slot, int n_tokens);
int k3mla_pool_cow(k3mla_pool* pool, int slot, int pos, int32_t* src_page, int32_t* dst_page);
int k3mla_pool_page_refs(const k3mla_pool* pool, int page);

/* ---- whole-page copy (PR #869, M1 commit: "whole-page copy on prefill
 * adoption") ---------------------------------------------------------------------
 * For i < n: page dst_ids[i] of dst_slab <- page src_ids[i] of src_slab, all
 * n_layers layers (a page of the page-first slab is one contiguous block of
 * n_layers * 64 * 576 bf16).  Adopting a prefilled sequence into a decode slot:
 * claim the slot's pages (k3mla_pool_ensure), then copy the prefill pool's pages
 * into them; un-sharing a page: the pair k3mla_pool_cow names, with
 * src_slab == dst_slab.
 * dst_slab / src_slab  device, [dst_n_pages | src_n_pages][n_layers][64][576]
 *                      bf16, 16-byte aligned (may be the same slab)
 * src_ids / dst_ids    device int32 [n], 0 <= n <= 65535
 * dev_err              device int32 or NULL: K3MLA_DEV_BAD_PAGE for a pair with
 *                      an id outside its slab (that pair is skipped)
 * The dst ids must be distinct and, within one slab, none may also be a src id
 * of the same call (the copies run concurrently).  One kernel on `stream`; it may
 * start while the kernel before it is still running and reads the ids and pages
 * only after that kernel has completed. */
int k3mla_copy_pages(uint16_t* dst_slab, int dst_n_pages, const uint16_t* src_slab, int src_n_pages,
                     int n_layers, const int32_t* src_ids, const int32_t* dst_ids, int n,
                     int32_t* dev_err, void* stream);

/* ---- paged decode with built-in scratch ---------------------------------------
 * The pegainfer PR #869 page has no counterpart to this call.  It is k3mla_paged_decode without the
 * `workspace` / `ws_bytes` pair, for callers that cannot allocate device memory at
 * the point where they decode: a serving process that reserves all device memory
 * for its own pool at start-up and forbids allocation while it serves, or a plugin
 * that its host framework hands only the pointers of its inputs and outputs.  The
 * scratch is a fixed array of K3MLA_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the
 * library; every GPU that loads the library holds it until the process exits.  The
 * call itself allocates and frees nothing.  Arguments, results and error behaviour
 * are those of k3mla_paged_decode (same kernels, same bits), and:
 *   - Limit: k3mla_decode_workspace_bytes(B, max_ctx, split_tokens) must not exceed
 *     K3MLA_NOALLOC_SCRATCH_BYTES: up to 168 slots when every slot has one split
 *     (max_ctx <= K3MLA_SPLIT_MAX under the default rule), fewer when slots can have
 *     several.  A larger request returns K3MLA_E_WORKSPACE before anything is
 *     launched; k3mla_last_error() gives the sizes.
 *   - The first call in a CUDA context of a device looks up the array's device
 *     address (once, with that device current); a later call in a new context of the
 *     same device (after cudaDeviceReset, for instance) looks it up again.  Make the
 *     first call before any stream capture begins.  This header makes no statement
 *     either way about capturing this call in a CUDA graph.
 *   - All calls on a device share the one array.  Calls whose kernels overlap on
 *     the GPU (different streams, or threads with no ordering between their calls)
 *     race on it and corrupt each other's results: order them, e.g. on one stream.
 *   - Nothing in the array needs to start at zero: a call writes every scratch value
 *     it reads, so what the previous call left there does not matter. */
#define K3MLA_NOALLOC_SCRATCH_BYTES (16u << 20)
int k3mla_paged_decode_noalloc(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers,
                               int layer, const int32_t* block_table, int max_pages_per_slot,
                               const int32_t* ctx_len, const uint16_t* w_kv_b, uint16_t scale_bf16,
                               uint16_t* out, int32_t* argmax_t, int B, int max_ctx, int split_tokens,
                               int32_t* dev_err, void* stream);

/* ---- the expanded-cache design, as an A/B baseline (PR #869, M2 commit) --------
 * The design the absorbed decode replaces: every token's latent expanded by kv_b
 * into per-head K (192 = 128 nope + the 64-wide rope key) and V (128) rows, about
 * 1.47 MB per token over 24 MLA layers (61,440 bytes per token and layer) against
 * the latent's 27.6 KB, and ordinary attention over them.  For timing the two
 * designs on the same workload; not part of the absorbed path.
 *
 * k3mla_expand_latent_cache: for every page p < n_pages of the slab, token t and
 * head h, at this layer:
 *   xcache[p][t][h][0:128]   = bf16( W_UK[h] c_t )      (f32 accumulation)
 *   xcache[p][t][h][128:192] = k_rope_t                  (copied)
 *   xcache[p][t][h][192:320] = bf16( W_UV[h] c_t )
 * slab   device [n_pages][n_layers][64][576] bf16, 16-byte aligned
 * w_kv_b device [24576][512] bf16, the layer's weights, 16-byte aligned
 * xcache device, k3mla_expanded_cache_bytes(n_pages) bytes, 16-byte aligned
 * One kernel on `stream`; it reads nothing before the kernel ahead of it completed.
 *
 * k3mla_expanded_decode: for each slot b < B and head h, over its n = ctx_len[b]
 * tokens (token t at page block_table[b][t / 64], row t % 64; -1 is a zero K / V
 * row that takes part in the softmax; ids outside [-1, n_pages) read as zero and
 * set K3MLA_DEV_BAD_PAGE; n is clamped to min(max_ctx, 64 * max_pages_per_slot)
 * with K3MLA_DEV_CTX):
 *   s_t = bf16( bf16( q[b][h] . K_h[t] ) * scale ),  p = softmax(s),
 *   out[b][h] = bf16( sum_t p_t V_h[t] )             (f32 online softmax)
 * q device [B][96][192] bf16 (q_nope | q_rope, not absorbed), 4-byte aligned;
 * out device [B][96][128] bf16, 8-byte aligned; n == 0 gives zeros.  One kernel on
 * `stream`, no workspace.
 * Both return K3MLA_E_INVALID, with nothing launched, for sizes out of range (a
 * layer past the slab, no pages, a grid past 65535 slots) or a null or misaligned
 * pointer; k3mla_expanded_decode with B == 0 does nothing.  The caller owns every
 * buffer. */
size_t k3mla_expanded_cache_bytes(int n_pages);
int k3mla_expand_latent_cache(const uint16_t* slab, int n_pages, int n_layers, int layer, const uint16_t* w_kv_b,
                              uint16_t* xcache, int32_t* dev_err, void* stream);
int k3mla_expanded_decode(const uint16_t* q, const uint16_t* xcache, int n_pages, const int32_t* block_table,
                          int max_pages_per_slot, const int32_t* ctx_len, uint16_t scale_bf16, uint16_t* out, int B,
                          int max_ctx, int32_t* dev_err, void* stream);

/* ---- diagnostic: the abort path of the bounded waits ---------------------------
 * Not part of the decode path.  k3mla_paged_decode with two changes that exist only
 * to exercise what happens when a device wait runs out: in every split, the first
 * third of logical page `withhold_page` (>= 1) of the split is never loaded, so the
 * waits on it cannot complete, and every bounded wait of the split kernel gives up
 * after `wait_us` microseconds (100 .. 100000) instead of 1 s.  The kernels then set
 * K3MLA_DEV_TIMEOUT in *dev_err, let every copy and MMA they issued land, free their
 * tensor memory and return; the outputs are invalid.  Returns as k3mla_paged_decode
 * (K3MLA_E_INVALID for the two arguments out of range). */
int k3mla_diag_decode_timeout(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers, int layer,
                              const int32_t* block_table, int max_pages_per_slot, const int32_t* ctx_len,
                              const uint16_t* w_kv_b, uint16_t scale_bf16, uint16_t* out, int32_t* argmax_t,
                              void* workspace, size_t ws_bytes, int B, int max_ctx, int split_tokens,
                              int withhold_page, uint32_t wait_us, int32_t* dev_err, void* stream);

/* ---- diagnostic: the exact-chain mode's exponential ------------------------------
 * y[i] = the f32 nearest to e^(x[i]) as the exact-chain mode computes it (the double
 * exponential rounded once to f32 -- the chain's definition of e_t -- evaluated first in
 * f32 pairs, the double exponential deciding where the pair is too close to a rounding
 * boundary); fast[i] (optional, may be NULL) = 1 where the f32 pair decided, else 0.
 * x, y, fast: device arrays of n elements, 4-byte aligned.  One kernel on `stream`.
 * Returns K3MLA_E_INVALID for n < 0 or a null / misaligned x or y; n == 0 does nothing. */
int k3mla_diag_exact_exp(const float* x, float* y, int32_t* fast, int n, void* stream);

/* ---- diagnostic --------------------------------------------------------------
 * Runs the decode kernel's two tensor-core contractions on one 64-token page in
 * isolation so that their operand layouts can be checked against a plain matrix
 * product.  Not part of the decode path.  `b` is one page, device [64][576] bf16.
 *   mode 0: S[128][64] f32 = Q[128][576] x T^T, Q from `a` (device [96][576]
 *           bf16, rows >= 96 zero), T the page -> d (device [128][64] f32).
 *   mode 1: O[512][96] f32 = T[:, 0:512]^T x P^T, P from `a` (device [96][64]
 *           bf16) -> d (device [512][96] f32).
 */
int k3mla_diag_umma(int mode, const uint16_t* a, const uint16_t* b, float* d, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* K3MLA_H_ */
