// common.cuh -- geometry constants and host-side helpers shared by the library's
// translation units (error text, launch checks, TMA descriptor creation).
#pragma once
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/k3mla.h"

namespace k3 {

constexpr int H = K3MLA_HEADS;          // 96
constexpr int NOPE = K3MLA_QK_NOPE;     // 128
constexpr int ROPE = K3MLA_QK_ROPE;     // 64
constexpr int QDIM = NOPE + ROPE;       // 192
constexpr int VH = K3MLA_V_HEAD;        // 128
constexpr int LORA = K3MLA_KV_LORA;     // 512
constexpr int ROW = K3MLA_ROW;          // 576
constexpr int PAGE = K3MLA_PAGE;        // 64
constexpr int TILE = K3MLA_TILE;        // 128
constexpr int WROWS_PER_HEAD = NOPE + VH;  // 256
constexpr int SPLIT_MAX = K3MLA_SPLIT_MAX;  // 4096: longest split of the default rule

// Split length of a slot whose (clamped) context is n tokens: split_tokens when positive, else the
// default rule -- ceil(n / SPLIT_MAX) splits of equal length rounded up to the 128-token tile.  It
// depends on n and constants only, never on the batch, the GPU or the page ids, so a slot is cut
// the same way whatever else is in the launch.
__host__ __device__ inline int slot_split(int n, int split_tokens)
{
    if (split_tokens > 0) return split_tokens;
    const int ns = n <= SPLIT_MAX ? 1 : (n + SPLIT_MAX - 1) / SPLIT_MAX;
    const int per = (n + ns - 1) / ns;
    const int t = (per + TILE - 1) / TILE * TILE;
    return t < TILE ? TILE : t;
}

// Splits that hold tokens for a slot of n tokens cut every `split` tokens (0 for an empty context).
__host__ __device__ inline int slot_nsplit(int n, int split) { return n <= 0 ? 0 : (n + split - 1) / split; }

// Upper bound of slot_nsplit over contexts up to max_ctx: the split count of the launch's grid.
__host__ __device__ inline int launch_nsplit(int max_ctx, int split_tokens)
{
    const int s = split_tokens > 0 ? split_tokens : SPLIT_MAX;
    return (max_ctx + s - 1) / s;
}

// Per-thread error text for k3mla_last_error().
void set_error(const char* fmt, ...);

// Check a kernel launch; returns K3MLA_OK or K3MLA_E_CUDA with the text recorded.
int check_launch(const char* what);

// True if the current device is an sm_103 part; records the reason otherwise.
bool device_ok();

// 2-D bf16 tensor map over `rows` rows of `cols` elements (row pitch = cols*2
// bytes) with a box of box_cols x box_rows and 128-byte swizzle.
int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows);

// 3-D bf16 tensor map over the latent slab viewed as (64 elements, rows, chunks):
// dim0 = 64 contiguous elements (128 bytes), dim1 = slab rows (pitch row_bytes),
// dim2 = 64-element chunks of a row (pitch 128 bytes).  A box of
// (64, box_rows, box_chunks) lands in shared memory as [chunk][row][128 B] with
// 128-byte swizzle -- the K-major / MN-major operand layout of the tensor cores.
int make_tmap_slab_3d(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems, uint32_t n_chunks,
                      uint32_t box_rows, uint32_t box_chunks);

// General tensor map (bulk tensor stores; also the multi-query q_abs loads): `rank` dims (innermost
// first), byte strides of dims 1.. (multiples of 16), the box, f32 or bf16 elements, with 128-byte
// swizzle (inner box extent 128 bytes) or none.
int make_tmap_store(CUtensorMap* map, bool f32, uint32_t rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box, bool swizzle128);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch `kernel` on `st` with programmatic stream serialization: it may be scheduled while the
// kernel before it in the stream is still running, and every kernel of this library calls
// griddep_wait() before it touches memory that an earlier kernel may write.  Returns K3MLA_OK or
// K3MLA_E_CUDA (text recorded under `what`).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const char* what,
               Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, args...);
    return check_launch(what);
}

// Byte offsets of the decode workspace's regions: final o_lat [96][B][512] bf16 (every slot with at
// most one split lands it there itself), f32 partial O [B][nsplit][96][512] (only when some slot can
// have several splits), and the split records [B][nsplit][96][4] f32 (m_ref, l, best score, best t).
struct WsLayout {
    size_t olat, o, ml, total;
};
inline WsLayout ws_layout(int B, int nsplit)
{
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    WsLayout w;
    w.olat = 0;
    w.o = up((size_t)B * H * LORA * 2);
    w.ml = w.o + (nsplit > 1 ? up((size_t)B * nsplit * H * LORA * 4) : 0);
    w.total = w.ml + (size_t)B * nsplit * H * 4 * 4;
    return w;
}

// Split partials -> o_lat -> W_UV expansion (merge_expand.cu).
struct MergeParams {
    const float* ws_o;     // [B][nsplit][96][512] f32 partial O (null when nsplit == 1)
    const float* ws_ml;    // [B][nsplit][96][4]: m_ref, l, best score, best t (int bits)
    const uint16_t* ws_olat;  // [96][B][512] bf16: final o_lat of the slots with at most one split
    const int32_t* ctx_len;
    const uint16_t* w_kv_b;
    uint16_t* out;         // [B][96][128] bf16
    int32_t* argmax;       // [B][96] or null
    int32_t* dev_err;      // K3MLA_DEV_* bits or null
    int B, max_ctx, max_pages, split_tokens, nsplit;  // split_tokens 0: the default per-slot rule
    int tile;              // slots per CTA: 64 (nsplit == 1, every o_lat landed) or 16 (merge)
};
int launch_merge_expand(const MergeParams& mp, cudaStream_t st);

// k3mla_absorb_q_append with each slot's write position ctx_len[b] - 1 (none when ctx_len[b] <= 0): the
// append of a decode step whose context lengths already count the new token (absorb_append.cu).
int launch_absorb_append_at_ctx(const uint16_t* q, const uint16_t* w_kv_b, uint16_t* q_abs, uint16_t* slab,
                                int n_pages, int n_layers, int layer, const int32_t* block_table,
                                int max_pages_per_slot, const int32_t* ctx_len, const uint16_t* c_kv,
                                int64_t c_stride, const uint16_t* k_rope, int64_t r_stride, int B, int32_t* dev_err,
                                cudaStream_t stream);

}  // namespace k3
