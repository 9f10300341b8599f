// plan.cpp -- an opt-in split length planned for a whole batch (batch-dependent numerics).
//
// pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode": the decode
// reduces each slot's context in splits and merges the partial results in a
// fixed order.  The default rule cuts every slot by its own context alone, so a
// slot's bits never depend on its batch; on a ragged batch of few slots that
// leaves most SM pairs idle.  The host that claims the pages knows every slot's
// context, and this call plans one split length for the batch instead: the
// shortest whose non-empty splits still fit one wave of SM pairs.  A slot's bits
// then depend on the other slots' contexts and on the SM count.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/k3mla.h"

namespace k3 {
void set_error(const char* fmt, ...);
}

// Splits that hold at least one token of their slot: sum over b of ceil(ctx_b / split).
static long long live_splits(const int32_t* ctx, int B, int max_ctx, int split)
{
    long long n = 0;
    for (int b = 0; b < B; ++b) {
        const int c = std::min(std::max(ctx[b], 0), max_ctx);
        n += (c + split - 1) / split;
    }
    return n;
}

extern "C" int k3mla_batch_planned_split_tokens(const int32_t* ctx_host, int B, int max_ctx)
{
    if (B <= 0 || max_ctx <= 0) return K3MLA_TILE;
    if (!ctx_host) {
        k3::set_error("k3mla_batch_planned_split_tokens: ctx_host is NULL");
        return K3MLA_E_INVALID;
    }
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long pairs = sms / 2;
    const int whole = (max_ctx + K3MLA_TILE - 1) / K3MLA_TILE * K3MLA_TILE;  // one split per slot
    int longest_ctx = 0;
    for (int b = 0; b < B; ++b) longest_ctx = std::max(longest_ctx, std::min(std::max(ctx_host[b], 0), max_ctx));
    // The live split count does not grow with the split, so the shortest split that fits one wave
    // is found by bisection; the longest split it leaves is the decode's critical path.  Once a
    // split covers the longest context, every slot has one live split whatever the length, and a
    // whole-context split does the same work without empty splits or a merge of partials.
    int lo = 1, hi = (std::min(whole, longest_ctx) + K3MLA_TILE - 1) / K3MLA_TILE;  // in tiles
    if (hi <= 1 || live_splits(ctx_host, B, max_ctx, (hi - 1) * K3MLA_TILE) > pairs) return whole;
    --hi;  // (hi) tiles fit; find the fewest that do
    while (lo < hi) {
        const int mid = (lo + hi) / 2;
        if (live_splits(ctx_host, B, max_ctx, mid * K3MLA_TILE) <= pairs) hi = mid;
        else lo = mid + 1;
    }
    return lo * K3MLA_TILE;
}
