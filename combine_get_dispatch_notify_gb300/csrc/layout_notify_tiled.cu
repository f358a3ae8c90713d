// Steps 1 and 2 in one launch for shapes of any size: the tiled form (see
// ln_tiled.cuh).  Persistent CTAs take tiles of TT tokens in (source rank,
// tile) order, the first by block index and later ones from a ticket; the
// grid is what the device holds at once, at most one CTA per tile.  The tile size grows from 512 tokens until the tiles
// fit one wave of 512-thread CTAs, then shrinks to the smallest multiple of 32
// that still does; CTAs have 512 threads then (256 when a caller-chosen tile
// size leaves more tiles than that).
#include "ln_tiled.cuh"

namespace ep {
namespace {

constexpr int kTiledThreads = 256;
constexpr int kTiledThreadsWide = 512;  // when the tiles fit one wave of 512-thread CTAs
constexpr long long kMaxTiles = 16384;  // the tile size grows beyond this many tiles

__global__ void __launch_bounds__(kTiledThreadsWide) layout_notify_tiled_kernel(TiledLnArgs p) {
    extern __shared__ __align__(16) int32_t dyn[];
    __shared__ TiledShared sh;
    griddep_launch_dependents();
    griddep_wait();  // top-k ids written by the preceding kernel are visible
    // The issuing thread is held while the prefetch is taken in: not the one
    // that takes the tickets.
    if (threadIdx.x == kWarp) tiled_prefetch_ids(p, static_cast<int>(blockIdx.x));
    int b = static_cast<int>(blockIdx.x);  // the grid is at most one CTA per tile
    while (b >= 0) b = tiled_tile(p, sh, dyn, b, 0);
}

}  // namespace

namespace {
// `base` tokens per tile (fewer when T is smaller, a multiple of 32), doubled
// (up to 8192) while there are more than kMaxTiles tiles.
int tile_tokens_from(const Shape& sh, int base) {
    int TT = base;
    if (sh.T < TT) TT = sh.T < kWarp ? kWarp : (sh.T + kWarp - 1) / kWarp * kWarp;
    while (TT < 8192 && static_cast<long long>(sh.R) * ((sh.T + TT - 1) / TT) > kMaxTiles) TT *= 2;
    return TT;
}
}  // namespace

// Tokens per tile the launcher starts from: 512 by that rule.
int tiled_tile_tokens(const Shape& sh, int requested) {
    return requested > 0 ? requested : tile_tokens_from(sh, 512);
}

// Tokens per tile the workspace is sized for: 256 by that rule, so that it
// holds at least as many tiles as the launcher takes (it never goes below
// half of a tile of 512 or more tokens, and checks against this).
int tiled_sizing_tokens(const Shape& sh) { return tile_tokens_from(sh, 256); }

size_t tiled_workspace_bytes(const Shape& sh, int TT) {
    const long long tps = sh.T > 0 ? (sh.T + TT - 1) / TT : 1;
    return tiled_workspace_layout(sh.R, sh.N, sh.R * tps).total;
}

size_t tiled_workspace_zero_bytes() { return tiled_workspace_layout(1, 1, 1).words; }

size_t tiled_smem_bytes(const Shape& sh, int TT) {
    return sizeof(int32_t) * tiled_smem_words(sh.E, TT, sh.R + sh.N);
}

cudaError_t launch_layout_notify_tiled(const Shape& sh, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                                       int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                                       uint8_t* is_token_in_rank, const NotifyArgs& a, void* workspace,
                                       int tile_tokens, int stall_tile, long long wait_limit_ns,
                                       cudaStream_t stream) {
    const void* kernel = reinterpret_cast<const void*>(layout_notify_tiled_kernel);
    const int sms = device_sm_count();
    int TT = tiled_tile_tokens(sh, tile_tokens);
    if (tile_tokens == 0) {
        // larger tiles while the tiles are more than one wave of resident
        // 512-thread CTAs
        while (TT < 8192) {
            const long long tiles = static_cast<long long>(sh.R) * ((sh.T + TT - 1) / TT);
            const int per = max_blocks_per_sm(kernel, kTiledThreadsWide, tiled_smem_bytes(sh, TT));
            if (tiles <= static_cast<long long>(per) * sms) break;
            TT *= 2;
        }
        // then the smallest tile (a multiple of 32) that still fits that wave:
        // spreading the tokens over every resident slot shortens the busiest
        // SM - within the tile count the workspace is sized for
        if (TT >= 512) {
            const long long slots =
                static_cast<long long>(max_blocks_per_sm(kernel, kTiledThreadsWide, tiled_smem_bytes(sh, TT))) * sms;
            const long long per_source = slots / sh.R;
            const int ts = tiled_sizing_tokens(sh);
            if (per_source >= 1) {
                const long long tt = ((sh.T + per_source - 1) / per_source + kWarp - 1) / kWarp * kWarp;
                if (tt < TT && tt * 2 > TT && tt >= ts) TT = static_cast<int>(tt);
            }
        }
    }
    TiledLnArgs p = tiled_args(sh, TT, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                               num_tokens_per_expert, is_token_in_rank, a, workspace);
    p.stall_tile = stall_tile;
    p.wait_limit_ns = wait_limit_ns;
    const size_t smem = tiled_smem_bytes(sh, TT);
    // 512 threads per CTA (half the ids per thread) when every tile still
    // gets a CTA of its own at once, else 256 (more CTAs resident)
    const int per_wide = max_blocks_per_sm(kernel, kTiledThreadsWide, smem);
    const int threads = p.n_tiles <= static_cast<long long>(per_wide) * sms ? kTiledThreadsWide : kTiledThreads;
    const int per_sm = threads == kTiledThreadsWide ? per_wide : max_blocks_per_sm(kernel, kTiledThreads, smem);
    if (per_sm <= 0 || sms <= 0) return cudaErrorInvalidConfiguration;
    const long long cap = static_cast<long long>(per_sm) * sms;
    const long long grid = p.n_tiles < cap ? p.n_tiles : cap;
    return launch_pdl(layout_notify_tiled_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, 0,
                      false, p);
}

}  // namespace ep
