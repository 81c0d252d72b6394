// internal.cuh -- declarations shared by the translation units of libmlora.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "mlora.h"

namespace mlora {

constexpr int kBlockM = MLORA_FORWARD_BLOCK_M;  // token rows per GEMM tile (MMA M)
constexpr int kBlockK = 64;                     // bf16 elements per 128-byte swizzle row
constexpr int kTileWidths = 3;                   // weight rows per experts tile: 256, 192 or 128
__host__ __device__ constexpr int tile_width(int wc) { return 256 - 64 * wc; }
// Tuned tile widths are kept per power-of-two bucket of a launch's block
// count: bucket b holds [2^b, 2^(b+1)) blocks, the last one everything above.
constexpr int kWidthBuckets = 16;
__host__ __device__ inline int width_bucket(int nblocks) {
    int b = 0;
    while (b + 1 < kWidthBuckets && (nblocks >> (b + 1)) > 0) ++b;
    return b;
}

// The tile width of a launch with nblocks blocks (I, H the projections'
// output widths) on a grid of `grid` CTAs when no tuned table applies.  One
// SM streams weights at a rate of its own (~44 GB/s measured, about the HBM
// rate divided by the SM count), so a phase whose tiles do not fill whole
// waves of the grid leaves HBM idle.  With at most two waves of wide
// gate_up tiles, the width that minimises (waves of gate_up tiles) x (bytes
// per gate_up tile) + the same for down is taken, the wider on a tie;
// larger batches keep wide tiles.
__host__ __device__ inline int choose_width(int nblocks, int I, int H, long grid) {
    const long wide = static_cast<long>(nblocks) * ((I + 127) / 128);
    if (wide > 2 * grid) return 0;
    int best = 0;
    long best_cost = -1;
    for (int wc = 0; wc < kTileWidths; ++wc) {
        const int n = tile_width(wc);
        const long tg = static_cast<long>(nblocks) * ((I + n / 2 - 1) / (n / 2));
        const long td = static_cast<long>(nblocks) * ((H + n - 1) / n);
        const long cost =
            ((tg + grid - 1) / grid) * n * static_cast<long>(H) + ((td + grid - 1) / grid) * n * static_cast<long>(I);
        if (best_cost < 0 || cost < best_cost) {
            best = wc;
            best_cost = cost;
        }
    }
    return best;
}
constexpr int kLoraTileCols = 64;               // shrink result row, padded to one swizzle row
constexpr int kRowBox = 32;                     // token rows per TMA box of an A operand
constexpr long long kWaitCycles = 4000000000LL;  // default spin limit of a device wait (~2 s at 2 GHz)

// Bounds-checked debug build (compiled with -DMLORA_CHECK_BOUNDS): every
// computed index into a workspace or output buffer is checked before the
// store; a bad one sets MLORA_DEV_BOUNDS in the status word and the store
// is skipped, so nothing faults.  The normal build compiles the checks away.
#ifdef MLORA_CHECK_BOUNDS
#define MLORA_IN_BOUNDS(cond, status) (::mlora::bounds_ok((cond), (status)))
#else
#define MLORA_IN_BOUNDS(cond, status) true
#endif
#ifdef __CUDACC__
__device__ __forceinline__ bool bounds_ok(bool ok, uint32_t* status) {
    if (!ok && status) atomicOr(status, MLORA_DEV_BOUNDS);
    return ok;
}
#endif

// Per-forward buffers carved out of the caller's workspace.
struct Workspace {
    uint32_t* status;      // [0] device status word
    int32_t* n_pad;        // padded slot total written by align
    int32_t* gt_total;     // number of shrink group tiles
    int32_t* max_rows;     // most real rows in any block
    int32_t* done13;       // [max_blocks] shrink tiles finished per block, gate_up projection
    int32_t* done2;        // [max_blocks] the same for the down projection
    int32_t* tile_next;    // experts tiles claimed so far
    int32_t* act_done;     // [max_blocks] gate_up tiles finished per block
    size_t zeroed_bytes;   // leading bytes cleared by every forward (header and counters)
    int32_t* sorted_ids;   // [max_padded]
    int32_t* expert_ids;   // [max_blocks]
    int32_t* blk_rows;     // [max_blocks] real (non-padding) rows of each block
    int32_t* lora_of;      // [max_padded] adapter of each sorted position (-1: none / pad)
    int32_t* blk_nad;      // [max_blocks] distinct adapters in the block
    int32_t* blk_lt_start; // [max_blocks] first LoRA tile of the block
    int32_t* blk_lora;     // [max_blocks * cap] the block's adapters, ascending
    int32_t* gt_block;     // [max_lt] block of each shrink group tile
    int32_t* gt_first;     // [max_lt] first adapter (index into the block's list) of each group
    void* x_perm;          // [max_padded, H] bf16: x rows gathered in sorted order
    void* act;             // [max_padded, I] bf16: SwiGLU output in sorted order
    void* lora_t13;        // [max_lt * 128, 64] bf16: s * x A13^T, one masked LoRA tile per (block, adapter)
    void* lora_t2;         // [max_lt * 128, 64] bf16: s * act A2^T, the same for the down projection
    void* y_slot;          // [M*K', H] fp32: each slot's expert output
    uint8_t* x_q;          // MXFP8 layer: [max_padded, H] E4M3 x rows in sorted order
    uint8_t* x_s;          // [max_blocks][ceil(H/128)][512] their scale atoms
    uint8_t* act_q;        // [max_padded, I] E4M3 SwiGLU rows
    uint8_t* act_s;        // [max_blocks][ceil(I/128)][512] their scale atoms
    size_t bytes;
};

struct Sizes {
    int M, H, I, E_tot, K_total, L, rank;
    bool lora;
    long S;           // M * K_total
    long max_padded;  // with block_m = kBlockM
    long max_blocks;
    int cap;          // adapters per block list: min(L, kBlockM)
    int gsize;        // adapters per shrink group tile: 256 / rank rounded up to 16
    long max_lt;
    bool mx;          // MXFP8 expert weights
    int nkc0, nkc1;   // K-chunks of 128 of H and of I (MXFP8)
    // CTA-pair experts tiles (pair_mode): every expert's blocks padded to
    // an even count, so that blocks 2u and 2u+1 always share an expert;
    // max_padded then counts padding up to 2 * kBlockM per expert
    bool pair;
};

Sizes make_sizes(int M, int H, int I, int E_tot, int K_total, int L, int rank, bool mx = false);
Workspace carve_workspace(const Sizes& z, void* base);  // base == nullptr: sizing only

long align_max_padded(long S, int E_tot, int block_m);

// Extra outputs of align used only inside the forward.  blk_rows is always
// written when set; the adapter fields only when token_lora_idx is set.
struct AlignExtra {
    uint32_t* zero;  // words cleared first thing (the forward's header and counters)
    int32_t* max_rows;  // most real rows in any block (<= block_m), or null
    long lt_cap;     // capacity of the group-tile lists (bounds checks)
    int zero_words;
    int32_t* blk_rows;
    const int32_t* token_lora_idx;
    int L;
    int K_total;
    int cap;
    int32_t* lora_of;
    int32_t* blk_nad;
    int32_t* blk_lora;
    int32_t* blk_lt_start;
    int gsize;
    int32_t* gt_block;
    int32_t* gt_first;
    int32_t* gt_total;
    int pair_pad;    // pad every expert's blocks to an even count (empty blocks: 0 rows)
};

cudaError_t launch_route(const float* logits, const float* bias, int M, int E, int top_k, int scoring,
                         int renormalize, int n_shared, float inv_rsf, int32_t* ids, float* w, cudaStream_t s);

cudaError_t launch_align(const int32_t* ids, long S, int E_tot, int block_m, long max_padded, int32_t* sorted,
                         int32_t* expert_ids, int32_t* n_pad, uint32_t* status, const AlignExtra* extra,
                         cudaStream_t s);

// Small batches (align_small.cu): at most kSmallMaxSlots slots, one
// latency-lean launch; with `gather` set the same launch also copies the x
// rows into sorted order (the row gather of the forward).
constexpr long kSmallMaxSlots = 2048;
struct GatherArgs {
    const void* x;  // [M, H] bf16
    void* x_perm;   // [max_padded, H] bf16 (may be null in the MXFP8 layer without adapters)
    int H;
    int K_total;
    uint8_t* x_q;   // MXFP8 layer: [max_padded, H] E4M3 rows, else null
    uint8_t* x_s;   // MXFP8 layer: [max_blocks][ceil(H/128)][512] scale atoms
};
bool align_small_fits(long S, int E_tot, int block_m, long max_padded, const AlignExtra* extra, bool gather);
cudaError_t launch_align_small(const int32_t* ids, long S, int E_tot, int block_m, long max_padded, int32_t* sorted,
                               int32_t* expert_ids, int32_t* n_pad, uint32_t* status, const AlignExtra* extra,
                               const GatherArgs* gather, cudaStream_t s);

cudaError_t launch_gather_rows(const void* x, int H, const int32_t* sorted, const int32_t* n_pad, long S,
                               int K_total, long max_padded, void* x_perm, uint32_t* status, cudaStream_t s);

cudaError_t launch_combine(const void* y_slot, const int32_t* topk_ids, const float* topk_w, int M, int H,
                           int K_total, int E_tot, float out_scale, void* y, cudaStream_t s);

// ------------------------------------------------------------ grouped GEMM --
// One projection of the expert MLP: gate_up (side 0) or down (side 1).
struct alignas(128) GemmSide {
    CUtensorMap tm_a;       // token rows [rows, K] (x in sorted order / act), box {64, kRowBox}
    CUtensorMap tm_a_full;  // the same with box {64, 128}: one box per full block
    // weight rows: w13 view {H, I, 2, E_tot} / w2 view {I, H, E_tot}, one
    // map per tile width (256, 192, 128 weight rows; a gate_up box takes
    // half the rows from the gate and half from the up half, gate first).
    // A CTA-pair launch (256-row tiles only) holds the 128-row box of one
    // gate_up half in width class 1's slot, here and in tm_lb.
    CUtensorMap tm_b[kTileWidths];
    CUtensorMap tm_sa;      // LoRA shrink weights: A13 / A2 view {K, rank, L*E_tot}
    // LoRA expand weights: B13 view {rank, I, 2, L*E_tot} / B2 view {rank, H, L*E_tot},
    // one map per tile width
    CUtensorMap tm_lb[kTileWidths];
    CUtensorMap tm_t;       // this side's LoRA tiles [tiles*128, 64], box {64, kRowBox}
    CUtensorMap tm_t_full;  // box {64, 128}
    // Maps of the launch kind.  MXFP8 layer: E4M3 token rows (x codes / act
    // codes [rows, K]), box {128, kRowBox} (tm_ax) and {128, 128}
    // (tm_ax_full); E4M3 weight rows (tm_bx: w13 codes view {H, I, 2,
    // E_tot}, box {128, 96, 2, 1} / w2 codes {I, H, E_tot}, box {128, 192,
    // 1}).  CTA-pair launch (bf16): two K-chunks of 64 per copy -- token rows
    // viewed as {64, rows, K/64} (chunk stride 128 B), box {64, 128, 2}
    // (tm_ax_full), and one CTA's half of a weight slab, w13 viewed as {64,
    // I, 2, E_tot, H/64}, box {64, 128, 1, 1, 2} / w2 as {64, H, E_tot,
    // I/64}, box {64, 128, 1, 2} (tm_bx); both land as [chunk][row][64].
    // A view covers only the whole chunks of K (a partial last chunk is
    // loaded with the 2D maps).
    CUtensorMap tm_ax;
    CUtensorMap tm_ax_full;
    CUtensorMap tm_bx;
    const uint8_t* a_scales;  // token-row scale atoms [max_blocks][nkc][512]
    const uint8_t* b_scales;  // packed weight scales [E_tot][slabs][nkc][1024]
    uint8_t* out_q;           // gate_up side: act codes [rows, I]
    uint8_t* out_s;           // gate_up side: act scale atoms [max_blocks][ceil(I/128)][512]
    int nkc;                  // K-chunks of 128 (MXFP8)
    void* lora_t;           // LoRA tiles: written by the shrink tiles, read by the expand stages
    int32_t* done;          // per block: finished shrink tiles (zero at launch)
    void* out;              // act [rows, I] bf16 / y_slot [M*K', H] fp32
    int K;                  // reduction length: H / I
    int n_out;              // output columns: I / H
    int ncb;                // column slabs per block, wide tiles: ceil(I/128) / ceil(H/256)
};

struct alignas(128) GemmParams {
    GemmSide side[2];
    const int32_t* n_pad;
    const int32_t* expert_ids;
    const int32_t* blk_rows;
    const int32_t* sorted_ids;
    const int32_t* lora_of;
    const int32_t* blk_nad;
    const int32_t* blk_lora;
    const int32_t* blk_lt_start;
    const int32_t* gt_block;
    const int32_t* gt_first;
    const int32_t* gt_total;
    int32_t* act_done;  // per block: finished gate_up tiles (zero at launch)
    long lt_cap;        // LoRA tiles the workspace holds (bounds checks)
    long pad_cap;       // sorted positions the workspace holds (bounds checks)
    int32_t* tile_next; // tiles claimed so far (zero at launch)
    const int32_t* max_rows;  // most real rows in any block (written by align)
    uint32_t* status;
    long long wait_limit;        // clock cycles a wait may take before the CTA gives up
    const int32_t* stall_flag;   // test hook: non-null = wait on this never-set flag first
    int E_tot;
    int cap;
    int gsize;
    int rank;
    int S;              // sentinel slot value M*K'
    int has_lora;
    int mx;             // MXFP8 expert weights (fixed 192-row tiles)
    int pair;           // CTA-pair tiles over blocks (2u, 2u+1): clusters of 2, 256-row MMAs
    // tuned tile width class per block-count bucket (-1: the rule, choose_width)
    int8_t width_table[kWidthBuckets];
    float scaling;
};

// The expert MLP of all blocks in one persistent kernel: gate_up shrink
// tiles, gate_up tiles (+ expand, SwiGLU), down shrink tiles, down tiles
// (+ expand); see gemm.cu.
cudaError_t launch_experts(const GemmParams& p, long max_tiles, cudaStream_t s);

// MXFP8 (mxfp8.cu): weights to E4M3 codes and packed scales; the row gather
// of the MXFP8 layer (x rows quantized into sorted order, plus the bf16 rows
// the adapters' shrink reads when x_perm is set).
cudaError_t launch_mx_quantize_weights(const void* w, long rows, int K, int which, int H, int I, uint8_t* codes,
                                       uint8_t* packed_scales, cudaStream_t s);
cudaError_t launch_mx_gather(const void* x, int H, int K_total, const int32_t* sorted, const int32_t* n_pad,
                             long S, long max_padded, uint8_t* x_q, uint8_t* x_s, void* x_perm, uint32_t* status,
                             cudaStream_t s);

int device_sm_count();

// Whether a bf16 layer runs its experts kernel as CTA pairs: only when the
// calling thread asked for it (mlora_set_pair_mode); the MXFP8 layer never.
bool use_pair_mode(bool mx);

// Launch with programmatic stream serialisation (see griddep_wait in ptx.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same as clusters of `cluster` CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cluster, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace mlora
