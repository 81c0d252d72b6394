/*
 * mlora.h -- C ABI of libmlora.so: the fused Mixture-of-Experts expert layer
 * with per-token multi-LoRA adapters, as hand-written CUDA kernels for
 * sm_103a (GB300).
 *
 * The operation (pages cited by title and section):
 *  - "Amazon SageMaker 및 Amazon Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA
 *    서빙 최적화", section "섹션별 상세" paragraph 1: every token carries its own
 *    adapter; the adapter's LoRA shrink (x A^T) and expand ((.) B^T) are
 *    folded into each routed expert's projections; section "이미지 분석 /
 *    Diagram": an adapter path on both the gate_up and the down projection;
 *    paragraph 2: layers without adapters exit at once, and the layer runs
 *    under CUDA graphs.
 *  - "[vllm] vLLM ROCm 환경에서 Shared-Expert Fusion을 통한 MoE 추론 성능 최적화",
 *    section "코드 분석" item 1: shared experts are appended after the routed
 *    top-k slots with ids E..E+n_shared-1; item 2: the sort-and-pad (align)
 *    runs over E_tot = w13.shape[0] experts; section "교훈" item 2: the
 *    shared slot weight 1/routed_scaling_factor keeps the fused layer equal
 *    to the separate shared MLP once the sum is scaled by that factor.
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller: contiguous,
 *    row-major, 16-byte aligned.  The library never allocates or frees
 *    device memory and never synchronises the stream, except
 *    mlora_moe_read_status(_static), which waits for the stream by design.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  All work is enqueued on it, so every call can be captured into
 *    a CUDA graph (mlora_moe_read_status(_static) excepted).
 *  - The work runs on the current device (cudaGetDevice).  Outside stream
 *    capture, a tensor pointer that is device memory of another GPU is
 *    refused with MLORA_ERR_INVALID_ARG before anything is enqueued.
 *  - bf16 tensors are passed as void*.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    failed check returns a non-zero status and enqueues nothing.  Values
 *    that live in device memory (expert ids, adapter ids) are checked on the
 *    device: a bad value is skipped (expert id) or treated as "no adapter"
 *    (adapter id) and recorded in the device status word that
 *    mlora_moe_read_status returns.  Kernels never trap.
 *  - Errors reported by the CUDA runtime at launch map to MLORA_ERR_CUDA;
 *    asynchronous faults surface at the caller's next synchronisation.
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mlora_status {
    MLORA_OK = 0,
    MLORA_ERR_INVALID_ARG = 1, /* NULL or misaligned pointer, bad enum value */
    MLORA_ERR_SHAPE = 2,       /* sizes out of range or inconsistent */
    MLORA_ERR_UNSUPPORTED = 3, /* valid in principle, not built (e.g. rank > 64) */
    MLORA_ERR_WORKSPACE = 4,   /* workspace NULL, misaligned or too small */
    MLORA_ERR_CUDA = 5         /* the CUDA runtime or driver reported an error */
} mlora_status;

enum { MLORA_SCORE_SOFTMAX = 0, MLORA_SCORE_SIGMOID_BIAS = 1 };

/* Bits of the device status word (mlora_moe_read_status). */
#define MLORA_DEV_TIMEOUT 1u        /* a pipeline wait gave up after ~2 s; outputs invalid */
#define MLORA_DEV_BAD_EXPERT_ID 2u  /* a topk id was outside [0, E_tot); that slot was dropped */
#define MLORA_DEV_BAD_LORA_IDX 4u   /* a token_lora_idx was outside [-1, L); treated as -1 */
#define MLORA_DEV_BOUNDS 8u         /* bounds-checked debug build only: an index left its buffer; the access was skipped */

#define MLORA_MAX_EXPERTS 1024 /* E (routing) and E_tot (align, forward) */
#define MLORA_MAX_TOPK 64      /* K' = top_k + n_shared */
#define MLORA_MAX_RANK 64      /* LoRA rank: a multiple of 8 in [8, 64] */
#define MLORA_MAX_ALIGN_BLOCK 1024
#define MLORA_FORWARD_BLOCK_M 128 /* block_m used inside mlora_moe_forward */

/*
 * Top-k routing with optional forced shared-expert slots.
 *
 * logits  [M, E] fp32.  bias [E] fp32, read only for SIGMOID_BIAS (may be
 * NULL there: zero bias).  Writes, for K' = top_k + n_shared,
 * topk_ids [M, K'] int32 and topk_w [M, K'] fp32:
 *  - SOFTMAX: the top_k experts by logit (the softmax is monotone), in
 *    descending order, ties to the lower id; weights are the softmax over the
 *    selected logits when renormalize != 0, else the full softmax's entries.
 *  - SIGMOID_BIAS: the top_k experts by sigmoid(l) + bias, computed in fp32,
 *    same order and tie rule; weights sigmoid(l) (no bias), divided by their
 *    sum over the routed slots when renormalize != 0.
 *  - slot top_k + j (j < n_shared) gets id E + j and weight
 *    1 / routed_scaling_factor.
 * Constraints: 0 <= M, 1 <= top_k <= E <= MLORA_MAX_EXPERTS, 0 <= n_shared,
 * K' <= MLORA_MAX_TOPK, routed_scaling_factor > 0 when n_shared > 0.
 * Logits should be finite.  A NaN key (NaN logit, or NaN bias) ranks below
 * every number, ties among NaN keys going to the lower id, so the ids stay
 * in [0, E) whatever the input; the weights of a token with NaN logits are
 * NaN.
 */
mlora_status mlora_moe_route(const float* logits, const float* bias, int M, int E, int top_k, int scoring,
                             int renormalize, int n_shared, float routed_scaling_factor, int32_t* topk_ids,
                             float* topk_w, void* stream);

/*
 * Length of the sorted_ids buffer mlora_moe_align writes:
 * round_up(M*K' + min(E_tot, M*K') * (block_m - 1), block_m).  expert_ids
 * holds max_padded / block_m entries.  Returns 0 for invalid arguments.
 */
size_t mlora_moe_align_max_padded(int M, int K_total, int E_tot, int block_m);

/*
 * Sort and pad the M*K' routed slots by expert (align).
 *
 * topk_ids [M, K_total] int32 with values in [0, E_tot).  Slot f = m*K'+k.
 * Writes sorted_ids [max_padded]: experts in ascending id, each expert's
 * slots in ascending f, padded with the sentinel M*K' to a multiple of
 * block_m; positions past the padded total hold the sentinel.
 * expert_ids [max_padded / block_m]: the expert of each block, -1 past the
 * end.  num_post_padded [1]: the padded total.  Bit-exact and deterministic
 * for a given block_m.  Slots whose id is out of range are skipped.
 * Constraints: 0 <= M, 1 <= K_total <= MLORA_MAX_TOPK,
 * 1 <= E_tot <= MLORA_MAX_EXPERTS, 1 <= block_m <= MLORA_MAX_ALIGN_BLOCK,
 * M*K_total < 2^31 - E_tot*block_m.
 */
mlora_status mlora_moe_align(const int32_t* topk_ids, int M, int K_total, int E_tot, int block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded, void* stream);

/*
 * Bytes of device workspace mlora_moe_forward needs for these sizes (with
 * L = 0 or rank = 0 for a layer without adapters).  Returns 0 for invalid
 * sizes.  The workspace is 256-byte aligned and caller-owned; it may be
 * reused by consecutive calls on the same stream.
 */
size_t mlora_moe_workspace_size(int M, int H, int I, int E_tot, int K_total, int L, int rank);

/*
 * The layer:
 *   y[m] = out_scale * sum_{k<K'} topk_w[m,k] * Expert_{topk_ids[m,k]}(x[m]; l_m)
 * with l_m = token_lora_idx[m] and, for expert e,
 *   h = x W13_e^T + s (x A13_{l,e}^T) B13_{l,e}^T        (2I values; LoRA only if l >= 0)
 *   a = silu(h[0:I]) * h[I:2I]                           (SwiGLU; silu(z) = z / (1 + e^-z))
 *   d = a W2_e^T + s (a A2_{l,e}^T) B2_{l,e}^T           (H values)
 * Shapes (bf16 unless noted): x [M, H]; w13 [E_tot, 2I, H] (rows [0,I) gate,
 * [I,2I) up); w2 [E_tot, H, I]; A13 [L, E_tot, rank, H]; B13 [L, E_tot, 2I,
 * rank]; A2 [L, E_tot, rank, I]; B2 [L, E_tot, H, rank]; token_lora_idx [M]
 * int32 (-1: no adapter); topk_ids [M, K'] int32 in [0, E_tot); topk_w
 * [M, K'] fp32; y [M, H] bf16.  s = scaling.  With shared-expert fusion the
 * route call appends the shared slots and out_scale is the routed scaling
 * factor; n_shared is the number of those trailing slots (0 <= n_shared <
 * K_total; only validated, the slots are ordinary experts here).
 * If any of A13, B13, A2, B2, token_lora_idx is NULL, or L == 0, or rank ==
 * 0, the layer runs without adapters and launches no LoRA work.  When the
 * adapter pointers are given but no token uses an adapter, the LoRA kernels
 * exit on the device and the result equals the adapter-free layer exactly.
 * Constraints: H, I multiples of 8 (16-byte rows), H, I >= 8;
 * rank in {8, 16, ..., 64}; E_tot <= MLORA_MAX_EXPERTS; K' <= MLORA_MAX_TOPK;
 * workspace_bytes >= mlora_moe_workspace_size(...).
 * Intermediates: the adapter shrink result is kept as bf16 (s * x A^T), the
 * SwiGLU output as bf16 (both feed the tensor cores), each slot's expert
 * output as fp32, all accumulation in fp32; y is rounded to bf16 (nearest
 * even).
 */
mlora_status mlora_moe_forward(const void* x, const void* w13, const void* w2, const void* A13, const void* B13,
                               const void* A2, const void* B2, const int32_t* token_lora_idx,
                               const int32_t* topk_ids, const float* topk_w, int M, int H, int I, int E_tot,
                               int K_total, int L, int rank, float scaling, int n_shared, float out_scale, void* y,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * ---- MXFP8 expert weights -------------------------------------------------
 * "[vllm] vLLM ROCm 환경에서 Shared-Expert Fusion을 통한 MoE 추론 성능 최적화",
 * section "코드 분석" item 2: the fused layer runs on an MXFP8 experts path.
 * The pages do not define the format; it is the OCP Microscaling (MX)
 * specification's MXFP8: along the reduction dimension (H for w13 and x, I
 * for w2 and the SwiGLU output) blocks of 32 elements share one E8M0 scale
 * 2^(s-127) (a byte s); elements are FP8 E4M3.  A block converts with
 * shared exponent floor(log2 max|v|) - 8 (a block of zeros: s = 0) and
 * elements v / 2^shared rounded to the nearest E4M3 value, ties to even,
 * saturated to +-448.  In the MXFP8 layer x and the SwiGLU output are
 * quantized this way on the device before they meet the expert weights; the
 * LoRA adapters stay bf16 and read the unquantized x and SwiGLU output
 * (shrink and expand as in the bf16 layer, accumulated with the base
 * product).  H and I must be multiples of 32.
 *
 * Packed scales (the order the tensor cores read them in; `which` 0 is
 * gate_up, 1 is down): for each expert e, tile slab cb and K-chunk kc of 128,
 * 1024 bytes = two 512-byte atoms, atom a holding tile rows 128a..128a+127,
 * row t's scale for K-block kb (0..3) of the chunk at byte
 * (t % 32) * 16 + ((t % 128) / 32) * 4 + kb of its atom.  gate_up: slabs of
 * 96 gate + 96 up rows, cb in [0, ceil(I/96)), kc in [0, ceil(H/128)); tile
 * row t < 96 is w13 row cb*96 + t (gate), t >= 96 is row I + cb*96 + t - 96
 * (up).  down: slabs of 192 rows of w2, cb in [0, ceil(H/192)), kc in
 * [0, ceil(I/128)); tile row t is w2 row cb*192 + t.  Bytes of rows or
 * blocks past the matrix are 0.
 */

/* Bytes of the packed scales of the gate_up (which = 0) or down (which = 1)
 * weights; 0 for invalid sizes. */
size_t mlora_mxfp8_scales_size(int E_tot, int H, int I, int which);

/*
 * Quantize bf16 expert weights to MXFP8 on the device (done once, when the
 * weights are loaded): w13 [E_tot, 2I, H] -> w13_q [E_tot, 2I, H] E4M3
 * codes (bytes, the weights' own layout) and w13_s packed scales
 * (mlora_mxfp8_scales_size(..., 0) bytes); w2 [E_tot, H, I] -> w2_q and
 * w2_s likewise.  All buffers are caller-owned device memory, 16-byte
 * aligned.  Enqueued on `stream`; nothing is allocated.
 */
mlora_status mlora_mxfp8_quantize_weights(const void* w13, const void* w2, int E_tot, int H, int I, void* w13_q,
                                          void* w13_s, void* w2_q, void* w2_s, void* stream);

/* Workspace bytes of mlora_moe_forward_mxfp8 (as mlora_moe_workspace_size). */
size_t mlora_moe_workspace_size_mxfp8(int M, int H, int I, int E_tot, int K_total, int L, int rank);

/*
 * The layer of mlora_moe_forward with MXFP8 expert weights (w13_q, w13_s,
 * w2_q, w2_s from mlora_mxfp8_quantize_weights); every other argument,
 * constraint and convention as there, plus H and I multiples of 32.  The
 * expert tiles are 192 weight rows wide.
 */
mlora_status mlora_moe_forward_mxfp8(const void* x, const void* w13_q, const void* w13_s, const void* w2_q,
                                     const void* w2_s, const void* A13, const void* B13, const void* A2,
                                     const void* B2, const int32_t* token_lora_idx, const int32_t* topk_ids,
                                     const float* topk_w, int M, int H, int I, int E_tot, int K_total, int L,
                                     int rank, float scaling, int n_shared, float out_scale, void* y,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * mlora_moe_forward_static -- the same layer as mlora_moe_forward, for
 * callers that cannot allocate device memory where they run it (their
 * device memory belongs to another allocator they must not bypass, they may
 * not allocate after start-up, or they only hold pointers to tensors).
 * The pages have no counterpart to this entry point; it is a deployment
 * convenience of this library.
 *
 * Arguments are those of mlora_moe_forward without the workspace: the
 * scratch is a fixed device array inside the library, of
 * MLORA_STATIC_WORKSPACE_BYTES, reserved on every GPU that loads the
 * library's kernels and held until the process exits.  Nothing is
 * allocated or freed by the call.
 *  - Sizes whose mlora_moe_workspace_size exceeds the array return
 *    MLORA_ERR_WORKSPACE and enqueue nothing (64 MiB holds, e.g., the
 *    M=64, H=I=2880, E=32, top_k=4, L=8, rank=16 layer).
 *  - The first call on a device looks up the array's device address
 *    (once per device and CUDA context, with that device current); make
 *    that first call before any stream capture on the device.  After
 *    cudaDeviceReset the device's context is a new one and the next call
 *    looks the address up again, so it too should precede any capture.
 *  - Every call shares the one array and it keeps the last call's
 *    contents.  The call clears what must start at zero (its status word)
 *    itself; everything else is written before it is read.  Calls whose
 *    work overlaps on the GPU (different streams, or concurrent host
 *    threads) race on the array: serialise them.
 *  - The device status bits of the last call on the current device are
 *    read with mlora_moe_read_status_static.
 */
#define MLORA_STATIC_WORKSPACE_BYTES (64u << 20)
mlora_status mlora_moe_forward_static(const void* x, const void* w13, const void* w2, const void* A13,
                                      const void* B13, const void* A2, const void* B2,
                                      const int32_t* token_lora_idx, const int32_t* topk_ids, const float* topk_w,
                                      int M, int H, int I, int E_tot, int K_total, int L, int rank, float scaling,
                                      int n_shared, float out_scale, void* y, void* stream);

/*
 * Copies the device status word of the last forward that used `workspace`
 * (MLORA_DEV_* bits, 0 = clean) to *host_status after waiting for `stream`.
 */
mlora_status mlora_moe_read_status(const void* workspace, uint32_t* host_status, void* stream);

/*
 * mlora_moe_read_status for mlora_moe_forward_static: copies the device
 * status word (MLORA_DEV_* bits, 0 = clean) of the last static forward on
 * the current device to *host_status after waiting for `stream`.  Like the
 * static forward itself it has no counterpart on the pages; it lets callers
 * without a workspace see a wait timeout or a bad expert or adapter id.
 * It allocates nothing.  The word belongs to whichever static call ran
 * last on the device: read it on the stream that call used, before another
 * static call is enqueued.
 */
mlora_status mlora_moe_read_status_static(uint32_t* host_status, void* stream);

/*
 * Measurement hook.  Sets, for the calling host thread, MLORA_STAGE_EVENTS
 * cudaEvent_t handles (passed as void*) that every later mlora_moe_forward
 * on this thread records on its stream at the stage boundaries:
 *   [0] before align, [1] after align, [2] after the row gather,
 *   [3] after the experts kernel (both projections with their LoRA shrink
 *       and expand, and SwiGLU), [4] after the combine.
 * The events are recorded with cudaEventRecordExternal while the stream is
 * being captured, so they become event nodes of a CUDA graph.
 * events == NULL (or count == 0) switches the hook off.  The caller owns
 * the events and keeps them alive while the hook is set.  Returns
 * MLORA_ERR_INVALID_ARG when 0 < count < MLORA_STAGE_EVENTS.
 */
#define MLORA_STAGE_EVENTS 5
mlora_status mlora_set_stage_events(void* const* events, int count);

/*
 * Test hook for the bounded waits of the experts kernel.  For the calling
 * host thread: wait_limit_cycles (> 0) replaces the ~2 s limit (in SM clock
 * cycles) after which a pipeline wait gives up; 0 restores it.  stall != 0
 * makes every CTA of later forwards first wait on a workspace flag that
 * nothing sets, so that the wait runs out: the forward then reports
 * MLORA_DEV_TIMEOUT in the device status word (mlora_moe_read_status), its
 * output is invalid, and the context stays usable.  No GPU fault is raised.
 * Returns MLORA_ERR_INVALID_ARG for a negative limit.
 */
mlora_status mlora_set_wait_test(long long wait_limit_cycles, int stall);

/*
 * Tile configuration of the experts kernel ("Amazon SageMaker 및 Amazon
 * Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA 서빙 최적화", section "섹션별
 * 상세" paragraph 4: block and split parameters found per deployment and
 * loaded automatically).  Each bf16 forward picks, for the number of
 * 128-slot blocks it finds on the device, a tile width of 256, 192 or 128
 * weight rows (width class 0, 1, 2), and a shrink group size (adapters per
 * shrink tile, 1-4): from the library's tuned table for the layer's shape
 * (H, I, E_tot, K', rank) when it has a row for it, else from the wave rule
 * (fill the grid's SMs with each projection's tiles) and at most 4
 * adapters (256 stacked rank rows) a group.  The table is written by the
 * offline tuner (python -m moe_layer_lora_gb300.autotune) and compiled in.
 * Neither choice changes any output bit: every output element sums the same
 * products in the same order.
 *
 * mlora_set_tile_config: for the calling host thread, force the width class
 * (-1: table or rule) and the shrink group size (0: table or rule; clamped to
 * what the rank allows) of later forwards -- the tuner's hook.  MXFP8
 * layers keep their 192-row width.  MLORA_ERR_INVALID_ARG out of range.
 *
 * mlora_tile_config: the width class and group size a bf16 layer of this
 * shape would use for `nblocks` blocks on a grid of `grid` CTAs (one per
 * SM), and whether a tuned row applied (*tuned, may be NULL).  Host only.
 */
mlora_status mlora_set_tile_config(int width_class, int gsize);
mlora_status mlora_tile_config(int H, int I, int E_tot, int K_total, int rank, int nblocks, int grid,
                               int* width_class, int* gsize, int* tuned);

/*
 * CTA-pair mode of the bf16 experts kernel (opt-in).  The experts kernel
 * runs as clusters of two CTAs on two SMs, each pair sharing 256-row MMAs
 * (tcgen05 cta_group::2) over two 128-slot blocks of one expert: each SM
 * loads its own block's token rows and half of the tile's 256 weight rows,
 * two K-chunks of 64 per copy, so a stage brings a third fewer bytes per
 * MMA and the producer issues half as many copies.  Align then pads every
 * expert's blocks to an even count (the second block of a pair may hold no
 * rows), which the workspace size accounts for: mlora_moe_workspace_size
 * reports the size for the mode in effect on the calling thread when it is
 * called.  Tiles are 256 weight rows wide in this mode, and a block's
 * shrink tiles occupy both SMs of a pair.  On prefill-sized layers the pair
 * kernel runs its MMAs faster but computes more padded rows, and the
 * adapter work costs more, so it is off by default.  With finite adapter
 * weights the mode changes no output bit except, possibly, the sign of an
 * exact zero: an adapter's expand adds zero products to the rows of a
 * pair's block that does not use it (a non-finite expand weight then turns
 * them into NaN).
 *
 * mlora_set_pair_mode: for the calling host thread, 1 runs later bf16
 * forwards in pair mode, 0 (default) with one CTA per SM; the MXFP8 layer
 * never pairs.  MLORA_ERR_INVALID_ARG for other values.
 * mlora_pair_mode: the calling thread's mode (1 or 0).  Host only.
 */
mlora_status mlora_set_pair_mode(int on);
int mlora_pair_mode(void);

/* Static, human-readable name of a status code. */
const char* mlora_status_string(mlora_status status);

#ifdef __cplusplus
}
#endif

#endif /* MLORA_H */
