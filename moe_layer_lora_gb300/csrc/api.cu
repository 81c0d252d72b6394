// api.cu -- the extern "C" entry points of libmlora.so: host-side argument
// validation, workspace layout, TMA tensor-map encoding and the launch
// sequence of the fused MoE-LoRA layer.
//
// Forward, all on the caller's stream, no host synchronisation, no
// allocation (capturable in a CUDA graph):
//   align (clears the status word and counters first; + per-block adapter lists)
//   -> gather x rows (in the align launch for batches of up to
//   kSmallMaxSlots slots) -> experts kernel (gate_up shrink, gate_up + expand +
//   SwiGLU, down shrink, down + expand, one persistent grid) -> combine
// Without adapters the experts kernel runs only base tiles; when adapters
// are given but no token uses one, align finds no shrink tiles on the
// device and the expand chunks are skipped, so the layer exits early
// without a host round trip ("Amazon SageMaker 및
// Amazon Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA 서빙 최적화", section
// "섹션별 상세" paragraph 2).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "internal.cuh"
#include "mx.cuh"

namespace mlora {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// bf16 tensor map with 128-byte swizzle; dims innermost first, strides in
// bytes for dims 1..rank-1.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 bytes (MXFP8 layer)
bool make_map_u8(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                 const cuuint32_t* box) {
    return make_map(m, base, rank, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

mlora_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLORA_OK : MLORA_ERR_CUDA; }

// Tuned tile widths and shrink group sizes per layer shape (tuned_tiles.inc,
// written by the offline tuner); the last row (H = 0) ends the table.
struct TunedShape {
    int H, I, E_tot, K_total, rank;
    int8_t wc[kWidthBuckets];
    int gsize;
};
const TunedShape kTunedShapes[] = {
#include "tuned_tiles.inc"
    {0, 0, 0, 0, 0, {0}, 0},
};

// tile override for the tuner (mlora_set_tile_config), per host thread
thread_local int g_force_wc = -1;
thread_local int g_force_gsize = 0;
thread_local bool g_pair_mode = false;

thread_local cudaEvent_t g_stage_events[MLORA_STAGE_EVENTS];
thread_local bool g_stage_events_on = false;
// wait-limit test hook (mlora_set_wait_test)
thread_local long long g_wait_limit = kWaitCycles;
thread_local bool g_stall_test = false;

// Inside stream capture the events become graph event-record nodes (the
// external flag); outside capture they are recorded normally.
cudaError_t mark_stage(int i, cudaStream_t s) {
    if (!g_stage_events_on) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(s, &cs);
    if (err != cudaSuccess) return err;
    if (cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(g_stage_events[i], s, cudaEventRecordExternal);
    return cudaEventRecord(g_stage_events[i], s);
}

// MLORA_DEBUG=1 in the environment prints the CUDA error behind an
// MLORA_ERR_CUDA return to stderr.
mlora_status cuda_fail(cudaError_t e, const char* where) {
    static const bool verbose = [] {
        const char* v = getenv("MLORA_DEBUG");
        return v && *v && *v != '0';
    }();
    if (verbose) fprintf(stderr, "libmlora: %s: %s\n", where, cudaGetErrorString(e));
    return MLORA_ERR_CUDA;
}

// Outside stream capture: does any of the pointers name device memory of
// a GPU other than the current one?  The kernels run on the current device,
// and their tensor maps and loads would then reach another GPU's memory.
// (During capture the check is skipped: the capture's own eager calls, made
// before it, ran it.)  Host, managed and unregistered pointers pass.
bool foreign_device_memory(cudaStream_t s, std::initializer_list<const void*> ptrs) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (cs != cudaStreamCaptureStatusNone) return false;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    for (const void* p : ptrs) {
        if (!p) continue;
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            (void)cudaGetLastError();
            continue;
        }
        if (a.type == cudaMemoryTypeDevice && a.device != dev) return true;
    }
    return false;
}

// The tile width table (per block-count bucket; -1 = the wave rule) and the
// shrink group size a layer of this shape uses: the thread's override if
// set, else the tuned row of this shape, else the rules.  MXFP8 layers keep
// their fixed width.  Returns whether a tuned row applied.
bool resolve_tiles(int H, int I, int E_tot, int K_total, int rank, bool mx, int8_t* table, int* gsize) {
    for (int b = 0; b < kWidthBuckets; ++b) table[b] = -1;
    bool tuned = false;
    const int rp = (rank + 15) / 16 * 16;
    const int gmax = rank > 0 ? std::min(4, (mx ? kMxWidth : 256) / rp) : 1;
    for (const TunedShape* t = kTunedShapes; t->H; ++t) {
        if (t->H == H && t->I == I && t->E_tot == E_tot && t->K_total == K_total && t->rank == rank) {
            tuned = true;
            if (!mx)
                for (int b = 0; b < kWidthBuckets; ++b)
                    table[b] = t->wc[b] >= 0 && t->wc[b] < kTileWidths ? t->wc[b] : -1;
            if (t->gsize > 0) *gsize = std::min(t->gsize, gmax);
            break;
        }
    }
    if (g_force_wc >= 0 && !mx)
        for (int b = 0; b < kWidthBuckets; ++b) table[b] = static_cast<int8_t>(g_force_wc);
    if (g_force_gsize > 0 && rank > 0) *gsize = std::min(g_force_gsize, gmax);
    return tuned;
}

}  // namespace

int device_sm_count() {
    // per-device cache, shared by host threads (idempotent relaxed writes)
    static std::atomic<int> counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64) {
        const int c = counts[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (dev >= 0 && dev < 64) counts[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool use_pair_mode(bool mx) { return g_pair_mode && !mx; }

Sizes make_sizes(int M, int H, int I, int E_tot, int K_total, int L, int rank, bool mx) {
    Sizes z{};
    z.mx = mx;
    z.nkc0 = static_cast<int>(mx_chunks(0, H, I));
    z.nkc1 = static_cast<int>(mx_chunks(1, H, I));
    z.M = M;
    z.H = H;
    z.I = I;
    z.E_tot = E_tot;
    z.K_total = K_total;
    z.L = L;
    z.rank = rank;
    z.lora = L > 0 && rank > 0;
    z.S = static_cast<long>(M) * K_total;
    z.pair = use_pair_mode(mx);
    z.max_padded = align_max_padded(z.S, E_tot, z.pair ? 2 * kBlockM : kBlockM);
    z.max_blocks = z.max_padded / kBlockM;
    z.cap = z.lora ? std::min(L, kBlockM) : 0;
    z.max_lt = z.max_blocks * z.cap;
    // adapters per shrink group tile: up to 256 stacked rank rows (the MMA's
    // N; 192, the accumulator width, in the MXFP8 layer), at most 4 so that
    // a block's shrink spreads over more SMs
    z.gsize = z.lora ? std::min(4, (mx ? kMxWidth : 256) / ((rank + 15) / 16 * 16)) : 1;
    return z;
}

Workspace carve_workspace(const Sizes& z, void* base) {
    Workspace w{};
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        const size_t o = off;
        off += round256(bytes);
        return base ? static_cast<char*>(base) + o : nullptr;
    };
    // cleared by every forward: the header and the per-block shrink counters
    char* header = take(256);
    w.status = reinterpret_cast<uint32_t*>(header);
    w.n_pad = reinterpret_cast<int32_t*>(header ? header + 4 : nullptr);
    w.gt_total = reinterpret_cast<int32_t*>(header ? header + 8 : nullptr);
    w.tile_next = reinterpret_cast<int32_t*>(header ? header + 12 : nullptr);
    w.max_rows = reinterpret_cast<int32_t*>(header ? header + 28 : nullptr);  // (+24: the wait test's flag)
    w.act_done = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
    if (z.lora) {
        w.done13 = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
        w.done2 = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
    }
    w.zeroed_bytes = off;
    w.sorted_ids = reinterpret_cast<int32_t*>(take(4 * z.max_padded));
    w.expert_ids = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
    w.blk_rows = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
    if (z.lora) {
        w.lora_of = reinterpret_cast<int32_t*>(take(4 * z.max_padded));
        w.blk_nad = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
        w.blk_lt_start = reinterpret_cast<int32_t*>(take(4 * z.max_blocks));
        w.blk_lora = reinterpret_cast<int32_t*>(take(4 * z.max_blocks * z.cap));
        w.gt_block = reinterpret_cast<int32_t*>(take(4 * z.max_lt));
        w.gt_first = reinterpret_cast<int32_t*>(take(4 * z.max_lt));
    }
    // bf16 token rows: the base GEMMs' A (bf16 layer) or the shrinks' (adapters)
    if (!z.mx || z.lora) {
        w.x_perm = take(2 * static_cast<size_t>(z.max_padded) * z.H);
        w.act = take(2 * static_cast<size_t>(z.max_padded) * z.I);
    }
    if (z.mx) {
        // MXFP8 token rows and their scale atoms (one per 128 rows and K-chunk)
        w.x_q = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(z.max_padded) * z.H));
        w.x_s = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(z.max_blocks) * z.nkc0 * kMxAtom));
        w.act_q = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(z.max_padded) * z.I));
        w.act_s = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(z.max_blocks) * z.nkc1 * kMxAtom));
    }
    if (z.lora) {
        w.lora_t13 = take(2 * static_cast<size_t>(z.max_lt) * kBlockM * kLoraTileCols);
        w.lora_t2 = take(2 * static_cast<size_t>(z.max_lt) * kBlockM * kLoraTileCols);
    }
    w.y_slot = take(4 * static_cast<size_t>(z.S) * z.H);
    w.bytes = off;
    return w;
}

}  // namespace mlora

using namespace mlora;

extern "C" {

const char* mlora_status_string(mlora_status status) {
    switch (status) {
        case MLORA_OK: return "ok";
        case MLORA_ERR_INVALID_ARG: return "invalid argument";
        case MLORA_ERR_SHAPE: return "invalid shape";
        case MLORA_ERR_UNSUPPORTED: return "unsupported configuration";
        case MLORA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MLORA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

mlora_status mlora_moe_route(const float* logits, const float* bias, int M, int E, int top_k, int scoring,
                             int renormalize, int n_shared, float routed_scaling_factor, int32_t* topk_ids,
                             float* topk_w, void* stream) {
    if (scoring != MLORA_SCORE_SOFTMAX && scoring != MLORA_SCORE_SIGMOID_BIAS) return MLORA_ERR_INVALID_ARG;
    if (M < 0 || E < 1 || E > MLORA_MAX_EXPERTS || top_k < 1 || top_k > E || n_shared < 0 ||
        top_k + n_shared > MLORA_MAX_TOPK)
        return MLORA_ERR_SHAPE;
    if (n_shared > 0 && !(routed_scaling_factor > 0.0f)) return MLORA_ERR_INVALID_ARG;
    if (M == 0) return MLORA_OK;
    if (!logits || !topk_ids || !topk_w) return MLORA_ERR_INVALID_ARG;
    if (foreign_device_memory(static_cast<cudaStream_t>(stream), {logits, bias, topk_ids, topk_w}))
        return MLORA_ERR_INVALID_ARG;
    const float inv_rsf = n_shared > 0 ? 1.0f / routed_scaling_factor : 0.0f;
    return cuda_status(launch_route(logits, scoring == MLORA_SCORE_SIGMOID_BIAS ? bias : nullptr, M, E, top_k,
                                    scoring, renormalize, n_shared, inv_rsf, topk_ids, topk_w,
                                    static_cast<cudaStream_t>(stream)));
}

size_t mlora_moe_align_max_padded(int M, int K_total, int E_tot, int block_m) {
    if (M < 0 || K_total < 1 || E_tot < 1 || block_m < 1 || block_m > MLORA_MAX_ALIGN_BLOCK) return 0;
    return static_cast<size_t>(align_max_padded(static_cast<long>(M) * K_total, E_tot, block_m));
}

mlora_status mlora_moe_align(const int32_t* topk_ids, int M, int K_total, int E_tot, int block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded, void* stream) {
    if (M < 0 || K_total < 1 || K_total > MLORA_MAX_TOPK || E_tot < 1 || E_tot > MLORA_MAX_EXPERTS ||
        block_m < 1 || block_m > MLORA_MAX_ALIGN_BLOCK)
        return MLORA_ERR_SHAPE;
    const long S = static_cast<long>(M) * K_total;
    if (S + static_cast<long>(E_tot) * block_m >= 0x7fffffffL) return MLORA_ERR_SHAPE;
    if (!num_post_padded || (S > 0 && (!topk_ids || !sorted_ids || !expert_ids))) return MLORA_ERR_INVALID_ARG;
    if (foreign_device_memory(static_cast<cudaStream_t>(stream), {topk_ids, sorted_ids, expert_ids, num_post_padded}))
        return MLORA_ERR_INVALID_ARG;
    const long mp = align_max_padded(S, E_tot, block_m);
    return cuda_status(launch_align(topk_ids, S, E_tot, block_m, mp, sorted_ids, expert_ids, num_post_padded,
                                    nullptr, nullptr, static_cast<cudaStream_t>(stream)));
}

static mlora_status check_forward_sizes(int M, int H, int I, int E_tot, int K_total, int L, int rank,
                                        bool mx = false) {
    if (M < 0 || H < 8 || I < 8 || (H % 8) || (I % 8) || E_tot < 1 || E_tot > MLORA_MAX_EXPERTS || K_total < 1 ||
        K_total > MLORA_MAX_TOPK || L < 0 || rank < 0)
        return MLORA_ERR_SHAPE;
    if (mx && (H % kMxBlock || I % kMxBlock)) return MLORA_ERR_SHAPE;
    if (L > 0 && rank > 0 && (rank % 8 || rank > MLORA_MAX_RANK)) return MLORA_ERR_UNSUPPORTED;
    const long S = static_cast<long>(M) * K_total;
    if (S + static_cast<long>(E_tot) * kBlockM >= 0x7fffffffL) return MLORA_ERR_SHAPE;
    if (static_cast<long>(L) * E_tot >= 0x7fffffffL) return MLORA_ERR_SHAPE;
    const Sizes z = make_sizes(M, H, I, E_tot, K_total, L, rank, mx);
    if (z.max_lt * kBlockM >= 0x7fffffffL) return MLORA_ERR_SHAPE;
    return MLORA_OK;
}

size_t mlora_moe_workspace_size(int M, int H, int I, int E_tot, int K_total, int L, int rank) {
    if (check_forward_sizes(M, H, I, E_tot, K_total, L, rank) != MLORA_OK) return 0;
    return carve_workspace(make_sizes(M, H, I, E_tot, K_total, L, rank), nullptr).bytes;
}

size_t mlora_moe_workspace_size_mxfp8(int M, int H, int I, int E_tot, int K_total, int L, int rank) {
    if (check_forward_sizes(M, H, I, E_tot, K_total, L, rank, true) != MLORA_OK) return 0;
    return carve_workspace(make_sizes(M, H, I, E_tot, K_total, L, rank, true), nullptr).bytes;
}

size_t mlora_mxfp8_scales_size(int E_tot, int H, int I, int which) {
    if (E_tot < 1 || E_tot > MLORA_MAX_EXPERTS || H < kMxBlock || I < kMxBlock || H % kMxBlock || I % kMxBlock ||
        (which != 0 && which != 1))
        return 0;
    return static_cast<size_t>(E_tot) * mx_slabs(which, H, I) * mx_chunks(which, H, I) * kMxTileScaleBytes;
}

mlora_status mlora_mxfp8_quantize_weights(const void* w13, const void* w2, int E_tot, int H, int I, void* w13_q,
                                          void* w13_s, void* w2_q, void* w2_s, void* stream) {
    const size_t s13 = mlora_mxfp8_scales_size(E_tot, H, I, 0), s2 = mlora_mxfp8_scales_size(E_tot, H, I, 1);
    if (!s13 || !s2) return MLORA_ERR_SHAPE;
    const void* ptrs[] = {w13, w2, w13_q, w13_s, w2_q, w2_s};
    for (const void* ptr : ptrs)
        if (!ptr || !aligned16(ptr)) return MLORA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (foreign_device_memory(s, {w13, w2, w13_q, w13_s, w2_q, w2_s})) return MLORA_ERR_INVALID_ARG;
    cudaError_t err;
    // bytes of the packed scales that no weight row fills (ragged last slab
    // or K-chunk) read as 2^-127
    if ((err = cudaMemsetAsync(w13_s, 0, s13, s)) != cudaSuccess) return cuda_fail(err, "scales");
    if ((err = cudaMemsetAsync(w2_s, 0, s2, s)) != cudaSuccess) return cuda_fail(err, "scales");
    err = launch_mx_quantize_weights(w13, 2L * I * E_tot, H, 0, H, I, static_cast<uint8_t*>(w13_q),
                                     static_cast<uint8_t*>(w13_s), s);
    if (err != cudaSuccess) return cuda_fail(err, "quantize w13");
    err = launch_mx_quantize_weights(w2, static_cast<long>(H) * E_tot, I, 1, H, I, static_cast<uint8_t*>(w2_q),
                                     static_cast<uint8_t*>(w2_s), s);
    if (err != cudaSuccess) return cuda_fail(err, "quantize w2");
    return MLORA_OK;
}

namespace {

// MXFP8 expert weights of a forward (null: the bf16 layer).
struct MxWeights {
    const void* w13_q;
    const void* w13_s;
    const void* w2_q;
    const void* w2_s;
};

mlora_status forward_impl(const void* x, const void* w13, const void* w2, const MxWeights* mxw, const void* A13,
                          const void* B13, const void* A2, const void* B2, const int32_t* token_lora_idx,
                          const int32_t* topk_ids, const float* topk_w, int M, int H, int I, int E_tot, int K_total,
                          int L, int rank, float scaling, int n_shared, float out_scale, void* y, void* workspace,
                          size_t workspace_bytes, void* stream) {
    const bool mx = mxw != nullptr;
    const bool lora = A13 && B13 && A2 && B2 && token_lora_idx && L > 0 && rank > 0;
    const int L_eff = lora ? L : 0, r_eff = lora ? rank : 0;
    mlora_status st = check_forward_sizes(M, H, I, E_tot, K_total, L, rank, mx);
    if (st != MLORA_OK) return st;
    if (n_shared < 0 || n_shared >= K_total || n_shared >= E_tot) return MLORA_ERR_SHAPE;
    if (M == 0) return MLORA_OK;
    if (mx) {
        w13 = mxw->w13_q;
        w2 = mxw->w2_q;
        if (!mxw->w13_s || !mxw->w2_s || !aligned16(mxw->w13_s) || !aligned16(mxw->w2_s))
            return MLORA_ERR_INVALID_ARG;
    }
    if (!x || !w13 || !w2 || !topk_ids || !topk_w || !y) return MLORA_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w13, w2, topk_ids, topk_w, y};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return MLORA_ERR_INVALID_ARG;
    if (lora) {
        const void* lp[] = {A13, B13, A2, B2};
        for (const void* ptr : lp)
            if (!aligned16(ptr)) return MLORA_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(token_lora_idx) & 3u) return MLORA_ERR_INVALID_ARG;
    }
    if (foreign_device_memory(static_cast<cudaStream_t>(stream),
                              {x, w13, w2, topk_ids, topk_w, y, workspace, lora ? A13 : nullptr,
                               lora ? token_lora_idx : nullptr, mx ? mxw->w13_s : nullptr}))
        return MLORA_ERR_INVALID_ARG;
    Sizes z = make_sizes(M, H, I, E_tot, K_total, L_eff, r_eff, mx);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MLORA_ERR_WORKSPACE;
    const Workspace ws = carve_workspace(z, workspace);
    if (workspace_bytes < ws.bytes) return MLORA_ERR_WORKSPACE;

    // ---- tensor maps (dims innermost first) ----
    GemmParams gp{};
    // tile widths and shrink group size: tuned table or rules (the group
    // size does not change the workspace layout)
    resolve_tiles(H, I, E_tot, K_total, r_eff, mx, gp.width_table, &z.gsize);
    GemmSide& up = gp.side[0];
    GemmSide& dn = gp.side[1];
    const cuuint64_t H_ = H, I_ = I, E_ = E_tot, MP = z.max_padded;
    bool ok = true;
    {
        const cuuint32_t bx[2] = {64, kRowBox};
        const cuuint32_t bxf[2] = {64, 128};
        // a gate_up tile of width n takes n/2 gate and n/2 up rows (one box
        // over both halves: gate rows, then up rows), a down tile n rows.
        // CTA pairs (256-row tiles only) load one half per CTA: width class
        // 1's slot holds that 128-row half box instead.
        cuuint32_t b13[kTileWidths][4], b2[kTileWidths][3];
        for (int wc = 0; wc < kTileWidths; ++wc) {
            const cuuint32_t n = static_cast<cuuint32_t>(tile_width(wc));
            b13[wc][0] = 64, b13[wc][1] = n / 2, b13[wc][2] = 2, b13[wc][3] = 1;
            b2[wc][0] = 64, b2[wc][1] = n, b2[wc][2] = 1;
        }
        if (z.pair) b13[1][1] = 128, b13[1][2] = 1;
        if (ws.x_perm) {
            const cuuint64_t dx[2] = {H_, MP}, sx[1] = {H_ * 2};
            ok &= make_map(&up.tm_a, ws.x_perm, 2, dx, sx, bx);
            ok &= make_map(&up.tm_a_full, ws.x_perm, 2, dx, sx, bxf);
            const cuuint64_t da[2] = {I_, MP}, sa[1] = {I_ * 2};
            ok &= make_map(&dn.tm_a, ws.act, 2, da, sa, bx);
            ok &= make_map(&dn.tm_a_full, ws.act, 2, da, sa, bxf);
        }
        if (mx) {
            const cuuint32_t qb[2] = {kMxChunk, kRowBox}, qbf[2] = {kMxChunk, 128};
            const cuuint64_t dx[2] = {H_, MP}, sx[1] = {H_};
            ok &= make_map_u8(&up.tm_ax, ws.x_q, 2, dx, sx, qb);
            ok &= make_map_u8(&up.tm_ax_full, ws.x_q, 2, dx, sx, qbf);
            const cuuint64_t da[2] = {I_, MP}, sa[1] = {I_};
            ok &= make_map_u8(&dn.tm_ax, ws.act_q, 2, da, sa, qb);
            ok &= make_map_u8(&dn.tm_ax_full, ws.act_q, 2, da, sa, qbf);
            const cuuint64_t d13[4] = {H_, I_, 2, E_}, s13[3] = {H_, I_ * H_, 2 * I_ * H_};
            const cuuint32_t q13[4] = {kMxChunk, kMxHalf, 2, 1};
            ok &= make_map_u8(&up.tm_bx, w13, 4, d13, s13, q13);
            const cuuint64_t d2[3] = {I_, H_, E_}, s2[2] = {I_, H_ * I_};
            const cuuint32_t q2[3] = {kMxChunk, kMxWidth, 1};
            ok &= make_map_u8(&dn.tm_bx, w2, 3, d2, s2, q2);
        } else {
            const cuuint64_t d13[4] = {H_, I_, 2, E_}, s13[3] = {H_ * 2, I_ * H_ * 2, 2 * I_ * H_ * 2};
            const cuuint64_t d2[3] = {I_, H_, E_}, s2[2] = {I_ * 2, H_ * I_ * 2};
            for (int wc = 0; wc < kTileWidths; ++wc) {
                ok &= make_map(&up.tm_b[wc], w13, 4, d13, s13, b13[wc]);
                ok &= make_map(&dn.tm_b[wc], w2, 3, d2, s2, b2[wc]);
            }
        }
        if (z.pair && !mx) {
            // CTA pairs: two K-chunks of 64 per copy, through views with a
            // chunk dimension of stride 128 B over the whole chunks of K
            // (at least two of them; otherwise every stage uses the 2D maps)
            const cuuint32_t bxc[3] = {64, 128, 2};
            if (H_ / 64 >= 2) {
                const cuuint64_t dx[3] = {64, MP, H_ / 64}, sx[2] = {H_ * 2, 128};
                ok &= make_map(&up.tm_ax_full, ws.x_perm, 3, dx, sx, bxc);
                const cuuint64_t dw[5] = {64, I_, 2, E_, H_ / 64}, sw[4] = {H_ * 2, I_ * H_ * 2, 2 * I_ * H_ * 2, 128};
                const cuuint32_t bw[5] = {64, 128, 1, 1, 2};
                ok &= make_map(&up.tm_bx, w13, 5, dw, sw, bw);
            }
            if (I_ / 64 >= 2) {
                const cuuint64_t da[3] = {64, MP, I_ / 64}, sa[2] = {I_ * 2, 128};
                ok &= make_map(&dn.tm_ax_full, ws.act, 3, da, sa, bxc);
                const cuuint64_t dw[4] = {64, H_, E_, I_ / 64}, sw[3] = {I_ * 2, H_ * I_ * 2, 128};
                const cuuint32_t bw[4] = {64, 128, 1, 2};
                ok &= make_map(&dn.tm_bx, w2, 4, dw, sw, bw);
            }
        }
        if (lora) {
            const cuuint64_t R = rank, LE = static_cast<cuuint64_t>(L) * E_tot;
            const cuuint32_t rp = static_cast<cuuint32_t>((rank + 15) / 16 * 16);
            const cuuint64_t dt[2] = {64, static_cast<cuuint64_t>(z.max_lt) * kBlockM}, st_[1] = {128};
            ok &= make_map(&up.tm_t, ws.lora_t13, 2, dt, st_, bx);
            ok &= make_map(&up.tm_t_full, ws.lora_t13, 2, dt, st_, bxf);
            ok &= make_map(&dn.tm_t, ws.lora_t2, 2, dt, st_, bx);
            ok &= make_map(&dn.tm_t_full, ws.lora_t2, 2, dt, st_, bxf);
            // shrink weights: rank rows past the rank read as zero
            const cuuint64_t dA13[3] = {H_, R, LE}, sA13[2] = {H_ * 2, R * H_ * 2};
            const cuuint32_t bA[3] = {64, rp, 1};
            ok &= make_map(&up.tm_sa, A13, 3, dA13, sA13, bA);
            const cuuint64_t dA2[3] = {I_, R, LE}, sA2[2] = {I_ * 2, R * I_ * 2};
            ok &= make_map(&dn.tm_sa, A2, 3, dA2, sA2, bA);
            // expand weights: columns past the rank read as zero
            const cuuint64_t dB13[4] = {R, I_, 2, LE}, sB13[3] = {R * 2, I_ * R * 2, 2 * I_ * R * 2};
            const cuuint64_t dB2[3] = {R, H_, LE}, sB2[2] = {R * 2, H_ * R * 2};
            for (int wc = 0; wc < kTileWidths; ++wc) {
                ok &= make_map(&up.tm_lb[wc], B13, 4, dB13, sB13, b13[wc]);
                ok &= make_map(&dn.tm_lb[wc], B2, 3, dB2, sB2, b2[wc]);
            }
        }
    }
    if (!ok) return cuda_fail(cudaErrorInvalidValue, "tensor map encoding");

    up.lora_t = ws.lora_t13;
    up.done = ws.done13;
    up.out = ws.act;
    up.K = H;
    up.n_out = I;
    up.ncb = (I + 127) / 128;
    dn.lora_t = ws.lora_t2;
    dn.done = ws.done2;
    dn.out = ws.y_slot;
    dn.K = I;
    dn.n_out = H;
    dn.ncb = (H + 255) / 256;
    if (mx) {
        up.a_scales = ws.x_s;
        up.b_scales = static_cast<const uint8_t*>(mxw->w13_s);
        up.out_q = ws.act_q;
        up.out_s = ws.act_s;
        up.nkc = z.nkc0;
        dn.a_scales = ws.act_s;
        dn.b_scales = static_cast<const uint8_t*>(mxw->w2_s);
        dn.nkc = z.nkc1;
    }
    gp.mx = mx ? 1 : 0;
    gp.pair = z.pair ? 1 : 0;
    gp.n_pad = ws.n_pad;
    gp.expert_ids = ws.expert_ids;
    gp.blk_rows = ws.blk_rows;
    gp.sorted_ids = ws.sorted_ids;
    gp.lora_of = ws.lora_of;
    gp.blk_nad = ws.blk_nad;
    gp.blk_lora = ws.blk_lora;
    gp.blk_lt_start = ws.blk_lt_start;
    gp.gt_block = ws.gt_block;
    gp.gt_first = ws.gt_first;
    gp.gt_total = ws.gt_total;
    gp.act_done = ws.act_done;
    gp.lt_cap = z.max_lt;
    gp.pad_cap = z.max_padded;
    gp.tile_next = ws.tile_next;
    gp.max_rows = ws.max_rows;
    gp.status = ws.status;
    gp.wait_limit = g_wait_limit;
    // the never-set flag: a header word that the reset clears and nothing writes
    gp.stall_flag = g_stall_test ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(ws.status) + 24)
                                 : nullptr;
    gp.E_tot = E_tot;
    gp.cap = z.cap;
    gp.gsize = z.gsize;
    gp.rank = r_eff;
    gp.S = static_cast<int>(z.S);
    gp.has_lora = lora ? 1 : 0;
    gp.scaling = scaling;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if ((err = mark_stage(0, s)) != cudaSuccess) return cuda_fail(err, "stage event");
    AlignExtra ex{};
    // the align kernel clears the header and the counters itself (no
    // memset node between the caller's route and align)
    ex.zero = ws.status;
    ex.zero_words = static_cast<int>(ws.zeroed_bytes / 4);
    ex.lt_cap = z.max_lt;
    ex.max_rows = ws.max_rows;
    ex.blk_rows = ws.blk_rows;
    ex.pair_pad = z.pair ? 1 : 0;
    if (lora) {
        ex.token_lora_idx = token_lora_idx;
        ex.L = L;
        ex.K_total = K_total;
        ex.cap = z.cap;
        ex.lora_of = ws.lora_of;
        ex.blk_nad = ws.blk_nad;
        ex.blk_lora = ws.blk_lora;
        ex.blk_lt_start = ws.blk_lt_start;
        ex.gsize = z.gsize;
        ex.gt_block = ws.gt_block;
        ex.gt_first = ws.gt_first;
        ex.gt_total = ws.gt_total;
    }
    if (align_small_fits(z.S, E_tot, kBlockM, z.max_padded, &ex, true)) {
        // small batches: align and the row gather in one launch (stage
        // boundaries 1 and 2 coincide)
        const GatherArgs ga{x, ws.x_perm, H, K_total, ws.x_q, ws.x_s};
        err = launch_align_small(topk_ids, z.S, E_tot, kBlockM, z.max_padded, ws.sorted_ids, ws.expert_ids,
                                 ws.n_pad, ws.status, &ex, &ga, s);
        if (err != cudaSuccess) return cuda_fail(err, "align + gather");
        if ((err = mark_stage(1, s)) != cudaSuccess) return cuda_fail(err, "stage event");
    } else {
        err = launch_align(topk_ids, z.S, E_tot, kBlockM, z.max_padded, ws.sorted_ids, ws.expert_ids, ws.n_pad,
                           ws.status, &ex, s);
        if (err != cudaSuccess) return cuda_fail(err, "align");
        if ((err = mark_stage(1, s)) != cudaSuccess) return cuda_fail(err, "stage event");
        if (mx)
            err = launch_mx_gather(x, H, K_total, ws.sorted_ids, ws.n_pad, z.S, z.max_padded, ws.x_q, ws.x_s,
                                   ws.x_perm, ws.status, s);
        else
            err = launch_gather_rows(x, H, ws.sorted_ids, ws.n_pad, z.S, K_total, z.max_padded, ws.x_perm,
                                     ws.status, s);
        if (err != cudaSuccess) return cuda_fail(err, "gather");
    }
    if ((err = mark_stage(2, s)) != cudaSuccess) return cuda_fail(err, "stage event");
    // narrow tiles (half width) at most double the slab count
    const long max_tiles = 2 * z.max_lt + z.max_blocks * (2L * up.ncb + 2L * dn.ncb);
    err = launch_experts(gp, max_tiles, s);
    if (err != cudaSuccess) return cuda_fail(err, "experts");
    if ((err = mark_stage(3, s)) != cudaSuccess) return cuda_fail(err, "stage event");
    err = launch_combine(ws.y_slot, topk_ids, topk_w, M, H, K_total, E_tot, out_scale, y, s);
    if (err != cudaSuccess) return cuda_fail(err, "combine");
    if ((err = mark_stage(4, s)) != cudaSuccess) return cuda_fail(err, "stage event");
    return MLORA_OK;
}

}  // namespace

mlora_status mlora_moe_forward(const void* x, const void* w13, const void* w2, const void* A13, const void* B13,
                               const void* A2, const void* B2, const int32_t* token_lora_idx,
                               const int32_t* topk_ids, const float* topk_w, int M, int H, int I, int E_tot,
                               int K_total, int L, int rank, float scaling, int n_shared, float out_scale, void* y,
                               void* workspace, size_t workspace_bytes, void* stream) {
    return forward_impl(x, w13, w2, nullptr, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, M, H, I, E_tot,
                        K_total, L, rank, scaling, n_shared, out_scale, y, workspace, workspace_bytes, stream);
}

mlora_status mlora_moe_forward_mxfp8(const void* x, const void* w13_q, const void* w13_s, const void* w2_q,
                                     const void* w2_s, const void* A13, const void* B13, const void* A2,
                                     const void* B2, const int32_t* token_lora_idx, const int32_t* topk_ids,
                                     const float* topk_w, int M, int H, int I, int E_tot, int K_total, int L,
                                     int rank, float scaling, int n_shared, float out_scale, void* y,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    const MxWeights mxw{w13_q, w13_s, w2_q, w2_s};
    return forward_impl(x, nullptr, nullptr, &mxw, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, M, H, I,
                        E_tot, K_total, L, rank, scaling, n_shared, out_scale, y, workspace, workspace_bytes,
                        stream);
}

mlora_status mlora_set_stage_events(void* const* events, int count) {
    if (!events || count == 0) {
        g_stage_events_on = false;
        return MLORA_OK;
    }
    if (count < MLORA_STAGE_EVENTS) return MLORA_ERR_INVALID_ARG;
    for (int i = 0; i < MLORA_STAGE_EVENTS; ++i) {
        if (!events[i]) return MLORA_ERR_INVALID_ARG;
        g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    g_stage_events_on = true;
    return MLORA_OK;
}

mlora_status mlora_set_pair_mode(int on) {
    if (on != 0 && on != 1) return MLORA_ERR_INVALID_ARG;
    g_pair_mode = on != 0;
    return MLORA_OK;
}

int mlora_pair_mode(void) { return g_pair_mode ? 1 : 0; }

mlora_status mlora_set_tile_config(int width_class, int gsize) {
    if (width_class < -1 || width_class >= kTileWidths || gsize < 0 || gsize > 4) return MLORA_ERR_INVALID_ARG;
    g_force_wc = width_class;
    g_force_gsize = gsize;
    return MLORA_OK;
}

mlora_status mlora_tile_config(int H, int I, int E_tot, int K_total, int rank, int nblocks, int grid,
                               int* width_class, int* gsize, int* tuned) {
    if (!width_class || !gsize || H < 8 || I < 8 || E_tot < 1 || K_total < 1 || rank < 0 || nblocks < 1 || grid < 1)
        return MLORA_ERR_INVALID_ARG;
    const Sizes z = make_sizes(1, H, I, E_tot, K_total, rank > 0 ? 1 : 0, rank);
    int8_t table[kWidthBuckets];
    int g = z.gsize;
    const bool t = resolve_tiles(H, I, E_tot, K_total, rank, false, table, &g);
    const int tw = table[width_bucket(nblocks)];
    *width_class = tw >= 0 ? tw : choose_width(nblocks, I, H, grid);
    *gsize = g;
    if (tuned) *tuned = t ? 1 : 0;
    return MLORA_OK;
}

mlora_status mlora_set_wait_test(long long wait_limit_cycles, int stall) {
    if (wait_limit_cycles < 0) return MLORA_ERR_INVALID_ARG;
    g_wait_limit = wait_limit_cycles == 0 ? kWaitCycles : wait_limit_cycles;
    g_stall_test = stall != 0;
    return MLORA_OK;
}

mlora_status mlora_moe_read_status(const void* workspace, uint32_t* host_status, void* stream) {
    if (!workspace || !host_status) return MLORA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MLORA_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

}  // extern "C"
