// gemm.cu -- the grouped expert GEMMs on the 5th-generation tensor cores.
//
// One persistent, warp-specialised kernel template serves three products
// over blocks of kBlockM = 128 sorted slots (all slots of a block share one
// expert e, from align):
//
//  kGateUp: h = X W13_e^T over a 128-column slab j0.. of the gate rows and
//           the same slab of the up rows (one MMA with N = 256: B rows 0..127
//           gate, 128..255 up), then, per adapter l present in the block,
//           h += T_l B13_{l,e}^T as extra K-chunks into the same TMEM
//           accumulator (the LoRA expand folded into the projection,
//           "Amazon SageMaker 및 Amazon Bedrock에서 vLLM을 활용한 MoE 모델
//           Multi-LoRA 서빙 최적화", section "섹션별 상세" paragraphs 1 and 3);
//           epilogue: act = silu(gate) * up -> bf16.
//  kDown:   d = act W2_e^T over 256 output columns, + T2_l B2_{l,e}^T chunks;
//           epilogue: bf16 row of the slot's expert output.
//  kShrink: t = X A_{l,e}^T for one (block, adapter) pair, N = rank rounded
//           up to 16; epilogue: the masked, scaled shrink tile T_l (rows of
//           other adapters zero, columns past the rank zero) in bf16.
//
// Roles (192 threads): warp 0 issues TMA loads into a ring of smem stages
// (A tile 128 x 64 bf16: one 128-row box for a full block, 32-row boxes
// covering only the real rows of a partial one; B tile N x 64 bf16; both
// K-major with 128-byte swizzle); warp 1 allocates TMEM and one lane issues tcgen05.mma (M = 128,
// K = 16 per instruction, fp32 accumulate) and tcgen05.commit; warps 2..5
// drain the double-buffered TMEM accumulator with tcgen05.ld while the next
// tile's MMAs run.  Tiles are strided over a grid of at most one CTA per SM.
// Every mbarrier wait is bounded (ptx.cuh).
#include "internal.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kThreads = 192;
constexpr int kATileBytes = kBlockM * kBlockK * 2;  // 16 KiB

template <int MODE>
struct Cfg {
    static constexpr int kStages = 4;
    static constexpr int kBRows = 256;
    static constexpr int kAccCols = 256;
    static constexpr int kTmemCols = 512;
};
template <>
struct Cfg<kShrink> {
    static constexpr int kStages = 6;
    static constexpr int kBRows = 64;
    static constexpr int kAccCols = 64;
    static constexpr int kTmemCols = 128;
};

template <int MODE>
constexpr int stage_bytes() {
    return kATileBytes + Cfg<MODE>::kBRows * kBlockK * 2;
}

template <int MODE>
constexpr int smem_bytes() {
    return Cfg<MODE>::kStages * stage_bytes<MODE>() + 1024 /* alignment slack */ + 256 /* barriers */;
}

// Bounded wait used only while unwinding after an abort: ignores the abort
// flag so that copies already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    int zero = 0;
    mbar_wait(bar, parity, &zero, nullptr, kWaitCycles / 8);
}

struct TileCoord {
    int b;   // block of kBlockM sorted positions
    int cb;  // column slab
    int e;   // expert
    int l;   // adapter (shrink only)
};

template <int MODE>
__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, long tile, int ncb) {
    TileCoord c;
    if (MODE == kShrink) {
        c.b = p.lt_block[tile];
        c.l = p.lt_lora[tile];
        c.cb = 0;
    } else {
        c.b = static_cast<int>(tile / ncb);
        c.cb = static_cast<int>(tile - static_cast<long>(c.b) * ncb);
        c.l = -1;
    }
    c.e = p.expert_ids[c.b];
    return c;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    using C = Cfg<MODE>;
    constexpr int kStages = C::kStages;
    constexpr int kStageBytes = stage_bytes<MODE>();

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tensormap(&p.tm_a);
        prefetch_tensormap(&p.tm_a_full);
        prefetch_tensormap(&p.tm_b);
        if (MODE != kShrink && p.has_lora) {
            prefetch_tensormap(&p.tm_t);
            prefetch_tensormap(&p.tm_t_full);
            prefetch_tensormap(&p.tm_lb);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::kTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Everything above overlapped the previous kernel.  With a shrink as the
    // previous kernel (pdl_early) only its shrink tiles are needed, and only
    // by the expand stages: the producer waits for it there, while the base
    // product (whose inputs were complete before the shrink started) runs.
    if (!p.pdl_early) griddep_wait();

    const int nblocks = *p.n_pad / kBlockM;
    int ncb = 1;
    long ntiles;
    if (MODE == kGateUp) {
        ncb = (p.n_out + 127) / 128;
        ntiles = static_cast<long>(nblocks) * ncb;
    } else if (MODE == kDown) {
        ncb = (p.n_out + 255) / 256;
        ntiles = static_cast<long>(nblocks) * ncb;
    } else {
        ntiles = *p.lt_total;
    }
    const int nk = (p.K + kBlockK - 1) / kBlockK;
    const int rp = (p.rank + 15) / 16 * 16;       // shrink N
    const int lora_ksteps = (p.rank + 15) / 16;   // expand K-steps of 16
    const bool expand = MODE != kShrink && p.has_lora;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            long it = 0;
            bool ok = true;
            bool waited = false;
            for (long tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TileCoord tc = decode_tile<MODE>(p, tile, ncb);
                const int row0 = tc.b * kBlockM;
                // only the block's real rows are loaded; the MMA rows past
                // them hold stale data and feed only discarded output rows
                const int nbox = (p.blk_rows[tc.b] + kRowBox - 1) / kRowBox;
                const bool full_block = nbox * kRowBox == kBlockM;
                const uint32_t a_bytes = static_cast<uint32_t>(nbox) * kRowBox * kBlockK * 2;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + s * kStageBytes;
                    uint8_t* sb = sa + kATileBytes;
                    const int k0 = kb * kBlockK;
                    if (MODE == kGateUp) {
                        mbar_arrive_expect_tx(&full[s], a_bytes + 2 * 128 * kBlockK * 2);
                        tma_load_4d(sb, &p.tm_b, &full[s], k0, tc.cb * 128, 0, tc.e);
                        tma_load_4d(sb + 128 * kBlockK * 2, &p.tm_b, &full[s], k0, tc.cb * 128, 1, tc.e);
                    } else if (MODE == kDown) {
                        mbar_arrive_expect_tx(&full[s], a_bytes + 256 * kBlockK * 2);
                        tma_load_3d(sb, &p.tm_b, &full[s], k0, tc.cb * 256, tc.e);
                    } else {
                        mbar_arrive_expect_tx(&full[s], a_bytes + rp * kBlockK * 2);
                        tma_load_3d(sb, &p.tm_b, &full[s], k0, 0, tc.l * p.E_tot + tc.e);
                    }
                    if (full_block)
                        tma_load_2d(sa, &p.tm_a_full, &full[s], k0, row0);
                    else
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d(sa + i * kRowBox * kBlockK * 2, &p.tm_a, &full[s], k0, row0 + i * kRowBox);
                }
                if (!ok || !expand) continue;
                const int nad = p.blk_nad[tc.b];
                const int lt0 = p.blk_lt_start[tc.b];
                if (p.pdl_early && nad > 0 && !waited) {
                    griddep_wait();  // the shrink tiles are complete from here on
                    waited = true;
                }
                for (int i = 0; i < nad; ++i, ++it) {
                    const int l = p.blk_lora[static_cast<long>(tc.b) * p.cap + i];
                    const int s = static_cast<int>(it % kStages);
                    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + s * kStageBytes;
                    uint8_t* sb = sa + kATileBytes;
                    const int le = l * p.E_tot + tc.e;
                    if (MODE == kGateUp) {
                        mbar_arrive_expect_tx(&full[s], a_bytes + 2 * 128 * kBlockK * 2);
                        tma_load_4d(sb, &p.tm_lb, &full[s], 0, tc.cb * 128, 0, le);
                        tma_load_4d(sb + 128 * kBlockK * 2, &p.tm_lb, &full[s], 0, tc.cb * 128, 1, le);
                    } else {
                        mbar_arrive_expect_tx(&full[s], a_bytes + 256 * kBlockK * 2);
                        tma_load_3d(sb, &p.tm_lb, &full[s], 0, tc.cb * 256, le);
                    }
                    if (full_block)
                        tma_load_2d(sa, &p.tm_t_full, &full[s], 0, (lt0 + i) * kBlockM);
                    else
                        for (int j = 0; j < nbox; ++j)
                            tma_load_2d(sa + j * kRowBox * kBlockK * 2, &p.tm_t, &full[s], 0,
                                        (lt0 + i) * kBlockM + j * kRowBox);
                }
            }
            if (!ok) {
                for (long j = it > kStages ? it - kStages : 0; j < it; ++j)
                    drain_wait(&full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(128, MODE == kShrink ? rp : 256);
            long it = 0;
            int lt = 0;
            bool ok = true;
            for (long tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++lt) {
                const TileCoord tc = decode_tile<MODE>(p, tile, ncb);
                const int acc = lt & 1;
                if (!mbar_wait(&tempty[acc], (static_cast<uint32_t>(lt >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    if (!mbar_wait(&full[s], static_cast<uint32_t>(it / kStages) & 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * kStageBytes);
                    const uint64_t ad = umma_desc_sw128(a_addr);
                    const uint64_t bd = umma_desc_sw128(a_addr + kATileBytes);
#pragma unroll
                    for (int k = 0; k < kBlockK / 16; ++k)
                        umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                if (!ok) break;
                if (expand) {
                    const int nad = p.blk_nad[tc.b];
                    for (int i = 0; i < nad; ++i, ++it) {
                        const int s = static_cast<int>(it % kStages);
                        if (!mbar_wait(&full[s], static_cast<uint32_t>(it / kStages) & 1u, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + s * kStageBytes);
                        const uint64_t ad = umma_desc_sw128(a_addr);
                        const uint64_t bd = umma_desc_sw128(a_addr + kATileBytes);
                        for (int k = 0; k < lora_ksteps; ++k) umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, 1u);
                        umma_commit(&empty[s]);
                    }
                    if (!ok) break;
                }
                umma_commit(&tfull[acc]);
            }
            // every MMA issued above completes before TMEM is released
            umma_commit(drain);
            drain_wait(drain, 0);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int lt = 0;
        for (long tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
            const TileCoord tc = decode_tile<MODE>(p, tile, ncb);
            const int acc = lt & 1;
            if (!mbar_wait(&tfull[acc], static_cast<uint32_t>(lt >> 1) & 1u, abort_flag, p.status)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * C::kAccCols) +
                                (static_cast<uint32_t>(q * 32) << 16);
            const int prow = tc.b * kBlockM + row;
            if (MODE == kGateUp) {
                const bool real = p.sorted_ids[prow] < p.S;
                const int j0 = tc.cb * 128;
                __nv_bfloat16* act = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(prow) * p.n_out;
                for (int c = 0; c < 128; c += 32) {
                    if (j0 + c >= p.n_out) break;
                    float g[32], u[32];
                    tmem_ld32(tb + c, g);
                    tmem_ld32(tb + 128 + c, u);
                    if (real) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int col = j0 + c + 8 * v;
                            if (col < p.n_out) {
                                uint4 o;
                                o.x = pack_bf16x2(silu(g[8 * v + 0]) * u[8 * v + 0], silu(g[8 * v + 1]) * u[8 * v + 1]);
                                o.y = pack_bf16x2(silu(g[8 * v + 2]) * u[8 * v + 2], silu(g[8 * v + 3]) * u[8 * v + 3]);
                                o.z = pack_bf16x2(silu(g[8 * v + 4]) * u[8 * v + 4], silu(g[8 * v + 5]) * u[8 * v + 5]);
                                o.w = pack_bf16x2(silu(g[8 * v + 6]) * u[8 * v + 6], silu(g[8 * v + 7]) * u[8 * v + 7]);
                                *reinterpret_cast<uint4*>(act + col) = o;
                            }
                        }
                    }
                }
            } else if (MODE == kDown) {
                const int f = p.sorted_ids[prow];
                const bool real = f < p.S;
                const int o0 = tc.cb * 256;
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(real ? f : 0) * p.n_out;
                for (int c = 0; c < 256; c += 32) {
                    if (o0 + c >= p.n_out) break;
                    float v[32];
                    tmem_ld32(tb + c, v);
                    if (real) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int col = o0 + c + 8 * j;
                            if (col < p.n_out) {
                                uint4 o;
                                o.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
                                o.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
                                o.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
                                o.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
                                *reinterpret_cast<uint4*>(dst + col) = o;
                            }
                        }
                    }
                }
            } else {
                const bool mine = p.lora_of[prow] == tc.l;
                __nv_bfloat16* dst =
                    static_cast<__nv_bfloat16*>(p.out) + (static_cast<size_t>(tile) * kBlockM + row) * kLoraTileCols;
                for (int c = 0; c < kLoraTileCols; c += 16) {
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                    if (c < rp) tmem_ld16(tb + c, v);
                    float o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = (mine && c + i < p.rank) ? p.scaling * v[i] : 0.f;
                    uint4 w0, w1;
                    w0.x = pack_bf16x2(o[0], o[1]);
                    w0.y = pack_bf16x2(o[2], o[3]);
                    w0.z = pack_bf16x2(o[4], o[5]);
                    w0.w = pack_bf16x2(o[6], o[7]);
                    w1.x = pack_bf16x2(o[8], o[9]);
                    w1.y = pack_bf16x2(o[10], o[11]);
                    w1.z = pack_bf16x2(o[12], o[13]);
                    w1.w = pack_bf16x2(o[14], o[15]);
                    reinterpret_cast<uint4*>(dst + c)[0] = w0;
                    reinterpret_cast<uint4*>(dst + c)[1] = w1;
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
    // the grid never completes before the one it follows, so whatever runs
    // after it may rely on both
    if (p.pdl_early) griddep_wait();
}

template <int MODE>
cudaError_t launch_mode(const GemmParams& p, long max_tiles, cudaStream_t s) {
    constexpr int smem = smem_bytes<MODE>();
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !((attr_done >> dev) & 1ull)) {
        err = cudaFuncSetAttribute(gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        attr_done |= 1ull << dev;
    }
    long grid = device_sm_count();
    if (grid > max_tiles) grid = max_tiles;
    return launch_pdl(gemm_kernel<MODE>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, s, p);
}

}  // namespace

cudaError_t launch_gemm(GemmMode mode, const GemmParams& p, long max_tiles, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    switch (mode) {
        case kGateUp: return launch_mode<kGateUp>(p, max_tiles, s);
        case kDown: return launch_mode<kDown>(p, max_tiles, s);
        default: return launch_mode<kShrink>(p, max_tiles, s);
    }
}

}  // namespace mlora
