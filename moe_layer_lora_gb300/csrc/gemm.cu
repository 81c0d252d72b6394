// gemm.cu -- the expert MLP of the layer on the 5th-generation tensor cores:
// both grouped GEMMs, their per-token LoRA shrink and expand, and SwiGLU,
// in one persistent kernel.
//
// The kernel works through four phases of tiles over blocks of kBlockM =
// 128 sorted slots (all slots of a block share one expert e, from align).
// Every CTA claims its tiles of the concatenated sequence from a global
// counter -- the first as it starts, each next one a few stages before the
// current tile's loads are all issued -- so tiles of unequal cost (shrink,
// gate_up, down, blocks with many adapters) spread evenly over the SMs:
//
//  1. gate_up shrink tiles (with adapters): T13_l = s * X A13_{l,e}^T for
//     up to `gsize` adapters l of one block at once -- their rank rows
//     stacked along N (N = g * rank rounded up to 16) -- written as one
//     masked bf16 tile per (block, adapter) (rows of other adapters and
//     columns past the rank zero); then the block's shrink counter is
//     bumped.
//  2. gate_up tiles: h = X W13_e^T over a 128-column slab of the gate rows
//     and the same slab of the up rows (one MMA with N = 256: B rows 0..127
//     gate, 128..255 up); with adapters, after the K loop, every adapter l
//     of the block adds T13_l B13_{l,e}^T as extra K-chunks into the same
//     TMEM accumulator -- the expand folded into the projection ("Amazon
//     SageMaker 및 Amazon Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA 서빙
//     최적화", section "섹션별 상세" paragraphs 1-3); epilogue act =
//     silu(g) * u in bf16, then the block's act counter is bumped.
//  3. down shrink tiles: T2_l = s * act A2_{l,e}^T, as in phase 1.
//  4. down tiles: d = act W2_e^T over 256 output columns + the T2 expand;
//     epilogue the slot's expert output in fp32.
// Batches with few blocks take tiles of 192 or 128 weight rows instead
// (N = 192 or 128; gate_up tiles half gate, half up rows) so that the
// tiles of each phase fill the grid's SMs.  Shrink tiles pack up to four
// 64-wide K-chunks per stage.
//
// A tile depends only on tiles of earlier phases of the same block, i.e.
// on tiles with smaller indices.  Every tile, a CTA's first included, is
// claimed from one counter in index order by a CTA that is already running,
// and a CTA works through its claims in order, so the unfinished claimed
// tile with the smallest index always has its inputs ready -- however many
// of the grid's CTAs are resident (other kernels may hold SMs): the
// producer can wait on the block's counters (act before a down-side tile
// starts, the shrink counter before the expand stages) without deadlock,
// and the phases overlap across CTAs:
// the gate_up base product streams while other CTAs run shrink tiles, and
// the down GEMM fills the gate_up tail.  (The pages overlap the shrink and
// expand kernels with PDL; here they share one grid.)
//
// Roles (224 threads): warps 0 and 6 issue TMA loads into a ring of smem
// stages, warp 0 the weight operand (B tile 256 x 64 bf16) and warp 6 the
// token rows (A tile 128 x 64 bf16: one 128-row box for a full block,
// 32-row boxes covering only the real rows of a partial one; both K-major
// with 128-byte swizzle); warp 1 allocates TMEM and one lane issues
// tcgen05.mma (M = 128, K = 16 per instruction, fp32 accumulate) and
// tcgen05.commit; warps 2..5 drain the double-buffered TMEM accumulator with
// tcgen05.ld while the next tile's MMAs run.  Grid: at most one CTA per SM.
// Every wait is bounded (~2 s unless a test sets a shorter limit): a
// timeout records MLORA_DEV_TIMEOUT, drains the copies in flight, frees
// TMEM and returns.
#include <atomic>

#include "internal.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

// 9 warps: weight producer (even stages, tiles), MMA, 4 epilogue, row
// producer (even stages), weight producer (odd), row producer (odd)
constexpr int kThreads = 288;
constexpr int kBN = 256;                                         // weight rows per wide tile (MMA N)
// The shared-memory ring: 4 stages of 48 KiB (A 16 KiB + B 32 KiB); when
// no block has more than 32 real rows (decode-like batches) the A part of a
// stage is one 32-row box, and 6 stages of 36 KiB hold 50 % more bytes in
// flight.
constexpr int kStages = 4;
constexpr int kSmallStages = 6;
// MXFP8 stages: A rows x 128 E4M3 (16 KiB for a full block, 4 KiB for one
// 32-row box), B 192 x 128 E4M3 (24 KiB), then the stage's scale atoms
// (512 B for A, 1 KiB for B), rounded up to the 1 KiB swizzle atom
constexpr int kMxBBytes = kMxWidth * kMxChunk;
constexpr int kMxStageBytes = (16384 + kMxBBytes + 3 * kMxAtom + 1023) / 1024 * 1024;  // 42 KiB
constexpr int kMxStages = 5;
constexpr int kMxSmallStageBytes = (4096 + kMxBBytes + 3 * kMxAtom + 1023) / 1024 * 1024;  // 30 KiB
constexpr int kMxSmallStages = 7;
// CTA-pair stages: two K-chunks of 64 (a copy moves both, so that the
// producer issues half as many copies per MMA): the CTA's A rows (2 x 16
// KiB), then its 128 of the tile's 256 weight rows (2 x 16 KiB)
constexpr int kPairABytes = 2 * 16384;
constexpr int kPairStageBytes = kPairABytes + 2 * 128 * 64 * 2;  // 64 KiB
constexpr int kPairStages = 3;
constexpr int kMaxStages = 7;  // barrier arrays: the deepest ring
static_assert(kMaxStages >= kStages && kMaxStages >= kSmallStages && kMaxStages >= kMxStages &&
                  kMaxStages >= kMxSmallStages && kMaxStages >= kPairStages, "barrier arrays");
// MXFP8 tensor memory: two 192-column accumulators, then two slots of
// scale factors (A at +0, B at +32 -- 32-column aligned -- of each 64)
constexpr int kMxAccCols = kMxWidth;
constexpr int kMxSfCol0 = 2 * kMxAccCols;
constexpr int kTileRing = 4;                                     // claimed tiles handed from producer to consumers
constexpr int kATileBytes = kBlockM * kBlockK * 2;               // 16 KiB
constexpr int kStageBytes = kATileBytes + kBN * kBlockK * 2;     // 48 KiB
constexpr int kSmallATileBytes = kRowBox * kBlockK * 2;          // 4 KiB
constexpr int kSmallStageBytes = kSmallATileBytes + kBN * kBlockK * 2;  // 36 KiB
constexpr int kRingBytes = kSmallStages * kSmallStageBytes;      // 216 KiB
constexpr int kAccCols = kBN;
constexpr int kTmemCols = 2 * kBN;
constexpr int kSmemBytes = kRingBytes + 1024 /* alignment slack */ + 256 /* barriers */;
static_assert(kStages * kStageBytes <= kRingBytes && kSmallStages * kSmallStageBytes <= kRingBytes, "ring");
static_assert(kSmemBytes <= 227 * 1024, "shared memory of a CTA");
static_assert(kStages * kStageBytes <= kRingBytes && kPairStages * kPairStageBytes <= kRingBytes, "ring");
static_assert(kMxStages * kMxStageBytes <= kRingBytes && kMxSmallStages * kMxSmallStageBytes <= kRingBytes, "ring");
static_assert(kMxSfCol0 + 2 * 64 <= 512, "tensor memory");
// one CTA per SM: each CTA allocates all 512 TMEM columns, so two CTAs of
// this kernel on one SM would wait on each other
static_assert(2 * kSmemBytes > 228 * 1024, "the experts kernel must not fit twice on an SM");

enum TileKind : int { kShrinkUp = 0, kGateUp = 1, kShrinkDown = 2, kDown = 3 };

// Bounded wait used only while unwinding after an abort: ignores the abort
// flag so that copies already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, long long limit) {
    int zero = 0;
    mbar_wait(bar, parity, &zero, nullptr, limit / 8 + 1000);
}

// Bounded wait until *flag >= target (acquire), then order this thread's
// later TMA (async-proxy) reads after it.
__device__ bool wait_counter(const int32_t* flag, int target, volatile int* abort_flag, uint32_t* status,
                             long long limit) {
    const long long t0 = clock64();
    for (uint32_t it = 0;; ++it) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= target) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return true;
        }
        if ((it & 63u) == 63u) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                atomicOr(status, MLORA_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

struct Tile {
    int kind;
    int side;  // 0: gate_up projection, 1: down projection
    bool shrink;
    int b;     // block of kBlockM sorted positions
    int cb;    // column slab (base tiles)
    int e;     // expert
    int i0;    // first adapter of the group in the block's list (shrink tiles)
    int g;     // adapters in the group (shrink tiles)
    bool rowless;  // CTA pair: this CTA holds none of the tile's token rows (the odd CTA of a shrink tile)
};

// Tile width of a launch: 256 weight rows (gate_up: 128 gate + 128 up),
// 192 or 128, the same for every tile of the launch.  Every CTA derives it
// from the padded slot count (choose_width).
struct Geom {
    int wc;      // width class: tile_width(wc) weight rows per tile
    int bn;      // weight rows per tile (MMA N)
    int half;    // gate (and up) rows of a gate_up tile
    int ncb0;    // column slabs per block, gate_up
    int ncb1;    // column slabs per block, down
};

// Phase boundaries of the tile sequence.
struct Phases {
    long s1, g, s2, d;  // ends of phases 1..4
};

// Tile `tile` of the sequence.  Base tiles run over units of rows: blocks,
// or in pair mode pairs of blocks (2u, 2u+1), where t.b is the block of
// this CTA (cluster rank `rank`); shrink tiles run over one block, whose
// rows the even CTA of a pair holds.
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, const Geom& gm, long tile, const Phases& ph, int ns,
                                            int nunits, int pair, uint32_t rank) {
    Tile t;
    long u;
    if (tile < ph.s1) {
        t.kind = kShrinkUp;
        u = tile;
    } else if (tile < ph.g) {
        t.kind = kGateUp;
        u = tile - ph.s1;
    } else if (tile < ph.s2) {
        t.kind = kShrinkDown;
        u = tile - ph.g;
    } else {
        t.kind = kDown;
        u = tile - ph.s2;
    }
    t.side = t.kind >= kShrinkDown ? 1 : 0;
    t.shrink = t.kind == kShrinkUp || t.kind == kShrinkDown;
    // blocks in descending order: the row gather writes x_perm in ascending
    // order, so the last blocks' rows are the ones still in L2
    if (t.shrink) {
        const long v = ns - 1 - u;
        t.b = p.gt_block[v];
        t.i0 = p.gt_first[v];
        t.g = min(p.gsize, p.blk_nad[t.b] - t.i0);
        t.cb = 0;
        t.rowless = pair && rank != 0;
    } else {
        const int ncb = t.side ? gm.ncb1 : gm.ncb0;
        const int bu = static_cast<int>(u / ncb);
        t.cb = static_cast<int>(u - static_cast<long>(bu) * ncb);
        const int unit = nunits - 1 - bu;
        t.b = pair ? 2 * unit + static_cast<int>(rank) : unit;
        t.i0 = 0;
        t.g = 0;
        t.rowless = false;
    }
    t.e = p.expert_ids[t.b];
    return t;
}

// K-chunks of 64 packed into one stage of a shrink tile.  A chunk is the A
// rows actually loaded (a_bytes) followed by the group's adapter rows
// (b_bytes); both are multiples of 2 KiB, so every chunk starts on a
// 1 KiB swizzle atom.  The MMA reads 128 A rows from a chunk's start, so
// that 16 KiB window must stay inside the stage as well.
constexpr int kMaxShrinkChunks = 4;
__device__ __forceinline__ int shrink_chunks(uint32_t a_bytes, uint32_t b_bytes, uint32_t stage_bytes) {
    const uint32_t chunk = a_bytes + b_bytes;
    int c = 1;
    while (c < kMaxShrinkChunks && (c + 1) * chunk <= stage_bytes && c * chunk + kATileBytes <= stage_bytes) ++c;
    return c;
}

// silu(z) = z * sigmoid(z); the fast divide returns 0 once 1 + e^-z
// overflows, the limit for very negative z
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Barriers and small shared state after the stage ring.
struct SmemLayout {
    uint64_t* full;        // [kMaxStages] a stage's loads landed
    uint64_t* empty;       // [kMaxStages] the MMAs reading a stage finished
    uint64_t* tfull;       // [2] an accumulator is ready for the epilogue
    uint64_t* tempty;      // [2] the epilogue drained an accumulator
    uint64_t* drain;       // the last MMAs of the CTA finished
    uint64_t* pub;         // the 128 epilogue threads finished writing a published tile
    uint64_t* tile_full;   // [kTileRing] a claimed tile index is in the ring
    uint64_t* tile_empty;  // [kTileRing] the MMA lane and 4 epilogue warps read it
    long long* tile_ring;
    uint32_t* tmem_holder;
    volatile int* abort_flag;
    __device__ __forceinline__ explicit SmemLayout(uint8_t* smem) {
        full = reinterpret_cast<uint64_t*>(smem + kRingBytes);
        empty = full + kMaxStages;
        tfull = empty + kMaxStages;
        tempty = tfull + 2;
        drain = tempty + 2;
        pub = drain + 1;
        tile_full = pub + 1;
        tile_empty = tile_full + kTileRing;
        tile_ring = reinterpret_cast<long long*>(tile_empty + kTileRing);
        tmem_holder = reinterpret_cast<uint32_t*>(tile_ring + kTileRing);
        abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    }
};

// What every role of a CTA derives once per launch: the shared-memory
// layout, the tile geometry and the phase boundaries of the tile list.
struct Ctx {
    const GemmParams* p;
    uint8_t* smem;
    SmemLayout L;
    Geom gm;
    Phases ph;
    int nblocks;
    int nunits;       // row units of the base tiles: blocks, or pairs of blocks
    int pair;         // CTA-pair launch
    uint32_t rank;    // cluster rank in a pair (0: the CTA that issues the MMAs)
    int ns;           // shrink tiles per projection
    int rp;           // rank padded to the MMA's N granule
    int lora_ksteps;  // expand K-steps of 16
    uint32_t tmem_base;
    long long lim;    // cycles a wait may take before the CTA gives up
    __device__ __forceinline__ Ctx(const GemmParams& prm, uint8_t* sm, uint32_t tmem)
        : p(&prm), smem(sm), L(sm), tmem_base(tmem), lim(prm.wait_limit) {
        nblocks = *prm.n_pad / kBlockM;
        pair = prm.pair;
        rank = pair ? cluster_ctarank() : 0u;
        // (align pads every expert to whole pairs of blocks in pair mode)
        nunits = pair ? nblocks / 2 : nblocks;
        ns = prm.has_lora ? *prm.gt_total : 0;
        // MXFP8 launches use 192-row tiles (the packed weight scales follow
        // them), CTA pairs 256-row tiles; otherwise the tuned table's width
        // for this many blocks, else the wave rule
        const int tuned = prm.width_table[width_bucket(nblocks)];
        gm.wc = prm.mx     ? 1
                : pair     ? 0
                : tuned >= 0 ? tuned
                             : choose_width(nblocks, prm.side[0].n_out, prm.side[1].n_out, gridDim.x);
        gm.bn = tile_width(gm.wc);
        gm.half = gm.bn / 2;
        gm.ncb0 = (prm.side[0].n_out + gm.half - 1) / gm.half;
        gm.ncb1 = (prm.side[1].n_out + gm.bn - 1) / gm.bn;
        ph.s1 = ns;
        ph.g = ph.s1 + static_cast<long>(nunits) * gm.ncb0;
        ph.s2 = ph.g + ns;
        ph.d = ph.s2 + static_cast<long>(nunits) * gm.ncb1;
        rp = (prm.rank + 15) / 16 * 16;
        lora_ksteps = (prm.rank + 15) / 16;
    }
};

// TMA producers, four threads in four warps over one ring of nst stages of
// stb bytes (the first ab of each holding A rows).  An issuing thread
// stalls for a while on every TMA copy it issues (a streaming probe: two
// copies a stage from one thread take ~600 ns, from two threads ~330 ns),
// so each stage's two operands come from two threads, and each operand's
// stages alternate between two threads (`par`: the stages it issues, by the
// parity of the stage count):
//  * the weight producer (kRows = false; warp 0) claims the tiles, hands
//    them to the other roles through the tile ring and streams each
//    stage's weight operand (B): expert weight rows, the adapters' B rows
//    of the expand stages, the adapters' A rows of the shrink stages;
//  * the row producer (kRows = true; warp 6) reads the tiles from the ring,
//    waits for the rows' producers (a down-side tile for the block's act
//    rows, an expand for the block's shrink tiles) and streams the
//    token-row operand (A): x or act rows, the LoRA tiles of the expands.
// Each announces its own bytes on the stage's full barrier (two arrivals),
// so the weight stream runs ahead of the row stream's waits by up to the
// ring's depth.  Only the even weight producer claims and hands out tiles;
// the other three read them from the ring.
template <int nst, uint32_t stb, uint32_t ab, bool kMx, bool kRows>
__device__ __forceinline__ void producer(const Ctx& c, long first_tile, int par) {
    const GemmParams& p = *c.p;
    uint64_t* const full = c.L.full;
    uint64_t* const empty = c.L.empty;
    uint64_t* const tile_full = c.L.tile_full;
    uint64_t* const tile_empty = c.L.tile_empty;
    long long* const tile_ring = c.L.tile_ring;
    volatile int* const abort_flag = c.L.abort_flag;
    const long long lim = c.lim;
    const int ns = c.ns;
    const Geom& gm = c.gm;
    const Phases& ph = c.ph;
    const long ntiles = c.ph.d;
    const int rp = c.rp;
    uint8_t* const smem = c.smem;
    long it = 0;  // stages issued
    bool ok = true;
    long tile = first_tile, next = -1;
    // the next tile is claimed a few stages before this one's base loads
    // are all issued: late enough that the CTA is about to be free (a
    // claim at the start of a tile hands work to CTAs that will be busy
    // for a whole tile while others idle), early enough that the atomic's
    // latency hides behind the last loads
    const bool master = !kRows && par == 0;
    auto claim = [&]() {
        if (master && next < 0) next = atomicAdd(p.tile_next, 1);
    };
    // whether this thread issues stage `it`.  It skips the other parity's
    // stages without waiting on them: its own wait two stages back (for
    // stage it - 2 - nst) already keeps it less than a ring cycle ahead of
    // the MMA lane, so a parity wait on a slot always refers to the slot's
    // latest use (nst >= 2)
    auto mine = [&]() { return static_cast<int>(it & 1) == par; };
    // waits for the next free stage; false after an abort
    auto stage_free = [&](int s) {
        return mbar_wait(&empty[s], (static_cast<uint32_t>(it / nst) & 1u) ^ 1u, abort_flag, p.status, lim);
    };
    // test hook: a wait on a flag that nothing sets, which must end
    // in a reported timeout and a clean exit
    if (master && p.stall_flag && !wait_counter(p.stall_flag, 1, abort_flag, p.status, lim)) ok = false;
    for (int jt = 0; ok; ++jt, tile = next, next = -1) {
        const int ts = jt % kTileRing;
        const uint32_t tph = static_cast<uint32_t>(jt / kTileRing) & 1u;
        if (master) {
            // hand the tile (or the end mark) to the row producer, the MMA
            // lane and the epilogue
            if (!mbar_wait(&tile_empty[ts], tph ^ 1u, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            const bool have = tile >= 0 && tile < ntiles;
            tile_ring[ts] = have ? tile : -1;
            mbar_arrive(&tile_full[ts]);
            if (!have) break;
        } else {
            if (!mbar_wait(&tile_full[ts], tph, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            tile = tile_ring[ts];
            mbar_arrive(&tile_empty[ts]);
            if (tile < 0) break;
        }
        const Tile tc = decode_tile(p, gm, tile, ph, ns, c.nunits, 0, 0u);
        const GemmSide& sd = p.side[tc.side];
        const int row0 = tc.b * kBlockM;
        // only the block's real rows are loaded; the MMA rows past
        // them hold stale data and feed only discarded output rows
        const int nbox = (p.blk_rows[tc.b] + kRowBox - 1) / kRowBox;
        const bool full_block = nbox * kRowBox == kBlockM;
        const uint32_t a_bytes = static_cast<uint32_t>(nbox) * kRowBox * kBlockK * 2;
        const int32_t* lora_list = p.blk_lora + static_cast<long>(tc.b) * p.cap;
        const int nk = (sd.K + kBlockK - 1) / kBlockK;
        // base tiles of the MXFP8 layer: K-chunks of 128 E4M3
        const int nk_base = kMx ? sd.nkc : nk;
        // the down side reads act rows, complete once the block's gate_up
        // tiles all are (the weight rows do not depend on them)
        if (kRows && tc.side == 1 && !wait_counter(p.act_done + tc.b, gm.ncb0, abort_flag, p.status, lim)) {
            ok = false;
            break;
        }
        if (tc.shrink) {
            // several K-chunks per stage: the shrink's operands are
            // small, and a stage of one chunk leaves the copy
            // engine latency-bound
            const uint32_t b_bytes = static_cast<uint32_t>(tc.g) * rp * kBlockK * 2;
            const uint32_t chunk = a_bytes + b_bytes;
            const int cps = shrink_chunks(a_bytes, b_bytes, stb);
            for (int kb0 = 0; kb0 < nk; kb0 += cps, ++it) {
                const int s = static_cast<int>(it % nst);
                const int nc = min(cps, nk - kb0);
                if (kb0 + nc >= nk) claim();
                if (!mine()) continue;
                if (!stage_free(s)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nc) * (kRows ? a_bytes : b_bytes));
                for (int cc = 0; cc < nc; ++cc) {
                    uint8_t* ca = smem + s * stb + cc * chunk;
                    const int k0 = (kb0 + cc) * kBlockK;
                    if (!kRows) {
                        for (int i = 0; i < tc.g; ++i)
                            tma_load_3d(ca + a_bytes + i * rp * kBlockK * 2, &sd.tm_sa, &full[s], k0, 0,
                                        lora_list[tc.i0 + i] * p.E_tot + tc.e);
                    } else if (full_block) {
                        tma_load_2d(ca, &sd.tm_a_full, &full[s], k0, row0);
                    } else {
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d(ca + i * kRowBox * kBlockK * 2, &sd.tm_a, &full[s], k0, row0 + i * kRowBox);
                    }
                }
            }
            continue;
        }
        // a base stage: the tile's weight rows of K-chunk kb (B; in the
        // MXFP8 layer E4M3 rows of 128 bytes, then the chunk's packed
        // weight scales) and the block's token rows (A; MXFP8: then the
        // chunk's scale atom of the activations)
        for (int kb = 0; kb < nk_base; ++kb, ++it) {
            const int s = static_cast<int>(it % nst);
            if (kb + 3 >= nk_base) claim();
            if (!mine()) continue;
            if (!stage_free(s)) {
                ok = false;
                break;
            }
            const int k0 = kb * (kMx ? kMxChunk : kBlockK);
            if (!kRows) {
                uint8_t* sb = smem + s * stb + ab;
                const CUtensorMap* map = kMx ? &sd.tm_bx : &sd.tm_b[gm.wc];
                mbar_arrive_expect_tx(&full[s], kMx ? gm.bn * kMxChunk + kMxTileScaleBytes : gm.bn * kBlockK * 2);
                if (tc.kind == kGateUp)
                    // one box over the slab's gate rows and then its up rows
                    tma_load_4d(sb, map, &full[s], k0, tc.cb * gm.half, 0, tc.e);
                else
                    tma_load_3d(sb, map, &full[s], k0, tc.cb * gm.bn, tc.e);
                if (kMx) {
                    const long ncb = tc.side ? gm.ncb1 : gm.ncb0;
                    bulk_load(sb + kMxBBytes + kMxAtom,
                              sd.b_scales + ((static_cast<size_t>(tc.e) * ncb + tc.cb) * sd.nkc + kb) * kMxTileScaleBytes,
                              kMxTileScaleBytes, &full[s]);
                }
            } else {
                uint8_t* sa = smem + s * stb;
                mbar_arrive_expect_tx(&full[s], kMx ? a_bytes + kMxAtom : a_bytes);
                const CUtensorMap* full_map = kMx ? &sd.tm_ax_full : &sd.tm_a_full;
                const CUtensorMap* box_map = kMx ? &sd.tm_ax : &sd.tm_a;
                if (full_block)
                    tma_load_2d(sa, full_map, &full[s], k0, row0);
                else
                    for (int i = 0; i < nbox; ++i)
                        tma_load_2d(sa + i * kRowBox * 128, box_map, &full[s], k0, row0 + i * kRowBox);
                if (kMx)
                    bulk_load(sa + ab + kMxBBytes, sd.a_scales + (static_cast<size_t>(tc.b) * sd.nkc + kb) * kMxAtom,
                              kMxAtom, &full[s]);
            }
        }
        if (!ok || !p.has_lora) continue;
        const int nad = p.blk_nad[tc.b];
        if (nad == 0) continue;
        // the expand needs every shrink tile of this block and side
        if (kRows && !wait_counter(sd.done + tc.b, (nad + p.gsize - 1) / p.gsize, abort_flag, p.status, lim)) {
            ok = false;
            break;
        }
        const int lt0 = p.blk_lt_start[tc.b];
        for (int i = 0; i < nad; ++i, ++it) {
            const int s = static_cast<int>(it % nst);
            if (!mine()) continue;
            if (!stage_free(s)) {
                ok = false;
                break;
            }
            uint8_t* sa = smem + s * stb;
            if (!kRows) {
                const int le = lora_list[i] * p.E_tot + tc.e;
                const CUtensorMap* lbmap = &sd.tm_lb[gm.wc];
                mbar_arrive_expect_tx(&full[s], gm.bn * kBlockK * 2);
                if (tc.kind == kGateUp)
                    tma_load_4d(sa + ab, lbmap, &full[s], 0, tc.cb * gm.half, 0, le);
                else
                    tma_load_3d(sa + ab, lbmap, &full[s], 0, tc.cb * gm.bn, le);
            } else {
                mbar_arrive_expect_tx(&full[s], a_bytes);
                if (full_block)
                    tma_load_2d(sa, &sd.tm_t_full, &full[s], 0, (lt0 + i) * kBlockM);
                else
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d(sa + j * kRowBox * kBlockK * 2, &sd.tm_t, &full[s], 0,
                                    (lt0 + i) * kBlockM + j * kRowBox);
            }
        }
    }
    if (!ok) {
        // this thread's stages among the last min(it, nst), walking back
        // from the ring position (a stage whose other operand never went
        // out ends the bounded wait)
        for (long j = it > nst ? it - nst : 0; j < it; ++j)
            if (static_cast<int>(j & 1) == par) drain_wait(&full[j % nst], static_cast<uint32_t>(j / nst) & 1u, lim);
    }
}

// MMA issuer (one thread), over the same ring geometry as the producer.
template <int nst, uint32_t stb, uint32_t ab, bool kMx>
__device__ __forceinline__ void mma_issuer(const Ctx& c) {
    const GemmParams& p = *c.p;
    uint64_t* const full = c.L.full;
    uint64_t* const empty = c.L.empty;
    uint64_t* const tfull = c.L.tfull;
    uint64_t* const tempty = c.L.tempty;
    uint64_t* const drain = c.L.drain;
    uint64_t* const tile_full = c.L.tile_full;
    uint64_t* const tile_empty = c.L.tile_empty;
    long long* const tile_ring = c.L.tile_ring;
    volatile int* const abort_flag = c.L.abort_flag;
    const long long lim = c.lim;
    const int ns = c.ns;
    const Geom& gm = c.gm;
    const Phases& ph = c.ph;
    const int rp = c.rp;
    const int lora_ksteps = c.lora_ksteps;
    uint8_t* const smem = c.smem;
    const uint32_t tmem_base = c.tmem_base;
    const uint32_t idesc_base = umma_idesc_bf16(128, gm.bn);
    long it = 0;  // stages consumed
    uint32_t sf_slot = 0;  // MXFP8: scale slot of the next base stage
    bool ok = true;
    for (int lt = 0; ok; ++lt) {
        const int ts = lt % kTileRing;
        if (!mbar_wait(&tile_full[ts], static_cast<uint32_t>(lt / kTileRing) & 1u, abort_flag, p.status, lim)) break;
        const long tile = tile_ring[ts];
        mbar_arrive(&tile_empty[ts]);
        if (tile < 0) break;
        const Tile tc = decode_tile(p, gm, tile, ph, ns, c.nunits, 0, 0u);
        const int nk = (p.side[tc.side].K + kBlockK - 1) / kBlockK;
        const int acc = lt & 1;
        if (!mbar_wait(&tempty[acc], (static_cast<uint32_t>(lt >> 1) & 1u) ^ 1u, abort_flag, p.status, lim)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * (kMx ? kMxAccCols : kAccCols));
        // a down tile whose slab runs past H multiplies only the
        // valid weight rows (rounded up to the MMA's N granule of 16)
        const int dn_valid = p.side[1].n_out - tc.cb * gm.bn;
        const uint32_t idesc = tc.shrink ? umma_idesc_bf16(128, tc.g * rp)
                               : (tc.kind == kDown && dn_valid < gm.bn)
                                   ? umma_idesc_bf16(128, (dn_valid + 15) / 16 * 16)
                                   : idesc_base;
        if (tc.shrink) {
            // the producer's packing: cps K-chunks of (A rows, adapter rows) per stage
            const int nbox = (p.blk_rows[tc.b] + kRowBox - 1) / kRowBox;
            const uint32_t a_bytes = nbox * kRowBox == kBlockM ? static_cast<uint32_t>(kATileBytes)
                                                               : static_cast<uint32_t>(nbox) * kRowBox * kBlockK * 2;
            const uint32_t chunk = a_bytes + static_cast<uint32_t>(tc.g) * rp * kBlockK * 2;
            const int cps = shrink_chunks(a_bytes, chunk - a_bytes, stb);
            for (int kb0 = 0; kb0 < nk; kb0 += cps, ++it) {
                const int s = static_cast<int>(it % nst);
                if (!mbar_wait(&full[s], static_cast<uint32_t>(it / nst) & 1u, abort_flag, p.status, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nc = min(cps, nk - kb0);
                for (int c = 0; c < nc; ++c) {
                    const uint32_t a_addr = smem_u32(smem + s * stb + c * chunk);
                    const uint64_t ad = umma_desc_sw128(a_addr);
                    const uint64_t bd = umma_desc_sw128(a_addr + a_bytes);
#pragma unroll
                    for (int k = 0; k < kBlockK / 16; ++k)
                        umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb0 | c | k) != 0 ? 1u : 0u);
                }
                umma_commit(&empty[s]);
            }
            if (!ok) break;
            umma_commit(&tfull[acc]);
            continue;
        }
        const int nk_base = kMx ? p.side[tc.side].nkc : nk;
        // MXFP8: N of the block-scaled MMA (the trimmed last down slab as above)
        const int n_mx = (tc.kind == kDown && dn_valid < gm.bn) ? (dn_valid + 15) / 16 * 16 : gm.bn;
        for (int kb = 0; kb < nk_base; ++kb, ++it) {
            const int s = static_cast<int>(it % nst);
            if (!mbar_wait(&full[s], static_cast<uint32_t>(it / nst) & 1u, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * stb);
            const uint64_t ad = umma_desc_sw128(a_addr);
            const uint64_t bd = umma_desc_sw128(a_addr + ab);
            if (kMx) {
                // the stage's scale atoms into tensor memory (ordered before
                // the MMAs that read them, and after the earlier MMAs that
                // read the same slot), then four K = 32 block-scaled MMAs,
                // each taking its byte of every scale word
                const uint32_t sf_smem = a_addr + ab + kMxBBytes;
                const uint32_t sfa = tmem_base + kMxSfCol0 + 64 * (sf_slot & 1u);
                const uint32_t sfb = sfa + 32;
                ++sf_slot;
                tmem_cp_32x128b_x4(sfa, smem_desc_plain(sf_smem, 128, 128));
                tmem_cp_32x128b_x4(sfb, smem_desc_plain(sf_smem + kMxAtom, 128, 128));
                tmem_cp_32x128b_x4(sfb + 4, smem_desc_plain(sf_smem + 2 * kMxAtom, 128, 128));
#pragma unroll
                for (int k = 0; k < kMxChunk / 32; ++k)
                    umma_mx(d, ad + 2 * k, bd + 2 * k, umma_idesc_mx(128, n_mx, k), sfa, sfb,
                            (kb | k) != 0 ? 1u : 0u);
            } else {
#pragma unroll
                for (int k = 0; k < kBlockK / 16; ++k)
                    umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            umma_commit(&empty[s]);
        }
        if (!ok) break;
        if (!tc.shrink && p.has_lora) {
            const int nad = p.blk_nad[tc.b];
            for (int i = 0; i < nad; ++i, ++it) {
                const int s = static_cast<int>(it % nst);
                if (!mbar_wait(&full[s], static_cast<uint32_t>(it / nst) & 1u, abort_flag, p.status, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * stb);
                const uint64_t ad = umma_desc_sw128(a_addr);
                const uint64_t bd = umma_desc_sw128(a_addr + ab);
                for (int k = 0; k < lora_ksteps; ++k) umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, 1u);
                umma_commit(&empty[s]);
            }
            if (!ok) break;
        }
        umma_commit(&tfull[acc]);
    }
    // every MMA issued above completes before TMEM is released
    umma_commit(drain);
    drain_wait(drain, 0, lim);
}

// Bytes of the token rows a CTA loads for block b: whole 32-row boxes
// covering its real rows (one 128-row box when the block is full).
__device__ __forceinline__ uint32_t block_a_bytes(const GemmParams& p, int b) {
    const int nbox = (p.blk_rows[b] + kRowBox - 1) / kRowBox;
    return static_cast<uint32_t>(nbox) * kRowBox * kBlockK * 2;
}

// Adapters of a pair of blocks: the ascending union of their lists.
__device__ __forceinline__ int pair_union_count(const GemmParams& p, int b0) {
    const int n0 = p.blk_nad[b0], n1 = p.blk_nad[b0 + 1];
    const int32_t* l0 = p.blk_lora + static_cast<long>(b0) * p.cap;
    const int32_t* l1 = l0 + p.cap;
    int i0 = 0, i1 = 0, n = 0;
    while (i0 < n0 || i1 < n1) {
        const int a = i0 < n0 ? l0[i0] : 0x7fffffff, b = i1 < n1 ? l1[i1] : 0x7fffffff;
        const int l = min(a, b);
        i0 += a == l;
        i1 += b == l;
        ++n;
    }
    return n;
}

// TMA producers of a CTA pair: in each CTA a weight producer (kRows =
// false; warp 0) and a row producer (kRows = true; warp 6), as in the
// one-CTA kernel.  The even CTA's weight producer claims the tiles and
// hands each to the rings of both CTAs.  Each CTA streams its own block's
// token rows (A) and its 128 of the tile's 256 weight rows (B: the gate
// rows of a gate_up slab in the even CTA, the up rows in the odd one; the
// first or second half of a down slab) into its own stage ring; every copy
// completes on the even CTA's stage barrier, on which all four producers
// arrive (the odd CTA's remotely), each announcing its own bytes before it
// issues them -- so that the barrier's transaction count never runs below
// zero, whichever CTA's copies land first.  Shrink
// tiles: the even CTA holds the block's rows, the adapters' rank rows are
// split between the two (a group of odd size gets a zero adapter in the odd
// CTA).  Expand stages run over the union of the two blocks' adapters; a
// block without the stage's adapter loads zero rows (a box at a negative
// row reads as zero).
template <int nst, uint32_t stb, uint32_t ab, bool kRows>
__device__ __forceinline__ void producer_pair(const Ctx& c, long first_tile) {
    const GemmParams& p = *c.p;
    uint64_t* const full = c.L.full;
    uint64_t* const empty = c.L.empty;
    uint64_t* const tile_full = c.L.tile_full;
    uint64_t* const tile_empty = c.L.tile_empty;
    long long* const tile_ring = c.L.tile_ring;
    volatile int* const abort_flag = c.L.abort_flag;
    const long long lim = c.lim;
    const Geom& gm = c.gm;
    const long ntiles = c.ph.d;
    const int rp = c.rp;
    uint8_t* const smem = c.smem;
    const uint32_t rank = c.rank;
    const bool lead = rank == 0;
    const bool master = lead && !kRows;
    constexpr uint32_t kChunkB = 128 * kBlockK * 2;  // a CTA's weight rows of one K-chunk
    long it = 0;  // stages passed
    bool ok = true;
    long tile = first_tile, next = -1;
    auto claim = [&]() {
        if (master && next < 0) next = atomicAdd(p.tile_next, 1);
    };
    auto stage_free = [&](int s) {
        return mbar_wait(&empty[s], (static_cast<uint32_t>(it / nst) & 1u) ^ 1u, abort_flag, p.status, lim);
    };
    // this producer's arrival on stage s of the even CTA, with its bytes
    auto arrive_stage = [&](int s, uint32_t fb, uint32_t bytes) {
        if (lead)
            mbar_arrive_expect_tx(&full[s], bytes);
        else
            mbar_arrive_expect_tx_cluster(fb, bytes);
    };
    if (master && p.stall_flag && !wait_counter(p.stall_flag, 1, abort_flag, p.status, lim)) ok = false;
    for (int jt = 0; ok; ++jt, tile = next, next = -1) {
        const int ts = jt % kTileRing;
        const uint32_t tph = static_cast<uint32_t>(jt / kTileRing) & 1u;
        if (master) {
            // the slot is free once its readers in both CTAs arrived
            if (!mbar_wait_cluster(&tile_empty[ts], tph ^ 1u, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            const bool have = tile >= 0 && tile < ntiles;
            const long v = have ? tile : -1;
            tile_ring[ts] = v;
            st_cluster_s64(mapa_shared(&tile_ring[ts], 1), v);
            mbar_arrive(&tile_full[ts]);
            mbar_arrive_cluster(mapa_shared(&tile_full[ts], 1));
            if (!have) break;
        } else {
            if (!mbar_wait_cluster(&tile_full[ts], tph, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            tile = tile_ring[ts];
            mbar_arrive_cluster(mapa_shared(&tile_empty[ts], 0));
            if (tile < 0) break;
        }
        const Tile tc = decode_tile(p, gm, tile, c.ph, c.ns, c.nunits, 1, rank);
        const GemmSide& sd = p.side[tc.side];
        const int nk = (sd.K + kBlockK - 1) / kBlockK;
        const int32_t* lora_list = p.blk_lora + static_cast<long>(tc.b) * p.cap;
        if (tc.shrink) {
            // the down shrink reads act rows (the even CTA's)
            if (kRows && lead && tc.side == 1 &&
                !wait_counter(p.act_done + tc.b, gm.ncb0, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            const uint32_t a0 = block_a_bytes(p, tc.b);
            const int nbox = static_cast<int>(a0 / (kRowBox * kBlockK * 2));
            const bool full_block = nbox * kRowBox == kBlockM;
            const int row0 = tc.b * kBlockM;
            const int g2 = (tc.g + 1) / 2;  // adapters per CTA
            const uint32_t bh = static_cast<uint32_t>(g2) * rp * kBlockK * 2;
            const uint32_t chunk = a0 + bh;  // the same layout in both CTAs
            const int cps = shrink_chunks(a0, bh, stb);
            for (int kb0 = 0; kb0 < nk; kb0 += cps, ++it) {
                const int s = static_cast<int>(it % nst);
                const int nc = min(cps, nk - kb0);
                if (kb0 + nc >= nk) claim();
                // every producer waits for every stage it passes, so that
                // it never runs a whole ring ahead of the MMA lane (a parity
                // wait cannot tell a phase two behind from a finished one)
                if (!stage_free(s)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = mapa_shared(&full[s], 0);
                // (the odd CTA holds no rows of a shrink tile)
                arrive_stage(s, fb, kRows ? (lead ? static_cast<uint32_t>(nc) * a0 : 0u)
                                                        : static_cast<uint32_t>(nc) * bh);
                if (kRows && !lead) continue;
                for (int cc = 0; cc < nc; ++cc) {
                    uint8_t* ca = smem + s * stb + cc * chunk;
                    const int k0 = (kb0 + cc) * kBlockK;
                    if (!kRows) {
                        for (int i = 0; i < g2; ++i) {
                            const int ai = static_cast<int>(rank) * g2 + i;
                            const int le = ai < tc.g ? lora_list[tc.i0 + ai] * p.E_tot + tc.e : -1;
                            tma_load_3d_pair(ca + a0 + i * rp * kBlockK * 2, &sd.tm_sa, fb, k0, 0, le);
                        }
                    } else if (full_block) {
                        tma_load_2d_pair(ca, &sd.tm_a_full, fb, k0, row0);
                    } else {
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d_pair(ca + i * kRowBox * kBlockK * 2, &sd.tm_a, fb, k0, row0 + i * kRowBox);
                    }
                }
            }
            continue;
        }
        const int b0 = tc.b & ~1;  // the pair's blocks: b0 (even CTA), b0 + 1
        const uint32_t a_mine = block_a_bytes(p, tc.b);
        const int nbox = static_cast<int>(a_mine / (kRowBox * kBlockK * 2));
        const bool full_block = nbox * kRowBox == kBlockM;
        const int row0 = tc.b * kBlockM;
        const int nst2 = (nk + 1) / 2;  // stages of two chunks (the last one's second may lie past K)
        const int kwhole = sd.K / kBlockK;
        // stage j copies chunks 2j and 2j+1 with one copy per operand when
        // both are whole chunks of K, or the second lies entirely past K
        // (the view's zero fill); the stage holding a partial last chunk
        // copies chunk by chunk through the 2D maps
        auto view_ok = [&](int j) {
            const int c1 = 2 * j + 1;
            return kwhole >= 2 && (c1 < kwhole || (c1 == kwhole && kwhole == nk));
        };
        // the down side reads act rows, complete once the block's gate_up
        // tiles all are (the weight rows do not depend on them)
        if (kRows && tc.side == 1 && !wait_counter(p.act_done + tc.b, gm.ncb0, abort_flag, p.status, lim)) {
            ok = false;
            break;
        }
        for (int j = 0; j < nst2; ++j, ++it) {
            const int s = static_cast<int>(it % nst);
            if (j + 2 >= nst2) claim();
            if (!stage_free(s)) {
                ok = false;
                break;
            }
            const uint32_t fb = mapa_shared(&full[s], 0);
            if (!kRows) {
                // (a pair launch keeps the 128-row half boxes of the gate_up
                // weights and expand weights in width class 1's map slot)
                arrive_stage(s, fb, 2 * kChunkB);
                uint8_t* sb = smem + s * stb + ab;
                if (view_ok(j)) {
                    if (tc.kind == kGateUp)
                        tma_load_5d_pair(sb, &sd.tm_bx, fb, 0, tc.cb * 128, static_cast<int>(rank), tc.e, 2 * j);
                    else
                        tma_load_4d_pair(sb, &sd.tm_bx, fb, 0, tc.cb * 256 + static_cast<int>(rank) * 128, tc.e,
                                         2 * j);
                } else {
                    for (int cc = 0; cc < 2; ++cc) {
                        const int k0 = (2 * j + cc) * kBlockK;
                        if (tc.kind == kGateUp)
                            tma_load_4d_pair(sb + cc * kChunkB, &sd.tm_b[1], fb, k0, tc.cb * 128,
                                             static_cast<int>(rank), tc.e);
                        else
                            tma_load_3d_pair(sb + cc * kChunkB, &sd.tm_b[2], fb, k0,
                                             tc.cb * 256 + static_cast<int>(rank) * 128, tc.e);
                    }
                }
            } else {
                arrive_stage(s, fb, 2 * a_mine);
                uint8_t* sa = smem + s * stb;
                if (nbox == 0) {
                } else if (full_block && view_ok(j)) {
                    tma_load_3d_pair(sa, &sd.tm_ax_full, fb, 0, row0, 2 * j);
                } else {
                    for (int cc = 0; cc < 2; ++cc) {
                        const int k0 = (2 * j + cc) * kBlockK;
                        uint8_t* ca = sa + cc * (kPairABytes / 2);
                        if (full_block)
                            tma_load_2d_pair(ca, &sd.tm_a_full, fb, k0, row0);
                        else
                            for (int i = 0; i < nbox; ++i)
                                tma_load_2d_pair(ca + i * kRowBox * kBlockK * 2, &sd.tm_a, fb, k0, row0 + i * kRowBox);
                    }
                }
            }
        }
        if (!ok || !p.has_lora) continue;
        const int n0 = p.blk_nad[b0], n1 = p.blk_nad[b0 + 1];
        if (n0 + n1 == 0) continue;
        // this block's LoRA tiles: every shrink tile of the block and side
        const int nmine = rank ? n1 : n0;
        if (kRows && nmine > 0 &&
            !wait_counter(sd.done + tc.b, (nmine + p.gsize - 1) / p.gsize, abort_flag, p.status, lim)) {
            ok = false;
            break;
        }
        const int32_t* l0 = p.blk_lora + static_cast<long>(b0) * p.cap;
        const int32_t* l1 = l0 + p.cap;
        const int lt0 = p.blk_lt_start[tc.b];
        const CUtensorMap* lb = tc.kind == kGateUp ? &sd.tm_lb[1] : &sd.tm_lb[2];
        int i0 = 0, i1 = 0;
        while (i0 < n0 || i1 < n1) {
            const int a = i0 < n0 ? l0[i0] : 0x7fffffff, b = i1 < n1 ? l1[i1] : 0x7fffffff;
            const int l = min(a, b);
            const int mine = rank ? (b == l ? i1 : -1) : (a == l ? i0 : -1);
            const int s = static_cast<int>(it % nst);
            if (!stage_free(s)) {
                ok = false;
                break;
            }
            const uint32_t fb = mapa_shared(&full[s], 0);
            uint8_t* sa = smem + s * stb;
            if (!kRows) {
                arrive_stage(s, fb, kChunkB);
                const int le = l * p.E_tot + tc.e;
                if (tc.kind == kGateUp)
                    tma_load_4d_pair(sa + ab, lb, fb, 0, tc.cb * 128, static_cast<int>(rank), le);
                else
                    tma_load_3d_pair(sa + ab, lb, fb, 0, tc.cb * 256 + static_cast<int>(rank) * 128, le);
            } else {
                arrive_stage(s, fb, a_mine);
                if (full_block)
                    tma_load_2d_pair(sa, &sd.tm_t_full, fb, 0, mine >= 0 ? (lt0 + mine) * kBlockM : -kBlockM);
                else
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d_pair(sa + j * kRowBox * kBlockK * 2, &sd.tm_t, fb, 0,
                                         mine >= 0 ? (lt0 + mine) * kBlockM + j * kRowBox : -kRowBox);
            }
            i0 += a == l;
            i1 += b == l;
            ++it;
        }
    }
    // after an abort the even CTA's producers wait (bounded) for the stages
    // issued: each barrier counts the bytes of both CTAs' copies (a stage
    // whose other operand never went out ends the bounded wait); the odd
    // CTA's copies land before the pair passes its final cluster barrier
    if (!ok && lead) {
        for (long j = it > nst ? it - nst : 0; j < it; ++j)
            drain_wait(&full[j % nst], static_cast<uint32_t>(j / nst) & 1u, lim);
    }
}

// MMA issuer of a CTA pair (one thread of the even CTA): the 256-row MMAs
// (cta_group::2) of every tile, each stage's completion signalled to the
// stage's empty barrier in both CTAs and each finished accumulator to both
// CTAs' epilogues.
template <int nst, uint32_t stb, uint32_t ab>
__device__ __forceinline__ void mma_issuer_pair(const Ctx& c) {
    const GemmParams& p = *c.p;
    uint64_t* const full = c.L.full;
    uint64_t* const empty = c.L.empty;
    uint64_t* const tfull = c.L.tfull;
    uint64_t* const tempty = c.L.tempty;
    uint64_t* const drain = c.L.drain;
    uint64_t* const tile_full = c.L.tile_full;
    uint64_t* const tile_empty = c.L.tile_empty;
    long long* const tile_ring = c.L.tile_ring;
    volatile int* const abort_flag = c.L.abort_flag;
    const long long lim = c.lim;
    const Geom& gm = c.gm;
    const int rp = c.rp;
    const int lora_ksteps = c.lora_ksteps;
    uint8_t* const smem = c.smem;
    const uint32_t tmem_base = c.tmem_base;
    const uint32_t idesc_base = umma_idesc_bf16(256, 256);
    long it = 0;  // stages consumed
    bool ok = true;
    for (int lt = 0; ok; ++lt) {
        const int ts = lt % kTileRing;
        if (!mbar_wait(&tile_full[ts], static_cast<uint32_t>(lt / kTileRing) & 1u, abort_flag, p.status, lim)) break;
        const long tile = tile_ring[ts];
        mbar_arrive(&tile_empty[ts]);
        if (tile < 0) break;
        const Tile tc = decode_tile(p, gm, tile, c.ph, c.ns, c.nunits, 1, 0u);
        const int nk = (p.side[tc.side].K + kBlockK - 1) / kBlockK;
        const int acc = lt & 1;
        // both CTAs' epilogues drained this accumulator
        if (!mbar_wait_cluster(&tempty[acc], (static_cast<uint32_t>(lt >> 1) & 1u) ^ 1u, abort_flag, p.status,
                               lim)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        if (tc.shrink) {
            const uint32_t a0 = block_a_bytes(p, tc.b);
            const int g2 = (tc.g + 1) / 2;
            const uint32_t bh = static_cast<uint32_t>(g2) * rp * kBlockK * 2;
            const uint32_t chunk = a0 + bh;
            const int cps = shrink_chunks(a0, bh, stb);
            const uint32_t idesc = umma_idesc_bf16(256, 2 * g2 * rp);
            for (int kb0 = 0; kb0 < nk; kb0 += cps, ++it) {
                const int s = static_cast<int>(it % nst);
                if (!mbar_wait(&full[s], static_cast<uint32_t>(it / nst) & 1u, abort_flag, p.status, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nc = min(cps, nk - kb0);
                for (int cc = 0; cc < nc; ++cc) {
                    const uint32_t a_addr = smem_u32(smem + s * stb + cc * chunk);
                    const uint64_t ad = umma_desc_sw128(a_addr);
                    const uint64_t bd = umma_desc_sw128(a_addr + a0);
#pragma unroll
                    for (int k = 0; k < kBlockK / 16; ++k)
                        umma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (kb0 | cc | k) != 0 ? 1u : 0u);
                }
                umma_commit_pair(&empty[s], 3);
            }
            if (!ok) break;
            umma_commit_pair(&tfull[acc], 3);
            continue;
        }
        // base stages: two K-chunks each (the last stage's second may lie
        // past K and is skipped)
        const int nst2 = (nk + 1) / 2;
        for (int j = 0; j < nst2; ++j, ++it) {
            const int s = static_cast<int>(it % nst);
            if (!mbar_wait(&full[s], static_cast<uint32_t>(it / nst) & 1u, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int nc = min(2, nk - 2 * j);
            for (int cc = 0; cc < nc; ++cc) {
                const uint32_t a_addr = smem_u32(smem + s * stb + cc * (kPairABytes / 2));
                const uint64_t ad = umma_desc_sw128(a_addr);
                const uint64_t bd = umma_desc_sw128(smem_u32(smem + s * stb + ab + cc * 128 * kBlockK * 2));
#pragma unroll
                for (int k = 0; k < kBlockK / 16; ++k)
                    umma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc_base, (j | cc | k) != 0 ? 1u : 0u);
            }
            umma_commit_pair(&empty[s], 3);
        }
        if (!ok) break;
        if (p.has_lora) {
            const int nu = pair_union_count(p, tc.b);
            for (int i = 0; i < nu; ++i, ++it) {
                const int s = static_cast<int>(it % nst);
                if (!mbar_wait(&full[s], static_cast<uint32_t>(it / nst) & 1u, abort_flag, p.status, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * stb);
                const uint64_t ad = umma_desc_sw128(a_addr);
                const uint64_t bd = umma_desc_sw128(a_addr + ab);
                for (int k = 0; k < lora_ksteps; ++k) umma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc_base, 1u);
                umma_commit_pair(&empty[s], 3);
            }
            if (!ok) break;
        }
        umma_commit_pair(&tfull[acc], 3);
    }
    // every MMA issued above (into both CTAs' tensor memory) completes
    // before either CTA releases it
    umma_commit_pair(drain, 1);
    drain_wait(drain, 0, lim);
}

// Epilogue (warps 2-5): drains the TMEM accumulators, writes shrink tiles,
// act rows or slot rows and publishes the per-block counters.  In a CTA
// pair each CTA drains its own accumulator rows (its own block) and reports
// the tile ring and the accumulator as read to the even CTA.
template <bool kMx, bool kPair>
__device__ __forceinline__ void epilogue(const Ctx& c) {
    const GemmParams& p = *c.p;
    uint64_t* const tfull = c.L.tfull;
    uint64_t* const tempty = c.L.tempty;
    uint64_t* const pub = c.L.pub;
    uint64_t* const tile_full = c.L.tile_full;
    uint64_t* const tile_empty = c.L.tile_empty;
    long long* const tile_ring = c.L.tile_ring;
    volatile int* const abort_flag = c.L.abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long lim = c.lim;
    const int ns = c.ns;
    const Geom& gm = c.gm;
    const Phases& ph = c.ph;
    const int rp = c.rp;
    const uint32_t tmem_base = c.tmem_base;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    uint32_t npub = 0;
    for (int lt = 0;; ++lt) {
        const int ts = lt % kTileRing;
        const uint32_t tph = static_cast<uint32_t>(lt / kTileRing) & 1u;
        if (!(kPair ? mbar_wait_cluster(&tile_full[ts], tph, abort_flag, p.status, lim)
                    : mbar_wait(&tile_full[ts], tph, abort_flag, p.status, lim)))
            break;
        const long tile = tile_ring[ts];
        __syncwarp();
        if (lane == 0) {
            if (kPair)
                mbar_arrive_cluster(mapa_shared(&tile_empty[ts], 0));
            else
                mbar_arrive(&tile_empty[ts]);
        }
        if (tile < 0) break;
        const Tile tc = decode_tile(p, gm, tile, ph, ns, c.nunits, kPair ? 1 : 0, c.rank);
        const GemmSide& sd = p.side[tc.side];
        const int acc = lt & 1;
        if (!mbar_wait(&tfull[acc], static_cast<uint32_t>(lt >> 1) & 1u, abort_flag, p.status, lim)) break;
        tc_fence_after();
        if (kPair && tc.rowless) {
            // the odd CTA of a shrink tile: its accumulator rows are unused
            tc_fence_before();
            mbar_arrive_cluster(mapa_shared(&tempty[acc], 0));
            continue;
        }
        const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * (kMx ? kMxAccCols : kAccCols)) +
                            (static_cast<uint32_t>(q * 32) << 16);
        const int prow = tc.b * kBlockM + row;
        int32_t* publish = nullptr;  // counter to bump once all 128 threads wrote
        if (tc.shrink) {
            const int my_l = row < p.blk_rows[tc.b] ? p.lora_of[prow] : -1;
            const int32_t* lora_list = p.blk_lora + static_cast<long>(tc.b) * p.cap;
            const int lt0 = p.blk_lt_start[tc.b] + tc.i0;
            for (int i = 0; i < tc.g; ++i) {
                if (!MLORA_IN_BOUNDS(lt0 + i < p.lt_cap, p.status)) break;
                const bool mine = my_l == lora_list[tc.i0 + i];
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(sd.lora_t) +
                                     (static_cast<size_t>(lt0 + i) * kBlockM + row) * kLoraTileCols;
                for (int c = 0; c < kLoraTileCols; c += 16) {
                    float v[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                    if (c < rp) tmem_ld16(tb + i * rp + c, v);
                    float o[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = (mine && c + j < p.rank) ? p.scaling * v[j] : 0.f;
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
            publish = sd.done + tc.b;
        } else if (tc.kind == kGateUp) {
            const bool real = MLORA_IN_BOUNDS(prow < p.pad_cap, p.status) && p.sorted_ids[prow] < p.S;
            const int j0 = tc.cb * gm.half;
            __nv_bfloat16* act = static_cast<__nv_bfloat16*>(sd.out) + static_cast<size_t>(prow) * sd.n_out;
            for (int c = 0; c < gm.half; c += 32) {
                if (j0 + c >= sd.n_out) break;
                float g[32], u[32];
                tmem_ld32(tb + c, g);
                tmem_ld32(tb + gm.half + c, u);
                if (real) {
                    // the SwiGLU output in place of g
#pragma unroll
                    for (int i = 0; i < 32; ++i) g[i] = silu(g[i]) * u[i];
                    // bf16 rows: the down GEMM's A (bf16 layer) or the down
                    // shrink's (adapters)
                    if (!kMx || p.has_lora) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int col = j0 + c + 8 * v;
                            if (col < sd.n_out) {
                                uint4 o;
                                o.x = pack_bf16x2(g[8 * v + 0], g[8 * v + 1]);
                                o.y = pack_bf16x2(g[8 * v + 2], g[8 * v + 3]);
                                o.z = pack_bf16x2(g[8 * v + 4], g[8 * v + 5]);
                                o.w = pack_bf16x2(g[8 * v + 6], g[8 * v + 7]);
                                *reinterpret_cast<uint4*>(act + col) = o;
                            }
                        }
                    }
                    if (kMx) {
                        // MXFP8 rows for the down GEMM: one block of 32 (I is a
                        // multiple of 32), its codes and its scale byte
                        uint4 q0, q1;
                        const uint8_t sc = mx_quantize32(g, q0, q1);
                        const int col = j0 + c;
                        uint4* dq = reinterpret_cast<uint4*>(sd.out_q + static_cast<size_t>(prow) * sd.n_out + col);
                        dq[0] = q0;
                        dq[1] = q1;
                        uint8_t* atoms = sd.out_s + static_cast<size_t>(tc.b) * p.side[1].nkc * kMxAtom;
                        atoms[(col / kMxChunk) * kMxAtom + mx_atom_byte(row, (col % kMxChunk) / kMxBlock)] = sc;
                        // after the last block of I: the rest of its K-chunk
                        // reads as zero data, with a zero scale byte rather
                        // than a stale NaN one
                        if (col + kMxBlock == sd.n_out)
                            for (int kb = (col % kMxChunk) / kMxBlock + 1; kb < kMxChunk / kMxBlock; ++kb)
                                atoms[(col / kMxChunk) * kMxAtom + mx_atom_byte(row, kb)] = 0;
                    }
                }
            }
            publish = p.act_done + tc.b;
        } else {
            const int f = MLORA_IN_BOUNDS(prow < p.pad_cap, p.status) ? p.sorted_ids[prow] : p.S;
            const bool real = f < p.S;
            const int o0 = tc.cb * gm.bn;
            // the slot's expert output stays fp32 until the combine
            float* dst = static_cast<float*>(sd.out) + static_cast<size_t>(real ? f : 0) * sd.n_out;
            for (int c = 0; c < gm.bn; c += 32) {
                if (o0 + c >= sd.n_out) break;
                float v[32];
                tmem_ld32(tb + c, v);
                if (real) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int col = o0 + c + 4 * j;
                        if (col < sd.n_out)
                            *reinterpret_cast<float4*>(dst + col) =
                                make_float4(v[4 * j + 0], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                }
            }
        }
        tc_fence_before();
        if (kPair)
            mbar_arrive_cluster(mapa_shared(&tempty[acc], 0));
        else
            mbar_arrive(&tempty[acc]);
        if (publish) {
            // other CTAs read what this tile wrote with TMA: every thread
            // orders its writes for the async proxy, arrives (release, CTA
            // scope) and waits (bounded, acquire) for all 128; then one
            // thread bumps the counter with a GPU-scope release, cumulative
            // over the writes it has synchronised with.  Every thread
            // waits, not only the one that publishes: a warp that ran on
            // to its next published tile would otherwise lend that tile's
            // arrival to this phase, completing it before a slower warp's
            // rows are written.
            asm volatile("fence.proxy.async.global;" ::: "memory");
            mbar_arrive(pub);
            const bool all_written = mbar_wait(pub, npub & 1u, abort_flag, p.status, lim);
            if (all_written && warp == 2 && lane == 0) red_add_release_gpu(publish, 1);
            ++npub;
        }
    }
}

template <bool kMx, bool kPair>
__global__ void __launch_bounds__(kThreads, 1) experts_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout L(smem);
    uint64_t* const full = L.full;
    uint64_t* const empty = L.empty;
    uint64_t* const tfull = L.tfull;
    uint64_t* const tempty = L.tempty;
    uint64_t* const drain = L.drain;
    uint64_t* const pub = L.pub;
    uint64_t* const tile_full = L.tile_full;
    uint64_t* const tile_empty = L.tile_empty;
    uint32_t* const tmem_holder = L.tmem_holder;
    volatile int* const abort_flag = L.abort_flag;

    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        // a stage is full once both producers' copies landed (a pair: the
        // even CTA's barrier counts the four producers of both CTAs)
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&full[s], kPair ? 4 : 2);
            mbar_init(&empty[s], 1);
        }
        // a pair: the even CTA's accumulator barriers count both CTAs'
        // epilogue threads, its tile-ring barriers the readers of both
        // (MMA lane + 4 epilogue warps + row producer; 2 producers + 4
        // epilogue warps); one CTA: MMA lane, 4 epilogue warps and three
        // producers
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], kPair ? 256 : 128);
        }
        mbar_init(drain, 1);
        mbar_init(pub, 128);
        for (int r = 0; r < kTileRing; ++r) {
            mbar_init(&tile_full[r], 1);
            mbar_init(&tile_empty[r], kPair ? 12 : 1 + 4 + 3);
        }
        *abort_flag = 0;
        fence_barrier_init();
        for (int sd = 0; sd < 2; ++sd) {
            // (the MXFP8 layer has bf16 token rows only for the adapters)
            if (!kMx || p.has_lora) {
                prefetch_tensormap(&p.side[sd].tm_a);
                prefetch_tensormap(&p.side[sd].tm_a_full);
            }
            if (!kMx)
                for (int wc = 0; wc < kTileWidths; ++wc) prefetch_tensormap(&p.side[sd].tm_b[wc]);
            if (kMx) {
                prefetch_tensormap(&p.side[sd].tm_ax);
                prefetch_tensormap(&p.side[sd].tm_ax_full);
                prefetch_tensormap(&p.side[sd].tm_bx);
            }
            if (kPair && p.side[sd].K >= 2 * kBlockK) {
                prefetch_tensormap(&p.side[sd].tm_ax_full);
                prefetch_tensormap(&p.side[sd].tm_bx);
            }
            if (p.has_lora) {
                prefetch_tensormap(&p.side[sd].tm_sa);
                for (int wc = 0; wc < kTileWidths; ++wc) prefetch_tensormap(&p.side[sd].tm_lb[wc]);
                prefetch_tensormap(&p.side[sd].tm_t);
                prefetch_tensormap(&p.side[sd].tm_t_full);
            }
        }
    }
    if (warp == 1) {
        if (kPair)
            tmem_alloc_pair(tmem_holder, kTmemCols);
        else
            tmem_alloc(tmem_holder, kTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    // a pair: both CTAs' barriers initialised and tensor memory allocated
    // before either touches the other's
    if (kPair) cluster_barrier();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // everything above overlapped the previous kernel in the stream
    griddep_wait();

    // the producer's first tile is claimed like every other (a CTA that
    // another kernel keeps waiting for an SM holds no tile that others
    // depend on), before the loads below so that the latencies overlap
    long first_tile = -1;
    if (threadIdx.x == 0 && (!kPair || cluster_ctarank() == 0)) first_tile = atomicAdd(p.tile_next, 1);
    const Ctx c(p, smem, tmem_base);
    // ring geometry of this launch (the same in every CTA): when no expert
    // has more than one 32-row box of slots, A stages shrink to 4 KiB and
    // the ring holds 6 stages instead of 4.  Only the two ring roles are
    // compiled per geometry; the epilogue exists once.
    const bool small_a = *p.max_rows <= kRowBox;
    constexpr int nst_s = kMx ? kMxSmallStages : kSmallStages, nst_f = kMx ? kMxStages : kStages;
    constexpr uint32_t stb_s = kMx ? kMxSmallStageBytes : kSmallStageBytes;
    constexpr uint32_t stb_f = kMx ? kMxStageBytes : kStageBytes;
    if (warp == 0 || warp >= 6) {
        if ((threadIdx.x & 31) == 0) {
            if constexpr (kPair) {
                if (warp == 0) producer_pair<kPairStages, kPairStageBytes, kPairABytes, false>(c, first_tile);
                if (warp == 6) producer_pair<kPairStages, kPairStageBytes, kPairABytes, true>(c, -1);
            } else {
                // warps 0 / 7: weight operand, even / odd stages; 6 / 8: rows
                const bool rows = warp == 6 || warp == 8;
                const int par = warp >= 7 ? 1 : 0;
                const long ft = warp == 0 ? first_tile : -1;
                if (small_a) {
                    if (rows)
                        producer<nst_s, stb_s, kSmallATileBytes, kMx, true>(c, ft, par);
                    else
                        producer<nst_s, stb_s, kSmallATileBytes, kMx, false>(c, ft, par);
                } else {
                    if (rows)
                        producer<nst_f, stb_f, kATileBytes, kMx, true>(c, ft, par);
                    else
                        producer<nst_f, stb_f, kATileBytes, kMx, false>(c, ft, par);
                }
            }
        }
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) {
            if constexpr (kPair) {
                if (c.rank == 0) mma_issuer_pair<kPairStages, kPairStageBytes, kPairABytes>(c);
            } else if (small_a) {
                mma_issuer<nst_s, stb_s, kSmallATileBytes, kMx>(c);
            } else {
                mma_issuer<nst_f, stb_f, kATileBytes, kMx>(c);
            }
        }
    } else {
        epilogue<kMx, kPair>(c);
    }

    tc_fence_before();
    __syncthreads();
    // a pair: the even CTA's MMAs into the odd CTA's tensor memory and the
    // odd CTA's copies and arrivals on the even CTA's barriers are over
    // before either CTA releases its tensor memory or exits
    if (kPair) cluster_barrier();
    if (warp == 1) {
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_experts(const GemmParams& p, long max_tiles, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    // per variant (bf16, MXFP8, bf16 pairs): one bit per device whose
    // shared-memory attribute is set, and the pairs a device keeps resident
    static std::atomic<unsigned long long> attr_done[3];
    static std::atomic<int> resident_pairs[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    const int v = p.pair ? 2 : p.mx ? 1 : 0;
    void (*const kernel)(GemmParams) =
        p.pair ? experts_kernel<false, true> : p.mx ? experts_kernel<true, false> : experts_kernel<false, false>;
    if (!(attr_done[v].load(std::memory_order_relaxed) & bit) || !bit) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (err != cudaSuccess) return err;
        attr_done[v].fetch_or(bit, std::memory_order_relaxed);
    }
    const long sms = device_sm_count();
    if (p.pair) {
        // one cluster of two CTAs per pair of SMs, as many as fit at once
        int pairs = dev >= 0 && dev < 64 ? resident_pairs[dev].load(std::memory_order_relaxed) : 0;
        if (pairs <= 0) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmemBytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&pairs, kernel, &cfg) != cudaSuccess || pairs <= 0) {
                (void)cudaGetLastError();
                pairs = static_cast<int>(sms / 2);
            }
            if (pairs > sms / 2) pairs = static_cast<int>(sms / 2);
            if (pairs < 1) pairs = 1;
            if (dev >= 0 && dev < 64) resident_pairs[dev].store(pairs, std::memory_order_relaxed);
        }
        long grid = 2L * pairs;
        if (grid > 2 * max_tiles) grid = 2 * max_tiles;
        return launch_pdl_cluster(kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, s, 2u, p);
    }
    long grid = sms;
    if (grid > max_tiles) grid = max_tiles;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, s, p);
}

}  // namespace mlora
