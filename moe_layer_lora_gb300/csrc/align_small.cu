// align_small.cu -- sort and pad the routed slots by expert (align) for
// batches of at most kSmallMaxSlots slots, and inside the forward the row
// gather in the same launch.
//
// "[vllm] vLLM ROCm 환경에서 Shared-Expert Fusion을 통한 MoE 추론 성능 최적화",
// section "코드 분석" item 2: the sort runs over E_tot = w13.shape[0]
// experts, shared ones included.  The output contract is the one of
// align.cu, bit for bit: experts ascending, each expert's slots f = m*K'+k
// ascending, each list padded with the sentinel M*K' to a multiple of
// block_m, sentinel / -1 tails; with adapters the same per-position adapter,
// per-block adapter lists and shrink group numbering.
//
// Small batches are latency-bound: the large-batch kernel spends most of
// its time in CTA-wide barriers.  Here 512 threads take at most 4 slots
// each; warp w owns one contiguous run of slots and ranks them in rounds of
// 32 (a slot's rank within its expert in the warp = the expert's slots in
// the warp's earlier rounds + the earlier lanes of its round with the same
// expert, from __match_any_sync), with no CTA barrier until every warp is
// done; one pass over the per-warp counts then gives each warp's first
// position per expert.  About eight barriers in all.
//
// The grid has several CTAs when the forward asks for the row gather: each
// CTA computes the same (cheap) sort, CTA 0 alone writes the sort's outputs,
// and every CTA copies the x rows of its share of the slots into their
// sorted positions -- one launch and one dependency instead of two.  Those
// rows depend on slot numbers only, so each CTA starts them into L2 before
// its grid wait, while the routing kernel still runs.  With adapters, a
// block's distinct adapters come from a 64-bit set when there are at most
// 64 adapters (one warp minimum per adapter otherwise).
#include <algorithm>
#include <atomic>

#include "internal.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = kSmallMaxSlots / kThreads;  // slots per thread
constexpr int kMaxSmem = 227 * 1024;
constexpr int kScratch = 64;  // ints: scan scratch [0, 34), flags [48], largest count [49], gather list length [50]
static_assert(kRounds * kThreads == kSmallMaxSlots, "slots per thread");

// Exclusive scan of one int per thread over the CTA; the CTA total goes to
// *total.  Three barriers (the last lets scratch be reused).
__device__ int cta_exclusive_scan(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += n;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int s = lane < kWarps ? scratch[lane] : 0;
        int si = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, si, off);
            if (lane >= off) si += n;
        }
        if (lane < kWarps) scratch[lane] = si - s;
        if (lane == kWarps - 1) scratch[kWarps] = si;
    }
    __syncthreads();
    const int excl = scratch[warp] + inc - v;
    *total = scratch[kWarps];
    __syncthreads();
    return excl;
}

// The same for two values at once (one set of barriers); scratch holds
// 2 * (kWarps + 1) ints.
__device__ void cta_exclusive_scan2(int va, int vb, int* scratch, int* ea, int* eb, int* ta, int* tb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = va, ib = vb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int na = __shfl_up_sync(0xffffffffu, ia, off);
        const int nb = __shfl_up_sync(0xffffffffu, ib, off);
        if (lane >= off) {
            ia += na;
            ib += nb;
        }
    }
    int* sa = scratch;
    int* sb = scratch + kWarps + 1;
    if (lane == 31) {
        sa[warp] = ia;
        sb[warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        const int a = lane < kWarps ? sa[lane] : 0;
        const int b = lane < kWarps ? sb[lane] : 0;
        int xa = a, xb = b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int na = __shfl_up_sync(0xffffffffu, xa, off);
            const int nb = __shfl_up_sync(0xffffffffu, xb, off);
            if (lane >= off) {
                xa += na;
                xb += nb;
            }
        }
        if (lane < kWarps) {
            sa[lane] = xa - a;
            sb[lane] = xb - b;
        }
        if (lane == kWarps - 1) {
            sa[kWarps] = xa;
            sb[kWarps] = xb;
        }
    }
    __syncthreads();
    *ea = sa[warp] + ia - va;
    *eb = sb[warp] + ib - vb;
    *ta = sa[kWarps];
    *tb = sb[kWarps];
    __syncthreads();
}

// x / block_m and rounding up to a multiple of it, for x >= 0: a shift when
// block_m is a power of two (the forward's 128), else a division.
struct BlockDiv {
    int bm, sh;
    __device__ int div(int x) const { return sh >= 0 ? x >> sh : x / bm; }
    __device__ int up(int x) const { return div(x + bm - 1) * bm; }
};

__device__ __forceinline__ BlockDiv block_div(int b) { return BlockDiv{b, (b & (b - 1)) == 0 ? __ffs(b) - 1 : -1}; }

// Position of the j-th (from 0) set bit of m; j < popc(m).  A binary search
// over halves of the remaining window by their population counts.
__device__ __forceinline__ int nth_set_bit(unsigned m, int j) {
    int pos = 0;
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
        const unsigned low = m & ((1u << w) - 1u);
        const int c = __popc(low);
        if (j >= c) {
            j -= c;
            m >>= w;
            pos += w;
        } else {
            m = low;
        }
    }
    return pos;
}

template <bool kWithLora, bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
    align_small_kernel(const int32_t* __restrict__ ids, int S, int E_tot, int BM, int max_padded,
                       int32_t* __restrict__ sorted, int32_t* __restrict__ expert_ids,
                       int32_t* __restrict__ n_pad_out, uint32_t* __restrict__ status, AlignExtra ex,
                       const uint4* __restrict__ x, int H8, int K_total, uint4* __restrict__ x_perm,
                       uint8_t* __restrict__ x_q, uint8_t* __restrict__ x_s) {
    extern __shared__ int smem_i[];
    int* wcnt = smem_i;                  // [kWarps][E_tot] a warp's slots per expert, then its first offset
    int* tot = wcnt + kWarps * E_tot;    // [E_tot] slots per expert
    int* first = tot + E_tot;            // [E_tot] padded start of each expert
    int* scratch = first + E_tot;        // [kScratch]
    int* nad_s = scratch + kScratch;     // with adapters: [max_padded / BM] adapters per block
    const BlockDiv bd = block_div(BM);
    const int max_blocks = bd.div(max_padded);
    int* glist = nad_s + (kWithLora ? max_blocks : 0);  // gather: [2 * S] (position, token) of this CTA's rows
    int* ints_end = glist + (kGather ? 2 * S : 0);
    // (8-byte aligned: the output sweep reads four entries at a time)
    uint16_t* st_sorted = reinterpret_cast<uint16_t*>(ints_end + ((ints_end - smem_i) & 1));  // [max_padded]
    int16_t* st_lora = reinterpret_cast<int16_t*>(st_sorted + max_padded);            // with adapters: [max_padded]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool writer = blockIdx.x == 0;  // CTA-uniform: the CTA that writes the sort's outputs
    int* flags = scratch + 48;
    if (kGather) {
        // the x rows this CTA copies are known before the ids are (slot f
        // reads token f / K_total): start them into L2 while the routing
        // kernel still runs (a prefetch reads nothing stale into a result)
        const int lines = (H8 * 16 + 127) / 128;
        const int nrows = (S - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
        for (int i = tid; i < nrows * lines; i += kThreads) {
            const int f = static_cast<int>(blockIdx.x) + (i / lines) * static_cast<int>(gridDim.x);
            const char* line = reinterpret_cast<const char*>(x + static_cast<size_t>(f / K_total) * H8) + (i % lines) * 128;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
        }
    }
    griddep_wait();
    griddep_launch_dependents();

    // this warp's contiguous run of slots, in rounds of 32 (all loads issued
    // first)
    const int per_warp = ((S + kWarps - 1) / kWarps + 31) & ~31;
    const int w0 = warp * per_warp;
    int e_r[kRounds], l_r[kRounds], rank_r[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int f = w0 + r * 32 + lane;
        const bool in = r * 32 < per_warp && f < S;
        e_r[r] = in ? __ldg(ids + f) : -1;
        l_r[r] = (kWithLora && in) ? __ldg(ex.token_lora_idx + f / ex.K_total) : -1;
        rank_r[r] = 0;
    }
    for (int e = lane; e < E_tot; e += 32) wcnt[warp * E_tot + e] = 0;
    if (tid == 0) {
        *flags = 0;
        scratch[49] = 0;
        scratch[50] = 0;
    }
    // the forward's status word, counts and per-block counters start at zero
    if (writer) {
        for (int i = tid; i < ex.zero_words; i += kThreads) ex.zero[i] = 0u;
        // every position starts as padding (the sentinel id S, no adapter);
        // the slots' positions are written over it below
        if ((max_padded & 1) == 0) {
            uint32_t* ss2 = reinterpret_cast<uint32_t*>(st_sorted);
            for (int i = tid; i < max_padded / 2; i += kThreads) ss2[i] = static_cast<uint32_t>(S) * 0x10001u;
            if (kWithLora) {
                uint32_t* sl2 = reinterpret_cast<uint32_t*>(st_lora);
                for (int i = tid; i < max_padded / 2; i += kThreads) sl2[i] = 0xFFFFFFFFu;
            }
        } else {
            for (int i = tid; i < max_padded; i += kThreads) {
                st_sorted[i] = static_cast<uint16_t>(S);
                if (kWithLora) st_lora[i] = -1;
            }
        }
    }
    __syncthreads();

    // 1. ranks within the warp, round by round in slot order
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        if (r * 32 >= per_warp) break;  // warp-uniform
        const int f = w0 + r * 32 + lane;
        const bool in = f < S;
        const bool valid = in && static_cast<unsigned>(e_r[r]) < static_cast<unsigned>(E_tot);
        if (in && !valid) atomicOr(flags, static_cast<int>(MLORA_DEV_BAD_EXPERT_ID));
        const int key = valid ? e_r[r] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int base = valid ? wcnt[warp * E_tot + key] : 0;
        rank_r[r] = base + __popc(peers & lt);
        __syncwarp();
        if (valid && (peers & lt) == 0) wcnt[warp * E_tot + key] = base + __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // 2. per expert: each warp's first offset (exclusive over the warps
    //    that hold slots, in place; all of an expert's counts read before
    //    any is written), the total and the padded size; thread t takes
    //    experts 2t and 2t+1 (E_tot <= 1024), then one scan of the padded
    //    sizes
    const int nw = min(kWarps, (S + per_warp - 1) / per_warp);  // warps holding slots
    int c_e[2] = {0, 0}, pad_e[2] = {0, 0};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int e = 2 * tid + q;
        if (e < E_tot) {
            int t[kWarps];
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t[w] = w < nw ? wcnt[w * E_tot + e] : 0;
            int run = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                if (w < nw) wcnt[w * E_tot + e] = run;
                run += t[w];
            }
            tot[e] = run;
            c_e[q] = run;
            pad_e[q] = bd.up(run);
            if (run > 0) atomicMax(&scratch[49], run);
        }
    }
    int total;
    const int start = cta_exclusive_scan(pad_e[0] + pad_e[1], scratch, &total);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int e = 2 * tid + q;
        if (e >= E_tot) break;
        const int s_e = start + (q ? pad_e[0] : 0);
        first[e] = s_e;
        if (writer) {
            // the block -> expert map and the real rows of each block
            const int b0 = bd.div(s_e);
            for (int b = b0; b < bd.div(s_e + pad_e[q]); ++b) {
                if (!MLORA_IN_BOUNDS(b < max_blocks, status)) break;
                expert_ids[b] = e;
                if (ex.blk_rows) ex.blk_rows[b] = min(BM, c_e[q] - (b - b0) * BM);
            }
        }
    }
    if (writer) {
        if (tid == 0) {
            *n_pad_out = total;
            if (ex.max_rows) *ex.max_rows = min(scratch[49], BM);
        }
        for (int b = bd.div(total) + tid; b < max_blocks; b += kThreads) expert_ids[b] = -1;
    }
    __syncthreads();

    // 3. every slot's sorted position: the expert's start + the warp's
    //    first offset + its rank in the warp
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        if (r * 32 >= per_warp) break;
        const int f = w0 + r * 32 + lane;
        const int e = e_r[r];
        if (f >= S || static_cast<unsigned>(e) >= static_cast<unsigned>(E_tot)) continue;
        const int pos = first[e] + wcnt[warp * E_tot + e] + rank_r[r];
        if (!MLORA_IN_BOUNDS(pos >= 0 && pos < max_padded, status)) continue;
        if (writer) {
            st_sorted[pos] = static_cast<uint16_t>(f);
            if (kWithLora) {
                int l = l_r[r];
                if (l < -1 || l >= ex.L) {
                    atomicOr(flags, static_cast<int>(MLORA_DEV_BAD_LORA_IDX));
                    l = -1;
                }
                st_lora[pos] = static_cast<int16_t>(l);
            }
        }
        if (kGather && f % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x)) {
            const int i = atomicAdd(&scratch[50], 1);
            glist[2 * i] = pos;
            glist[2 * i + 1] = f / K_total;
        }
    }
    __syncthreads();

    // 4. this CTA's x rows into their sorted positions: one warp per row,
    //    four 16-byte loads in flight per lane (MXFP8 layer: the rows
    //    quantized, and copied in bf16 only when adapters read them)
    if (kGather && x_q) {
        const int n = scratch[50];
        const int nchunk = (8 * H8 + kMxChunk - 1) / kMxChunk;
        for (int i = warp; i < n; i += kWarps) {
            const int pos = glist[2 * i];
            mx_gather_row(x + static_cast<size_t>(glist[2 * i + 1]) * H8, 8 * H8, pos % kBlockM,
                          x_q + static_cast<size_t>(pos) * 8 * H8,
                          x_s + static_cast<size_t>(pos / kBlockM) * nchunk * kMxAtom,
                          x_perm ? x_perm + static_cast<size_t>(pos) * H8 : nullptr, lane);
        }
    } else if (kGather) {
        const int n = scratch[50];
        for (int i = warp; i < n; i += kWarps) {
            const int pos = glist[2 * i];
            const uint4* src = x + static_cast<size_t>(glist[2 * i + 1]) * H8;
            uint4* dst = x_perm + static_cast<size_t>(pos) * H8;
            for (int i0 = lane; i0 < H8; i0 += 128) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i0 + 32 * j < H8) v[j] = __ldg(src + i0 + 32 * j);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i0 + 32 * j < H8) dst[i0 + 32 * j] = v[j];
            }
        }
    }
    if (!writer) return;

    // 5. the sorted ids (padding and the tail past the last block
    //    included) and the adapters of the used positions out in coalesced
    //    sweeps, four entries per thread and step where alignment allows
    const bool vec = (max_padded & 3) == 0 && (total & 3) == 0 &&
                     ((reinterpret_cast<uintptr_t>(sorted) |
                       (kWithLora ? reinterpret_cast<uintptr_t>(ex.lora_of) : uintptr_t(0))) & 15) == 0;
    if (vec) {
        const uint2* s4 = reinterpret_cast<const uint2*>(st_sorted);
        for (int i = tid; i < max_padded / 4; i += kThreads) {
            const uint2 v = s4[i];
            reinterpret_cast<int4*>(sorted)[i] = make_int4(static_cast<int>(v.x & 0xFFFFu), static_cast<int>(v.x >> 16),
                                                           static_cast<int>(v.y & 0xFFFFu), static_cast<int>(v.y >> 16));
        }
        if (kWithLora) {
            const uint2* l4 = reinterpret_cast<const uint2*>(st_lora);
            for (int i = tid; i < total / 4; i += kThreads) {
                const uint2 v = l4[i];
                reinterpret_cast<int4*>(ex.lora_of)[i] =
                    make_int4(static_cast<int16_t>(v.x & 0xFFFFu), static_cast<int16_t>(v.x >> 16),
                              static_cast<int16_t>(v.y & 0xFFFFu), static_cast<int16_t>(v.y >> 16));
            }
        }
    } else {
        for (int p = tid; p < max_padded; p += kThreads) {
            sorted[p] = st_sorted[p];
            if (kWithLora && p < total) ex.lora_of[p] = st_lora[p];
        }
    }
    if (!kWithLora) {
        if (tid == 0 && *flags && status) atomicOr(status, static_cast<uint32_t>(*flags));
        return;
    }

    // 6. distinct adapters of each block (ascending), one warp per block:
    //    with at most 64 adapters the block's set as a 64-bit mask, whose
    //    j-th member lane j writes; else one warp minimum per adapter
    constexpr int kMaxPerLane = MLORA_FORWARD_BLOCK_M / 32;
    const int nblocks = bd.div(total);
    for (int b = warp; b < nblocks; b += kWarps) {
        int mine[kMaxPerLane];
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int r = lane + 32 * i;
            mine[i] = r >= BM ? -1 : st_lora[b * BM + r];
        }
        int count = 0;
        if (ex.L <= 64) {
            unsigned lo = 0u, hi = 0u;
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i) {
                const int l = mine[i];
                if (l >= 0 && l < 32) lo |= 1u << l;
                if (l >= 32) hi |= 1u << (l - 32);
            }
            lo = __reduce_or_sync(0xffffffffu, lo);
            hi = __reduce_or_sync(0xffffffffu, hi);
            const int nlo = __popc(lo);
            count = nlo + __popc(hi);
            if (!MLORA_IN_BOUNDS(count <= ex.cap, status)) count = ex.cap;
            for (int j = lane; j < count; j += 32)
                ex.blk_lora[static_cast<long>(b) * ex.cap + j] = j < nlo ? nth_set_bit(lo, j) : 32 + nth_set_bit(hi, j - nlo);
        } else {
            int prev = -1;
            for (;;) {
                int cand = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < kMaxPerLane; ++i)
                    if (mine[i] > prev && mine[i] < cand) cand = mine[i];
                cand = static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<unsigned>(cand)));
                if (cand == 0x7fffffff) break;
                if (!MLORA_IN_BOUNDS(count < ex.cap, status)) break;
                if (lane == 0) ex.blk_lora[static_cast<long>(b) * ex.cap + count] = cand;
                ++count;
                prev = cand;
            }
        }
        if (lane == 0) {
            ex.blk_nad[b] = count;
            nad_s[b] = count;
        }
    }
    __syncthreads();
    if (tid == 0 && *flags && status) atomicOr(status, static_cast<uint32_t>(*flags));

    // 7. number the blocks' LoRA tiles (one per (block, adapter)) and the
    //    shrink group tiles (up to gsize adapters of one block each)
    int run_lt = 0, run_gt = 0;
    for (int cb = 0; cb < nblocks; cb += kThreads) {
        const int b = cb + tid;
        const int v = b < nblocks ? nad_s[b] : 0;
        const int ng = (v + ex.gsize - 1) / ex.gsize;
        int lt_chunk, gt_chunk, lt_excl, gt_excl;
        cta_exclusive_scan2(v, ng, scratch, &lt_excl, &gt_excl, &lt_chunk, &gt_chunk);
        if (b < nblocks) {
            ex.blk_lt_start[b] = run_lt + lt_excl;
            for (int j = 0; j < ng; ++j) {
                if (!MLORA_IN_BOUNDS(run_gt + gt_excl + j < ex.lt_cap, status)) break;
                ex.gt_block[run_gt + gt_excl + j] = b;
                ex.gt_first[run_gt + gt_excl + j] = j * ex.gsize;
            }
        }
        run_lt += lt_chunk;
        run_gt += gt_chunk;
    }
    if (tid == 0) *ex.gt_total = run_gt;
}

template <bool kWithLora, bool kGather>
cudaError_t launch_variant(int variant, const cudaLaunchConfig_t& cfg, const int32_t* ids, int S, int E_tot, int BM,
                           int max_padded, int32_t* sorted, int32_t* expert_ids, int32_t* n_pad, uint32_t* status,
                           const AlignExtra& ex, const uint4* x, int H8, int K_total, uint4* x_perm,
                           uint8_t* x_q, uint8_t* x_s) {
    static std::atomic<unsigned long long> attr_set[4];  // one bit per device (shared by host threads)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (!(attr_set[variant].load(std::memory_order_relaxed) & bit) || !bit) {
        err = cudaFuncSetAttribute(align_small_kernel<kWithLora, kGather>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (err != cudaSuccess) return err;
        attr_set[variant].fetch_or(bit, std::memory_order_relaxed);
    }
    return cudaLaunchKernelEx(&cfg, align_small_kernel<kWithLora, kGather>, ids, S, E_tot, BM, max_padded, sorted,
                              expert_ids, n_pad, status, ex, x, H8, K_total, x_perm, x_q, x_s);
}

}  // namespace

size_t align_small_smem(long S, int E_tot, int block_m, long max_padded, bool with_lora, bool gather) {
    size_t ints = static_cast<size_t>(kWarps + 2) * E_tot + kScratch +
                  (with_lora ? static_cast<size_t>(max_padded / block_m) : 0) + (gather ? 2 * static_cast<size_t>(S) : 0);
    ints += ints & 1;  // the staged ids start on an 8-byte boundary
    return sizeof(int) * ints +
           (sizeof(uint16_t) + (with_lora ? sizeof(int16_t) : 0)) * static_cast<size_t>(max_padded);
}

bool align_small_fits(long S, int E_tot, int block_m, long max_padded, const AlignExtra* extra, bool gather) {
    const bool with_lora = extra && extra->token_lora_idx;
    // (blocks padded to pairs: the cluster kernel only)
    if (extra && extra->pair_pad) return false;
    if (S < 1 || S > kSmallMaxSlots || E_tot > 2 * kThreads) return false;
    if (with_lora && (extra->L > 32767 || block_m != MLORA_FORWARD_BLOCK_M)) return false;
    return align_small_smem(S, E_tot, block_m, max_padded, with_lora, gather) <= static_cast<size_t>(kMaxSmem);
}

cudaError_t launch_align_small(const int32_t* ids, long S, int E_tot, int block_m, long max_padded, int32_t* sorted,
                               int32_t* expert_ids, int32_t* n_pad, uint32_t* status, const AlignExtra* extra,
                               const GatherArgs* gather, cudaStream_t s) {
    const bool with_lora = extra && extra->token_lora_idx;
    const bool g = gather != nullptr;
    // with the gather: about two slots' rows per CTA, at most one CTA per SM
    const int grid = g ? static_cast<int>(std::min<long>(device_sm_count(), (S + 1) / 2)) : 1;
    AlignExtra ex{};
    if (extra) ex = *extra;
    const uint4* x = g ? static_cast<const uint4*>(gather->x) : nullptr;
    uint4* x_perm = g ? static_cast<uint4*>(gather->x_perm) : nullptr;
    const int H8 = g ? gather->H / 8 : 0;
    const int K_total = g ? gather->K_total : 1;
    uint8_t* x_q = g ? gather->x_q : nullptr;
    uint8_t* x_s = g ? gather->x_s : nullptr;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = align_small_smem(S, E_tot, block_m, max_padded, with_lora, g);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int Si = static_cast<int>(S), mpi = static_cast<int>(max_padded);
    cudaError_t err;
    if (with_lora)
        err = g ? launch_variant<true, true>(3, cfg, ids, Si, E_tot, block_m, mpi, sorted, expert_ids, n_pad, status,
                                             ex, x, H8, K_total, x_perm, x_q, x_s)
                : launch_variant<true, false>(2, cfg, ids, Si, E_tot, block_m, mpi, sorted, expert_ids, n_pad,
                                              status, ex, x, H8, K_total, x_perm, x_q, x_s);
    else
        err = g ? launch_variant<false, true>(1, cfg, ids, Si, E_tot, block_m, mpi, sorted, expert_ids, n_pad,
                                              status, ex, x, H8, K_total, x_perm, x_q, x_s)
                : launch_variant<false, false>(0, cfg, ids, Si, E_tot, block_m, mpi, sorted, expert_ids, n_pad,
                                               status, ex, x, H8, K_total, x_perm, x_q, x_s);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace mlora
