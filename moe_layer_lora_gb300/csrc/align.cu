// align.cu -- sort and pad the routed slots by expert (moe_align).
//
// "[vllm] vLLM ROCm 환경에서 Shared-Expert Fusion을 통한 MoE 추론 성능 최적화",
// section "코드 분석" item 2: the sort runs over E_tot = w13.shape[0] experts,
// shared ones included.  Output contract (bit-exact): experts ascending,
// each expert's slots f = m*K'+k ascending, each list padded with the
// sentinel M*K' to a multiple of block_m, sentinel / -1 tails.
//
// One CTA of 1024 threads: shared-memory histogram, a block scan of the
// padded counts, then a stable scatter.  Two ways to make it stable:
//  * passes of 1024 slots (one pass of slots, or many experts): within a
//    pass a slot's rank is (slots of its expert in earlier warps) + (earlier
//    lanes of its warp with the same expert, from __match_any_sync); the
//    per-warp per-expert counts live in a small shared table that one warp
//    per expert turns into exclusive prefixes with a shuffle scan;
//  * runs (more slots, up to 96 experts): each thread owns one contiguous
//    run of slots and counts it into its own column of a [E_tot][1024]
//    table; a scan along each expert's row gives every thread its first
//    position per expert, and the thread places its run in order.
// Either way, when the padded list fits in shared memory (16-bit slot ids
// and adapters) it is built there and copied out in one coalesced sweep
// instead of scattered 4-byte stores.
// From 2048 slots a thread-block cluster of up to 8 such CTAs (about 1024
// slots each) shares the work:
// each sorts one contiguous chunk of the slots, the chunks' per-expert
// counts are exchanged through distributed shared memory (cluster barrier,
// then mapa + ld.shared::cluster), and every CTA places its chunk after the
// slots of the same expert in earlier chunks -- still experts ascending,
// slots ascending within an expert.  The block lists are split over the
// CTAs and the first CTA numbers them after a last cluster barrier.
//
// Inside the forward the same pass also records the real (non-padding) row
// count of every block and, with adapters, per sorted position the token's
// adapter and per block of kBlockM positions the ascending list of distinct
// adapters; each (block, adapter) pair gets a masked LoRA tile, and the
// adapters of a block are cut into shrink group tiles of up to gsize.
#include <algorithm>
#include <atomic>

#include "internal.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kRunsMaxExperts = 96;      // per-thread count columns: 96 x 1024 x 2 B
constexpr int kMaxSmem = 227 * 1024;
constexpr long kClusterMinSlots = 2 * 1024;  // from here a cluster of CTAs sorts the slots

// Exclusive block scan of one int per thread; returns the exclusive prefix
// and writes the block total to *total.  Uses 33 ints of scratch.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
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
        int s = scratch[lane];
        int si = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, si, off);
            if (lane >= off) si += n;
        }
        scratch[lane] = si - s;  // exclusive warp offsets
        if (lane == 31) scratch[32] = si;
    }
    __syncthreads();
    const int excl = scratch[warp] + inc - v;
    *total = scratch[32];
    __syncthreads();
    return excl;
}

// ids[f .. f+4) clipped to end (missing entries read as -1); one 16-byte
// load when the run is aligned
__device__ __forceinline__ void load_ids4(const int32_t* __restrict__ ids, int f, int end, bool vec_ok, int* e4) {
    if (vec_ok && f + 4 <= end) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(ids + f));
        e4[0] = v.x; e4[1] = v.y; e4[2] = v.z; e4[3] = v.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) e4[j] = f + j < end ? ids[f + j] : -1;
    }
}

// Thread-block cluster helpers (large batches run one cluster of kCluster
// CTAs, each sorting a contiguous chunk of the slots).
constexpr int kCluster = 8;
__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// An int in the shared memory of CTA `rank` of the cluster, at the offset
// of `local` in this CTA.
__device__ __forceinline__ int dsmem_load(const int* local, unsigned rank) {
    uint32_t ra;
    int v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

template <bool kWithLora>
__global__ void __launch_bounds__(kThreads, 1)
    align_kernel(const int32_t* __restrict__ ids, int S, int E_tot, int BM, int max_padded,
                 int32_t* __restrict__ sorted, int32_t* __restrict__ expert_ids, int32_t* __restrict__ n_pad_out,
                 uint32_t* __restrict__ status, int runs, int staged, int ncl, AlignExtra ex) {
    // ncl CTAs (one thread-block cluster when > 1): CTA crank sorts the
    // slots [c0, c1); the per-expert counts of all chunks are exchanged through
    // distributed shared memory, so each CTA knows where its chunk's slots
    // of each expert start
    extern __shared__ int smem_i[];
    int* cnt = smem_i;                                            // [E_tot] this chunk's slots per expert
    int* first = cnt + E_tot;                                     // [E_tot] padded start of each expert
    int* cursor = first + E_tot;                                  // [E_tot] next free position
    int* tot = cursor + E_tot;                                    // [E_tot] all chunks' slots per expert
    int* cbase = tot + E_tot;                                     // [E_tot] slots of the expert in earlier chunks
    int* scratch = cbase + E_tot;                                 // [40] (scratch[39]: flags)
    int* nad_s = scratch + 40;  // with adapters: [max_padded / BM] adapters per block
    // passes: [kWarps][E_tot] per-warp counts; runs: [E_tot][kThreads] per-thread counts
    // (16-byte aligned: the runs' row scan reads it as uint4)
    uint16_t* wcnt =
        reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(nad_s + (kWithLora ? max_padded / BM : 0)) + 15) &
                                    ~uintptr_t(15));
    // staged: [max_padded] sorted slot ids, then [max_padded] adapters
    uint16_t* st_sorted = wcnt + static_cast<size_t>(E_tot) * (runs ? kThreads : kWarps);
    int16_t* st_lora = reinterpret_cast<int16_t*>(st_sorted + max_padded);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int crank = ncl > 1 ? static_cast<int>(cluster_rank()) : 0;
    // this CTA's chunk, a multiple of 4 slots long (16-byte aligned runs)
    const int chunk = ((S + ncl - 1) / ncl + 3) & ~3;
    const int c0 = min(S, crank * chunk), c1 = min(S, c0 + chunk);
    int* flags = scratch + 39;  // bad ids seen by this CTA, written to status at the end
    griddep_wait();
    griddep_launch_dependents();
    // passes: the first pass's expert and adapter ids, loaded now so that
    // their latency hides behind the clearing below
    int e_next = (!runs && c0 + tid < c1) ? __ldg(ids + c0 + tid) : -1;
    int l_next = (kWithLora && !runs && c0 + tid < c1) ? __ldg(ex.token_lora_idx + (c0 + tid) / ex.K_total) : -1;
    // the forward's status word, counts and per-block counters start at
    // zero (this kernel is the forward's first; the CTAs of a cluster report
    // their flags only at the end, after the cluster barriers)
    if (crank == 0)
        for (int i = tid; i < ex.zero_words; i += kThreads) ex.zero[i] = 0u;
    if (tid == 0) {
        *flags = 0;
        scratch[38] = 0;  // most slots of one expert
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    // runs: slots per thread, a multiple of 4 so that a run starts on a
    // 16-byte boundary when ids does
    const int run_len = ((c1 - c0 + kThreads - 1) / kThreads + 3) & ~3;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    const int run0 = min(c1, c0 + tid * run_len), run1 = min(c1, run0 + run_len);

    for (int e = tid; e < E_tot; e += kThreads) cnt[e] = 0;
    if (runs) {
        for (int e = 0; e < E_tot; ++e) wcnt[e * kThreads + tid] = 0;
    } else {
        for (int i = tid; i < kWarps * E_tot; i += kThreads) wcnt[i] = 0;
    }
    __syncthreads();

    // 1. histogram
    if (runs) {
        // each thread counts its own run of slots into its own column, then
        // one warp per expert turns the row into exclusive prefixes (in slot
        // order) and the expert's total
        for (int f = run0; f < run1; f += 4) {
            int e4[4];
            load_ids4(ids, f, run1, vec_ok, e4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (f + j >= run1) break;
                if (static_cast<unsigned>(e4[j]) < static_cast<unsigned>(E_tot))
                    ++wcnt[e4[j] * kThreads + tid];
                else
                    atomicOr(flags, static_cast<int>(MLORA_DEV_BAD_EXPERT_ID));
            }
        }
        __syncthreads();
        // two levels: each lane sums its 32 consecutive columns (four
        // 16-byte reads), one shuffle scan over the lanes, then each lane
        // writes its columns' exclusive prefixes
        for (int e = warp; e < E_tot; e += kWarps) {
            uint4* row = reinterpret_cast<uint4*>(wcnt + e * kThreads) + lane * 4;
            uint4 v[4];
            int sum = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[q] = row[q];
                const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) sum += static_cast<int>(w[h] & 0xffffu) + static_cast<int>(w[h] >> 16);
            }
            int inc = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += nb;
            }
            int run = inc - sum;  // columns of earlier lanes
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int lo = static_cast<int>(w[h] & 0xffffu), hi = static_cast<int>(w[h] >> 16);
                    w[h] = static_cast<uint32_t>(run) | (static_cast<uint32_t>(run + lo) << 16);
                    run += lo + hi;
                }
                row[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (lane == 31) cnt[e] = inc;
        }
    } else {
        for (int f = c0 + tid; f < c1; f += kThreads) {
            const int e = f == c0 + tid ? e_next : ids[f];
            if (static_cast<unsigned>(e) < static_cast<unsigned>(E_tot))
                atomicAdd(&cnt[e], 1);
            else
                atomicOr(flags, static_cast<int>(MLORA_DEV_BAD_EXPERT_ID));
        }
    }
    __syncthreads();

    // 1b. every chunk's counts: the expert totals, and this chunk's first
    //     position inside each expert (slots of earlier chunks)
    if (ncl > 1) cluster_sync_all();
    for (int e = tid; e < E_tot; e += kThreads) {
        int t = 0, b = 0;
        for (int q = 0; q < ncl; ++q) {
            const int v = ncl > 1 ? dsmem_load(cnt + e, static_cast<unsigned>(q)) : cnt[e];
            t += v;
            if (q < crank) b += v;
        }
        tot[e] = t;
        cbase[e] = b;
    }
    __syncthreads();

    // 2. exclusive scan of the padded counts (E_tot <= 1024: one expert per
    //    thread), the block -> expert map and the real rows of each block
    //    (pair_pad: padded to whole pairs of blocks, the second of a pair
    //    possibly empty)
    const int PB = ex.pair_pad ? 2 * BM : BM;
    const int c = tid < E_tot ? tot[tid] : 0;
    const int padded = (c + PB - 1) / PB * PB;
    int total;
    const int start = block_exclusive_scan(padded, scratch, &total);
    if (tid < E_tot) {
        first[tid] = start;
        cursor[tid] = start + cbase[tid];
    }
    if (tid < E_tot && c > 0) atomicMax(&scratch[38], c);
    if (tid < E_tot && crank == 0) {
        for (int b = start / BM; b < (start + padded) / BM; ++b) {
            if (!MLORA_IN_BOUNDS(b < max_padded / BM, status)) break;
            expert_ids[b] = tid;
            if (ex.blk_rows) ex.blk_rows[b] = max(0, min(BM, c - (b - start / BM) * BM));
        }
    }
    if (crank == 0) {
        if (tid == 0) *n_pad_out = total;
        for (int p = total + tid; p < max_padded; p += kThreads) sorted[p] = S;
        for (int b = total / BM + tid; b < max_padded / BM; b += kThreads) expert_ids[b] = -1;
    }
    __syncthreads();
    if (crank == 0 && tid == 0 && ex.max_rows) *ex.max_rows = min(scratch[38], BM);

    // 3. per-expert padding, one warp per expert
    for (int e = warp * ncl + crank; e < E_tot; e += kWarps * ncl) {
        const int n = tot[e];
        const int pad_end = first[e] + (n + PB - 1) / PB * PB;
        for (int p = first[e] + n + lane; p < pad_end; p += 32) {
            if (!MLORA_IN_BOUNDS(p < max_padded, status)) break;
            if (staged) {
                st_sorted[p] = static_cast<uint16_t>(S);
                st_lora[p] = -1;
            } else {
                sorted[p] = S;
                if (kWithLora) ex.lora_of[p] = -1;
            }
        }
    }

    // 4a. runs: every thread places its own run in order
    if (runs) {
        for (int f0 = run0; f0 < run1; f0 += 4) {
            int e4[4];
            load_ids4(ids, f0, run1, vec_ok, e4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int f = f0 + j, e = e4[j];
                if (f >= run1) break;
                if (static_cast<unsigned>(e) >= static_cast<unsigned>(E_tot)) continue;
                const int p = cursor[e] + wcnt[e * kThreads + tid]++;
                if (!MLORA_IN_BOUNDS(p >= 0 && p < max_padded, status)) continue;
                int l = -1;
                if (kWithLora) {
                    l = ex.token_lora_idx[f / ex.K_total];
                    if (l < -1 || l >= ex.L) {
                        atomicOr(flags, static_cast<int>(MLORA_DEV_BAD_LORA_IDX));
                        l = -1;
                    }
                }
                if (staged) {
                    st_sorted[p] = static_cast<uint16_t>(f);
                    st_lora[p] = static_cast<int16_t>(l);
                } else {
                    sorted[p] = f;
                    if (kWithLora) ex.lora_of[p] = l;
                }
            }
        }
        __syncthreads();
    }

    // 4b. passes: stable scatter, 1024 slots per pass.  Within a pass a slot's rank
    //    among the slots of its expert is (its expert's slots in earlier
    //    warps) + (earlier lanes of its warp with the same expert); the first
    //    term comes from a per-expert scan over the warps' counts, done one
    //    expert column per warp.
    // the next pass's expert and adapter ids are loaded during this one
    for (int base = c0; !runs && base < c1; base += kThreads) {
        const int f = base + tid;
        const int e = e_next;
        const int l_in = l_next;
        const bool more = f + kThreads < c1;
        e_next = more ? ids[f + kThreads] : -1;
        if (kWithLora) l_next = more ? ex.token_lora_idx[(f + kThreads) / ex.K_total] : -1;
        const bool valid = static_cast<unsigned>(e) < static_cast<unsigned>(E_tot);
        const int key = valid ? e : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & lt_mask);
        const int n_same = __popc(peers);
        const bool leader = (peers & lt_mask) == 0;
        if (valid && leader) wcnt[warp * E_tot + e] = static_cast<uint16_t>(n_same);
        __syncthreads();
        for (int ex_col = warp; ex_col < E_tot; ex_col += kWarps) {
            const int c_w = wcnt[lane * E_tot + ex_col];
            int inc = c_w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += nb;
            }
            if (c_w) wcnt[lane * E_tot + ex_col] = static_cast<uint16_t>(inc - c_w);
        }
        __syncthreads();
        int pos = 0;
        if (valid && leader) pos = cursor[e] + wcnt[warp * E_tot + e];
        pos = __shfl_sync(0xffffffffu, pos, __ffs(peers) - 1);
        if (valid) {
            const int p = pos + rank;
            const bool in_range = MLORA_IN_BOUNDS(p >= 0 && p < max_padded, status);
            int l = l_in;
            if (kWithLora && (l < -1 || l >= ex.L)) {
                atomicOr(flags, static_cast<int>(MLORA_DEV_BAD_LORA_IDX));
                l = -1;
            }
            if (!in_range) {
            } else if (staged) {
                st_sorted[p] = static_cast<uint16_t>(f);
                st_lora[p] = static_cast<int16_t>(l);
            } else {
                sorted[p] = f;
                if (kWithLora) ex.lora_of[p] = l;
            }
        }
        __syncthreads();
        if (valid && leader) {
            atomicAdd(&cursor[e], n_same);
            wcnt[warp * E_tot + e] = 0;
        }
        __syncthreads();
    }

    // staged: one coalesced copy of the sorted ids (and adapters) out
    if (staged) {
        for (int p = tid; p < total; p += kThreads) {
            sorted[p] = st_sorted[p];
            if (kWithLora) ex.lora_of[p] = st_lora[p];
        }
    }
    // a cluster: every chunk placed (and every peer done reading this CTA's
    // counts) before the block lists read the adapters of all positions
    if (ncl > 1) cluster_sync_all();

    if (!kWithLora) {
        __syncthreads();
        if (tid == 0 && *flags && status) atomicOr(status, static_cast<uint32_t>(*flags));
        return;
    }

    // 5. distinct adapters of each block (ascending), one warp per block;
    //    the block's adapter ids are read once into registers
    constexpr int kMaxPerLane = MLORA_FORWARD_BLOCK_M / 32;
    const int nblocks = total / BM;
    for (int b = warp * ncl + crank; b < nblocks; b += kWarps * ncl) {
        int mine[kMaxPerLane];
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int r = lane + 32 * i;
            // (a cluster's other CTAs wrote these positions: read through L2)
            mine[i] = r >= BM ? -1 : staged ? st_lora[b * BM + r] : ncl > 1 ? __ldcg(ex.lora_of + b * BM + r)
                                                                                : ex.lora_of[b * BM + r];
        }
        int prev = -1, count = 0;
        for (;;) {
            int cand = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i)
                if (mine[i] > prev && mine[i] < cand) cand = mine[i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, off));
            if (cand == 0x7fffffff) break;
            if (!MLORA_IN_BOUNDS(count < ex.cap, status)) break;
            if (lane == 0) ex.blk_lora[static_cast<long>(b) * ex.cap + count] = cand;
            ++count;
            prev = cand;
        }
        if (lane == 0) {
            ex.blk_nad[b] = count;
            nad_s[b] = count;
        }
    }
    __syncthreads();
    if (tid == 0 && *flags && status) atomicOr(status, static_cast<uint32_t>(*flags));
    // a cluster: the first CTA numbers all blocks once every list is written
    if (ncl > 1) {
        cluster_sync_all();
        if (crank != 0) return;
    }

    // 6. number the blocks' LoRA tiles (one per (block, adapter)) and the
    //    shrink group tiles (up to gsize adapters of one block each)
    int run_lt = 0, run_gt = 0;
    for (int cb = 0; cb < nblocks; cb += kThreads) {
        const int b = cb + tid;
        const int v = b < nblocks ? (ncl > 1 ? __ldcg(ex.blk_nad + b) : nad_s[b]) : 0;
        const int ng = (v + ex.gsize - 1) / ex.gsize;
        int lt_chunk, gt_chunk;
        const int lt_excl = block_exclusive_scan(v, scratch, &lt_chunk);
        const int gt_excl = block_exclusive_scan(ng, scratch, &gt_chunk);
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

}  // namespace

long align_max_padded(long S, int E_tot, int block_m) {
    const long nonempty = S < E_tot ? S : E_tot;
    const long bound = S + nonempty * (block_m - 1);
    return (bound + block_m - 1) / block_m * block_m;
}

cudaError_t launch_align(const int32_t* ids, long S, int E_tot, int block_m, long max_padded, int32_t* sorted,
                         int32_t* expert_ids, int32_t* n_pad, uint32_t* status, const AlignExtra* extra,
                         cudaStream_t s) {
    // small batches take the latency-lean kernel (same outputs, bit for bit)
    if (align_small_fits(S, E_tot, block_m, max_padded, extra, false))
        return launch_align_small(ids, S, E_tot, block_m, max_padded, sorted, expert_ids, n_pad, status, extra,
                                  nullptr, s);
    const bool with_lora = extra && extra->token_lora_idx;
    void (*kernel)(const int32_t*, int, int, int, int, int32_t*, int32_t*, int32_t*, uint32_t*, int, int, int,
                   AlignExtra) = with_lora ? align_kernel<true> : align_kernel<false>;
    static std::atomic<unsigned long long> attr_set[2];  // one bit per device (shared by host threads)
    static std::atomic<unsigned long long> cluster_ok[2], cluster_known[2];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    const int v = with_lora ? 1 : 0;
    if (!(attr_set[v].load(std::memory_order_relaxed) & bit) || !bit) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (err != cudaSuccess) return err;
        attr_set[v].fetch_or(bit, std::memory_order_relaxed);
    }
    // large batches: one cluster of kCluster CTAs, each sorting a chunk
    // (when the device can host such a cluster at full shared memory)
    int ncl = 1;
    if (S >= kClusterMinSlots) {
        if (!(cluster_known[v].load(std::memory_order_relaxed) & bit) || !bit) {
            cudaLaunchConfig_t q{};
            q.gridDim = dim3(kCluster);
            q.blockDim = dim3(kThreads);
            q.dynamicSmemBytes = kMaxSmem;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = kCluster;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, kernel, &q) != cudaSuccess) {
                (void)cudaGetLastError();
                nclusters = 0;
            }
            if (nclusters > 0) cluster_ok[v].fetch_or(bit, std::memory_order_relaxed);
            cluster_known[v].fetch_or(bit, std::memory_order_relaxed);
        }
        // about one pass of 1024 slots per CTA, at most kCluster CTAs
        if (cluster_ok[v].load(std::memory_order_relaxed) & bit)
            ncl = static_cast<int>(std::min<long>(kCluster, (S + kThreads - 1) / kThreads));
    }
    // several passes over the slots, or (more than one pass of slots per
    // CTA, few experts) per-thread runs with one count column per thread;
    // one CTA builds the padded list in shared memory when it fits there
    const long chunk = (S + ncl - 1) / ncl;
    const int runs = chunk > kThreads && E_tot <= kRunsMaxExperts && S <= 65535 ? 1 : 0;
    size_t smem = sizeof(int) * (5 * static_cast<size_t>(E_tot) + 40 +
                                 (with_lora ? static_cast<size_t>(max_padded / block_m) : 0)) +
                  16 /* alignment of the count table */ +
                  sizeof(uint16_t) * static_cast<size_t>(runs ? kThreads : kWarps) * E_tot;
    const size_t stage_bytes = (sizeof(uint16_t) + sizeof(int16_t)) * static_cast<size_t>(max_padded);
    const bool small_ids = S <= 65535 && (!extra || extra->L <= 32767);
    int staged = 0;
    if (ncl == 1 && small_ids && smem + stage_bytes <= static_cast<size_t>(kMaxSmem)) {
        staged = 1;
        smem += stage_bytes;
    }
    AlignExtra ex{};
    if (extra) ex = *extra;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ncl);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = ncl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ncl > 1 ? 2 : 1;
    err = cudaLaunchKernelEx(&cfg, kernel, ids, static_cast<int>(S), E_tot, block_m, static_cast<int>(max_padded),
                             sorted, expert_ids, n_pad, status, runs, staged, ncl, ex);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace mlora
