// shrink.cu -- the LoRA shrink on CUDA cores for small batches, split over
// K across the CTAs of a thread-block cluster.
//
// "Amazon SageMaker 및 Amazon Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA 서빙
// 최적화", section "섹션별 상세" paragraphs 1 and 3: the shrink x A^T of each
// token's adapter is a skinny product (rank r of 8..64 outputs per row),
// parallelised with Split-K.  In decode-sized batches a (block, adapter)
// tile holds a handful of rows, so the work is streaming A_{l,e} once from
// HBM and the limit is how many loads are in flight, not arithmetic.
//
// One cluster of kSplit CTAs owns one tile; CTA `rank` takes the rank-th
// 1/kSplit of K.  It copies its K-slice of the r rows of A and of the
// tile's n rows of X into shared memory with cp.async (all copies in
// flight at once), then each thread computes whole (row, q) dot products
// over the slice from shared memory into a per-CTA fp32 partial.  The
// split-K sum runs over distributed shared memory: after a cluster barrier
// every CTA writes 16 rows of the output tile, adding the kSplit partials
// in rank order (deterministic, no atomics).  Output: the same masked tile
// as the tensor-core shrink, T[t][row][q] = bf16(s * sum_k X[row][k]
// A[q][k]) for rows whose adapter is the tile's, zero elsewhere and past
// the rank.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace mlora {
namespace {

constexpr int kThreads = kBlockM;  // one thread per row of the block when building the row list
constexpr int kSplit = 8;
constexpr int kSmemBytes = 24 * 1024;  // leaves room for one GEMM CTA on the same SM
constexpr int kPartialBytes = 8 * 1024;
constexpr int kRowsPerRank = kBlockM / kSplit;

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
    const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(ha[i]);
        const float2 fb = __bfloat1622float2(hb[i]);
        s = fmaf(fa.x, fb.x, s);
        s = fmaf(fa.y, fb.y, s);
    }
    return s;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kThreads)
    shrink_split_kernel(const ShrinkParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = static_cast<int>(cluster.block_rank());
    const int cid = blockIdx.x / kSplit, ncl = gridDim.x / kSplit;
    extern __shared__ uint4 dyn[];
    __shared__ int rowlist[kBlockM];
    __shared__ int rowpos[kBlockM];
    __shared__ int wcnt[kThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_wait();
    // the consuming GEMM may start now and stream its base weights beside
    // this kernel; it waits for this grid only before its expand stages
    griddep_launch_dependents();
    const int ntiles = *p.lt_total;
    const int K8 = p.K / 8;
    const int r = p.rank;
    const int per = (K8 + kSplit - 1) / kSplit;
    const int k_begin = min(K8, crank * per), k_end = min(K8, k_begin + per);
    const uint4* X = static_cast<const uint4*>(p.X);
    const uint4* A = static_cast<const uint4*>(p.A);
    float* part = reinterpret_cast<float*>(dyn);  // [n][r] fp32 partial of this CTA's K-slice

    for (int t = cid; t < ntiles; t += ncl) {
        const int b = p.lt_block[t];
        const int l = p.lt_lora[t];
        const int e = p.expert_ids[b];
        const int real = p.blk_rows[b];
        // rows of the block with this adapter, in ascending row order (the
        // same list in every CTA of the cluster)
        const bool mine = tid < real && p.lora_of[b * kBlockM + tid] == l;
        const unsigned bal = __ballot_sync(0xffffffffu, mine);
        if (lane == 0) wcnt[warp] = __popc(bal);
        __syncthreads();
        int base = 0, n = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            base += w < warp ? wcnt[w] : 0;
            n += wcnt[w];
        }
        const int pos = mine ? base + __popc(bal & ((1u << lane) - 1u)) : -1;
        rowpos[tid] = pos;
        if (mine) rowlist[pos] = tid;
        const uint4* Ab = A + static_cast<size_t>(l * p.E_tot + e) * r * K8;
        __syncthreads();

        // the rows go in groups small enough for their fp32 partials to take
        // at most a third of the budget; the rest stages K-chunks of A (r rows)
        // and X (the group's rows), rows padded by one 16-byte vector
        const int group = min(kBlockM, kPartialBytes / (4 * r));
        for (int g0 = 0; g0 == 0 || g0 < n; g0 += group) {
            const int gn = max(0, min(group, n - g0));
            for (int i = tid; i < gn * r; i += kThreads) part[i] = 0.f;
            uint4* stage = dyn + (gn * r * 4 + 15) / 16;
            const int stage_u4 = kSmemBytes / 16 - (gn * r * 4 + 15) / 16;
            const int kc8 = max(1, stage_u4 / (r + gn) - 1);
            const int stride = kc8 + 1;
            __syncthreads();
            for (int kc = k_begin; gn > 0 && kc < k_end; kc += kc8) {
                const int width = min(kc8, k_end - kc);
                for (int idx = tid; idx < (r + gn) * width; idx += kThreads) {
                    const int row = idx / width, i = idx - row * width;
                    const uint4* src =
                        row < r ? Ab + static_cast<size_t>(row) * K8 + kc + i
                                : X + static_cast<size_t>(b * kBlockM + rowlist[g0 + row - r]) * K8 + kc + i;
                    cp_async16(stage + row * stride + i, src);
                }
                cp_async_wait_all();
                __syncthreads();
                // `sub` consecutive threads share one output when there are
                // few outputs, each taking every sub-th vector of the chunk
                const int outs = gn * r;
                const int sub = outs >= kThreads ? 1 : min(32, 1 << (31 - __clz(kThreads / outs)));
                for (int o0 = 0; o0 < outs * sub; o0 += kThreads) {
                    const int slot = o0 + tid;
                    const int o = slot / sub, part_i = slot - o * sub;
                    float sum = 0.f;
                    if (o < outs) {
                        const int j = o / r, q = o - j * r;
                        const uint4* av = stage + q * stride;
                        const uint4* xv = stage + (r + j) * stride;
                        for (int i = part_i; i < width; i += sub) sum += dot8(av[i], xv[i]);
                    }
                    for (int off = sub >> 1; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                    if (o < outs && part_i == 0) part[o] += sum;
                }
                __syncthreads();
            }

            // split-K reduction over the cluster: this CTA writes rows
            // [kRowsPerRank * crank, +kRowsPerRank) of the tile, 8 columns per
            // thread -- the group's rows, and the rows of other adapters
            // (zero) in the first pass
            cluster.sync();
            const int row = kRowsPerRank * crank + (tid >> 3);
            const int c0 = (tid & 7) * 8;
            const int j = rowpos[row];
            const bool in_group = j >= g0 && j < g0 + gn;
            if (in_group || (g0 == 0 && j < 0)) {
                float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (in_group) {
                    for (int src = 0; src < kSplit; ++src) {
                        const float* rp = cluster.map_shared_rank(part, src);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            if (c0 + c < r) v[c] += rp[(j - g0) * r + c0 + c];
                    }
                }
                uint4 o;
                o.x = pack_bf16x2(p.scaling * v[0], p.scaling * v[1]);
                o.y = pack_bf16x2(p.scaling * v[2], p.scaling * v[3]);
                o.z = pack_bf16x2(p.scaling * v[4], p.scaling * v[5]);
                o.w = pack_bf16x2(p.scaling * v[6], p.scaling * v[7]);
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.T) +
                                          (static_cast<size_t>(t) * kBlockM + row) * kLoraTileCols + c0) = o;
            }
            cluster.sync();  // partials are reused by the next group or tile
        }
    }
}

}  // namespace

cudaError_t launch_shrink_rows(const ShrinkParams& p, long max_tiles, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !((attr_done >> dev) & 1ull)) {
        err = cudaFuncSetAttribute(shrink_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (err != cudaSuccess) return err;
        // the same L1/shared split as the GEMMs, so that a GEMM CTA can join
        // a shrink CTA on one SM without the SM being reconfigured
        err = cudaFuncSetAttribute(shrink_split_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        attr_done |= 1ull << dev;
    }
    // one CTA per SM: the consuming GEMM's CTA fits beside it
    long clusters = device_sm_count() / kSplit;
    if (clusters > max_tiles) clusters = max_tiles;
    if (clusters < 1) clusters = 1;
    return launch_pdl(shrink_split_kernel, dim3(static_cast<unsigned>(clusters * kSplit)), dim3(kThreads),
                      kSmemBytes, s, p);
}

}  // namespace mlora
