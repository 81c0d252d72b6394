// rows.cu -- the two bandwidth-bound row kernels around the grouped GEMMs:
//  * gather: x rows copied into sorted (expert-grouped) order so each GEMM
//    tile reads 128 consecutive rows with one TMA box;
//  * combine: y[m] = out_scale * sum_k topk_w[m,k] * y_slot[m*K'+k] (fp32
//    slot rows, fp32 sum, y rounded once to bf16), the weighted top-k sum ("[vllm] vLLM ROCm 환경에서 Shared-Expert Fusion을 통한
//    MoE 추론 성능 최적화", section "코드 분석" item 1: the routing weights,
//    shared slots included, weight each slot's expert output).
// The gather moves 16-byte vectors, one warp a row.  The combine reads 32
// bytes of fp32 per slot and writes eight bf16 outputs a thread; a launch
// too small to fill the GPU with more than eight slots a token takes 16
// bytes and four outputs a thread, so that its twelve-slot groups keep one
// memory round trip.
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int H8,
                                                          const int32_t* __restrict__ sorted,
                                                          const int32_t* __restrict__ n_pad, int S, int K_total,
                                                          uint4* __restrict__ x_perm, int max_padded,
                                                          uint32_t* __restrict__ status) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int np = *n_pad;
    const int stride = gridDim.x * warps;
    int p = blockIdx.x * warps + (threadIdx.x >> 5);
    // the next row's source slot is read one row ahead, so that its latency
    // overlaps the current row's copy
    int f_next = p < np && p < max_padded ? sorted[p] : S;
    for (; p < np; p += stride) {
        if (!MLORA_IN_BOUNDS(p < max_padded, status)) break;
        const int f = f_next;
        const int pn = p + stride;
        f_next = pn < np && pn < max_padded ? sorted[pn] : S;
        if (f >= S) continue;  // padding row: never stored downstream
        const uint4* src = x + static_cast<size_t>(f / K_total) * H8;
        uint4* dst = x_perm + static_cast<size_t>(p) * H8;
        // eight independent 16-byte loads in flight per lane
        for (int i0 = lane; i0 < H8; i0 += 256) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + 32 * j < H8) v[j] = __ldg(src + i0 + 32 * j);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + 32 * j < H8) dst[i0 + 32 * j] = v[j];
        }
    }
}

__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ y_slot,
                                                      const int32_t* __restrict__ topk_ids,
                                                      const float* __restrict__ topk_w, int M, int H8, int K_total,
                                                      int E_tot, float out_scale, uint4* __restrict__ y) {
    griddep_wait();
    griddep_launch_dependents();
    const long total = static_cast<long>(M) * H8;
    for (long idx = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long>(gridDim.x) * blockDim.x) {
        const int m = static_cast<int>(idx / H8);
        const int c = static_cast<int>(idx - static_cast<long>(m) * H8);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // slots in groups of eight, every load of a group issued at once --
        // ids, weights and slot rows, so that a group costs one memory
        // round trip (a dropped slot's row lies inside y_slot as well; it is
        // read and left out of the sum); the sum still runs over k in
        // ascending order
        for (int k0 = 0; k0 < K_total; k0 += 8) {
            float4 raw[8][2];
            float wk[8];
            int e[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const long f = static_cast<long>(m) * K_total + k0 + j;
                e[j] = -1;
                if (k0 + j < K_total) {
                    e[j] = __ldg(topk_ids + f);
                    wk[j] = __ldg(topk_w + f);
                    const float4* src = y_slot + (f * H8 + c) * 2;
                    raw[j][0] = __ldcs(src);
                    raw[j][1] = __ldcs(src + 1);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // a dropped slot (id outside [0, E_tot)) adds nothing
                if (static_cast<unsigned>(e[j]) >= static_cast<unsigned>(E_tot)) continue;
                const float v[8] = {raw[j][0].x, raw[j][0].y, raw[j][0].z, raw[j][0].w,
                                    raw[j][1].x, raw[j][1].y, raw[j][1].z, raw[j][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(wk[j], v[i], acc[i]);
            }
        }
        uint4 o;
        o.x = pack_bf16x2(out_scale * acc[0], out_scale * acc[1]);
        o.y = pack_bf16x2(out_scale * acc[2], out_scale * acc[3]);
        o.z = pack_bf16x2(out_scale * acc[4], out_scale * acc[5]);
        o.w = pack_bf16x2(out_scale * acc[6], out_scale * acc[7]);
        y[idx] = o;
    }
}

__global__ void __launch_bounds__(256) combine_narrow_kernel(const float4* __restrict__ y_slot,
                                                      const int32_t* __restrict__ topk_ids,
                                                      const float* __restrict__ topk_w, int M, int H4, int K_total,
                                                      int E_tot, float out_scale, uint2* __restrict__ y) {
    griddep_wait();
    griddep_launch_dependents();
    constexpr int kGroup = 12;
    const long total = static_cast<long>(M) * H4;
    for (long idx = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long>(gridDim.x) * blockDim.x) {
        const int m = static_cast<int>(idx / H4);
        const int c = static_cast<int>(idx - static_cast<long>(m) * H4);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        // slots in groups of twelve, every load of a group issued at once --
        // ids, weights and slot rows, so that a group costs one memory
        // round trip (a dropped slot's row lies inside y_slot as well; it is
        // read and left out of the sum); the sum still runs over k in
        // ascending order
        for (int k0 = 0; k0 < K_total; k0 += kGroup) {
            float4 raw[kGroup];
            float wk[kGroup];
            int e[kGroup];
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                const long f = static_cast<long>(m) * K_total + k0 + j;
                e[j] = -1;
                if (k0 + j < K_total) {
                    e[j] = __ldg(topk_ids + f);
                    wk[j] = __ldg(topk_w + f);
                    raw[j] = __ldcs(y_slot + f * H4 + c);
                }
            }
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                // a dropped slot (id outside [0, E_tot)) adds nothing
                if (static_cast<unsigned>(e[j]) >= static_cast<unsigned>(E_tot)) continue;
                acc[0] = fmaf(wk[j], raw[j].x, acc[0]);
                acc[1] = fmaf(wk[j], raw[j].y, acc[1]);
                acc[2] = fmaf(wk[j], raw[j].z, acc[2]);
                acc[3] = fmaf(wk[j], raw[j].w, acc[3]);
            }
        }
        uint2 o;
        o.x = pack_bf16x2(out_scale * acc[0], out_scale * acc[1]);
        o.y = pack_bf16x2(out_scale * acc[2], out_scale * acc[3]);
        y[idx] = o;
    }
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, int H, const int32_t* sorted, const int32_t* n_pad, long S,
                               int K_total, long max_padded, void* x_perm, uint32_t* status, cudaStream_t s) {
    if (max_padded == 0) return cudaSuccess;
    const int warps_per_block = 8;
    long blocks = (max_padded + warps_per_block - 1) / warps_per_block;
    const long cap = 8L * device_sm_count();
    if (blocks > cap) blocks = cap;
    return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(32 * warps_per_block), 0, s,
                      static_cast<const uint4*>(x), H / 8, sorted, n_pad, static_cast<int>(S), K_total,
                      static_cast<uint4*>(x_perm), static_cast<int>(max_padded), status);
}

cudaError_t launch_combine(const void* y_slot, const int32_t* topk_ids, const float* topk_w, int M, int H,
                           int K_total, int E_tot, float out_scale, void* y, cudaStream_t s) {
    const long sms = device_sm_count();
    const long wide = static_cast<long>(M) * (H / 8);
    if (wide == 0) return cudaSuccess;
    // more than eight slots a token in a launch too small to fill the GPU:
    // four outputs a thread and groups of twelve slots, one memory round
    // trip where eight outputs a thread would take two (a launch that fills
    // the GPU keeps the wider threads, whose larger loads hold more bytes
    // in flight)
    if (K_total > 8 && wide <= 256L * sms) {
        const long total = static_cast<long>(M) * (H / 4);
        const long blocks = (total + 255) / 256;
        return launch_pdl(combine_narrow_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                          static_cast<const float4*>(y_slot), topk_ids, topk_w, M, H / 4, K_total, E_tot, out_scale,
                          static_cast<uint2*>(y));
    }
    long blocks = (wide + 255) / 256;
    const long cap = 16L * sms;
    if (blocks > cap) blocks = cap;
    return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                      static_cast<const float4*>(y_slot), topk_ids, topk_w, M, H / 8, K_total, E_tot, out_scale,
                      static_cast<uint4*>(y));
}

}  // namespace mlora
