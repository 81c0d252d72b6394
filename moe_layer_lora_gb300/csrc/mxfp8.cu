// mxfp8.cu -- the MXFP8 side of the layer around the experts kernel:
//  * weights to MXFP8 once (E4M3 codes in the weights' own layout, E8M0
//    scales packed per 192-row tile slab and 128-wide K-chunk in the order
//    the tensor cores read them, mx.cuh);
//  * the row gather of the MXFP8 layer: each routed x row quantized (blocks
//    of 32 along H) into its sorted position, its scales into the block's
//    scale atoms, and the plain bf16 row too when adapters read it.
// The pages name an MXFP8 experts path for the fused layer ("[vllm] vLLM
// ROCm 환경에서 Shared-Expert Fusion을 통한 MoE 추론 성능 최적화", section
// "코드 분석" item 2); the format is the OCP Microscaling specification's
// MXFP8 (E4M3 elements, one E8M0 scale per 32).
#include <cuda_bf16.h>

#include "internal.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

// 32 bf16 (four uint4) to fp32
__device__ __forceinline__ void bf16x32_to_f32(const uint4 (&r)[4], float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r[q]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __bfloat1622float2(h[i]);
            v[8 * q + 2 * i] = t.x;
            v[8 * q + 2 * i + 1] = t.y;
        }
    }
}

// One warp per weight row; each lane takes whole blocks of 32.  which = 0:
// rows of w13 [E_tot * 2I, H]; which = 1: rows of w2 [E_tot * H, I].
__global__ void __launch_bounds__(256) mx_quantize_weights_kernel(const uint4* __restrict__ w, long rows, int K,
                                                                  int which, int H, int I,
                                                                  uint8_t* __restrict__ codes,
                                                                  uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const long warps = static_cast<long>(gridDim.x) * (blockDim.x >> 5);
    const int nblk = K / kMxBlock;
    const long nslab = mx_slabs(which, H, I), nchunk = mx_chunks(which, H, I);
    for (long R = blockIdx.x * static_cast<long>(blockDim.x >> 5) + (threadIdx.x >> 5); R < rows; R += warps) {
        // this row's place in the packed scales: its expert, tile slab and
        // row n of the 192-row tile
        long e, cb;
        int n;
        if (which == 0) {
            e = R / (2L * I);
            const int j2 = static_cast<int>(R - e * 2L * I);
            const int up = j2 >= I ? 1 : 0;
            const int j = j2 - up * I;
            cb = j / kMxHalf;
            n = up * kMxHalf + j % kMxHalf;
        } else {
            e = R / H;
            const int o = static_cast<int>(R - e * H);
            cb = o / kMxWidth;
            n = o % kMxWidth;
        }
        const uint4* src = w + R * (K / 8);
        for (int b = lane; b < nblk; b += 32) {
            uint4 r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) r[q] = __ldg(src + b * 4 + q);
            float v[32];
            bf16x32_to_f32(r, v);
            uint4 q0, q1;
            const uint8_t sc = mx_quantize32(v, q0, q1);
            uint4* dst = reinterpret_cast<uint4*>(codes + R * K + b * kMxBlock);
            dst[0] = q0;
            dst[1] = q1;
            const long kc = b / (kMxChunk / kMxBlock);
            scales[((e * nslab + cb) * nchunk + kc) * kMxTileScaleBytes + (n / 128) * kMxAtom +
                   mx_atom_byte(n % 128, b % (kMxChunk / kMxBlock))] = sc;
        }
    }
}

// One warp per sorted position p < n_pad holding a real slot: x row
// f / K' quantized into x_q[p] and its scales into the atoms of block
// p / 128; the bf16 row copied into x_perm[p] as well when x_perm is set.
__global__ void __launch_bounds__(256) mx_gather_kernel(const uint4* __restrict__ x, int H, int K_total,
                                                        const int32_t* __restrict__ sorted,
                                                        const int32_t* __restrict__ n_pad, int S, int max_padded,
                                                        uint8_t* __restrict__ x_q, uint8_t* __restrict__ x_s,
                                                        uint4* __restrict__ x_perm, uint32_t* __restrict__ status) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int np = *n_pad;
    const int nchunk = (H + kMxChunk - 1) / kMxChunk;
    for (int p = blockIdx.x * warps + (threadIdx.x >> 5); p < np; p += gridDim.x * warps) {
        if (!MLORA_IN_BOUNDS(p < max_padded, status)) break;
        const int f = sorted[p];
        if (f >= S) continue;  // padding row: its outputs are discarded
        mx_gather_row(x + static_cast<size_t>(f / K_total) * (H / 8), H, p % kBlockM, x_q + static_cast<size_t>(p) * H,
                      x_s + static_cast<size_t>(p / kBlockM) * nchunk * kMxAtom,
                      x_perm ? x_perm + static_cast<size_t>(p) * (H / 8) : nullptr, lane);
    }
}

}  // namespace

cudaError_t launch_mx_quantize_weights(const void* w, long rows, int K, int which, int H, int I, uint8_t* codes,
                                       uint8_t* packed_scales, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    long blocks = (rows + 7) / 8;
    const long cap = 16L * device_sm_count();
    if (blocks > cap) blocks = cap;
    mx_quantize_weights_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint4*>(w), rows, K,
                                                                             which, H, I, codes, packed_scales);
    return cudaGetLastError();
}

cudaError_t launch_mx_gather(const void* x, int H, int K_total, const int32_t* sorted, const int32_t* n_pad,
                             long S, long max_padded, uint8_t* x_q, uint8_t* x_s, void* x_perm, uint32_t* status,
                             cudaStream_t s) {
    if (max_padded == 0) return cudaSuccess;
    const int warps_per_block = 8;
    long blocks = (max_padded + warps_per_block - 1) / warps_per_block;
    const long cap = 8L * device_sm_count();
    if (blocks > cap) blocks = cap;
    return launch_pdl(mx_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(32 * warps_per_block), 0, s,
                      static_cast<const uint4*>(x), H, K_total, sorted, n_pad, static_cast<int>(S),
                      static_cast<int>(max_padded), x_q, x_s, static_cast<uint4*>(x_perm), status);
}

}  // namespace mlora
