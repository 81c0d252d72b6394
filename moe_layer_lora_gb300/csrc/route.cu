// route.cu -- top-k routing, one warp per token.
//
// Softmax top-k (selection on the raw logits, weights = softmax of the
// selected logits, or of all when not renormalising) and sigmoid+bias top-k
// (selection on sigmoid(l)+b in fp32, weights sigmoid(l)), followed by the
// forced shared-expert slots of "[vllm] vLLM ROCm 환경에서 Shared-Expert
// Fusion을 통한 MoE 추론 성능 최적화", section "코드 분석" item 1 (ids E..E+n-1
// after the routed slots) with weight 1/routed_scaling_factor (section
// "교훈" item 2).  Ranking: descending key, ties to the lower expert id.
//
// Each lane holds experts lane, lane+32, ... in registers (coalesced row
// read); every selection step is one arg-max over the warp.
// Non-finite input never yields an id outside [0, E): a NaN key ranks
// last (ties among them to the lower id); the weights of such a token are
// then NaN as well.
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace mlora {
namespace {

__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// A non-NaN float as an unsigned integer of the same order (-0 folded into
// +0, which compare equal as floats), for the warp's integer max reduction.
__device__ __forceinline__ unsigned ordered(float k) {
    const unsigned u = __float_as_uint(k == 0.0f ? 0.0f : k);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                    int M, int E, int top_k, int scoring, int renormalize,
                                                    int n_shared, float inv_rsf, int32_t* __restrict__ ids,
                                                    float* __restrict__ w) {
    griddep_wait();
    griddep_launch_dependents();
    const int token = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (token >= M) return;  // whole warp leaves together
    const float* l = logits + static_cast<size_t>(token) * E;

    float raw[VPL], key[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        const int e = lane + 32 * v;
        if (e < E) {
            raw[v] = l[e];
            const float k = scoring == MLORA_SCORE_SOFTMAX ? raw[v]
                                                           : 1.0f / (1.0f + expf(-raw[v])) + (bias ? bias[e] : 0.0f);
            // a NaN key ranks below every number (and equal NaN keys go to
            // the lower id), so every selected id is a real expert
            key[v] = isnan(k) ? -INFINITY : k;
        } else {
            raw[v] = -INFINITY;
            key[v] = -INFINITY;
        }
    }

    const int KT = top_k + n_shared;
    int32_t* oid = ids + static_cast<size_t>(token) * KT;
    float* ow = w + static_cast<size_t>(token) * KT;

    float my_raw[2] = {0.f, 0.f};  // raw logit of slots k = lane and k = lane + 32
    int my_id[2] = {0, 0};
    if constexpr (VPL <= 8) {
        // each lane's candidates as a queue, best first (descending key,
        // then ascending id; ids ascend with v, so a stable sort keeps equal
        // keys in id order).  A selection is the head of the lane whose head
        // is the warp's best -- the largest key, then (only when lanes tie)
        // the lowest id -- and only that lane's queue moves.  Slots past E
        // rank below every key.
        unsigned q_ok[VPL];
        int q_id[VPL];
        float q_raw[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const int e = lane + 32 * v;
            q_ok[v] = e < E ? ordered(key[v]) : 0u;
            q_id[v] = e;
            q_raw[v] = raw[v];
        }
#pragma unroll
        for (int i = 1; i < VPL; ++i) {
#pragma unroll
            for (int j = i; j > 0; --j) {
                if (q_ok[j] > q_ok[j - 1]) {
                    const unsigned to = q_ok[j];
                    const int ti = q_id[j];
                    const float tr = q_raw[j];
                    q_ok[j] = q_ok[j - 1];
                    q_id[j] = q_id[j - 1];
                    q_raw[j] = q_raw[j - 1];
                    q_ok[j - 1] = to;
                    q_id[j - 1] = ti;
                    q_raw[j - 1] = tr;
                }
            }
        }
        for (int k = 0; k < top_k; ++k) {
            const unsigned kmax = __reduce_max_sync(0xffffffffu, q_ok[0]);
            const unsigned tied = __ballot_sync(0xffffffffu, q_ok[0] == kmax);
            int owner;
            if (__popc(tied) == 1)  // the same for every lane
                owner = __ffs(tied) - 1;
            else
                owner = static_cast<int>(
                    __reduce_min_sync(0xffffffffu, q_ok[0] == kmax ? static_cast<unsigned>(q_id[0]) : 0xffffffffu) &
                    31u);
            const int sid = __shfl_sync(0xffffffffu, q_id[0], owner);
            const float sraw = __shfl_sync(0xffffffffu, q_raw[0], owner);
            if ((k & 31) == lane) {
                my_raw[k >> 5] = sraw;
                my_id[k >> 5] = sid;
            }
            if (lane == owner) {
#pragma unroll
                for (int v = 0; v + 1 < VPL; ++v) {
                    q_ok[v] = q_ok[v + 1];
                    q_id[v] = q_id[v + 1];
                    q_raw[v] = q_raw[v + 1];
                }
                q_ok[VPL - 1] = 0u;
            }
        }
    } else {
        uint32_t taken = 0;
        for (int k = 0; k < top_k; ++k) {
            float bk = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int e = lane + 32 * v;
                if (e < E && !((taken >> v) & 1u) && better(key[v], e, bk, bi)) {
                    bk = key[v];
                    bi = e;
                }
            }
            // the warp's arg-max: the largest key, then the lowest id among
            // the lanes holding it (two warp reductions)
            const unsigned ok = ordered(bk);
            const unsigned kmax = __reduce_max_sync(0xffffffffu, ok);
            bi = static_cast<int>(__reduce_min_sync(0xffffffffu, ok == kmax ? static_cast<unsigned>(bi) : 0x7fffffffu));
            const int owner = bi & 31, vsel = bi >> 5;
            float r = 0.f;
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                if (v == vsel) r = raw[v];
            r = __shfl_sync(0xffffffffu, r, owner);
            if (lane == owner) taken |= 1u << vsel;
            if ((k & 31) == lane) {
                my_raw[k >> 5] = r;
                my_id[k >> 5] = bi;
            }
        }
    }

    // weights of the routed slots this lane owns
    float val[2] = {0.f, 0.f};
    float part = 0.f;
    if (scoring == MLORA_SCORE_SOFTMAX) {
        // the first selected logit is the row maximum
        const float lmax = __shfl_sync(0xffffffffu, my_raw[0], 0);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (lane + 32 * h < top_k) val[h] = expf(my_raw[h] - lmax);
        if (renormalize) {
            part = val[0] + val[1];
        } else {
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                if (lane + 32 * v < E) part += expf(raw[v] - lmax);
        }
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (lane + 32 * h < top_k) val[h] = 1.0f / (1.0f + expf(-my_raw[h]));
        part = val[0] + val[1];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const bool divide = scoring == MLORA_SCORE_SOFTMAX || renormalize;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int k = lane + 32 * h;
        if (k < top_k) {
            oid[k] = my_id[h];
            ow[k] = divide ? val[h] / part : val[h];
        }
    }
    for (int j = lane; j < n_shared; j += 32) {
        oid[top_k + j] = E + j;
        ow[top_k + j] = inv_rsf;
    }
}

}  // namespace

cudaError_t launch_route(const float* logits, const float* bias, int M, int E, int top_k, int scoring,
                         int renormalize, int n_shared, float inv_rsf, int32_t* ids, float* w, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    const dim3 block(256);
    const dim3 grid((M + 7) / 8);
    const int vpl = (E + 31) / 32;
#define MLORA_ROUTE_CASE(V)                                                                                 \
    return launch_pdl(route_kernel<V>, grid, block, 0, s, logits, bias, M, E, top_k, scoring, renormalize, n_shared, \
                      inv_rsf, ids, w);
    switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32) {
        case 1: MLORA_ROUTE_CASE(1)
        case 2: MLORA_ROUTE_CASE(2)
        case 4: MLORA_ROUTE_CASE(4)
        case 8: MLORA_ROUTE_CASE(8)
        case 16: MLORA_ROUTE_CASE(16)
        default: MLORA_ROUTE_CASE(32)
    }
#undef MLORA_ROUTE_CASE
}

}  // namespace mlora
