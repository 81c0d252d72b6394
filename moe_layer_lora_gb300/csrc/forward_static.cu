// forward_static.cu -- mlora_moe_forward_static: the fused MoE-LoRA layer
// with its scratch memory in a fixed device array of this library instead
// of a workspace the caller allocates.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at
// the point where they run the layer -- code embedded in a host program
// whose device memory is owned by another allocator it must not bypass,
// code that may not allocate after start-up (fixed memory budgets,
// latency-critical paths where an allocation can synchronise the device),
// or thin bindings that only receive pointers to tensors.  Those callers
// still pass every input and output; only the scratch is provided here.
//
// The array lives in the module's global memory: each GPU on which the
// library's kernels are loaded reserves MLORA_STATIC_WORKSPACE_BYTES for it
// and keeps that memory until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kStaticBytes = MLORA_STATIC_WORKSPACE_BYTES;

// Shared by every call on a device; it keeps the contents of the last call.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct StaticSlot {
    void* ptr = nullptr;
    unsigned long long ctx_id = 0;  // context the address belongs to
};
StaticSlot g_static[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the current CUDA context (0 when it cannot be told).  A device's
// primary context is re-created after cudaDeviceReset, and the array then
// has a new address: the cached one belongs to the old context.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the array on the current device.  In host code the
// symbol is only a host-side stand-in, so the address has to be asked for,
// once per device and context, with that device current.
mlora_status static_workspace(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLORA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLORA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    StaticSlot& slot = g_static[dev];
    if (!slot.ptr || slot.ctx_id != current_context_id()) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) {
            slot.ptr = nullptr;
            return MLORA_ERR_CUDA;
        }
        slot.ptr = p;
        // the lookup made the device's context current: its id is the one
        // later calls compare against
        slot.ctx_id = current_context_id();
    }
    *out = slot.ptr;
    return MLORA_OK;
}

}  // namespace

extern "C" mlora_status mlora_moe_forward_static(const void* x, const void* w13, const void* w2, const void* A13,
                                                 const void* B13, const void* A2, const void* B2,
                                                 const int32_t* token_lora_idx, const int32_t* topk_ids,
                                                 const float* topk_w, int M, int H, int I, int E_tot, int K_total,
                                                 int L, int rank, float scaling, int n_shared, float out_scale,
                                                 void* y, void* stream) {
    const bool lora = A13 && B13 && A2 && B2 && token_lora_idx && L > 0 && rank > 0;
    const size_t need = mlora_moe_workspace_size(M, H, I, E_tot, K_total, lora ? L : 0, lora ? rank : 0);
    if (need == 0) {
        // invalid sizes: the regular entry point reports which check failed
        // before it touches the workspace or the device
        return mlora_moe_forward(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, M, H, I, E_tot,
                                 K_total, L, rank, scaling, n_shared, out_scale, y, nullptr, 0, stream);
    }
    if (need > kStaticBytes) return MLORA_ERR_WORKSPACE;
    void* ws = nullptr;
    const mlora_status st = static_workspace(&ws);
    if (st != MLORA_OK) return st;
    return mlora_moe_forward(x, w13, w2, A13, B13, A2, B2, token_lora_idx, topk_ids, topk_w, M, H, I, E_tot,
                             K_total, L, rank, scaling, n_shared, out_scale, y, ws, kStaticBytes, stream);
}

// The status word sits at the start of the array, as at the start of a
// caller's workspace.
extern "C" mlora_status mlora_moe_read_status_static(uint32_t* host_status, void* stream) {
    if (!host_status) return MLORA_ERR_INVALID_ARG;
    void* ws = nullptr;
    const mlora_status st = static_workspace(&ws);
    if (st != MLORA_OK) return st;
    return mlora_moe_read_status(ws, host_status, stream);
}
