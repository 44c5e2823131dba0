// static_scratch.cu -- moe_decode_layer_static: the decode layer for callers
// that cannot allocate device memory.
//
// Some callers have no way to provide a workspace: a plugin whose host
// engine owns all device memory and forbids allocation while it runs, a
// runtime that freezes allocation after start-up to keep latency
// deterministic, or code with no handle to its framework's allocator.  This
// entry point runs the same kernels as moe_decode_layer, with the scratch
// taken from one fixed array in the library's device memory instead of the
// caller's workspace.  It allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine.
#include <cstddef>
#include <cstdio>

#include "common.cuh"

namespace moe {
moe_status report_error(moe_status status, const char* message);
}

namespace {

// The fixed scratch array.  Every GPU that loads the library holds it until
// the process exits.  Calls share it and it keeps the last call's contents.
constexpr size_t kScratchBytes = MOE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch on the current device (in host code the
// symbol is only a host-side stand-in).  Looked up on every call: the lookup
// allocates nothing, and an address kept across calls would be stale after
// the device's context is reset and the module loaded again.
moe_status scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return moe::report_error(MOE_ERR_CUDA, cudaGetErrorString(e));
    *out = p;
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_decode_layer_static(const void* hidden, const void* w_router, const float* router_bias,
                                              const void* w_gate, const void* w_up, const void* w_down,
                                              int32_t d_ff, const moe_route_params* params,
                                              const moe_routing* routing, void* out, moe_stream_t stream) {
    const size_t need = moe_workspace_bytes(params, d_ff);
    if (need == 0) return MOE_ERR_ARG;   // the reason is already recorded
    if (need > kScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof msg, "this batch needs %zu bytes of scratch; the fixed array holds %zu", need,
                 kScratchBytes);
        return moe::report_error(MOE_ERR_WORKSPACE, msg);
    }
    void* ws = nullptr;
    moe_status st = scratch_address(&ws);
    if (st != MOE_OK) return st;
    // The counters at the front of the scratch must start at zero.  The flag
    // word (the header's first four bytes) is kept, so that flags raised by
    // earlier calls stay readable with moe_device_status_static().
    const moe::WsLayout L = moe::ws_layout(params->B, params->N, params->d, moe_num_slots(params), d_ff,
                                           params->dtype == MOE_DTYPE_BF16 ? 2 : 4);
    static_assert(offsetof(moe::WsHeader, flags) == 0, "the flag word leads the header");
    cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(ws) + sizeof(uint32_t), 0,
                                    L.pos_of - sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return moe::report_error(MOE_ERR_CUDA, cudaGetErrorString(e));
    return moe_decode_layer(hidden, w_router, router_bias, w_gate, w_up, w_down, d_ff, params, routing, out, ws,
                            kScratchBytes, stream);
}

extern "C" moe_status moe_device_status_static(moe_stream_t stream, uint32_t* flags) {
    void* ws = nullptr;
    moe_status st = scratch_address(&ws);
    if (st != MOE_OK) return st;
    return moe_device_status(ws, stream, flags);
}
