// tp_static_ws.cu -- tp_mlp_block_static_ws: the MLP block for callers that
// cannot allocate device memory.
//
// tp_mlp_block needs scratch for the hidden activation H [M, f] and takes it
// from the caller.  Some callers have no way to provide it: a serving loop
// that must not call cudaMalloc once it is running (cudaMalloc can
// synchronise the whole device and stall every other stream), or a host
// framework that owns all device memory through its own pool and hands a
// library only the input and output tensors.  For them this entry point keeps
// the scratch in a fixed array that is part of the library's device image:
// it is reserved when the library's module is loaded on a device and stays
// reserved on every device that loads the library until the process exits.
//
// The array's name seen from host code is only a host-side stand-in for the
// symbol, not a device address (a kernel given it would fault, or silently
// use the wrong memory where the GPU can reach host memory).  Its device
// address is obtained once per device with cudaGetSymbolAddress, with that
// device current, and then passed on like any caller-owned workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tp.h"

namespace {

// The fixed scratch: holds H for one call at a time.
static __device__ __align__(256) unsigned char g_static_ws[TP_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mutex;
void *g_ws_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, looked up on the
// first call for that device and cached.  Returns nullptr on failure.
void *static_ws_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if (g_ws_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess) return nullptr;
        g_ws_ptr[dev] = p;
    }
    return g_ws_ptr[dev];
}

}  // namespace

extern "C" tp_status tp_mlp_block_static_ws(const void *X, const void *W1, const void *W2,
                                            void *Y, int64_t M, int64_t d, int64_t f,
                                            int n_shards, tp_dtype in_t, tp_dtype out_t,
                                            cudaStream_t s) {
    const size_t need = tp_mlp_block_workspace_size(M, f, in_t);
    if (need > static_cast<size_t>(TP_STATIC_WS_BYTES)) return TP_ERR_WORKSPACE;
    void *ws = nullptr;
    if (need > 0) {
        ws = static_ws_address();
        if (ws == nullptr) return TP_ERR_CUDA;
    }
    return tp_mlp_block(X, W1, W2, Y, ws, static_cast<size_t>(TP_STATIC_WS_BYTES), M, d, f,
                        n_shards, in_t, out_t, s);
}
