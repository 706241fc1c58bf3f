// tp_mlp_forward with the library's own static device scratch instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is a file-scope __device__ array.  Its host-side name is only a
// stand-in for the symbol, not a device address, so host code never passes it
// to a kernel: the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[TPL_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (nullptr on error).
// The first call on a device does the lookup; later calls return the cache.
void* static_ws_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return nullptr;
        g_static_ptr[dev] = p;
    }
    return g_static_ptr[dev];
}

}  // namespace

extern "C" tpl_status tpl_tp_mlp_forward_static_ws(const void* X, const void* Wg, const void* Wu, const void* Wd,
                                                   void* Y, float* partials, int64_t B, int64_t D, int64_t F,
                                                   int tp, int dtype, int out_dtype, void* stream) {
    TPL_NVTX_RANGE("tpl_tp_mlp_forward_static_ws");
    if (!X || !Wg || !Wu || !Wd || !Y) return TPL_ERR_NULL;
    size_t any = 0;
    const tpl_status s = tpl_tp_mlp_forward_workspace(B, D, F, tp, dtype, &any);   // shape and dtype checks
    if (s != TPL_OK) return s;
    if (!tpl::mlp_out_dtype_ok(dtype, out_dtype)) return TPL_ERR_DTYPE;
    // the scratch this call needs: the plan for the partials argument given
    if (tpl::mlp_plan_bytes(B, D, F, tp, dtype, partials != nullptr) > (size_t)TPL_STATIC_WS_BYTES)
        return TPL_ERR_STATIC_LIMIT;
    // the array used is the current device's, so the stream must be that
    // device's too (the tensors are the caller's to place on it)
    int cur = -1, sdev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return TPL_ERR_CUDA;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return TPL_ERR_CUDA;
    if (sdev != cur) return TPL_ERR_UNSUPPORTED;
    void* ws = static_ws_address();
    if (!ws) return TPL_ERR_CUDA;
    // Nothing in the MLP's scratch has to start at zero: every element of the
    // hidden activations and of the split partials is written before it is
    // read, so what an earlier call left in the array does not matter.
    return tpl_tp_mlp_forward(X, Wg, Wu, Wd, Y, partials, B, D, F, tp, dtype, out_dtype, ws,
                              (size_t)TPL_STATIC_WS_BYTES, stream);
}
