// A forward pass that allocates nothing: the workspace is a fixed device
// array compiled into this library instead of a buffer the caller provides.
//
// For callers that cannot hand the library a workspace -- for example a
// plugin inside a host application that owns every device allocation and
// gives plugins no allocator, or code on a latency-critical path where
// cudaMalloc's implicit device-wide synchronisation is not acceptable.  They
// pass only the weight, the input and the output.
//
// The array is kStaticWorkspaceBytes (32 MiB).  Every GPU on which this
// library's device code is loaded holds those 32 MiB until the process
// exits.  Problems whose workspace (convt3d_workspace_bytes) is larger are
// rejected with CONVT3D_ERR_WORKSPACE before anything is launched.  A
// device-side condition of a call (a bounded wait that ran out) lands in the
// status word at the start of the array; convt3d_check(plan, NULL, stream)
// reads and clears it, and the next call's weight packing clears it too.
#include <mutex>

#include "convt3d_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = (size_t)32 << 20;

// The shared workspace.  In host code this name is only a handle for
// cudaGetSymbolAddress; it is never dereferenced or passed to a kernel.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_device_ptr[kMaxDevices];  // device address of g_static_workspace, per device

}  // namespace

namespace convt3d {
// Device address of the built-in workspace on the current device (looked up
// with that device current on first use, then cached); NULL on failure, with
// the reason recorded for convt3d_last_error.  The cached address stays valid
// for the life of the device's primary context: after cudaDeviceReset the
// library must not be used again in this process.
void *static_workspace_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        report_error("no usable current CUDA device");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_device_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess || !p) {
            report_error("cudaGetSymbolAddress of the built-in workspace: %s", cudaGetErrorString(e));
            return nullptr;
        }
        g_device_ptr[dev] = p;
    }
    return g_device_ptr[dev];
}
}  // namespace convt3d

extern "C" convt3d_status_t convt3d_forward_static_workspace(convt3d_plan_t plan, const void *w, const void *x,
                                                             const float *bias, const float *gamma,
                                                             const float *beta, void *y, void *stream) {
    if (!plan || !w || !x || !y) {
        convt3d::report_error("NULL plan, w, x or y");
        return CONVT3D_ERR_INVALID_ARG;
    }
    const size_t need = convt3d_workspace_bytes(plan);
    if (need > kStaticWorkspaceBytes) {
        convt3d::report_error("problem needs %zu workspace bytes; the built-in workspace holds %zu", need,
                              kStaticWorkspaceBytes);
        return CONVT3D_ERR_WORKSPACE;
    }
    // First call on a device: look up the array's device address with that device current.
    void *ws = convt3d::static_workspace_address();
    if (!ws) return CONVT3D_ERR_CUDA;
    // pack_weights clears the status word at the start of the workspace; every
    // other workspace region is fully rewritten by pack_weights and forward.
    convt3d_status_t st = convt3d_pack_weights(plan, w, ws, kStaticWorkspaceBytes, stream);
    if (st != CONVT3D_OK) return st;
    return convt3d_forward(plan, x, bias, gamma, beta, y, ws, kStaticWorkspaceBytes, stream);
}
