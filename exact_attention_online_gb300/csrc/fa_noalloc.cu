// fa_bwd_static_scratch: the backward pass for callers that cannot allocate
// device memory.
//
// fa_bwd() needs a caller-provided workspace (D, a padded base-2 copy of LSE
// and the fp32 dQ accumulator).  Some callers cannot obtain one: they run
// where cudaMalloc is not allowed or not wanted - a runtime that hands out
// all device memory from its own fixed pool and forbids other allocations, a
// latency-critical loop that must not risk the device-wide synchronisation
// cudaMalloc can cause, or a plugin with no handle on the host application's
// allocator.  This entry point keeps that scratch in a fixed array in device
// memory that belongs to the library, so the caller passes only inputs and
// outputs.
//
// The array has a fixed size (kScratchBytes, 32 MiB) and every GPU that
// loads the library holds it until the process exits.  Problems whose
// workspace (fa_bwd_workspace_size) is larger are rejected with
// FA_ERR_WORKSPACE.  All calls on a device share the one array: calls whose
// kernels overlap on the GPU (on different streams, or from different
// threads without ordering) race on it; serialise them on one stream.  The
// array keeps the previous call's contents; every region the kernels read is
// rewritten by the first kernel of each call (D, LSE copy, zeroed dQ
// accumulator), so nothing stale is used.
//
// In host code the array's name is only a host-side stand-in for the device
// symbol, so its device address is fetched with cudaGetSymbolAddress, once
// per device, with that device current, by the first call made on the device.
// That first call on each device should therefore come before any stream
// capture.  No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// The backward's scratch: D, LSE copy and dQ accumulator, carved exactly as
// the caller-provided workspace of fa_bwd().
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on `dev` (the current device), looked up
// once per device.
fa_status scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_static_scratch(const void* q, const void* k, const void* v,
                                           const void* o, const void* dout, const float* lse,
                                           void* dq, void* dk, void* dv, int B, int H, int Hkv,
                                           int N, int d, int causal, float scale,
                                           fa_stream_t stream) {
    fa_status st = fa::validate_bwd_args(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (fa_bwd_workspace_size(B, H, Hkv, N, d) > kScratchBytes) return FA_ERR_WORKSPACE;
    int dev = -1;
    fa::DeviceStatus* status = nullptr;
    if ((st = fa::ready_device(&dev, &status)) != FA_OK) return st;
    void* scratch = nullptr;
    if ((st = scratch_address(dev, &scratch)) != FA_OK) return st;
    const fa::Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale};
    const fa::BwdWorkspace ws = fa::bwd_workspace_carve(scratch, s);
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e = fa::launch_bwd_preprocess(s, o, false, dout, lse, ws, status, cs);
    if (e == cudaSuccess) e = fa::launch_bwd_dkdv(s, q, k, v, dout, dk, dv, ws, status, cs);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_convert(s, ws, dq, cs);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
