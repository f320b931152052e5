// C ABI of libfa.so (declared in include/fa.h): argument validation, workspace
// layout, tensor-map encoding, the device status word and the launches.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

// One status word per device context (see DeviceStatus).
__device__ DeviceStatus g_status_word;

namespace {

std::atomic<long long> g_launches{0};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr int kMaxDevices = 64;
DeviceStatus* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};   // 0 unknown, 1 sm_103, -1 other
DeviceStatus g_last_detail{};      // last non-zero status word read by the host

bool load_encode() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Checks that the current device is an sm_103 part and fills the per-device
// caches (status word address, SM count).
fa_status device_ready(int* dev_out) {
    const int dev = current_device();
    if (dev < 0) return FA_ERR_CUDA;
    *dev_out = dev;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_sm_count[dev] = sms;
        if (g_arch_ok[dev] == 1) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) {
                g_arch_ok[dev] = 0;
                return FA_ERR_CUDA;
            }
            g_status_ptr[dev] = static_cast<DeviceStatus*>(ptr);
        }
    }
    return g_arch_ok[dev] == 1 ? FA_OK : FA_ERR_UNSUPPORTED;
}

fa_status check_shape(int B, int H, int Hkv, int N, int d) {
    if (B < 1 || H < 1 || Hkv < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const long long np = padded_rows(N);
    if ((long long)B * H * np * d >= (1LL << 31) || (long long)B * H * np >= (1LL << 31))
        return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status check_scale(float scale) {
    return (std::isfinite(scale) && scale > 0.0f) ? FA_OK : FA_ERR_INVALID_ARG;
}

fa_status check_ptr(const void* p) {
    if (!p) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return FA_ERR_ALIGNMENT;
    return FA_OK;
}

fa_status first_error(std::initializer_list<fa_status> l) {
    for (fa_status s : l)
        if (s != FA_OK) return s;
    return FA_OK;
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// For entry points defined in other files: the same argument checks as
// fa_bwd() (without the workspace) and the same per-device set-up.
fa_status validate_bwd_args(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, const void* dq, const void* dk,
                            const void* dv, int B, int H, int Hkv, int N, int d, float scale) {
    return first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                        check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(dout), check_ptr(lse),
                        check_ptr(dq), check_ptr(dk), check_ptr(dv)});
}

fa_status ready_device(int* dev, DeviceStatus** status) {
    const fa_status st = device_ready(dev);
    if (st == FA_OK) *status = g_status_ptr[*dev];
    return st;
}

int device_sm_count() {
    const int dev = current_device();
    return dev < 0 ? 0 : g_sm_count[dev];
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int rows, int outer,
                       int box_rows) {
    if (!load_encode()) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_f32_2d(CUtensorMap* map, const void* base, int inner, long long rows,
                      int box_inner, int box_rows) {
    if (!load_encode()) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 4};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_u8_3d(CUtensorMap* map, const void* base, int inner, int rows, int outer) {
    if (!load_encode()) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)inner * (cuuint64_t)rows};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t bwd_workspace_bytes(const Shape& s) {
    const size_t rows = (size_t)s.B * s.H * padded_rows(s.N);
    return align256(rows * kExtCols * 2) * 2 + align256(rows * (size_t)s.d * 4) + align256(4);
}

BwdWorkspace bwd_workspace_carve(void* base, const Shape& s) {
    const size_t rows = (size_t)s.B * s.H * padded_rows(s.N);
    char* p = static_cast<char*>(base);
    BwdWorkspace w;
    w.lse_ext = reinterpret_cast<uint16_t*>(p);
    w.d_ext = reinterpret_cast<uint16_t*>(p + align256(rows * kExtCols * 2));
    w.dq_acc = reinterpret_cast<float*>(p + 2 * align256(rows * kExtCols * 2));
    w.work = reinterpret_cast<int*>(p + 2 * align256(rows * kExtCols * 2) +
                                    align256(rows * (size_t)s.d * 4));
    return w;
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Hkv, int N, int d, int causal, float scale, fa_stream_t stream) {
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(lse)});
    if (st != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale};
    return from_cuda(
        launch_fwd(s, q, k, v, o, lse, false, g_status_ptr[dev], (cudaStream_t)stream));
}

fa_status fa_fwd_precise(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                         int H, int Hkv, int N, int d, int causal, float scale,
                         fa_stream_t stream) {
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(lse)});
    if (st != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale};
    return from_cuda(
        launch_fwd(s, q, k, v, o, lse, true, g_status_ptr[dev], (cudaStream_t)stream));
}

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Hkv, int N, int d, int window, float scale,
                        fa_stream_t stream) {
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(lse)});
    if (st != FA_OK) return st;
    if (window < 1) return FA_ERR_INVALID_ARG;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const Shape s{B, H, Hkv, N, d, 1, scale, window};
    return from_cuda(
        launch_fwd(s, q, k, v, o, lse, false, g_status_ptr[dev], (cudaStream_t)stream));
}

size_t fa_bwd_workspace_size(int B, int H, int Hkv, int N, int d) {
    if (check_shape(B, H, Hkv, N, d) != FA_OK) return 0;
    return bwd_workspace_bytes(Shape{B, H, Hkv, N, d, 0, 1.0f});
}

static fa_status check_workspace(const void* ws, size_t bytes, const Shape& s) {
    if (!ws) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return FA_ERR_ALIGNMENT;
    if (bytes < bwd_workspace_bytes(s)) return FA_ERR_WORKSPACE;
    return FA_OK;
}

static fa_status bwd_preprocess_impl(const void* o, bool o_f32, const void* dout,
                                     const float* lse, void* workspace, size_t workspace_bytes,
                                     int B, int H, int Hkv, int N, int d, fa_stream_t stream) {
    const Shape s{B, H, Hkv, N, d, 0, 1.0f};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_ptr(o), check_ptr(dout),
                                check_ptr(lse)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_bwd_preprocess(s, o, o_f32, dout, lse,
                                           bwd_workspace_carve(workspace, s), g_status_ptr[dev],
                                           (cudaStream_t)stream));
}

fa_status fa_bwd_preprocess(const void* o, const void* dout, const float* lse, void* workspace,
                            size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                            fa_stream_t stream) {
    return bwd_preprocess_impl(o, false, dout, lse, workspace, workspace_bytes, B, H, Hkv, N, d,
                               stream);
}

fa_status fa_bwd_preprocess_precise(const float* o, const void* dout, const float* lse,
                                    void* workspace, size_t workspace_bytes, int B, int H,
                                    int Hkv, int N, int d, fa_stream_t stream) {
    return bwd_preprocess_impl(o, true, dout, lse, workspace, workspace_bytes, B, H, Hkv, N, d,
                               stream);
}

static fa_status bwd_dkdv_impl(const void* q, const void* k, const void* v, const void* dout,
                               void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                               int H, int Hkv, int N, int d, int causal, float scale, int window,
                               fa_stream_t stream) {
    const Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale, window};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(dout), check_ptr(dk),
                                check_ptr(dv)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_bwd_dkdv(s, q, k, v, dout, dk, dv, bwd_workspace_carve(workspace, s),
                                     g_status_ptr[dev], (cudaStream_t)stream));
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                      int N, int d, int causal, float scale, fa_stream_t stream) {
    return bwd_dkdv_impl(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d,
                         causal, scale, 0, stream);
}

fa_status fa_bwd_dkdv_window(const void* q, const void* k, const void* v, const void* dout,
                             void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                             int H, int Hkv, int N, int d, int window, float scale,
                             fa_stream_t stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return bwd_dkdv_impl(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, 1,
                         scale, window, stream);
}

fa_status fa_bwd_dq_convert(const void* workspace, size_t workspace_bytes, void* dq, int B, int H,
                            int Hkv, int N, int d, float scale, fa_stream_t stream) {
    const Shape s{B, H, Hkv, N, d, 0, scale};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(dq)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_bwd_dq_convert(s, bwd_workspace_carve(const_cast<void*>(workspace), s),
                                           dq, (cudaStream_t)stream));
}

static fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, bool o_f32,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                          int d, int causal, float scale, fa_stream_t stream, int window = 0) {
    const Shape s{B, H, Hkv, N, d, (causal || window > 0) ? 1 : 0, scale, window};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(dout),
                                check_ptr(lse), check_ptr(dq), check_ptr(dk), check_ptr(dv)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const BwdWorkspace ws = bwd_workspace_carve(workspace, s);
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e = launch_bwd_preprocess(s, o, o_f32, dout, lse, ws, g_status_ptr[dev], cs);
    if (e == cudaSuccess) e = launch_bwd_dkdv(s, q, k, v, dout, dk, dv, ws, g_status_ptr[dev], cs);
    if (e == cudaSuccess) e = launch_bwd_dq_convert(s, ws, dq, cs);
    return from_cuda(e);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int causal,
                 float scale, fa_stream_t stream) {
    return bwd_impl(q, k, v, o, false, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H,
                    Hkv, N, d, causal, scale, stream);
}

fa_status fa_bwd_precise(const void* q, const void* k, const void* v, const float* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                         int d, int causal, float scale, fa_stream_t stream) {
    return bwd_impl(q, k, v, o, true, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H,
                    Hkv, N, d, causal, scale, stream);
}

fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                        int d, int window, float scale, fa_stream_t stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, false, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H,
                    Hkv, N, d, 1, scale, stream, window);
}

static fa_status fwd_train_impl(const void* q, const void* k, const void* v, void* o,
                                bool precise, float* lse, void* workspace,
                                size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                                int causal, float scale, fa_stream_t stream, int window = 0) {
    const Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale, window};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(lse)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const BwdWorkspace ws = bwd_workspace_carve(workspace, s);
    return from_cuda(launch_fwd(s, q, k, v, o, lse, precise, g_status_ptr[dev],
                                (cudaStream_t)stream, &ws));
}

fa_status fa_fwd_train(const void* q, const void* k, const void* v, void* o, float* lse,
                       void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                       int d, int causal, float scale, fa_stream_t stream) {
    return fwd_train_impl(q, k, v, o, false, lse, workspace, workspace_bytes, B, H, Hkv, N, d,
                          causal, scale, stream);
}

fa_status fa_fwd_train_precise(const void* q, const void* k, const void* v, float* o,
                               float* lse, void* workspace, size_t workspace_bytes, int B,
                               int H, int Hkv, int N, int d, int causal, float scale,
                               fa_stream_t stream) {
    return fwd_train_impl(q, k, v, o, true, lse, workspace, workspace_bytes, B, H, Hkv, N, d,
                          causal, scale, stream);
}

static fa_status bwd_train_impl(const void* q, const void* k, const void* v, const void* o,
                                bool o_f32, const void* dout, void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                                int N, int d, int causal, float scale, fa_stream_t stream,
                                int window = 0) {
    const Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale, window};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(v), check_ptr(o), check_ptr(dout),
                                check_ptr(dq), check_ptr(dk), check_ptr(dv)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const BwdWorkspace ws = bwd_workspace_carve(workspace, s);
    cudaStream_t cs = (cudaStream_t)stream;
    // -D only (the training forward wrote the -LSE table and zeroed the
    // accumulator), then dK/dV and the dQ conversion.
    cudaError_t e = launch_bwd_preprocess(s, o, o_f32, dout, nullptr, ws, g_status_ptr[dev], cs,
                                          /*full=*/false);
    if (e == cudaSuccess) e = launch_bwd_dkdv(s, q, k, v, dout, dk, dv, ws, g_status_ptr[dev], cs);
    if (e == cudaSuccess) e = launch_bwd_dq_convert(s, ws, dq, cs);
    return from_cuda(e);
}

fa_status fa_bwd_train(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, void* dq, void* dk, void* dv, void* workspace,
                       size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int causal,
                       float scale, fa_stream_t stream) {
    return bwd_train_impl(q, k, v, o, false, dout, dq, dk, dv, workspace, workspace_bytes, B, H,
                          Hkv, N, d, causal, scale, stream);
}

fa_status fa_bwd_train_precise(const void* q, const void* k, const void* v, const float* o,
                               const void* dout, void* dq, void* dk, void* dv, void* workspace,
                               size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                               int causal, float scale, fa_stream_t stream) {
    return bwd_train_impl(q, k, v, o, true, dout, dq, dk, dv, workspace, workspace_bytes, B, H,
                          Hkv, N, d, causal, scale, stream);
}

fa_status fa_fwd_window_train(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                              int N, int d, int window, float scale, fa_stream_t stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return fwd_train_impl(q, k, v, o, false, lse, workspace, workspace_bytes, B, H, Hkv, N, d, 1,
                          scale, stream, window);
}

fa_status fa_bwd_window_train(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                              int window, float scale, fa_stream_t stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return bwd_train_impl(q, k, v, o, false, dout, dq, dk, dv, workspace, workspace_bytes, B, H,
                          Hkv, N, d, 1, scale, stream, window);
}

static fa_status pre_train_impl(const void* o, bool o_f32, const void* dout, void* workspace,
                                size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                                fa_stream_t stream) {
    const Shape s{B, H, Hkv, N, d, 0, 1.0f};
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_ptr(o), check_ptr(dout)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_bwd_preprocess(s, o, o_f32, dout, nullptr,
                                           bwd_workspace_carve(workspace, s), g_status_ptr[dev],
                                           (cudaStream_t)stream, /*full=*/false));
}

fa_status fa_bwd_preprocess_train(const void* o, const void* dout, void* workspace,
                                  size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                                  fa_stream_t stream) {
    return pre_train_impl(o, false, dout, workspace, workspace_bytes, B, H, Hkv, N, d, stream);
}

fa_status fa_bwd_preprocess_train_precise(const float* o, const void* dout, void* workspace,
                                          size_t workspace_bytes, int B, int H, int Hkv, int N,
                                          int d, fa_stream_t stream) {
    return pre_train_impl(o, true, dout, workspace, workspace_bytes, B, H, Hkv, N, d, stream);
}

static fa_status check_varlen(const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                              int Hkv, int d) {
    fa_status st = check_shape(B, H, Hkv, max_seqlen, d);
    if (st != FA_OK) return st;
    if (!cu_seqlens || total < 1) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cu_seqlens) % alignof(int) != 0) return FA_ERR_ALIGNMENT;
    if ((long long)H * total * d >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens, int B, int max_seqlen, int total, int H, int Hkv,
                        int d, int causal, float scale, fa_stream_t stream) {
    fa_status st = first_error({check_varlen(cu_seqlens, B, max_seqlen, total, H, Hkv, d),
                                check_scale(scale), check_ptr(q), check_ptr(k), check_ptr(v),
                                check_ptr(o), check_ptr(lse)});
    if (st != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    Shape s{B, H, Hkv, max_seqlen, d, causal ? 1 : 0, scale};
    s.cu_seqlens = cu_seqlens;
    s.total = total;
    return from_cuda(
        launch_fwd(s, q, k, v, o, lse, false, g_status_ptr[dev], (cudaStream_t)stream));
}

size_t fa_bwd_varlen_workspace_size(int B, int H, int Hkv, int max_seqlen, int d) {
    return fa_bwd_workspace_size(B, H, Hkv, max_seqlen, d);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, const int* cu_seqlens, int B,
                        int max_seqlen, int total, int H, int Hkv, int d, int causal, float scale,
                        fa_stream_t stream) {
    Shape s{B, H, Hkv, max_seqlen, d, causal ? 1 : 0, scale};
    s.cu_seqlens = cu_seqlens;
    s.total = total;
    fa_status st = first_error({check_varlen(cu_seqlens, B, max_seqlen, total, H, Hkv, d),
                                check_scale(scale), check_ptr(q), check_ptr(k), check_ptr(v),
                                check_ptr(o), check_ptr(dout), check_ptr(lse), check_ptr(dq),
                                check_ptr(dk), check_ptr(dv)});
    if (st != FA_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    const BwdWorkspace ws = bwd_workspace_carve(workspace, s);
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e = launch_bwd_preprocess(s, o, false, dout, lse, ws, g_status_ptr[dev], cs);
    if (e == cudaSuccess) e = launch_bwd_dkdv(s, q, k, v, dout, dk, dv, ws, g_status_ptr[dev], cs);
    if (e == cudaSuccess) e = launch_bwd_dq_convert(s, ws, dq, cs);
    return from_cuda(e);
}

fa_status fa_device_status(fa_stream_t stream) {
    int dev;
    fa_status st = device_ready(&dev);
    if (st != FA_OK) return st;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FA_ERR_CUDA;
    DeviceStatus w{};
    if (cudaMemcpyFromSymbol(&w, g_status_word, sizeof(w)) != cudaSuccess) return FA_ERR_CUDA;
    if (w.code != 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        g_last_detail = w;
    }
    const DeviceStatus zero{};
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return static_cast<fa_status>(w.code);
}

void fa_device_status_detail(int* site, int* block) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (site) *site = g_last_detail.site;
    if (block) *block = g_last_detail.block;
}

fa_status fa_watchdog_selftest(long long timeout_ns, fa_stream_t stream) {
    int dev;
    fa_status st = device_ready(&dev);
    if (st != FA_OK) return st;
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 5000000000LL) timeout_ns = 5000000000LL;
    return from_cuda(launch_watchdog_selftest(timeout_ns, g_status_ptr[dev], (cudaStream_t)stream));
}

fa_status fa_exp2_check(const float* x, float* y_fma, float* y_ex2, int n, fa_stream_t stream) {
    if (n < 1 || !x || !y_fma || !y_ex2) return FA_ERR_INVALID_ARG;
    int dev;
    fa_status st = device_ready(&dev);
    if (st != FA_OK) return st;
    return from_cuda(launch_exp2_check(x, y_fma, y_ex2, n, (cudaStream_t)stream));
}

fa_status fa_ex2_rate(float* out, int blocks, int iters, fa_stream_t stream) {
    if (!out || blocks < 1 || iters < 1 || blocks > (1 << 20) || iters > (1 << 24))
        return FA_ERR_INVALID_ARG;
    int dev;
    fa_status st = device_ready(&dev);
    if (st != FA_OK) return st;
    return from_cuda(launch_ex2_rate(out, blocks, iters, (cudaStream_t)stream));
}

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

long long fa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t fa_fp8_buffer_size(int B, int H, int Hkv, int N, int d) {
    if (check_shape(B, H, Hkv, N, d) != FA_OK || d != 128) return 0;
    return fp8_buffer_bytes(Shape{B, H, Hkv, N, d, 0, 1.0f});
}

static fa_status check_fp8_buffer(const void* buf, size_t bytes, const Shape& s) {
    if (!buf) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(buf) % 256 != 0) return FA_ERR_ALIGNMENT;
    if (bytes < fp8_buffer_bytes(s)) return FA_ERR_WORKSPACE;
    return FA_OK;
}

fa_status fa_fp8_quantize(const void* v, void* fp8_buf, size_t fp8_buf_bytes, int B, int H,
                          int Hkv, int N, int d, fa_stream_t stream) {
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_ptr(v)});
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    const Shape s{B, H, Hkv, N, d, 0, 1.0f};
    if ((st = check_fp8_buffer(fp8_buf, fp8_buf_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_fp8_quantize(s, v, fp8_buffer_carve(fp8_buf, s), (cudaStream_t)stream));
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* fp8_buf, size_t fp8_buf_bytes,
                     void* o, float* lse, int B, int H, int Hkv, int N, int d, int causal,
                     float scale, fa_stream_t stream) {
    fa_status st = first_error({check_shape(B, H, Hkv, N, d), check_scale(scale), check_ptr(q),
                                check_ptr(k), check_ptr(o), check_ptr(lse)});
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    const Shape s{B, H, Hkv, N, d, causal ? 1 : 0, scale};
    if ((st = check_fp8_buffer(fp8_buf, fp8_buf_bytes, s)) != FA_OK) return st;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_fwd_fp8(s, q, k, fp8_buffer_carve(const_cast<void*>(fp8_buf), s), o,
                                    lse, g_status_ptr[dev], (cudaStream_t)stream));
}

static fa_status check_decode_shape(int B, int H, int Hkv, int Nq, int Nk, int d) {
    if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < Nq || d < 1 || H % Hkv != 0)
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if ((long long)(H / Hkv) * Nq > kDecodeMaxRows) return FA_ERR_UNSUPPORTED;
    if ((long long)B * Hkv * Nk * d >= (1LL << 31) || (long long)B * H * Nq * d >= (1LL << 31))
        return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

size_t fa_fwd_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d) {
    if (check_decode_shape(B, H, Hkv, Nq, Nk, d) != FA_OK) return 0;
    return decode_workspace_bytes(B, H, Hkv, Nq, Nk, d);
}

fa_status fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                        void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nq,
                        int Nk, int d, int causal, float scale, fa_stream_t stream) {
    fa_status st = first_error({check_decode_shape(B, H, Hkv, Nq, Nk, d), check_scale(scale),
                                check_ptr(q), check_ptr(k), check_ptr(v), check_ptr(o),
                                check_ptr(lse)});
    if (st != FA_OK) return st;
    if (!workspace || workspace_bytes < decode_workspace_bytes(B, H, Hkv, Nq, Nk, d))
        return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return FA_ERR_ALIGNMENT;
    int dev;
    if ((st = device_ready(&dev)) != FA_OK) return st;
    return from_cuda(launch_fwd_decode(q, k, v, o, lse, workspace, B, H, Hkv, Nq, Nk, d,
                                       causal ? 1 : 0, scale, g_status_ptr[dev],
                                       (cudaStream_t)stream));
}

}  // extern "C"
