// Internal launch interface between the C ABI (api.cu) and the kernel files,
// plus the few device helpers that two kernel files share.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "exp2_poly.h"
#include "fa.h"
#include "sm103_ptx.cuh"

namespace fa {

// Shapes of one call, validated by the C ABI before any launcher runs.
struct Shape {
    int B, H, Hkv, N, d;
    int causal;
    float scale;
    int window = 0;   // causal sliding window W (query i sees keys i - W < j <= i); 0 = none
    // Packed variable-length batches: device array of B + 1 row offsets and
    // the total row count; N is then the longest sequence.  nullptr = dense.
    const int* cu_seqlens = nullptr;
    int total = 0;
};

// Rows [t0, t0 + len) of sequence b of a packed variable-length batch (cu =
// the B + 1 row offsets), clamped to the tensor's rows and to the longest
// sequence N: whatever the offsets hold, every access stays in bounds.
__device__ __forceinline__ int packed_seq(const int* __restrict__ cu, int b, int N,
                                          long long rows, int& t0) {
    long long a = __ldg(cu + b), e = __ldg(cu + b + 1);
    a = a < 0 ? 0 : (a > rows ? rows : a);
    e = e > rows ? rows : e;
    long long len = e - a;
    len = len < 0 ? 0 : (len > N ? N : len);
    t0 = (int)a;
    return (int)len;
}

// 2^x for two fp32 values on the FMA pipe instead of the exponential unit:
// x = n + f with n = rint(x), from the fp32 rounding of x + 1.5 * 2^23 (exact
// for |x| < 2^22), and f = x - n in [-1/2, 1/2], also exact; 2^f by the
// minimax polynomial of exp2_poly.h (Horner, paired FMAs); 2^n by adding n to
// the exponent field (t = x + 1.5 * 2^23 holds 2^22 + n in its mantissa, so
// bits(t) << 23 is n << 23 modulo 2^32).  x is clamped below at -126, so
// -inf (a masked score) gives a value under 2^-126, which the softmax's bf16
// P and fp32 sums treat as zero.  Relative error at most kExp2PolyMaxRelErr
// for results in the normal range.
__device__ __forceinline__ uint64_t exp2_fma2(uint64_t x2) {
    float x0, x1;
    f2_split(x2, x0, x1);
    const uint64_t x = f2(fmaxf(x0, -126.0f), fmaxf(x1, -126.0f));
    const uint64_t magic = f2(12582912.0f, 12582912.0f);
    const uint64_t t = f2_add(x, magic);
    const uint64_t f = f2_sub(x, f2_sub(t, magic));
    uint64_t p = f2_fma(f2(kExp2C3, kExp2C3), f, f2(kExp2C2, kExp2C2));
    p = f2_fma(p, f, f2(kExp2C1, kExp2C1));
    p = f2_fma(p, f, f2(kExp2C0, kExp2C0));
    float t0, t1, p0, p1;
    f2_split(t, t0, t1);
    f2_split(p, p0, p1);
    return f2(__uint_as_float(__float_as_uint(p0) + (__float_as_uint(t0) << 23)),
              __uint_as_float(__float_as_uint(p1) + (__float_as_uint(t1) << 23)));
}
static_assert(kExp2PolyDegree == 3, "exp2_fma2 evaluates a cubic");

// Window value the kernels carry when there is none: the lower edge i - W + 1
// lies below every key index.
constexpr int kNoWindow = 1 << 30;

// Rows of every per-head buffer in the backward workspace are padded to this.
constexpr int kRowPad = 128;
inline int padded_rows(int N) { return (N + kRowPad - 1) / kRowPad * kRowPad; }

// Backward workspace: [lse_ext bf16 B*H*Np x 16][d_ext bf16 B*H*Np x 16]
// [dQacc fp32 B*H*Np*d][work int32], each region 256-byte aligned.  The two
// ext tables
// are the B operands of the K = 16 MMAs that add -LSE (scaled) to S^T and -D
// to dP^T inside the tensor core: per row 16 bf16 columns, stored as
// 8-row x 16-byte core matrices (row group g, K half kc at (2 g + kc) * 128
// bytes), the layout of an unswizzled K-major MMA operand.
struct BwdWorkspace {
    uint16_t* lse_ext;  // cols 0-8: -LSE log2(e) as three bf16 terms, three times
    uint16_t* d_ext;    // cols 9-11: -D = -rowsum(dO o O) as three bf16 terms
    float* dq_acc;      // fp32 accumulator of dQ / scale
    // The dK/dV kernel's work counter (next work item); zeroed by the
    // preprocess, left zero by the dK/dV kernel.
    int* work;
};
constexpr int kExtCols = 16;   // bf16 columns per row of an ext table

// One row of the -LSE table: x = -LSE log2(e) (or -1e30 on a padded row)
// split into three bf16 terms h + m + l (about 24 bits of x), written three
// times into columns 0-8 of workspace row r; columns 9-15 are zero.
__device__ __forceinline__ void write_lse_ext_row(uint16_t* lse_ext, long long r, float x) {
    const float h = bf16_round(x), m = bf16_round(x - h), l = bf16_round(x - h - m);
    uint16_t* row = lse_ext + ((r >> 3) * 2 * 8 + (r & 7)) * 8;   // (2 g + 0) * 64 + (r % 8) * 8
    *reinterpret_cast<uint4*>(row) =
        make_uint4(pack_bf16x2(h, m), pack_bf16x2(l, h), pack_bf16x2(m, l), pack_bf16x2(h, m));
    *reinterpret_cast<uint4*>(row + 64) = make_uint4(pack_bf16x2(l, 0.0f), 0u, 0u, 0u);
}
size_t bwd_workspace_bytes(const Shape& s);
BwdWorkspace bwd_workspace_carve(void* base, const Shape& s);

// Launchers (return a cudaError_t from the launch).
// launch_fwd: train_ws non-null = training forward, which also writes the
// -LSE table and zeroes the dQ accumulator of that backward workspace.
cudaError_t launch_fwd(const Shape& s, const void* q, const void* k, const void* v, void* o,
                       float* lse, bool precise, DeviceStatus* status, cudaStream_t stream,
                       const BwdWorkspace* train_ws = nullptr);
// full = false: only -D (the rest was prepared by the training forward).
cudaError_t launch_bwd_preprocess(const Shape& s, const void* o, bool o_f32, const void* dout,
                                  const float* lse, const BwdWorkspace& ws,
                                  DeviceStatus* status, cudaStream_t stream, bool full = true);
cudaError_t launch_bwd_dkdv(const Shape& s, const void* q, const void* k, const void* v,
                            const void* dout, void* dk, void* dv, const BwdWorkspace& ws,
                            DeviceStatus* status, cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const Shape& s, const BwdWorkspace& ws, void* dq,
                                  cudaStream_t stream);
cudaError_t launch_watchdog_selftest(long long timeout_ns, DeviceStatus* status,
                                     cudaStream_t stream);
// Evaluates exp2_fma2 and ex2.approx.ftz.f32 on n inputs (diagnostic).
cudaError_t launch_exp2_check(const float* x, float* y_fma, float* y_ex2, int n,
                              cudaStream_t stream);
// Exponential-unit throughput microbenchmark (diagnostic): blocks x 256
// threads, each 8 x iters ex2.approx; out holds blocks x 256 floats.
cudaError_t launch_ex2_rate(float* out, int blocks, int iters, cudaStream_t stream);

// Tensor-map encoding through the driver entry point (no libcuda link).
// Builds a 3-D map over a bf16 tensor [outer][rows][d] with a {64, box_rows, 1}
// box and 128-byte swizzle.  Returns false on failure.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int rows, int outer,
                       int box_rows);

// 2-D map over an fp32 matrix [rows][inner] with a {box_inner, box_rows} box
// and 128-byte swizzle (box_inner * 4 <= 128).
bool make_tmap_f32_2d(CUtensorMap* map, const void* base, int inner, long long rows,
                      int box_inner, int box_rows);

// 3-D map over a byte tensor [outer][rows][inner] with a {128, 128, 1} box and
// 128-byte swizzle (inner and rows multiples of 128).
bool make_tmap_u8_3d(CUtensorMap* map, const void* base, int inner, int rows, int outer);

// FP8 buffer: e4m3 codes of V transposed [B*Hkv][d][Np], then fp32 block
// scales of V [B*Hkv][Np/128] and the largest V scale of each kv head
// [B*Hkv]; each region 256-byte aligned.
struct Fp8Buffer {
    uint8_t* v8t;
    float* sv;
    float* svmax;
};
size_t fp8_buffer_bytes(const Shape& s);
Fp8Buffer fp8_buffer_carve(void* base, const Shape& s);
cudaError_t launch_fp8_quantize(const Shape& s, const void* v, const Fp8Buffer& buf,
                                cudaStream_t stream);
cudaError_t launch_fwd_fp8(const Shape& s, const void* q, const void* k, const Fp8Buffer& buf,
                           void* o, float* lse, DeviceStatus* status, cudaStream_t stream);

// Split-KV decoding forward (fa_decode.cu).  Workspace: fp32 partial outputs
// [B][H][Nq][n_split][d] (256-byte aligned end), then fp32 partial LSEs
// [B][H][Nq][n_split]; n_split from decode_split_plan().
void decode_split_plan(int B, int Hkv, int Nk, int d, int* n_split, int* keys_per_split);
size_t decode_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d);
cudaError_t launch_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, int B, int H, int Hkv, int Nq, int Nk, int d,
                              int causal, float scale, DeviceStatus* status,
                              cudaStream_t stream);
constexpr int kDecodeMaxRows = 16;   // (H / Hkv) * Nq rows per kv group

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Counts one kernel launch for fa_kernel_launches().
void count_launch();

// Argument checks of fa_bwd() (without the workspace) and the per-device
// set-up (sm_103 check, status word), for entry points in other files.
fa_status validate_bwd_args(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, const void* dq, const void* dk,
                            const void* dv, int B, int H, int Hkv, int N, int d, float scale);
fa_status ready_device(int* dev, DeviceStatus** status);

}  // namespace fa
