// Forward kernel: exact attention with the online-softmax recurrence, tiled so
// the N x N score matrix never leaves the SM (FlashAttention blog, "From Online
// Softmax to FlashAttention" and "FlashAttention"; FlashAttention-2 review
// thread, author answers on non-matmul FLOPs and on Figure 2).
//
// One CTA owns two 128-row query tiles (t = 0, 1) of one (batch, head) and
// streams 128-key K/V tiles through a shared-memory ring:
//   warp 8      TMA producer: Q tiles once, then K_j, V_j into the ring.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (SS MMA),
//               O_t += P_t V_j with P_t read from TMEM (TS MMA).
//   warps 0-3   softmax for tile 0, warps 4-7 for tile 1: one query row per
//               thread (warps 10-11 are idle).  While one group does its softmax the tensor core
//               runs the other tile's MMAs.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  P_t (bf16 pairs) overwrites the
// first half of S_t; the MMA that next writes S_t is issued after the MMA
// that reads P_t, and tcgen05 MMAs of one thread execute in order.
//
// Softmax in base 2: p = 2^(S*c - m) with c = scale*log2(e).  The running max
// m is only raised when the block max exceeds it by more than 8 (a factor
// 256), so most blocks skip the O rescale; numerator and denominator always
// use the same m, so the result is unchanged in exact arithmetic.  O is
// divided by l once, in the epilogue, and LSE = ln2 * (m + log2 l).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kTiles = 2;         // query tiles per CTA
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = 12 * 32;   // 3 warpgroups: softmax 0, softmax 1, control
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;         // warps 10-11 only take part in set-up and teardown
// Register split (setmaxnreg): the launch gives 384 x 168; the control
// warpgroup drops to 56 so each softmax thread can hold a full 128-score row:
// 128 x 56 + 256 x 224 = 64512 <= 384 x 168 = 64512.
constexpr int kRegsControl = 56;
constexpr int kRegsSoftmax = 224;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct FwdCfg {
    static constexpr int kStages = (D == 128) ? 2 : 3;
    static constexpr int kTileBytes = kBM * D * 2;          // one Q, K or V tile
    static constexpr int kChunks = D / 64;                  // 128-byte swizzle chunks
    static constexpr int kChunkBytes = 128 * 128;           // 128 rows x 128 bytes
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTiles * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kSmemBytes = kOffV + kStages * kTileBytes;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;    // alignment slack
    // TMEM columns
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
};

struct FwdParams {
    int H, Hkv, N, BH, n_mblk, causal;
    float scale_log2;                 // scale * log2(e)
    __nv_bfloat16* o;
    float* lse;
    DeviceStatus* status;
};

// K-major operand tile with 128-byte swizzle: 16-element K step kk.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
    return sdesc_sw128(base + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
}
// MN-major V tile (keys x d, d contiguous): 16-key step kk.
__device__ __forceinline__ uint64_t vmn_desc(uint32_t base, int kk) {
    return sdesc_sw128(base + kk * (16 * 128), 128 * 128, 1024);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using Cfg = FwdCfg<D>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_q, bar_k[S], bar_v[S], bar_kv_empty[S];
    __shared__ uint64_t bar_s[kTiles], bar_p[kTiles], bar_o[kTiles];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    const WaitCtx wc{p.status, &abort_sh};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Tile -> (query block pair, batch*head).  Under the causal mask the
    // longest query blocks are dispatched first.
    const int idx = blockIdx.x;
    const int mb_rank = idx / p.BH;
    const int bh = idx % p.BH;
    const int m_blk = CAUSAL ? (p.n_mblk - 1 - mb_rank) : mb_rank;
    const int b = bh / p.H, h = bh % p.H;
    const int kv_bh = b * p.Hkv + h / (p.H / p.Hkv);
    const int n_kv_all = (p.N + kBN - 1) / kBN;
    const int n_kv = CAUSAL ? min(n_kv_all, 2 * m_blk + 2) : n_kv_all;
    const int row_base = m_blk * (kTiles * kBM);

    if (threadIdx.x == 0) {
        abort_sh = 0;
        mbar_init(&bar_q, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(&bar_k[s], 1);
            mbar_init(&bar_v[s], 1);
            mbar_init(&bar_kv_empty[s], 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bar_s[t], 1);
            mbar_init(&bar_p[t], 128);
            mbar_init(&bar_o[t], 1);
        }
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    uint8_t* sQ = smem + Cfg::kOffQ;
    uint8_t* sK = smem + Cfg::kOffK;
    uint8_t* sV = smem + Cfg::kOffV;

    // One register-budget change per warpgroup, executed by all its warps at
    // the same instruction; each role's code is dominated by exactly one.
    if (warp < kSoftmaxWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;                 // query tile of this group
        const int quarter = warp & 3;            // TMEM lane quarter
        const int rl = quarter * 32 + lane;      // row within the tile
        const int row0 = row_base + t * kBM;
        const int row = row0 + rl;
        const uint32_t col_s = t ? Cfg::kColS1 : Cfg::kColS0;
        const uint32_t col_o = t ? Cfg::kColO1 : Cfg::kColO0;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const float c = p.scale_log2;
        float m2 = -CUDART_INF_F;   // running max, log2-scaled
        float l = 0.0f;
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            if (!fa_wait_warp(&bar_s[t], j & 1, 30 + t, wc)) { ok = false; break; }
            tc_fence_after();
            uint32_t r[4][32];
            tmem_ld32(lane_addr + col_s + 0, r[0]);
            tmem_ld32(lane_addr + col_s + 32, r[1]);
            tmem_ld32(lane_addr + col_s + 64, r[2]);
            tmem_ld32(lane_addr + col_s + 96, r[3]);
            tmem_ld_wait(r[0]);
            asm volatile("" : FA_R32(r[1]) : : "memory");
            asm volatile("" : FA_R32(r[2]) : : "memory");
            asm volatile("" : FA_R32(r[3]) : : "memory");
            float sv[kBN];
#pragma unroll
            for (int e = 0; e < kBN; ++e) sv[e] = __uint_as_float(r[e >> 5][e & 31]);

            const int col0 = j * kBN;
            const bool need_mask = (CAUSAL && col0 + kBN - 1 > row0) || (col0 + kBN > p.N);
            if (need_mask) {
                const int lim_causal = CAUSAL ? row - col0 : kBN;   // keep e <= row - col0
                const int lim_n = p.N - col0;                        // keep e < N - col0
#pragma unroll
                for (int e = 0; e < kBN; ++e)
                    if (e > lim_causal || e >= lim_n) sv[e] = -CUDART_INF_F;
            }
            float mx4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
            for (int e = 4; e < kBN; e += 4) {
                mx4[0] = fmaxf(mx4[0], sv[e]);
                mx4[1] = fmaxf(mx4[1], sv[e + 1]);
                mx4[2] = fmaxf(mx4[2], sv[e + 2]);
                mx4[3] = fmaxf(mx4[3], sv[e + 3]);
            }
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            const float mx2 = mx * c;
            const bool need = mx2 > m2 + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? mx2 : m2;
                const float alpha = (m_new == m2) ? 1.0f : ex2(m2 - m_new);
                l *= alpha;
                if (j > 0) {
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32(lane_addr + col_o + c0, ov);
                        tmem_ld_wait(ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(lane_addr + col_o + c0, ov);
                    }
                }
                m2 = m_new;
            }
            const float m_use = (m2 == -CUDART_INF_F) ? 0.0f : m2;
            float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            uint32_t pk[2][32];
#pragma unroll
            for (int e = 0; e < kBN; e += 2) {
                const float p0 = ex2(fmaf(sv[e], c, -m_use));
                const float p1 = ex2(fmaf(sv[e + 1], c, -m_use));
                rs4[(e >> 1) & 3] += p0 + p1;
                pk[e >> 6][(e >> 1) & 31] = pack_bf16x2(p0, p1);
            }
            const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
            l += rs;
            tmem_st32(lane_addr + col_s + 0, pk[0]);
            tmem_st32(lane_addr + col_s + 32, pk[1]);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_p[t]);
        }

        // ----------------------------------------------------------- epilogue
        if (ok && fa_wait_warp(&bar_o[t], 0, 32 + t, wc)) {
            tc_fence_after();
            const bool valid = row < p.N;
            const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
            __nv_bfloat16* orow = p.o + ((size_t)bh * p.N + (valid ? row : 0)) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32(lane_addr + col_o + c0, ov);
                tmem_ld_wait(ov);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 0]) * inv_l,
                                          __uint_as_float(ov[q4 * 8 + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 2]) * inv_l,
                                          __uint_as_float(ov[q4 * 8 + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 4]) * inv_l,
                                          __uint_as_float(ov[q4 * 8 + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 6]) * inv_l,
                                          __uint_as_float(ov[q4 * 8 + 7]) * inv_l);
                        dst[q4] = w;
                    }
                }
            }
            if (valid)
                p.lse[(size_t)bh * p.N + row] =
                    (l > 0.0f) ? (m2 + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (warp == kProducerWarp) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                mbar_arrive_expect_tx(&bar_q, kTiles * Cfg::kTileBytes);
                for (int t = 0; t < kTiles; ++t)
                    for (int c = 0; c < Cfg::kChunks; ++c)
                        tma_load_3d(sQ + t * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_q, &bar_q,
                                    c * 64, row_base + t * kBM, bh);
                int issued = 0;
                for (int j = 0; j < n_kv; ++j) {
                    const int s = j % S, u = j / S;
                    if (j >= S && !fa_wait(&bar_kv_empty[s], (u - 1) & 1, 10, wc)) break;
                    mbar_arrive_expect_tx(&bar_k[s], Cfg::kTileBytes);
                    for (int c = 0; c < Cfg::kChunks; ++c)
                        tma_load_3d(sK + s * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_k, &bar_k[s],
                                    c * 64, j * kBN, kv_bh);
                    mbar_arrive_expect_tx(&bar_v[s], Cfg::kTileBytes);
                    for (int c = 0; c < Cfg::kChunks; ++c)
                        tma_load_3d(sV + s * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_v, &bar_v[s],
                                    c * 64, j * kBN, kv_bh);
                    issued = j + 1;
                }
                // Drain: on an abort, wait (bounded) for the copies still in flight
                // so none lands after the CTA has exited.
                if (abort_sh) {
                    for (int j = max(0, issued - S); j < issued; ++j) {
                        fa_wait(&bar_k[j % S], (j / S) & 1, 11, WaitCtx{p.status, nullptr});
                        fa_wait(&bar_v[j % S], (j / S) & 1, 11, WaitCtx{p.status, nullptr});
                    }
                }
            }
        } else if (warp == kMmaWarp) {
            if (lane == 0) {
                constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
                constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, false, true);
                const uint32_t sq = smem_u32(sQ), sk = smem_u32(sK), sv = smem_u32(sV);
                bool ok = fa_wait(&bar_q, 0, 20, wc) && fa_wait(&bar_k[0], 0, 21, wc);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < kTiles; ++t) {
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + (Cfg::kColS0 + t * (Cfg::kColS1 - Cfg::kColS0)), kmajor_desc(sq + t * Cfg::kTileBytes, kk),
                                   kmajor_desc(sk, kk), idesc_s, kk > 0);
                        mma_commit(&bar_s[t]);
                    }
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int s = j % S, u = j / S;
                    const bool next = j + 1 < n_kv;
                    const int s1 = (j + 1) % S, u1 = (j + 1) / S;
                    if (!fa_wait(&bar_v[s], u & 1, 22, wc)) { ok = false; break; }
                    if (next && !fa_wait(&bar_k[s1], u1 & 1, 23, wc)) { ok = false; break; }
                    for (int t = 0; t < kTiles; ++t) {
                        if (!fa_wait(&bar_p[t], j & 1, 24 + t, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t vb = sv + s * Cfg::kTileBytes;
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            mma_ts(tmem + (Cfg::kColO0 + t * (Cfg::kColO1 - Cfg::kColO0)), tmem + (Cfg::kColS0 + t * (Cfg::kColS1 - Cfg::kColS0)) + kk * 8, vmn_desc(vb, kk),
                                   idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                        if (next) {
                            const uint32_t kb = sk + s1 * Cfg::kTileBytes;
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tmem + (Cfg::kColS0 + t * (Cfg::kColS1 - Cfg::kColS0)), kmajor_desc(sq + t * Cfg::kTileBytes, kk),
                                       kmajor_desc(kb, kk), idesc_s, kk > 0);
                            mma_commit(&bar_s[t]);
                        } else {
                            mma_commit(&bar_o[t]);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&bar_kv_empty[s]);
                }
                // Make sure no MMA is still writing TMEM when the CTA tears down.
                if (!ok) {
                    __shared__ uint64_t bar_drain;
                    mbar_init(&bar_drain, 1);
                    fence_mbar_init();
                    mma_commit(&bar_drain);
                    fa_wait(&bar_drain, 0, 29, WaitCtx{p.status, nullptr});
                }
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const Shape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const FwdParams& p, int grid,
                         cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D, CAUSAL>;
    static int configured_device = -1;   // attribute is per device; cheap to repeat
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             FwdCfg<D>::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<grid, kThreads, FwdCfg<D>::kSmemAlloc, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Shape& s, const void* q, const void* k, const void* v, void* o,
                       float* lse, DeviceStatus* status, cudaStream_t stream) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_3d(&tq, q, s.d, s.N, s.B * s.H, kBM) ||
        !make_tmap_bf16_3d(&tk, k, s.d, s.N, s.B * s.Hkv, kBN) ||
        !make_tmap_bf16_3d(&tv, v, s.d, s.N, s.B * s.Hkv, kBN))
        return cudaErrorInvalidValue;
    FwdParams p;
    p.H = s.H;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.BH = s.B * s.H;
    p.n_mblk = (s.N + kTiles * kBM - 1) / (kTiles * kBM);
    p.causal = s.causal;
    p.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.status = status;
    const int grid = p.n_mblk * p.BH;
    count_launch();
    if (s.d == 128)
        return s.causal ? launch_fwd_t<128, true>(s, tq, tk, tv, p, grid, stream)
                        : launch_fwd_t<128, false>(s, tq, tk, tv, p, grid, stream);
    return s.causal ? launch_fwd_t<64, true>(s, tq, tk, tv, p, grid, stream)
                    : launch_fwd_t<64, false>(s, tq, tk, tv, p, grid, stream);
}

}  // namespace fa
