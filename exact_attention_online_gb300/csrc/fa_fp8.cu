// FP8 (e4m3) forward: exact attention with the P V product in e4m3
// (FlashAttention-3 summary, abstract: FP8 with block quantization; the
// granularity is this library's reading: one scale per (batch, head, block of
// 128 rows), scale = amax / 448).
//
// Which product runs in e4m3.  Rounding Q and K to e4m3's 3 mantissa bits puts
// a relative error of about 2.7 % RMS on each, so the scores S = Q K^T carry an
// absolute error of about 0.04 |S|-scale, and every P = 2^(S c - m) inherits
// it through the exponential; outliers in Q or K multiply it.  A model of this
// quantisation (e4m3 from its definition, the kernel's block scales and P
// rounding) gives 0.048 relative RMS error of O on N(0,1) inputs and 0.086 /
// 0.116 on the outlier / x20-channel inputs with Q, K, V and P all in e4m3,
// against 0.034 / 0.021 / 0.034 with S computed from the bf16 Q and K and
// only P and V in e4m3 (a random Hadamard rotation of Q and K, incoherent
// processing, brings the all-e4m3 outlier case only to 0.074: e4m3 is a
// floating-point format, so spreading an outlier over the channels does not
// shrink the relative rounding of the products).  So S = Q K^T is a bf16
// tcgen05 MMA (kind::f16) and O += P V a kind::f8f6f4 MMA.
//
// Two steps.
//   quantize   bf16 V -> e4m3 codes, transposed ([d][keys], so that the MMA's
//              B operand is K-major), and fp32 block scales sv, in one
//              caller-owned buffer (layout in fa.h); a second small kernel
//              takes each kv head's largest block scale svmax.
//   forward    the bf16 forward's structure at d = 128 (persistent CTAs,
//              two 128-row query tiles per item, K/V rings, S and P V MMA
//              issuers in two warps, two softmax warpgroups):
//                S_t = Q_t K_j^T (bf16, fp32 in TMEM);
//                P is quantised as e4m3(p * 448 * sv_j / svmax) (the V block
//                scale moves into P, so one descale remains), written over the
//                first 32 columns of S_t, and O_t += P8_t V8_j^T (K = 32 per
//                instruction); epilogue O = O_t * (svmax / 448) / l.
//              The running max is exact (raised whenever a block exceeds it),
//              so p <= 1 and p * 448 stays within e4m3's range.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <type_traits>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kD = 128;           // head dim (one 128-byte e4m3 row)
constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kTiles = 2;
constexpr int kThreads = 12 * 32;
constexpr int kProducerWarp = 8;    // K tiles
constexpr int kMmaWarp = 9;         // S MMA issuer; allocates TMEM
constexpr int kVProducerWarp = 10;  // V and Q tiles
constexpr int kPvWarp = 11;         // P V MMA issuer
// 128 x 72 + 256 x 216 = 64512 = 384 x 168: no role spills (the softmax
// warps did at 208).
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsNeeded = 128 * kRegsControl + 256 * kRegsSoftmax;
constexpr int kStagesK = 3, kStagesV = 3;
constexpr int kChunkBytes = 128 * 128;            // 128 rows x 128 bytes (64 bf16 or 128 e4m3)
constexpr int kQKTileBytes = 2 * kChunkBytes;     // a bf16 Q or K tile: two 64-column chunks
constexpr int kVTileBytes = kChunkBytes;          // an e4m3 V^T tile: 128 x 128 codes
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTiles * kQKTileBytes;
constexpr int kOffV = kOffK + kStagesK * kQKTileBytes;
constexpr int kSmemBytes = kOffV + kStagesV * kVTileBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;

struct Fp8Params {
    int H, Hkv, N, BH, n_mblk, n_items, nblk;
    float scale_log2;
    const float* sv;     // [B*Hkv][nblk]
    const float* svmax;  // [B*Hkv]
    __nv_bfloat16* o;
    float* lse;
    DeviceStatus* status;
};

struct Tile {
    int bh, kv_bh, row_base;
    int n_kv[kTiles];
};

// Item of this CTA in round rd: the cost-ranked items are dealt in rounds of
// gridDim.x with the order of the CTAs reversed every other round, which
// evens out the causal costs per CTA (as in the bf16 forward).
__device__ __forceinline__ int snake_item(int rd) {
    const int G = gridDim.x, c = blockIdx.x;
    return rd * G + ((rd & 1) ? G - 1 - c : c);
}

__device__ __forceinline__ Tile fp8_tile(int item, const Fp8Params& p, bool causal) {
    Tile w;
    const int mb_rank = item / p.BH;
    w.bh = item % p.BH;
    const int m_blk = causal ? (p.n_mblk - 1 - mb_rank) : mb_rank;
    const int b = w.bh / p.H, h = w.bh % p.H;
    w.kv_bh = b * p.Hkv + h / (p.H / p.Hkv);
    w.row_base = m_blk * (kTiles * kBM);
    const int n_kv_all = (p.N + kBN - 1) / kBN;
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
        w.n_kv[t] = causal ? min(n_kv_all, 2 * m_blk + t + 1) : n_kv_all;
    return w;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_vt, const Fp8Params p) {
    constexpr int SK = kStagesK, SV = kStagesV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_k[SK], bar_k_empty[SK], bar_v[SV], bar_v_empty[SV];
    __shared__ uint64_t bar_q[kTiles], bar_q_free[kTiles];
    __shared__ uint64_t bar_s[kTiles], bar_p[kTiles], bar_pv[kTiles], bar_o[kTiles], bar_o_free[kTiles];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    const WaitCtx wc{p.status, &abort_sh};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int s = 0; s < SK; ++s) {
            mbar_init(&bar_k[s], 1);
            mbar_init(&bar_k_empty[s], 1);
        }
        for (int s = 0; s < SV; ++s) {
            mbar_init(&bar_v[s], 1);
            mbar_init(&bar_v_empty[s], 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bar_q[t], 1);
            mbar_init(&bar_q_free[t], 1);
            mbar_init(&bar_s[t], 1);
            mbar_init(&bar_p[t], 128);
            mbar_init(&bar_pv[t], 1);
            mbar_init(&bar_o[t], 1);
            mbar_init(&bar_o_free[t], 128);
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

    uint8_t* sQ = smem + kOffQ;
    uint8_t* sK = smem + kOffK;
    uint8_t* sV = smem + kOffV;

    if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int rl = quarter * 32 + lane;
        const uint32_t col_s = t ? kColS1 : kColS0;
        const uint32_t col_o = t ? kColO1 : kColO0;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t cs = 0;
        bool ok = true;
        int lt = 0;
        for (int rd = 0, item = snake_item(0); ok && item < p.n_items;
             item = snake_item(++rd), ++lt) {
            const Tile wt = fp8_tile(item, p, CAUSAL);
            const int row0 = wt.row_base + t * kBM;
            const int row = row0 + rl;
            const int n_kv = wt.n_kv[t];
            const float svmax = __ldg(p.svmax + wt.kv_bh);
            const float c = p.scale_log2;
            const float pw = (svmax > 0.0f) ? 448.0f / svmax : 0.0f;   // times sv_j per block
            float m2 = -CUDART_INF_F;
            float l = 0.0f;
            for (int j = 0; j < n_kv; ++j) {
                const float w = pw * __ldg(p.sv + (size_t)wt.kv_bh * p.nblk + j);
                if (!fa_wait_warp(&bar_s[t], cs & 1, 30 + t, wc)) { ok = false; break; }
                ++cs;
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
                    const int lim_causal = CAUSAL ? row - col0 : kBN;
                    const int lim_n = p.N - col0;
#pragma unroll
                    for (int e = 0; e < kBN; ++e)
                        if (e > lim_causal || e >= lim_n) sv[e] = -CUDART_INF_F;
                }
                float mx8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(sv[2 * u], sv[2 * u + 1]);
#pragma unroll
                for (int e = 16; e < kBN; e += 16)
#pragma unroll
                    for (int u = 0; u < 8; ++u) mx8[u] = fmax3(mx8[u], sv[e + 2 * u], sv[e + 2 * u + 1]);
                const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                       fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                // c > 0, so the max of s * c is c times the max of s.  The running
                // max is exact here: p <= 1 keeps p * 448 inside e4m3's range.
                const float mx2 = mx * c;
                const bool need = mx2 > m2;
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = need ? mx2 : m2;
                    const float alpha = (m_new == m2) ? 1.0f : ex2(m2 - m_new);
                    l *= alpha;
                    if (j > 0) {
#pragma unroll
                        for (int c0 = 0; c0 < kD; c0 += 32) {
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
                const uint64_t c2 = f2(c, c), negm2 = f2(-m_use, -m_use);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pk[32];
#pragma unroll
                for (int e4 = 0; e4 < 32; ++e4) {
                    float x0, x1, x2, x3;
                    f2_split(f2_fma(f2(sv[4 * e4], sv[4 * e4 + 1]), c2, negm2), x0, x1);
                    f2_split(f2_fma(f2(sv[4 * e4 + 2], sv[4 * e4 + 3]), c2, negm2), x2, x3);
                    const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
                    acc2[e4 & 3] = f2_add(acc2[e4 & 3], f2_add(f2(p0, p1), f2(p2, p3)));
                    pk[e4] = pack_e4m3x4(p0 * w, p1 * w, p2 * w, p3 * w);
                }
                tmem_st32(lane_addr + col_s, pk);   // P8 over the first 32 S columns
                {
                    float a0, a1;
                    f2_split(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), a0, a1);
                    l += a0 + a1;
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_p[t]);
            }
            if (!ok) break;
            // ------------------------------------------------------- epilogue
            if (!fa_wait_warp(&bar_o[t], lt & 1, 32 + t, wc)) { ok = false; break; }
            tc_fence_after();
            uint32_t ov[kD / 32][32];
#pragma unroll
            for (int c0 = 0; c0 < kD / 32; ++c0) tmem_ld32(lane_addr + col_o + c0 * 32, ov[c0]);
            tmem_ld_wait(ov[0]);
#pragma unroll
            for (int c0 = 1; c0 < kD / 32; ++c0) asm volatile("" : FA_R32(ov[c0]) : : "memory");
            tc_fence_before();
            mbar_arrive(&bar_o_free[t]);
            const bool valid = row < p.N;
            const float out_mul = (l > 0.0f) ? (svmax * (1.0f / 448.0f)) / l : 0.0f;
            if (valid) {
                const size_t orow = ((size_t)wt.bh * p.N + row) * kD;
#pragma unroll
                for (int c0 = 0; c0 < kD / 32; ++c0) {
                    uint4* dst = reinterpret_cast<uint4*>(p.o + orow + c0 * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 0]) * out_mul,
                                          __uint_as_float(ov[c0][q4 * 8 + 1]) * out_mul);
                        v.y = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 2]) * out_mul,
                                          __uint_as_float(ov[c0][q4 * 8 + 3]) * out_mul);
                        v.z = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 4]) * out_mul,
                                          __uint_as_float(ov[c0][q4 * 8 + 5]) * out_mul);
                        v.w = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 6]) * out_mul,
                                          __uint_as_float(ov[c0][q4 * 8 + 7]) * out_mul);
                        dst[q4] = v;
                    }
                }
                p.lse[(size_t)wt.bh * p.N + row] =
                    (l > 0.0f) ? (m2 + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
            }
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (warp == kProducerWarp && lane == 0) {
            // ------------------------------------------------- K producer
            tma_prefetch_desc(&tm_k);
            uint32_t g = 0;
            bool ok = true;
            for (int rd = 0, item = snake_item(0); ok && item < p.n_items;
                 item = snake_item(++rd)) {
                const Tile wt = fp8_tile(item, p, CAUSAL);
                for (int j = 0; j < wt.n_kv[kTiles - 1]; ++j, ++g) {
                    const int s = g % SK;
                    if (g >= (uint32_t)SK && !fa_wait(&bar_k_empty[s], ((g / SK) - 1) & 1, 10, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_k[s], kQKTileBytes);
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(sK + s * kQKTileBytes + c * kChunkBytes, &tm_k, &bar_k[s],
                                    c * 64, j * kBN, wt.kv_bh);
                }
            }
            if (abort_sh) {
                const WaitCtx dc{p.status, nullptr};
                for (uint32_t x = (g > (uint32_t)SK ? g - SK : 0); x < g; ++x)
                    fa_wait(&bar_k[x % SK], (x / SK) & 1, 11, dc);
            }
        } else if (warp == kVProducerWarp && lane == 0) {
            // ---------------------------------------------- V and Q producer
            tma_prefetch_desc(&tm_vt);
            tma_prefetch_desc(&tm_q);
            uint32_t g = 0;
            int lt = 0, q_loaded = -1;
            bool ok = true;
            for (int rd = 0, item = snake_item(0); ok && item < p.n_items;
                 item = snake_item(++rd), ++lt) {
                const Tile wt = fp8_tile(item, p, CAUSAL);
                for (int t = 0; t < kTiles; ++t) {
                    if (lt > 0 && !fa_wait(&bar_q_free[t], (lt - 1) & 1, 12, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar_q[t], kQKTileBytes);
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(sQ + t * kQKTileBytes + c * kChunkBytes, &tm_q, &bar_q[t],
                                    c * 64, wt.row_base + t * kBM, wt.bh);
                }
                if (!ok) break;
                q_loaded = lt;
                for (int j = 0; j < wt.n_kv[kTiles - 1]; ++j, ++g) {
                    const int s = g % SV;
                    if (g >= (uint32_t)SV && !fa_wait(&bar_v_empty[s], ((g / SV) - 1) & 1, 13, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_v[s], kVTileBytes);
                    // V^T block: rows = head-dim index, 128 keys per row
                    tma_load_3d(sV + s * kVTileBytes, &tm_vt, &bar_v[s], j * kBN, 0, wt.kv_bh);
                }
            }
            if (abort_sh) {
                const WaitCtx dc{p.status, nullptr};
                for (uint32_t x = (g > (uint32_t)SV ? g - SV : 0); x < g; ++x)
                    fa_wait(&bar_v[x % SV], (x / SV) & 1, 14, dc);
                if (q_loaded >= 0)
                    for (int t = 0; t < kTiles; ++t) fa_wait(&bar_q[t], q_loaded & 1, 15, dc);
            }
        } else if (warp == kPvWarp && lane == 0) {
            // ------------------------------------------- P V MMA issuer
            // O_t += P8_t V8_j: A = P8_t from TMEM (four codes per column),
            // B = the V^T block, K-major over the keys.
            constexpr uint32_t idesc_o = idesc_e4m3_f32(kBM, kD);
            const uint32_t svs = smem_u32(sV);
            uint32_t g = 0, cp0 = 0, cp1 = 0;
            bool ok = true;
            int lt = 0;
            auto pv = [&](auto tc, uint32_t vstage, bool first, bool last, bool wait_o) -> bool {
                constexpr int T = decltype(tc)::value;
                constexpr uint32_t col_o = T ? kColO1 : kColO0;
                constexpr uint32_t col_s = T ? kColS1 : kColS0;
                uint32_t& c = T ? cp1 : cp0;
                if (!fa_wait(&bar_p[T], c & 1, 24 + T, wc)) return false;
                ++c;
                if (wait_o && !fa_wait(&bar_o_free[T], (lt - 1) & 1, 26 + T, wc)) return false;
                tc_fence_after();
                const uint64_t vd = sdesc_sw128(svs + vstage * kVTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kBN / 32; ++kk)
                    mma_ts_f8(tmem + col_o, tmem + col_s + kk * 8, vd + kmajor_step(kk, kVTileBytes),
                              idesc_o, (!first || kk > 0) ? 1u : 0u);
                mma_commit(&bar_pv[T]);
                if (last) mma_commit(&bar_o[T]);
                return true;
            };
            for (int rd = 0, item = snake_item(0); ok && item < p.n_items;
                 item = snake_item(++rd), ++lt) {
                const Tile wt = fp8_tile(item, p, CAUSAL);
                const int n0 = wt.n_kv[0], n1 = wt.n_kv[1];
                for (int j = 0; j < n1; ++j) {
                    const uint32_t gj = g + j, vs = gj % SV;
                    if (!fa_wait(&bar_v[vs], (gj / SV) & 1, 22, wc)) { ok = false; break; }
                    const bool wait_o = (j == 0 && lt > 0);
                    if (j < n0 &&
                        !pv(std::integral_constant<int, 0>{}, vs, j == 0, j + 1 == n0, wait_o)) {
                        ok = false;
                        break;
                    }
                    if (!pv(std::integral_constant<int, 1>{}, vs, j == 0, j + 1 == n1, wait_o)) {
                        ok = false;
                        break;
                    }
                    mma_commit(&bar_v_empty[vs]);
                }
                g += n1;
            }
            if (!ok) {
                __shared__ uint64_t bar_drain_pv;
                mbar_init(&bar_drain_pv, 1);
                fence_mbar_init();
                mma_commit(&bar_drain_pv);
                fa_wait(&bar_drain_pv, 0, 29, WaitCtx{p.status, nullptr});
            }
        } else if (warp == kMmaWarp && lane == 0) {
            // ---------------------------------------------- S MMA issuer
            // S_t(j) = Q_t K_j^T (bf16) once K_j has landed and the P_t V MMA
            // that reads the previous P_t (written over S_t) has completed.
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
            const uint32_t sq = smem_u32(sQ), sk = smem_u32(sK);
            uint32_t g = 0, ns0 = 0, ns1 = 0;
            bool ok = true;
            int lt = 0;
            auto s_mma = [&](auto tc, uint32_t kstage) -> bool {
                constexpr int T = decltype(tc)::value;
                uint32_t& n = T ? ns1 : ns0;
                if (n > 0 && !fa_wait(&bar_pv[T], (n - 1) & 1, 36 + T, wc)) return false;
                ++n;
                tc_fence_after();
                const uint64_t qd = sdesc_sw128(sq + T * kQKTileBytes, 16, 1024);
                const uint64_t kd = sdesc_sw128(sk + kstage * kQKTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_ss(tmem + (T ? kColS1 : kColS0), qd + kmajor_step(kk, kChunkBytes),
                           kd + kmajor_step(kk, kChunkBytes), idesc_s, kk > 0);
                mma_commit(&bar_s[T]);
                return true;
            };
            for (int rd = 0, item = snake_item(0); ok && item < p.n_items;
                 item = snake_item(++rd), ++lt) {
                const Tile wt = fp8_tile(item, p, CAUSAL);
                const int n0 = wt.n_kv[0], n1 = wt.n_kv[1];
                if (!fa_wait(&bar_q[0], lt & 1, 20, wc) || !fa_wait(&bar_q[1], lt & 1, 20, wc)) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < n1; ++j) {
                    const uint32_t gj = g + j, ks = gj % SK;
                    if (!fa_wait(&bar_k[ks], (gj / SK) & 1, 21, wc)) { ok = false; break; }
                    if (j < n0) {
                        if (!s_mma(std::integral_constant<int, 0>{}, ks)) { ok = false; break; }
                        if (j + 1 == n0) mma_commit(&bar_q_free[0]);
                    }
                    if (!s_mma(std::integral_constant<int, 1>{}, ks)) { ok = false; break; }
                    if (j + 1 == n1) mma_commit(&bar_q_free[1]);
                    mma_commit(&bar_k_empty[ks]);
                }
                g += n1;
            }
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

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- quantize
// One CTA (256 threads) per 128-row block of one kv head of V.  Thread t
// holds row t / 2, columns (t % 2) * 64 ... + 63.  amax over the block's valid
// rows; scale = amax / 448 and inv = 448 / amax as fp32 divisions (1 and 1 for
// an all-zero block); code = e4m3(fp32(x * inv)), nearest even, saturating.
// Rows past N are written as zero codes.  The block goes out transposed.
__global__ void __launch_bounds__(256)
fa_fp8_quant_kernel(const __nv_bfloat16* __restrict__ v, Fp8Buffer buf, int N, int Np) {
    __shared__ float warp_max[8];
    __shared__ __align__(16) uint8_t tile_t[128][128 + 16];   // transpose staging
    const int nblk = Np / 128;
    const int g = blockIdx.x / nblk, b = blockIdx.x % nblk;
    const __nv_bfloat16* src = v;
    const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int row = b * 128 + r;
    const bool valid = row < N;
    float x[64];
    if (valid) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src + ((size_t)g * N + row) * kD + half * 64);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 w = s4[u];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[u * 8 + 2 * e] = __uint_as_float(ww[e] << 16);
                x[u * 8 + 2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = 0.0f;
    }
    float am = 0.0f;
#pragma unroll
    for (int e = 0; e < 64; ++e) am = fmaxf(am, fabsf(x[e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = am;
    __syncthreads();
    float amax = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, warp_max[w]);
    const float inv = (amax > 0.0f) ? __fdiv_rn(448.0f, amax) : 1.0f;
    const float sc = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint32_t codes[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        codes[e] = pack_e4m3x4(__fmul_rn(x[4 * e], inv), __fmul_rn(x[4 * e + 1], inv),
                               __fmul_rn(x[4 * e + 2], inv), __fmul_rn(x[4 * e + 3], inv));
    {
        // stage the block [row][col], then write [col][row] runs of 64 keys
        uint4* t4 = reinterpret_cast<uint4*>(&tile_t[r][half * 64]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            t4[u] = make_uint4(codes[4 * u], codes[4 * u + 1], codes[4 * u + 2], codes[4 * u + 3]);
        __syncthreads();
        const int c = threadIdx.x >> 1, r0 = (threadIdx.x & 1) * 64;
        uint32_t col[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            col[e] = (uint32_t)tile_t[r0 + 4 * e][c] | ((uint32_t)tile_t[r0 + 4 * e + 1][c] << 8) |
                     ((uint32_t)tile_t[r0 + 4 * e + 2][c] << 16) |
                     ((uint32_t)tile_t[r0 + 4 * e + 3][c] << 24);
        uint4* d4 = reinterpret_cast<uint4*>(buf.v8t + ((size_t)g * kD + c) * Np + b * 128 + r0);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            d4[u] = make_uint4(col[4 * u], col[4 * u + 1], col[4 * u + 2], col[4 * u + 3]);
    }
    if (threadIdx.x == 0) buf.sv[(size_t)g * nblk + b] = sc;
}

// Largest V block scale of each kv head; one warp per head.
__global__ void fa_fp8_vmax_kernel(Fp8Buffer buf, int BHkv, int nblk) {
    const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (g >= BHkv) return;
    float m = 0.0f;
    for (int b = lane; b < nblk; b += 32) m = fmaxf(m, buf.sv[(size_t)g * nblk + b]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) buf.svmax[g] = m;
}

template <bool CAUSAL>
cudaError_t launch_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const Fp8Params& p, int grid, cudaStream_t stream) {
    auto kern = fa_fwd_fp8_kernel<CAUSAL>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        if (attr.numRegs * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<grid, kThreads, kSmemAlloc, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

size_t fp8_buffer_bytes(const Shape& s) {
    const size_t Np = padded_rows(s.N), nblk = Np / 128;
    auto a = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t bkv = (size_t)s.B * s.Hkv;
    return a(bkv * Np * s.d) + a(bkv * nblk * 4) + a(bkv * 4);
}

Fp8Buffer fp8_buffer_carve(void* base, const Shape& s) {
    const size_t Np = padded_rows(s.N), nblk = Np / 128;
    auto a = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t bkv = (size_t)s.B * s.Hkv;
    char* p = static_cast<char*>(base);
    Fp8Buffer f;
    f.v8t = reinterpret_cast<uint8_t*>(p);
    p += a(bkv * Np * s.d);
    f.sv = reinterpret_cast<float*>(p);
    p += a(bkv * nblk * 4);
    f.svmax = reinterpret_cast<float*>(p);
    return f;
}

cudaError_t launch_fp8_quantize(const Shape& s, const void* v, const Fp8Buffer& buf,
                                cudaStream_t stream) {
    const int Np = padded_rows(s.N), nblk = Np / 128;
    const int BHkv = s.B * s.Hkv;
    const long long blocks = (long long)BHkv * nblk;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    count_launch();
    fa_fp8_quant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(v), buf, s.N, Np);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
    fa_fp8_vmax_kernel<<<(BHkv + 7) / 8, 256, 0, stream>>>(buf, BHkv, nblk);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const Shape& s, const void* q, const void* k, const Fp8Buffer& buf,
                           void* o, float* lse, DeviceStatus* status, cudaStream_t stream) {
    const int Np = padded_rows(s.N);
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_3d(&tq, q, kD, s.N, s.B * s.H, kBM) ||
        !make_tmap_bf16_3d(&tk, k, kD, s.N, s.B * s.Hkv, kBN) ||
        !make_tmap_u8_3d(&tv, buf.v8t, Np, kD, s.B * s.Hkv))
        return cudaErrorInvalidValue;
    Fp8Params p;
    p.H = s.H;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.BH = s.B * s.H;
    p.n_mblk = (s.N + kTiles * kBM - 1) / (kTiles * kBM);
    p.n_items = p.n_mblk * p.BH;
    p.nblk = Np / 128;
    p.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
    p.sv = buf.sv;
    p.svmax = buf.svmax;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.status = status;
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    const int grid = p.n_items < sms ? p.n_items : sms;
    count_launch();
    return s.causal ? launch_fp8_t<true>(tq, tk, tv, p, grid, stream)
                    : launch_fp8_t<false>(tq, tk, tv, p, grid, stream);
}

}  // namespace fa
