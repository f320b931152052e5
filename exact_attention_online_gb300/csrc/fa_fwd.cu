// Forward kernel: exact attention with the online-softmax recurrence, tiled so
// the N x N score matrix never leaves the SM (FlashAttention blog, "From Online
// Softmax to FlashAttention" and "FlashAttention"; FlashAttention-2 review
// thread, author answers on non-matmul FLOPs and on Figure 2).
//
// Persistent grid, one CTA per SM.  A work item is two 128-row query tiles
// (t = 0, 1) of one (batch, head); CTA c takes items c, c + gridDim.x, ...
// (longest causal items first) and streams 128-key K and V tiles through two
// shared-memory rings:
//   warp 8      TMA producer of K_j; K_j is released when both S MMAs that
//               read it have completed, so K loads run whole blocks ahead.
//               In the PRECISE variant the whole warp also re-encodes the
//               second half of each landed V_j as fp16, in place.
//   warp 10     TMA producer of V_j and of the Q tiles (each item's Q ahead of
//               its V blocks); V_j is released after both P V MMAs.  In the
//               PRECISE variant the whole warp also re-encodes the first half
//               of each landed V_j as fp16, in place.
//   warp 9      S MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (SS MMA).
//   warp 11     P V MMA issuer (one thread): O_t += P_t V_j, P_t read from
//               TMEM (TS MMA).  An MMA issue blocks while the tensor pipe is
//               busy, and every barrier wait, fence and commit of an issuing
//               thread costs on the order of a hundred cycles; with two
//               issuers one thread's waits overlap the other's MMAs.
//   warps 0-3   softmax for tile 0, warps 4-7 for tile 1: one query row per
//               thread.  While one group does its softmax the tensor core
//               runs the other tile's MMAs.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  At d = 128, P_t (bf16 pairs)
// overwrites the first half of S_t; the MMA that next writes S_t is issued
// only after the P_t V MMA that reads P_t has completed.
// At d = 64 (bf16 output) P_t has columns of its own after O_1, which breaks
// that chain: the softmax releases S_t as soon as it has loaded it, the next
// S_t MMA is issued at once, and the softmax waits for the previous P V MMA
// only just before it writes P_t.  The tensor core then works on S_t(j+1) and
// P_t(j-1) V while the softmax of block j runs.
//
// Softmax in base 2: p = 2^(S*c - m) with c = scale*log2(e).  The running max
// m is only raised when the block max exceeds it by more than 8 (a factor
// 256), so most blocks skip the O rescale; numerator and denominator always
// use the same m, so the result is unchanged in exact arithmetic.  O is
// divided by l once, in the epilogue, and LSE = ln2 * (m + log2 l).
//
// PRECISE variant: the P V product runs in fp16 instead of bf16 (same tensor
// rate): P is rounded to fp16 (11 significant bits against bf16's 8), V_j is
// re-encoded as fp16 in shared memory (exact for magnitudes in [2^-14,
// 65280]; 65536 and above overflow to infinity), and O is written in fp32.
// This takes the bf16 rounding of O out of the error (half a bf16 ulp of 30 is
// 0.06) and cuts that of P eightfold: each p is off by at most 2^-11 of
// itself (2^-25 absolute below 2^-14).  The row sum l is corrected by what
// the rounding added to each key block's largest p, so a row whose weight
// sits on one key returns that key's V row unrounded; in general a row of O
// moves by at most 2^-11 (sum over block maxima of w |v - O| + sum over the
// other keys of w |v|) <= 2^-10 max|V|, w = p / l.
#include <cuda_bf16.h>
#include <type_traits>
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
constexpr int kProducerWarp = 8;    // K tiles
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;  // V and Q tiles
constexpr int kPvWarp = 11;         // P V MMA issuer
// Register split (setmaxnreg): the launch gives 384 x 168; the control
// warpgroup drops to 72 so each softmax thread can hold a full 128-score row:
// 128 x 72 + 256 x 216 = 64512 <= 384 x 168 = 64512.  At 216 no role spills
// (at 208 the softmax warps did, d = 128: forward 3 % slower).
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsNeeded = 128 * kRegsControl + 256 * kRegsSoftmax;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// One pair in every kExp2FmaEvery of a row's exps is computed on the FMA pipe
// (exp2_fma2) instead of the exponential unit, 0 = none.  Measured on the
// forward alone: d = 128 one pair in 8: +1.8 % (one in 16 +0.6 %, one in 4
// -4.6 %); d = 64, where the softmax is bound by instruction issue rather than
// by the exponential unit: one in 16 -4 %, one in 8 -6.5 %.
template <int D, bool PRECISE>
struct Exp2FmaEvery {
    static constexpr int value = (D == 128 && !PRECISE) ? 8 : 0;
    static constexpr int mod = value > 0 ? value : 1;
};

template <int D, bool PRECISE = false>
struct FwdCfg {
    // K and V have rings of their own: K is released as soon as both S MMAs of
    // a block are issued, V after both P V MMAs.  The PRECISE variant holds
    // each V_j longer (its fp16 re-encoding sits between landing and use) and
    // at d = 128 trades a K stage for a third V stage.
    static constexpr int kStagesK = (D == 128) ? (PRECISE ? 2 : 3) : 4;
    static constexpr int kStagesV = (D == 128) ? (PRECISE ? 3 : 2) : 3;
    static constexpr int kTileBytes = kBM * D * 2;          // one Q, K or V tile
    static constexpr int kChunks = D / 64;                  // 128-byte swizzle chunks
    static constexpr int kChunkBytes = 128 * 128;           // 128 rows x 128 bytes
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTiles * kTileBytes;
    static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
    static constexpr int kSmemBytes = kOffV + kStagesV * kTileBytes;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;    // alignment slack
    // TMEM columns
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
    // At d = 64, S_0 | S_1 | O_0 | O_1 fill 384 columns and P_t (64 columns of
    // bf16 pairs) gets columns of its own.
    static constexpr uint32_t kColP0 = 384, kColP1 = 448;
};

struct FwdParams {
    int H, Hkv, N, BH, n_mblk, n_items, causal;
    // Causal sliding window W: query i sees keys i - W < j <= i.  Without a
    // window this holds kNoWindow, so large that the lower edge never binds.
    int window;
    // Packed variable-length batches: sequence b is rows cu_seqlens[b] ..
    // cu_seqlens[b+1] - 1 of every head ([H][rows][d]); N is then the
    // longest sequence.  Dense batches: rows = N, cu_seqlens unused.
    int rows;
    const int* cu_seqlens;
    float scale_log2;                 // scale * log2(e)
    void* o;                          // bf16, or fp32 in the precise variant
    float* lse;
    DeviceStatus* status;
    // Training forward (dense batches): the backward workspace rows this
    // forward prepares, Np (= N rounded up to 128) rows per (batch, head):
    // the -LSE table row and a zeroed dQ accumulator row.  nullptr = none.
    uint16_t* lse_ext;
    float* dq_acc;
    int Np;
};

// Work item (query-block pair, batch*head) -> coordinates.  Under the causal
// mask the longest query blocks come first (the tile list is in decreasing
// cost order, and each CTA takes every gridDim.x-th item).
struct FwdTile {
    int bh, row_base;
    int q_z, kv_z;             // head coordinate of the Q / O and K / V tensor maps
    int tok0, len;             // first row of the sequence in its head, its length
    int lo[kTiles];            // first key block each query tile needs
    int n_kv[kTiles];          // one past its last key block
};

__device__ __forceinline__ int fwd_m_blk(int item, const FwdParams& p, bool causal) {
    const int mb_rank = item / p.BH;
    return causal ? (p.n_mblk - 1 - mb_rank) : mb_rank;
}

// The work items of this CTA, the same sequence for every role.  Items are
// ranked in decreasing cost (under the causal mask) and dealt out in rounds
// of gridDim.x, the order of the CTAs reversed every other round ("snake"),
// so that the sum of costs per CTA evens out (CPU model of the bench
// workloads: 0.98-1.00 of the mean load per CTA, against 0.88-0.94 for
// plain round robin).  With variable lengths the ranks count only the items
// that have rows (query-block pairs past a sequence's end are passed over):
// a cursor walks the (level, sequence) list forward, ranks only grow.
template <bool VARLEN>
struct FwdSched {
    int round = 0;
    int mb = 0, b = 0, base = 0;   // cursor: level, sequence, rank of (b, head 0)

    __device__ __forceinline__ int next(const FwdParams& p, bool causal) {
        const int G = gridDim.x, c = blockIdx.x;
        const int t = round * G + ((round & 1) ? G - 1 - c : c);   // rank
        ++round;
        if (!VARLEN) return t < p.n_items ? t : p.n_items;
        const int B = p.BH / p.H;
        while (mb < p.n_mblk) {
            if (b >= B) {
                ++mb;
                b = 0;
                continue;
            }
            int t0;
            const int len = packed_seq(p.cu_seqlens, b, p.N, p.rows, t0);
            if (fwd_m_blk(mb * p.BH, p, causal) * (kTiles * kBM) < len) {
                if (t < base + p.H) return mb * p.BH + b * p.H + (t - base);
                base += p.H;
            }
            ++b;
        }
        return p.n_items;
    }
};

template <bool WINDOW, bool VARLEN>
__device__ __forceinline__ FwdTile fwd_tile(int item, const FwdParams& p, bool causal) {
    FwdTile w;
    w.bh = item % p.BH;
    const int m_blk = fwd_m_blk(item, p, causal);
    const int b = w.bh / p.H, h = w.bh % p.H;
    if (VARLEN) {
        w.len = packed_seq(p.cu_seqlens, b, p.N, p.rows, w.tok0);
        w.q_z = h;
        w.kv_z = h / (p.H / p.Hkv);
    } else {
        w.tok0 = 0;
        w.len = p.N;
        w.q_z = w.bh;
        w.kv_z = b * p.Hkv + h / (p.H / p.Hkv);
    }
    w.row_base = m_blk * (kTiles * kBM);
    const int n_kv_all = (w.len + kBN - 1) / kBN;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        w.n_kv[t] = causal ? min(n_kv_all, 2 * m_blk + t + 1) : n_kv_all;
        // The tile's first row sees keys from row0 - W + 1 on.  A tile wholly
        // past N (the second tile of the last pair) keeps one block, which
        // the masks empty, so that every tile takes at least one block.
        w.lo[t] = WINDOW ? min(max(0, w.row_base + t * kBM - p.window + 1) / kBN, w.n_kv[t] - 1)
                         : 0;
    }
    return w;
}

// WINDOW (with CAUSAL): the causal sliding window of p.window keys.
// VARLEN: packed variable-length sequences (p.cu_seqlens).
// PRECISE: one warp's half (part 0 or 1) of the fp16 re-encoding of V_x, in
// place, once V_x has landed; the P V issuer waits for both halves (bar_v_cvt
// counts two arrivals).  Spread over two warps on two SM sub-partitions, the
// conversion takes issue slots from fewer softmax warps each.
template <int SV, int TILE_BYTES>
__device__ __forceinline__ bool convert_v_half(uint8_t* sV, uint64_t* bar_v, uint64_t* bar_v_cvt,
                                               uint32_t x, int part, int lane, const WaitCtx& wc) {
    const uint32_t s = x % SV;
    if (!fa_wait_warp(&bar_v[s], (x / SV) & 1, 16 + part, wc)) return false;
    constexpr int kHalf = TILE_BYTES / 32;   // 16-byte pieces in half a tile
    uint4* v4 = reinterpret_cast<uint4*>(sV + s * TILE_BYTES) + part * kHalf;
#pragma unroll 8
    for (int i = lane; i < kHalf; i += 32) {
        uint4 w = v4[i];
        w.x = bf16x2_to_f16x2(w.x);
        w.y = bf16x2_to_f16x2(w.y);
        w.z = bf16x2_to_f16x2(w.z);
        w.w = bf16x2_to_f16x2(w.w);
        v4[i] = w;
    }
    fence_proxy_async_smem();   // visible to the tensor core's reads
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_v_cvt[s]);
    return true;
}

template <int D, bool CAUSAL, bool PRECISE, bool WINDOW, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using Cfg = FwdCfg<D, PRECISE>;
    constexpr int SK = Cfg::kStagesK, SV = Cfg::kStagesV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_k[SK], bar_k_empty[SK], bar_v[SV], bar_v_empty[SV];
    __shared__ uint64_t bar_v_cvt[SV];        // PRECISE: V_j re-encoded as fp16
    __shared__ uint64_t bar_q[kTiles], bar_q_free[kTiles];
    __shared__ uint64_t bar_s[kTiles], bar_p[kTiles], bar_pv[kTiles], bar_o_free[kTiles];
    __shared__ uint64_t bar_s_free[kTiles];   // separate-P form only
    constexpr bool SEP = (D == 64) && !PRECISE;
    constexpr int kExp2FmaEvery = Exp2FmaEvery<D, PRECISE>::value;
    constexpr int kExp2FmaMod = Exp2FmaEvery<D, PRECISE>::mod;
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
            mbar_init(&bar_v_cvt[s], 2);   // one arrival per converting warp
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bar_q[t], 1);
            mbar_init(&bar_q_free[t], 1);
            mbar_init(&bar_s[t], 1);
            mbar_init(&bar_p[t], 128);
            mbar_init(&bar_o_free[t], 128);
            mbar_init(&bar_s_free[t], 128);
            mbar_init(&bar_pv[t], 1);
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
        const uint32_t col_s = t ? Cfg::kColS1 : Cfg::kColS0;
        const uint32_t col_o = t ? Cfg::kColO1 : Cfg::kColO0;
        const uint32_t col_p = SEP ? (t ? Cfg::kColP1 : Cfg::kColP0) : col_s;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const float c = p.scale_log2;
        uint32_t cs = 0;                         // S_t completions seen so far
        uint32_t cpv = 0;                        // P_t V completions seen (separate P)
        bool ok = true;
        int lt = 0;
        FwdSched<VARLEN> sch;
        for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
             item = sch.next(p, CAUSAL), ++lt) {
            const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
            const int row0 = wt.row_base + t * kBM;
            const int row = row0 + rl;
            // (selects, not a run-time index: the arrays stay in registers)
            const int lo = t ? wt.lo[1] : wt.lo[0], n_kv = t ? wt.n_kv[1] : wt.n_kv[0];
            float m2 = -CUDART_INF_F;   // running max, log2-scaled
            float l = 0.0f;
            // PRECISE: what the fp16 rounding of each block's largest p added
            // to the P V product, scaled like l.  O is divided by l + lc, so a
            // row whose weight sits on one key returns that key's V row
            // without the rounding of its p (up to 2^-11 |V| otherwise); the
            // LSE keeps l.
            float lc = 0.0f;
            for (int j = lo; j < n_kv; ++j) {
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
                if (SEP) {   // S_t is in registers: the next S_t MMA may overwrite it
                    tc_fence_before();
                    mbar_arrive(&bar_s_free[t]);
                }
                float sv[kBN];
#pragma unroll
                for (int e = 0; e < kBN; ++e) sv[e] = __uint_as_float(r[e >> 5][e & 31]);

                const int col0 = j * kBN;
                const bool need_mask = (CAUSAL && (col0 + kBN - 1 > row0 ||
                                                   (WINDOW && col0 < row0 + kBM - p.window))) ||
                                       (col0 + kBN > wt.len);
                if (need_mask) {
                    const int lim_causal = CAUSAL ? row - col0 : kBN;   // keep e <= row - col0
                    const int lim_n = wt.len - col0;                     // keep e < N - col0
                    const int lim_lo = WINDOW ? row - p.window + 1 - col0 : 0;  // keep e >= this
#pragma unroll
                    for (int e = 0; e < kBN; ++e)
                        if (e > lim_causal || e >= lim_n || e < lim_lo) sv[e] = -CUDART_INF_F;
                }
                // Row max: three-input max, eight independent chains.
                float mx8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(sv[2 * u], sv[2 * u + 1]);
#pragma unroll
                for (int e = 16; e < kBN; e += 16)
#pragma unroll
                    for (int u = 0; u < 8; ++u) mx8[u] = fmax3(mx8[u], sv[e + 2 * u], sv[e + 2 * u + 1]);
                const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                       fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                const float mx2 = mx * c;
                const bool need = mx2 > m2 + kRescaleThreshold;
                // O rescale of this block (only when some row raised its max);
                // the O columns may be touched only after the P V MMA of the
                // previous block has completed.
                auto rescale_o = [&](float alpha) {
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
                };
                const bool any_need = __any_sync(0xffffffffu, need);
                float alpha = 1.0f;
                if (any_need) {
                    const float m_new = need ? mx2 : m2;
                    alpha = (m_new == m2) ? 1.0f : ex2(m2 - m_new);
                    l *= alpha;
                    if (PRECISE) lc *= alpha;
                    if (!SEP && j > lo) rescale_o(alpha);
                    m2 = m_new;
                }
                const float m_use = (m2 == -CUDART_INF_F) ? 0.0f : m2;
                if (PRECISE) {   // the block max's p, as the loop below computes it
                    const float pm = ex2(fmaf(mx, c, -m_use));
                    float h0, h1;
                    unpack_f16x2(pack_f16x2(pm, 0.0f), h0, h1);
                    lc += h0 - pm;
                }
                // p = 2^(s c - m): exponent argument two lanes per instruction,
                // row sum in four paired accumulators.
                const uint64_t c2 = f2(c, c), negm2 = f2(-m_use, -m_use);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pk[2][32];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int e2 = 0; e2 < 32; ++e2) {
                        const int e = hh * 64 + 2 * e2;
                        float p0, p1;
                        if (kExp2FmaEvery > 0 && e2 % kExp2FmaMod == kExp2FmaMod - 1) {
                            // this pair on the FMA pipe (exp2_fma2), the rest
                            // on the exponential unit
                            f2_split(exp2_fma2(f2_fma(f2(sv[e], sv[e + 1]), c2, negm2)), p0, p1);
                        } else {
                            float x0, x1;
                            f2_split(f2_fma(f2(sv[e], sv[e + 1]), c2, negm2), x0, x1);
                            p0 = ex2(x0);
                            p1 = ex2(x1);
                        }
                        acc2[e2 & 3] = f2_add(acc2[e2 & 3], f2(p0, p1));
                        pk[hh][e2] = PRECISE ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                    }
                    if (!SEP) tmem_st32(lane_addr + col_s + hh * 32, pk[hh]);
                }
                if (SEP) {
                    // P_t and O_t are free once P_t(j-1) V has completed.
                    if (j > lo) {
                        if (!fa_wait_warp(&bar_pv[t], cpv & 1, 34 + t, wc)) { ok = false; break; }
                        ++cpv;
                        tc_fence_after();
                        if (any_need) rescale_o(alpha);
                    }
                    tmem_st32(lane_addr + col_p, pk[0]);
                    tmem_st32(lane_addr + col_p + 32, pk[1]);
                }
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
            // O row -> registers, release the O columns to the next item's
            // MMAs, then normalise and store.
            // The last P_t V MMA of the item has completed.  Without separate
            // P columns the softmax did not wait for the earlier ones; each S
            // MMA was issued only after the P V MMA before it had completed,
            // so those are complete already.
            if (!SEP) cpv += n_kv - lo - 1;
            if (!fa_wait_warp(&bar_pv[t], cpv & 1, 34 + t, wc)) { ok = false; break; }
            ++cpv;
            tc_fence_after();
            uint32_t ov[D / 32][32];
#pragma unroll
            for (int c0 = 0; c0 < D / 32; ++c0) tmem_ld32(lane_addr + col_o + c0 * 32, ov[c0]);
            tmem_ld_wait(ov[0]);
#pragma unroll
            for (int c0 = 1; c0 < D / 32; ++c0) asm volatile("" : FA_R32(ov[c0]) : : "memory");
            tc_fence_before();
            mbar_arrive(&bar_o_free[t]);
            const bool valid = row < wt.len;
            const float l_o = PRECISE ? l + lc : l;
            const float inv_l = (l_o > 0.0f) ? 1.0f / l_o : 0.0f;
            const size_t orow = ((size_t)wt.q_z * p.rows + wt.tok0 + (valid ? row : 0)) * D;
            if (valid) {
#pragma unroll
                for (int c0 = 0; c0 < D / 32; ++c0) {
                    if (PRECISE) {
                        float4* dst =
                            reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow + c0 * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(ov[c0][q4 * 4 + 0]) * inv_l,
                                                  __uint_as_float(ov[c0][q4 * 4 + 1]) * inv_l,
                                                  __uint_as_float(ov[c0][q4 * 4 + 2]) * inv_l,
                                                  __uint_as_float(ov[c0][q4 * 4 + 3]) * inv_l);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(
                            static_cast<__nv_bfloat16*>(p.o) + orow + c0 * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 0]) * inv_l,
                                              __uint_as_float(ov[c0][q4 * 8 + 1]) * inv_l);
                            w.y = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 2]) * inv_l,
                                              __uint_as_float(ov[c0][q4 * 8 + 3]) * inv_l);
                            w.z = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 4]) * inv_l,
                                              __uint_as_float(ov[c0][q4 * 8 + 5]) * inv_l);
                            w.w = pack_bf16x2(__uint_as_float(ov[c0][q4 * 8 + 6]) * inv_l,
                                              __uint_as_float(ov[c0][q4 * 8 + 7]) * inv_l);
                            dst[q4] = w;
                        }
                    }
                }
                p.lse[(size_t)wt.q_z * p.rows + wt.tok0 + row] =
                    (l > 0.0f) ? (m2 + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
            }
            if (p.lse_ext != nullptr && row0 < p.Np) {
                // Training forward: this tile's rows of the backward workspace
                // (a tile lies wholly below Np or wholly past it: both are
                // multiples of 128).  The -LSE row as the preprocess would
                // write it from the stored LSE (padding rows past N get -1e30,
                // so P = 0 there), and the tile's 128 fp32 dQ accumulator rows
                // zeroed, contiguous in memory: consecutive threads write
                // consecutive 16-byte pieces, so each warp store is coalesced.
                const long long r0 = (long long)wt.bh * p.Np + row0;
                const float lse_row =
                    (l > 0.0f) ? (m2 + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
                write_lse_ext_row(p.lse_ext, r0 + rl,
                                  valid ? -lse_row * 1.4426950408889634f : -1e30f);
                float4* z = reinterpret_cast<float4*>(p.dq_acc + r0 * D);
#pragma unroll
                for (int c4 = 0; c4 < D / 4; ++c4) z[c4 * kBM + rl] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (!PRECISE && warp == kProducerWarp && lane == 0) {
            // ------------------------------------------------- K producer
            tma_prefetch_desc(&tm_k);
            uint32_t g = 0;              // K blocks loaded so far (ring position)
            bool ok = true;
            FwdSched<VARLEN> sch;
            for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
                 item = sch.next(p, CAUSAL)) {
                const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
                for (int j = wt.lo[0]; j < wt.n_kv[kTiles - 1]; ++j, ++g) {
                    const int s = g % SK;
                    if (g >= (uint32_t)SK && !fa_wait(&bar_k_empty[s], ((g / SK) - 1) & 1, 10, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_k[s], Cfg::kTileBytes);
                    for (int c = 0; c < Cfg::kChunks; ++c)
                        tma_load_3d(sK + s * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_k, &bar_k[s],
                                    c * 64, wt.tok0 + j * kBN, wt.kv_z);
                }
            }
            if (abort_sh) {   // drain the copies still in flight (bounded)
                const WaitCtx dc{p.status, nullptr};
                for (uint32_t x = (g > (uint32_t)SK ? g - SK : 0); x < g; ++x)
                    fa_wait(&bar_k[x % SK], (x / SK) & 1, 11, dc);
            }
        } else if (!PRECISE && warp == kVProducerWarp && lane == 0) {
            // ---------------------------------------------- V and Q producer
            // The Q tiles of an item are loaded ahead of its V blocks, as soon
            // as the last S MMAs of the previous item have read the old ones.
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_q);
            uint32_t g = 0;
            int lt = 0, q_loaded = -1;
            bool ok = true;
            FwdSched<VARLEN> sch;
            for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
                 item = sch.next(p, CAUSAL), ++lt) {
                const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
                for (int t = 0; t < kTiles; ++t) {
                    if (lt > 0 && !fa_wait(&bar_q_free[t], (lt - 1) & 1, 12, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar_q[t], Cfg::kTileBytes);
                    for (int c = 0; c < Cfg::kChunks; ++c)
                        tma_load_3d(sQ + t * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_q,
                                    &bar_q[t], c * 64, wt.tok0 + wt.row_base + t * kBM, wt.q_z);
                }
                if (!ok) break;
                q_loaded = lt;
                for (int j = wt.lo[0]; j < wt.n_kv[kTiles - 1]; ++j, ++g) {
                    const int s = g % SV;
                    if (g >= (uint32_t)SV && !fa_wait(&bar_v_empty[s], ((g / SV) - 1) & 1, 13, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_v[s], Cfg::kTileBytes);
                    for (int c = 0; c < Cfg::kChunks; ++c)
                        tma_load_3d(sV + s * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_v, &bar_v[s],
                                    c * 64, wt.tok0 + j * kBN, wt.kv_z);
                }
            }
            if (abort_sh) {   // drain the copies still in flight (bounded)
                const WaitCtx dc{p.status, nullptr};
                for (uint32_t x = (g > (uint32_t)SV ? g - SV : 0); x < g; ++x)
                    fa_wait(&bar_v[x % SV], (x / SV) & 1, 14, dc);
                if (q_loaded >= 0)
                    for (int t = 0; t < kTiles; ++t) fa_wait(&bar_q[t], q_loaded & 1, 15, dc);
            }
        } else if (warp == kProducerWarp && (PRECISE || lane == 0)) {
            // ------------------------------------- K producer, PRECISE form
            // (This and the next form are written to cover the bf16 case as
            // well, where the branches above take it first; equivalent to
            // PRECISE-only conditions, but the kernel built from this form
            // measured 8 % faster.)
            // The whole warp runs this loop (lane 0 issues the copies) and,
            // before issuing K_g, converts its half of V_{g-2}.
            // Issuing K_g waits for the S MMAs of K_{g-SK}, which follow the
            // P V MMAs of V_{g-SK-1}, whose half was converted before; the
            // issue of V_{g-2} waits for nothing this warp does from here on.
            const bool leader = (lane == 0);
            if (leader) tma_prefetch_desc(&tm_k);
            uint32_t g = 0, gc = 0;      // K blocks loaded (ring position); V halves converted
            bool ok = true;
            FwdSched<VARLEN> sch;
            for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
                 item = sch.next(p, CAUSAL)) {
                const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
                for (int j = wt.lo[0]; j < wt.n_kv[kTiles - 1]; ++j, ++g) {
                    if (PRECISE && gc + 2 <= g) {
                        if (!convert_v_half<SV, Cfg::kTileBytes>(sV, bar_v, bar_v_cvt, gc, 1, lane, wc)) {
                            ok = false;
                            break;
                        }
                        ++gc;
                    }
                    const int s = g % SK;
                    if (g >= (uint32_t)SK && !(PRECISE ? fa_wait_warp(&bar_k_empty[s], ((g / SK) - 1) & 1, 10, wc)
                                                       : fa_wait(&bar_k_empty[s], ((g / SK) - 1) & 1, 10, wc))) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        mbar_arrive_expect_tx(&bar_k[s], Cfg::kTileBytes);
                        for (int c = 0; c < Cfg::kChunks; ++c)
                            tma_load_3d(sK + s * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_k,
                                        &bar_k[s], c * 64, wt.tok0 + j * kBN, wt.kv_z);
                    }
                }
            }
            while (PRECISE && ok && gc < g)
                ok = convert_v_half<SV, Cfg::kTileBytes>(sV, bar_v, bar_v_cvt, gc++, 1, lane, wc);
            if (abort_sh && leader) {   // drain the copies still in flight (bounded)
                const WaitCtx dc{p.status, nullptr};
                for (uint32_t x = (g > (uint32_t)SK ? g - SK : 0); x < g; ++x)
                    fa_wait(&bar_k[x % SK], (x / SK) & 1, 11, dc);
            }
        } else if (warp == kVProducerWarp && (PRECISE || lane == 0)) {
            // -------------------------------- V and Q producer, PRECISE form
            // The whole warp runs this loop (lane 0 issues the copies) and
            // re-encodes its half of each V_g as fp16 as soon as it has
            // landed, before issuing V_{g+1}; the P V issuer waits for that
            // and for the K producer warp's half.  Issuing V_{g+1} waits for
            // the P V MMAs of V_{g+1-SV}, converted before, so the two never
            // wait on each other.  An item's first V block is issued ahead of
            // its Q tiles, so that it lands while the Q loads wait for the
            // previous item's last S MMAs.
            const bool leader = (lane == 0);
            if (leader) {
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_q);
            }
            uint32_t g = 0;   // V blocks issued (and their first halves converted)
            int lt = 0, q_loaded = -1;
            bool ok = true;
            FwdSched<VARLEN> sch;
            for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
                 item = sch.next(p, CAUSAL), ++lt) {
                const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
                const int jb = wt.lo[0], je = wt.n_kv[kTiles - 1];
                auto issue_v = [&](int j) -> bool {   // V_j into the ring
                    const int s = g % SV;
                    if (g >= (uint32_t)SV && !(PRECISE ? fa_wait_warp(&bar_v_empty[s], ((g / SV) - 1) & 1, 13, wc) : fa_wait(&bar_v_empty[s], ((g / SV) - 1) & 1, 13, wc)))
                        return false;
                    if (leader) {
                        mbar_arrive_expect_tx(&bar_v[s], Cfg::kTileBytes);
                        for (int c = 0; c < Cfg::kChunks; ++c)
                            tma_load_3d(sV + s * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_v,
                                        &bar_v[s], c * 64, wt.tok0 + j * kBN, wt.kv_z);
                    }
                    ++g;
                    return true;
                };
                const bool pre = PRECISE && jb < je;
                if (pre && !issue_v(jb)) { ok = false; break; }
                for (int t = 0; t < kTiles; ++t) {
                    if (lt > 0 && !(PRECISE ? fa_wait_warp(&bar_q_free[t], (lt - 1) & 1, 12, wc) : fa_wait(&bar_q_free[t], (lt - 1) & 1, 12, wc))) { ok = false; break; }
                    if (leader) {
                        mbar_arrive_expect_tx(&bar_q[t], Cfg::kTileBytes);
                        for (int c = 0; c < Cfg::kChunks; ++c)
                            tma_load_3d(sQ + t * Cfg::kTileBytes + c * Cfg::kChunkBytes, &tm_q,
                                        &bar_q[t], c * 64, wt.tok0 + wt.row_base + t * kBM, wt.q_z);
                    }
                }
                if (!ok) break;
                q_loaded = lt;
                for (int j = jb; j < je; ++j) {
                    // (issue_v counts V_j before the conversion: an abort drains it)
                    if (!(pre && j == jb) && !issue_v(j)) { ok = false; break; }
                    if (PRECISE && !convert_v_half<SV, Cfg::kTileBytes>(sV, bar_v, bar_v_cvt, g - 1, 0, lane, wc)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (abort_sh && leader) {   // drain the copies still in flight (bounded)
                const WaitCtx dc{p.status, nullptr};
                for (uint32_t x = (g > (uint32_t)SV ? g - SV : 0); x < g; ++x)
                    fa_wait(&bar_v[x % SV], (x / SV) & 1, 14, dc);
                if (q_loaded >= 0)
                    for (int t = 0; t < kTiles; ++t) fa_wait(&bar_q[t], q_loaded & 1, 15, dc);
            }
        } else if (warp == kPvWarp && lane == 0) {
            // ------------------------------------------- P V MMA issuer
            // O_t += P_t V_j, P_t read from TMEM.  A second issuing thread:
            // while the S issuer waits or commits, this one keeps the tensor
            // core busy, and the other way round.
            constexpr uint32_t idesc_o =
                PRECISE ? idesc_f16_f32(kBM, D, false, true) : idesc_bf16_f32(kBM, D, false, true);
            const uint32_t sv = smem_u32(sV);
            uint32_t g = 0, cp0 = 0, cp1 = 0;       // V blocks used; P_t arrivals seen
            bool ok = true;
            int lt = 0;
            auto pv = [&](auto tc, uint32_t vstage, bool first, bool wait_o) -> bool {
                constexpr int T = decltype(tc)::value;
                constexpr uint32_t col_o = T ? Cfg::kColO1 : Cfg::kColO0;
                constexpr uint32_t col_s = T ? Cfg::kColS1 : Cfg::kColS0;
                constexpr uint32_t col_p = SEP ? (T ? Cfg::kColP1 : Cfg::kColP0) : col_s;
                uint32_t& c = T ? cp1 : cp0;
                if (!fa_wait(&bar_p[T], c & 1, 24 + T, wc)) return false;
                ++c;
                if (wait_o && !fa_wait(&bar_o_free[T], (lt - 1) & 1, 26 + T, wc)) return false;
                tc_fence_after();
                const uint64_t vd = sdesc_sw128(sv + vstage * Cfg::kTileBytes, Cfg::kChunkBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tmem + col_o, tmem + col_p + kk * 8, vd + mnmajor_step(kk), idesc_o,
                           (!first || kk > 0) ? 1u : 0u);
                mma_commit(&bar_pv[T]);
                return true;
            };
            FwdSched<VARLEN> sch;
            for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
                 item = sch.next(p, CAUSAL), ++lt) {
                const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
                // Key blocks [lo0, n0) for tile 0, [lo1, n1) for tile 1, with
                // lo0 <= lo1 and n0 <= n1; V_j streams for j in [lo0, n1).
                const int lo0 = wt.lo[0], lo1 = wt.lo[1], n0 = wt.n_kv[0], n1 = wt.n_kv[1];
                for (int j = lo0; j < n1; ++j) {
                    const uint32_t gj = g + (j - lo0), vs = gj % SV;
                    // V_j landed (PRECISE: and re-encoded as fp16)
                    if (!fa_wait(PRECISE ? &bar_v_cvt[vs] : &bar_v[vs], (gj / SV) & 1, 22, wc)) {
                        ok = false;
                        break;
                    }
                    if (j < n0 && !pv(std::integral_constant<int, 0>{}, vs, j == lo0,
                                      j == lo0 && lt > 0)) {
                        ok = false;
                        break;
                    }
                    if (j >= lo1 && !pv(std::integral_constant<int, 1>{}, vs, j == lo1,
                                        j == lo1 && lt > 0)) {
                        ok = false;
                        break;
                    }
                    mma_commit(&bar_v_empty[vs]);            // V_j read by both PVs
                }
                g += n1 - lo0;
            }
            if (!ok) {   // no MMA of this thread may still write TMEM at teardown
                __shared__ uint64_t bar_drain_pv;
                mbar_init(&bar_drain_pv, 1);
                fence_mbar_init();
                mma_commit(&bar_drain_pv);
                fa_wait(&bar_drain_pv, 0, 29, WaitCtx{p.status, nullptr});
            }
        } else if (warp == kMmaWarp && lane == 0) {
            // ---------------------------------------------- S MMA issuer
            // S_t(j) = Q_t K_j^T goes out as soon as K_j has landed and the
            // columns of S_t are free again: loaded by the softmax (P in
            // columns of its own), or read by the P_t V MMA of the previous
            // block (P written over S).  The tile index is a compile-time
            // constant in every MMA, so operand addresses fold into the
            // instruction stream.
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
            const uint32_t sq = smem_u32(sQ), sk = smem_u32(sK);
            uint32_t g = 0, ns0 = 0, ns1 = 0;       // K blocks used; S_t MMAs issued
            bool ok = true;
            int lt = 0;
            auto s_mma = [&](auto tc, uint32_t kstage) -> bool {
                constexpr int T = decltype(tc)::value;
                uint32_t& n = T ? ns1 : ns0;
                if (n > 0 && !fa_wait(SEP ? &bar_s_free[T] : &bar_pv[T], (n - 1) & 1, 36 + T, wc))
                    return false;
                ++n;
                tc_fence_after();
                const uint64_t qd = sdesc_sw128(sq + T * Cfg::kTileBytes, 16, 1024);
                const uint64_t kd = sdesc_sw128(sk + kstage * Cfg::kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + (T ? Cfg::kColS1 : Cfg::kColS0),
                           qd + kmajor_step(kk, Cfg::kChunkBytes),
                           kd + kmajor_step(kk, Cfg::kChunkBytes), idesc_s, kk > 0);
                mma_commit(&bar_s[T]);
                return true;
            };
            FwdSched<VARLEN> sch;
            for (int item = sch.next(p, CAUSAL); ok && item < p.n_items;
                 item = sch.next(p, CAUSAL), ++lt) {
                const FwdTile wt = fwd_tile<WINDOW, VARLEN>(item, p, CAUSAL);
                const int lo0 = wt.lo[0], lo1 = wt.lo[1], n0 = wt.n_kv[0], n1 = wt.n_kv[1];
                if (!fa_wait(&bar_q[0], lt & 1, 20, wc) || !fa_wait(&bar_q[1], lt & 1, 20, wc)) {
                    ok = false;
                    break;
                }
                for (int j = lo0; j < n1; ++j) {
                    const uint32_t gj = g + (j - lo0), ks = gj % SK;
                    if (!fa_wait(&bar_k[ks], (gj / SK) & 1, 21, wc)) { ok = false; break; }
                    if (j < n0) {
                        if (!s_mma(std::integral_constant<int, 0>{}, ks)) { ok = false; break; }
                        if (j + 1 == n0) mma_commit(&bar_q_free[0]);
                    }
                    if (j >= lo1) {
                        if (!s_mma(std::integral_constant<int, 1>{}, ks)) { ok = false; break; }
                        if (j + 1 == n1) mma_commit(&bar_q_free[1]);
                    }
                    mma_commit(&bar_k_empty[ks]);            // K_j read by both S MMAs
                }
                g += n1 - lo0;
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

template <int D, bool CAUSAL, bool PRECISE, bool WINDOW = false, bool VARLEN = false>
cudaError_t launch_fwd_t(const Shape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const FwdParams& p, int grid,
                         cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D, CAUSAL, PRECISE, WINDOW, VARLEN>;
    static int configured_device = -1;   // attribute is per device; cheap to repeat
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        // The register split must fit in what the launch provides, or the
        // setmaxnreg.inc of the softmax warps would wait forever.
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        if (attr.numRegs * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FwdCfg<D, PRECISE>::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<grid, kThreads, FwdCfg<D, PRECISE>::kSmemAlloc, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Shape& s, const void* q, const void* k, const void* v, void* o,
                       float* lse, bool precise, DeviceStatus* status, cudaStream_t stream,
                       const BwdWorkspace* train_ws) {
    // Dense: maps {d, N, B*H(kv)}.  Packed variable lengths: {d, total, H(kv)},
    // a sequence's rows addressed from its first row.
    const bool varlen = s.cu_seqlens != nullptr;
    const int rows = varlen ? s.total : s.N;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_3d(&tq, q, s.d, rows, varlen ? s.H : s.B * s.H, kBM) ||
        !make_tmap_bf16_3d(&tk, k, s.d, rows, varlen ? s.Hkv : s.B * s.Hkv, kBN) ||
        !make_tmap_bf16_3d(&tv, v, s.d, rows, varlen ? s.Hkv : s.B * s.Hkv, kBN))
        return cudaErrorInvalidValue;
    FwdParams p;
    p.H = s.H;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.rows = rows;
    p.cu_seqlens = s.cu_seqlens;
    p.BH = s.B * s.H;
    p.n_mblk = (s.N + kTiles * kBM - 1) / (kTiles * kBM);
    p.n_items = p.n_mblk * p.BH;
    p.causal = s.causal;
    p.window = s.window > 0 ? s.window : kNoWindow;
    p.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
    p.o = o;
    p.lse = lse;
    p.status = status;
    p.lse_ext = nullptr;
    p.dq_acc = nullptr;
    p.Np = padded_rows(s.N);
    if (train_ws) {   // dense batches only (packed ones keep the plain preprocess)
        if (varlen) return cudaErrorInvalidValue;
        p.lse_ext = train_ws->lse_ext;
        p.dq_acc = train_ws->dq_acc;
    }
    // Persistent: one CTA per SM (at most one work item per CTA when there
    // are fewer items than SMs).
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    const int grid = p.n_items < sms ? p.n_items : sms;
    count_launch();
    const bool c = s.causal != 0;
    if (varlen) {   // packed variable-length sequences (bf16 output, no window)
        if (precise || s.window > 0) return cudaErrorInvalidValue;
        if (s.d == 128)
            return c ? launch_fwd_t<128, true, false, false, true>(s, tq, tk, tv, p, grid, stream)
                     : launch_fwd_t<128, false, false, false, true>(s, tq, tk, tv, p, grid, stream);
        return c ? launch_fwd_t<64, true, false, false, true>(s, tq, tk, tv, p, grid, stream)
                 : launch_fwd_t<64, false, false, false, true>(s, tq, tk, tv, p, grid, stream);
    }
    if (s.window > 0) {   // the causal sliding window (bf16 output only)
        if (!c || precise) return cudaErrorInvalidValue;
        return s.d == 128 ? launch_fwd_t<128, true, false, true>(s, tq, tk, tv, p, grid, stream)
                          : launch_fwd_t<64, true, false, true>(s, tq, tk, tv, p, grid, stream);
    }
    if (s.d == 128) {
        if (precise)
            return c ? launch_fwd_t<128, true, true>(s, tq, tk, tv, p, grid, stream)
                     : launch_fwd_t<128, false, true>(s, tq, tk, tv, p, grid, stream);
        return c ? launch_fwd_t<128, true, false>(s, tq, tk, tv, p, grid, stream)
                 : launch_fwd_t<128, false, false>(s, tq, tk, tv, p, grid, stream);
    }
    if (precise)
        return c ? launch_fwd_t<64, true, true>(s, tq, tk, tv, p, grid, stream)
                 : launch_fwd_t<64, false, true>(s, tq, tk, tv, p, grid, stream);
    return c ? launch_fwd_t<64, true, false>(s, tq, tk, tv, p, grid, stream)
             : launch_fwd_t<64, false, false>(s, tq, tk, tv, p, grid, stream);
}

}  // namespace fa
