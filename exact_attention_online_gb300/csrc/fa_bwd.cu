// Backward kernels: recomputation-based attention backward (FlashAttention
// blog, "Backward - Recomputation"; dV = P^T dO from the FlashAttention-2
// review thread's public comment; the other gradients by the calculus of
// softmax attention: dP = dO V^T, D = rowsum(dO o O), dS = P o (dP - D),
// dQ = scale dS K, dK = scale dS^T Q).
//
//   preprocess  writes -D_i = -<dO_i, O_i> and -LSE_i * log2(e) (padded rows:
//               -inf, so P = 0 there), both negated so that the main kernel
//               adds them in paired fp32 FMAs; zeroes the dQ accumulator and
//               the dkdv kernel's work counter.
//   dkdv        one work item per (batch, kv head, block j of 128 keys), taken
//               by persistent CTAs (one an SM) from a counter in the
//               workspace.  K_j and V_j
//               stay in shared memory; dK_j and dV_j accumulate in TMEM over
//               every query head of the GQA group and every query block i that
//               can see the keys (causal: i*Br + Br - 1 >= 128 j).  Per block i:
//                 S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T          (SS MMA)
//                 P^T  = 2^(S^T c - lse2),  dS^T = P^T o (dP^T - D)  (threads)
//                 dV  += P^T dO_i  (A = P^T in TMEM),  dK += dS^T Q_i  (SS)
//                 d=128: dQ_i^T = K_j^T dS^T;  d=64: dQ_i = dS K_j    (SS)
//               and the dQ partial is staged in shared memory and added into
//               the fp32 accumulator by one bulk (d=128) or tensor (d=64)
//               reduce per query block (FlashAttention-2 review 2: the
//               query-derivative update is shared between the workers of one
//               query block).  At d=128 K_j is also copied into tensor memory
//               once per CTA (the last 64 columns), so S^T = K_j Q_i^T is a TS
//               MMA that reads only Q_i from shared memory.
//   dq_convert  dQ = bf16(scale * accumulator).
//
// Roles in dkdv: warps 0-7 compute (one key row per thread, two warps per row
// splitting the query columns), warp 8 TMA producer, warps 9 and 10 MMA
// issuers, warps 12-15 read the dQ partial out of TMEM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kBN = 128;   // keys per CTA
// 16 warps: 0-7 compute (two warpgroups), 8 TMA producer, 9 and 10 MMA
// issuers, 11 idle, 12-15 dQ read-out.
constexpr int kThreads = 512;
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;      // dV and S^T MMAs; allocates TMEM
constexpr int kMma2Warp = 10;    // dK, dQ and dP^T MMAs
constexpr int kReadoutWarp0 = 12;
constexpr int kReadoutThreads = 128;
// Register split (setmaxnreg) of the 512 x 128 launch registers:
// 256 x 152 + 128 x 96 + 128 x 112 = 65536.  With 112 for the control warps
// (producer, MMA issuers) no role spills; 96 left the MMA issuers spilling.
constexpr int kRegsCompute = 152;
constexpr int kRegsReadout = 96;
constexpr int kRegsControl = 112;
constexpr int kRegsNeeded = 256 * kRegsCompute + 128 * kRegsReadout + 128 * kRegsControl;

template <int D, bool KV2 = false>
struct BwdCfg {
    static constexpr int kBR = (D == 128) ? 64 : 128;        // queries per step
    static constexpr int kKVBytes = kBN * D * 2;              // K_j or V_j
    static constexpr int kQBytes = kBR * D * 2;               // Q_i or dO_i
    static constexpr int kDSBytes = kBN * kBR * 2;            // dS^T tile
    // KV2 (causal d = 64): two K/V slots, the next work item's K_j, V_j
    // loading while the current item runs, and one dQ staging tile to make
    // room.  Otherwise one K/V slot and two staging tiles: at d = 128 a second
    // slot does not fit, and without the mask the items are long enough that
    // the second staging tile is worth more (-2 % vs +2 % at d = 64).
    static_assert(!KV2 || D == 64, "two K/V slots fit at d = 64 only");
    static constexpr int kKVSlots = KV2 ? 2 : 1;
    static constexpr int kStageTiles = KV2 ? 1 : 2;
    static constexpr int kKVSlotBytes = 2 * kKVBytes;         // K_j, then V_j
    static constexpr int kOffK = 0;                           // + slot * kKVSlotBytes
    static constexpr int kOffV = kOffK + kKVBytes;            // + slot * kKVSlotBytes
    static constexpr int kOffQ = kKVSlots * kKVSlotBytes;     // 2 stages
    static constexpr int kOffDO = kOffQ + 2 * kQBytes;        // 2 stages
    static constexpr int kOffDS = kOffDO + 2 * kQBytes;
    static constexpr int kOffStage = kOffDS + kDSBytes;       // kStageTiles fp32 dQ staging tiles
    static constexpr int kStageTileBytes = kBR * D * 4;        // 32 KB for both head dims
    // The K = 16 extension operands (unswizzled core matrices, 32 bytes a
    // row): the constant A tile for the 128 key rows, and per stage the -LSE
    // and -D tables of the BR query rows.
    static constexpr int kOnesBytes = kBN * 32;
    static constexpr int kExtBytes = kBR * 32;
    static constexpr int kOffOnes = kOffStage + kStageTiles * kStageTileBytes;
    static constexpr int kOffExt = kOffOnes + kOnesBytes;     // [2 stages][lse, d]
    static constexpr int kSmemBytes = kOffExt + 4 * kExtBytes;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;
    static constexpr int kStageBytes = 2 * kQBytes + 2 * kExtBytes;
    // TMEM columns
    static constexpr uint32_t kColDK = 0, kColDV = D, kColS = 2 * D, kColDP = 2 * D + kBR,
                              kColDQ = 2 * D + 2 * kBR;
    // d = 128: K_j as bf16 pairs (128 key lanes x 64 columns) in the last 64
    // columns, the A operand of S^T = K_j Q_i^T read from tensor memory
    // instead of shared memory.
    static constexpr uint32_t kColKT = kColDQ + 64;
    static constexpr bool kKInTmem = (D == 128);
};

struct BwdParams {
    int H, Hkv, N, Np, G, causal;
    int rows;                         // rows per head of q, k, v, dk, dv: N, or the packed total
    int chunk;                        // key/value heads per key-block-major chunk (causal)
    // Causal sliding window W: key k is seen by queries k <= i < k + W.
    // Without a window this holds kNoWindow.
    int window;
    // Packed variable-length batches: sequence b is rows cu_seqlens[b] ..
    // cu_seqlens[b+1] - 1 of every head; N is then the longest sequence and
    // the workspace keeps N-row (padded) regions per (batch, head).
    const int* cu_seqlens;
    float scale, scale_log2;
    const uint16_t* lse_ext;          // workspace tables (fa_internal.h)
    const uint16_t* d_ext;
    float* dq_acc;
    int* work;                        // next work item (zero on entry, left zero)
    int n_bg, n_items;                // B * Hkv; work items (B * Hkv * key blocks)
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    DeviceStatus* status;
};

// What one dK/dV work item covers: (batch, kv head, key block j) and the
// range of query blocks (of br rows) that see some key of the block.  The
// persistent CTAs take the items in index order from the work counter, so
// that, as with one CTA per item, the hardware-like first-come order decides
// which SM runs which item.  Dense causal batches: key-block-major, so that the
// longest CTAs (small j, every query block after them) start first and the
// shortest fill the tail (a CPU model of the bench workloads puts the busiest
// SM within 1-2 % of the mean instead of 7-14 %; measured: dK/dV +2 % to
// +13 %).  Otherwise head-major: without the mask every CTA costs the same and
// the CTAs that run at the same time share Q and dO in L2 (key-block-major
// measured 12 % slower there), and with packed sequences of different lengths
// j does not rank the cost (measured 12 % slower).  Key-block-major runs over
// chunks of p.chunk heads at a time, sized so that a chunk's Q, dO and dQ
// accumulator stay in L2 while its key blocks re-read them.
struct BwdCta {
    int jblk, b, g, bg, tok0, seq_len, z_kv, i_start, n_i, n_it;
    bool idle;   // a key block past its packed sequence's end: nothing to do
};
template <bool CAUSAL, bool WINDOW, bool VARLEN>
__device__ __forceinline__ BwdCta bwd_cta(const BwdParams& p, int br, int item) {
    BwdCta c;
    constexpr bool kKeyMajor = CAUSAL && !VARLEN;
    const int n_kblk = (p.N + kBN - 1) / kBN;
    const int n_bg = p.n_bg;                      // B * Hkv
    if (kKeyMajor) {
        const int chunk = item / (p.chunk * n_kblk), loc = item % (p.chunk * n_kblk);
        const int width = min(p.chunk, n_bg - chunk * p.chunk);
        c.jblk = loc / width;
        c.bg = chunk * p.chunk + loc % width;
    } else {
        c.jblk = item % n_kblk;
        c.bg = item / n_kblk;
    }
    c.b = c.bg / p.Hkv;
    c.g = c.bg % p.Hkv;
    // The sequence: its first row in the tensors and its length.  Dense
    // batches address rows of head b*H(kv) + h; packed ones rows tok0 + i of
    // head h.
    c.tok0 = 0;
    c.seq_len = VARLEN ? packed_seq(p.cu_seqlens, c.b, p.N, p.rows, c.tok0) : p.N;
    c.idle = VARLEN && c.jblk * kBN >= c.seq_len;
    c.z_kv = VARLEN ? c.g : c.bg;
    const int n_qblk = (c.seq_len + br - 1) / br;
    // Query blocks that see some key of the block: rows 128 j .. 128 j + 127
    // + W - 1 under the causal (windowed) mask.
    c.i_start = CAUSAL ? (c.jblk * kBN) / br : 0;
    const int i_end = WINDOW ? min(n_qblk, (c.jblk * kBN + kBN - 1 + (p.window - 1)) / br + 1)
                             : n_qblk;
    c.n_i = i_end - c.i_start;
    c.n_it = p.G * c.n_i;                         // (head in group) x (query block)
    return c;
}

// The constant A operand of the extension MMAs, 128 key rows x 16 columns:
// cols 0-8 hold 1/c as three bf16 terms (h h h m m m l l l), against the B
// columns (x_h x_m x_l) x 3 of -LSE log2(e), so that the nine products sum to
// (-LSE log2 e) / c; cols 9-11 hold 1 against the three terms of -D; the rest
// 0.  One 16-byte piece per thread of the first 256.
__device__ __forceinline__ void bwd_fill_ones(uint8_t* sOnes, float scale_log2) {
    if (threadIdx.x < kBN * 32 / 16) {
        const float inv = 1.0f / scale_log2;
        const float ih = bf16_round(inv), im = bf16_round(inv - ih),
                    il = bf16_round(inv - ih - im);
        const int kc = (threadIdx.x >> 3) & 1;   // K half of this core-matrix row
        uint4 w;
        if (kc == 0) {
            w.x = pack_bf16x2(ih, ih);
            w.y = pack_bf16x2(ih, im);
            w.z = pack_bf16x2(im, im);
            w.w = pack_bf16x2(il, il);
        } else {
            w.x = pack_bf16x2(il, 1.0f);
            w.y = pack_bf16x2(1.0f, 1.0f);
            w.z = 0u;
            w.w = 0u;
        }
        *reinterpret_cast<uint4*>(sOnes + threadIdx.x * 16) = w;
        fence_proxy_async_smem();
    }
}

// WINDOW (with CAUSAL): the causal sliding window of p.window keys.
// VARLEN: packed variable-length sequences (p.cu_seqlens).
template <int D, bool CAUSAL, bool WINDOW, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using Cfg = BwdCfg<D, (D == 64 && CAUSAL)>;
    constexpr int BR = Cfg::kBR;
    // Two MMA-issuing threads at d = 128 and without the mask (d = 64: +8 %);
    // one for causal d = 64 (two measured 3 % slower there).
    constexpr bool kTwoIssuers = (D == 128) || !CAUSAL;
    constexpr int HALF = BR / 2;                  // query columns per compute warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    constexpr int KVS = Cfg::kKVSlots;
    // bar_kv[s]: K_j, V_j of slot s landed; bar_kv_free[s]: every MMA that
    // reads slot s's K_j, V_j has completed (one arrival per MMA issuer)
    __shared__ uint64_t bar_kv[KVS], bar_kv_free[KVS];
    __shared__ uint64_t bar_full[2], bar_empty[2], bar_s, bar_dp, bar_p, bar_ds, bar_dq_full,
        bar_dq_free, bar_done, bar_ktm;
    // Persistent CTAs: the producer takes work items from p.work and passes
    // them on through a two-slot ring (-1: no more); an item's dK, dV leave
    // tensor memory (bar_acc_free) before the next item's MMAs overwrite them.
    __shared__ uint64_t bar_item_full[2], bar_item_empty[2], bar_acc_free;
    __shared__ int item_sh[2];
    constexpr int kItemConsumers = kComputeWarps + 4 + (kTwoIssuers ? 2 : 1);
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    const WaitCtx wc{p.status, &abort_sh};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;


    uint8_t* sK = smem + Cfg::kOffK;
    uint8_t* sV = smem + Cfg::kOffV;
    uint8_t* sQ = smem + Cfg::kOffQ;
    uint8_t* sDO = smem + Cfg::kOffDO;
    uint8_t* sDS = smem + Cfg::kOffDS;
    float* sStage = reinterpret_cast<float*>(smem + Cfg::kOffStage);   // [tiles][BR*D] fp32
    uint8_t* sOnes = smem + Cfg::kOffOnes;
    uint8_t* sExt = smem + Cfg::kOffExt;      // stage st: lse at 2 st, d at 2 st + 1

    bwd_fill_ones(sOnes, p.scale_log2);

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int s = 0; s < KVS; ++s) {
            mbar_init(&bar_kv[s], 1);
            mbar_init(&bar_kv_free[s], kTwoIssuers ? 2 : 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], kTwoIssuers ? 2 : 1);   // every MMA issuer lets go of the stage
        }
        mbar_init(&bar_s, 1);
        mbar_init(&bar_dp, 1);
        mbar_init(&bar_p, kComputeThreads);
        mbar_init(&bar_ds, kComputeThreads);
        mbar_init(&bar_dq_full, 1);
        mbar_init(&bar_dq_free, kReadoutThreads);
        mbar_init(&bar_done, kTwoIssuers ? 2 : 1);   // one arrival per MMA issuer
        mbar_init(&bar_ktm, kComputeThreads);        // K_j copied into tensor memory
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_item_full[s], 1);
            mbar_init(&bar_item_empty[s], kItemConsumers);
        }
        mbar_init(&bar_acc_free, kComputeThreads);
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

    // The work item of rank n for a consumer warp (all lanes) or thread: false
    // if the wait gave up; item < 0 when there is no more work.
    auto next_item_warp = [&](int n, int& item) -> bool {
        const int slot = n & 1;
        if (!fa_wait_warp(&bar_item_full[slot], (n >> 1) & 1, 65, wc)) return false;
        item = item_sh[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_item_empty[slot]);
        return true;
    };
    auto next_item_thread = [&](int n, int& item) -> bool {
        const int slot = n & 1;
        if (!fa_wait(&bar_item_full[slot], (n >> 1) & 1, 65, wc)) return false;
        item = item_sh[slot];
        mbar_arrive(&bar_item_empty[slot]);
        return true;
    };

    // One register-budget change per warpgroup (all its warps, same
    // instruction); each role below is dominated by exactly one of them.
    if (warp < kComputeWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
        // ---------------------------------------------------------- compute
        // warp w: TMEM lane quarter w % 4 (= 32 key rows), query half w / 4.
        const int quarter = warp & 3, hf = warp >> 2;
        const int rl = quarter * 32 + lane;          // key row within the block
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const int cb = hf * HALF;                    // first query column of this warp
        const float c = p.scale_log2;
        bool ok = true;
        int gi = 0, nb = 0;   // query-block steps and work items of this CTA so far
        for (int n = 0; ok; ++n) {
            int item;
            if (!next_item_warp(n, item) || item < 0) break;
            const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
            if (cta.idle || cta.n_it == 0) continue;
            const int jblk = cta.jblk, tok0 = cta.tok0, seq_len = cta.seq_len, z_kv = cta.z_kv;
            const int i_start = cta.i_start, n_i = cta.n_i, n_it = cta.n_it;
            const int key = jblk * kBN + rl;
            if (Cfg::kKInTmem) {
                // K_j -> tensor memory: this thread's key row, the 64 head-dim
                // columns of its half (one 128-byte swizzled row of chunk hf),
                // as 32 bf16 pairs; the S^T MMAs take it from there.
                if (!fa_wait_warp(&bar_kv[nb % KVS], (nb / KVS) & 1, 64, wc)) {
                    ok = false;
                } else {
                    const uint8_t* rowp =
                        sK + (nb % KVS) * Cfg::kKVSlotBytes + hf * (kBN * 128) + rl * 128;
                    uint32_t kw[32];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint4 x = *reinterpret_cast<const uint4*>(rowp + ((u ^ (rl & 7)) * 16));
                        kw[4 * u + 0] = x.x;
                        kw[4 * u + 1] = x.y;
                        kw[4 * u + 2] = x.z;
                        kw[4 * u + 3] = x.w;
                    }
                    tmem_st32(lane_addr + Cfg::kColKT + hf * 32, kw);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bar_ktm);
                }
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int git = gi + it;
                const int i = i_start + it % n_i;
                // (no wait for the Q_i / dO_i stage: these warps read neither, and
                // S^T(i) completing implies the stage has landed)
                if (!fa_wait_warp(&bar_s, git & 1, 61, wc)) { ok = false; break; }
                tc_fence_after();
                const int q0 = i * BR;
                const bool need_mask = (CAUSAL && (q0 < jblk * kBN + kBN - 1 ||
                                                   (WINDOW && q0 + BR - 1 > jblk * kBN + p.window - 1))) ||
                                       (jblk * kBN + kBN > seq_len);
                // column e visible iff key_lim <= e <= key_hi
                const int key_lim = CAUSAL ? key - q0 : -1;
                const int key_hi = WINDOW ? key + p.window - 1 - q0 : BR;
                const bool key_valid = key < seq_len;
                // P^T = 2^(S'^T c) with S'^T = S^T - LSE log2(e) / c from the
                // tensor core, kept in fp32 for dS; bf16 copy into TMEM over this
                // warp's own S^T columns (already read).  Two columns per
                // paired-fp32 instruction.
                float pf[HALF];
                const uint64_t c2 = f2(c, c);
#pragma unroll
                for (int ch = 0; ch < HALF / 32; ++ch) {
                    uint32_t sr[32];
                    tmem_ld32(lane_addr + Cfg::kColS + cb + ch * 32, sr);
                    tmem_ld_wait(sr);
                    uint32_t pk[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const int qe = cb + ch * 32 + 2 * e2;
                        float x0, x1;
                        f2_split(f2_mul(f2(__uint_as_float(sr[2 * e2]), __uint_as_float(sr[2 * e2 + 1])),
                                        c2),
                                 x0, x1);
                        float p0 = ex2(x0), p1 = ex2(x1);
                        if (need_mask) {
                            if (qe < key_lim || qe > key_hi || !key_valid) p0 = 0.0f;
                            if (qe + 1 < key_lim || qe + 1 > key_hi || !key_valid) p1 = 0.0f;
                        }
                        pf[ch * 32 + 2 * e2] = p0;
                        pf[ch * 32 + 2 * e2 + 1] = p1;
                        pk[e2] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(lane_addr + Cfg::kColS + cb + ch * 16, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_p);

                // dS^T = P^T o (dP^T - D) -> bf16, swizzled [key][query] tile in
                // smem; dP^T - D comes from the tensor core.
                if (!fa_wait_warp(&bar_dp, git & 1, 62, wc)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int ch = 0; ch < HALF / 32; ++ch) {
                    uint32_t dpr[32];
                    tmem_ld32(lane_addr + Cfg::kColDP + cb + ch * 32, dpr);
                    tmem_ld_wait(dpr);
                    uint32_t dsk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float d0, d1;
                        f2_split(f2_mul(f2(pf[ch * 32 + 2 * e], pf[ch * 32 + 2 * e + 1]),
                                        f2(__uint_as_float(dpr[2 * e]), __uint_as_float(dpr[2 * e + 1]))),
                                 d0, d1);
                        dsk[e] = pack_bf16x2(d0, d1);
                    }
                    const int qc = (cb + ch * 32) >> 6;       // 64-query chunk of the tile
                    const int u0 = ((cb + ch * 32) & 63) >> 3;  // first 16-byte unit in the row
                    uint8_t* rowp = sDS + qc * (kBN * 128) + rl * 128;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const int unit = u0 + u4;
                        *reinterpret_cast<uint4*>(rowp + ((unit ^ (rl & 7)) * 16)) =
                            make_uint4(dsk[u4 * 4 + 0], dsk[u4 * 4 + 1], dsk[u4 * 4 + 2],
                                       dsk[u4 * 4 + 3]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&bar_ds);
            }
            // ---------------------------------------------------- dK, dV epilogue
            if (ok && fa_wait_warp(&bar_done, nb & 1, 63, wc)) {
                tc_fence_after();
                const bool valid = key < seq_len;
                const size_t row = ((size_t)z_kv * p.rows + tok0 + (valid ? key : 0)) * D;
                const int c_lo = hf * (D / 2);
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const uint32_t col = which ? Cfg::kColDV : Cfg::kColDK;
                    const float mul = which ? 1.0f : p.scale;
                    __nv_bfloat16* dst = (which ? p.dv : p.dk) + row;
#pragma unroll
                    for (int c0 = c_lo; c0 < c_lo + D / 2; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(lane_addr + col + c0, r);
                        tmem_ld_wait(r);
                        if (valid) {
                            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                uint4 w;
                                w.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * mul,
                                                  __uint_as_float(r[q4 * 8 + 1]) * mul);
                                w.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * mul,
                                                  __uint_as_float(r[q4 * 8 + 3]) * mul);
                                w.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * mul,
                                                  __uint_as_float(r[q4 * 8 + 5]) * mul);
                                w.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * mul,
                                                  __uint_as_float(r[q4 * 8 + 7]) * mul);
                                d4[q4] = w;
                            }
                        }
                    }
                }
                // dK, dV read out: the next item's first dV / dK MMA may overwrite them
                tc_fence_before();
                mbar_arrive(&bar_acc_free);
            } else {
                ok = false;
            }
            gi += n_it;
            ++nb;
        }
    } else if (warp >= kReadoutWarp0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsReadout));
        // ----------------------------------------------------- dQ read-out
        // TMEM -> registers -> fp32 staging tile laid out like the accumulator
        // rows -> one bulk reduce-add of BR*D*4 = 32 KB per query block.
        const int quarter = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const int rl = quarter * 32 + lane;
        const bool leader = (warp == kReadoutWarp0 && lane == 0);
        bool ok = true;
        int gi = 0;   // query-block steps of this CTA so far
        for (int n = 0; ok; ++n) {
            int item;
            if (!next_item_warp(n, item) || item < 0) break;
            const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
            if (cta.idle || cta.n_it == 0) continue;
            const int b = cta.b, g = cta.g, i_start = cta.i_start, n_i = cta.n_i, n_it = cta.n_it;
            for (int it = 0; ok && it < n_it; ++it) {
                const int git = gi + it;
                const int hq = g * p.G + it / n_i;
                const int i = i_start + it % n_i;
                const int bh = b * p.H + hq;
                // The four read-out warps leave together (they meet at named
                // barriers below), so a failed wait in one of them stops all.
                const bool w_ok = fa_wait_warp(&bar_dq_full, git & 1, 70, wc);
                if (named_bar_or(1, kReadoutThreads, !w_ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + Cfg::kColDQ, r0);
                tmem_ld32(lane_addr + Cfg::kColDQ + 32, r1);
                tmem_ld_wait(r0);
                asm volatile("" : FA_R32(r1) : : "memory");
                tc_fence_before();
                mbar_arrive(&bar_dq_free);
                float* stg = sStage + (git % Cfg::kStageTiles) * (BR * D);
                // the copy that last read this tile
                if (leader) bulk_wait_group_read<Cfg::kStageTiles - 1>();
                named_bar_sync(1, kReadoutThreads);
                if (D == 128) {
                    // dQ^T: lane = head-dim index dd, column = query -> stg[q][dd]
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        stg[e * D + rl] = __uint_as_float(r0[e]);
                        stg[(32 + e) * D + rl] = __uint_as_float(r1[e]);
                    }
                } else {
                    // dQ: lane = query row, column = head-dim index.  Two boxes of
                    // 32 columns, 128-byte swizzled (16-byte piece u of row r at
                    // u ^ (r & 7)), so eight neighbouring rows write eight
                    // different bank groups; a tensor reduce undoes the swizzle.
#pragma unroll
                    for (int box = 0; box < 2; ++box) {
                        uint8_t* rowp = reinterpret_cast<uint8_t*>(stg) + box * (128 * 128) + rl * 128;
                        const uint32_t* src = box ? r1 : r0;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            *reinterpret_cast<uint4*>(rowp + ((u ^ (rl & 7)) * 16)) =
                                make_uint4(src[4 * u], src[4 * u + 1], src[4 * u + 2], src[4 * u + 3]);
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(1, kReadoutThreads);
                if (leader) {
                    if (D == 128) {
                        bulk_reduce_add_f32(p.dq_acc + ((size_t)bh * p.Np + (size_t)i * BR) * D, stg,
                                            BR * D * 4);
                    } else {
                        const int y = bh * p.Np + i * BR;
                        tma_reduce_add_2d(&tm_dq, stg, 0, y);
                        tma_reduce_add_2d(&tm_dq, reinterpret_cast<uint8_t*>(stg) + 128 * 128, 32, y);
                    }
                    bulk_commit_group();
                }
            }
            gi += n_it;
        }
        if (leader) bulk_wait_group<0>();
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (warp == kProducerWarp) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_do);
                int gi = 0, nb = 0;          // query-block steps and work items so far
                int issued = 0, kv_issued = 0;
                bool ok = true;
                for (int n = 0; ok; ++n) {
                        const int slot = n & 1;
                        if (n >= 2 && !fa_wait(&bar_item_empty[slot], ((n >> 1) - 1) & 1, 66, wc))
                            break;
                        // Every CTA's last take finds no item; the last of those
                        // takes leaves the counter zero for the next launch.
                        const int old = atomicAdd(p.work, 1);
                        const int item = old < p.n_items ? old : -1;
                        if (old == p.n_items + (int)gridDim.x - 1) *p.work = 0;
                        item_sh[slot] = item;
                        mbar_arrive(&bar_item_full[slot]);
                        if (item < 0) break;
                        const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
                        if (cta.idle || cta.n_it == 0) continue;
                        const int jblk = cta.jblk, b = cta.b, g = cta.g, tok0 = cta.tok0;
                        const int z_kv = cta.z_kv, i_start = cta.i_start, n_i = cta.n_i;
                        const int n_it = cta.n_it;
                        // K_j, V_j into slot nb % KVS, over the item there
                        // before, whose MMAs have completed (with two slots
                        // this load runs while the previous item's MMAs do)
                        const int kvs = nb % KVS;
                        if (nb >= KVS &&
                            !fa_wait(&bar_kv_free[kvs], ((nb / KVS) - 1) & 1, 42, wc))
                            break;
                        uint8_t* sk_ = sK + kvs * Cfg::kKVSlotBytes;
                        uint8_t* sv_ = sV + kvs * Cfg::kKVSlotBytes;
                        mbar_arrive_expect_tx(&bar_kv[kvs], 2 * Cfg::kKVBytes);
                        for (int c = 0; c < D / 64; ++c) {
                            tma_load_3d(sk_ + c * (kBN * 128), &tm_k, &bar_kv[kvs], c * 64,
                                        tok0 + jblk * kBN, z_kv);
                            tma_load_3d(sv_ + c * (kBN * 128), &tm_v, &bar_kv[kvs], c * 64,
                                        tok0 + jblk * kBN, z_kv);
                        }
                        ++kv_issued;
                        for (int it = 0; it < n_it; ++it) {
                            const int git = gi + it;
                            const int st = git & 1, u = git >> 1;
                            if (git >= 2 && !fa_wait(&bar_empty[st], (u - 1) & 1, 40, wc)) {
                                ok = false;
                                break;
                            }
                            const int hq = g * p.G + it / n_i;
                            const int i = i_start + it % n_i;
                            const int bh = b * p.H + hq;
                            const int z_q = VARLEN ? hq : bh;
                            mbar_arrive_expect_tx(&bar_full[st], Cfg::kStageBytes);
                            for (int c = 0; c < D / 64; ++c) {
                                tma_load_3d(sQ + st * Cfg::kQBytes + c * (BR * 128), &tm_q,
                                            &bar_full[st], c * 64, tok0 + i * BR, z_q);
                                tma_load_3d(sDO + st * Cfg::kQBytes + c * (BR * 128), &tm_do,
                                            &bar_full[st], c * 64, tok0 + i * BR, z_q);
                            }
                            const size_t xrow = (size_t)bh * p.Np + (size_t)i * BR;
                            bulk_load(sExt + (2 * st) * Cfg::kExtBytes, p.lse_ext + xrow * kExtCols,
                                      Cfg::kExtBytes, &bar_full[st]);
                            bulk_load(sExt + (2 * st + 1) * Cfg::kExtBytes,
                                      p.d_ext + xrow * kExtCols, Cfg::kExtBytes, &bar_full[st]);
                            issued = git + 1;
                        }
                        gi += n_it;
                        ++nb;
                    }
                    if (abort_sh) {   // drain the copies still in flight (bounded)
                        const WaitCtx dc{p.status, nullptr};
                        for (int x = max(0, kv_issued - KVS); x < kv_issued; ++x)
                            fa_wait(&bar_kv[x % KVS], (x / KVS) & 1, 41, dc);
                        for (int x = max(0, issued - 2); x < issued; ++x)
                            fa_wait(&bar_full[x & 1], (x >> 1) & 1, 41, dc);
                    }
                }
                __syncwarp();
            } else if (!kTwoIssuers && warp == kMmaWarp) {
                // One MMA-issuing thread (d = 64): dV, S^T for the next block, dK,
                // the dQ partial, dP^T for the next block, in that order.
                if (lane == 0) {
                    constexpr uint32_t id_s = idesc_bf16_f32(128, BR, false, false);
                    constexpr uint32_t id_kv = idesc_bf16_f32(128, D, false, true);
                    constexpr uint32_t id_dq = idesc_bf16_f32(128, 64, true, true);
                    const uint32_t sq = smem_u32(sQ), sdo = smem_u32(sDO), sds = smem_u32(sDS);
                    // Descriptors are built once per operand tile and stepped by
                    // constants, keeping the issuing thread's work between MMAs small;
                    // K_j's and V_j's are set per item (their slot alternates).
                    uint32_t sk = smem_u32(sK);
                    uint64_t kd = 0, vd = 0;
                    const uint32_t sext = smem_u32(sExt);
                    const uint64_t onesd = sdesc_plain(smem_u32(sOnes), 128, 256);
                    auto issue_s = [&](int st) {      // S^T = K_j Q_i^T - LSE log2(e) / c
                        const uint64_t qd = sdesc_sw128(sq + st * Cfg::kQBytes, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            if constexpr (Cfg::kKInTmem)
                                mma_ts(tmem + Cfg::kColS, tmem + Cfg::kColKT + kk * 8,
                                       qd + kmajor_step(kk, BR * 128), id_s, kk > 0);
                            else
                                mma_ss(tmem + Cfg::kColS, kd + kmajor_step(kk, kBN * 128),
                                       qd + kmajor_step(kk, BR * 128), id_s, kk > 0);
                        }
                        mma_ss(tmem + Cfg::kColS, onesd, sdesc_plain(sext + 2 * st * Cfg::kExtBytes,
                                                                     128, 256), id_s, 1u);
                        mma_commit(&bar_s);
                    };
                    auto issue_dp = [&](int st) {     // dP^T - D = V_j dO_i^T - D
                        const uint64_t dod = sdesc_sw128(sdo + st * Cfg::kQBytes, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + Cfg::kColDP, vd + kmajor_step(kk, kBN * 128),
                                   dod + kmajor_step(kk, BR * 128), id_s, kk > 0);
                        mma_ss(tmem + Cfg::kColDP, onesd,
                               sdesc_plain(sext + (2 * st + 1) * Cfg::kExtBytes, 128, 256), id_s, 1u);
                        mma_commit(&bar_dp);
                    };
                    bool ok = true;
                    int gi = 0, nb = 0;   // query-block steps and work items so far
                    for (int n = 0; ok; ++n) {
                    int item;
                    if (!next_item_thread(n, item)) { ok = false; break; }
                    if (item < 0) break;
                    const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
                    if (cta.idle || cta.n_it == 0) continue;
                    const int n_it = cta.n_it;
                    // K_j, V_j (and K_j in tensor memory) of this item, its first
                    // stage, and the previous item's dK, dV read out
                    const int kvs = nb % KVS;
                    sk = smem_u32(sK) + kvs * Cfg::kKVSlotBytes;
                    kd = sdesc_sw128(sk, 16, 1024);
                    vd = sdesc_sw128(smem_u32(sV) + kvs * Cfg::kKVSlotBytes, 16, 1024);
                    ok = fa_wait(&bar_kv[kvs], (nb / KVS) & 1, 50, wc) &&
                         fa_wait(&bar_full[gi & 1], (gi >> 1) & 1, 51, wc) &&
                         (!Cfg::kKInTmem || fa_wait(&bar_ktm, nb & 1, 57, wc)) &&
                         (nb == 0 || fa_wait(&bar_acc_free, (nb - 1) & 1, 58, wc));
                    if (ok) {
                        tc_fence_after();
                        issue_s(gi & 1);
                        issue_dp(gi & 1);
                    }
                    for (int it = 0; ok && it < n_it; ++it) {
                        const int git = gi + it;
                        const int st = git & 1, st1 = (git + 1) & 1;
                        const bool next = it + 1 < n_it;
                        const uint32_t q_ = sq + st * Cfg::kQBytes, do_ = sdo + st * Cfg::kQBytes;
                        // dV += P^T dO_i  (P^T in TMEM; query half h of the K dimension
                        // sits in the S^T columns of the warps of half h)
                        if (!fa_wait(&bar_p, git & 1, 52, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dod_mn = sdesc_sw128(do_, BR * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < BR / 16; ++kk) {
                            const int qs = kk * 16;
                            const uint32_t pcol = Cfg::kColS + (qs / HALF) * HALF + (qs % HALF) / 2;
                            mma_ts(tmem + Cfg::kColDV, tmem + pcol, dod_mn + mnmajor_step(kk), id_kv,
                                   (it > 0 || kk > 0) ? 1u : 0u);
                        }
                        if (next) {
                            if (!fa_wait(&bar_full[st1], ((git + 1) >> 1) & 1, 54, wc)) { ok = false; break; }
                            tc_fence_after();
                            issue_s(st1);
                        }
                        // dK += dS^T Q_i
                        if (!fa_wait(&bar_ds, git & 1, 55, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dsd = sdesc_sw128(sds, 16, 1024);
                        const uint64_t qd_mn = sdesc_sw128(q_, BR * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < BR / 16; ++kk)
                            mma_ss(tmem + Cfg::kColDK, dsd + kmajor_step(kk, kBN * 128),
                                   qd_mn + mnmajor_step(kk), id_kv, (it > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bar_empty[st]);
                        // dQ partial (K dimension = the 128 keys)
                        if (git > 0 && !fa_wait(&bar_dq_free, (git - 1) & 1, 53, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a_ = (D == 128) ? sk : sds;
                        const uint32_t b_ = (D == 128) ? sds : sk;
                        const uint64_t ad_mn = sdesc_sw128(a_, kBN * 128, 1024);
                        const uint64_t bd_mn = sdesc_sw128(b_, kBN * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            mma_ss(tmem + Cfg::kColDQ, ad_mn + mnmajor_step(kk), bd_mn + mnmajor_step(kk),
                                   id_dq, kk > 0);
                        mma_commit(&bar_dq_full);
                        if (next) issue_dp(st1);
                    }
                    if (ok) {   // every MMA of the item, and so every read of its slot
                        mma_commit(&bar_done);
                        mma_commit(&bar_kv_free[kvs]);
                    }
                    gi += n_it;
                    ++nb;
                }
                if (!ok) {   // no MMA of this thread may still write TMEM at teardown
                    __shared__ uint64_t bar_drain1;
                    mbar_init(&bar_drain1, 1);
                    fence_mbar_init();
                    mma_commit(&bar_drain1);
                    fa_wait(&bar_drain1, 0, 59, WaitCtx{p.status, nullptr});
                }
            }
            __syncwarp();
        } else if (kTwoIssuers && (warp == kMmaWarp || warp == kMma2Warp)) {
          if (lane == 0) {
            // MMA issue.  Half A: dV += P^T dO_i, then S^T for block i+1 (it
            // overwrites P^T, so after the dV MMA, in issue order).  Half B:
            // dK += dS^T Q_i, the dQ partial, then dP^T for block i+1 (its
            // completion also tells the compute warps that dS^T may be
            // overwritten).  An MMA issue blocks while the tensor pipe is busy
            // and each barrier wait and commit of an issuing thread costs on
            // the order of a hundred cycles; at d = 128, and at d = 64 without
            // the mask, the halves go to two threads (warps kMmaWarp and
            // kMma2Warp) so that one's waits overlap the other's MMAs.  For
            // causal d = 64 one thread issues both, in the order A, B.
            constexpr uint32_t id_s = idesc_bf16_f32(128, BR, false, false);
            constexpr uint32_t id_kv = idesc_bf16_f32(128, D, false, true);
            constexpr uint32_t id_dq = idesc_bf16_f32(128, 64, true, true);
            const uint32_t sq = smem_u32(sQ), sdo = smem_u32(sDO), sds = smem_u32(sDS);
            uint32_t sk = smem_u32(sK);   // K_j's, V_j's slot is set per item
            uint64_t kd = 0, vd = 0;
            const uint32_t sext = smem_u32(sExt);
            const uint64_t onesd = sdesc_plain(smem_u32(sOnes), 128, 256);
            const bool half_a = (warp == kMmaWarp);
            const bool half_b = (warp == kMma2Warp);
            auto issue_s = [&](int st) {      // S^T = K_j Q_i^T - LSE log2(e) / c
                const uint64_t qd = sdesc_sw128(sq + st * Cfg::kQBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // S^T: A = K_j from tensor memory at d = 128, else shared memory
                    if constexpr (Cfg::kKInTmem)
                        mma_ts(tmem + Cfg::kColS, tmem + Cfg::kColKT + kk * 8,
                               qd + kmajor_step(kk, BR * 128), id_s, kk > 0);
                    else
                        mma_ss(tmem + Cfg::kColS, kd + kmajor_step(kk, kBN * 128),
                               qd + kmajor_step(kk, BR * 128), id_s, kk > 0);
                }
                mma_ss(tmem + Cfg::kColS, onesd, sdesc_plain(sext + 2 * st * Cfg::kExtBytes, 128,
                                                             256), id_s, 1u);
                mma_commit(&bar_s);
            };
            auto issue_dp = [&](int st) {     // dP^T - D = V_j dO_i^T - D
                const uint64_t dod = sdesc_sw128(sdo + st * Cfg::kQBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + Cfg::kColDP, vd + kmajor_step(kk, kBN * 128),
                           dod + kmajor_step(kk, BR * 128), id_s, kk > 0);
                mma_ss(tmem + Cfg::kColDP, onesd,
                       sdesc_plain(sext + (2 * st + 1) * Cfg::kExtBytes, 128, 256), id_s, 1u);
                mma_commit(&bar_dp);
            };
            bool ok = true;
            int gi = 0, nb = 0;   // query-block steps and work items so far
            for (int n = 0; ok; ++n) {
                int item;
                if (!next_item_thread(n, item)) { ok = false; break; }
                if (item < 0) break;
                const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
                if (cta.idle || cta.n_it == 0) continue;
                const int n_it = cta.n_it;
                // K_j, V_j (and for half A K_j in tensor memory) of this item, its
                // first stage, and the previous item's dK, dV read out
                const int kvs = nb % KVS;
                sk = smem_u32(sK) + kvs * Cfg::kKVSlotBytes;
                kd = sdesc_sw128(sk, 16, 1024);
                vd = sdesc_sw128(smem_u32(sV) + kvs * Cfg::kKVSlotBytes, 16, 1024);
                ok = fa_wait(&bar_kv[kvs], (nb / KVS) & 1, 50, wc) &&
                     fa_wait(&bar_full[gi & 1], (gi >> 1) & 1, 51, wc) &&
                     (!(Cfg::kKInTmem && half_a) || fa_wait(&bar_ktm, nb & 1, 57, wc)) &&
                     (nb == 0 || fa_wait(&bar_acc_free, (nb - 1) & 1, 58, wc));
                if (ok) {
                    tc_fence_after();
                    if (half_a) issue_s(gi & 1);
                    if (half_b) issue_dp(gi & 1);
                }
                for (int it = 0; ok && it < n_it; ++it) {
                    const int git = gi + it;
                    const int st = git & 1, st1 = (git + 1) & 1;
                    const bool next = it + 1 < n_it;
                    if (half_a) {
                        // dV += P^T dO_i  (P^T in TMEM; query half h of the K
                        // dimension sits in the S^T columns of the warps of half h)
                        if (!fa_wait(&bar_p, git & 1, 52, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dod_mn = sdesc_sw128(sdo + st * Cfg::kQBytes, BR * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < BR / 16; ++kk) {
                            const int qs = kk * 16;
                            const uint32_t pcol = Cfg::kColS + (qs / HALF) * HALF + (qs % HALF) / 2;
                            mma_ts(tmem + Cfg::kColDV, tmem + pcol, dod_mn + mnmajor_step(kk), id_kv,
                                   (it > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bar_empty[st]);      // half A is done with Q_i, dO_i
                        if (next) {
                            if (!fa_wait(&bar_full[st1], ((git + 1) >> 1) & 1, 54, wc)) { ok = false; break; }
                            tc_fence_after();
                            issue_s(st1);
                        }
                    }
                    if (half_b) {
                        // dK += dS^T Q_i
                        if (!fa_wait(&bar_ds, git & 1, 55, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dsd = sdesc_sw128(sds, 16, 1024);
                        const uint64_t qd_mn = sdesc_sw128(sq + st * Cfg::kQBytes, BR * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < BR / 16; ++kk)
                            mma_ss(tmem + Cfg::kColDK, dsd + kmajor_step(kk, kBN * 128),
                                   qd_mn + mnmajor_step(kk), id_kv, (it > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bar_empty[st]);      // half B is done with Q_i, dO_i
                        // dQ partial (K dimension = the 128 keys)
                        if (git > 0 && !fa_wait(&bar_dq_free, (git - 1) & 1, 53, wc)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a_ = (D == 128) ? sk : sds;
                        const uint32_t b_ = (D == 128) ? sds : sk;
                        const uint64_t ad_mn = sdesc_sw128(a_, kBN * 128, 1024);
                        const uint64_t bd_mn = sdesc_sw128(b_, kBN * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            mma_ss(tmem + Cfg::kColDQ, ad_mn + mnmajor_step(kk), bd_mn + mnmajor_step(kk),
                                   id_dq, kk > 0);
                        mma_commit(&bar_dq_full);
                        if (next) {
                            if (!fa_wait(&bar_full[st1], ((git + 1) >> 1) & 1, 56, wc)) { ok = false; break; }
                            tc_fence_after();
                            issue_dp(st1);
                        }
                    }
                }
                if (ok) {   // one arrival per issuing thread, per item
                    mma_commit(&bar_done);
                    mma_commit(&bar_kv_free[kvs]);
                }
                gi += n_it;
                ++nb;
            }
            const bool first = half_a;
            if (!ok) {   // no MMA of this thread may still write TMEM at teardown
                __shared__ uint64_t bar_drain[2];
                uint64_t* dbar = &bar_drain[first ? 0 : 1];
                mbar_init(dbar, 1);
                fence_mbar_init();
                mma_commit(dbar);
                fa_wait(dbar, 0, 59, WaitCtx{p.status, nullptr});
            }
          }
          __syncwarp();   // reconverge before the block-wide barrier below
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Row i of (batch b, head h) in the caller's [.][rows][d] tensors: dense
// batches keep head b*H + h with rows = N; packed variable-length batches
// (cu != nullptr) keep head h with rows = the total, sequence b starting at
// row cu[b].  Returns the sequence length.
__device__ __forceinline__ int seq_row(const int* __restrict__ cu, long long bh, int H, int N,
                                       long long rows, long long& base) {
    if (!cu) {
        base = bh * N;
        return N;
    }
    const int b = (int)(bh / H), h = (int)(bh % H);
    int t0;
    const int len = packed_seq(cu, b, N, rows, t0);
    base = (long long)h * rows + t0;
    return len;
}

// Per workspace row (b, h, i) that the dK/dV kernel reads (i below the
// sequence's length rounded up to 128: every one of the Np rows of a dense
// batch): the two K = 16 extension tables of the dK/dV kernel and a zeroed dQ
// accumulator row.  x = -LSE log2(e) (padded
// rows: -1e30, so that P = 0 there) and y = -D = -<dO_i, O_i> are each split
// into three bf16 terms (h + m + l holds x to about 24 bits):
//   lse_ext row: cols 0-8 = x_h x_m x_l x_h x_m x_l x_h x_m x_l, 9-15 = 0
//   d_ext row:   cols 9-11 = y_h y_m y_l, the rest 0
// stored as unswizzled K-major core matrices (row group g = r / 8, K half kc:
// 16 bytes at ((2 g + kc) * 8 + r % 8) * 16).  D / 8 lanes per row (16-byte
// loads), 256 / D rows per warp, grid-stride over the B*H*Np rows.  O is
// bf16, or fp32 when it comes from the precise forward.  FULL = false (after
// a training forward, which wrote the -LSE table and zeroed the accumulator):
// the -D table only.
template <int D, typename OT, bool FULL>
__global__ void __launch_bounds__(256)
fa_bwd_pre_kernel(const OT* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                  const float* __restrict__ lse, uint16_t* __restrict__ lse_ext,
                  uint16_t* __restrict__ d_ext, float* __restrict__ dq_acc,
                  int* __restrict__ work, int N, int Np, long long rows,
                  const int* __restrict__ cu, int H, long long seq_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *work = 0;   // the dK/dV kernel's work counter
    constexpr int LPR = D / 8;          // lanes per row, 8 elements each
    constexpr int RPW = 32 / LPR;       // rows per warp
    const int lane = threadIdx.x & 31, sub = lane / LPR, sl = lane % LPR;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r0 = wid * RPW; r0 < rows; r0 += nw * RPW) {
        const long long r = r0 + sub;
        const bool in = r < rows;
        const long long bh = r / Np;
        const int i = (int)(r % Np);
        long long base = 0;
        const int len = in ? seq_row(cu, bh, H, N, seq_rows, base) : 0;
        const bool valid = in && i < len;
        // Rows the dK/dV kernel reads or reduces into: the query blocks of the
        // sequence, up to its length rounded up to 128 (all Np rows of a dense
        // batch; packed sequences shorter than the longest one skip the rest).
        const bool used = in && i < (len + kRowPad - 1) / kRowPad * kRowPad;
        float x = -1e30f;
        if (FULL && valid) x = -lse[base + i] * 1.4426950408889634f;
        float acc = 0.0f;
        if (valid) {
            const long long src = (base + i) * D + sl * 8;
            const uint4 dd = *reinterpret_cast<const uint4*>(dout + src);
            const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dd);
            float ov[8];
            if constexpr (sizeof(OT) == 4) {
                const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(o) + src);
                const float4 b = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(o) + src + 4);
                ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
                ov[4] = b.x; ov[5] = b.y; ov[6] = b.z; ov[7] = b.w;
            } else {
                const uint4 oo = *reinterpret_cast<const uint4*>(o + src);
                const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&oo);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 f = __bfloat1622float2(o2[t]);
                    ov[2 * t] = f.x;
                    ov[2 * t + 1] = f.y;
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 f = __bfloat1622float2(d2[t]);
                acc = fmaf(ov[2 * t], f.x, acc);
                acc = fmaf(ov[2 * t + 1], f.y, acc);
            }
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (used && sl == 0 && FULL) write_lse_ext_row(lse_ext, r, x);   // lane 0: -LSE row
        if (used && sl == 1) {
            // lane 1 of the row: the d_ext row, -D in columns 9-11
            const float v = -acc;
            const float h = bf16_round(v), m = bf16_round(v - h), l = bf16_round(v - h - m);
            uint16_t* row = d_ext + ((r >> 3) * 2 * 8 + (r & 7)) * 8;   // (2 g) * 64 + (r % 8) * 8
            *reinterpret_cast<uint4*>(row) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(row + 64) =                       // K half 1: + 8 rows x 8
                make_uint4(pack_bf16x2(0.0f, h), pack_bf16x2(m, l), 0u, 0u);
        }
        if (FULL && used) {
            float4* z = reinterpret_cast<float4*>(dq_acc + r * D) + sl * 2;
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// dQ = bf16(scale * accumulator), 8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, int N,
                         int Np, float scale, long long n_vec) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n_vec; t += stride) {
        const long long e = t * 8;                  // element index in dq
        const long long row = e / D;                // bh * N + i
        const int col = (int)(e % D);
        const long long bh = row / N;
        const int i = (int)(row % N);
        const float4* src = reinterpret_cast<const float4*>(acc + (bh * Np + i) * D + col);
        const float4 a = src[0], bb = src[1];
        uint4 w;
        w.x = pack_bf16x2(a.x * scale, a.y * scale);
        w.y = pack_bf16x2(a.z * scale, a.w * scale);
        w.z = pack_bf16x2(bb.x * scale, bb.y * scale);
        w.w = pack_bf16x2(bb.z * scale, bb.w * scale);
        *reinterpret_cast<uint4*>(dq + e) = w;
    }
}

// The same for packed variable-length batches: walks the B*H*Np workspace
// rows and writes the rows inside their sequence.
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_dq_convert_varlen_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                const int* __restrict__ cu, int H, int N, int Np,
                                long long seq_rows, float scale, long long n_vec) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n_vec; t += stride) {
        const long long e = t * 8;                  // element index in the accumulator
        const long long row = e / D;                // bh * Np + i
        const int col = (int)(e % D);
        const long long bh = row / Np;
        const int i = (int)(row % Np);
        long long base;
        if (i >= seq_row(cu, bh, H, N, seq_rows, base)) continue;
        const float4* src = reinterpret_cast<const float4*>(acc + e);
        const float4 a = src[0], bb = src[1];
        uint4 w;
        w.x = pack_bf16x2(a.x * scale, a.y * scale);
        w.y = pack_bf16x2(a.z * scale, a.w * scale);
        w.z = pack_bf16x2(bb.x * scale, bb.y * scale);
        w.w = pack_bf16x2(bb.z * scale, bb.w * scale);
        *reinterpret_cast<uint4*>(dq + (base + i) * D + col) = w;
    }
}

// Bounded-wait self-test: one CTA waits on an mbarrier nobody completes.
__global__ void fa_watchdog_kernel(DeviceStatus* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_sh;
    if (threadIdx.x == 0) {
        abort_sh = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    fa_wait(&bar, 0, 99, WaitCtx{status, &abort_sh}, limit_ns);
    __syncthreads();
}

// exp2 on the FMA pipe and on the exponential unit, side by side (diagnostic).
__global__ void fa_exp2_check_kernel(const float* __restrict__ x, float* __restrict__ y_fma,
                                     float* __restrict__ y_ex2, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float a = x[i], b = (i + 1 < n) ? x[i + 1] : 0.0f;
    float r0, r1;
    f2_split(exp2_fma2(f2(a, b)), r0, r1);
    y_fma[i] = r0;
    y_ex2[i] = ex2(a);
    if (i + 1 < n) {
        y_fma[i + 1] = r1;
        y_ex2[i + 1] = ex2(b);
    }
}

int grid_for(long long work_items, int per_block) {
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    long long blocks = (work_items + per_block - 1) / per_block;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

template <int D, bool CAUSAL, bool WINDOW = false, bool VARLEN = false>
cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                          int grid, cudaStream_t stream) {
    auto kern = fa_bwd_dkdv_kernel<D, CAUSAL, WINDOW, VARLEN>;
    using Cfg = BwdCfg<D, (D == 64 && CAUSAL)>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        // The register split must fit in what the launch provides, or the
        // setmaxnreg.inc of the compute warps would wait forever.
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        if (attr.numRegs * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<grid, kThreads, Cfg::kSmemAlloc, stream>>>(tq, tk, tv, tdo, tdq, p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// d = 128 with two query blocks in flight.
//
// The kernel above keeps one query block in flight at d = 128: its period is
// the hand-off chain S^T -> P -> dV -> next S^T and dP^T -> dS -> dK, dQ ->
// next dP^T through the compute warps, over which the tensor pipe idles about
// half the time.  This form runs two pipelines, the even and the odd
// query-block steps of a CTA, each with its own tensor-memory columns, four
// compute warps, dS^T tile and MMA-issuing thread, so that one pipeline's MMAs
// run while the other waits for its compute warps:
//   TMEM  dK 0-127 | dV 128-255 | S^T_0 | dP^T_0 / dQ^T_0 | S^T_1 | dP^T_1 / dQ^T_1
// (64 columns each).  A step's dQ^T goes over its pipeline's dP^T columns
// once the compute warps have read them (they have when dS^T is written), and
// the pipeline's next dP^T waits until the read-out warps have taken dQ^T.
// K_j is read from shared memory (no columns left for a tensor-memory copy).
// Both pipelines accumulate into dK and dV, so the compute warps zero them
// before an item's first dV / dK MMA instead of an accumulate flag doing it,
// and each issuing thread issues step git's dV (dK) MMAs only after the other
// has issued step git - 1's (a turn barrier per accumulator): the tensor core
// takes MMAs in issue order, so dK and dV sum their terms in step order and
// come out bit-reproducible.
// Used at d = 128 except with the sliding window (dense or packed batches,
// with or without the causal mask), where it measured faster (A/B on one
// box: dK/dV -2.1 % gpt_long, -2.8 % gqa; steps +0.7 to +2.6 %, +1.9 %
// packed; the whole backward without the mask -3.5 to -4 % at B4 H16 N4096
// and B8 H16 N2048); with the window it measured 3.5 % slower, so the window
// keeps the one-pipeline kernel.
// Q_i / dO_i stream through three stages so that a pipeline's next block has
// landed while its current one is in use; a stage's landing is signalled on
// one of six barriers (step mod 6), so that each issuing thread waits on
// barriers only it waits on, phase after phase.  The dQ partial leaves
// through a 16 KB staging tile in two halves.
struct Bwd2Cfg {
    static constexpr int D = 128;
    static constexpr int kBR = 64;
    static constexpr int kStages = 3;
    static constexpr int kKVBytes = kBN * D * 2;               // 32 KB
    static constexpr int kQBytes = kBR * D * 2;                // 16 KB
    static constexpr int kDSBytes = kBN * kBR * 2;             // 16 KB
    static constexpr int kStageTileBytes = (kBR / 2) * D * 4;  // 16 KB: half a dQ partial
    static constexpr int kOnesBytes = kBN * 32;
    static constexpr int kExtBytes = kBR * 32;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKVBytes;
    static constexpr int kOffQ = kOffV + kKVBytes;               // kStages
    static constexpr int kOffDO = kOffQ + kStages * kQBytes;     // kStages
    static constexpr int kOffDS = kOffDO + kStages * kQBytes;    // one per pipeline
    static constexpr int kOffStage = kOffDS + 2 * kDSBytes;
    static constexpr int kOffOnes = kOffStage + kStageTileBytes;
    static constexpr int kOffExt = kOffOnes + kOnesBytes;        // [stage][lse, d]
    static constexpr int kSmemBytes = kOffExt + kStages * 2 * kExtBytes;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;
    static constexpr int kStepBytes = 2 * kQBytes + 2 * kExtBytes;
    static constexpr uint32_t kColDK = 0, kColDV = 128;
    __host__ __device__ static constexpr uint32_t col_s(int pp) { return 256 + 128 * pp; }
    __host__ __device__ static constexpr uint32_t col_dpq(int pp) { return 320 + 128 * pp; }
};
static_assert(Bwd2Cfg::kSmemAlloc <= 227 * 1024 - 1024, "shared memory of the two-pipeline kernel");

template <bool CAUSAL, bool WINDOW, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_dkdv2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
    using Cfg = Bwd2Cfg;
    constexpr int D = Cfg::D, BR = Cfg::kBR, NS = Cfg::kStages;
    constexpr int kPipeThreads = 128;            // compute threads of one pipeline
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    // bar_full[git % 6]: step git's Q_i, dO_i and tables landed (stage git % 3)
    __shared__ uint64_t bar_kv, bar_kv_free, bar_full[2 * NS], bar_empty[NS];
    __shared__ uint64_t bar_s[2], bar_dp[2], bar_p[2], bar_ds[2], bar_dq_full[2], bar_dq_free[2];
    __shared__ uint64_t bar_done, bar_acc_free;
    // bar_dv_turn / bar_dk_turn: phase git completes when step git's dV (dK)
    // MMAs have been issued
    __shared__ uint64_t bar_dv_turn, bar_dk_turn;
    __shared__ uint64_t bar_item_full[2], bar_item_empty[2];
    __shared__ int item_sh[2];
    constexpr int kItemConsumers = kComputeWarps + 4 + 2;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    const WaitCtx wc{p.status, &abort_sh};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint8_t* sK = smem + Cfg::kOffK;
    uint8_t* sV = smem + Cfg::kOffV;
    uint8_t* sQ = smem + Cfg::kOffQ;
    uint8_t* sDO = smem + Cfg::kOffDO;
    uint8_t* sDS = smem + Cfg::kOffDS;
    float* sStage = reinterpret_cast<float*>(smem + Cfg::kOffStage);
    uint8_t* sOnes = smem + Cfg::kOffOnes;
    uint8_t* sExt = smem + Cfg::kOffExt;      // stage st: lse at 2 st, d at 2 st + 1

    bwd_fill_ones(sOnes, p.scale_log2);

    if (threadIdx.x == 0) {
        abort_sh = 0;
        mbar_init(&bar_kv, 1);
        mbar_init(&bar_kv_free, 2);                  // one commit per MMA issuer
        for (int s = 0; s < 2 * NS; ++s) mbar_init(&bar_full[s], 1);
        for (int s = 0; s < NS; ++s) mbar_init(&bar_empty[s], 1);   // the step's MMA issuer
        for (int q = 0; q < 2; ++q) {
            mbar_init(&bar_s[q], 1);
            mbar_init(&bar_dp[q], 1);
            mbar_init(&bar_p[q], kPipeThreads);
            mbar_init(&bar_ds[q], kPipeThreads);
            mbar_init(&bar_dq_full[q], 1);
            mbar_init(&bar_dq_free[q], kReadoutThreads);
            mbar_init(&bar_item_full[q], 1);
            mbar_init(&bar_item_empty[q], kItemConsumers);
        }
        mbar_init(&bar_done, 2);                     // one commit per MMA issuer, per item
        mbar_init(&bar_acc_free, kComputeThreads);   // dK, dV zeroed for the item
        mbar_init(&bar_dv_turn, 1);
        mbar_init(&bar_dk_turn, 1);
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

    auto next_item_warp = [&](int n, int& item) -> bool {
        const int slot = n & 1;
        if (!fa_wait_warp(&bar_item_full[slot], (n >> 1) & 1, 65, wc)) return false;
        item = item_sh[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_item_empty[slot]);
        return true;
    };
    auto next_item_thread = [&](int n, int& item) -> bool {
        const int slot = n & 1;
        if (!fa_wait(&bar_item_full[slot], (n >> 1) & 1, 65, wc)) return false;
        item = item_sh[slot];
        mbar_arrive(&bar_item_empty[slot]);
        return true;
    };

    if (warp < kComputeWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
        // ------------------------------------------------------------ compute
        // warp w: pipeline w / 4 (the steps of that parity), TMEM lane quarter
        // w % 4 (= 32 key rows), all 64 query columns of the step.
        const int cp = warp >> 2, quarter = warp & 3;
        const int rl = quarter * 32 + lane;          // key row within the block
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t col_s = Cfg::col_s(cp), col_dp = Cfg::col_dpq(cp);
        uint8_t* const sds = sDS + cp * Cfg::kDSBytes;
        const float c = p.scale_log2;
        bool ok = true;
        int gi = 0, nb = 0;   // query-block steps and work items of this CTA so far
        for (int n = 0; ok; ++n) {
            int item;
            if (!next_item_warp(n, item) || item < 0) break;
            const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
            if (cta.idle || cta.n_it == 0) continue;
            const int jblk = cta.jblk, tok0 = cta.tok0, seq_len = cta.seq_len, z_kv = cta.z_kv;
            const int i_start = cta.i_start, n_i = cta.n_i, n_it = cta.n_it;
            const int key = jblk * kBN + rl;
            // dK (pipeline 0's warps) and dV (pipeline 1's) of this item start
            // from zero; the previous item's were read out below
            {
                uint32_t z[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) z[e] = 0u;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32)
                    tmem_st32(lane_addr + (cp ? Cfg::kColDV : Cfg::kColDK) + c0, z);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_acc_free);
            }
            for (int it = (gi & 1) == cp ? 0 : 1; ok && it < n_it; it += 2) {
                const int git = gi + it;
                const uint32_t k = (uint32_t)git >> 1;       // this pipeline's step count
                const int i = i_start + it % n_i;
                if (!fa_wait_warp(&bar_s[cp], k & 1, 61, wc)) { ok = false; break; }
                tc_fence_after();
                const int q0 = i * BR;
                const bool need_mask = (CAUSAL && (q0 < jblk * kBN + kBN - 1 ||
                                                   (WINDOW && q0 + BR - 1 > jblk * kBN + p.window - 1))) ||
                                       (jblk * kBN + kBN > seq_len);
                const int key_lim = CAUSAL ? key - q0 : -1;
                const int key_hi = WINDOW ? key + p.window - 1 - q0 : BR;
                const bool key_valid = key < seq_len;
                // P^T = 2^(S'^T c), S'^T = S^T - LSE log2(e) / c from the tensor
                // core; fp32 kept for dS, the bf16 pairs written over the first
                // 32 columns of S^T (already read) for the dV MMA.
                float pf[BR];
                const uint64_t c2 = f2(c, c);
#pragma unroll
                for (int ch = 0; ch < BR / 32; ++ch) {
                    uint32_t sr[32];
                    tmem_ld32(lane_addr + col_s + ch * 32, sr);
                    tmem_ld_wait(sr);
                    uint32_t pk[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const int qe = ch * 32 + 2 * e2;
                        float x0, x1;
                        f2_split(f2_mul(f2(__uint_as_float(sr[2 * e2]), __uint_as_float(sr[2 * e2 + 1])),
                                        c2),
                                 x0, x1);
                        float p0 = ex2(x0), p1 = ex2(x1);
                        if (need_mask) {
                            if (qe < key_lim || qe > key_hi || !key_valid) p0 = 0.0f;
                            if (qe + 1 < key_lim || qe + 1 > key_hi || !key_valid) p1 = 0.0f;
                        }
                        pf[qe] = p0;
                        pf[qe + 1] = p1;
                        pk[e2] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(lane_addr + col_s + ch * 16, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_p[cp]);

                // dS^T = P^T o (dP^T - D) -> bf16, swizzled [key][query] tile;
                // dP^T - D comes from the tensor core.  The pipeline's previous
                // dK and dQ MMAs, which read this tile, were issued before this
                // dP^T, so its completion frees the tile.
                if (!fa_wait_warp(&bar_dp[cp], k & 1, 62, wc)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int ch = 0; ch < BR / 32; ++ch) {
                    uint32_t dpr[32];
                    tmem_ld32(lane_addr + col_dp + ch * 32, dpr);
                    tmem_ld_wait(dpr);
                    uint32_t dsk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float d0, d1;
                        f2_split(f2_mul(f2(pf[ch * 32 + 2 * e], pf[ch * 32 + 2 * e + 1]),
                                        f2(__uint_as_float(dpr[2 * e]), __uint_as_float(dpr[2 * e + 1]))),
                                 d0, d1);
                        dsk[e] = pack_bf16x2(d0, d1);
                    }
                    uint8_t* rowp = sds + rl * 128;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const int unit = ch * 4 + u4;
                        *reinterpret_cast<uint4*>(rowp + ((unit ^ (rl & 7)) * 16)) =
                            make_uint4(dsk[u4 * 4 + 0], dsk[u4 * 4 + 1], dsk[u4 * 4 + 2],
                                       dsk[u4 * 4 + 3]);
                    }
                }
                tc_fence_before();   // the dP^T reads precede the dQ^T MMA over them
                fence_proxy_async_smem();
                mbar_arrive(&bar_ds[cp]);
            }
            // ---------------------------------------------------- dK, dV epilogue
            if (ok && fa_wait_warp(&bar_done, nb & 1, 63, wc)) {
                tc_fence_after();
                const bool valid = key < seq_len;
                const size_t row = ((size_t)z_kv * p.rows + tok0 + (valid ? key : 0)) * D;
                const uint32_t col = cp ? Cfg::kColDV : Cfg::kColDK;
                const float mul = cp ? 1.0f : p.scale;
                __nv_bfloat16* dst = (cp ? p.dv : p.dk) + row;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_addr + col + c0, r);
                    tmem_ld_wait(r);
                    if (valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * mul,
                                              __uint_as_float(r[q4 * 8 + 1]) * mul);
                            w.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * mul,
                                              __uint_as_float(r[q4 * 8 + 3]) * mul);
                            w.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * mul,
                                              __uint_as_float(r[q4 * 8 + 5]) * mul);
                            w.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * mul,
                                              __uint_as_float(r[q4 * 8 + 7]) * mul);
                            d4[q4] = w;
                        }
                    }
                }
            } else {
                ok = false;
            }
            gi += n_it;
            ++nb;
        }
    } else if (warp >= kReadoutWarp0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsReadout));
        // ----------------------------------------------------- dQ read-out
        // TMEM (the step's pipeline) -> registers -> fp32 staging tile in two
        // halves of 32 query rows -> a 16 KB bulk reduce-add each.
        const int quarter = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const int rl = quarter * 32 + lane;          // head-dim index
        const bool leader = (warp == kReadoutWarp0 && lane == 0);
        bool ok = true;
        int gi = 0;
        for (int n = 0; ok; ++n) {
            int item;
            if (!next_item_warp(n, item) || item < 0) break;
            const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
            if (cta.idle || cta.n_it == 0) continue;
            const int b = cta.b, g = cta.g, i_start = cta.i_start, n_i = cta.n_i, n_it = cta.n_it;
            for (int it = 0; ok && it < n_it; ++it) {
                const int git = gi + it;
                const int pp = git & 1;
                const uint32_t k = (uint32_t)git >> 1;
                const int hq = g * p.G + it / n_i;
                const int i = i_start + it % n_i;
                const int bh = b * p.H + hq;
                const bool w_ok = fa_wait_warp(&bar_dq_full[pp], k & 1, 70, wc);
                if (named_bar_or(1, kReadoutThreads, !w_ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + Cfg::col_dpq(pp), r0);
                tmem_ld32(lane_addr + Cfg::col_dpq(pp) + 32, r1);
                tmem_ld_wait(r0);
                asm volatile("" : FA_R32(r1) : : "memory");
                tc_fence_before();
                mbar_arrive(&bar_dq_free[pp]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // the copy that last read the staging tile
                    if (leader) bulk_wait_group_read<0>();
                    named_bar_sync(1, kReadoutThreads);
                    // dQ^T: lane = head-dim index, column = query -> stg[q][dd]
                    const uint32_t* src = h ? r1 : r0;
#pragma unroll
                    for (int e = 0; e < 32; ++e) sStage[e * D + rl] = __uint_as_float(src[e]);
                    fence_proxy_async_smem();
                    named_bar_sync(1, kReadoutThreads);
                    if (leader) {
                        bulk_reduce_add_f32(
                            p.dq_acc + ((size_t)bh * p.Np + (size_t)i * BR + h * (BR / 2)) * D, sStage,
                            Cfg::kStageTileBytes);
                        bulk_commit_group();
                    }
                }
            }
            gi += n_it;
        }
        if (leader) bulk_wait_group<0>();
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (warp == kProducerWarp) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_do);
                int gi = 0, nb = 0;
                int issued = 0, kv_issued = 0;
                bool ok = true;
                for (int n = 0; ok; ++n) {
                    const int slot = n & 1;
                    if (n >= 2 && !fa_wait(&bar_item_empty[slot], ((n >> 1) - 1) & 1, 66, wc)) break;
                    // Every CTA's last take finds no item; the last of those
                    // takes leaves the counter zero for the next launch.
                    const int old = atomicAdd(p.work, 1);
                    const int item = old < p.n_items ? old : -1;
                    if (old == p.n_items + (int)gridDim.x - 1) *p.work = 0;
                    item_sh[slot] = item;
                    mbar_arrive(&bar_item_full[slot]);
                    if (item < 0) break;
                    const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
                    if (cta.idle || cta.n_it == 0) continue;
                    const int jblk = cta.jblk, b = cta.b, g = cta.g, tok0 = cta.tok0;
                    const int z_kv = cta.z_kv, i_start = cta.i_start, n_i = cta.n_i;
                    const int n_it = cta.n_it;
                    // K_j, V_j over the previous item's, whose MMAs have completed
                    if (nb > 0 && !fa_wait(&bar_kv_free, (nb - 1) & 1, 42, wc)) break;
                    mbar_arrive_expect_tx(&bar_kv, 2 * Cfg::kKVBytes);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_3d(sK + c * (kBN * 128), &tm_k, &bar_kv, c * 64, tok0 + jblk * kBN,
                                    z_kv);
                        tma_load_3d(sV + c * (kBN * 128), &tm_v, &bar_kv, c * 64, tok0 + jblk * kBN,
                                    z_kv);
                    }
                    ++kv_issued;
                    for (int it = 0; it < n_it; ++it) {
                        const int git = gi + it;
                        const int st = git % NS, u = git / NS;
                        if (git >= NS && !fa_wait(&bar_empty[st], (u - 1) & 1, 40, wc)) {
                            ok = false;
                            break;
                        }
                        const int hq = g * p.G + it / n_i;
                        const int i = i_start + it % n_i;
                        const int bh = b * p.H + hq;
                        const int z_q = VARLEN ? hq : bh;
                        uint64_t* full = &bar_full[git % (2 * NS)];
                        mbar_arrive_expect_tx(full, Cfg::kStepBytes);
                        for (int c = 0; c < D / 64; ++c) {
                            tma_load_3d(sQ + st * Cfg::kQBytes + c * (BR * 128), &tm_q, full, c * 64,
                                        tok0 + i * BR, z_q);
                            tma_load_3d(sDO + st * Cfg::kQBytes + c * (BR * 128), &tm_do, full, c * 64,
                                        tok0 + i * BR, z_q);
                        }
                        const size_t xrow = (size_t)bh * p.Np + (size_t)i * BR;
                        bulk_load(sExt + (2 * st) * Cfg::kExtBytes, p.lse_ext + xrow * kExtCols,
                                  Cfg::kExtBytes, full);
                        bulk_load(sExt + (2 * st + 1) * Cfg::kExtBytes, p.d_ext + xrow * kExtCols,
                                  Cfg::kExtBytes, full);
                        issued = git + 1;
                    }
                    gi += n_it;
                    ++nb;
                }
                if (abort_sh) {   // drain the copies still in flight (bounded)
                    const WaitCtx dc{p.status, nullptr};
                    if (kv_issued > 0) fa_wait(&bar_kv, (kv_issued - 1) & 1, 41, dc);
                    for (int x = max(0, issued - NS); x < issued; ++x)
                        fa_wait(&bar_full[x % (2 * NS)], (x / (2 * NS)) & 1, 41, dc);
                }
            }
            __syncwarp();
        } else if (warp == kMmaWarp || warp == kMma2Warp) {
            if (lane == 0) {
                // MMA issue for pipeline pp: per step S^T, dP^T (once the
                // read-out has taken the pipeline's previous dQ^T), dV (once P^T
                // is in TMEM), dK and dQ^T (once dS^T is in SMEM).
                const int pp = (warp == kMmaWarp) ? 0 : 1;
                constexpr uint32_t id_s = idesc_bf16_f32(128, BR, false, false);
                constexpr uint32_t id_kv = idesc_bf16_f32(128, D, false, true);
                constexpr uint32_t id_dq = idesc_bf16_f32(128, 64, true, true);
                const uint32_t sk = smem_u32(sK), sv = smem_u32(sV), sq = smem_u32(sQ),
                               sdo = smem_u32(sDO), sds = smem_u32(sDS) + pp * Cfg::kDSBytes;
                const uint64_t kd = sdesc_sw128(sk, 16, 1024), vd = sdesc_sw128(sv, 16, 1024);
                const uint64_t dsd = sdesc_sw128(sds, 16, 1024);
                const uint64_t kd_mn = sdesc_sw128(sk, kBN * 128, 1024);
                const uint64_t dsd_mn = sdesc_sw128(sds, kBN * 128, 1024);
                const uint32_t sext = smem_u32(sExt);
                const uint64_t onesd = sdesc_plain(smem_u32(sOnes), 128, 256);
                const uint32_t col_s = Cfg::col_s(pp), col_dpq = Cfg::col_dpq(pp);
                bool ok = true;
                int gi = 0, nb = 0;
                for (int n = 0; ok; ++n) {
                    int item;
                    if (!next_item_thread(n, item)) { ok = false; break; }
                    if (item < 0) break;
                    const BwdCta cta = bwd_cta<CAUSAL, WINDOW, VARLEN>(p, BR, item);
                    if (cta.idle || cta.n_it == 0) continue;
                    const int n_it = cta.n_it;
                    // Every per-item phase is waited on by both issuers, whether
                    // or not the item has steps of their parity: K_j, V_j landed
                    // and dK, dV zeroed (a waiter never falls two phases behind).
                    ok = fa_wait(&bar_kv, nb & 1, 50, wc) && fa_wait(&bar_acc_free, nb & 1, 58, wc);
                    for (int it = (gi & 1) == pp ? 0 : 1; ok && it < n_it; it += 2) {
                        const int git = gi + it;
                        const uint32_t k = (uint32_t)git >> 1;
                        const int st = git % NS;
                        if (!fa_wait(&bar_full[git % (2 * NS)], (git / (2 * NS)) & 1, 51, wc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t q_ = sq + st * Cfg::kQBytes, do_ = sdo + st * Cfg::kQBytes;
                        // S^T = K_j Q_i^T - LSE log2(e) / c
                        {
                            const uint64_t qd = sdesc_sw128(q_, 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tmem + col_s, kd + kmajor_step(kk, kBN * 128),
                                       qd + kmajor_step(kk, BR * 128), id_s, kk > 0);
                            mma_ss(tmem + col_s, onesd,
                                   sdesc_plain(sext + 2 * st * Cfg::kExtBytes, 128, 256), id_s, 1u);
                            mma_commit(&bar_s[pp]);
                        }
                        // dP^T - D = V_j dO_i^T - D, over the previous dQ^T
                        if (k > 0 && !fa_wait(&bar_dq_free[pp], (k - 1) & 1, 53, wc)) { ok = false; break; }
                        tc_fence_after();
                        {
                            const uint64_t dod = sdesc_sw128(do_, 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tmem + col_dpq, vd + kmajor_step(kk, kBN * 128),
                                       dod + kmajor_step(kk, BR * 128), id_s, kk > 0);
                            mma_ss(tmem + col_dpq, onesd,
                                   sdesc_plain(sext + (2 * st + 1) * Cfg::kExtBytes, 128, 256), id_s,
                                   1u);
                            mma_commit(&bar_dp[pp]);
                        }
                        // dV += P^T dO_i (P^T: bf16 pairs in the first 32 S^T columns),
                        // after step git - 1's dV MMAs
                        if (!fa_wait(&bar_p[pp], k & 1, 52, wc) ||
                            (git > 0 && !fa_wait(&bar_dv_turn, (git - 1) & 1, 46, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        {
                            const uint64_t dod_mn = sdesc_sw128(do_, BR * 128, 1024);
#pragma unroll
                            for (int kk = 0; kk < BR / 16; ++kk)
                                mma_ts(tmem + Cfg::kColDV, tmem + col_s + kk * 8,
                                       dod_mn + mnmajor_step(kk), id_kv, 1u);
                        }
                        tc_fence_before();   // the MMAs above precede the turn's arrival
                        mbar_arrive(&bar_dv_turn);
                        // dK += dS^T Q_i, after step git - 1's dK MMAs
                        if (!fa_wait(&bar_ds[pp], k & 1, 55, wc) ||
                            (git > 0 && !fa_wait(&bar_dk_turn, (git - 1) & 1, 47, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        {
                            const uint64_t qd_mn = sdesc_sw128(q_, BR * 128, 1024);
#pragma unroll
                            for (int kk = 0; kk < BR / 16; ++kk)
                                mma_ss(tmem + Cfg::kColDK, dsd + kmajor_step(kk, kBN * 128),
                                       qd_mn + mnmajor_step(kk), id_kv, 1u);
                        }
                        tc_fence_before();   // the MMAs above precede the turn's arrival
                        mbar_arrive(&bar_dk_turn);
                        mma_commit(&bar_empty[st]);      // Q_i, dO_i no longer read
                        // dQ^T partial = K_j^T dS^T (K dimension = the 128 keys),
                        // over dP^T, which the compute warps have read
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            mma_ss(tmem + col_dpq, kd_mn + mnmajor_step(kk), dsd_mn + mnmajor_step(kk),
                                   id_dq, kk > 0);
                        mma_commit(&bar_dq_full[pp]);
                    }
                    if (ok) {   // every MMA of the item from this thread (possibly none)
                        mma_commit(&bar_done);
                        mma_commit(&bar_kv_free);
                    }
                    gi += n_it;
                    ++nb;
                }
                if (!ok) {   // no MMA of this thread may still write TMEM at teardown
                    __shared__ uint64_t bar_drain2[2];
                    mbar_init(&bar_drain2[pp], 1);
                    fence_mbar_init();
                    mma_commit(&bar_drain2[pp]);
                    fa_wait(&bar_drain2[pp], 0, 59, WaitCtx{p.status, nullptr});
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

template <bool CAUSAL, bool WINDOW = false, bool VARLEN = false>
cudaError_t launch_dkdv2_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const BwdParams& p, int grid,
                           cudaStream_t stream) {
    auto kern = fa_bwd_dkdv2_kernel<CAUSAL, WINDOW, VARLEN>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        if (attr.numRegs * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Bwd2Cfg::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<grid, kThreads, Bwd2Cfg::kSmemAlloc, stream>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const Shape& s, const void* o, bool o_f32, const void* dout,
                                  const float* lse, const BwdWorkspace& ws, DeviceStatus* status,
                                  cudaStream_t stream, bool full) {
    (void)status;
    const int Np = padded_rows(s.N);
    const long long rows = (long long)s.B * s.H * Np;
    const long long seq_rows = s.cu_seqlens ? s.total : s.N;
    const int grid = grid_for(rows, 8 * (256 / s.d));   // 8 warps a block, 256/d rows a warp
    count_launch();
    auto* d_ = static_cast<const __nv_bfloat16*>(dout);
    auto go = [&](auto kern, auto* o_) {
        kern<<<grid, 256, 0, stream>>>(o_, d_, lse, ws.lse_ext, ws.d_ext, ws.dq_acc, ws.work, s.N,
                                       Np, rows, s.cu_seqlens, s.H, seq_rows);
        return cudaGetLastError();
    };
    auto* ob = static_cast<const __nv_bfloat16*>(o);
    auto* of = static_cast<const float*>(o);
    if (s.d == 128) {
        if (o_f32)
            return full ? go(fa_bwd_pre_kernel<128, float, true>, of)
                        : go(fa_bwd_pre_kernel<128, float, false>, of);
        return full ? go(fa_bwd_pre_kernel<128, __nv_bfloat16, true>, ob)
                    : go(fa_bwd_pre_kernel<128, __nv_bfloat16, false>, ob);
    }
    if (o_f32)
        return full ? go(fa_bwd_pre_kernel<64, float, true>, of)
                    : go(fa_bwd_pre_kernel<64, float, false>, of);
    return full ? go(fa_bwd_pre_kernel<64, __nv_bfloat16, true>, ob)
                : go(fa_bwd_pre_kernel<64, __nv_bfloat16, false>, ob);
}

cudaError_t launch_bwd_dkdv(const Shape& s, const void* q, const void* k, const void* v,
                            const void* dout, void* dk, void* dv, const BwdWorkspace& ws,
                            DeviceStatus* status, cudaStream_t stream) {
    const int br = (s.d == 128) ? BwdCfg<128>::kBR : BwdCfg<64>::kBR;
    const bool varlen = s.cu_seqlens != nullptr;
    const int rows = varlen ? s.total : s.N;
    const int zq = varlen ? s.H : s.B * s.H, zkv = varlen ? s.Hkv : s.B * s.Hkv;
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!make_tmap_bf16_3d(&tq, q, s.d, rows, zq, br) ||
        !make_tmap_bf16_3d(&tdo, dout, s.d, rows, zq, br) ||
        !make_tmap_bf16_3d(&tk, k, s.d, rows, zkv, kBN) ||
        !make_tmap_bf16_3d(&tv, v, s.d, rows, zkv, kBN) ||
        !make_tmap_f32_2d(&tdq, ws.dq_acc, s.d, (long long)s.B * s.H * padded_rows(s.N), 32, br))
        return cudaErrorInvalidValue;
    BwdParams p;
    p.H = s.H;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.Np = padded_rows(s.N);
    p.rows = rows;
    p.cu_seqlens = s.cu_seqlens;
    p.G = s.H / s.Hkv;
    // Chunk size: what fits a 64 MB L2 budget of Q, dO (bf16) and dQ
    // accumulator (fp32) rows, 8 G N d bytes per key/value head, but at least
    // a quarter of the heads: with many small chunks the heavy CTAs of the last
    // one start late and the balance is lost (CPU model: gqa 0.88 of the mean
    // load at 3 heads a chunk, 0.98 at 8).
    {
        const long long n_bg = (long long)s.B * s.Hkv;
        const long long per = 8LL * p.G * s.N * s.d;
        long long c = (64LL << 20) / (per > 0 ? per : 1);
        c = c > (n_bg + 3) / 4 ? c : (n_bg + 3) / 4;
        // A window bounds every key block's query range, so the working set
        // of all heads at once is small: one chunk (measured 1 % faster).
        if (s.window > 0) c = n_bg;
        p.chunk = (int)(c < 1 ? 1 : (c > n_bg ? n_bg : c));
    }
    p.causal = s.causal;
    p.window = s.window > 0 ? s.window : kNoWindow;
    p.scale = s.scale;
    p.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
    p.lse_ext = ws.lse_ext;
    p.d_ext = ws.d_ext;
    p.dq_acc = ws.dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.status = status;
    p.work = ws.work;
    const int n_kblk = (s.N + kBN - 1) / kBN;
    p.n_bg = s.B * s.Hkv;
    p.n_items = n_kblk * s.B * s.Hkv;
    // Persistent: one CTA per SM (fewer when there are fewer work items),
    // taking items in the order above from the work counter.
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    const int grid = p.n_items < sms ? p.n_items : sms;
    count_launch();
    if (varlen) {   // packed variable-length sequences (no window)
        if (s.window > 0) return cudaErrorInvalidValue;
        if (s.d == 128)
            return s.causal ? launch_dkdv2_t<true, false, true>(tq, tk, tv, tdo, p, grid, stream)
                            : launch_dkdv2_t<false, false, true>(tq, tk, tv, tdo, p, grid, stream);
        return s.causal
                   ? launch_dkdv_t<64, true, false, true>(tq, tk, tv, tdo, tdq, p, grid, stream)
                   : launch_dkdv_t<64, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, stream);
    }
    if (s.window > 0) {   // the causal sliding window
        if (!s.causal) return cudaErrorInvalidValue;
        return s.d == 128 ? launch_dkdv_t<128, true, true>(tq, tk, tv, tdo, tdq, p, grid, stream)
                          : launch_dkdv_t<64, true, true>(tq, tk, tv, tdo, tdq, p, grid, stream);
    }
    if (s.d == 128)
        return s.causal ? launch_dkdv2_t<true>(tq, tk, tv, tdo, p, grid, stream)
                        : launch_dkdv2_t<false>(tq, tk, tv, tdo, p, grid, stream);
    return s.causal ? launch_dkdv_t<64, true>(tq, tk, tv, tdo, tdq, p, grid, stream)
                    : launch_dkdv_t<64, false>(tq, tk, tv, tdo, tdq, p, grid, stream);
}

cudaError_t launch_bwd_dq_convert(const Shape& s, const BwdWorkspace& ws, void* dq,
                                  cudaStream_t stream) {
    auto* dq_ = static_cast<__nv_bfloat16*>(dq);
    if (s.cu_seqlens) {
        const int Np = padded_rows(s.N);
        const long long nv = (long long)s.B * s.H * Np * s.d / 8;
        const int g = grid_for(nv, 256);
        count_launch();
        if (s.d == 128)
            fa_bwd_dq_convert_varlen_kernel<128><<<g, 256, 0, stream>>>(
                ws.dq_acc, dq_, s.cu_seqlens, s.H, s.N, Np, s.total, s.scale, nv);
        else
            fa_bwd_dq_convert_varlen_kernel<64><<<g, 256, 0, stream>>>(
                ws.dq_acc, dq_, s.cu_seqlens, s.H, s.N, Np, s.total, s.scale, nv);
        return cudaGetLastError();
    }
    const long long n_vec = (long long)s.B * s.H * s.N * s.d / 8;
    const int grid = grid_for(n_vec, 256);
    count_launch();
    if (s.d == 128)
        fa_bwd_dq_convert_kernel<128><<<grid, 256, 0, stream>>>(ws.dq_acc, dq_, s.N,
                                                                padded_rows(s.N), s.scale, n_vec);
    else
        fa_bwd_dq_convert_kernel<64><<<grid, 256, 0, stream>>>(ws.dq_acc, dq_, s.N,
                                                               padded_rows(s.N), s.scale, n_vec);
    return cudaGetLastError();
}

cudaError_t launch_exp2_check(const float* x, float* y_fma, float* y_ex2, int n,
                              cudaStream_t stream) {
    count_launch();
    const int pairs = (n + 1) / 2;
    fa_exp2_check_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y_fma, y_ex2, n);
    return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(long long timeout_ns, DeviceStatus* status,
                                     cudaStream_t stream) {
    count_launch();
    fa_watchdog_kernel<<<1, 32, 0, stream>>>(status, (unsigned long long)timeout_ns);
    return cudaGetLastError();
}

}  // namespace fa
