// Split-KV decoding forward: a few new query rows (Nq) against a long key /
// value sequence (Nk), the decoding setting of the FlashAttention blog
// ("Flash-Decoding": split the keys, compute partial softmax results in
// parallel, combine them with their log-sum-exp) and of the FA2 review thread.
//
// The queries are the last Nq positions: under the causal mask query row r
// sees key j iff j <= r + Nk - Nq (bottom-right alignment; the forward's
// j <= i when Nq == Nk).
//
// Every key and value row is read once and used for only R = G * Nq query
// rows (G = H / Hkv), so the work is bandwidth-bound; the arithmetic still
// goes to the tensor core, which leaves the CUDA cores only the softmax:
//   split kernel   one CTA (three warps) per (batch, kv head, key split).  The
//                  R query rows of the group sit in the first rows of a
//                  128-row Q tile (the rest zero) and the split's keys stream
//                  through a TMA ring in tiles of 128:
//                    S_t = Q K_t^T   (SS MMA, M = N = 128, two TMEM buffers)
//                    O  += P_t V_t   (TS MMA, P over the first half of S_t)
//                  so the tensor core does 128 / R times the useful work and
//                  still idles most of the time (a 64 KB tile takes about
//                  3000 cycles of one SM's share of HBM bandwidth, its MMAs
//                  about 700).  Warp 0 holds rows 0-31 of S and runs the
//                  online softmax (base 2, conditional rescale of O in TMEM)
//                  for the rows below R; warp 1 loads; warp 2 issues the
//                  MMAs (S one tile ahead of P V).  The split writes o / l
//                  (fp32) and its LSE.
//   combine kernel one warp per output row: LSE = log sum_s exp(LSE_s),
//                  O = sum_s exp(LSE_s - LSE) O_s, bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kTileKeys = 128;        // keys per tile (the MMA's N)
constexpr int kThreads = 96;          // softmax warp, producer warp, MMA warp
constexpr int kQRows = 16;            // query rows loaded (R <= 16), rest of the tile zero
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kRescale = 8.0f;      // log2 units, as in the forward

struct DecodeParams {
    float* o_part;            // [B][H][Nq][n_split][d]
    float* lse_part;          // [B][H][Nq][n_split], natural log
    int H, Hkv, Nq, Nk, G, R, n_split, keys_per_split, causal;
    int n_items;              // B * Hkv * n_split work items (batch, kv head, key split)
    float scale_log2;
    DeviceStatus* status;
};

// d = 128: a K/V ring of 3 stages of 64 KB (K and V tiles) and two S buffers
// in TMEM (512 columns with O): one CTA fills an SM.  d = 64: 2 stages of
// 32 KB and one S buffer (256 columns), so that two CTAs share an SM and
// each one's MMA and softmax chain hides behind the other's loads.
template <int D>
__host__ __device__ constexpr int decode_stages() { return D == 128 ? 3 : 2; }
template <int D>
__host__ __device__ constexpr int decode_ctas_per_sm() { return D == 128 ? 1 : 2; }
template <int D>
__host__ __device__ constexpr int decode_tile_bytes() { return kTileKeys * D * 2; }
// d = 64: persistent CTAs (two an SM) that take work items c, c + grid, ...
// and stream the next item's tiles through the same rings without draining
// them, with two Q tiles (the next item's Q loads while the current one is
// used); d = 128: one item per CTA.
template <int D>
__host__ __device__ constexpr bool decode_persistent() { return D == 64; }
template <int D>
__host__ __device__ constexpr int decode_q_bufs() { return decode_persistent<D>() ? 2 : 1; }
template <int D>
__host__ __device__ constexpr int decode_smem_bytes() {
    return decode_q_bufs<D>() * 128 * D * 2 + decode_stages<D>() * 2 * decode_tile_bytes<D>() +
           1024;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    constexpr int S = decode_stages<D>();
    constexpr int TB = decode_tile_bytes<D>();
    constexpr int kChunkBytes = 128 * 128;        // 64 columns x 128 rows, one SW128 chunk
    constexpr bool kTwoS = (D == 128);            // two S buffers (else S_t+1 after P_t V)
    constexpr uint32_t kColS0 = 0, kColS1 = kTwoS ? 128 : 0, kColO = kTwoS ? 256 : 128;
    constexpr uint32_t kTmemCols = kTwoS ? 512 : 256;
    constexpr int QB = decode_q_bufs<D>();
    constexpr int kQBytes = 128 * D * 2;
    extern __shared__ uint8_t dsm_raw[];
    uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = dsm;                            // [QB] x 128 x D, rows >= kQRows zero
    uint8_t* sK = dsm + QB * kQBytes;             // [S] tiles
    uint8_t* sV = sK + S * TB;                    // [S] tiles
    __shared__ uint64_t bar_q[QB], bar_q_free[QB], bar_k[S], bar_k_empty[S], bar_v[S],
        bar_v_empty[S];
    // the softmax warp has read an item's O: the next item's first P V may
    // overwrite it
    __shared__ uint64_t bar_o_free;
    // S_t, P_t and P_t V_t signal barrier t & 1 (completion k of barrier b
    // is tile b + 2k; t counts the CTA's tiles over all its work items): a
    // waiter for tile t never finds tile t + 2 complete
    __shared__ uint64_t bar_s[2], bar_p[2], bar_pv[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    const WaitCtx wc{p.status, &abort_sh};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Work item -> (kv group bg = b * Hkv + g, key split, its keys and tiles).
    struct Item { int split, bg, b, g, j_begin, j_end, n_tiles; };
    auto item_at = [&](int item) {
        Item it;
        it.split = item % p.n_split;
        it.bg = item / p.n_split;
        it.b = it.bg / p.Hkv;
        it.g = it.bg % p.Hkv;
        it.j_begin = it.split * p.keys_per_split;
        it.j_end = min(p.Nk, it.j_begin + p.keys_per_split);
        it.n_tiles = (it.j_end - it.j_begin + kTileKeys - 1) / kTileKeys;   // >= 1 by the plan
        return it;
    };

    // The Q tiles' rows past the loaded ones are MMA rows whose results nobody
    // reads; they are zeroed so that they hold plain numbers.
    for (int e = threadIdx.x; e < QB * kQBytes / 16; e += kThreads)
        reinterpret_cast<uint4*>(sQ)[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int qb = 0; qb < QB; ++qb) {
            mbar_init(&bar_q[qb], 1);
            mbar_init(&bar_q_free[qb], 1);
        }
        mbar_init(&bar_o_free, 32);
        for (int s = 0; s < S; ++s) {
            mbar_init(&bar_k[s], 1);
            mbar_init(&bar_k_empty[s], 1);
            mbar_init(&bar_v[s], 1);
            mbar_init(&bar_v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar_s[t], 1);
            mbar_init(&bar_p[t], 32);
            mbar_init(&bar_pv[t], 1);
        }
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 1) {
        // -------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int gt = 0, q_issued = 0;   // tiles and Q tiles loaded so far
            bool ok = true;
            for (int item = blockIdx.x, n = 0; ok && item < p.n_items; item += gridDim.x, ++n) {
                const Item it = item_at(item);
                const int qb = n % QB;
                // the Q tile of item n - QB has been read by its last S MMA
                if (n >= QB && !fa_wait(&bar_q_free[qb], ((n / QB) - 1) & 1, 79, wc)) break;
                mbar_arrive_expect_tx(&bar_q[qb], kQRows * 128 * (D / 64));
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sQ + qb * kQBytes + c * kChunkBytes, &tm_q, &bar_q[qb], c * 64,
                                it.bg * p.R, 0);
                ++q_issued;
                for (int t = 0; t < it.n_tiles; ++t, ++gt) {
                    const int s = gt % S;
                    const int j0 = it.j_begin + t * kTileKeys;
                    if (gt >= S && !fa_wait(&bar_k_empty[s], ((gt / S) - 1) & 1, 80, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_k[s], TB);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(sK + s * TB + c * kChunkBytes, &tm_k, &bar_k[s], c * 64, j0,
                                    it.bg);
                    if (gt >= S && !fa_wait(&bar_v_empty[s], ((gt / S) - 1) & 1, 81, wc)) {
                        // K of this tile is in flight: count it for the drain
                        fa_wait(&bar_k[s], (gt / S) & 1, 82, WaitCtx{p.status, nullptr});
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_v[s], TB);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(sV + s * TB + c * kChunkBytes, &tm_v, &bar_v[s], c * 64, j0,
                                    it.bg);
                }
            }
            if (abort_sh) {   // drain the copies still in flight (bounded)
                const WaitCtx dc{p.status, nullptr};
                for (int x = max(0, q_issued - QB); x < q_issued; ++x)
                    fa_wait(&bar_q[x % QB], (x / QB) & 1, 82, dc);
                for (int t = max(0, gt - S); t < gt; ++t) {
                    fa_wait(&bar_k[t % S], (t / S) & 1, 82, dc);
                    fa_wait(&bar_v[t % S], (t / S) & 1, 82, dc);
                }
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTileKeys, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
            const uint32_t sq = smem_u32(sQ), sk = smem_u32(sK), sv = smem_u32(sV);
            bool ok = true;
            int gt = 0;   // tiles of this CTA so far (all items)
            int n = 0;    // current item's rank among this CTA's items
            // O += P_u V_u for tile u; first = the item's first tile, whose
            // P V overwrites O once the previous item's O has been read out.
            auto pv = [&](int u, bool first) -> bool {
                const int s = u % S;
                if (!fa_wait(&bar_p[u & 1], (u >> 1) & 1, 84, wc) ||
                    !fa_wait(&bar_v[s], (u / S) & 1, 85, wc))
                    return false;
                if (first && n > 0 && !fa_wait(&bar_o_free, (n - 1) & 1, 78, wc)) return false;
                tc_fence_after();
                const uint32_t col_p = (u & 1) ? kColS1 : kColS0;
                const uint64_t vd = sdesc_sw128(sv + s * TB, kChunkBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk)
                    mma_ts(tmem + kColO, tmem + col_p + kk * 8, vd + mnmajor_step(kk), idesc_o,
                           (!first || kk > 0) ? 1u : 0u);
                mma_commit(&bar_pv[u & 1]);
                mma_commit(&bar_v_empty[s]);
                return true;
            };
            for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++n) {
                const Item it = item_at(item);
                const int qb = n % QB;
                if (!fa_wait(&bar_q[qb], (n / QB) & 1, 83, wc)) { ok = false; break; }
                tc_fence_after();
                const uint64_t qd = sdesc_sw128(sq + qb * kQBytes, 16, 1024);
                for (int t = 0; ok && t < it.n_tiles; ++t) {
                    const int g_t = gt + t;
                    const int s = g_t % S;
                    if (!fa_wait(&bar_k[s], (g_t / S) & 1, 86, wc)) { ok = false; break; }
                    tc_fence_after();
                    // S_t over P_{t-2} (P_{t-1} with one buffer): in issue order
                    // after the P V MMA that read it
                    const uint32_t col_s = (g_t & 1) ? kColS1 : kColS0;
                    const uint64_t kd = sdesc_sw128(sk + s * TB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + col_s, qd + kmajor_step(kk, kChunkBytes),
                               kd + kmajor_step(kk, kChunkBytes), idesc_s, kk > 0);
                    mma_commit(&bar_s[g_t & 1]);
                    mma_commit(&bar_k_empty[s]);
                    if (t + 1 == it.n_tiles) mma_commit(&bar_q_free[qb]);   // Q tile read
                    if (kTwoS) {
                        if (t > 0 && !pv(g_t - 1, t == 1)) { ok = false; break; }
                    } else if (!pv(g_t, t == 0)) {   // one S buffer: P V before S_t+1
                        ok = false;
                        break;
                    }
                }
                if (kTwoS && ok) ok = pv(gt + it.n_tiles - 1, it.n_tiles == 1);
                gt += it.n_tiles;
            }
            if (!ok) {   // no MMA of this thread may still write TMEM at teardown
                __shared__ uint64_t bar_drain;
                mbar_init(&bar_drain, 1);
                fence_mbar_init();
                mma_commit(&bar_drain);
                fa_wait(&bar_drain, 0, 87, WaitCtx{p.status, nullptr});
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax (rows = lanes)
        const int r = lane;                       // query row of the group
        const bool row_ok = r < p.R;
        const int last_vis = p.causal ? (r % p.Nq) + (p.Nk - p.Nq) : p.Nk - 1;
        const float c = p.scale_log2;
        bool ok = true;
        int gt = 0;   // tiles of this CTA so far (all items)
        for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
            const Item it = item_at(item);
            const int b = it.b, g = it.g, split = it.split;
            const int j_begin = it.j_begin, j_end = it.j_end, n_tiles = it.n_tiles;
            float m2 = -CUDART_INF_F, l = 0.0f;
            for (int t = 0; t < n_tiles; ++t) {
                const int g_t = gt + t;
                if (!fa_wait_warp(&bar_s[g_t & 1], (g_t >> 1) & 1, 88, wc)) { ok = false; break; }
                tc_fence_after();
                const uint32_t col_s = (g_t & 1) ? kColS1 : kColS0;
                uint32_t sr[4][32];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tmem + col_s + q4 * 32, sr[q4]);
                tmem_ld_wait(sr[0]);
#pragma unroll
                for (int q4 = 1; q4 < 4; ++q4) asm volatile("" : FA_R32(sr[q4]) : : "memory");
                // visible keys of the tile for this row: j0 + e <= lim
                const int j0 = j_begin + t * kTileKeys;
                const int lim = min(last_vis, j_end - 1) - j0;   // keep e <= lim
                float x[kTileKeys];
#pragma unroll
                for (int e = 0; e < kTileKeys; ++e) x[e] = __uint_as_float(sr[e >> 5][e & 31]);
                if (lim < kTileKeys - 1) {
#pragma unroll
                    for (int e = 0; e < kTileKeys; ++e)
                        if (e > lim) x[e] = -CUDART_INF_F;
                }
                // Row max of the raw scores in eight independent chains of
                // three-input maxima, then scaled (c > 0): a short dependency
                // chain where a single running max would be 128 deep.
                float mx8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(x[2 * u], x[2 * u + 1]);
#pragma unroll
                for (int e = 16; e < kTileKeys; e += 16)
#pragma unroll
                    for (int u = 0; u < 8; ++u) mx8[u] = fmax3(mx8[u], x[e + 2 * u], x[e + 2 * u + 1]);
                const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                       fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7])) * c;
                const bool need = row_ok && mx > m2 + kRescale;
                float alpha = 1.0f;
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = need ? mx : m2;
                    alpha = (m_new == m2) ? 1.0f : ex2(m2 - m_new);
                    m2 = m_new;
                    // O holds P V of the earlier tiles: rescale it once the last
                    // of those P V MMAs (and so every earlier one) has completed
                    if (t > 0) {
                        if (!fa_wait_warp(&bar_pv[(g_t - 1) & 1], ((g_t - 1) >> 1) & 1, 89, wc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t ov[32];
                            tmem_ld32(tmem + kColO + c0, ov);
                            tmem_ld_wait(ov);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            tmem_st32(tmem + kColO + c0, ov);
                        }
                    }
                    l *= alpha;
                }
                const float m_use = (m2 == -CUDART_INF_F) ? 0.0f : m2;
                // p = 2^(s c - m): the exponent argument two lanes per paired
                // FMA, the row sum in four paired accumulators.
                const uint64_t c2 = f2(c, c), negm2 = f2(-m_use, -m_use);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pk[2][32];
#pragma unroll
                for (int e2 = 0; e2 < kTileKeys / 2; ++e2) {
                    float a0, a1;
                    f2_split(f2_fma(f2(x[2 * e2], x[2 * e2 + 1]), c2, negm2), a0, a1);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    acc2[e2 & 3] = f2_add(acc2[e2 & 3], f2(p0, p1));
                    pk[e2 >> 5][e2 & 31] = pack_bf16x2(p0, p1);
                }
                {
                    float a0, a1;
                    f2_split(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), a0, a1);
                    l += a0 + a1;
                }
                tmem_st32(tmem + col_s, pk[0]);
                tmem_st32(tmem + col_s + 32, pk[1]);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_p[g_t & 1]);
            }
            const int g_last = gt + n_tiles - 1;
            gt += n_tiles;
            if (!ok) break;
            if (!fa_wait_warp(&bar_pv[g_last & 1], (g_last >> 1) & 1, 90, wc)) break;
            {
                tc_fence_after();
                // split outputs: O_s = o / l, LSE_s = ln2 (m + log2 l); zeros and
                // -inf when no key of the split is visible to the row
                const int hl = r / max(p.Nq, 1), qi = r % max(p.Nq, 1);
                const size_t row = ((size_t)b * p.H + g * p.G + hl) * p.Nq + qi;
                const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
                // O into registers, then released to the next item's first P V
                uint32_t ov[D / 32][32];
#pragma unroll
                for (int c0 = 0; c0 < D / 32; ++c0) tmem_ld32(tmem + kColO + c0 * 32, ov[c0]);
                tmem_ld_wait(ov[0]);
#pragma unroll
                for (int c0 = 1; c0 < D / 32; ++c0) asm volatile("" : FA_R32(ov[c0]) : : "memory");
                tc_fence_before();
                mbar_arrive(&bar_o_free);
                if (row_ok) {
#pragma unroll
                    for (int c0 = 0; c0 < D / 32; ++c0) {
                        float4* dst = reinterpret_cast<float4*>(
                            p.o_part + (row * p.n_split + split) * D + c0 * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(ov[c0][4 * q4]) * inv,
                                                  __uint_as_float(ov[c0][4 * q4 + 1]) * inv,
                                                  __uint_as_float(ov[c0][4 * q4 + 2]) * inv,
                                                  __uint_as_float(ov[c0][4 * q4 + 3]) * inv);
                    }
                    p.lse_part[row * p.n_split + split] =
                        (l > 0.0f) ? (m2 + log2f(l)) * kLn2 : -CUDART_INF_F;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One warp per output row: combine the splits by their log-sum-exp.
template <int D>
__global__ void __launch_bounds__(256)
fa_decode_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse, long long rows,
                         int n_split) {
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* lp = lse_part + row * n_split;
    const float* os = o_part + row * n_split * D + lane;
    // The partial O of the first kPre splits is loaded together with the
    // LSEs (one memory round trip when n_split <= kPre, the usual case);
    // rows past n_split read as zero and get weight zero.
    constexpr int kPre = 8;
    float pre[kPre][D / 32];
#pragma unroll
    for (int k = 0; k < kPre; ++k)
#pragma unroll
        for (int c = 0; c < D / 32; ++c) pre[k][c] = (k < n_split) ? os[k * D + 32 * c] : 0.0f;
    const float l0 = lane < n_split ? lp[lane] : -CUDART_INF_F;
    float mx = l0;
    for (int s = lane + 32; s < n_split; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float acc[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = 0.0f;
    float wsum = 0.0f;
    if (mx != -CUDART_INF_F) {
        // 32 splits at a time: lane k computes the weight of split base + k
        // (0 for a split that saw no key: its partial O is zero), then every
        // lane adds its columns of each split's partial O, the loads of
        // different splits independent of one another.
        for (int base = 0; base < n_split; base += 32) {
            const int sl = base + lane;
            const float ls = (base == 0) ? l0 : (sl < n_split ? lp[sl] : -CUDART_INF_F);
            const float w = (ls == -CUDART_INF_F) ? 0.0f : expf(ls - mx);
            wsum += w;
            const int cnt = min(32, n_split - base);
            int k = 0;
            if (base == 0) {
#pragma unroll
                for (int kp = 0; kp < kPre; ++kp) {
                    const float wk = __shfl_sync(0xffffffffu, w, kp);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(wk, pre[kp][c], acc[c]);
                }
                k = kPre;
            }
#pragma unroll 4
            for (; k < cnt; ++k) {
                const float wk = __shfl_sync(0xffffffffu, w, k);
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
                    acc[c] = fmaf(wk, os[(base + k) * D + 32 * c], acc[c]);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    }
    const float inv = (wsum > 0.0f) ? 1.0f / wsum : 0.0f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) o[row * D + lane + 32 * c] = __float2bfloat16_rn(acc[c] * inv);
    if (lane == 0) lse[row] = (wsum > 0.0f) ? mx + logf(wsum) : -CUDART_INF_F;
}

}  // namespace

// Split policy: the number of CTAs, B * Hkv * n_split, is chosen for the
// fullest waves of 152 x (CTAs per SM: 1 at d = 128, 2 at d = 64) among
// n_split in [ceil(slots / (B Hkv)), 4 ceil(slots / (B Hkv))], each split a
// whole number of 128-key tiles.  The target is fixed, so the workspace size
// does not depend on the device.
void decode_split_plan(int B, int Hkv, int Nk, int d, int* n_split, int* keys_per_split) {
    const int kSms = 152 * (d == 128 ? decode_ctas_per_sm<128>() : decode_ctas_per_sm<64>());
    const int tiles = (Nk + kTileKeys - 1) / kTileKeys;
    const long long groups = (long long)B * Hkv;
    int lo = (int)((kSms + groups - 1) / groups);
    if (lo > tiles) lo = tiles;
    if (lo < 1) lo = 1;
    int hi = 4 * lo < tiles ? 4 * lo : tiles;
    int best = lo;
    double best_eff = -1.0;
    for (int n = lo; n <= hi; ++n) {
        const int tiles_per = (tiles + n - 1) / n;
        const int n_eff = (tiles + tiles_per - 1) / tiles_per;      // splits actually used
        const long long ctas = groups * n_eff;
        const long long waves = (ctas + kSms - 1) / kSms;
        const double eff = (double)ctas / (double)(waves * kSms);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = n;
        }
    }
    const int tiles_per = (tiles + best - 1) / best;
    *keys_per_split = tiles_per * kTileKeys;
    *n_split = (Nk + *keys_per_split - 1) / *keys_per_split;
}

size_t decode_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d) {
    int ns, kps;
    decode_split_plan(B, Hkv, Nk, d, &ns, &kps);
    const size_t rows = (size_t)B * H * Nq;
    const size_t o_bytes = (rows * ns * d * 4 + 255) / 256 * 256;
    return o_bytes + rows * ns * 4;
}

template <int D>
static cudaError_t launch_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const DecodeParams& p, long long blocks, cudaStream_t stream) {
    auto kern = fa_decode_split_kernel<D>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             decode_smem_bytes<D>());
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<(unsigned)blocks, kThreads, decode_smem_bytes<D>(), stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, int B, int H, int Hkv, int Nq, int Nk, int d,
                              int causal, float scale, DeviceStatus* status,
                              cudaStream_t stream) {
    DecodeParams p;
    int ns, kps;
    decode_split_plan(B, Hkv, Nk, d, &ns, &kps);
    const size_t rows = (size_t)B * H * Nq;
    // q as one column of rows: the group (b, g) is rows (b Hkv + g) R ...
    // (heads of a group are adjacent); 16 rows are loaded, rows past R are
    // never read back.  K and V: {d, Nk, B Hkv}, 128-key tiles.
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_3d(&tq, q, d, (int)rows, 1, kQRows) ||
        !make_tmap_bf16_3d(&tk, k, d, Nk, B * Hkv, kTileKeys) ||
        !make_tmap_bf16_3d(&tv, v, d, Nk, B * Hkv, kTileKeys))
        return cudaErrorInvalidValue;
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          (rows * ns * d * 4 + 255) / 256 * 256);
    p.H = H;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nk = Nk;
    p.G = H / Hkv;
    p.R = p.G * Nq;
    p.n_split = ns;
    p.keys_per_split = kps;
    p.causal = causal;
    p.scale_log2 = scale * kLog2e;
    p.status = status;
    const long long items = (long long)B * Hkv * ns;
    if (items > 0x7fffffffLL || rows * 32 / 256 + 1 > 0x7fffffffULL) return cudaErrorInvalidValue;
    p.n_items = (int)items;
    // One CTA per work item, or (persistent, d = 64) as many CTAs as stay
    // resident, each taking every grid-th item.
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    const long long resident = (long long)sms * decode_ctas_per_sm<64>();
    const long long grid64 = decode_persistent<64>() ? (items < resident ? items : resident) : items;
    count_launch();
    cudaError_t e = d == 128 ? launch_split<128>(tq, tk, tv, p, items, stream)
                             : launch_split<64>(tq, tk, tv, p, grid64, stream);
    if (e != cudaSuccess) return e;
    count_launch();
    const unsigned cblocks = (unsigned)((rows * 32 + 255) / 256);
    if (d == 128)
        fa_decode_combine_kernel<128><<<cblocks, 256, 0, stream>>>(
            p.o_part, p.lse_part, static_cast<__nv_bfloat16*>(o), lse, (long long)rows, ns);
    else
        fa_decode_combine_kernel<64><<<cblocks, 256, 0, stream>>>(
            p.o_part, p.lse_part, static_cast<__nv_bfloat16*>(o), lse, (long long)rows, ns);
    return cudaGetLastError();
}

}  // namespace fa
