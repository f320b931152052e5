// Split-KV decoding forward: a few new query rows (Nq) against a long key /
// value sequence (Nk), the decoding setting of the FlashAttention blog
// ("Flash-Decoding": split the keys, compute partial softmax results in
// parallel, combine them with their log-sum-exp) and of the FA2 review thread.
//
// The queries are the last Nq positions: under the causal mask query row r
// sees key j iff j <= r + Nk - Nq (bottom-right alignment; the forward's
// j <= i when Nq == Nk).
//
// The work is bandwidth-bound (every key and value row is read once and used
// for only R = G * Nq query rows, G = H / Hkv), so it runs on the CUDA cores:
//   split kernel   one CTA per (batch, kv head, key split): one producer warp
//                  streams the split's contiguous K and V rows, 64 keys per
//                  tile, into a 96 KB shared-memory ring by bulk copies (two
//                  CTAs per SM for up to 8 rows); eight compute warps, per tile:
//                  (1) warp w scores keys w, w + 8, ...: lane l holds head-dim
//                  elements [EPL l, EPL l + EPL) of K and of the q rows
//                  (registers), and a key's R partial dot products are summed
//                  over the lanes by a reduce-scatter butterfly; (2) one warp
//                  per row updates the running max m and sum l over the tile
//                  (online softmax, base 2) and turns the scores into p;
//                  (3) thread t owns four columns (t % (d/4)) and every
//                  (256 / (d/4))-th key of the tile, and accumulates all R
//                  output rows over its keys after scaling them by
//                  2^(m_old - m_new).  At the end of the split the key groups'
//                  sums are added through shared memory, and the split writes
//                  o / l (fp32) and its LSE.
//   combine kernel one warp per output row: LSE = log sum_s exp(LSE_s),
//                  O = sum_s exp(LSE_s - LSE) O_s, bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kTileKeys = 64;         // keys per tile
constexpr int kThreads = 256;         // compute threads; one more warp produces
constexpr int kMaxRows = kDecodeMaxRows;   // G * Nq
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

struct DecodeParams {
    const __nv_bfloat16* q;   // [B][H][Nq][d]
    const __nv_bfloat16* k;   // [B][Hkv][Nk][d]
    const __nv_bfloat16* v;
    float* o_part;            // [B][H][Nq][n_split][d]
    float* lse_part;          // [B][H][Nq][n_split], natural log
    int H, Hkv, Nq, Nk, G, R, n_split, keys_per_split, causal;
    float scale_log2;
    DeviceStatus* status;
};

// K/V ring depth: 3 stages of 32 KB at d = 128, 6 of 16 KB at d = 64 (96 KB,
// so two CTAs fit on an SM when their registers allow).
template <int D>
__host__ __device__ constexpr int decode_stages() { return D == 128 ? 3 : 6; }
template <int D>
__host__ __device__ constexpr int decode_smem_bytes() { return decode_stages<D>() * 2 * kTileKeys * D * 2; }

template <int D, int RP>
__global__ void __launch_bounds__(kThreads + 32, 1)
fa_decode_split_kernel(const DecodeParams p) {
    constexpr int EPL = D / 32;               // head-dim elements per lane in (1)
    constexpr int CG = D / 4;                 // column groups of four
    constexpr int KG = kThreads / CG;         // key groups: 8 at d = 128, 16 at d = 64
    constexpr int KPT = kTileKeys / KG;       // keys of a tile per thread in (3)
    constexpr int KV_BYTES = kTileKeys * D * 2;
    constexpr int kStages = decode_stages<D>();
    extern __shared__ __align__(128) uint8_t dsm[];
    uint8_t* sK = dsm;                                   // [kStages][T][D] bf16
    uint8_t* sV = dsm + kStages * KV_BYTES;              // [kStages][T][D] bf16
    __shared__ __align__(16) float q_s[kMaxRows][D];     // q * scale * log2(e)
    __shared__ __align__(16) float p_s[kMaxRows][kTileKeys];
    __shared__ float alpha_s[kMaxRows], l_s[kMaxRows], m_s[kMaxRows];
    __shared__ uint64_t bar_full[kStages], bar_empty[kStages];
    __shared__ int abort_sh;
    const WaitCtx wc{p.status, &abort_sh};
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x % p.n_split;
    const int bg = blockIdx.x / p.n_split;                  // b * Hkv + g
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int j_begin = split * p.keys_per_split;
    const int j_end = min(p.Nk, j_begin + p.keys_per_split);
    const int n_tiles = (j_end - j_begin + kTileKeys - 1) / kTileKeys;
    const int R = p.R;
    const __nv_bfloat16* kh = p.k + (size_t)bg * p.Nk * D;
    const __nv_bfloat16* vh = p.v + (size_t)bg * p.Nk * D;

    if (tid == 0) {
        abort_sh = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], kThreads);
        }
        fence_mbar_init();
    }
    // q rows of the group: row r = hl * Nq + qi reads head g * G + hl.
    for (int e = tid; e < R * D; e += kThreads + 32) {
        const int r = e / D, c = e % D;
        const int hl = r / p.Nq, qi = r % p.Nq;
        const size_t src = (((size_t)b * p.H + g * p.G + hl) * p.Nq + qi) * D + c;
        q_s[r][c] = __bfloat162float(p.q[src]) * p.scale_log2;
    }
    __syncthreads();

    if (warp == kThreads / 32) {
        // ------------------------------------------------------ producer
        // K and V tiles are contiguous rows: one bulk copy each per tile.
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t, ++issued) {
                const int s = t % kStages;
                if (t >= kStages && !fa_wait(&bar_empty[s], ((t / kStages) - 1) & 1, 80, wc)) break;
                const int j0 = j_begin + t * kTileKeys;
                const uint32_t bytes = (uint32_t)min(kTileKeys, j_end - j0) * D * 2;
                mbar_arrive_expect_tx(&bar_full[s], 2 * bytes);
                bulk_load(sK + s * KV_BYTES, kh + (size_t)j0 * D, bytes, &bar_full[s]);
                bulk_load(sV + s * KV_BYTES, vh + (size_t)j0 * D, bytes, &bar_full[s]);
            }
            if (abort_sh) {   // copies still in flight (bounded)
                const WaitCtx dc{p.status, nullptr};
                for (int t = max(0, issued - kStages); t < issued; ++t)
                    fa_wait(&bar_full[t % kStages], (t / kStages) & 1, 81, dc);
            }
        }
        __syncwarp();
        return;   // the compute threads use named barrier 1 below, not __syncthreads
    }

    // ---------------------------------------------------------- compute
    float q_reg[RP][EPL];                     // this lane's slice of every q row
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int e = 0; e < EPL; ++e) q_reg[r][e] = (r < R) ? q_s[r][lane * EPL + e] : 0.0f;
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.0f, 0.0f};
    const int cg = tid % CG, kg = tid / CG;
    float acc[RP][4];
#pragma unroll
    for (int r = 0; r < RP; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.0f;
    const int shift = p.Nk - p.Nq;            // query row qi sees keys j <= qi + shift
    bool ok = true;

    for (int t = 0; ok && t < n_tiles; ++t) {
        const int s = t % kStages;
        // every compute thread waits (bounded); all of them stop if any gave up
        const bool got = fa_wait(&bar_full[s], (t / kStages) & 1, 82, wc);
        if (named_bar_or(1, kThreads, !got)) { ok = false; break; }
        const int t0 = j_begin + t * kTileKeys;
        const int nk = min(kTileKeys, j_end - t0);
        const uint8_t* kt = sK + s * KV_BYTES;
        const uint8_t* vt = sV + s * KV_BYTES;
        // (1) scores: warp w takes keys w, w + 8, ...; lane l holds head-dim
        // elements [EPL l, EPL l + EPL) of K (one conflict-free shared-memory
        // read per key) and of the RP q rows (registers); the RP partial dot
        // products are summed over the 32 lanes by a reduce-scatter butterfly
        // (RP - 1 + 5 - log2 RP shuffles per key), after which lanes with
        // l % (32 / RP) == 0 hold the score of row l / (32 / RP).
#pragma unroll
        for (int key = warp; key < kTileKeys; key += kThreads / 32) {
            float vals[RP];
            if (key < nk) {
                float kf[EPL];
                if (EPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(kt + (size_t)key * D * 2 + lane * 8);
                    kf[0] = __uint_as_float(w.x << 16);
                    kf[1] = __uint_as_float(w.x & 0xffff0000u);
                    kf[EPL > 2 ? 2 : 0] = __uint_as_float(w.y << 16);
                    kf[EPL > 2 ? 3 : 1] = __uint_as_float(w.y & 0xffff0000u);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(kt + (size_t)key * D * 2 + lane * 4);
                    kf[0] = __uint_as_float(w << 16);
                    kf[1] = __uint_as_float(w & 0xffff0000u);
                }
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    float a = 0.0f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) a = fmaf(q_reg[r][e], kf[e], a);
                    vals[r] = a;
                }
            } else {
#pragma unroll
                for (int r = 0; r < RP; ++r) vals[r] = 0.0f;
            }
            // reduce-scatter: at each step a lane keeps half of its rows and
            // adds the partner's copy of them
#pragma unroll
            for (int cnt = RP, o = 16; cnt > 1; cnt >>= 1, o >>= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i2 = 0; i2 < cnt / 2; ++i2) {
                    const float send = upper ? vals[i2] : vals[i2 + cnt / 2];
                    const float keep = upper ? vals[i2 + cnt / 2] : vals[i2];
                    vals[i2] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
#pragma unroll
            for (int o = 16 / RP; o > 0; o >>= 1) vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], o);
            const int span = 32 / RP;
            if ((lane % span) == 0) {
                const int r = lane / span;
                if (r < R) {
                    const int j = t0 + key;
                    const bool vis = key < nk && (!p.causal || j <= r % p.Nq + shift);
                    p_s[r][key] = vis ? vals[0] : -CUDART_INF_F;
                }
            }
        }
        named_bar_sync(1, kThreads);
        // (2) one warp per row: tile max, running max and sum, p in place
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = warp + 8 * i;
            if (r < R) {
                float sv[kTileKeys / 32];
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int e = 0; e < kTileKeys / 32; ++e) {
                    sv[e] = p_s[r][lane + 32 * e];
                    mx = fmaxf(mx, sv[e]);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_new = fmaxf(m_run[i], mx);
                // no visible key so far: keep everything at zero
                const float alpha = (m_new == -CUDART_INF_F) ? 1.0f : exp2f(m_run[i] - m_new);
                float sum = 0.0f;
#pragma unroll
                for (int e = 0; e < kTileKeys / 32; ++e) {
                    const float pe = (m_new == -CUDART_INF_F) ? 0.0f : exp2f(sv[e] - m_new);
                    p_s[r][lane + 32 * e] = pe;
                    sum += pe;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                l_run[i] = l_run[i] * alpha + sum;
                m_run[i] = m_new;
                if (lane == 0) alpha_s[r] = alpha;
            }
        }
        named_bar_sync(1, kThreads);
        // (3) O rows += p V over this thread's keys of the tile (rows of V in
        // shared memory, a warp reading one contiguous row segment)
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            if (r < R) {
                const float a = alpha_s[r];
                acc[r][0] *= a;
                acc[r][1] *= a;
                acc[r][2] *= a;
                acc[r][3] *= a;
            }
        }
#pragma unroll 4
        for (int i = 0; i < KPT; ++i) {
            const int jj = kg + KG * i;
            if (jj < nk) {
                const uint2 w = *reinterpret_cast<const uint2*>(vt + (size_t)jj * D * 2 + cg * 8);
                const float v0 = __uint_as_float(w.x << 16), v1 = __uint_as_float(w.x & 0xffff0000u);
                const float v2 = __uint_as_float(w.y << 16), v3 = __uint_as_float(w.y & 0xffff0000u);
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    if (r < R) {
                        const float pe = p_s[r][jj];
                        acc[r][0] = fmaf(pe, v0, acc[r][0]);
                        acc[r][1] = fmaf(pe, v1, acc[r][1]);
                        acc[r][2] = fmaf(pe, v2, acc[r][2]);
                        acc[r][3] = fmaf(pe, v3, acc[r][3]);
                    }
                }
            }
        }
        mbar_arrive(&bar_empty[s]);           // K and V of this stage are no longer read
        named_bar_sync(1, kThreads);          // p_s and alpha_s are rewritten next tile
    }
    if (!ok) return;

    // split outputs: O_s = o / l, LSE_s = ln2 (m + log2 l); -inf and zeros
    // when no key of the split is visible to the row.  The key groups' partial
    // sums meet in shared memory (p_s is free now), one row at a time.
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = warp + 8 * i;
        if (r < R && lane == 0) {
            l_s[r] = l_run[i];
            m_s[r] = m_run[i];
        }
    }
    float* red = &p_s[0][0];                  // [KG][D] floats: KG * D <= 16 * T
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        if (r >= R) break;                    // uniform across the compute threads
        named_bar_sync(1, kThreads);
        *reinterpret_cast<float4*>(red + kg * D + 4 * cg) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        named_bar_sync(1, kThreads);
        if (tid < D) {
            float sum = 0.0f;
#pragma unroll
            for (int k2 = 0; k2 < KG; ++k2) sum += red[k2 * D + tid];
            const int hl = r / p.Nq, qi = r % p.Nq;
            const size_t row = ((size_t)b * p.H + g * p.G + hl) * p.Nq + qi;
            const float l = l_s[r];
            p.o_part[(row * p.n_split + split) * D + tid] = (l > 0.0f) ? sum / l : 0.0f;
            if (tid == 0)
                p.lse_part[row * p.n_split + split] =
                    (l > 0.0f) ? (m_s[r] + log2f(l)) * kLn2 : -CUDART_INF_F;
        }
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
    float mx = -CUDART_INF_F;
    for (int s = lane; s < n_split; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float acc[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = 0.0f;
    float wsum = 0.0f;
    if (mx != -CUDART_INF_F) {
        for (int s = 0; s < n_split; ++s) {
            const float ls = lp[s];
            if (ls == -CUDART_INF_F) continue;
            const float w = expf(ls - mx);
            wsum += w;
            const float* os = o_part + (row * n_split + s) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(w, os[lane + 32 * c], acc[c]);
        }
    }
    const float inv = (wsum > 0.0f) ? 1.0f / wsum : 0.0f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) o[row * D + lane + 32 * c] = __float2bfloat16_rn(acc[c] * inv);
    if (lane == 0) lse[row] = (wsum > 0.0f) ? mx + logf(wsum) : -CUDART_INF_F;
}

}  // namespace

// Split policy: with its 96 KB K/V ring the split kernel fits two CTAs per SM
// for up to 8 rows per kv group (one for 16, by registers), so the number of
// CTAs, B * Hkv * n_split, is chosen for the fullest waves of that many
// slots on a 152-SM part among n_split in [ceil(slots / (B Hkv)),
// 4 ceil(slots / (B Hkv))], each split a whole number of 64-key tiles.  The
// target is fixed, so the workspace size does not depend on the device.
void decode_split_plan(int B, int Hkv, int R, int Nk, int* n_split, int* keys_per_split) {
    const int kSms = R <= 8 ? 2 * 152 : 152;
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
    decode_split_plan(B, Hkv, (H / Hkv) * Nq, Nk, &ns, &kps);
    const size_t rows = (size_t)B * H * Nq;
    const size_t o_bytes = (rows * ns * d * 4 + 255) / 256 * 256;
    return o_bytes + rows * ns * 4;
}

template <int D, int RP>
static cudaError_t launch_split(const DecodeParams& p, long long blocks, cudaStream_t stream) {
    auto kern = fa_decode_split_kernel<D, RP>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             decode_smem_bytes<D>());
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    kern<<<(unsigned)blocks, kThreads + 32, decode_smem_bytes<D>(), stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, int B, int H, int Hkv, int Nq, int Nk, int d,
                              int causal, float scale, DeviceStatus* status,
                              cudaStream_t stream) {
    DecodeParams p;
    int ns, kps;
    decode_split_plan(B, Hkv, (H / Hkv) * Nq, Nk, &ns, &kps);
    const size_t rows = (size_t)B * H * Nq;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
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
    const long long blocks = (long long)B * Hkv * ns;
    if (blocks > 0x7fffffffLL || rows * 32 / 256 + 1 > 0x7fffffffULL) return cudaErrorInvalidValue;
    count_launch();
    // rows padded to a power of two: 1, 2, 4, 8 or 16
    const int R = p.R;
    cudaError_t e;
    if (d == 128)
        e = R <= 1 ? launch_split<128, 1>(p, blocks, stream)
          : R <= 2 ? launch_split<128, 2>(p, blocks, stream)
          : R <= 4 ? launch_split<128, 4>(p, blocks, stream)
          : R <= 8 ? launch_split<128, 8>(p, blocks, stream)
                   : launch_split<128, 16>(p, blocks, stream);
    else
        e = R <= 1 ? launch_split<64, 1>(p, blocks, stream)
          : R <= 2 ? launch_split<64, 2>(p, blocks, stream)
          : R <= 4 ? launch_split<64, 4>(p, blocks, stream)
          : R <= 8 ? launch_split<64, 8>(p, blocks, stream)
                   : launch_split<64, 16>(p, blocks, stream);
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
