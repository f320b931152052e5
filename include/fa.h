/*
 * fa.h: C ABI of the GB300 (sm_103a) exact-attention library, libfa.so.
 *
 * The operation (pages of exact_attention_online):
 *   Forward, for every batch b and query head h, with key/value head
 *   g = h / (H / Hkv):
 *       S = scale * Q K^T   (key j > query i masked out when causal)
 *       P = softmax(S) row by row,   O = P V,   LSE_i = ln sum_j exp(S_ij)
 *   This is exact standard attention (FlashAttention blog, "From Online
 *   Softmax to FlashAttention"), computed tile by tile with the online-softmax
 *   recurrence (same page, "Online Softmax" and "FlashAttention") so the N x N
 *   score matrix never reaches device memory.  The division by the softmax
 *   denominator is deferred to the end, and LSE is saved instead of (m, l)
 *   (FlashAttention-2 review thread, author answer on non-matmul FLOPs and
 *   review 2).  Fully masked key blocks are skipped and the mask is applied to
 *   the diagonal block only (FlashAttention-2 review thread, answers on
 *   Figure 2 and on non-matmul FLOPs).
 *
 *   Backward, by recomputation (FlashAttention blog, "Backward -
 *   Recomputation"): from Q, K, V, O, dO and LSE it recomputes
 *   P = exp(S - LSE) and returns
 *       dV = P^T dO   (FlashAttention-2 review thread, public comment)
 *       dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P o (dP - D)
 *       dQ = scale * dS K,  dK = scale * dS^T Q
 *   with dK and dV summed over the query heads that share a key/value head
 *   (MQA/GQA).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA tensors) on the
 *     current device, except where stated.  The caller owns all memory; the
 *     library never allocates or frees device memory.
 *   - Layout: q, o, dout, dq are bf16 [B][H][N][d] contiguous; k, v, dk, dv
 *     are bf16 [B][Hkv][N][d] contiguous; lse is fp32 [B][H][N] (natural
 *     log).  Every tensor pointer must be 16-byte aligned.
 *   - Supported: d in {64, 128}; H % Hkv == 0; B, H, Hkv, N >= 1;
 *     B*H*N*d < 2^31; scale finite and > 0.  N need not be a multiple of the
 *     tile size.  Queries and keys have the same length N; the causal mask
 *     keeps key j for query i iff j <= i.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronize, except fa_device_status().
 *   - Arguments are validated before anything is launched.  A rejected call
 *     returns a negative fa_status and launches nothing.  A launch failure
 *     returns FA_ERR_CUDA.  Faults detected inside a kernel (a bounded wait
 *     that ran out) are recorded in a device status word that
 *     fa_device_status() reads.
 *   - Outputs may not alias inputs.  The library is thread-safe.
 *   - The library caches, per device, the device addresses of its own
 *     device variables (the status word, the fixed scratch array of
 *     fa_bwd_static_scratch) from the first call on that device.  Do not use
 *     it across a cudaDeviceReset() (or any teardown of the device's primary
 *     context) in the same process: the cached addresses would then point
 *     into memory that no longer belongs to the library.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1, /* null pointer, bad size, non-finite scale, H % Hkv != 0 */
    FA_ERR_UNSUPPORTED = -2, /* head dim not 64/128, sizes past the 32-bit index range,
                                device is not sm_103 */
    FA_ERR_ALIGNMENT = -3,   /* a tensor pointer is not 16-byte aligned */
    FA_ERR_WORKSPACE = -4,   /* workspace null or smaller than fa_bwd_workspace_size() */
    FA_ERR_CUDA = -5,        /* a CUDA runtime / driver call failed */
    FA_ERR_TIMEOUT = -6      /* a kernel's bounded wait ran out (device-side report) */
} fa_status;

/*
 * Forward.  Writes o (bf16, [B][H][N][d]) and lse (fp32, [B][H][N]).
 * One launch of the forward kernel.
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Hkv, int N, int d, int causal, float scale,
                 fa_stream_t stream);

/*
 * Forward with an fp32 output and an fp16 P V product.  Same operation,
 * layouts and errors as fa_fwd() except that o is fp32 [B][H][N][d] and that
 * the P V product runs in fp16 instead of bf16: P is rounded to fp16 (11
 * significant bits instead of 8) and each V tile is re-encoded as fp16 in
 * shared memory, exactly for magnitudes in [2^-14, 65280].  fa_fwd() rounds P
 * and O to bf16 (unit roundoff 2^-8 each), an error that grows with the
 * magnitude of V and O (up to 0.06 at |O| = 30, already 0.016 for |O| in
 * [4, 8)); here each p is off by at most 2^-11 of itself, and with the row
 * sum corrected for the rounding of each key block's largest p a row of O
 * moves by at most 2^-10 max|V| (in practice far less: a row whose weight
 * sits on one key returns that key's V row unrounded), the rest being the
 * fp32 accumulation's.  V entries of magnitude 65536 or more (beyond fp16)
 * make O non-finite; below 2^-14 they enter as fp16 subnormals (absolute
 * error at most 2^-25).
 * One launch of the forward kernel.
 */
FA_API fa_status fa_fwd_precise(const void* q, const void* k, const void* v, float* o,
                                float* lse, int B, int H, int Hkv, int N, int d, int causal,
                                float scale, fa_stream_t stream);

/*
 * Causal sliding-window ("local") forward: query i attends to the `window`
 * most recent keys, i - window < j <= i (FlashAttention-2 review thread, the
 * authors' common response, "Collaborations on open source models", names
 * local attention; the pages do not spell out the mask, and this is the
 * plain reading: the causal mask with a lower edge).  window >= N is plain
 * causal attention.  Arguments, layouts, ownership and errors as fa_fwd()
 * with causal = 1, plus FA_ERR_INVALID_ARG for window < 1.  Key blocks
 * wholly outside every window of a query tile are neither loaded nor
 * multiplied, so the cost grows with N * window instead of N^2 / 2.
 * One launch of the forward kernel.
 */
FA_API fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int Hkv, int N, int d, int window, float scale,
                               fa_stream_t stream);

/*
 * Packed variable-length batch forward ("varlen"): B sequences of different
 * lengths, concatenated without padding (FlashAttention-2 review thread, the
 * authors' answer "FA2 with variable sequence lengths": the lengths come as
 * an array; here as their running sums, so each sequence's first row needs
 * no scan).
 * Sequence b occupies rows cu_seqlens[b] .. cu_seqlens[b+1] - 1 of every
 * head; attention (with the causal mask when causal != 0) runs inside each
 * sequence only.
 *   q, o: bf16 [H][total][d];  k, v: bf16 [Hkv][total][d];  lse: fp32 [H][total].
 *   cu_seqlens: DEVICE int32 [B + 1], 0 = cu[0] <= cu[1] <= ... <= cu[B] = total,
 *     each length <= max_seqlen (read by the kernels; owned by the caller).
 *   max_seqlen: the longest sequence (sizes the work decomposition).
 * Offsets outside these rules give unspecified results but no access
 * outside the tensors: the kernels clamp each sequence to [0, total) and to
 * max_seqlen.  Errors as fa_fwd(), plus FA_ERR_INVALID_ARG for a null
 * cu_seqlens or total < 1.  bf16 output; no sliding window.
 * One launch of the forward kernel.
 */
FA_API fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                               int Hkv, int d, int causal, float scale, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd_varlen() needs: that of fa_bwd() for B
 * sequences of max_seqlen rows (the workspace keeps a padded max_seqlen-row
 * region per sequence and head).
 */
FA_API size_t fa_bwd_varlen_workspace_size(int B, int H, int Hkv, int max_seqlen, int d);

/*
 * Backward of fa_fwd_varlen(): layouts as there (dq like q; dk, dv like k),
 * lse as fa_fwd_varlen() wrote it, workspace as in fa_bwd() (>=
 * fa_bwd_varlen_workspace_size bytes).  Errors as fa_bwd() and
 * fa_fwd_varlen().  Three kernel launches.
 */
FA_API fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                               int B, int max_seqlen, int total, int H, int Hkv, int d,
                               int causal, float scale, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd() needs: -LSE and -D as 16-column bf16
 * tables ([B][H][Np][16] each, the operands of the small MMAs that fold them
 * into S and dP) and the fp32 dQ accumulator ([B][H][Np][d]), where Np is N
 * rounded up to 128.  Returns 0 for arguments fa_bwd() would reject.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * Backward.  Reads q, k, v, o, dout (bf16) and lse (fp32, as written by
 * fa_fwd), writes dq (bf16 [B][H][N][d]), dk, dv (bf16 [B][Hkv][N][d]).
 * `workspace` (device, >= fa_bwd_workspace_size bytes, 16-byte aligned) is
 * scratch owned by the caller; its contents on entry do not matter.
 * Equivalent to fa_bwd_preprocess, fa_bwd_dkdv and fa_bwd_dq_convert in that
 * order on `stream` (three kernel launches).  dk and dv are the same bit for
 * bit on every call with the same inputs (each key block's sums run in a
 * fixed order); dq sums the key blocks' partials with reduce-adds in the
 * order the CTAs finish, so its last bits can differ between calls.
 */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const void* dout, const float* lse, void* dq, void* dk, void* dv,
                 void* workspace, size_t workspace_bytes,
                 int B, int H, int Hkv, int N, int d, int causal, float scale,
                 fa_stream_t stream);

/*
 * Backward after fa_fwd_precise(): identical to fa_bwd() except that o is the
 * fp32 [B][H][N][d] output of fa_fwd_precise (used for D = rowsum(dO o O)).
 * Gradients are bf16 as in fa_bwd().  Three kernel launches.
 */
FA_API fa_status fa_bwd_precise(const void* q, const void* k, const void* v, const float* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes,
                                int B, int H, int Hkv, int N, int d, int causal, float scale,
                                fa_stream_t stream);

/*
 * Backward of fa_fwd_window(): arguments, layouts, workspace and errors as
 * fa_bwd() with causal = 1, plus FA_ERR_INVALID_ARG for window < 1; lse is the
 * one fa_fwd_window() wrote.  Each key block is paired only with the query
 * blocks whose windows reach it.  Three kernel launches.
 */
FA_API fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               void* workspace, size_t workspace_bytes,
                               int B, int H, int Hkv, int N, int d, int window, float scale,
                               fa_stream_t stream);

/*
 * Backward, stage 1 of 3: D_i = sum_c dO_ic O_ic (fp32); -D and -LSE (base-2
 * units, padding rows that give P = 0) written into the workspace tables as
 * three bf16 terms each; the fp32 dQ accumulator zeroed.  One launch.
 */
FA_API fa_status fa_bwd_preprocess(const void* o, const void* dout, const float* lse,
                            void* workspace, size_t workspace_bytes,
                            int B, int H, int Hkv, int N, int d, fa_stream_t stream);

/* Stage 1 for an fp32 o from fa_fwd_precise().  One launch. */
FA_API fa_status fa_bwd_preprocess_precise(const float* o, const void* dout, const float* lse,
                                           void* workspace, size_t workspace_bytes,
                                           int B, int H, int Hkv, int N, int d,
                                           fa_stream_t stream);

/*
 * Backward, stage 2 of 3: the main recomputation kernel.  One CTA per
 * (batch, key/value head, block of 128 keys) keeps K_j and V_j on chip, loops
 * over every query head of its group and every query block that can see the
 * keys, writes dK_j and dV_j, and adds its dQ partials into the fp32
 * accumulator in the workspace.  One launch.
 */
FA_API fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout,
                      void* dk, void* dv, void* workspace, size_t workspace_bytes,
                      int B, int H, int Hkv, int N, int d, int causal, float scale,
                      fa_stream_t stream);

/*
 * Backward stage 2 of fa_bwd_window(): fa_bwd_dkdv() with the causal
 * sliding-window mask (query i sees keys i - window < j <= i); window < 1 is
 * FA_ERR_INVALID_ARG.  Stages 1 and 3 do not depend on the mask.  One launch.
 */
FA_API fa_status fa_bwd_dkdv_window(const void* q, const void* k, const void* v,
                                    const void* dout, void* dk, void* dv, void* workspace,
                                    size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                                    int window, float scale, fa_stream_t stream);

/* Backward, stage 3 of 3: dq = bf16(scale * accumulator).  One launch. */
FA_API fa_status fa_bwd_dq_convert(const void* workspace, size_t workspace_bytes, void* dq,
                            int B, int H, int Hkv, int N, int d, float scale,
                            fa_stream_t stream);

/*
 * Training pair: a forward that also prepares its backward, and that
 * backward.  The backward of this library starts with a pass that writes a
 * -LSE table and zeroes the fp32 dQ accumulator in the workspace (stage 1);
 * a training step runs the forward and the backward back to back, and
 * fa_fwd_train writes those rows from its own epilogue, where LSE is
 * computed, so the backward's first pass only computes D = rowsum(dO o O).
 * Splitting stage 1 this way is this library's; the pages describe the
 * backward's inputs (O, dO, LSE), not this schedule.
 *
 * fa_fwd_train: fa_fwd() (same arguments, outputs and errors), plus
 * `workspace` (>= fa_bwd_workspace_size(B, H, Hkv, N, d) bytes, 16-byte
 * aligned, owned by the caller) prepared for fa_bwd_train().  One launch.
 * fa_bwd_train: the backward of that forward.  q, k, v, o, dout as in
 * fa_bwd(); the workspace must be the one the last fa_fwd_train() with the
 * same shapes prepared, unchanged since (no lse argument: its -LSE table is
 * in the workspace).  Same results as fa_bwd() on the lse that forward wrote.
 * Three launches.  The _precise forms take and give the fp32 o of
 * fa_fwd_precise().
 */
FA_API fa_status fa_fwd_train(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                              int N, int d, int causal, float scale, fa_stream_t stream);
FA_API fa_status fa_fwd_train_precise(const void* q, const void* k, const void* v, float* o,
                                      float* lse, void* workspace, size_t workspace_bytes,
                                      int B, int H, int Hkv, int N, int d, int causal,
                                      float scale, fa_stream_t stream);
FA_API fa_status fa_bwd_train(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                              int causal, float scale, fa_stream_t stream);
FA_API fa_status fa_bwd_train_precise(const void* q, const void* k, const void* v,
                                      const float* o, const void* dout, void* dq, void* dk,
                                      void* dv, void* workspace, size_t workspace_bytes, int B,
                                      int H, int Hkv, int N, int d, int causal, float scale,
                                      fa_stream_t stream);

/*
 * The training pair for the causal sliding window of fa_fwd_window() /
 * fa_bwd_window(): fa_fwd_window_train is fa_fwd_window() (same arguments,
 * outputs and errors) plus the workspace prepared as by fa_fwd_train();
 * fa_bwd_window_train is fa_bwd_window() on that workspace (no lse
 * argument), three launches.  window < 1 is FA_ERR_INVALID_ARG.
 */
FA_API fa_status fa_fwd_window_train(const void* q, const void* k, const void* v, void* o,
                                     float* lse, void* workspace, size_t workspace_bytes, int B,
                                     int H, int Hkv, int N, int d, int window, float scale,
                                     fa_stream_t stream);
FA_API fa_status fa_bwd_window_train(const void* q, const void* k, const void* v, const void* o,
                                     const void* dout, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, int B, int H,
                                     int Hkv, int N, int d, int window, float scale,
                                     fa_stream_t stream);

/*
 * Stage 1 of fa_bwd_train(), for callers that time or interleave the stages:
 * -D into the workspace a training forward prepared (one launch; _precise:
 * fp32 o).  fa_bwd_train() is fa_bwd_preprocess_train() + fa_bwd_dkdv() +
 * fa_bwd_dq_convert().
 */
FA_API fa_status fa_bwd_preprocess_train(const void* o, const void* dout, void* workspace,
                                         size_t workspace_bytes, int B, int H, int Hkv, int N,
                                         int d, fa_stream_t stream);
FA_API fa_status fa_bwd_preprocess_train_precise(const float* o, const void* dout,
                                                 void* workspace, size_t workspace_bytes, int B,
                                                 int H, int Hkv, int N, int d,
                                                 fa_stream_t stream);

/*
 * Backward without a workspace argument, for callers that cannot allocate
 * device memory (a runtime that owns all device memory in a fixed pool, a
 * latency-critical loop that must not risk the synchronisation cudaMalloc can
 * cause, a plugin without access to the host application's allocator).  The
 * pages have no counterpart to this; it is a deployment convenience.
 * Same operation, arguments (minus workspace) and results as fa_bwd().  The
 * scratch fa_bwd() takes from the caller lives instead in one fixed 32 MiB
 * array in device memory owned by the library; every GPU that loads the
 * library holds it until the process exits.  Calls whose
 * fa_bwd_workspace_size() exceeds 32 MiB return FA_ERR_WORKSPACE.  All calls
 * on a device share the array: calls that overlap on the GPU race, so order
 * them on one stream.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  Allocates nothing.  Three launches.
 */
FA_API fa_status fa_bwd_static_scratch(const void* q, const void* k, const void* v,
                                       const void* o, const void* dout, const float* lse,
                                       void* dq, void* dk, void* dv,
                                       int B, int H, int Hkv, int N, int d, int causal,
                                       float scale, fa_stream_t stream);

/*
 * FP8 forward (FlashAttention-3 summary, abstract: FP8 with block
 * quantization): the P V product in e4m3, S = Q K^T in bf16.  Two calls:
 * quantize V once, then run the forward.  Head dimension 128 only
 * (FA_ERR_UNSUPPORTED otherwise).
 *
 * Why only P V: e4m3 keeps 3 mantissa bits, so rounding Q and K puts a relative
 * error of about 2.7 % RMS on each and the scores inherit it before the
 * exponential; with Q, K, V and P all in e4m3 the output's relative RMS error
 * is about 0.05 on N(0,1) inputs and up to 0.12 on inputs with outliers.
 * Keeping the scores in bf16 and only P and V in e4m3 halves that.
 *
 * Quantization (the block granularity is this library's reading of "block
 * quantization"): for each (batch, kv head) of V and each block of 128 rows,
 * amax = max |x| over the block, scale = amax / 448 and inv = 448 / amax
 * (fp32 divisions; 1 and 1 for an all-zero block), and each element becomes
 * the e4m3 code of fp32(x * inv): 1 sign, 4 exponent (bias 7) and 3 mantissa
 * bits, round to nearest even, magnitudes beyond 448 saturate to 448.
 *
 * fp8_buf is one caller-owned device buffer of fa_fp8_buffer_size() bytes,
 * 256-byte aligned, laid out as consecutive regions each starting on a
 * 256-byte boundary (Np = N rounded up to 128, nblk = Np / 128):
 *   v8t   uint8 [B*Hkv][128][Np]     e4m3 codes of V, transposed (keys last;
 *                                    zero on keys >= N)
 *   sv    fp32  [B*Hkv][nblk]        block scales of V
 *   svmax fp32  [B*Hkv]              largest V block scale of each kv head
 * fa_fp8_buffer_size() returns 0 for an invalid shape or d != 128.
 */
FA_API size_t fa_fp8_buffer_size(int B, int H, int Hkv, int N, int d);

/*
 * Fills fp8_buf from bf16 v [B][Hkv][N][d] (H only checks H % Hkv).  Errors:
 * FA_ERR_INVALID_ARG (shape, null tensor), FA_ERR_UNSUPPORTED (d != 128),
 * FA_ERR_WORKSPACE (null or too small buffer), FA_ERR_ALIGNMENT (buffer not
 * 256-byte aligned), FA_ERR_CUDA.  Asynchronous on `stream`; two launches.
 */
FA_API fa_status fa_fp8_quantize(const void* v, void* fp8_buf, size_t fp8_buf_bytes, int B, int H,
                                 int Hkv, int N, int d, fa_stream_t stream);

/*
 * Attention forward with the P V product in e4m3: S = Q K^T from the bf16
 * q [B][H][N][d] and k [B][Hkv][N][d] (tcgen05 kind::f16, fp32 in tensor
 * memory), the online softmax in fp32, P quantized to e4m3 as
 * e4m3(p * 448 * sv_j / svmax) for key block j (p <= 1: the running max is
 * exact), O += P8 V8 (kind::f8f6f4, fp32 accumulation) with V from the buffer
 * fa_fp8_quantize() filled, O = O * (svmax / 448) / l written as bf16
 * o [B][H][N][d], and the fp32 natural-log LSE [B][H][N] (the same LSE as
 * fa_fwd(): it depends on S only).  Same shapes, causal convention and errors
 * as fa_fwd() (plus FA_ERR_UNSUPPORTED for d != 128 and the buffer errors
 * above).  Asynchronous on `stream`; one launch.
 */
FA_API fa_status fa_fwd_fp8(const void* q, const void* k, const void* fp8_buf,
                            size_t fp8_buf_bytes, void* o, float* lse, int B, int H, int Hkv,
                            int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * Split-KV decoding forward (FlashAttention blog, "Flash-Decoding"; the
 * decoding setting of the FA2 review thread): Nq new query rows against Nk >=
 * Nq keys.  q and o are bf16 [B][H][Nq][d], k and v bf16 [B][Hkv][Nk][d], lse
 * fp32 [B][H][Nq] (natural log).  The queries are the last Nq positions:
 * with causal != 0 query row r sees keys j <= r + Nk - Nq (bottom-right
 * alignment; the same rule as fa_fwd() when Nq == Nk).  The keys are split
 * across CTAs, each split's partial output and LSE go to the workspace, and a
 * second kernel combines them (two launches).  d in {64, 128}; (H / Hkv) * Nq
 * <= 16 (FA_ERR_UNSUPPORTED otherwise).  workspace: caller-owned device
 * memory of fa_fwd_decode_workspace_size() bytes, 256-byte aligned
 * (FA_ERR_WORKSPACE if null or smaller, FA_ERR_ALIGNMENT if misaligned).
 * Tensors 16-byte aligned.  Asynchronous on `stream`.
 */
FA_API size_t fa_fwd_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d);
FA_API fa_status fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                               void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                               int Nq, int Nk, int d, int causal, float scale,
                               fa_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the device status word of the
 * current device: FA_OK, or the first error a kernel recorded (for example
 * FA_ERR_TIMEOUT when a bounded wait ran out).  Returns FA_ERR_CUDA if the
 * synchronization itself fails.
 */
FA_API fa_status fa_device_status(fa_stream_t stream);

/*
 * Where the last recorded device error came from: writes the wait-site id and
 * the linear block index (either pointer may be NULL).  Host-side read of the
 * status word; call after fa_device_status() reported an error.
 */
FA_API void fa_device_status_detail(int* site, int* block);

/* Static English name of a status code ("FA_OK", ...).  Never NULL. */
FA_API const char* fa_status_string(fa_status s);

/*
 * Number of kernels this library has launched in this process (all devices),
 * a host-side counter for diagnostics.
 */
FA_API long long fa_kernel_launches(void);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier that nothing completes, with a limit of `timeout_ns` nanoseconds
 * (clamped to [1e3, 5e9]).  The kernel gives up, records FA_ERR_TIMEOUT in
 * the status word and returns; the context stays usable.  Returns FA_OK if
 * the launch succeeded (read the outcome with fa_device_status()).
 */
FA_API fa_status fa_watchdog_selftest(long long timeout_ns, fa_stream_t stream);

/*
 * Diagnostic of the exponential used when part of a softmax row's exps run on
 * the FMA pipe instead of the exponential unit (the pages' argument that every
 * non-matmul cycle counts, FlashAttention-2 review thread, author answer on
 * non-matmul FLOPs, applied to the GPU's second bottleneck): for n device
 * floats x, writes y_fma = 2^x computed as 2^rint(x) * p(x - rint(x)), p the
 * fp32 minimax cubic fitted by csrc/fit_exp2_poly.py (relative error at most
 * 7.5e-5 in the normal range, x clamped below at -126), and y_ex2 = 2^x from
 * ex2.approx.ftz.f32.  Device pointers; one launch; FA_ERR_INVALID_ARG for
 * n < 1 or a null pointer.
 */
FA_API fa_status fa_exp2_check(const float* x, float* y_fma, float* y_ex2, int n,
                               fa_stream_t stream);

/*
 * Throughput microbenchmark of the exponential unit, the second bound of the
 * attention kernels after the tensor core (one 2^x per score element; the
 * FlashAttention-2 review thread, author answer on non-matmul FLOPs): `blocks`
 * CTAs of 256 threads, each thread running eight independent chains
 * x <- 2^(-x) of ex2.approx.ftz.f32 for `iters` rounds, so one launch
 * evaluates blocks * 256 * 8 * iters exps; `out` (device, blocks * 256 floats,
 * owned by the caller) receives each thread's sum of its eight final values
 * (each in [1/2, 1]).  Time the launch on `stream` to get the unit's rate.
 * FA_ERR_INVALID_ARG for a null pointer, blocks outside [1, 2^20] or iters
 * outside [1, 2^24].
 */
FA_API fa_status fa_ex2_rate(float* out, int blocks, int iters, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
