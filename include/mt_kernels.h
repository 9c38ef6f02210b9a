/*
 * mt_kernels.h - C ABI of the individual sm_103a kernels of the stateless
 * layer template (libmt.so). The training step (mt.h) is built from these;
 * they are exported so each one can be checked on its own.
 *
 * The template is the per-layer compute of the RAM-centric method
 * ("MegaTrain：单卡训百亿大模型的突破与实践", zhichai.net, section
 * "以内存为中心的训练新范式" point 4: a lightweight stateless template per
 * layer, parameters bound at run time; travelaiplan blog "單卡也能練 100B+",
 * 核心功能 point 3: hand-written backward per layer instead of autograd).
 *
 * Conventions for every function below:
 *  - all array arguments are DEVICE pointers, caller-owned; nothing is
 *    allocated or freed; outputs are fully overwritten unless stated;
 *  - bf16 = IEEE bfloat16 bits (uint16), fp32 = float; matrices are
 *    row-major with the given leading dimension (elements);
 *  - tokens are laid out row-major (batch, position): row m = b * s + t;
 *  - `stream` is a cudaStream_t (NULL = legacy default stream); the call only
 *    enqueues work and returns;
 *  - return MT_OK, MT_EINVAL (bad shape / alignment; nothing enqueued) or
 *    MT_ECUDA (launch failed).
 */
#ifndef MT_KERNELS_H_
#define MT_KERNELS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Dense product on tcgen05 tensor cores: C[M,N] = A[M,K] * B[N,K]^T (+ R).
 * A, B bf16 K-contiguous, 16-byte aligned, lda/ldb multiples of 8. C is bf16
 * (c_f32 = 0, ldc multiple of 8) or fp32 (c_f32 = 1, ldc multiple of 4). R is
 * an optional [M,N] residual of C's element type (bf16 or fp32; 16-byte
 * aligned, ldr multiple of 8) added to the fp32 accumulator before the store.
 * The linear layers y = x W^T of a decoder layer (W stored [out, in]); with
 * fp32 C and R the output and down projections add into the fp32 residual
 * stream.
 */
int mt_k_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int c_f32,
              const void* R, int64_t ldr, int M, int N, int K, void* stream);

/*
 * The same product with either operand read in place in the other layout:
 * a_mn_major = 1 means A is stored [K, M] (M contiguous, row pitch lda >= M),
 * i.e. the product uses A^T of that array; b_mn_major = 1 means B is stored
 * [K, N] (row pitch ldb >= N). This covers a linear layer's backward without
 * transposing anything: dX = dY W (B = W [out, in] as [K, N]) and
 * dW = dY^T X (A = dY [tokens, out], B = X [tokens, in], both [K, *]).
 * Pitches are multiples of 8 elements; other rules as mt_k_gemm.
 */
int mt_k_gemm_ex(const void* A, int64_t lda, int a_mn_major, const void* B, int64_t ldb, int b_mn_major, void* C,
                 int64_t ldc, int c_f32, const void* R, int64_t ldr, int M, int N, int K, void* stream);

/*
 * QKV projection with RoPE in the epilogue: C = A B^T as mt_k_gemm (bf16 C),
 * where each row's columns [0, rot_cols) - heads of hd columns - are rotated
 * like mt_k_rope (inverse = 0) at position (row mod seq) from the fp32
 * products and rounded to bf16 once (mt_k_gemm followed by mt_k_rope rounds
 * twice: before and after the rotation). The attention input of one layer
 * (the zhichai.net article's stateless template, point 4). hd 64 or 128, N
 * and rot_cols multiples of hd; cos/sin fp32 [seq_max, hd/2].
 */
int mt_k_gemm_rope(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int M, int N, int K,
                   const float* cos_t, const float* sin_t, int rot_cols, int hd, int seq, void* stream);

/*
 * Gate/up projection with SwiGLU in the epilogue: W bf16 [2f, K] holds the
 * gate rows then the up rows (K-major, like mt_k_gemm's B). Writes
 * gu = A W^T (bf16 [M, 2f], row pitch ldgu; kept for the backward) and
 * a = silu(gate) * up computed from the fp32 gate and up (bf16 [M, f], row
 * pitch lda_out). mt_k_gemm then mt_k_swiglu_fwd computes a from the
 * bf16-rounded gate and up instead. f a multiple of 128.
 */
int mt_k_gemm_swiglu_fwd(const void* A, int64_t lda, const void* W, int64_t ldw, void* gu, int64_t ldgu, void* a,
                         int64_t lda_out, int M, int f, int K, void* stream);

/*
 * Down projection input gradient with the SwiGLU backward in the epilogue:
 * the fp32 da = dy W (dy bf16 [M, K], W the down weight bf16 [K, f] read in
 * place, as mt_k_gemm_ex with b_mn_major = 1) is turned into
 * dgu = (d gate | d up) [M, 2f] (bf16) with gate | up read from gu [M, 2f];
 * da is never written or rounded (mt_k_gemm_ex then mt_k_swiglu_bwd rounds
 * it to bf16 first). f a multiple of 32.
 */
int mt_k_gemm_swiglu_bwd(const void* dy, int64_t lddy, const void* W, int64_t ldw, const void* gu, int64_t ldgu,
                         void* dgu, int64_t lddgu, int M, int f, int K, void* stream);

/*
 * Weight gradient of a linear layer, G = dY^T X over K tokens: dY bf16
 * [K, M] (pitch lddy), X bf16 [K, N] (pitch ldx), G bf16 [M, N] (pitch ldg,
 * a multiple of 8; G 16-byte aligned). When M x N has too few 128 x 256
 * output tiles to fill the 152 SMs (mt_k_gemm_splitk(M, N, K) > 1), the K
 * tokens are split into that many contiguous ranges, each range's fp32
 * product goes to its own slice of the device workspace ws (ws_elems fp32
 * elements, at least mt_k_gemm_wgrad_ws(M, N); caller-owned) and the slices
 * are summed in slice order and rounded once to bf16: deterministic, and
 * equal to the unsplit product up to fp32 summation order. With ws NULL or
 * too small it is the plain product (mt_k_gemm_ex, a_mn = b_mn = 1). The
 * layer-wise backward of the streamed template (the zhichai.net article,
 * point 5) computes every dW this way before the slab copy.
 */
int mt_k_gemm_wgrad(const void* dY, int64_t lddy, const void* X, int64_t ldx, void* G, int64_t ldg, int M, int N,
                    int K, float* ws, int64_t ws_elems, void* stream);
/*
 * Tile shape of plain products (no fused epilogue, no K split), process-wide:
 * 0 = the library's choice (default; 256 x 256 tiles for products with many
 * tiles, where an SM's operand bytes per product are the limit, else
 * 128 x 256), 1 = always 128 x 256, 2 = always 256 x 256. Results are the
 * same up to fp32 summation order within a tile (none: both shapes sum K in
 * the same order, so they are bitwise equal). Not thread-safe against
 * concurrent launches. Returns MT_EINVAL for other values.
 */
int mt_k_gemm_tile_policy(int policy);
/* Split factor mt_k_gemm_wgrad uses for G [M, N] over K tokens (1: none). */
int mt_k_gemm_splitk(int M, int N, int K);
/* fp32 workspace elements mt_k_gemm_wgrad may use for G [M, N] at any K. */
int64_t mt_k_gemm_wgrad_ws(int M, int N);

/*
 * RMSNorm forward: y[m,:] = x[m,:] * rstd[m] * w, rstd = 1/sqrt(mean(x^2)+eps).
 * x [M, d] is bf16 (x_f32 = 0) or fp32 (x_f32 = 1: the residual stream);
 * y bf16 [M, d] (ld = d), w bf16 [d], rstd fp32 [M]. d multiple of 8.
 */
int mt_k_rmsnorm_fwd(const void* x, int x_f32, const void* w, void* y, float* rstd, int M, int d, float eps,
                     void* stream);

/*
 * RMSNorm backward. dy: gradient w.r.t. y, fp32 [M, d]; x [M, d] bf16
 * (x_f32 = 0) or fp32 (x_f32 = 1);
 * dres: optional fp32 [M, d] added to dx (the residual branch). Writes
 * dx_f32 (fp32 [M,d], may be NULL) and dx_bf16 (bf16 [M,d], may be NULL),
 * per-block partial sums of dw into `partial` (fp32 [n_part, d], scratch)
 * and the final dw (summed over rows in a fixed order) as bf16 into dw_out.
 * dx_f32 may alias dres. mt_k_rmsnorm_bwd_parts() gives n_part for M.
 */
int mt_k_rmsnorm_bwd(const float* dy, const void* x, int x_f32, const void* w, const float* rstd, const float* dres,
                     float* dx_f32, void* dx_bf16, float* partial, void* dw_out, int M, int d, void* stream);
int mt_k_rmsnorm_bwd_parts(int M);

/*
 * Rotate-half RoPE in place on the first `n_rot_heads` heads of each token
 * row of a bf16 [B*s, ld] buffer (heads of hd contiguous elements starting at
 * column 0). cos/sin fp32 [s_max, hd/2] tables. inverse = 1 rotates by the
 * negative angle (the backward).
 */
int mt_k_rope(void* x, int64_t ld, int B, int s, int n_rot_heads, int hd, const float* cos_t, const float* sin_t,
              int inverse, void* stream);

/* a[m, j] = silu(gu[m, j]) * gu[m, f + j]; gu bf16 [M, 2f], a bf16 [M, f]. */
int mt_k_swiglu_fwd(const void* gu, void* a, int M, int f, void* stream);

/* dgu[m, j] = da*u*sig(g)*(1+g(1-sig(g))), dgu[m, f+j] = da*silu(g); da bf16 [M, f]. */
int mt_k_swiglu_bwd(const void* da, const void* gu, void* dgu, int M, int f, void* stream);

/*
 * Causal grouped-query attention forward (flash style, KV streamed in tiles).
 * qkv bf16 [B*s, ldqkv]: q heads at columns [0, H*hd), k heads at
 * [H*hd, (H+Hkv)*hd), v heads after; o bf16 [B*s, ldo] (H*hd columns);
 * lse fp32 [B, H, s] natural-log softmax denominators. hd in {16, 64, 128};
 * hd 64 / 128 run on tcgen05 (o 16-byte aligned, ldo multiple of 8).
 */
int mt_k_attn_fwd(const void* qkv, int64_t ldqkv, void* o, int64_t ldo, float* lse, int B, int s, int H, int Hkv,
                  int hd, void* stream);

/*
 * The same forward on the legacy warp-level mma.sync tensor-core path
 * (any hd in {16, 64, 128}); mt_k_attn_fwd uses it for hd = 16 and runs
 * hd 64 / 128 on tcgen05 with TMEM accumulators. Kept for comparison.
 */
int mt_k_attn_fwd_mma(const void* qkv, int64_t ldqkv, void* o, int64_t ldo, float* lse, int B, int s, int H,
                      int Hkv, int hd, void* stream);

/*
 * Attention backward, deterministic (no float atomics). Inputs as the
 * forward plus dout bf16 [B*s, lddo] and the forward's lse. delta is fp32
 * scratch [B, H, s]. Writes dq, dk, dv into dqkv bf16 [B*s, lddqkv] in the
 * qkv column layout.
 */
int mt_k_attn_bwd(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout, int64_t lddo,
                  const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B, int s, int H, int Hkv, int hd,
                  void* stream);

/*
 * The same backward with RoPE's inverse rotation applied to dq and dk before
 * they are stored (position = row mod s; cos_t / sin_t fp32 [s_max, hd/2],
 * 16-byte aligned, as mt_k_rope), so dqkv holds the gradients w.r.t. the
 * un-rotated q, k and v. At hd 64 / 128 the rotation runs on the fp32
 * accumulators in the tcgen05 kernels' stores (dq and dk rounded to bf16
 * once); at hd 16 it is mt_k_attn_bwd followed by mt_k_rope (inverse = 1).
 * The backward of the decoder layer's "RoPE then attention" (the stateless
 * template, zhichai.net article point 4).
 */
int mt_k_attn_bwd_rope(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout, int64_t lddo,
                       const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B, int s, int H, int Hkv,
                       int hd, const float* cos_t, const float* sin_t, void* stream);

/* The same backward on the legacy mma.sync path (any hd); mt_k_attn_bwd uses
 * it for hd = 16 and runs hd 64 / 128 on tcgen05. Kept for comparison. */
int mt_k_attn_bwd_mma(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout, int64_t lddo,
                      const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B, int s, int H, int Hkv,
                      int hd, void* stream);

/*
 * Cross entropy over a vocabulary row block: logits fp32 [M, ldl], labels
 * int32 [M]. Writes dz bf16 [M, lddz] = (softmax - onehot) * scale and
 * loss_rows fp32 [M] = logsumexp - z[label] (unscaled).
 */
int mt_k_cross_entropy(const float* logits, int64_t ldl, const int32_t* labels, void* dz, int64_t lddz,
                       float* loss_rows, int M, int V, float scale, void* stream);

/* out[0] = sum of x[0..n) in a fixed order (fp64 accumulation), fp32 result. */
int mt_k_sum(const float* x, int n, float* out, void* stream);

/* x[m, :] = E[tok[m], :]; E bf16 [V, d], x [M, d] bf16 (x_f32 = 0) or fp32
 * (x_f32 = 1, exact). Ids outside [0, V) give a zero row and set the device
 * error word. */
int mt_k_embedding_fwd(const void* E, const int32_t* tok, void* x, int x_f32, int M, int d, int V, void* stream);

/*
 * dE[v, :] = sum over m with tok[m] = v of dx[m, :], bf16 [V, d] output,
 * fp32 dx [M, d]. Deterministic: rows are summed in increasing m. `work` is
 * int32 scratch of mt_k_embedding_bwd_work(M, V) elements.
 */
int mt_k_embedding_bwd(const float* dx, const int32_t* tok, void* dE, int M, int d, int V, int32_t* work,
                       void* stream);
int64_t mt_k_embedding_bwd_work(int M, int V);

/*
 * Embedding backward for callers that cannot allocate device memory (for
 * example code running inside another framework's memory pool, or a
 * process whose allocator is owned by someone else), so they cannot pass the
 * `work` buffer mt_k_embedding_bwd needs. The articles describe no such
 * entry point; it exists for this library's users only.
 *
 * Same arguments and result as mt_k_embedding_bwd without `work`: the sort
 * workspace is a fixed array of (2 * 262144 + 1 + 524288) int32 (4 MiB) in
 * the library's device memory, held by every GPU that loads the library
 * until the process exits. It therefore accepts at most
 * MT_NOALLOC_EMBED_MAX_TOKENS tokens (M) and MT_NOALLOC_EMBED_MAX_VOCAB rows
 * (V); larger sizes return MT_EINVAL with a message in mt_last_error(NULL).
 * It calls no allocation routine. The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture. The address is kept for
 * the life of the process: after cudaDeviceReset (or anything else that
 * replaces the device's primary context) it is stale and the entry point
 * must not be called again in that process. All calls share the one
 * array: calls that can overlap on the GPU (other streams, other threads)
 * race and must be serialised by the caller. Nothing a previous call left in
 * the array affects the result. Ids outside [0, V) are left out of the sums
 * without a report (check them first with mt_k_check_ids if needed).
 */
#define MT_NOALLOC_EMBED_MAX_TOKENS 524288
#define MT_NOALLOC_EMBED_MAX_VOCAB 262144
int mt_k_embedding_bwd_noalloc(const float* dx, const int32_t* tok, void* dE, int M, int d, int V, void* stream);

/* Sets *bad = 1 if any of the n ids lies outside [0, V) (device check). */
int mt_k_check_ids(const int32_t* ids, int n, int V, int32_t* bad, void* stream);

/* Reads (and with reset = 1 clears) the device error word of the current device. */
int mt_k_device_error(int* code, int reset);

#ifdef __cplusplus
}
#endif
#endif /* MT_KERNELS_H_ */
