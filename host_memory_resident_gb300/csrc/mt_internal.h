// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "../../include/mt.h"
#include "../../include/mt_kernels.h"

namespace mt {

// Address of the current device's error word (allocated on first use,
// zero-initialised, kept until process exit); null if allocation failed.
int* device_error_word();

// Sets the calling thread's message returned by mt_last_error(NULL).
void set_last_error_message(const std::string& msg);

// C = op(A) * op(B) (+ R) with either operand K-major or MN-major; see mt_k_gemm_ex.
int gemm_ex(const void* A, long long lda, int a_mn, const void* B, long long ldb, int b_mn, void* C, long long ldc,
            int c_f32, const void* R, long long ldr, int M, int N, int K, cudaStream_t stream);

// Heads per chunk of the attention kernels' launch order: as many as keep
// the streamed operands of the CTAs in flight (bytes_per_head each) within
// about 48 MiB of the 129 MB L2; at least 1, at most nh.
inline int attn_head_chunk(long long bytes_per_head, int nh) {
  const long long budget = 48LL << 20;
  long long hc = bytes_per_head > 0 ? budget / bytes_per_head : nh;
  if (hc < 1) hc = 1;
  if (hc > nh) hc = nh;
  return (int)hc;
}

// Tile shape of plain products: 0 the built-in choice, 1 always 128 x 256,
// 2 always 256 x 256 where allowed (plain epilogue, no split). Process-wide.
int gemm_tile_policy(int policy);

// Split-K factor the library uses for C[M, N] over K (1: no split; depends
// on the shape only, so planning needs no GPU).
int splitk_factor(int M, int N, int K);
// Workspace elements gemm_wgrad needs to split C[M, N] for any K (0: never).
size_t splitk_ws_elems(int M, int N);
// C (bf16) = op(A) op(B)^T over K, split along K into fp32 slices of ws
// (splitk_factor(M, N, K) * M * N elements) and summed in a fixed order when
// that is faster; a plain product otherwise. Deterministic.
int gemm_wgrad(const void* A, long long lda, int a_mn, const void* B, long long ldb, int b_mn, void* C, long long ldc,
               int M, int N, int K, float* ws, size_t ws_elems, cudaStream_t stream);

// GEMMs with fused epilogues; see mt_k_gemm_rope, mt_k_gemm_swiglu_fwd,
// mt_k_gemm_swiglu_bwd.
int gemm_rope(const void* A, long long lda, const void* B, long long ldb, void* C, long long ldc, int M, int N, int K,
              const float* cos_t, const float* sin_t, int rot_cols, int hd, int seq, cudaStream_t stream);
int gemm_swiglu_fwd(const void* A, long long lda, const void* W, long long ldw, void* gu, long long ldgu, void* a,
                    long long lda_out, int M, int f, int K, cudaStream_t stream);
int gemm_swiglu_bwd(const void* dy, long long lddy, const void* W, long long ldw, const void* gu, long long ldgu,
                    void* dgu, long long lddgu, int M, int f, int K, cudaStream_t stream);

// Causal GQA attention forward on tcgen05 (hd 64 or 128); see mt_k_attn_fwd.
int attn_fwd_tc(const void* qkv, long long ld, void* o, long long ldo, float* lse, int B, int s, int H, int Hkv,
                int hd, cudaStream_t stream);

// Attention backward products on tcgen05 (hd 64 or 128); delta precomputed.
// With cos_t / sin_t non-null, dq and dk are stored rotated back (RoPE's
// inverse at position row mod s).
int attn_bwd_tc(const void* qkv, long long ld, const void* dout, long long lddo, const float* lse,
                const float* delta, void* dqkv, long long lddq, int B, int s, int H, int Hkv, int hd,
                const float* cos_t, const float* sin_t, cudaStream_t stream);

// dst[i] = bf16(src[i]) for i < n (round to nearest even).
int convert_f32_bf16(const float* src, void* dst, long long n, cudaStream_t stream);

// C = A * B^T (+ R); see mt_k_gemm.
int gemm_abt(const void* A, long long lda, const void* B, long long ldb, void* C, long long ldc, int c_f32,
             const void* R, long long ldr, int M, int N, int K, cudaStream_t stream);

}  // namespace mt
