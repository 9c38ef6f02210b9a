// Dense bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   C[M, N] = A[M, K] * B[N, K]^T  (+ R[M, N])      fp32 accumulate
//
// A and B are row-major with K contiguous ("K-major"), which is the layout of
// a linear layer's forward product y = x W^T with W stored [out, in]. The
// backward products are expressed in the same form by the caller (dgrad with
// W^T, wgrad with transposed activations). This is the dense contraction of
// the stateless layer template (zhichai.net article, "以内存为中心的训练新范式"
// point 4; lqnn.cn article section 三: the per-layer compute the streamed
// weights feed).
//
// Design (one CTA per SM, persistent over output tiles):
//   * tile 128 x 256, K step 64 (one 128-byte swizzle row of bf16), 4-stage
//     shared-memory ring filled by TMA (warp 0, one elected lane);
//   * warp 1 allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//     one lane issues tcgen05.mma (M=128, N=256, K=16), committing each stage
//     back to the producer and each finished accumulator to the epilogue;
//   * warps 2-5 drain an accumulator with tcgen05.ld while the MMA warp fills
//     the other one, add the optional bf16 residual, round and store.
// Tiles are visited in groups of kGroupM row blocks so the A panel of a group
// stays in L2 while the group sweeps all column blocks.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "mt_internal.h"

namespace mt {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kGroupM = 32;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr size_t kSmemBytes = 1024 /*align slack*/ + (size_t)kStages * kStageBytes + 256 /*barriers*/;

struct GemmArgs {
  int M, N, K;
  void* C;
  long long ldc;
  const bf16* R;
  long long ldr;
  int c_f32;
  int num_mb, num_nb;
  int* err;
};

__device__ __forceinline__ void tile_coords(int t, int num_mb, int num_nb, int& mb, int& nb) {
  const int per_group = kGroupM * num_nb;
  const int group = t / per_group;
  const int first_m = group * kGroupM;
  const int gsz = min(kGroupM, num_mb - first_m);
  const int r = t - group * per_group;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

// A_MN / B_MN: the operand is stored MN-major in global memory (A as
// [K][M], B as [K][N], MN contiguous) and staged as 64 x 64 boxes.
constexpr uint32_t kBoxBytes = 64 * 64 * 2;  // one 64 MN x 64 K box

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_abt_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* tfull_bar = empty_bar + kStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = args.num_mb * args.num_nb;
  const int num_kb = (args.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 4 * 32);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, args.num_mb, args.num_nb, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, args.err)) { *abort_flag = 1; break; }
          uint8_t* sa = smem + stage * kStageBytes;
          uint8_t* sb = sa + kABytes;
          mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
          if (A_MN) {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j)
              tma_load_2d(sa + j * kBoxBytes, &tmap_a, mb * kBM + j * 64, kb * kBK, &full_bar[stage]);
          } else {
            tma_load_2d(sa, &tmap_a, kb * kBK, mb * kBM, &full_bar[stage]);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              tma_load_2d(sb + j * kBoxBytes, &tmap_b, nb * kBN + j * 64, kb * kBK, &full_bar[stage]);
          } else {
            tma_load_2d(sb, &tmap_b, kb * kBK, nb * kBN, &full_bar[stage]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty_bar[acc], (use & 1) ^ 1, args.err)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K step of 16: 32 bytes along a K-major row, or 16 K rows (2 KiB) down an MN-major box
            const uint64_t ad = A_MN ? smem_desc_mnmajor_sw128(sa + kk * 2048, kBoxBytes)
                                     : smem_desc_kmajor_sw128(sa + kk * 32);
            const uint64_t bd = B_MN ? smem_desc_mnmajor_sw128(sb + kk * 2048, kBoxBytes)
                                     : smem_desc_kmajor_sw128(sb + kk * 32);
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        tc_commit(&tfull_bar[acc]);
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5 cover TMEM lane quarters (warp % 4)
    const int q = warp & 3;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull_bar[acc], use & 1, args.err)) { *abort_flag = 1; break; }
      tc_fence_after();
      int mb, nb;
      tile_coords(t, args.num_mb, args.num_nb, mb, nb);
      const int row = mb * kBM + q * 32 + lane;
      const bool row_ok = row < args.M;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (uint32_t)(acc * kBN + c * 32) + ((uint32_t)(q * 32) << 16), r);
        tmem_ld_wait();
        const int col0 = nb * kBN + c * 32;
        if (!row_ok || col0 >= args.N) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        const bool full = col0 + 32 <= args.N;
        if (args.R != nullptr) {
          const bf16* rp = args.R + (long long)row * args.ldr + col0;
          if (full) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 u = reinterpret_cast<const uint4*>(rp)[j];
              float2 f0 = unpack_bf16x2(u.x), f1 = unpack_bf16x2(u.y), f2 = unpack_bf16x2(u.z),
                     f3 = unpack_bf16x2(u.w);
              v[j * 8 + 0] += f0.x; v[j * 8 + 1] += f0.y; v[j * 8 + 2] += f1.x; v[j * 8 + 3] += f1.y;
              v[j * 8 + 4] += f2.x; v[j * 8 + 5] += f2.y; v[j * 8 + 6] += f3.x; v[j * 8 + 7] += f3.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < args.N) v[i] += __bfloat162float(rp[i]);
          }
        }
        if (args.c_f32) {
          float* cp = reinterpret_cast<float*>(args.C) + (long long)row * args.ldc + col0;
          if (full) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(cp)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < args.N) cp[i] = v[i];
          }
        } else {
          bf16* cp = reinterpret_cast<bf16*>(args.C) + (long long)row * args.ldc + col0;
          if (full) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 u;
              u.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
              u.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
              u.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
              u.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
              reinterpret_cast<uint4*>(cp)[j] = u;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < args.N) cp[i] = __float2bfloat16_rn(v[i]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int g_num_sms = 0;

int get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(gemm_abt_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    cudaFuncSetAttribute(gemm_abt_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    cudaFuncSetAttribute(gemm_abt_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    cudaFuncSetAttribute(gemm_abt_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  });
  return g_encode ? 0 : -1;
}

// Row-major bf16 matrix [rows, cols] with row pitch `ld` elements, boxes of
// box_rows x box_cols with 128-byte swizzle (box_cols * 2 bytes = 128).
int make_tmap(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld, int box_rows,
              int box_cols) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

}  // namespace

int gemm_ex(const void* A, long long lda, int a_mn, const void* B, long long ldb, int b_mn, void* C, long long ldc,
            int c_f32, const void* R, long long ldr, int M, int N, int K, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0) return MT_EINVAL;
  if (M == 0 || N == 0) return MT_OK;
  if (K == 0) return MT_EINVAL;
  if (get_encode() != 0) return MT_ECUDA;
  // TMA: 16-byte aligned bases and row pitches; vector epilogue: 16-byte rows.
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(A) || !al16(B) || !al16(C) || (R && !al16(R))) return MT_EINVAL;
  if ((lda * 2) % 16 || (ldb * 2) % 16) return MT_EINVAL;
  if (a_mn ? lda < M : lda < K) return MT_EINVAL;
  if (b_mn ? ldb < N : ldb < K) return MT_EINVAL;
  if (ldc < N || (c_f32 ? (ldc % 4) : (ldc % 8))) return MT_EINVAL;
  if (R && (ldr % 8 || ldr < N)) return MT_EINVAL;
  CUtensorMap ta, tb;
  // K-major: rows = M (or N), cols = K, box kBM (kBN) x 64; MN-major: rows = K,
  // cols = M (or N), box 64 x 64.
  const int ea = a_mn ? make_tmap(&ta, A, K, M, lda, kBK, 64) : make_tmap(&ta, A, M, K, lda, kBM, kBK);
  const int eb = b_mn ? make_tmap(&tb, B, K, N, ldb, kBK, 64) : make_tmap(&tb, B, N, K, ldb, kBN, kBK);
  if (ea || eb) return MT_EINVAL;
  GemmArgs args;
  args.M = M;
  args.N = N;
  args.K = K;
  args.C = C;
  args.ldc = ldc;
  args.R = reinterpret_cast<const bf16*>(R);
  args.ldr = ldr;
  args.c_f32 = c_f32;
  args.num_mb = (M + kBM - 1) / kBM;
  args.num_nb = (N + kBN - 1) / kBN;
  args.err = device_error_word();
  const int tiles = args.num_mb * args.num_nb;
  const int grid = tiles < g_num_sms ? tiles : g_num_sms;
  if (!a_mn && !b_mn) gemm_abt_kernel<false, false><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  else if (!a_mn) gemm_abt_kernel<false, true><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  else if (!b_mn) gemm_abt_kernel<true, false><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  else gemm_abt_kernel<true, true><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

int gemm_abt(const void* A, long long lda, const void* B, long long ldb, void* C, long long ldc, int c_f32,
             const void* R, long long ldr, int M, int N, int K, cudaStream_t stream) {
  return gemm_ex(A, lda, 0, B, ldb, 0, C, ldc, c_f32, R, ldr, M, N, K, stream);
}

}  // namespace mt
