// Causal grouped-query attention forward on the 5th-generation tensor cores.
//
// One CTA per (128-query tile, head, batch), warp-specialised:
//   warp 0   TMA producer: Q once, then K and V tiles of 128 keys into a
//            two-stage ring (3-D tensor map over the qkv rows of one
//            sequence, so rows past its end arrive as zeros);
//   warp 1   allocates TMEM and issues tcgen05.mma:
//              S_j = Q K_j^T      (M 128, N 128, K = hd)  into one of two
//                                  128-column TMEM buffers,
//              O  += P_j V_j      (M 128, N = hd, K 128) with P from shared
//                                  memory and V read MN-major in place;
//   warps 2-9 softmax: two threads per query row (one TMEM lane), each
//            reading half of the row's 128 scores with tcgen05.ld; the halves
//            combine their max and sum through shared memory. The causal mask
//            and the online softmax run in fp32 (log2 domain); P is written as
//            bf16 into 128-byte-swizzled shared memory (each half fills one
//            64-key box). O is rescaled in TMEM only when a row's running
//            maximum grows by more than 2^8, so P stays below 256 and the
//            final O / l is unchanged.
// This is the attention of the stateless layer template (zhichai.net
// article, "以内存为中心的训练新范式" point 4); streaming the keys in tiles keeps
// its memory O(s), the basis of the long-context runs the travelaiplan blog
// describes (section 3, 7B at 512K context).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "mt_internal.h"

namespace mt {
namespace {

constexpr int kQ = 128;                 // queries per CTA (MMA M)
constexpr int kKV = 128;                // keys per tile
constexpr int kThr = 320;               // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr uint32_t kBox = 128 * 128;    // one 64-column x 128-row bf16 box (16 KiB)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;        // rescale O only when the max grows by > 2^8

template <int HD>
struct TcCfg {
  static constexpr int kBoxes = HD / 64;
  static constexpr uint32_t kTile = kBoxes * kBox;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kTile;
  static constexpr uint32_t kVOff = kKOff + 2 * kTile;
  static constexpr uint32_t kPOff = kVOff + 2 * kTile;
  static constexpr uint32_t kPBuf = 2 * kBox;          // one P tile (128 keys)
  static constexpr uint32_t kBarOff = kPOff + 2 * kPBuf;  // two P buffers
  static constexpr uint32_t kRedOff = kBarOff + 128;  // [2 halves][128 rows] floats for max / sum
  // at least 120 KiB so that one CTA (and its 512 TMEM columns) owns the SM
  static constexpr size_t kSmemRaw = 1024 + kRedOff + 2 * 128 * 4;
  static constexpr size_t kSmem = kSmemRaw < 122880 ? 122880 : kSmemRaw;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int HD>
__global__ void __launch_bounds__(kThr, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, bf16* __restrict__ o, long long ldo,
                       float* __restrict__ lse, int s, int H, int Hkv, int* err) {
  using C = TcCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* s_empty = bars + 7;   // [2]
  uint64_t* p_full = bars + 9;    // [2]
  uint64_t* p_empty = bars + 11;  // [2]: PV with that P buffer finished (O current)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 13);

  const int nqt = (s + kQ - 1) / kQ;
  const int qt = nqt - 1 - blockIdx.x;  // heaviest tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (H / Hkv);
  const int q0 = qt * kQ;
  const int n_kv = qt + 1;  // causal: key tiles 0..qt
  const int qcol = h * HD, kcol = (H + g) * HD, vcol = (H + Hkv + g) * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm);
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 256);
      mbar_init(&p_empty[i], 1);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ loads
      mbar_arrive_expect_tx(q_full, C::kTile);
      for (int bx = 0; bx < C::kBoxes; ++bx)
        tma_load_3d(sm + C::kQOff + bx * kBox, &tm, qcol + bx * 64, q0, b, q_full);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, err)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::kTile);
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_3d(sm + C::kKOff + st * C::kTile + bx * kBox, &tm, kcol + bx * 64, j * kKV, b, &kv_full[st]);
          tma_load_3d(sm + C::kVOff + st * C::kTile + bx * kBox, &tm, vcol + bx * 64, j * kKV, b, &kv_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMAs
      constexpr uint32_t idesc_s = idesc_bf16_f32(kQ, kKV, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kQ, HD, false, true);
      const uint32_t sQ = smem_u32(sm + C::kQOff);
      const uint32_t sP = smem_u32(sm + C::kPOff);
      bool ok = mbar_wait(q_full, 0, err);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&kv_full[st], (j >> 1) & 1, err)) return false;
        if (!mbar_wait(&s_empty[st], ((j >> 1) & 1) ^ 1, err)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + C::kKOff + st * C::kTile);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          tc_mma_bf16(tS[st], smem_desc_kmajor_sw128(sQ + off), smem_desc_kmajor_sw128(sK + off), idesc_s,
                      kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv && !issue_s(j + 1)) break;
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, err)) break;
        tc_fence_after();
        const uint32_t sV = smem_u32(sm + C::kVOff + (j & 1) * C::kTile);
        const uint32_t sPj = sP + (j & 1) * C::kPBuf;
#pragma unroll
        for (int kk = 0; kk < kKV / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
          tc_mma_bf16(tO, smem_desc_kmajor_sw128(sPj + aoff), smem_desc_mnmajor_sw128(sV + kk * 2048, kBox), idesc_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&p_empty[j & 1]);
        tc_commit(&kv_empty[j & 1]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                 // TMEM lane quarter
    const int half = (warp - 2) >> 2;       // which 64 keys / which half of O
    const int row = q * 32 + lane;
    const int qpos = q0 + row;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc = rsqrtf((float)HD) * kLog2e;
    float* red = reinterpret_cast<float*>(sm + C::kRedOff);  // [2][128]
    float m_ref = -INFINITY, l = 0.f;
    uint8_t* sP = sm + C::kPOff + half * kBox;
    constexpr int kOCols = HD / 2;          // O columns this thread rescales / stores
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory"); };
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int st = j & 1;
      if (!mbar_wait(&s_full[st], (j >> 1) & 1, err)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld_32x32b_x32(tS[st] + lane_off + half * 64 + c * 32, r[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s_empty[st]);
      // raw scores; only the diagonal tile (the last one) needs the causal mask
      float v[64];
      float mraw = -INFINITY;
      if (j == n_kv - 1) {
        const int kbase = j * kKV + half * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = (kbase + c * 32 + i > qpos) ? -INFINITY : __uint_as_float(r[c][i]);
            v[c * 32 + i] = x;
            mraw = fmaxf(mraw, x);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[c * 32 + i] = __uint_as_float(r[c][i]);
            mraw = fmaxf(mraw, v[c * 32 + i]);
          }
      }
      float mx = mraw * sc;  // row max in the scaled log2 domain (sc > 0)
      red[half * 128 + row] = mx;
      pair_sync();
      mx = fmaxf(mx, red[(half ^ 1) * 128 + row]);
      if (j == 0) m_ref = mx;
      const bool need = j > 0 && mx > m_ref + kRescale;
      const float m_use = need ? mx : m_ref;
      // P = exp2(v - m_use) as packed bf16, computed before any wait
      uint32_t pk[32];
      float lt0 = 0.f, lt1 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2_approx(fmaf(v[2 * i], sc, -m_use));
        const float p1 = ex2_approx(fmaf(v[2 * i + 1], sc, -m_use));
        lt0 += p0;
        lt1 += p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      const float lt = lt0 + lt1;
      // this P buffer was last read by PV_{j-2}
      if (j >= 2 && !mbar_wait(&p_empty[st], ((j >> 1) - 1) & 1, err)) { ok = false; break; }
      if (__any_sync(0xffffffffu, need)) {
        // O must be current (PV_{j-1} finished) before it is rescaled
        if (!mbar_wait(&p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, err)) { ok = false; break; }
        tc_fence_after();
        const float factor = need ? exp2f(m_ref - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t ov[32];
          const uint32_t ta = tO + lane_off + half * kOCols + c * 32;
          tmem_ld_32x32b_x32(ta, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * factor);
          tmem_st_32x32b_x32(ta, ov);
        }
        tmem_st_wait();
        if (need) {
          l *= factor;
          m_ref = mx;
        }
      } else if (j >= 2) {
        tc_fence_after();
      }
      l += lt;
      // write this half's 64-key box of P buffer st (128-byte swizzle)
      uint8_t* sPb = sP + st * C::kPBuf;
      const uint32_t rsw = (uint32_t)(row & 7);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 u = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        *reinterpret_cast<uint4*>(sPb + row * 128 + (((uint32_t)c ^ rsw) * 16)) = u;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[st]);
      pair_sync();  // both halves read red[] before it is rewritten
    }
    if (ok) {
      red[half * 128 + row] = l;
      pair_sync();
      l += red[(half ^ 1) * 128 + row];
    }
    if (ok && mbar_wait(&p_empty[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1, err)) {
      tc_fence_after();
      const float inv = 1.f / l;
      bf16* orow = o + ((long long)b * s + qpos) * ldo + (long long)h * HD + half * kOCols;
#pragma unroll 1
      for (int c = 0; c < kOCols / 32; ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tO + lane_off + half * kOCols + c * 32, ov);
        tmem_ld_wait();
        if (qpos < s) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(ov[8 * k + 0]) * inv, __uint_as_float(ov[8 * k + 1]) * inv);
            u.y = pack_bf16x2(__uint_as_float(ov[8 * k + 2]) * inv, __uint_as_float(ov[8 * k + 3]) * inv);
            u.z = pack_bf16x2(__uint_as_float(ov[8 * k + 4]) * inv, __uint_as_float(ov[8 * k + 5]) * inv);
            u.w = pack_bf16x2(__uint_as_float(ov[8 * k + 6]) * inv, __uint_as_float(ov[8 * k + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * k) = u;
          }
        }
      }
      if (qpos < s && half == 0) lse[((long long)b * H + h) * s + qpos] = (m_ref + log2f(l)) / kLog2e;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_once;

void init_once() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  cudaFuncSetAttribute(attn_fwd_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<64>::kSmem);
  cudaFuncSetAttribute(attn_fwd_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<128>::kSmem);
}

}  // namespace

// qkv bf16 [B*s, ld]; see mt_k_attn_fwd. hd must be 64 or 128.
int attn_fwd_tc(const void* qkv, long long ld, void* o, long long ldo, float* lse, int B, int s, int H, int Hkv,
                int hd, cudaStream_t stream) {
  std::call_once(g_once, init_once);
  if (!g_enc) return MT_ECUDA;
  if (hd != 64 && hd != 128) return MT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(qkv) & 15) || ld % 8 || ldo % 8 || (reinterpret_cast<uintptr_t>(o) & 15))
    return MT_EINVAL;
  CUtensorMap tm;
  cuuint64_t dims[3] = {(cuuint64_t)ld, (cuuint64_t)s, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)s * ld * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kKV, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (g_enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MT_EINVAL;
  dim3 grid((s + kQ - 1) / kQ, H, B);
  int* err = device_error_word();
  if (hd == 64)
    attn_fwd_tc_kernel<64><<<grid, kThr, TcCfg<64>::kSmem, stream>>>(tm, (bf16*)o, ldo, lse, s, H, Hkv, err);
  else
    attn_fwd_tc_kernel<128><<<grid, kThr, TcCfg<128>::kSmem, stream>>>(tm, (bf16*)o, ldo, lse, s, H, Hkv, err);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

}  // namespace mt
