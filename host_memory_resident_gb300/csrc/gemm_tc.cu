// Dense bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   C[M, N] = A[M, K] * B[N, K]^T  (+ R[M, N])      fp32 accumulate
//
// C and the optional residual R are both bf16 or both fp32 (the decoder's
// residual stream is kept in fp32: x + O Wo^T and h + a Wdown^T add the
// fp32 accumulator to the fp32 stream and store fp32).
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
//   * warps 2-9 drain an accumulator with tcgen05.ld while the MMA warp fills
//     the other one (two warps per TMEM lane quarter, each taking half of the
//     tile's columns), add the optional residual and store (bf16 or fp32).
// Tiles are visited in groups of kGroupM row blocks so the A panel of a group
// stays in L2 while the group sweeps all column blocks.
//
// Fused epilogues. Each works on the fp32 accumulator and rounds to bf16 only
// what it stores, so the only bf16 roundings are those of the stored
// operands of later products:
//   * RoPE: the QKV projection rotates the q and k heads of its tile
//     (rotate-half pairs, position = row mod seq) from the fp32 products
//     and stores the rotated values;
//   * SwiGLU forward: the gate/up projection's B tile pairs 128 gate rows
//     with the matching 128 up rows, so the epilogue computes
//     a = silu(gate) * up from the fp32 gate and up and stores a and (for
//     the backward) gate | up;
//   * SwiGLU backward: the down projection's input gradient da never leaves
//     the SM; the epilogue turns the fp32 da and the stored gate | up into
//     d(gate) | d(up).
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
constexpr int kThreads = 320;       // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr size_t kSmemBytes = 1024 /*align slack*/ + (size_t)kStages * kStageBytes + 256 /*barriers*/;

enum : int { kEpiPlain = 0, kEpiRope = 1, kEpiSwigluFwd = 2, kEpiSwigluBwd = 3 };

struct GemmArgs {
  int M, N, K;
  void* C;
  long long ldc;
  const void* R;          // residual of C's type (bf16, or fp32 when c_f32)
  long long ldr;
  int c_f32;
  int num_mb, num_nb;
  int* err;
  // fused epilogues
  bf16* C2;               // SwiGLU forward: a [M, f]
  long long ldc2;
  const bf16* X;          // SwiGLU backward: gate | up [M, 2f]
  long long ldx;
  int f;                  // SwiGLU: ffn width (gate columns [0, f), up [f, 2f))
  const float* cos_t;     // RoPE tables [seq, hd/2]
  const float* sin_t;
  int rot_cols, hd, seq;  // RoPE: rotate columns [0, rot_cols) in heads of hd
  int st32;               // C (and C2) rows 32-byte aligned: whole-sector 32-byte stores
  // split K: work unit t is output tile t % tiles over K blocks
  // [s * kbps, (s + 1) * kbps) with s = t / tiles; slice s of the (fp32)
  // output starts split_stride elements after slice s - 1
  int splits, kbps;
  long long split_stride;
};

// One 32-byte store (a whole L2 sector); p 32-byte aligned.
__device__ __forceinline__ void st_global_32b(void* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t w4,
                                              uint32_t w5, uint32_t w6, uint32_t w7) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w0), "r"(w1), "r"(w2), "r"(w3),
               "r"(w4), "r"(w5), "r"(w6), "r"(w7)
               : "memory");
}

// 32 values as bf16 at p (16-byte aligned; 32-byte aligned when st32).
__device__ __forceinline__ void store_bf16x32(bf16* p, const float (&v)[32], int st32 = 0) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  if (st32) {
    st_global_32b(p, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
    st_global_32b(p + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      reinterpret_cast<uint4*>(p)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// The 32 gate and 32 up values (bf16, packed) of one row at ffn column col0
// for the SwiGLU-backward epilogue; zeros outside the matrix.
__device__ __forceinline__ void load_gate_up(const GemmArgs& a, int row, bool row_ok, int col0, uint4 (&g)[4],
                                             uint4 (&u)[4]) {
  if (row_ok && col0 < a.N) {
    const uint4* gp = reinterpret_cast<const uint4*>(a.X + (long long)row * a.ldx + col0);
    const uint4* up = reinterpret_cast<const uint4*>(a.X + (long long)row * a.ldx + a.f + col0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      g[j] = gp[j];
      u[j] = up[j];
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = u[j] = make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ void load_f32x32(const float* p, float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 u = reinterpret_cast<const float4*>(p)[j];
    v[4 * j + 0] = u.x; v[4 * j + 1] = u.y; v[4 * j + 2] = u.z; v[4 * j + 3] = u.w;
  }
}

__device__ __forceinline__ void tile_coords(int t, int num_mb, int num_nb, int& mb, int& nb);

// Work unit t: its output tile (mb, nb), split sp and K-block range [kb0, kb1).
__device__ __forceinline__ void unit_coords(int t, const GemmArgs& a, int num_kb, int& mb, int& nb, int& sp, int& kb0,
                                            int& kb1) {
  const int tiles = a.num_mb * a.num_nb;
  sp = t / tiles;
  tile_coords(t - sp * tiles, a.num_mb, a.num_nb, mb, nb);
  kb0 = sp * a.kbps;
  kb1 = min(num_kb, kb0 + a.kbps);
}

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

// out[m, n] = bf16(sum over s = 0 .. S-1, in order, of ws[s][m][n]); one
// thread per 8 columns. The split-K weight gradients end here.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int S, long long slice, int M, int N,
                                     bf16* __restrict__ out, long long ldo) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int nv = N >> 3;
  if (idx >= (long long)M * nv) return;
  const int row = (int)(idx / nv), v = (int)(idx % nv);
  const float* p = ws + (long long)row * N + v * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int sp = 0; sp < S; ++sp) {
    const float4 a = reinterpret_cast<const float4*>(p + sp * slice)[0];
    const float4 b = reinterpret_cast<const float4*>(p + sp * slice)[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  *reinterpret_cast<uint4*>(out + (long long)row * ldo + v * 8) =
      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                 pack_bf16x2(acc[6], acc[7]));
}

// W2: 256 x 256 tiles, each K step two products (A rows 0-127 and 128-255)
// sharing the B operand, into two 256-column accumulators that fill TMEM (so
// one tile's epilogue is not overlapped with the next tile's products) and a
// 3-stage ring of 64 KiB stages. Per 64-deep K block an SM then takes in 64
// KiB for 8 products instead of 48 KiB for 4.
template <bool W2>
struct TileCfg {
  static constexpr int kBMt = W2 ? 256 : kBM;
  static constexpr int kSt = W2 ? 3 : kStages;
  static constexpr uint32_t kAB = (uint32_t)kBMt * kBK * 2;
  static constexpr uint32_t kStB = kAB + kBBytes;
  static constexpr size_t kSmem = 1024 + (size_t)kSt * kStB + 256;
  static_assert(kSmem <= 232448, "shared memory per block");
};

template <bool A_MN, bool B_MN, int EPI, bool W2 = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_abt_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    GemmArgs args) {
  static_assert(!W2 || EPI == kEpiPlain, "256-row tiles only with the plain epilogue");
  using T = TileCfg<W2>;
  constexpr int kBM = T::kBMt;            // rows of a tile (shadows the 128-row default)
  constexpr int kStages = T::kSt;
  constexpr uint32_t kABytes = T::kAB;
  constexpr uint32_t kStageBytes = T::kStB;
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
  const int num_tiles = args.num_mb * args.num_nb * args.splits;  // work units
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
      mbar_init(&tempty_bar[a], kEpiWarps * 32);
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
        int mb, nb, sp, kb0, kb1;
        unit_coords(t, args, num_kb, mb, nb, sp, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
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
          if (EPI == kEpiSwigluFwd) {
            // 128 gate rows, then the 128 up rows of the same ffn columns
            tma_load_2d(sb, &tmap_b, kb * kBK, nb * (kBN / 2), &full_bar[stage]);
            tma_load_2d(sb + (kBN / 2) * kBK * 2, &tmap_b, kb * kBK, args.f + nb * (kBN / 2), &full_bar[stage]);
          } else if (B_MN) {
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
      constexpr uint32_t idesc = idesc_bf16_f32(128, kBN, A_MN, B_MN);  // one M = 128 product
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x, ++it) {
        // two accumulators used in turn, or (W2) one pair of them per tile
        const int acc = W2 ? 0 : (it & 1);
        const uint32_t use = W2 ? (uint32_t)it : (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty_bar[acc], (use & 1) ^ 1, args.err)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        int mb, nb, sp, kb0, kb1;
        unit_coords(t, args, num_kb, mb, nb, sp, kb0, kb1);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
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
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
            if (W2)  // A rows 128-255 start 16 KiB into the stage in both layouts
              tc_mma_bf16(d_tmem + (uint32_t)kBN, desc_advance(ad, kABytes / 2), bd, idesc,
                          (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        tc_commit(&tfull_bar[acc]);
      }
    }
  } else {
    // ---------------- epilogue: warps 2..9; warp % 4 is the TMEM lane quarter,
    // (warp - 2) / 4 the half of the tile's columns (or heads) it stores
    const int q = warp & 3;
    const int hs = (warp - 2) >> 2;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int acc = W2 ? 0 : (it & 1);
      const uint32_t use = W2 ? (uint32_t)it : (uint32_t)(it >> 1);
      int mb, nb, sp, kb0, kb1;
      unit_coords(t, args, (args.K + kBK - 1) / kBK, mb, nb, sp, kb0, kb1);
      // W2: warp half hs reads the accumulator of tile rows hs * 128 + [0, 128)
      // (all 256 columns); otherwise half hs of the columns of all 128 rows
      const int row = mb * kBM + (W2 ? hs * 128 : 0) + q * 32 + lane;
      const bool row_ok = row < args.M;
      // SwiGLU backward: the gate | up values of this warp's first chunk do
      // not depend on the accumulator; their loads overlap the wait for it
      uint4 xg[4], xu[4];
      const int xc0 = hs * (kBN / 64);
      if (EPI == kEpiSwigluBwd) load_gate_up(args, row, row_ok, nb * kBN + xc0 * 32, xg, xu);
      if (!mbar_wait(&tfull_bar[acc], use & 1, args.err)) { *abort_flag = 1; break; }
      tc_fence_after();
      const uint32_t tacc = tmem_base + (uint32_t)((W2 ? hs : acc) * kBN) + ((uint32_t)(q * 32) << 16);
      if (EPI == kEpiRope) {
        // heads of hd columns; dims i and i + hd/2 of a head form a pair, so
        // chunk j of the first half pairs with chunk j of the second half
        const int hd = args.hd, half = hd >> 1;
        const int pos = row_ok ? row % args.seq : 0;
        const int nh = kBN / hd;  // heads per tile, split between the two halves
#pragma unroll 1
        for (int hb = hs * (nh / 2); hb < (hs + 1) * (nh / 2); ++hb) {
          const int col_h = nb * kBN + hb * hd;
#pragma unroll 1
          for (int j = 0; j < hd / 64; ++j) {
            __syncwarp();
            uint32_t ra[32], rb[32];
            tmem_ld_32x32b_x32(tacc + (uint32_t)(hb * hd + j * 32), ra);
            tmem_ld_32x32b_x32(tacc + (uint32_t)(hb * hd + j * 32 + half), rb);
            tmem_ld_wait();
            if (!row_ok || col_h >= args.N) continue;
            float va[32], vb[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              va[i] = __uint_as_float(ra[i]);
              vb[i] = __uint_as_float(rb[i]);
            }
            if (col_h < args.rot_cols) {
              float cs[32], sn[32];
              load_f32x32(args.cos_t + (long long)pos * half + j * 32, cs);
              load_f32x32(args.sin_t + (long long)pos * half + j * 32, sn);
#pragma unroll
              for (int i = 0; i < 32; ++i) rope_pair(va[i], vb[i], cs[i], sn[i], va[i], vb[i]);
            }
            bf16* cp = reinterpret_cast<bf16*>(args.C) + (long long)row * args.ldc + col_h + j * 32;
            store_bf16x32(cp, va, args.st32);
            store_bf16x32(cp + half, vb, args.st32);
          }
        }
      } else if (EPI == kEpiSwigluFwd) {
        // accumulator columns [0, 128) are gate, [128, 256) up, of ffn
        // columns nb * 128 + [0, 128)
#pragma unroll 1
        for (int c = hs * (kBN / 128); c < (hs + 1) * (kBN / 128); ++c) {
          __syncwarp();
          uint32_t rg[32], ru[32];
          tmem_ld_32x32b_x32(tacc + (uint32_t)(c * 32), rg);
          tmem_ld_32x32b_x32(tacc + (uint32_t)(kBN / 2 + c * 32), ru);
          tmem_ld_wait();
          if (!row_ok) continue;
          const int fc = nb * (kBN / 2) + c * 32;
          float g[32], u[32], a[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            g[i] = __uint_as_float(rg[i]);
            u[i] = __uint_as_float(ru[i]);
            a[i] = swiglu_fwd_elem(g[i], u[i]);
          }
          bf16* cp = reinterpret_cast<bf16*>(args.C) + (long long)row * args.ldc;
          store_bf16x32(cp + fc, g, args.st32);
          store_bf16x32(cp + args.f + fc, u, args.st32);
          store_bf16x32(args.C2 + (long long)row * args.ldc2 + fc, a, args.st32);
        }
      } else if (EPI == kEpiSwigluBwd) {
        // the tile is da for ffn columns nb * 256 + [0, 256); the next
        // chunk's gate | up loads are issued before this chunk's arithmetic
#pragma unroll 1
        for (int c = xc0; c < xc0 + kBN / 64; ++c) {
          __syncwarp();
          uint4 ng[4], nu[4];
          if (c + 1 < xc0 + kBN / 64) load_gate_up(args, row, row_ok, nb * kBN + (c + 1) * 32, ng, nu);
          uint32_t r[32];
          tmem_ld_32x32b_x32(tacc + (uint32_t)(c * 32), r);
          tmem_ld_wait();
          const int col0 = nb * kBN + c * 32;
          if (row_ok && col0 < args.N) {
            float dg[32], du[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t gw[4] = {xg[j].x, xg[j].y, xg[j].z, xg[j].w};
              const uint32_t uw[4] = {xu[j].x, xu[j].y, xu[j].z, xu[j].w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 g2 = unpack_bf16x2(gw[k]), u2 = unpack_bf16x2(uw[k]);
                const int i = 8 * j + 2 * k;
                swiglu_bwd_elem(__uint_as_float(r[i]), g2.x, u2.x, dg[i], du[i]);
                swiglu_bwd_elem(__uint_as_float(r[i + 1]), g2.y, u2.y, dg[i + 1], du[i + 1]);
              }
            }
            bf16* cp = reinterpret_cast<bf16*>(args.C) + (long long)row * args.ldc + col0;
            store_bf16x32(cp, dg, args.st32);
            store_bf16x32(cp + args.f, du, args.st32);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            xg[j] = ng[j];
            xu[j] = nu[j];
          }
        }
      } else {
#pragma unroll 1
        for (int c = W2 ? 0 : hs * (kBN / 64); c < (W2 ? kBN / 32 : (hs + 1) * (kBN / 64)); ++c) {
          __syncwarp();
          uint32_t r[32];
          tmem_ld_32x32b_x32(tacc + (uint32_t)(c * 32), r);
          tmem_ld_wait();
          const int col0 = nb * kBN + c * 32;
          if (!row_ok || col0 >= args.N) continue;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          const bool full = col0 + 32 <= args.N;
          if (args.R != nullptr && args.c_f32) {
            const float* rp = reinterpret_cast<const float*>(args.R) + (long long)row * args.ldr + col0;
            if (full) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 u = reinterpret_cast<const float4*>(rp)[j];
                v[4 * j + 0] += u.x; v[4 * j + 1] += u.y; v[4 * j + 2] += u.z; v[4 * j + 3] += u.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (col0 + i < args.N) v[i] += rp[i];
            }
          } else if (args.R != nullptr) {
            const bf16* rp = reinterpret_cast<const bf16*>(args.R) + (long long)row * args.ldr + col0;
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
            float* cp = reinterpret_cast<float*>(args.C) + sp * args.split_stride + (long long)row * args.ldc + col0;
            if (full && args.st32) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_global_32b(cp + 8 * j, __float_as_uint(v[8 * j]), __float_as_uint(v[8 * j + 1]),
                              __float_as_uint(v[8 * j + 2]), __float_as_uint(v[8 * j + 3]),
                              __float_as_uint(v[8 * j + 4]), __float_as_uint(v[8 * j + 5]),
                              __float_as_uint(v[8 * j + 6]), __float_as_uint(v[8 * j + 7]));
            } else if (full) {
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
              store_bf16x32(cp, v, args.st32);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (col0 + i < args.N) cp[i] = __float2bfloat16_rn(v[i]);
            }
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
    const int sm = (int)kSmemBytes;
    cudaFuncSetAttribute(gemm_abt_kernel<false, false, kEpiPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(gemm_abt_kernel<false, true, kEpiPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(gemm_abt_kernel<true, false, kEpiPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(gemm_abt_kernel<true, true, kEpiPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    const int sw = (int)TileCfg<true>::kSmem;
    cudaFuncSetAttribute(gemm_abt_kernel<false, false, kEpiPlain, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         sw);
    cudaFuncSetAttribute(gemm_abt_kernel<false, true, kEpiPlain, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         sw);
    cudaFuncSetAttribute(gemm_abt_kernel<true, false, kEpiPlain, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         sw);
    cudaFuncSetAttribute(gemm_abt_kernel<true, true, kEpiPlain, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         sw);
    cudaFuncSetAttribute(gemm_abt_kernel<false, false, kEpiRope>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(gemm_abt_kernel<false, false, kEpiSwigluFwd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         sm);
    cudaFuncSetAttribute(gemm_abt_kernel<false, true, kEpiSwigluBwd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         sm);
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

namespace {

int g_tile_policy = 0;  // 0: the choice below; 1: 128-row tiles; 2: 256-row tiles where allowed

// Whether a plain product takes 256 x 256 tiles: time in units of one
// 128 x 256 x 64 tile step, waves of 152 tiles times K blocks; a 256-row
// tile step costs 2 x 0.97 of them. Measured on GB300 (CUDA events, both
// shapes forced): the wide tiles gain 2-4% where the wave counts match
// (8192 x 8192 x 4096, 16384 x 11264 x 2048, 16384 x 32000 x 2048) and lose
// 3-16% where halving the tile count leaves a thin last wave (16384 x 2048
// by 2048 or 5632, 16384 x 2560 x 2048).
bool wide_tiles(int M, int N, int K) {
  if (g_tile_policy != 0) return g_tile_policy == 2;
  constexpr int kSMs = 152;
  const long long t128 = (long long)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const long long t256 = (long long)((M + 255) / 256) * ((N + kBN - 1) / kBN);
  const double c128 = (double)((t128 + kSMs - 1) / kSMs);
  const double c256 = (double)((t256 + kSMs - 1) / kSMs) * 2.0 * 0.97;
  return c256 < c128 * 0.995;
}

// Validates the operands, builds the tensor maps and launches one GEMM with
// the epilogue `epi` (whose extra fields `args` already holds).
int launch(int epi, const void* A, long long lda, int a_mn, const void* B, long long ldb, int b_mn, GemmArgs& args,
           cudaStream_t stream) {
  const int M = args.M, N = args.N, K = args.K;
  if (M < 0 || N < 0 || K < 0) return MT_EINVAL;
  if (M == 0 || N == 0) return MT_OK;
  if (K == 0) return MT_EINVAL;
  if (get_encode() != 0) return MT_ECUDA;
  // TMA: 16-byte aligned bases and row pitches; vector epilogue: 16-byte rows.
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(A) || !al16(B) || !al16(args.C) || (args.R && !al16(args.R))) return MT_EINVAL;
  if ((lda * 2) % 16 || (ldb * 2) % 16) return MT_EINVAL;
  if (a_mn ? lda < M : lda < K) return MT_EINVAL;
  if (b_mn ? ldb < N : ldb < K) return MT_EINVAL;
  if (args.ldc < N || (args.c_f32 ? (args.ldc % 4) : (args.ldc % 8))) return MT_EINVAL;
  if (args.R && (args.ldr % 8 || args.ldr < N)) return MT_EINVAL;
  if (args.R && args.splits > 1) return MT_EINVAL;
  // split K: every split gets at least one K block
  const int num_kb = (K + kBK - 1) / kBK;
  if (args.splits < 1) args.splits = 1;
  args.kbps = (num_kb + args.splits - 1) / args.splits;
  args.splits = (num_kb + args.kbps - 1) / args.kbps;
  // 256 x 256 tiles for plain unsplit products with enough of them
  const bool w2 = epi == kEpiPlain && args.splits == 1 && wide_tiles(M, N, K);
  const int bm = w2 ? 256 : kBM;
  CUtensorMap ta, tb;
  // K-major: rows = M (or N), cols = K, box bm (kBN) x 64; MN-major: rows = K,
  // cols = M (or N), box 64 x 64. The SwiGLU forward loads its B tile as two
  // 128-row boxes (gate rows, then up rows).
  const int ea = a_mn ? make_tmap(&ta, A, K, M, lda, kBK, 64) : make_tmap(&ta, A, M, K, lda, bm, kBK);
  const int eb = b_mn ? make_tmap(&tb, B, K, N, ldb, kBK, 64)
                      : make_tmap(&tb, B, N, K, ldb, epi == kEpiSwigluFwd ? kBN / 2 : kBN, kBK);
  if (ea || eb) return MT_EINVAL;
  args.num_mb = (M + bm - 1) / bm;
  args.num_nb = (N + kBN - 1) / kBN;
  args.err = device_error_word();
  auto al32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; };
  args.st32 = al32(args.C) && (args.c_f32 ? args.ldc % 8 == 0 : args.ldc % 16 == 0) &&
              (args.C2 == nullptr || (al32(args.C2) && args.ldc2 % 16 == 0)) ? 1 : 0;
  const int tiles = args.num_mb * args.num_nb * args.splits;
  const int grid = tiles < g_num_sms ? tiles : g_num_sms;
  if (epi == kEpiRope) {
    if (a_mn || b_mn) return MT_EINVAL;
    gemm_abt_kernel<false, false, kEpiRope><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  } else if (epi == kEpiSwigluFwd) {
    if (a_mn || b_mn) return MT_EINVAL;
    gemm_abt_kernel<false, false, kEpiSwigluFwd><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  } else if (epi == kEpiSwigluBwd) {
    if (a_mn || !b_mn) return MT_EINVAL;
    gemm_abt_kernel<false, true, kEpiSwigluBwd><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  } else if (w2) {
    constexpr size_t sw = TileCfg<true>::kSmem;
    if (!a_mn && !b_mn)
      gemm_abt_kernel<false, false, kEpiPlain, true><<<grid, kThreads, sw, stream>>>(ta, tb, args);
    else if (!a_mn)
      gemm_abt_kernel<false, true, kEpiPlain, true><<<grid, kThreads, sw, stream>>>(ta, tb, args);
    else if (!b_mn)
      gemm_abt_kernel<true, false, kEpiPlain, true><<<grid, kThreads, sw, stream>>>(ta, tb, args);
    else
      gemm_abt_kernel<true, true, kEpiPlain, true><<<grid, kThreads, sw, stream>>>(ta, tb, args);
  } else if (!a_mn && !b_mn) {
    gemm_abt_kernel<false, false, kEpiPlain><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  } else if (!a_mn) {
    gemm_abt_kernel<false, true, kEpiPlain><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  } else if (!b_mn) {
    gemm_abt_kernel<true, false, kEpiPlain><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  } else {
    gemm_abt_kernel<true, true, kEpiPlain><<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, args);
  }
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

GemmArgs base_args(int M, int N, int K, void* C, long long ldc, int c_f32) {
  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = C;
  a.ldc = ldc;
  a.c_f32 = c_f32;
  a.splits = 1;
  return a;
}

bool al16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int gemm_tile_policy(int policy) {
  if (policy < 0 || policy > 2) return MT_EINVAL;
  g_tile_policy = policy;
  return MT_OK;
}

int gemm_ex(const void* A, long long lda, int a_mn, const void* B, long long ldb, int b_mn, void* C, long long ldc,
            int c_f32, const void* R, long long ldr, int M, int N, int K, cudaStream_t stream) {
  GemmArgs args = base_args(M, N, K, C, ldc, c_f32);
  args.R = R;
  args.ldr = ldr;
  return launch(kEpiPlain, A, lda, a_mn, B, ldb, b_mn, args, stream);
}

int splitk_factor(int M, int N, int K) {
  // Output tiles that leave a large share of the 152 SMs idle in the last
  // wave are split along K when that shortens the launch: time in K-block
  // units, waves x K blocks per split, plus the reduction's bytes at HBM
  // speed (one K block of one tile: about 0.37 us; HBM: about 6.5 TB/s).
  constexpr int kSMs = 152;
  constexpr double kKBlockUs = 0.371, kHbmBytesPerUs = 6.5e6;
  const long long tiles = (long long)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const int num_kb = (K + kBK - 1) / kBK;
  if (N % 8 || tiles >= 4 * kSMs || num_kb < 16) return 1;
  int best = 1;
  double best_us = 0.0;
  for (int sp = 1; sp <= 4; ++sp) {
    const int kbps = (num_kb + sp - 1) / sp;
    const int spe = (num_kb + kbps - 1) / kbps;
    const double waves = (double)((tiles * spe + kSMs - 1) / kSMs);
    double us = waves * kbps * kKBlockUs;
    if (spe > 1) us += (double)(spe * 4 + 2) * M * N / kHbmBytesPerUs;
    if (sp == 1 || us < best_us) {
      best = spe;
      best_us = us;
    }
  }
  return best;
}

size_t splitk_ws_elems(int M, int N) {
  const long long tiles = (long long)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  return (N % 8 || tiles >= 4 * 152) ? 0 : (size_t)4 * M * N;
}

int gemm_wgrad(const void* A, long long lda, int a_mn, const void* B, long long ldb, int b_mn, void* C, long long ldc,
               int M, int N, int K, float* ws, size_t ws_elems, cudaStream_t stream) {
  const int sp = splitk_factor(M, N, K);
  if (sp <= 1 || ws == nullptr || (size_t)sp * M * N > ws_elems || ldc % 8 ||
      (reinterpret_cast<uintptr_t>(C) & 15))
    return gemm_ex(A, lda, a_mn, B, ldb, b_mn, C, ldc, 0, nullptr, 0, M, N, K, stream);
  GemmArgs args = base_args(M, N, K, ws, N, 1);
  args.splits = sp;
  args.split_stride = (long long)M * N;
  const int r = launch(kEpiPlain, A, lda, a_mn, B, ldb, b_mn, args, stream);
  if (r != MT_OK) return r;
  const long long threads = (long long)M * (N / 8);
  splitk_reduce_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(ws, args.splits, args.split_stride, M, N,
                                                                              reinterpret_cast<bf16*>(C), ldc);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

int gemm_rope(const void* A, long long lda, const void* B, long long ldb, void* C, long long ldc, int M, int N, int K,
              const float* cos_t, const float* sin_t, int rot_cols, int hd, int seq, cudaStream_t stream) {
  if (hd <= 0 || hd % 64 || (kBN / 2) % hd || N % hd || rot_cols < 0 || rot_cols % hd || rot_cols > N || seq <= 0 ||
      !cos_t || !sin_t || ldc % 8)
    return MT_EINVAL;
  GemmArgs args = base_args(M, N, K, C, ldc, 0);
  args.cos_t = cos_t;
  args.sin_t = sin_t;
  args.rot_cols = rot_cols;
  args.hd = hd;
  args.seq = seq;
  return launch(kEpiRope, A, lda, 0, B, ldb, 0, args, stream);
}

int gemm_swiglu_fwd(const void* A, long long lda, const void* W, long long ldw, void* gu, long long ldgu, void* a,
                    long long lda_out, int M, int f, int K, cudaStream_t stream) {
  if (f <= 0 || f % (kBN / 2) || ldgu < 2LL * f || ldgu % 8 || lda_out < f || lda_out % 8 || !al16p(a))
    return MT_EINVAL;
  GemmArgs args = base_args(M, 2 * f, K, gu, ldgu, 0);
  args.C2 = reinterpret_cast<bf16*>(a);
  args.ldc2 = lda_out;
  args.f = f;
  return launch(kEpiSwigluFwd, A, lda, 0, W, ldw, 0, args, stream);
}

int gemm_swiglu_bwd(const void* dy, long long lddy, const void* W, long long ldw, const void* gu, long long ldgu,
                    void* dgu, long long lddgu, int M, int f, int K, cudaStream_t stream) {
  if (f <= 0 || f % 32 || ldgu < 2LL * f || ldgu % 8 || lddgu < 2LL * f || lddgu % 8 || !al16p(gu)) return MT_EINVAL;
  GemmArgs args = base_args(M, f, K, dgu, lddgu, 0);
  args.X = reinterpret_cast<const bf16*>(gu);
  args.ldx = ldgu;
  args.f = f;
  return launch(kEpiSwigluBwd, dy, lddy, 0, W, ldw, 1, args, stream);
}

int gemm_abt(const void* A, long long lda, const void* B, long long ldb, void* C, long long ldc, int c_f32,
             const void* R, long long ldr, int M, int N, int K, cudaStream_t stream) {
  return gemm_ex(A, lda, 0, B, ldb, 0, C, ldc, c_f32, R, ldr, M, N, K, stream);
}

}  // namespace mt
