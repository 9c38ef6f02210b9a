// Causal grouped-query attention, forward and backward, KV streamed through
// shared memory in tiles (memory O(s) per head, no s x s matrix), which is
// what lets the long-context configuration run one layer at a time (the
// travelaiplan blog "單卡也能練 100B+", section 3 on 7B at 512K context, and
// the zhichai.net article, "MegaTrain 的性能与能力", long context as a
// by-product of the layer-wise design).
//
// Forward: one CTA per (64-query tile, head, batch); 4 warps x 16 query rows;
// online softmax in fp32; writes O (bf16) and the row log-sum-exp (fp32).
// Backward (deterministic, no float atomics):
//   delta  = rowsum(dO * O)                                  (per row, head)
//   dK, dV : one CTA per (key tile, KV head, batch), looping over the query
//            heads of the group and the query tiles at or after the diagonal;
//   dQ     : one CTA per (query tile, head, batch), looping over key tiles.
// Matrix products use the bf16 m16n8k16 tensor-core instruction with fp32
// accumulation; tiles are staged with cp.async into 128-byte-row swizzled
// shared memory and read with ldmatrix.
#include <cfloat>

#include "common.cuh"
#include "mt_internal.h"

namespace mt {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Element offset of (row, col) in a [rows][HD] bf16 tile whose 16-byte chunks
// are XOR-swizzled by row (conflict-free ldmatrix for HD >= 64).
template <int HD>
__device__ __forceinline__ int swz(int row, int col) {
  if constexpr (HD >= 64) {
    const int chunk = (col >> 3) ^ (row & 7);
    return row * HD + (chunk << 3) + (col & 7);
  } else {
    return row * HD + col;
  }
}

// Load `rows` x HD bf16 rows from global (row pitch ld, first row r0 of a
// sequence of length s; rows >= s are zero-filled) into a swizzled tile.
template <int HD, int NT>
__device__ __forceinline__ void load_tile(bf16* sm, const bf16* g, long long ld, int r0, int rows, int s) {
  constexpr int CH = HD / 8;  // 16-byte chunks per row
  for (int i = threadIdx.x; i < rows * CH; i += NT) {
    const int r = i / CH, c = (i % CH) * 8;
    const bool ok = r0 + r < s;
    const bf16* src = g + (long long)(ok ? r0 + r : 0) * ld + c;
    cp_async_16(smem_u32(sm + swz<HD>(r, c)), src, ok);
  }
}

// A fragment (16 x 16) of rows [r0, r0+16) and cols [k0, k0+16) of a tile.
template <int HD>
__device__ __forceinline__ void lds_a(const bf16* sm, int r0, int k0, uint32_t (&a)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
  const int c = k0 + 8 * (lane >> 4);
  ldmatrix_x4(smem_u32(sm + swz<HD>(r, c)), a[0], a[1], a[2], a[3]);
}

// B fragments for two n-tiles (rows n0..n0+15 of the tile are the n index,
// cols k0..k0+15 the k index): b[0],b[1] n-tile 0; b[2],b[3] n-tile 1.
template <int HD>
__device__ __forceinline__ void lds_b(const bf16* sm, int n0, int k0, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = n0 + (lane & 7) + 8 * (lane >> 4);
  const int c = k0 + 8 * ((lane >> 3) & 1);
  ldmatrix_x4(smem_u32(sm + swz<HD>(r, c)), b[0], b[1], b[2], b[3]);
}

// B fragments from a tile stored [k][n] (rows k0..k0+15, cols n0..n0+15).
template <int HD>
__device__ __forceinline__ void lds_bt(const bf16* sm, int k0, int n0, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = k0 + (lane & 7) + 8 * ((lane >> 3) & 1);
  const int c = n0 + 8 * (lane >> 4);
  ldmatrix_x4_trans(smem_u32(sm + swz<HD>(r, c)), b[0], b[1], b[2], b[3]);
}

// ------------------------------------------------------------------ forward
template <int HD>
struct FwdCfg {
  static constexpr int BM = 64, BN = 64, NT = 128;
  static constexpr size_t smem = (size_t)(BM + 4 * BN) * HD * sizeof(bf16);
};

template <int HD>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const bf16* __restrict__ qkv, long long ld, bf16* __restrict__ o,
                                                       long long ldo, float* __restrict__ lse, int s, int H, int Hkv) {
  using C = FwdCfg<HD>;
  extern __shared__ __align__(128) uint8_t smraw[];
  bf16* Qs = reinterpret_cast<bf16*>(smraw);
  bf16* Ks = Qs + C::BM * HD;
  bf16* Vs = Ks + 2 * C::BN * HD;

  const int nqt = (s + C::BM - 1) / C::BM;
  const int qt = nqt - 1 - blockIdx.x;  // heaviest tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (H / Hkv);
  const int q0 = qt * C::BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bf16* base = qkv + (long long)b * s * ld;
  const bf16* qg = base + (long long)h * HD;
  const bf16* kg = base + (long long)(H + g) * HD;
  const bf16* vg = base + (long long)(H + Hkv + g) * HD;

  load_tile<HD, C::NT>(Qs, qg, ld, q0, C::BM, s);
  cp_async_commit();
  const int kv_end = min(q0 + C::BM, s);
  const int nkt = (kv_end + C::BN - 1) / C::BN;
  load_tile<HD, C::NT>(Ks, kg, ld, 0, C::BN, s);
  load_tile<HD, C::NT>(Vs, vg, ld, 0, C::BN, s);
  cp_async_commit();

  cp_async_wait<1>();
  __syncthreads();
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) lds_a<HD>(Qs, warp * 16, kk * 16, qf[kk]);

  const float sc = rsqrtf((float)HD) * kLog2e;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  float acc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int row_a = q0 + warp * 16 + (lane >> 2);  // rows row_a and row_a + 8

  for (int j = 0; j < nkt; ++j) {
    const int buf = j & 1;
    if (j + 1 < nkt) {
      load_tile<HD, C::NT>(Ks + (buf ^ 1) * C::BN * HD, kg, ld, (j + 1) * C::BN, C::BN, s);
      load_tile<HD, C::NT>(Vs + (buf ^ 1) * C::BN * HD, vg, ld, (j + 1) * C::BN, C::BN, s);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16* Kt = Ks + buf * C::BN * HD;
    const bf16* Vt = Vs + buf * C::BN * HD;

    float S[C::BN / 8][4];
#pragma unroll
    for (int n = 0; n < C::BN / 8; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int n2 = 0; n2 < C::BN / 16; ++n2) {
        uint32_t bb[4];
        lds_b<HD>(Kt, n2 * 16, kk * 16, bb);
        mma_bf16_16816(S[2 * n2], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], bb[0], bb[1]);
        mma_bf16_16816(S[2 * n2 + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], bb[2], bb[3]);
      }
    }
    // scale, causal mask, online softmax (log2 domain)
    const int k_base = j * C::BN + 2 * (lane & 3);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < C::BN / 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k_base + n * 8 + (e & 1);
        const int row = row_a + 8 * (e >> 1);
        float v = S[n][e] * sc;
        if (key > row || key >= s) v = -INFINITY;
        S[n][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
    float corr[2], mnew[2], msafe[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      mnew[r] = fmaxf(mrow[r], mx[r]);
      msafe[r] = mnew[r] == -INFINITY ? 0.f : mnew[r];
      corr[r] = exp2f(mrow[r] - msafe[r]);
      mrow[r] = mnew[r];
      lrow[r] *= corr[r];
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      acc[i][0] *= corr[0]; acc[i][1] *= corr[0];
      acc[i][2] *= corr[1]; acc[i][3] *= corr[1];
    }
    uint32_t pf[C::BN / 8][2];
#pragma unroll
    for (int n = 0; n < C::BN / 8; ++n) {
      const float p0 = exp2f(S[n][0] - msafe[0]), p1 = exp2f(S[n][1] - msafe[0]);
      const float p2 = exp2f(S[n][2] - msafe[1]), p3 = exp2f(S[n][3] - msafe[1]);
      lrow[0] += p0 + p1;
      lrow[1] += p2 + p3;
      pf[n][0] = pack_bf16x2(p0, p1);
      pf[n][1] = pack_bf16x2(p2, p3);
    }
#pragma unroll
    for (int kk = 0; kk < C::BN / 16; ++kk) {
#pragma unroll
      for (int n2 = 0; n2 < HD / 16; ++n2) {
        uint32_t bb[4];
        lds_bt<HD>(Vt, kk * 16, n2 * 16, bb);
        mma_bf16_16816(acc[2 * n2], pf[2 * kk][0], pf[2 * kk][1], pf[2 * kk + 1][0], pf[2 * kk + 1][1], bb[0],
                       bb[1]);
        mma_bf16_16816(acc[2 * n2 + 1], pf[2 * kk][0], pf[2 * kk][1], pf[2 * kk + 1][0], pf[2 * kk + 1][1], bb[2],
                       bb[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
  const float inv0 = 1.f / lrow[0], inv1 = 1.f / lrow[1];
  bf16* og = o + (long long)b * s * ldo + (long long)h * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * (lane & 3);
    if (row_a < s)
      *reinterpret_cast<uint32_t*>(og + (long long)row_a * ldo + col) = pack_bf16x2(acc[i][0] * inv0, acc[i][1] * inv0);
    if (row_a + 8 < s)
      *reinterpret_cast<uint32_t*>(og + (long long)(row_a + 8) * ldo + col) =
          pack_bf16x2(acc[i][2] * inv1, acc[i][3] * inv1);
  }
  if ((lane & 3) == 0) {
    float* lg = lse + ((long long)b * H + h) * s;
    if (row_a < s) lg[row_a] = (mrow[0] + log2f(lrow[0])) / kLog2e;
    if (row_a + 8 < s) lg[row_a + 8] = (mrow[1] + log2f(lrow[1])) / kLog2e;
  }
}

// ------------------------------------------------------------------- delta
template <int HD>
__global__ void attn_delta_kernel(const bf16* __restrict__ o, long long ldo, const bf16* __restrict__ dout,
                                  long long lddo, float* __restrict__ delta, int B, int s, int H) {
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= (long long)B * s * H) return;
  const int h = (int)(w % H);
  const long long row = w / H;  // b * s + t
  const bf16* op = o + row * ldo + (long long)h * HD;
  const bf16* dp = dout + row * lddo + (long long)h * HD;
  float acc = 0.f;
  for (int c = 2 * lane; c < HD; c += 64) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(op + c));
    const float2 d = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dp + c));
    acc += a.x * d.x + a.y * d.y;
  }
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
  if (lane == 0) {
    const int b = (int)(row / s), t = (int)(row % s);
    delta[((long long)b * H + h) * s + t] = acc;
  }
}

// ----------------------------------------------------------------- dK / dV
template <int HD>
struct KvCfg {
  static constexpr int BN = 64;                   // keys per CTA (4 warps x 16)
  static constexpr int BQ = HD == 128 ? 32 : 64;  // queries per inner step
  static constexpr int NT = 128;
  static constexpr size_t smem = (size_t)(2 * BN + 4 * BQ) * HD * sizeof(bf16) + 4 * BQ * sizeof(float);
};

template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_kernel(const bf16* __restrict__ qkv, long long ld,
                                                            const bf16* __restrict__ dout, long long lddo,
                                                            const float* __restrict__ lse,
                                                            const float* __restrict__ delta, bf16* __restrict__ dqkv,
                                                            long long lddq, int s, int H, int Hkv) {
  using C = KvCfg<HD>;
  extern __shared__ __align__(128) uint8_t smraw[];
  bf16* Ks = reinterpret_cast<bf16*>(smraw);
  bf16* Vs = Ks + C::BN * HD;
  bf16* Qs = Vs + C::BN * HD;          // [2][BQ][HD]
  bf16* Ds = Qs + 2 * C::BQ * HD;      // dO tiles [2][BQ][HD]
  float* Ls = reinterpret_cast<float*>(Ds + 2 * C::BQ * HD);  // [2][BQ]
  float* Es = Ls + 2 * C::BQ;                                 // delta [2][BQ]

  const int kt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int k0 = kt * C::BN;
  const int grp = H / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bf16* base = qkv + (long long)b * s * ld;
  const bf16* dbase = dout + (long long)b * s * lddo;
  load_tile<HD, C::NT>(Ks, base + (long long)(H + g) * HD, ld, k0, C::BN, s);
  load_tile<HD, C::NT>(Vs, base + (long long)(H + Hkv + g) * HD, ld, k0, C::BN, s);
  cp_async_commit();

  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  const float sc = rsqrtf((float)HD) * kLog2e;
  const int qt_first = k0 / C::BQ;
  const int nqt = (s + C::BQ - 1) / C::BQ;
  const int steps_per_head = nqt - qt_first;
  const int total = steps_per_head * grp;
  const int key_a = k0 + warp * 16 + (lane >> 2);  // this thread's key rows: key_a, key_a + 8

  auto issue = [&](int step, int buf) {
    const int h = g * grp + step / steps_per_head;
    const int q0 = (qt_first + step % steps_per_head) * C::BQ;
    load_tile<HD, C::NT>(Qs + buf * C::BQ * HD, base + (long long)h * HD, ld, q0, C::BQ, s);
    load_tile<HD, C::NT>(Ds + buf * C::BQ * HD, dbase + (long long)h * HD, lddo, q0, C::BQ, s);
    const float* lg = lse + ((long long)b * H + h) * s;
    const float* eg = delta + ((long long)b * H + h) * s;
    for (int i = threadIdx.x; i < C::BQ; i += C::NT) {
      const int q = q0 + i;
      Ls[buf * C::BQ + i] = q < s ? lg[q] * kLog2e : 0.f;
      Es[buf * C::BQ + i] = q < s ? eg[q] : 0.f;
    }
  };
  if (total > 0) issue(0, 0);
  cp_async_commit();

  for (int step = 0; step < total; ++step) {
    const int buf = step & 1;
    if (step + 1 < total) issue(step + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int q0 = (qt_first + step % steps_per_head) * C::BQ;
    const bf16* Qt = Qs + buf * C::BQ * HD;
    const bf16* Dt = Ds + buf * C::BQ * HD;
    const float* Lt = Ls + buf * C::BQ;
    const float* Et = Es + buf * C::BQ;

    // S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x BQ queries
    float St[C::BQ / 8][4], Pt[C::BQ / 8][4];
#pragma unroll
    for (int n = 0; n < C::BQ / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) St[n][e] = Pt[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t ka[4], va[4];
      lds_a<HD>(Ks, warp * 16, kk * 16, ka);
      lds_a<HD>(Vs, warp * 16, kk * 16, va);
#pragma unroll
      for (int n2 = 0; n2 < C::BQ / 16; ++n2) {
        uint32_t qb[4], db[4];
        lds_b<HD>(Qt, n2 * 16, kk * 16, qb);
        lds_b<HD>(Dt, n2 * 16, kk * 16, db);
        mma_bf16_16816(St[2 * n2], ka[0], ka[1], ka[2], ka[3], qb[0], qb[1]);
        mma_bf16_16816(St[2 * n2 + 1], ka[0], ka[1], ka[2], ka[3], qb[2], qb[3]);
        mma_bf16_16816(Pt[2 * n2], va[0], va[1], va[2], va[3], db[0], db[1]);
        mma_bf16_16816(Pt[2 * n2 + 1], va[0], va[1], va[2], va[3], db[2], db[3]);
      }
    }
    // P^T = exp(S^T * scale - lse[q]), dS^T = P^T * (dP^T - delta[q])
    uint32_t pa[C::BQ / 8][2], da[C::BQ / 8][2];
#pragma unroll
    for (int n = 0; n < C::BQ / 8; ++n) {
      float p[4], ds[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qi = n * 8 + 2 * (lane & 3) + (e & 1);
        const int q = q0 + qi;
        const int key = key_a + 8 * (e >> 1);
        const bool live = q < s && key <= q;
        p[e] = live ? exp2f(St[n][e] * sc - Lt[qi]) : 0.f;
        ds[e] = p[e] * (Pt[n][e] - Et[qi]);
      }
      pa[n][0] = pack_bf16x2(p[0], p[1]);
      pa[n][1] = pack_bf16x2(p[2], p[3]);
      da[n][0] = pack_bf16x2(ds[0], ds[1]);
      da[n][1] = pack_bf16x2(ds[2], ds[3]);
    }
    // dV += P^T dO ; dK += dS^T Q   (k index = queries)
#pragma unroll
    for (int kk = 0; kk < C::BQ / 16; ++kk) {
#pragma unroll
      for (int n2 = 0; n2 < HD / 16; ++n2) {
        uint32_t db[4], qb[4];
        lds_bt<HD>(Dt, kk * 16, n2 * 16, db);
        lds_bt<HD>(Qt, kk * 16, n2 * 16, qb);
        mma_bf16_16816(dv[2 * n2], pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1], db[0], db[1]);
        mma_bf16_16816(dv[2 * n2 + 1], pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1], db[2],
                       db[3]);
        mma_bf16_16816(dk[2 * n2], da[2 * kk][0], da[2 * kk][1], da[2 * kk + 1][0], da[2 * kk + 1][1], qb[0], qb[1]);
        mma_bf16_16816(dk[2 * n2 + 1], da[2 * kk][0], da[2 * kk][1], da[2 * kk + 1][0], da[2 * kk + 1][1], qb[2],
                       qb[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  const float scale = rsqrtf((float)HD);
  bf16* dkg = dqkv + (long long)b * s * lddq + (long long)(H + g) * HD;
  bf16* dvg = dqkv + (long long)b * s * lddq + (long long)(H + Hkv + g) * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * (lane & 3);
    if (key_a < s) {
      *reinterpret_cast<uint32_t*>(dkg + (long long)key_a * lddq + col) = pack_bf16x2(dk[i][0] * scale, dk[i][1] * scale);
      *reinterpret_cast<uint32_t*>(dvg + (long long)key_a * lddq + col) = pack_bf16x2(dv[i][0], dv[i][1]);
    }
    if (key_a + 8 < s) {
      *reinterpret_cast<uint32_t*>(dkg + (long long)(key_a + 8) * lddq + col) =
          pack_bf16x2(dk[i][2] * scale, dk[i][3] * scale);
      *reinterpret_cast<uint32_t*>(dvg + (long long)(key_a + 8) * lddq + col) = pack_bf16x2(dv[i][2], dv[i][3]);
    }
  }
}

// --------------------------------------------------------------------- dQ
template <int HD>
struct QCfg {
  static constexpr int BM = 64;                   // queries per CTA
  static constexpr int BN = HD == 128 ? 32 : 64;  // keys per inner step
  static constexpr int NT = 128;
  static constexpr size_t smem = (size_t)(2 * BM + 4 * BN) * HD * sizeof(bf16);
};

template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const bf16* __restrict__ qkv, long long ld,
                                                          const bf16* __restrict__ dout, long long lddo,
                                                          const float* __restrict__ lse,
                                                          const float* __restrict__ delta, bf16* __restrict__ dqkv,
                                                          long long lddq, int s, int H, int Hkv) {
  using C = QCfg<HD>;
  extern __shared__ __align__(128) uint8_t smraw[];
  bf16* Qs = reinterpret_cast<bf16*>(smraw);
  bf16* Ds = Qs + C::BM * HD;
  bf16* Ks = Ds + C::BM * HD;   // [2][BN][HD]
  bf16* Vs = Ks + 2 * C::BN * HD;

  const int nqt = (s + C::BM - 1) / C::BM;
  const int qt = nqt - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (H / Hkv);
  const int q0 = qt * C::BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bf16* base = qkv + (long long)b * s * ld;
  const bf16* kg = base + (long long)(H + g) * HD;
  const bf16* vg = base + (long long)(H + Hkv + g) * HD;
  load_tile<HD, C::NT>(Qs, base + (long long)h * HD, ld, q0, C::BM, s);
  load_tile<HD, C::NT>(Ds, dout + (long long)b * s * lddo + (long long)h * HD, lddo, q0, C::BM, s);
  cp_async_commit();
  const int kv_end = min(q0 + C::BM, s);
  const int nkt = (kv_end + C::BN - 1) / C::BN;
  load_tile<HD, C::NT>(Ks, kg, ld, 0, C::BN, s);
  load_tile<HD, C::NT>(Vs, vg, ld, 0, C::BN, s);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();

  uint32_t qf[HD / 16][4], df[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    lds_a<HD>(Qs, warp * 16, kk * 16, qf[kk]);
    lds_a<HD>(Ds, warp * 16, kk * 16, df[kk]);
  }
  const int row_a = q0 + warp * 16 + (lane >> 2);
  const float* lg = lse + ((long long)b * H + h) * s;
  const float* eg = delta + ((long long)b * H + h) * s;
  float lrow[2], erow[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int q = row_a + 8 * r;
    lrow[r] = q < s ? lg[q] * kLog2e : 0.f;
    erow[r] = q < s ? eg[q] : 0.f;
  }
  float dq[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
  const float sc = rsqrtf((float)HD) * kLog2e;

  for (int j = 0; j < nkt; ++j) {
    const int buf = j & 1;
    if (j + 1 < nkt) {
      load_tile<HD, C::NT>(Ks + (buf ^ 1) * C::BN * HD, kg, ld, (j + 1) * C::BN, C::BN, s);
      load_tile<HD, C::NT>(Vs + (buf ^ 1) * C::BN * HD, vg, ld, (j + 1) * C::BN, C::BN, s);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16* Kt = Ks + buf * C::BN * HD;
    const bf16* Vt = Vs + buf * C::BN * HD;
    float S[C::BN / 8][4], P[C::BN / 8][4];
#pragma unroll
    for (int n = 0; n < C::BN / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) S[n][e] = P[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int n2 = 0; n2 < C::BN / 16; ++n2) {
        uint32_t kb[4], vb[4];
        lds_b<HD>(Kt, n2 * 16, kk * 16, kb);
        lds_b<HD>(Vt, n2 * 16, kk * 16, vb);
        mma_bf16_16816(S[2 * n2], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], kb[0], kb[1]);
        mma_bf16_16816(S[2 * n2 + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], kb[2], kb[3]);
        mma_bf16_16816(P[2 * n2], df[kk][0], df[kk][1], df[kk][2], df[kk][3], vb[0], vb[1]);
        mma_bf16_16816(P[2 * n2 + 1], df[kk][0], df[kk][1], df[kk][2], df[kk][3], vb[2], vb[3]);
      }
    }
    uint32_t dsf[C::BN / 8][2];
    const int k_base = j * C::BN + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < C::BN / 8; ++n) {
      float ds[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k_base + n * 8 + (e & 1);
        const int r = e >> 1;
        const int row = row_a + 8 * r;
        const bool live = row < s && key <= row;
        const float p = live ? exp2f(S[n][e] * sc - lrow[r]) : 0.f;
        ds[e] = p * (P[n][e] - erow[r]);
      }
      dsf[n][0] = pack_bf16x2(ds[0], ds[1]);
      dsf[n][1] = pack_bf16x2(ds[2], ds[3]);
    }
    // dQ += dS K   (k index = keys; K stored [key][hd] = [k][n])
#pragma unroll
    for (int kk = 0; kk < C::BN / 16; ++kk) {
#pragma unroll
      for (int n2 = 0; n2 < HD / 16; ++n2) {
        uint32_t kb[4];
        lds_bt<HD>(Kt, kk * 16, n2 * 16, kb);
        mma_bf16_16816(dq[2 * n2], dsf[2 * kk][0], dsf[2 * kk][1], dsf[2 * kk + 1][0], dsf[2 * kk + 1][1], kb[0],
                       kb[1]);
        mma_bf16_16816(dq[2 * n2 + 1], dsf[2 * kk][0], dsf[2 * kk][1], dsf[2 * kk + 1][0], dsf[2 * kk + 1][1],
                       kb[2], kb[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  const float scale = rsqrtf((float)HD);
  bf16* dqg = dqkv + (long long)b * s * lddq + (long long)h * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * (lane & 3);
    if (row_a < s)
      *reinterpret_cast<uint32_t*>(dqg + (long long)row_a * lddq + col) = pack_bf16x2(dq[i][0] * scale, dq[i][1] * scale);
    if (row_a + 8 < s)
      *reinterpret_cast<uint32_t*>(dqg + (long long)(row_a + 8) * lddq + col) =
          pack_bf16x2(dq[i][2] * scale, dq[i][3] * scale);
  }
}

template <int HD>
int launch_fwd(const bf16* qkv, long long ld, bf16* o, long long ldo, float* lse, int B, int s, int H, int Hkv,
               cudaStream_t st) {
  using C = FwdCfg<HD>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem);
    attr = true;
  }
  dim3 grid((s + C::BM - 1) / C::BM, H, B);
  attn_fwd_kernel<HD><<<grid, C::NT, C::smem, st>>>(qkv, ld, o, ldo, lse, s, H, Hkv);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

template <int HD>
int launch_bwd(const bf16* qkv, long long ld, const bf16* o, long long ldo, const bf16* dout, long long lddo,
               const float* lse, float* delta, bf16* dqkv, long long lddq, int B, int s, int H, int Hkv,
               cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_bwd_dkdv_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)KvCfg<HD>::smem);
    cudaFuncSetAttribute(attn_bwd_dq_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QCfg<HD>::smem);
    attr = true;
  }
  const long long warps = (long long)B * s * H;
  attn_delta_kernel<HD><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(o, ldo, dout, lddo, delta, B, s, H);
  dim3 g1((s + KvCfg<HD>::BN - 1) / KvCfg<HD>::BN, Hkv, B);
  attn_bwd_dkdv_kernel<HD><<<g1, KvCfg<HD>::NT, KvCfg<HD>::smem, st>>>(qkv, ld, dout, lddo, lse, delta, dqkv, lddq,
                                                                        s, H, Hkv);
  dim3 g2((s + QCfg<HD>::BM - 1) / QCfg<HD>::BM, H, B);
  attn_bwd_dq_kernel<HD><<<g2, QCfg<HD>::NT, QCfg<HD>::smem, st>>>(qkv, ld, dout, lddo, lse, delta, dqkv, lddq, s,
                                                                    H, Hkv);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

bool attn_args_ok(const void* p, long long ld, int B, int s, int H, int Hkv, int hd) {
  if (B < 0 || s < 0 || H <= 0 || Hkv <= 0 || H % Hkv) return false;
  if (hd != 16 && hd != 64 && hd != 128) return false;
  if ((reinterpret_cast<uintptr_t>(p) & 15) || ld % 8) return false;
  return true;
}

}  // namespace
}  // namespace mt

using namespace mt;

extern "C" int mt_k_attn_fwd(const void* qkv, int64_t ldqkv, void* o, int64_t ldo, float* lse, int B, int s, int H,
                             int Hkv, int hd, void* stream) {
  if ((hd == 64 || hd == 128) && attn_args_ok(qkv, ldqkv, B, s, H, Hkv, hd) &&
      ldqkv >= (int64_t)(H + 2 * Hkv) * hd && ldo >= (int64_t)H * hd && ldo % 8 == 0 &&
      (reinterpret_cast<uintptr_t>(o) & 15) == 0) {
    if (B == 0 || s == 0) return MT_OK;
    return attn_fwd_tc(qkv, ldqkv, o, ldo, lse, B, s, H, Hkv, hd, (cudaStream_t)stream);
  }
  return mt_k_attn_fwd_mma(qkv, ldqkv, o, ldo, lse, B, s, H, Hkv, hd, stream);
}

extern "C" int mt_k_attn_fwd_mma(const void* qkv, int64_t ldqkv, void* o, int64_t ldo, float* lse, int B, int s,
                                 int H, int Hkv, int hd, void* stream) {
  if (!attn_args_ok(qkv, ldqkv, B, s, H, Hkv, hd) || ldqkv < (int64_t)(H + 2 * Hkv) * hd || ldo < (int64_t)H * hd ||
      ldo % 2 || (reinterpret_cast<uintptr_t>(o) & 3))
    return MT_EINVAL;
  if (B == 0 || s == 0) return MT_OK;
  const bf16* q = (const bf16*)qkv;
  cudaStream_t st = (cudaStream_t)stream;
  switch (hd) {
    case 16: return launch_fwd<16>(q, ldqkv, (bf16*)o, ldo, lse, B, s, H, Hkv, st);
    case 64: return launch_fwd<64>(q, ldqkv, (bf16*)o, ldo, lse, B, s, H, Hkv, st);
    default: return launch_fwd<128>(q, ldqkv, (bf16*)o, ldo, lse, B, s, H, Hkv, st);
  }
}

namespace {
int attn_bwd_any(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout, int64_t lddo,
                 const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B, int s, int H, int Hkv, int hd,
                 const float* cos_t, const float* sin_t, void* stream) {
  if ((hd == 64 || hd == 128) && attn_args_ok(qkv, ldqkv, B, s, H, Hkv, hd) &&
      attn_args_ok(dout, lddo, B, s, H, Hkv, hd) && attn_args_ok(dqkv, lddqkv, B, s, H, Hkv, hd) &&
      ldqkv >= (int64_t)(H + 2 * Hkv) * hd && lddqkv >= (int64_t)(H + 2 * Hkv) * hd && ldo % 2 == 0 &&
      lddo >= (int64_t)H * hd) {
    if (B == 0 || s == 0) return MT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    const long long warps = (long long)B * s * H;
    if (hd == 64)
      attn_delta_kernel<64><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>((const bf16*)o, ldo, (const bf16*)dout,
                                                                        lddo, delta, B, s, H);
    else
      attn_delta_kernel<128><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>((const bf16*)o, ldo, (const bf16*)dout,
                                                                         lddo, delta, B, s, H);
    if (cudaGetLastError() != cudaSuccess) return MT_ECUDA;
    return attn_bwd_tc(qkv, ldqkv, dout, lddo, lse, delta, dqkv, lddqkv, B, s, H, Hkv, hd, cos_t, sin_t, st);
  }
  const int r = mt_k_attn_bwd_mma(qkv, ldqkv, o, ldo, dout, lddo, lse, delta, dqkv, lddqkv, B, s, H, Hkv, hd, stream);
  if (r != MT_OK || cos_t == nullptr) return r;
  // the legacy path rotates back in a separate pass (bf16 in, bf16 out)
  return mt_k_rope(dqkv, lddqkv, B, s, H + Hkv, hd, cos_t, sin_t, 1, stream);
}
}  // namespace

extern "C" int mt_k_attn_bwd(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout,
                             int64_t lddo, const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B, int s,
                             int H, int Hkv, int hd, void* stream) {
  return attn_bwd_any(qkv, ldqkv, o, ldo, dout, lddo, lse, delta, dqkv, lddqkv, B, s, H, Hkv, hd, nullptr, nullptr,
                      stream);
}

extern "C" int mt_k_attn_bwd_rope(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout,
                                  int64_t lddo, const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B,
                                  int s, int H, int Hkv, int hd, const float* cos_t, const float* sin_t, void* stream) {
  if (cos_t == nullptr || sin_t == nullptr || (reinterpret_cast<uintptr_t>(cos_t) & 15) ||
      (reinterpret_cast<uintptr_t>(sin_t) & 15))
    return MT_EINVAL;
  return attn_bwd_any(qkv, ldqkv, o, ldo, dout, lddo, lse, delta, dqkv, lddqkv, B, s, H, Hkv, hd, cos_t, sin_t, stream);
}

extern "C" int mt_k_attn_bwd_mma(const void* qkv, int64_t ldqkv, const void* o, int64_t ldo, const void* dout,
                                 int64_t lddo, const float* lse, float* delta, void* dqkv, int64_t lddqkv, int B,
                                 int s, int H, int Hkv, int hd, void* stream) {
  if (!attn_args_ok(qkv, ldqkv, B, s, H, Hkv, hd) || !attn_args_ok(dout, lddo, B, s, H, Hkv, hd) ||
      !attn_args_ok(dqkv, lddqkv, B, s, H, Hkv, hd) || ldqkv < (int64_t)(H + 2 * Hkv) * hd ||
      lddqkv < (int64_t)(H + 2 * Hkv) * hd || ldo % 2 || lddo < (int64_t)H * hd)
    return MT_EINVAL;
  if (B == 0 || s == 0) return MT_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const bf16* q = (const bf16*)qkv;
  switch (hd) {
    case 16:
      return launch_bwd<16>(q, ldqkv, (const bf16*)o, ldo, (const bf16*)dout, lddo, lse, delta, (bf16*)dqkv, lddqkv,
                            B, s, H, Hkv, st);
    case 64:
      return launch_bwd<64>(q, ldqkv, (const bf16*)o, ldo, (const bf16*)dout, lddo, lse, delta, (bf16*)dqkv, lddqkv,
                            B, s, H, Hkv, st);
    default:
      return launch_bwd<128>(q, ldqkv, (const bf16*)o, ldo, (const bf16*)dout, lddo, lse, delta, (bf16*)dqkv,
                             lddqkv, B, s, H, Hkv, st);
  }
}
