// Causal grouped-query attention backward on the 5th-generation tensor cores.
// Deterministic: every gradient element is accumulated by one CTA in a fixed
// order (no atomics). Two kernels, warp-specialised like the forward (warp 0
// TMA, warp 1 TMEM allocation + tcgen05.mma, warps 2-9 element-wise work):
//
//  dK/dV: one CTA per (128-key tile, KV head, batch). For every query head
//         of the group and every 128-query sub-tile at or after the diagonal:
//           S^T  = K Q^T, then dP^T = V dO^T, in one TMEM buffer
//           P^T  = exp(S^T * scale - lse[q]),  dS^T = P^T (dP^T - delta[q])
//                                                     (bf16, a second buffer)
//           dV  += P^T dO,  dK += dS^T Q   with dO and Q read MN-major
//         then dK *= scale. Every product is 128 x 128 or 128 x hd; all
//         eight element-wise warps work on one sub-tile, two threads per key.
//  dQ:    one CTA per (128-query tile, head, batch), two threads per query
//         row. For every 128-key tile up to the diagonal: S = Q K^T,
//         dP = dO V^T (TMEM); dS (bf16, TMEM); dQ += dS K with K read
//         MN-major; then dQ *= scale.
// delta = rowsum(dO * O) comes from the pre-pass in attention.cu. This is the
// backward of the stateless layer template's attention (travelaiplan blog,
// 核心功能 point 3: a hand-written backward per layer instead of autograd).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <string>
#include <type_traits>

#include "common.cuh"
#include "mt_internal.h"

namespace mt {
namespace {

constexpr int kT = 128;               // rows of a tile (keys or queries)
constexpr int kThr = 320;
constexpr uint32_t kBox = 128 * 128;  // 64 columns x 128 rows of bf16
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint8_t* align1024b(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Write `ncols` fp32 TMEM columns of this thread's lane as bf16 (times scale).
__device__ __forceinline__ void tmem_row_to_bf16(uint32_t taddr, int ncols, float scale, bf16* dst, bool store) {
#pragma unroll 1
  for (int c = 0; c < ncols / 32; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + c * 32, v);
    tmem_ld_wait();
    if (store) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(v[8 * k + 0]) * scale, __uint_as_float(v[8 * k + 1]) * scale);
        u.y = pack_bf16x2(__uint_as_float(v[8 * k + 2]) * scale, __uint_as_float(v[8 * k + 3]) * scale);
        u.z = pack_bf16x2(__uint_as_float(v[8 * k + 4]) * scale, __uint_as_float(v[8 * k + 5]) * scale);
        u.w = pack_bf16x2(__uint_as_float(v[8 * k + 6]) * scale, __uint_as_float(v[8 * k + 7]) * scale);
        *reinterpret_cast<uint4*>(dst + c * 32 + 8 * k) = u;
      }
    }
  }
}

// N consecutive fp32 values from a 16-byte-aligned address, in 16-byte loads
// (a RoPE table row: one position's cos or sin entries).
template <int N>
__device__ __forceinline__ void load_f32_vec(const float* p, float (&v)[N]) {
  static_assert(N % 4 == 0, "16-byte loads");
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p) + j);
    v[4 * j] = u.x;
    v[4 * j + 1] = u.y;
    v[4 * j + 2] = u.z;
    v[4 * j + 3] = u.w;
  }
}

// RoPE's inverse rotation on N columns of this thread's TMEM lane and their
// partners hd/2 further (times scale), stored as bf16: (x1, x2) ->
// (x1 c + x2 s, x2 c - x1 s) at the row's position, so dq / dk leave the
// kernel as gradients of the un-rotated q / k, rounded once. cs / sn hold
// the position's cos / sin entries of the N pairs (loaded by the caller
// ahead of time: each thread's row is a different position, so the loads
// cannot coalesce across the warp and their latency is best hidden).
template <int N>
__device__ __forceinline__ void tmem_pair_rope_to_bf16(uint32_t ta, uint32_t tb, float scale, const float (&cs)[N],
                                                       const float (&sn)[N], bf16* da, bf16* db, bool store) {
  uint32_t va[N], vb[N];
  if constexpr (N == 32) {
    tmem_ld_32x32b_x32(ta, va);
    tmem_ld_32x32b_x32(tb, vb);
  } else {
    tmem_ld_32x32b_x16(ta, va);
    tmem_ld_32x32b_x16(tb, vb);
  }
  tmem_ld_wait();
  if (!store) return;
  uint32_t pa[N / 2], pb[N / 2];
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    float o[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 2 * k + e;
      rope_pair(__uint_as_float(va[i]) * scale, __uint_as_float(vb[i]) * scale, cs[i], -sn[i], o[0][e], o[1][e]);
    }
    pa[k] = pack_bf16x2(o[0][0], o[0][1]);
    pb[k] = pack_bf16x2(o[1][0], o[1][1]);
  }
#pragma unroll
  for (int j = 0; j < N / 8; ++j) {
    reinterpret_cast<uint4*>(da)[j] = make_uint4(pa[4 * j], pa[4 * j + 1], pa[4 * j + 2], pa[4 * j + 3]);
    reinterpret_cast<uint4*>(db)[j] = make_uint4(pb[4 * j], pb[4 * j + 1], pb[4 * j + 2], pb[4 * j + 3]);
  }
}

// ------------------------------------------ dK / dV, 128-query sub-tiles
// One CTA per (128-key tile, KV head, batch); it walks the group's query
// heads and, per head, the 128-query sub-tiles from the diagonal on. Per
// sub-tile j the MMA thread issues, in this order,
//   dP^T j   (into tA, once the element-wise warps have copied S^T j out),
//   dV += P^T j dO   (once they have stored P^T j in tB),
//   S^T j + 1   (into tA, once they have copied dP^T j out),
//   dK += dS^T j Q   (once they have stored dS^T j in tB),
// so the element-wise warps compute P^T j while dP^T j runs, and dS^T j
// while dV j and S^T j + 1 run. Every product is M 128 x N 128 (or hd):
// a product with N = 64 costs about 1.5 times its arithmetic in issue, and
// the issue slots it needs are the ones the element-wise warps take. TMEM
// holds tA (S^T then dP^T, fp32), tB (P^T | dS^T packed as bf16 pairs, the
// A operands of the dV and dK products), dV and dK: 128 + 128 + 2 hd <= 512
// columns. Q and dO tiles of 128 queries share four shared-memory slots
// (see slot_q / slot_o); one element-wise warp checks that they have landed
// and releases them, so the MMA thread makes four waits and two commits per
// sub-tile (each of its waits and commits lets the products it has queued
// drain). The element-wise warps stage the sub-tile's 128
// lse and 128 delta values in shared memory, double-buffered, one barrier
// per sub-tile; each thread reads four query columns per 16-byte broadcast
// load, in two-wide fp32 instructions.
template <int HD>
struct KvTc2 {
  static constexpr int kBoxes = HD / 64;
  static constexpr uint32_t kKV = kBoxes * kBox;         // K, V, Q or dO tile of 128 rows
  static constexpr int kSlots = 4;                       // Q / dO slots, shared by both
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kKV;
  static constexpr uint32_t kSlotOff = 2 * kKV;          // [slot]
  static constexpr uint32_t kBarOff = kSlotOff + kSlots * kKV;
  static constexpr uint32_t kVecOff = kBarOff + 256;     // [2][lse * log2e x 128 | delta x 128]
  static constexpr size_t kSmem = 1024 + kVecOff + 2 * 128 * 8;
  static_assert(kSmem <= 232448, "shared memory per block");
};

// Slots of Q(j) and dO(j), the operands of 128-query sub-tile j: a slot is
// released by the product that last reads it (dO by dV, Q by dK, which runs
// later), and sub-tile j + 2 takes the slots in that order, Q(j + 2) the one
// dO(j) held and dO(j + 2) the one Q(j) held. Each slot is used once per two
// sub-tiles, so both slots of sub-tile j are in their use j / 2.
__device__ __forceinline__ int slot_q(int j) { return (0x3120 >> (4 * (j & 3))) & 15; }
__device__ __forceinline__ int slot_o(int j) { return (0x2031 >> (4 * (j & 3))) & 15; }

template <int HD>
__global__ void __launch_bounds__(kThr, 1)
    attn_bwd_dkdv_tc2_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                             const float* __restrict__ lse, const float* __restrict__ delta,
                             bf16* __restrict__ dqkv, long long lddq, int s, int H, int Hkv, int hc,
                             const float* __restrict__ cos_t, const float* __restrict__ sin_t, int* err) {
  using C = KvTc2<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024b(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
  uint64_t* kv_full = bars;                       // K and V tiles
  uint64_t* slot_full = bars + 1;                 // [kSlots]
  uint64_t* slot_empty = slot_full + C::kSlots;   // [kSlots] released by the loads warp
  uint64_t* s_full = slot_empty + C::kSlots;      // S^T j in tA (so dV j - 1, issued before it, is done)
  uint64_t* s_read = s_full + 1;                  // S^T copied out of tA, dO j landed (8 warps)
  uint64_t* d_full = s_full + 2;                  // dP^T j in tA (so dK j - 1, issued before it, is done)
  uint64_t* d_read = s_full + 3;                  // dP^T copied out of tA, Q j + 1 landed (8 warps)
  uint64_t* pv_full = s_full + 4;                 // P^T stored in tB (8 warps)
  uint64_t* ds_full = s_full + 5;                 // dS^T stored in tB (8 warps)
  uint64_t* done = s_full + 6;                    // all products done (completes once)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(s_full + 7);

  const int nqt = (s + kT - 1) / kT;
  int hb, kt;  // (batch, KV head) pair and key tile; kt = 0 is the longest
  chunked_tile_order(blockIdx.x, (int)gridDim.x / nqt, nqt, hc, hb, kt);
  const int g = hb % Hkv, b = hb / Hkv;
  const int grp = H / Hkv;
  const int k0 = kt * kT;
  const int per_head = nqt - kt;  // 128-query sub-tiles from the diagonal on
  const int total = grp * per_head;
  const int kcol = (H + g) * HD, vcol = (H + Hkv + g) * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tqkv);
    tma_prefetch_desc(&tdo);
    mbar_init(kv_full, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&slot_full[i], 1);
      mbar_init(&slot_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, 8);  // one arrival per element-wise warp
    mbar_init(d_full, 1);
    mbar_init(d_read, 8);
    mbar_init(pv_full, 8);
    mbar_init(ds_full, 8);
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: tA holds S^T, then dP^T, of the sub-tile (fp32, 128
  // queries); tB holds P^T (columns 0-63) and dS^T (64-127) packed as bf16
  // pairs, the A operands of the dV and dK products; then dV and dK.
  const uint32_t tA = tmem, tB = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + HD;

  if (warp == 0) {
    if (lane == 0) {
      int nld = 0;  // Q / dO loads issued
      bool ok = true;
      mbar_arrive_expect_tx(kv_full, 2 * C::kKV);
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_3d(sm + C::kKOff + bx * kBox, &tqkv, kcol + bx * 64, k0, b, kv_full);
        tma_load_3d(sm + C::kVOff + bx * kBox, &tqkv, vcol + bx * 64, k0, b, kv_full);
      }
      for (int j = 0; j < total && ok; ++j) {
        const int h = g * grp + j / per_head;
        const int q0 = k0 + (j % per_head) * kT;
        const int u = j >> 1;
        for (int w = 0; w < 2; ++w) {  // Q, then dO
          const int sl = w == 0 ? slot_q(j) : slot_o(j);
          if (u > 0 && !mbar_wait(&slot_empty[sl], (u - 1) & 1, err)) { ok = false; break; }
          uint8_t* dst = sm + C::kSlotOff + sl * C::kKV;
          mbar_arrive_expect_tx(&slot_full[sl], C::kKV);
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            if (w == 0)
              tma_load_3d(dst + bx * kBox, &tqkv, h * HD + bx * 64, q0, b, &slot_full[sl]);
            else
              tma_load_3d(dst + bx * kBox, &tdo, h * HD + bx * 64, q0, b, &slot_full[sl]);
          }
          ++nld;
        }
      }
      if (!ok) {
        // wait (bounded) for this CTA's copies still in flight before it exits
        mbar_wait(kv_full, 0, err);
        for (int i = nld - 1; i >= 0 && i >= nld - C::kSlots; --i) {
          const int j = i >> 1;
          const int sl = (i & 1) ? slot_o(j) : slot_q(j);
          mbar_wait(&slot_full[sl], (j >> 1) & 1, err);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kT, kT, false, false);  // S^T, dP^T: 128 keys x 128 queries
      constexpr uint32_t id_g = idesc_bf16_f32(kT, HD, false, true);   // dV, dK: B (dO, Q) MN-major
      const uint64_t dK = smem_desc_kmajor_sw128(smem_u32(sm + C::kKOff));
      const uint64_t dV = smem_desc_kmajor_sw128(smem_u32(sm + C::kVOff));
      auto slot_addr = [&](int sl) { return smem_u32(sm + C::kSlotOff + sl * C::kKV); };
      // A (K or V rows) and B (Q or dO rows) both K-major over hd
      auto scores = [&](uint64_t da, int sl) {
        const uint64_t db = smem_desc_kmajor_sw128(slot_addr(sl));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          tc_mma_bf16(tA, desc_advance(da, off), desc_advance(db, off), id_s, kk > 0);
        }
      };
      // dX += (P^T or dS^T, from tB at column ta) x (dO or Q, MN-major), over the 128 queries
      auto grads = [&](uint32_t dacc, uint32_t ta, int sl, bool first) {
        const uint64_t mb = smem_desc_mnmajor_sw128(slot_addr(sl), kBox);
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          tc_mma_bf16_ta(dacc, ta + kk * 8, desc_advance(mb, kk * 2048), id_g, (first && kk == 0) ? 0u : 1u);
      };
      bool ok = mbar_wait(kv_full, 0, err) && mbar_wait(&slot_full[slot_q(0)], 0, err);
      if (ok) {
        tc_fence_after();
        scores(dK, slot_q(0));
        tc_commit(s_full);
      }
      // per sub-tile j: dP^T j, dV j, S^T j + 1, dK j, so the element-wise
      // warps' work on one product's result overlaps the next product. Each
      // wait or commit of this thread stalls the tensor pipe until what it
      // has queued drains, so it makes four waits and two commits per
      // sub-tile: the loads warp checks that Q / dO have landed before the
      // group's arrivals, and releases their slots, and since products run
      // in issue order s_full j and d_full j also report dV j - 1 and
      // dK j - 1 done
      for (int j = 0; ok && j < total; ++j) {
        const uint32_t ph = j & 1;
        if (!(ok = mbar_wait(s_read, ph, err))) break;
        tc_fence_after();
        scores(dV, slot_o(j));
        tc_commit(d_full);
        if (!(ok = mbar_wait(pv_full, ph, err))) break;
        tc_fence_after();
        grads(tdV, tB, slot_o(j), j == 0);
        if (j + 1 < total) {
          if (!(ok = mbar_wait(d_read, ph, err))) break;
          tc_fence_after();
          scores(dK, slot_q(j + 1));
          tc_commit(s_full);
        }
        if (!(ok = mbar_wait(ds_full, ph, err))) break;
        tc_fence_after();
        grads(tdK, tB + 64, slot_q(j), j == 0);
      }
      if (ok) tc_commit(done);
    }
  } else {
    // two threads per key row: quarter q of the rows, half hf of the queries
    const int q = warp & 3, hf = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int key = k0 + row;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc = rsqrtf((float)HD) * kLog2e;
    float* vecs = reinterpret_cast<float*>(sm + C::kVecOff);  // [2][256]
    const int te = threadIdx.x - 64;  // 0..255
    auto all_sync = [&]() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) { return mbar_wait_warp(bar, parity, err); };
    // one warp also checks that the Q / dO tiles the next products read have
    // landed, before the group's arrival that lets the MMA thread issue them,
    // and releases each slot once its last reader is known to be done
    const bool loads_warp = warp == 2;
    auto wait_slot = [&](int sl, int jj) { return !loads_warp || wait_all(&slot_full[sl], (jj >> 1) & 1); };
    auto release = [&](int sl) {
      if (loads_warp) mbar_arrive_warp(&slot_empty[sl]);
    };
    bool ok = true;
    // (lse * log2e, delta) of query te of sub-tile j, read one sub-tile ahead
    auto load_vec = [&](int j) -> float2 {
      const int hh = g * grp + j / per_head;
      const int qq = k0 + (j % per_head) * kT + te;
      const long long vi = ((long long)b * H + hh) * s + qq;
      return qq < s ? make_float2(lse[vi] * kLog2e, delta[vi]) : make_float2(INFINITY, 0.f);
    };
    float2 vnext = make_float2(0.f, 0.f);
    if (te < kT && total > 0) vnext = load_vec(0);
    // every thread runs every sub-tile's barrier, also after a failed wait
    for (int j = 0; j < total; ++j) {
      const uint32_t ph = j & 1;
      const bool diag = (j % per_head) == 0;
      const int q0 = k0 + (j % per_head) * kT;
      float* vec = vecs + (j & 1) * 2 * kT;
      // the buffer written here was last read in sub-tile j - 2, which every
      // thread finished before the barrier of sub-tile j - 1
      if (te < kT) {
        vec[te] = vnext.x;
        vec[kT + te] = vnext.y;
      }
      all_sync();
      if (te < kT && j + 1 < total) vnext = load_vec(j + 1);
      if (!ok) continue;
      if (!wait_slot(slot_o(j), j) || !wait_all(s_full, ph)) { ok = false; continue; }
      // S^T j done, so dV j - 1, the last reader of dO j - 1's slot, is too
      if (j > 0) release(slot_o(j - 1));
      tc_fence_after();
      uint32_t rs[64], rp[64];
      tmem_ld_32x32b_x64_sync(tA + lane_off + hf * 64, rs);
      tc_fence_before();
      mbar_arrive_warp(s_read);
      // P^T = exp2(S^T * scale - lse); the diagonal sub-tile masks key > query.
      // P stays in rs (fp32, for dS^T); pw gets it packed as bf16 pairs.
      const float4* l4 = reinterpret_cast<const float4*>(vec + hf * 64);
      const float4* d4 = reinterpret_cast<const float4*>(vec + kT + hf * 64);
      const float2 sc2 = make_float2(sc, sc);
      uint32_t pw[32];
      auto probs = [&](auto masked_tag) {
        constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 l = l4[i];  // columns 4i .. 4i + 3 of this half
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int c = 4 * i + 2 * h2;
            const float2 x = ffma2(make_float2(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])), sc2,
                                   h2 == 0 ? make_float2(-l.x, -l.y) : make_float2(-l.z, -l.w));
            float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            if (kMasked) {
              if (q0 + hf * 64 + c < key) p0 = 0.f;
              if (q0 + hf * 64 + c + 1 < key) p1 = 0.f;
            }
            rs[c] = __float_as_uint(p0);
            rs[c + 1] = __float_as_uint(p1);
            pw[c >> 1] = pack_bf16x2(p0, p1);
          }
        }
      };
      if (diag)
        probs(std::true_type{});
      else
        probs(std::false_type{});
      {
        // P^T j - 1 was read by dV j - 1, done before S^T j
        tmem_st_32x32b_x32_sync(tB + lane_off + hf * 32, pw);
        tc_fence_before();
        mbar_arrive_warp(pv_full);
      }
      if ((j + 1 < total && !wait_slot(slot_q(j + 1), j + 1)) || !wait_all(d_full, ph)) { ok = false; continue; }
      // dP^T j done, so dK j - 1, the last reader of Q j - 1's slot, is too
      if (j > 0) release(slot_q(j - 1));
      tc_fence_after();
      tmem_ld_32x32b_x64_sync(tA + lane_off + hf * 64, rp);
      tc_fence_before();
      mbar_arrive_warp(d_read);
      // dS^T = P^T (dP^T - delta), packed in place
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 d = d4[i];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = 4 * i + 2 * h2;
          const float2 pp = make_float2(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1]));
          const float2 dp = make_float2(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1]));
          const float2 dv = fmul2(pp, fadd2(dp, h2 == 0 ? make_float2(-d.x, -d.y) : make_float2(-d.z, -d.w)));
          rp[c >> 1] = pack_bf16x2(dv.x, dv.y);  // in place: word c / 2 was read at this step or before
        }
      }
      {
        // dS^T j - 1 was read by dK j - 1, done before dP^T j
        tmem_st_32x32b_x32_sync(tB + 64 + lane_off + hf * 32, *reinterpret_cast<const uint32_t(*)[32]>(rp));
        tc_fence_before();
        mbar_arrive_warp(ds_full);
      }
    }
    // the dk rows' first RoPE chunk is read while the last products run
    const bool store = key < s;
    const bool rot = hf == 1 && cos_t != nullptr;
    const long long tb = (long long)(store ? key : 0) * (HD / 2);
    float rc[32], rsn[32];
    if (rot && ok && total > 0) {
      load_f32_vec<32>(cos_t + tb, rc);
      load_f32_vec<32>(sin_t + tb, rsn);
    }
    if (ok && total > 0 && wait_all(done, 0)) {
      tc_fence_after();
      const long long r0 = (long long)b * s + key;
      bf16* dkrow = dqkv + r0 * lddq + (long long)kcol;
      if (hf == 0) {
        tmem_row_to_bf16(tdV + lane_off, HD, 1.f, dqkv + r0 * lddq + (long long)vcol, store);
      } else if (!rot) {
        tmem_row_to_bf16(tdK + lane_off, HD, rsqrtf((float)HD), dkrow, store);
      } else {
        // dk rotated back at the key's position, one 32-pair chunk per step
#pragma unroll 1
        for (int jj = 0; jj < HD / 64; ++jj) {
          if (jj > 0) {
            load_f32_vec<32>(cos_t + tb + jj * 32, rc);
            load_f32_vec<32>(sin_t + tb + jj * 32, rsn);
          }
          tmem_pair_rope_to_bf16<32>(tdK + lane_off + jj * 32, tdK + lane_off + HD / 2 + jj * 32, rsqrtf((float)HD),
                                     rc, rsn, dkrow + jj * 32, dkrow + HD / 2 + jj * 32, store);
        }
      }
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

// ---------------------------------------------------------------------- dQ
// One CTA per (128-query tile, head, batch), two threads per query row (one
// per 64-key half). Per 128-key tile j: S = Q K^T and dP = dO V^T into TMEM;
// the element-wise warps write dS (packed bf16) into one of two 64-column
// TMEM buffers, where dQ += dS K reads it as its A operand. K and V stream
// through separate TMA rings: V is free as soon as dP has run, K once dQ
// has, so the loads of tile j + 1 are issued while tile j - 1 is still being
// multiplied instead of after it. Both land on one barrier per tile, which
// one element-wise warp checks (and it frees each V stage once S / dP of its
// tile are done): every wait or commit of the MMA thread lets the products
// it has queued drain, and it makes two of each per key tile.
template <int HD>
struct QTc {
  static constexpr int kBoxes = HD / 64;
  static constexpr uint32_t kTile = kBoxes * kBox;
  static constexpr int kKS = HD == 64 ? 4 : 3;             // K ring stages
  static constexpr int kVS = HD == 64 ? 4 : 2;             // V ring stages
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kOOff = kTile;                 // dO
  static constexpr uint32_t kKOff = 2 * kTile;             // [kKS]
  static constexpr uint32_t kVOff = kKOff + kKS * kTile;   // [kVS]
  static constexpr uint32_t kBarOff = kVOff + kVS * kTile;
  static constexpr size_t kSmem = 1024 + kBarOff + 256;
  static_assert(kSmem <= 232448, "shared memory per block");
  static_assert(kKS + 2 * kVS + 6 <= 256 / 8, "barrier area");
  static_assert(kVS <= kKS, "tiles in flight are bounded by the V ring");
};

template <int HD>
__global__ void __launch_bounds__(kThr, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                          const float* __restrict__ lse, const float* __restrict__ delta, bf16* __restrict__ dqkv,
                          long long lddq, int s, int H, int Hkv, int hc, const float* __restrict__ cos_t,
                          const float* __restrict__ sin_t, int* err) {
  using C = QTc<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024b(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;           // [kVS] K and V of tile j, on barrier j % kVS
  uint64_t* k_empty = kv_full + C::kVS;   // [kKS]
  uint64_t* v_empty = k_empty + C::kKS;   // [kVS]
  uint64_t* s_full = v_empty + C::kVS;   // S and dP in TMEM
  uint64_t* s_empty = s_full + 1;        // S and dP copied out of TMEM
  uint64_t* p_full = s_full + 2;         // dS stored in TMEM
  uint64_t* done = s_full + 3;           // every dQ product done (completes once)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(s_full + 4);

  const int nt = (s + kT - 1) / kT;
  int hb, rank;  // (batch, head) pair; rank 0 is the longest query tile
  chunked_tile_order(blockIdx.x, (int)gridDim.x / nt, nt, hc, hb, rank);
  const int qt = nt - 1 - rank;
  const int h = hb % H, b = hb / H;
  const int g = h / (H / Hkv);
  const int q0 = qt * kT;
  const int n_kv = qt + 1;
  const int kcol = (H + g) * HD, vcol = (H + Hkv + g) * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tqkv);
    tma_prefetch_desc(&tdo);
    mbar_init(q_full, 1);
    for (int i = 0; i < C::kKS; ++i) mbar_init(&k_empty[i], 1);
    for (int i = 0; i < C::kVS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 8);  // one arrival per element-wise warp
    mbar_init(p_full, 8);
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
  // dS of even / odd key tiles, 64 packed columns each
  auto tDS = [&](int j_) { return tmem + 384u + 64u * (uint32_t)(j_ & 1); };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::kTile);
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_3d(sm + C::kQOff + bx * kBox, &tqkv, h * HD + bx * 64, q0, b, q_full);
        tma_load_3d(sm + C::kOOff + bx * kBox, &tdo, h * HD + bx * 64, q0, b, q_full);
      }
      // K and V of tile j land on one barrier (kv_full[j % kVS]), so the MMA
      // thread makes one wait for both; the V ring is the shallower, so at
      // most kVS tiles are in flight
      int nkv = 0;  // tiles whose loads were issued
      for (int j = 0; j < n_kv; ++j) {
        const int ks = j % C::kKS, vs = j % C::kVS;
        if (!mbar_wait(&k_empty[ks], ((j / C::kKS) & 1) ^ 1, err)) break;
        if (!mbar_wait(&v_empty[vs], ((j / C::kVS) & 1) ^ 1, err)) break;
        mbar_arrive_expect_tx(&kv_full[vs], 2 * C::kTile);
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_3d(sm + C::kKOff + ks * C::kTile + bx * kBox, &tqkv, kcol + bx * 64, j * kT, b, &kv_full[vs]);
          tma_load_3d(sm + C::kVOff + vs * C::kTile + bx * kBox, &tqkv, vcol + bx * 64, j * kT, b, &kv_full[vs]);
        }
        ++nkv;
      }
      if (nkv < n_kv) {
        // a wait gave up: wait (bounded) for this CTA's copies still in
        // flight before it exits
        mbar_wait(q_full, 0, err);
        for (int i = 0; i < C::kVS && i < nkv; ++i) {
          const int last = nkv - 1 - i;
          mbar_wait(&kv_full[last % C::kVS], (last / C::kVS) & 1, err);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kT, kT, false, false);
      constexpr uint32_t id_q = idesc_bf16_f32(kT, HD, false, true);
      const uint64_t dQ = smem_desc_kmajor_sw128(smem_u32(sm + C::kQOff));
      const uint64_t dO = smem_desc_kmajor_sw128(smem_u32(sm + C::kOOff));
      bool ok = mbar_wait(q_full, 0, err);
      // S / dP of key tile j (its K and V loaded, the TMEM they overwrite
      // copied out by the element-wise warps); V is released when dP is done
      auto issue_s = [&](int j) -> bool {
        const int ks = j % C::kKS, vs = j % C::kVS;
        // tile 0's K / V are checked here; later tiles' by the element-wise
        // loads warp before its s_empty arrival (each wait of this thread
        // lets the products it has queued drain)
        if (j == 0 && !mbar_wait(&kv_full[0], 0, err)) return false;
        if (j > 0 && !mbar_wait(s_empty, (j - 1) & 1, err)) return false;
        tc_fence_after();
        const uint64_t dK = smem_desc_kmajor_sw128(smem_u32(sm + C::kKOff + ks * C::kTile));
        const uint64_t dV = smem_desc_kmajor_sw128(smem_u32(sm + C::kVOff + vs * C::kTile));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          tc_mma_bf16(tS, desc_advance(dQ, off), desc_advance(dK, off), id_s, kk > 0);
          tc_mma_bf16(tdP, desc_advance(dO, off), desc_advance(dV, off), id_s, kk > 0);
        }
        tc_commit(s_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        // the next tile's scores overlap this tile's element-wise work
        if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
        if (!(ok = mbar_wait(p_full, j & 1, err))) break;
        tc_fence_after();
        const uint64_t mK = smem_desc_mnmajor_sw128(smem_u32(sm + C::kKOff + (j % C::kKS) * C::kTile), kBox);
        // A operand from TMEM: 16 keys of dS are 8 packed columns
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          tc_mma_bf16_ta(tdQ, tDS(j) + kk * 8, desc_advance(mK, kk * 2048), id_q, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&k_empty[j % C::kKS]);
      }
      if (ok) tc_commit(done);
    }
  } else {
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int qpos = q0 + row;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc = rsqrtf((float)HD) * kLog2e;
    const long long vidx = ((long long)b * H + h) * s + qpos;
    const float l2 = qpos < s ? lse[vidx] * kLog2e : INFINITY;
    const float dl = qpos < s ? delta[vidx] : 0.f;
    bool ok = true;
    // one warp checks that the next tile's K / V have landed (before the
    // arrival that lets the MMA thread issue its products) and frees each V
    // stage once S / dP of its tile are done
    const bool loads_warp = warp == 2;
    for (int j = 0; j < n_kv && ok; ++j) {
      if (loads_warp && j + 1 < n_kv &&
          !mbar_wait_warp(&kv_full[(j + 1) % C::kVS], ((j + 1) / C::kVS) & 1, err)) {
        ok = false;
        break;
      }
      if (!mbar_wait_warp(s_full, j & 1, err)) { ok = false; break; }
      if (loads_warp) mbar_arrive_warp(&v_empty[j % C::kVS]);
      tc_fence_after();
      uint32_t rs[64], rp[64];
      tmem_ld_32x32b_x64_sync(tS + lane_off + half * 64, rs);
      tmem_ld_32x32b_x64_sync(tdP + lane_off + half * 64, rp);
      tc_fence_before();
      mbar_arrive_warp(s_empty);
      const int kb = j * kT + half * 64;
      uint32_t dk[32];
      const float2 sc2 = make_float2(sc, sc), nl2 = make_float2(-l2, -l2), ndl = make_float2(-dl, -dl);
      // only the diagonal key tile (the last) masks key > query; the others
      // run a copy of the loop without the compares
      auto elementwise = [&](auto masked_tag) {
        constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int ci = 2 * i;
          const float2 x = ffma2(make_float2(__uint_as_float(rs[ci]), __uint_as_float(rs[ci + 1])), sc2, nl2);
          float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (kMasked) {
            if (kb + ci > qpos) pp.x = 0.f;
            if (kb + ci + 1 > qpos) pp.y = 0.f;
          }
          const float2 dp = make_float2(__uint_as_float(rp[ci]), __uint_as_float(rp[ci + 1]));
          const float2 dv = fmul2(pp, fadd2(dp, ndl));
          dk[i] = pack_bf16x2(dv.x, dv.y);
        }
      };
      if (j == n_kv - 1)
        elementwise(std::true_type{});
      else
        elementwise(std::false_type{});
      // dS of this half's 64 keys into its 32 columns of buffer j % 2. The
      // product that last read that buffer (dQ of tile j - 2) completed
      // before S of tile j did, which s_full reported.
      tmem_st_32x32b_x32(tDS(j) + lane_off + half * 32, dk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(p_full);
    }
    // dq rotated back at the query's position: this thread takes pairs
    // [half * HD/4, (half + 1) * HD/4) and their partners HD/2 further; their
    // cos / sin entries are read while the last products run
    constexpr int N = HD / 4;
    const long long tb = (long long)(qpos < s ? qpos : 0) * (HD / 2) + half * N;
    float rc[N], rsn[N];
    if (cos_t != nullptr && ok) {
      load_f32_vec<N>(cos_t + tb, rc);
      load_f32_vec<N>(sin_t + tb, rsn);
    }
    if (ok && mbar_wait_warp(done, 0, err)) {
      tc_fence_after();
      bf16* dqh = dqkv + ((long long)b * s + qpos) * lddq + (long long)h * HD;
      if (cos_t == nullptr) {
        tmem_row_to_bf16(tdQ + lane_off + half * (HD / 2), HD / 2, rsqrtf((float)HD), dqh + half * (HD / 2), qpos < s);
      } else {
        tmem_pair_rope_to_bf16<N>(tdQ + lane_off + half * N, tdQ + lane_off + HD / 2 + half * N, rsqrtf((float)HD),
                                  rc, rsn, dqh + half * N, dqh + HD / 2 + half * N, qpos < s);
      }
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
  cudaFuncSetAttribute(attn_bwd_dkdv_tc2_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)KvTc2<64>::kSmem);
  cudaFuncSetAttribute(attn_bwd_dkdv_tc2_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)KvTc2<128>::kSmem);
  cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QTc<64>::kSmem);
  cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QTc<128>::kSmem);
}

bool make_map3(CUtensorMap* m, const void* p, long long ld, int s, int B) {
  cuuint64_t dims[3] = {(cuuint64_t)ld, (cuuint64_t)s, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)s * ld * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kT, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Backward matrix products of attention on tcgen05 (hd 64 or 128); delta must
// already hold rowsum(dO * O). Writes dq, dk, dv into dqkv; with cos_t /
// sin_t (RoPE tables [s_max, hd/2]) dq and dk are rotated back first.
int attn_bwd_tc(const void* qkv, long long ld, const void* dout, long long lddo, const float* lse,
                const float* delta, void* dqkv, long long lddq, int B, int s, int H, int Hkv, int hd,
                const float* cos_t, const float* sin_t, cudaStream_t stream) {
  std::call_once(g_once, init_once);
  if (!g_enc) return MT_ECUDA;
  if (hd != 64 && hd != 128) return MT_EINVAL;
  // the rotation reads each position's table row in 16-byte loads
  if ((cos_t == nullptr) != (sin_t == nullptr) || (reinterpret_cast<uintptr_t>(cos_t) & 15) ||
      (reinterpret_cast<uintptr_t>(sin_t) & 15))
    return MT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(dout) & 15) ||
      (reinterpret_cast<uintptr_t>(dqkv) & 15) || ld % 8 || lddo % 8 || lddq % 8)
    return MT_EINVAL;
  CUtensorMap tq, td;
  if (!make_map3(&tq, qkv, ld, s, B) || !make_map3(&td, dout, lddo, s, B)) return MT_EINVAL;
  const int nt = (s + kT - 1) / kT;
  // one CTA per (tile, head, batch) on a 1-D grid, in the chunked order
  if ((long long)nt * H * B > 0x7fffffffLL) return MT_EINVAL;
  const int grp = H / Hkv;
  // dK/dV of a KV head streams its group's Q and dO; dQ of a query head
  // streams its KV head's K and V, shared by the group's query heads
  const int hc1 = attn_head_chunk((long long)grp * s * hd * 4, B * Hkv);
  const int hc2 = attn_head_chunk((long long)s * hd * 4 / grp, B * H);
  int* err = device_error_word();
  const unsigned g1 = (unsigned)(nt * Hkv * B), g2 = (unsigned)(nt * H * B);
  if (hd == 64) {
    attn_bwd_dkdv_tc2_kernel<64><<<g1, kThr, KvTc2<64>::kSmem, stream>>>(tq, td, lse, delta, (bf16*)dqkv,
                                                                         lddq, s, H, Hkv, hc1, cos_t, sin_t, err);
    attn_bwd_dq_tc_kernel<64><<<g2, kThr, QTc<64>::kSmem, stream>>>(tq, td, lse, delta, (bf16*)dqkv, lddq, s, H, Hkv,
                                                                   hc2, cos_t, sin_t, err);
  } else {
    attn_bwd_dkdv_tc2_kernel<128><<<g1, kThr, KvTc2<128>::kSmem, stream>>>(tq, td, lse, delta, (bf16*)dqkv,
                                                                           lddq, s, H, Hkv, hc1, cos_t, sin_t, err);
    attn_bwd_dq_tc_kernel<128><<<g2, kThr, QTc<128>::kSmem, stream>>>(tq, td, lse, delta, (bf16*)dqkv, lddq, s, H,
                                                                     Hkv, hc2, cos_t, sin_t, err);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_error_message(std::string("attention backward launch: ") + cudaGetErrorString(e));
    return MT_ECUDA;
  }
  return MT_OK;
}

}  // namespace mt
