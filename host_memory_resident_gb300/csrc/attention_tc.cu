// Causal grouped-query attention forward on the 5th-generation tensor cores.
//
// One CTA per (pair of adjacent 128-query tiles, head, batch); the two tiles
// share every K and V tile the CTA loads. Warp-specialised:
//   warp 0   TMA producer: both Q tiles once, then K and V tiles of 128 keys
//            into separate rings (3-D tensor map over the qkv rows of one
//            sequence, so rows past its end arrive as zeros); K runs one
//            tile ahead of V;
//   warp 1   allocates TMEM and issues tcgen05.mma for both tiles t:
//              S_t = Q_t K_j^T    (M 128, N 128, K = hd) into t's 128-column
//                                  TMEM buffer,
//              O_t += P_t V_j     (M 128, N = hd, K 128) with P_t read from
//                                  TMEM as the A operand and V read MN-major
//                                  in place;
//   warps 2-5, 6-9: one softmax group per query tile, one thread per query
//            row (its TMEM lane) holding the row's 128 scores in registers.
//            The causal mask and the online softmax run in fp32 (log2
//            domain); P is written back as bf16 into TMEM: at hd 64 into
//            columns of its own, so S_t of the next key tile is issued as
//            soon as the group has copied S_t out; at hd 128, where S and O
//            fill TMEM, into the first 64 columns of S_t's own buffer, so
//            S_t of the next key tile is issued right after P_t V (the
//            products run in issue order). No P tile passes through shared
//            memory, whose port the operand reads and the TMA writes share.
//            O is rescaled in TMEM only when a row's running maximum grows
//            by more than 2^8, so P stays below 256 and the final O / l is
//            unchanged.
// While one group exponentiates, the tensor core computes the other group's
// products and both groups' next scores, so neither the exponential units nor
// the tensor core waits on a single chain of dependencies. Every wait or
// commit of the MMA thread lets the products it has queued drain; at hd 128
// it makes one of each per tile and key tile (a softmax warp checks the K / V
// loads and frees their stages).
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

constexpr int kQ = 128;                 // queries per tile (MMA M)
constexpr int kKV = 128;                // keys per tile
constexpr int kThr = 320;               // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (two groups)
constexpr uint32_t kBox = 128 * 128;    // one 64-column x 128-row bf16 box (16 KiB)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;        // rescale O only when the max grows by > 2^8

template <int HD>
struct TcCfg {
  static constexpr int kBoxes = HD / 64;
  static constexpr uint32_t kTile = kBoxes * kBox;     // 128 rows x HD
  static constexpr int kKS = 3;                        // K ring slots
  static constexpr int kVS = HD == 64 ? 3 : 2;         // V ring slots
  static constexpr uint32_t kQOff = 0;                 // two Q tiles
  static constexpr uint32_t kKOff = 2 * kTile;
  static constexpr uint32_t kVOff = kKOff + kKS * kTile;
  static constexpr uint32_t kBarOff = kVOff + kVS * kTile;
  static constexpr size_t kSmem = 1024 + kBarOff + 256;
  static_assert(kSmem <= 232448, "shared memory per block");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int HD>
__global__ void __launch_bounds__(kThr, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, bf16* __restrict__ o, long long ldo,
                       float* __restrict__ lse, int s, int H, int Hkv, int hc, int* err) {
  using C = TcCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
  uint64_t* q_full = bars;                   // [1]
  uint64_t* k_full = bars + 1;               // [kKS]
  uint64_t* k_empty = k_full + C::kKS;       // [kKS]
  uint64_t* v_full = k_empty + C::kKS;       // [kVS]
  uint64_t* v_empty = v_full + C::kVS;       // [kVS]
  uint64_t* s_full = v_empty + C::kVS;       // [2] per tile: S_t written
  uint64_t* s_empty = s_full + 2;            // [2] per tile: S_t copied out by its softmax group
  uint64_t* p_full = s_empty + 2;            // [2] per tile: P_t written (and O_t rescaled)
  uint64_t* p_empty = p_full + 2;            // [2] per tile: P_t V finished (hd 64: every key tile; hd 128: the last)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(p_empty + 2);

  const int nqt = (s + kQ - 1) / kQ;
  const int npair = (nqt + 1) / 2;
  int hb, rank;  // (batch, head) pair; rank 0 is the longest pair of query tiles
  chunked_tile_order(blockIdx.x, (int)gridDim.x / npair, npair, hc, hb, rank);
  const int pr = npair - 1 - rank;
  const int h = hb % H, b = hb / H;
  const int g = h / (H / Hkv);
  const int qt0 = 2 * pr;
  const int ntile = (qt0 + 1 < nqt) ? 2 : 1;
  const int nkv[2] = {qt0 + 1, ntile == 2 ? qt0 + 2 : 0};  // causal: key tiles 0..qt
  const int n_kv = ntile == 2 ? nkv[1] : nkv[0];
  const int qcol = h * HD, kcol = (H + g) * HD, vcol = (H + Hkv + g) * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm);
    mbar_init(q_full, 1);
    // at hd 128 each softmax group frees the K / V stages its tile has
    // finished with (one arrival per query tile); at hd 64 the MMA thread does
    const uint32_t rel = HD == 128 ? (uint32_t)ntile : 1u;
    for (int i = 0; i < C::kKS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], rel);
    }
    for (int i = 0; i < C::kVS; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], rel);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_empty[t], 4);  // one arrival per softmax warp
      mbar_init(&p_full[t], 4);
      mbar_init(&p_empty[t], 1);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // per-tile TMEM buffers, as arithmetic (an array indexed by the tile
  // would live in local memory)
  auto tS = [&](int t_) { return tmem + 128u * (uint32_t)t_; };
  auto tO = [&](int t_) { return tmem + 256u + (uint32_t)HD * (uint32_t)t_; };
  // P_t in TMEM: hd 64 leaves columns 384-511 free for it; at hd 128 it
  // takes the first 64 columns of S_t's buffer (kAlias)
  constexpr bool kAlias = HD == 128;
  auto tP = [&](int t_) { return kAlias ? tS(t_) : tmem + 384u + 64u * (uint32_t)t_; };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ loads
      int nk = 0, nv = 0;  // tiles issued into each ring
      bool ok = true;
      auto load_k = [&](int j) -> bool {
        const int st = j % C::kKS, use = j / C::kKS;
        if (!mbar_wait(&k_empty[st], (use & 1) ^ 1, err)) return false;
        mbar_arrive_expect_tx(&k_full[st], C::kTile);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_3d(sm + C::kKOff + st * C::kTile + bx * kBox, &tm, kcol + bx * 64, j * kKV, b, &k_full[st]);
        ++nk;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int st = j % C::kVS, use = j / C::kVS;
        if (!mbar_wait(&v_empty[st], (use & 1) ^ 1, err)) return false;
        mbar_arrive_expect_tx(&v_full[st], C::kTile);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_3d(sm + C::kVOff + st * C::kTile + bx * kBox, &tm, vcol + bx * 64, j * kKV, b, &v_full[st]);
        ++nv;
        return true;
      };
      mbar_arrive_expect_tx(q_full, ntile * C::kTile);
      for (int t = 0; t < ntile; ++t)
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_3d(sm + C::kQOff + t * C::kTile + bx * kBox, &tm, qcol + bx * 64, (qt0 + t) * kQ, b, q_full);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) ok = load_k(j);
        if (ok && j > 0) ok = load_v(j - 1);
      }
      if (!ok) {
        // wait (bounded) for this CTA's copies still in flight before it exits
        mbar_wait(q_full, 0, err);
        for (int i = 0; i < C::kKS && i < nk; ++i) {
          const int last = nk - 1 - ((nk - 1 - i) % C::kKS);  // last tile issued into slot last % kKS
          mbar_wait(&k_full[last % C::kKS], (last / C::kKS) & 1, err);
        }
        for (int i = 0; i < C::kVS && i < nv; ++i) {
          const int last = nv - 1 - ((nv - 1 - i) % C::kVS);
          mbar_wait(&v_full[last % C::kVS], (last / C::kVS) & 1, err);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMAs
      constexpr uint32_t idesc_s = idesc_bf16_f32(kQ, kKV, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kQ, HD, false, true);
      bool ok = mbar_wait(q_full, 0, err);
      const uint64_t dQ0 = smem_desc_kmajor_sw128(smem_u32(sm + C::kQOff));
      // S_t(j) = Q_t K_j^T; K_j has landed (the caller waited for it)
      auto mma_s = [&](int j, int t) {
        const uint64_t dK = smem_desc_kmajor_sw128(smem_u32(sm + C::kKOff + (j % C::kKS) * C::kTile));
        const uint64_t dQ = desc_advance(dQ0, t * C::kTile);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          tc_mma_bf16(tS(t), desc_advance(dQ, off), desc_advance(dK, off), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t]);
      };
      // O_t += P_t(j) V_j, P_t from TMEM (16 keys = 8 packed columns per step)
      auto mma_pv = [&](int j, int t, uint64_t mV) {
#pragma unroll
        for (int kk = 0; kk < kKV / 16; ++kk)
          tc_mma_bf16_ta(tO(t), tP(t) + kk * 8, desc_advance(mV, kk * 2048), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&p_empty[t]);
      };
      auto wait_k = [&](int j) { return mbar_wait(&k_full[j % C::kKS], (j / C::kKS) & 1, err); };
      if (kAlias) {
        // P_t(j) occupies S_t's columns until P_t(j) V has read it, so
        // S_t(j + 1) is issued right after that product. Every wait or
        // commit of this thread lets the products it has queued drain, so
        // it makes one wait (p_full) and one commit (s_full) per tile and
        // key tile: the softmax group checks that V j and K j + 1 have
        // landed before its p_full arrival and frees the K / V stages, and
        // S_t(j + 1) done also reports P_t(j) V done; only a tile's last
        // P V commits to p_empty
        if (ok && (ok = wait_k(0))) {
          tc_fence_after();
          for (int t = 0; t < 2; ++t)
            if (nkv[t] > 0) mma_s(0, t);
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          const int vs = j % C::kVS;
          const uint64_t mV = smem_desc_mnmajor_sw128(smem_u32(sm + C::kVOff + vs * C::kTile), kBox);
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= nkv[t]) continue;
            if (!(ok = mbar_wait(&p_full[t], j & 1, err))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kKV / 16; ++kk)
              tc_mma_bf16_ta(tO(t), tP(t) + kk * 8, desc_advance(mV, kk * 2048), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            if (j + 1 < nkv[t])
              mma_s(j + 1, t);
            else
              tc_commit(&p_empty[t]);
          }
        }
      } else {
        // S_t(j) for both tiles that still need key tile j, then release K_j;
        // S_t(j) overwrites S_t(j-1) once the group has copied it out
        auto issue_s = [&](int j) -> bool {
          if (!wait_k(j)) return false;
          for (int t = 0; t < 2; ++t) {
            if (j >= nkv[t]) continue;
            if (j > 0 && !mbar_wait(&s_empty[t], (j - 1) & 1, err)) return false;
            tc_fence_after();
            mma_s(j, t);
          }
          tc_commit(&k_empty[j % C::kKS]);
          return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 0; ok && j < n_kv; ++j) {
          if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
          const int vs = j % C::kVS;
          if (!(ok = mbar_wait(&v_full[vs], (j / C::kVS) & 1, err))) break;
          const uint64_t mV = smem_desc_mnmajor_sw128(smem_u32(sm + C::kVOff + vs * C::kTile), kBox);
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= nkv[t]) continue;
            if (!(ok = mbar_wait(&p_full[t], j & 1, err))) break;
            tc_fence_after();
            mma_pv(j, t, mV);
          }
          if (ok) tc_commit(&v_empty[vs]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) >> 2;          // query tile of this group
    const int q = warp & 3;                 // TMEM lane quarter
    const int row = q * 32 + lane;
    const int qpos = (qt0 + t) * kQ + row;
    const int nk = nkv[t];
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sc = rsqrtf((float)HD) * kLog2e;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // at hd 128, one warp of the group checks that V j and K j + 1 have
    // landed (while the group waits for S_t(j) anyway) and frees the K / V
    // stages this tile has finished with
    const bool loads_warp = kAlias && q == 2;
    for (int j = 0; j < nk && ok; ++j) {
      if (loads_warp) {
        if (!mbar_wait_warp(&v_full[j % C::kVS], (j / C::kVS) & 1, err)) { ok = false; break; }
        if (j + 1 < nk && !mbar_wait_warp(&k_full[(j + 1) % C::kKS], ((j + 1) / C::kKS) & 1, err)) {
          ok = false;
          break;
        }
      }
      if (!mbar_wait_warp(&s_full[t], j & 1, err)) { ok = false; break; }
      if (loads_warp) {
        // S_t(j) done: K j read; P_t(j-1) V, issued before S_t(j), done: V j-1 read
        mbar_arrive_warp(&k_empty[j % C::kKS]);
        if (j > 0) mbar_arrive_warp(&v_empty[(j - 1) % C::kVS]);
      }
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tS(t) + lane_off + c * 32, r[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive_warp(&s_empty[t]);
      // only the diagonal tile (the last one) needs the causal mask
      if (j == nk - 1) {
        const int kbase = j * kKV;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (kbase + c * 32 + i > qpos) r[c][i] = __float_as_uint(-INFINITY);
      }
      float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          m0 = fmax3(m0, __uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1]));
          m1 = fmax3(m1, __uint_as_float(r[c][i + 2]), __uint_as_float(r[c][i + 3]));
        }
      const float mx = fmaxf(m0, m1) * sc;  // row max in the scaled log2 domain (sc > 0)
      if (j == 0) m_ref = mx;
      const bool need = j > 0 && mx > m_ref + kRescale;
      const float m_use = need ? mx : m_ref;
      // P = exp2(s * sc - m_use), packed to bf16 in place
      float2 lt = make_float2(0.f, 0.f);
      const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_use, -m_use);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = ffma2(make_float2(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), sc2, nm2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          lt = fadd2(lt, pp);
          r[c][i] = pack_bf16x2(pp.x, pp.y);
        }
      const float lt0 = lt.x, lt1 = lt.y;
      // P_t(j-1) V has finished: O_t is current and the P buffer is free (at
      // hd 128 S_t(j), issued after it, has completed)
      if (j > 0 && !kAlias) {
        if (!mbar_wait_warp(&p_empty[t], (j - 1) & 1, err)) { ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need)) {
        const float factor = need ? exp2f(m_ref - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t ov[32];
          const uint32_t ta = tO(t) + lane_off + c * 32;
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
      }
      l += lt0 + lt1;
      // the row's 64 packed words into its TMEM lane, keys in order
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t pw[32];
#pragma unroll
        for (int w = 0; w < 32; ++w) pw[w] = r[(32 * h2 + w) >> 4][(32 * h2 + w) & 15];
        tmem_st_32x32b_x32(tP(t) + lane_off + h2 * 32, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&p_full[t]);
    }
    if (ok && nk > 0 && mbar_wait_warp(&p_empty[t], kAlias ? 0u : (uint32_t)((nk - 1) & 1), err)) {
      tc_fence_after();
      const float inv = 1.f / l;
      bf16* orow = o + ((long long)b * s + qpos) * ldo + (long long)h * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tO(t) + lane_off + c * 32, ov);
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
      if (qpos < s) lse[((long long)b * H + h) * s + qpos] = (m_ref + log2f(l)) / kLog2e;
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
  const int npair = ((s + kQ - 1) / kQ + 1) / 2;
  // one CTA per (pair of query tiles, head, batch) on a 1-D grid, in the
  // chunked order; a query head streams its KV head's K and V, shared by
  // the group's query heads
  if ((long long)npair * H * B > 0x7fffffffLL) return MT_EINVAL;
  const int hc = attn_head_chunk((long long)s * hd * 4 / (H / Hkv), B * H);
  const unsigned grid = (unsigned)(npair * H * B);
  int* err = device_error_word();
  if (hd == 64)
    attn_fwd_tc_kernel<64><<<grid, kThr, TcCfg<64>::kSmem, stream>>>(tm, (bf16*)o, ldo, lse, s, H, Hkv, hc, err);
  else
    attn_fwd_tc_kernel<128><<<grid, kThr, TcCfg<128>::kSmem, stream>>>(tm, (bf16*)o, ldo, lse, s, H, Hkv, hc, err);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

}  // namespace mt
