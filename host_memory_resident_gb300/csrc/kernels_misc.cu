// Memory-bound kernels of the stateless layer template: RMSNorm, RoPE,
// SwiGLU, embedding gather / deterministic scatter-add, cross
// entropy, fixed-order sums. Each is a plain streaming pass with 16-byte
// vector accesses where the layout allows; their cost is HBM bandwidth.
// The operators are those of a Llama-style decoder layer run through the
// per-layer template of the zhichai.net article ("以内存为中心的训练新范式",
// point 4) with the backward written by hand (travelaiplan blog, 核心功能
// point 3).
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <mutex>
#include <string>
#include <type_traits>

#include "common.cuh"
#include "mt_internal.h"

namespace mt {

int* device_error_word() {
  static int* words[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!words[dev]) {
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess || cudaMemset(p, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    words[dev] = p;
  }
  return words[dev];
}

namespace {

constexpr int kNormBwdVec = 4;          // 8-element vectors per thread and row, at most: 32 elements
constexpr int kNormBwdMaxWarps = 8;     // warps per row: d <= 8 * 32 * 32 = 8192
constexpr int kNormBwdMaxParts = 1216;  // row groups (dw partial sums): 8 per SM on 152 SMs (2 blocks of 4)

inline int launch_ok() { return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA; }

__device__ __forceinline__ void load_bf16x8(const bf16* p, float (&f)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

__device__ __forceinline__ void load_f32x8(const float* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Eight consecutive values of a bf16 or fp32 row as fp32.
__device__ __forceinline__ void load_x8(const bf16* p, float (&f)[8]) { load_bf16x8(p, f); }
__device__ __forceinline__ void load_x8(const float* p, float (&f)[8]) { load_f32x8(p, f); }

// Eight x values held in registers: packed bf16 pairs, or fp32.
template <typename TX>
struct XReg;
template <>
struct XReg<bf16> {
  uint4 p;
  __device__ __forceinline__ void load(const bf16* q) { p = *reinterpret_cast<const uint4*>(q); }
  __device__ __forceinline__ void zero() { p = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ float2 pair(int i) const {
    const uint32_t w = i == 0 ? p.x : i == 1 ? p.y : i == 2 ? p.z : p.w;
    return unpack_bf16x2(w);
  }
};
template <>
struct XReg<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* q) {
    a = reinterpret_cast<const float4*>(q)[0];
    b = reinterpret_cast<const float4*>(q)[1];
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ float2 pair(int i) const {
    return i == 0 ? make_float2(a.x, a.y) : i == 1 ? make_float2(a.z, a.w) : i == 2 ? make_float2(b.x, b.y)
                                                                                    : make_float2(b.z, b.w);
  }
};

__device__ __forceinline__ void store_bf16x8(bf16* p, const float (&f)[8]) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------ RMSNorm fwd
// One warp per row: sum of squares, then y = x * rstd * w. x is the
// residual stream (fp32) or any bf16 row.
template <typename TX>
__global__ void rmsnorm_fwd_kernel(const TX* __restrict__ x, const bf16* __restrict__ w, bf16* __restrict__ y,
                                   float* __restrict__ rstd, int M, int d, float eps) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const TX* xr = x + (long long)row * d;
  const int nvec = d >> 3;
  float ss = 0.f;
  for (int v = lane; v < nvec; v += 32) {
    float f[8];
    load_x8(xr + v * 8, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += f[i] * f[i];
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)d + eps);
  if (lane == 0) rstd[row] = r;
  bf16* yr = y + (long long)row * d;
  for (int v = lane; v < nvec; v += 32) {
    float f[8], g[8];
    load_x8(xr + v * 8, f);
    load_bf16x8(w + v * 8, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * r * g[i];
    store_bf16x8(yr + v * 8, f);
  }
}

// One row per block of kNormFwdThreads threads, each holding up to VPT
// vectors of 8 elements of the row in registers: x is read from HBM once
// (sum of squares, fixed-order block sum, then y = x * rstd * w from the
// registers). Rows up to 8 * VPT * kNormFwdThreads elements.
constexpr int kNormFwdThreads = 128;
template <typename TX, int VPT>
__global__ void __launch_bounds__(kNormFwdThreads)
    rmsnorm_fwd_row_kernel(const TX* __restrict__ x, const bf16* __restrict__ w, bf16* __restrict__ y,
                           float* __restrict__ rstd, int d, float eps) {
  __shared__ float red[kNormFwdThreads / 32];
  const int row = blockIdx.x, tid = threadIdx.x;
  const int nvec = d >> 3;
  const TX* xr = x + (long long)row * d;
  float v[VPT][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int vi = tid + k * kNormFwdThreads;
    if (vi < nvec) {
      load_x8(xr + vi * 8, v[k]);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[k][i] * v[k][i];
    }
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormFwdThreads / 32; ++i) tot += red[i];
  const float r = rsqrtf(tot / (float)d + eps);
  if (tid == 0) rstd[row] = r;
  bf16* yr = y + (long long)row * d;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int vi = tid + k * kNormFwdThreads;
    if (vi < nvec) {
      float g[8];
      load_bf16x8(w + vi * 8, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[k][i] = v[k][i] * r * g[i];
      store_bf16x8(yr + vi * 8, v[k]);
    }
  }
}

// ------------------------------------------------------------ RMSNorm bwd
// Row groups of W warps (W = ceil(d / 1024)); each thread holds up to 32
// elements of a row. Group g takes a contiguous range of rows; per row:
// dot = sum(dy*w*x) (warp shuffles, then one named barrier across the
// group's warps), dx = rstd*w*dy - x*rstd^3*dot/d (+ dres), and the thread's
// dw partial += dy*x*rstd. The group's partial goes to partial[g] and the
// column sums run in a fixed order, so dw is deterministic.
template <int W, typename TX, int VEC>
__global__ void __launch_bounds__(256, VEC == 2 ? 3 : 2)
    rmsnorm_bwd_kernel(const float* __restrict__ dy, const TX* __restrict__ x, const bf16* __restrict__ w,
                       const float* __restrict__ rstd, const float* dres, float* dx_f32, bf16* __restrict__ dx_bf16,
                       float* __restrict__ partial, int M, int d, int n_groups, int rows_per_group) {
  constexpr int G = 8 / W > 0 ? 8 / W : 1;  // groups per block
  __shared__ float red[G][2][W];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gl = warp / W, wg = warp % W;   // group within the block, warp within the group
  const int gid = blockIdx.x * G + gl;
  if (gid >= n_groups) return;  // whole groups leave together (named barriers count only their warps)
  const int nvec = d >> 3;
  const int r0 = gid * rows_per_group, r1 = min(M, r0 + rows_per_group);
  uint4 wp[VEC];                    // w as packed bf16 pairs
  float acc[VEC][8];
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int v = lane + 32 * (wg + W * k);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[k][i] = 0.f;
    wp[k] = v < nvec ? *reinterpret_cast<const uint4*>(w + v * 8) : make_uint4(0, 0, 0, 0);
  }
  for (int row = r0, it = 0; row < r1; ++row, ++it) {
    const float r = rstd[row];
    const float* dyr = dy + (long long)row * d;
    const TX* xr = x + (long long)row * d;
    float dyv[VEC][8];
    XReg<TX> xp[VEC];
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int v = lane + 32 * (wg + W * k);
      if (v < nvec) {
        const float4 a = reinterpret_cast<const float4*>(dyr + v * 8)[0];
        const float4 b = reinterpret_cast<const float4*>(dyr + v * 8)[1];
        dyv[k][0] = a.x; dyv[k][1] = a.y; dyv[k][2] = a.z; dyv[k][3] = a.w;
        dyv[k][4] = b.x; dyv[k][5] = b.y; dyv[k][6] = b.z; dyv[k][7] = b.w;
        xp[k].load(xr + v * 8);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) dyv[k][i] = 0.f;
        xp[k].zero();
      }
    }
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const uint32_t ww[4] = {wp[k].x, wp[k].y, wp[k].z, wp[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 xf = xp[k].pair(i), wf = unpack_bf16x2(ww[i]);
        dot += dyv[k][2 * i] * wf.x * xf.x;
        dot += dyv[k][2 * i + 1] * wf.y * xf.y;
      }
    }
    dot = warp_sum(dot);
    float tot = dot;
    if (W > 1) {
      if (lane == 0) red[gl][it & 1][wg] = dot;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + gl), "r"(32 * W) : "memory");
      tot = 0.f;
#pragma unroll
      for (int i = 0; i < W; ++i) tot += red[gl][it & 1][i];
    }
    const float c = r * r * r * tot / (float)d;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int v = lane + 32 * (wg + W * k);
      if (v < nvec) {
        const uint32_t ww[4] = {wp[k].x, wp[k].y, wp[k].z, wp[k].w};
        float o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 xf = xp[k].pair(i), wf = unpack_bf16x2(ww[i]);
          o[2 * i] = r * wf.x * dyv[k][2 * i] - xf.x * c;
          o[2 * i + 1] = r * wf.y * dyv[k][2 * i + 1] - xf.y * c;
          acc[k][2 * i] += dyv[k][2 * i] * xf.x * r;
          acc[k][2 * i + 1] += dyv[k][2 * i + 1] * xf.y * r;
        }
        const long long off = (long long)row * d + v * 8;
        if (dres != nullptr) {
          const float4 a = reinterpret_cast<const float4*>(dres + off)[0];
          const float4 b = reinterpret_cast<const float4*>(dres + off)[1];
          o[0] += a.x; o[1] += a.y; o[2] += a.z; o[3] += a.w;
          o[4] += b.x; o[5] += b.y; o[6] += b.z; o[7] += b.w;
        }
        if (dx_f32 != nullptr) {
          reinterpret_cast<float4*>(dx_f32 + off)[0] = make_float4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<float4*>(dx_f32 + off)[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
        if (dx_bf16 != nullptr) store_bf16x8(dx_bf16 + off, o);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int v = lane + 32 * (wg + W * k);
    if (v < nvec) {
      float* p = partial + (long long)gid * d + v * 8;
      reinterpret_cast<float4*>(p)[0] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
      reinterpret_cast<float4*>(p)[1] = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
    }
  }
}

// dw[c] = sum over parts p of partial[p, c], rounded to bf16. Block: 32
// columns x 16 part classes; class j sums parts j, j+16, ... in order, then
// the 16 class sums are added in order (a fixed order for every launch).
constexpr int kColsumClasses = 16;
__global__ void __launch_bounds__(32 * kColsumClasses)
    colsum_to_bf16_kernel(const float* __restrict__ partial, int n_part, int d, bf16* __restrict__ out) {
  __shared__ float cls[kColsumClasses][32];
  const int cl = threadIdx.x & 31, j = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + cl;
  float s = 0.f;
  if (c < d)
    for (int p = j; p < n_part; p += kColsumClasses) s += partial[(long long)p * d + c];
  cls[j][cl] = s;
  __syncthreads();
  if (j == 0 && c < d) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kColsumClasses; ++i) t += cls[i][cl];
    out[c] = __float2bfloat16_rn(t);
  }
}

// ------------------------------------------------------------------ RoPE
// Thread per (row, head, pair of adjacent rotation pairs).
__global__ void rope_kernel(bf16* __restrict__ xbuf, long long ld, int M, int s, int nheads, int hd,
                            const float* __restrict__ cos_t, const float* __restrict__ sin_t, float sign) {
  const int half = hd >> 1;
  const int quarter = half >> 1;  // thread handles pairs 2p, 2p+1
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)M * nheads * quarter;
  if (idx >= total) return;
  const int p = (int)(idx % quarter);
  const long long rh = idx / quarter;
  const int head = (int)(rh % nheads);
  const int row = (int)(rh / nheads);
  const int t = row % s;
  bf16* base = xbuf + (long long)row * ld + (long long)head * hd;
  const int i = 2 * p;
  __nv_bfloat162* pa = reinterpret_cast<__nv_bfloat162*>(base + i);
  __nv_bfloat162* pb = reinterpret_cast<__nv_bfloat162*>(base + i + half);
  const float2 a = __bfloat1622float2(*pa);
  const float2 b = __bfloat1622float2(*pb);
  const float c0 = cos_t[(long long)t * half + i], c1 = cos_t[(long long)t * half + i + 1];
  const float s0 = sign * sin_t[(long long)t * half + i], s1 = sign * sin_t[(long long)t * half + i + 1];
  float o1x, o2x, o1y, o2y;
  rope_pair(a.x, b.x, c0, s0, o1x, o2x);
  rope_pair(a.y, b.y, c1, s1, o1y, o2y);
  *pa = __floats2bfloat162_rn(o1x, o1y);
  *pb = __floats2bfloat162_rn(o2x, o2y);
}

// Same rotation, 8 consecutive pairs per thread with 16-byte loads and
// stores (row pitch a multiple of 8 elements, hd a multiple of 16).
__global__ void rope_vec_kernel(bf16* __restrict__ xbuf, long long ld, int M, int s, int nheads, int hd,
                                const float* __restrict__ cos_t, const float* __restrict__ sin_t, float sign) {
  const int half = hd >> 1;
  const int per = half >> 3;  // threads per (row, head)
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)M * nheads * per;
  if (idx >= total) return;
  const int p = (int)(idx % per);
  const long long rh = idx / per;
  const int head = (int)(rh % nheads);
  const int row = (int)(rh / nheads);
  const int t = row % s;
  const int i = 8 * p;
  bf16* base = xbuf + (long long)row * ld + (long long)head * hd;
  uint4* pa = reinterpret_cast<uint4*>(base + i);
  uint4* pb = reinterpret_cast<uint4*>(base + i + half);
  const uint4 ua = *pa, ub = *pb;
  const float4* ct = reinterpret_cast<const float4*>(cos_t + (long long)t * half + i);
  const float4* st = reinterpret_cast<const float4*>(sin_t + (long long)t * half + i);
  const float4 c0 = ct[0], c1 = ct[1], s0 = st[0], s1 = st[1];
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float sn[8] = {sign * s0.x, sign * s0.y, sign * s0.z, sign * s0.w,
                       sign * s1.x, sign * s1.y, sign * s1.z, sign * s1.w};
  const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 a = unpack_bf16x2(wa[k]), b = unpack_bf16x2(wb[k]);
    float o1x, o2x, o1y, o2y;
    rope_pair(a.x, b.x, c[2 * k], sn[2 * k], o1x, o2x);
    rope_pair(a.y, b.y, c[2 * k + 1], sn[2 * k + 1], o1y, o2y);
    oa[k] = pack_bf16x2(o1x, o1y);
    ob[k] = pack_bf16x2(o2x, o2y);
  }
  *pa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *pb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// ---------------------------------------------------------------- SwiGLU
__global__ void swiglu_fwd_kernel(const bf16* __restrict__ gu, bf16* __restrict__ a, int M, int f) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int nv = f >> 3;
  if (idx >= (long long)M * nv) return;
  const int row = (int)(idx / nv);
  const int v = (int)(idx % nv);
  const bf16* gr = gu + (long long)row * 2 * f + v * 8;
  float g[8], u[8], o[8];
  load_bf16x8(gr, g);
  load_bf16x8(gr + f, u);
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = swiglu_fwd_elem(g[i], u[i]);
  store_bf16x8(a + (long long)row * f + v * 8, o);
}

__global__ void swiglu_bwd_kernel(const bf16* __restrict__ da, const bf16* __restrict__ gu, bf16* __restrict__ dgu,
                                  int M, int f) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int nv = f >> 3;
  if (idx >= (long long)M * nv) return;
  const int row = (int)(idx / nv);
  const int v = (int)(idx % nv);
  const bf16* gr = gu + (long long)row * 2 * f + v * 8;
  float g[8], u[8], d[8], dg[8], du[8];
  load_bf16x8(gr, g);
  load_bf16x8(gr + f, u);
  load_bf16x8(da + (long long)row * f + v * 8, d);
#pragma unroll
  for (int i = 0; i < 8; ++i) swiglu_bwd_elem(d[i], g[i], u[i], dg[i], du[i]);
  bf16* o = dgu + (long long)row * 2 * f + v * 8;
  store_bf16x8(o, dg);
  store_bf16x8(o + f, du);
}

// ------------------------------------------------------------- embedding
__global__ void embedding_fwd_kernel(const bf16* __restrict__ E, const int32_t* __restrict__ tok, bf16* __restrict__ x,
                                     int M, int d, int V, int* err) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const int id = tok[row];
  const bool ok = id >= 0 && id < V;
  if (!ok && lane == 0) set_device_error(err, kDevErrBadToken);
  const uint4* src = reinterpret_cast<const uint4*>(E + (long long)(ok ? id : 0) * d);
  uint4* dst = reinterpret_cast<uint4*>(x + (long long)row * d);
  for (int v = lane; v < (d >> 3); v += 32) dst[v] = ok ? src[v] : make_uint4(0, 0, 0, 0);
}

// The same gather into an fp32 row (the start of the fp32 residual stream;
// every bf16 value is exact in fp32).
__global__ void embedding_fwd_f32_kernel(const bf16* __restrict__ E, const int32_t* __restrict__ tok,
                                         float* __restrict__ x, int M, int d, int V, int* err) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const int id = tok[row];
  const bool ok = id >= 0 && id < V;
  if (!ok && lane == 0) set_device_error(err, kDevErrBadToken);
  const bf16* src = E + (long long)(ok ? id : 0) * d;
  float* dst = x + (long long)row * d;
  for (int v = lane; v < (d >> 3); v += 32) {
    float f[8];
    load_bf16x8(src + v * 8, f);
    if (!ok) {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
    reinterpret_cast<float4*>(dst + v * 8)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(dst + v * 8)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

// Stable counting sort of token positions by id, in one CTA of 1024 threads.
// work layout (int32): start[V + 1] | cursor[V] | perm[M].
constexpr int kSortThreads = 1024;

__device__ __forceinline__ int block_inclusive_max(int v, int* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = max(v, n);
  }
  if (lane == 31) scratch[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = max(w, n);
    }
    scratch[lane] = w;
  }
  __syncthreads();
  if (wid > 0) v = max(v, scratch[wid - 1]);
  __syncthreads();
  return v;
}

__device__ __forceinline__ int block_exclusive_sum(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const int before = (wid > 0 ? scratch[wid - 1] : 0) + x - v;
  *total = scratch[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kSortThreads) token_sort_kernel(const int32_t* __restrict__ tok, int M, int V,
                                                                  int32_t* __restrict__ work, int* err) {
  __shared__ unsigned long long keys[kSortThreads];
  __shared__ int scratch[32];
  int32_t* start = work;
  int32_t* cursor = work + V + 1;
  int32_t* perm = cursor + V;
  const int tid = threadIdx.x;
  for (int v = tid; v < V; v += kSortThreads) cursor[v] = 0;
  __syncthreads();
  for (int m = tid; m < M; m += kSortThreads) {
    const int id = tok[m];
    if (id >= 0 && id < V) atomicAdd(&cursor[id], 1);
    else set_device_error(err, kDevErrBadToken);
  }
  __syncthreads();
  int carry = 0;
  for (int v0 = 0; v0 < V; v0 += kSortThreads) {
    const int v = v0 + tid;
    const int c = v < V ? cursor[v] : 0;
    int total;
    const int ex = block_exclusive_sum(c, scratch, &total);
    if (v < V) start[v] = carry + ex;
    carry += total;
  }
  if (tid == 0) start[V] = carry;
  for (int v = tid; v < V; v += kSortThreads) cursor[v] = 0;
  __syncthreads();
  for (int m0 = 0; m0 < M; m0 += kSortThreads) {
    const int m = m0 + tid;
    unsigned long long key = ~0ull;
    if (m < M) {
      const int id = tok[m];
      if (id >= 0 && id < V) key = ((unsigned long long)(unsigned)id << 32) | (unsigned)m;
    }
    keys[tid] = key;
    __syncthreads();
    // bitonic sort of 1024 keys, ascending
    for (int k = 2; k <= kSortThreads; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        const int p = tid ^ j;
        if (p > tid) {
          const unsigned long long a = keys[tid], b = keys[p];
          const bool up = (tid & k) == 0;
          if ((a > b) == up) { keys[tid] = b; keys[p] = a; }
        }
        __syncthreads();
      }
    }
    const unsigned long long me = keys[tid];
    const bool valid = me != ~0ull;
    const unsigned id = (unsigned)(me >> 32);
    const bool head = tid == 0 || (keys[tid - 1] >> 32) != id;
    const int seg = block_inclusive_max(head ? tid : 0, scratch);
    const int rank = tid - seg;
    if (valid) perm[start[id] + cursor[id] + rank] = (int)(me & 0xffffffffu);
    const bool tail = tid == kSortThreads - 1 || (keys[tid + 1] >> 32) != id;
    __syncthreads();
    if (valid && tail) cursor[id] += rank + 1;
    __syncthreads();
  }
}

// dE[v, c..c+3] = sum_{p in [start[v], start[v+1])} dx[perm[p], c..c+3]
__global__ void embedding_bwd_reduce_kernel(const float* __restrict__ dx, const int32_t* __restrict__ work,
                                            bf16* __restrict__ dE, int d, int V) {
  const int v = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (c >= d) return;
  const int32_t* start = work;
  const int32_t* perm = work + 2 * V + 1;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int p1 = start[v + 1];
  for (int p = start[v]; p < p1; ++p) {
    const float4 x = *reinterpret_cast<const float4*>(dx + (long long)perm[p] * d + c);
    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
  }
  uint2 u;
  u.x = pack_bf16x2(acc.x, acc.y);
  u.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(dE + (long long)v * d + c) = u;
}

// ---------------------------------------------------------- cross entropy
constexpr int kCeThreads = 512;
constexpr int kCeUnroll = 4;  // independent 16-byte loads in flight per thread


// Merge of two (max, sum of 2^(y - max)) pairs in log2 units.
__device__ __forceinline__ void online_merge2(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * ex2_approx(m - m2) + s2;
    m = m2;
  } else if (m2 != -INFINITY) {
    s += s2 * ex2_approx(m2 - m);
  }
}

// Persistent: a grid of one or two 512-thread blocks per SM walks the rows,
// so the rows in flight (blocks x V x 4 bytes) stay well inside L2 and the
// second pass over a row (the gradient) reads it from L2 instead of HBM;
// each thread keeps kCeUnroll 16-byte loads in flight. The exponentials run
// in base 2 (e^x = 2^(x log2 e)) on the special-function unit: one fused
// multiply-add and one ex2 per logit and pass.
__global__ void __launch_bounds__(kCeThreads, 2)
    cross_entropy_kernel(const float* __restrict__ logits, long long ldl, const int32_t* __restrict__ labels,
                         bf16* __restrict__ dz, long long lddz, float* __restrict__ loss_rows, int M, int V,
                         float scale, int* err) {
  constexpr float kL2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
  __shared__ float sm_m[kCeThreads / 32], sm_s[kCeThreads / 32];
  const int tid = threadIdx.x;
  const int nv = V >> 2;
  for (int row = blockIdx.x; row < M; row += gridDim.x) {
    const float* z = logits + (long long)row * ldl;
    float m = -INFINITY, s = 0.f;  // log2 units: m = max of z log2 e, s = sum of 2^(z log2 e - m)
    for (int v0 = tid; v0 < nv; v0 += kCeUnroll * kCeThreads) {
      float4 q[kCeUnroll];
#pragma unroll
      for (int u = 0; u < kCeUnroll; ++u) {
        const int v = v0 + u * kCeThreads;
        if (v < nv) q[u] = reinterpret_cast<const float4*>(z)[v];
      }
#pragma unroll
      for (int u = 0; u < kCeUnroll; ++u) {
        if (v0 + u * kCeThreads < nv) {
          const float mx = fmaxf(fmaxf(q[u].x, q[u].y), fmaxf(q[u].z, q[u].w)) * kL2e;
          const float ls = ex2_approx(fmaf(q[u].x, kL2e, -mx)) + ex2_approx(fmaf(q[u].y, kL2e, -mx)) +
                           ex2_approx(fmaf(q[u].z, kL2e, -mx)) + ex2_approx(fmaf(q[u].w, kL2e, -mx));
          online_merge2(m, s, mx, ls);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      online_merge2(m, s, m2, s2);
    }
    __syncthreads();  // the previous row's reads of sm_m / sm_s are done
    if ((tid & 31) == 0) { sm_m[tid >> 5] = m; sm_s[tid >> 5] = s; }
    __syncthreads();
    m = sm_m[0];
    s = sm_s[0];
    for (int i = 1; i < kCeThreads / 32; ++i) online_merge2(m, s, sm_m[i], sm_s[i]);
    const float lse2 = m + log2f(s);  // log2 of the softmax denominator
    const int label = labels[row];
    const bool lab_ok = label >= 0 && label < V;
    if (tid == 0) {
      if (!lab_ok) set_device_error(err, kDevErrBadToken);
      loss_rows[row] = lse2 * kLn2 - (lab_ok ? z[label] : 0.f);
    }
    bf16* dr = dz + (long long)row * lddz;
    for (int v0 = tid; v0 < nv; v0 += kCeUnroll * kCeThreads) {
      float4 q[kCeUnroll];
#pragma unroll
      for (int u = 0; u < kCeUnroll; ++u) {
        const int v = v0 + u * kCeThreads;
        if (v < nv) q[u] = reinterpret_cast<const float4*>(z)[v];
      }
#pragma unroll
      for (int u = 0; u < kCeUnroll; ++u) {
        const int v = v0 + u * kCeThreads;
        if (v >= nv) continue;
        const int j = v * 4;
        float p0 = ex2_approx(fmaf(q[u].x, kL2e, -lse2)), p1 = ex2_approx(fmaf(q[u].y, kL2e, -lse2));
        float p2 = ex2_approx(fmaf(q[u].z, kL2e, -lse2)), p3 = ex2_approx(fmaf(q[u].w, kL2e, -lse2));
        if (j == label) p0 -= 1.f;
        if (j + 1 == label) p1 -= 1.f;
        if (j + 2 == label) p2 -= 1.f;
        if (j + 3 == label) p3 -= 1.f;
        uint2 w;
        w.x = pack_bf16x2(p0 * scale, p1 * scale);
        w.y = pack_bf16x2(p2 * scale, p3 * scale);
        *reinterpret_cast<uint2*>(dr + j) = w;
      }
    }
  }
}

// dst = bf16(src), 8 elements per thread where the tail allows.
__global__ void f32_to_bf16_kernel(const float* __restrict__ src, bf16* __restrict__ dst, long long n) {
  const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i + 8 <= n) {
    float f[8];
    load_f32x8(src + i, f);
    store_bf16x8(dst + i, f);
  } else {
    for (long long j = i; j < n; ++j) dst[j] = __float2bfloat16_rn(src[j]);
  }
}

// Single-block fixed-order sum (fp64 accumulation).
__global__ void sum_kernel(const float* __restrict__ x, int n, float* __restrict__ out) {
  __shared__ double red[1024];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += (double)x[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = (float)red[0];
}

__global__ void check_ids_kernel(const int32_t* __restrict__ ids, int n, int V, int32_t* bad) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int v = ids[i];
    if (v < 0 || v >= V) *bad = 1;
  }
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int convert_f32_bf16(const float* src, void* dst, long long n, cudaStream_t stream) {
  if (n < 0 || !al16(src) || !al16(dst)) return MT_EINVAL;
  if (n == 0) return MT_OK;
  const long long threads = (n + 7) / 8;
  f32_to_bf16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(src, (bf16*)dst, n);
  return launch_ok();
}
}  // namespace mt

using namespace mt;

extern "C" {

int mt_k_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int c_f32,
              const void* R, int64_t ldr, int M, int N, int K, void* stream) {
  return gemm_abt(A, lda, B, ldb, C, ldc, c_f32, R, ldr, M, N, K, (cudaStream_t)stream);
}

int mt_k_gemm_ex(const void* A, int64_t lda, int a_mn_major, const void* B, int64_t ldb, int b_mn_major, void* C,
                 int64_t ldc, int c_f32, const void* R, int64_t ldr, int M, int N, int K, void* stream) {
  return gemm_ex(A, lda, a_mn_major, B, ldb, b_mn_major, C, ldc, c_f32, R, ldr, M, N, K, (cudaStream_t)stream);
}

int mt_k_gemm_rope(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int M, int N, int K,
                   const float* cos_t, const float* sin_t, int rot_cols, int hd, int seq, void* stream) {
  return gemm_rope(A, lda, B, ldb, C, ldc, M, N, K, cos_t, sin_t, rot_cols, hd, seq, (cudaStream_t)stream);
}

int mt_k_gemm_swiglu_fwd(const void* A, int64_t lda, const void* W, int64_t ldw, void* gu, int64_t ldgu, void* a,
                         int64_t lda_out, int M, int f, int K, void* stream) {
  return gemm_swiglu_fwd(A, lda, W, ldw, gu, ldgu, a, lda_out, M, f, K, (cudaStream_t)stream);
}

int mt_k_gemm_swiglu_bwd(const void* dy, int64_t lddy, const void* W, int64_t ldw, const void* gu, int64_t ldgu,
                         void* dgu, int64_t lddgu, int M, int f, int K, void* stream) {
  return gemm_swiglu_bwd(dy, lddy, W, ldw, gu, ldgu, dgu, lddgu, M, f, K, (cudaStream_t)stream);
}

int mt_k_gemm_wgrad(const void* dY, int64_t lddy, const void* X, int64_t ldx, void* G, int64_t ldg, int M, int N,
                    int K, float* ws, int64_t ws_elems, void* stream) {
  if (ws_elems < 0) return MT_EINVAL;
  return gemm_wgrad(dY, lddy, 1, X, ldx, 1, G, ldg, M, N, K, ws, (size_t)ws_elems, (cudaStream_t)stream);
}

int mt_k_gemm_tile_policy(int policy) { return gemm_tile_policy(policy); }

int mt_k_gemm_splitk(int M, int N, int K) { return (M <= 0 || N <= 0 || K <= 0) ? 1 : splitk_factor(M, N, K); }

int64_t mt_k_gemm_wgrad_ws(int M, int N) { return (M <= 0 || N <= 0) ? 0 : (int64_t)splitk_ws_elems(M, N); }

int mt_k_rmsnorm_fwd(const void* x, int x_f32, const void* w, void* y, float* rstd, int M, int d, float eps,
                     void* stream) {
  if (M < 0 || d <= 0 || d % 8 || !al16(x) || !al16(w) || !al16(y)) return MT_EINVAL;
  if (M == 0) return MT_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int vpt = (d / 8 + kNormFwdThreads - 1) / kNormFwdThreads;
  if (vpt <= 8) {
    auto go = [&](auto xt, auto vt) {
      using TX = decltype(xt);
      constexpr int V = decltype(vt)::value;
      rmsnorm_fwd_row_kernel<TX, V><<<M, kNormFwdThreads, 0, st>>>((const TX*)x, (const bf16*)w, (bf16*)y, rstd, d,
                                                                    eps);
    };
    auto by_vpt = [&](auto xt) {
      switch (vpt) {
        case 1: go(xt, std::integral_constant<int, 1>{}); break;
        case 2: go(xt, std::integral_constant<int, 2>{}); break;
        case 3: go(xt, std::integral_constant<int, 3>{}); break;
        case 4: go(xt, std::integral_constant<int, 4>{}); break;
        case 5: go(xt, std::integral_constant<int, 5>{}); break;
        case 6: go(xt, std::integral_constant<int, 6>{}); break;
        case 7: go(xt, std::integral_constant<int, 7>{}); break;
        default: go(xt, std::integral_constant<int, 8>{}); break;
      }
    };
    if (x_f32) by_vpt(0.f);
    else by_vpt(bf16{});
    return launch_ok();
  }
  // longer rows: one warp per row, two passes over x
  const int rows_per_block = 8;
  const dim3 grid((M + rows_per_block - 1) / rows_per_block), block(32 * rows_per_block);
  if (x_f32)
    rmsnorm_fwd_kernel<float><<<grid, block, 0, (cudaStream_t)stream>>>((const float*)x, (const bf16*)w, (bf16*)y,
                                                                        rstd, M, d, eps);
  else
    rmsnorm_fwd_kernel<bf16><<<grid, block, 0, (cudaStream_t)stream>>>((const bf16*)x, (const bf16*)w, (bf16*)y,
                                                                       rstd, M, d, eps);
  return launch_ok();
}

int mt_k_rmsnorm_bwd_parts(int M) { return M < kNormBwdMaxParts ? (M > 0 ? M : 1) : kNormBwdMaxParts; }

int mt_k_rmsnorm_bwd(const float* dy, const void* x, int x_f32, const void* w, const float* rstd, const float* dres,
                     float* dx_f32, void* dx_bf16, float* partial, void* dw_out, int M, int d, void* stream) {
  if (M < 0 || d <= 0 || d % 8 || d > 8 * kNormBwdVec * 32 * kNormBwdMaxWarps) return MT_EINVAL;
  if (!al16(dy) || !al16(x) || !al16(w) || (dres && !al16(dres)) || (dx_f32 && !al16(dx_f32)) ||
      (dx_bf16 && !al16(dx_bf16)) || !al16(partial))
    return MT_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  // 16 elements a thread (more warps per row, more loads in flight) where
  // 8 warps cover the row, else 32
  const int vec = d <= 8 * 2 * 32 * kNormBwdMaxWarps ? 2 : kNormBwdVec;
  // row groups: one wave of resident blocks (no tail wave, and fewer dw
  // partial rows for the column sums), at most mt_k_rmsnorm_bwd_parts(M)
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MT_ECUDA;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  const int w_row = (d + 8 * vec * 32 - 1) / (8 * vec * 32);
  const int resident = sms[dev] * (vec == 2 ? 3 : 2) * (8 / w_row > 0 ? 8 / w_row : 1);
  const int parts = std::min(mt_k_rmsnorm_bwd_parts(M), std::max(resident, 1));
  if (M > 0) {
    const int W = w_row;  // warps per row
    const int rpg = (M + parts - 1) / parts;
    const int ngroups = (M + rpg - 1) / rpg;  // every group has at least one row
    auto go = [&](auto kernel, int w_, auto xt) {
      using TX = decltype(xt);
      const int g = 8 / w_ > 0 ? 8 / w_ : 1;
      kernel<<<(ngroups + g - 1) / g, 32 * w_ * g, 0, st>>>(dy, (const TX*)x, (const bf16*)w, rstd, dres, dx_f32,
                                                           (bf16*)dx_bf16, partial, M, d, ngroups, rpg);
    };
    auto by_w = [&](auto xt, auto vt) {
      using TX = decltype(xt);
      constexpr int V = decltype(vt)::value;
      switch (W) {
        case 1: go(rmsnorm_bwd_kernel<1, TX, V>, 1, xt); break;
        case 2: go(rmsnorm_bwd_kernel<2, TX, V>, 2, xt); break;
        case 3: go(rmsnorm_bwd_kernel<3, TX, V>, 3, xt); break;
        case 4: go(rmsnorm_bwd_kernel<4, TX, V>, 4, xt); break;
        case 5: go(rmsnorm_bwd_kernel<5, TX, V>, 5, xt); break;
        case 6: go(rmsnorm_bwd_kernel<6, TX, V>, 6, xt); break;
        case 7: go(rmsnorm_bwd_kernel<7, TX, V>, 7, xt); break;
        default: go(rmsnorm_bwd_kernel<8, TX, V>, 8, xt); break;
      }
    };
    auto dispatch = [&](auto xt) {
      if (vec == 2) by_w(xt, std::integral_constant<int, 2>{});
      else by_w(xt, std::integral_constant<int, kNormBwdVec>{});
    };
    if (x_f32) dispatch(0.f);
    else dispatch(bf16{});
    colsum_to_bf16_kernel<<<(d + 31) / 32, 32 * kColsumClasses, 0, st>>>(partial, ngroups, d, (bf16*)dw_out);
  } else {
    cudaMemsetAsync(partial, 0, sizeof(float) * d, st);
    colsum_to_bf16_kernel<<<(d + 31) / 32, 32 * kColsumClasses, 0, st>>>(partial, 1, d, (bf16*)dw_out);
  }
  return launch_ok();
}

int mt_k_rope(void* x, int64_t ld, int B, int s, int n_rot_heads, int hd, const float* cos_t, const float* sin_t,
              int inverse, void* stream) {
  if (B < 0 || s <= 0 || n_rot_heads < 0 || hd < 4 || hd % 4 || ld < (int64_t)n_rot_heads * hd || ld % 2)
    return MT_EINVAL;
  const int threads = 256;
  if (hd % 16 == 0 && ld % 8 == 0 && al16(x) && al16(cos_t) && al16(sin_t)) {
    const long long total = (long long)B * s * n_rot_heads * (hd / 16);
    if (total == 0) return MT_OK;
    rope_vec_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, (cudaStream_t)stream>>>(
        (bf16*)x, ld, B * s, s, n_rot_heads, hd, cos_t, sin_t, inverse ? -1.f : 1.f);
    return launch_ok();
  }
  const long long total = (long long)B * s * n_rot_heads * (hd / 4);
  if (total == 0) return MT_OK;
  rope_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, (cudaStream_t)stream>>>(
      (bf16*)x, ld, B * s, s, n_rot_heads, hd, cos_t, sin_t, inverse ? -1.f : 1.f);
  return launch_ok();
}

int mt_k_swiglu_fwd(const void* gu, void* a, int M, int f, void* stream) {
  if (M < 0 || f <= 0 || f % 8 || !al16(gu) || !al16(a)) return MT_EINVAL;
  const long long total = (long long)M * (f / 8);
  if (total == 0) return MT_OK;
  swiglu_fwd_kernel<<<(unsigned)((total + 255) / 256), 256, 0, (cudaStream_t)stream>>>((const bf16*)gu, (bf16*)a,
                                                                                      M, f);
  return launch_ok();
}

int mt_k_swiglu_bwd(const void* da, const void* gu, void* dgu, int M, int f, void* stream) {
  if (M < 0 || f <= 0 || f % 8 || !al16(da) || !al16(gu) || !al16(dgu)) return MT_EINVAL;
  const long long total = (long long)M * (f / 8);
  if (total == 0) return MT_OK;
  swiglu_bwd_kernel<<<(unsigned)((total + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
      (const bf16*)da, (const bf16*)gu, (bf16*)dgu, M, f);
  return launch_ok();
}

int mt_k_cross_entropy(const float* logits, int64_t ldl, const int32_t* labels, void* dz, int64_t lddz,
                       float* loss_rows, int M, int V, float scale, void* stream) {
  if (M < 0 || V <= 0 || V % 4 || ldl < V || ldl % 4 || lddz < V || lddz % 4 || !al16(logits)) return MT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(dz) & 7) != 0) return MT_EINVAL;
  if (M == 0) return MT_OK;
  // rows in flight: two blocks per SM, one for long rows (about 48 MB of
  // logits in flight at most where the rows allow)
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MT_ECUDA;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  const long long per_row = 4LL * V;
  long long blocks = (48LL << 20) / per_row;
  blocks = std::max<long long>(sms[dev], std::min<long long>(blocks, 2LL * sms[dev]));
  blocks = std::min<long long>(blocks, M);
  cross_entropy_kernel<<<(unsigned)blocks, kCeThreads, 0, (cudaStream_t)stream>>>(
      logits, ldl, labels, (bf16*)dz, lddz, loss_rows, M, V, scale, device_error_word());
  return launch_ok();
}

int mt_k_sum(const float* x, int n, float* out, void* stream) {
  if (n < 0) return MT_EINVAL;
  sum_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(x, n, out);
  return launch_ok();
}

int mt_k_embedding_fwd(const void* E, const int32_t* tok, void* x, int x_f32, int M, int d, int V, void* stream) {
  if (M < 0 || d <= 0 || d % 8 || V <= 0 || !al16(E) || !al16(x)) return MT_EINVAL;
  if (M == 0) return MT_OK;
  if (x_f32)
    embedding_fwd_f32_kernel<<<(M + 7) / 8, 256, 0, (cudaStream_t)stream>>>((const bf16*)E, tok, (float*)x, M, d, V,
                                                                            device_error_word());
  else
    embedding_fwd_kernel<<<(M + 7) / 8, 256, 0, (cudaStream_t)stream>>>((const bf16*)E, tok, (bf16*)x, M, d, V,
                                                                        device_error_word());
  return launch_ok();
}

int64_t mt_k_embedding_bwd_work(int M, int V) { return 2LL * V + 1 + (M > 0 ? M : 0); }

int mt_k_embedding_bwd(const float* dx, const int32_t* tok, void* dE, int M, int d, int V, int32_t* work,
                       void* stream) {
  if (M < 0 || d <= 0 || d % 4 || V <= 0 || !al16(dx) || (reinterpret_cast<uintptr_t>(dE) & 7)) return MT_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  token_sort_kernel<<<1, kSortThreads, 0, st>>>(tok, M, V, work, device_error_word());
  dim3 grid(V, (d / 4 + 255) / 256);
  embedding_bwd_reduce_kernel<<<grid, 256, 0, st>>>(dx, work, (bf16*)dE, d, V);
  return launch_ok();
}

int mt_k_check_ids(const int32_t* ids, int n, int V, int32_t* bad, void* stream) {
  if (n < 0 || V <= 0) return MT_EINVAL;
  if (n == 0) return MT_OK;
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  check_ids_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(ids, n, V, bad);
  return launch_ok();
}

int mt_k_device_error(int* code, int reset) {
  if (!code) return MT_EINVAL;
  int* w = device_error_word();
  if (!w) return MT_ECUDA;
  if (cudaMemcpy(code, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MT_ECUDA;
  if (reset && cudaMemset(w, 0, sizeof(int)) != cudaSuccess) return MT_ECUDA;
  return MT_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Embedding backward that allocates nothing (see mt_k_embedding_bwd_noalloc
// in mt_kernels.h). Its sort workspace lives in this fixed device array,
// which every GPU that loads the library keeps until the process exits.
namespace {

constexpr int kNoAllocMaxV = MT_NOALLOC_EMBED_MAX_VOCAB;
constexpr int kNoAllocMaxM = MT_NOALLOC_EMBED_MAX_TOKENS;
static __device__ __align__(256) int32_t g_embed_bwd_scratch[2 * kNoAllocMaxV + 1 + kNoAllocMaxM];

// Device address of g_embed_bwd_scratch for the current device, looked up
// once per device (host code may not use the symbol itself: on the host it
// names a stand-in, not device memory).
int32_t* embed_scratch_address(cudaError_t* err) {
  static int32_t* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_embed_bwd_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" int mt_k_embedding_bwd_noalloc(const float* dx, const int32_t* tok, void* dE, int M, int d, int V,
                                          void* stream) {
  if (M > kNoAllocMaxM || V > kNoAllocMaxV) {
    set_last_error_message("mt_k_embedding_bwd_noalloc: M (" + std::to_string(M) + ") or V (" +
                           std::to_string(V) + ") above the fixed workspace limits of " +
                           std::to_string(kNoAllocMaxM) + " tokens and " + std::to_string(kNoAllocMaxV) +
                           " vocabulary rows");
    return MT_EINVAL;
  }
  if (M < 0 || d <= 0 || d % 4 || V <= 0 || !al16(dx) || (reinterpret_cast<uintptr_t>(dE) & 7)) return MT_EINVAL;
  cudaError_t err = cudaSuccess;
  int32_t* work = embed_scratch_address(&err);
  if (!work) {
    set_last_error_message(std::string("mt_k_embedding_bwd_noalloc: cudaGetSymbolAddress failed: ") +
                           cudaGetErrorString(err));
    return MT_ECUDA;
  }
  // The sort kernel clears its own counters and rewrites every bucket start
  // and every position it later reads, so nothing left by an earlier call
  // is used. No error word is passed: the library's error word is allocated
  // on first use, which this entry point must not do.
  cudaStream_t st = (cudaStream_t)stream;
  token_sort_kernel<<<1, kSortThreads, 0, st>>>(tok, M, V, work, nullptr);
  dim3 grid(V, (d / 4 + 255) / 256);
  embedding_bwd_reduce_kernel<<<grid, 256, 0, st>>>(dx, work, (bf16*)dE, d, V);
  return launch_ok();
}
