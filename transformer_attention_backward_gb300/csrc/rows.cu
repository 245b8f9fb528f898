// Row-wise memory-bound kernels: softmax backward, RoPE backward, RMSNorm
// backward, and the bounded-wait self test.
//
//   softmax_bwd : softmaxBackward, "Hesper.Training.VerifiedBackward" section Softmax
//   rope_bwd    : ropeBackward, section RoPE (rotation by -theta)
//   rmsnorm_bwd_dgamma : the same plus the scale gradient dgamma = sum over
//                 rows of dy x / rms (the forward y = gamma x / rms is linear
//                 in gamma; the norm's other gradient)
//   rmsnorm_bwd : rmsNormBackward, section RMSNorm; the two row reductions the
//                 Hesper WGSL kernel runs as separate shared-memory phases
//                 ("RMSNorm backward kernel" fix, Hesper pull request #1) are
//                 independent sums, so they are taken here in one pass over
//                 registers.
#include <math.h>

#include "abw_host.h"

namespace abw {
namespace {

constexpr int kRowThreads = 256;

// Sum of two values across a block of kRowThreads threads.
__device__ __forceinline__ float2 block_sum2(float a, float b, float2 *red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = make_float2(a, b);
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  if (w == 0) {
    t = l < kRowThreads / 32 ? red[l] : make_float2(0.f, 0.f);
    t.x = warp_sum(t.x);
    t.y = warp_sum(t.y);
    if (l == 0) red[kRowThreads / 32] = t;
  }
  __syncthreads();
  return red[kRowThreads / 32];
}

// ---------------------------------------------------------------------------
// softmax backward: one warp per row, the row held in registers
// (n <= 128 * NV, n % 4 == 0), 16-byte loads.
// ---------------------------------------------------------------------------
template <int NV>
__global__ void __launch_bounds__(256) softmax_bwd_warp_v4(const float *__restrict__ s,
                                                           const float *__restrict__ dy,
                                                           float *__restrict__ dx, int rows, int n) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4 *s4 = reinterpret_cast<const float4 *>(s + static_cast<size_t>(row) * n);
  const float4 *d4 = reinterpret_cast<const float4 *>(dy + static_cast<size_t>(row) * n);
  float4 *o4 = reinterpret_cast<float4 *>(dx + static_cast<size_t>(row) * n);
  const int n4 = n >> 2;
  float4 sv[NV], dv[NV];
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = lane + 32 * k;
    if (i < n4) {
      sv[k] = __ldg(s4 + i);
      dv[k] = __ldg(d4 + i);
      acc += sv[k].x * dv[k].x + sv[k].y * dv[k].y + sv[k].z * dv[k].z + sv[k].w * dv[k].w;
    }
  }
  const float dot = warp_sum(acc);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = lane + 32 * k;
    if (i < n4) {
      float4 r;
      r.x = sv[k].x * (dv[k].x - dot);
      r.y = sv[k].y * (dv[k].y - dot);
      r.z = sv[k].z * (dv[k].z - dot);
      r.w = sv[k].w * (dv[k].w - dot);
      o4[i] = r;
    }
  }
}

// Any n: one block per row, two passes (the second mostly from L1/L2).
__global__ void __launch_bounds__(kRowThreads) softmax_bwd_block(const float *__restrict__ s,
                                                                 const float *__restrict__ dy,
                                                                 float *__restrict__ dx, int n) {
  __shared__ float2 red[kRowThreads / 32 + 1];
  const size_t base = static_cast<size_t>(blockIdx.x) * n;
  float acc = 0.f;
  for (int i = threadIdx.x; i < n; i += kRowThreads) acc += s[base + i] * dy[base + i];
  const float dot = block_sum2(acc, 0.f, red).x;
  for (int i = threadIdx.x; i < n; i += kRowThreads) dx[base + i] = s[base + i] * (dy[base + i] - dot);
}

// ---------------------------------------------------------------------------
// RoPE backward.  One block per (b, t) row of H*D values.  The D/2 angles of
// the row are formed once per block: with explicit theta they are read; else
// theta_i = (pos0 + t) * inv_freq_i is formed in double precision, reduced
// modulo 2 pi in double, and only then rounded to float for sincosf (an fp32
// product p * inv_freq loses ~p * 2^-24 rad, which at p ~ 8e3 is ~5e-4 rad).
// ---------------------------------------------------------------------------
struct RopeParams {
  const float *dy;
  float *dx;
  const float *theta;     // [B*T][D/2] or null
  int T, H, D, pos0, interleaved;
  double inv_freq[256];   // base^(-2i/D), formed on the host in double
};

constexpr int kRopeBatch = 8;
__global__ void __launch_bounds__(128) rope_bwd_kernel(const __grid_constant__ RopeParams p) {
  __shared__ float2 cs[256];
  const int row = blockIdx.x;           // b * T + t
  const int t = row % p.T;
  const int half = p.D >> 1;
  const size_t base = static_cast<size_t>(row) * p.H * p.D;
  const int npairs = p.H * half;
  const bool vec = p.interleaved && (p.D & 3) == 0;   // two pairs per float4
  const float4 *src = reinterpret_cast<const float4 *>(p.dy + base);
  float4 *dst = reinterpret_cast<float4 *>(p.dx + base);
  const int n4 = npairs >> 1;
  // The first batch of row values is requested before the angles are
  // formed, so the angle arithmetic runs while the loads are in flight.
  // kRopeBatch vectors per thread are loaded before the first is written,
  // so a thread waits for one memory latency per batch, not per vector
  // (each element is read before it is written, so dx may be dy).
  float4 y[kRopeBatch];
  if (vec) {
#pragma unroll
    for (int u = 0; u < kRopeBatch; ++u) {
      const int i = threadIdx.x + u * blockDim.x;
      if (i < n4) y[u] = src[i];
    }
  }
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    float th;
    if (p.theta) {
      th = p.theta[static_cast<size_t>(row) * half + i];
    } else {
      // reduced to [-pi, pi] in double (a multiply by 1 / 2 pi, not a divide:
      // double division is slow on this GPU, and a last-bit difference in
      // the quotient only picks another multiple of 2 pi)
      const double a = static_cast<double>(p.pos0 + t) * p.inv_freq[i];
      const double twopi = 6.283185307179586476925286766559, inv_twopi = 0.15915494309189533576888376337251;
      th = static_cast<float>(fma(-twopi, rint(a * inv_twopi), a));
    }
    float sn, c;
    sincosf(th, &sn, &c);
    cs[i] = make_float2(c, sn);
  }
  __syncthreads();
  if (vec) {
    const int q4 = p.D >> 2;
    for (int i0 = threadIdx.x;;) {
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < n4) {
          const int pi = (i % q4) * 2;   // pair index within the head
          const float2 a = cs[pi], b = cs[pi + 1];
          float4 r;
          r.x = y[u].x * a.x + y[u].y * a.y;
          r.y = -y[u].x * a.y + y[u].y * a.x;
          r.z = y[u].z * b.x + y[u].w * b.y;
          r.w = -y[u].z * b.y + y[u].w * b.x;
          dst[i] = r;
        }
      }
      i0 += kRopeBatch * blockDim.x;
      if (i0 >= n4) break;
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < n4) y[u] = src[i];
      }
    }
  } else {
    for (int i0 = threadIdx.x; i0 < npairs; i0 += kRopeBatch * blockDim.x) {
      float y0[kRopeBatch], y1[kRopeBatch];
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < npairs) {
          const int h = i / half, pi = i % half;
          const size_t o = base + static_cast<size_t>(h) * p.D;
          y0[u] = p.dy[o + (p.interleaved ? 2 * pi : pi)];
          y1[u] = p.dy[o + (p.interleaved ? 2 * pi + 1 : pi + half)];
        }
      }
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < npairs) {
          const int h = i / half, pi = i % half;
          const size_t o = base + static_cast<size_t>(h) * p.D;
          const float2 a = cs[pi];
          p.dx[o + (p.interleaved ? 2 * pi : pi)] = y0[u] * a.x + y1[u] * a.y;
          p.dx[o + (p.interleaved ? 2 * pi + 1 : pi + half)] = -y0[u] * a.y + y1[u] * a.x;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// RMSNorm backward.  One block per row; with n % 4 == 0 and n <= 1024 * NV the
// row stays in registers between the reduction and the output.
// ---------------------------------------------------------------------------
template <bool XBF16>
__device__ __forceinline__ float4 load_x4(const void *x, size_t idx4) {
  if (XBF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(x) + idx4);
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
  } else {
    return __ldg(reinterpret_cast<const float4 *>(x) + idx4);
  }
}

template <bool DXBF16>
__device__ __forceinline__ void store_dx4(void *dx, size_t idx4, float4 v) {
  if (DXBF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    reinterpret_cast<uint2 *>(dx)[idx4] = u;
  } else {
    reinterpret_cast<float4 *>(dx)[idx4] = v;
  }
}

// For calls of many rows (kCap), rows of up to 2 x 1024 elements keep 8
// blocks (2048 threads) resident per SM and rows of up to 3 x 1024 keep 7, so
// about 1,000 rows run in one wave and long calls keep more rows in flight
// (the row keeps x and dy * gamma in registers, not dy and gamma apart; at 7
// blocks a few values of the longer rows go to the stack, which calls of few
// rows, one wave anyway, do without).
template <int NV, bool kCap>
constexpr int rms_min_blocks() { return !kCap ? 1 : NV <= 2 ? 8 : NV == 3 ? 7 : 1; }

template <bool XBF16, bool DXBF16, int NV, bool kCap>
__global__ void __launch_bounds__(kRowThreads, rms_min_blocks<NV, kCap>()) rmsnorm_bwd_v4(const void *__restrict__ x,
                                                              const float *__restrict__ gamma,
                                                              const float *__restrict__ dy,
                                                              void *__restrict__ dx, int n, float eps) {
  __shared__ float2 red[kRowThreads / 32 + 1];
  const int n4 = n >> 2;
  const size_t rb = static_cast<size_t>(blockIdx.x) * n4;
  float4 xv[NV], gv[NV];   // x and dy * gamma
  float ss = 0.f, cs = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = threadIdx.x + kRowThreads * k;
    if (i < n4) {
      xv[k] = load_x4<XBF16>(x, rb + i);
      const float4 d = __ldg(reinterpret_cast<const float4 *>(dy) + rb + i);
      const float4 g = __ldg(reinterpret_cast<const float4 *>(gamma) + i);
      gv[k] = make_float4(d.x * g.x, d.y * g.y, d.z * g.z, d.w * g.w);
      ss += xv[k].x * xv[k].x + xv[k].y * xv[k].y + xv[k].z * xv[k].z + xv[k].w * xv[k].w;
      cs += gv[k].x * xv[k].x + gv[k].y * xv[k].y + gv[k].z * xv[k].z + gv[k].w * xv[k].w;
    }
  }
  const float2 sums = block_sum2(ss, cs, red);
  const float ms = sums.x / static_cast<float>(n) + eps;   // rms^2
  const float inv_rms = rsqrtf(ms);
  const float coef = sums.y / (static_cast<float>(n) * ms);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = threadIdx.x + kRowThreads * k;
    if (i < n4) {
      float4 r;
      r.x = (gv[k].x - xv[k].x * coef) * inv_rms;
      r.y = (gv[k].y - xv[k].y * coef) * inv_rms;
      r.z = (gv[k].z - xv[k].z * coef) * inv_rms;
      r.w = (gv[k].w - xv[k].w * coef) * inv_rms;
      store_dx4<DXBF16>(dx, rb + i, r);
    }
  }
}

// Any n: two passes over global memory.
template <bool XBF16, bool DXBF16>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_bwd_any(const void *__restrict__ x,
                                                               const float *__restrict__ gamma,
                                                               const float *__restrict__ dy,
                                                               void *__restrict__ dx, int n, float eps) {
  __shared__ float2 red[kRowThreads / 32 + 1];
  const size_t rb = static_cast<size_t>(blockIdx.x) * n;
  auto ldx = [&](size_t i) -> float {
    return XBF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(x)[i])
                 : reinterpret_cast<const float *>(x)[i];
  };
  float ss = 0.f, cs = 0.f;
  for (int i = threadIdx.x; i < n; i += kRowThreads) {
    const float xi = ldx(rb + i);
    ss += xi * xi;
    cs += dy[rb + i] * gamma[i] * xi;
  }
  const float2 sums = block_sum2(ss, cs, red);
  const float ms = sums.x / static_cast<float>(n) + eps;
  const float inv_rms = rsqrtf(ms);
  const float coef = sums.y / (static_cast<float>(n) * ms);
  for (int i = threadIdx.x; i < n; i += kRowThreads) {
    const float r = (dy[rb + i] * gamma[i] - ldx(rb + i) * coef) * inv_rms;
    if (DXBF16)
      reinterpret_cast<__nv_bfloat16 *>(dx)[rb + i] = __float2bfloat16_rn(r);
    else
      reinterpret_cast<float *>(dx)[rb + i] = r;
  }
}

template <bool XB, bool DB, bool kCap>
void rms_launch(int nv, const void *x, const float *g, const float *dy, void *dx, int rows, int n, float eps,
                cudaStream_t st) {
  if (nv <= 1)
    rmsnorm_bwd_v4<XB, DB, 1, kCap><<<rows, kRowThreads, 0, st>>>(x, g, dy, dx, n, eps);
  else if (nv <= 2)
    rmsnorm_bwd_v4<XB, DB, 2, kCap><<<rows, kRowThreads, 0, st>>>(x, g, dy, dx, n, eps);
  else if (nv <= 3)
    rmsnorm_bwd_v4<XB, DB, 3, kCap><<<rows, kRowThreads, 0, st>>>(x, g, dy, dx, n, eps);
  else if (nv <= 4)
    rmsnorm_bwd_v4<XB, DB, 4, kCap><<<rows, kRowThreads, 0, st>>>(x, g, dy, dx, n, eps);
  else
    rmsnorm_bwd_v4<XB, DB, 8, kCap><<<rows, kRowThreads, 0, st>>>(x, g, dy, dx, n, eps);
}

template <bool XB, bool DB>
cudaError_t rms_dispatch(const void *x, const float *g, const float *dy, void *dx, int rows, int n, float eps,
                         cudaStream_t st) {
  const int n4 = n / 4;
  const int nv = (n4 + kRowThreads - 1) / kRowThreads;
  if (n % 4 != 0 || nv > 8) {
    rmsnorm_bwd_any<XB, DB><<<rows, kRowThreads, 0, st>>>(x, g, dy, dx, n, eps);
    return cudaGetLastError();
  }
  // more rows than 4 blocks per SM hold: the register-capped form
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (rows > 4 * sms)
    rms_launch<XB, DB, true>(nv, x, g, dy, dx, rows, n, eps, st);
  else
    rms_launch<XB, DB, false>(nv, x, g, dy, dx, rows, n, eps, st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RMSNorm backward with the scale gradient: dx as above (optional) and
// dgamma_i = sum over rows of dy_i x_i / rms.  Blocks stride over the rows;
// each thread keeps its columns' dgamma partial sums in registers across its
// block's rows and adds them into the zeroed output once, with 16-byte
// vector reductions.
// ---------------------------------------------------------------------------
// The launch puts up to 4 blocks per SM; rows of up to 3 x 1024 elements are
// held to the registers that lets all of them be resident at once.
template <int NV>
constexpr int rms_dg_min_blocks() { return NV <= 3 ? 4 : 1; }

template <bool XBF16, bool DXBF16, int NV, bool DX>
__global__ void __launch_bounds__(kRowThreads, rms_dg_min_blocks<NV>()) rmsnorm_bwd_dgamma_v4(const void *__restrict__ x,
                                                                     const float *__restrict__ gamma,
                                                                     const float *__restrict__ dy,
                                                                     void *__restrict__ dx, float *__restrict__ dgamma,
                                                                     int rows, int n, float eps) {
  __shared__ float2 red[kRowThreads / 32 + 1];
  const int n4 = n >> 2;
  float4 gv[NV], ga[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = threadIdx.x + kRowThreads * k;
    gv[k] = (DX && i < n4) ? __ldg(reinterpret_cast<const float4 *>(gamma) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    ga[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const size_t rb = static_cast<size_t>(row) * n4;
    float4 xv[NV], dv[NV];
    float ss = 0.f, cs = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int i = threadIdx.x + kRowThreads * k;
      if (i < n4) {
        xv[k] = load_x4<XBF16>(x, rb + i);
        dv[k] = __ldg(reinterpret_cast<const float4 *>(dy) + rb + i);
        ss += xv[k].x * xv[k].x + xv[k].y * xv[k].y + xv[k].z * xv[k].z + xv[k].w * xv[k].w;
        if (DX)
          cs += dv[k].x * gv[k].x * xv[k].x + dv[k].y * gv[k].y * xv[k].y + dv[k].z * gv[k].z * xv[k].z +
                dv[k].w * gv[k].w * xv[k].w;
      }
    }
    const float2 sums = block_sum2(ss, cs, red);
    const float ms = sums.x / static_cast<float>(n) + eps;   // rms^2
    const float inv_rms = rsqrtf(ms);
    const float coef = sums.y / (static_cast<float>(n) * ms);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int i = threadIdx.x + kRowThreads * k;
      if (i < n4) {
        ga[k].x = fmaf(dv[k].x * xv[k].x, inv_rms, ga[k].x);
        ga[k].y = fmaf(dv[k].y * xv[k].y, inv_rms, ga[k].y);
        ga[k].z = fmaf(dv[k].z * xv[k].z, inv_rms, ga[k].z);
        ga[k].w = fmaf(dv[k].w * xv[k].w, inv_rms, ga[k].w);
        if (DX) {
          float4 r;
          r.x = (dv[k].x * gv[k].x - xv[k].x * coef) * inv_rms;
          r.y = (dv[k].y * gv[k].y - xv[k].y * coef) * inv_rms;
          r.z = (dv[k].z * gv[k].z - xv[k].z * coef) * inv_rms;
          r.w = (dv[k].w * gv[k].w - xv[k].w * coef) * inv_rms;
          store_dx4<DXBF16>(dx, rb + i, r);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = threadIdx.x + kRowThreads * k;
    if (i < n4 && blockIdx.x < rows) red_add_f4(dgamma + 4 * i, ga[k]);
  }
}

// Any n: one block per row in turn, per-element reductions into dgamma.
template <bool XBF16, bool DXBF16>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_bwd_dgamma_any(const void *__restrict__ x,
                                                                      const float *__restrict__ gamma,
                                                                      const float *__restrict__ dy,
                                                                      void *__restrict__ dx,
                                                                      float *__restrict__ dgamma, int rows, int n,
                                                                      float eps) {
  __shared__ float2 red[kRowThreads / 32 + 1];
  auto ldx = [&](size_t i) -> float {
    return XBF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(x)[i])
                 : reinterpret_cast<const float *>(x)[i];
  };
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const size_t rb = static_cast<size_t>(row) * n;
    float ss = 0.f, cs = 0.f;
    for (int i = threadIdx.x; i < n; i += kRowThreads) {
      const float xi = ldx(rb + i);
      ss += xi * xi;
      if (dx) cs += dy[rb + i] * gamma[i] * xi;
    }
    const float2 sums = block_sum2(ss, cs, red);
    const float ms = sums.x / static_cast<float>(n) + eps;
    const float inv_rms = rsqrtf(ms);
    const float coef = sums.y / (static_cast<float>(n) * ms);
    for (int i = threadIdx.x; i < n; i += kRowThreads) {
      const float xi = ldx(rb + i), d = dy[rb + i];
      atomicAdd(dgamma + i, d * xi * inv_rms);
      if (dx) {
        const float r = (d * gamma[i] - xi * coef) * inv_rms;
        if (DXBF16)
          reinterpret_cast<__nv_bfloat16 *>(dx)[rb + i] = __float2bfloat16_rn(r);
        else
          reinterpret_cast<float *>(dx)[rb + i] = r;
      }
    }
  }
}

template <bool XB, bool DB, int NV>
void rms_dg_launch(int grid, const void *x, const float *g, const float *dy, void *dx, float *dgamma, int rows, int n,
                   float eps, cudaStream_t st) {
  if (dx)
    rmsnorm_bwd_dgamma_v4<XB, DB, NV, true><<<grid, kRowThreads, 0, st>>>(x, g, dy, dx, dgamma, rows, n, eps);
  else
    rmsnorm_bwd_dgamma_v4<XB, DB, NV, false><<<grid, kRowThreads, 0, st>>>(x, g, dy, dx, dgamma, rows, n, eps);
}

template <bool XB, bool DB>
cudaError_t rms_dg_dispatch(const void *x, const float *g, const float *dy, void *dx, float *dgamma, int rows, int n,
                            float eps, int sms, cudaStream_t st) {
  const int n4 = n / 4;
  const int nv = (n4 + kRowThreads - 1) / kRowThreads;
  const int grid = rows < 4 * sms ? rows : 4 * sms;
  if (n % 4 != 0 || nv > 8)
    rmsnorm_bwd_dgamma_any<XB, DB><<<grid, kRowThreads, 0, st>>>(x, g, dy, dx, dgamma, rows, n, eps);
  else if (nv <= 1)
    rms_dg_launch<XB, DB, 1>(grid, x, g, dy, dx, dgamma, rows, n, eps, st);
  else if (nv <= 2)
    rms_dg_launch<XB, DB, 2>(grid, x, g, dy, dx, dgamma, rows, n, eps, st);
  else if (nv <= 3)
    rms_dg_launch<XB, DB, 3>(grid, x, g, dy, dx, dgamma, rows, n, eps, st);
  else if (nv <= 4)
    rms_dg_launch<XB, DB, 4>(grid, x, g, dy, dx, dgamma, rows, n, eps, st);
  else
    rms_dg_launch<XB, DB, 8>(grid, x, g, dy, dx, dgamma, rows, n, eps, st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self test of the bounded wait: a barrier that expects one arrival which
// never comes.
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(WaitCtl w) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(smem_u32(&bar), 0, w.limit_ns)) atomicOr(w.err, kErrSelfTest);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_softmax_bwd(const float *s, const float *dy, float *dx, int rows, int n, cudaStream_t st) {
  const int n4 = n / 4;
  const int nv = (n4 + 31) / 32;
  const bool vec = (n % 4) == 0 && nv <= 8;
  if (vec) {
    const int blocks = (rows + 7) / 8;   // 8 warps per block, one row each
    if (nv <= 1)
      softmax_bwd_warp_v4<1><<<blocks, 256, 0, st>>>(s, dy, dx, rows, n);
    else if (nv <= 2)
      softmax_bwd_warp_v4<2><<<blocks, 256, 0, st>>>(s, dy, dx, rows, n);
    else if (nv <= 4)
      softmax_bwd_warp_v4<4><<<blocks, 256, 0, st>>>(s, dy, dx, rows, n);
    else
      softmax_bwd_warp_v4<8><<<blocks, 256, 0, st>>>(s, dy, dx, rows, n);
  } else {
    softmax_bwd_block<<<rows, kRowThreads, 0, st>>>(s, dy, dx, n);
  }
  return cudaGetLastError();
}

cudaError_t launch_rope_bwd(const float *dy, float *dx, int B, int T, int H, int D, const float *theta, int pos0,
                            double base, int interleaved, cudaStream_t st) {
  RopeParams p;
  p.dy = dy;
  p.dx = dx;
  p.theta = theta;
  p.T = T;
  p.H = H;
  p.D = D;
  p.pos0 = pos0;
  p.interleaved = interleaved;
  for (int i = 0; i < 256; ++i) p.inv_freq[i] = (i < D / 2 && base > 0) ? pow(base, -2.0 * i / D) : 0.0;
  const long long rows = static_cast<long long>(B) * T;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  rope_bwd_kernel<<<static_cast<unsigned>(rows), 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bwd(const void *x, int x_bf16, const float *gamma, const float *dy, void *dx,
                               int dx_bf16, int rows, int n, float eps, cudaStream_t st) {
  if (x_bf16 && dx_bf16) return rms_dispatch<true, true>(x, gamma, dy, dx, rows, n, eps, st);
  if (x_bf16) return rms_dispatch<true, false>(x, gamma, dy, dx, rows, n, eps, st);
  if (dx_bf16) return rms_dispatch<false, true>(x, gamma, dy, dx, rows, n, eps, st);
  return rms_dispatch<false, false>(x, gamma, dy, dx, rows, n, eps, st);
}

cudaError_t launch_rmsnorm_bwd_dgamma(const void *x, int x_bf16, const float *gamma, const float *dy, void *dx,
                                      int dx_bf16, float *dgamma, int rows, int n, float eps, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(dgamma, 0, static_cast<size_t>(n) * 4, st);
  if (e != cudaSuccess || rows == 0) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (x_bf16 && dx_bf16) return rms_dg_dispatch<true, true>(x, gamma, dy, dx, dgamma, rows, n, eps, sms, st);
  if (x_bf16) return rms_dg_dispatch<true, false>(x, gamma, dy, dx, dgamma, rows, n, eps, sms, st);
  if (dx_bf16) return rms_dg_dispatch<false, true>(x, gamma, dy, dx, dgamma, rows, n, eps, sms, st);
  return rms_dg_dispatch<false, false>(x, gamma, dy, dx, dgamma, rows, n, eps, sms, st);
}

cudaError_t launch_selftest_wait(const WaitCtl &w, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(w);
  return cudaGetLastError();
}

}  // namespace abw
