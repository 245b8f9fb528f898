// The steps of the layer backward around the attention backward, all bound
// by HBM bandwidth:
//
//   relu2_mul_bwd : the FFN's gated activation hidden = ReLU(gate)^2 * up
//                   (Hesper pull request #1, FFN-backward commit, "ReLU^2 x
//                   Mul backward"): dGate = dH up 2 ReLU(gate),
//                   dUp = dH ReLU(gate)^2, element by element.
//   lora_bwd      : parameter gradients of a rank-r adapter y = s B (A x) on
//                   a projection (pull request #1: the chain ends "RoPE
//                   backward -> dQ -> LoRA backward", with the adapter's
//                   input the layer's saved normed activations):
//                   h = x A^T, dB = s dy^T h, dh = s dy B, dA = dh^T x.
//
// The adapter products have rank r <= 16, so they are skinny: per row of x
// and dy the work is r dot products, and the whole step is a stream over x
// and dy.  Two kernels: a row pass forms h and dh (r values per row each,
// into the caller's workspace) and zeroes dA / dB; a column pass adds each
// chunk of rows' outer-product sums into dA and dB with vector reductions.
// x and dy are read twice; the second read comes from L2 for the chain's
// shapes (1024 rows of 2560).
#include "abw_host.h"

namespace abw {
namespace {

// ----------------------------------------------------------------- ReLU^2 x Mul
__device__ __forceinline__ float4 ld_cs_f4(const float *p) {
  float4 v;
  asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

template <bool BF16>
__device__ __forceinline__ float4 ld_act4(const void *p, long long i4) {
  if (BF16) {
    uint2 u;
    asm volatile("ld.global.cs.v2.u32 {%0, %1}, [%2];"
                 : "=r"(u.x), "=r"(u.y)
                 : "l"(reinterpret_cast<const uint2 *>(p) + i4));
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
  } else {
    return ld_cs_f4(reinterpret_cast<const float *>(p) + 4 * i4);
  }
}

template <bool BF16>
__device__ __forceinline__ float ld_act1(const void *p, long long i) {
  return BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]) : reinterpret_cast<const float *>(p)[i];
}

// grid-stride over groups of four elements; the (n % 4) tail by block 0.
// Registers held to 64 so that 4 blocks (1,024 threads) are resident per SM
// (75 left 3; 32 spilled).
template <bool BF16>
__global__ void __launch_bounds__(256, 4) relu2_mul_bwd_kernel(const void *__restrict__ gate, const void *__restrict__ up,
                                                            const float *__restrict__ dh, float *__restrict__ dgate,
                                                            float *__restrict__ dup, long long n) {
  const long long n4 = n >> 2;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 g = ld_act4<BF16>(gate, i), u = ld_act4<BF16>(up, i), d = ld_cs_f4(dh + 4 * i);
    const float rx = fmaxf(g.x, 0.f), ry = fmaxf(g.y, 0.f), rz = fmaxf(g.z, 0.f), rw = fmaxf(g.w, 0.f);
    st_cs_f4(dgate + 4 * i, make_float4(2.f * d.x * u.x * rx, 2.f * d.y * u.y * ry, 2.f * d.z * u.z * rz,
                                        2.f * d.w * u.w * rw));
    st_cs_f4(dup + 4 * i, make_float4(d.x * rx * rx, d.y * ry * ry, d.z * rz * rz, d.w * rw * rw));
  }
  if (blockIdx.x == 0) {
    const long long e = 4 * n4 + threadIdx.x;
    if (e < n) {
      const float g = ld_act1<BF16>(gate, e), u = ld_act1<BF16>(up, e), d = dh[e];
      const float r = fmaxf(g, 0.f);
      dgate[e] = 2.f * d * u * r;
      dup[e] = d * r * r;
    }
  }
}

// ----------------------------------------------------------------- LoRA
constexpr int kLoraRows = 4;     // rows per block of the row pass

template <bool XBF16>
__device__ __forceinline__ float4 ldg_x4(const void *x, size_t i4) {
  if (XBF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(x) + i4);
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
  } else {
    return __ldg(reinterpret_cast<const float4 *>(x) + i4);
  }
}

// Row pass: block b takes rows kLoraRows b .. + kLoraRows - 1 and writes
// h[t][j] = x_t . A_j and dh[t][j] = s dy_t . B[:, j] (j < r) to the
// workspace; every thread also zeroes its share of dA and dB.
template <bool XBF16, int RK>
__global__ void __launch_bounds__(256) lora_rows_kernel(const void *__restrict__ x, const float *__restrict__ dy,
                                                        const float *__restrict__ A, const float *__restrict__ B,
                                                        float *__restrict__ h, float *__restrict__ dh,
                                                        float *__restrict__ dA, float *__restrict__ dB, int rows,
                                                        int n_in, int n_out, int r, float scale) {
  __shared__ float red[8][2 * kLoraRows * RK];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {
    const long long nz = static_cast<long long>(r) * (n_in + n_out);
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + tid; e < nz; e += stride) {
      if (e < static_cast<long long>(r) * n_in)
        dA[e] = 0.f;
      else
        dB[e - static_cast<long long>(r) * n_in] = 0.f;
    }
  }
  const int t0 = blockIdx.x * kLoraRows;
  float acc[kLoraRows][RK], acc2[kLoraRows][RK];
#pragma unroll
  for (int t = 0; t < kLoraRows; ++t)
#pragma unroll
    for (int j = 0; j < RK; ++j) acc[t][j] = acc2[t][j] = 0.f;
  // h: four input columns per step
  const int c4 = n_in >> 2;
  for (int c = tid; c < c4; c += 256) {
    float4 a[RK];
#pragma unroll
    for (int j = 0; j < RK; ++j)
      a[j] = j < r ? __ldg(reinterpret_cast<const float4 *>(A + static_cast<size_t>(j) * n_in) + c)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 xv[kLoraRows];
#pragma unroll
    for (int t = 0; t < kLoraRows; ++t)
      xv[t] = t0 + t < rows ? ldg_x4<XBF16>(x, static_cast<size_t>(t0 + t) * c4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < kLoraRows; ++t)
#pragma unroll
      for (int j = 0; j < RK; ++j)
        acc[t][j] += xv[t].x * a[j].x + xv[t].y * a[j].y + xv[t].z * a[j].z + xv[t].w * a[j].w;
  }
  // dh: one output column per step (B row o holds its r rank entries); the
  // loads of a step are issued before its products
#pragma unroll 2
  for (int o = tid; o < n_out; o += 256) {
    float bo[RK], d[kLoraRows];
#pragma unroll
    for (int j = 0; j < RK; ++j) bo[j] = j < r ? __ldg(B + static_cast<size_t>(o) * r + j) : 0.f;
#pragma unroll
    for (int t = 0; t < kLoraRows; ++t) d[t] = t0 + t < rows ? __ldg(dy + static_cast<size_t>(t0 + t) * n_out + o) : 0.f;
#pragma unroll
    for (int t = 0; t < kLoraRows; ++t)
#pragma unroll
      for (int j = 0; j < RK; ++j) acc2[t][j] = fmaf(d[t], bo[j], acc2[t][j]);
  }
#pragma unroll
  for (int t = 0; t < kLoraRows; ++t)
#pragma unroll
    for (int j = 0; j < RK; ++j) {
      const float s1 = warp_sum(acc[t][j]), s2 = warp_sum(acc2[t][j]);
      if (lane == 0) {
        red[warp][t * RK + j] = s1;
        red[warp][kLoraRows * RK + t * RK + j] = s2;
      }
    }
  __syncthreads();
  if (tid < 2 * kLoraRows * RK) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w][tid];
    const int second = tid >= kLoraRows * RK;
    const int k = second ? tid - kLoraRows * RK : tid;
    const int t = k / RK, j = k % RK;
    if (t0 + t < rows && j < r) {
      if (second)
        dh[static_cast<size_t>(t0 + t) * r + j] = scale * s;
      else
        h[static_cast<size_t>(t0 + t) * r + j] = s;
    }
  }
}

// Column pass: block (column tile, row chunk) covers kLoraColG groups of four
// columns (of dA's n_in, then of dB's n_out) over 32 or 64 rows and adds its
// partial sums
//   dA[j][i] += sum_t dh[t][j] x[t][i],   dB[o][j] += s sum_t dy[t][o] h[t][j]
// with vector reductions.  Thread = (column group, row slice of kLoraColK
// rows, all loaded before the first product); the row slices' sums meet in
// shared memory, so one reduction per output group and rank leaves the
// block, and many small blocks keep many rows in flight.
constexpr int kLoraColG = 32;    // 4-column groups per block
constexpr int kLoraColK = 8;     // rows per row slice
// row slices per block (their partial sums share 37 KB of shared memory)
template <int RK>
constexpr int lora_col_slices() { return RK <= 8 ? 8 : 4; }
template <int RK>
constexpr int lora_col_rows() { return lora_col_slices<RK>() * kLoraColK; }

template <bool XBF16, int RK>
__global__ void __launch_bounds__(lora_col_slices<RK>() * kLoraColG) lora_cols_kernel(
    const void *__restrict__ x, const float *__restrict__ dy, const float *__restrict__ h,
    const float *__restrict__ dh, float *__restrict__ dA, float *__restrict__ dB, int rows, int n_in, int n_out,
    int r, float scale) {
  constexpr int kS = lora_col_slices<RK>(), kR = lora_col_rows<RK>(), kT = kS * kLoraColG;
  __shared__ float coef[kR][RK];
  __shared__ __align__(16) float part[kS][kLoraColG][4 * RK + 4];   // +4: spread the banks
  const int tid = threadIdx.x, cg = tid & (kLoraColG - 1), sl = tid / kLoraColG;
  const int r0 = blockIdx.y * kR;
  const int nr = min(kR, rows - r0);
  const int in4 = n_in >> 2, out4 = n_out >> 2;
  const int xtiles = (in4 + kLoraColG - 1) / kLoraColG;
  const bool xcol = static_cast<int>(blockIdx.x) < xtiles;
  const int c0 = (xcol ? blockIdx.x : blockIdx.x - xtiles) * kLoraColG;
  const int c = c0 + cg;   // this thread's 4-column group
  const bool on = c < (xcol ? in4 : out4);
  float4 v[kLoraColK];
#pragma unroll
  for (int k = 0; k < kLoraColK; ++k) {
    const int tt = sl * kLoraColK + k;
    if (on && tt < nr)
      v[k] = xcol ? ldg_x4<XBF16>(x, static_cast<size_t>(r0 + tt) * in4 + c)
                  : __ldg(reinterpret_cast<const float4 *>(dy + static_cast<size_t>(r0 + tt) * n_out) + c);
    else
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  {
    const float *src = xcol ? dh : h;   // dA needs dh, dB needs h
    for (int e = tid; e < kR * RK; e += kT) {
      const int tt = e / RK, j = e % RK;
      coef[tt][j] = (tt < nr && j < r) ? src[static_cast<size_t>(r0 + tt) * r + j] : 0.f;
    }
  }
  __syncthreads();
  float4 acc[RK];
#pragma unroll
  for (int j = 0; j < RK; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kLoraColK; ++k)
#pragma unroll
    for (int j = 0; j < RK; ++j) {
      const float w = coef[sl * kLoraColK + k][j];   // rows past nr have v = 0
      acc[j].x = fmaf(w, v[k].x, acc[j].x);
      acc[j].y = fmaf(w, v[k].y, acc[j].y);
      acc[j].z = fmaf(w, v[k].z, acc[j].z);
      acc[j].w = fmaf(w, v[k].w, acc[j].w);
    }
#pragma unroll
  for (int j = 0; j < RK; ++j) *reinterpret_cast<float4 *>(&part[sl][cg][4 * j]) = acc[j];
  __syncthreads();
  // thread -> (group g, rank j): the slices' sums of columns 4 (c0 + g) ..
  // + 3 for rank j
  for (int e = tid; e < kLoraColG * RK; e += kT) {
    const int g = e / RK, j = e % RK;
    const int cc = c0 + g;
    if (cc >= (xcol ? in4 : out4) || j >= r) continue;
    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kS; ++q) {
      const float4 u = *reinterpret_cast<const float4 *>(&part[q][g][4 * j]);
      s4.x += u.x;
      s4.y += u.y;
      s4.z += u.z;
      s4.w += u.w;
    }
    if (xcol) {
      red_add_f4(dA + static_cast<size_t>(j) * n_in + 4 * cc, s4);
    } else {
      // column 4 cc + e of dy is row 4 cc + e of dB
      float *col = dB + static_cast<size_t>(4 * cc) * r + j;
      atomicAdd(col, scale * s4.x);
      atomicAdd(col + r, scale * s4.y);
      atomicAdd(col + 2 * r, scale * s4.z);
      atomicAdd(col + 3 * r, scale * s4.w);
    }
  }
}

template <bool XB, int RK>
cudaError_t lora_launch(const void *x, const float *dy, const float *A, const float *B, float *dA, float *dB,
                        float *h, float *dh, int rows, int n_in, int n_out, int r, float scale, cudaStream_t st) {
  const int rblocks = rows > 0 ? (rows + kLoraRows - 1) / kLoraRows : 1;
  lora_rows_kernel<XB, RK><<<rblocks, 256, 0, st>>>(x, dy, A, B, h, dh, dA, dB, rows, n_in, n_out, r, scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || rows == 0) return e;
  const int tiles = ((n_in >> 2) + kLoraColG - 1) / kLoraColG + ((n_out >> 2) + kLoraColG - 1) / kLoraColG;
  const dim3 grid(tiles, (rows + lora_col_rows<RK>() - 1) / lora_col_rows<RK>());
  lora_cols_kernel<XB, RK><<<grid, lora_col_slices<RK>() * kLoraColG, 0, st>>>(x, dy, h, dh, dA, dB, rows, n_in,
                                                                              n_out, r, scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_relu2_mul_bwd(const void *gate, const void *up, int bf16, const float *dh, float *dgate,
                                 float *dup, long long n, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long groups = (n + 3) / 4;
  long long blocks = (groups + 255) / 256;
  blocks = blocks < 1 ? 1 : blocks;
  if (blocks > 8LL * sms) blocks = 8LL * sms;   // 2048 threads per SM, each looping
  if (bf16)
    relu2_mul_bwd_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(gate, up, dh, dgate, dup, n);
  else
    relu2_mul_bwd_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(gate, up, dh, dgate, dup, n);
  return cudaGetLastError();
}

size_t lora_workspace_bytes(int rows, int r) { return static_cast<size_t>(rows) * r * 2 * 4 + 256; }

cudaError_t launch_lora_bwd(const void *x, int x_bf16, const float *dy, const float *A, const float *B, float *dA,
                            float *dB, int rows, int n_in, int n_out, int r, float scale, void *ws,
                            cudaStream_t st) {
  char *p = static_cast<char *>(ws);
  p += (256 - (reinterpret_cast<uintptr_t>(p) & 255)) & 255;
  float *h = reinterpret_cast<float *>(p);
  float *dh = h + static_cast<size_t>(rows) * r;
  if (r <= 8)
    return x_bf16 ? lora_launch<true, 8>(x, dy, A, B, dA, dB, h, dh, rows, n_in, n_out, r, scale, st)
                  : lora_launch<false, 8>(x, dy, A, B, dA, dB, h, dh, rows, n_in, n_out, r, scale, st);
  return x_bf16 ? lora_launch<true, 16>(x, dy, A, B, dA, dB, h, dh, rows, n_in, n_out, r, scale, st)
                : lora_launch<false, 16>(x, dy, A, B, dA, dB, h, dh, rows, n_in, n_out, r, scale, st);
}

}  // namespace abw
