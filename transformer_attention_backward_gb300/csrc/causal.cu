// Causal multi-query attention backward (keys j <= query i), probabilities
// recomputed from the saved log-sum-exp; RoPE backward fused on dq and dk.
//
// Spec: DaisyChain-Train transformer.js, backward(): dV = A^T dctx,
// dA = dctx V^T, dS = A (dA - sum_j A dA) scale, dQ = dS K, dK = dS^T Q,
// over the causal softmax of forward(); "Hesper.Training.VerifiedBackward"
// sections Softmax / Scaled Dot-Product / RoPE for the per-element steps.
//
// Three launches per call:
//   1. prep     : delta_i = dout_i . o_i (the identity sum_j P_ij dP_ij =
//                 dout_i . o_i), the RoPE cos/sin table, zeroed dq accumulator
//   2. main     : one CTA per (64-key block, KV head, batch); loops over the
//                 query heads of the group and the query blocks at or after
//                 the key block; dK/dV accumulate in registers, dq through
//                 fp32 atomics into the workspace
//   3. finalize : dq = R(-theta) (scale * accumulator)
#include <math.h>

#include "abw_host.h"

namespace abw {
namespace {

constexpr int kD = 128;
constexpr int kBK = 64;   // keys per CTA
constexpr int kBQ = 64;   // queries per inner block
constexpr int kThr = 256;

struct CausalWs {
  float *dq_acc;     // [B][T][Hq][D]
  float *delta;      // [B][Hq][T]
  float2 *rope;      // [T][D/2] (cos, sin)
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

CausalWs carve(void *ws, int B, int T, int Hq, int D) {
  CausalWs w;
  char *p = static_cast<char *>(ws);
  p += (256 - (reinterpret_cast<uintptr_t>(p) & 255)) & 255;
  w.dq_acc = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * T * Hq * D * 4);
  w.delta = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * Hq * T * 4);
  w.rope = reinterpret_cast<float2 *>(p);
  return w;
}

// delta_i = dout_i . o_i, one warp per (b, t, h) row of D = 128 bf16.
__global__ void __launch_bounds__(256) causal_delta_kernel(const __nv_bfloat16 *__restrict__ o,
                                                           const __nv_bfloat16 *__restrict__ dout,
                                                           float *__restrict__ delta, int B, int T, int Hq) {
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(B) * T * Hq) return;
  const uint2 a = reinterpret_cast<const uint2 *>(o + row * kD)[lane];
  const uint2 g = reinterpret_cast<const uint2 *>(dout + row * kD)[lane];
  float s = bf16_lo(a.x) * bf16_lo(g.x) + bf16_hi(a.x) * bf16_hi(g.x) + bf16_lo(a.y) * bf16_lo(g.y) +
            bf16_hi(a.y) * bf16_hi(g.y);
  s = warp_sum(s);
  if (lane == 0) {
    const int h = static_cast<int>(row % Hq);
    const long long bt = row / Hq;
    const int t = static_cast<int>(bt % T);
    const int b = static_cast<int>(bt / T);
    delta[(static_cast<size_t>(b) * Hq + h) * T + t] = s;
  }
}

// RoPE table: cos/sin of theta = (pos0 + t) * base^(-2i/D), angle formed and
// reduced modulo 2 pi in double, rounded to float only for sincosf.
__global__ void causal_rope_table_kernel(float2 *__restrict__ tab, int T, int pos0, double log2_base) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= T * (kD / 2)) return;
  const int t = idx / (kD / 2), i = idx % (kD / 2);
  const double inv_freq = exp2(-log2_base * (2.0 * i / kD));
  const double a = static_cast<double>(pos0 + t) * inv_freq;
  const double twopi = 6.283185307179586476925286766559;
  const float th = static_cast<float>(a - twopi * rint(a / twopi));
  float s, c;
  sincosf(th, &s, &c);
  tab[idx] = make_float2(c, s);
}

struct MainParams {
  const __nv_bfloat16 *q, *k, *v, *dout;
  const float *lse;
  float *dk, *dv;
  CausalWs ws;
  int B, T, Hq, Hkv, G;
  float scale;
  int rope;
};

// SIMT reference kernel: correct for any T, D = 128.
__global__ void __launch_bounds__(kThr, 1) causal_bwd_simt(const __grid_constant__ MainParams p) {
  extern __shared__ float sm[];
  float *Ks = sm;                          // [64][128]
  float *Vs = Ks + kBK * kD;               // [64][128]
  float *Qs = Vs + kBK * kD;               // [64][128]
  float *Os = Qs + kBQ * kD;               // dout [64][128]
  float *Ps = Os + kBQ * kD;               // [64][65]
  float *Ds = Ps + kBQ * 65;               // [64][65]
  float *ls = Ds + kBQ * 65;               // lse [64]
  float *dl = ls + kBQ;                    // delta [64]

  const int nkb = (p.T + kBK - 1) / kBK;
  const int kb = nkb - 1 - blockIdx.x;     // heavy (early) key blocks first
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int k0 = kb * kBK;
  const int tid = threadIdx.x;

  // load K, V block (rows beyond T are zero)
  for (int i = tid; i < kBK * kD; i += kThr) {
    const int r = i / kD, d = i % kD;
    const int j = k0 + r;
    float kv = 0.f, vv = 0.f;
    if (j < p.T) {
      const size_t off = ((static_cast<size_t>(b) * p.T + j) * p.Hkv + kvh) * kD + d;
      kv = __bfloat162float(p.k[off]);
      vv = __bfloat162float(p.v[off]);
    }
    Ks[i] = kv;
    Vs[i] = vv;
  }

  // dK, dV accumulators: thread owns key row jr, dims c + 4m (m < 32)
  const int jr = tid >> 2, c4 = tid & 3;
  float aK[32], aV[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) aK[m] = aV[m] = 0.f;

  const float l2e = 1.4426950408889634f;
  for (int hh = 0; hh < p.G; ++hh) {
    const int h = kvh * p.G + hh;
    for (int q0 = (k0 / kBQ) * kBQ; q0 < p.T; q0 += kBQ) {
      __syncthreads();
      for (int i = tid; i < kBQ * kD; i += kThr) {
        const int r = i / kD, d = i % kD;
        const int t = q0 + r;
        float qv = 0.f, ov = 0.f;
        if (t < p.T) {
          const size_t off = ((static_cast<size_t>(b) * p.T + t) * p.Hq + h) * kD + d;
          qv = __bfloat162float(p.q[off]);
          ov = __bfloat162float(p.dout[off]);
        }
        Qs[i] = qv;
        Os[i] = ov;
      }
      if (tid < kBQ) {
        const int t = q0 + tid;
        const size_t lo = (static_cast<size_t>(b) * p.Hq + h) * p.T + t;
        ls[tid] = t < p.T ? p.lse[lo] : 0.f;
        dl[tid] = t < p.T ? p.ws.delta[lo] : 0.f;
      }
      __syncthreads();
      // S, dP: thread computes rows 4*ti..4*ti+3, cols tj + 16*m
      {
        const int ti = tid >> 4, tj = tid & 15;
        float s[4][4], dp[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) s[a][c] = dp[a][c] = 0.f;
        for (int d = 0; d < kD; ++d) {
          float qa[4], oa[4], kc[4], vc[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            qa[a] = Qs[(4 * ti + a) * kD + d];
            oa[a] = Os[(4 * ti + a) * kD + d];
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            kc[c] = Ks[(tj + 16 * c) * kD + d];
            vc[c] = Vs[(tj + 16 * c) * kD + d];
          }
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              s[a][c] = fmaf(qa[a], kc[c], s[a][c]);
              dp[a][c] = fmaf(oa[a], vc[c], dp[a][c]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int i = 4 * ti + a, t = q0 + i;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int jj = tj + 16 * c, j = k0 + jj;
            float P = 0.f;
            if (t < p.T && j <= t) P = exp2f((s[a][c] * p.scale - ls[i]) * l2e);
            Ps[i * 65 + jj] = P;
            Ds[i * 65 + jj] = P * (dp[a][c] - dl[i]);
          }
        }
      }
      __syncthreads();
      // dV[jr] += sum_i P[i][jr] dO[i];  dK[jr] += sum_i dS[i][jr] Q[i]
      for (int i = 0; i < kBQ; ++i) {
        const float P = Ps[i * 65 + jr], dS = Ds[i * 65 + jr];
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          aV[m] = fmaf(P, Os[i * kD + c4 + 4 * m], aV[m]);
          aK[m] = fmaf(dS, Qs[i * kD + c4 + 4 * m], aK[m]);
        }
      }
      // dQ[i] += sum_j dS[i][j] K[j]  (thread: row i = jr, dims c4 + 4m)
      {
        float aq[32];
#pragma unroll
        for (int m = 0; m < 32; ++m) aq[m] = 0.f;
        for (int jj = 0; jj < kBK; ++jj) {
          const float dS = Ds[jr * 65 + jj];
#pragma unroll
          for (int m = 0; m < 32; ++m) aq[m] = fmaf(dS, Ks[jj * kD + c4 + 4 * m], aq[m]);
        }
        const int t = q0 + jr;
        if (t < p.T) {
          float *dst = p.ws.dq_acc + ((static_cast<size_t>(b) * p.T + t) * p.Hq + h) * kD;
#pragma unroll
          for (int m = 0; m < 32; ++m) atomicAdd(dst + c4 + 4 * m, aq[m]);
        }
      }
    }
  }
  __syncthreads();
  // epilogue: dK (scaled, rotated) and dV
  float *Kout = Qs;   // reuse: [64][128]
#pragma unroll
  for (int m = 0; m < 32; ++m) Kout[jr * kD + c4 + 4 * m] = aK[m] * p.scale;
  __syncthreads();
  for (int i = tid; i < kBK * (kD / 2); i += kThr) {
    const int r = i / (kD / 2), pi = i % (kD / 2);
    const int j = k0 + r;
    if (j >= p.T) continue;
    float y0 = Kout[r * kD + 2 * pi], y1 = Kout[r * kD + 2 * pi + 1];
    if (p.rope) {
      const float2 cs = p.ws.rope[j * (kD / 2) + pi];
      const float z0 = y0 * cs.x + y1 * cs.y, z1 = -y0 * cs.y + y1 * cs.x;
      y0 = z0;
      y1 = z1;
    }
    float *dst = p.dk + ((static_cast<size_t>(b) * p.T + j) * p.Hkv + kvh) * kD + 2 * pi;
    dst[0] = y0;
    dst[1] = y1;
  }
  const int j = k0 + jr;
  if (j < p.T) {
    float *dst = p.dv + ((static_cast<size_t>(b) * p.T + j) * p.Hkv + kvh) * kD;
#pragma unroll
    for (int m = 0; m < 32; ++m) dst[c4 + 4 * m] = aV[m];
  }
}

// dq = R(-theta_t) (scale * acc), one thread per rotary pair.
__global__ void __launch_bounds__(256) causal_dq_finalize(const float *__restrict__ acc, const float2 *__restrict__ rope,
                                                          float *__restrict__ dq, long long npairs, int T, int Hq,
                                                          float scale, int use_rope) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= npairs) return;
  const int pi = static_cast<int>(i % (kD / 2));
  const long long row = i / (kD / 2);          // (b * T + t) * Hq + h
  const int t = static_cast<int>((row / Hq) % T);
  const float2 y = reinterpret_cast<const float2 *>(acc)[i];
  float z0 = y.x * scale, z1 = y.y * scale;
  if (use_rope) {
    const float2 cs = rope[t * (kD / 2) + pi];
    const float a = z0 * cs.x + z1 * cs.y, c = -z0 * cs.y + z1 * cs.x;
    z0 = a;
    z1 = c;
  }
  reinterpret_cast<float2 *>(dq)[i] = make_float2(z0, z1);
}

}  // namespace

size_t causal_workspace_bytes(int B, int T, int Hq, int D) {
  return 256 + up256(static_cast<size_t>(B) * T * Hq * D * 4) + up256(static_cast<size_t>(B) * Hq * T * 4) +
         up256(static_cast<size_t>(T) * (D / 2) * 8);
}

cudaError_t launch_attn_bwd_causal(const void *q, const void *k, const void *v, const void *o, const void *dout,
                                   const float *lse, float *dq, float *dk, float *dv, int B, int T, int Hq, int Hkv,
                                   int D, float scale, double rope_base, int pos0, void *ws, size_t ws_bytes,
                                   const WaitCtl &w, cudaStream_t st, const char **why) {
  (void)ws_bytes;
  (void)w;
  if (D != kD) {
    *why = "D != 128";
    return cudaErrorNotSupported;
  }
  const int nkb = (T + kBK - 1) / kBK;
  if (Hkv > 65535 || B > 65535) {
    *why = "B or Hkv > 65535";
    return cudaErrorNotSupported;
  }
  CausalWs cw = carve(ws, B, T, Hq, D);
  const size_t qn = static_cast<size_t>(B) * T * Hq * D;
  cudaError_t e = cudaMemsetAsync(cw.dq_acc, 0, qn * 4, st);
  if (e != cudaSuccess) return e;
  {
    const long long rows = static_cast<long long>(B) * T * Hq;
    const long long blocks = (rows * 32 + 255) / 256;
    causal_delta_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), cw.delta, B, T, Hq);
  }
  const int rope = rope_base > 0.0;
  if (rope) {
    const int n = T * (kD / 2);
    causal_rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(cw.rope, T, pos0, log2(rope_base));
  }
  MainParams p;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k = static_cast<const __nv_bfloat16 *>(k);
  p.v = static_cast<const __nv_bfloat16 *>(v);
  p.dout = static_cast<const __nv_bfloat16 *>(dout);
  p.lse = lse;
  p.dk = dk;
  p.dv = dv;
  p.ws = cw;
  p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.scale = scale;
  p.rope = rope;
  const int smem = (4 * 64 * kD + 2 * 64 * 65 + 2 * 64) * 4;
  e = cudaFuncSetAttribute(causal_bwd_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  causal_bwd_simt<<<dim3(nkb, Hkv, B), kThr, smem, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long npairs = static_cast<long long>(qn / 2);
  causal_dq_finalize<<<static_cast<unsigned>((npairs + 255) / 256), 256, 0, st>>>(cw.dq_acc, cw.rope, dq, npairs, T,
                                                                                 Hq, scale, rope);
  return cudaGetLastError();
}

}  // namespace abw
