// Causal multi-query attention backward (keys j <= query i), probabilities
// recomputed from the saved log-sum-exp; RoPE backward fused on dq and dk.
//
// Spec: DaisyChain-Train transformer.js, backward(): dV = A^T dctx,
// dA = dctx V^T, dS = A (dA - sum_j A dA) scale, dQ = dS K, dK = dS^T Q,
// over the causal softmax of forward(); "Hesper.Training.VerifiedBackward"
// sections Softmax / Scaled Dot-Product / RoPE for the per-element steps.
//
// Launches per call:
//   1. memset   : fp32 dq accumulator
//   2. prep     : delta_i = dout_i . o_i (the identity sum_j P_ij dP_ij =
//                 dout_i . o_i) and lse_i * log2(e), both padded to a multiple
//                 of 64 queries (padding: delta 0, lse +inf so P = 0 there)
//   3. rope     : cos/sin table of theta(t, i) (only with RoPE)
//   4. main     : tcgen05 kernel, one CTA per (128-key block, KV head, batch)
//   5. finalize : dq = R(-theta) (scale * accumulator)
//
// Main kernel (sm_103a, 12 warps, one CTA per SM).  Per CTA the K and V
// block stays in shared memory; the CTA loops over the query heads of its KV
// group and the 64-query blocks at or after its key block:
//   MMA1  S^T  = K Q^T          M=128 keys, N=64 queries, K=128 (TMEM)
//   MMA2  dP^T = V dO^T         same shape
//   softmax warps: P = exp2(S scale log2e - lse log2e) (causal mask),
//          dS = P (dP - delta), both rounded to bf16 into swizzled smem
//   MMA3  dV  += P^T dO          M=128 keys, N=128, K=64 queries
//   MMA4  dK  += dS^T Q          same shape
//   MMA5  dQ^T = K^T dS^T        M=128 (head dim), N=64 queries, K=128 keys,
//          written over the S columns the softmax warps have finished with;
//          dq warps transpose it through shared memory (32 queries at a
//          time) and fold it into the fp32 dq accumulator with 16-byte
//          vector reductions (kept off the TMA queue, which carries the
//          Q/dO loads).
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 4-7 softmax
// (and the dK epilogue: scale + RoPE), 8-11 dq reduction (and the dV
// epilogue).  S/dP are double-buffered in TMEM so the tensor core computes
// block n+1 while the softmax warps work on block n.  TMEM (512 columns):
//   [0,64) S0 / dQ^T0   [64,128) dP0   [128,192) S1 / dQ^T1   [192,256) dP1
//   [256,384) dV        [384,512) dK
// Q / dO / lse / delta arrive through a 3-deep TMA ring, so the load for block
// n+3 is in flight while blocks n+1 and n+2 compute.
#include <math.h>

#include <mutex>

#include "abw_host.h"
#include "tcgen05.cuh"

namespace abw {
namespace {

constexpr int kD = 128;
constexpr int kBK = 128;   // keys per CTA
constexpr int kBQ = 64;    // queries per block
constexpr int kThr = 384;  // 12 warps

// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kOffK = 0;                 // [2 D-halves][128 keys][128 B], 128B-swizzled
constexpr int kOffV = 32768;
constexpr int kStages = 3;               // Q / dO / lse / delta ring depth
constexpr int kOffStage = 65536;
constexpr int kStageBytes = 33792;       // Q 16 KB, dO 16 KB, lse2 256 B, delta 256 B (1 KB aligned)
constexpr int kStQ = 0, kStDO = 16384, kStLse = 32768, kStDelta = 33024;
constexpr int kOffP = kOffStage + kStages * kStageBytes;   // P^T [128 keys][64 queries] bf16, swizzled
constexpr int kOffDS = kOffP + 16384;                 // dS^T [128 keys][64 queries] bf16, swizzled
constexpr int kOffDQ = kOffDS + 16384;                // dQ staging: [32 queries][128] fp32
constexpr int kOffBar = kOffDQ + 16384;
constexpr int kSmem = kOffBar + 256 + 1024;           // + alignment slack

// Barrier slots (8 bytes each) after kOffBar.
enum {
  kBarKV = 0, kBarQFull = 1, kBarQEmpty = 4, kBarSFull = 7, kBarPFull = 9, kBarPEmpty = 10,
  kBarDQFull = 11, kBarTEmpty = 13, kBarDKV = 15, kBarFinal = 16, kNumBars = 17
};
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;

constexpr uint32_t kColS0 = 0, kColDP0 = 64, kColS1 = 128, kColDP1 = 192, kColDV = 256, kColDK = 384;

struct CausalWs {
  float *dq_acc;     // [B][T][Hq][D]
  float *delta;      // [B][Hq][Tp]
  float *lse2;       // [B][Hq][Tp]  lse * log2(e), +inf past T
  float2 *rope;      // [T][D/2] (cos, sin)
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

int padded_T(int T) { return (T + kBQ - 1) / kBQ * kBQ; }

CausalWs carve(void *ws, int B, int T, int Hq, int D) {
  const size_t Tp = static_cast<size_t>(padded_T(T));
  CausalWs w;
  char *p = static_cast<char *>(ws);
  p += (256 - (reinterpret_cast<uintptr_t>(p) & 255)) & 255;
  w.dq_acc = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * T * Hq * D * 4);
  w.delta = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * Hq * Tp * 4);
  w.lse2 = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * Hq * Tp * 4);
  w.rope = reinterpret_cast<float2 *>(p);
  return w;
}

// delta and lse*log2(e) for every (b, h, t < Tp): one warp per (b, t, h) row
// of D = 128 bf16 for t < T; padding rows get delta 0 and lse +inf.
__global__ void __launch_bounds__(256) causal_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                                                          const __nv_bfloat16 *__restrict__ dout,
                                                          const float *__restrict__ lse, float *__restrict__ delta,
                                                          float *__restrict__ lse2, int B, int T, int Tp, int Hq) {
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(B) * Tp * Hq) return;
  const int h = static_cast<int>(row % Hq);
  const long long bt = row / Hq;
  const int t = static_cast<int>(bt % Tp);
  const int b = static_cast<int>(bt / Tp);
  const size_t out = (static_cast<size_t>(b) * Hq + h) * Tp + t;
  if (t >= T) {
    if (lane == 0) {
      delta[out] = 0.f;
      lse2[out] = INFINITY;
    }
    return;
  }
  const size_t src = ((static_cast<size_t>(b) * T + t) * Hq + h) * kD;
  const uint2 a = reinterpret_cast<const uint2 *>(o + src)[lane];
  const uint2 g = reinterpret_cast<const uint2 *>(dout + src)[lane];
  float s = bf16_lo(a.x) * bf16_lo(g.x) + bf16_hi(a.x) * bf16_hi(g.x) + bf16_lo(a.y) * bf16_lo(g.y) +
            bf16_hi(a.y) * bf16_hi(g.y);
  s = warp_sum(s);
  if (lane == 0) {
    delta[out] = s;
    lse2[out] = lse[(static_cast<size_t>(b) * Hq + h) * T + t] * 1.4426950408889634f;
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

struct TcParams {
  CausalWs ws;
  float *dk, *dv;
  int B, T, Tp, Hq, Hkv, G, nkb, nqb;
  float scale;
  int rope;
  WaitCtl wait;
};

// 2^x on the MUFU unit (relative error ~2^-22, which is far below the bf16
// rounding P gets next); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThr, 1)
    causal_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // work item: heavy (early) key blocks first across the whole grid
  const int per_kb = p.Hkv * p.B;
  const int kb = blockIdx.x / per_kb;
  const int rem = blockIdx.x - kb * per_kb;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int k0 = kb * kBK;
  const int qb0 = k0 / kBQ;
  const int nq = p.nqb - qb0;            // query blocks per head
  const int N = p.G * nq;                // iterations of this CTA
  // Query block of iteration n.  Each CTA walks its query blocks from a
  // different starting point (rotated by its key block), so CTAs of the same
  // head working at the same time reduce into different dq rows.
  const int rot = (kb * 5) % nq;
  auto qblock = [&](int n) -> int {
    int i = n % nq + rot;
    if (i >= nq) i -= nq;
    return qb0 + i;
  };

  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + i * 8; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
  auto wt = [&](uint32_t br, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(br, parity, p.wait.limit_ns)) return true;
    *abort_flag = 1;
    atomicOr(p.wait.err, kErrWaitTimeout);
    return false;
  };

  if (tid == 0) {
    mbar_init(bar(kBarKV), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarDQFull + s), 1);
      mbar_init(bar(kBarTEmpty + s), 128);
    }
    mbar_init(bar(kBarPFull), 128);
    mbar_init(bar(kBarPEmpty), 1);
    mbar_init(bar(kBarDKV), 1);
    mbar_init(bar(kBarFinal), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) tc::tmem_alloc(sb + kOffTmemSlot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kOffTmemSlot);

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmDO);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_arrive_expect_tx(bar(kBarKV), 4 * 16384);
      for (int hx = 0; hx < 2; ++hx) {
        tma_load_4d(sb + kOffK + hx * 16384, &tmK, hx * 64, kvh, k0, b, bar(kBarKV));
        tma_load_4d(sb + kOffV + hx * 16384, &tmV, hx * 64, kvh, k0, b, bar(kBarKV));
      }
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int s = n % kStages, cyc = n / kStages;
        if (!wt(bar(kBarQEmpty + s), (cyc & 1) ^ 1)) break;
        const int h = kvh * p.G + n / nq;
        const int q0 = qblock(n) * kBQ;
        const uint32_t st = sb + kOffStage + s * kStageBytes;
        const uint32_t fb = bar(kBarQFull + s);
        mbar_arrive_expect_tx(fb, 2 * 16384 + 2 * 256);
        for (int hx = 0; hx < 2; ++hx) {
          tma_load_4d(st + kStQ + hx * 8192, &tmQ, hx * 64, h, q0, b, fb);
          tma_load_4d(st + kStDO + hx * 8192, &tmDO, hx * 64, h, q0, b, fb);
        }
        const size_t ro = (static_cast<size_t>(b) * p.Hq + h) * p.Tp + q0;
        bulk_load(st + kStLse, p.ws.lse2 + ro, 256, fb);
        bulk_load(st + kStDelta, p.ws.delta + ro, 256, fb);
        issued = n + 1;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        for (int n = (issued > kStages ? issued - kStages : 0); n < issued; ++n)
          mbar_wait_bounded(bar(kBarQFull + n % kStages), (n / kStages) & 1, 2000000000ull);
        mbar_wait_bounded(bar(kBarKV), 0, 2000000000ull);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      constexpr uint32_t id_sdp = tc::idesc_bf16_f32(128, 64, 0, 0);    // S^T, dP^T
      constexpr uint32_t id_kv = tc::idesc_bf16_f32(128, 128, 0, 1);    // dV, dK
      constexpr uint32_t id_dq = tc::idesc_bf16_f32(128, 64, 1, 1);     // dQ^T
      bool ok = wt(bar(kBarKV), 0);
      tc::fence_after_sync();
      auto issue_sdp = [&](int n) -> bool {
        const int s = n & 1, cyc = n >> 1;                       // TMEM buffer
        const int qs = n % kStages, qc = n / kStages;             // smem stage
        if (!wt(bar(kBarQFull + qs), qc & 1)) return false;
        if (!wt(bar(kBarTEmpty + s), (cyc & 1) ^ 1)) return false;
        tc::fence_after_sync();
        const uint32_t st = sb + kOffStage + qs * kStageBytes;
        const uint32_t dS = tmem + (s ? kColS1 : kColS0), dP = tmem + (s ? kColDP1 : kColDP0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32, qo = (kk >> 2) * 8192 + (kk & 3) * 32;
          tc::mma_bf16(dS, tc::sdesc_sw128(sb + kOffK + ko, 16, 1024), tc::sdesc_sw128(st + kStQ + qo, 16, 1024),
                       id_sdp, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32, qo = (kk >> 2) * 8192 + (kk & 3) * 32;
          tc::mma_bf16(dP, tc::sdesc_sw128(sb + kOffV + ko, 16, 1024), tc::sdesc_sw128(st + kStDO + qo, 16, 1024),
                       id_sdp, kk > 0);
        }
        tc::commit(bar(kBarSFull + s));
        return true;
      };
      if (ok) ok = issue_sdp(0);
      for (int n = 0; ok && n < N; ++n) {
        const int s = n & 1;
        if (n + 1 < N && !issue_sdp(n + 1)) break;
        if (!wt(bar(kBarPFull), n & 1)) break;
        tc::fence_after_sync();
        const int qs = n % kStages;
        const uint32_t st = sb + kOffStage + qs * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // dV += P^T dO
          tc::mma_bf16(tmem + kColDV, tc::sdesc_sw128(sb + kOffP + kk * 32, 16, 1024),
                       tc::sdesc_sw128(st + kStDO + kk * 2048, 8192, 1024), id_kv, (n > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // dK += dS^T Q
          tc::mma_bf16(tmem + kColDK, tc::sdesc_sw128(sb + kOffDS + kk * 32, 16, 1024),
                       tc::sdesc_sw128(st + kStQ + kk * 2048, 8192, 1024), id_kv, (n > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // dQ^T = K^T dS^T
          tc::mma_bf16(tmem + (s ? kColS1 : kColS0), tc::sdesc_sw128(sb + kOffK + kk * 2048, 16384, 1024),
                       tc::sdesc_sw128(sb + kOffDS + kk * 2048, 8192, 1024), id_dq, kk > 0);
        tc::commit(bar(kBarQEmpty + qs));
        tc::commit(bar(kBarPEmpty));
        tc::commit(bar(kBarDQFull + s));
      }
      tc::commit(bar(kBarDKV));
      tc::commit(bar(kBarFinal));
      mbar_wait_bounded(bar(kBarFinal), 0, 2000000000ull);   // every MMA has completed
    }
  } else if (warp >= 4 && warp < 8) {
    // ============================ softmax warps ===========================
    const int qd = warp & 3;
    const int j = 32 * qd + lane;                       // key row in the block
    const int key = k0 + j;
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;
    for (int n = 0; n < N; ++n) {
      const int s = n & 1, cyc = n >> 1;
      const int q0 = qblock(n) * kBQ;
      if (!wt(bar(kBarSFull + s), cyc & 1)) break;
      tc::fence_after_sync();
      const int qs = n % kStages;
      const float *lse2 = reinterpret_cast<const float *>(smem + kOffStage + qs * kStageBytes + kStLse);
      const float *dl = reinterpret_cast<const float *>(smem + kOffStage + qs * kStageBytes + kStDelta);
      // only the two query blocks that overlap the key block need the causal
      // mask; queries past T have lse = +inf, so their P is exactly 0
      const bool diag = q0 < k0 + kBK;
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float sv[32], pv[32];
        tc::ld32x2_wait(tmem + lanebase + (s ? kColS1 : kColS0) + 32 * hf,
                        tmem + lanebase + (s ? kColDP1 : kColDP0) + 32 * hf, sv, pv);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + 32 * hf + c);
          const float4 d4 = *reinterpret_cast<const float4 *>(dl + 32 * hf + c);
          float P0 = fast_exp2(fmaf(sv[c], sl2, -l4.x));
          float P1 = fast_exp2(fmaf(sv[c + 1], sl2, -l4.y));
          float P2 = fast_exp2(fmaf(sv[c + 2], sl2, -l4.z));
          float P3 = fast_exp2(fmaf(sv[c + 3], sl2, -l4.w));
          if (diag) {
            const int q = q0 + 32 * hf + c;
            P0 = key <= q ? P0 : 0.f;
            P1 = key <= q + 1 ? P1 : 0.f;
            P2 = key <= q + 2 ? P2 : 0.f;
            P3 = key <= q + 3 ? P3 : 0.f;
          }
          const float dS0 = P0 * (pv[c] - d4.x), dS1 = P1 * (pv[c + 1] - d4.y);
          const float dS2 = P2 * (pv[c + 2] - d4.z), dS3 = P3 * (pv[c + 3] - d4.w);
          pk[16 * hf + c / 2] = pack_bf16x2(P0, P1);
          pk[16 * hf + c / 2 + 1] = pack_bf16x2(P2, P3);
          dk[16 * hf + c / 2] = pack_bf16x2(dS0, dS1);
          dk[16 * hf + c / 2 + 1] = pack_bf16x2(dS2, dS3);
        }
      }
      if (!wt(bar(kBarPEmpty), (n & 1) ^ 1)) break;
      unsigned char *prow = smem + kOffP + j * 128;
      unsigned char *drow = smem + kOffDS + j * 128;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const int o = (c8 ^ (j & 7)) << 4;
        *reinterpret_cast<uint4 *>(prow + o) = make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        *reinterpret_cast<uint4 *>(drow + o) = make_uint4(dk[4 * c8], dk[4 * c8 + 1], dk[4 * c8 + 2], dk[4 * c8 + 3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(bar(kBarPFull));
    }
    // ---- dK epilogue: scale, RoPE backward, store
    if (wt(bar(kBarDKV), 0)) {
      tc::fence_after_sync();
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tc::ld32_wait(tmem + lanebase + kColDK + 32 * c, v);
        if (key < p.T) {
          float *dst = p.dk + ((static_cast<size_t>(b) * p.T + key) * p.Hkv + kvh) * kD + 32 * c;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float y0 = v[i] * p.scale, y1 = v[i + 1] * p.scale, y2 = v[i + 2] * p.scale, y3 = v[i + 3] * p.scale;
            if (p.rope) {
              const float4 cs = *reinterpret_cast<const float4 *>(p.ws.rope + key * (kD / 2) + 16 * c + i / 2);
              const float z0 = y0 * cs.x + y1 * cs.y, z1 = -y0 * cs.y + y1 * cs.x;
              const float z2 = y2 * cs.z + y3 * cs.w, z3 = -y2 * cs.w + y3 * cs.z;
              y0 = z0; y1 = z1; y2 = z2; y3 = z3;
            }
            *reinterpret_cast<float4 *>(dst + i) = make_float4(y0, y1, y2, y3);
          }
        }
      }
    }
  } else if (warp >= 8) {
    // ============================ dq reduction warps ======================
    const int qd = warp & 3;
    const int d = 32 * qd + lane;                       // head-dim row of dQ^T
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    for (int n = 0; n < N; ++n) {
      const int s = n & 1, cyc = n >> 1;
      // the four dq warps share named barriers: leave the loop together
      if (!named_barrier_and(1, 128, wt(bar(kBarDQFull + s), cyc & 1))) break;
      tc::fence_after_sync();
      float v0[32], v1[32];
      tc::ld32x2_wait(tmem + lanebase + (s ? kColS1 : kColS0), tmem + lanebase + (s ? kColS1 : kColS0) + 32, v0, v1);
      tc::fence_before_sync();
      mbar_arrive(bar(kBarTEmpty + s));
      const int h = kvh * p.G + n / nq;
      const int q0 = qblock(n) * kBQ;
      // dQ^T rows (one head-dim index per thread) -> shared memory, transposed
      // to query rows; each warp then adds whole 512-byte dq rows with
      // 16-byte vector reductions (32 queries per pass through the buffer)
      float *stage = reinterpret_cast<float *>(smem + kOffDQ);
      float *dst = p.ws.dq_acc + ((static_cast<size_t>(b) * p.T + q0) * p.Hq + h) * kD + 4 * lane;
      const size_t rstride = static_cast<size_t>(p.Hq) * kD;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        if (hf == 1) named_barrier(1, 128);            // first half has been read
#pragma unroll
        for (int c = 0; c < 32; ++c) stage[c * kD + d] = hf ? v1[c] : v0[c];
        named_barrier(1, 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = qd * 8 + k;                    // query row within the half
          const int q = q0 + 32 * hf + r;
          if (q < p.T) red_add_f4(dst + (32 * hf + r) * rstride, *reinterpret_cast<const float4 *>(stage + r * kD + 4 * lane));
        }
      }
      named_barrier(1, 128);
    }
    // ---- dV epilogue
    const int key = k0 + d;   // TMEM lane == key row for dV
    if (wt(bar(kBarDKV), 0)) {
      tc::fence_after_sync();
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tc::ld32_wait(tmem + lanebase + kColDV + 32 * c, v);
        if (key < p.T) {
          float *dst = p.dv + ((static_cast<size_t>(b) * p.T + key) * p.Hkv + kvh) * kD + 32 * c;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
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

bool make_map(CUtensorMap *m, const void *base, int H, int T, int B, uint32_t rows, const char **why) {
  const uint64_t dims[4] = {kD, static_cast<uint64_t>(H), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {kD * 2, static_cast<uint64_t>(H) * kD * 2, static_cast<uint64_t>(T) * H * kD * 2};
  const uint32_t box[4] = {64, 1, rows, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, why);
}

// Scratch for attn_bwd_causal_noalloc: a fixed device array the library
// owns, so that entry point never allocates.  Every GPU that loads the
// library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace

cudaError_t noalloc_scratch(void **ptr, const char **why) {
  // Resolved once per device, with that device current.  A symbol's name in
  // host code is only a host-side stand-in; the device address must come
  // from the runtime.
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) {
    *why = "device ordinal out of range";
    return cudaErrorInvalidDevice;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *why = "cudaGetSymbolAddress of the built-in scratch failed";
      return e;
    }
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

size_t causal_workspace_bytes(int B, int T, int Hq, int D) {
  const size_t Tp = static_cast<size_t>(padded_T(T));
  return 256 + up256(static_cast<size_t>(B) * T * Hq * D * 4) + 2 * up256(static_cast<size_t>(B) * Hq * Tp * 4) +
         up256(static_cast<size_t>(T) * (D / 2) * 8);
}

cudaError_t launch_attn_bwd_causal(const void *q, const void *k, const void *v, const void *o, const void *dout,
                                   const float *lse, float *dq, float *dk, float *dv, int B, int T, int Hq, int Hkv,
                                   int D, float scale, double rope_base, int pos0, void *ws, size_t ws_bytes,
                                   const WaitCtl &w, cudaStream_t st, const char **why) {
  (void)ws_bytes;
  if (D != kD) {
    *why = "D != 128";
    return cudaErrorNotSupported;
  }
  const int nkb = (T + kBK - 1) / kBK;
  const int Tp = padded_T(T);
  const long long ctas = static_cast<long long>(nkb) * Hkv * B;
  if (ctas > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorNotSupported;
  }
  CausalWs cw = carve(ws, B, T, Hq, D);
  const size_t qn = static_cast<size_t>(B) * T * Hq * D;
  cudaError_t e = cudaMemsetAsync(cw.dq_acc, 0, qn * 4, st);
  if (e != cudaSuccess) return e;
  {
    const long long rows = static_cast<long long>(B) * Tp * Hq;
    const long long blocks = (rows * 32 + 255) / 256;
    causal_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse, cw.delta, cw.lse2, B,
        T, Tp, Hq);
  }
  const int rope = rope_base > 0.0;
  if (rope) {
    const int n = T * (kD / 2);
    causal_rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(cw.rope, T, pos0, log2(rope_base));
  }
  CUtensorMap tq, tdo, tk, tv;
  if (!make_map(&tq, q, Hq, T, B, kBQ, why) || !make_map(&tdo, dout, Hq, T, B, kBQ, why) ||
      !make_map(&tk, k, Hkv, T, B, kBK, why) || !make_map(&tv, v, Hkv, T, B, kBK, why))
    return cudaErrorInvalidValue;
  TcParams p;
  p.ws = cw;
  p.dk = dk;
  p.dv = dv;
  p.B = B; p.T = T; p.Tp = Tp; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.nkb = nkb;
  p.nqb = Tp / kBQ;
  p.scale = scale;
  p.rope = rope;
  p.wait = w;
  e = cudaFuncSetAttribute(causal_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  causal_bwd_tc_kernel<<<static_cast<unsigned>(ctas), kThr, kSmem, st>>>(tq, tdo, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long npairs = static_cast<long long>(qn / 2);
  causal_dq_finalize<<<static_cast<unsigned>((npairs + 255) / 256), 256, 0, st>>>(cw.dq_acc, cw.rope, dq, npairs, T,
                                                                                 Hq, scale, rope);
  return cudaGetLastError();
}

}  // namespace abw
