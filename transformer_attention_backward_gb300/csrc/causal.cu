// Causal multi-query attention backward (keys j <= query i), probabilities
// recomputed from the saved log-sum-exp; RoPE backward fused on dq and dk.
//
// Spec: DaisyChain-Train transformer.js, backward(): dV = A^T dctx,
// dA = dctx V^T, dS = A (dA - sum_j A dA) scale, dQ = dS K, dK = dS^T Q,
// over the causal softmax of forward(); "Hesper.Training.VerifiedBackward"
// sections Softmax / Scaled Dot-Product / RoPE for the per-element steps.
//
// Launches per call:
//   1. prep : delta_i = dout_i . o_i (the identity sum_j P_ij dP_ij =
//             dout_i . o_i) and lse_i * log2(e), both padded to a multiple of
//             128 queries (padding: delta 0, lse +inf so P = 0 there); the
//             table of scale * (cos, sin) of theta(t, i) with RoPE
//   2. kv   : tcgen05 kernel, one CTA per (128-key block, KV head, batch):
//             dK and dV accumulate in TMEM over every query block at or after
//             the key block; each bf16 dS tile leaves for the workspace
//   3. dq   : tcgen05 kernel, one CTA per (128-query block, head, batch):
//             dQ^T = K^T dS^T accumulates in TMEM over the key blocks at or
//             before the query block; dq is written once, scaled and rotated
//
// Splitting dQ off trades an fp32 reduction of every (query block, key block)
// partial into dq (32 KB of L2 atomics per 64 x 128 tile, which sets the pace
// of a fused kernel) for a plain 16 KB store and load of the bf16 dS tile the
// dK product already uses; no product is recomputed.
//
// kv kernel (sm_103a, 12 warps, one CTA per SM).  Per CTA the K and V block
// stays in shared memory; the CTA loops over the query heads of its KV group
// and the 64-query blocks at or after its key block:
//   MMA1  S^T  = K Q^T          M=128 keys, N=64 queries, K=128 (TMEM)
//   MMA2  dP^T = V dO^T         same shape
//   softmax warps: P = exp2(S scale log2e - lse log2e) (causal mask),
//          dS = P (dP - delta), both rounded to bf16 into swizzled smem
//   MMA3  dV  += P^T dO          M=128 keys, N=128, K=64 queries
//   MMA4  dK  += dS^T Q          same shape
//   dS store warp: the 16 KB dS^T tile -> workspace (bulk async copy)
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 3 dS store, 4-11
// softmax (8 warps: four 32-key lane quarters x two 32-query halves), then
// the dK (4-7: scale + RoPE) and dV (8-11) epilogues.  S/dP are
// double-buffered in TMEM so the tensor core computes block n+1 while the
// softmax warps work on block n.  TMEM (512 columns):
//   [0,64) S0   [64,128) dP0   [128,192) S1   [192,256) dP1
//   [256,384) dV   [384,512) dK
// Q / dO / lse / delta arrive through a 4-deep TMA ring.
//
// dq kernel (12 warps, one CTA per SM): per key block the K block (32 KB)
// and the two dS^T tiles of the CTA's query blocks (2 x 16 KB, adjacent in
// the workspace) arrive through a 3-deep ring; MMA dQ^T += K^T dS^T with
// M=128 (head dim), N=128 queries, K=128 keys.  Epilogue warps 4-11 read
// dQ^T from TMEM (lane = head-dim index), pair lanes d and d^1 for RoPE and
// store dq rows.
#include <math.h>

#include <mutex>

#include "abw_host.h"
#include "tcgen05.cuh"

namespace abw {
namespace {

constexpr int kD = 128;
constexpr int kBK = 128;   // keys per kv CTA, queries per dq CTA
constexpr int kBQ = 64;    // queries per block (one dS tile)
constexpr int kThr = 384;  // 12 warps
constexpr int kTileBytes = kBK * kBQ * 2;   // one bf16 dS^T tile

// kv kernel shared memory.  It fills all but a few hundred bytes of the 227
// KB a CTA may have, so there is no slack to align the base by hand: the
// kernel checks that the dynamic shared memory starts on a 1024-byte boundary
// (which the 128B-swizzled tiles need) and otherwise reports and returns.
constexpr int kOffK = 0;                 // [2 D-halves][128 keys][128 B], 128B-swizzled
constexpr int kOffV = 32768;
constexpr int kStages = 4;               // Q / dO / lse / delta ring depth
constexpr int kOffStage = 65536;
constexpr int kStageBytes = 32768;       // Q 16 KB, dO 16 KB
constexpr int kStQ = 0, kStDO = 16384;
constexpr int kOffP = kOffStage + kStages * kStageBytes;   // P^T [128 keys][64 queries] bf16, swizzled
constexpr int kOffDS = kOffP + 16384;                 // dS^T [128 keys][64 queries] bf16, swizzled
constexpr int kOffLD = kOffDS + 16384;                // per stage: lse2 [64] f32, delta [64] f32
constexpr int kOffBar = kOffLD + kStages * 512;
constexpr int kSmem = kOffBar + 256;

// kv kernel barrier slots (8 bytes each) after kOffBar.
enum {
  kBarKV = 0, kBarQFull = 1, kBarQEmpty = 5, kBarSFull = 9, kBarPFull = 11, kBarPEmpty = 12,
  kBarTEmpty = 13, kBarDKV = 15, kBarFinal = 16, kNumBars = 17
};
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
static_assert(kOffAbort + 4 <= kSmem && kSmem <= 232448, "kv kernel shared memory");

constexpr uint32_t kColS0 = 0, kColDP0 = 64, kColS1 = 128, kColDP1 = 192, kColDV = 256, kColDK = 384;

// dq kernel shared memory: 3 stages of [K block 32 KB | two dS^T tiles 32 KB].
constexpr int kQStages = 3;
constexpr int kQStageBytes = 65536;
constexpr int kQOffDS = 32768;
constexpr int kQOffBar = kQStages * kQStageBytes;
enum { kQBarFull = 0, kQBarEmpty = 3, kQBarDone = 6, kQNumBars = 7 };
constexpr int kQOffTmemSlot = kQOffBar + kQNumBars * 8;
constexpr int kQOffAbort = kQOffTmemSlot + 4;
constexpr int kQSmem = kQOffBar + 256 + 1024;

struct CausalWs {
  float *delta;        // [B][Hq][Tp]
  float *lse2;         // [B][Hq][Tp]  lse * log2(e), +inf past T
  float2 *rope;        // [T][D/2] scale * (cos, sin)
  __nv_bfloat16 *ds;   // [B][Hq][tiles per head][128 keys][64 queries], swizzled tiles
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Queries and keys padded to whole 128-blocks: every key block then sees an
// even number of 64-query blocks, and the dq kernel's two tiles always exist.
int padded_T(int T) { return (T + kBK - 1) / kBK * kBK; }

// dS^T tiles of one head: key block kb pairs with query blocks 2 kb ..
// nqb - 1 (nqb = 2 nkb), stored key block by key block.
long long tiles_per_head(int nkb) { return static_cast<long long>(nkb) * nkb + nkb; }

CausalWs carve(void *ws, int B, int T, int Hq, int D) {
  const size_t Tp = static_cast<size_t>(padded_T(T));
  CausalWs w;
  char *p = static_cast<char *>(ws);
  p += (256 - (reinterpret_cast<uintptr_t>(p) & 255)) & 255;
  w.delta = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * Hq * Tp * 4);
  w.lse2 = reinterpret_cast<float *>(p);
  p += up256(static_cast<size_t>(B) * Hq * Tp * 4);
  w.rope = reinterpret_cast<float2 *>(p);
  p += up256(static_cast<size_t>(T) * (D / 2) * 8);
  w.ds = reinterpret_cast<__nv_bfloat16 *>(p);
  return w;
}

// One warp per (b, t, h) row, t < Tp: delta and lse*log2(e) (padding rows:
// 0 and +inf) and -- for b = h = 0, with RoPE -- the row of the table
// scale * (cos, sin) of theta = (pos0 + t) * base^(-2i/D).  The angle is
// formed and reduced modulo 2 pi in double and rounded to float only for
// sincosf.
__global__ void __launch_bounds__(256) causal_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                                                          const __nv_bfloat16 *__restrict__ dout,
                                                          const float *__restrict__ lse, float *__restrict__ delta,
                                                          float *__restrict__ lse2, float2 *__restrict__ rope, int B,
                                                          int T, int Tp, int Hq, float scale, int use_rope, int pos0,
                                                          double log2_base) {
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
  if (use_rope && b == 0 && h == 0) {
    const double twopi = 6.283185307179586476925286766559;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      const double a_ = static_cast<double>(pos0 + t) * exp2(-log2_base * (2.0 * i / kD));
      const float th = static_cast<float>(a_ - twopi * rint(a_ / twopi));
      float sn, c;
      sincosf(th, &sn, &c);
      rope[t * (kD / 2) + i] = make_float2(scale * c, scale * sn);
    }
  }
}

struct TcParams {
  CausalWs ws;
  float *dq, *dk, *dv;
  int B, T, Tp, Hq, Hkv, G, nkb, nqb;
  long long tph;   // dS^T tiles per head
  float scale;
  int rope;
  WaitCtl wait;
};

// Index of the dS^T tile (key block kb, query block qb >= 2 kb) within its head.
__device__ __forceinline__ long long tile_index(int kb, int qb, int nqb) {
  return static_cast<long long>(kb) * nqb - static_cast<long long>(kb) * (kb - 1) + (qb - 2 * kb);
}

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
    causal_kv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (sb & 1023) {
    if (tid == 0) atomicOr(p.wait.err, kErrSmemAlign);
    return;
  }

  // work item: heavy (early) key blocks first across the whole grid
  const int per_kb = p.Hkv * p.B;
  const int kb = blockIdx.x / per_kb;
  const int rem = blockIdx.x - kb * per_kb;
  const int kvh = rem % p.Hkv, b = rem / p.Hkv;
  const int k0 = kb * kBK;
  const int qb0 = k0 / kBQ;
  const int nq = p.nqb - qb0;            // query blocks per head
  const int N = p.G * nq;                // iterations of this CTA

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
      mbar_init(bar(kBarTEmpty + s), 256);   // the eight softmax warps have read S and dP
    }
    mbar_init(bar(kBarPFull), 256);
    mbar_init(bar(kBarPEmpty), 2);           // MMA3/4 done + dS tile copied out
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
        const int q0 = (qb0 + n % nq) * kBQ;
        const uint32_t st = sb + kOffStage + s * kStageBytes;
        const uint32_t fb = bar(kBarQFull + s);
        mbar_arrive_expect_tx(fb, 2 * 16384 + 2 * 256);
        for (int hx = 0; hx < 2; ++hx) {
          tma_load_4d(st + kStQ + hx * 8192, &tmQ, hx * 64, h, q0, b, fb);
          tma_load_4d(st + kStDO + hx * 8192, &tmDO, hx * 64, h, q0, b, fb);
        }
        const size_t ro = (static_cast<size_t>(b) * p.Hq + h) * p.Tp + q0;
        bulk_load(sb + kOffLD + s * 512, p.ws.lse2 + ro, 256, fb);
        bulk_load(sb + kOffLD + s * 512 + 256, p.ws.delta + ro, 256, fb);
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
      if (ok && N > 0) ok = issue_sdp(0);
      for (int n = 0; ok && n < N; ++n) {
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
        tc::commit(bar(kBarQEmpty + qs));
        tc::commit(bar(kBarPEmpty));
      }
      tc::commit(bar(kBarDKV));
      tc::commit(bar(kBarFinal));
      mbar_wait_bounded(bar(kBarFinal), 0, 2000000000ull);   // every MMA has completed
    }
  } else if (warp == 3) {
    // ============================ dS store ================================
    if (lane == 0) {
      for (int n = 0; n < N; ++n) {
        if (!wt(bar(kBarPFull), n & 1)) break;
        const int h = kvh * p.G + n / nq;
        const int qb = qb0 + n % nq;
        __nv_bfloat16 *head_tiles = p.ws.ds + (static_cast<size_t>(b) * p.Hq + h) * p.tph * (kTileBytes / 2);
        bulk_store(head_tiles + tile_index(kb, qb, p.nqb) * (kTileBytes / 2), sb + kOffDS, kTileBytes);
        bulk_commit_group();
        bulk_wait_group_read0();   // the dS buffer may be rewritten
        mbar_arrive(bar(kBarPEmpty));
      }
      bulk_wait_group0();          // the tiles are in global memory
    }
  } else if (warp >= 4) {
    // ============================ softmax warps ===========================
    const int qd = warp & 3;                            // TMEM lane quarter
    const int ch = (warp - 4) >> 2;                     // 32-query half
    const int j = 32 * qd + lane;                       // key row in the block
    const int key = k0 + j;
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;
    for (int n = 0; n < N; ++n) {
      const int s = n & 1, cyc = n >> 1;
      const int q0 = (qb0 + n % nq) * kBQ;
      if (!wt(bar(kBarSFull + s), cyc & 1)) break;
      tc::fence_after_sync();
      const int qs = n % kStages;
      const float *lse2 = reinterpret_cast<const float *>(smem + kOffLD + qs * 512) + 32 * ch;
      const float *dl = reinterpret_cast<const float *>(smem + kOffLD + qs * 512 + 256) + 32 * ch;
      float sv[32], pv[32];
      tc::ld32x2_wait(tmem + lanebase + (s ? kColS1 : kColS0) + 32 * ch,
                      tmem + lanebase + (s ? kColDP1 : kColDP0) + 32 * ch, sv, pv);
      tc::fence_before_sync();
      mbar_arrive(bar(kBarTEmpty + s));                 // S/dP buffer free for block n + 2
      // only the two query blocks that overlap the key block need the causal
      // mask; queries past T have lse = +inf, so their P is exactly 0
      const bool diag = q0 < k0 + kBK;
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + c);
        const float4 d4 = *reinterpret_cast<const float4 *>(dl + c);
        float P0 = fast_exp2(fmaf(sv[c], sl2, -l4.x));
        float P1 = fast_exp2(fmaf(sv[c + 1], sl2, -l4.y));
        float P2 = fast_exp2(fmaf(sv[c + 2], sl2, -l4.z));
        float P3 = fast_exp2(fmaf(sv[c + 3], sl2, -l4.w));
        if (diag) {
          const int q = q0 + 32 * ch + c;
          P0 = key <= q ? P0 : 0.f;
          P1 = key <= q + 1 ? P1 : 0.f;
          P2 = key <= q + 2 ? P2 : 0.f;
          P3 = key <= q + 3 ? P3 : 0.f;
        }
        const float dS0 = P0 * (pv[c] - d4.x), dS1 = P1 * (pv[c + 1] - d4.y);
        const float dS2 = P2 * (pv[c + 2] - d4.z), dS3 = P3 * (pv[c + 3] - d4.w);
        pk[c / 2] = pack_bf16x2(P0, P1);
        pk[c / 2 + 1] = pack_bf16x2(P2, P3);
        dk[c / 2] = pack_bf16x2(dS0, dS1);
        dk[c / 2 + 1] = pack_bf16x2(dS2, dS3);
      }
      if (!wt(bar(kBarPEmpty), (n & 1) ^ 1)) break;
      unsigned char *prow = smem + kOffP + j * 128;
      unsigned char *drow = smem + kOffDS + j * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int o = ((4 * ch + c4) ^ (j & 7)) << 4;   // 128B swizzle of 16-byte chunk 4 ch + c4
        *reinterpret_cast<uint4 *>(prow + o) = make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
        *reinterpret_cast<uint4 *>(drow + o) = make_uint4(dk[4 * c4], dk[4 * c4 + 1], dk[4 * c4 + 2], dk[4 * c4 + 3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(bar(kBarPFull));
    }
    if (wt(bar(kBarDKV), 0)) {
      tc::fence_after_sync();
      if (ch == 0) {
        // ---- dK epilogue: scale, RoPE backward, store
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tc::ld32_wait(tmem + lanebase + kColDK + 32 * c, v);
          if (key < p.T) {
            float *dst = p.dk + ((static_cast<size_t>(b) * p.T + key) * p.Hkv + kvh) * kD + 32 * c;
            // scale * (cos, sin) of the chunk's 16 pairs; the table holds
            // the scale already.  All loads come before the first store: a
            // load after a store to possibly the same memory would wait for it.
            float4 cs[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              cs[i] = p.rope ? *reinterpret_cast<const float4 *>(p.ws.rope + key * (kD / 2) + 16 * c + 2 * i)
                             : make_float4(p.scale, 0.f, p.scale, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float *x = v + 4 * i;
              *reinterpret_cast<float4 *>(dst + 4 * i) =
                  make_float4(x[0] * cs[i].x + x[1] * cs[i].y, -x[0] * cs[i].y + x[1] * cs[i].x,
                              x[2] * cs[i].z + x[3] * cs[i].w, -x[2] * cs[i].w + x[3] * cs[i].z);
            }
          }
        }
      } else {
        // ---- dV epilogue
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
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(kThr, 1)
    causal_dq_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // work item: query block pair m (queries 128 m .. 128 m + 127), heavy first
  const int per_m = p.Hq * p.B;
  const int m = p.nkb - 1 - static_cast<int>(blockIdx.x / per_m);
  const int rem = blockIdx.x % per_m;
  const int h = rem % p.Hq, b = rem / p.Hq;
  const int kvh = h / p.G;
  const int nsteps = m + 1;              // key blocks 0 .. m
  const __nv_bfloat16 *head_tiles = p.ws.ds + (static_cast<size_t>(b) * p.Hq + h) * p.tph * (kTileBytes / 2);

  auto bar = [&](int i) -> uint32_t { return sb + kQOffBar + i * 8; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kQOffAbort);
  auto wt = [&](uint32_t br, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(br, parity, p.wait.limit_ns)) return true;
    *abort_flag = 1;
    atomicOr(p.wait.err, kErrWaitTimeout);
    return false;
  };

  if (tid == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bar(kQBarFull + s), 1);
      mbar_init(bar(kQBarEmpty + s), 1);
    }
    mbar_init(bar(kQBarDone), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) tc::tmem_alloc(sb + kQOffTmemSlot, 128);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kQOffTmemSlot);

  if (warp == 0) {
    // ============================ producer ================================
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      int issued = 0;
      for (int i = 0; i < nsteps; ++i) {
        const int s = i % kQStages, cyc = i / kQStages;
        if (!wt(bar(kQBarEmpty + s), (cyc & 1) ^ 1)) break;
        const uint32_t st = sb + s * kQStageBytes;
        const uint32_t fb = bar(kQBarFull + s);
        mbar_arrive_expect_tx(fb, 2 * 16384 + 2 * kTileBytes);
        for (int hx = 0; hx < 2; ++hx) tma_load_4d(st + hx * 16384, &tmK, hx * 64, kvh, i * kBK, b, fb);
        // tiles (i, 2m) and (i, 2m + 1) are adjacent
        bulk_load(st + kQOffDS, head_tiles + tile_index(i, 2 * m, p.nqb) * (kTileBytes / 2), 2 * kTileBytes, fb);
        issued = i + 1;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        for (int i = (issued > kQStages ? issued - kQStages : 0); i < issued; ++i)
          mbar_wait_bounded(bar(kQBarFull + i % kQStages), (i / kQStages) & 1, 2000000000ull);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      constexpr uint32_t id_dq = tc::idesc_bf16_f32(128, 128, 1, 1);    // dQ^T += K^T dS^T
      for (int i = 0; i < nsteps; ++i) {
        const int s = i % kQStages, cyc = i / kQStages;
        if (!wt(bar(kQBarFull + s), cyc & 1)) break;
        tc::fence_after_sync();
        const uint32_t st = sb + s * kQStageBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_bf16(tmem, tc::sdesc_sw128(st + kk * 2048, 16384, 1024),
                       tc::sdesc_sw128(st + kQOffDS + kk * 2048, kTileBytes, 1024), id_dq, (i > 0 || kk > 0));
        tc::commit(bar(kQBarEmpty + s));
      }
      tc::commit(bar(kQBarDone));
      mbar_wait_bounded(bar(kQBarDone), 0, 2000000000ull);   // every MMA has completed
    }
  } else if (warp >= 4) {
    // ============================ epilogue ================================
    const int qd = warp & 3;                 // TMEM lane quarter = 32 head-dim rows
    const int ch = (warp - 4) >> 2;          // 64-query half
    const int d = 32 * qd + lane;
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    const bool odd = d & 1;
    if (wt(bar(kQBarDone), 0)) {
      tc::fence_after_sync();
      for (int cc = 0; cc < 2; ++cc) {
        float v[32];
        tc::ld32_wait(tmem + lanebase + 64 * ch + 32 * cc, v);
        const int qbase = m * kBK + 64 * ch + 32 * cc;
        // pair (2i, 2i+1) rotated by -theta; the table holds scale * (cos,
        // sin).  All 32 loads come before the first store: a load after a
        // store to possibly the same memory would wait for it.
        float2 cs[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int q = qbase + c;
          cs[c] = !p.rope ? make_float2(p.scale, 0.f)
                  : q < p.T ? p.ws.rope[q * (kD / 2) + (d >> 1)] : make_float2(0.f, 0.f);
        }
        float *dst = p.dq + ((static_cast<size_t>(b) * p.T + qbase) * p.Hq + h) * kD + d;
        const size_t qstride = static_cast<size_t>(p.Hq) * kD;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float partner = __shfl_xor_sync(0xffffffffu, v[c], 1);
          if (qbase + c < p.T) dst[c * qstride] = v[c] * cs[c].x + (odd ? -partner : partner) * cs[c].y;
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 128);
  }
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
  const int nkb = static_cast<int>(Tp / kBK);
  return 256 + 2 * up256(static_cast<size_t>(B) * Hq * Tp * 4) + up256(static_cast<size_t>(T) * (D / 2) * 8) +
         up256(static_cast<size_t>(B) * Hq * static_cast<size_t>(tiles_per_head(nkb)) * kTileBytes);
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
  const int Tp = padded_T(T);
  const int nkb = Tp / kBK;
  const long long kv_ctas = static_cast<long long>(nkb) * Hkv * B;
  const long long dq_ctas = static_cast<long long>(nkb) * Hq * B;
  if (kv_ctas > 0x7fffffffLL || dq_ctas > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorNotSupported;
  }
  CausalWs cw = carve(ws, B, T, Hq, D);
  const int rope = rope_base > 0.0;
  {
    const long long rows = static_cast<long long>(B) * Tp * Hq;
    const long long blocks = (rows * 32 + 255) / 256;
    causal_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse, cw.delta, cw.lse2,
        cw.rope, B, T, Tp, Hq, scale, rope, pos0, rope ? log2(rope_base) : 0.0);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tdo, tk, tv;
  if (!make_map(&tq, q, Hq, T, B, kBQ, why) || !make_map(&tdo, dout, Hq, T, B, kBQ, why) ||
      !make_map(&tk, k, Hkv, T, B, kBK, why) || !make_map(&tv, v, Hkv, T, B, kBK, why))
    return cudaErrorInvalidValue;
  TcParams p;
  p.ws = cw;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B; p.T = T; p.Tp = Tp; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.nkb = nkb;
  p.nqb = Tp / kBQ;
  p.tph = tiles_per_head(nkb);
  p.scale = scale;
  p.rope = rope;
  p.wait = w;
  e = cudaFuncSetAttribute(causal_kv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  causal_kv_tc_kernel<<<static_cast<unsigned>(kv_ctas), kThr, kSmem, st>>>(tq, tdo, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(causal_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  if (e != cudaSuccess) return e;
  causal_dq_tc_kernel<<<static_cast<unsigned>(dq_ctas), kThr, kQSmem, st>>>(tk, p);
  return cudaGetLastError();
}

}  // namespace abw
