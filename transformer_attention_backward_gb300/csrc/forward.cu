// Causal attention forward that produces what the backward consumes: the
// output O (bf16) and the log-sum-exp of the scaled scores (fp32).
//
// Spec: the online-softmax attention of the FlashAttention commits of Hesper
// pull request #1 (flashAttentionSpec, shown equal to the three-step
// standardAttention: scores, softmax, apply), over the causal mask of
// DaisyChain-Train transformer.js forward().  Per query row i, over key
// blocks j = 0, 1, ...: m = running max, l = running sum of exp(s - m),
// O = running sum of exp(s - m) v; a block whose max exceeds m rescales l
// and O by exp(m_old - m_new).  At the end O / l is the attention output and
// m + log l the log-sum-exp.
//
// Design (sm_103a, tcgen05): one CTA per (128-query block, head, batch),
// heads in groups of 8 with the heaviest query blocks of a group first.  Warp 0 loads Q once and K / V blocks of 128
// keys through a 3-deep TMA ring; warp 1 issues
//   S = Q K^T   (M=128 queries, N=128 keys, K=128: TMEM, two buffers)
//   O += P V    (M=128 queries, N=128 dims, K=128 keys: A = P in TMEM)
// in the order S(0) S(1) | PV(0) S(2) | PV(1) S(3) ..., so the softmax warps
// work on S(n+1) while PV(n) and S(n+2) run (K / V through a 3-deep ring); warps 2-5 (one TMEM lane
// quarter each, thread = query row) form P and write it as bf16 over S.  The
// rescale is lazy: the running max moves only when a block's max exceeds it
// by more than 8 (base 2), so P <= 2^8 between rescales; a rescale waits for
// the previous PV product and scales the row's O accumulator in TMEM.
// TMEM: [0,128) O, [128,256) S0 / P0, [256,384) S1 / P1.
#include <math.h>

#include "abw_host.h"
#include "tcgen05.cuh"

namespace abw {
namespace {

constexpr int kFD = 128;              // head dim
constexpr int kFB = 128;              // queries per CTA, keys per block
constexpr int kFThr = 192;            // 6 warps
constexpr int kFOffQ = 0;             // [2 D-halves][128 rows][128 B]
constexpr int kFOffKV = 32768;        // kFStages stages of [K 32 KB | V 32 KB]
constexpr int kFStages = 3;
constexpr int kFStage = 65536;
constexpr int kFOffBar = kFOffKV + kFStages * kFStage;
enum {
  kFBarQ = 0, kFBarKVFull = 1, kFBarKVEmpty = kFBarKVFull + kFStages, kFBarSFull = kFBarKVEmpty + kFStages,
  kFBarPFull = kFBarSFull + 2, kFBarO = kFBarPFull + 2, kFBarFinal = kFBarO + 1, kFNumBars = kFBarFinal + 1
};
constexpr int kFOffTmem = kFOffBar + kFNumBars * 8;
constexpr int kFOffAbort = kFOffTmem + 4;
constexpr int kFSmem = kFOffBar + 256 + 1024;   // + alignment slack
static_assert(kFOffTmem + 8 <= kFOffBar + 256 && kFSmem <= 232448, "forward kernel shared memory");
constexpr uint32_t kFColO = 0, kFColS0 = 128, kFColS1 = 256;
constexpr float kRescale = 8.f;       // lazy-rescale threshold (base-2 units)
constexpr int kFHeadGroup = 8;        // (batch, head) pairs per scheduling group

struct FwdParams {
  __nv_bfloat16 *o;
  float *lse;
  int B, T, Hq, Hkv, G, nqb;
  float scale;
  WaitCtl wait;
};

__device__ __forceinline__ float fexp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// 32 lanes x 32 columns, four times (columns c0, c0 + 32, c0 + 64, c0 + 96),
// one wait: a thread's whole 128-column row.
__device__ __forceinline__ void ld128_wait(uint32_t taddr, float (&v)[128]) {
  float (&a)[32] = *reinterpret_cast<float (*)[32]>(&v[0]);
  float (&b)[32] = *reinterpret_cast<float (*)[32]>(&v[32]);
  float (&c)[32] = *reinterpret_cast<float (*)[32]>(&v[64]);
  float (&d)[32] = *reinterpret_cast<float (*)[32]>(&v[96]);
  tc::ld32x2_wait(taddr, taddr + 32, a, b);
  tc::ld32x2_wait(taddr + 64, taddr + 96, c, d);
}

__global__ void __launch_bounds__(kFThr, 1)
    causal_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // item: (query block m, head h, batch b).  The (batch, head) pairs go in
  // groups of kFHeadGroup; within a group the heavy (late) query blocks come
  // first.  The CTAs that run at one time then cover few heads, whose K and
  // V (every query block of a head re-reads them) stay in L2.
  const int nh = p.Hq * p.B;
  const int grp = static_cast<int>(blockIdx.x) / (kFHeadGroup * p.nqb);
  const int gsz = min(kFHeadGroup, nh - grp * kFHeadGroup);
  const int in_grp = static_cast<int>(blockIdx.x) - grp * kFHeadGroup * p.nqb;
  const int m = p.nqb - 1 - in_grp / gsz;
  const int hb = grp * kFHeadGroup + in_grp % gsz;   // b * Hq + h
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int kvh = h / p.G;
  const int q0 = m * kFB;
  const int N = m + 1;                    // key blocks 0 .. m

  auto bar = [&](int i) -> uint32_t { return sb + kFOffBar + i * 8; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kFOffAbort);
  auto wt = [&](uint32_t br, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(br, parity, p.wait.limit_ns)) return true;
    *abort_flag = 1;
    report_timeout(p.wait.err, kSiteFwd, (br - sb - kFOffBar) / 8);
    return false;
  };
  auto wtw = [&](uint32_t br, uint32_t parity) -> bool { return __shfl_sync(0xffffffffu, wt(br, parity), 0); };

  if (tid == 0) {
    mbar_init(bar(kFBarQ), 1);
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(bar(kFBarKVFull + s), 1);
      mbar_init(bar(kFBarKVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kFBarSFull + s), 1);
      mbar_init(bar(kFBarPFull + s), 128);   // every softmax thread has written its P row
    }
    mbar_init(bar(kFBarO), 1);
    mbar_init(bar(kFBarFinal), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(sb + kFOffTmem, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kFOffTmem);

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_arrive_expect_tx(bar(kFBarQ), 2 * 16384);
      for (int hx = 0; hx < 2; ++hx) tma_load_4d(sb + kFOffQ + hx * 16384, &tmQ, hx * 64, h, q0, b, bar(kFBarQ));
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int s = n % kFStages;
        if (!wt(bar(kFBarKVEmpty + s), ((n / kFStages) & 1) ^ 1)) break;
        const uint32_t st = sb + kFOffKV + s * kFStage;
        const uint32_t fb = bar(kFBarKVFull + s);
        mbar_arrive_expect_tx(fb, 4 * 16384);
        for (int hx = 0; hx < 2; ++hx) {
          tma_load_4d(st + hx * 16384, &tmK, hx * 64, kvh, n * kFB, b, fb);
          tma_load_4d(st + 32768 + hx * 16384, &tmV, hx * 64, kvh, n * kFB, b, fb);
        }
        issued = n + 1;
      }
      if (*abort_flag) {
        for (int n = (issued > kFStages ? issued - kFStages : 0); n < issued; ++n)
          mbar_wait_bounded(bar(kFBarKVFull + n % kFStages), (n / kFStages) & 1, 2000000000ull);
        mbar_wait_bounded(bar(kFBarQ), 0, 2000000000ull);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    constexpr uint32_t id_s = tc::idesc_bf16_f32(128, 128, 0, 0);    // S = Q K^T, both K-major
    constexpr uint32_t id_o = tc::idesc_bf16_f32(128, 128, 0, 1);    // O += P V, V MN-major
    const uint64_t dQ = tc::sdesc_sw128(sb + kFOffQ, 16, 1024);
    const uint64_t dK = tc::sdesc_sw128(sb + kFOffKV, 16, 1024);
    const uint64_t dVm = tc::sdesc_sw128(sb + kFOffKV + 32768, 16384, 1024);
    auto kstep = [](int kk) -> uint32_t { return static_cast<uint32_t>((kk >> 2) * 16384 + (kk & 3) * 32) >> 4; };
    bool ok = wtw(bar(kFBarQ), 0);
    tc::fence_after_sync();
    // S(n) into buffer n & 1.  That buffer last held P(n - 2), read by
    // PV(n - 2), which was issued before (in-order execution).
    auto issue_s = [&](int n) -> bool {
      if (!wtw(bar(kFBarKVFull + n % kFStages), (n / kFStages) & 1)) return false;
      tc::fence_after_sync();
      const uint64_t so = static_cast<uint64_t>((n % kFStages) * kFStage) >> 4;
      const uint32_t tS = tmem + ((n & 1) ? kFColS1 : kFColS0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_w(tS, dQ + kstep(kk), dK + so + kstep(kk), id_s, kk > 0);
      tc::commit_w(bar(kFBarSFull + (n & 1)));
      return true;
    };
    if (ok) ok = issue_s(0);
    if (ok && N > 1) ok = issue_s(1);
    for (int n = 0; ok && n < N; ++n) {
      if (!wtw(bar(kFBarPFull + (n & 1)), (n >> 1) & 1)) break;
      tc::fence_after_sync();
      const uint64_t so = static_cast<uint64_t>((n % kFStages) * kFStage) >> 4;
      const uint32_t tP = tmem + ((n & 1) ? kFColS1 : kFColS0);
      // P chunk c (16 keys) sits in the 8 columns 32 (c / 2) + 8 (c % 2)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16_ts_w(tmem + kFColO, tP + (kk >> 1) * 32 + (kk & 1) * 8, dVm + so + ((kk * 2048) >> 4), id_o,
                          (n > 0 || kk > 0));
      tc::commit_w(bar(kFBarO));                    // O holds blocks 0 .. n
      tc::commit_w(bar(kFBarKVEmpty + n % kFStages));   // K / V stage of block n is free
      if (n + 2 < N && !issue_s(n + 2)) break;
    }
    tc::commit_w(bar(kFBarFinal));
    mbar_wait_bounded(bar(kFBarFinal), 0, 2000000000ull);   // every MMA has completed
  } else {
    // ============================ softmax warps ===========================
    const int qd = warp & 3;                           // TMEM lane quarter
    const int i = 32 * qd + lane;                      // query row in the block
    const int q = q0 + i;
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;   // scores in base-2 units
    float mrun = -INFINITY, lrun = 0.f;
    bool ok = true;
    for (int n = 0; n < N; ++n) {
      if (!wtw(bar(kFBarSFull + (n & 1)), (n >> 1) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t tS = tmem + lanebase + ((n & 1) ? kFColS1 : kFColS0);
      float s[128];
      ld128_wait(tS, s);
      // only the diagonal block is masked; a separate copy of the loop keeps
      // the common one free of the test
      float mb = -INFINITY;
      if (n == m) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          s[c] = n * kFB + c > q ? -INFINITY : s[c] * sl2;
          mb = fmaxf(mb, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          s[c] *= sl2;
          mb = fmaxf(mb, s[c]);
        }
      }
      // lazy rescale: only when some row of the warp moves its max by > 8.
      // Every phase of the O barrier (one per PV product) is waited for, in
      // order, once per block: here when the block rescales, else just before
      // P(n) is handed over.  A wait that skipped phases could be satisfied
      // by the parity of an older phase whose arrival lands late (measured:
      // sporadic rows whose rescale raced with PV(n - 1)).
      bool waited = false;
      const bool need = mb > mrun + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float mnew = need ? mb : mrun;
        const float f = (mrun == -INFINITY) ? 0.f : fexp2(mrun - mnew);
        lrun *= f;
        mrun = mnew;
        if (n > 0) {
          // O holds blocks 0 .. n - 1 once PV(n - 1) has completed
          if (!wtw(bar(kFBarO), (n - 1) & 1)) {
            ok = false;
            break;
          }
          waited = true;
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {   // 32 columns at a time: s[] stays live
            float o[32];
            tc::ld32_wait(tmem + lanebase + kFColO + c, o);
            uint32_t ra[16], rb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              ra[e] = __float_as_uint(o[e] * f);
              rb[e] = __float_as_uint(o[16 + e] * f);
            }
            tc::st16x2_wait(tmem + lanebase + kFColO + c, ra, tmem + lanebase + kFColO + c + 16, rb);
          }
        }
      }
      // P = 2^(s - m), summed into l, written as bf16 over S: chunk c of 16
      // keys to columns 32 (c / 2) + 8 (c % 2)
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 8; c += 2) {
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float a0 = fexp2(s[16 * c + e] - mrun), a1 = fexp2(s[16 * c + e + 1] - mrun);
          const float b0 = fexp2(s[16 * c + 16 + e] - mrun), b1 = fexp2(s[16 * c + 16 + e + 1] - mrun);
          ls += (a0 + a1) + (b0 + b1);
          pa[e / 2] = pack2(a0, a1);
          pb[e / 2] = pack2(b0, b1);
        }
        tc::st8x2_async(tS + 32 * (c >> 1), pa, tS + 32 * (c >> 1) + 8, pb);
      }
      lrun += ls;
      if (n > 0 && !waited && !wtw(bar(kFBarO), (n - 1) & 1)) {
        ok = false;
        break;
      }
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(kFBarPFull + (n & 1)));
    }
    // ---- epilogue: O / l as bf16 rows, lse = (m + log2 l) ln 2
    if (ok && wtw(bar(kFBarO), (N - 1) & 1)) {
      tc::fence_after_sync();
      float o[128];
      ld128_wait(tmem + lanebase + kFColO, o);
      if (q < p.T) {
        const float inv = 1.f / lrun;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((static_cast<size_t>(b) * p.T + q) * p.Hq + h) * kFD);
#pragma unroll
        for (int c = 0; c < 128; c += 8)
          dst[c / 8] = make_uint4(pack2(o[c] * inv, o[c + 1] * inv), pack2(o[c + 2] * inv, o[c + 3] * inv),
                                  pack2(o[c + 4] * inv, o[c + 5] * inv), pack2(o[c + 6] * inv, o[c + 7] * inv));
        p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.T + q] = (mrun + __log2f(lrun)) * 0.69314718055994531f;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

bool fmap(CUtensorMap *mp, const void *base, int H, int T, int B, const char **why) {
  const uint64_t dims[4] = {kFD, static_cast<uint64_t>(H), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {kFD * 2, static_cast<uint64_t>(H) * kFD * 2, static_cast<uint64_t>(T) * H * kFD * 2};
  const uint32_t box[4] = {64, 1, kFB, 1};
  return encode_tiled(mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                      why);
}

}  // namespace

cudaError_t launch_attn_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse, int B, int T,
                                   int Hq, int Hkv, int D, float scale, const WaitCtl &w, cudaStream_t st,
                                   const char **why) {
  if (D != kFD) {
    *why = "D != 128";
    return cudaErrorNotSupported;
  }
  const int nqb = (T + kFB - 1) / kFB;
  const long long ctas = static_cast<long long>(nqb) * Hq * B;
  if (ctas > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorNotSupported;
  }
  CUtensorMap tq, tk, tv;
  if (!fmap(&tq, q, Hq, T, B, why) || !fmap(&tk, k, Hkv, T, B, why) || !fmap(&tv, v, Hkv, T, B, why))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.nqb = nqb;
  p.scale = scale;
  p.wait = w;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(causal_fwd_kernel), kFSmem);
  if (e != cudaSuccess) return e;
  causal_fwd_kernel<<<static_cast<unsigned>(ctas), kFThr, kFSmem, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace abw
