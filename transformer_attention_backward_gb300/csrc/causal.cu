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
//             dK and dV accumulate in TMEM over every 128-query block at or
//             after the key block; each bf16 dS tile leaves for the workspace
//   3. dq   : persistent tcgen05 kernel over (128-query block, head, batch):
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
// and the 128-query blocks at or after its key block:
//   MMA1  S^T  = K Q^T          M=128 keys, N=128 queries, K=128 (TMEM)
//   MMA2  dP^T = V dO^T         same shape
//   softmax warps: P = exp2(S scale log2e - lse log2e) (causal mask on the
//          diagonal block), written back as bf16 into TMEM over the S values
//          just read; then dS = P (dP - delta), written over dP and, as a
//          128B-swizzled tile row, to the workspace
//   MMA3  dV  += P^T dO          M=128 keys, N=128, K=128 queries, A in TMEM
//   MMA4  dK  += dS^T Q          same shape
// S/dP are single-buffered; what keeps the tensor core busy is the order of
// the products and four separate signals (S ready, dP ready, P ready, dS
// ready): per block n the issue order is S(n) dP(n) | dV(n) S(n+1) |
// dK(n) dP(n+1), so P(n) is formed while dP(n) runs and dS(n) while dV(n)
// and S(n+1) run.  Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner,
// 4-11 softmax (warp w: 32-key lane quarter w % 4, query half (w - 4) / 4),
// then the dK (scale + RoPE) and dV epilogues, each half of the softmax
// warps taking half the columns of both.  TMEM (512 columns):
//   [0,128) S / P   [128,256) dP / dS   [256,384) dV   [384,512) dK
// Q (with lse) and dO (with delta) of one query block arrive through a
// 3-deep and a 2-deep TMA ring.
//
// dq kernel (persistent, 12 warps, one CTA per SM): for each work item (128
// queries of one head) and each key block at or before it, the K block
// (32 KB) and the item's two dS^T tiles (2 x 16 KB, adjacent in the
// workspace) arrive through a 3-deep ring that runs on across items; MMA
// dQ^T += K^T dS^T with M=128 (head dim), N=128 queries, K=128 keys into one
// of two TMEM accumulators.  Epilogue warps 4-11 read dQ^T (lane = head-dim
// index), free the accumulator, pair lanes d and d^1 for RoPE and store dq
// rows while the next item accumulates.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "abw_host.h"
#include "tcgen05.cuh"

namespace abw {
namespace {

constexpr int kD = 128;
constexpr int kBK = 128;   // keys per kv CTA, queries per dq CTA
constexpr int kBQ = 64;    // queries per dS tile
constexpr int kThr = 384;  // 12 warps
constexpr int kTileBytes = kBK * kBQ * 2;   // one bf16 dS^T tile
constexpr int kHeadGroup = 8;               // kv kernel: (batch, KV head) pairs per scheduling group

// kv kernel shared memory.  It fills all but a few hundred bytes of the 227
// KB a CTA may have, so there is no slack to align the base by hand: the
// kernel checks that the dynamic shared memory starts on a 1024-byte
// boundary (which the 128B-swizzled tiles need) and otherwise reports and
// returns.  One query block is 128 queries; its Q and its dO are each
// [2 D-halves][128 rows][128 B] 128B-swizzled (32 KB).  Q goes through a
// 3-deep ring (read by S and, last, dK) and dO through a 2-deep one (read by
// dP and, last, dV, which comes earlier in the block; after dV the slot
// stages the block's dS^T rows for their bulk copy to the workspace before
// it is refilled), so each block's copies are issued well before its first
// product.  The block's lse (512 B) rides with its Q copy into a ring of the
// Q ring's depth and its delta (512 B) with its dO copy into one of the dO
// ring's depth: the softmax warps are done with both before the slot they
// ride with is released, so no copy waits for the softmax.  At the end the K / V
// region stages the dV tiles (after the last dV), two Q slots the key
// block's RoPE rows (after the last dP) and the dO ring the dK tiles (after
// the last dK).
constexpr int kKvBQ = 128;               // queries per kv block (two dS^T tiles)
constexpr int kOffK = 0;                 // [2 D-halves][128 keys][128 B], 128B-swizzled
constexpr int kOffV = 32768;
constexpr int kQStagesKv = 3, kDOStages = 2;
constexpr int kBlockBytes = 32768;       // one Q or dO block
constexpr int kOffQ = 65536;
constexpr int kOffDO = kOffQ + kQStagesKv * kBlockBytes;
constexpr int kHalfQ = 16384;            // one 64-dim half of a Q / dO block
constexpr int kOffLse = kOffDO + kDOStages * kBlockBytes;      // per Q slot: lse2 [128] f32
constexpr int kOffDelta = kOffLse + kQStagesKv * 512;          // per dO slot: delta [128] f32
constexpr int kOffBar = kOffDelta + kDOStages * 512;

// kv kernel barrier slots (8 bytes each) after kOffBar.
enum {
  kBarKV = 0, kBarV = 1, kBarQFull = 2, kBarQEmpty = kBarQFull + kQStagesKv, kBarDOFull = kBarQEmpty + kQStagesKv,
  kBarDOEmpty = kBarDOFull + kDOStages, kBarSFull = kBarDOEmpty + kDOStages,
  kBarDPFull = kBarSFull + 1, kBarPFull = kBarDPFull + 1, kBarDSFull = kBarPFull + 1, kBarDVDone = kBarDSFull + 1,
  kBarStaged = kBarDVDone + 1, kBarRope = kBarStaged + 2, kBarDVFinal = kBarRope + 1, kBarDKV = kBarDVFinal + 1,
  kBarFinal = kBarDKV + 1, kNumBars = kBarFinal + 1
};
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
// dO slot 1's two staged barriers (slot 0's are kBarStaged, kBarStaged + 1),
// placed after the other words so that those keep their offsets (moving the
// barrier block by 16 bytes measured 2 % slower)
constexpr int kOffStaged1 = kOffAbort + 4;
static_assert(kDOStages == 2, "one pair of staged barriers per dO slot");
constexpr int kSmem = kOffBar + 256;
static_assert(kOffStaged1 % 8 == 0 && kOffStaged1 + 16 <= kSmem && kSmem <= 232448, "kv kernel shared memory");

// kv kernel TMEM columns: S^T / P^T, dP^T / dS^T (one query block each), dV, dK.
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

// dq kernel shared memory: 3 stages of [K block 32 KB | two dS^T tiles 32 KB].
constexpr int kQStages = 3;
constexpr int kQStageBytes = 65536;
constexpr int kQOffDS = 32768;
constexpr int kQOffBar = kQStages * kQStageBytes;
enum { kQBarFull = 0, kQBarEmpty = 3, kQBarAccFull = 6, kQBarAccEmpty = 8, kQBarFinal = 10, kQNumBars = 11 };
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

// Position of RoPE pair i of position t in the table: rows of 64 pairs
// (512 B), the 16-byte units (two pairs) of a row XOR-swizzled by t % 8, so
// that a warp reading one unit of 32 consecutive rows out of shared memory
// touches every bank the same number of times.
__host__ __device__ __forceinline__ int rope_slot(int t, int i) {
  return t * (kD / 2) + ((((i >> 1) ^ (t & 7)) << 1) | (i & 1));
}

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

// delta and lse*log2(e) per (b, h, t < Tp) and, with RoPE, the table
// scale * (cos, sin) of theta = (pos0 + t) * base^(-2i/D).  A half-warp takes
// kPrepRows rows of o and dout, consecutive in (b, t, h) order (16 bytes per
// lane and tensor, all loads issued before the first reduction); table
// entries are strided over the grid's threads; padding entries t in [T, Tp) get delta 0 and lse +inf,
// one per thread.  The RoPE angle is formed and reduced modulo 2 pi in
// double and rounded to float only for sincosf.
constexpr int kPrepRows = 4;

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 g) {
  return bf16_lo(a.x) * bf16_lo(g.x) + bf16_hi(a.x) * bf16_hi(g.x) + bf16_lo(a.y) * bf16_lo(g.y) +
         bf16_hi(a.y) * bf16_hi(g.y) + bf16_lo(a.z) * bf16_lo(g.z) + bf16_hi(a.z) * bf16_hi(g.z) +
         bf16_lo(a.w) * bf16_lo(g.w) + bf16_hi(a.w) * bf16_hi(g.w);
}

struct PrepRope {
  double inv_freq[kD / 2];   // base^(-2i/D), formed on the host in double
  float scale;
  int use_rope, pos0;
  float *zero_dk, *zero_dv;  // zeroed when zero_n4 > 0 (float4 count of each)
  long long zero_n4;
};

__global__ void __launch_bounds__(256) causal_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                                                          const __nv_bfloat16 *__restrict__ dout,
                                                          const float *__restrict__ lse, float *__restrict__ delta,
                                                          float *__restrict__ lse2, float2 *__restrict__ rope, int B,
                                                          int T, int Tp, int Hq, const __grid_constant__ PrepRope rp) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  // with the kv kernel's head groups split over CTAs, dK and dV receive
  // partial sums by reduction: zero them first (16 bytes per thread, strided
  // over the grid)
  if (rp.zero_n4 > 0) {
    const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = gid; e < rp.zero_n4; e += nthr) {
      reinterpret_cast<float4 *>(rp.zero_dk)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4 *>(rp.zero_dv)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const int sub = threadIdx.x & 15;
  // padding entries
  const long long npad = static_cast<long long>(B) * Hq * (Tp - T);
  if (gid < npad) {
    const long long bh = gid / (Tp - T);
    const int t = T + static_cast<int>(gid % (Tp - T));
    delta[bh * Tp + t] = 0.f;
    lse2[bh * Tp + t] = INFINITY;
  }
  // Rows are taken in memory order (b, t, h): a block's rows of o and dout
  // are one contiguous stretch (DRAM pages are read whole), and only the
  // small delta / lse accesses are strided.
  const long long nrows = static_cast<long long>(B) * T * Hq;
  const long long r0 = (gid >> 4) * kPrepRows;
  int hh = static_cast<int>(r0 % Hq), tt, bb;
  {
    const long long bt = r0 / Hq;
    tt = static_cast<int>(bt % T);
    bb = static_cast<int>(bt / T);
  }
  int rh[kPrepRows], rt[kPrepRows], rb[kPrepRows];
#pragma unroll
  for (int k = 0; k < kPrepRows; ++k) {
    rh[k] = hh;
    rt[k] = tt;
    rb[k] = bb;
    if (++hh == Hq) {
      hh = 0;
      if (++tt == T) {
        tt = 0;
        ++bb;
      }
    }
  }
  uint4 a[kPrepRows], g[kPrepRows];
  float l[kPrepRows];
#pragma unroll
  for (int k = 0; k < kPrepRows; ++k) {
    if (r0 + k < nrows) {
      const size_t src = ((static_cast<size_t>(rb[k]) * T + rt[k]) * Hq + rh[k]) * kD;
      a[k] = reinterpret_cast<const uint4 *>(o + src)[sub];
      g[k] = reinterpret_cast<const uint4 *>(dout + src)[sub];
      l[k] = lse ? lse[(static_cast<size_t>(rb[k]) * Hq + rh[k]) * T + rt[k]] : 0.f;
    } else {
      a[k] = make_uint4(0, 0, 0, 0);
      g[k] = a[k];
      l[k] = 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < kPrepRows; ++k) {
    float v = dot8_bf16(a[k], g[k]);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);   // within the half-warp
    if (r0 + k < nrows) {
      const size_t out = (static_cast<size_t>(rb[k]) * Hq + rh[k]) * Tp + rt[k];
      if (sub == 0) {
        delta[out] = v;
        lse2[out] = l[k] * 1.4426950408889634f;
      }
    }
  }
  // RoPE table: (t, i) entries strided over every thread of the grid (one
  // each once B * Hq >= 16), so the double-precision angle reduction is
  // spread over all SMs instead of a few half-warps
  if (rp.use_rope) {
    const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
    const double twopi = 6.283185307179586476925286766559, inv_twopi = 0.15915494309189533576888376337251;
    for (long long e = gid; e < static_cast<long long>(T) * (kD / 2); e += nthr) {
      const int t = static_cast<int>(e / (kD / 2)), i = static_cast<int>(e % (kD / 2));
      const double ang = static_cast<double>(rp.pos0 + t) * rp.inv_freq[i];
      const float th = static_cast<float>(fma(-twopi, rint(ang * inv_twopi), ang));
      float sn, c;
      __sincosf(th, &sn, &c);   // |th| <= pi: absolute error ~1e-6, far below the bf16 inputs' rounding
      rope[rope_slot(t, i)] = make_float2(rp.scale * c, rp.scale * sn);
    }
  }
}

constexpr int kMaxVarKb = 32;   // key blocks up to which the kv split may vary per key block
struct TcParams {
  CausalWs ws;
  float *dq, *dk, *dv;
  const __nv_bfloat16 *pattn;   // saved probabilities [B][Hq][T][T] (row = query), or null: recompute from lse
  int B, T, Tp, Hq, Hkv, G, nkb, nqb;
  int hsplit, gs;  // kv kernel: each KV head's G query heads go to hsplit CTAs, gs = G / hsplit each
  // kv kernel, small grids: the split chosen per key block instead (nsplit[kb]
  // CTAs per (batch, KV head), kb_first[kb] the index of the key block's
  // first CTA), so that a CTA's blocks (heads x query blocks) stay within
  // one key block row's worth; var_split = 0 uses hsplit for every key block.
  int var_split;
  int nsplit[kMaxVarKb], kb_first[kMaxVarKb + 1];
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

// kSavedP: P comes from the saved probabilities (no S product) instead of
// being recomputed from lse; one instantiation per form keeps the softmax
// loop free of the test.
template <bool kSavedP>
__global__ void __launch_bounds__(kThr, 1)
    causal_kv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                        const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The dq kernel (launched as this grid's programmatic dependent) may take
  // the SMs this grid's last CTAs leave idle; it waits for this grid's
  // completion before it reads any dS tile.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (sb & 1023) {
    if (tid == 0) atomicOr(p.wait.err, kErrSmemAlign);
    return;
  }

  // Work item: (key block, batch, KV head, head split).  The (batch, KV head,
  // split) units go in groups of kHeadGroup; within a group the heavy (early)
  // key blocks come first.  The CTAs that run at one time then cover few
  // heads, whose Q and dO (every key block of a head re-reads them) stay in
  // L2 between the key blocks.
  int kb, b, kvh, h_first, gs;   // query heads h_first .. h_first + gs - 1
  if (p.var_split) {
    // key blocks in order (the heaviest first); within one, nsplit[kb] CTAs
    // per (batch, KV head)
    kb = 0;
    while (kb + 1 < p.nkb && static_cast<int>(blockIdx.x) >= p.kb_first[kb + 1]) ++kb;
    const int u = blockIdx.x - p.kb_first[kb], ns = p.nsplit[kb];
    const int unit = u / ns;   // b * Hkv + kvh
    kvh = unit % p.Hkv;
    b = unit / p.Hkv;
    gs = p.G / ns;
    h_first = kvh * p.G + (u % ns) * gs;
  } else {
    const int nh = p.Hkv * p.B * p.hsplit;
    const int grp = blockIdx.x / (kHeadGroup * p.nkb);
    const int gsz = min(kHeadGroup, nh - grp * kHeadGroup);
    const int in_grp = blockIdx.x - grp * kHeadGroup * p.nkb;
    kb = in_grp / gsz;
    const int hb = grp * kHeadGroup + in_grp % gsz;   // (b * Hkv + kvh) * hsplit + split
    kvh = (hb / p.hsplit) % p.Hkv;
    b = hb / (p.hsplit * p.Hkv);
    gs = p.gs;
    h_first = kvh * p.G + (hb % p.hsplit) * gs;
  }
  // with the group split over CTAs, dK / dV receive partial sums
  const bool split_group = gs < p.G;
  const int k0 = kb * kBK;
  const int nq = p.nkb - kb;             // 128-query blocks at or after the key block, per head
  const int N = gs * nq;                 // iterations of this CTA

  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + i * 8; };
  // Block n's dS is staged in dO slot n % 2, and each slot has its own pair
  // of staged barriers (query halves): the softmax warps can stage block
  // n + 2 only after the copy warp has released the slot from block n, so a
  // barrier is never two phases ahead of the copy warp's parity wait.  (One
  // pair for all blocks could be, when the copy warp falls a block behind,
  // and its wait would then be for a phase that needs the copy warp itself.)
  auto staged_bar = [&](int slot, int half) -> uint32_t {
    return slot == 0 ? bar(kBarStaged + half) : sb + kOffStaged1 + 8 * half;
  };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
  auto wt = [&](uint32_t br, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(br, parity, p.wait.limit_ns)) return true;
    *abort_flag = 1;
    report_timeout(p.wait.err, kSiteKv, (br - sb - kOffBar) / 8);
    return false;
  };
  // Whole-warp form: lane 0's outcome for every lane, so that a warp never
  // splits in front of a warp-collective tcgen05 instruction.
  auto wtw = [&](uint32_t br, uint32_t parity) -> bool { return __shfl_sync(0xffffffffu, wt(br, parity), 0); };

  if (tid == 0) {
    mbar_init(bar(kBarKV), 1);   // K landed
    mbar_init(bar(kBarV), 1);    // V landed
    for (int s = 0; s < kQStagesKv; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
    }
    for (int s = 0; s < kDOStages; ++s) {
      mbar_init(bar(kBarDOFull + s), 1);
      mbar_init(bar(kBarDOEmpty + s), 1);   // the block's dS copy has read the slot
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarDPFull), 1);
    mbar_init(bar(kBarPFull), 256);    // every softmax thread has put its P row into TMEM
    mbar_init(bar(kBarDSFull), 256);   // ... and its dS row
    mbar_init(bar(kBarDVDone), 1);     // dV(n) has read dO(n) for the last time
    for (int s = 0; s < 2; ++s)
      mbar_init(bar(kBarStaged + s), 128);   // slot 0: every thread of query half s has staged its dS row
    for (int s = 0; s < 2; ++s) mbar_init(sb + kOffStaged1 + 8 * s, 128);   // ... slot 1
    mbar_init(bar(kBarRope), 1);       // the key block's RoPE rows landed
    mbar_init(bar(kBarDVFinal), 1);    // the last dV product has completed
    mbar_init(bar(kBarDKV), 1);
    mbar_init(bar(kBarFinal), 1);
    *abort_flag = 0;
    fence_barrier_init();
    // This thread is the producer: K, Q(0) with its lse, then V and dO(0)
    // with its delta go out before the TMEM allocation and the block barrier.  The
    // first S product waits for 64 KB rather than for every block's 128 KB.
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmQ);
    mbar_arrive_expect_tx(bar(kBarKV), 2 * 16384);
    for (int hx = 0; hx < 2; ++hx) tma_load_4d(sb + kOffK + hx * 16384, &tmK, hx * 64, kvh, k0, b, bar(kBarKV));
    mbar_arrive_expect_tx(bar(kBarQFull), 2 * kHalfQ + 512);
    for (int hx = 0; hx < 2; ++hx)
      tma_load_4d(sb + kOffQ + hx * kHalfQ, &tmQ, hx * 64, h_first, kb * kKvBQ, b, bar(kBarQFull));
    const size_t ro = (static_cast<size_t>(b) * p.Hq + h_first) * p.Tp + kb * kKvBQ;
    bulk_load(sb + kOffLse, p.ws.lse2 + ro, 512, bar(kBarQFull));
    prefetch_tensormap(&tmV);
    mbar_arrive_expect_tx(bar(kBarV), 2 * 16384);
    for (int hx = 0; hx < 2; ++hx) tma_load_4d(sb + kOffV + hx * 16384, &tmV, hx * 64, kvh, k0, b, bar(kBarV));
    prefetch_tensormap(&tmDO);
    mbar_arrive_expect_tx(bar(kBarDOFull), 2 * kHalfQ + 512);
    for (int hx = 0; hx < 2; ++hx)
      tma_load_4d(sb + kOffDO + hx * kHalfQ, &tmDO, hx * 64, h_first, kb * kKvBQ, b, bar(kBarDOFull));
    bulk_load(sb + kOffDelta, p.ws.delta + ro, 512, bar(kBarDOFull));
  }
  if (warp == 2) tc::tmem_alloc(sb + kOffTmemSlot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kOffTmemSlot);

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      // K, Q(0), V and dO(0) are already on their way (issued with the barriers)
      const bool v_issued = true;
      int q_issued = 1, d_issued = 1;
      for (int n = 0; n < N; ++n) {
        const int h = h_first + n / nq;
        const int q0 = (kb + n % nq) * kKvBQ;
        const int qs = n % kQStagesKv, ds = n % kDOStages;
        const size_t ro = (static_cast<size_t>(b) * p.Hq + h) * p.Tp + q0;
        if (n > 0) {
          if (!wt(bar(kBarQEmpty + qs), ((n / kQStagesKv) & 1) ^ 1)) break;
          mbar_arrive_expect_tx(bar(kBarQFull + qs), 2 * kHalfQ + 512);
          for (int hx = 0; hx < 2; ++hx)
            tma_load_4d(sb + kOffQ + qs * kBlockBytes + hx * kHalfQ, &tmQ, hx * 64, h, q0, b, bar(kBarQFull + qs));
          bulk_load(sb + kOffLse + qs * 512, p.ws.lse2 + ro, 512, bar(kBarQFull + qs));
          q_issued = n + 1;
        }
        if (n > 0) {
          if (!wt(bar(kBarDOEmpty + ds), ((n / kDOStages) & 1) ^ 1)) break;
          mbar_arrive_expect_tx(bar(kBarDOFull + ds), 2 * kHalfQ + 512);
          for (int hx = 0; hx < 2; ++hx)
            tma_load_4d(sb + kOffDO + ds * kBlockBytes + hx * kHalfQ, &tmDO, hx * 64, h, q0, b, bar(kBarDOFull + ds));
          bulk_load(sb + kOffDelta + ds * 512, p.ws.delta + ro, 512, bar(kBarDOFull + ds));
          d_issued = n + 1;
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        for (int n = (q_issued > kQStagesKv ? q_issued - kQStagesKv : 0); n < q_issued; ++n)
          mbar_wait_bounded(bar(kBarQFull + n % kQStagesKv), (n / kQStagesKv) & 1, 2000000000ull);
        for (int n = (d_issued > kDOStages ? d_issued - kDOStages : 0); n < d_issued; ++n)
          mbar_wait_bounded(bar(kBarDOFull + n % kDOStages), (n / kDOStages) & 1, 2000000000ull);
        mbar_wait_bounded(bar(kBarKV), 0, 2000000000ull);
        if (v_issued) mbar_wait_bounded(bar(kBarV), 0, 2000000000ull);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    // The whole warp runs this loop in step (so descriptors and addresses stay
    // warp-uniform); one elected lane issues each MMA and commit.  Per query
    // block n the products go out in the order
    //   S(n) dP(n) | P(n) ready: dV(n) S(n+1) | dS(n) ready: dK(n) dP(n+1)
    // so that the softmax warps turn S(n) into P(n) while dP(n) runs, and
    // dP(n) into dS(n) while dV(n) and S(n+1) run.  S(n+1) overwrites the
    // P(n) columns dV(n) reads, and dP(n+1) the dS(n) columns dK(n) reads:
    // tcgen05 MMAs of one thread run in issue order, so each reads its
    // operand before the next product writes there.
    {
      constexpr uint32_t id_sdp = tc::idesc_bf16_f32(128, 128, 0, 0);   // S^T, dP^T
      constexpr uint32_t id_kv = tc::idesc_bf16_f32(128, 128, 0, 1);    // dV, dK (A from TMEM)
      // Descriptors are built once; moving by a byte offset inside shared
      // memory adds offset / 16 to the address field (all offsets stay below
      // 256 KB, so the 14-bit field never carries).
      const uint64_t dK = tc::sdesc_sw128(sb + kOffK, 16, 1024), dV = tc::sdesc_sw128(sb + kOffV, 16, 1024);
      const uint64_t dQk = tc::sdesc_sw128(sb + kOffQ, 16, 1024);          // Q as K-major B of S^T
      const uint64_t dOk = tc::sdesc_sw128(sb + kOffDO, 16, 1024);         // dO as K-major B of dP^T
      const uint64_t dQm = tc::sdesc_sw128(sb + kOffQ, kHalfQ, 1024);      // Q as MN-major B of dK
      const uint64_t dOm = tc::sdesc_sw128(sb + kOffDO, kHalfQ, 1024);     // dO as MN-major B of dV
      bool ok = wtw(bar(kBarKV), 0);   // K (V is waited for before the first dP product)
      tc::fence_after_sync();
      auto qoff = [](int n) -> uint64_t { return static_cast<uint64_t>((n % kQStagesKv) * kBlockBytes) >> 4; };
      auto dooff = [](int n) -> uint64_t { return static_cast<uint64_t>((n % kDOStages) * kBlockBytes) >> 4; };
      // K-step kk (16 of the 128 head dims): half kk / 4, 32 bytes per step inside it
      auto kstep = [](int kk, int half) -> uint32_t { return static_cast<uint32_t>((kk >> 2) * half + (kk & 3) * 32) >> 4; };
      // With saved probabilities there is no S product: the S signal then
      // only says that the P columns are free again (every product issued
      // so far, dV(n - 1) included, has completed).
      constexpr bool saved_p = kSavedP;
      auto issue_s = [&](int n) -> bool {
        if (!wtw(bar(kBarQFull + n % kQStagesKv), (n / kQStagesKv) & 1)) return false;
        tc::fence_after_sync();
        if constexpr (!saved_p) {
          const uint64_t so = qoff(n);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_bf16_w(tmem + kColS, dK + kstep(kk, 16384), dQk + so + kstep(kk, kHalfQ), id_sdp, kk > 0);
        }
        tc::commit_w(bar(kBarSFull));
        return true;
      };
      auto issue_dp = [&](int n) -> bool {
        if (!wtw(bar(kBarDOFull + n % kDOStages), (n / kDOStages) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t so = dooff(n);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_bf16_w(tmem + kColDP, dV + kstep(kk, 16384), dOk + so + kstep(kk, kHalfQ), id_sdp, kk > 0);
        tc::commit_w(bar(kBarDPFull));
        return true;
      };
      if (ok && N > 0) ok = issue_s(0) && wtw(bar(kBarV), 0) && issue_dp(0);
      // P^T / dS^T of query chunk c (16 queries) sit in the 8 TMEM columns
      // 32 (c / 2) + 8 (c % 2) of the S (P) and dP (dS) columns.
      for (int n = 0; ok && n < N; ++n) {
        if (!wtw(bar(kBarPFull), n & 1)) break;
        tc::fence_after_sync();
        const uint64_t dso = dooff(n), qso = qoff(n);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // dV += P^T dO
          tc::mma_bf16_ts_w(tmem + kColDV, tmem + kColS + (kk >> 1) * 32 + (kk & 1) * 8, dOm + dso + ((kk * 2048) >> 4),
                            id_kv, (n > 0 || kk > 0));
        tc::commit_w(bar(kBarDVDone));   // dO(n) has been read for the last time
        if (n == N - 1) tc::commit_w(bar(kBarDVFinal));
        if (n + 1 < N && !issue_s(n + 1)) break;
        if (!wtw(bar(kBarDSFull), n & 1)) break;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // dK += dS^T Q
          tc::mma_bf16_ts_w(tmem + kColDK, tmem + kColDP + (kk >> 1) * 32 + (kk & 1) * 8, dQm + qso + ((kk * 2048) >> 4),
                            id_kv, (n > 0 || kk > 0));
        tc::commit_w(bar(kBarQEmpty + n % kQStagesKv));   // and Q(n)
        if (n + 1 < N && !issue_dp(n + 1)) break;
      }
      tc::commit_w(bar(kBarDKV));
      tc::commit_w(bar(kBarFinal));   // waited for after the epilogue
    }
  } else if (warp == 3) {
    // ============================ dS copy warp ============================
    // Block n's two dS^T tiles (one per query half, adjacent in the
    // workspace) are copied from the dO(n) slot by two 16 KB bulk copies.
    // Waiting for the copies to read the slot (they queue behind the ring's
    // loads) happens here, not in the softmax warps.
    if (lane == 0) {
      for (int n = 0; n < N; ++n) {
        const int h = h_first + n / nq, qb = kb + n % nq;
        __nv_bfloat16 *dst =
            p.ws.ds + ((static_cast<size_t>(b) * p.Hq + h) * p.tph + tile_index(kb, 2 * qb, p.nqb)) * (kTileBytes / 2);
        // each query half's tile goes out as soon as its four warps staged it
        bool staged = true;
        for (int hf = 0; hf < 2 && staged; ++hf) {
          staged = wt(staged_bar(n % kDOStages, hf), (n / kDOStages) & 1);
          if (staged) bulk_store(dst + hf * (kTileBytes / 2), sb + kOffDO + (n % kDOStages) * kBlockBytes + hf * kTileBytes,
                                 kTileBytes);
        }
        bulk_commit_group();
        if (!staged) break;
        bulk_wait_group_read0();
        mbar_arrive(bar(kBarDOEmpty + n % kDOStages));
      }
      bulk_wait_group0();
    }
    // the softmax warps stage dK in the dO ring once the last copy has read it
    named_barrier(3, 288);
  } else if (warp >= 4) {
    // ============================ softmax warps ===========================
    // Warp w covers the 32-key TMEM lane quarter w % 4 and half g of the 128
    // queries of every block (64 queries: S / dP columns 64 g .. 64 g + 63).
    // Per block: wait for S, form P (kept in fp32 registers), write it back
    // as bf16 over the S values just read, arrive; then wait for dP, form
    // dS = P (dP - delta), write it over dP and to the workspace, arrive.
    const int qd = warp & 3;                            // TMEM lane quarter
    const int ch = (warp - 4) >> 2;                     // query half (then dK / dV epilogue half)
    const int j = 32 * qd + lane;                       // key row in the block
    const int key = k0 + j;
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;
    const uint32_t tS = tmem + lanebase + kColS + 64 * ch;
    const uint32_t tD = tmem + lanebase + kColDP + 64 * ch;
    bool rope_issued = false;
    int blocks_done = 0;
    for (int n = 0; n < N; ++n) {
      const int h = h_first + n / nq;
      const int qb = kb + n % nq;                       // 128-query block
      const int q0 = qb * kKvBQ + 64 * ch;              // this half's first query
      // lse * log2 e and delta of this half's 64 queries: lse arrived with
      // Q(n), which S(n) waited for (with saved probabilities too), delta
      // with dO(n), which dP(n) waited for
      const float *lse2 = reinterpret_cast<const float *>(smem + kOffLse + (n % kQStagesKv) * 512) + 64 * ch;
      const float *dl = reinterpret_cast<const float *>(smem + kOffDelta + (n % kDOStages) * 512) + 64 * ch;
      // only the diagonal block needs the causal mask; queries past T have
      // lse = +inf, so their P is exactly 0
      const bool diag = qb == kb;
      float P[64];
      uint32_t pk[32];
      if constexpr (kSavedP) {
        // ---- P from the saved probabilities: this thread's key column of
        // the 64 query rows, read before the P columns are free
        const __nv_bfloat16 *pc = p.pattn + (static_cast<size_t>(b) * p.Hq + h) * p.T * p.T + key;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int q = q0 + e;
          P[e] = (q < p.T && key <= q) ? __bfloat162float(pc[static_cast<size_t>(q) * p.T]) : 0.f;
        }
        if (!wtw(bar(kBarSFull), n & 1)) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < 64; e += 2) pk[e / 2] = pack_bf16x2(P[e], P[e + 1]);
      } else {
      // ---- P = 2^(S scale log2 e - lse log2 e)
      if (!wtw(bar(kBarSFull), n & 1)) break;
      tc::fence_after_sync();
      {
        float (&lo)[32] = *reinterpret_cast<float (*)[32]>(&P[0]);
        float (&hi)[32] = *reinterpret_cast<float (*)[32]>(&P[32]);
        tc::ld32x2_wait(tS, tS + 32, lo, hi);
      }
      // two copies of the loop, so that the common, unmasked one is straight-line code
      auto p_loop = [&](const bool masked) {
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + e);
          P[e] = fast_exp2(fmaf(P[e], sl2, -l4.x));
          P[e + 1] = fast_exp2(fmaf(P[e + 1], sl2, -l4.y));
          P[e + 2] = fast_exp2(fmaf(P[e + 2], sl2, -l4.z));
          P[e + 3] = fast_exp2(fmaf(P[e + 3], sl2, -l4.w));
          if (masked) {
            const int q = q0 + e;
            P[e] = key <= q ? P[e] : 0.f;
            P[e + 1] = key <= q + 1 ? P[e + 1] : 0.f;
            P[e + 2] = key <= q + 2 ? P[e + 2] : 0.f;
            P[e + 3] = key <= q + 3 ? P[e + 3] : 0.f;
          }
          pk[e / 2] = pack_bf16x2(P[e], P[e + 1]);
          pk[e / 2 + 1] = pack_bf16x2(P[e + 2], P[e + 3]);
        }
      };
      if (diag)
        p_loop(true);
      else
        p_loop(false);
      }
      // chunk c (16 queries = 8 packed columns) goes to column 32 (c / 2) +
      // 8 (c % 2) of this half: the A-operand layout of the dV product
      {
        const uint32_t (&c0)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&pk[0]);
        const uint32_t (&c1)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&pk[8]);
        const uint32_t (&c2)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&pk[16]);
        const uint32_t (&c3)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&pk[24]);
        tc::st8x2_async(tS, c0, tS + 8, c1);
        tc::st8x2_async(tS + 32, c2, tS + 40, c3);
      }
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(kBarPFull));
      // ---- dS = P (dP - delta), to TMEM (A operand of dK) and to the workspace
      if (!wtw(bar(kBarDPFull), n & 1)) break;
      tc::fence_after_sync();
      uint4 U[8];   // this key row's dS^T as eight 16-byte units of 8 queries
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float d[32];
        tc::ld32_wait(tD + 32 * half, d);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dl + 32 * half + e);
          const float s0 = P[32 * half + e] * (d[e] - d4.x);
          const float s1 = P[32 * half + e + 1] * (d[e + 1] - d4.y);
          const float s2 = P[32 * half + e + 2] * (d[e + 2] - d4.z);
          const float s3 = P[32 * half + e + 3] * (d[e + 3] - d4.w);
          dk[e / 2] = pack_bf16x2(s0, s1);
          dk[e / 2 + 1] = pack_bf16x2(s2, s3);
        }
        {
          const uint32_t (&c0)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&dk[0]);
          const uint32_t (&c1)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&dk[8]);
          tc::st8x2_async(tD + 32 * half, c0, tD + 32 * half + 8, c1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) U[4 * half + u] = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
      }
      // dS is in TMEM: the dK product (and after it dP(n + 1)) may start
      // while the workspace copy below is still being written
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(kBarDSFull));
      // Once dV(n) has read dO(n) for the last time, its ring slot stages
      // the block's two dS^T tiles (32 KB in the tiles' own 128B-swizzled
      // layout: unit u of row r at 16 (u ^ (r % 8))); the copy warp moves
      // them to the workspace and hands the slot back to the producer.
      if (!wtw(bar(kBarDVDone), n & 1)) break;
      tc::fence_after_sync();
      {
        const uint32_t stg = kOffDO + (n % kDOStages) * kBlockBytes + ch * 16384 + qd * 4096 + lane * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4 *>(smem + stg + ((u ^ (lane & 7)) << 4)) = U[u];
        fence_proxy_async_smem();
        mbar_arrive(staged_bar(n % kDOStages, ch));
      }
      blocks_done = n + 1;
    }
    if (blocks_done == N && p.rope && warp == 4 && lane == 0) {
      // dP(N - 1) has completed, so have dK(N - 2) and dK(N - 3): the two Q
      // slots other than Q(N - 1)'s are free.  They take this key block's
      // RoPE rows for the dK epilogue (keys 0-63, then 64-127).
      const int rows = min(kBK, p.T - k0);
      mbar_arrive_expect_tx(bar(kBarRope), rows * 512);
      bulk_load(sb + kOffQ + (N % kQStagesKv) * kBlockBytes, p.ws.rope + k0 * (kD / 2), min(rows, 64) * 512,
                bar(kBarRope));
      if (rows > 64)
        bulk_load(sb + kOffQ + ((N + 1) % kQStagesKv) * kBlockBytes, p.ws.rope + (k0 + 64) * (kD / 2),
                  (rows - 64) * 512, bar(kBarRope));
      rope_issued = true;
    }
    // ---- dK (scale + RoPE backward) and dV epilogues.  Group ch takes the
    // 32-column chunks 2 ch and 2 ch + 1 of both, staged as 128B-swizzled
    // [128 rows][32] fp32 tiles and written by TMA tensor stores (rows past T
    // are not written; with the head group split over CTAs the partial sums
    // are added into the zeroed outputs).  dV first, as soon as the last dV
    // product has completed, into the K / V region (no product reads it
    // after the last S and dP); then dK after the last dK product, into the
    // dO ring once the copy warp has seen its last workspace copy read, with
    // the RoPE rows from the two Q slots filled above.  All 256 threads agree
    // on each outcome at their named barriers.
    bool eok = wtw(bar(kBarDVFinal), 0);
    if (eok) {
      tc::fence_after_sync();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * ch + cc;
        float u[32];
        tc::ld32_wait(tmem + lanebase + kColDV + 32 * c, u);
        unsigned char *vrow = smem + kOffK + c * 16384 + j * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4 *>(vrow + ((i ^ (j & 7)) << 4)) =
              make_float4(u[4 * i], u[4 * i + 1], u[4 * i + 2], u[4 * i + 3]);
      }
    }
    fence_proxy_async_smem();
    eok = named_barrier_and(4, 256, eok);
    if (eok && warp == 4 && lane == 0) {
      for (int c = 0; c < 4; ++c) {
        if (split_group)
          tma_reduce_add_4d(&tmdV, sb + kOffK + c * 16384, 32 * c, kvh, k0, b);
        else
          tma_store_4d(&tmdV, sb + kOffK + c * 16384, 32 * c, kvh, k0, b);
      }
      bulk_commit_group();
    }
    bool kok = eok && wtw(bar(kBarDKV), 0);
    if (p.rope) kok = kok && wtw(bar(kBarRope), 0);
    named_barrier(3, 288);
    if (kok) {
      tc::fence_after_sync();
      const unsigned char *rrow =
          smem + kOffQ + ((j < 64 ? N : N + 1) % kQStagesKv) * kBlockBytes + (j & 63) * 512;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * ch + cc;
        float v[32];
        tc::ld32_wait(tmem + lanebase + kColDK + 32 * c, v);
        unsigned char *krow = smem + kOffDO + c * 16384 + j * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // pairs (4i, 4i+1), (4i+2, 4i+3); the table holds scale * (cos, sin)
          const float4 t = (p.rope && key < p.T)
                               ? *reinterpret_cast<const float4 *>(rrow + ((8 * c + (i ^ (j & 7))) << 4))
                               : make_float4(p.scale, 0.f, p.scale, 0.f);
          const float *x = v + 4 * i;
          *reinterpret_cast<float4 *>(krow + ((i ^ (j & 7)) << 4)) =
              make_float4(x[0] * t.x + x[1] * t.y, -x[0] * t.y + x[1] * t.x, x[2] * t.z + x[3] * t.w,
                          -x[2] * t.w + x[3] * t.z);
        }
      }
    }
    fence_proxy_async_smem();
    kok = named_barrier_and(4, 256, kok);
    if (warp == 4 && lane == 0) {
      if (kok) {
        for (int c = 0; c < 4; ++c) {
          if (split_group)
            tma_reduce_add_4d(&tmdK, sb + kOffDO + c * 16384, 32 * c, kvh, k0, b);
          else
            tma_store_4d(&tmdK, sb + kOffDO + c * 16384, 32 * c, kvh, k0, b);
        }
        bulk_commit_group();
      }
      bulk_wait_group_read0();   // shared memory may be released; the writes complete on their own
    }
    // a RoPE copy still in flight (after a timeout) lands before the CTA exits
    if (rope_issued) mbar_wait_bounded(bar(kBarRope), 0, 2000000000ull);
  }
  if (warp == 1) mbar_wait_bounded(bar(kBarFinal), 0, 2000000000ull);   // every MMA has completed
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

  // Persistent: work items are (query block pair m, head, batch), heaviest
  // (largest m) first, dealt to the CTAs in alternating-direction rounds.  Item j of a CTA
  // accumulates into TMEM buffer j & 1, so its epilogue overlaps the loads
  // and products of item j + 1.
  const int per_m = p.Hq * p.B;
  const int items = p.nkb * per_m;
  struct Item { int m, h, b; };
  auto item = [&](int it) -> Item {
    Item r;
    r.m = p.nkb - 1 - it / per_m;
    const int rem = it % per_m;
    r.h = rem % p.Hq;
    r.b = rem / p.Hq;
    return r;
  };

  // The r-th item of this CTA: rounds over the CTAs alternate direction, so
  // the heaviest-first item list spreads evenly (a plain round-robin leaves
  // the busiest CTA 12 % above the mean at T = 2048, this within 1 %).
  auto nth = [&](int r) -> int {
    const int c = (r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
    return r * static_cast<int>(gridDim.x) + c;
  };

  auto bar = [&](int i) -> uint32_t { return sb + kQOffBar + i * 8; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kQOffAbort);
  auto wt = [&](uint32_t br, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(br, parity, p.wait.limit_ns)) return true;
    *abort_flag = 1;
    report_timeout(p.wait.err, kSiteDq, (br - sb - kQOffBar) / 8);
    return false;
  };
  // Whole-warp form: lane 0's outcome for every lane, so that a warp never
  // splits in front of a warp-collective tcgen05 instruction.
  auto wtw = [&](uint32_t br, uint32_t parity) -> bool { return __shfl_sync(0xffffffffu, wt(br, parity), 0); };

  if (tid == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bar(kQBarFull + s), 1);
      mbar_init(bar(kQBarEmpty + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(kQBarAccFull + a), 1);
      mbar_init(bar(kQBarAccEmpty + a), 256);
    }
    mbar_init(bar(kQBarFinal), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) tc::tmem_alloc(sb + kQOffTmemSlot, 256);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kQOffTmemSlot);

  if (warp == 0) {
    // ============================ producer ================================
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      const uint64_t keep = l2_evict_last(), stream = l2_evict_first();
      // the dS tiles come from the kv kernel: wait for that grid to have
      // completed (a no-op when this grid was launched after it completed)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int g = 0;   // steps issued so far (ring position)
      bool ok = true;
      for (int r = 0, it = nth(0); ok && it < items; it = nth(++r)) {
        const Item w = item(it);
        const int kvh = w.h / p.G;
        const __nv_bfloat16 *tiles = p.ws.ds + (static_cast<size_t>(w.b) * p.Hq + w.h) * p.tph * (kTileBytes / 2);
        for (int i = 0; i <= w.m; ++i, ++g) {
          const int s = g % kQStages, cyc = g / kQStages;
          if (!wt(bar(kQBarEmpty + s), (cyc & 1) ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t st = sb + s * kQStageBytes;
          const uint32_t fb = bar(kQBarFull + s);
          mbar_arrive_expect_tx(fb, 2 * 16384 + 2 * kTileBytes);
          for (int hx = 0; hx < 2; ++hx)
            tma_load_4d_hint(st + hx * 16384, &tmK, hx * 64, kvh, i * kBK, w.b, fb, keep);
          // tiles (i, 2m) and (i, 2m + 1) are adjacent; each is read once
          bulk_load_hint(st + kQOffDS, tiles + tile_index(i, 2 * w.m, p.nqb) * (kTileBytes / 2), 2 * kTileBytes,
                         fb, stream);
        }
      }
      if (!ok) {
        // let copies already in flight land before the CTA can exit
        for (int i = (g > kQStages ? g - kQStages : 0); i < g; ++i)
          mbar_wait_bounded(bar(kQBarFull + i % kQStages), (i / kQStages) & 1, 2000000000ull);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    // whole warp in step, one elected lane issues
    {
      constexpr uint32_t id_dq = tc::idesc_bf16_f32(128, 128, 1, 1);    // dQ^T += K^T dS^T
      // built once; a byte offset inside shared memory adds offset / 16
      const uint64_t dKt = tc::sdesc_sw128(sb, 16384, 1024);                  // K^T, MN-major A
      const uint64_t dSt = tc::sdesc_sw128(sb + kQOffDS, kTileBytes, 1024);   // dS^T, MN-major B
      int g = 0, j = 0;
      bool ok = true;
      for (int r = 0, it = nth(0); ok && it < items; it = nth(++r), ++j) {
        const Item w = item(it);
        const int a = j & 1;
        if (!wtw(bar(kQBarAccEmpty + a), ((j >> 1) & 1) ^ 1)) break;
        tc::fence_after_sync();
        for (int i = 0; i <= w.m; ++i, ++g) {
          const int s = g % kQStages, cyc = g / kQStages;
          if (!wtw(bar(kQBarFull + s), cyc & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t so = static_cast<uint64_t>(s * kQStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_bf16_w(tmem + a * 128, dKt + so + ((kk * 2048) >> 4), dSt + so + ((kk * 2048) >> 4), id_dq,
                         (i > 0 || kk > 0));
          tc::commit_w(bar(kQBarEmpty + s));
        }
        if (ok) tc::commit_w(bar(kQBarAccFull + a));
      }
      tc::commit_w(bar(kQBarFinal));
      mbar_wait_bounded(bar(kQBarFinal), 0, 2000000000ull);   // every MMA has completed
    }
  } else if (warp >= 4) {
    // ============================ epilogue ================================
    const int qd = warp & 3;                 // TMEM lane quarter = 32 head-dim rows
    const int ch = (warp - 4) >> 2;          // 64-query half
    const int d = 32 * qd + lane;
    const uint32_t lanebase = static_cast<uint32_t>(32 * qd) << 16;
    const bool odd = d & 1;
    const size_t qstride = static_cast<size_t>(p.Hq) * kD;
    // RoPE: the table holds scale * e^{i (pos0 + t) theta} for pair d / 2;
    // consecutive positions differ by the rotation e^{i theta}, taken once
    // from the first two rows.  A chunk reads the table at every 8th query
    // and rotates in between (7 complex products add ~1e-5 relative error),
    // so the epilogue waits for 4 table reads instead of 32.
    float2 stp = make_float2(1.f, 0.f);
    if (p.rope && p.T >= 2) {
      const float2 t0 = p.ws.rope[rope_slot(0, d >> 1)], t1 = p.ws.rope[rope_slot(1, d >> 1)];
      const float is2 = 1.f / (p.scale * p.scale);
      stp = make_float2((t1.x * t0.x + t1.y * t0.y) * is2, (t1.y * t0.x - t1.x * t0.y) * is2);
    }
    int j = 0;
    for (int r = 0, it = nth(0); it < items; it = nth(++r), ++j) {
      const Item w = item(it);
      const int a = j & 1;
      if (!wtw(bar(kQBarAccFull + a), (j >> 1) & 1)) break;
      tc::fence_after_sync();
      float v[2][32];
      tc::ld32x2_wait(tmem + lanebase + a * 128 + 64 * ch, tmem + lanebase + a * 128 + 64 * ch + 32, v[0], v[1]);
      tc::fence_before_sync();
      mbar_arrive(bar(kQBarAccEmpty + a));   // the accumulator may be reused
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int qbase = w.m * kBK + 64 * ch + 32 * cc;
        // pair (2i, 2i+1) rotated by -theta; the factors are scale * (cos,
        // sin).  The table reads come before the first store: a load after
        // a store to possibly the same memory would wait for it.
        float2 cs[32];
        if (!p.rope) {
#pragma unroll
          for (int c = 0; c < 32; ++c) cs[c] = make_float2(p.scale, 0.f);
        } else {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int q = qbase + 8 * g8;
            cs[8 * g8] = q < p.T ? p.ws.rope[rope_slot(q, d >> 1)] : make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8)
#pragma unroll
            for (int c = 8 * g8 + 1; c < 8 * g8 + 8; ++c)
              cs[c] = make_float2(cs[c - 1].x * stp.x - cs[c - 1].y * stp.y, cs[c - 1].x * stp.y + cs[c - 1].y * stp.x);
        }
        float *dst = p.dq + ((static_cast<size_t>(w.b) * p.T + qbase) * p.Hq + w.h) * kD + d;
        // the bound is tested once per chunk: only the last chunk can pass T
        auto store = [&](const bool bounded) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float x = v[cc][c];
            const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
            if (!bounded || qbase + c < p.T) dst[c * qstride] = x * cs[c].x + (odd ? -partner : partner) * cs[c].y;
          }
        };
        if (qbase + 32 <= p.T)
          store(false);
        else
          store(true);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 256);
  }
}

bool make_map(CUtensorMap *m, const void *base, int H, int T, int B, uint32_t rows, const char **why) {
  const uint64_t dims[4] = {kD, static_cast<uint64_t>(H), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {kD * 2, static_cast<uint64_t>(H) * kD * 2, static_cast<uint64_t>(T) * H * kD * 2};
  const uint32_t box[4] = {64, 1, rows, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, why);
}

// fp32 [B][T][H][128] tensor stored in [128 rows][32 floats] 128B-swizzled tiles.
bool make_map_f32(CUtensorMap *m, void *base, int H, int T, int B, const char **why) {
  const uint64_t dims[4] = {kD, static_cast<uint64_t>(H), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {kD * 4, static_cast<uint64_t>(H) * kD * 4, static_cast<uint64_t>(T) * H * kD * 4};
  const uint32_t box[4] = {32, 1, static_cast<uint32_t>(kBK), 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                      why);
}

// Scratch for attn_bwd_causal_noalloc: a fixed device array the library
// owns, so that entry point never allocates.  Every GPU that loads the
// library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace

cudaError_t noalloc_scratch(void **ptr, const char **why) {
  // Resolved once per device and context, with that device current.  A
  // symbol's name in host code is only a host-side stand-in; the device
  // address must come from the runtime.  The context id in the key makes a
  // context created after cudaDeviceReset resolve the address again.
  static std::mutex mu;
  static void *addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) {
    *why = "device ordinal out of range";
    return cudaErrorInvalidDevice;
  }
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx_of[dev] != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *why = "cudaGetSymbolAddress of the built-in scratch failed";
      return e;
    }
    addr[dev] = p;
    ctx_of[dev] = ctx;
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

cudaError_t launch_attn_bwd_causal(const void *q, const void *k, const void *v, const void *pattn, const void *o,
                                   const void *dout, const float *lse, float *dq, float *dk, float *dv, int B, int T,
                                   int Hq, int Hkv, int D, float scale, double rope_base, int pos0, void *ws,
                                   size_t ws_bytes, const WaitCtl &w, cudaStream_t st, const char **why) {
  (void)ws_bytes;
  if (D != kD) {
    *why = "D != 128";
    return cudaErrorNotSupported;
  }
  const int Tp = padded_T(T);
  const int nkb = Tp / kBK;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // Split each KV head's query heads over more CTAs while the grid would not
  // fill the GPU (partial dK / dV are then added into zeroed outputs).
  const int G = Hq / Hkv;
  int hsplit = 1;
  while (hsplit < G && G % (2 * hsplit) == 0 && static_cast<long long>(nkb) * Hkv * B * hsplit < sms) hsplit *= 2;
  long long kv_ctas = static_cast<long long>(nkb) * Hkv * B * hsplit;
  // When the group is split (the grid would not fill the GPU otherwise),
  // choose the split per key block: key block kb gives each head nkb - kb
  // query blocks, so it takes the largest share of the group (a divisor of
  // G) whose blocks stay within nkb, the count of the heaviest key block
  // with one head per CTA.  Every CTA then holds at most nkb blocks and the
  // light key blocks use fewer CTAs: fewer CTAs and no second partial wave.
  int nsplit[kMaxVarKb] = {}, kb_first[kMaxVarKb + 1] = {};
  const bool var_split = hsplit > 1 && nkb <= kMaxVarKb;
  if (var_split) {
    kv_ctas = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      int share = 1;   // heads per CTA
      for (int d = 1; d <= G; ++d)
        if (G % d == 0 && d * (nkb - kb) <= nkb) share = d;
      nsplit[kb] = G / share;
      kb_first[kb] = static_cast<int>(kv_ctas);
      kv_ctas += static_cast<long long>(B) * Hkv * nsplit[kb];
    }
    kb_first[nkb] = static_cast<int>(kv_ctas);
  }
  const long long dq_ctas = static_cast<long long>(nkb) * Hq * B;
  if (kv_ctas > 0x7fffffffLL || dq_ctas > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorNotSupported;
  }
  CausalWs cw = carve(ws, B, T, Hq, D);
  const int rope = rope_base > 0.0;
  PrepRope rp;
  rp.zero_dk = dk;
  rp.zero_dv = dv;
  rp.zero_n4 = hsplit > 1 ? static_cast<long long>(B) * T * Hkv * kD / 4 : 0;
  for (int i = 0; i < kD / 2; ++i) rp.inv_freq[i] = rope ? pow(rope_base, -2.0 * i / kD) : 0.0;
  rp.scale = scale;
  rp.use_rope = rope;
  rp.pos0 = pos0;
  {
    const long long rows = static_cast<long long>(B) * T * Hq;
    const long long threads = std::max((rows + kPrepRows - 1) / kPrepRows * 16,
                                       static_cast<long long>(B) * Hq * (Tp - T));
    const long long blocks = (threads + 255) / 256;
    causal_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse, cw.delta, cw.lse2,
        cw.rope, B, T, Tp, Hq, rp);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tdo, tk, tv, tdk, tdv;
  if (!make_map(&tq, q, Hq, T, B, kKvBQ, why) || !make_map(&tdo, dout, Hq, T, B, kKvBQ, why) ||
      !make_map(&tk, k, Hkv, T, B, kBK, why) || !make_map(&tv, v, Hkv, T, B, kBK, why) ||
      !make_map_f32(&tdk, dk, Hkv, T, B, why) || !make_map_f32(&tdv, dv, Hkv, T, B, why))
    return cudaErrorInvalidValue;
  TcParams p;
  p.ws = cw;
  p.pattn = static_cast<const __nv_bfloat16 *>(pattn);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B; p.T = T; p.Tp = Tp; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.nkb = nkb;
  p.nqb = Tp / kBQ;
  p.tph = tiles_per_head(nkb);
  p.hsplit = hsplit;
  p.gs = G / hsplit;
  p.var_split = var_split;
  for (int kb = 0; kb < kMaxVarKb; ++kb) p.nsplit[kb] = nsplit[kb];
  for (int kb = 0; kb <= kMaxVarKb; ++kb) p.kb_first[kb] = kb_first[kb];
  p.scale = scale;
  p.rope = rope;
  p.wait = w;
  auto kv_kernel = pattn ? causal_kv_tc_kernel<true> : causal_kv_tc_kernel<false>;
  e = ensure_dynamic_smem(reinterpret_cast<const void *>(kv_kernel), kSmem);
  if (e != cudaSuccess) return e;
  kv_kernel<<<static_cast<unsigned>(kv_ctas), kThr, kSmem, st>>>(tq, tdo, tk, tv, tdk, tdv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = ensure_dynamic_smem(reinterpret_cast<const void *>(causal_dq_tc_kernel), kQSmem);
  if (e != cudaSuccess) return e;
  const long long dq_grid = std::min<long long>(dq_ctas, sms);
  // launched as the kv grid's programmatic dependent: its CTAs start on SMs
  // the kv grid's tail leaves idle and set up while the last kv CTAs finish
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(dq_grid));
  cfg.blockDim = dim3(kThr);
  cfg.dynamicSmemBytes = kQSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, causal_dq_tc_kernel, tk, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace abw
