// Decode-style attention backward: one query per sequence against a KV cache,
// grouped KV heads, RoPE backward fused on dq.
//
// Spec: "Hesper.Training.VerifiedBackward", section Attention (full
// single-head) -- attentionBackwardQ (dAttn = dOut V^T, softmax backward,
// dQ = scale dScores K), attentionBackwardV (dV[s] = attn[s] dOut) -- and
// section Scaled Dot-Product (dk = scale dScore q), summed over the query
// heads that share a KV head; section RoPE (ropeBackward) on dq.
//
// Design (GB300): the work is bound by HBM -- K and V are read once (bf16) and
// dK, dV are written once (fp32).  One (batch, KV head) unit is split over a
// thread-block cluster of up to 8 CTAs, each owning a contiguous chunk of
// keys; K/V tiles of 64 rows arrive by TMA.  Per key the CTA keeps two
// scalars per query head (score, dP) in shared memory.  The cluster merges the
// per-CTA softmax statistics (max, normaliser, sum e dP) through distributed
// shared memory -- the online-softmax merge Hesper's split-KV flash attention
// applies to its tile partials (pull request #1, "Phase 2: Merge partial
// results") -- and every CTA then writes its dK/dV rows straight from the
// two scalars per head with streaming 16-byte stores.
//
// Two shapes of the same kernel:
//  * resident (a CTA's chunk fits its two TMA stages -- e.g. 1024 keys over 8
//    CTAs): the K tiles stay in shared memory, so the CTA's share of dq is
//    summed with the final dS straight from them.  With
//    a bf16 head dim of 64, 128 or 256 the tiles arrive 128B-swizzled and
//    each key row is split over 4 lanes, every lane owning a quarter of the
//    head dim, with scale*q and dout broadcast from shared memory
//    (conflict-free on both operands).
//  * streaming (longer chunks): tiles cycle through the two stages and the
//    dq partials sum_j e_j dP_j K_j and sum_j e_j K_j are carried as running
//    max-rescaled sums, merged across the cluster with the statistics.
// Either way no byte of K/V is read twice and nothing goes through a global
// scratch buffer.
#include <cooperative_groups.h>
#include <math.h>

#include <type_traits>

#include "abw_host.h"
#include "tcgen05.cuh"

namespace cg = cooperative_groups;

namespace abw {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 64;       // K/V rows per TMA tile
constexpr int kStages = 2;      // TMA stages
constexpr int kMaxCluster = 8;  // portable cluster size
constexpr int kMaxG = 8;

struct DecodeParams {
  const float *q;
  const float *dout;
  float *dq;
  float *dk;
  float *dv;
  int B, Hq, Hkv, S, D, G;
  int chunk;      // keys per CTA (multiple of kTile)
  int ncl;        // CTAs per (b, kv head) == cluster size
  int resident;   // chunk <= kStages * kTile: K stays in shared memory
  int lpr_log2;   // generic dot phase: log2(lanes per K/V row), 16 bytes per lane
  int rs_log2;    // streaming: log2(row splits) of the dq partial sums
  int rowbytes;   // D * sizeof(kv)
  int tc;         // bf16, D = 128, 128 keys per CTA: score / dP products on the tensor core
  float scale;
  int rope;
  float rcos[128];
  float rsin[128];
  WaitCtl wait;
};

// Byte offsets of the dynamic shared-memory regions (same in every CTA).
// Per-key scalars are key-major with a stride of gs (the kernel's
// power-of-two head capacity), so one vector load fetches all heads of a key.
struct Layout {
  int kv, qs, sbuf, pbuf, etile, edp, xm, xl, xc, xa, xb, glob, rstat, alpha, runm, runl, runc, rsc, bars, tcs, total;
  __host__ __device__ static int up(int x, int a) { return (x + a - 1) / a * a; }
  // swz: the quarter-row layout of scale*q / dout is used; resident: the
  // streaming-only regions (running statistics, tile exponentials, dq
  // partial exchange) are left out -- every region a path uses is present.
  __host__ __device__ Layout(int G, int gs, int D, int chunk, int rowbytes, int rs, bool swz, bool resident) {
    int o = 0;
    const int tiles = 2 * kStages * kTile * rowbytes;        // [K st0][K st1][V st0][V st1]
    const int scratch = resident ? 0 : 2 * rs * G * D * 4;    // streaming: row-split dq partials
    const int ns = resident ? 0 : 1;
    kv = o;    o += tiles > scratch ? tiles : scratch;   o = up(o, 16);
    // The tensor-core path (128-key chunk, D = 128) stages its [16 rows]
    // [128] bf16 B operands at qs: first s / dP's two (8 KB, which may run on
    // into sbuf / pbuf, written only after those products complete), later
    // dq's one (4 KB, written while pbuf is read, so within qs alone).
    int qsz = swz ? 2 * gs * 4 * (D / 4 + 4) * 4 : 0;
    if (swz && D == 128 && chunk == 2 * kTile) {
      const int need = 8192 - 2 * gs * chunk * 4;
      qsz = qsz > need ? qsz : need;
      qsz = qsz > 4096 ? qsz : 4096;
    }
    qs = o;    o += qsz;
    sbuf = o;  o += gs * chunk * 4;
    pbuf = o;  o += gs * chunk * 4;
    etile = o; o += ns * gs * kTile * 4;
    edp = o;   o += ns * gs * kTile * 4;
    xm = o;    o += kMaxG * 4;
    xl = o;    o += kMaxG * 4;
    xc = o;    o += kMaxG * 4;
    xa = o;    o += ns * G * D * 4;
    xb = o;    o += ns * G * D * 4;    o = up(o, 16);
    glob = o;  o += kMaxG * 16;
    rstat = o; o += kMaxCluster * gs * 16;
    alpha = o; o += kMaxG * 4;
    runm = o;  o += kMaxG * 4;
    runl = o;  o += kMaxG * 4;
    runc = o;  o += kMaxG * 4;
    rsc = o;   o += kMaxCluster * kMaxG * 4;  o = up(o, 16);
    bars = o;  o += kStages * 8;
    tcs = o;   o += 16;                                     // tensor-core path: mbarrier, TMEM address
    total = up(o, 16);
  }
};

// 16 bytes of a K/V row as floats.
__device__ __forceinline__ void load16(const unsigned char *p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void load16(const unsigned char *p, float (&f)[4]) {
  const float4 u = *reinterpret_cast<const float4 *>(p);
  f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}

// Four consecutive row elements at p.
__device__ __forceinline__ float4 load4(const unsigned char *p, __nv_bfloat16 *) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}
__device__ __forceinline__ float4 load4(const unsigned char *p, float *) {
  return *reinterpret_cast<const float4 *>(p);
}

// Loads the N consecutive floats at p (16-byte aligned when N >= 4).
template <int N>
__device__ __forceinline__ void ld_heads(const float *p, float (&x)[N]) {
  if constexpr (N >= 4) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 v = *reinterpret_cast<const float4 *>(p + i);
      x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
    }
  } else if constexpr (N == 2) {
    const float2 v = *reinterpret_cast<const float2 *>(p);
    x[0] = v.x; x[1] = v.y;
  } else {
    x[0] = p[0];
  }
}

// Sums NV values over an aligned group of `lpr` lanes (a power of two) while
// spreading them out: each exchange step halves the values a lane keeps, so
// the group needs log2(NV) + log2(lpr / NV) shuffles per value set instead of
// NV * log2(lpr).  On return lane l holds the group sums of values
// idx0 .. idx0 + nf - 1 in v[0 .. nf).
template <int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lpr, int lane, int &idx0, int &nf) {
  int o = lpr >> 1;
  idx0 = 0;
  nf = NV;
#pragma unroll
  for (int s = 0; (NV >> s) > 1; ++s) {
    if (o == 0) break;
    const int h = NV >> (s + 1);
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < (NV >> (s + 1)); ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (up) idx0 += h;
    nf = h;
    o >>= 1;
  }
  for (; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
}

// DT > 0: resident chunk, 128B-swizzled bf16 tiles, head dim DT, quarter-row
// lanes.  DT == 0: any supported head dim, resident or streaming, unswizzled.
template <typename KV, int GMAX, int DT>
__global__ void __launch_bounds__(kThreads, GMAX >= 8 ? 1 : (DT > 0 ? 3 : 2))
    decode_bwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ DecodeParams p) {
  constexpr bool SWZ = DT > 0;
  constexpr int ES = static_cast<int>(sizeof(KV));
  constexpr int EPL = 16 / ES;                 // elements per 16-byte granule
  constexpr int NV = 2 * GMAX;                 // per-row values: s_h and dP_h
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int G = p.G;
  const int D = SWZ ? DT : p.D;
  const int rowbytes = SWZ ? DT * ES : p.rowbytes;
  const bool resident = SWZ || p.resident;
  const int RS = 1 << p.rs_log2;
  const Layout L(G, GMAX, D, p.chunk, rowbytes, RS, SWZ, resident);
  const int rank = static_cast<int>(cluster.block_rank());
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int key0 = rank * p.chunk;
  const int nkeys = min(p.chunk, p.S - key0);   // >= 1 by construction of chunk / ncl
  const int ntiles = (nkeys + kTile - 1) / kTile;
  const uint32_t tile_bytes = static_cast<uint32_t>(kTile * rowbytes);

  float *sbuf = reinterpret_cast<float *>(smem + L.sbuf);
  float *pbuf = reinterpret_cast<float *>(smem + L.pbuf);
  float *etile = reinterpret_cast<float *>(smem + L.etile);
  float *edp = reinterpret_cast<float *>(smem + L.edp);
  float *xm = reinterpret_cast<float *>(smem + L.xm);
  float *xl = reinterpret_cast<float *>(smem + L.xl);
  float *xc = reinterpret_cast<float *>(smem + L.xc);
  float *xa = reinterpret_cast<float *>(smem + L.xa);
  float *xb = reinterpret_cast<float *>(smem + L.xb);
  float4 *glob = reinterpret_cast<float4 *>(smem + L.glob);
  float4 *rstat = reinterpret_cast<float4 *>(smem + L.rstat);
  float *alph = reinterpret_cast<float *>(smem + L.alpha);
  float *runm = reinterpret_cast<float *>(smem + L.runm);
  float *runl = reinterpret_cast<float *>(smem + L.runl);
  float *runc = reinterpret_cast<float *>(smem + L.runc);
  float *rsc = reinterpret_cast<float *>(smem + L.rsc);
  float *qsm = reinterpret_cast<float *>(smem + L.qs);    // [GMAX][4 parts][D/4 + 4]: scale*q
  float *dsm = qsm + GMAX * 4 * (D / 4 + 4);              // same for dout
  const uint32_t bar0 = smem_u32(smem + L.bars);
  const uint32_t kv0 = smem_u32(smem + L.kv);
  // Tensor-core path (bf16, D = 128, a full 128-key chunk): K and V arrive as
  // one 128-row block each, [2 halves of 64 dims][128 rows][128 B] swizzled,
  // and s = K (scale q)^T, dP = V dout^T come from two M=128, N=16, K=128
  // MMA chains whose B operands carry each head's vector split into bf16
  // high and low parts (q = hi + lo to ~2^-17), so the fp32 results match
  // fp32 dot products closely.  The B operands [16 rows][128 dims] sit in the
  // q/dout staging area, which the score buffers overlap once the products
  // are done.
  constexpr bool TCP = (DT == 128);
  const bool tc = TCP && p.tc != 0;
  const uint32_t tcbar = smem_u32(smem + L.tcs);

  auto ktile = [&](int st) -> const unsigned char * { return smem + L.kv + st * tile_bytes; };
  auto vtile = [&](int st) -> const unsigned char * { return smem + L.kv + (kStages + st) * tile_bytes; };
  // address of element d of row r in a tile
  auto elem = [&](const unsigned char *tile, int r, int d) -> const unsigned char * {
    if constexpr (SWZ) {
      const int off = d * ES;
      return tile + (off >> 7) * (kTile * 128) + r * 128 + ((((off & 127) >> 4) ^ (r & 7)) << 4) + (off & 15);
    } else {
      return tile + r * rowbytes + d * ES;
    }
  };

  auto issue = [&](int t) {
    const int st = t % kStages;
    const uint32_t bar = bar0 + st * 8;
    const uint32_t kd = kv0 + st * tile_bytes, vd = kv0 + (kStages + st) * tile_bytes;
    mbar_arrive_expect_tx(bar, 2 * tile_bytes);
    if constexpr (SWZ) {
      // one 128-byte-wide box per 128 bytes of row; box bx lands at bx * 8 KiB
#pragma unroll
      for (int bx = 0; bx < DT * ES / 128; ++bx) {
        tma_load_4d(kd + bx * (kTile * 128), &tmK, bx * (128 / ES), kvh, key0 + t * kTile, b, bar);
        tma_load_4d(vd + bx * (kTile * 128), &tmV, bx * (128 / ES), kvh, key0 + t * kTile, b, bar);
      }
    } else {
      tma_load_4d(kd, &tmK, 0, kvh, key0 + t * kTile, b, bar);
      tma_load_4d(vd, &tmV, 0, kvh, key0 + t * kTile, b, bar);
    }
  };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + s * 8, 1);
    mbar_init(tcbar, 1);
    fence_barrier_init();
    if (tc) {
      // the K / V copies go out first; everything below overlaps them
      mbar_arrive_expect_tx(bar0, 4 * 16384);
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        tma_load_4d(kv0 + hx * 16384, &tmK, hx * 64, kvh, key0, b, bar0);
        tma_load_4d(kv0 + 32768 + hx * 16384, &tmV, hx * 64, kvh, key0, b, bar0);
      }
    }
  }
  if (tid < kMaxG) {
    runm[tid] = -INFINITY;
    runl[tid] = 0.f;
    runc[tid] = 0.f;
  }
  if (tc && warp == 0) tc::tmem_alloc(tcbar + 8, 64);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tc ? *reinterpret_cast<volatile uint32_t *>(smem + L.tcs + 8) : 0u;
  if (tid == 0 && !tc)
    for (int t = 0; t < min(kStages, ntiles); ++t) issue(t);
  // announce that this CTA runs (its shared memory may be written by its
  // peers once they have waited on this phase of the cluster barrier)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---- scale*q and dout for the dot products
  const size_t qrow0 = (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * G) * D;
  const int lpr = 1 << p.lpr_log2;                      // generic: lanes per row
  const int sub = lane & (lpr - 1);
  const int rgrp = lane >> p.lpr_log2;
  const int rows_per_warp = 32 >> p.lpr_log2;
  const int rows_per_step = kWarps * rows_per_warp;
  const bool lane_on = sub * 16 < rowbytes;
  constexpr int QR = SWZ ? 1 : GMAX;                    // register copies (generic only)
  float qr[QR][EPL], dr[QR][EPL];
  if (tc) {
    // B operands: row n < GMAX holds the bf16 high part of head n's vector,
    // row GMAX + n its low part, rows past 2 GMAX (and heads >= G) zero
    unsigned char *qb = smem + L.qs, *db = qb + 4096;
    for (int idx = tid; idx < 16 * 128; idx += kThreads) {
      const int n = idx >> 7, d = idx & 127;
      const int h = n < GMAX ? n : n - GMAX;
      float xq = 0.f, xd = 0.f;
      if (n < 2 * GMAX && h < G) {
        xq = p.q[qrow0 + static_cast<size_t>(h) * D + d] * p.scale;
        xd = p.dout[qrow0 + static_cast<size_t>(h) * D + d];
      }
      const __nv_bfloat16 qh = __float2bfloat16_rn(xq), dh = __float2bfloat16_rn(xd);
      const __nv_bfloat16 vq = n < GMAX ? qh : __float2bfloat16_rn(xq - __bfloat162float(qh));
      const __nv_bfloat16 vd = n < GMAX ? dh : __float2bfloat16_rn(xd - __bfloat162float(dh));
      const int off = (d >> 6) * 2048 + n * 128 + ((((d & 63) >> 3) ^ (n & 7)) << 4) + (d & 7) * 2;
      *reinterpret_cast<__nv_bfloat16 *>(qb + off) = vq;
      *reinterpret_cast<__nv_bfloat16 *>(db + off) = vd;
    }
    fence_proxy_async_smem();
    __syncthreads();
  } else if constexpr (SWZ) {
    constexpr int DPL = DT / 4;
    for (int idx = tid; idx < GMAX * DT; idx += kThreads) {
      const int h = idx / DT, d = idx - h * DT;
      const int o = (h * 4 + d / DPL) * (DPL + 4) + d % DPL;
      const bool on = h < G;
      qsm[o] = on ? p.q[qrow0 + idx] * p.scale : 0.f;
      dsm[o] = on ? p.dout[qrow0 + idx] : 0.f;
    }
    __syncthreads();
  } else {
#pragma unroll
    for (int h = 0; h < QR; ++h)
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const int d = sub * EPL + e;
        const bool on = h < G && lane_on;
        qr[h][e] = on ? p.q[qrow0 + static_cast<size_t>(h) * D + d] * p.scale : 0.f;
        dr[h][e] = on ? p.dout[qrow0 + static_cast<size_t>(h) * D + d] : 0.f;
      }
  }
  const int wmask = (lpr > NV ? lpr / NV : 1) - 1;   // generic: lanes of a group holding identical sums

  // (a) s_hj = (scale q_h) . K_j and dP_hj = dout_h . V_j.
  // Swizzled path: thread (r, pp) owns quarter pp of row r of NR tiles
  // (st0, st0 + 1, ...), so each broadcast q/dout load feeds NR rows; the dot
  // products use packed fp32x2 FMAs and a 4-lane reduce-scatter.
  auto dots_swz = [&](auto nr_tag, int st0, int rows0, int rows1) {
    constexpr int NR = decltype(nr_tag)::value;
    constexpr int DPL = (DT > 0 ? DT : 4) / 4;
    constexpr int NCH = DPL * ES / 16;
    const int r = tid >> 2, pp = tid & 3;             // 64 rows x 4 quarter-rows
    float2 acc[NR][NV];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr)
#pragma unroll
      for (int i = 0; i < NV; ++i) acc[rr][i] = make_float2(0.f, 0.f);
    const float *qp = qsm + pp * (DPL + 4);
    const float *dp_ = dsm + pp * (DPL + 4);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int d0 = pp * DPL + c * 8;
      float2 kf[NR][4], vf[NR][4];
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        const uint4 ku = *reinterpret_cast<const uint4 *>(elem(ktile(st0 + rr), r, d0));
        const uint4 vu = *reinterpret_cast<const uint4 *>(elem(vtile(st0 + rr), r, d0));
        kf[rr][0] = make_float2(bf16_lo(ku.x), bf16_hi(ku.x)); kf[rr][1] = make_float2(bf16_lo(ku.y), bf16_hi(ku.y));
        kf[rr][2] = make_float2(bf16_lo(ku.z), bf16_hi(ku.z)); kf[rr][3] = make_float2(bf16_lo(ku.w), bf16_hi(ku.w));
        vf[rr][0] = make_float2(bf16_lo(vu.x), bf16_hi(vu.x)); vf[rr][1] = make_float2(bf16_lo(vu.y), bf16_hi(vu.y));
        vf[rr][2] = make_float2(bf16_lo(vu.z), bf16_hi(vu.z)); vf[rr][3] = make_float2(bf16_lo(vu.w), bf16_hi(vu.w));
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        const float4 qa = *reinterpret_cast<const float4 *>(qp + h * 4 * (DPL + 4) + c * 8);
        const float4 qb = *reinterpret_cast<const float4 *>(qp + h * 4 * (DPL + 4) + c * 8 + 4);
        const float4 da = *reinterpret_cast<const float4 *>(dp_ + h * 4 * (DPL + 4) + c * 8);
        const float4 db = *reinterpret_cast<const float4 *>(dp_ + h * 4 * (DPL + 4) + c * 8 + 4);
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) {
          acc[rr][h] = __ffma2_rn(make_float2(qa.x, qa.y), kf[rr][0], acc[rr][h]);
          acc[rr][h] = __ffma2_rn(make_float2(qa.z, qa.w), kf[rr][1], acc[rr][h]);
          acc[rr][h] = __ffma2_rn(make_float2(qb.x, qb.y), kf[rr][2], acc[rr][h]);
          acc[rr][h] = __ffma2_rn(make_float2(qb.z, qb.w), kf[rr][3], acc[rr][h]);
          acc[rr][GMAX + h] = __ffma2_rn(make_float2(da.x, da.y), vf[rr][0], acc[rr][GMAX + h]);
          acc[rr][GMAX + h] = __ffma2_rn(make_float2(da.z, da.w), vf[rr][1], acc[rr][GMAX + h]);
          acc[rr][GMAX + h] = __ffma2_rn(make_float2(db.x, db.y), vf[rr][2], acc[rr][GMAX + h]);
          acc[rr][GMAX + h] = __ffma2_rn(make_float2(db.z, db.w), vf[rr][3], acc[rr][GMAX + h]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      float val[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) val[i] = acc[rr][i].x + acc[rr][i].y;
      int idx0, nf;
      reduce_scatter<NV>(val, 4, pp, idx0, nf);
      // each of the 4 lanes keeps NV/4 sums (all scores or all dP, heads
      // idx0 % GMAX onward); with NV = 2, lanes 0 and 2 hold the two sums
      constexpr int NF = NV >= 4 ? NV / 4 : 1;
      if (r < (rr == 0 ? rows0 : rows1) && (NV >= 4 || (pp & 1) == 0)) {
        float *dst = (idx0 < GMAX ? sbuf : pbuf) + ((st0 + rr) * kTile + r) * GMAX + (idx0 & (GMAX - 1));
        if constexpr (NF == 4) {
          *reinterpret_cast<float4 *>(dst) = make_float4(val[0], val[1], val[2], val[3]);
        } else if constexpr (NF == 2) {
          *reinterpret_cast<float2 *>(dst) = make_float2(val[0], val[1]);
        } else {
          dst[0] = val[0];
        }
      }
    }
  };
  // Generic path: a row split over `lpr` lanes of 16 bytes, q/dout in registers.
  auto dots = [&](int st, int jt, int rows_valid) {
    const unsigned char *Kt = ktile(st), *Vt = vtile(st);
    if constexpr (SWZ) {
      dots_swz(std::integral_constant<int, 1>{}, st, rows_valid, 0);
    } else {
      for (int r = warp * rows_per_warp + rgrp; r < kTile; r += rows_per_step) {
        float kf[EPL], vf[EPL];
        if (lane_on) {
          load16(Kt + r * rowbytes + sub * 16, kf);
          load16(Vt + r * rowbytes + sub * 16, vf);
        } else {
#pragma unroll
          for (int e = 0; e < EPL; ++e) kf[e] = vf[e] = 0.f;
        }
        float val[NV];
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          float a = 0.f, c = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            a = fmaf(qr[h][e], kf[e], a);
            c = fmaf(dr[h][e], vf[e], c);
          }
          val[h] = a;
          val[GMAX + h] = c;
        }
        int idx0, nf;
        reduce_scatter<NV>(val, lpr, sub, idx0, nf);
        if ((sub & wmask) == 0 && r < rows_valid) {
#pragma unroll
          for (int i = 0; i < NV; ++i) {
            if (i < nf) {
              const int idx = idx0 + i;
              const int h = idx < GMAX ? idx : idx - GMAX;
              if (h < G) (idx < GMAX ? sbuf : pbuf)[(jt + r) * GMAX + h] = val[i];
            }
          }
        }
      }
    }
  };

  // ======================= phase 1 =========================================
  const int D4 = D >> 2;
  if (resident) {
    if (tc) {
      if (warp == 0) {
        mbar_wait_or_flag(bar0, 0, p.wait);
        tc::fence_after_sync();
        if (lane == 0) {
          constexpr uint32_t id = tc::idesc_bf16_f32(128, 16, 0, 0);
          const uint32_t qb = smem_u32(smem + L.qs), db = qb + 4096;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = (kk >> 2) * 2048 + (kk & 3) * 32;
            tc::mma_bf16(tmem, tc::sdesc_sw128(kv0 + ao, 16, 1024), tc::sdesc_sw128(qb + bo, 16, 1024), id, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = (kk >> 2) * 2048 + (kk & 3) * 32;
            tc::mma_bf16(tmem + 16, tc::sdesc_sw128(kv0 + 32768 + ao, 16, 1024), tc::sdesc_sw128(db + bo, 16, 1024),
                         id, kk > 0);
          }
          tc::commit(tcbar);
        }
        __syncwarp();
      }
      mbar_wait_or_flag(tcbar, 0, p.wait);
      tc::fence_after_sync();
      if (warp < 4) {
        // TMEM lane = key; columns: s hi | s lo | pad (16), dP hi | dP lo | pad (16)
        float v[32];
        tc::ld32_wait(tmem + (static_cast<uint32_t>(32 * warp) << 16), v);
        const int key = 32 * warp + lane;
        if (key < nkeys) {
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            sbuf[key * GMAX + h] = h < G ? v[h] + v[GMAX + h] : 0.f;
            pbuf[key * GMAX + h] = h < G ? v[16 + h] + v[16 + GMAX + h] : 0.f;
          }
        }
      }
      tc::fence_before_sync();
    } else if (SWZ && ntiles == 2) {
      mbar_wait_or_flag(bar0, 0, p.wait);
      mbar_wait_or_flag(bar0 + 8, 0, p.wait);
      dots_swz(std::integral_constant<int, 2>{}, 0, kTile, nkeys - kTile);
    } else {
      for (int t = 0; t < ntiles; ++t) {
        mbar_wait_or_flag(bar0 + t * 8, 0, p.wait);
        dots(t, t * kTile, min(kTile, nkeys - t * kTile));
      }
    }
    __syncthreads();
    // chunk statistics per head (warp h): max, sum e, sum e dP
    if (warp < G) {
      const int h = warp;
      float m = -INFINITY;
      for (int j = lane; j < nkeys; j += 32) m = fmaxf(m, sbuf[j * GMAX + h]);
      m = warp_max(m);
      float ls = 0.f, cs = 0.f;
      for (int j = lane; j < nkeys; j += 32) {
        const float e = expf(sbuf[j * GMAX + h] - m);
        ls += e;
        cs = fmaf(e, pbuf[j * GMAX + h], cs);
      }
      ls = warp_sum(ls);
      cs = warp_sum(cs);
      if (lane == 0) {
        xm[h] = m;
        xl[h] = ls;
        xc[h] = cs;
      }
    }
  } else {
    // streaming: running statistics and running dq partials
    const int dc = tid % D4, rsp = tid / D4;
    const bool c_on = rsp < RS;
    float accA[GMAX][4], accB[GMAX][4];
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) accA[h][i] = accB[h][i] = 0.f;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kStages;
      mbar_wait_or_flag(bar0 + st * 8, (t / kStages) & 1, p.wait);
      const int rows_valid = min(kTile, nkeys - t * kTile);
      const int jt = t * kTile;
      dots(st, jt, rows_valid);
      __syncthreads();
      if (warp < G) {
        const int h = warp;
        const float s0 = lane < rows_valid ? sbuf[(jt + lane) * GMAX + h] : -INFINITY;
        const float s1 = lane + 32 < rows_valid ? sbuf[(jt + lane + 32) * GMAX + h] : -INFINITY;
        const float d0 = lane < rows_valid ? pbuf[(jt + lane) * GMAX + h] : 0.f;
        const float d1 = lane + 32 < rows_valid ? pbuf[(jt + lane + 32) * GMAX + h] : 0.f;
        const float mt = warp_max(fmaxf(s0, s1));
        const float m_old = runm[h];
        const float m_new = fmaxf(m_old, mt);
        const float a = expf(m_old - m_new);   // 0 on the first tile
        const float e0 = lane < rows_valid ? expf(s0 - m_new) : 0.f;
        const float e1 = lane + 32 < rows_valid ? expf(s1 - m_new) : 0.f;
        etile[lane * GMAX + h] = e0;
        etile[(lane + 32) * GMAX + h] = e1;
        edp[lane * GMAX + h] = e0 * d0;
        edp[(lane + 32) * GMAX + h] = e1 * d1;
        const float ls = warp_sum(e0 + e1);
        const float csum = warp_sum(e0 * d0 + e1 * d1);
        if (lane == 0) {
          runl[h] = runl[h] * a + ls;
          runc[h] = runc[h] * a + csum;
          runm[h] = m_new;
          alph[h] = a;
        }
      }
      __syncthreads();
      // A_h[d] = sum_j e_hj dP_hj K_jd, B_h[d] = sum_j e_hj K_jd (max-rescaled)
      if (c_on) {
        const unsigned char *Kt = ktile(st);
        float al[GMAX];
        ld_heads<GMAX>(alph, al);
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            accA[h][i] *= al[h];
            accB[h][i] *= al[h];
          }
        for (int r = rsp; r < rows_valid; r += RS) {
          const float4 kv = load4(elem(Kt, r, 4 * dc), static_cast<KV *>(nullptr));
          float e[GMAX], w[GMAX];
          ld_heads<GMAX>(etile + r * GMAX, e);
          ld_heads<GMAX>(edp + r * GMAX, w);
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            accA[h][0] = fmaf(w[h], kv.x, accA[h][0]); accA[h][1] = fmaf(w[h], kv.y, accA[h][1]);
            accA[h][2] = fmaf(w[h], kv.z, accA[h][2]); accA[h][3] = fmaf(w[h], kv.w, accA[h][3]);
            accB[h][0] = fmaf(e[h], kv.x, accB[h][0]); accB[h][1] = fmaf(e[h], kv.y, accB[h][1]);
            accB[h][2] = fmaf(e[h], kv.z, accB[h][2]); accB[h][3] = fmaf(e[h], kv.w, accB[h][3]);
          }
        }
      }
      __syncthreads();
      if (tid == 0 && t + kStages < ntiles) {
        fence_proxy_async_smem();
        issue(t + kStages);
      }
    }
    // row-split partials -> scratch (the tiles are consumed), summed in a
    // fixed order so results do not depend on scheduling
    float *sa = reinterpret_cast<float *>(smem + L.kv);
    float *sb = sa + RS * G * D;
    if (c_on) {
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h < G) {
          float *pa = sa + rsp * G * D + h * D + 4 * dc;
          float *pb = sb + rsp * G * D + h * D + 4 * dc;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pa[i] = accA[h][i];
            pb[i] = accB[h][i];
          }
        }
      }
    }
    if (tid < G) {
      xm[tid] = runm[tid];
      xl[tid] = runl[tid];
      xc[tid] = runc[tid];
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kThreads) {
      float a = 0.f, c = 0.f;
      for (int rs = 0; rs < RS; ++rs) {
        a += sa[rs * G * D + idx];
        c += sb[rs * G * D + idx];
      }
      xa[idx] = a;
      xb[idx] = c;
    }
  }
  // every CTA pushes its statistics into slot `rank` of each CTA's table, so
  // after the cluster barrier the merge reads only local shared memory (every
  // peer has started: the first cluster-barrier phase has completed)
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (tid < p.ncl * G) {
    const int r = tid / G, h = tid - r * G;
    cluster.map_shared_rank(rstat, r)[rank * GMAX + h] = make_float4(xm[h], xl[h], xc[h], 0.f);
  }
  cluster.sync();

  // ======================= merge the softmax statistics ====================
  if (tid < G) {
    const int h = tid;
    float M = -INFINITY;
    for (int r = 0; r < p.ncl; ++r) M = fmaxf(M, rstat[r * GMAX + h].x);
    float Ls = 0.f, Cs = 0.f;
    for (int r = 0; r < p.ncl; ++r) {
      const float4 st = rstat[r * GMAX + h];
      const float w = expf(st.x - M);
      Ls = fmaf(st.y, w, Ls);
      Cs = fmaf(st.z, w, Cs);
      rsc[r * kMaxG + h] = w;
    }
    glob[h] = make_float4(M, 1.f / Ls, Cs / Ls, 0.f);
  }
  __syncthreads();

  // P and scale * dS of this CTA's keys, in place of the score and dP
  // (heads G .. GMAX-1 of the padded layout get 0, so later loops need no
  // head predicate)
  for (int i = tid; i < GMAX * nkeys; i += kThreads) {
    const int h = i & (GMAX - 1);
    float P = 0.f, dS = 0.f;
    if (h < G) {
      const float4 g = glob[h];
      P = expf(sbuf[i] - g.x) * g.y;
      dS = p.scale * P * (pbuf[i] - g.z);
    }
    sbuf[i] = P;
    pbuf[i] = dS;
  }
  __syncthreads();

  // ======================= dq partial of this CTA ==========================
  // Resident K: sum_j dS'_hj K_j over this CTA's keys, pushed into a slot of
  // rank 0's (consumed) V tiles.  Streaming: rank 0 merges the running
  // partials of every CTA now.  Either way this happens before any dK/dV
  // store is issued, and the cluster barrier that publishes it is split: its
  // arrive goes out here and its wait comes after the stores, so neither side
  // stalls on the other.
  float *slots = reinterpret_cast<float *>(smem + L.kv + kStages * tile_bytes);   // [ncl][G*D] in rank 0
  const int half = D >> 1;
  // phase 2: dK / dV rows of this CTA's keys, over the warps [w0, w0 + nw)
  auto store_rows = [&](int w0, int nw) {
    const int F4 = D >> 2;                                  // float4 per output row
    int olog = 0;
    while ((1 << olog) < F4 && olog < 5) ++olog;
    const int olpr = 1 << olog;                             // lanes per row (<= 32)
    const int osub = lane & (olpr - 1), ogrp = lane >> olog;
    const int orows_w = 32 >> olog;
    const int npass = (F4 + 31) / 32;
    for (int pass = 0; pass < npass; ++pass) {
      const int f = osub + 32 * pass;
      const bool on = f < F4;
      float2 qo[GMAX][2], go[GMAX][2];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
        if (on && h < G) {
          a = *reinterpret_cast<const float4 *>(p.q + qrow0 + static_cast<size_t>(h) * D + 4 * f);
          c = *reinterpret_cast<const float4 *>(p.dout + qrow0 + static_cast<size_t>(h) * D + 4 * f);
        }
        qo[h][0] = make_float2(a.x, a.y); qo[h][1] = make_float2(a.z, a.w);
        go[h][0] = make_float2(c.x, c.y); go[h][1] = make_float2(c.z, c.w);
      }
      float *dkp = p.dk + ((static_cast<size_t>(b) * p.S + key0) * p.Hkv + kvh) * D + 4 * f;
      float *dvp = p.dv + ((static_cast<size_t>(b) * p.S + key0) * p.Hkv + kvh) * D + 4 * f;
      const size_t rstride = static_cast<size_t>(p.Hkv) * D;
      for (int j = (warp - w0) * orows_w + ogrp; j < nkeys; j += nw * orows_w) {
        float2 k0 = make_float2(0.f, 0.f), k1 = k0, v0 = k0, v1 = k0;
        float Ph[GMAX], dSh[GMAX];
        ld_heads<GMAX>(sbuf + j * GMAX, Ph);
        ld_heads<GMAX>(pbuf + j * GMAX, dSh);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          const float2 ds = make_float2(dSh[h], dSh[h]), pw = make_float2(Ph[h], Ph[h]);
          k0 = __ffma2_rn(ds, qo[h][0], k0);
          k1 = __ffma2_rn(ds, qo[h][1], k1);
          v0 = __ffma2_rn(pw, go[h][0], v0);
          v1 = __ffma2_rn(pw, go[h][1], v1);
        }
        if (on) {
          st_cs_f4(dkp + j * rstride, make_float4(k0.x, k0.y, k1.x, k1.y));
          st_cs_f4(dvp + j * rstride, make_float4(v0.x, v0.y, v1.x, v1.y));
        }
      }
    }
  };
  if (resident) {
    // Resident K: warps 0-3 form sum_j dS'_hj K_j over this CTA's keys and
    // push it into a slot of rank 0's (consumed) V tiles while warps 4-7
    // write the dK / dV rows; the two use different units (shared memory and
    // ALU against the store path) and overlap.  The cluster barrier that
    // publishes the slots is split: every warp arrives once (warps 0-3 after
    // their push, with release), and all wait after their own work.
    if (tc && warp < 4) {
      // dq^T [128 dims][16] = K^T dS on the tensor core: A = the resident K
      // block read MN-major (M = head dims), B = [16 rows][128 keys] with
      // row n < GMAX the bf16 high part of head n's scale * dS, row GMAX + n
      // its low part; the result (TMEM lane = head dim) goes to rank 0.
      unsigned char *bq = smem + L.qs;                   // free since the score / dP products completed
      for (int idx = tid; idx < 16 * 128; idx += 128) {
        const int n = idx >> 7, j = idx & 127;
        const int h = n < GMAX ? n : n - GMAX;
        const float x = (n < 2 * GMAX && j < nkeys) ? pbuf[j * GMAX + h] : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const __nv_bfloat16 val = n < GMAX ? hi : __float2bfloat16_rn(x - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16 *>(bq + (j >> 6) * 2048 + n * 128 + ((((j & 63) >> 3) ^ (n & 7)) << 4) +
                                           (j & 7) * 2) = val;
      }
      fence_proxy_async_smem();
      named_barrier(1, 128);
      if (warp == 0) {
        tc::fence_after_sync();
        if (lane == 0) {
          constexpr uint32_t id = tc::idesc_bf16_f32(128, 16, 1, 0);
          const uint32_t bqa = smem_u32(bq);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_bf16(tmem + 32, tc::sdesc_sw128(kv0 + kk * 2048, 16384, 1024),
                         tc::sdesc_sw128(bqa + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024), id, kk > 0);
          tc::commit(tcbar);
        }
        __syncwarp();
      }
      mbar_wait_or_flag(tcbar, 1, p.wait);
      tc::fence_after_sync();
      float v[32];
      tc::ld32_wait(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32, v);
      tc::fence_before_sync();
      const int d = 32 * warp + lane;
      float *dst0 = cluster.map_shared_rank(slots, 0) + rank * G * D;
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) dst0[h * D + d] = v[h] + v[GMAX + h];
      asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    } else if (warp < 4) {
      const int dc = tid % D4, rsp = tid / D4;           // (row split, 4-dim chunk)
      // row splits among the 128 threads, capped so nrs * G * D floats fit
      // the K tiles once consumed
      const int nrs = min(128 / D4, 32 * ES / GMAX);
      float2 aq[GMAX][2];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) aq[h][0] = aq[h][1] = make_float2(0.f, 0.f);
      if (rsp < nrs) {
        for (int j = rsp; j < nkeys; j += nrs) {
          const float4 kv = load4(elem(ktile(j / kTile), j % kTile, 4 * dc), static_cast<KV *>(nullptr));
          const float2 k01 = make_float2(kv.x, kv.y), k23 = make_float2(kv.z, kv.w);
          float dSh[GMAX];
          ld_heads<GMAX>(pbuf + j * GMAX, dSh);
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            const float2 w = make_float2(dSh[h], dSh[h]);
            aq[h][0] = __ffma2_rn(w, k01, aq[h][0]);
            aq[h][1] = __ffma2_rn(w, k23, aq[h][1]);
          }
        }
      }
      named_barrier(1, 128);                             // K tiles consumed
      float *red = reinterpret_cast<float *>(smem + L.kv);
      if (rsp < nrs) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
          if (h < G)
            *reinterpret_cast<float4 *>(red + (rsp * G + h) * D + 4 * dc) =
                make_float4(aq[h][0].x, aq[h][0].y, aq[h][1].x, aq[h][1].y);
      }
      named_barrier(1, 128);
      float *dst0 = cluster.map_shared_rank(slots, 0) + rank * G * D;
      for (int idx = tid; idx < G * D; idx += 128) {
        float a = 0.f;
        for (int r = 0; r < nrs; ++r) a += red[r * G * D + idx];
        dst0[idx] = a;
      }
      asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    } else {
      asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
      store_rows(4, kWarps - 4);
    }
  } else {
    // Streaming: rank 0 merges the running partials of every CTA, then all
    // warps write their dK / dV rows.
    if (rank == 0) {
      for (int pr = tid; pr < G * half; pr += kThreads) {
        const int h = pr / half, pi = pr - h * half;
        const int idx = h * D + 2 * pi;
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          if (r < p.ncl) {
            const float w = rsc[r * kMaxG + h];
            const float2 ra = *reinterpret_cast<const float2 *>(cluster.map_shared_rank(xa, r) + idx);
            const float2 rb = *reinterpret_cast<const float2 *>(cluster.map_shared_rank(xb, r) + idx);
            a0 = fmaf(w, ra.x, a0); a1 = fmaf(w, ra.y, a1);
            b0 = fmaf(w, rb.x, b0); b1 = fmaf(w, rb.y, b1);
          }
        }
        const float4 g = glob[h];
        const float y0 = p.scale * (a0 - g.z * b0) * g.y;
        const float y1 = p.scale * (a1 - g.z * b1) * g.y;
        float z0 = y0, z1 = y1;
        if (p.rope) {
          const float c = p.rcos[pi], sn = p.rsin[pi];
          z0 = y0 * c + y1 * sn;
          z1 = -y0 * sn + y1 * c;
        }
        *reinterpret_cast<float2 *>(p.dq + qrow0 + idx) = make_float2(z0, z1);
      }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    store_rows(0, kWarps);
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");

  // ======================= dq (resident): rank 0 sums the slots ============
  if (resident && rank == 0) {
    for (int pr = tid; pr < G * half; pr += kThreads) {
      const int h = pr / half, pi = pr - h * half;
      const int idx = h * D + 2 * pi;
      float y0 = 0.f, y1 = 0.f;
      for (int r = 0; r < p.ncl; ++r) {
        const float2 v = *reinterpret_cast<const float2 *>(slots + r * G * D + idx);
        y0 += v.x;
        y1 += v.y;
      }
      float z0 = y0, z1 = y1;
      if (p.rope) {
        const float c = p.rcos[pi], sn = p.rsin[pi];
        z0 = y0 * c + y1 * sn;
        z1 = -y0 * sn + y1 * c;
      }
      *reinterpret_cast<float2 *>(p.dq + qrow0 + idx) = make_float2(z0, z1);
    }
  }
  if (tc) {
    __syncthreads();   // every TMEM read has completed (waited on, fenced) before this
    if (warp == 0) {
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, 64);
    }
  }
}

template <typename KV, int GMAX, int DT>
cudaError_t launch_typed(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int smem,
                         cudaStream_t st) {
  auto kern = decode_bwd_kernel<KV, GMAX, DT>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ncl, p.Hkv, p.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

template <typename KV, int DT>
cudaError_t launch_g(int gmax, const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int smem,
                     cudaStream_t st) {
  switch (gmax) {
    case 1: return launch_typed<KV, 1, DT>(tk, tv, p, smem, st);
    case 2: return launch_typed<KV, 2, DT>(tk, tv, p, smem, st);
    case 4: return launch_typed<KV, 4, DT>(tk, tv, p, smem, st);
    default: return launch_typed<KV, 8, DT>(tk, tv, p, smem, st);
  }
}

}  // namespace

cudaError_t launch_attn_bwd_decode(const float *q, const void *k, const void *v, const float *dout, float *dq,
                                   float *dk, float *dv, int B, int Hq, int Hkv, int S, int D, int kv_bf16,
                                   float scale, double rope_base, int q_pos, const WaitCtl &w, cudaStream_t st,
                                   const char **why) {
  const int es = kv_bf16 ? 2 : 4;
  const int rowbytes = D * es;
  if (rowbytes > 512 || rowbytes % 16 != 0) {
    *why = "row width";
    return cudaErrorNotSupported;
  }
  if (Hkv > 65535 || B > 65535) {
    *why = "B or Hkv > 65535";
    return cudaErrorNotSupported;
  }
  int lpr_log2 = 0;
  while ((16 << lpr_log2) < rowbytes) ++lpr_log2;  // generic: lanes per row (16 B each), power of two
  const int G = Hq / Hkv;
  const int gmax = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
  int rs_log2 = 0;                                 // streaming: row splits of the dq partial sums
  while ((1 << (rs_log2 + 1)) <= kTile && (D / 4) << (rs_log2 + 1) <= kThreads) ++rs_log2;
  const int tiles = (S + kTile - 1) / kTile;
  int ncl = tiles < kMaxCluster ? tiles : kMaxCluster;
  const int chunk = ((tiles + ncl - 1) / ncl) * kTile;
  ncl = (S + chunk - 1) / chunk;                   // every CTA owns at least one key
  const bool resident = chunk <= kStages * kTile;
  // specialised head dims: bf16 rows of 128 / 256 / 512 bytes with a resident chunk
  const int dt = (kv_bf16 && resident && (D == 64 || D == 128 || D == 256)) ? D : 0;
  const Layout L(G, gmax, D, chunk, rowbytes, 1 << rs_log2, dt > 0, resident);
  const int smem = L.total + 1024;                 // + alignment slack
  if (smem > 227 * 1024) {
    *why = "KV length too long for the per-CTA score buffers";
    return cudaErrorNotSupported;
  }

  DecodeParams p;
  p.q = q; p.dout = dout; p.dq = dq; p.dk = dk; p.dv = dv;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.S = S; p.D = D; p.G = G;
  p.chunk = chunk; p.ncl = ncl; p.resident = resident ? 1 : 0;
  p.lpr_log2 = lpr_log2; p.rs_log2 = rs_log2; p.rowbytes = rowbytes;
  p.tc = (dt == 128 && chunk == 2 * kTile) ? 1 : 0;
  p.scale = scale;
  p.rope = rope_base > 0.0 && q_pos >= 0;
  for (int i = 0; i < 128; ++i) {
    if (p.rope && i < D / 2) {
      const double th = static_cast<double>(q_pos) * pow(rope_base, -2.0 * i / D);
      p.rcos[i] = static_cast<float>(cos(th));
      p.rsin[i] = static_cast<float>(sin(th));
    } else {
      p.rcos[i] = 1.f;
      p.rsin[i] = 0.f;
    }
  }
  p.wait = w;

  CUtensorMap tk, tv;
  const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv), static_cast<uint64_t>(S),
                            static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>(rowbytes), static_cast<uint64_t>(Hkv) * rowbytes,
                               static_cast<uint64_t>(S) * Hkv * rowbytes};
  const uint32_t box[4] = {static_cast<uint32_t>(dt ? 128 / es : D), 1, static_cast<uint32_t>(p.tc ? 2 * kTile : kTile),
                           1};
  const CUtensorMapDataType dtp = kv_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapSwizzle sw = dt ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (!encode_tiled(&tk, dtp, 4, k, dims, strides, box, sw, why) ||
      !encode_tiled(&tv, dtp, 4, v, dims, strides, box, sw, why))
    return cudaErrorInvalidValue;

  switch (dt) {
    case 64: return launch_g<__nv_bfloat16, 64>(gmax, tk, tv, p, smem, st);
    case 128: return launch_g<__nv_bfloat16, 128>(gmax, tk, tv, p, smem, st);
    case 256: return launch_g<__nv_bfloat16, 256>(gmax, tk, tv, p, smem, st);
    default:
      return kv_bf16 ? launch_g<__nv_bfloat16, 0>(gmax, tk, tv, p, smem, st)
                     : launch_g<float, 0>(gmax, tk, tv, p, smem, st);
  }
}

}  // namespace abw
