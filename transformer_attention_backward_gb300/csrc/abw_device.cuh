// Device-side helpers shared by the kernels: shared-memory barriers with
// bounded waits, TMA (cp.async.bulk.tensor) loads, bf16 conversion and warp
// reductions.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace abw {

// Bits of the device error word.
enum : unsigned int {
  kErrWaitTimeout = 1u,   // a bounded barrier wait ran out
  kErrSelfTest = 2u,      // the self-test kernel's wait ran out (expected)
  kErrSmemAlign = 4u,     // a kernel found its shared memory misaligned and did no work
};

// Everything a kernel needs to report a failed wait.
struct WaitCtl {
  unsigned int *err;              // device error words (library-owned): [0] bits, [1] first timeout site
  unsigned long long limit_ns;    // time limit of one wait
};

// Where a wait ran out, for the report: kernel (bits 28-31), barrier slot
// (bits 20-27), warp (bits 16-19) and the low 16 bits of the block index.
enum : unsigned int { kSiteKv = 1u, kSiteDq = 2u, kSiteFwd = 3u, kSiteDecode = 4u };
__device__ __forceinline__ unsigned int wait_site(unsigned int kernel, unsigned int slot) {
  return (kernel << 28) | ((slot & 0xffu) << 20) | (((threadIdx.x >> 5) & 0xfu) << 16) | (blockIdx.x & 0xffffu);
}
// Records a timeout: the error bit, and the site if it is the first one.
// Kept out of line: it runs only on the failure path.
static __device__ __noinline__ void report_timeout(unsigned int *err, unsigned int kernel, unsigned int slot) {
  atomicOr(err, kErrWaitTimeout);
  atomicCAS(err + 1, 0u, wait_site(kernel, slot));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Time spent in a bounded wait.  The global timer can be re-synchronised
// while a kernel runs, so it may step backwards or leap ahead between two
// readings; the wait sums the steps between successive readings and drops
// any step that is negative or longer than kWaitStepMaxNs (one polling round
// takes microseconds).  As a second bound, independent of the timer, the
// wait gives up after limit_ns / 128 polling rounds: a round of 32 barrier
// probes takes well over 128 ns, so this cap is never reached before the
// timed limit while the timer advances.
constexpr unsigned long long kWaitStepMaxNs = 50000000ull;   // 50 ms
struct WaitClock {
  unsigned long long prev, waited, rounds, limit;
  __device__ __forceinline__ explicit WaitClock(unsigned long long limit_ns)
      : prev(globaltimer_ns()), waited(0), rounds(0), limit(limit_ns) {}
  // one polling round has passed; true once the wait has lasted limit_ns
  __device__ __forceinline__ bool expired() {
    const unsigned long long now = globaltimer_ns();
    const unsigned long long step = now - prev;   // huge when the timer stepped back
    if (step < kWaitStepMaxNs) waited += step;
    prev = now;
    return waited > limit || ++rounds > (limit >> 7);
  }
};

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA / tensor core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Cluster-scope variant: pairs with a peer CTA's release-arrive on this
// barrier, making the peer's shared-memory writes visible to this thread.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                          unsigned long long limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  WaitClock wc(limit_ns);
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (wc.expired()) return false;
  }
}

// Arrives (release, cluster scope) on the barrier at the same shared-memory
// offset in CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}

// Waits for phase `parity` of the barrier to complete, giving up after
// `limit_ns`.  Returns false on timeout (the caller records it and drains).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  WaitClock wc(limit_ns);
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (wc.expired()) return false;
  }
}

// Bounded wait that reports a timeout in the error word and then waits once
// more (again bounded) so that copies in flight land before the block moves
// on or exits.  Returns true iff the first wait succeeded.
__device__ __forceinline__ bool mbar_wait_or_flag(uint32_t bar, uint32_t parity, const WaitCtl &w) {
  if (mbar_wait_bounded(bar, parity, w.limit_ns)) return true;
  report_timeout(w.err, kSiteDecode, bar >> 3);
  const unsigned long long drain = w.limit_ns < 2000000000ull ? 2000000000ull : w.limit_ns;
  mbar_wait_bounded(bar, parity, drain);
  return false;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// L2 eviction-priority policies for the cache-hinted copies below.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                                 int c3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Plain bulk copy global -> shared (both addresses 16-byte aligned, size a
// multiple of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Element-wise add of a shared-memory tile into global memory through a
// tensor map (rows past the tensor's extent are dropped).  Completion is
// tracked by bulk groups: commit, then wait until the source has been read.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2,
                                                  int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// Plain bulk copy shared -> global, tracked by bulk groups (both addresses
// 16-byte aligned, size a multiple of 16 bytes).
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}
// Tile copy shared -> global through a tensor map, tracked by bulk groups
// (elements outside the tensor are not written).  Coordinates must not be
// negative.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Barrier over a subset of the block's warps (id 1..15, `count` threads).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier over `count` threads that also returns the AND of `pred` across
// them, so a group of warps can leave a loop together.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.b32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1 : 0), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Vector fp32 reduction into global memory (four consecutive floats), done
// in the L2 without returning a value.
__device__ __forceinline__ void red_add_f4(float *p, float4 v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// Streaming (evict-first) 16-byte store for outputs that are not re-read.
__device__ __forceinline__ void st_cs_f4(float *p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

}  // namespace abw
