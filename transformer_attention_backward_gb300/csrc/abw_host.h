// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "abw_device.cuh"

namespace abw {

// Unique id of the calling thread's current CUDA context (0 if none).
// Per-device caches (symbol addresses, raised attribute limits) are keyed on
// it as well as on the ordinal, so that they are resolved again in a context
// created after cudaDeviceReset.
unsigned long long context_id();

// Error word + wait limit for the current device (resolved once per device
// and context).  `err` is null if the symbol address could not be obtained.
WaitCtl wait_ctl();

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).  Returns false and fills `why` on failure.
bool encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, uint32_t rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                  CUtensorMapSwizzle swizzle, const char **why);

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`, calling the runtime only when the limit has to grow: calls
// after the first make no runtime call for it (which keeps them free of
// anything but launches, e.g. under stream capture).
cudaError_t ensure_dynamic_smem(const void *func, int bytes);

// Launchers: validate nothing (api.cu has done it), enqueue, and return the
// launch error.
cudaError_t launch_softmax_bwd(const float *s, const float *dy, float *dx, int rows, int n,
                               cudaStream_t st);
cudaError_t launch_rope_bwd(const float *dy, float *dx, int B, int T, int H, int D, const float *theta,
                            int pos0, double base, int interleaved, cudaStream_t st);
cudaError_t launch_rmsnorm_bwd(const void *x, int x_bf16, const float *gamma, const float *dy, void *dx,
                               int dx_bf16, int rows, int n, float eps, cudaStream_t st);

// Zeroes dgamma, then adds every row's dy x / rms into it; dx may be null.
cudaError_t launch_rmsnorm_bwd_dgamma(const void *x, int x_bf16, const float *gamma, const float *dy, void *dx,
                                      int dx_bf16, float *dgamma, int rows, int n, float eps, cudaStream_t st);
cudaError_t launch_relu2_mul_bwd(const void *gate, const void *up, int bf16, const float *dh, float *dgate,
                                 float *dup, long long n, cudaStream_t st);
size_t lora_workspace_bytes(int rows, int r);
cudaError_t launch_lora_bwd(const void *x, int x_bf16, const float *dy, const float *A, const float *B, float *dA,
                            float *dB, int rows, int n_in, int n_out, int r, float scale, void *ws,
                            cudaStream_t st);

// Returns cudaErrorNotSupported (and sets *why) when a shape has no kernel.
cudaError_t launch_attn_bwd_decode(const float *q, const void *k, const void *v, const float *dout,
                                   float *dq, float *dk, float *dv, int B, int Hq, int Hkv, int S, int D,
                                   int kv_bf16, float scale, double rope_base, int q_pos,
                                   const WaitCtl &w, cudaStream_t st, const char **why);

cudaError_t launch_attn_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse, int B, int T,
                                   int Hq, int Hkv, int D, float scale, const WaitCtl &w, cudaStream_t st,
                                   const char **why);

size_t causal_workspace_bytes(int B, int T, int Hq, int D);
// pattn: saved probabilities [B][Hq][T][T] bf16 (then lse may be null), or
// null to recompute them from lse.
cudaError_t launch_attn_bwd_causal(const void *q, const void *k, const void *v, const void *pattn, const void *o,
                                   const void *dout, const float *lse, float *dq, float *dk, float *dv,
                                   int B, int T, int Hq, int Hkv, int D, float scale, double rope_base,
                                   int pos0, void *ws, size_t ws_bytes, const WaitCtl &w,
                                   cudaStream_t st, const char **why);

cudaError_t launch_selftest_wait(const WaitCtl &w, cudaStream_t st);

// Size of the fixed device scratch behind attn_bwd_causal_noalloc.
constexpr size_t kNoAllocScratchBytes = 32ull << 20;   // 32 MiB

// Device address of that scratch on the current device (resolved once per
// device).  Never allocates.
cudaError_t noalloc_scratch(void **ptr, const char **why);

}  // namespace abw
