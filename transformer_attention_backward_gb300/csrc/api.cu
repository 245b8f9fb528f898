// The C ABI: argument validation, status codes, the per-thread error message,
// the device error word, and the TMA descriptor encoder.  Every compute step
// runs in the kernels of the other translation units.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/attn_bwd.h"
#include "abw_host.h"

namespace {

thread_local std::string g_last_error;
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

// The device error word.  Kernels receive its device address (resolved per
// device with cudaGetSymbolAddress) and atomically OR failure bits into it.
__device__ unsigned int g_abw_err_word[2];   // bits, first timeout site

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
unsigned int *g_err_addr[kMaxDevices] = {};
unsigned long long g_err_ctx[kMaxDevices] = {};   // context the cached address belongs to

abw_status fail(abw_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

abw_status from_cuda(cudaError_t e, const char *what, const char *why = nullptr) {
  if (e == cudaSuccess) return ABW_OK;
  if (e == cudaErrorNotSupported) return fail(ABW_ENOTSUP, "%s: %s", what, why ? why : "unsupported shape");
  return fail(ABW_ECUDA, "%s: %s (%s)%s%s", what, cudaGetErrorString(e), cudaGetErrorName(e),
              why ? ": " : "", why ? why : "");
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  const char *name;
  const void *p;
  size_t bytes;
};

bool overlaps(const Range &a, const Range &b) {
  if (a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Null / alignment checks for every buffer, and no output overlapping any
// other buffer.
abw_status check_buffers(const char *op, const Range *in, int nin, const Range *out, int nout) {
  for (int i = 0; i < nin + nout; ++i) {
    const Range &r = i < nin ? in[i] : out[i - nin];
    if (r.bytes == 0) continue;
    if (r.p == nullptr) return fail(ABW_EINVAL, "%s: %s is NULL", op, r.name);
    if (!aligned16(r.p)) return fail(ABW_EINVAL, "%s: %s is not 16-byte aligned", op, r.name);
  }
  for (int i = 0; i < nout; ++i) {
    for (int j = 0; j < nin; ++j)
      if (overlaps(out[i], in[j]))
        return fail(ABW_EINVAL, "%s: output %s overlaps input %s", op, out[i].name, in[j].name);
    for (int j = i + 1; j < nout; ++j)
      if (overlaps(out[i], out[j]))
        return fail(ABW_EINVAL, "%s: outputs %s and %s overlap", op, out[i].name, out[j].name);
  }
  return ABW_OK;
}

size_t dt_size(abw_dtype d) { return d == ABW_BF16 ? 2 : 4; }

}  // namespace

namespace abw {

unsigned long long context_id() {
  // cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points
  // (no link against libcuda).  The id is unique for the life of the
  // process, so a context created after cudaDeviceReset never matches a
  // cached entry of the one it replaced, even at the same handle address.
  using GetCur = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCur get_cur = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<GetCur>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

cudaError_t ensure_dynamic_smem(const void *func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = context_id();
  struct Entry {
    const void *func;
    int dev, bytes;
    unsigned long long ctx;
  };
  static std::mutex mu;
  static Entry seen[64];
  static int nseen = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < nseen; ++i) {
    if (seen[i].func != func || seen[i].dev != dev) continue;
    if (ctx != 0 && seen[i].ctx == ctx && seen[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
      seen[i].bytes = bytes;
      seen[i].ctx = ctx;
    }
    return e;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && nseen < 64) seen[nseen++] = Entry{func, dev, bytes, ctx};
  return e;
}

WaitCtl wait_ctl() {
  WaitCtl w{nullptr, g_wait_limit_ns.load()};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return w;
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_err_addr[dev] == nullptr || ctx == 0 || g_err_ctx[dev] != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_abw_err_word) != cudaSuccess) return w;
    g_err_addr[dev] = static_cast<unsigned int *>(p);
    g_err_ctx[dev] = ctx;
  }
  w.err = g_err_addr[dev];
  return w;
}

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, uint32_t rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                  CUtensorMapSwizzle swizzle, const char **why) {
  using Fn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                          const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                          CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(p);
  });
  if (!fn) {
    if (why) *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dt, rank, const_cast<void *>(base), dims, strides_bytes, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (why) *why = "cuTensorMapEncodeTiled failed";
    return false;
  }
  return true;
}

}  // namespace abw

// ============================================================================
// extern "C" entry points
// ============================================================================
extern "C" {

const char *abw_last_error(void) { return g_last_error.c_str(); }

int abw_version(void) { return 100; }

void abw_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns); }

abw_status abw_device_check(abw_stream stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return from_cuda(e, "abw_device_check");
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "abw_device_check: device error word unavailable");
  unsigned int words[2] = {0, 0};
  e = cudaMemcpyAsync(words, w.err, sizeof(words), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(w.err, 0, sizeof(words), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return from_cuda(e, "abw_device_check");
  const unsigned int word = words[0], site = words[1];
  if (word & (abw::kErrWaitTimeout | abw::kErrSelfTest)) {
    static const char *const kernels[] = {"?", "causal kv", "causal dq", "causal forward", "decode"};
    const unsigned int k = site >> 28;
    return fail(ABW_ETIMEOUT,
                "a device-side bounded wait ran out (error word 0x%x; first in the %s kernel, barrier slot %u, "
                "warp %u, block %u)",
                word, kernels[k < 5 ? k : 0], (site >> 20) & 0xffu, (site >> 16) & 0xfu, site & 0xffffu);
  }
  if (word & abw::kErrSmemAlign)
    return fail(ABW_ECUDA, "a kernel's dynamic shared memory was not 1024-byte aligned; it did no work");
  return ABW_OK;
}

abw_status abw_selftest_wait_timeout(unsigned long long limit_ns, abw_stream stream) {
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "abw_selftest_wait_timeout: device error word unavailable");
  w.limit_ns = limit_ns;
  return from_cuda(abw::launch_selftest_wait(w, reinterpret_cast<cudaStream_t>(stream)),
                   "abw_selftest_wait_timeout");
}

abw_status softmax_bwd(const float *s, const float *dy, float *dx, int rows, int n, abw_stream stream) {
  if (rows < 0 || n < 1) return fail(ABW_EINVAL, "softmax_bwd: rows=%d n=%d (need rows >= 0, n >= 1)", rows, n);
  if (rows == 0) return ABW_OK;
  const size_t bytes = static_cast<size_t>(rows) * n * 4;
  Range in[] = {{"s", s, bytes}, {"dy", dy, bytes}};
  Range out[] = {{"dx", dx, bytes}};
  abw_status st = check_buffers("softmax_bwd", in, 2, out, 1);
  if (st != ABW_OK) return st;
  return from_cuda(abw::launch_softmax_bwd(s, dy, dx, rows, n, reinterpret_cast<cudaStream_t>(stream)),
                   "softmax_bwd");
}

abw_status rope_bwd(const float *dy, float *dx, int B, int T, int H, int D, const float *theta, int pos0,
                    float base, int interleaved, abw_stream stream) {
  if (B < 0 || T < 0 || H < 0) return fail(ABW_EINVAL, "rope_bwd: negative size");
  if (D < 2 || (D & 1)) return fail(ABW_EINVAL, "rope_bwd: D=%d must be even and >= 2", D);
  if (D > 512) return fail(ABW_ENOTSUP, "rope_bwd: D=%d > 512", D);
  if (!theta && !(base > 0.0f)) return fail(ABW_EINVAL, "rope_bwd: base must be > 0 when theta is NULL");
  if (!theta && pos0 < 0) return fail(ABW_EINVAL, "rope_bwd: pos0 must be >= 0");
  if (B == 0 || T == 0 || H == 0) return ABW_OK;
  const size_t bytes = static_cast<size_t>(B) * T * H * D * 4;
  const size_t tbytes = theta ? static_cast<size_t>(B) * T * (D / 2) * 4 : 0;
  Range in[] = {{"dy", dy, bytes}, {"theta", theta, tbytes}};
  if (dx != dy) {
    Range out[] = {{"dx", dx, bytes}};
    abw_status st = check_buffers("rope_bwd", in, 2, out, 1);
    if (st != ABW_OK) return st;
  } else {
    Range out[] = {{"dx", dx, bytes}};
    abw_status st = check_buffers("rope_bwd", in + 1, 1, out, 1);   // in place: only theta must not overlap
    if (st != ABW_OK) return st;
  }
  return from_cuda(abw::launch_rope_bwd(dy, dx, B, T, H, D, theta, pos0, static_cast<double>(base),
                                        interleaved ? 1 : 0, reinterpret_cast<cudaStream_t>(stream)),
                   "rope_bwd");
}

abw_status rmsnorm_bwd(const void *x, abw_dtype x_dtype, const float *gamma, const float *dy, void *dx,
                       abw_dtype dx_dtype, int rows, int n, float eps, abw_stream stream) {
  if (rows < 0 || n < 1) return fail(ABW_EINVAL, "rmsnorm_bwd: rows=%d n=%d", rows, n);
  if ((x_dtype != ABW_F32 && x_dtype != ABW_BF16) || (dx_dtype != ABW_F32 && dx_dtype != ABW_BF16))
    return fail(ABW_EINVAL, "rmsnorm_bwd: bad dtype");
  if (!(eps >= 0.0f)) return fail(ABW_EINVAL, "rmsnorm_bwd: eps must be >= 0");
  if (rows == 0) return ABW_OK;
  const size_t rn = static_cast<size_t>(rows) * n;
  Range in[] = {{"x", x, rn * dt_size(x_dtype)}, {"gamma", gamma, static_cast<size_t>(n) * 4}, {"dy", dy, rn * 4}};
  Range out[] = {{"dx", dx, rn * dt_size(dx_dtype)}};
  abw_status st = check_buffers("rmsnorm_bwd", in, 3, out, 1);
  if (st != ABW_OK) return st;
  return from_cuda(abw::launch_rmsnorm_bwd(x, x_dtype == ABW_BF16, gamma, dy, dx, dx_dtype == ABW_BF16, rows, n,
                                           eps, reinterpret_cast<cudaStream_t>(stream)),
                   "rmsnorm_bwd");
}

abw_status rmsnorm_bwd_dgamma(const void *x, abw_dtype x_dtype, const float *gamma, const float *dy, void *dx,
                              abw_dtype dx_dtype, float *dgamma, int rows, int n, float eps, abw_stream stream) {
  if (rows < 0 || n < 1) return fail(ABW_EINVAL, "rmsnorm_bwd_dgamma: rows=%d n=%d", rows, n);
  if ((x_dtype != ABW_F32 && x_dtype != ABW_BF16) || (dx_dtype != ABW_F32 && dx_dtype != ABW_BF16))
    return fail(ABW_EINVAL, "rmsnorm_bwd_dgamma: bad dtype");
  if (!(eps >= 0.0f)) return fail(ABW_EINVAL, "rmsnorm_bwd_dgamma: eps must be >= 0");
  const size_t rn = static_cast<size_t>(rows) * n;
  Range in[] = {{"x", x, rn * dt_size(x_dtype)},
                {"gamma", gamma, dx ? static_cast<size_t>(n) * 4 : 0},
                {"dy", dy, rn * 4}};
  Range out[] = {{"dgamma", dgamma, static_cast<size_t>(n) * 4}, {"dx", dx, dx ? rn * dt_size(dx_dtype) : 0}};
  abw_status st = check_buffers("rmsnorm_bwd_dgamma", in, 3, out, 2);
  if (st != ABW_OK) return st;
  return from_cuda(abw::launch_rmsnorm_bwd_dgamma(x, x_dtype == ABW_BF16, gamma, dy, dx, dx_dtype == ABW_BF16,
                                                  dgamma, rows, n, eps, reinterpret_cast<cudaStream_t>(stream)),
                   "rmsnorm_bwd_dgamma");
}

abw_status relu2_mul_bwd(const void *gate, const void *up, abw_dtype act_dtype, const float *dh, float *dgate,
                         float *dup, long long n, abw_stream stream) {
  if (n < 0) return fail(ABW_EINVAL, "relu2_mul_bwd: n=%lld", n);
  if (act_dtype != ABW_F32 && act_dtype != ABW_BF16) return fail(ABW_EINVAL, "relu2_mul_bwd: bad dtype");
  if (n == 0) return ABW_OK;
  const size_t nb = static_cast<size_t>(n);
  Range in[] = {{"gate", gate, nb * dt_size(act_dtype)}, {"up", up, nb * dt_size(act_dtype)}, {"dh", dh, nb * 4}};
  Range out[] = {{"dgate", dgate, nb * 4}, {"dup", dup, nb * 4}};
  abw_status st = check_buffers("relu2_mul_bwd", in, 3, out, 2);
  if (st != ABW_OK) return st;
  return from_cuda(abw::launch_relu2_mul_bwd(gate, up, act_dtype == ABW_BF16, dh, dgate, dup, n,
                                             reinterpret_cast<cudaStream_t>(stream)),
                   "relu2_mul_bwd");
}

size_t lora_bwd_workspace_bytes(int rows, int r) {
  if (rows < 0 || r < 1) return 0;
  return abw::lora_workspace_bytes(rows, r);
}

abw_status lora_bwd(const void *x, abw_dtype x_dtype, const float *dy, const float *A, const float *B, float *dA,
                    float *dB, int rows, int n_in, int n_out, int r, float scale, void *workspace,
                    size_t workspace_bytes, abw_stream stream) {
  if (rows < 0 || n_in < 1 || n_out < 1) return fail(ABW_EINVAL, "lora_bwd: rows=%d n_in=%d n_out=%d", rows, n_in, n_out);
  if (x_dtype != ABW_F32 && x_dtype != ABW_BF16) return fail(ABW_EINVAL, "lora_bwd: bad dtype");
  if (r < 1 || r > 16) return fail(ABW_ENOTSUP, "lora_bwd: rank r=%d unsupported (1 <= r <= 16)", r);
  if (n_in % 4 != 0 || n_out % 4 != 0)
    return fail(ABW_ENOTSUP, "lora_bwd: n_in=%d, n_out=%d must be multiples of 4", n_in, n_out);
  if (!(scale == scale)) return fail(ABW_EINVAL, "lora_bwd: scale is NaN");
  const size_t need = abw::lora_workspace_bytes(rows, r);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ABW_EWORKSPACE, "lora_bwd: workspace %zu bytes at %p, need %zu", workspace_bytes, workspace, need);
  const size_t rb = static_cast<size_t>(rows);
  Range in[] = {{"x", x, rb * n_in * dt_size(x_dtype)}, {"dy", dy, rb * n_out * 4},
                {"A", A, static_cast<size_t>(r) * n_in * 4}, {"B", B, static_cast<size_t>(n_out) * r * 4}};
  Range out[] = {{"dA", dA, static_cast<size_t>(r) * n_in * 4}, {"dB", dB, static_cast<size_t>(n_out) * r * 4},
                 {"workspace", workspace, need}};
  abw_status st = check_buffers("lora_bwd", in, 4, out, 3);
  if (st != ABW_OK) return st;
  return from_cuda(abw::launch_lora_bwd(x, x_dtype == ABW_BF16, dy, A, B, dA, dB, rows, n_in, n_out, r, scale,
                                        workspace, reinterpret_cast<cudaStream_t>(stream)),
                   "lora_bwd");
}

abw_status attn_bwd_decode(const float *q, const void *k, const void *v, const float *dout, float *dq, float *dk,
                           float *dv, int B, int Hq, int Hkv, int S, int D, abw_dtype kv_dtype, float scale,
                           float rope_base, int q_pos, abw_stream stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || D < 0) return fail(ABW_EINVAL, "attn_bwd_decode: negative size");
  if (S < 1) return fail(ABW_EINVAL, "attn_bwd_decode: S=%d (softmax over no keys is undefined)", S);
  if (kv_dtype != ABW_F32 && kv_dtype != ABW_BF16) return fail(ABW_EINVAL, "attn_bwd_decode: bad kv dtype");
  if (Hkv == 0 || Hq % Hkv != 0) return fail(ABW_EINVAL, "attn_bwd_decode: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (Hq / Hkv > 8) return fail(ABW_ENOTSUP, "attn_bwd_decode: Hq/Hkv=%d > 8", Hq / Hkv);
  const size_t es = dt_size(kv_dtype);
  if (D < 2 || (D & 1) || (D * es) % 16 != 0 || D * es > 512)
    return fail(ABW_ENOTSUP, "attn_bwd_decode: D=%d unsupported (even, D*sizeof(kv) %% 16 == 0, <= 512 B)", D);
  if (!(scale == scale)) return fail(ABW_EINVAL, "attn_bwd_decode: scale is NaN");
  if (B == 0 || Hq == 0) return ABW_OK;
  const size_t qb = static_cast<size_t>(B) * Hq * D * 4;
  const size_t kvn = static_cast<size_t>(B) * S * Hkv * D;
  Range in[] = {{"q", q, qb}, {"k", k, kvn * es}, {"v", v, kvn * es}, {"dout", dout, qb}};
  Range out[] = {{"dq", dq, qb}, {"dk", dk, kvn * 4}, {"dv", dv, kvn * 4}};
  abw_status st = check_buffers("attn_bwd_decode", in, 4, out, 3);
  if (st != ABW_OK) return st;
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "attn_bwd_decode: no CUDA device");
  const char *why = nullptr;
  const double rb = (rope_base > 0.0f && q_pos >= 0) ? static_cast<double>(rope_base) : 0.0;
  return from_cuda(abw::launch_attn_bwd_decode(q, k, v, dout, dq, dk, dv, B, Hq, Hkv, S, D, kv_dtype == ABW_BF16,
                                               scale, rb, q_pos, w, reinterpret_cast<cudaStream_t>(stream), &why),
                   "attn_bwd_decode", why);
}

abw_status attn_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse, int B, int T, int Hq,
                           int Hkv, int D, float scale, abw_stream stream) {
  if (B < 0 || T < 0 || Hq < 0 || Hkv < 0) return fail(ABW_EINVAL, "attn_fwd_causal: negative size");
  if (Hkv == 0 || Hq % Hkv != 0) return fail(ABW_EINVAL, "attn_fwd_causal: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (D != 128) return fail(ABW_ENOTSUP, "attn_fwd_causal: D=%d unsupported (D == 128)", D);
  if (!(scale == scale)) return fail(ABW_EINVAL, "attn_fwd_causal: scale is NaN");
  if (B == 0 || T == 0 || Hq == 0) return ABW_OK;
  const size_t qn = static_cast<size_t>(B) * T * Hq * D, kn = static_cast<size_t>(B) * T * Hkv * D;
  Range in[] = {{"q", q, qn * 2}, {"k", k, kn * 2}, {"v", v, kn * 2}};
  Range out[] = {{"o", o, qn * 2}, {"lse", lse, static_cast<size_t>(B) * Hq * T * 4}};
  abw_status st = check_buffers("attn_fwd_causal", in, 3, out, 2);
  if (st != ABW_OK) return st;
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "attn_fwd_causal: no CUDA device");
  const char *why = nullptr;
  return from_cuda(abw::launch_attn_fwd_causal(q, k, v, o, lse, B, T, Hq, Hkv, D, scale, w,
                                               reinterpret_cast<cudaStream_t>(stream), &why),
                   "attn_fwd_causal", why);
}

size_t attn_bwd_causal_workspace_bytes(int B, int T, int Hq, int D) {
  if (B < 0 || T < 0 || Hq < 0 || D < 0) return 0;
  return abw::causal_workspace_bytes(B, T, Hq, D);
}

abw_status attn_bwd_causal(const void *q, const void *k, const void *v, const void *o, const void *dout,
                           const float *lse, float *dq, float *dk, float *dv, int B, int T, int Hq, int Hkv, int D,
                           float scale, float rope_base, int pos0, void *workspace, size_t workspace_bytes,
                           abw_stream stream) {
  if (B < 0 || T < 0 || Hq < 0 || Hkv < 0) return fail(ABW_EINVAL, "attn_bwd_causal: negative size");
  if (Hkv == 0 || Hq % Hkv != 0) return fail(ABW_EINVAL, "attn_bwd_causal: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (D != 128) return fail(ABW_ENOTSUP, "attn_bwd_causal: D=%d unsupported (D == 128)", D);
  if (rope_base > 0.0f && pos0 < 0) return fail(ABW_EINVAL, "attn_bwd_causal: pos0 must be >= 0");
  if (!(scale == scale)) return fail(ABW_EINVAL, "attn_bwd_causal: scale is NaN");
  if (B == 0 || T == 0 || Hq == 0) return ABW_OK;
  const size_t need = abw::causal_workspace_bytes(B, T, Hq, D);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ABW_EWORKSPACE, "attn_bwd_causal: workspace %zu bytes at %p, need %zu", workspace_bytes, workspace,
                need);
  const size_t qn = static_cast<size_t>(B) * T * Hq * D, kn = static_cast<size_t>(B) * T * Hkv * D;
  Range in[] = {{"q", q, qn * 2},    {"k", k, kn * 2},
                {"v", v, kn * 2},    {"o", o, qn * 2},
                {"dout", dout, qn * 2}, {"lse", lse, static_cast<size_t>(B) * Hq * T * 4}};
  Range out[] = {{"dq", dq, qn * 4}, {"dk", dk, kn * 4}, {"dv", dv, kn * 4}, {"workspace", workspace, need}};
  abw_status st = check_buffers("attn_bwd_causal", in, 6, out, 4);
  if (st != ABW_OK) return st;
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "attn_bwd_causal: no CUDA device");
  const char *why = nullptr;
  const double rb = rope_base > 0.0f ? static_cast<double>(rope_base) : 0.0;
  return from_cuda(abw::launch_attn_bwd_causal(q, k, v, nullptr, o, dout, lse, dq, dk, dv, B, T, Hq, Hkv, D, scale, rb, pos0,
                                               workspace, workspace_bytes, w,
                                               reinterpret_cast<cudaStream_t>(stream), &why),
                   "attn_bwd_causal", why);
}

abw_status attn_bwd_causal_saved_p(const void *q, const void *k, const void *v, const void *p_attn, const void *o,
                                   const void *dout, float *dq, float *dk, float *dv, int B, int T, int Hq, int Hkv,
                                   int D, float scale, float rope_base, int pos0, void *workspace,
                                   size_t workspace_bytes, abw_stream stream) {
  if (B < 0 || T < 0 || Hq < 0 || Hkv < 0) return fail(ABW_EINVAL, "attn_bwd_causal_saved_p: negative size");
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(ABW_EINVAL, "attn_bwd_causal_saved_p: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (D != 128) return fail(ABW_ENOTSUP, "attn_bwd_causal_saved_p: D=%d unsupported (D == 128)", D);
  if (rope_base > 0.0f && pos0 < 0) return fail(ABW_EINVAL, "attn_bwd_causal_saved_p: pos0 must be >= 0");
  if (!(scale == scale)) return fail(ABW_EINVAL, "attn_bwd_causal_saved_p: scale is NaN");
  if (B == 0 || T == 0 || Hq == 0) return ABW_OK;
  const size_t need = abw::causal_workspace_bytes(B, T, Hq, D);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ABW_EWORKSPACE, "attn_bwd_causal_saved_p: workspace %zu bytes at %p, need %zu", workspace_bytes,
                workspace, need);
  const size_t qn = static_cast<size_t>(B) * T * Hq * D, kn = static_cast<size_t>(B) * T * Hkv * D;
  const size_t pn = static_cast<size_t>(B) * Hq * T * T;
  Range in[] = {{"q", q, qn * 2},    {"k", k, kn * 2},      {"v", v, kn * 2},
                {"p_attn", p_attn, pn * 2}, {"o", o, qn * 2}, {"dout", dout, qn * 2}};
  Range out[] = {{"dq", dq, qn * 4}, {"dk", dk, kn * 4}, {"dv", dv, kn * 4}, {"workspace", workspace, need}};
  abw_status st = check_buffers("attn_bwd_causal_saved_p", in, 6, out, 4);
  if (st != ABW_OK) return st;
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "attn_bwd_causal_saved_p: no CUDA device");
  const char *why = nullptr;
  const double rb = rope_base > 0.0f ? static_cast<double>(rope_base) : 0.0;
  return from_cuda(abw::launch_attn_bwd_causal(q, k, v, p_attn, o, dout, nullptr, dq, dk, dv, B, T, Hq, Hkv, D, scale,
                                               rb, pos0, workspace, workspace_bytes, w,
                                               reinterpret_cast<cudaStream_t>(stream), &why),
                   "attn_bwd_causal_saved_p", why);
}

abw_status attn_bwd_causal_noalloc(const void *q, const void *k, const void *v, const void *o, const void *dout,
                                   const float *lse, float *dq, float *dk, float *dv, int B, int T, int Hq, int Hkv,
                                   int D, float scale, float rope_base, int pos0, abw_stream stream) {
  // Same checks and kernels as attn_bwd_causal; the workspace is the
  // library's built-in device scratch instead of a caller allocation.
  if (B < 0 || T < 0 || Hq < 0 || Hkv < 0) return fail(ABW_EINVAL, "attn_bwd_causal_noalloc: negative size");
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(ABW_EINVAL, "attn_bwd_causal_noalloc: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (D != 128) return fail(ABW_ENOTSUP, "attn_bwd_causal_noalloc: D=%d unsupported (D == 128)", D);
  if (rope_base > 0.0f && pos0 < 0) return fail(ABW_EINVAL, "attn_bwd_causal_noalloc: pos0 must be >= 0");
  if (!(scale == scale)) return fail(ABW_EINVAL, "attn_bwd_causal_noalloc: scale is NaN");
  if (B == 0 || T == 0 || Hq == 0) return ABW_OK;
  const size_t need = abw::causal_workspace_bytes(B, T, Hq, D);
  if (need > abw::kNoAllocScratchBytes)
    return fail(ABW_EWORKSPACE,
                "attn_bwd_causal_noalloc: these sizes need %zu bytes of scratch, more than the built-in %zu "
                "(about B*Hq*T^2 bytes); use attn_bwd_causal with a workspace",
                need, static_cast<size_t>(abw::kNoAllocScratchBytes));
  const size_t qn = static_cast<size_t>(B) * T * Hq * D, kn = static_cast<size_t>(B) * T * Hkv * D;
  Range in[] = {{"q", q, qn * 2},    {"k", k, kn * 2},
                {"v", v, kn * 2},    {"o", o, qn * 2},
                {"dout", dout, qn * 2}, {"lse", lse, static_cast<size_t>(B) * Hq * T * 4}};
  Range out[] = {{"dq", dq, qn * 4}, {"dk", dk, kn * 4}, {"dv", dv, kn * 4}};
  abw_status st = check_buffers("attn_bwd_causal_noalloc", in, 6, out, 3);
  if (st != ABW_OK) return st;
  abw::WaitCtl w = abw::wait_ctl();
  if (!w.err) return fail(ABW_ECUDA, "attn_bwd_causal_noalloc: no CUDA device");
  const char *why = nullptr;
  void *scratch = nullptr;
  cudaError_t e = abw::noalloc_scratch(&scratch, &why);
  if (e != cudaSuccess) return from_cuda(e, "attn_bwd_causal_noalloc", why);
  const double rb = rope_base > 0.0f ? static_cast<double>(rope_base) : 0.0;
  return from_cuda(abw::launch_attn_bwd_causal(q, k, v, nullptr, o, dout, lse, dq, dk, dv, B, T, Hq, Hkv, D, scale, rb, pos0,
                                               scratch, abw::kNoAllocScratchBytes, w,
                                               reinterpret_cast<cudaStream_t>(stream), &why),
                   "attn_bwd_causal_noalloc", why);
}

}  // extern "C"
