/*
 * attn_bwd.h -- C ABI of the attention backward chain for NVIDIA GB300 (sm_103a).
 *
 * The backward (vector-Jacobian product) of each step of a transformer
 * attention layer, as specified by the CPU specs of the
 * "Hesper.Training.VerifiedBackward" API page and the backward chain of
 * Hesper pull request #1 ("Attention backward GPU kernels"), plus the steps
 * around it that the chain runs (the norm's scale gradient, the FFN's gated
 * activation, the LoRA adapter gradients):
 *
 *   softmax_bwd      dx = s * (dy - sum(s * dy))                     (section Softmax)
 *   rope_bwd         dx = R(-theta) dy per rotary pair               (section RoPE)
 *   rmsnorm_bwd      dx = (dy g - x sum(dy g x) / (n rms^2)) / rms   (section RMSNorm)
 *   attn_bwd_decode  one query per sequence over a KV cache, GQA     (section Attention
 *                    (full single-head): attentionBackwardQ/V; Scaled Dot-Product:
 *                    scaledDotBackwardK), with RoPE backward fused on dq
 *   attn_bwd_causal  T queries over T keys under a causal mask, recomputing the
 *                    probabilities from the saved log-sum-exp; RoPE backward fused on
 *                    dq and dk (DaisyChain-Train transformer.js, backward(): dV = A^T dctx,
 *                    dA = dctx V^T, dS = A (dA - sum A dA), dQ = dS K, dK = dS^T Q)
 *   attn_bwd_causal_saved_p  the same from the saved attention weights (PR #1 softmax fix)
 *   attn_fwd_causal  the forward whose O and log-sum-exp attn_bwd_causal consumes
 *   rmsnorm_bwd_dgamma  rmsnorm_bwd plus dgamma = sum_rows dy x / rms
 *   relu2_mul_bwd    dgate = dh up 2 ReLU(gate), dup = dh ReLU(gate)^2  (PR #1, FFN backward)
 *   lora_bwd         dA, dB of y = s B A x                             (PR #1, LoRA backward)
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers (cudaMalloc'd or equivalent), owned by
 *     the caller.  The library never allocates device memory.  Scratch memory,
 *     where an operation needs it, is a caller-provided workspace.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *     call returns without synchronizing.  Outputs are overwritten, never
 *     accumulated into.
 *   - Inputs and outputs must not overlap, except where stated (rope_bwd allows
 *     dx == dy).
 *   - Every tensor is dense and row-major in the layout given, with its base
 *     address 16-byte aligned.
 *   - A non-OK status leaves the outputs unspecified; abw_last_error() returns
 *     a message for the last non-OK status of the calling thread.
 *   - Nothing crosses the ABI as a C++ exception, and nothing aborts.
 *   - Calls neither synchronise nor allocate: the work they enqueue on
 *     `stream` is kernel launches (and, for rmsnorm_bwd_dgamma, a memset of
 *     its output).  The first call of an operation on a device also resolves
 *     per-device state and raises the kernels' shared-memory limits.  So the
 *     calls can be captured into CUDA graphs; make one call of each operation
 *     on the device before capturing.
 *
 * Notation: B batch, Hq query heads, Hkv KV heads (Hq % Hkv == 0; query head
 * h reads KV head h / (Hq / Hkv)), D head dim, S KV length (decode), T
 * sequence length (causal), n row length.  bf16 tensors are IEEE bfloat16
 * (passed as `const void*`).
 */
#ifndef ATTN_BWD_H
#define ATTN_BWD_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ABW_OK = 0,
    ABW_EINVAL = 1,      /* a null pointer, a negative size, a misaligned pointer, overlap */
    ABW_ENOTSUP = 2,     /* valid but unsupported shape (e.g. head dim) */
    ABW_ECUDA = 3,       /* a CUDA launch or runtime error; message has the CUDA string */
    ABW_ETIMEOUT = 4,    /* a device-side bounded wait ran out (see abw_device_check) */
    ABW_EWORKSPACE = 5   /* workspace null or smaller than *_workspace_bytes() */
} abw_status;

typedef enum { ABW_F32 = 0, ABW_BF16 = 1 } abw_dtype;

/* Same type as cudaStream_t. */
typedef struct CUstream_st *abw_stream;

/* Message for the last non-OK status returned to this thread ("" if none). */
const char *abw_last_error(void);

/* ABI version (major * 100 + minor). */
int abw_version(void);

/* Synchronizes `stream`, then reads and clears the library's device error
 * word.  Returns ABW_ETIMEOUT if any kernel since the last check gave up on a
 * bounded wait (it then drained its own copies and returned instead of
 * hanging), ABW_ECUDA on a CUDA error, else ABW_OK. */
abw_status abw_device_check(abw_stream stream);

/* Sets the time limit, in nanoseconds, of every device-side wait of the
 * library's kernels (default 2e9, i.e. 2 s).  For tests. */
void abw_set_wait_limit_ns(unsigned long long ns);

/* Launches one block that waits, with the library's bounded wait, on a
 * shared-memory barrier nothing ever arrives at.  The wait runs out after
 * `limit_ns`, the kernel records the timeout in the device error word and
 * returns, so abw_device_check() then reports ABW_ETIMEOUT.  Exercises the
 * failure path of the bounded waits without faulting or hanging the GPU. */
abw_status abw_selftest_wait_timeout(unsigned long long limit_ns, abw_stream stream);

/*
 * softmax_bwd -- softmaxBackward ("Hesper.Training.VerifiedBackward", section
 * Softmax): dx_i = s_i (dy_i - sum_j s_j dy_j), row by row.
 *   s   [rows][n] f32  probabilities (the softmax output saved by the forward)
 *   dy  [rows][n] f32  upstream gradient
 *   dx  [rows][n] f32  output
 * rows >= 0, n >= 1.
 */
abw_status softmax_bwd(const float *s, const float *dy, float *dx, int rows, int n,
                       abw_stream stream);

/*
 * rope_bwd -- ropeBackward (section RoPE): every rotary pair (y0, y1) of dy is
 * rotated by -theta: (y0 cos t + y1 sin t, -y0 sin t + y1 cos t).
 *   dy, dx [B][T][H][D] f32 (dx == dy allowed: in place)
 *   theta  [B*T][D/2] f32 explicit angles, or NULL: theta(b, t, i) =
 *          (pos0 + t) * base^(-2i/D) with the angle formed in double precision
 *   interleaved  1: pairs (2i, 2i+1);  0: pairs (i, i + D/2)
 * D even, 2 <= D <= 512; base > 0 when theta is NULL.
 */
abw_status rope_bwd(const float *dy, float *dx, int B, int T, int H, int D,
                    const float *theta, int pos0, float base, int interleaved,
                    abw_stream stream);

/*
 * rmsnorm_bwd -- rmsNormBackward (section RMSNorm), per row of length n:
 *   rms = sqrt(sum_j x_j^2 / n + eps),  c = sum_j dy_j g_j x_j,
 *   dx_i = (dy_i g_i - x_i c / (n rms^2)) / rms.
 *   x     [rows][n] f32 or bf16 (x_dtype)   the saved forward input
 *   gamma [n] f32
 *   dy    [rows][n] f32
 *   dx    [rows][n] f32 or bf16 (dx_dtype)
 * Both row sums are taken in one pass with fp32 accumulation.
 */
abw_status rmsnorm_bwd(const void *x, abw_dtype x_dtype, const float *gamma,
                       const float *dy, void *dx, abw_dtype dx_dtype, int rows, int n,
                       float eps, abw_stream stream);

/*
 * rmsnorm_bwd_dgamma -- rmsNormBackward (section RMSNorm) together with the
 * gradient of the norm's scale.  The page states dx only; the forward
 * y_i = gamma_i x_i / rms is linear in gamma, so its scale gradient is
 *   dgamma_i = sum over rows of dy_i x_i / rms.
 *   x, gamma, dy, dx as rmsnorm_bwd; dx may be NULL (then gamma may be NULL
 *   too, and only dgamma is produced)
 *   dgamma [n] f32, overwritten (the call zeroes it, then adds every row)
 * The row sums are fp32; the order in which the rows' terms are added into
 * dgamma varies from call to call (reductions in L2), so results agree to
 * fp32 rounding, not bit for bit.
 */
abw_status rmsnorm_bwd_dgamma(const void *x, abw_dtype x_dtype, const float *gamma, const float *dy,
                              void *dx, abw_dtype dx_dtype, float *dgamma, int rows, int n, float eps,
                              abw_stream stream);

/*
 * relu2_mul_bwd -- backward of the FFN's gated activation
 * hidden = ReLU(gate)^2 * up (Hesper pull request #1, the FFN-backward
 * commit's "ReLU^2 x Mul backward"), element by element:
 *   dgate = dh * up * 2 ReLU(gate),   dup = dh * ReLU(gate)^2.
 *   gate, up  [n] act_dtype (f32 or bf16)  saved forward activations
 *   dh        [n] f32                      upstream gradient of hidden
 *   dgate, dup [n] f32                     outputs
 * n >= 0 (any layout: the operation is element-wise).
 */
abw_status relu2_mul_bwd(const void *gate, const void *up, abw_dtype act_dtype, const float *dh,
                         float *dgate, float *dup, long long n, abw_stream stream);

/*
 * lora_bwd -- parameter gradients of a rank-r LoRA adapter on a projection
 * (Hesper pull request #1: the backward chain ends "RoPE backward -> dQ ->
 * LoRA backward", the adapter's input being the layer's saved normed
 * activations, and its input gradient feeds only dA and dB).  The adapter
 * adds y = scale * B (A x) per row; with h = x A^T:
 *   dB = scale dy^T h,   dA = (scale dy B)^T x      (sums over the rows)
 *   x   [rows][n_in] f32 or bf16 (x_dtype)   saved adapter input
 *   dy  [rows][n_out] f32                    gradient of the projection's output
 *                                            (e.g. dq as [tokens][Hq*D])
 *   A   [r][n_in] f32;   B [n_out][r] f32
 *   dA  [r][n_in] f32;   dB [n_out][r] f32   overwritten
 *   workspace  device memory of at least lora_bwd_workspace_bytes(rows, r)
 * Supported: 1 <= r <= 16; n_in and n_out multiples of 4.  Sums over rows are
 * fp32, added in an order that varies from call to call.
 */
size_t lora_bwd_workspace_bytes(int rows, int r);
abw_status lora_bwd(const void *x, abw_dtype x_dtype, const float *dy, const float *A, const float *B,
                    float *dA, float *dB, int rows, int n_in, int n_out, int r, float scale,
                    void *workspace, size_t workspace_bytes, abw_stream stream);

/*
 * attn_bwd_decode -- one query per sequence against a KV cache (attentionBackwardQ,
 * attentionBackwardV, scaledDotBackwardK of section Attention / Scaled Dot-Product),
 * with grouped KV heads:
 *   s_hj = scale q_h . K_j,  P_h = softmax_j(s_h),  dP_hj = dout_h . V_j,
 *   delta_h = sum_j P_hj dP_hj,  dS_hj = P_hj (dP_hj - delta_h),
 *   dq_h = scale sum_j dS_hj K_j        (then R(-theta(q_pos)) when RoPE is on)
 *   dK_j = scale sum_{h in group} dS_hj q_h,   dV_j = sum_{h in group} P_hj dout_h
 *   q, dout, dq [B][Hq][D] f32
 *   k, v        [B][S][Hkv][D] kv_dtype (f32 or bf16); dk, dv the same shape, f32
 *   rope_base > 0 and q_pos >= 0: RoPE backward at position q_pos on dq
 *   (pairs (2i, 2i+1), theta_i = q_pos base^(-2i/D)); otherwise none.
 * Supported: S >= 1; Hq % Hkv == 0 with Hq / Hkv <= 8; D even with
 * D * sizeof(kv) a multiple of 16 bytes and at most 512 bytes.
 */
abw_status attn_bwd_decode(const float *q, const void *k, const void *v, const float *dout,
                           float *dq, float *dk, float *dv,
                           int B, int Hq, int Hkv, int S, int D, abw_dtype kv_dtype,
                           float scale, float rope_base, int q_pos, abw_stream stream);

/*
 * attn_fwd_causal -- the causal attention forward that produces the
 * activations attn_bwd_causal consumes: online-softmax attention (Hesper
 * pull request #1, FlashAttention commits: flashAttentionSpec, equal to the
 * three-step standardAttention) under the causal mask (keys j <= query i):
 *   s_ij = scale q_i . k_j,  lse_i = log sum_{j<=i} exp(s_ij),
 *   o_i = sum_{j<=i} exp(s_ij - lse_i) v_j
 *   q [B][T][Hq][D] bf16;  k, v [B][T][Hkv][D] bf16 (query head h reads KV
 *   head h / (Hq / Hkv))
 *   o [B][T][Hq][D] bf16 (rounded from fp32);  lse [B][Hq][T] f32, natural log
 * The probabilities enter the o product rounded to bf16; sums are fp32.
 * Supported: D == 128; T >= 1; Hq % Hkv == 0.
 */
abw_status attn_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int T, int Hq, int Hkv, int D, float scale, abw_stream stream);

/*
 * attn_bwd_causal_workspace_bytes -- workspace size attn_bwd_causal needs for
 * these sizes, with Tp = T rounded up to 128 and nb = Tp / 128: delta and
 * lse * log2(e), each f32 [B][Hq][Tp]; the RoPE table [T][D/2] of
 * scale * (cos, sin); the bf16 dS tiles of the causal half, 16 KB per
 * (128-key block, 64-query block) pair, B * Hq * (nb^2 + nb) of them; and
 * 256-byte alignment slack.  About B * Hq * Tp * (Tp + 136) bytes.
 */
size_t attn_bwd_causal_workspace_bytes(int B, int T, int Hq, int D);

/*
 * attn_bwd_causal -- causal multi-query attention backward (keys j <= query i).
 * The probabilities are recomputed from the saved log-sum-exp:
 *   P_ij = exp(scale q_i . k_j - lse_i) for j <= i, else 0,
 *   dP = dout V^T,  delta_i = dout_i . o_i (= sum_j P_ij dP_ij),
 *   dS = P (dP - delta),  dq = scale dS K,  dk = scale dS^T Q,  dv = P^T dout,
 * dk and dv summed over the query heads that share a KV head.  With
 * rope_base > 0, RoPE backward R(-theta(pos0 + t)) (pairs (2i, 2i+1),
 * theta_i = (pos0 + t) base^(-2i/D)) is applied to dq and dk.
 *   q, o, dout [B][T][Hq][D] bf16;   k, v [B][T][Hkv][D] bf16
 *   lse        [B][Hq][T] f32 natural-log log-sum-exp of the scaled scores
 *   dq [B][T][Hq][D] f32;  dk, dv [B][T][Hkv][D] f32
 *   workspace  device memory of at least attn_bwd_causal_workspace_bytes()
 * Supported: D == 128; T >= 1; Hq % Hkv == 0.
 */
abw_status attn_bwd_causal(const void *q, const void *k, const void *v, const void *o,
                           const void *dout, const float *lse,
                           float *dq, float *dk, float *dv,
                           int B, int T, int Hq, int Hkv, int D, float scale,
                           float rope_base, int pos0,
                           void *workspace, size_t workspace_bytes, abw_stream stream);

/*
 * attn_bwd_causal_saved_p -- attn_bwd_causal reading the attention weights
 * the forward saved instead of recomputing them from the log-sum-exp: the
 * form of Hesper pull request #1's softmax-backward fix ("save per-layer
 * attention weights ... use saved attnBuf": dScores = attn (dAttn -
 * sum attn dAttn)) and of transformer.js backward(), which reads the cached
 * attention A.
 *   p_attn [B][Hq][T][T] bf16  the softmax output, row = query i, column =
 *          key j; entries with j > i are not read (the causal mask makes
 *          them 0)
 *   o      [B][T][Hq][D] bf16  the forward's output, for
 *          delta_i = sum_j P_ij dP_ij = dout_i . o_i (the identity holds
 *          because o = P v)
 *   everything else as attn_bwd_causal (no lse), with the same workspace
 *   size (attn_bwd_causal_workspace_bytes).
 */
abw_status attn_bwd_causal_saved_p(const void *q, const void *k, const void *v, const void *p_attn,
                                   const void *o, const void *dout, float *dq, float *dk, float *dv,
                                   int B, int T, int Hq, int Hkv, int D, float scale,
                                   float rope_base, int pos0, void *workspace, size_t workspace_bytes,
                                   abw_stream stream);

/*
 * attn_bwd_causal_noalloc -- attn_bwd_causal for callers that cannot allocate
 * device memory: no workspace argument, and the call allocates nothing.  (The
 * pages have no counterpart; this is an interface convenience.)
 *
 * Who needs it: code that runs where cudaMalloc is off limits -- inside a
 * CUDA stream capture or a custom allocator's callback, in a process whose
 * device memory is owned by another framework's pool, or in a plugin given
 * only the tensors it works on.  Such a caller passes the inputs and outputs
 * as for attn_bwd_causal; the scratch comes from a 32 MiB array in the
 * library's device image (a file-scope __device__ variable), which every GPU
 * that loads the library keeps until the process exits.
 *
 *   Arguments, layouts and results: as attn_bwd_causal.
 *   Limit: the sizes must need at most 32 MiB of scratch
 *   (attn_bwd_causal_workspace_bytes(B, T, Hq, D) <= 33554432, roughly
 *   B * Hq * T^2 < 32 MiB, e.g. B=2, T=512, Hq=20 needs about 13 MB); larger
 *   sizes return ABW_EWORKSPACE without launching anything.
 *   First call on a device: looks up the array's device address on that
 *   device (cudaGetSymbolAddress) and caches it; make that first call before
 *   any stream capture that should contain it.
 *   Sharing: every call on a device uses the same array.  Each call writes
 *   every part of it that it later reads, so consecutive calls are
 *   independent -- but calls that overlap on the GPU (different streams, no
 *   ordering between them) race on the array.
 */
abw_status attn_bwd_causal_noalloc(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse,
                                   float *dq, float *dk, float *dv,
                                   int B, int T, int Hq, int Hkv, int D, float scale,
                                   float rope_base, int pos0, abw_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H */
