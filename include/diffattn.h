/*
 * diffattn.h -- C ABI of the GB300 (sm_103a) multi-head differential-attention
 * forward library (libdiffattn.so).
 *
 * The operator, as the pages on the Differential Transformer state it:
 *
 *   DiffAttn(Q1,Q2,K1,K2,V) = (softmax(Q1 K1^T / sqrt d) - lambda softmax(Q2 K2^T / sqrt d)) V
 *
 * ("Differential Transformer", ultralytics.com glossary, section "How
 * differential attention works", with its worked example; "Differential
 * Transformer V2 (DIFF V2) 기술적 혁신 분석", section "차등 어텐션 메커니즘의 핵심 원리").
 *
 * Conventions shared by every entry point
 *  - Layout is BSHD, contiguous, row-major: element (b, t, h, c) of a tensor
 *    [B, n, H, W] sits at ((b*n + t)*H + h)*W + c.
 *  - Every pointer argument except those documented as host values is a
 *    DEVICE pointer owned by the caller.  The library allocates no device
 *    memory and keeps no pointer after the call returns.
 *  - All entry points are asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL means the legacy default stream), except
 *    diffattn_lambda_init (pure host) and diffattn_device_status (syncs).
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a non-zero status and leaves all buffers untouched.
 *    diffattn_last_error() then returns a message (thread-local).
 *  - Kernels never trap.  Every wait inside a kernel is bounded (2e9 SM clock
 *    cycles, about one second); a wait that runs out records
 *    DIFFATTN_ERR_TIMEOUT in a device status word that diffattn_device_status()
 *    reads and clears.
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DIFFATTN_OK = 0,
    DIFFATTN_ERR_NULL = 1,        /* a required pointer is NULL                      */
    DIFFATTN_ERR_SHAPE = 2,       /* a size is negative, zero where it may not be,
                                     or inconsistent (e.g. Hq not a multiple of Hkv) */
    DIFFATTN_ERR_ALIGN = 3,       /* a bf16 tensor is not 16-byte aligned            */
    DIFFATTN_ERR_DTYPE = 4,       /* unknown dtype code                              */
    DIFFATTN_ERR_UNSUPPORTED = 5, /* valid but not implemented (e.g. bf16 with d not
                                     in {64, 128})                                   */
    DIFFATTN_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed               */
    DIFFATTN_ERR_TIMEOUT = 7,     /* a bounded in-kernel wait ran out                */
    DIFFATTN_ERR_BOUNDS = 8       /* bounds-check build only: an index check in a
                                     kernel failed and the access was skipped       */
} diffattn_status;

typedef enum {
    DIFFATTN_F32 = 0,  /* fp32 in, fp32 out, fp32 arithmetic (CUDA-core kernel)         */
    DIFFATTN_BF16 = 1  /* bf16 in, bf16 out; fp32 accumulation on tcgen05 tensor cores */
} diffattn_dtype;

/*
 * lambda_init for the 1-based layer index l: 0.8 - 0.6 * exp(-0.3 * (l - 1)).
 * Differential Transformer news article (esgcw.com.cn), section "差分注意力";
 * DIFF V2 analysis page, section "DIFF V1의 한계와 문제점".
 * Pure host function.  Returns NaN for l < 1.  A constant lambda_init (the
 * article's alternative, e.g. 0.8 in every layer) is passed directly as a
 * float to the calls below.
 */
float diffattn_lambda_init(int layer_index);

/*
 * lambda = exp(<lq1, lk1>) - exp(<lq2, lk2>) + lambda_init, computed on the
 * device in fp32 by one warp (the re-parameterisation of the learnable scalar;
 * news article section "差分注意力", DIFF V2 analysis page section 5 of
 * "DIFF V2의 핵심 기술적 혁신").
 *   lq1, lk1, lq2, lk2 : device fp32 vectors of length `dim` (dim >= 1).
 *   lambda_out         : device fp32 scalar, written by the kernel.  Pass it to
 *                        diffattn_forward on the same stream; no host sync.
 * Errors: NULL pointers -> ERR_NULL; dim < 1 -> ERR_SHAPE.
 */
diffattn_status lambda_reparam(const float* lq1, const float* lk1, const float* lq2,
                               const float* lk2, int dim, float lambda_init,
                               float* lambda_out, void* stream);

/*
 * Multi-head DIFF V1 forward with the per-head RMSNorm (the pages' "GroupNorm")
 * scaled by the fixed multiplier (1 - lambda_init):
 *
 *   O   = (softmax(Q1 K1^T / sqrt d) - lambda softmax(Q2 K2^T / sqrt d)) V   per (b, h)
 *   out = (1 - lambda_init) * gamma * O / sqrt(mean_c O^2 + eps)             per (b, t, h)
 *
 * (news article section "差分注意力": multi-head, lambda shared across the heads
 * of a layer, LN = RMSNorm per head, concat along channels.)
 *   dt          : DIFFATTN_BF16 or DIFFATTN_F32; q*, k*, v and out share it.
 *   B, H, n, d  : batch, diff heads, tokens, per-map query/key width.  The
 *                 value width is 2d.  bf16 needs d in {64, 128}; f32 needs
 *                 d in [1, 128].  n = 0 or B = 0 or H = 0 is a no-op.
 *   q1, q2, k1, k2 : [B, n, H, d];  v, out : [B, n, H, 2d].
 *   lambda      : device fp32 scalar (e.g. written by lambda_reparam).
 *   lambda_init : host float, the fixed norm multiplier is (1 - lambda_init).
 *   gamma       : device fp32 [2d] RMSNorm weight shared by all heads, or NULL
 *                 for all ones.
 *   eps         : RMSNorm epsilon; eps <= 0 selects 1e-5.
 *   causal      : non-zero: query t sees key j iff j <= t.
 * Errors: NULL -> ERR_NULL; bad sizes -> ERR_SHAPE; bf16 pointers not 16-byte
 * aligned -> ERR_ALIGN; unsupported d -> ERR_UNSUPPORTED; launch failure ->
 * ERR_CUDA.  `out` may not alias an input.
 */
diffattn_status diffattn_forward(diffattn_dtype dt, int B, int H, int n, int d,
                                 const void* q1, const void* q2, const void* k1,
                                 const void* k2, const void* v, const float* lambda,
                                 float lambda_init, const float* gamma, float eps,
                                 int causal, void* out, void* stream);

/*
 * diffattn_forward with the queries and keys in FP8: the low-bit attention
 * that the "Differential Transformer" glossary page (section on the reported
 * benefits) motivates by DIFF's smaller activation outliers, applied to the
 * score products Q_r K_r^T on the tensor cores' e4m3 path (kind::f8f6f4,
 * twice the bf16 rate); the values, P.V, the combine and the norm stay as in
 * the bf16 forward.
 *   q1, q2, k1, k2 : [B, n, H, d] device arrays of e4m3 bytes (OCP FP8 E4M3,
 *                    "fn") holding Q_r / q_scale_r and K_r / k_scale_r, one
 *                    scale per tensor (how they were quantised is the
 *                    caller's; e.g. amax / 448).
 *   q1_scale, q2_scale, k1_scale, k2_scale : finite and positive, else ERR_SHAPE.
 *   v, out, lambda, lambda_init, gamma, eps, causal : as for diffattn_forward (bf16).
 * The result is diffattn_forward's for Q_r = q_scale_r e4m3(q_r) and
 * K_r = k_scale_r e4m3(k_r): every e4m3 product is exact in the fp32
 * accumulator and each map's two scales fold into its softmax exponent.
 * d = 128 (one 128-byte row a box) or d = 64 with H >= 2 (a 128-byte box
 * covers a head's 64-byte row and the next head's, whose bytes the MMAs do
 * not read; the last head's box ends in zeros), else ERR_UNSUPPORTED.
 * Errors otherwise as for diffattn_forward.
 */
diffattn_status diffattn_forward_fp8qk(int B, int H, int n, int d, const void* q1, const void* q2,
                                       const void* k1, const void* k2, float q1_scale,
                                       float q2_scale, float k1_scale, float k2_scale, const void* v,
                                       const float* lambda, float lambda_init, const float* gamma,
                                       float eps, int causal, void* out, void* stream);

/*
 * diffattn_v2_forward with the queries and keys in FP8 (e4m3), one
 * dequantisation scale per tensor: the low-bit score products that the
 * "Differential Transformer" glossary page (section on the reported
 * benefits) motivates by the smaller activation outliers, as in
 * diffattn_forward_fp8qk, applied to the DIFF V2 operator (DIFF V2 analysis page, "2. 커스텀 커널
 * 제거", "GQA와의 호환성").  The two query heads of a pair score against
 * their shared key head with kind::f8f6f4 MMAs (fp32 accumulation); P and V
 * stay bf16.
 *   q : [B, n, Hq, d] device bytes (e4m3 codes) holding q / q_scale;
 *   k : [B, n, Hkv, d] device bytes holding k / k_scale;
 *   q_scale, k_scale : finite and positive, else ERR_SHAPE.
 *   v, lam_logits, sb, st, softmax_scale, causal, out : as for
 *         diffattn_v2_forward with dt = DIFFATTN_BF16.
 * The result is diffattn_v2_forward's for Q = q_scale e4m3(q) and
 * K = k_scale e4m3(k).  d = 128 only, else ERR_UNSUPPORTED; errors otherwise
 * as for diffattn_v2_forward.
 */
diffattn_status diffattn_v2_forward_fp8qk(int B, int Hq, int Hkv, int n, int d, const void* q, const void* k,
                                          float q_scale, float k_scale, const void* v, const float* lam_logits,
                                          long long sb, long long st, float softmax_scale, int causal,
                                          void* out, void* stream);

/*
 * diffattn_forward on inputs and output in HOST memory: the call copies the
 * inputs in, runs the forward and copies the output back, pipelined over
 * chunks (the copy of chunk c + 1 in, the forward of chunk c and the copy of
 * chunk c - 1 out overlap on internal copy streams).  The chunks are batch
 * entries, except for a causal bf16 forward of fewer than four sequences:
 * then they are ranges of 128-token tiles of every sequence (the queries of
 * a range see only keys copied in by it and the ranges before it), whose
 * forwards alternate between `stream` and an internal compute stream; at
 * most eight chunks.  The output is identical to diffattn_forward's either
 * way.  Same operation, layouts, arguments and errors as diffattn_forward,
 * except:
 *   q1, q2, k1, k2, v (in), out : host memory, [B, n, H, d] / [B, n, H, 2d];
 *                 page-locked (cudaHostAlloc / cudaHostRegister) for the
 *                 copies to be asynchronous; pageable memory still works
 *                 but each copy then blocks the host.
 *   lambda, gamma : device memory as for diffattn_forward (parameters of the
 *                 layer, resident on the device).
 *   workspace   : device memory the caller owns, at least
 *                 diffattn_forward_host_workspace(dt, B, H, n, d) bytes,
 *                 256-byte aligned; it holds the device copies of the inputs
 *                 and of the output (the library allocates nothing per call).
 * Asynchronous on `stream`: the output in host memory is complete when the
 * stream's work up to this call is; the workspace and the host buffers must
 * not be touched before that.  A smaller workspace -> ERR_SHAPE; an
 * unaligned workspace -> ERR_ALIGN.
 */
size_t diffattn_forward_host_workspace(diffattn_dtype dt, int B, int H, int n, int d);

diffattn_status diffattn_forward_host(diffattn_dtype dt, int B, int H, int n, int d,
                                      const void* q1, const void* q2, const void* k1,
                                      const void* k2, const void* v, const float* lambda,
                                      float lambda_init, const float* gamma, float eps,
                                      int causal, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * DIFF V1 decode step: one new token per sequence over a key/value cache
 * ("Differential Transformer" glossary page, "How differential attention
 * works"; news article section "差分注意力" for the per-head RMSNorm):
 *
 *   O   = (softmax(q1 K1^T / sqrt d) - lambda softmax(q2 K2^T / sqrt d)) V   per (b, h), keys j < lens[b]
 *   out = (1 - lambda_init) * gamma * O / sqrt(mean_c O^2 + eps)
 *
 * i.e. diffattn_forward's last row of a causal sequence whose keys and
 * values (the new token's included) are already in the cache.
 *   dt          : DIFFATTN_BF16 (d in {64, 128}); other types -> ERR_UNSUPPORTED.
 *   q1, q2      : [B, H, d] device, the new token's queries.
 *   k1, k2      : [B, n, H, d] device key caches; v : [B, n, H, 2d] value cache.
 *   lens        : device int32 [B], keys visible to each sequence, clamped to
 *                 [0, n]; NULL: n for every sequence.  A sequence with no
 *                 visible key gets an all-zero output.
 *   lambda, lambda_init, gamma, eps : as for diffattn_forward.
 *   out         : [B, H, 2d] device.
 *   workspace   : NULL, or device memory the caller owns of at least
 *                 diffattn_decode_workspace(B, H, d) bytes (4-byte aligned).
 *                 With it, when there are too few (b, h) pairs to fill the GPU,
 *                 several thread-block clusters share a pair's keys and a second
 *                 small kernel merges their states; results are the same up
 *                 to fp32 rounding order.  Without it nothing is allocated.
 *                 A non-NULL workspace smaller than that -> ERR_SHAPE; one
 *                 not 4-byte aligned -> ERR_ALIGN.
 * Memory-bound: K1, K2 and V are read once (V for both maps); asynchronous
 * on `stream`.  Errors as for diffattn_forward.
 */
size_t diffattn_decode_workspace(int B, int H, int d);

diffattn_status diffattn_decode(diffattn_dtype dt, int B, int H, int n, int d, const void* q1,
                                const void* q2, const void* k1, const void* k2, const void* v,
                                const int* lens, const float* lambda, float lambda_init,
                                const float* gamma, float eps, void* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * diffattn_decode for callers that cannot allocate device memory.  The paper
 * has no counterpart: this is a deployment variant of the decode step above.
 *
 * Who needs it: the split form of diffattn_decode (several clusters share
 * the keys of one (batch, head) pair when there are too few pairs to fill
 * the GPU) keeps partial softmax states in a workspace that the caller
 * allocates.  Some callers cannot: a plugin inside a host framework that
 * owns every byte of device memory, a plain C caller with no device
 * allocator at hand, or a serving loop that forbids cudaMalloc after
 * start-up because it can synchronise the device and take milliseconds.
 * This call takes no workspace; it uses a fixed scratch array compiled
 * into the library instead, and calls no cudaMalloc, cudaFree or any
 * other allocating routine.
 *
 * Same operation, arguments, layouts and errors as diffattn_decode with a
 * workspace (bf16, d in {64, 128}), and the same result: the pairs are split
 * over clusters exactly as diffattn_decode splits them when given one.
 *
 * Limits and sharing:
 *  - the scratch holds 4 MiB (4194304 bytes) on every GPU that loads the
 *    library, until the process exits;
 *  - a call needs diffattn_decode_workspace(B, H, d) <= 4194304, i.e.
 *    B*H <= 504 pairs at d = 64 and B*H <= 254 at d = 128; a larger batch is
 *    rejected with ERR_SHAPE before anything is launched (such a batch fills
 *    the GPU without splitting: call diffattn_decode with a NULL workspace,
 *    which also allocates nothing);
 *  - the first call on a device looks up the scratch's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture;
 *  - every call on a device uses the same scratch, and each call writes
 *    every value it later reads (nothing needs clearing between calls).
 *    Calls whose kernels can overlap on the GPU (other streams, other host
 *    threads) race on the scratch and corrupt each other's results:
 *    serialise them on one stream.
 */
diffattn_status diffattn_decode_noalloc(diffattn_dtype dt, int B, int H, int n, int d,
                                        const void* q1, const void* q2, const void* k1,
                                        const void* k2, const void* v, const int* lens,
                                        const float* lambda, float lambda_init,
                                        const float* gamma, float eps, void* out,
                                        void* stream);

/*
 * diffattn_decode with the key caches in FP8 (the low-bit attention that the
 * "Differential Transformer" glossary page motivates by DIFF's smaller
 * activation outliers): k1, k2 are [B, n, H, d] device arrays of e4m3 bytes
 * (OCP FP8 E4M3, "fn": no infinities, 0x7f / 0xff are NaN) holding
 * K_r / k_scale_r, one scale per tensor; the kernel computes exactly what
 * diffattn_decode computes for the bf16 caches K_r = k_scale_r * e4m3(k_r)
 * (fp32 arithmetic; each e4m3 value is converted exactly).  q1, q2, v, out,
 * lens, lambda, gamma, workspace: as for diffattn_decode (bf16, d in {64, 128};
 * workspace size diffattn_decode_workspace).  k1_scale, k2_scale: finite and
 * positive, else ERR_SHAPE.  6 d bytes read a key instead of 8 d.
 */
diffattn_status diffattn_decode_fp8k(int B, int H, int n, int d, const void* q1, const void* q2,
                                     const void* k1, const void* k2, float k1_scale,
                                     float k2_scale, const void* v, const int* lens,
                                     const float* lambda, float lambda_init, const float* gamma,
                                     float eps, void* out, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * DIFF V2 decode step: one new token per sequence over a key/value cache
 * (DIFF V2 analysis page, sections "2. 커스텀 커널 제거", "5. 간소화된 λ
 * 매개변수화" and "GQA와의 호환성"): per head pair g of sequence b,
 *
 *   out_g = softmax(q_{2g} K_kv^T * scale) V_kv - sigmoid(logit[b*sb + g]) softmax(q_{2g+1} K_kv^T * scale) V_kv
 *
 * over the keys j < lens[b], kv = 2g / (Hq / Hkv); no norm.  The last row of
 * diffattn_v2_forward for a causal sequence whose keys and values (the new
 * token's included) are in the cache; each K/V tile is read once for both
 * query heads of a pair.
 *   dt          : DIFFATTN_BF16 with d = 128; other types / widths -> ERR_UNSUPPORTED.
 *   q           : [B, Hq, d] device; k, v : [B, n, Hkv, d] device caches.
 *   Hq even, Hq % Hkv == 0, (Hq / Hkv) even.
 *   lens        : device int32 [B] (clamped to [0, n]) or NULL (n); a
 *                 sequence with no visible key gets zeros.
 *   lam_logits  : device fp32, the logit of pair g of sequence b at
 *                 lam_logits[b*sb + g] (sb = 0: one logit per pair).
 *   softmax_scale : <= 0 selects 1/sqrt(d).
 *   out         : [B, Hq/2, d] device.
 *   workspace   : NULL, or at least diffattn_v2_decode_workspace(B, Hq, d)
 *                 bytes of device memory, as for diffattn_decode (smaller ->
 *                 ERR_SHAPE, not 4-byte aligned -> ERR_ALIGN).
 * Asynchronous on `stream`.  Errors as for diffattn_forward.
 */
size_t diffattn_v2_decode_workspace(int B, int Hq, int d);

diffattn_status diffattn_v2_decode(diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d,
                                   const void* q, const void* k, const void* v, const int* lens,
                                   const float* lam_logits, long long sb, float softmax_scale,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * diffattn_v2_decode with the key cache in FP8: k is a [B, n, Hkv, d] device
 * array of e4m3 bytes holding K / k_scale (k_scale finite and positive, else
 * ERR_SHAPE); the result is diffattn_v2_decode's for K = k_scale * e4m3(k).
 * Everything else as for diffattn_v2_decode (bf16, d = 128; workspace size
 * diffattn_v2_decode_workspace).  3 d bytes read a key instead of 4 d.
 */
diffattn_status diffattn_v2_decode_fp8k(int B, int Hq, int Hkv, int n, int d, const void* q,
                                        const void* k, float k_scale, const void* v,
                                        const int* lens, const float* lam_logits, long long sb,
                                        float softmax_scale, void* out, void* workspace,
                                        size_t workspace_bytes, void* stream);

/*
 * DIFF V2 forward (DIFF V2 analysis page, sections "2. 커스텀 커널 제거",
 * "5. 간소화된 λ 매개변수화" and "GQA와의 호환성"): 2h query heads over h KV
 * heads, grouped-query attention, each even/odd pair of query heads inside
 * one KV group differenced with a sigmoid lambda, no norm:
 *
 *   A_j   = softmax(q_j K_kv(j)^T * scale) V_kv(j),   kv(j) = j / (Hq / Hkv)
 *   out_g = A_{2g} - sigmoid(logit[b, t, g]) * A_{2g+1},   g < Hq/2
 *
 *   q   : [B, n, Hq, d];  k, v : [B, n, Hkv, d];  out : [B, n, Hq/2, d].
 *   Hq even, Hq % Hkv == 0 and (Hq / Hkv) even (so a pair never straddles
 *   two KV heads).  bf16 needs d = 128; f32 needs d in [1, 128].
 *   lam_logits : device fp32; the logit of (b, t, g) is
 *                lam_logits[b*sb + t*st + g]  (sb = st = 0: one logit per pair).
 *   softmax_scale : <= 0 selects 1/sqrt(d).
 * Errors as for diffattn_forward.
 */
diffattn_status diffattn_v2_forward(diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d,
                                    const void* q, const void* k, const void* v,
                                    const float* lam_logits, long long sb, long long st,
                                    float softmax_scale, int causal, void* out,
                                    void* stream);

/*
 * Projection on the tensor cores: c = a w^T, bf16 operands, fp32 accumulation,
 * bf16 result rounded once to nearest.  The projections X W^Q, X W^K, X W^V
 * (and X W^lambda for DIFF V2) and Concat(heads) W^O around the operator
 * (news article section "差分注意力"; see diffattn_layer_forward) are this
 * product with the weight stored as [out features, in features].
 *   a : [M, K] device bf16;  w : [N, K] device bf16;  c : [M, N] device bf16,
 *       all contiguous and 16-byte aligned.
 *   K >= 1 and N multiples of 8 (16-byte rows), else ERR_SHAPE; M = 0 or
 *   N = 0 is a no-op.  Asynchronous on `stream`.  Errors as for diffattn_forward.
 */
diffattn_status diffattn_projection(int M, int N, int K, const void* a, const void* w, void* c,
                                    void* stream);

/*
 * The DIFF V1 attention layer around the operator (news article section
 * "差分注意力": X is projected by W^Q, W^K, W^V with per-head matrices, every
 * head's output is normalised on its own with the fixed multiplier
 * (1 - lambda_init), the heads are concatenated along the channels and
 * projected by W^O; lambda is re-parameterised from four vectors):
 *
 *   [Q | K | V] = X [W^Q | W^K | W^V];   head i: Q_1, Q_2 = first and last d of
 *                 Q's 2d columns [2 d i, 2 d (i + 1)), the same for K; V's 2d
 *   y_i = diffattn_forward of head i (lambda = lambda_reparam(lq1, lk1, lq2, lk2))
 *   out = Concat(y_1 .. y_H) W^O
 *
 *   x     : [B, n, D] device bf16 (tokens).
 *   w_qkv : [3 H 2d, D] device bf16: rows [0, H 2d) are the columns of W^Q
 *           ([D, H 2d]), then those of W^K, then W^V (the weight of one fused
 *           linear layer, [out features, in features]).
 *   w_o   : [D, H 2d] device bf16 (W^O as [out features, in features]).
 *   lq1, lk1, lq2, lk2 : device fp32 [d];  lambda_init, gamma, eps, causal:
 *           as for diffattn_forward.
 *   out   : [B, n, D] device bf16.
 *   workspace : device memory the caller owns, at least
 *           diffattn_layer_workspace(B, n, H, d) bytes, 256-byte aligned; it
 *           holds the projections, the normalised heads and lambda.
 * bf16 with d in {64, 128} (else ERR_UNSUPPORTED); D a multiple of 8; B = 0 or
 * n = 0 is a no-op.  Four kernels in stream order (projection GEMM, lambda,
 * the fused operator reading the projections in place, W^O GEMM);
 * asynchronous on `stream`.  Errors as for diffattn_forward; a small or
 * unaligned workspace -> ERR_SHAPE / ERR_ALIGN.
 */
size_t diffattn_layer_workspace(int B, int n, int H, int d);

diffattn_status diffattn_layer_forward(int B, int n, int D, int H, int d, const void* x,
                                       const void* w_qkv, const void* w_o, const float* lq1,
                                       const float* lk1, const float* lq2, const float* lk2,
                                       float lambda_init, const float* gamma, float eps, int causal,
                                       void* out, void* workspace, size_t workspace_bytes,
                                       void* stream);

/*
 * The DIFF V2 attention layer (DIFF V2 analysis page, sections "2. 커스텀 커널
 * 제거", "5. 간소화된 λ 매개변수화" (lambda per token and head, a sigmoid of a
 * projection of the token) and "GQA와의 호환성"):
 *
 *   [q | k | v | z] = X [W^Q | W^K | W^V | W^lambda]    z: one logit per token and pair
 *   y   = diffattn_v2_forward(q, k, v, logits z per token, scale 1/sqrt(d))
 *   out = Concat(pairs) W^O
 *
 *   x      : [B, n, D] device bf16.
 *   w_qkvl : [(Hq + 2 Hkv) d + Hq/2, D] device bf16: the columns of W^Q
 *            ([D, Hq d]), W^K, W^V ([D, Hkv d] each), then W^lambda ([D, Hq/2]).
 *   w_o    : [D, Hq/2 d] device bf16.   out : [B, n, D] device bf16.
 *   workspace : at least diffattn_v2_layer_workspace(B, n, Hq, Hkv, d) bytes,
 *            256-byte aligned (projections, fp32 logits, pair outputs).
 * bf16 with d = 128; Hq, Hkv rules as for diffattn_v2_forward; D a multiple of
 * 8.  Three kernels in stream order; the logits leave the projection in fp32.
 */
size_t diffattn_v2_layer_workspace(int B, int n, int Hq, int Hkv, int d);

diffattn_status diffattn_v2_layer_forward(int B, int n, int D, int Hq, int Hkv, int d,
                                          const void* x, const void* w_qkvl, const void* w_o,
                                          int causal, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * Backward pass of diffattn_forward (DIFF V1): fp32 inputs on CUDA cores, or
 * bf16 inputs on the tensor cores (tcgen05; d = 64).  The pages
 * ("Differential Transformer" glossary page, "How differential attention
 * works"; news article section "差分注意力") define the forward and report
 * trained models; the gradients are the chain rule of that forward:
 *
 *   A_r = softmax(Q_r K_r^T / sqrt d),  O = (A_1 - lambda A_2) V,
 *   y = (1 - lambda_init) gamma O / sqrt(mean_c O^2 + eps)
 *
 * Given dy = dL/dy it writes dL/dq1, dq2, dk1, dk2, dv, dL/dlambda and
 * dL/dgamma; the maps are recomputed, never stored.
 *   dt          : DIFFATTN_F32 (d in [1, 128]) or DIFFATTN_BF16 (d = 64; other d ->
 *                 ERR_UNSUPPORTED).  q1, q2, k1, k2, v and dy are of type dt; the
 *                 gradients dq1 .. dv are fp32 for both.  bf16: every tensor 16-byte
 *                 aligned, else ERR_ALIGN; P, dS and dO are rounded to bf16 for the
 *                 tensor cores, sums run in fp32.
 *   q1, q2, k1, k2, dq1, dq2, dk1, dk2 : [B, n, H, d] device; v, dy, dv : [B, n, H, 2d].
 *   lambda      : device scalar (as for the forward); lambda_init, eps, causal, gamma
 *                 (device [2d] or NULL for ones): as for diffattn_forward.
 *   dlambda     : device scalar (required); dgamma : device [2d] or NULL (not written).
 *   workspace   : device memory of at least diffattn_backward_workspace(B, H, n, d)
 *                 bytes, 16-byte aligned (per-row statistics, dO, dgamma shares);
 *                 smaller -> ERR_SHAPE.  The library allocates nothing.
 * fp32: sums for dlambda and dgamma run in a fixed order (same inputs, same
 * bits); bf16: dq is accumulated by TMA reduce-adds whose order varies from run
 * to run (dlambda, dgamma, dk and dv still in a fixed order).  Asynchronous on
 * `stream` (fp32: four kernels; bf16: two memsets and three kernels).  Errors as
 * for diffattn_forward.
 */
size_t diffattn_backward_workspace(int B, int H, int n, int d);

diffattn_status diffattn_backward(diffattn_dtype dt, int B, int H, int n, int d, const void* q1,
                                  const void* q2, const void* k1, const void* k2, const void* v,
                                  const float* lambda, float lambda_init, const float* gamma,
                                  float eps, int causal, const void* dy, void* dq1, void* dq2,
                                  void* dk1, void* dk2, void* dv, float* dlambda, float* dgamma,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass of diffattn_v2_forward (DIFF V2), fp32 on CUDA cores or bf16
 * (d = 128) on the tensor cores: per head
 * pair g of query heads 2g, 2g + 1 over KV head kv = 2g / (Hq / Hkv), with
 * s = sigmoid(logit) of the row, out = A_2g V - s A_2g+1 V (DIFF V2 analysis
 * page, "2. 커스텀 커널 제거", "5. 간소화된 λ 매개변수화", "GQA와의 호환성").
 * Given dy [B, n, Hq/2, d] it writes dq [B, n, Hq, d], dk and dv [B, n, Hkv, d]
 * (summed over every query head that reads the KV head) and dlogits, laid out
 * like lam_logits: strides (sb, st) = (n*Hq/2, Hq/2) (one logit per token and
 * pair), (Hq/2, 0) (per sequence and pair) or (0, 0) (per pair), the
 * gradient summed over the tokens (and sequences) that share a logit; other
 * strides -> ERR_UNSUPPORTED.
 *   dt : DIFFATTN_F32 (d in [1, 128]) or DIFFATTN_BF16 (d = 128, every tensor
 *        16-byte aligned, else ERR_UNSUPPORTED / ERR_ALIGN); q, k, v, dy of type
 *        dt, the gradients dq, dk, dv and dlogits fp32 for both.
 *   softmax_scale, causal, Hq / Hkv rules: as for diffattn_v2_forward.
 *   workspace : at least diffattn_v2_backward_workspace(B, Hq, n, d) bytes of
 *               device memory, 16-byte aligned; the library allocates nothing.
 * fp32: fixed summation orders (same inputs, same bits); bf16: dq by TMA
 * reduce-adds in a varying order.  Asynchronous on `stream`.  Errors as for
 * diffattn_forward.
 */
size_t diffattn_v2_backward_workspace(int B, int Hq, int n, int d);

diffattn_status diffattn_v2_backward(diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d,
                                     const void* q, const void* k, const void* v,
                                     const float* lam_logits, long long sb, long long st,
                                     float softmax_scale, int causal, const void* dy, void* dq,
                                     void* dk, void* dv, float* dlogits, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * Training forward and the backward from its saved statistics (bf16, tensor
 * cores).  The pages describe the forward and report trained models; how a
 * training step splits its work between forward and backward is this
 * library's: as in the usual attention backward, the forward keeps what the
 * backward would otherwise recompute.
 *
 * diffattn_forward_train: diffattn_forward (bf16, d = 64; same arguments,
 * same output bits) that also writes, per (batch, head, token) row, lse_1 and
 * lse_2 (the base-2 log-sum-exp of each map's scaled scores) and the
 * normalised map outputs O_1 = A_1 V and O_2 = A_2 V in bf16 to `saved`:
 *   saved : device memory of at least diffattn_forward_saved_bytes(B, H, n, d)
 *           bytes, 256-byte aligned (else ERR_SHAPE / ERR_ALIGN); the caller
 *           keeps it until the backward of this forward.
 * diffattn_backward_saved: diffattn_backward with dt = DIFFATTN_BF16 (same
 * arguments, gradients and workspace) given the same inputs and the `saved`
 * of their training forward; it does not recompute the forward's maps (a
 * per-row pass turns dy, O_1, O_2 into dO and the softmax-gradient row sums),
 * so it takes less time.  The result equals diffattn_backward's up to the
 * bf16 rounding of O_1, O_2.
 * The V2 pair is the same for diffattn_v2_forward / diffattn_v2_backward
 * (bf16, d = 128; rows are (batch, head pair, token)).  Other d ->
 * ERR_UNSUPPORTED; errors otherwise as for the calls they extend.
 */
size_t diffattn_forward_saved_bytes(int B, int H, int n, int d);

diffattn_status diffattn_forward_train(int B, int H, int n, int d, const void* q1, const void* q2,
                                       const void* k1, const void* k2, const void* v,
                                       const float* lambda, float lambda_init, const float* gamma,
                                       float eps, int causal, void* out, void* saved,
                                       size_t saved_bytes, void* stream);

diffattn_status diffattn_backward_saved(int B, int H, int n, int d, const void* q1, const void* q2,
                                        const void* k1, const void* k2, const void* v,
                                        const float* lambda, float lambda_init, const float* gamma,
                                        float eps, int causal, const void* dy, const void* saved,
                                        size_t saved_bytes, void* dq1, void* dq2, void* dk1,
                                        void* dk2, void* dv, float* dlambda, float* dgamma,
                                        void* workspace, size_t workspace_bytes, void* stream);

size_t diffattn_v2_forward_saved_bytes(int B, int Hq, int n, int d);

diffattn_status diffattn_v2_forward_train(int B, int Hq, int Hkv, int n, int d, const void* q,
                                          const void* k, const void* v, const float* lam_logits,
                                          long long sb, long long st, float softmax_scale,
                                          int causal, void* out, void* saved, size_t saved_bytes,
                                          void* stream);

diffattn_status diffattn_v2_backward_saved(int B, int Hq, int Hkv, int n, int d, const void* q,
                                           const void* k, const void* v, const float* lam_logits,
                                           long long sb, long long st, float softmax_scale,
                                           int causal, const void* dy, const void* saved,
                                           size_t saved_bytes, void* dq, void* dk, void* dv,
                                           float* dlogits, void* workspace, size_t workspace_bytes,
                                           void* stream);

/*
 * Gradients of lambda = exp(<lq1, lk1>) - exp(<lq2, lk2>) + lambda_init
 * (news article section "差分注意力") with respect to the four vectors of
 * length dim, given the device scalar dlambda: dlq1 = dlambda exp(<lq1, lk1>) lk1,
 * dlk1 = dlambda exp(<lq1, lk1>) lq1, and the second pair with the opposite
 * sign.  All pointers are device fp32.  One warp, asynchronous on `stream`.
 */
diffattn_status lambda_reparam_backward(const float* lq1, const float* lk1, const float* lq2,
                                        const float* lk2, int dim, const float* dlambda,
                                        float* dlq1, float* dlk1, float* dlq2, float* dlk2,
                                        void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns DIFFATTN_OK, DIFFATTN_ERR_TIMEOUT if a
 * bounded in-kernel wait ran out since the last call, DIFFATTN_ERR_BOUNDS (the
 * bounds-check build only) if an index check failed, or DIFFATTN_ERR_CUDA if
 * the stream reported an error.
 */
diffattn_status diffattn_device_status(void* stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* diffattn_last_error(void);

/*
 * 1 if this library is the bounds-check build (libdiffattn_bounds.so, built
 * with -DDIFFATTN_BOUNDS), else 0.  That build checks every TMA coordinate,
 * tensor-memory address and global store of its kernels before the access;
 * a failed check skips the access and diffattn_device_status returns
 * DIFFATTN_ERR_BOUNDS with the first failing site in diffattn_last_error.  It
 * is slower and meant for small cases; the results are otherwise identical.
 */
int diffattn_bounds_checked(void);

/*
 * Bounds-check build only (else ERR_UNSUPPORTED, nothing launched): launches
 * one thread that stores through the checked store at index 5 of a limit of
 * 4 (into a library-internal 8-element array, so the store could not leave
 * it either way).  The check must skip the store, and the next
 * diffattn_device_status must return DIFFATTN_ERR_BOUNDS.
 */
diffattn_status diffattn_debug_bounds_selftest(void* stream);

/*
 * Host only (nothing launched): the item plan that a persistent d = 128
 * forward over `units` (batch, head) units and query tiles
 * [qt0, qt0 + nqt) of an n-token sequence would run on `grid` CTAs, for the
 * tests.  Items are indices of the unit-major item map (unit u, query tile
 * qt0 + nqt - 1 - (item mod nqt) for item = u nqt + ...); CTA c runs
 * items[first[c]] .. items[first[c + 1] - 1] in that order.
 *   first : host array of at least grid + 1 entries (written);
 *   items : host array of at least units * nqt entries (written);
 *   kv_unit_bytes : K/V bytes of one unit (it sets the group size).
 * Returns the number of CTAs with a list (grid), or 0 when the launch is too
 * large for a plan (more than 256 CTAs or 4096 items: the snake order runs).
 */
int diffattn_debug_item_plan(int grid, long long units, int nqt, int qt0, int n, int causal,
                             long long kv_unit_bytes, unsigned short* first, unsigned short* items);

/*
 * Diagnostics: launches one CTA whose thread waits on an mbarrier that nothing
 * arrives on, with a budget of about `budget_ns` nanoseconds (1 .. 1e9; the
 * kernel counts 2 SM clock cycles per nanosecond).  The wait
 * must run out and record DIFFATTN_ERR_TIMEOUT in the status word; this is how
 * the bounded-wait path is exercised without hanging a GPU.  No copy is in
 * flight while it waits.
 */
diffattn_status diffattn_debug_wait_timeout(long long budget_ns, void* stream);

/*
 * Number of kernels the library has launched in this process (all devices).
 * Lets a caller count the kernels of a timed region.
 */
long long diffattn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
