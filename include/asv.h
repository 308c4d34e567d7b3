/*
 * asv.h -- C ABI of the GB300 logit-space speculative verification library (libasv).
 *
 * One shared library with plain C entry points over caller-owned device
 * buffers.  It covers the verification step of three speculative-decoding
 * methods described on these pages:
 *
 *   [ASYM]  "AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs"
 *           (reading notes), sec. 4.1 (contrastive delta-fusion) and sec. 4.2
 *           (context-divergence-aware acceptance, the CDA gate).
 *   [RAPID] "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
 *           Decoding" (paper notes), Key designs 2-4 (retrieval-augmented target,
 *           tail protection, adjusted residual sampling).
 *   [SCI]   "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia"
 *           (paper notes), Key design 3 (JSD test against an adaptive threshold
 *           driven by an EWMA of the acceptance rate).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Logit tensors are row-major [B, K+1, V]: request b, position i (K draft
 *    positions plus the bonus position K), vocabulary entry k; a row is V
 *    contiguous elements, element type fp32 or bf16 (ASV_F32 / ASV_BF16).
 *  - Every pointer argument is a DEVICE pointer owned by the caller unless the
 *    name ends in _host.  The library never allocates, frees or retains memory.
 *  - Calls are asynchronous on `stream`; nothing waits for the GPU.  The return
 *    value reports argument validation and launch failures only.  Conditions
 *    that depend on the data are written per request to out_req_status
 *    (ASV_REQ_* bits); a flagged request gets accept length 0 and tokens -1.
 *  - Output tokens per request: the accepted drafts, then one token chosen by the
 *    verifier at the first rejection (or at the bonus position), then -1 padding.
 *  - Two kernels serve the AsymSpec / E2-SCI entry points, with the same
 *    decisions and tokens.  The cluster kernel (the default): thread-block
 *    clusters that stream their rows with 16-byte loads (element loads for
 *    unaligned rows).  The staged kernel (asv_set_kernel(ASV_KERNEL_STAGED)):
 *    one CTA per SM (a cooperative launch, so all of them are resident at once),
 *    rows cut into units that bulk copies stage in shared memory, the CTAs of a
 *    row exchanging partial sums through the workspace; it takes rows whose base
 *    address is 16-byte aligned (V * element size a multiple of 16 and 16-byte
 *    aligned base pointers) given a workspace of asv_workspace_bytes(...), and
 *    leaves the E2-SCI pre-hit, cluster-size overrides (asv_set_tuning) and
 *    workspaces only as large as the cluster kernel needs to the cluster kernel.
 *  - `workspace` is device scratch of at least asv_workspace_bytes(...) bytes.
 *    It must be zero-filled before its first use (asv_workspace_init does that);
 *    every call leaves it zero-filled again.  Two calls that may run at the
 *    same time must not share a workspace.
 *  - Thread safety: the entry points keep no host state except the tuning
 *    override and a per-device cache of launch attributes.
 */
#ifndef ASV_H_
#define ASV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ASV_OK = 0,
  ASV_ERR_NULL = 1,      /* a required pointer is NULL */
  ASV_ERR_SHAPE = 2,     /* B < 0, K < 0 (K < 1 for SCI), V < 2, or V too large for one cluster */
  ASV_ERR_ALIGN = 3,     /* a pointer is not aligned to its element size */
  ASV_ERR_DTYPE = 4,     /* unknown element type, or a type the mode does not take */
  ASV_ERR_PARAM = 5,     /* a scalar parameter is non-finite or out of range */
  ASV_ERR_WORKSPACE = 6, /* workspace NULL or smaller than asv_workspace_bytes() */
  ASV_ERR_CUDA = 7       /* a CUDA runtime call or the launch failed (see asv_last_cuda_error) */
} asv_status;

typedef enum { ASV_F32 = 0, ASV_BF16 = 1 } asv_dtype;

typedef enum {
  ASV_MODE_ASYMSPEC = 0,
  ASV_MODE_RAPID = 1,
  ASV_MODE_SCI = 2,
  ASV_MODE_SWEEP = 3,        /* asymspec_verify_sweep */
  ASV_MODE_ASYMSPEC_SCI = 4  /* asymspec_sci_verify */
} asv_mode;

/* Per-request status bits written by the kernels (never a trap). */
#define ASV_REQ_NONFINITE 1u /* a row holds NaN or +inf, or is entirely -inf */
#define ASV_REQ_BAD_DRAFT 2u /* a draft id lies outside [0, V) */
#define ASV_REQ_TIMEOUT 4u   /* a bounded wait of the staged kernel expired (its launch keeps every CTA
                                resident, so this marks a fault, not a load condition): the request's
                                outputs are unspecified and the workspace must be zero-filled again */

/* Human-readable name of a status code (static string). */
const char* asv_status_string(asv_status s);

/* cudaError_t value of the most recent ASV_ERR_CUDA on the calling thread (0 if none). */
int asv_last_cuda_error(void);

/* Bytes of device workspace one call of `mode` needs for a [B, K+1, V] batch. */
size_t asv_workspace_bytes(int mode, int B, int K, int V, int dtype);

/* Zero-fill `ws_bytes` bytes of workspace on `stream` (cudaMemsetAsync). */
asv_status asv_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Tuning override for the launch plan: cluster size (CTAs per row, 1..16; 0
 * restores the automatic choice).  threads_per_cta must be 0 or 256, the size
 * the kernels are compiled for (anything else is ASV_ERR_PARAM).  Applies to
 * later calls from any thread.
 */
asv_status asv_set_tuning(int cluster_ctas, int threads_per_cta);

/* Kernel selection for the AsymSpec / E2-SCI entry points, for later calls from any thread:
 * ASV_KERNEL_DEFAULT and ASV_KERNEL_CLUSTER select the cluster kernel, ASV_KERNEL_STAGED the
 * staged kernel where it applies (see the conventions above).  Anything else is ASV_ERR_PARAM. */
#define ASV_KERNEL_DEFAULT 0
#define ASV_KERNEL_CLUSTER 1
#define ASV_KERNEL_STAGED 2
asv_status asv_set_kernel(int which);

/* The plan the next call with these shapes would use, and how many of its clusters the device
 * can hold at once (cudaOccupancyMaxActiveClusters).  Any output may be NULL.
 * - Cluster kernel: cluster size, threads, dynamic shared memory bytes, bulk_copy = 1 if rows take
 *   16-byte vector loads (0 element loads), active clusters.
 * - Staged kernel (when selected, for AsymSpec, E2-SCI, the sweep and the fused mode on rows whose
 *   V * element size is a multiple of 16, with no cluster-size override): units per row in
 *   cluster_ctas, its threads, dynamic shared memory bytes, bulk_copy = 2, and its CTAs in
 *   max_active_clusters. */
asv_status asv_query_plan(int mode, int B, int K, int V, int dtype, int* cluster_ctas, int* threads_per_cta,
                          int* smem_bytes, int* bulk_copy, int* max_active_clusters);

/*
 * asymspec_verify -- the AsymSpec verification step.  [ASYM] sec. 4.1-4.2.
 *
 * Inputs, each [B, K+1, V] of element type `dtype`:
 *   a  drafter logits on the full context, b  drafter logits on the compressed
 *   context, t  verifier logits on the compressed context.
 *   draft_ids [B, K] int32: the drafted token at each of the K positions.
 * Per row i:  D_i = JSD(softmax a_i || softmax b_i) (natural log, weights 1/2);
 *   c_i = argmax_k (t_ik + beta * (a_ik - b_ik)), the fp32 score formed as one
 *   rounded subtraction and one fused multiply-add, lowest index on ties.
 * Draft i < K is accepted iff softmax(t_i)[d_i] > gamma * exp(-D_i) * softmax(b_i)[d_i]
 * (strict; decided in double in the log domain).  The scan stops at the first
 * rejection n (n = K if none); the request emits d_0..d_{n-1}, then c_n.
 *
 * beta: any finite value.  gamma: finite, > 0.
 * Outputs: out_accept_len [B] int32; out_tokens [B, K+1] int32 (-1 padded);
 *   out_D [B, K+1] float (clamped to [0, ln 2], may be NULL);
 *   out_lse [B, K+1, 3] float, log-sum-exp of a, b, t (may be NULL);
 *   out_req_status [B] uint32 ASV_REQ_* bits.
 * B = 0 is a no-op that returns ASV_OK.
 * Checks, in this order, each returning before anything is queued on the GPU: B, K, V
 * (ASV_ERR_SHAPE), dtype (ASV_ERR_DTYPE); for B > 0: beta, gamma (ASV_ERR_PARAM), the alignment
 * of every pointer given, NULL counting as aligned (ASV_ERR_ALIGN), the required pointers
 * (ASV_ERR_NULL), then the workspace (ASV_ERR_WORKSPACE, ASV_ERR_ALIGN for a workspace not
 * 256-byte aligned).
 */
asv_status asymspec_verify(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids, int B,
                           int K, int V, float beta, float gamma, int32_t* out_accept_len, int32_t* out_tokens,
                           float* out_D, float* out_lse, uint32_t* out_req_status, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/* Context-gain signal used in the delta-fusion score ([ASYM] sec. 5, mechanism ablation). */
typedef enum {
  ASV_DELTA_A_MINUS_B = 0, /* delta = a - b: the method (same drafter, two context views) */
  ASV_DELTA_A = 1,         /* delta = a: the raw full-context drafter logits */
  ASV_DELTA_T_MINUS_B = 2  /* delta = t - b: a two-model difference on the compressed view */
} asv_delta_source;

typedef struct {
  int delta_source; /* asv_delta_source; ASV_DELTA_A_MINUS_B in asymspec_verify */
} asv_asym_options;

/*
 * asymspec_verify_ex -- asymspec_verify with options (NULL options = the defaults).  With
 * delta_source != ASV_DELTA_A_MINUS_B the emitted token is argmax_k (t_k + beta * delta_k) for
 * the chosen delta, formed the same way (one rounded fp32 operation, then one FMA); the gate,
 * D and the log-sum-exps are unchanged.  Any other delta_source value is ASV_ERR_PARAM.
 */
asv_status asymspec_verify_ex(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                              int B, int K, int V, float beta, float gamma, const asv_asym_options* options,
                              int32_t* out_accept_len, int32_t* out_tokens, float* out_D, float* out_lse,
                              uint32_t* out_req_status, void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * asymspec_verify_sweep -- AsymSpec for every (beta, gamma) of a grid from one read of a, b, t.
 * [ASYM] sec. 5 sweeps beta and gamma over a flat region; D and the log-sum-exps do not depend on
 * them, the emitted token depends on beta only and the gate on gamma only, so one pass over the
 * inputs serves the whole grid.  betas [n_beta] (1..ASV_SWEEP_MAX_BETA, finite) and gammas
 * [n_gamma] (1..ASV_SWEEP_MAX_GAMMA, > 0) are HOST arrays.  For grid point (beta_i, gamma_j) the
 * results equal asymspec_verify(..., beta_i, gamma_j, ...):
 *   out_accept_len [n_gamma, B]        (the accepted prefix depends on gamma only)
 *   out_tokens     [n_beta, n_gamma, B, K+1]
 *   out_D [B, K+1], out_lse [B, K+1, 3] (may be NULL), out_req_status [B].
 * The workspace is asv_workspace_bytes(ASV_MODE_SWEEP, ...).
 */
#define ASV_SWEEP_MAX_BETA 4
#define ASV_SWEEP_MAX_GAMMA 8
asv_status asymspec_verify_sweep(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                                 int B, int K, int V, const float* betas, int n_beta, const float* gammas,
                                 int n_gamma, int32_t* out_accept_len, int32_t* out_tokens, float* out_D,
                                 float* out_lse, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream);

/*
 * asymspec_verify_host -- asymspec_verify over HOST buffers, for callers whose
 * logits live in host memory.  Copies a, b, t and draft_ids to the device arena,
 * runs the verification, and copies accept lengths, tokens, D and request status
 * back, all on `stream` (the call returns before the copies finish; synchronise
 * the stream before reading the outputs).  Host buffers should be pinned.
 * `arena` is caller-owned device memory of at least asv_host_arena_bytes(...)
 * bytes, zero-filled before its first use; it holds the staged inputs, the
 * outputs and the workspace.  out_D_host may be NULL.
 */
size_t asv_host_arena_bytes(int B, int K, int V, int dtype);
asv_status asymspec_verify_host(const void* a_host, const void* b_host, const void* t_host, int dtype,
                                const int32_t* draft_ids_host, int B, int K, int V, float beta, float gamma,
                                int32_t* out_accept_len_host, int32_t* out_tokens_host, float* out_D_host,
                                uint32_t* out_req_status_host, void* arena, size_t arena_bytes,
                                cudaStream_t stream);

/*
 * asymspec_verify_static -- asymspec_verify without a caller workspace, for callers that cannot
 * allocate device memory: code handed only its input and output buffers (for instance a plugin
 * inside a serving framework whose memory pool it does not own), or code that must not allocate
 * once it is running.  The paper has no counterpart; this is a packaging variant.
 *
 * The scratch lives in a file-scope device array of ASV_STATIC_SCRATCH_BYTES bytes (1 MiB),
 * reserved on every GPU that loads the library's device code and held until the process exits.
 * The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 * - Batches whose workspace (asv_workspace_bytes) exceeds ASV_STATIC_SCRATCH_BYTES are rejected
 *   with ASV_ERR_WORKSPACE (at K = 8 that is a little over 7,000 requests).
 * - Every call made outside stream capture looks up the array's device address
 *   (cudaGetSymbolAddress) with the current device, so a device reset between calls (which reloads
 *   the module and may move the array) is picked up.  A call made while `stream` is capturing uses
 *   the address found by the last call outside capture on that device: make the first call on a
 *   device, and the first call after any device reset, before capturing.
 * - Every argument check of asymspec_verify, and the size limit, comes before the GPU or the array
 *   is touched: a rejected call queues nothing.
 * - Every call shares the one array.  Each call clears the part that must start at zero (one
 *   cudaMemsetAsync on `stream`) before its kernel; calls that may overlap on the GPU (other
 *   streams, other host threads) race on the array and must not be issued.
 * Everything else is as asymspec_verify.
 */
#define ASV_STATIC_SCRATCH_BYTES (1u << 20)
asv_status asymspec_verify_static(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                                  int B, int K, int V, float beta, float gamma, int32_t* out_accept_len,
                                  int32_t* out_tokens, float* out_D, float* out_lse, uint32_t* out_req_status,
                                  cudaStream_t stream);

/*
 * rapid_verify -- RAPID verification with the retrieval-augmented target.
 * [RAPID] Workflow; Key designs 2 (augmented target), 3 (tail protection),
 * 4 (adjusted residual sampling).
 *
 * Inputs (fp32, [B, G+1, V]): z  target logits; q  drafter probabilities.
 *   draft_ids [B, G] int32.
 * Per row: p = softmax(z/T); zhat = z + eta*T*(q - p); phat = softmax(zhat/T);
 *   tail = {k : phat_k < tail_frac * max phat};  protected target p' keeps p on
 *   the tail and rescales phat on the rest so that p' sums to 1.
 * Draft i is accepted iff u_i * q_i(d_i) < p'_i(d_i) with u_i a Philox4x32-10
 * uniform; at the first rejection n the token is drawn from
 * norm(max(p_n - p'_n, p_n - q_n, 0)) (from p_n if that is all zero); if all G
 * drafts pass, the bonus token is drawn from p'_G.  Draws use an exponential
 * race over Philox uniforms.
 * Random numbers: key = (seed low 32 bits, seed high 32 bits); counter =
 * (word / 4, position i, request b, stream + 4*offset); the uniform is
 * ((word32 >> 9) + 0.5) * 2^-23 from word (word % 4) of the block; streams are
 * 0 = accept test (word 0), 1 = residual draw (word k), 2 = bonus draw (word k).
 * T > 0, eta >= 0, 0 <= tail_frac < 1, all finite.
 * Outputs: out_accept_len [B], out_tokens [B, G+1], out_req_status [B].
 * Launches: two kernels on `stream`, the verification and then the draw; the draw
 * is a programmatic dependent launch of the verification (it may be scheduled
 * while the verification's last CTAs run and waits for the verification to
 * complete before it reads anything), so work the caller enqueues on `stream`
 * after this call runs after both, as in plain stream order; inside stream
 * capture the pair becomes two graph nodes joined by a programmatic edge.
 */
asv_status rapid_verify(const float* z, const float* q, const int32_t* draft_ids, int B, int G, int V, float T,
                        float eta, float tail_frac, uint64_t seed, uint32_t offset, int32_t* out_accept_len,
                        int32_t* out_tokens, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                        cudaStream_t stream);

/* RAPID options ([RAPID] Key design 3 leaves the renormalisation of the protected target open). */
typedef struct {
  int tail_mode; /* 0: tail entries keep p exactly and the head is rescaled so the protected target
                    sums to 1 (the reading rapid_verify uses); 1: p substitutes phat on the tail and
                    every entry is renormalised (tail p/Z, head phat/Z, Z = tail p-mass + head
                    phat-mass) */
} asv_rapid_options;

/* rapid_verify with options (NULL = the defaults).  An unknown tail_mode is ASV_ERR_PARAM. */
asv_status rapid_verify_ex(const float* z, const float* q, const int32_t* draft_ids, int B, int G, int V, float T,
                           float eta, float tail_frac, uint64_t seed, uint32_t offset, const asv_rapid_options* options,
                           int32_t* out_accept_len, int32_t* out_tokens, uint32_t* out_req_status, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/* E2-SCI threshold and credit parameters.  [SCI] Key design 3. */
typedef struct {
  double T_base;      /* base threshold */
  double alpha_omega; /* alpha * omega, the credit gain */
  double tau_credit;  /* neutral credit level */
  double T_min;       /* lower clamp */
  double T_max;       /* upper clamp */
  double ewma_beta;   /* EWMA weight of the newest window (0.3) */
} asv_sci_params;

/*
 * sci_verify -- one E2-SCI verification window per request.  [SCI] Key design 3.
 *
 * Inputs, [B, K+1, V] of `dtype`: draft logits and target logits; draft_ids [B, K].
 * r_hat [B] double: the credit state, read and updated in place.
 * Per request: T = clamp(T_base + alpha_omega*(r_hat - tau_credit), T_min, T_max);
 *   J_i = JSD(softmax draft_i || softmax target_i); drafts are accepted while
 *   J_i <= T; n = the accepted prefix; tokens = d_0..d_{n-1}, argmax(target_n);
 *   r_hat <- (1 - ewma_beta)*r_hat + ewma_beta*(n/K).  A flagged request leaves
 *   r_hat unchanged.  K >= 1.
 * Outputs: out_accept_len [B], out_tokens [B, K+1], out_jsd [B, K+1] float (may be
 *   NULL), out_T [B] float (may be NULL), out_req_status [B].
 */
asv_status sci_verify(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                      int B, int K, int V, const asv_sci_params* params, double* r_hat, int32_t* out_accept_len,
                      int32_t* out_tokens, float* out_jsd, float* out_T, uint32_t* out_req_status,
                      void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * sci_verify_prehit -- sci_verify with the first-token pre-hit of [SCI] Key design 4 (PLC): the
 * first draft of every window is verified first, and a window whose first draft fails the
 * threshold is dropped without reading its later rows (accept length 0, the target's argmax at
 * position 0, r_hat updated with acceptance 0).  Two launches on `stream`: row 0 of every request,
 * then rows 1..K of the windows kept.  For finite inputs the outputs equal sci_verify's, except
 * that out_jsd holds only row 0 of a dropped window (its later entries are not written); a
 * dropped window never sees non-finite values past its first row, so such a request is flagged
 * by sci_verify but not here.  Draft ids are all checked.  K >= 1.
 */
asv_status sci_verify_prehit(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                             int B, int K, int V, const asv_sci_params* params, double* r_hat, int32_t* out_accept_len,
                             int32_t* out_tokens, float* out_jsd, float* out_T, uint32_t* out_req_status,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * E2-SCI stabilisers.  [SCI] Key design 3 adds hysteresis, a minimum refresh interval and a
 * fallback to a conservative threshold when accuracy under the predicted threshold drops below a
 * bound, and gives no constants; these are the parameters.  One window's threshold, from the
 * candidate T_cand = clamp(T_base + alpha_omega*(r_hat - tau_credit), T_min, T_max) and the
 * request's state:
 *   first window (state not set)                               -> T_cand
 *   fallback pending                                           -> fallback_T
 *   age >= min_refresh and |T_cand - T_applied| > hysteresis   -> T_cand
 *   otherwise                                                  -> T_applied
 * A change sets age to 1, keeping T_applied adds one.  After the window, a fallback is pending
 * for the next window iff n / K < fallback_acc.  hysteresis = 0, min_refresh = 1 and
 * fallback_acc = 0 reproduce sci_verify.
 */
typedef struct {
  double hysteresis;   /* >= 0 */
  int32_t min_refresh; /* >= 1 windows */
  int32_t reserved;    /* 0 */
  double fallback_acc; /* acceptance rate below which the next window falls back */
  double fallback_T;   /* the conservative threshold */
} asv_sci_stabilisers;

/* Per-request stabiliser state, device memory, zero-filled before a request's first window. */
typedef struct {
  double T_applied; /* threshold used by the last window */
  int32_t age;      /* windows since T_applied last changed */
  uint32_t flags;   /* 1: a threshold has been applied; 2: fallback pending */
} asv_sci_state;

/*
 * sci_verify_ex -- sci_verify with stabilisers.  `stab` NULL is sci_verify; otherwise `state`
 * [B] (16-byte aligned) is read and updated in place with r_hat (a flagged request leaves both
 * unchanged) and out_T reports the threshold the window used.  Invalid stabiliser values are
 * ASV_ERR_PARAM.
 */
asv_status sci_verify_ex(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                         int B, int K, int V, const asv_sci_params* params, const asv_sci_stabilisers* stab,
                         double* r_hat, asv_sci_state* state, int32_t* out_accept_len, int32_t* out_tokens,
                         float* out_jsd, float* out_T, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * asymspec_sci_verify -- AsymSpec and one E2-SCI window on the same tensors from one read.
 * E2-SCI takes draft = a and target = t; its divergence JSD(a || t) is summed in the same pass
 * as D = JSD(a || b).  The AsymSpec outputs equal asymspec_verify(a, b, t, ..., beta, gamma);
 * the SCI outputs equal sci_verify(a, t, ..., params, r_hat) (r_hat updated in place):
 * out_sci_accept_len [B], out_sci_tokens [B, K+1], out_jsd [B, K+1] (may be NULL), out_T [B]
 * (may be NULL).  out_req_status [B] is shared (a flagged request gets accept length 0 and
 * tokens -1 in both modes and keeps its r_hat).  K >= 1.  The workspace is
 * asv_workspace_bytes(ASV_MODE_ASYMSPEC_SCI, ...).
 */
asv_status asymspec_sci_verify(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                               int B, int K, int V, float beta, float gamma, const asv_sci_params* params,
                               double* r_hat, int32_t* out_accept_len, int32_t* out_tokens, float* out_D,
                               float* out_lse, int32_t* out_sci_accept_len, int32_t* out_sci_tokens, float* out_jsd,
                               float* out_T, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                               cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ASV_H_ */
