// asv_internal.h -- host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "asv.h"

namespace asv {

constexpr int kMaxCluster = 16;  // CTAs per row (16 needs the non-portable cluster attribute)

// One row's result as the row's cluster leaves it in the workspace for the
// request-level scan.  `value` is the row's divergence (SCI) or unused;
// `token` the row's emitted-token candidate; `bits` the kBit* flags.
struct __align__(16) RowRecord {
  double value;
  int32_t token;
  uint32_t bits;
};

// RAPID row state kept for the request-level scan and for the residual/bonus draw, which the
// last row of a request to finish recomputes for the emitted position.  With zs = z / T:
//   p_k = ex2(fma(zs_k, log2e, -zs_max*log2e)) * inv_sum, zhat_k = z_k + eta*T*(q_k - p_k),
//   tail_k <=> zhat_k / T < zhat_max + ln(tail_frac),
//   protected_k = p_k * tail_scale on the tail, ex2((zhat_k / T - zhat_max) * log2e) * head_scale on
//   the head.
// One row's result in the multi-outcome kernels (the all-(beta, gamma) sweep; AsymSpec fused with
// E2-SCI): JSD(a || t) (fused), the emitted-token candidates of the argmax slots, one gate bit per
// gamma, and the kBit* problem flags.
struct __align__(16) MultiRecord {
  double J;
  int32_t tok[4];
  uint32_t gate_bits;
  uint32_t flags;
};

struct __align__(32) RapidRecord {
  float zs_max;
  float inv_sum;
  float zhat_max;   // max of zhat / T
  float head_scale;
  uint32_t bits;
  float tail_scale;  // 1, or 1/Z under the alternative tail reading
  uint32_t pad[2];
};

// RAPID: the draw the verification's scan leaves for the draw launch (one per request): the stop
// row and its record's row constants, then the draw launch's own race slots and counter.
struct __align__(64) RapidJob {
  float zs_max;
  float inv_sum;
  float zhat_max;
  float head_scale;
  float tail_scale;
  int32_t row;      // stop position n (residual draw if n < G, bonus draw if n == G)
  uint32_t active;  // 1 while the draw is pending
  uint32_t ticket;  // CTAs of the draw launch done with this request
  // Race winners as ~((key bits << 32) | index), combined with atomic max (zero = none yet):
  // [0] the residual (bonus position: the protected target), [1] p, used if [0] has no entry.
  unsigned long long slot[2];
  uint32_t pad[4];
};

// Per-request E2-SCI stabiliser state (layout of asv_sci_state).
struct __align__(16) SciState {
  double T_applied;
  int32_t age;
  uint32_t flags;  // 1: a threshold has been applied; 2: fallback pending
};

struct LaunchPlan {
  int cluster;    // CTAs per row
  int threads;    // threads per CTA
  int n_slice;    // vocabulary entries per CTA (multiple of the 16-byte vector width)
  int smem;       // dynamic shared memory bytes
  int bulk;       // 1: rows staged with bulk copies
};

constexpr int kModeAsym = 0;
constexpr int kModeSci = 1;

struct JsdArgs {
  const void* x[3];  // AsymSpec: a, b, t.  SCI: draft, target (x[2] unused)
  const int32_t* draft_ids;
  int B, K, V;
  int n_slice;
  int bulk;
  int variant;       // 0 single outcome; 1 all-(beta, gamma) sweep; 2 AsymSpec fused with E2-SCI
  float betas[4];    // betas[0] is the AsymSpec beta; the sweep uses n_beta of them
  int n_beta;
  int delta_source;  // AsymSpec: 0 a - b, 1 a, 2 t - b
  double ln_gamma;
  double ln_gammas[8];  // sweep: n_gamma values of ln(gamma); fused: ln_gammas[0] = ln_gamma
  int n_gamma;
  // SCI
  double T_base, alpha_omega, tau_credit, T_min, T_max, ewma_beta;
  double* r_hat;
  // E2-SCI pre-hit: 0 off; 1 row 0 of every request; 2 rows 1..K of requests not dropped
  int prehit_phase;
  uint32_t* dropped;  // [B] 1 when phase 1 dropped the request's window
  // SCI stabilisers (state == nullptr: off)
  SciState* sci_state;
  double hyst, fb_acc, fb_T;
  int min_refresh;
  // outputs
  int32_t* out_accept_len;
  int32_t* out_tokens;
  float* out_D;      // AsymSpec: JSD(a,b); SCI: JSD(draft,target)
  float* out_lse;    // AsymSpec only, [R, 3]
  float* out_T;      // SCI only
  float* out_J;               // fused: JSD(a || t) [R]
  int32_t* out_sci_accept_len;  // fused: E2-SCI accept lengths [B]
  int32_t* out_sci_tokens;      // fused: E2-SCI tokens [B, K+1]
  uint32_t* out_req_status;
  // workspace
  uint32_t* tickets;
  RowRecord* records;
  MultiRecord* mrecords;  // multi-outcome variants (the same workspace bytes as `records`)
  // staged kernel: rows cut into `n_unit` units of n_slice entries, each staged in one CTA's shared
  // memory; the CTAs of a row exchange partial statistics through the workspace
  int n_unit;            // units per row
  int units;             // rows * n_unit
  int chunk_units;       // consecutive units of a row one CTA takes at a time (divides n_unit)
  uint32_t* row_cnt;     // [rows] pass-A partials published
  uint32_t* row_jcnt;    // [rows] pass-B partials published
  void* part_a;          // [units] 64-byte pass-A partials
  float* part_b;         // [units] 16 floats: pass-B sums as (hi, lo) pairs
  uint32_t* abort_flag;  // set by a CTA whose bounded wait expired
  uint32_t* check_log;   // checked build: [count of failed index tests, line of the first]
};

struct RapidArgs {
  const float* z;
  const float* q;
  const int32_t* draft_ids;
  int B, G, V;
  int n_slice;
  int bulk;
  float T, inv_T, eta, tail_frac, ln_tail_frac;
  int tail_mode;  // 0: tail keeps p, head rescaled; 1: substitute p on the tail, renormalise all
  uint32_t seed_lo, seed_hi, offset;
  int32_t* out_accept_len;
  int32_t* out_tokens;
  uint32_t* out_req_status;
  uint32_t* tickets;
  RapidRecord* records;
  RapidJob* jobs;
  int draw_ctas;  // CTAs per request of the draw launch
  uint32_t* check_log;  // checked build: [count of failed index tests, line of the first]
};

// Staged AsymSpec / E2-SCI kernel (asv_staged.cu): units per row and entries per unit for a row of
// V entries of `elem_bytes` bytes, `nt` inputs read by pass A and `nb` by pass B (the two rings of
// unit buffers fill a fixed shared-memory budget), dynamic shared memory of one CTA, threads per
// CTA, and the launch (cooperative: one CTA per SM, all resident at once).
struct StagedPlan {
  int n_unit;    // units per row
  int n;         // entries per unit (multiple of the 16-byte vector width)
  int smem;      // dynamic shared memory bytes per CTA
  int chunk;     // largest number of units per chunk
};
int staged_chunk_for(const StagedPlan& pl, long long rows, int grid);
StagedPlan staged_plan(int V, int elem_bytes, int nt, int nb);  // nb: inputs pass B reads
int staged_max_units();
int staged_threads();
size_t staged_workspace_bytes(long long rows, int n_unit);
// Workspace bytes of the cluster AsymSpec kernel alone (tickets and row records); a call given
// no more than this runs the cluster kernel.
size_t asym_cluster_workspace_bytes(int B, int K);
cudaError_t launch_jsd_staged(int mode, int dtype, const JsdArgs& args, const StagedPlan& plan, int grid,
                              cudaStream_t s);
int staged_grid(int mode, int dtype, const JsdArgs& args, const StagedPlan& plan);  // 0: cannot launch

// The checked build appends a 256-byte check log to every workspace (zero-filled like the rest).
#ifdef ASV_CHECKED
constexpr size_t kCheckLogBytes = 256;
#else
constexpr size_t kCheckLogBytes = 0;
#endif

// Kernel launchers (return the cudaError_t of the launch).
cudaError_t launch_jsd_family(int mode, int dtype, const JsdArgs& args, const LaunchPlan& plan, cudaStream_t s);
cudaError_t launch_rapid(const RapidArgs& args, const LaunchPlan& plan, cudaStream_t s);

int jsd_threads();      // threads per CTA of the AsymSpec / SCI kernel
int jsd_ctas_per_sm();  // CTAs of it that share an SM (its launch bounds)
bool rapid_needs_all_sums(int tail_mode, float ln_tail_frac);  // all-entry sums: dense pass B
int rapid_umax_bytes(bool all_sums, int n_slice);                 // the per-vector-group bounds of U
int rapid_smem_bytes(bool all_sums, int n_slice, bool aligned);   // dynamic shared memory per CTA
int rapid_ring_bytes();                                           // the pass-A ring of one CTA
int rapid_draw_smem_bytes(int n_slice, bool aligned);            // ... of the draw launch
int rapid_draw_ctas_per_sm();                                     // draw CTAs resident per SM
int rapid_threads();      // threads per CTA of the RAPID kernel
int rapid_ctas_per_sm();  // CTAs of it that share an SM (its launch bounds)

// Host-side argument checks shared by asymspec_verify and asymspec_verify_static (asv_api.cu):
// check_asym_shape covers B, K, V and the element type; check_asym_args (for B > 0) the scalar
// parameters, then the alignment of every pointer given, then the required pointers.
asv_status check_asym_shape(int B, int K, int V, int dtype);
asv_status check_asym_args(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids, int K,
                           float beta, float gamma, const int32_t* out_accept_len, const int32_t* out_tokens,
                           const float* out_D, const float* out_lse, const uint32_t* out_req_status);

// Occupancy query: clusters of `plan` that can be resident at once (0 = cannot launch).
int jsd_max_active_clusters(int mode, int dtype, const LaunchPlan& plan);
int rapid_max_active_clusters(const LaunchPlan& plan);

}  // namespace asv
