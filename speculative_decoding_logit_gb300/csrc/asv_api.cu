// asv_api.cu -- the extern "C" entry points declared in include/asv.h: argument validation,
// workspace layout, launch planning (cluster size, threads, shared memory) and dispatch.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "asv.h"
#include "asv_internal.h"

static_assert(sizeof(asv_sci_state) == sizeof(asv::SciState), "asv_sci_state layout");

using asv::LaunchPlan;

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<int> g_tune_cluster{0};
std::atomic<int> g_use_staged{0};  // asv_set_kernel: 1 selects the staged kernel where it applies

asv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = int(e);
  return ASV_ERR_CUDA;
}

struct DevInfo {
  int sms = 0;
};

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

cudaError_t dev_info(DevInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.sms == 0) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  }
  *out = d;
  return cudaSuccess;
}

inline size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// CTAs of the staged kernel that fit the device at once, per (device, kernel instantiation); the
// first query of an instantiation on a device also raises its shared-memory limit.
struct StagedKey {
  int dev, mode, dtype, dsrc, variant;
  bool operator<(const StagedKey& o) const {
    return std::tie(dev, mode, dtype, dsrc, variant) < std::tie(o.dev, o.mode, o.dtype, o.dsrc, o.variant);
  }
};
std::map<StagedKey, int> g_staged_grid;
std::mutex g_staged_mu;

cudaError_t staged_grid_cached(int mode, int dtype, const asv::JsdArgs& a, const asv::StagedPlan& plan, int* grid) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const StagedKey key{dev, mode, dtype, a.delta_source, a.variant};
  std::lock_guard<std::mutex> lk(g_staged_mu);
  auto it = g_staged_grid.find(key);
  if (it == g_staged_grid.end()) it = g_staged_grid.emplace(key, asv::staged_grid(mode, dtype, a, plan)).first;
  *grid = it->second;
  return cudaSuccess;
}
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace layout: [tickets: B x u32, padded to 256 B][records: R x record].
size_t tickets_bytes(int B) { return round_up(size_t(B) * 4, 256); }

size_t record_bytes(int mode) {
  if (mode == ASV_MODE_RAPID) return sizeof(asv::RapidRecord);
  if (mode == ASV_MODE_SWEEP || mode == ASV_MODE_ASYMSPEC_SCI) return sizeof(asv::MultiRecord);
  return sizeof(asv::RowRecord);
}

// Cluster size for the streaming kernels, which stage nothing, so `ctas_per_sm` CTAs (their
// launch bounds) share an SM and each pass re-reads its slice from L2.  The smallest C whose R*C
// CTAs fill at least 90% of one wave of resident CTAs and whose last wave is at least 85% full --
// fewer CTAs per row mean fewer cluster exchanges, while a partly empty last wave leaves SMs idle.
// A batch too small to fill a wave even at C = 16 takes the largest C (at least 1024 entries per
// CTA).  A tuning override replaces the choice.
int wave_fill_cluster(int V, long long R, int ctas_per_sm, int sms) {
  int C = g_tune_cluster.load();
  if (C > 0) return C;
  const int c_max = std::max(1, std::min(asv::kMaxCluster, V / 1024));
  const double resident = double(ctas_per_sm) * sms;
  for (int c = 1; c <= c_max; ++c) {
    const double waves = double(R) * c / resident;
    if (waves < 0.9) continue;
    if (waves / std::ceil(waves) >= 0.85) return c;
  }
  return c_max;
}

// Plan for the AsymSpec / SCI kernel.
cudaError_t plan_jsd(int elem_bytes, int V, long long R, bool aligned, LaunchPlan* out) {
  DevInfo di;
  cudaError_t e = dev_info(&di);
  if (e != cudaSuccess) return e;
  const int vec = 16 / elem_bytes;
  int C = wave_fill_cluster(V, R, asv::jsd_ctas_per_sm(), di.sms);
  // fp32 rows carry half the arithmetic per byte of bf16 ones, so the pass-B re-reads that L2 misses
  // weigh more: slices of at most 512 KB of the three inputs keep more of each CTA's pair in L2
  // (measured on 1280 fp32 rows of V = 151936: 0.507 ms at C = 4 against 0.519 ms at C = 3; bf16
  // batches measured best at the wave-filling choice).
  if (elem_bytes == 4 && g_tune_cluster.load() <= 0)
    while (C < asv::kMaxCluster && V / (C + 1) >= 1024 && 3LL * elem_bytes * ceil_div(V, C) > 512LL * 1024) ++C;
  out->cluster = C;
  out->threads = asv::jsd_threads();
  out->n_slice = int(round_up(size_t(ceil_div(V, C)), size_t(vec)));
  out->smem = 0;
  out->bulk = aligned ? 1 : 0;
  return cudaSuccess;
}

// Plan for the RAPID kernel (fp32 rows, four entries per 16-byte vector).  Aligned rows under the
// default tail reading stream pass A through the shared-memory ring: the verification is then bound
// by the bytes in flight while it streams, and every CTA pays its exchanges and sparse re-reads
// once, so the fewest CTAs per row that keep at least 8 MB in flight over the batch (each CTA's ring
// holds 32 KB), with the ring and the per-group bounds within 72 KB (three CTAs per SM).  Otherwise
// (the dense pass B of the all-entry sums, or element loads) the wave-filling choice, with the
// bounds within 52 KB (four CTAs per SM).
cudaError_t plan_rapid(int V, long long R, bool aligned, bool all_sums, LaunchPlan* out) {
  DevInfo di;
  cudaError_t e = dev_info(&di);
  if (e != cudaSuccess) return e;
  auto n_slice = [&](int c) { return int(round_up(size_t(ceil_div(V, c)), 4)); };
  auto smem = [&](int c) { return asv::rapid_smem_bytes(all_sums, n_slice(c), aligned); };
  const int c_max = std::max(1, std::min(asv::kMaxCluster, V / 1024));
  int C = g_tune_cluster.load();
  if (C <= 0) {
    if (aligned && !all_sums) {
      const long long per_row = std::max<long long>(1, R) * asv::rapid_ring_bytes();
      C = int(std::min<long long>(c_max, std::max<long long>(1, ((8LL << 20) + per_row - 1) / per_row)));
      while (C < asv::kMaxCluster && smem(C) > 72 * 1024) ++C;
    } else {
      C = wave_fill_cluster(V, R, asv::rapid_ctas_per_sm(), di.sms);
      while (C < asv::kMaxCluster && smem(C) > 52 * 1024) ++C;
    }
  }
  if (smem(C) > 200 * 1024) return cudaErrorInvalidValue;  // V too large
  out->cluster = C;
  out->threads = asv::rapid_threads();
  out->n_slice = n_slice(C);
  out->smem = smem(C);
  out->bulk = aligned ? 1 : 0;
  return cudaSuccess;
}

// CTAs per request of the RAPID draw launch.  The draw reads the B stop rows once, so a second,
// partial wave of CTAs would nearly double its time: while the batch fits one wave of resident
// draw CTAs, as many CTAs per request as 95 % of that wave holds (a CTA streams its slice through a
// ring of six vectors per thread; measured, a few SMs hold one draw CTA fewer right after the
// verification, whose last CTAs the draw's first ones overlap); larger batches take slices of at
// most one ring's worth (6144 entries) over several waves.  At least 1024 entries per CTA.
int rapid_draw_ctas(int V, int B) {
  DevInfo di;
  const int sms = dev_info(&di) == cudaSuccess ? di.sms : 1;
  const long long slots = 1LL * asv::rapid_draw_ctas_per_sm() * sms * 95 / 100;
  long long want = slots / std::max(B, 1);
  if (want < 1) want = (V + 6143) / 6144;
  return int(std::max(1LL, std::min<long long>(want, std::max(1, V / 1024))));
}

bool valid_dtype(int dt) { return dt == ASV_F32 || dt == ASV_BF16; }
int elem_size(int dt) { return dt == ASV_F32 ? 4 : 2; }

}  // namespace

namespace asv {

// Argument checks of asymspec_verify, in the order they are applied: shapes and element type, then
// (for B > 0) the scalar parameters, the alignment of every pointer given (NULL counts as
// aligned), and last the required pointers.  A call that fails any of them touches neither the
// GPU nor the workspace.
asv_status check_asym_shape(int B, int K, int V, int dtype) {
  if (B < 0 || K < 0 || V < 2) return ASV_ERR_SHAPE;
  if ((long long)B * ((long long)K + 1) * asv::kMaxCluster > 0x7fffffffLL) return ASV_ERR_SHAPE;
  if (!valid_dtype(dtype)) return ASV_ERR_DTYPE;
  return ASV_OK;
}

asv_status check_asym_args(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids, int K,
                           float beta, float gamma, const int32_t* out_accept_len, const int32_t* out_tokens,
                           const float* out_D, const float* out_lse, const uint32_t* out_req_status) {
  if (!std::isfinite(beta) || !std::isfinite(gamma) || !(gamma > 0.0f)) return ASV_ERR_PARAM;
  const size_t eb = size_t(elem_size(dtype));
  if (!aligned(a, eb) || !aligned(b, eb) || !aligned(t, eb) || !aligned(draft_ids, 4) || !aligned(out_accept_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(out_req_status, 4) || !aligned(out_D, 4) || !aligned(out_lse, 4))
    return ASV_ERR_ALIGN;
  if (!a || !b || !t || (K > 0 && !draft_ids) || !out_accept_len || !out_tokens || !out_req_status) return ASV_ERR_NULL;
  return ASV_OK;
}

}  // namespace asv

extern "C" {

const char* asv_status_string(asv_status s) {
  switch (s) {
    case ASV_OK: return "ASV_OK";
    case ASV_ERR_NULL: return "ASV_ERR_NULL: a required pointer is NULL";
    case ASV_ERR_SHAPE: return "ASV_ERR_SHAPE: invalid B, K or V";
    case ASV_ERR_ALIGN: return "ASV_ERR_ALIGN: misaligned pointer";
    case ASV_ERR_DTYPE: return "ASV_ERR_DTYPE: unsupported element type";
    case ASV_ERR_PARAM: return "ASV_ERR_PARAM: scalar parameter out of range";
    case ASV_ERR_WORKSPACE: return "ASV_ERR_WORKSPACE: workspace missing or too small";
    case ASV_ERR_CUDA: return "ASV_ERR_CUDA: CUDA runtime error";
  }
  return "unknown asv_status";
}

int asv_last_cuda_error(void) { return g_last_cuda_error; }

// Workspace: [tickets: B x u32, padded to 256 B][records: R x record]; E2-SCI adds the pre-hit
// drop flags [B x u32] after the records (256-byte aligned).
static size_t records_end(int mode, int B, int K) {
  return round_up(tickets_bytes(B) + size_t(B) * size_t(K + 1) * record_bytes(mode), 256);
}

// A workspace region followed by the checked build's check log (256-byte aligned); the ordinary
// build has no log and uses the region's exact size.
static size_t with_log(size_t bytes) {
  return asv::kCheckLogBytes ? round_up(bytes, 256) + asv::kCheckLogBytes : bytes;
}

// The check log of a call whose workspace region (without the log) is `region` bytes.
static uint32_t* check_log_at(void* workspace, size_t region) {
  if (!asv::kCheckLogBytes) return nullptr;
  return reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + round_up(region, 256));
}

// Workspace of the cluster kernels (and of RAPID).
static size_t cluster_workspace_bytes(int mode, int B, int K) {
  if (B < 0 || K < 0) return 0;
  if (mode == ASV_MODE_SCI) return records_end(mode, B, K) + size_t(B) * 4;
  if (mode == ASV_MODE_RAPID) return records_end(mode, B, K) + size_t(B) * sizeof(asv::RapidJob);
  return tickets_bytes(B) + size_t(B) * size_t(K + 1) * record_bytes(mode);
}

}  // extern "C"

namespace asv {
size_t asym_cluster_workspace_bytes(int B, int K) { return with_log(cluster_workspace_bytes(ASV_MODE_ASYMSPEC, B, K)); }
}  // namespace asv

extern "C" {

// The staged kernel's plan for a mode, or n_unit = 0 when it does not apply: rows must be whole
// 16-byte vectors (V * element size a multiple of 16), at most staged_max_units() units per row,
// and the unit count must fit the launch's index arithmetic.
static asv::StagedPlan staged_plan_for(int mode, int B, int K, int V, int dtype) {
  asv::StagedPlan pl{0, 0, 0, 0};
  if (mode == ASV_MODE_RAPID || !valid_dtype(dtype) || B < 1 || K < 0 || V < 2) return pl;
  const int eb = elem_size(dtype);
  if ((size_t(V) * size_t(eb)) % 16 != 0) return pl;
  const int nt = mode == ASV_MODE_SCI ? 2 : 3;
  const int nb = mode == ASV_MODE_ASYMSPEC_SCI ? 3 : 2;
  asv::StagedPlan p = asv::staged_plan(V, eb, nt, nb);
  if (p.n_unit > asv::staged_max_units()) return pl;
  if ((long long)B * ((long long)K + 1) * p.n_unit > 0x7fffffffLL) return pl;
  return p;
}

// The staged kernel's workspace follows the cluster kernels', 256-byte aligned.
static size_t staged_offset(int mode, int B, int K) { return round_up(cluster_workspace_bytes(mode, B, K), 256); }

// Sized for the kernel the current selection (asv_set_kernel) would use; a call given less than the
// staged kernel's size runs the cluster kernel.
size_t asv_workspace_bytes(int mode, int B, int K, int V, int dtype) {
  if (B < 0 || K < 0) return 0;
  const asv::StagedPlan sp = staged_plan_for(mode, B, K, V, dtype);
  if (sp.n_unit == 0 || g_use_staged.load() != 1) return with_log(cluster_workspace_bytes(mode, B, K));
  return with_log(staged_offset(mode, B, K) + asv::staged_workspace_bytes((long long)B * (K + 1), sp.n_unit));
}

asv_status asv_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!workspace) return ASV_ERR_NULL;
  cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, stream);
  return e == cudaSuccess ? ASV_OK : cuda_fail(e);
}

asv_status asv_set_tuning(int cluster_ctas, int threads_per_cta) {
  if (cluster_ctas < 0 || cluster_ctas > asv::kMaxCluster) return ASV_ERR_PARAM;
  if (threads_per_cta != 0 && threads_per_cta != asv::jsd_threads()) return ASV_ERR_PARAM;
  g_tune_cluster.store(cluster_ctas);
  return ASV_OK;
}

asv_status asv_set_kernel(int which) {
  if (which < ASV_KERNEL_DEFAULT || which > ASV_KERNEL_STAGED) return ASV_ERR_PARAM;
  g_use_staged.store(which == ASV_KERNEL_STAGED ? 1 : 0);
  return ASV_OK;
}

asv_status asv_query_plan(int mode, int B, int K, int V, int dtype, int* cluster_ctas, int* threads_per_cta,
                          int* smem_bytes, int* bulk_copy, int* max_active_clusters) {
  if (B < 1 || K < 0 || V < 2) return ASV_ERR_SHAPE;
  if (!valid_dtype(dtype)) return ASV_ERR_DTYPE;
  if (mode == ASV_MODE_RAPID && dtype != ASV_F32) return ASV_ERR_DTYPE;
  const int eb = elem_size(dtype);
  const bool bulk = (size_t(V) * eb) % 16 == 0;
  // The staged kernel (when a call with 16-byte aligned pointers and a full workspace would take it):
  // units per row, its threads, dynamic shared memory, 2, and its CTAs (one per SM).
  const asv::StagedPlan sp = staged_plan_for(mode, B, K, V, dtype);
  if (sp.n_unit > 0 && g_tune_cluster.load() == 0 && g_use_staged.load() == 1) {
    asv::JsdArgs a;
    std::memset(&a, 0, sizeof(a));
    a.variant = mode == ASV_MODE_SWEEP ? 1 : mode == ASV_MODE_ASYMSPEC_SCI ? 2 : 0;
    const int kmode = mode == ASV_MODE_SCI ? asv::kModeSci : asv::kModeAsym;
    int grid = 0;
    cudaError_t e = staged_grid_cached(kmode, dtype, a, sp, &grid);
    if (e != cudaSuccess) return cuda_fail(e);
    if (grid >= 2 * sp.n_unit) {
      if (cluster_ctas) *cluster_ctas = sp.n_unit;
      if (threads_per_cta) *threads_per_cta = asv::staged_threads();
      if (smem_bytes) *smem_bytes = sp.smem;
      if (bulk_copy) *bulk_copy = 2;
      if (max_active_clusters) *max_active_clusters = grid;
      return ASV_OK;
    }
  }
  LaunchPlan pl;
  cudaError_t e = mode == ASV_MODE_RAPID
                      ? plan_rapid(V, (long long)B * (K + 1), bulk, false, &pl)
                      : plan_jsd(eb, V, (long long)B * (K + 1), bulk, &pl);
  if (e == cudaErrorInvalidValue) return ASV_ERR_SHAPE;
  if (e != cudaSuccess) return cuda_fail(e);
  if (cluster_ctas) *cluster_ctas = pl.cluster;
  if (threads_per_cta) *threads_per_cta = pl.threads;
  if (smem_bytes) *smem_bytes = pl.smem;
  if (bulk_copy) *bulk_copy = pl.bulk;
  if (max_active_clusters) {
    *max_active_clusters = mode == ASV_MODE_RAPID
                               ? asv::rapid_max_active_clusters(pl)
                               : asv::jsd_max_active_clusters(mode == ASV_MODE_SCI ? asv::kModeSci : asv::kModeAsym,
                                                              dtype, pl);
  }
  return ASV_OK;
}

static asv_status run_jsd(int mode, asv::JsdArgs& a, int dtype, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
  int amode = mode == asv::kModeAsym ? ASV_MODE_ASYMSPEC : ASV_MODE_SCI;
  if (a.variant == 1) amode = ASV_MODE_SWEEP;
  if (a.variant == 2) amode = ASV_MODE_ASYMSPEC_SCI;
  if (ws_bytes < with_log(cluster_workspace_bytes(amode, a.B, a.K))) return ASV_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return ASV_ERR_ALIGN;
  const int eb = elem_size(dtype);
  const int NT = mode == asv::kModeAsym ? 3 : 2;
  bool bulk = (size_t(a.V) * eb) % 16 == 0;
  for (int j = 0; j < NT; ++j) bulk = bulk && aligned(a.x[j], 16);
  a.tickets = reinterpret_cast<uint32_t*>(workspace);
  a.records = reinterpret_cast<asv::RowRecord*>(static_cast<char*>(workspace) + tickets_bytes(a.B));
  a.mrecords = reinterpret_cast<asv::MultiRecord*>(static_cast<char*>(workspace) + tickets_bytes(a.B));
  a.check_log = check_log_at(workspace, cluster_workspace_bytes(amode, a.B, a.K));
  // The staged kernel: aligned rows, no pre-hit, no cluster-size override, and a workspace that
  // holds its exchange area (a smaller one, enough for the cluster kernel, selects that kernel).
  const asv::StagedPlan sp = staged_plan_for(amode, a.B, a.K, a.V, dtype);
  if (bulk && sp.n_unit > 0 && a.prehit_phase == 0 && g_tune_cluster.load() == 0 && g_use_staged.load() == 1 &&
      ws_bytes >= asv_workspace_bytes(amode, a.B, a.K, a.V, dtype)) {
    int grid = 0;
    cudaError_t e = staged_grid_cached(mode, dtype, a, sp, &grid);
    if (e != cudaSuccess) return cuda_fail(e);
    if (grid >= 2 * sp.n_unit) {
      const long long rows = (long long)a.B * (a.K + 1);
      char* st = static_cast<char*>(workspace) + staged_offset(amode, a.B, a.K);
      const size_t cnt = (size_t(rows) * 8 + 255) / 256 * 256;
      a.n_slice = sp.n;
      a.n_unit = sp.n_unit;
      a.units = int(rows * sp.n_unit);
      a.chunk_units = asv::staged_chunk_for(sp, rows, grid);
      a.row_cnt = reinterpret_cast<uint32_t*>(st);
      a.row_jcnt = a.row_cnt + rows;
      a.abort_flag = reinterpret_cast<uint32_t*>(st + cnt);
      a.part_a = st + cnt + 256;
      a.part_b = reinterpret_cast<float*>(st + cnt + 256 + size_t(a.units) * 128);
      a.bulk = 2;
      a.check_log = check_log_at(workspace, staged_offset(amode, a.B, a.K) +
                                                asv::staged_workspace_bytes(rows, sp.n_unit));
      e = asv::launch_jsd_staged(mode, dtype, a, sp, std::min(grid, a.units / a.chunk_units), stream);
      if (e != cudaSuccess) return cuda_fail(e);
      return ASV_OK;
    }
  }
  LaunchPlan pl;
  cudaError_t e = plan_jsd(eb, a.V, (long long)a.B * (a.K + 1), bulk, &pl);
  if (e == cudaErrorInvalidValue) return ASV_ERR_SHAPE;
  if (e != cudaSuccess) return cuda_fail(e);
  a.n_slice = pl.n_slice;
  a.bulk = pl.bulk;
  if (mode == asv::kModeSci && a.prehit_phase != 0) {
    // E2-SCI pre-hit: phase 1 over row 0 of every request, phase 2 over rows 1..K of the requests
    // phase 1 kept, then the drop flags are cleared (the workspace is left zeroed).
    a.dropped = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + records_end(ASV_MODE_SCI, a.B, a.K));
    a.prehit_phase = 1;
    e = asv::launch_jsd_family(mode, dtype, a, pl, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    a.prehit_phase = 2;
    e = asv::launch_jsd_family(mode, dtype, a, pl, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemsetAsync(a.dropped, 0, size_t(a.B) * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return ASV_OK;
  }
  e = asv::launch_jsd_family(mode, dtype, a, pl, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return ASV_OK;
}

asv_status asymspec_verify(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids, int B,
                           int K, int V, float beta, float gamma, int32_t* out_accept_len, int32_t* out_tokens,
                           float* out_D, float* out_lse, uint32_t* out_req_status, void* workspace,
                           size_t ws_bytes, cudaStream_t stream) {
  return asymspec_verify_ex(a, b, t, dtype, draft_ids, B, K, V, beta, gamma, nullptr, out_accept_len, out_tokens,
                            out_D, out_lse, out_req_status, workspace, ws_bytes, stream);
}

asv_status asymspec_verify_ex(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                              int B, int K, int V, float beta, float gamma, const asv_asym_options* options,
                              int32_t* out_accept_len, int32_t* out_tokens, float* out_D, float* out_lse,
                              uint32_t* out_req_status, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  const int dsrc = options ? options->delta_source : ASV_DELTA_A_MINUS_B;
  if (dsrc < ASV_DELTA_A_MINUS_B || dsrc > ASV_DELTA_T_MINUS_B) return ASV_ERR_PARAM;
  asv_status st = asv::check_asym_shape(B, K, V, dtype);
  if (st != ASV_OK || B == 0) return st;
  st = asv::check_asym_args(a, b, t, dtype, draft_ids, K, beta, gamma, out_accept_len, out_tokens, out_D, out_lse,
                           out_req_status);
  if (st != ASV_OK) return st;
  if (!workspace) return ASV_ERR_WORKSPACE;
  asv::JsdArgs args;
  std::memset(&args, 0, sizeof(args));
  args.x[0] = a;
  args.x[1] = b;
  args.x[2] = t;
  args.draft_ids = draft_ids;
  args.B = B;
  args.K = K;
  args.V = V;
  args.betas[0] = beta;
  args.n_beta = 1;
  args.delta_source = dsrc;
  args.ln_gamma = std::log(double(gamma));
  args.out_accept_len = out_accept_len;
  args.out_tokens = out_tokens;
  args.out_D = out_D;
  args.out_lse = out_lse;
  args.out_req_status = out_req_status;
  return run_jsd(asv::kModeAsym, args, dtype, workspace, ws_bytes, stream);
}

asv_status sci_verify(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                      int B, int K, int V, const asv_sci_params* params, double* r_hat, int32_t* out_accept_len,
                      int32_t* out_tokens, float* out_jsd, float* out_T, uint32_t* out_req_status,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return sci_verify_ex(draft_logits, target_logits, dtype, draft_ids, B, K, V, params, nullptr, r_hat, nullptr,
                       out_accept_len, out_tokens, out_jsd, out_T, out_req_status, workspace, ws_bytes, stream);
}

static asv_status sci_run(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                          int B, int K, int V, const asv_sci_params* params, const asv_sci_stabilisers* stab,
                          double* r_hat, asv_sci_state* state, int prehit, int32_t* out_accept_len,
                          int32_t* out_tokens, float* out_jsd, float* out_T, uint32_t* out_req_status,
                          void* workspace, size_t ws_bytes, cudaStream_t stream);

asv_status sci_verify_ex(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                         int B, int K, int V, const asv_sci_params* params, const asv_sci_stabilisers* stab,
                         double* r_hat, asv_sci_state* state, int32_t* out_accept_len, int32_t* out_tokens,
                         float* out_jsd, float* out_T, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                         cudaStream_t stream) {
  return sci_run(draft_logits, target_logits, dtype, draft_ids, B, K, V, params, stab, r_hat, state, 0,
                 out_accept_len, out_tokens, out_jsd, out_T, out_req_status, workspace, ws_bytes, stream);
}

asv_status sci_verify_prehit(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                             int B, int K, int V, const asv_sci_params* params, double* r_hat, int32_t* out_accept_len,
                             int32_t* out_tokens, float* out_jsd, float* out_T, uint32_t* out_req_status,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return sci_run(draft_logits, target_logits, dtype, draft_ids, B, K, V, params, nullptr, r_hat, nullptr, 1,
                 out_accept_len, out_tokens, out_jsd, out_T, out_req_status, workspace, ws_bytes, stream);
}

static asv_status sci_run(const void* draft_logits, const void* target_logits, int dtype, const int32_t* draft_ids,
                          int B, int K, int V, const asv_sci_params* params, const asv_sci_stabilisers* stab,
                          double* r_hat, asv_sci_state* state, int prehit, int32_t* out_accept_len,
                          int32_t* out_tokens, float* out_jsd, float* out_T, uint32_t* out_req_status,
                          void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || K < 1 || V < 2) return ASV_ERR_SHAPE;
  if ((long long)B * (K + 1) * asv::kMaxCluster > 0x7fffffffLL) return ASV_ERR_SHAPE;
  if (!valid_dtype(dtype)) return ASV_ERR_DTYPE;
  if (B == 0) return ASV_OK;
  if (!draft_logits || !target_logits || !draft_ids || !params || !r_hat || !out_accept_len || !out_tokens ||
      !out_req_status)
    return ASV_ERR_NULL;
  if (!workspace) return ASV_ERR_WORKSPACE;
  const size_t eb = size_t(elem_size(dtype));
  if (!aligned(draft_logits, eb) || !aligned(target_logits, eb) || !aligned(draft_ids, 4) || !aligned(r_hat, 8) ||
      !aligned(out_accept_len, 4) || !aligned(out_tokens, 4) || !aligned(out_jsd, 4) || !aligned(out_T, 4) ||
      !aligned(out_req_status, 4))
    return ASV_ERR_ALIGN;
  const asv_sci_params& P = *params;
  const double vals[6] = {P.T_base, P.alpha_omega, P.tau_credit, P.T_min, P.T_max, P.ewma_beta};
  for (double v : vals)
    if (!std::isfinite(v)) return ASV_ERR_PARAM;
  if (P.T_min > P.T_max || P.ewma_beta < 0.0 || P.ewma_beta > 1.0) return ASV_ERR_PARAM;
  if (stab) {
    if (!state) return ASV_ERR_NULL;
    if (!aligned(state, 16)) return ASV_ERR_ALIGN;
    if (!std::isfinite(stab->hysteresis) || stab->hysteresis < 0.0 || stab->min_refresh < 1 ||
        !std::isfinite(stab->fallback_acc) || !std::isfinite(stab->fallback_T))
      return ASV_ERR_PARAM;
  }
  asv::JsdArgs args;
  std::memset(&args, 0, sizeof(args));
  args.x[0] = draft_logits;
  args.x[1] = target_logits;
  args.draft_ids = draft_ids;
  args.B = B;
  args.K = K;
  args.V = V;
  args.T_base = P.T_base;
  args.alpha_omega = P.alpha_omega;
  args.tau_credit = P.tau_credit;
  args.T_min = P.T_min;
  args.T_max = P.T_max;
  args.ewma_beta = P.ewma_beta;
  args.r_hat = r_hat;
  args.prehit_phase = prehit;
  if (stab) {
    args.sci_state = reinterpret_cast<asv::SciState*>(state);
    args.hyst = stab->hysteresis;
    args.min_refresh = stab->min_refresh;
    args.fb_acc = stab->fallback_acc;
    args.fb_T = stab->fallback_T;
  }
  args.out_accept_len = out_accept_len;
  args.out_tokens = out_tokens;
  args.out_D = out_jsd;
  args.out_T = out_T;
  args.out_req_status = out_req_status;
  return run_jsd(asv::kModeSci, args, dtype, workspace, ws_bytes, stream);
}

// Shared checks of the AsymSpec-family entry points over three [B, K+1, V] inputs.
static asv_status check_asym_inputs(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                                    int B, int K, int V) {
  if (B < 0 || K < 0 || V < 2) return ASV_ERR_SHAPE;
  if ((long long)B * (K + 1) * asv::kMaxCluster > 0x7fffffffLL) return ASV_ERR_SHAPE;
  if (!valid_dtype(dtype)) return ASV_ERR_DTYPE;
  if (B == 0) return ASV_OK;
  if (!a || !b || !t || (K > 0 && !draft_ids)) return ASV_ERR_NULL;
  const size_t eb = size_t(elem_size(dtype));
  if (!aligned(a, eb) || !aligned(b, eb) || !aligned(t, eb) || !aligned(draft_ids, 4)) return ASV_ERR_ALIGN;
  return ASV_OK;
}

asv_status asymspec_verify_sweep(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                                 int B, int K, int V, const float* betas, int n_beta, const float* gammas,
                                 int n_gamma, int32_t* out_accept_len, int32_t* out_tokens, float* out_D,
                                 float* out_lse, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream) {
  asv_status st = check_asym_inputs(a, b, t, dtype, draft_ids, B, K, V);
  if (st != ASV_OK || B == 0) return st;
  if (!betas || !gammas || !out_accept_len || !out_tokens || !out_req_status) return ASV_ERR_NULL;
  if (!workspace) return ASV_ERR_WORKSPACE;
  if (n_beta < 1 || n_beta > ASV_SWEEP_MAX_BETA || n_gamma < 1 || n_gamma > ASV_SWEEP_MAX_GAMMA) return ASV_ERR_PARAM;
  if (!aligned(out_accept_len, 4) || !aligned(out_tokens, 4) || !aligned(out_req_status, 4) || !aligned(out_D, 4) ||
      !aligned(out_lse, 4))
    return ASV_ERR_ALIGN;
  asv::JsdArgs args;
  std::memset(&args, 0, sizeof(args));
  for (int i = 0; i < 4; ++i) {
    const float be = betas[i < n_beta ? i : 0];
    if (!std::isfinite(be)) return ASV_ERR_PARAM;
    args.betas[i] = be;
  }
  for (int g = 0; g < n_gamma; ++g) {
    if (!std::isfinite(gammas[g]) || !(gammas[g] > 0.0f)) return ASV_ERR_PARAM;
    args.ln_gammas[g] = std::log(double(gammas[g]));
  }
  args.variant = 1;
  args.n_beta = n_beta;
  args.n_gamma = n_gamma;
  args.x[0] = a;
  args.x[1] = b;
  args.x[2] = t;
  args.draft_ids = draft_ids;
  args.B = B;
  args.K = K;
  args.V = V;
  args.out_accept_len = out_accept_len;
  args.out_tokens = out_tokens;
  args.out_D = out_D;
  args.out_lse = out_lse;
  args.out_req_status = out_req_status;
  return run_jsd(asv::kModeAsym, args, dtype, workspace, ws_bytes, stream);
}

asv_status asymspec_sci_verify(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids,
                               int B, int K, int V, float beta, float gamma, const asv_sci_params* params,
                               double* r_hat, int32_t* out_accept_len, int32_t* out_tokens, float* out_D,
                               float* out_lse, int32_t* out_sci_accept_len, int32_t* out_sci_tokens, float* out_jsd,
                               float* out_T, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                               cudaStream_t stream) {
  if (K < 1 && B > 0) return ASV_ERR_SHAPE;
  asv_status st = check_asym_inputs(a, b, t, dtype, draft_ids, B, K, V);
  if (st != ASV_OK || B == 0) return st;
  if (!params || !r_hat || !out_accept_len || !out_tokens || !out_sci_accept_len || !out_sci_tokens ||
      !out_req_status)
    return ASV_ERR_NULL;
  if (!workspace) return ASV_ERR_WORKSPACE;
  if (!aligned(r_hat, 8) || !aligned(out_accept_len, 4) || !aligned(out_tokens, 4) || !aligned(out_D, 4) ||
      !aligned(out_lse, 4) || !aligned(out_sci_accept_len, 4) || !aligned(out_sci_tokens, 4) ||
      !aligned(out_jsd, 4) || !aligned(out_T, 4) || !aligned(out_req_status, 4))
    return ASV_ERR_ALIGN;
  if (!std::isfinite(beta) || !std::isfinite(gamma) || !(gamma > 0.0f)) return ASV_ERR_PARAM;
  const asv_sci_params& P = *params;
  const double vals[6] = {P.T_base, P.alpha_omega, P.tau_credit, P.T_min, P.T_max, P.ewma_beta};
  for (double v : vals)
    if (!std::isfinite(v)) return ASV_ERR_PARAM;
  if (P.T_min > P.T_max || P.ewma_beta < 0.0 || P.ewma_beta > 1.0) return ASV_ERR_PARAM;
  asv::JsdArgs args;
  std::memset(&args, 0, sizeof(args));
  args.variant = 2;
  args.betas[0] = args.betas[1] = args.betas[2] = args.betas[3] = beta;
  args.n_beta = 1;
  args.ln_gamma = std::log(double(gamma));
  args.ln_gammas[0] = args.ln_gamma;
  args.n_gamma = 1;
  args.x[0] = a;
  args.x[1] = b;
  args.x[2] = t;
  args.draft_ids = draft_ids;
  args.B = B;
  args.K = K;
  args.V = V;
  args.T_base = P.T_base;
  args.alpha_omega = P.alpha_omega;
  args.tau_credit = P.tau_credit;
  args.T_min = P.T_min;
  args.T_max = P.T_max;
  args.ewma_beta = P.ewma_beta;
  args.r_hat = r_hat;
  args.out_accept_len = out_accept_len;
  args.out_tokens = out_tokens;
  args.out_D = out_D;
  args.out_lse = out_lse;
  args.out_J = out_jsd;
  args.out_sci_accept_len = out_sci_accept_len;
  args.out_sci_tokens = out_sci_tokens;
  args.out_T = out_T;
  args.out_req_status = out_req_status;
  return run_jsd(asv::kModeAsym, args, dtype, workspace, ws_bytes, stream);
}

// Host-buffer variant: arena = [a | b | t | draft_ids | accept_len | tokens | D | status | workspace],
// each part aligned to 256 bytes.
static size_t host_arena_layout(int B, int K, int V, int dtype, size_t off[9]) {
  const size_t R = size_t(B) * size_t(K + 1);
  const size_t in_bytes = R * size_t(V) * size_t(elem_size(dtype));
  const size_t sizes[9] = {in_bytes, in_bytes, in_bytes, size_t(B) * size_t(K) * 4, size_t(B) * 4, R * 4, R * 4,
                           size_t(B) * 4, asv_workspace_bytes(ASV_MODE_ASYMSPEC, B, K, V, dtype)};
  size_t o = 0;
  for (int i = 0; i < 9; ++i) {
    off[i] = o;
    o = round_up(o + sizes[i], 256);
  }
  return o;
}

size_t asv_host_arena_bytes(int B, int K, int V, int dtype) {
  if (B < 0 || K < 0 || V < 2 || !valid_dtype(dtype)) return 0;
  size_t off[9];
  return host_arena_layout(B, K, V, dtype, off);
}

asv_status asymspec_verify_host(const void* a_host, const void* b_host, const void* t_host, int dtype,
                                const int32_t* draft_ids_host, int B, int K, int V, float beta, float gamma,
                                int32_t* out_accept_len_host, int32_t* out_tokens_host, float* out_D_host,
                                uint32_t* out_req_status_host, void* arena, size_t arena_bytes,
                                cudaStream_t stream) {
  if (B < 0 || K < 0 || V < 2) return ASV_ERR_SHAPE;
  if (!valid_dtype(dtype)) return ASV_ERR_DTYPE;
  if (B == 0) return ASV_OK;
  if (!a_host || !b_host || !t_host || (K > 0 && !draft_ids_host) || !out_accept_len_host || !out_tokens_host ||
      !out_req_status_host)
    return ASV_ERR_NULL;
  if (!arena) return ASV_ERR_WORKSPACE;
  if (!aligned(arena, 256)) return ASV_ERR_ALIGN;
  size_t off[9];
  const size_t need = host_arena_layout(B, K, V, dtype, off);
  if (arena_bytes < need) return ASV_ERR_WORKSPACE;
  char* base = static_cast<char*>(arena);
  const size_t R = size_t(B) * size_t(K + 1);
  const size_t in_bytes = R * size_t(V) * size_t(elem_size(dtype));
  const void* src[4] = {a_host, b_host, t_host, draft_ids_host};
  const size_t nbytes[4] = {in_bytes, in_bytes, in_bytes, size_t(B) * size_t(K) * 4};
  for (int i = 0; i < 4; ++i) {
    if (nbytes[i] == 0) continue;
    cudaError_t e = cudaMemcpyAsync(base + off[i], src[i], nbytes[i], cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  asv_status st = asymspec_verify(base + off[0], base + off[1], base + off[2], dtype,
                                  reinterpret_cast<const int32_t*>(base + off[3]), B, K, V, beta, gamma,
                                  reinterpret_cast<int32_t*>(base + off[4]), reinterpret_cast<int32_t*>(base + off[5]),
                                  reinterpret_cast<float*>(base + off[6]), nullptr,
                                  reinterpret_cast<uint32_t*>(base + off[7]), base + off[8],
                                  need - off[8], stream);
  if (st != ASV_OK) return st;
  struct {
    void* dst;
    size_t o;
    size_t n;
  } outs[4] = {{out_accept_len_host, off[4], size_t(B) * 4},
               {out_tokens_host, off[5], R * 4},
               {out_D_host, off[6], R * 4},
               {out_req_status_host, off[7], size_t(B) * 4}};
  for (auto& o : outs) {
    if (!o.dst) continue;
    cudaError_t e = cudaMemcpyAsync(o.dst, base + o.o, o.n, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return ASV_OK;
}

asv_status rapid_verify(const float* z, const float* q, const int32_t* draft_ids, int B, int G, int V, float T,
                        float eta, float tail_frac, uint64_t seed, uint32_t offset, int32_t* out_accept_len,
                        int32_t* out_tokens, uint32_t* out_req_status, void* workspace, size_t ws_bytes,
                        cudaStream_t stream) {
  return rapid_verify_ex(z, q, draft_ids, B, G, V, T, eta, tail_frac, seed, offset, nullptr, out_accept_len,
                         out_tokens, out_req_status, workspace, ws_bytes, stream);
}

asv_status rapid_verify_ex(const float* z, const float* q, const int32_t* draft_ids, int B, int G, int V, float T,
                           float eta, float tail_frac, uint64_t seed, uint32_t offset, const asv_rapid_options* options,
                           int32_t* out_accept_len, int32_t* out_tokens, uint32_t* out_req_status, void* workspace,
                           size_t ws_bytes, cudaStream_t stream) {
  const int tail_mode = options ? options->tail_mode : 0;
  if (tail_mode != 0 && tail_mode != 1) return ASV_ERR_PARAM;
  if (B < 0 || G < 0 || V < 2) return ASV_ERR_SHAPE;
  if ((long long)B * (G + 1) * asv::kMaxCluster > 0x7fffffffLL) return ASV_ERR_SHAPE;
  if (B == 0) return ASV_OK;
  if (!z || !q || (G > 0 && !draft_ids) || !out_accept_len || !out_tokens || !out_req_status) return ASV_ERR_NULL;
  if (!workspace) return ASV_ERR_WORKSPACE;
  if (!aligned(z, 4) || !aligned(q, 4) || !aligned(draft_ids, 4) || !aligned(out_accept_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(out_req_status, 4) || !aligned(workspace, 256))
    return ASV_ERR_ALIGN;
  if (!std::isfinite(T) || !(T > 0.0f) || !std::isfinite(eta) || eta < 0.0f || !std::isfinite(tail_frac) ||
      tail_frac < 0.0f || tail_frac >= 1.0f)
    return ASV_ERR_PARAM;
  if (ws_bytes < asv_workspace_bytes(ASV_MODE_RAPID, B, G, V, ASV_F32)) return ASV_ERR_WORKSPACE;
  uint32_t* rapid_log = check_log_at(workspace, cluster_workspace_bytes(ASV_MODE_RAPID, B, G));
  bool bulk = (size_t(V) * 4) % 16 == 0 && aligned(z, 16) && aligned(q, 16);
  LaunchPlan pl;
  const float ln_tf = tail_frac > 0.0f ? std::log(tail_frac) : -INFINITY;
  cudaError_t e = plan_rapid(V, (long long)B * (G + 1), bulk, asv::rapid_needs_all_sums(tail_mode, ln_tf), &pl);
  if (e == cudaErrorInvalidValue) return ASV_ERR_SHAPE;
  if (e != cudaSuccess) return cuda_fail(e);
  asv::RapidArgs a;
  std::memset(&a, 0, sizeof(a));
  a.z = z;
  a.q = q;
  a.draft_ids = draft_ids;
  a.B = B;
  a.G = G;
  a.V = V;
  a.n_slice = pl.n_slice;
  a.bulk = pl.bulk;
  a.T = T;
  a.inv_T = 1.0f / T;
  a.eta = eta;
  a.tail_frac = tail_frac;
  a.ln_tail_frac = ln_tf;
  a.tail_mode = tail_mode;
  a.seed_lo = uint32_t(seed);
  a.seed_hi = uint32_t(seed >> 32);
  a.offset = offset;
  a.out_accept_len = out_accept_len;
  a.out_tokens = out_tokens;
  a.out_req_status = out_req_status;
  a.tickets = reinterpret_cast<uint32_t*>(workspace);
  a.records = reinterpret_cast<asv::RapidRecord*>(static_cast<char*>(workspace) + tickets_bytes(B));
  a.jobs = reinterpret_cast<asv::RapidJob*>(static_cast<char*>(workspace) + records_end(ASV_MODE_RAPID, B, G));
  a.draw_ctas = rapid_draw_ctas(V, B);
  a.check_log = rapid_log;
  e = asv::launch_rapid(a, pl, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return ASV_OK;
}

}  // extern "C"
