// asv_staged.cu -- the staged AsymSpec / E2-SCI verification kernel: one persistent CTA per SM,
// rows cut into units that bulk copies stage in shared memory, so that every input byte is read
// from HBM once and the arithmetic of one unit overlaps the copies of the next ones.
//
// Sources (web pages):
//   "AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs" (reading notes),
//     sec. 4.1 (delta-fusion token), sec. 4.2 (D = JSD(softmax a || softmax b), the CDA gate),
//     sec. 5 (delta-source ablation; beta and gamma over a grid);
//   "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia" (paper notes), Key design 3
//     (JSD(draft || target) against a threshold driven by an EWMA of the acceptance rate).
//
// Work decomposition.  A row (request r, position i) is V entries of each input; it is cut into
// n_unit units of n entries (the last one shorter).  Unit u = row * n_unit + q.  CTA c of a grid of
// G CTAs (one per SM, launched cooperatively, so all are resident at once) takes the units
// c, c + G, c + 2G, ... in that order.  Its warps:
//   producer   one lane copies each unit's slices of the inputs into one of kBuf shared-memory
//              buffers (cp.async.bulk, completing on the buffer's `full` mbarrier) and refills a
//              buffer when the compute warps release it (`empty`);
//   compute    kW warps run pass A of unit s (running maxima, sums of exp against a lazily moved
//              reference, the verifier argmax) and pass B of unit s - kLag (the per-entry
//              Jensen-Shannon terms against the row constants), both from shared memory.  After each
//              pass the warps' partials are combined in warp order and published to the workspace:
//              pass A with a release increment of the row's counter, pass B with an acq_rel ticket
//              on the row's second counter;
//   stats      waits for the row of each unit to have all n_unit pass-A partials, combines them in
//              unit order into the row constants (log-sum-exps, lse_b - lse_a, the argmax) and
//              hands them to the compute warps (`rc_ready`);
//   finaliser  takes the rows whose pass-B ticket this CTA drew last: D from the row's pass-B
//              sums, the gate, the outputs and the request-level scan (the last row of a request
//              scans its records), then clears the row's workspace entries.
// A row's units are consecutive and n_unit <= G, so they fall in at most two consecutive steps of
// the CTAs' unit sequences.  Pass B of step s waits for the pass-A partials of steps <= s + 1, and
// every CTA publishes those before it waits for anything another CTA does, so every wait ends while
// all CTAs are resident.  The waits are bounded all the same: a CTA whose wait expires marks the
// request ASV_REQ_TIMEOUT, raises the workspace's abort flag (the other CTAs' polls then stop),
// waits for its own copies in flight and leaves.
//
// Numerics are those of the cluster kernel (asv_jsd.cu): inputs widened exactly to fp32, exp2 of
// fma(x, log2e, -reference) on the special-function unit, compensated fp32 sums across warps and
// units, the even-symmetric narrow and wide divergence forms, the gate in double.
#include "asv_jsd_common.cuh"

namespace asv {
namespace {

constexpr int kW = 16;               // compute warps
constexpr int kWT = kW * 32;         // compute threads
constexpr int kProducerWarp = kW;    // the other roles' warps
constexpr int kStatsWarp = kW + 1;
constexpr int kFinalWarp = kW + 2;
constexpr int kThreads = (kW + 3) * 32;
constexpr int kBuf = 4;              // unit buffers
constexpr int kLag = 2;              // pass B runs kLag units behind pass A
constexpr int kSlots = 4;            // row-constant slots (>= kLag + 1, a power of 2)
constexpr int kFq = 4;               // finalisation queue entries
constexpr int kMaxUnits = 64;        // units per row the staging arrays hold
constexpr int kBudget = 200 * 1024;  // dynamic shared memory for the unit buffers
constexpr int kPartAStride = 32;     // words per pass-A partial in the workspace (128 bytes)
constexpr int kPartBStride = 16;     // words per pass-B partial (64 bytes)
constexpr unsigned long long kWaitNs = 1000000000ull;  // a wait is abandoned after 1 s

static_assert(kSlots >= kLag + 1 && (kSlots & (kSlots - 1)) == 0, "row-constant slots");
static_assert(kBuf >= kLag + 2, "the producer must never wait for a unit whose pass B waits on later units");
static_assert(sizeof(JsdPart) <= 4 * kPartAStride, "pass-A partial slot");

// ------------------------------------------------------------------ mbarriers, bulk copies, time

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false if `abort` is raised or a second passes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitNs) return false;
    }
  }
}

// The same wait by a whole warp, with one answer for every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global memory into
// this CTA's shared memory, completing on mbarrier `bar` (transaction bytes).
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void named_sync_compute() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWT) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void st_cg_zero4(void* p) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1, %1, %1, %1};" ::"l"(p), "r"(0u) : "memory");
}

// ------------------------------------------------------------------ shared state

struct FinJob {
  int32_t row;
  int32_t stop;
  int32_t pad[2];
  JsdRowConsts rc;
};

struct __align__(16) StagedShared {
  uint64_t full[kBuf];
  uint64_t empty[kBuf];
  uint64_t rc_ready[kSlots];
  uint64_t fq_full[kFq];
  uint64_t fq_free[kFq];
  JsdRowConsts rc[kSlots];
  FinJob fq[kFq];
  // per-warp partials of the last two units (pass A: maxima, sums, argmax slots; pass B: sums)
  float wa_m[2][kW][3];
  float wa_s[2][kW][3];
  float wa_av[2][kW][kMaxArg];
  int32_t wa_ai[2][kW][kMaxArg];
  float wb[2][kW][6];
  JsdPart from[kMaxUnits];          // stats warp: a row's pass-A partials
  float jsd_from[kMaxUnits][12];    // finaliser: a row's pass-B sums
  volatile int abort;
};

// ------------------------------------------------------------------ pass A state

template <typename T, int MODE, int DSRC, int NB, bool FUSE>
struct PassA {
  using G = GVec<T>;
  static constexpr int NT = JsdTraits<MODE>::NT;
  static constexpr int NP = G::kPairs;
  static constexpr int NA = NB + (FUSE ? 1 : 0);
  RunMax<T> rmax[NT];
  float mL[NT];
  float2 acc[NT];
  float bv[NA];
  int bi[NA];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      rmax[j] = RunMax<T>();
      mL[j] = 0.0f;
      acc[j] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int s = 0; s < NA; ++s) {
      bv[s] = -INFINITY;
      bi[s] = INT_MAX;
    }
  }

  // One vector (entries idx0 .. idx0 + VEC - 1 of the row) of every input.
  __device__ __forceinline__ void body(const uint4 (&cur)[NT], const int idx0, const float2 (&beta2)[NB]) {
    bool far = false;
#pragma unroll
    for (int j = 0; j < NT; ++j) far |= rmax[j].update(cur[j]);
    if (far) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float M = rmax[j].value();
        if (isfinite(M)) {
          const float nL = M * kLog2e;
          if (!rmax[j].started() || nL > mL[j] + kRefSlack) {
            const float f = (acc[j].x != 0.0f || acc[j].y != 0.0f) ? exp2f(mL[j] - nL) : 0.0f;
            acc[j] = fmul2(acc[j], make_float2(f, f));
            mL[j] = nL;
            rmax[j].set_threshold(nL);
          }
        }
      }
    }
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    float2 x[NT][NP];
#pragma unroll
    for (int j = 0; j < NT; ++j) G::pairs(cur[j], x[j]);
#pragma unroll
    for (int q2 = 0; q2 < NP; ++q2) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float2 y = ffma2(x[j][q2], l2e2, make_float2(-mL[j], -mL[j]));
        acc[j] = fadd2(acc[j], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
      }
    }
#pragma unroll
    for (int sl = 0; sl < NA; ++sl) {
      float2 sc[NP];
#pragma unroll
      for (int q2 = 0; q2 < NP; ++q2) {
        if constexpr (MODE == kModeAsym) {
          if (FUSE && sl == NB) sc[q2] = x[2][q2];
          else sc[q2] = ffma2(beta2[sl < NB ? sl : 0], delta2<DSRC>(x[0][q2], x[1][q2], x[2][q2]), x[2][q2]);
        } else {
          sc[q2] = x[JsdTraits<MODE>::TGT][q2];
        }
      }
      float vm = fmaxf(sc[0].x, sc[0].y);
#pragma unroll
      for (int q2 = 1; q2 < NP; ++q2) vm = fmaxf(vm, fmaxf(sc[q2].x, sc[q2].y));
      if (vm > bv[sl]) {
        int e_first = 2 * NP - 1;
#pragma unroll
        for (int q2 = NP - 1; q2 >= 0; --q2) {
          if (sc[q2].y == vm) e_first = 2 * q2 + 1;
          if (sc[q2].x == vm) e_first = 2 * q2;
        }
        bv[sl] = vm;
        bi[sl] = idx0 + e_first;
      }
    }
  }
};

// One vector of the divergence pair (xa, xb) against row constants r: narrow form for the whole
// vector when its largest u^2 is inside the domain (short form for the AsymSpec pair), else the
// per-entry path.
template <int NP>
__device__ __forceinline__ void pair_terms(const float2 (&xa)[NP], const float2 (&xb)[NP], const RowB& r, float2& acn,
                                           float& sn, float& sp, float& sq, const bool sh) {
  const float kS0 = sh ? ASV_JSD_SHORT_S0 : ASV_JSD_EVEN_S0;
  const float2 dl2 = make_float2(r.dL, r.dL);
  const float2 hl2e2 = make_float2(0.5f * kLog2e, 0.5f * kLog2e);
  const float2 nhml2 = make_float2(-r.hML, -r.hML);
  float2 s2[NP];
#pragma unroll
  for (int q2 = 0; q2 < NP; ++q2) {
    const float2 uu = fsub2(fsub2(xb[q2], xa[q2]), dl2);
    s2[q2] = fmul2(uu, uu);
  }
  float smax = fmax_nan(s2[0].x, s2[0].y);
#pragma unroll
  for (int q2 = 1; q2 < NP; ++q2) smax = fmax_nan(smax, fmax_nan(s2[q2].x, s2[q2].y));
  if (smax <= kS0) {
#pragma unroll
    for (int q2 = 0; q2 < NP; ++q2) {
      const float2 y = ffma2(fadd2(xa[q2], xb[q2]), hl2e2, nhml2);
      const float2 e = make_float2(ex2_approx(y.x), ex2_approx(y.y));
      acn = ffma2(fmul2(e, s2[q2]), sh ? asv_jsd_short2(s2[q2]) : asv_jsd_even2(s2[q2]), acn);
    }
  } else {
#pragma unroll
    for (int q2 = 0; q2 < NP; ++q2) {
      jsd_entry(xa[q2].x, xb[q2].x, r, sn, sp, sq);
      jsd_entry(xa[q2].y, xb[q2].y, r, sn, sp, sq);
    }
  }
}

// Row constants from a row's pass-A partials (`from[q]`, q < C, in unit order), by one whole warp;
// lane 0 writes them to `rc`.  Lane j < NT combines input j, lane NT + s argmax slot s, four units
// at a time; the running sum moves to a new reference when a later group holds a larger maximum.
template <int MODE, int NA, bool FUSE>
__device__ __forceinline__ void combine_row(const JsdPart* from, const uint32_t C, const int lane,
                                            JsdRowConsts& rc) {
  constexpr int NT = JsdTraits<MODE>::NT;
  const int j = lane < NT ? lane : 0;
  const int sl = (lane >= NT && lane < NT + NA) ? lane - NT : 0;
  float Mj = -INFINITY;
  DF Sj{0.0f, 0.0f};
  float av = -INFINITY;
  int ai = INT_MAX;
  for (uint32_t q0 = 0; q0 < C; q0 += 4) {
    float mx4[4], hi4[4], lo4[4], av4[4];
    int ai4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = q0 + u < C;
      const JsdPart& f = from[ok ? q0 + u : 0];
      mx4[u] = ok ? f.mx[j] : -INFINITY;
      hi4[u] = ok ? f.sum_hi[j] : 0.0f;
      lo4[u] = ok ? f.sum_lo[j] : 0.0f;
      av4[u] = ok ? f.argv[sl] : -INFINITY;
      ai4[u] = ok ? f.argi[sl] : INT_MAX;
    }
    float Mn = Mj;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      Mn = fmaxf(Mn, mx4[u]);
      argmax_merge(av, ai, av4[u], ai4[u]);
    }
    const float Rn = ref_of(Mn);
    if (Sj.hi != 0.0f) {
      const float g = exp2f(ref_of(Mj) - Rn);
      Sj = DF{Sj.hi * g, Sj.lo * g};
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (hi4[u] != 0.0f) {
        const float g = exp2f(ref_of(mx4[u]) - Rn);
        Sj = df_add(Sj, DF{hi4[u] * g, lo4[u] * g});
      }
    }
    Mj = Mn;
  }
  DF S[NT];
  float M[NT], MLr[NT];
#pragma unroll
  for (int jj = 0; jj < NT; ++jj) {
    M[jj] = __shfl_sync(0xffffffffu, Mj, jj);
    S[jj].hi = __shfl_sync(0xffffffffu, Sj.hi, jj);
    S[jj].lo = __shfl_sync(0xffffffffu, Sj.lo, jj);
    MLr[jj] = ref_of(M[jj]);
  }
  int i2[NA];
#pragma unroll
  for (int s2 = 0; s2 < NA; ++s2) i2[s2] = __shfl_sync(0xffffffffu, ai, NT + s2);
  if (lane == 0) {
    bool finite = true;
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      finite = finite && isfinite(M[jj]) && isfinite(S[jj].hi) && S[jj].hi > 0.0f;
      rc.M[jj] = M[jj];
      rc.ML[jj] = MLr[jj];
      rc.S_hi[jj] = S[jj].hi;
      rc.S_lo[jj] = S[jj].lo;
    }
    // lse_b - lse_a = (Mb - Ma) + ln(Sb / Sa) - (cb - ca) ln2, c = fma(M, log2e, -ML) the exact
    // rounding error of ML (the sums are against ML).
    float dL = 0.0f;
    if (finite) {
      const float ca = fmaf(M[0], kLog2e, -MLr[0]);
      const float cb = fmaf(M[1], kLog2e, -MLr[1]);
      const float ratio = (S[1].hi + S[1].lo) / (S[0].hi + S[0].lo);
      dL = (M[1] - M[0]) + (ln_split(ratio) - (cb - ca) * kLn2f);
    }
    rc.finite = finite ? 1 : 0;
    rc.dL = dL;
    rc.hML = 0.5f * MLr[0] + 0.5f * MLr[1];
    rc.dL2 = 0.0f;
    rc.hML2 = 0.0f;
    if constexpr (FUSE) {
      float dL2 = 0.0f;
      if (finite) {
        const float ca = fmaf(M[0], kLog2e, -MLr[0]);
        const float ct = fmaf(M[2], kLog2e, -MLr[2]);
        const float ratio = (S[2].hi + S[2].lo) / (S[0].hi + S[0].lo);
        dL2 = (M[2] - M[0]) + (ln_split(ratio) - (ct - ca) * kLn2f);
      }
      rc.dL2 = dL2;
      rc.hML2 = 0.5f * MLr[0] + 0.5f * MLr[2];
    }
#pragma unroll
    for (int s2 = 0; s2 < kMaxArg; ++s2) rc.rowi[s2] = s2 < NA ? i2[s2] : INT_MAX;
  }
}

// A request's outputs when its verification could not complete (a bounded wait expired).
__device__ void mark_timeout(const JsdArgs& p, const int row, const int lane) {
  const int R1 = p.K + 1;
  const int req = row / R1;
  for (int i = lane; i < R1; i += 32) p.out_tokens[size_t(req) * R1 + i] = -1;
  if (lane == 0) {
    p.out_accept_len[req] = 0;
    atomicOr(p.out_req_status + req, 4u);
    atomicExch(p.abort_flag, 1u);
  }
}

// ------------------------------------------------------------------ the kernel

template <typename T, int MODE, int DSRC, int NB, bool FUSE>
__global__ void __launch_bounds__(kThreads, 1) jsd_staged_kernel(const JsdArgs p) {
  using G = GVec<T>;
  using PA = PassA<T, MODE, DSRC, NB, FUSE>;
  constexpr int NT = JsdTraits<MODE>::NT;
  constexpr int VEC = G::kVec;
  constexpr int NP = G::kPairs;
  constexpr int NA = PA::NA;
  constexpr int NS = FUSE ? 6 : 3;   // pass-B sums
  constexpr bool kMulti = (NB > 1) || FUSE;
  static_assert(NA <= kMaxArg, "argmax slots");

  extern __shared__ __align__(128) unsigned char s_buf[];
  __shared__ StagedShared sh;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int G_ = int(gridDim.x);
  const int cta = int(blockIdx.x);
  const int C = p.n_unit;
  const int n = p.n_slice;
  const int V = p.V;
  const int my_units = cta < p.units ? (p.units - cta + G_ - 1) / G_ : 0;
  const size_t in_bytes = size_t(n) * G::kBytes;  // one input's slice in a buffer
  auto buf_addr = [&](int b, int j) { return s_buf + (size_t(b) * NT + j) * in_bytes; };

  if (tid == 0) {
    for (int b = 0; b < kBuf; ++b) {
      mbar_init(smem_addr(&sh.full[b]), 1);
      mbar_init(smem_addr(&sh.empty[b]), kW);
    }
    for (int k = 0; k < kSlots; ++k) mbar_init(smem_addr(&sh.rc_ready[k]), 1);
    for (int k = 0; k < kFq; ++k) {
      mbar_init(smem_addr(&sh.fq_full[k]), 1);
      mbar_init(smem_addr(&sh.fq_free[k]), 1);
    }
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < my_units; ++s) {
        const int b = s % kBuf;
        if (s >= kBuf && !mbar_wait(smem_addr(&sh.empty[b]), uint32_t((s / kBuf) - 1) & 1u, &sh.abort)) {
          sh.abort = 1;
          break;
        }
        if (sh.abort) break;
        const long long u = (long long)s * G_ + cta;
        const int row = int(u / C);
        const int v0 = int(u - (long long)row * C) * n;
        const int len = min(n, V - v0);
        const uint32_t bytes = uint32_t(len) * G::kBytes;
        mbar_arrive_expect_tx(smem_addr(&sh.full[b]), bytes * NT);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const char* src = static_cast<const char*>(p.x[j]) + (size_t(row) * size_t(V) + size_t(v0)) * G::kBytes;
          bulk_copy(smem_addr(buf_addr(b, j)), src, bytes, smem_addr(&sh.full[b]));
        }
        issued = s + 1;
      }
      // Never leave with copies in flight into this CTA's shared memory: wait for the last copies
      // of every buffer (earlier ones were consumed before their buffer was refilled).
      for (int s = max(0, issued - kBuf); s < issued; ++s) {
        const uint32_t bar = smem_addr(&sh.full[s % kBuf]);
        const unsigned long long t0 = global_ns();
        while (!mbar_try(bar, uint32_t(s / kBuf) & 1u) && global_ns() - t0 < kWaitNs) {
        }
      }
    }
    return;
  }

  if (warp == kStatsWarp) {
    // ---------------------------------------------------------------- stats
    const JsdPart* part_a = static_cast<const JsdPart*>(p.part_a);
    for (int s = 0; s < my_units; ++s) {
      const long long u = (long long)s * G_ + cta;
      const int row = int(u / C);
      // every lane polls the row's counter with acquire semantics
      bool ok = true;
      const unsigned long long t0 = global_ns();
      for (uint32_t it = 0;; ++it) {
        const uint32_t c = ld_acquire_gpu(p.row_cnt + row);
        if (__all_sync(0xffffffffu, c >= uint32_t(C))) break;
        if ((it & 15u) == 15u) {
          const bool stop = sh.abort || *reinterpret_cast<volatile uint32_t*>(p.abort_flag) != 0u ||
                            global_ns() - t0 > kWaitNs;
          if (__any_sync(0xffffffffu, stop)) {
            ok = false;
            break;
          }
        }
        __nanosleep(64);
      }
      const int k = s % kSlots;
      if (ok) {
        for (int q = lane; q < C; q += 32) {
          const char* src = reinterpret_cast<const char*>(part_a) + (size_t(row) * C + q) * (4 * kPartAStride);
          float4* dst = reinterpret_cast<float4*>(&sh.from[q]);
#pragma unroll
          for (int w4 = 0; w4 < int(sizeof(JsdPart) / 16); ++w4) dst[w4] = ld_cg_f4(src + 16 * w4);
        }
        __syncwarp();
        combine_row<MODE, NA, FUSE>(sh.from, uint32_t(C), lane, sh.rc[k]);
      } else {
        mark_timeout(p, row, lane);
        if (lane == 0) sh.abort = 1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh.rc_ready[k]));
      if (!ok) break;
    }
    return;
  }

  if (warp == kFinalWarp) {
    // ---------------------------------------------------------------- finaliser
    for (uint32_t jf = 0;; ++jf) {
      const int slot = int(jf % kFq);
      if (!warp_wait(smem_addr(&sh.fq_full[slot]), (jf / kFq) & 1u, &sh.abort)) break;
      const FinJob& job = sh.fq[slot];
      if (job.stop) break;
      const int row = job.row;
      for (int q = lane; q < C; q += 32) {
        const float* src = p.part_b + (size_t(row) * C + q) * kPartBStride;
#pragma unroll
        for (int w4 = 0; w4 < 3; ++w4) {
          const float4 v = ld_cg_f4(src + 4 * w4);
          sh.jsd_from[q][4 * w4 + 0] = v.x;
          sh.jsd_from[q][4 * w4 + 1] = v.y;
          sh.jsd_from[q][4 * w4 + 2] = v.z;
          sh.jsd_from[q][4 * w4 + 3] = v.w;
        }
      }
      // The draft token and its verifier / compressed-drafter logits (single-outcome kernels).
      const int R1 = p.K + 1;
      const int req = row / R1;
      const int pos = row - req * R1;
      int d = -1;
      float xd = 0.0f;
      if (!kMulti && (lane == 1 || lane == 2) && pos < p.K) {
        d = p.draft_ids[size_t(req) * p.K + pos];
        if (MODE == kModeAsym && job.rc.finite && d >= 0 && d < V)
          xd = G::at(p.x[lane == 1 ? NT - 1 : 1], size_t(row) * size_t(V) + size_t(d));
      }
      __syncwarp();
      jsd_finalize_row<T, MODE, NB, FUSE>(p, row, job.rc, sh.jsd_from, uint32_t(C), lane, d, xd);
      __syncwarp();
      // The row's workspace entries back to zero (every unit of the row has read its pass-A
      // partials before its pass-B ticket, so nobody reads them any more).
      for (int q = lane; q < C; q += 32) {
        char* a = reinterpret_cast<char*>(p.part_a) + (size_t(row) * C + q) * (4 * kPartAStride);
#pragma unroll
        for (int w4 = 0; w4 < int(sizeof(JsdPart) / 16); ++w4) st_cg_zero4(a + 16 * w4);
        float* bsum = p.part_b + (size_t(row) * C + q) * kPartBStride;
#pragma unroll
        for (int w4 = 0; w4 < 3; ++w4) st_cg_zero4(bsum + 4 * w4);
      }
      if (lane == 0) {
        p.row_cnt[row] = 0u;
        p.row_jcnt[row] = 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh.fq_free[slot]));
    }
    return;
  }

  // ------------------------------------------------------------------ compute warps
  float2 beta2[NB];
#pragma unroll
  for (int sl = 0; sl < NB; ++sl) beta2[sl] = make_float2(p.betas[sl], p.betas[sl]);
  constexpr bool kPairShort = MODE == kModeAsym;
  uint32_t jq = 0;  // finalisation jobs queued (warp 0, lane 0)

  // Queue a job for the finaliser (warp 0): the row and its constants, or the stop mark.
  auto enqueue = [&](int row, bool stop, const JsdRowConsts* rc) {
    const int slot = int(jq % kFq);
    bool ok = true;
    if (lane == 0 && jq >= uint32_t(kFq))
      ok = mbar_wait(smem_addr(&sh.fq_free[slot]), ((jq / kFq) - 1) & 1u, &sh.abort);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) sh.abort = 1;
      return false;
    }
    FinJob& job = sh.fq[slot];
    if (rc) {
      constexpr int kWords = int(sizeof(JsdRowConsts) / 4);
      static_assert(kWords <= 32, "row constants");
      if (lane < kWords) reinterpret_cast<uint32_t*>(&job.rc)[lane] = reinterpret_cast<const uint32_t*>(rc)[lane];
    }
    if (lane == 0) {
      job.row = row;
      job.stop = stop ? 1 : 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&sh.fq_full[slot]));
    ++jq;
    return true;
  };

  // Every compute warp runs the same sequence of named barriers, so a warp that gives up a wait
  // (`dead`) keeps going through the loop without touching data until the end.
  bool dead = false;
  for (int s = 0; s < my_units + kLag; ++s) {
    if (s < my_units) {
      // ---------------------------------------------------------------- pass A of unit s
      const int b = s % kBuf;
      if (!dead && !warp_wait(smem_addr(&sh.full[b]), uint32_t(s / kBuf) & 1u, &sh.abort)) {
        sh.abort = 1;
        dead = true;
      }
      const long long u = (long long)s * G_ + cta;
      const int row = int(u / C);
      const int v0 = int(u - (long long)row * C) * n;
      const int len = min(n, V - v0);
      const int nvec = dead ? 0 : len / VEC;
      PA st;
      st.reset();
      const char* bin[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) bin[j] = reinterpret_cast<const char*>(buf_addr(b, j));
      {
        int vi = tid;
        uint4 cur[NT], nxt[NT];
        if (vi < nvec) {
#pragma unroll
          for (int j = 0; j < NT; ++j) cur[j] = lds128(bin[j] + size_t(vi) * 16);
        }
        for (; vi < nvec; vi += kWT) {
          const int vn = vi + kWT;
          if (vn < nvec) {
#pragma unroll
            for (int j = 0; j < NT; ++j) nxt[j] = lds128(bin[j] + size_t(vn) * 16);
          }
          st.body(cur, v0 + vi * VEC, beta2);
#pragma unroll
          for (int j = 0; j < NT; ++j) cur[j] = nxt[j];
        }
      }
      // warp partials: maxima, argmax slots, sums against the warp maximum
      const int ws = s & 1;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float wm = warp_max(st.rmax[j].value());
        const float sm = st.acc[j].x + st.acc[j].y;
        const float moved = (sm != 0.0f) ? sm * exp2f(st.mL[j] - ref_of(wm)) : 0.0f;
        const float wsum = warp_sumf(moved);
        if (lane == 0) {
          sh.wa_m[ws][warp][j] = wm;
          sh.wa_s[ws][warp][j] = wsum;
        }
      }
#pragma unroll
      for (int sl = 0; sl < NA; ++sl) {
        warp_argmax(st.bv[sl], st.bi[sl]);
        if (lane == 0) {
          sh.wa_av[ws][warp][sl] = st.bv[sl];
          sh.wa_ai[ws][warp][sl] = st.bi[sl];
        }
      }
      named_sync_compute();
      if (warp == 0 && __all_sync(0xffffffffu, !dead && sh.abort == 0)) {
        // the unit's partial: lane j < NT input j, lane NT + s argmax slot s, over the warps in order
        char* dst = reinterpret_cast<char*>(p.part_a) + size_t(u) * (4 * kPartAStride);
        JsdPart* dp = reinterpret_cast<JsdPart*>(dst);
        if (lane < NT) {
          const int j = lane;
          float Mc = sh.wa_m[ws][0][j];
#pragma unroll
          for (int w = 1; w < kW; ++w) Mc = fmaxf(Mc, sh.wa_m[ws][w][j]);
          const float Rc = ref_of(Mc);
          DF dsum{0.0f, 0.0f};
#pragma unroll
          for (int w = 0; w < kW; ++w) {
            const float sw = sh.wa_s[ws][w][j];
            if (sw != 0.0f) dsum = df_add(dsum, DF{sw * exp2f(ref_of(sh.wa_m[ws][w][j]) - Rc), 0.0f});
          }
          dp->mx[j] = Mc;
          dp->sum_hi[j] = dsum.hi;
          dp->sum_lo[j] = dsum.lo;
        } else if (lane < NT + NA) {
          const int sl = lane - NT;
          float v = sh.wa_av[ws][0][sl];
          int i = sh.wa_ai[ws][0][sl];
#pragma unroll
          for (int w = 1; w < kW; ++w) argmax_merge(v, i, sh.wa_av[ws][w][sl], sh.wa_ai[ws][w][sl]);
          dp->argv[sl] = v;
          dp->argi[sl] = i;
        }
        __syncwarp();
        if (lane == 0) red_add_release_gpu(p.row_cnt + row, 1u);
      }
    }
    if (s >= kLag) {
      // ---------------------------------------------------------------- pass B of unit s - kLag
      const int s2 = s - kLag;
      const int b2 = s2 % kBuf;
      const int k = s2 % kSlots;
      if (!dead && (!warp_wait(smem_addr(&sh.rc_ready[k]), uint32_t(s2 / kSlots) & 1u, &sh.abort) ||
                    __any_sync(0xffffffffu, sh.abort != 0))) {
        sh.abort = 1;
        dead = true;
      }
      const long long u2 = (long long)s2 * G_ + cta;
      const int row2 = int(u2 / C);
      const int v02 = int(u2 - (long long)row2 * C) * n;
      const int len2 = min(n, V - v02);
      const int nvec2 = len2 / VEC;
      const JsdRowConsts& rc = sh.rc[k];
      const bool finite = !dead && rc.finite != 0;
      RowB rb, rbt;
      rb.dL = rc.dL;
      rb.MaL = rc.ML[0];
      rb.MbL = rc.ML[1];
      rb.hML = rc.hML;
      rbt = rb;
      if constexpr (FUSE) {
        rbt.dL = rc.dL2;
        rbt.MbL = rc.ML[2];
        rbt.hML = rc.hML2;
      }
      float2 accn = make_float2(0.0f, 0.0f), accn2 = make_float2(0.0f, 0.0f);
      float an = 0.0f, ap = 0.0f, aq = 0.0f, an2 = 0.0f, ap2 = 0.0f, aq2 = 0.0f;
      if (finite) {
        const char* ba = reinterpret_cast<const char*>(buf_addr(b2, 0));
        const char* bb = reinterpret_cast<const char*>(buf_addr(b2, 1));
        const char* bt = reinterpret_cast<const char*>(buf_addr(b2, NT - 1));
        for (int vi = tid; vi < nvec2; vi += kWT) {
          float2 xa[NP], xb[NP];
          G::pairs(lds128(ba + size_t(vi) * 16), xa);
          G::pairs(lds128(bb + size_t(vi) * 16), xb);
          pair_terms<NP>(xa, xb, rb, accn, an, ap, aq, kPairShort);
          if constexpr (FUSE) {
            float2 xt[NP];
            G::pairs(lds128(bt + size_t(vi) * 16), xt);
            pair_terms<NP>(xa, xt, rbt, accn2, an2, ap2, aq2, false);
          }
        }
      }
      // the buffer is free once every lane of every compute warp has read it
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(smem_addr(&sh.empty[b2]));
      const int wsb = s2 & 1;
      {
        const float wn = warp_sumf((accn.x + accn.y) + an);
        const float wp = warp_sumf(ap);
        const float wq = warp_sumf(aq);
        if (lane == 0) {
          sh.wb[wsb][warp][0] = wn;
          sh.wb[wsb][warp][1] = wp;
          sh.wb[wsb][warp][2] = wq;
        }
        if constexpr (FUSE) {
          const float wn2 = warp_sumf((accn2.x + accn2.y) + an2);
          const float wp2 = warp_sumf(ap2);
          const float wq2 = warp_sumf(aq2);
          if (lane == 0) {
            sh.wb[wsb][warp][3] = wn2;
            sh.wb[wsb][warp][4] = wp2;
            sh.wb[wsb][warp][5] = wq2;
          }
        }
      }
      named_sync_compute();
      if (warp == 0 && __all_sync(0xffffffffu, !dead && sh.abort == 0)) {
        float* dst = p.part_b + size_t(u2) * kPartBStride;
        if (lane < NS) {
          DF dm{sh.wb[wsb][0][lane], 0.0f};
#pragma unroll
          for (int w = 1; w < kW; ++w) dm = df_add(dm, DF{sh.wb[wsb][w][lane], 0.0f});
          dst[2 * lane] = dm.hi;
          dst[2 * lane + 1] = dm.lo;
        }
        __syncwarp();
        uint32_t ticket = 0;
        if (lane == 0) ticket = atom_add_acq_rel_gpu(p.row_jcnt + row2, 1u);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        // The unit that completes the row hands it to this CTA's finaliser.
        if (ticket == uint32_t(C - 1) && !enqueue(row2, false, &rc)) dead = true;
      }
    }
  }
  if (warp == 0) enqueue(0, true, nullptr);
  (void)kMulti;
}

using StagedKernel = void (*)(const JsdArgs);

// variant 0: single outcome; 1: the all-(beta, gamma) sweep (4 betas); 2: AsymSpec fused with E2-SCI.
template <typename T>
StagedKernel pick_typed(int mode, int dsrc, int variant) {
  if (variant == 1) return jsd_staged_kernel<T, kModeAsym, 0, 4, false>;
  if (variant == 2) return jsd_staged_kernel<T, kModeAsym, 0, 1, true>;
  if (mode == kModeSci) return jsd_staged_kernel<T, kModeSci, 0, 1, false>;
  if (dsrc == 1) return jsd_staged_kernel<T, kModeAsym, 1, 1, false>;
  if (dsrc == 2) return jsd_staged_kernel<T, kModeAsym, 2, 1, false>;
  return jsd_staged_kernel<T, kModeAsym, 0, 1, false>;
}

StagedKernel pick(int mode, int dtype, int dsrc, int variant) {
  return dtype == 0 ? pick_typed<float>(mode, dsrc, variant) : pick_typed<bf16_t>(mode, dsrc, variant);
}

}  // namespace

StagedPlan staged_plan(int V, int elem_bytes, int nt) {
  const int vec = 16 / elem_bytes;
  int n_max = kBudget / (kBuf * nt * elem_bytes);
  n_max -= n_max % vec;
  StagedPlan pl;
  pl.n_unit = (V + n_max - 1) / n_max;
  int n = (V + pl.n_unit - 1) / pl.n_unit;
  n = (n + vec - 1) / vec * vec;
  pl.n = n;
  pl.smem = kBuf * nt * n * elem_bytes;
  return pl;
}

int staged_threads() { return kThreads; }

// Workspace of the staged kernel: [row_cnt: rows][row_jcnt: rows] (256-byte padded), the abort flag
// (256 bytes), the pass-A partials (128 bytes per unit) and the pass-B partials (64 bytes per unit).
size_t staged_workspace_bytes(long long rows, int n_unit) {
  const size_t cnt = (size_t(rows) * 8 + 255) / 256 * 256;
  const size_t units = size_t(rows) * size_t(n_unit);
  return cnt + 256 + units * size_t(4 * (kPartAStride + kPartBStride));
}

// Raises the instantiation's dynamic shared-memory limit to the whole buffer budget (every plan's
// buffers fit in it) and returns how many of its CTAs the device holds at once with that much.
int staged_grid(int mode, int dtype, const JsdArgs& a, const StagedPlan& plan) {
  (void)plan;
  StagedKernel kern = pick(mode, dtype, a.delta_source, a.variant);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBudget) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kBudget) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm * sms;
}

cudaError_t launch_jsd_staged(int mode, int dtype, const JsdArgs& a, const StagedPlan& plan, int grid,
                              cudaStream_t s) {
  StagedKernel kern = pick(mode, dtype, a.delta_source, a.variant);  // (its limit was raised by staged_grid)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(unsigned(kThreads), 1, 1);
  cfg.dynamicSmemBytes = size_t(plan.smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace asv
