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
// n_unit units of n entries (the last one shorter), and m consecutive units form a chunk (n_unit =
// n_chunk * m).  Chunk ch = row * n_chunk + qc.  CTA c of a grid of G CTAs (one per SM, launched
// cooperatively, so all are resident at once) takes the chunks c, c + G, c + 2G, ... in that order,
// a unit at a time.  Its warps:
//   producers    two warps (one lane each) issue cp.async.bulk copies into two rings of shared-memory
//                buffers: the A ring receives each unit's slices of every input from HBM; the B
//                ring, refilled as pass B frees it (kLag units behind), receives the divergence
//                pair's slices again, which L2 still holds;
//   compute      kW warps run pass A of unit s from the A ring (running maxima, sums of exp against
//                a lazily moved reference, the verifier argmax) and pass B of unit s - kLag from the
//                B ring (the per-entry Jensen-Shannon terms against the row constants), carrying
//                per-thread state across the units of a chunk; at a chunk's last unit each warp
//                reduces its state and leaves it in a shared-memory slot;
//   publishers   one warp combines the compute warps' pass-A partials of a chunk in warp order and
//                publishes them to the workspace with a release increment of the row's counter;
//                another does the same for pass B;
//   stats        kStatsN warps (chunk t of this CTA to warp t % kStatsN) wait for the row of a chunk
//                to have all n_chunk pass-A partials, combine them in chunk order into the row
//                constants (log-sum-exps, lse_b - lse_a, the argmax) and hand them to the compute
//                warps;
//   finaliser    for every row whose last chunk is this CTA's, waits for all n_chunk pass-B
//                partials, then computes D, the gate, the outputs and the request-level scan (the
//                last row of a request scans its records), and clears the row's workspace entries.
// Every hand-over inside a CTA goes through an mbarrier pair (ready / free), so no warp waits for a
// slower one except for data it needs.  A row's chunks are consecutive and n_chunk <= G / 2, so they
// fall in at most two consecutive steps of the CTAs' chunk sequences; the row constants of step t
// need the pass-A partials of steps <= t + 1, which a CTA publishes without waiting for anything
// another CTA does, so every wait ends while all CTAs are resident.  The waits are bounded all the
// same: a CTA whose wait expires marks the request ASV_REQ_TIMEOUT, raises the workspace's abort
// flag (the other CTAs' polls then stop), waits for its own copies in flight and leaves.
//
// Numerics are those of the cluster kernel (asv_jsd.cu): inputs widened exactly to fp32, exp2 of
// fma(x, log2e, -reference) on the special-function unit, compensated fp32 sums across warps and
// units, the even-symmetric narrow and wide divergence forms, the gate in double.
#include "asv_jsd_common.cuh"

namespace asv {
namespace {

constexpr int kW = 16;               // compute warps
constexpr int kWT = kW * 32;         // compute threads
constexpr int kStatsN = 4;           // stats warps (unit s goes to stats warp s % kStatsN)
constexpr int kProducerWarp = kW;    // the other roles' warps: A-ring producer,
constexpr int kProducerBWarp = kW + 1;  // B-ring producer,
constexpr int kPubAWarp = kW + 2;    // publishers,
constexpr int kPubBWarp = kW + 3;
constexpr int kStatsWarp0 = kW + 4;  // stats warps and the finaliser
constexpr int kFinalWarp = kW + 4 + kStatsN;
constexpr int kThreads = (kW + 5 + kStatsN) * 32;
constexpr int kRingA = 3;            // A-ring buffers (every input of a unit, from HBM)
constexpr int kRingB = 2;            // B-ring buffers (the divergence pair of a unit, from L2)
constexpr int kChunk = 4;            // largest number of units per chunk
constexpr int kLag = kChunk + 2;     // pass B runs kLag units behind pass A
constexpr int kSlots = 4;            // chunk slots: partials and row constants (a power of 2)
constexpr int kMaxUnits = 40;        // chunks per row the staging arrays hold
constexpr int kBudget = 198 * 1024;  // dynamic shared memory for the two rings
constexpr int kPartAStride = 32;     // words per pass-A partial in the workspace (128 bytes)
constexpr int kPartBStride = 16;     // words per pass-B partial (64 bytes)
constexpr unsigned long long kWaitNs = 1000000000ull;  // a wait is abandoned after 1 s

static_assert((kSlots & (kSlots - 1)) == 0 && kSlots >= 2, "chunk slots");
static_assert(kRingB >= 2, "the producer's B-ring wait must not depend on the compute warps' current unit");
static_assert(kSlots % kStatsN == 0, "a stats warp reuses only its own row-constant slots");
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

// The same test, but the thread may be suspended for up to `hint_ns` while the phase is incomplete
// (it resumes when the phase completes), so a waiting warp takes no issue slots from the others.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false if `abort` is raised or a second passes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitNs) return false;
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

__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void st_cg_zero4(void* p) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1, %1, %1, %1};" ::"l"(p), "r"(0u) : "memory");
}

// ------------------------------------------------------------------ shared state

struct __align__(16) StagedShared {
  uint64_t full_a[kRingA], empty_a[kRingA];
  uint64_t full_b[kRingB], empty_b[kRingB];
  uint64_t a_ready[kSlots], a_free[kSlots];    // compute -> pass-A publisher
  uint64_t b_ready[kSlots], b_free[kSlots];    // compute -> pass-B publisher
  uint64_t rc_ready[kSlots], rc_free[kSlots];  // stats -> compute
  JsdRowConsts rc[kSlots];
  JsdRowConsts fin_rc;
  // per-warp partials (pass A: maxima, sums, argmax slots; pass B: sums)
  float wa_m[kSlots][kW][3];
  float wa_s[kSlots][kW][3];
  float wa_av[kSlots][kW][kMaxArg];
  int32_t wa_ai[kSlots][kW][kMaxArg];
  float wb[kSlots][kW][6];
  JsdPart from[kStatsN + 1][kMaxUnits];  // a row's pass-A partials: the stats warps and the finaliser
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

// Where unit s of this CTA lies: its chunk (the CTA's chunk counter t, the global chunk id), its
// position j in the chunk, its row, unit index q in the row, first entry and length.
struct UnitPos {
  int t, j, ch, row, qc, q, v0, len;
};

__device__ __forceinline__ UnitPos unit_pos(int s, int G, int cta, int nch, int m, int n, int V) {
  UnitPos r;
  r.t = s / m;
  r.j = s - r.t * m;
  const long long ch = (long long)r.t * G + cta;
  r.row = int(ch / nch);
  r.qc = int(ch - (long long)r.row * nch);
  r.ch = r.row * nch + r.qc;
  r.q = r.qc * m + r.j;
  r.v0 = r.q * n;
  r.len = min(n, V - r.v0);
  return r;
}

// A row's pass-A partials (one per chunk) from the workspace into `from` (lanes take chunks), then
// the row constants into `rc` (whole warp).
template <int MODE, int NA, bool FUSE>
__device__ __forceinline__ void gather_row(const JsdArgs& p, int row, int nch, int lane, JsdPart* from,
                                           JsdRowConsts& rc) {
  for (int q = lane; q < nch; q += 32) {
    const char* src = static_cast<const char*>(p.part_a) + (size_t(row) * nch + q) * (4 * kPartAStride);
    float4* dst = reinterpret_cast<float4*>(&from[q]);
#pragma unroll
    for (int w4 = 0; w4 < int(sizeof(JsdPart) / 16); ++w4) dst[w4] = ld_cg_f4(src + 16 * w4);
  }
  __syncwarp();
  combine_row<MODE, NA, FUSE>(from, uint32_t(nch), lane, rc);
  __syncwarp();
}

// Every lane polls `*cnt` (acquire) until it reaches `target`; false if the workspace's abort flag
// or this CTA's is raised, or a second passes.
__device__ __forceinline__ bool poll_count(const uint32_t* cnt, uint32_t target, const JsdArgs& p,
                                           const volatile int* abort) {
  const unsigned long long t0 = global_ns();
  uint32_t nap = 32;
  for (uint32_t it = 0;; ++it) {
    const uint32_t c = ld_acquire_gpu(cnt);
    if (__all_sync(0xffffffffu, c >= target)) return true;
    if ((it & 7u) == 7u) {
      const bool stop = *abort || *reinterpret_cast<volatile uint32_t*>(p.abort_flag) != 0u ||
                        global_ns() - t0 > kWaitNs;
      if (__any_sync(0xffffffffu, stop)) return false;
    }
    __nanosleep(nap);  // back off (up to 1 us) while the other CTAs catch up
    if (nap < 1024u) nap *= 2u;
  }
}

template <typename T, int MODE, int DSRC, int NB, bool FUSE>
__global__ void __launch_bounds__(kThreads, 1) jsd_staged_kernel(const JsdArgs p) {
  using G = GVec<T>;
  using PA = PassA<T, MODE, DSRC, NB, FUSE>;
  constexpr int NT = JsdTraits<MODE>::NT;
  constexpr int NBI = FUSE ? 3 : 2;  // inputs pass B reads: the pair (fused: and the target)
  constexpr int VEC = G::kVec;
  constexpr int NP = G::kPairs;
  constexpr int NA = PA::NA;
  constexpr int NS = FUSE ? 6 : 3;   // pass-B sums
  constexpr bool kMulti = (NB > 1) || FUSE;
  static_assert(NA <= kMaxArg, "argmax slots");
  (void)kMulti;

  extern __shared__ __align__(128) unsigned char s_buf[];
  __shared__ StagedShared sh;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int G_ = int(gridDim.x);
  const int cta = int(blockIdx.x);
  const int m = p.chunk_units;
  const int nch = p.n_unit / m;  // chunks per row
  const int n = p.n_slice;
  const int V = p.V;
  const int chunks = p.units / m;
  const int my_chunks = cta < chunks ? (chunks - cta + G_ - 1) / G_ : 0;
  const int my_units = my_chunks * m;
  const size_t in_bytes = size_t(n) * G::kBytes;  // one input's slice in a buffer
  unsigned char* ring_a = s_buf;
  unsigned char* ring_b = s_buf + size_t(kRingA) * NT * in_bytes;
  auto a_addr = [&](int i, int j) { return ring_a + (size_t(i) * NT + j) * in_bytes; };
  auto b_addr = [&](int i, int j) { return ring_b + (size_t(i) * NBI + j) * in_bytes; };
  auto bar = [](uint64_t& b) { return smem_addr(&b); };
#ifdef ASV_CHECKED
  uint32_t dyn_smem = 0;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_smem));
#else
  const uint32_t dyn_smem = 0;
#endif
  (void)dyn_smem;
  const int rows = p.B * (p.K + 1);

  if (tid == 0) {
    for (int i = 0; i < kRingA; ++i) {
      mbar_init(bar(sh.full_a[i]), 1);
      mbar_init(bar(sh.empty_a[i]), kW);
    }
    for (int i = 0; i < kRingB; ++i) {
      mbar_init(bar(sh.full_b[i]), 1);
      mbar_init(bar(sh.empty_b[i]), kW);
    }
    for (int k = 0; k < kSlots; ++k) {
      mbar_init(bar(sh.a_ready[k]), kW);
      mbar_init(bar(sh.a_free[k]), 1);
      mbar_init(bar(sh.b_ready[k]), kW);
      mbar_init(bar(sh.b_free[k]), 1);
      mbar_init(bar(sh.rc_ready[k]), 1);
      mbar_init(bar(sh.rc_free[k]), kW);
    }
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == kProducerWarp || warp == kProducerBWarp) {
    // ---------------------------------------------------------------- producers
    // A ring: unit y's slices of every input as soon as its buffer is free.  B ring (its own warp,
    // so that its waits never hold up the A ring): the divergence pair of unit s2 -- pass B of a
    // unit runs at compute step unit + kLag; the wait for a free B buffer is on pass B of unit
    // s2 - kRingB, never on a unit the compute warps need before they can free it.
    const bool ring_a_role = warp == kProducerWarp;
    if (lane == 0) {
      const int nbuf = ring_a_role ? kRingA : kRingB;
      const int nin = ring_a_role ? NT : NBI;
      uint64_t* full = ring_a_role ? sh.full_a : sh.full_b;
      uint64_t* empty = ring_a_role ? sh.empty_a : sh.empty_b;
      int issued = 0;
      for (int y = 0; y < my_units && !sh.abort; ++y) {
        const int i = y % nbuf;
        if (y >= nbuf && !mbar_wait(bar(empty[i]), uint32_t(y / nbuf - 1) & 1u, &sh.abort)) break;
        const UnitPos up = unit_pos(y, G_, cta, nch, m, n, V);
        const uint32_t bytes = uint32_t(up.len) * G::kBytes;
        const size_t off = (size_t(up.row) * size_t(V) + size_t(up.v0)) * G::kBytes;
        // (checked build: the unit inside the batch and its row, the buffers inside shared memory;
        // a unit that fails is not copied, and the waits for it run out -- the call then aborts)
        if (!ASV_GUARD(p, up.row < rows && up.len > 0 && up.v0 + up.len <= V && nch <= kMaxUnits &&
                              uint32_t(((ring_a_role ? a_addr(i, nin - 1) : b_addr(i, nin - 1)) - s_buf) + bytes) <=
                                  dyn_smem))
          break;
        mbar_arrive_expect_tx(bar(full[i]), bytes * nin);
        for (int j = 0; j < nin; ++j) {
          const int src = ring_a_role ? j : (j < 2 ? j : NT - 1);
          unsigned char* dst = ring_a_role ? a_addr(i, j) : b_addr(i, j);
          bulk_copy(smem_addr(dst), static_cast<const char*>(p.x[src]) + off, bytes, bar(full[i]));
        }
        issued = y + 1;
      }
      if (sh.abort) {
        // Never leave with copies in flight into this CTA's shared memory: wait for the last copies
        // of every buffer (earlier ones were consumed before their buffer was refilled).
        for (int y = max(0, issued - nbuf); y < issued; ++y) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try(bar(full[y % nbuf]), uint32_t(y / nbuf) & 1u) && global_ns() - t0 < kWaitNs) {
          }
        }
      }
    }
    return;
  }

  if (warp == kPubAWarp || warp == kPubBWarp) {
    // ---------------------------------------------------------------- publishers (one chunk a step)
    const bool is_a = warp == kPubAWarp;
    for (int t = 0; t < my_chunks; ++t) {
      const int k = t % kSlots;
      if (!warp_wait(bar(is_a ? sh.a_ready[k] : sh.b_ready[k]), uint32_t(t / kSlots) & 1u, &sh.abort)) {
        if (lane == 0) sh.abort = 1;
        break;
      }
      const UnitPos up = unit_pos(t * m, G_, cta, nch, m, n, V);
      const size_t ch = size_t(up.ch);
      if (!ASV_GUARD(p, up.row < rows && ch < size_t(p.units))) {
        if (lane == 0) sh.abort = 1;
        break;
      }
      if (is_a) {
        // lane j < NT: input j; lane NT + s: argmax slot s -- over the compute warps in order
        JsdPart* dp = reinterpret_cast<JsdPart*>(static_cast<char*>(p.part_a) + ch * (4 * kPartAStride));
        if (lane < NT) {
          const int j = lane;
          float mw[kW], sw[kW];
#pragma unroll
          for (int w = 0; w < kW; ++w) {
            mw[w] = sh.wa_m[k][w][j];
            sw[w] = sh.wa_s[k][w][j];
          }
          float Mc = mw[0];
#pragma unroll
          for (int w = 1; w < kW; ++w) Mc = fmaxf(Mc, mw[w]);
          const float Rc = ref_of(Mc);
          DF dsum{0.0f, 0.0f};
#pragma unroll
          for (int w = 0; w < kW; ++w)
            if (sw[w] != 0.0f) dsum = df_add(dsum, DF{sw[w] * exp2f(ref_of(mw[w]) - Rc), 0.0f});
          dp->mx[j] = Mc;
          dp->sum_hi[j] = dsum.hi;
          dp->sum_lo[j] = dsum.lo;
        } else if (lane < NT + NA) {
          const int sl = lane - NT;
          float v = sh.wa_av[k][0][sl];
          int i = sh.wa_ai[k][0][sl];
#pragma unroll
          for (int w = 1; w < kW; ++w) argmax_merge(v, i, sh.wa_av[k][w][sl], sh.wa_ai[k][w][sl]);
          dp->argv[sl] = v;
          dp->argi[sl] = i;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(sh.a_free[k]));
          red_add_release_gpu(p.row_cnt + up.row, 1u);
        }
      } else {
        float* dst = p.part_b + ch * kPartBStride;
        if (lane < NS) {
          DF dm{sh.wb[k][0][lane], 0.0f};
#pragma unroll
          for (int w = 1; w < kW; ++w) dm = df_add(dm, DF{sh.wb[k][w][lane], 0.0f});
          dst[2 * lane] = dm.hi;
          dst[2 * lane + 1] = dm.lo;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(sh.b_free[k]));
          red_add_release_gpu(p.row_jcnt + up.row, 1u);
        }
      }
    }
    return;
  }

  if (warp >= kStatsWarp0 && warp < kStatsWarp0 + kStatsN) {
    // ---------------------------------------------------------------- stats (chunks t with t % kStatsN == w)
    const int sw = warp - kStatsWarp0;
    for (int t = sw; t < my_chunks; t += kStatsN) {
      const int k = t % kSlots;
      const UnitPos up = unit_pos(t * m, G_, cta, nch, m, n, V);
      bool ok = t < kSlots || warp_wait(bar(sh.rc_free[k]), uint32_t(t / kSlots - 1) & 1u, &sh.abort);
      ok = ok && ASV_GUARD(p, up.row < rows && nch <= kMaxUnits);
      ok = ok && poll_count(p.row_cnt + up.row, uint32_t(nch), p, &sh.abort);
      if (ok) {
        gather_row<MODE, NA, FUSE>(p, up.row, nch, lane, sh.from[sw], sh.rc[k]);
      } else {
        mark_timeout(p, up.row, lane);
        if (lane == 0) sh.abort = 1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sh.rc_ready[k]));
      if (!ok) break;
    }
    return;
  }

  if (warp == kFinalWarp) {
    // ---------------------------------------------------------------- finaliser
    // The rows whose last chunk is this CTA's, in order.
    for (int t = 0; t < my_chunks; ++t) {
      const UnitPos up = unit_pos(t * m, G_, cta, nch, m, n, V);
      if (up.qc != nch - 1) continue;
      const int row = up.row;
      if (!ASV_GUARD(p, row < rows && nch <= kMaxUnits)) break;
      if (!poll_count(p.row_jcnt + row, uint32_t(nch), p, &sh.abort)) {
        mark_timeout(p, row, lane);
        if (lane == 0) sh.abort = 1;
        break;
      }
      gather_row<MODE, NA, FUSE>(p, row, nch, lane, sh.from[kStatsN], sh.fin_rc);
      for (int q = lane; q < nch; q += 32) {
        const float* src = p.part_b + (size_t(row) * nch + q) * kPartBStride;
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
        if (MODE == kModeAsym && sh.fin_rc.finite && d >= 0 && d < V)
          xd = G::at(p.x[lane == 1 ? NT - 1 : 1], size_t(row) * size_t(V) + size_t(d));
      }
      __syncwarp();
      jsd_finalize_row<T, MODE, NB, FUSE>(p, row, sh.fin_rc, sh.jsd_from, uint32_t(nch), lane, d, xd);
      __syncwarp();
      // The row's workspace entries back to zero (every chunk of the row read its pass-A partials
      // before its pass B, so nobody reads them any more).
      for (int q = lane; q < nch; q += 32) {
        char* a = static_cast<char*>(p.part_a) + (size_t(row) * nch + q) * (4 * kPartAStride);
#pragma unroll
        for (int w4 = 0; w4 < int(sizeof(JsdPart) / 16); ++w4) st_cg_zero4(a + 16 * w4);
        float* bsum = p.part_b + (size_t(row) * nch + q) * kPartBStride;
#pragma unroll
        for (int w4 = 0; w4 < 3; ++w4) st_cg_zero4(bsum + 4 * w4);
      }
      if (lane == 0) {
        p.row_cnt[row] = 0u;
        p.row_jcnt[row] = 0u;
      }
      __syncwarp();
    }
    return;
  }

  // ------------------------------------------------------------------ compute warps
  float2 beta2[NB];
#pragma unroll
  for (int sl = 0; sl < NB; ++sl) beta2[sl] = make_float2(p.betas[sl], p.betas[sl]);
  constexpr bool kPairShort = MODE == kModeAsym;
  PA st;                   // pass-A state of the current chunk
  RowB rb, rbt;            // pass-B row constants of the chunk pass B is in
  bool finite_b = false;
  float2 accn = make_float2(0.0f, 0.0f), accn2 = make_float2(0.0f, 0.0f);
  float an = 0.0f, ap = 0.0f, aq = 0.0f, an2 = 0.0f, ap2 = 0.0f, aq2 = 0.0f;
  for (int x = 0; x < my_units + kLag; ++x) {
    if (x < my_units) {
      // ---------------------------------------------------------------- pass A of unit x
      const int i = x % kRingA;
      const UnitPos up = unit_pos(x, G_, cta, nch, m, n, V);
      if (up.j == 0) st.reset();
      if (!warp_wait(bar(sh.full_a[i]), uint32_t(x / kRingA) & 1u, &sh.abort)) break;
      const int nvec = up.len / VEC;
      const char* bin[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) bin[j] = reinterpret_cast<const char*>(a_addr(i, j));
      for (int vi = tid; vi < nvec; vi += kWT) {
        uint4 cur[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) cur[j] = lds128(bin[j] + size_t(vi) * 16);
        st.body(cur, up.v0 + vi * VEC, beta2);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sh.empty_a[i]));
      if (up.j == m - 1) {
        // chunk done: warp partials (maxima, argmax slots, sums against the warp maximum)
        const int k = up.t % kSlots;
        float wm[NT], wsum[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          wm[j] = warp_max(st.rmax[j].value());
          const float sm = st.acc[j].x + st.acc[j].y;
          const float moved = (sm != 0.0f) ? sm * exp2f(st.mL[j] - ref_of(wm[j])) : 0.0f;
          wsum[j] = warp_sumf(moved);
        }
#pragma unroll
        for (int sl = 0; sl < NA; ++sl) warp_argmax(st.bv[sl], st.bi[sl]);
        if (up.t >= kSlots && !warp_wait(bar(sh.a_free[k]), uint32_t(up.t / kSlots - 1) & 1u, &sh.abort)) break;
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            sh.wa_m[k][warp][j] = wm[j];
            sh.wa_s[k][warp][j] = wsum[j];
          }
#pragma unroll
          for (int sl = 0; sl < NA; ++sl) {
            sh.wa_av[k][warp][sl] = st.bv[sl];
            sh.wa_ai[k][warp][sl] = st.bi[sl];
          }
          mbar_arrive(bar(sh.a_ready[k]));
        }
      }
    }
    const int s2 = x - kLag;
    if (s2 >= 0) {
      // ---------------------------------------------------------------- pass B of unit s2
      const int i = s2 % kRingB;
      const UnitPos up = unit_pos(s2, G_, cta, nch, m, n, V);
      const int k = up.t % kSlots;
      if (up.j == 0) {
        // a new chunk: its row constants into registers, the accumulators to zero
        if (!warp_wait(bar(sh.rc_ready[k]), uint32_t(up.t / kSlots) & 1u, &sh.abort)) break;
        if (sh.abort) break;
        const JsdRowConsts& rc = sh.rc[k];
        finite_b = rc.finite != 0;
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
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sh.rc_free[k]));
        accn = accn2 = make_float2(0.0f, 0.0f);
        an = ap = aq = an2 = ap2 = aq2 = 0.0f;
      }
      if (!warp_wait(bar(sh.full_b[i]), uint32_t(s2 / kRingB) & 1u, &sh.abort)) break;
      const int nvec = up.len / VEC;
      if (finite_b) {
        const char* ba = reinterpret_cast<const char*>(b_addr(i, 0));
        const char* bb = reinterpret_cast<const char*>(b_addr(i, 1));
        const char* bt = reinterpret_cast<const char*>(b_addr(i, NBI - 1));
        for (int vi = tid; vi < nvec; vi += kWT) {
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
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sh.empty_b[i]));
      if (up.j == m - 1) {
        float sums[6];
        sums[0] = warp_sumf((accn.x + accn.y) + an);
        sums[1] = warp_sumf(ap);
        sums[2] = warp_sumf(aq);
        if constexpr (FUSE) {
          sums[3] = warp_sumf((accn2.x + accn2.y) + an2);
          sums[4] = warp_sumf(ap2);
          sums[5] = warp_sumf(aq2);
        }
        if (up.t >= kSlots && !warp_wait(bar(sh.b_free[k]), uint32_t(up.t / kSlots - 1) & 1u, &sh.abort)) break;
        if (lane == 0) {
#pragma unroll
          for (int mm = 0; mm < NS; ++mm) sh.wb[k][warp][mm] = sums[mm];
          mbar_arrive(bar(sh.b_ready[k]));
        }
      }
    }
  }
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

StagedPlan staged_plan(int V, int elem_bytes, int nt, int nb) {
  const int vec = 16 / elem_bytes;
  int n_max = kBudget / ((kRingA * nt + kRingB * nb) * elem_bytes);
  n_max -= n_max % vec;
  StagedPlan pl;
  pl.n_unit = (V + n_max - 1) / n_max;
  pl.chunk = pl.n_unit < kChunk ? pl.n_unit : kChunk;
  int n = (V + pl.n_unit - 1) / pl.n_unit;
  n = (n + vec - 1) / vec * vec;
  pl.n = n;
  pl.smem = (kRingA * nt + kRingB * nb) * n * elem_bytes;
  return pl;
}

// Units per chunk for a batch of `rows` rows on `grid` CTAs: the largest m <= kChunk dividing the
// row's units such that the busiest CTA does at most 5 % more units than the average (chunks are
// the unit of work a CTA takes, so large chunks of few rows leave CTAs idle at the end).
int staged_chunk_for(const StagedPlan& pl, long long rows, int grid) {
  const double avg = double(rows) * pl.n_unit / grid;
  for (int m = pl.chunk; m > 1; --m) {
    if (pl.n_unit % m) continue;
    const long long chunks = rows * (pl.n_unit / m);
    const long long busiest = (chunks + grid - 1) / grid * m;
    if (double(busiest) <= 1.05 * avg + 1e-9 || busiest <= m) return m;
  }
  return 1;
}

int staged_max_units() { return kMaxUnits; }

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
