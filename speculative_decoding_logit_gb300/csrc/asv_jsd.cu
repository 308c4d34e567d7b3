// asv_jsd.cu -- the AsymSpec and E2-SCI verification kernels.
//
// Sources (web pages):
//   "AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs" (reading notes),
//     sec. 4.1: context-gain signal delta = a - b and the delta-fusion token argmax(t + beta*delta);
//     sec. 4.2: D = JSD(softmax a || softmax b), gamma_eff = gamma * exp(-D), accept while
//     softmax(t)[d] > gamma_eff * softmax(b)[d], emit the delta-fusion token at the first rejection;
//     sec. 5: the delta-source ablation (delta := a, delta := t - b).
//   "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia" (paper notes), Key design 3:
//     JSD(draft || target) against a threshold driven by an EWMA of the acceptance rate.
//
// Work decomposition.  One row (request r, position i) is V vocabulary entries of each input.  A
// thread-block cluster of C CTAs owns one row; CTA q owns entries [q*n_slice, (q+1)*n_slice):
//   pass A  reads the slice of every input from HBM once into registers (16-byte loads that bypass
//           L1, two vectors per trip) and keeps per thread a running maximum and a sum of
//           exp(x - max) (rescaled on the rare occasions the maximum grows) for each input, plus the
//           argmax of the verifier score;
//   exchange the CTA's statistics go to every CTA of the cluster through distributed shared
//           memory; one warp combines the C partials in rank order, so every CTA holds bit-identical
//           row statistics (log-sum-exps, the lse difference used below, the argmax);
//   pass B  re-reads the slice of the divergence pair (a and b; SCI: draft and target), which the
//           L2 cache still holds from pass A (the resident CTAs' slices are a few tens of MB),
//           through a per-thread ring of 16-byte cp.async copies in shared memory (aligned slices),
//           and sums the per-entry Jensen-Shannon terms; this loop is bound by the fp32 pipe;
//   finish  every CTA pushes its pass-B sums into CTA 0 and leaves; CTA 0 finalises the row (gate,
//           outputs, a 16-byte row record) and takes a ticket on the request's counter.  The last of
//           the K+1 rows to finish runs the left-to-right scan and resets the counter, so the whole
//           step is one launch with no spin-waits.
// A CTA holds no slice in shared memory (the ring is 32 KB), so four CTAs share an SM and hide
// each other's exchanges.  Arithmetic on entries is two-lane packed fp32 (fma/add/mul/sub .f32x2)
// where it pairs up.  Sums that cross warps and CTAs are carried as compensated fp32 pairs: this
// GPU's fp64 rate is a small fraction of its fp32 rate, so fp64 appears only in CTA 0's few
// finalisation steps.
//
// Numerics.  Inputs are widened exactly to fp32.  exp(x - M) is formed as ex2(fma(x, log2e, -M*log2e))
// against the current reference maximum; partial sums move between references with exp2f of the
// difference of the (rounded) references, and the row sums end up against ML = M*log2e rounded, the
// reference pass B uses, so the divergence sums and the row sums share one scale.  The constant
// rounding error of ML is removed from the log-sum-exps.  The gate is decided in double in the log
// domain.  The per-entry divergence term is evaluated from u = (xb - xa) - (lse_b - lse_a):
//   narrow form (|u| <= 4): sqrt(p q) u^2 R(u^2), R an even-symmetric fitted polynomial (a shorter
//                           one on |u| <= 3 for the AsymSpec pair), taken by a whole vector when the
//                           largest u^2 of its entries is inside the domain;
//   wide form (any u):      max(p,q) (A(r) - |u| r), r = exp(-|u|), A(r) = (1 - r) B(r).
// Both are sums of non-negative terms (no cancellation between large entropies), and identical rows
// give exactly 0.  Loads carry L2 cache policies: the divergence pair is marked evict-last in pass A
// (pass B reads it again) and evict-first in pass B, the verifier input evict-first.
#include "asv_jsd_common.cuh"

namespace asv {

constexpr int kJsdThreads = 256;  // threads per CTA the kernel is compiled for (launch bounds)
constexpr int kJsdCtasPerSm = 4;  // CTAs per SM the kernel is compiled for (launch bounds)

constexpr int kRing = 4;  // pass-B vectors in flight per input per thread (a power of 2)

struct __align__(16) JsdXchg {
  // Every CTA pushes its pass-A partials into from[its rank] of every CTA of the cluster before the
  // first exchange, so each CTA combines them from its own shared memory afterwards.
  JsdPart from[kMaxCluster];
  // Pushed into CTA 0 by every CTA before the second exchange; only CTA 0 reads them afterwards.
  // Pass-B sums (hi, lo): narrow form, wide p-form, wide q-form; then the second pair's (fused).
  float jsd_from[kMaxCluster][12];
};

// NB: fused scores t + beta_b * delta for NB betas (AsymSpec; the all-(beta, gamma) sweep takes 4).
// FUSE: AsymSpec and E2-SCI in one read -- pass B also sums JSD(a || t), and an extra argmax slot
// holds the plain target argmax.
template <typename T, int MODE, int DSRC, bool ALIGNED, int NB, bool FUSE>
__global__ void __launch_bounds__(kJsdThreads, kJsdCtasPerSm) jsd_family_kernel(const JsdArgs p) {
  using G = GVec<T>;
  constexpr int NT = JsdTraits<MODE>::NT;
  constexpr int TGT = JsdTraits<MODE>::TGT;
  constexpr int VEC = G::kVec;
  constexpr int NP = G::kPairs;
  constexpr int kWarps = kJsdThreads / 32;
  constexpr int NA = NB + (FUSE ? 1 : 0);  // argmax slots
  constexpr bool kMulti = (NB > 1) || FUSE;
  static_assert(NA <= kMaxArg, "argmax slots");
  static_assert(!FUSE || (MODE == kModeAsym && NB == 1), "fused mode pairs one AsymSpec beta with E2-SCI");

  __shared__ JsdXchg xchg;
  __shared__ JsdRowConsts rc;
  // Pass B ring (aligned slices): [kRing][NPB][kJsdThreads] 16-byte vectors.
  constexpr int NPB = FUSE ? 3 : 2;
  extern __shared__ __align__(16) uint4 s_ring[];
  __shared__ float s_wf[kWarps][6];
  __shared__ float s_av[kWarps][kMaxArg];
  __shared__ int32_t s_ai[kWarps][kMaxArg];
  __shared__ float s_wm[kWarps][3];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();
  const int R1 = p.K + 1;
  // Rows: one per cluster.  E2-SCI pre-hit: phase 1 takes row 0 of every request, phase 2 rows
  // 1..K of every request, skipping requests that phase 1 dropped (the whole cluster returns).
  int row = blockIdx.x / C;
  if (MODE == kModeSci && p.prehit_phase == 1) {
    row *= R1;
  } else if (MODE == kModeSci && p.prehit_phase == 2) {
    const int rq = row / p.K;
    if (*reinterpret_cast<const volatile uint32_t*>(p.dropped + rq)) return;
    row = rq * R1 + 1 + (row - rq * p.K);
  }
  // Split cluster barrier: every thread arrives now and waits after pass A, before the first write
  // into another CTA's shared memory, so every CTA of the cluster has started by then.
  cluster_arrive_relaxed();
  const int req = row / R1;
  const int pos = row - req * R1;
  const int V = p.V;
  const int v0 = int(rank) * p.n_slice;
  // (checked build: a row outside the batch, or a cluster larger than the exchange arrays, reads
  // nothing; every CTA still takes part in the cluster barriers)
  const bool row_ok = ASV_GUARD(p, row >= 0 && row < p.B * R1 && rank < uint32_t(kMaxCluster) && C <= uint32_t(kMaxCluster));
  const int len = row_ok ? max(0, min(V - v0, p.n_slice)) : 0;
  const int nvec = (len + VEC - 1) / VEC;
  constexpr bool aligned = ALIGNED;
  const size_t row_base = size_t(row) * size_t(V);

  const void* slice[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) slice[j] = static_cast<const char*>(p.x[j]) + (row_base + size_t(v0)) * G::kBytes;

  // The finalising warp (warp 0 of CTA 0) needs the row's draft token and, for the gate, its
  // verifier and compressed-drafter logits: lanes 1 and 2 load the token now and the logits after
  // pass A, so the loads' latency is not on the row's critical path (single-outcome kernels; the
  // multi-outcome ones, short of registers, load them when they finalise).
  const bool fin_lane = !kMulti && rank == 0 && warp == 0 && (lane == 1 || lane == 2);
  int d_pre = -1;
  if (fin_lane && pos < p.K && ASV_GUARD(p, row_ok && req < p.B)) d_pre = __ldg(p.draft_ids + size_t(req) * p.K + pos);

  // L2 policies: the verifier input is read once (evict first; fused: pass B reads it again); the
  // divergence pair is read again by pass B (evict last until then, evict first on that last read).
  const uint64_t pol_evict_first = policy_evict_first();
  const uint64_t pol_keep = policy_evict_last();
  const uint64_t pol_t = FUSE ? pol_keep : pol_evict_first;

  // ---------------------------------------------------------------- pass A: maxima, exp sums, argmax
  RunMax<T> rmax[NT];
  float mL[NT];
  float2 acc[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    mL[j] = 0.0f;
    acc[j] = make_float2(0.0f, 0.0f);
  }
  float bv[NA];
  int bi[NA];
#pragma unroll
  for (int s = 0; s < NA; ++s) {
    bv[s] = -INFINITY;
    bi[s] = INT_MAX;
  }
  {
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    float2 beta2[NB];
#pragma unroll
    for (int s = 0; s < NB; ++s) beta2[s] = make_float2(p.betas[s], p.betas[s]);
    // One vector (entries [vi*VEC, vi*VEC + VEC) of the slice) of every input into the pass-A state.
    auto a_body = [&](const uint4 (&cur)[NT], const int vi) {
      // Running maxima; when a value passes the reference's slack, move the partial sum to a new
      // reference at the current maximum.
      bool far = false;
#pragma unroll
      for (int j = 0; j < NT; ++j) far |= rmax[j].update(cur[j]);
      if (far) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float M = rmax[j].value();
          // Nothing finite seen yet (-inf), or a +inf/NaN row (flagged later): keep waiting.
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
      // Verifier scores; one comparison per vector and score against the best so far.
#pragma unroll
      for (int sl = 0; sl < NA; ++sl) {
        float2 sc[NP];
#pragma unroll
        for (int q2 = 0; q2 < NP; ++q2) {
          if constexpr (MODE == kModeAsym) {
            if (FUSE && sl == NB) sc[q2] = x[2][q2];  // the plain target argmax (E2-SCI's emitted token)
            else sc[q2] = ffma2(beta2[sl < NB ? sl : 0], delta2<DSRC>(x[0][q2], x[1][q2], x[2][q2]), x[2][q2]);
          } else {
            sc[q2] = x[TGT][q2];
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
          bi[sl] = v0 + vi * VEC + e_first;
        }
      }
    };
    // One vector of input j (checked build: its entries must lie in the slice).
    auto ldA = [&](int j, int v) {
      return ASV_GUARD(p, v >= 0 && (!aligned || v * VEC + VEC <= len)) ? G::load(slice[j], v * VEC, len, aligned, true,
                                                                            j == 2 ? pol_t : pol_keep)
                                                                  : G::pad();
    };
    uint4 cur[NT], nxt[NT];
    int vi = tid;
    if (vi < nvec) {
#pragma unroll
      for (int j = 0; j < NT; ++j) cur[j] = ldA(j, vi);
    }
    // (bf16 multi-outcome kernels, short of registers, keep one vector per trip.)
    if constexpr (ALIGNED && (!kMulti || std::is_same<T, float>::value)) {
      // Two vectors per trip, the prefetch alternating between cur and nxt (no register copies);
      // a prefetched vector is consumed only while it is in range.
      for (; vi < nvec; vi += 2 * kJsdThreads) {
        if (vi + kJsdThreads < nvec) {
#pragma unroll
          for (int j = 0; j < NT; ++j) nxt[j] = ldA(j, vi + kJsdThreads);
        }
        a_body(cur, vi);
        if (vi + kJsdThreads >= nvec) break;
        if (vi + 2 * kJsdThreads < nvec) {
#pragma unroll
          for (int j = 0; j < NT; ++j) cur[j] = ldA(j, vi + 2 * kJsdThreads);
        }
        a_body(nxt, vi + kJsdThreads);
      }
    } else {
      // bf16 multi-outcome kernels and element-wise loads of unaligned rows: one vector per trip.
      for (; vi < nvec; vi += kJsdThreads) {
        if (vi + kJsdThreads < nvec) {
#pragma unroll
          for (int j = 0; j < NT; ++j) nxt[j] = ldA(j, vi + kJsdThreads);
        }
        a_body(cur, vi);
#pragma unroll
        for (int j = 0; j < NT; ++j) cur[j] = nxt[j];
      }
    }
  }

  float xd_pre = 0.0f;
  if (MODE == kModeAsym && fin_lane && d_pre >= 0 && d_pre < V && row_ok)
    xd_pre = G::at(p.x[lane == 1 ? NT - 1 : 1], row_base + size_t(d_pre));

  // Pass B of aligned slices streams the divergence pair (fused: and the verifier input) from L2
  // through a ring of kRing vectors per input per thread in shared memory, filled by 16-byte
  // cp.async copies (no registers held by copies in flight); each thread reads only its own slots
  // and refills a slot only after the arithmetic has consumed it.  The first kRing slots are filled
  // now, so that their reads overlap the row's exchange.  A thread takes its vectors in the reverse
  // of pass A's order: those pass A read last are the likeliest to be still in L2.
  const int jn = nvec > tid ? (nvec - tid + kJsdThreads - 1) / kJsdThreads : 0;  // this thread's vectors
  auto ring_issue = [&](int j) {
    const int vi = tid + (jn - 1 - j) * kJsdThreads;
    if (j < jn) {
#pragma unroll
      for (int m = 0; m < NPB; ++m) {
        const int slot = ((j & (kRing - 1)) * NPB + m) * kJsdThreads + tid;
        if (ASV_GUARD(p, slot < kRing * NPB * kJsdThreads && vi * VEC + VEC <= len))
          cp_async16(smem_addr(&s_ring[slot]), static_cast<const char*>(slice[m < 2 ? m : NT - 1]) + size_t(vi) * 16u,
                     pol_evict_first);
      }
    }
    cp_async_commit();
  };
  if constexpr (ALIGNED) {
#pragma unroll
    for (int j = 0; j < kRing; ++j) ring_issue(j);
  }

  // CTA partials.  Each warp reduces its maxima and argmax slots, then its sums against its own
  // maximum; warp 0 combines the warps' results -- lane j < NT input j, lane NT + s argmax slot s,
  // each reading its values of every warp (reads issued together) and adding them in registers in
  // warp order -- and pushes them into every CTA of the cluster.  The serial sections of the row
  // keep dependent shuffle and shared-memory round trips few: while other CTAs on the SM stream
  // their loads, each such round trip waits behind those loads (a few hundred cycles).
  float wmax[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) wmax[j] = warp_max(rmax[j].value());
#pragma unroll
  for (int sl = 0; sl < NA; ++sl) warp_argmax(bv[sl], bi[sl]);
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float s = acc[j].x + acc[j].y;
    const float moved = (s != 0.0f) ? s * exp2f(mL[j] - ref_of(wmax[j])) : 0.0f;
    const float ws = warp_sumf(moved);
    if (lane == 0) {
      s_wm[warp][j] = wmax[j];
      s_wf[warp][j] = ws;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int sl = 0; sl < NA; ++sl) {
      s_av[warp][sl] = bv[sl];
      s_ai[warp][sl] = bi[sl];
    }
  }
  __syncthreads();
  cluster_wait();
  if (warp == 0 && lane < NT + NA && ASV_GUARD(p, rank < uint32_t(kMaxCluster) && C <= uint32_t(kMaxCluster))) {
    const uint32_t dst = smem_addr(&xchg.from[rank]);
    if (lane < NT) {
      const int j = lane;
      float m[kWarps], sw[kWarps];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        m[w] = s_wm[w][j];
        sw[w] = s_wf[w][j];
      }
      float Mc = m[0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) Mc = fmaxf(Mc, m[w]);
      const float Rc = ref_of(Mc);
      DF d{0.0f, 0.0f};
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (sw[w] != 0.0f) d = df_add(d, DF{sw[w] * exp2f(ref_of(m[w]) - Rc), 0.0f});
      }
      for (uint32_t q = 0; q < C; ++q) {
        dsmem_st_f32(dsmem_map(dst + offsetof(JsdPart, mx) + 4u * j, q), Mc);
        dsmem_st_f32(dsmem_map(dst + offsetof(JsdPart, sum_hi) + 4u * j, q), d.hi);
        dsmem_st_f32(dsmem_map(dst + offsetof(JsdPart, sum_lo) + 4u * j, q), d.lo);
      }
    } else {
      const int sl = lane - NT;
      float v = s_av[0][sl];
      int i = s_ai[0][sl];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) argmax_merge(v, i, s_av[w][sl], s_ai[w][sl]);
      for (uint32_t q = 0; q < C; ++q) {
        dsmem_st_f32(dsmem_map(dst + offsetof(JsdPart, argv) + 4u * sl, q), v);
        dsmem_st_u32(dsmem_map(dst + offsetof(JsdPart, argi) + 4u * sl, q), uint32_t(i));
      }
    }
  }
  cluster_sync_w0(warp);  // #1

  // ---------------------------------------------------------------- row statistics (warp 0)
  if (warp == 0) {
    // Lane j < NT combines input j's maxima and sums over the cluster's CTAs, lane NT + s argmax
    // slot s: each lane reads its values of four CTAs at a time (reads issued together) and combines
    // them in registers in rank order; one batch of independent shuffles brings them to lane 0.
    const int j = lane < NT ? lane : 0;
    const int sl = (lane >= NT && lane < NT + NA) ? lane - NT : 0;
    float Mj = -INFINITY;
    DF Sj{0.0f, 0.0f};  // against ref_of(Mj)
    float av = -INFINITY;
    int ai = INT_MAX;
    for (uint32_t q0 = 0; q0 < C; q0 += 4) {
      float mx4[4], hi4[4], lo4[4], av4[4];
      int ai4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool ok = q0 + u < C;
        const JsdPart& f = xchg.from[ok ? q0 + u : 0];
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
      if (Sj.hi != 0.0f) {  // (more than four CTAs) move the running sum to the new reference
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
      for (int j = 0; j < NT; ++j) {
        finite = finite && isfinite(M[j]) && isfinite(S[j].hi) && S[j].hi > 0.0f;
        rc.M[j] = M[j];
        rc.ML[j] = MLr[j];
        rc.S_hi[j] = S[j].hi;
        rc.S_lo[j] = S[j].lo;
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
      // hML = fl(ML[0]/2 + ML[1]/2); its rounding error is removed from the narrow sum at the end.
      rc.hML = 0.5f * MLr[0] + 0.5f * MLr[1];
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
      for (int sl = 0; sl < NA; ++sl) rc.rowi[sl] = i2[sl];
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- pass B: divergence terms
  {
    const bool finite = rc.finite != 0;
    RowB rb, rb2;
    rb.dL = rc.dL;
    rb.MaL = rc.ML[0];
    rb.MbL = rc.ML[1];
    rb.hML = rc.hML;
    if constexpr (FUSE) {
      rb2.dL = rc.dL2;
      rb2.MaL = rc.ML[0];
      rb2.MbL = rc.ML[2];
      rb2.hML = rc.hML2;
    }
    // Accumulators per pair: narrow (packed), narrow/wide p-form/wide q-form (scalar).
    float2 accn = make_float2(0.0f, 0.0f), accn2 = make_float2(0.0f, 0.0f);
    float an = 0.0f, ap = 0.0f, aq = 0.0f, an2 = 0.0f, ap2 = 0.0f, aq2 = 0.0f;
    // One vector of the pair (xa, xb) against row constants rb.
    // sh: the short narrow form (|u| <= 3, two fewer terms), for the AsymSpec pair, whose u stays
    // small; the E2-SCI pair (draft, target) spreads wider and takes the |u| <= 4 form.
    auto pair_terms = [&](const float2 (&xa)[NP], const float2 (&xb)[NP], const RowB& r, float2& acn, float& sn,
                          float& sp, float& sq, const bool sh) {
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
      // Narrow form for the whole vector unless one entry is outside it (or NaN: -inf pairs): the
      // largest u^2 by NaN-propagating maxima, which run on the ALU pipe -- this loop is bound by
      // the fp32 pipe (about 13 fp32 operations per entry), so the test costs it nothing there.
      float smax = fmax_nan(s2[0].x, s2[0].y);
#pragma unroll
      for (int q2 = 1; q2 < NP; ++q2) smax = fmax_nan(smax, fmax_nan(s2[q2].x, s2[q2].y));
      const bool narrow = smax <= kS0;
      if (narrow) {
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
    };
    constexpr bool kPairShort = MODE == kModeAsym;
    if (finite && ALIGNED) {
      // (the ring's first kRing slots were filled before the exchange)
      for (int j = 0; j < jn; ++j) {
        cp_async_wait_group<kRing - 1>();  // the copies of vector j have landed
        const int slot = (j & (kRing - 1)) * NPB;
        if (!ASV_GUARD(p, (slot + NPB - 1) * kJsdThreads + tid < kRing * NPB * kJsdThreads)) continue;
        float2 xa[NP], xb[NP];
        G::pairs(s_ring[(slot + 0) * kJsdThreads + tid], xa);
        G::pairs(s_ring[(slot + 1) * kJsdThreads + tid], xb);
        pair_terms(xa, xb, rb, accn, an, ap, aq, kPairShort);
        if constexpr (FUSE) {
          float2 xt[NP];
          G::pairs(s_ring[(slot + 2) * kJsdThreads + tid], xt);
          pair_terms(xa, xt, rb2, accn2, an2, ap2, aq2, false);
        }
        ring_issue(j + kRing);
      }
      cp_async_wait_all();
    } else if (finite) {
      int vi = tid;
      uint4 ca, cb, ct, na, nb, nt;
      if (vi < nvec && ASV_GUARD(p, vi >= 0)) {
        ca = G::load(slice[0], vi * VEC, len, aligned, true, pol_evict_first);
        cb = G::load(slice[1], vi * VEC, len, aligned, true, pol_evict_first);
        if constexpr (FUSE) ct = G::load(slice[NT - 1], vi * VEC, len, aligned, true, pol_evict_first);
      }
      for (; vi < nvec; vi += kJsdThreads) {
        const int vn = vi + kJsdThreads;
        if (vn < nvec) {
          na = G::load(slice[0], vn * VEC, len, aligned, true, pol_evict_first);
          nb = G::load(slice[1], vn * VEC, len, aligned, true, pol_evict_first);
          if constexpr (FUSE) nt = G::load(slice[NT - 1], vn * VEC, len, aligned, true, pol_evict_first);
        }
        float2 xa[NP], xb[NP];
        G::pairs(ca, xa);
        G::pairs(cb, xb);
        pair_terms(xa, xb, rb, accn, an, ap, aq, kPairShort);
        if constexpr (FUSE) {
          float2 xt[NP];
          G::pairs(ct, xt);
          pair_terms(xa, xt, rb2, accn2, an2, ap2, aq2, false);
          ct = nt;
        }
        ca = na;
        cb = nb;
      }
    }
    if (ALIGNED && !finite) cp_async_wait_all();  // the ring's first copies, unused
    const float wn = warp_sumf((accn.x + accn.y) + an);
    const float wp = warp_sumf(ap);
    const float wq = warp_sumf(aq);
    if (lane == 0) {
      s_wf[warp][0] = wn;
      s_wf[warp][1] = wp;
      s_wf[warp][2] = wq;
    }
    if constexpr (FUSE) {
      const float wn2 = warp_sumf((accn2.x + accn2.y) + an2);
      const float wp2 = warp_sumf(ap2);
      const float wq2 = warp_sumf(aq2);
      if (lane == 0) {
        s_wf[warp][3] = wn2;
        s_wf[warp][4] = wp2;
        s_wf[warp][5] = wq2;
      }
    }
  }
  __syncthreads();
  constexpr int NS = FUSE ? 6 : 3;
  if (warp == 0 && lane < NS && ASV_GUARD(p, rank < uint32_t(kMaxCluster))) {
    // Lane m adds sum m of the CTA's warps in warp order (reads issued together) and pushes it into
    // CTA 0.
    float v[kWarps];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v[w] = s_wf[w][lane];
    DF dm{v[0], 0.0f};
#pragma unroll
    for (int w = 1; w < kWarps; ++w) dm = df_add(dm, DF{v[w], 0.0f});
    const uint32_t base = smem_addr(&xchg.jsd_from[rank][2 * lane]);
    dsmem_st_f32(dsmem_map(base + 0, 0), dm.hi);
    dsmem_st_f32(dsmem_map(base + 4, 0), dm.lo);
  }
  cluster_sync_w0(warp);  // #2: after this only CTA 0 touches shared memory, and only its own
  if (rank != 0 || warp != 0) return;

  // ---------------------------------------------------------------- row finalisation (CTA 0, warp 0)
  if (!row_ok) return;
  jsd_finalize_row<T, MODE, NB, FUSE>(p, row, rc, xchg.jsd_from, C, lane, d_pre, xd_pre);
}

int jsd_threads() { return kJsdThreads; }
int jsd_ctas_per_sm() { return kJsdCtasPerSm; }

using JsdKernel = void (*)(const JsdArgs);

// variant 0: the single-outcome kernels; 1: the all-(beta, gamma) sweep (4 betas); 2: AsymSpec and
// E2-SCI fused (AsymSpec mode, delta = a - b).
template <bool AL>
static JsdKernel pick_aligned(int mode, int dtype, int dsrc, int variant) {
  if (variant == 1)
    return dtype == 0 ? jsd_family_kernel<float, kModeAsym, 0, AL, 4, false>
                      : jsd_family_kernel<bf16_t, kModeAsym, 0, AL, 4, false>;
  if (variant == 2)
    return dtype == 0 ? jsd_family_kernel<float, kModeAsym, 0, AL, 1, true>
                      : jsd_family_kernel<bf16_t, kModeAsym, 0, AL, 1, true>;
  if (mode == kModeSci)
    return dtype == 0 ? jsd_family_kernel<float, kModeSci, 0, AL, 1, false>
                      : jsd_family_kernel<bf16_t, kModeSci, 0, AL, 1, false>;
  if (dtype == 0) {
    if (dsrc == 1) return jsd_family_kernel<float, kModeAsym, 1, AL, 1, false>;
    if (dsrc == 2) return jsd_family_kernel<float, kModeAsym, 2, AL, 1, false>;
    return jsd_family_kernel<float, kModeAsym, 0, AL, 1, false>;
  }
  if (dsrc == 1) return jsd_family_kernel<bf16_t, kModeAsym, 1, AL, 1, false>;
  if (dsrc == 2) return jsd_family_kernel<bf16_t, kModeAsym, 2, AL, 1, false>;
  return jsd_family_kernel<bf16_t, kModeAsym, 0, AL, 1, false>;
}

static JsdKernel pick_kernel(int mode, int dtype, int dsrc, bool aligned, int variant) {
  return aligned ? pick_aligned<true>(mode, dtype, dsrc, variant) : pick_aligned<false>(mode, dtype, dsrc, variant);
}

// Dynamic shared memory: the pass-B ring of the aligned instantiations.
static int ring_bytes(bool aligned, int variant) {
  return aligned ? kRing * (variant == 2 ? 3 : 2) * kJsdThreads * 16 : 0;
}

static cudaLaunchConfig_t make_config(const LaunchPlan& plan, unsigned grid, int smem, cudaStream_t s,
                                      cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(unsigned(kJsdThreads), 1, 1);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(plan.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

static cudaError_t prepare(JsdKernel kern, const LaunchPlan& plan, int smem) {
  if (plan.cluster > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_jsd_family(int mode, int dtype, const JsdArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  JsdKernel kern = pick_kernel(mode, dtype, a.delta_source, a.bulk != 0, a.variant);
  const int smem = ring_bytes(a.bulk != 0, a.variant);
  cudaError_t e = prepare(kern, plan, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  // Rows launched: every row, or (E2-SCI pre-hit) row 0 of each request, then rows 1..K.
  const unsigned rows = a.prehit_phase == 1 ? unsigned(a.B)
                        : a.prehit_phase == 2 ? unsigned(a.B) * unsigned(a.K)
                                              : unsigned(a.B) * unsigned(a.K + 1);
  const unsigned grid = rows * unsigned(plan.cluster);
  cudaLaunchConfig_t cfg = make_config(plan, grid, smem, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

int jsd_max_active_clusters(int mode, int dtype, const LaunchPlan& plan) {
  JsdKernel kern = pick_kernel(mode, dtype, 0, plan.bulk != 0, 0);
  const int smem = ring_bytes(plan.bulk != 0, 0);
  if (prepare(kern, plan, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config(plan, unsigned(plan.cluster), smem, 0, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace asv
