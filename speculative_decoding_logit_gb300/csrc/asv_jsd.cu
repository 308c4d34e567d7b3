// asv_jsd.cu -- the AsymSpec and E2-SCI verification kernels.
//
// Sources (web pages):
//   "AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs" (reading notes),
//     sec. 4.1: context-gain signal delta = a - b and the delta-fusion token argmax(t + beta*delta);
//     sec. 4.2: D = JSD(softmax a || softmax b), gamma_eff = gamma * exp(-D), accept while
//     softmax(t)[d] > gamma_eff * softmax(b)[d], emit the delta-fusion token at the first rejection.
//   "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia" (paper notes), Key design 3:
//     JSD(draft || target) against a threshold driven by an EWMA of the acceptance rate.
//
// Work decomposition.  One row (request r, position i) is V vocabulary entries of each input.  A
// thread-block cluster of C CTAs owns one row; CTA q of the cluster owns entries
// [q*n_slice, (q+1)*n_slice).  Each CTA stages its slice of every input in shared memory once (1-D
// bulk copies in kNumChunks chunks, one mbarrier per chunk, so work starts on the first chunk while
// the rest is in flight), and the three passes the divergence needs run out of shared memory:
//   sweep 1: row maxima of every input and the argmax of the verifier score;
//   sweep 2: sums of exp(x - max) (exponentials on the special-function unit);
//   sweep 3: the per-entry Jensen-Shannon terms.
// Between sweeps the CTAs exchange partial results through distributed shared memory; every CTA
// combines the partials in rank order, so all CTAs hold bit-identical row statistics.  HBM is read
// exactly once per input byte.  CTA 0 finalises the row (gate, outputs, a 16-byte row record) and
// takes a ticket on the request's counter; the last of the K+1 rows to finish runs the left-to-right
// scan for its request and resets the counter, so the whole step is one launch with no spin-waits.
//
// Numerics.  Inputs are widened exactly to fp32.  exp(x - M) is formed as ex2(fma(x, log2e, -M*log2e)),
// whose constant rounding error c is known exactly and removed from the log-sum-exp in double; the
// divergence sums use the same form, so the factor cancels in their ratio with the row sums.
// Per-thread partial sums are fp32 (two accumulators), combined across the CTA and cluster in fp64.
// The gate is decided in double in the log domain.  The per-entry divergence term is evaluated from
// u = (xb - xa) - (lse_b - lse_a):
//   narrow form (|u| <= 2, AsymSpec's pair): p * u^2 * P(u), P a fitted polynomial;
//   wide form (any u): max(p,q) * (A(r) - |u| r), r = exp(-|u|), A(r) = (1-r) B(r).
// Both are sums of non-negative terms (no cancellation between large entropies), and identical rows
// give exactly 0.
#include <cfloat>
#include <climits>
#include <cstdlib>
#include <type_traits>

#include "asv_device.cuh"
#include "asv_internal.h"
#include "jsd_poly.inc"

namespace asv {

struct __align__(16) JsdXchg {
  float mx[3];       // row-slice maxima of the inputs
  float argv;        // best verifier score in the slice
  int32_t argi;      // its vocabulary index
  uint32_t err;      // staged-data wait expired in this CTA
  double sum[3];     // sums of ex2(fma(x, log2e, -M*log2e)) over the slice
  double jsd[2];     // divergence partial sums (p-form, q-form)
  float argv2;       // lean variant: argmax partials exchanged after the second sweep
  int32_t argi2;
};

template <int MODE>
struct JsdTraits {
  static constexpr int NT = (MODE == kModeAsym) ? 3 : 2;  // staged inputs
  static constexpr int TGT = NT - 1;                       // index of the verifier/target input
  static constexpr bool kWide = (MODE == kModeSci);        // divergence term form
};

// Per-entry Jensen-Shannon contribution, accumulated un-normalised:
// acc_p += exp(xa - Ma) * f(u) for entries in p-form, acc_q += exp(xb - Mb) * f(-u) in q-form.
template <bool WIDE>
__device__ __forceinline__ void jsd_entry(float xa, float xb, float dL, float MaL, float MbL, float& acc_p,
                                          float& acc_q) {
  const float u = (xb - xa) - dL;
  if (!WIDE && fabsf(u) <= ASV_JSD_POLY_U0) {
    const float ep = ex2_approx(fmaf(xa, kLog2e, -MaL));
    acc_p = fmaf(ep * (u * u), asv_jsd_poly(u), acc_p);
    return;
  }
  // Wide form.  u <= 0: p >= q, term = p * h(|u|); u > 0 (or NaN): term = q * h(|u|).
  const bool pform = (u <= 0.0f);
  const float s = fabsf(u);
  const float em = ex2_approx(pform ? fmaf(xa, kLog2e, -MaL) : fmaf(xb, kLog2e, -MbL));
  const float r = ex2_approx(-s * kLog2e);
  const float sr = (r > 0.0f) ? s * r : 0.0f;
  const float h = fmaf(1.0f - r, asv_jsd_wide_b(r), -sr);
  const float v = (em > 0.0f) ? em * h : 0.0f;
  if (pform) acc_p += v;
  else acc_q += v;
}

// Lean variant of the sweeps: maxima on raw data in sweep 1 (bf16x2 maxima), the argmax folded
// into sweep 2 with one comparison per 16-byte vector, and packed two-lane fp32 arithmetic.
template <typename T, int MODE, bool LEAN>
__global__ void __launch_bounds__(512) jsd_family_kernel(const JsdArgs p) {
  using E = Elem<T>;
  using S = typename E::storage;
  constexpr int NT = JsdTraits<MODE>::NT;
  constexpr int TGT = JsdTraits<MODE>::TGT;
  constexpr int VEC = E::kVec;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ JsdXchg xchg;
  __shared__ float s_wf[32][4];
  __shared__ int32_t s_wi[32];
  __shared__ double s_wd[32][3];
  __shared__ __align__(8) uint64_t s_bar[kNumChunks];
  __shared__ uint32_t s_err;

  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = nthr >> 5;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();
  const int row = blockIdx.x / C;
  const int R1 = p.K + 1;
  const int req = row / R1;
  const int pos = row - req * R1;
  const int V = p.V;
  const int v0 = int(rank) * p.n_slice;
  const int len = max(0, min(V - v0, p.n_slice));
  const int nvec = (len + VEC - 1) / VEC;
  const size_t row_base = size_t(row) * size_t(V);
  const size_t stage_stride = (size_t(p.n_slice) * sizeof(S) + 127) & ~size_t(127);

  S* stage[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) stage[j] = reinterpret_cast<S*>(smem_raw + j * stage_stride);

  const int chunk_vec = (nvec + kNumChunks - 1) / kNumChunks;

  // ---------------------------------------------------------------- staging
  if (tid == 0) {
    s_err = 0;
#pragma unroll
    for (int c = 0; c < kNumChunks; ++c) mbar_init(smem_addr(&s_bar[c]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (p.bulk) {
    if (tid == 0) {
      for (int c = 0; c < kNumChunks; ++c) {
        const int cv0 = c * chunk_vec;
        const int cv1 = min(nvec, cv0 + chunk_vec);
        if (cv1 <= cv0) break;
        const uint32_t bytes = uint32_t(cv1 - cv0) * VEC * sizeof(S);
        const uint32_t bar = smem_addr(&s_bar[c]);
        mbar_arrive_expect_tx(bar, bytes * NT);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const S* src = reinterpret_cast<const S*>(p.x[j]) + row_base + v0 + size_t(cv0) * VEC;
          bulk_g2s(smem_addr(stage[j] + size_t(cv0) * VEC), src, bytes, bar);
        }
      }
    }
  } else {
    // Unaligned rows: ordinary loads, the slice padded to the vector width with -inf.
    const int npad = nvec * VEC;
    for (int k = tid; k < npad; k += nthr) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const S* src = reinterpret_cast<const S*>(p.x[j]);
        stage[j][k] = (k < len) ? src[row_base + v0 + k] : E::neg_inf();
      }
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- sweep 1: maxima + argmax
  float mx[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) mx[j] = -INFINITY;
  float bv = -INFINITY;
  int bi = INT_MAX;
  if constexpr (LEAN) {
    if constexpr (std::is_same<T, bf16_t>::value) {
      uint32_t m2[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) m2[j] = 0xff80ff80u;
      for (int c = 0; c < kNumChunks; ++c) {
        const int cv0 = c * chunk_vec;
        const int cv1 = min(nvec, cv0 + chunk_vec);
        if (cv1 <= cv0) break;
        if (p.bulk && !mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls)) atomicOr(&s_err, 1u);
        for (int vi = cv0 + tid; vi < cv1; vi += nthr) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const uint4 w = reinterpret_cast<const uint4*>(stage[j])[vi];
            m2[j] = bmax2(bmax2(m2[j], w.x), bmax2(w.y, bmax2(w.z, w.w)));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) mx[j] = fmaxf(bf16_lo(m2[j]), bf16_hi(m2[j]));
    } else {
      for (int c = 0; c < kNumChunks; ++c) {
        const int cv0 = c * chunk_vec;
        const int cv1 = min(nvec, cv0 + chunk_vec);
        if (cv1 <= cv0) break;
        if (p.bulk && !mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls)) atomicOr(&s_err, 1u);
        for (int vi = cv0 + tid; vi < cv1; vi += nthr) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const float4 v = reinterpret_cast<const float4*>(stage[j])[vi];
            mx[j] = fmaxf(fmaxf(mx[j], v.x), fmaxf(v.y, fmaxf(v.z, v.w)));
          }
        }
      }
    }
  } else {
    for (int c = 0; c < kNumChunks; ++c) {
      const int cv0 = c * chunk_vec;
      const int cv1 = min(nvec, cv0 + chunk_vec);
      if (cv1 <= cv0) break;
      if (p.bulk && !mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls)) atomicOr(&s_err, 1u);
      for (int vi = cv0 + tid; vi < cv1; vi += nthr) {
        float x[NT][VEC];
  #pragma unroll
        for (int j = 0; j < NT; ++j) E::load_vec(stage[j], vi, x[j]);
        const int k0 = v0 + vi * VEC;
  #pragma unroll
        for (int e = 0; e < VEC; ++e) {
  #pragma unroll
          for (int j = 0; j < NT; ++j) mx[j] = fmaxf(mx[j], x[j][e]);
          float s;
          if (MODE == kModeAsym) s = fmaf(p.beta, x[0][e] - x[1][e], x[2][e]);
          else s = x[TGT][e];
          if (s > bv) {
            bv = s;
            bi = k0 + e;
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) mx[j] = warp_max(mx[j]);
  warp_argmax(bv, bi);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j) s_wf[warp][j] = mx[j];
    s_wf[warp][3] = bv;
    s_wi[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    float m2[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) m2[j] = (lane < nwarps) ? s_wf[lane][j] : -INFINITY;
    float v2 = (lane < nwarps) ? s_wf[lane][3] : -INFINITY;
    int i2 = (lane < nwarps) ? s_wi[lane] : INT_MAX;
#pragma unroll
    for (int j = 0; j < NT; ++j) m2[j] = warp_max(m2[j]);
    warp_argmax(v2, i2);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j) xchg.mx[j] = m2[j];
      xchg.argv = v2;
      xchg.argi = i2;
      xchg.err = s_err;
    }
  }
  cluster_sync();  // #1

  // Row maxima and argmax: every CTA combines all ranks in the same order.
  float M[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) M[j] = -INFINITY;
  float rowv = -INFINITY;
  int rowi = INT_MAX;
  {
    const uint32_t base_mx = smem_addr(&xchg.mx[0]);
    const uint32_t base_v = smem_addr(&xchg.argv);
    const uint32_t base_i = smem_addr(&xchg.argi);
    for (uint32_t q = 0; q < C; ++q) {
#pragma unroll
      for (int j = 0; j < NT; ++j) M[j] = fmaxf(M[j], dsmem_ld_f32(dsmem_map(base_mx + 4 * j, q)));
      argmax_merge(rowv, rowi, dsmem_ld_f32(dsmem_map(base_v, q)), dsmem_ld_s32(dsmem_map(base_i, q)));
    }
  }

  // ---------------------------------------------------------------- sweep 2: sums of exponentials
  float ML[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) ML[j] = isfinite(M[j]) ? M[j] * kLog2e : 0.0f;
  float bv2 = -INFINITY;
  int bi2 = INT_MAX;
  {
    float s0[NT], s1[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) s0[j] = s1[j] = 0.0f;
    if constexpr (LEAN) {
      constexpr int NP = E::kPairs;
      const float2 l2e2 = make_float2(kLog2e, kLog2e);
      const float2 beta2 = make_float2(p.beta, p.beta);
      float2 nml[NT], acc[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        nml[j] = make_float2(-ML[j], -ML[j]);
        acc[j] = make_float2(0.0f, 0.0f);
      }
      for (int vi = tid; vi < nvec; vi += nthr) {
        float2 x[NT][NP];
#pragma unroll
        for (int j = 0; j < NT; ++j) E::load_pairs(stage[j], vi, x[j]);
#pragma unroll
        for (int q2 = 0; q2 < NP; ++q2) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const float2 y = ffma2(x[j][q2], l2e2, nml[j]);
            acc[j] = fadd2(acc[j], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
          }
        }
        // verifier score of the vector's entries; one comparison per vector against the best so far
        float2 sc[NP];
#pragma unroll
        for (int q2 = 0; q2 < NP; ++q2) {
          if (MODE == kModeAsym) sc[q2] = ffma2(beta2, fsub2(x[0][q2], x[1][q2]), x[2][q2]);
          else sc[q2] = x[TGT][q2];
        }
        float vm = fmaxf(sc[0].x, sc[0].y);
#pragma unroll
        for (int q2 = 1; q2 < NP; ++q2) vm = fmaxf(vm, fmaxf(sc[q2].x, sc[q2].y));
        if (vm > bv2) {
          int e_first = 2 * NP - 1;
#pragma unroll
          for (int q2 = NP - 1; q2 >= 0; --q2) {
            if (sc[q2].y == vm) e_first = 2 * q2 + 1;
            if (sc[q2].x == vm) e_first = 2 * q2;
          }
          bv2 = vm;
          bi2 = v0 + vi * VEC + e_first;
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        s0[j] = acc[j].x;
        s1[j] = acc[j].y;
      }
    } else {
      for (int vi = tid; vi < nvec; vi += nthr) {
        float x[NT][VEC];
#pragma unroll
        for (int j = 0; j < NT; ++j) E::load_vec(stage[j], vi, x[j]);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            s0[j] += ex2_approx(fmaf(x[j][e], kLog2e, -ML[j]));
            s1[j] += ex2_approx(fmaf(x[j][e + 1], kLog2e, -ML[j]));
          }
        }
      }
    }
    if constexpr (LEAN) {
      warp_argmax(bv2, bi2);
      if (lane == 0) {
        s_wf[warp][3] = bv2;
        s_wi[warp] = bi2;
      }
    }
    double d[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) d[j] = warp_sum(double(s0[j]) + double(s1[j]));
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j) s_wd[warp][j] = d[j];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        double v = (lane < nwarps) ? s_wd[lane][j] : 0.0;
        v = warp_sum(v);
        if (lane == 0) xchg.sum[j] = v;
      }
      if constexpr (LEAN) {
        float v2 = (lane < nwarps) ? s_wf[lane][3] : -INFINITY;
        int i2 = (lane < nwarps) ? s_wi[lane] : INT_MAX;
        warp_argmax(v2, i2);
        if (lane == 0) {
          xchg.argv2 = v2;
          xchg.argi2 = i2;
        }
      }
    }
  }
  cluster_sync();  // #2
  if constexpr (LEAN) {
    const uint32_t base_v = smem_addr(&xchg.argv2);
    const uint32_t base_i = smem_addr(&xchg.argi2);
    for (uint32_t q = 0; q < C; ++q)
      argmax_merge(rowv, rowi, dsmem_ld_f32(dsmem_map(base_v, q)), dsmem_ld_s32(dsmem_map(base_i, q)));
  }

  double Ssum[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) Ssum[j] = 0.0;
  {
    const uint32_t base = smem_addr(&xchg.sum[0]);
    for (uint32_t q = 0; q < C; ++q) {
#pragma unroll
      for (int j = 0; j < NT; ++j) Ssum[j] += dsmem_ld_f64(dsmem_map(base + 8 * j, q));
    }
  }
  // lse = M + ln(S') - c ln2 with c = fma(M, log2e, -ML) the exact rounding error of ML.
  double lse[NT];
  bool finite = true;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float c = fmaf(M[j], kLog2e, -ML[j]);
    lse[j] = double(M[j]) + log(Ssum[j]) - double(c) * kLn2;
    finite = finite && isfinite(M[j]) && isfinite(Ssum[j]) && Ssum[j] > 0.0;
  }

  // ---------------------------------------------------------------- sweep 3: divergence terms
  {
    const float dL = finite ? float(lse[1] - lse[0]) : 0.0f;
    float ap0 = 0.0f, ap1 = 0.0f, aq0 = 0.0f, aq1 = 0.0f;
    if (finite) {
      if constexpr (LEAN && !JsdTraits<MODE>::kWide) {
        constexpr int NP = E::kPairs;
        const float2 l2e2 = make_float2(kLog2e, kLog2e);
        const float2 dl2 = make_float2(dL, dL);
        const float2 nmal = make_float2(-ML[0], -ML[0]);
        float2 accp = make_float2(0.0f, 0.0f);
        for (int vi = tid; vi < nvec; vi += nthr) {
          float2 xa[NP], xb[NP];
          E::load_pairs(stage[0], vi, xa);
          E::load_pairs(stage[1], vi, xb);
#pragma unroll
          for (int q2 = 0; q2 < NP; ++q2) {
            const float2 u = fsub2(fsub2(xb[q2], xa[q2]), dl2);
            if (fabsf(u.x) <= ASV_JSD_POLY_U0 && fabsf(u.y) <= ASV_JSD_POLY_U0) {
              const float2 y = ffma2(xa[q2], l2e2, nmal);
              const float2 ep = make_float2(ex2_approx(y.x), ex2_approx(y.y));
              accp = ffma2(fmul2(ep, fmul2(u, u)), asv_jsd_poly2(u), accp);
            } else {
              jsd_entry<false>(xa[q2].x, xb[q2].x, dL, ML[0], ML[1], ap0, aq0);
              jsd_entry<false>(xa[q2].y, xb[q2].y, dL, ML[0], ML[1], ap1, aq1);
            }
          }
        }
        ap0 += accp.x;
        ap1 += accp.y;
      } else {
        for (int vi = tid; vi < nvec; vi += nthr) {
          float xa[VEC], xb[VEC];
          E::load_vec(stage[0], vi, xa);
          E::load_vec(stage[1], vi, xb);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            jsd_entry<JsdTraits<MODE>::kWide>(xa[e], xb[e], dL, ML[0], ML[1], ap0, aq0);
            jsd_entry<JsdTraits<MODE>::kWide>(xa[e + 1], xb[e + 1], dL, ML[0], ML[1], ap1, aq1);
          }
        }
      }
    }
    double dp = warp_sum(double(ap0) + double(ap1));
    double dq = warp_sum(double(aq0) + double(aq1));
    if (lane == 0) {
      s_wd[warp][0] = dp;
      s_wd[warp][1] = dq;
    }
    __syncthreads();
    if (warp == 0) {
      double vp = (lane < nwarps) ? s_wd[lane][0] : 0.0;
      double vq = (lane < nwarps) ? s_wd[lane][1] : 0.0;
      vp = warp_sum(vp);
      vq = warp_sum(vq);
      if (lane == 0) {
        xchg.jsd[0] = vp;
        xchg.jsd[1] = vq;
        xchg.err = s_err;
      }
    }
  }
  cluster_sync();  // #3

  // ---------------------------------------------------------------- row finalisation (CTA 0)
  if (rank == 0 && tid == 0) {
    double jp = 0.0, jq = 0.0;
    uint32_t err = 0;
    {
      const uint32_t bp = smem_addr(&xchg.jsd[0]);
      const uint32_t be = smem_addr(&xchg.err);
      for (uint32_t q = 0; q < C; ++q) {
        jp += dsmem_ld_f64(dsmem_map(bp, q));
        jq += dsmem_ld_f64(dsmem_map(bp + 8, q));
        err |= dsmem_ld_u32(dsmem_map(be, q));
      }
    }
    double D = 0.5 * (jp / Ssum[0] + jq / Ssum[1]);
    D = fmin(fmax(D, 0.0), kLn2);
    uint32_t bits = 0;
    if (!finite) bits |= kBitNonfinite;
    if (err) bits |= kBitTimeout;
    const int token = (rowi == INT_MAX) ? 0 : rowi;
    if (MODE == kModeAsym && pos < p.K) {
      const int d = p.draft_ids[size_t(req) * p.K + pos];
      if (d < 0 || d >= V) {
        bits |= kBitBadDraft;
      } else if (finite) {
        // t_d and b_d from the slice of the CTA that staged entry d.
        const uint32_t owner = uint32_t(d / p.n_slice);
        const int off = d - int(owner) * p.n_slice;
        const float td = E::from_smem_remote(dsmem_map(smem_addr(stage[2] + off), owner));
        const float bd = E::from_smem_remote(dsmem_map(smem_addr(stage[1] + off), owner));
        const double margin = (double(td) - lse[2]) - p.ln_gamma + D - (double(bd) - lse[1]);
        if (margin > 0.0) bits |= kBitAccept;
      }
    }
    if (MODE == kModeSci && pos < p.K) {
      const int d = p.draft_ids[size_t(req) * p.K + pos];
      if (d < 0 || d >= V) bits |= kBitBadDraft;
    }
    if (p.out_D) p.out_D[row] = finite ? float(D) : __int_as_float(0x7fc00000);
    if (MODE == kModeAsym && p.out_lse) {
#pragma unroll
      for (int j = 0; j < 3; ++j) p.out_lse[size_t(row) * 3 + j] = float(lse[j]);
    }
    RowRecord rec;
    rec.value = D;
    rec.token = token;
    rec.bits = bits;
    p.records[row] = rec;
    __threadfence();
    const uint32_t ticket = atomicAdd(&p.tickets[req], 1u);
    if (ticket == uint32_t(p.K)) {
      // Last row of this request: the left-to-right scan.
      __threadfence();
      const volatile RowRecord* recs = p.records + size_t(req) * R1;
      uint32_t any = 0;
      for (int i = 0; i < R1; ++i) any |= recs[i].bits;
      const uint32_t status = ((any & kBitNonfinite) ? 1u : 0u) | ((any & kBitBadDraft) ? 2u : 0u) |
                              ((any & kBitTimeout) ? 4u : 0u);
      int32_t* toks = p.out_tokens + size_t(req) * R1;
      if (status) {
        p.out_accept_len[req] = 0;
        for (int i = 0; i < R1; ++i) toks[i] = -1;
      } else {
        int n = p.K;
        if (MODE == kModeAsym) {
          for (int i = 0; i < p.K; ++i)
            if (!(recs[i].bits & kBitAccept)) {
              n = i;
              break;
            }
        } else {
          double thr = p.T_base + p.alpha_omega * (p.r_hat[req] - p.tau_credit);
          thr = fmax(p.T_min, fmin(thr, p.T_max));
          if (p.out_T) p.out_T[req] = float(thr);
          for (int i = 0; i < p.K; ++i)
            if (recs[i].value > thr) {
              n = i;
              break;
            }
          const double pacc = double(n) / double(p.K);
          p.r_hat[req] = (1.0 - p.ewma_beta) * p.r_hat[req] + p.ewma_beta * pacc;
        }
        p.out_accept_len[req] = n;
        const int32_t* dr = p.draft_ids + size_t(req) * p.K;
        for (int i = 0; i < R1; ++i) toks[i] = (i < n) ? dr[i] : (i == n ? recs[n].token : -1);
      }
      if (MODE == kModeSci && status && p.out_T) {
        const double thr = p.T_base + p.alpha_omega * (p.r_hat[req] - p.tau_credit);
        p.out_T[req] = float(fmax(p.T_min, fmin(thr, p.T_max)));
      }
      p.out_req_status[req] = status;
      p.tickets[req] = 0u;
    }
  }

  // A CTA whose staged-data wait expired waits (bounded) for its copies before leaving.
  if (p.bulk && tid == 0 && s_err) {
    for (int c = 0; c < kNumChunks; ++c) {
      const int cv0 = c * chunk_vec;
      if (min(nvec, cv0 + chunk_vec) <= cv0) break;
      mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls);
    }
  }
  // Keep this CTA's shared memory alive until CTA 0 has finished its remote reads.
  cluster_sync();  // #4
}

int jsd_static_smem_bytes() { return int(sizeof(JsdXchg) + 32 * 4 * 4 + 32 * 4 + 32 * 3 * 8 + kNumChunks * 8 + 4); }

static bool lean_variant() {
  static const bool v = [] {
    const char* e = std::getenv("ASV_JSD_VARIANT");
    return !(e && e[0] == '0');
  }();
  return v;
}

template <typename T, int MODE>
static cudaError_t launch_one(const JsdArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  auto kern = lean_variant() ? jsd_family_kernel<T, MODE, true> : jsd_family_kernel<T, MODE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
  if (e != cudaSuccess) return e;
  if (plan.cluster > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const int R = a.B * (a.K + 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(R) * unsigned(plan.cluster), 1, 1);
  cfg.blockDim = dim3(unsigned(plan.threads), 1, 1);
  cfg.dynamicSmemBytes = size_t(plan.smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(plan.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int MODE>
static int max_clusters_one(const LaunchPlan& plan) {
  auto kern = lean_variant() ? jsd_family_kernel<T, MODE, true> : jsd_family_kernel<T, MODE, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem) != cudaSuccess) return 0;
  if (plan.cluster > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(plan.cluster), 1, 1);
  cfg.blockDim = dim3(unsigned(plan.threads), 1, 1);
  cfg.dynamicSmemBytes = size_t(plan.smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(plan.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_jsd_family(int mode, int dtype, const JsdArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  if (mode == kModeAsym) return dtype == 0 ? launch_one<float, kModeAsym>(a, plan, s) : launch_one<bf16_t, kModeAsym>(a, plan, s);
  return dtype == 0 ? launch_one<float, kModeSci>(a, plan, s) : launch_one<bf16_t, kModeSci>(a, plan, s);
}

int jsd_max_active_clusters(int mode, int dtype, const LaunchPlan& plan) {
  if (mode == kModeAsym) return dtype == 0 ? max_clusters_one<float, kModeAsym>(plan) : max_clusters_one<bf16_t, kModeAsym>(plan);
  return dtype == 0 ? max_clusters_one<float, kModeSci>(plan) : max_clusters_one<bf16_t, kModeSci>(plan);
}

}  // namespace asv
