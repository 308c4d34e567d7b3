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
// thread-block cluster of C CTAs owns one row; CTA q of the cluster owns entries
// [q*n_slice, (q+1)*n_slice).  Each CTA stages its slice of every input in shared memory once (1-D
// bulk copies in kNumChunks chunks, one mbarrier each, so work starts on the first chunk while the
// rest is in flight), and the three passes the divergence needs run out of shared memory:
//   sweep 1: row maxima of every input (bf16: two-lane bf16 maxima on the raw words);
//   sweep 2: sums of exp(x - max) on the special-function unit, and the argmax of the verifier
//            score (one comparison per 16-byte vector against the best so far);
//   sweep 3: the per-entry Jensen-Shannon terms.
// Arithmetic on entries is two-lane packed fp32 (fma/add/mul .f32x2) where it pairs up.  After each
// sweep: warp shuffles, per-warp partials combined by one warp, a cluster exchange through
// distributed shared memory, and one warp that combines the C partials in rank order and
// broadcasts the row constants, so every CTA holds bit-identical row statistics.  Sums that cross
// warps and CTAs are carried as compensated fp32 pairs: this GPU's fp64 rate is a small fraction of
// its fp32 rate, so fp64 appears only in CTA 0's few finalisation steps.  HBM is read exactly once
// per input byte.  Before the last exchange every CTA pushes its final partials (and the CTA holding
// the draft's entry pushes t_d and b_d) into CTA 0, so the other CTAs leave right after it.  CTA 0
// finalises the row (gate, outputs, a 16-byte row record) and takes a ticket on the request's
// counter; the last of the K+1 rows to finish runs the left-to-right scan and resets the counter,
// so the whole step is one launch with no spin-waits.
//
// Numerics.  Inputs are widened exactly to fp32.  exp(x - M) is formed as ex2(fma(x, log2e, -M*log2e)),
// whose constant rounding error c is known exactly and removed from the log-sum-exp; the divergence
// sums use the same form, so the factor cancels in their ratio with the row sums.  The gate is
// decided in double in the log domain.  The per-entry divergence term is evaluated from
// u = (xb - xa) - (lse_b - lse_a):
//   narrow form (|u| <= 2, AsymSpec's pair): p * u^2 * P(u), P a fitted polynomial;
//   wide form (any u): max(p,q) * (A(r) - |u| r), r = exp(-|u|), A(r) = (1-r) B(r).
// Both are sums of non-negative terms (no cancellation between large entropies), and identical rows
// give exactly 0.
#include <cfloat>
#include <climits>
#include <type_traits>

#include "asv_device.cuh"
#include "asv_internal.h"
#include "jsd_poly.inc"

// Polynomial evaluation in the narrow divergence form: 0 packed with coefficient immediates,
// 1 packed with the coefficient pairs held in registers, 2 scalar with immediates.
#ifndef ASV_POLY_MODE
#define ASV_POLY_MODE 1
#endif

namespace asv {

struct __align__(16) JsdXchg {
  float mx[3];        // slice maxima of the inputs
  float argv;         // best verifier score in the slice
  int32_t argi;       // its vocabulary index
  float sum_hi[3];    // slice sums of ex2(fma(x, log2e, -M*log2e)) as hi + lo
  float sum_lo[3];
  // Pushed into CTA 0 by every CTA before the third exchange, so that CTA 0 alone reads
  // them afterwards and the other CTAs can leave:
  float jsd_from[kMaxCluster][4];  // slice divergence sums: p-form hi, lo, q-form hi, lo
  uint32_t err_from[kMaxCluster];  // a staged-data wait expired in that CTA
  float td, bd;                    // t_d and b_d, from the CTA that staged entry d
};

// Row constants, computed by one thread after each cluster exchange and broadcast through shared memory.
struct __align__(16) JsdRowConsts {
  float M[3];
  float ML[3];     // M * log2e, rounded
  float S_hi[3];   // row sums of ex2(fma(x, log2e, -ML)) as hi + lo
  float S_lo[3];
  float dL;        // lse_b - lse_a (pair inputs 1 and 0)
  int32_t finite;
  float rowv;
  int32_t rowi;
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

// Natural log of a positive finite double without fp64 transcendental code: exponent from
// the bits, the mantissa's log with log1pf (absolute error below 1e-7).
__device__ __forceinline__ double ln_pos(double S) {
  const long long bits = __double_as_longlong(S);
  const int e = int((bits >> 52) & 0x7ff) - 1023;
  const double m = __longlong_as_double((bits & 0x000fffffffffffffLL) | 0x3ff0000000000000LL);  // [1, 2)
  return double(e) * kLn2 + double(log1pf(float(m - 1.0)));
}

__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The context-gain signal for the delta-fusion score: 0 -> a - b, 1 -> a, 2 -> t - b.
template <int DSRC>
__device__ __forceinline__ float2 delta2(float2 a, float2 b, float2 t) {
  if constexpr (DSRC == 1) return a;
  else if constexpr (DSRC == 2) return fsub2(t, b);
  else return fsub2(a, b);
}

template <typename T, int MODE, int DSRC>
__global__ void __launch_bounds__(512) jsd_family_kernel(const JsdArgs p) {
  using E = Elem<T>;
  using S = typename E::storage;
  constexpr int NT = JsdTraits<MODE>::NT;
  constexpr int TGT = JsdTraits<MODE>::TGT;
  constexpr int VEC = E::kVec;
  constexpr int NP = E::kPairs;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ JsdXchg xchg;
  __shared__ JsdRowConsts rc;
  __shared__ float s_wf[32][4];
  __shared__ int32_t s_wi[32];
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

  // ---------------------------------------------------------------- sweep 1: maxima
  float mx[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) mx[j] = -INFINITY;
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
#pragma unroll
  for (int j = 0; j < NT; ++j) mx[j] = warp_max(mx[j]);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j) s_wf[warp][j] = mx[j];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float v = warp_max(lane < nwarps ? s_wf[lane][j] : -INFINITY);
      if (lane == 0) xchg.mx[j] = v;
    }
  }
  cluster_sync_w0(warp);  // #1
  if (warp == 0) {
    // lane q < C reads CTA q's maxima; a warp max combines them.
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float v = -INFINITY;
      if (lane < int(C)) v = dsmem_ld_f32(dsmem_map(smem_addr(&xchg.mx[j]), uint32_t(lane)));
      v = warp_max(v);
      if (lane == 0) {
        rc.M[j] = v;
        rc.ML[j] = isfinite(v) ? v * kLog2e : 0.0f;
      }
    }
  }
  __syncthreads();
  float ML[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) ML[j] = rc.ML[j];

  // ---------------------------------------------------------------- sweep 2: exponential sums + argmax
  {
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    const float2 beta2 = make_float2(p.beta, p.beta);
    float2 nml[NT], acc[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      nml[j] = make_float2(-ML[j], -ML[j]);
      acc[j] = make_float2(0.0f, 0.0f);
    }
    float bv = -INFINITY;
    int bi = INT_MAX;
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
      // Verifier score of the vector's entries; one comparison per vector against the best so far.
      float2 sc[NP];
#pragma unroll
      for (int q2 = 0; q2 < NP; ++q2) {
        if constexpr (MODE == kModeAsym) sc[q2] = ffma2(beta2, delta2<DSRC>(x[0][q2], x[1][q2], x[2][q2]), x[2][q2]);
        else sc[q2] = x[TGT][q2];
      }
      float vm = fmaxf(sc[0].x, sc[0].y);
#pragma unroll
      for (int q2 = 1; q2 < NP; ++q2) vm = fmaxf(vm, fmaxf(sc[q2].x, sc[q2].y));
      if (vm > bv) {
        int e_first = 2 * NP - 1;
#pragma unroll
        for (int q2 = NP - 1; q2 >= 0; --q2) {
          if (sc[q2].y == vm) e_first = 2 * q2 + 1;
          if (sc[q2].x == vm) e_first = 2 * q2;
        }
        bv = vm;
        bi = v0 + vi * VEC + e_first;
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float v = warp_sumf(acc[j].x + acc[j].y);
      if (lane == 0) s_wf[warp][j] = v;
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      s_wf[warp][3] = bv;
      s_wi[warp] = bi;
    }
  }
  __syncthreads();
  if (warp == 0) {
    float v2 = (lane < nwarps) ? s_wf[lane][3] : -INFINITY;
    int i2 = (lane < nwarps) ? s_wi[lane] : INT_MAX;
    warp_argmax(v2, i2);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const DF d = warp_sum_df(DF{lane < nwarps ? s_wf[lane][j] : 0.0f, 0.0f});
      if (lane == 0) {
        xchg.sum_hi[j] = d.hi;
        xchg.sum_lo[j] = d.lo;
      }
    }
    if (lane == 0) {
      xchg.argv = v2;
      xchg.argi = i2;
    }
  }
  cluster_sync_w0(warp);  // #2
  if (warp == 0) {
    float v2 = -INFINITY;
    int i2 = INT_MAX;
    if (lane < int(C)) {
      v2 = dsmem_ld_f32(dsmem_map(smem_addr(&xchg.argv), uint32_t(lane)));
      i2 = dsmem_ld_s32(dsmem_map(smem_addr(&xchg.argi), uint32_t(lane)));
    }
    warp_argmax(v2, i2);
    DF Sj[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      DF d{0.0f, 0.0f};
      if (lane < int(C)) {
        d.hi = dsmem_ld_f32(dsmem_map(smem_addr(&xchg.sum_hi[j]), uint32_t(lane)));
        d.lo = dsmem_ld_f32(dsmem_map(smem_addr(&xchg.sum_lo[j]), uint32_t(lane)));
      }
      Sj[j] = warp_sum_df(d);
    }
    if (lane == 0) {
      bool finite = true;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        finite = finite && isfinite(rc.M[j]) && isfinite(Sj[j].hi) && Sj[j].hi > 0.0f;
        rc.S_hi[j] = Sj[j].hi;
        rc.S_lo[j] = Sj[j].lo;
      }
      // lse_b - lse_a = (Mb - Ma) + ln(Sb / Sa) - (cb - ca) ln2, c = fma(M, log2e, -ML) the exact
      // rounding error of ML (the sums carry a factor 2^c).
      float dL = 0.0f;
      if (finite) {
        const float ca = fmaf(rc.M[0], kLog2e, -rc.ML[0]);
        const float cb = fmaf(rc.M[1], kLog2e, -rc.ML[1]);
        const float ratio = (Sj[1].hi + Sj[1].lo) / (Sj[0].hi + Sj[0].lo);
        dL = (rc.M[1] - rc.M[0]) + (ln_split(ratio) - (cb - ca) * kLn2f);
      }
      rc.finite = finite ? 1 : 0;
      rc.dL = dL;
      rc.rowv = v2;
      rc.rowi = i2;
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- sweep 3: divergence terms
  {
    const bool finite = rc.finite != 0;
    const float dL = rc.dL;
    float ap0 = 0.0f, ap1 = 0.0f, aq0 = 0.0f, aq1 = 0.0f;
    if (finite) {
      if constexpr (!JsdTraits<MODE>::kWide) {
        const float2 l2e2 = make_float2(kLog2e, kLog2e);
        const float2 dl2 = make_float2(dL, dL);
        const float2 nmal = make_float2(-ML[0], -ML[0]);
#if ASV_POLY_MODE == 1
        const asv_jsd_poly2h_coeffs pk = asv_jsd_poly2h_load();
#endif
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
#if ASV_POLY_MODE == 1
              accp = ffma2(fmul2(ep, fmul2(u, u)), asv_jsd_poly2h(u, pk), accp);
#elif ASV_POLY_MODE == 2
              accp = ffma2(fmul2(ep, fmul2(u, u)), make_float2(asv_jsd_poly(u.x), asv_jsd_poly(u.y)), accp);
#else
              accp = ffma2(fmul2(ep, fmul2(u, u)), asv_jsd_poly2(u), accp);
#endif
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
          float2 xa[NP], xb[NP];
          E::load_pairs(stage[0], vi, xa);
          E::load_pairs(stage[1], vi, xb);
#pragma unroll
          for (int q2 = 0; q2 < NP; ++q2) {
            jsd_entry<true>(xa[q2].x, xb[q2].x, dL, ML[0], ML[1], ap0, aq0);
            jsd_entry<true>(xa[q2].y, xb[q2].y, dL, ML[0], ML[1], ap1, aq1);
          }
        }
      }
    }
    const float wp = warp_sumf(ap0 + ap1);
    const float wq = warp_sumf(aq0 + aq1);
    if (lane == 0) {
      s_wf[warp][0] = wp;
      s_wf[warp][1] = wq;
    }
  }
  __syncthreads();
  const int dpos = (pos < p.K) ? p.draft_ids[size_t(req) * p.K + pos] : -1;
  if (warp == 0) {
    const DF dp = warp_sum_df(DF{lane < nwarps ? s_wf[lane][0] : 0.0f, 0.0f});
    const DF dq = warp_sum_df(DF{lane < nwarps ? s_wf[lane][1] : 0.0f, 0.0f});
    if (lane == 0) {
      // Push this CTA's partials into CTA 0.
      const uint32_t base = smem_addr(&xchg.jsd_from[rank][0]);
      dsmem_st_f32(dsmem_map(base + 0, 0), dp.hi);
      dsmem_st_f32(dsmem_map(base + 4, 0), dp.lo);
      dsmem_st_f32(dsmem_map(base + 8, 0), dq.hi);
      dsmem_st_f32(dsmem_map(base + 12, 0), dq.lo);
      dsmem_st_u32(dsmem_map(smem_addr(&xchg.err_from[rank]), 0), s_err);
      // The CTA that staged the draft's entry pushes t_d and b_d.
      if (MODE == kModeAsym && dpos >= v0 && dpos < v0 + len) {
        const int off = dpos - v0;
        dsmem_st_f32(dsmem_map(smem_addr(&xchg.td), 0), E::to_float(stage[NT - 1][off]));
        dsmem_st_f32(dsmem_map(smem_addr(&xchg.bd), 0), E::to_float(stage[1][off]));
      }
    }
  }
  cluster_sync_w0(warp);  // #3: after this only CTA 0 touches shared memory, and only its own

  // A CTA whose staged-data wait expired waits (bounded) for its copies before leaving.
  if (p.bulk && tid == 0 && s_err) {
    for (int c = 0; c < kNumChunks; ++c) {
      const int cv0 = c * chunk_vec;
      if (min(nvec, cv0 + chunk_vec) <= cv0) break;
      mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls);
    }
  }
  if (rank != 0 || tid != 0) return;

  // ---------------------------------------------------------------- row finalisation (CTA 0)
  DF jp{0.0f, 0.0f}, jq{0.0f, 0.0f};
  uint32_t err = 0;
  for (uint32_t q = 0; q < C; ++q) {
    jp = df_add(jp, DF{xchg.jsd_from[q][0], xchg.jsd_from[q][1]});
    jq = df_add(jq, DF{xchg.jsd_from[q][2], xchg.jsd_from[q][3]});
    err |= xchg.err_from[q];
  }
  const bool finite = rc.finite != 0;
  float D = 0.0f;
  if (finite) {
    D = 0.5f * ((jp.hi + jp.lo) / (rc.S_hi[0] + rc.S_lo[0]) + (jq.hi + jq.lo) / (rc.S_hi[1] + rc.S_lo[1]));
    D = fminf(fmaxf(D, 0.0f), kLn2f);
  }
  // Log-sum-exps (double, this thread only): lse = M + ln(S) - c ln2.
  double lse[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float c = fmaf(rc.M[j], kLog2e, -rc.ML[j]);
    lse[j] = finite ? double(rc.M[j]) + ln_pos(double(rc.S_hi[j]) + double(rc.S_lo[j])) - double(c) * kLn2 : 0.0;
  }
  uint32_t bits = 0;
  if (!finite) bits |= kBitNonfinite;
  if (err) bits |= kBitTimeout;
  const int token = (rc.rowi == INT_MAX) ? 0 : rc.rowi;
  if (pos < p.K) {
    if (dpos < 0 || dpos >= V) {
      bits |= kBitBadDraft;
    } else if (MODE == kModeAsym && finite) {
      const double margin = (double(xchg.td) - lse[NT - 1]) - p.ln_gamma + double(D) - (double(xchg.bd) - lse[1]);
      if (margin > 0.0) bits |= kBitAccept;
    }
  }
  if (p.out_D) p.out_D[row] = finite ? D : __int_as_float(0x7fc00000);
  if (MODE == kModeAsym && p.out_lse) {
#pragma unroll
    for (int j = 0; j < NT; ++j) p.out_lse[size_t(row) * 3 + j] = float(lse[j]);
  }
  RowRecord rec;
  rec.value = double(D);
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
    double thr = 0.0;
    if (MODE == kModeSci) {
      thr = p.T_base + p.alpha_omega * (p.r_hat[req] - p.tau_credit);
      thr = fmax(p.T_min, fmin(thr, p.T_max));
      if (p.out_T) p.out_T[req] = float(thr);
    }
    if (status) {
      p.out_accept_len[req] = 0;
      for (int i = 0; i < R1; ++i) toks[i] = -1;
    } else {
      int n = p.K;
      for (int i = 0; i < p.K; ++i) {
        const bool ok = (MODE == kModeAsym) ? (recs[i].bits & kBitAccept) != 0 : !(recs[i].value > thr);
        if (!ok) {
          n = i;
          break;
        }
      }
      if (MODE == kModeSci) {
        const double pacc = double(n) / double(p.K);
        p.r_hat[req] = (1.0 - p.ewma_beta) * p.r_hat[req] + p.ewma_beta * pacc;
      }
      p.out_accept_len[req] = n;
      const int32_t* dr = p.draft_ids + size_t(req) * p.K;
      for (int i = 0; i < R1; ++i) toks[i] = (i < n) ? dr[i] : (i == n ? recs[n].token : -1);
    }
    p.out_req_status[req] = status;
    p.tickets[req] = 0u;
  }
}

int jsd_static_smem_bytes() {
  return int(sizeof(JsdXchg) + sizeof(JsdRowConsts) + 32 * 4 * 4 + 32 * 4 + kNumChunks * 8 + 4 + 64);
}

using JsdKernel = void (*)(const JsdArgs);

static JsdKernel pick_kernel(int mode, int dtype, int dsrc) {
  if (mode == kModeSci) return dtype == 0 ? jsd_family_kernel<float, kModeSci, 0> : jsd_family_kernel<bf16_t, kModeSci, 0>;
  if (dtype == 0) {
    if (dsrc == 1) return jsd_family_kernel<float, kModeAsym, 1>;
    if (dsrc == 2) return jsd_family_kernel<float, kModeAsym, 2>;
    return jsd_family_kernel<float, kModeAsym, 0>;
  }
  if (dsrc == 1) return jsd_family_kernel<bf16_t, kModeAsym, 1>;
  if (dsrc == 2) return jsd_family_kernel<bf16_t, kModeAsym, 2>;
  return jsd_family_kernel<bf16_t, kModeAsym, 0>;
}

static cudaLaunchConfig_t make_config(const LaunchPlan& plan, unsigned grid, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(unsigned(plan.threads), 1, 1);
  cfg.dynamicSmemBytes = size_t(plan.smem);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(plan.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

static cudaError_t prepare(JsdKernel kern, const LaunchPlan& plan) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
  if (e != cudaSuccess) return e;
  if (plan.cluster > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t launch_jsd_family(int mode, int dtype, const JsdArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  JsdKernel kern = pick_kernel(mode, dtype, a.delta_source);
  cudaError_t e = prepare(kern, plan);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  const unsigned grid = unsigned(a.B) * unsigned(a.K + 1) * unsigned(plan.cluster);
  cudaLaunchConfig_t cfg = make_config(plan, grid, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

int jsd_max_active_clusters(int mode, int dtype, const LaunchPlan& plan) {
  JsdKernel kern = pick_kernel(mode, dtype, 0);
  if (prepare(kern, plan) != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config(plan, unsigned(plan.cluster), 0, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace asv
