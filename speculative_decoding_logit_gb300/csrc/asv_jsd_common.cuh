// asv_jsd_common.cuh -- the building blocks of the AsymSpec / E2-SCI verification kernel
// (asv_jsd.cu): 16-byte vector access, running maxima, the per-entry Jensen-Shannon term, and the
// row finalisation (divergence from the pass-B sums, log-sum-exps, the CDA gate or the E2-SCI test,
// the row record and the left-to-right scan by the last row of a request), kept out of line of the
// kernel body.
//
// Sources (web pages): "AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs"
// (reading notes), sec. 4.1-4.2; "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit
// Inertia" (paper notes), Key design 3.
#pragma once

#include <cfloat>
#include <cstddef>
#include <climits>
#include <type_traits>

#include "asv_device.cuh"
#include "asv_internal.h"
#include "jsd_poly.inc"

namespace asv {

constexpr int kMaxArg = 4;  // argmax slots: fused scores for up to 4 betas, or 1 beta and the plain target
constexpr int kMaxGamma = 8;  // gammas of one sweep

// One CTA's pass-A partials.
struct __align__(16) JsdPart {
  float mx[3];        // CTA maxima of the inputs
  float sum_hi[3];    // CTA sums of exp2(x log2e - mL_cta), mL_cta = mx * log2e rounded, as hi + lo
  float sum_lo[3];
  float argv[kMaxArg];    // best scores in the CTA's slice
  int32_t argi[kMaxArg];  // their vocabulary indices
};

// Row constants, computed by warp 0 after the exchange and broadcast through shared memory.
struct __align__(16) JsdRowConsts {
  float M[3];
  float ML[3];     // M * log2e, rounded
  float S_hi[3];   // row sums of exp2(x log2e - ML) as hi + lo
  float S_lo[3];
  float dL;        // lse_b - lse_a (pair inputs 1 and 0)
  float hML;       // fl(ML[0]/2 + ML[1]/2), the narrow form's reference
  float dL2;       // fused: lse_t - lse_a (pair inputs 2 and 0)
  float hML2;      // fused: fl(ML[0]/2 + ML[2]/2)
  int32_t finite;
  int32_t rowi[kMaxArg];
};

template <int MODE>
struct JsdTraits {
  static constexpr int NT = (MODE == kModeAsym) ? 3 : 2;  // streamed inputs
  static constexpr int TGT = NT - 1;                       // index of the verifier/target input
};

// ------------------------------------------------------------------ global vector access

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 16-byte load with an L2 cache policy (evict-first for data read for the last time, evict-last
// for the divergence pair, which pass B reads again).
__device__ __forceinline__ uint4 ldg_stream_pol(const void* p, uint64_t pol) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(pol));
  return v;
}

// A 16-byte vector of one input: 8 bf16 or 4 fp32 entries, as raw words.
template <typename T>
struct GVec;

template <>
struct GVec<bf16_t> {
  static constexpr int kVec = 8;
  static constexpr int kPairs = 4;
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ uint4 pad() {
    return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  }
  // Entries [k, k+8) of a row slice; `aligned` slices use one 16-byte load, others ordinary loads
  // with -inf at and beyond `lim`.
  // With a policy (`hint`), the load carries that L2 cache policy.
  __device__ static __forceinline__ uint4 load(const void* base, int k, int lim, bool aligned, bool hint = false,
                                               uint64_t pol = 0) {
    const uint16_t* r = static_cast<const uint16_t*>(base);
    if (aligned) return hint ? ldg_stream_pol(r + k, pol) : ldg_stream(r + k);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (k + 2 * i < lim) ? uint32_t(__ldg(r + k + 2 * i)) : 0xff80u;
      const uint32_t hi = (k + 2 * i + 1 < lim) ? uint32_t(__ldg(r + k + 2 * i + 1)) : 0xff80u;
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static __forceinline__ void pairs(const uint4& v, float2 (&x)[4]) {
    x[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
    x[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
    x[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
    x[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
  }
  __device__ static __forceinline__ float at(const void* base, size_t k) {
    return __uint_as_float(uint32_t(__ldg(static_cast<const uint16_t*>(base) + k)) << 16);
  }
};

template <>
struct GVec<float> {
  static constexpr int kVec = 4;
  static constexpr int kPairs = 2;
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ uint4 pad() {
    return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
  }
  __device__ static __forceinline__ uint4 load(const void* base, int k, int lim, bool aligned, bool hint = false,
                                               uint64_t pol = 0) {
    const float* r = static_cast<const float*>(base);
    if (aligned) return hint ? ldg_stream_pol(r + k, pol) : ldg_stream(r + k);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = (k + i < lim) ? __float_as_uint(__ldg(r + k + i)) : 0xff800000u;
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static __forceinline__ void pairs(const uint4& v, float2 (&x)[2]) {
    x[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    x[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ static __forceinline__ float at(const void* base, size_t k) {
    return __ldg(static_cast<const float*>(base) + k);
  }
};

// Running maximum of one input over the vectors a thread has seen, and the reference the
// thread's exponentials are taken against.  The reference moves only when a value exceeds it by
// more than kRefSlack (in log2 units): terms then stay below 2^kRefSlack, far from fp32 overflow,
// and the rescale of the partial sum is needed about once per thread (on its first finite value)
// instead of on every growth of the maximum.  bf16 compares raw bf16x2 words (exact), fp32 floats.
constexpr float kRefSlack = 64.0f;

template <typename T>
struct RunMax;

template <>
struct RunMax<bf16_t> {
  uint32_t m2 = 0xff80ff80u;   // two-lane running maximum
  uint32_t thr2 = 0xff80ff80u; // two-lane bf16 threshold (rounded down): a larger value moves the reference
  // Returns true when a value of the vector exceeds the threshold.
  __device__ __forceinline__ bool update(const uint4& v) {
    const uint32_t vm = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
    m2 = bmax2(m2, vm);
    return bmax2(vm, thr2) != thr2;
  }
  __device__ __forceinline__ float value() const { return fmaxf(bf16_lo(m2), bf16_hi(m2)); }
  __device__ __forceinline__ bool started() const { return thr2 != 0xff80ff80u; }
  // New threshold for reference L (log2 units): the largest bf16 not above (L + slack) / log2e.
  __device__ __forceinline__ void set_threshold(float L) {
    const float t = (L + kRefSlack) * 0.693147180559945f;
    uint32_t b = __float_as_uint(t) >> 16;              // truncate toward zero
    if (t > 0.0f && __uint_as_float(b << 16) > t) b -= 1;  // (truncation of a positive value is not above it)
    if (t < 0.0f && __uint_as_float(b << 16) > t) b += 1;  // negative: move away from zero
    thr2 = b | (b << 16);
  }
};

template <>
struct RunMax<float> {
  float m = -INFINITY;
  float thr = -INFINITY;
  __device__ __forceinline__ bool update(const uint4& v) {
    const float vm = fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                           fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    m = fmaxf(m, vm);
    return vm > thr;
  }
  __device__ __forceinline__ float value() const { return m; }
  __device__ __forceinline__ bool started() const { return thr != -INFINITY; }
  __device__ __forceinline__ void set_threshold(float L) { thr = (L + kRefSlack) * 0.693147180559945f; }
};

// ------------------------------------------------------------------ per-entry divergence term

// Row constants pass B needs.
struct RowB {
  float dL;   // lse_b - lse_a
  float MaL;  // references of the pair (M log2e, rounded)
  float MbL;
  float hML;  // fl((MaL + MbL) / 2), the narrow form's reference
};

// One entry, either form.  acc_n: narrow terms sqrt(ea eb) u^2 R(u^2), with ea = exp2(xa log2e -
// MaL) and eb likewise; acc_p / acc_q: wide terms in p-form (ea h) / q-form (eb h).
__device__ __forceinline__ void jsd_entry(float xa, float xb, const RowB& rb, float& acc_n, float& acc_p,
                                          float& acc_q) {
  const float u = (xb - xa) - rb.dL;
  const float s2 = u * u;
  if (s2 <= ASV_JSD_EVEN_S0) {
    const float e = ex2_approx(fmaf(xa + xb, 0.5f * kLog2e, -rb.hML));
    acc_n = fmaf(e * s2, asv_jsd_even(s2), acc_n);
    return;
  }
  // Wide form.  u <= 0: p >= q, term = p * h(|u|); u > 0 (or NaN): term = q * h(|u|).
  const bool pform = (u <= 0.0f);
  const float s = fabsf(u);
  const float em = ex2_approx(pform ? fmaf(xa, kLog2e, -rb.MaL) : fmaf(xb, kLog2e, -rb.MbL));
  const float r = ex2_approx(-s * kLog2e);
  const float sr = (r > 0.0f) ? s * r : 0.0f;
  const float h = fmaf(1.0f - r, asv_jsd_wide_b(r), -sr);
  const float v = (em > 0.0f) ? em * h : 0.0f;
  if (pform) acc_p += v;
  else acc_q += v;
}

// Maximum that propagates NaN (fmaxf drops it), so a NaN entry fails the narrow-form test.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
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

// Reference for exponentials against a maximum M: M * log2e, or 0 while M is -inf (then every
// exponential is exp2(-inf) = 0 and a finite stand-in avoids inf - inf).
__device__ __forceinline__ float ref_of(float M) { return isfinite(M) ? M * kLog2e : 0.0f; }

// The context-gain signal for the delta-fusion score: 0 -> a - b, 1 -> a, 2 -> t - b.
template <int DSRC>
__device__ __forceinline__ float2 delta2(float2 a, float2 b, float2 t) {
  if constexpr (DSRC == 1) return a;
  else if constexpr (DSRC == 2) return fsub2(t, b);
  else return fsub2(a, b);
}

// Row finalisation by one warp of the row's CTA 0: D from the cluster's pass-B sums (`jsd_from[q]`
// holds CTA q's, q < C), the log-sum-exps, the gate, the outputs and a 16- or 32-byte row record;
// the warp that completes its request runs the left-to-right scan.  Single-outcome callers pass the
// row's draft token in lane 1 of `d_in` and its verifier / compressed-drafter logits in lanes 1 and
// 2 of `xd_in`.
template <typename T, int MODE, int NB, bool FUSE>
__device__ __forceinline__ void jsd_finalize_row(const JsdArgs& p, const int row, const JsdRowConsts& rc,
                                                 const float (*jsd_from)[12], const uint32_t C, const int lane,
                                                 const int d_in, const float xd_in) {
  using G = GVec<T>;
  constexpr int NT = JsdTraits<MODE>::NT;
  constexpr int NA = NB + (FUSE ? 1 : 0);
  constexpr bool kMulti = (NB > 1) || FUSE;
  const int R1 = p.K + 1;
  const int req = row / R1;
  const int pos = row - req * R1;
  const int V = p.V;
  const size_t row_base = size_t(row) * size_t(V);
  const unsigned kAll = 0xffffffffu;
  const int K = p.K;
  const bool finite = rc.finite != 0;
  // (checked build: the row and its request inside the batch, the grid sizes inside their arrays)
  if (!ASV_GUARD(p, row >= 0 && row < p.B * R1 && req < p.B && p.n_gamma <= kMaxGamma && p.n_beta <= kMaxArg))
    return;
  // The draft token and its verifier / compressed-drafter logits: single-outcome callers pass them
  // in (loaded early by lanes 1 and 2); the multi-outcome kernels load them here.
  const int d = (pos < K) ? (kMulti ? p.draft_ids[size_t(req) * K + pos] : __shfl_sync(kAll, d_in, 1)) : -1;
  const bool d_ok = d >= 0 && d < V;
  float xd = xd_in;
  if (kMulti && MODE == kModeAsym && finite && d_ok && (lane == 1 || lane == 2))
    xd = G::at(p.x[lane == 1 ? NT - 1 : 1], row_base + size_t(d));
  // Pass-B sums of the cluster's CTAs: lane m < NS adds sum m over the CTAs in rank order (reads
  // issued four CTAs at a time), then one batch of independent shuffles gives every lane all of them.
  constexpr int NS = FUSE ? 6 : 3;
  DF mine{0.0f, 0.0f};
  if (lane < NS) {
    for (uint32_t q0 = 0; q0 < C; q0 += 4) {
      float h4[4], l4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool ok = q0 + u < C;
        const float* f = jsd_from[ok ? q0 + u : 0];
        h4[u] = ok ? f[2 * lane] : 0.0f;
        l4[u] = ok ? f[2 * lane + 1] : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (q0 + u < C) mine = df_add(mine, DF{h4[u], l4[u]});
      }
    }
  }
  auto from_lane = [&](int m) { return DF{__shfl_sync(kAll, mine.hi, m), __shfl_sync(kAll, mine.lo, m)}; };
  const DF jn = from_lane(0), jp = from_lane(1), jq = from_lane(2);
  float D = 0.0f;
  if (finite) {
    // Narrow terms are against sqrt(ea eb) 2^(MaL/2 + MbL/2 - hML); the row sums Sa, Sb against
    // MaL, MbL.  delta = hML - (MaL/2 + MbL/2) exactly (TwoSum of the two halves).
    const float ha = 0.5f * rc.ML[0], hb = 0.5f * rc.ML[1];
    const float bb = rc.hML - ha;
    const float delta = -((ha - (rc.hML - bb)) + (hb - bb));
    const float Sa = rc.S_hi[0] + rc.S_lo[0];
    const float Sb = rc.S_hi[1] + rc.S_lo[1];
    const float narrow = __fdiv_rn((jn.hi + jn.lo) * exp2f(delta), __fsqrt_rn(Sa) * __fsqrt_rn(Sb));
    const float wide = __fdiv_rn(jp.hi + jp.lo, Sa) + __fdiv_rn(jq.hi + jq.lo, Sb);
    D = fminf(fmaxf(0.5f * (narrow + wide), 0.0f), kLn2f);
  }
  // Fused: J = JSD(a || t) from the second pair's sums, the same way.
  float J = 0.0f;
  if constexpr (FUSE) {
    const DF kn = from_lane(3), kp = from_lane(4), kq = from_lane(5);
    if (finite) {
      const float ha = 0.5f * rc.ML[0], ht = 0.5f * rc.ML[2];
      const float bb = rc.hML2 - ha;
      const float delta = -((ha - (rc.hML2 - bb)) + (ht - bb));
      const float Sa = rc.S_hi[0] + rc.S_lo[0];
      const float St = rc.S_hi[2] + rc.S_lo[2];
      const float narrow = __fdiv_rn((kn.hi + kn.lo) * exp2f(delta), __fsqrt_rn(Sa) * __fsqrt_rn(St));
      const float wide = __fdiv_rn(kp.hi + kp.lo, Sa) + __fdiv_rn(kq.hi + kq.lo, St);
      J = fminf(fmaxf(0.5f * (narrow + wide), 0.0f), kLn2f);
    }
  }
  // Log-sum-exps, one input per lane (double): lse = M + ln(S) - c ln2.
  double my_lse = 0.0;
  if (lane < NT && finite) {
    const float c = fmaf(rc.M[lane], kLog2e, -rc.ML[lane]);
    my_lse = double(rc.M[lane]) + ln_pos(double(rc.S_hi[lane]) + double(rc.S_lo[lane])) - double(c) * kLn2;
  }
  const double lse_b = __shfl_sync(kAll, my_lse, 1);
  const double lse_v = __shfl_sync(kAll, my_lse, NT - 1);
  const float td = __shfl_sync(kAll, xd, 1);
  const float bd = __shfl_sync(kAll, xd, 2);
  if constexpr (!kMulti) {
  uint32_t bits = 0;
  if (!finite) bits |= kBitNonfinite;
  if (pos < K) {
    if (!d_ok) {
      bits |= kBitBadDraft;
    } else if (MODE == kModeAsym && finite) {
      const double margin = (double(td) - lse_v) - p.ln_gamma + double(D) - (double(bd) - lse_b);
      if (margin > 0.0) bits |= kBitAccept;
    }
  }
  if (lane == 0 && p.out_D) p.out_D[row] = finite ? D : __int_as_float(0x7fc00000);
  if (MODE == kModeAsym && p.out_lse && lane < NT) p.out_lse[size_t(row) * 3 + lane] = float(my_lse);
  if (MODE == kModeSci && p.prehit_phase == 1) {
    // Pre-hit: the window is dropped when its first draft fails the threshold (or row 0 is not
    // finite, or a draft id is out of range); the request then finishes here with n = 0.
    double thr = __dadd_rn(p.T_base, __dmul_rn(p.alpha_omega, __dsub_rn(p.r_hat[req], p.tau_credit)));
    thr = fmax(p.T_min, fmin(thr, p.T_max));
    const int32_t* dr = p.draft_ids + size_t(req) * K;
    bool bad = false;
    for (int i = lane; i < K; i += 32) bad = bad || dr[i] < 0 || dr[i] >= V;
    bad = __any_sync(kAll, bad);
    const bool drop = !finite || bad || double(D) > thr;
    if (drop) {
      const uint32_t status = (finite ? 0u : 1u) | (bad ? 2u : 0u);
      int32_t* toks = p.out_tokens + size_t(req) * R1;
      const int tok0 = (rc.rowi[0] == INT_MAX) ? 0 : rc.rowi[0];
      for (int i = lane; i < R1; i += 32) toks[i] = status ? -1 : (i == 0 ? tok0 : -1);
      if (lane == 0) {
        if (p.out_T) p.out_T[req] = float(thr);
        if (!status) {
          const double pacc = 0.0;
          p.r_hat[req] = __dadd_rn(__dmul_rn(__dsub_rn(1.0, p.ewma_beta), p.r_hat[req]), __dmul_rn(p.ewma_beta, pacc));
        }
        p.out_accept_len[req] = 0;
        p.out_req_status[req] = status;
        p.dropped[req] = 1u;
      }
      return;
    }
  }
  uint32_t ticket = 0;
  if (lane == 0) {
    RowRecord rec;
    rec.value = double(D);
    rec.token = (rc.rowi[0] == INT_MAX) ? 0 : rc.rowi[0];
    rec.bits = bits;
    p.records[row] = rec;
    ticket = atom_add_acq_rel_gpu(&p.tickets[req], 1u);
  }
  ticket = __shfl_sync(kAll, ticket, 0);
  if (ticket != uint32_t(K)) return;

  // Last row of this request: the left-to-right scan, 32 records per step.
  (void)ld_acquire_gpu(&p.tickets[req]);  // every lane acquires the other rows' records
  RowRecord* recs = p.records + size_t(req) * R1;
  // SCI threshold (double, each operation rounded once as written), then the stabilisers.
  double thr = 0.0;
  int32_t new_age = 0;
  if (MODE == kModeSci) {
    thr = __dadd_rn(p.T_base, __dmul_rn(p.alpha_omega, __dsub_rn(p.r_hat[req], p.tau_credit)));
    thr = fmax(p.T_min, fmin(thr, p.T_max));
    if (p.sci_state) {
      const SciState st = p.sci_state[req];
      if (!(st.flags & 1u)) {
        new_age = 1;
      } else if (st.flags & 2u) {
        thr = p.fb_T;
        new_age = 1;
      } else if (st.age >= p.min_refresh && fabs(__dsub_rn(thr, st.T_applied)) > p.hyst) {
        new_age = 1;
      } else {
        thr = st.T_applied;
        new_age = st.age + 1;
      }
    }
  }
  uint32_t any = 0;
  int n = K;      // accepted prefix
  int tok_n = 0;  // token of row n
  for (int base = 0; base < R1; base += 32) {
    const int i = base + lane;
    uint32_t b = 0;
    double v = 0.0;
    int tk = 0;
    if (i < R1) {
      const float4 w = ld_cg_f4(recs + i);
      v = __hiloint2double(__float_as_int(w.y), __float_as_int(w.x));
      tk = __float_as_int(w.z);
      b = __float_as_uint(w.w);
    }
    any |= __reduce_or_sync(kAll, b);
    const bool ok = (MODE == kModeAsym) ? (b & kBitAccept) != 0 : !(v > thr);
    const unsigned rej = __ballot_sync(kAll, i < K && !ok);
    if (n == K && rej != 0u) n = base + __ffs(rej) - 1;
    const int src = (n >= base && n < base + 32) ? n - base : 0;
    const int tk_src = __shfl_sync(kAll, tk, src);
    if (n >= base && n < base + 32) tok_n = tk_src;
  }
  const uint32_t status = ((any & kBitNonfinite) ? 1u : 0u) | ((any & kBitBadDraft) ? 2u : 0u) |
                          ((any & kBitTimeout) ? 4u : 0u);
  int32_t* toks = p.out_tokens + size_t(req) * R1;
  const int32_t* dr = p.draft_ids + size_t(req) * K;
  for (int i = lane; i < R1; i += 32) {
    toks[i] = status ? -1 : ((i < n) ? dr[i] : (i == n ? tok_n : -1));
    recs[i] = RowRecord{};  // consumed: a call leaves the workspace zeroed
  }
  if (lane == 0) {
    if (MODE == kModeSci) {
      if (p.out_T) p.out_T[req] = float(thr);
      if (!status) {
        const double pacc = __ddiv_rn(double(n), double(K));
        p.r_hat[req] = __dadd_rn(__dmul_rn(__dsub_rn(1.0, p.ewma_beta), p.r_hat[req]), __dmul_rn(p.ewma_beta, pacc));
        if (p.sci_state) {
          SciState st;
          st.T_applied = thr;
          st.age = new_age;
          st.flags = 1u | (pacc < p.fb_acc ? 2u : 0u);
          p.sci_state[req] = st;
        }
      }
    }
    p.out_accept_len[req] = status ? 0 : n;
    p.out_req_status[req] = status;
    p.tickets[req] = 0u;
  }
  } else {
    // ---------------------------------------------------------------- multi-outcome row (sweep / fused)
    uint32_t flags = finite ? 0u : kBitNonfinite;
    uint32_t gate_bits = 0;
    if (pos < K) {
      if (!d_ok) {
        flags |= kBitBadDraft;
      } else if (finite) {
        // margin without ln(gamma); the gate for gamma_g is margin0 - ln(gamma_g) > 0.
        const double margin0 = (double(td) - lse_v) + double(D) - (double(bd) - lse_b);
        for (int g = 0; g < p.n_gamma; ++g)
          if (margin0 - p.ln_gammas[g] > 0.0) gate_bits |= 1u << g;
      }
    }
    if (lane == 0) {
      if (p.out_D) p.out_D[row] = finite ? D : __int_as_float(0x7fc00000);
      if (FUSE && p.out_J) p.out_J[row] = finite ? J : __int_as_float(0x7fc00000);
    }
    if (p.out_lse && lane < NT) p.out_lse[size_t(row) * 3 + lane] = float(my_lse);
    uint32_t ticket = 0;
    if (lane == 0) {
      MultiRecord rec;
      rec.J = double(J);
#pragma unroll
      for (int sl = 0; sl < kMaxArg; ++sl) rec.tok[sl] = (sl < NA && rc.rowi[sl] != INT_MAX) ? rc.rowi[sl] : 0;
      rec.gate_bits = gate_bits;
      rec.flags = flags;
      p.mrecords[row] = rec;
      ticket = atom_add_acq_rel_gpu(&p.tickets[req], 1u);
    }
    ticket = __shfl_sync(kAll, ticket, 0);
    if (ticket != uint32_t(K)) return;

    // Last row of this request: one scan per gamma (and, fused, the E2-SCI scan), 32 records a step.
    (void)ld_acquire_gpu(&p.tickets[req]);
    MultiRecord* recs = p.mrecords + size_t(req) * R1;
    double thr = 0.0;
    if (FUSE) {
      thr = __dadd_rn(p.T_base, __dmul_rn(p.alpha_omega, __dsub_rn(p.r_hat[req], p.tau_credit)));
      thr = fmax(p.T_min, fmin(thr, p.T_max));
    }
    uint32_t any = 0;
    int n_g[kMaxGamma];
#pragma unroll
    for (int g = 0; g < kMaxGamma; ++g) n_g[g] = K;
    int n_sci = K;
    for (int base = 0; base < R1; base += 32) {
      const int i = base + lane;
      uint32_t gb = 0, fl = 0;
      double jv = 0.0;
      if (i < R1) {
        const float4 w0 = ld_cg_f4(recs + i);
        const float4 w1 = ld_cg_f4(reinterpret_cast<const char*>(recs + i) + 16);
        jv = __hiloint2double(__float_as_int(w0.y), __float_as_int(w0.x));
        gb = __float_as_uint(w1.z);
        fl = __float_as_uint(w1.w);
      }
      any |= __reduce_or_sync(kAll, fl);
#pragma unroll
      for (int g = 0; g < kMaxGamma; ++g) {
        const unsigned rej = __ballot_sync(kAll, i < K && !((gb >> g) & 1u));
        if (n_g[g] == K && rej != 0u) n_g[g] = base + __ffs(rej) - 1;
      }
      if (FUSE) {
        const unsigned rej = __ballot_sync(kAll, i < K && jv > thr);
        if (n_sci == K && rej != 0u) n_sci = base + __ffs(rej) - 1;
      }
    }
    const uint32_t status = ((any & kBitNonfinite) ? 1u : 0u) | ((any & kBitBadDraft) ? 2u : 0u) |
                            ((any & kBitTimeout) ? 4u : 0u);
    const int32_t* dr = p.draft_ids + size_t(req) * K;
    const int B = p.B;
    for (int g = 0; g < p.n_gamma; ++g) {
      const int n = n_g[g];
      if (lane == 0) p.out_accept_len[size_t(g) * B + req] = status ? 0 : n;
      for (int b2 = 0; b2 < NB && b2 < p.n_beta; ++b2) {
        const int tok_n = __ldcg(&recs[n].tok[b2]);  // (L2: another SM wrote it)
        int32_t* toks = p.out_tokens + ((size_t(b2) * p.n_gamma + g) * B + req) * R1;
        for (int i = lane; i < R1; i += 32) toks[i] = status ? -1 : ((i < n) ? dr[i] : (i == n ? tok_n : -1));
      }
    }
    if constexpr (FUSE) {
      const int tok_n = __ldcg(&recs[n_sci].tok[NB]);
      int32_t* toks = p.out_sci_tokens + size_t(req) * R1;
      for (int i = lane; i < R1; i += 32) toks[i] = status ? -1 : ((i < n_sci) ? dr[i] : (i == n_sci ? tok_n : -1));
      if (lane == 0) {
        if (p.out_T) p.out_T[req] = float(thr);
        p.out_sci_accept_len[req] = status ? 0 : n_sci;
        if (!status) {
          const double pacc = __ddiv_rn(double(n_sci), double(K));
          p.r_hat[req] = __dadd_rn(__dmul_rn(__dsub_rn(1.0, p.ewma_beta), p.r_hat[req]), __dmul_rn(p.ewma_beta, pacc));
        }
      }
    }
    __syncwarp();
    for (int i = lane; i < R1; i += 32) recs[i] = MultiRecord{};  // consumed: the workspace is left zeroed
    if (lane == 0) {
      p.out_req_status[req] = status;
      p.tickets[req] = 0u;
    }
  }
}

}  // namespace asv
