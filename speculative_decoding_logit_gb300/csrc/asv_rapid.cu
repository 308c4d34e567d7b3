// asv_rapid.cu -- the RAPID verification kernel.
//
// Source: "RAPID: Long-Context Inference with Retrieval-Augmented Speculative Decoding" (paper
// notes): Workflow (rejection sampling against the augmented target); Key design 2 (augmented
// target zhat = z + eta*T*(q - p), p = softmax(z/T), phat = softmax(zhat/T)); Key design 3 (tokens
// whose augmented probability is below 10% of the peak keep the original target probability);
// Key design 4 (at a rejection the token is drawn from norm(max(p - phat, p - q, 0))).
//
// Decomposition as in the AsymSpec kernel: a cluster of C CTAs per row, CTA q owning entries
// [q*n_slice, (q+1)*n_slice) of z and q.  The kernel streams; it stages nothing in shared memory:
//   pass A  reads z and q from HBM once (16-byte loads that bypass L1, one vector prefetched):
//           running maximum of z/T and a sum of exp(z/T - ref) against a lazily moved reference,
//           the sum of q (finiteness), and the entries where z/T and q peak;
//   exch 1  row maximum M and S = sum exp(z/T - M), so p = exp(z/T - M) / S from here on; a lower
//           bound L0 on max zhat/T: zhat/T at the two peak entries;
//   pass B  re-reads z and q (the L2 cache still holds them: evict-last in pass A) and forms p and
//           zhat/T of every entry; running maximum of zhat/T.  An entry at or above (bound so far) +
//           ln(tail_frac), the bound being L0 or the thread's own maximum, may lie in the head
//           {zhat/T >= max + ln(tail_frac)}; a thread keeps up to two such candidates in registers
//           (dropping those the rising bound excludes); a third marks its CTA.  Under the second
//           tail reading (and for tail_frac = 0) pass B also sums p and exp(zhat/T - ref) over
//           every entry;
//   exch 2  row maximum Mh of zhat/T and the head boundary Mh + ln(tail_frac);
//   head    head sums (p-mass, exp(zhat/T - Mh)-mass) over the candidates -- every head entry is a
//           candidate, because the bound never exceeds Mh -- or, in a marked CTA, over a third read
//           of the slice (pass C, from L2);
//   exch 3  every CTA pushes its head sums into CTA 0 and leaves.
// The protected target is then p on the tail and exp(zhat/T - Mh) * (head p-mass / head exp-mass)
// on the head, which sums to 1 without a further normalisation pass.  The alternative reading of
// the protection (tail_mode 1: substitute p for phat on the tail, then renormalise every entry)
// makes the tail p / Z and the head phat / Z with Z = (tail p-mass) + (head phat-mass), the tail
// p-mass being (all p-mass) - (head p-mass).  CTA 0 of the row decides the draft's accept test
// u*q(d) < protected(d) (u from Philox4x32-10) and files a row record; the last row of a request
// to finish runs the scan, writes the outputs and leaves a draw job (the stop row and its
// constants).  A second launch, a group of CTAs per request, draws the emitted token at the stop
// position with an exponential race over that row (re-read from global memory): argmin_k E_k / w_k,
// E_k = -ln u_k, with w the residual max(p - protected, p - q, 0) or, at the bonus position, the
// protected target.  The draw is a programmatic dependent launch: every verification CTA signals
// at its start that the draw may be scheduled, so the draw's CTAs take the SM slots the
// verification's last CTAs leave free, and each waits (griddepcontrol.wait) for the whole
// verification to complete, its writes visible, before it reads anything.  No CTA waits on another
// cluster, and no CTA of the verification waits for its row's finalisation.
//
// Every quantity of an entry (p, zhat/T, the protected value) is formed by the same sequence of
// correctly rounded operations wherever it is needed -- pass B (two lanes per instruction), pass C,
// the accept test and the draw (one lane) -- so the head test gives the same answer everywhere.
#include <algorithm>
#include <climits>

#include "asv_device.cuh"
#include "asv_internal.h"

namespace asv {

constexpr int kRapidThreads = 256;    // threads per CTA (launch bounds)
constexpr int kRapidCtasPerSm = 4;    // CTAs per SM the kernel is compiled for (launch bounds)
constexpr float kRapidSlack = 64.0f;  // reference slack (log2 units), as in the AsymSpec kernel
constexpr int kDrawThreads = 256;     // threads per CTA of the draw launch
constexpr int kDrawStage = 6;         // slots of a draw thread's ring of vectors in shared memory
constexpr int kGroup = 4;             // vectors of a thread per stored bound of U (a power of 2)
// Pass A of aligned slices under the default tail reading streams through a per-thread ring of
// kRingA vectors of z and of q in shared memory, filled by 16-byte cp.async copies: the copies in
// flight hold no registers, so a thread keeps kRingA vectors per input on the way from HBM instead
// of the two a register prefetch affords (the verification is bound by the bytes in flight).
constexpr int kRingA = 4;  // a power of 2
constexpr int kRingABytes = kRingA * 2 * kRapidThreads * 16;

struct __align__(16) RapidXchg {
  // Exchange 1 (read by every CTA of the cluster).
  float zmax;  // CTA maximum of z/T
  float se[2];  // CTA sum of exp2(z/T log2e - ref(zmax)), hi + lo
  float sq[2];  // CTA sum of q, hi + lo
  float pk_v[2];    // peaks of z/T and of q in the CTA's slice: value,
  int32_t pk_i[2];  // index,
  float pk_z[2];    // z there,
  float pk_q[2];    // q there
  // Exchange 2.
  float zhmax;  // CTA maximum of zhat/T (at least L0)
  float ae[2];  // sum of exp2(zhat/T log2e - ref(zhmax)) over the slice (AE)
  float pa[2];  // sum of p over the slice (AE)
  // Exchange 3: pushed into CTA 0 by every CTA.  Head p-mass (hi, lo), head exp-mass (hi, lo).
  float head[kMaxCluster][4];
};

struct RowConsts {
  float invT, etaT, ML, inv_sum, zhmax, thr, head_scale, tail_scale;
};

// Row statistics, computed identically by warp 0 of every CTA and broadcast through shared memory.
struct __align__(16) RapidShared {
  float M;        // max z/T
  float inv_sum;  // 1 / sum exp2(z/T log2e - ML)
  float L0;       // lower bound of max zhat/T
  float zhmax;    // max zhat/T
  float ae_hi, ae_lo;  // row sum of exp2(zhat/T log2e - ref(zhmax)) (AE)
  float pa_hi, pa_lo;  // row sum of p (AE)
  int32_t finite;
};

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float ref_of(float M) { return isfinite(M) ? M * kLog2e : 0.0f; }

// Argmax over a warp carrying two payload values with the winner (larger value; ties: lower index).
__device__ __forceinline__ void warp_argmax_pl(float& v, int& i, float& a, float& b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    const float oa = __shfl_xor_sync(0xffffffffu, a, o);
    const float ob = __shfl_xor_sync(0xffffffffu, b, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
      a = oa;
      b = ob;
    }
  }
}

// p and zhat/T of one entry.  Explicitly rounded operations (no contraction), matching the
// two-lane forms of pass B bit for bit.
__device__ __forceinline__ void rapid_p_zhs(float z, float q, const RowConsts& c, float& p, float& zhs) {
  const float zs = __fmul_rn(z, c.invT);
  p = __fmul_rn(ex2_approx(__fmaf_rn(zs, kLog2e, -c.ML)), c.inv_sum);
  zhs = __fmul_rn(__fmaf_rn(c.etaT, __fsub_rn(q, p), z), c.invT);
}

// exp(zhat/T - Mh): the head weight.
__device__ __forceinline__ float head_exp(float zhs, float zhmax) {
  return ex2_approx(__fmul_rn(__fsub_rn(zhs, zhmax), kLog2e));
}

// p, zhat/T and the protected target of one entry.
__device__ __forceinline__ void rapid_entry(float z, float q, const RowConsts& c, float& p, float& zhs, float& prot) {
  rapid_p_zhs(z, q, c, p, zhs);
  prot = (zhs < c.thr) ? __fmul_rn(p, c.tail_scale) : __fmul_rn(head_exp(zhs, c.zhmax), c.head_scale);
}

// Four entries [k, k+4) of a row slice: one 16-byte load with an L2 policy when the slice is
// aligned, else element loads with `pad` at and beyond `lim`.
__device__ __forceinline__ float4 ld4(const float* base, int k, int lim, bool aligned, uint64_t pol, float pad) {
  float4 v;
  if (aligned) {
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(base + k), "l"(pol));
    return v;
  }
  v.x = (k + 0 < lim) ? __ldg(base + k + 0) : pad;
  v.y = (k + 1 < lim) ? __ldg(base + k + 1) : pad;
  v.z = (k + 2 < lim) ? __ldg(base + k + 2) : pad;
  v.w = (k + 3 < lim) ? __ldg(base + k + 3) : pad;
  return v;
}

// Four entries for a sparse re-read: an L1-allocating load (the same vector is read again soon).
__device__ __forceinline__ float4 ld4c(const float* base, int k, int lim, bool aligned, float pad) {
  if (aligned) return __ldg(reinterpret_cast<const float4*>(base + k));
  float4 v;
  v.x = (k + 0 < lim) ? __ldg(base + k + 0) : pad;
  v.y = (k + 1 < lim) ? __ldg(base + k + 1) : pad;
  v.z = (k + 2 < lim) ? __ldg(base + k + 2) : pad;
  v.w = (k + 3 < lim) ? __ldg(base + k + 3) : pad;
  return v;
}

// Two-lane p and zhat/T of the pairs (z, q) -- the operations of rapid_p_zhs, lane by lane.
__device__ __forceinline__ void pzhs2(float2 z, float2 q, float2 invT2, float2 nML2, float2 inv2, float2 etaT2,
                                      float2& pk, float2& zh) {
  const float2 zs = fmul2(z, invT2);
  const float2 y = ffma2(zs, make_float2(kLog2e, kLog2e), nML2);
  pk = fmul2(make_float2(ex2_approx(y.x), ex2_approx(y.y)), inv2);
  zh = fmul2(ffma2(etaT2, fsub2(q, pk), z), invT2);
}

// AE: the second tail reading (or tail_frac = 0) needs the all-entry sums of p and exp(zhat/T).
template <bool ALIGNED, bool AE>
__global__ void __launch_bounds__(kRapidThreads, kRapidCtasPerSm) rapid_kernel(const RapidArgs p) {
  constexpr int VEC = 4;
  constexpr int kWarps = kRapidThreads / 32;
  __shared__ RapidXchg xchg;
  __shared__ RapidShared rs;
  __shared__ float s_w[kWarps][4];
  __shared__ float s_pv[kWarps][2], s_pz[kWarps][2], s_pq[kWarps][2];
  __shared__ int32_t s_pi[kWarps][2];
  __shared__ int32_t s_cnt[kWarps];  // kRing, pass B: candidate groups per warp (list offsets)
  // Dynamic shared memory: the pass-A ring (kRing: [kRingA][z, q][kRapidThreads] 16-byte vectors),
  // then, !AE, for each thread and each group of kGroup of its vectors (vi = tid + j T, j = g kGroup
  // ... g kGroup + kGroup - 1), the maximum of U = fl(fl(fma(eta T, q, z)) / T) over their entries;
  // entry [g][tid].
  constexpr bool kRing = ALIGNED && !AE;
  constexpr uint32_t kUmaxOff = kRing ? uint32_t(kRingABytes) : 0u;
  extern __shared__ __align__(16) float4 s_dyn[];
  float4* const s_ring = s_dyn;
  float* const s_umax = reinterpret_cast<float*>(reinterpret_cast<char*>(s_dyn) + kUmaxOff);

  // The draw launch may be scheduled once every CTA of this grid has started (it waits for this
  // grid's completion before reading anything).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();
  const int row = blockIdx.x / C;
  const int G = p.G;
  const int R1 = G + 1;
  const int req = row / R1;
  const int pos = row - req * R1;
  const int V = p.V;
  const int v0 = int(rank) * p.n_slice;
  // (checked build: a row outside the batch, or a cluster larger than the exchange arrays, reads
  // nothing; every CTA still takes part in the cluster barriers)
  const bool row_ok = ASV_GUARD(p, row >= 0 && row < p.B * R1 && rank < uint32_t(kMaxCluster) && C <= uint32_t(kMaxCluster));
  const int len = row_ok ? max(0, min(V - v0, p.n_slice)) : 0;
  const int nvec = (len + VEC - 1) / VEC;
  const size_t row_base = size_t(row) * size_t(V);
  const float* zsl = p.z + row_base + v0;
#ifdef ASV_CHECKED
  uint32_t dyn_smem = 0;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_smem));
#endif
  // One vector of the slice (checked build: its entries must lie in the slice).
  auto LD4 = [&](const float* base, int k, uint64_t pol, float pad) {
    return ASV_GUARD(p, k >= 0 && (!ALIGNED || k + VEC <= len)) ? ld4(base, k, len, ALIGNED, pol, pad)
                                                            : make_float4(pad, pad, pad, pad);
  };
  auto LD4C = [&](const float* base, int k, float pad) {
    return ASV_GUARD(p, k >= 0 && (!ALIGNED || k + VEC <= len)) ? ld4c(base, k, len, ALIGNED, pad)
                                                            : make_float4(pad, pad, pad, pad);
  };
  const float* qsl = p.q + row_base + v0;
  const uint64_t pol_keep = policy_evict_last();
  const uint64_t pol_evict_first = policy_evict_first();
  const float invT = p.inv_T;
  const float etaT = p.eta * p.T;
  const float ln_tf = p.ln_tail_frac;
  const bool cand_on = ln_tf > -INFINITY;  // tail_frac = 0 puts every entry in the head
  const float2 invT2 = make_float2(invT, invT);
  const float2 etaT2 = make_float2(etaT, etaT);

  // The draft token's z and q for the accept test in CTA 0 (loaded now, used at the end).
  int d = -1;
  float zd = 0.0f, qd = 0.0f;
  if (rank == 0 && tid == 0 && pos < G && row_ok) {
    d = p.draft_ids[size_t(req) * G + pos];
    if (d >= 0 && d < V) {
      zd = __ldg(p.z + row_base + d);
      qd = __ldg(p.q + row_base + d);
    }
  }

  // ---------------------------------------------------------------- pass A (HBM)
  float thr = -INFINITY, mL = 0.0f;
  float2 acc = make_float2(0.0f, 0.0f), qacc = make_float2(0.0f, 0.0f);
  float ub_t = -INFINITY;  // !AE: the largest bound this thread stored
  // Peaks: [0] of z/T (its value is the thread's running maximum; payload z, q), [1] of the second
  // key below (payload z, q).
  float pv[2] = {-INFINITY, -INFINITY}, pz[2] = {0.0f, 0.0f}, pq[2] = {0.0f, 0.0f};
  int pi[2] = {INT_MAX, INT_MAX};
  {
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    // AE: pass B re-reads the whole slice (keep it in L2); else only a few vectors.
    const uint64_t polA = AE ? pol_keep : pol_evict_first;
    float gmax = -INFINITY;
    int it = 0;
    int vi = tid;
    // One vector (entries [vi*VEC, vi*VEC + VEC) of the slice) of z and q into the pass-A state.
    auto a_body = [&](const float4& cz, const float4& cq, const int vi) {
      const int vn = vi + kRapidThreads;
      const float2 s0 = fmul2(make_float2(cz.x, cz.y), invT2);
      const float2 s1 = fmul2(make_float2(cz.z, cz.w), invT2);
      const float vm = fmaxf(fmaxf(s0.x, s0.y), fmaxf(s1.x, s1.y));
      // The second peak's key: !AE, U = fl(fl(fma(eta T, q, z)) / T), which bounds zhat/T entry by
      // entry (p >= 0, every operation monotone and correctly rounded); AE, q.
      float2 k0, k1;
      if constexpr (!AE) {
        k0 = fmul2(ffma2(etaT2, make_float2(cq.x, cq.y), make_float2(cz.x, cz.y)), invT2);
        k1 = fmul2(ffma2(etaT2, make_float2(cq.z, cq.w), make_float2(cz.z, cz.w)), invT2);
      } else {
        k0 = make_float2(cq.x, cq.y);
        k1 = make_float2(cq.z, cq.w);
      }
      const float vk = fmaxf(fmaxf(k0.x, k0.y), fmaxf(k1.x, k1.y));
      if constexpr (!AE) {
        // One bound per kGroup consecutive vectors of this thread.
        gmax = fmaxf(gmax, vk);
        if ((it & (kGroup - 1)) == kGroup - 1 || vn >= nvec) {
#ifdef ASV_CHECKED
          if (ASV_GUARD(p, kUmaxOff + uint32_t(((it / kGroup) * kRapidThreads + tid) * 4) < dyn_smem))
#endif
            s_umax[(it / kGroup) * kRapidThreads + tid] = gmax;
          ub_t = fmaxf(ub_t, gmax);
          gmax = -INFINITY;
        }
        ++it;
      }
      if (vm > pv[0] || vk > pv[1]) {
        const float zv[4] = {cz.x, cz.y, cz.z, cz.w};
        const float qv[4] = {cq.x, cq.y, cq.z, cq.w};
        const int kb = v0 + vi * VEC;
        // The first entry holding the vector's peak, and its payload (unrolled selects).
        if (vm > pv[0]) {
          const float sv[4] = {s0.x, s0.y, s1.x, s1.y};
          int e = 3;
          float a = zv[3], b = qv[3];
#pragma unroll
          for (int j = 2; j >= 0; --j)
            if (sv[j] == vm) {
              e = j;
              a = zv[j];
              b = qv[j];
            }
          pv[0] = vm;
          pi[0] = kb + e;
          pz[0] = a;
          pq[0] = b;
          if (vm > thr && isfinite(vm)) {
            // Move the partial sum to a reference at the new maximum (about once per thread).
            const float nL = vm * kLog2e;
            if (thr == -INFINITY || nL > mL + kRapidSlack) {
              const float f = (acc.x != 0.0f || acc.y != 0.0f) ? exp2f(mL - nL) : 0.0f;
              acc = fmul2(acc, make_float2(f, f));
              mL = nL;
              thr = (nL + kRapidSlack) * 0.693147180559945f;
            }
          }
        }
        if (vk > pv[1]) {
          const float kv[4] = {k0.x, k0.y, k1.x, k1.y};
          int e = 3;
          float a = zv[3], b = qv[3];
#pragma unroll
          for (int j = 2; j >= 0; --j)
            if (kv[j] == vk) {
              e = j;
              a = zv[j];
              b = qv[j];
            }
          pv[1] = vk;
          pi[1] = kb + e;
          pz[1] = a;
          pq[1] = b;
        }
      }
      const float2 y0 = ffma2(s0, l2e2, make_float2(-mL, -mL));
      const float2 y1 = ffma2(s1, l2e2, make_float2(-mL, -mL));
      acc = fadd2(acc, make_float2(ex2_approx(y0.x), ex2_approx(y0.y)));
      acc = fadd2(acc, make_float2(ex2_approx(y1.x), ex2_approx(y1.y)));
      qacc = fadd2(qacc, make_float2(cq.x, cq.y));
      qacc = fadd2(qacc, make_float2(cq.z, cq.w));
    };
    if constexpr (kRing) {
      // Vector j of the thread (vi = tid + j T) goes to slot j mod kRingA; each thread reads only its
      // own slots and refills a slot only after the arithmetic has consumed it.
      auto ring_issue = [&](int j) {
        const int v = tid + j * kRapidThreads;
        if (v < nvec) {
          const int slot = (j & (kRingA - 1)) * 2;
          if (ASV_GUARD(p, v * VEC + VEC <= len &&
                               uint32_t(((slot + 1) * kRapidThreads + tid + 1) * 16) <= dyn_smem)) {
            cp_async16(smem_addr(&s_ring[(slot + 0) * kRapidThreads + tid]), zsl + v * VEC, pol_evict_first);
            cp_async16(smem_addr(&s_ring[(slot + 1) * kRapidThreads + tid]), qsl + v * VEC, pol_evict_first);
          }
        }
        cp_async_commit();
      };
#pragma unroll
      for (int j = 0; j < kRingA; ++j) ring_issue(j);
      for (int j = 0; vi < nvec; ++j, vi += kRapidThreads) {
        cp_async_wait_group<kRingA - 1>();  // the copies of vector j have landed
        const int slot = (j & (kRingA - 1)) * 2;
        const float4 cz = s_ring[(slot + 0) * kRapidThreads + tid];
        const float4 cq = s_ring[(slot + 1) * kRapidThreads + tid];
        a_body(cz, cq, vi);
        ring_issue(j + kRingA);
      }
      cp_async_wait_all();
    } else {
      float4 cz, cq, nz, nq;
      if (vi < nvec) {
        cz = LD4(zsl, vi * VEC, polA, -INFINITY);
        cq = LD4(qsl, vi * VEC, polA, 0.0f);
      }
      // Two vectors per trip, the prefetch alternating between (cz, cq) and (nz, nq) (no register
      // copies); a prefetched vector is consumed only while it is in range.
      for (; vi < nvec; vi += 2 * kRapidThreads) {
        if (vi + kRapidThreads < nvec) {
          nz = LD4(zsl, (vi + kRapidThreads) * VEC, polA, -INFINITY);
          nq = LD4(qsl, (vi + kRapidThreads) * VEC, polA, 0.0f);
        }
        a_body(cz, cq, vi);
        if (vi + kRapidThreads >= nvec) break;
        if (vi + 2 * kRapidThreads < nvec) {
          cz = LD4(zsl, (vi + 2 * kRapidThreads) * VEC, polA, -INFINITY);
          cq = LD4(qsl, (vi + 2 * kRapidThreads) * VEC, polA, 0.0f);
        }
        a_body(nz, nq, vi + kRapidThreads);
      }
    }
  }

  // CTA statistics: maximum; sums moved to the CTA reference; peaks.  Each warp reduces its own
  // (its sum against its own maximum), then lanes of warp 0 combine the warps' results, each reading
  // its values of every warp (reads issued together) and adding them in registers in warp order.
  // The serial sections of a row keep dependent shuffle and shared-memory round trips few: while
  // other CTAs on the SM stream their loads, each such round trip waits behind those loads.
  {
    const float w = warp_max(pv[0]);
#pragma unroll
    for (int k = 0; k < 2; ++k) warp_argmax_pl(pv[k], pi[k], pz[k], pq[k]);
    const float s = acc.x + acc.y;
    const float ws = warp_sum_f((s != 0.0f) ? s * exp2f(mL - ref_of(w)) : 0.0f);
    const float wq = warp_sum_f(qacc.x + qacc.y);
    if (lane == 0) {
      s_w[warp][0] = ws;
      s_w[warp][1] = wq;
      s_w[warp][3] = w;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        s_pv[warp][k] = pv[k];
        s_pi[warp][k] = pi[k];
        s_pz[warp][k] = pz[k];
        s_pq[warp][k] = pq[k];
      }
    }
    __syncthreads();
    if (warp == 0 && lane < 4) {
      if (lane == 0) {  // maximum of z/T and the exp sum against it
        float m[kWarps], sw[kWarps];
#pragma unroll
        for (int k = 0; k < kWarps; ++k) {
          m[k] = s_w[k][3];
          sw[k] = s_w[k][0];
        }
        float Mc = m[0];
#pragma unroll
        for (int k = 1; k < kWarps; ++k) Mc = fmaxf(Mc, m[k]);
        const float Rc = ref_of(Mc);
        DF d{0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < kWarps; ++k) {
          if (sw[k] != 0.0f) d = df_add(d, DF{sw[k] * exp2f(ref_of(m[k]) - Rc), 0.0f});
        }
        xchg.zmax = Mc;
        xchg.se[0] = d.hi;
        xchg.se[1] = d.lo;
      } else if (lane == 1) {  // sum of q
        float x[kWarps];
#pragma unroll
        for (int k = 0; k < kWarps; ++k) x[k] = s_w[k][1];
        DF d{x[0], 0.0f};
#pragma unroll
        for (int k = 1; k < kWarps; ++k) d = df_add(d, DF{x[k], 0.0f});
        xchg.sq[0] = d.hi;
        xchg.sq[1] = d.lo;
      } else {  // peak slot lane - 2
        const int k = lane - 2;
        float v = s_pv[0][k], a = s_pz[0][k], b = s_pq[0][k];
        int i = s_pi[0][k];
#pragma unroll
        for (int w2 = 1; w2 < kWarps; ++w2) {
          const float ov = s_pv[w2][k];
          const int oi = s_pi[w2][k];
          if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
            a = s_pz[w2][k];
            b = s_pq[w2][k];
          }
        }
        xchg.pk_v[k] = v;
        xchg.pk_i[k] = i;
        xchg.pk_z[k] = a;
        xchg.pk_q[k] = b;
      }
    }
  }
  cluster_sync_w0(warp);  // #1

  // ---------------------------------------------------------------- row statistics (warp 0)
  if (warp == 0) {
    // Lane 0: maximum of z/T and the exp sum; lane 1: sum of q; lanes 2, 3: peak slot lane - 2 --
    // each over the cluster's CTAs, four CTAs' values read at a time (remote reads issued together)
    // and combined in registers in rank order; one batch of shuffles brings them to lane 0.
    const int ks = (lane == 3) ? 1 : 0;
    const uint32_t o0 = (lane >= 2) ? uint32_t(offsetof(RapidXchg, pk_v)) + 4u * ks : uint32_t(offsetof(RapidXchg, zmax));
    const uint32_t o1 = (lane == 0) ? uint32_t(offsetof(RapidXchg, se))
                        : (lane == 1) ? uint32_t(offsetof(RapidXchg, sq)) : uint32_t(offsetof(RapidXchg, pk_z)) + 4u * ks;
    const uint32_t o2 = (lane < 2) ? o1 + 4u : uint32_t(offsetof(RapidXchg, pk_q)) + 4u * ks;
    const uint32_t o3 = uint32_t(offsetof(RapidXchg, pk_i)) + 4u * ks;
    const uint32_t base = smem_addr(&xchg);
    float mq = -INFINITY;  // lane 0: maximum so far; lanes 2, 3: peak value so far
    DF sx{0.0f, 0.0f};     // lane 0: exp sum against ref_of(mq); lane 1: q sum
    float pa_ = 0.0f, pb_ = 0.0f;
    int pi_ = INT_MAX;
    for (uint32_t q0 = 0; q0 < C; q0 += 4) {
      float f0[4], f1[4], f2[4];
      int f3[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t q = (q0 + u < C) ? q0 + u : 0u;
        f0[u] = dsmem_ld_f32(dsmem_map(base + o0, q));
        f1[u] = dsmem_ld_f32(dsmem_map(base + o1, q));
        f2[u] = dsmem_ld_f32(dsmem_map(base + o2, q));
        f3[u] = dsmem_ld_s32(dsmem_map(base + o3, q));
      }
      if (lane == 0) {
        float Mn = mq;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q0 + u < C) Mn = fmaxf(Mn, f0[u]);
        const float Rn = ref_of(Mn);
        if (sx.hi != 0.0f) {  // (more than four CTAs) move the running sum to the new reference
          const float g = exp2f(ref_of(mq) - Rn);
          sx = DF{sx.hi * g, sx.lo * g};
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (q0 + u < C && f1[u] != 0.0f) {
            const float g = exp2f(ref_of(f0[u]) - Rn);
            sx = df_add(sx, DF{f1[u] * g, f2[u] * g});
          }
        }
        mq = Mn;
      } else if (lane == 1) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q0 + u < C) sx = df_add(sx, DF{f1[u], f2[u]});
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (q0 + u < C && (f0[u] > mq || (f0[u] == mq && f3[u] < pi_))) {
            mq = f0[u];
            pi_ = f3[u];
            pa_ = f1[u];
            pb_ = f2[u];
          }
        }
      }
    }
    const unsigned kAll = 0xffffffffu;
    const float M = mq;  // lane 0
    const DF S = sx;     // lane 0
    const DF Q{__shfl_sync(kAll, sx.hi, 1), __shfl_sync(kAll, sx.lo, 1)};
    float v[2], a[2], b[2];
    int i[2];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      v[kk] = __shfl_sync(kAll, mq, 2 + kk);
      i[kk] = __shfl_sync(kAll, pi_, 2 + kk);
      a[kk] = __shfl_sync(kAll, pa_, 2 + kk);
      b[kk] = __shfl_sync(kAll, pb_, 2 + kk);
    }
    (void)v;
    const float ML = ref_of(M);
    if (lane == 0) {
      const bool fin = isfinite(M) && isfinite(S.hi) && S.hi > 0.0f && isfinite(Q.hi);
      rs.M = M;
      rs.finite = fin ? 1 : 0;
      rs.inv_sum = fin ? 1.0f / (S.hi + S.lo) : 0.0f;
      // L0: zhat/T at the peaks of z/T and of q (entries of this row, so L0 <= max zhat/T).
      float L0 = -INFINITY;
      if (fin) {
        RowConsts c;
        c.invT = invT;
        c.etaT = etaT;
        c.ML = ML;
        c.inv_sum = rs.inv_sum;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (i[k] != INT_MAX) {
            float pk, zh;
            rapid_p_zhs(a[k], b[k], c, pk, zh);
            L0 = fmaxf(L0, zh);
          }
        }
      }
      rs.L0 = L0;
    }
  }
  __syncthreads();
  const bool finite = rs.finite != 0;
  RowConsts rc;
  rc.invT = invT;
  rc.etaT = etaT;
  rc.ML = ref_of(rs.M);
  rc.inv_sum = rs.inv_sum;
  rc.zhmax = 0.0f;
  rc.thr = 0.0f;
  rc.head_scale = 0.0f;
  rc.tail_scale = 1.0f;

  // ---------------------------------------------------------------- pass B
  // AE: every entry (L2), with head candidates and the all-entry sums.  Otherwise only the vectors
  // whose bound max U reaches L0 + ln(tail_frac): the maximum of zhat/T (>= L0) and every head entry
  // (>= Mh + ln(tail_frac) >= L0 + ln(tail_frac)) lie there, since zhat/T <= U.
  float L = rs.L0;  // bound: L0, raised by this thread's own entries; ends as its max of zhat/T
  float c0z = 0.0f, c0p = 0.0f, c1z = 0.0f, c1p = 0.0f;  // head candidates (zhat/T, p)
  int nc = 0;
  bool ovf = false;
  float2 aacc = make_float2(0.0f, 0.0f), pall = make_float2(0.0f, 0.0f);
  float aL = ref_of(L), athr = isfinite(L) ? (aL + kRapidSlack) * 0.693147180559945f : -INFINITY;
  if (AE && finite) {
    const float2 nML2 = make_float2(-rc.ML, -rc.ML);
    const float2 inv2 = make_float2(rc.inv_sum, rc.inv_sum);
    float cthr = cand_on ? L + ln_tf : INFINITY;
    int vi = tid;
    float4 cz, cq, nz, nq;
    if (vi < nvec) {
      cz = LD4(zsl, vi * VEC, pol_evict_first, -INFINITY);
      cq = LD4(qsl, vi * VEC, pol_evict_first, 0.0f);
    }
    for (; vi < nvec; vi += kRapidThreads) {
      const int vn = vi + kRapidThreads;
      if (vn < nvec) {
        nz = LD4(zsl, vn * VEC, pol_evict_first, -INFINITY);
        nq = LD4(qsl, vn * VEC, pol_evict_first, 0.0f);
      }
      float2 p0, p1, h0, h1;
      pzhs2(make_float2(cz.x, cz.y), make_float2(cq.x, cq.y), invT2, nML2, inv2, etaT2, p0, h0);
      pzhs2(make_float2(cz.z, cz.w), make_float2(cq.z, cq.w), invT2, nML2, inv2, etaT2, p1, h1);
      const float vm = fmaxf(fmaxf(h0.x, h0.y), fmaxf(h1.x, h1.y));
      const float Ln = fmaxf(L, vm);
      if (vm >= cthr || (AE && vm > athr)) {
        if (cand_on) {
          if (Ln > L) {
            // The bound rose: drop candidates below the new boundary (they cannot be head entries).
            cthr = Ln + ln_tf;
            if (nc == 2 && c1z < cthr) nc = 1;
            if (nc >= 1 && c0z < cthr) {
              c0z = c1z;
              c0p = c1p;
              nc -= 1;
            }
          }
          const float hv[4] = {h0.x, h0.y, h1.x, h1.y};
          const float pv4[4] = {p0.x, p0.y, p1.x, p1.y};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (hv[e] >= cthr) {
              if (nc == 0) {
                c0z = hv[e];
                c0p = pv4[e];
                nc = 1;
              } else if (nc == 1) {
                c1z = hv[e];
                c1p = pv4[e];
                nc = 2;
              } else {
                ovf = true;
              }
            }
          }
        }
        if (AE && vm > athr && isfinite(Ln)) {
          const float nL = Ln * kLog2e;
          if (athr == -INFINITY || nL > aL + kRapidSlack) {
            const float f = (aacc.x != 0.0f || aacc.y != 0.0f) ? exp2f(aL - nL) : 0.0f;
            aacc = fmul2(aacc, make_float2(f, f));
            aL = nL;
            athr = (nL + kRapidSlack) * 0.693147180559945f;
          }
        }
      }
      L = Ln;
      if constexpr (AE) {
        const float2 l2e2 = make_float2(kLog2e, kLog2e);
        const float2 y0 = ffma2(h0, l2e2, make_float2(-aL, -aL));
        const float2 y1 = ffma2(h1, l2e2, make_float2(-aL, -aL));
        aacc = fadd2(aacc, make_float2(ex2_approx(y0.x), ex2_approx(y0.y)));
        aacc = fadd2(aacc, make_float2(ex2_approx(y1.x), ex2_approx(y1.y)));
        pall = fadd2(pall, p0);
        pall = fadd2(pall, p1);
      }
      cz = nz;
      cq = nq;
    }
  }
  // kRing: the vector groups whose bound reaches L0 + ln(tail_frac) are listed for the whole CTA
  // (in the pass-A ring, free now; thread order, then group order: a deterministic list) and the
  // CTA's threads share them out, so a slice whose candidates crowd into a few threads' groups
  // costs a few memory round trips per thread rather than one per group on those threads.  The
  // head sums walk the same list.  (A list that would not fit falls back to each thread's own
  // groups.)
  int n_list = -1;  // kRing: entries of the list (-1: not used)
  if (kRing && finite) {
    const float thrU = L + ln_tf;  // L = L0 here, the same in every thread
    const int ng = (nvec - tid + kGroup * kRapidThreads - 1) / (kGroup * kRapidThreads);  // this thread's groups
    int cnt = 0;
    if (ub_t >= thrU)
      for (int g = 0; g < ng; ++g) cnt += (s_umax[g * kRapidThreads + tid] >= thrU) ? 1 : 0;
    int incl = cnt;  // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_cnt[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      const int c = s_cnt[w2];
      base += (w2 < warp) ? c : 0;
      total += c;
    }
    constexpr int kListCap = kRingABytes / 4;
    if (total <= kListCap) {
      int32_t* const s_list = reinterpret_cast<int32_t*>(s_ring);
      int off = base + incl - cnt;
      if (cnt > 0)
        for (int g = 0; g < ng; ++g)
          if (s_umax[g * kRapidThreads + tid] >= thrU && ASV_GUARD(p, off < kListCap)) s_list[off++] = g * kRapidThreads + tid;
      n_list = total;
    }
    __syncthreads();
  }
  if (n_list >= 0) {
    const float2 nML2 = make_float2(-rc.ML, -rc.ML);
    const float2 inv2 = make_float2(rc.inv_sum, rc.inv_sum);
    const int32_t* const s_list = reinterpret_cast<const int32_t*>(s_ring);
    for (int e = tid; e < n_list; e += kRapidThreads) {
      const int u = s_list[e];
      const int g = u / kRapidThreads, t = u - g * kRapidThreads;
#pragma unroll
      for (int r = 0; r < kGroup; ++r) {
        const int vi = (g * kGroup + r) * kRapidThreads + t;
        if (vi < nvec) {
          const float4 z4 = LD4C(zsl, vi * VEC, -INFINITY);
          const float4 q4 = LD4C(qsl, vi * VEC, 0.0f);
          float2 p0, p1, h0, h1;
          pzhs2(make_float2(z4.x, z4.y), make_float2(q4.x, q4.y), invT2, nML2, inv2, etaT2, p0, h0);
          pzhs2(make_float2(z4.z, z4.w), make_float2(q4.z, q4.w), invT2, nML2, inv2, etaT2, p1, h1);
          L = fmaxf(L, fmaxf(fmaxf(h0.x, h0.y), fmaxf(h1.x, h1.y)));
        }
      }
    }
  } else if (!AE && finite && ub_t >= L + ln_tf) {
    const float2 nML2 = make_float2(-rc.ML, -rc.ML);
    const float2 inv2 = make_float2(rc.inv_sum, rc.inv_sum);
    const float thrU = L + ln_tf;
    for (int g = 0; g * kGroup * kRapidThreads + tid < nvec; ++g) {
      if (s_umax[g * kRapidThreads + tid] >= thrU) {
#pragma unroll
        for (int r = 0; r < kGroup; ++r) {
          const int vi = (g * kGroup + r) * kRapidThreads + tid;
          if (vi < nvec) {
            const float4 z4 = LD4C(zsl, vi * VEC, -INFINITY);
            const float4 q4 = LD4C(qsl, vi * VEC, 0.0f);
            float2 p0, p1, h0, h1;
            pzhs2(make_float2(z4.x, z4.y), make_float2(q4.x, q4.y), invT2, nML2, inv2, etaT2, p0, h0);
            pzhs2(make_float2(z4.z, z4.w), make_float2(q4.z, q4.w), invT2, nML2, inv2, etaT2, p1, h1);
            L = fmaxf(L, fmaxf(fmaxf(h0.x, h0.y), fmaxf(h1.x, h1.y)));
          }
        }
      }
    }
  }
  {
    // As at the first exchange: each warp reduces against its own maximum, lanes 0 and 1 of warp 0
    // combine the warps' results in registers.
    const float w = warp_max(L);
    float wa = 0.0f, wp = 0.0f;
    if constexpr (AE) {
      const float s = aacc.x + aacc.y;
      wa = warp_sum_f((s != 0.0f) ? s * exp2f(aL - ref_of(w)) : 0.0f);
      wp = warp_sum_f(pall.x + pall.y);
    }
    if (lane == 0) {
      s_w[warp][0] = wa;
      s_w[warp][1] = wp;
      s_w[warp][3] = w;
    }
    __syncthreads();
    if (warp == 0 && lane < 2) {
      if (lane == 0) {  // maximum of zhat/T and (AE) the exp sum against it
        float m[kWarps], sw[kWarps];
#pragma unroll
        for (int k = 0; k < kWarps; ++k) {
          m[k] = s_w[k][3];
          sw[k] = s_w[k][0];
        }
        float Mc = m[0];
#pragma unroll
        for (int k = 1; k < kWarps; ++k) Mc = fmaxf(Mc, m[k]);
        DF d{0.0f, 0.0f};
        if constexpr (AE) {
          const float Rc = ref_of(Mc);
#pragma unroll
          for (int k = 0; k < kWarps; ++k) {
            if (sw[k] != 0.0f) d = df_add(d, DF{sw[k] * exp2f(ref_of(m[k]) - Rc), 0.0f});
          }
        }
        xchg.zhmax = Mc;
        xchg.ae[0] = d.hi;
        xchg.ae[1] = d.lo;
      } else {  // (AE) sum of p
        DF d{0.0f, 0.0f};
        if constexpr (AE) {
          float x[kWarps];
#pragma unroll
          for (int k = 0; k < kWarps; ++k) x[k] = s_w[k][1];
          d = DF{x[0], 0.0f};
#pragma unroll
          for (int k = 1; k < kWarps; ++k) d = df_add(d, DF{x[k], 0.0f});
        }
        xchg.pa[0] = d.hi;
        xchg.pa[1] = d.lo;
      }
    }
  }
  const bool cta_ovf = __syncthreads_or(ovf ? 1 : 0) != 0;
  cluster_sync_w0(warp);  // #2

  if (warp == 0) {
    // Lane 0: maximum of zhat/T and (AE) the exp sum; lane 1: (AE) sum of p -- over the cluster's
    // CTAs, four CTAs' values read at a time, combined in registers in rank order.
    const uint32_t base = smem_addr(&xchg);
    const uint32_t o0 = uint32_t(offsetof(RapidXchg, zhmax));
    const uint32_t o1 = (lane == 0) ? uint32_t(offsetof(RapidXchg, ae)) : uint32_t(offsetof(RapidXchg, pa));
    float mq = -INFINITY;
    DF sx{0.0f, 0.0f};
    for (uint32_t q0 = 0; q0 < C; q0 += 4) {
      float f0[4], f1[4], f2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t q = (q0 + u < C) ? q0 + u : 0u;
        f0[u] = dsmem_ld_f32(dsmem_map(base + o0, q));
        if constexpr (AE) {
          f1[u] = dsmem_ld_f32(dsmem_map(base + o1, q));
          f2[u] = dsmem_ld_f32(dsmem_map(base + o1 + 4u, q));
        } else {
          f1[u] = 0.0f;
          f2[u] = 0.0f;
        }
      }
      if (lane == 0) {
        float Mn = mq;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q0 + u < C) Mn = fmaxf(Mn, f0[u]);
        if constexpr (AE) {
          const float Rn = ref_of(Mn);
          if (sx.hi != 0.0f) {
            const float g = exp2f(ref_of(mq) - Rn);
            sx = DF{sx.hi * g, sx.lo * g};
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (q0 + u < C && f1[u] != 0.0f) {
              const float g = exp2f(ref_of(f0[u]) - Rn);
              sx = df_add(sx, DF{f1[u] * g, f2[u] * g});
            }
          }
        }
        mq = Mn;
      } else if (AE) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q0 + u < C) sx = df_add(sx, DF{f1[u], f2[u]});
      }
    }
    const DF sp{__shfl_sync(0xffffffffu, sx.hi, 1), __shfl_sync(0xffffffffu, sx.lo, 1)};
    if (lane == 0) {
      rs.zhmax = mq;
      rs.ae_hi = sx.hi;
      rs.ae_lo = sx.lo;
      rs.pa_hi = sp.hi;
      rs.pa_lo = sp.lo;
    }
  }
  __syncthreads();
  rc.zhmax = rs.zhmax;
  rc.thr = rs.zhmax + ln_tf;

  // ---------------------------------------------------------------- head sums
  {
    float hp = 0.0f, he = 0.0f;
    // One vector of the slice into the head sums.
    auto head_vec = [&](int vi) {
      const float4 z4 = LD4C(zsl, vi * VEC, -INFINITY);
      const float4 q4 = LD4C(qsl, vi * VEC, 0.0f);
      const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
      const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float pk, zh;
        rapid_p_zhs(zz[e], qq[e], rc, pk, zh);
        if (zh >= rc.thr) {
          hp += pk;
          he += head_exp(zh, rc.zhmax);
        }
      }
    };
    if (n_list >= 0) {
      // The head lies in the listed groups whose bound reaches the boundary (re-read, normally
      // from L1).
      const int32_t* const s_list = reinterpret_cast<const int32_t*>(s_ring);
      for (int e = tid; e < n_list; e += kRapidThreads) {
        const int u = s_list[e];
        if (s_umax[u] >= rc.thr) {
          const int g = u / kRapidThreads, t = u - g * kRapidThreads;
          for (int r = 0; r < kGroup; ++r) {
            const int vi = (g * kGroup + r) * kRapidThreads + t;
            if (vi >= nvec) break;
            head_vec(vi);
          }
        }
      }
    } else if (!AE && finite && ub_t >= rc.thr) {
      // The head lies in the vectors whose bound reaches the boundary (re-read, normally from L1).
      for (int g = 0; g * kGroup * kRapidThreads + tid < nvec; ++g) {
        if (s_umax[g * kRapidThreads + tid] >= rc.thr) {
          for (int r = 0; r < kGroup; ++r) {
            const int vi = (g * kGroup + r) * kRapidThreads + tid;
            if (vi >= nvec) break;
            head_vec(vi);
          }
        }
      }
    }
    if (AE && finite && cand_on) {
      if (!cta_ovf) {
        if (nc >= 1 && c0z >= rc.thr) {
          hp += c0p;
          he += head_exp(c0z, rc.zhmax);
        }
        if (nc >= 2 && c1z >= rc.thr) {
          hp += c1p;
          he += head_exp(c1z, rc.zhmax);
        }
      } else {
        // Pass C: a thread ran out of candidate slots; test every entry of the slice.
        for (int vi = tid; vi < nvec; vi += kRapidThreads) {
          const float4 z4 = LD4(zsl, vi * VEC, pol_evict_first, -INFINITY);
          const float4 q4 = LD4(qsl, vi * VEC, pol_evict_first, 0.0f);
          const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
          const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pk, zh;
            rapid_p_zhs(zz[e], qq[e], rc, pk, zh);
            if (zh >= rc.thr) {
              hp += pk;
              he += head_exp(zh, rc.zhmax);
            }
          }
        }
      }
    }
    const float wh = warp_sum_f(hp);
    const float we = warp_sum_f(he);
    if (lane == 0) {
      s_w[warp][0] = wh;
      s_w[warp][1] = we;
    }
    __syncthreads();
    if (warp == 0) {
      // Lane k < kWarps holds warp k's sums; a butterfly over those lanes only (three steps).
      DF dh{lane < kWarps ? s_w[lane][0] : 0.0f, 0.0f}, de{lane < kWarps ? s_w[lane][1] : 0.0f, 0.0f};
#pragma unroll
      for (int o = kWarps / 2; o > 0; o >>= 1) {
        dh = df_add(dh, DF{__shfl_xor_sync(0xffffffffu, dh.hi, o), __shfl_xor_sync(0xffffffffu, dh.lo, o)});
        de = df_add(de, DF{__shfl_xor_sync(0xffffffffu, de.hi, o), __shfl_xor_sync(0xffffffffu, de.lo, o)});
      }
      if (lane == 0 && ASV_GUARD(p, rank < uint32_t(kMaxCluster))) {
        const uint32_t base = smem_addr(&xchg.head[rank][0]);
        dsmem_st_f32(dsmem_map(base + 0, 0), dh.hi);
        dsmem_st_f32(dsmem_map(base + 4, 0), dh.lo);
        dsmem_st_f32(dsmem_map(base + 8, 0), de.hi);
        dsmem_st_f32(dsmem_map(base + 12, 0), de.lo);
      }
    }
  }
  cluster_sync_w0(warp);  // #3: after this only CTA 0 touches shared memory, and only its own
  if (rank != 0 || warp != 0) return;

  // ---------------------------------------------------------------- row finalisation (CTA 0, warp 0)
  // Lane m < 2 adds head sum m over the cluster's CTAs in rank order (reads issued four CTAs at a
  // time); lane 0 takes lane 1's by one shuffle.
  DF hm{0.0f, 0.0f};
  if (lane < 2) {
    for (uint32_t q0 = 0; q0 < C; q0 += 4) {
      float h4[4], l4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t q = (q0 + u < C && ASV_GUARD(p, q0 + u < uint32_t(kMaxCluster))) ? q0 + u : 0u;
        h4[u] = xchg.head[q][2 * lane];
        l4[u] = xchg.head[q][2 * lane + 1];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (q0 + u < C) hm = df_add(hm, DF{h4[u], l4[u]});
    }
  }
  const DF Hp = hm;
  const DF He{__shfl_sync(0xffffffffu, hm.hi, 1), __shfl_sync(0xffffffffu, hm.lo, 1)};
  if (lane != 0) return;
  {
    float hp = Hp.hi + Hp.lo, he = He.hi + He.lo;
    const float ae = rs.ae_hi + rs.ae_lo, pa = rs.pa_hi + rs.pa_lo;
    if (!cand_on) {  // tail_frac = 0: the head is the whole row
      hp = pa;
      he = ae;
    }
    if (p.tail_mode == 0) {
      rc.head_scale = (he > 0.0f) ? hp / he : 0.0f;
      rc.tail_scale = 1.0f;
    } else {
      // Z = tail p-mass + head phat-mass, phat = exp(zhat/T - max) / ae:
      // tail p / Z, head exp(zhat/T - max) / (ae Z) = exp(..) / (ae tp + he).
      const float tp = pa - hp;
      const float zz = tp + (ae > 0.0f ? he / ae : 0.0f);
      rc.tail_scale = (zz > 0.0f) ? 1.0f / zz : 0.0f;
      const float den = fmaf(ae, tp, he);
      rc.head_scale = (den > 0.0f) ? 1.0f / den : 0.0f;
    }
  }
  uint32_t bits = 0;
  if (!finite) bits |= kBitNonfinite;
  if (pos < G) {
    if (d < 0 || d >= V) {
      bits |= kBitBadDraft;
    } else if (finite) {
      float pd, zhsd, protd;
      rapid_entry(zd, qd, rc, pd, zhsd, protd);
      const Philox4 r4 = philox4x32_10(0u, uint32_t(pos), uint32_t(req), 0u + 4u * p.offset, p.seed_lo, p.seed_hi);
      const float u = uniform_from_word(r4.v[0]);
      if (u * qd < protd) bits |= kBitAccept;
    }
  }
  if (!ASV_GUARD(p, row_ok && req < p.B)) return;
  RapidRecord rec;
  rec.zs_max = rs.M;
  rec.inv_sum = rc.inv_sum;
  rec.zhat_max = rc.zhmax;
  rec.head_scale = rc.head_scale;
  rec.tail_scale = rc.tail_scale;
  rec.bits = bits;
  rec.pad[0] = rec.pad[1] = 0;
  p.records[row] = rec;
  __threadfence();
  const uint32_t ticket = atomicAdd(&p.tickets[req], 1u);
  if (ticket != uint32_t(G)) return;
  // The last row of the request: scan the records, write the outputs and leave the draw job.
  __threadfence();
  const volatile RapidRecord* recs = p.records + size_t(req) * R1;
  uint32_t any = 0;
  for (int i = 0; i < R1; ++i) any |= recs[i].bits;
  const uint32_t status = ((any & kBitNonfinite) ? 1u : 0u) | ((any & kBitBadDraft) ? 2u : 0u);
  int32_t* toks = p.out_tokens + size_t(req) * R1;
  if (status) {
    p.out_accept_len[req] = 0;
    for (int i = 0; i < R1; ++i) toks[i] = -1;
    p.out_req_status[req] = status;
  } else {
    int n = G;
    for (int i = 0; i < G; ++i)
      if (!(recs[i].bits & kBitAccept)) {
        n = i;
        break;
      }
    RapidJob job = {};
    job.zs_max = recs[n].zs_max;
    job.inv_sum = recs[n].inv_sum;
    job.zhat_max = recs[n].zhat_max;
    job.head_scale = recs[n].head_scale;
    job.tail_scale = recs[n].tail_scale;
    job.row = n;
    job.active = 1u;
    p.jobs[req] = job;
    const int32_t* dr = p.draft_ids + size_t(req) * G;
    for (int i = 0; i < R1; ++i) toks[i] = (i < n) ? dr[i] : -1;  // toks[n]: the draw launch
    p.out_accept_len[req] = n;
    p.out_req_status[req] = 0u;
  }
  // The request's records and counter are consumed: clear them (a call leaves the workspace zeroed).
  for (int i = 0; i < R1; ++i) p.records[size_t(req) * R1 + i] = RapidRecord{};
  p.tickets[req] = 0u;
}

// The residual / bonus draw of every request whose verification left a job.  draw_ctas CTAs per
// request (no cluster), each over its slice of the stop row, race all entries once for both
// weightings (exponential race, argmin_k E_k / w_k, E_k = -ln u_k with the same uniform): the
// residual max(p - protected, p - q, 0) (at the bonus position the protected target), and p, which
// decides only if every residual weight is zero.  Pruning keeps the result exact: E_k > 1 - u_k
// (1 - u_k exact, at least 2^-24), so an entry with (1 - u_k) >= w_k K (1 + 2^-20), K the best key
// its warp has seen, has a key (as computed: logf, one division) above K and cannot win; the
// logarithm and the division are skipped for it.  A CTA's winners go into the job's slots with one
// 64-bit atomic max each (key bits above the index, inverted, so the smaller key and then the lower
// index win); the last CTA of the request writes the token and clears the job.
__global__ void __launch_bounds__(kDrawThreads) rapid_draw_kernel(const RapidArgs p) {
  constexpr int VEC = 4;
  constexpr int kWarps = kDrawThreads / 32;
  constexpr float kMargin = 1.0f + 0x1p-20f;
  __shared__ unsigned long long s_best[kWarps][2];
  __shared__ uint32_t s_last;
  // Launched as a programmatic dependent of the verification: wait until it has completed and its
  // writes (jobs, outputs) are visible.  (Without that launch attribute this returns at once.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int parts = p.draw_ctas;
  const int req = blockIdx.x / parts;
  const int part = blockIdx.x - req * parts;
  if (!ASV_GUARD(p, req < p.B && part < parts)) return;
  RapidJob* job = p.jobs + req;
  if (!job->active) return;  // uniform over the CTA
  if (!ASV_GUARD(p, job->row >= 0 && job->row <= p.G)) return;
  const int G = p.G;
  const int R1 = G + 1;
  const int V = p.V;
  const int n = job->row;
  const int v0 = part * p.n_slice;
  const int len = max(0, min(V - v0, p.n_slice));
  const int nvec = (len + VEC - 1) / VEC;
  const uint32_t stream = (n < G) ? 1u : 2u;
  const bool resid = n < G;  // the residual race (else the bonus: the protected target)
  RowConsts dc;
  dc.invT = p.inv_T;
  dc.etaT = p.eta * p.T;
  dc.ML = ref_of(job->zs_max);
  dc.inv_sum = job->inv_sum;
  dc.zhmax = job->zhat_max;
  dc.thr = job->zhat_max + p.ln_tail_frac;
  dc.head_scale = job->head_scale;
  dc.tail_scale = job->tail_scale;
  const size_t nbase = (size_t(req) * R1 + n) * size_t(V) + size_t(v0);
  const float* zr = p.z + nbase;
  const float* qr = p.q + nbase;
  const bool al = p.bulk != 0;
  const uint64_t pol = policy_evict_first();
  const int iters = (nvec + kDrawThreads - 1) / kDrawThreads;  // uniform over the CTA
  // Aligned rows: a ring of kDrawStage vectors per thread in shared memory, filled by cp.async
  // (vector `it` of the thread in slot it mod kDrawStage): the first kDrawStage are requested at
  // once, and each slot is refilled with the vector kDrawStage further on as soon as the arithmetic
  // has consumed it, so the copies overlap the arithmetic.  Each thread reads only its own slots.
  extern __shared__ float4 s_stage[];  // [min(iters, kDrawStage)][z, q][kDrawThreads]
#ifdef ASV_CHECKED
  uint32_t dyn_smem = 0;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_smem));
#endif
  auto stage = [&](int it) {
    const int vi = it * kDrawThreads + tid;
    if (al && it < iters && vi < nvec) {
      const int sl = it % kDrawStage;
      if (ASV_GUARD(p, vi * VEC + VEC <= len && uint32_t(((2 * sl + 1) * kDrawThreads + tid + 1) * 16) <= dyn_smem)) {
        cp_async16(smem_addr(&s_stage[(2 * sl + 0) * kDrawThreads + tid]), zr + vi * VEC, pol);
        cp_async16(smem_addr(&s_stage[(2 * sl + 1) * kDrawThreads + tid]), qr + vi * VEC, pol);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < kDrawStage; ++j) stage(j);
  float key[2] = {INFINITY, INFINITY};  // this thread's best keys and their indices
  int idx[2] = {INT_MAX, INT_MAX};
  float bound[2] = {INFINITY, INFINITY};  // the best keys its warp has seen (pruning bound)
  // Keep the better of (k, i) and (key, idx): the smaller key, on equal keys the lower index.
  auto offer = [&](int s, float k, int i) {
    if (k < key[s] || (k == key[s] && i < idx[s])) {
      key[s] = k;
      idx[s] = i;
    }
  };
  for (int it = 0; it < iters; ++it) {
    cp_async_wait_group<kDrawStage - 1>();  // the copies of vector it have landed
    const int vi = it * kDrawThreads + tid;
    const int sl = it % kDrawStage;
    const int kl = vi * VEC;
    const int kb = v0 + kl;
    // K (1 + 2^-20) for the pruning tests below, formed once per vector (w * that product rounds
    // within the margin's allowance); a zero weight gives 0 or NaN there, and both tests fail on it.
    float bm[2] = {bound[0] * kMargin, bound[1] * kMargin};
    float w[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
    uint32_t rw[4] = {0u, 0u, 0u, 0u};
    // Every vector in range takes its Philox block: the p-weighted race keeps nearly every vector
    // above the pruning threshold, so a test that could skip it would cost more than it saves.
    const bool any = vi < nvec;
    if (any) {
      const float4 z4 = al ? s_stage[(2 * sl + 0) * kDrawThreads + tid] : ld4(zr, kl, len, false, pol, -INFINITY);
      const float4 q4 = al ? s_stage[(2 * sl + 1) * kDrawThreads + tid] : ld4(qr, kl, len, false, pol, 0.0f);
      const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
      const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
      const bool full = kl + VEC <= len;  // (always, on aligned rows)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        // p, zhat/T and the protected target as rapid_entry forms them; the head term (an exp2) only
        // for the few head entries.
        float pk, zhs;
        rapid_p_zhs(zz[e], qq[e], dc, pk, zhs);
        float prot = __fmul_rn(pk, dc.tail_scale);
        if (!(zhs < dc.thr)) prot = __fmul_rn(head_exp(zhs, dc.zhmax), dc.head_scale);
        const bool in = full || kl + e < len;
        w[0][e] = in ? (resid ? fmaxf(fmaxf(pk - prot, pk - qq[e]), 0.0f) : prot) : 0.0f;
        w[1][e] = in ? pk : 0.0f;
      }
      const Philox4 r4 =
          philox4x32_10(uint32_t(kb >> 2), uint32_t(n), uint32_t(req), stream + 4u * p.offset, p.seed_lo, p.seed_hi);
#pragma unroll
      for (int e = 0; e < VEC; ++e) rw[e] = r4.v[e];
    }
    if (it == 0) {
      // Before any key is known every entry would take the logarithm and the division: seed the
      // warp's bounds with the keys of each thread's largest weight of its first vector (a key
      // some entry reaches, so a valid bound), then test the rest against them.
      float ks[2] = {INFINITY, INFINITY};
      if (any) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          float wb = w[s][0];  // (selects over the unrolled entries: no indexed local array)
          uint32_t rb = rw[0];
          int eb = 0;
#pragma unroll
          for (int e = 1; e < VEC; ++e) {
            if (w[s][e] > wb) {
              wb = w[s][e];
              rb = rw[e];
              eb = e;
            }
          }
          if (wb > 0.0f) {
            ks[s] = -logf(uniform_from_word(rb)) / wb;
            offer(s, ks[s], kb + eb);
          }
        }
      }
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        bound[s] = __uint_as_float(__reduce_min_sync(0xffffffffu, __float_as_uint(fminf(bound[s], ks[s]))));
        bm[s] = bound[s] * kMargin;
      }
    }
    if (any) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float u = uniform_from_word(rw[e]);
        const float lo = 1.0f - u;  // exact
        bool cand[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) cand[s] = lo < w[s][e] * bm[s];
        if (cand[0] || cand[1]) {
          const float E = -logf(u);
#pragma unroll
          for (int s = 0; s < 2; ++s)
            if (cand[s]) offer(s, E / w[s][e], kb + e);
        }
      }
    }
    // Share the bound across the warp (non-negative floats order like their bit patterns).
#pragma unroll
    for (int s = 0; s < 2; ++s)
      bound[s] = __uint_as_float(__reduce_min_sync(0xffffffffu, __float_as_uint(fminf(bound[s], key[s]))));
    stage(it + kDrawStage);  // slot sl is consumed: refill it
  }
  cp_async_wait_all();
  unsigned long long best[2];
#pragma unroll
  for (int s = 0; s < 2; ++s)
    best[s] = (idx[s] == INT_MAX) ? 0ull
                                  : ~((static_cast<unsigned long long>(__float_as_uint(key[s])) << 32) | uint32_t(idx[s]));
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best[k], o);
      best[k] = other > best[k] ? other : best[k];
    }
    if (lane == 0) s_best[warp][k] = best[k];
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long b0 = 0ull, b1 = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      b0 = s_best[w][0] > b0 ? s_best[w][0] : b0;
      b1 = s_best[w][1] > b1 ? s_best[w][1] : b1;
    }
    if (b0) atomicMax(&job->slot[0], b0);
    if (b1) atomicMax(&job->slot[1], b1);
    __threadfence();
    s_last = (atomicAdd(&job->ticket, 1u) == uint32_t(parts - 1)) ? 1u : 0u;
    if (s_last) {
      __threadfence();
      const unsigned long long w0 = atomicAdd(&job->slot[0], 0ull);
      const unsigned long long w1 = atomicAdd(&job->slot[1], 0ull);
      const unsigned long long w = w0 ? w0 : w1;
      const int tok = w ? int(uint32_t(~w)) : 0;
      p.out_tokens[size_t(req) * R1 + n] = tok;
      *job = RapidJob{};  // the job is consumed (a call leaves the workspace zeroed)
    }
  }
}

int rapid_threads() { return kRapidThreads; }
int rapid_ctas_per_sm() { return kRapidCtasPerSm; }

namespace {

cudaLaunchConfig_t cluster_config(unsigned ctas, unsigned cluster, size_t smem, cudaLaunchAttribute* attr,
                                  cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(unsigned(kRapidThreads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <typename K>
cudaError_t allow_cluster(K kern, int cluster) {
  if (cluster <= 8) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename K>
cudaError_t prepare(K kern, const LaunchPlan& plan) {
  cudaError_t e = allow_cluster(kern, plan.cluster);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
}

template <bool AL, bool AE>
cudaError_t launch_verify(const RapidArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  auto kern = rapid_kernel<AL, AE>;
  cudaError_t e = prepare(kern, plan);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = cluster_config(unsigned(a.B * (a.G + 1)) * unsigned(plan.cluster),
                                                unsigned(plan.cluster), size_t(plan.smem), attr, s);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool rapid_needs_all_sums(int tail_mode, float ln_tail_frac) { return tail_mode != 0 || !(ln_tail_frac > -INFINITY); }

int rapid_draw_smem_bytes(int n_slice, bool aligned) {
  const int iters = (n_slice / 4 + kDrawThreads - 1) / kDrawThreads;
  return aligned ? std::min(iters, kDrawStage) * 2 * kDrawThreads * 16 : 0;
}

int rapid_draw_ctas_per_sm() { return 4; }  // 48 KB of staging each

int rapid_umax_bytes(bool all_sums, int n_slice) {
  const int iters = (n_slice / 4 + kRapidThreads - 1) / kRapidThreads;
  return all_sums ? 0 : (iters + kGroup - 1) / kGroup * kRapidThreads * 4;
}

int rapid_ring_bytes() { return kRingABytes; }

int rapid_smem_bytes(bool all_sums, int n_slice, bool aligned) {
  return ((aligned && !all_sums) ? kRingABytes : 0) + rapid_umax_bytes(all_sums, n_slice);
}

// Two launches on the stream: the verification (every row), then the draws (draw_ctas CTAs per
// request, with slices of their own: n_slice is recomputed for them).
cudaError_t launch_rapid(const RapidArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  const bool ae = rapid_needs_all_sums(a.tail_mode, a.ln_tail_frac);
  cudaError_t e;
  if (plan.bulk) e = ae ? launch_verify<true, true>(a, plan, s) : launch_verify<true, false>(a, plan, s);
  else e = ae ? launch_verify<false, true>(a, plan, s) : launch_verify<false, false>(a, plan, s);
  if (e != cudaSuccess) return e;
  RapidArgs b = a;
  const int parts = a.draw_ctas;
  b.n_slice = ((a.V + parts - 1) / parts + 3) / 4 * 4;
  const int smem = rapid_draw_smem_bytes(b.n_slice, a.bulk != 0);
  e = cudaFuncSetAttribute(rapid_draw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.B) * unsigned(parts), 1, 1);
  cfg.blockDim = dim3(unsigned(kDrawThreads), 1, 1);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rapid_draw_kernel, b);
}

int rapid_max_active_clusters(const LaunchPlan& plan) {
  auto kern = rapid_kernel<true, false>;
  if (prepare(kern, plan) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = cluster_config(unsigned(plan.cluster), unsigned(plan.cluster), size_t(plan.smem),
                                                attr, nullptr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace asv
