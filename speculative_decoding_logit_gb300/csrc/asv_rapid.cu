// asv_rapid.cu -- the RAPID verification kernel.
//
// Source: "RAPID: Long-Context Inference with Retrieval-Augmented Speculative Decoding" (paper
// notes): Workflow (rejection sampling against the augmented target); Key design 2 (augmented
// target zhat = z + eta*T*(q - p), p = softmax(z/T), phat = softmax(zhat/T)); Key design 3 (tokens
// whose augmented probability is below 10% of the peak keep the original target probability);
// Key design 4 (at a rejection the token is drawn from norm(max(p - phat, p - q, 0))).
//
// Decomposition as in the AsymSpec kernel: a cluster of C CTAs per row, each CTA staging its slice
// of z and q in shared memory once.  Four sweeps over the staged slice, each followed by a cluster
// exchange through distributed shared memory:
//   1. max of z/T;  2. sum of exp(z/T - max) (and sum of q, for the finiteness check);
//   3. max of zhat/T;  4. head sums: sum of p and of exp(zhat/T - max) over entries at or above
//      the tail boundary zhat/T >= max + ln(tail_frac).
// The protected target is then p on the tail and exp(zhat/T - max) * (head p-mass / head
// exp-mass) on the head, which sums to 1 without a further normalisation pass.  The alternative
// reading of the protection (tail_mode 1: substitute p for phat on the tail, then renormalise
// every entry) also sums p over the tail and exp(zhat/T - max) over every entry in sweep 4; then
// the tail is p / Z and the head phat / Z with Z = (tail p-mass) + (head phat-mass).  CTA 0 of the row
// decides the draft's accept test u*q(d) < protected(d) (u from Philox4x32-10) and files a row
// record.  The last row of a request to finish runs the scan and, in the same cluster, draws the
// emitted token at the stop position with an exponential race over that row (re-read from global
// memory, normally still in L2): argmin_k E_k / w_k, E_k = -ln u_k, with w the residual
// max(p - protected, p - q, 0) or, at the bonus position, the protected target.
#include <climits>

#include "asv_device.cuh"
#include "asv_internal.h"

namespace asv {

struct __align__(16) RapidXchg {
  float zmax;
  float zhmax;
  uint32_t err;
  uint32_t draw_active;  // set remotely by CTA 0 when this cluster draws for its request
  float sum_e[2];   // hi, lo
  float sum_q[2];
  float head_p[2];
  float head_e[2];
  float race_key;
  int32_t race_idx;
  int32_t draw_row;
  float d_zs_max;  // the drawn row's record, broadcast by CTA 0
  float d_inv_sum;
  float d_zhat_max;
  float d_head_scale;
  float d_tail_scale;
  float tail_p[2];  // tail_mode 1: sum of p over the tail
  float all_e[2];   // tail_mode 1: sum of exp(zhat/T - max) over every entry
};

struct RowConsts {
  float invT, etaT, ML, inv_sum, zhmax, thr, head_scale, tail_scale;
};

// Row statistics broadcast by one thread after each cluster exchange.
struct __align__(16) RapidShared {
  float M;
  float inv_sum;
  float zhmax;
  int32_t finite;
};

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// p, zhat/T and the protected target of one entry, recomputed identically everywhere.
__device__ __forceinline__ void rapid_entry(float z, float q, const RowConsts& c, float& p, float& zhs, float& prot) {
  const float zs = z * c.invT;
  p = ex2_approx(fmaf(zs, kLog2e, -c.ML)) * c.inv_sum;
  const float zh = fmaf(c.etaT, q - p, z);
  zhs = zh * c.invT;
  prot = (zhs < c.thr) ? p * c.tail_scale : ex2_approx((zhs - c.zhmax) * kLog2e) * c.head_scale;
}

__global__ void __launch_bounds__(512) rapid_kernel(const RapidArgs p) {
  constexpr int VEC = 4;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ RapidXchg xchg;
  __shared__ RapidShared rs;
  __shared__ float s_wf[32];
  __shared__ int32_t s_wi[32];
  __shared__ float s_w2[32][2];
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
  const int G = p.G;
  const int R1 = G + 1;
  const int req = row / R1;
  const int pos = row - req * R1;
  const int V = p.V;
  const int v0 = int(rank) * p.n_slice;
  const int len = max(0, min(V - v0, p.n_slice));
  const int nvec = (len + VEC - 1) / VEC;
  const size_t row_base = size_t(row) * size_t(V);
  const size_t stage_stride = (size_t(p.n_slice) * sizeof(float) + 127) & ~size_t(127);
  float* zst = reinterpret_cast<float*>(smem_raw);
  float* qst = reinterpret_cast<float*>(smem_raw + stage_stride);
  const int chunk_vec = (nvec + kNumChunks - 1) / kNumChunks;

  // ---------------------------------------------------------------- staging
  if (tid == 0) {
    s_err = 0;
    xchg.draw_active = 0;
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
        const uint32_t bytes = uint32_t(cv1 - cv0) * VEC * 4u;
        const uint32_t bar = smem_addr(&s_bar[c]);
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s(smem_addr(zst + cv0 * VEC), p.z + row_base + v0 + cv0 * VEC, bytes, bar);
        bulk_g2s(smem_addr(qst + cv0 * VEC), p.q + row_base + v0 + cv0 * VEC, bytes, bar);
      }
    }
  } else {
    const int npad = nvec * VEC;
    for (int k = tid; k < npad; k += nthr) {
      zst[k] = (k < len) ? p.z[row_base + v0 + k] : -INFINITY;
      qst[k] = (k < len) ? p.q[row_base + v0 + k] : 0.0f;
    }
    __syncthreads();
  }

  auto block_max = [&](float v) -> float {
    v = warp_max(v);
    if (lane == 0) s_wf[warp] = v;
    __syncthreads();
    float r = -INFINITY;
    if (warp == 0) r = warp_max(lane < nwarps ? s_wf[lane] : -INFINITY);
    __syncthreads();
    return r;  // valid in warp 0
  };
  // fp32 warp sums; the per-warp partials are combined by warp 0 as compensated pairs and
  // written to dst_a / dst_b (hi, lo) in this CTA's exchange slot.
  auto block_sum2 = [&](float a, float b, float* dst_a, float* dst_b) {
    a = warp_sum_f(a);
    b = warp_sum_f(b);
    if (lane == 0) {
      s_w2[warp][0] = a;
      s_w2[warp][1] = b;
    }
    __syncthreads();
    if (warp == 0) {
      const DF ra = warp_sum_df(DF{lane < nwarps ? s_w2[lane][0] : 0.0f, 0.0f});
      const DF rb = warp_sum_df(DF{lane < nwarps ? s_w2[lane][1] : 0.0f, 0.0f});
      if (lane == 0) {
        dst_a[0] = ra.hi;
        dst_a[1] = ra.lo;
        dst_b[0] = rb.hi;
        dst_b[1] = rb.lo;
      }
    }
    __syncthreads();
  };
  // Sum over the cluster of a (hi, lo) slot, in warp 0 (result valid in lane 0).
  auto cluster_sum = [&](const float* slot) -> DF {
    DF d{0.0f, 0.0f};
    if (lane < int(C)) {
      d.hi = dsmem_ld_f32(dsmem_map(smem_addr(&slot[0]), uint32_t(lane)));
      d.lo = dsmem_ld_f32(dsmem_map(smem_addr(&slot[1]), uint32_t(lane)));
    }
    return warp_sum_df(d);
  };

  const float invT = p.inv_T;
  // ---------------------------------------------------------------- sweep 1: max of z/T
  {
    float m = -INFINITY;
    for (int c = 0; c < kNumChunks; ++c) {
      const int cv0 = c * chunk_vec;
      const int cv1 = min(nvec, cv0 + chunk_vec);
      if (cv1 <= cv0) break;
      if (p.bulk && !mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls)) atomicOr(&s_err, 1u);
      for (int vi = cv0 + tid; vi < cv1; vi += nthr) {
        const float4 z4 = reinterpret_cast<const float4*>(zst)[vi];
        m = fmaxf(m, fmaxf(fmaxf(z4.x * invT, z4.y * invT), fmaxf(z4.z * invT, z4.w * invT)));
      }
    }
    const float r = block_max(m);
    if (tid == 0) {
      xchg.zmax = r;
      xchg.err = s_err;
    }
  }
  cluster_sync();  // #1
  if (warp == 0) {
    float v = -INFINITY;
    if (lane < int(C)) v = dsmem_ld_f32(dsmem_map(smem_addr(&xchg.zmax), uint32_t(lane)));
    v = warp_max(v);
    if (lane == 0) rs.M = v;
  }
  __syncthreads();
  const float M = rs.M;
  RowConsts rc;
  rc.invT = invT;
  rc.etaT = p.eta * p.T;
  rc.ML = isfinite(M) ? M * kLog2e : 0.0f;

  // ---------------------------------------------------------------- sweep 2: sum of exp, sum of q
  {
    float e0 = 0.f, e1 = 0.f, q0 = 0.f, q1 = 0.f;
    for (int vi = tid; vi < nvec; vi += nthr) {
      const float4 z4 = reinterpret_cast<const float4*>(zst)[vi];
      const float4 q4 = reinterpret_cast<const float4*>(qst)[vi];
      e0 += ex2_approx(fmaf(z4.x * invT, kLog2e, -rc.ML)) + ex2_approx(fmaf(z4.z * invT, kLog2e, -rc.ML));
      e1 += ex2_approx(fmaf(z4.y * invT, kLog2e, -rc.ML)) + ex2_approx(fmaf(z4.w * invT, kLog2e, -rc.ML));
      q0 += q4.x + q4.z;
      q1 += q4.y + q4.w;
    }
    block_sum2(e0 + e1, q0 + q1, xchg.sum_e, xchg.sum_q);
  }
  cluster_sync();  // #2
  if (warp == 0) {
    const DF Se = cluster_sum(xchg.sum_e);
    const DF Sq = cluster_sum(xchg.sum_q);
    if (lane == 0) {
      const bool fin = isfinite(M) && isfinite(Se.hi) && Se.hi > 0.0f && isfinite(Sq.hi);
      rs.finite = fin ? 1 : 0;
      rs.inv_sum = fin ? 1.0f / (Se.hi + Se.lo) : 0.0f;
    }
  }
  __syncthreads();
  const bool finite = rs.finite != 0;
  rc.inv_sum = rs.inv_sum;
  rc.zhmax = 0.f;
  rc.thr = 0.f;
  rc.head_scale = 0.f;
  rc.tail_scale = 1.0f;

  // ---------------------------------------------------------------- sweep 3: max of zhat/T
  {
    float m = -INFINITY;
    if (finite) {
      for (int vi = tid; vi < nvec; vi += nthr) {
        const float4 z4 = reinterpret_cast<const float4*>(zst)[vi];
        const float4 q4 = reinterpret_cast<const float4*>(qst)[vi];
        const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
        const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pk = ex2_approx(fmaf(zz[e] * invT, kLog2e, -rc.ML)) * rc.inv_sum;
          m = fmaxf(m, fmaf(rc.etaT, qq[e] - pk, zz[e]) * invT);
        }
      }
    }
    const float r = block_max(m);
    if (tid == 0) xchg.zhmax = r;
  }
  cluster_sync();  // #3
  if (warp == 0) {
    float v = -INFINITY;
    if (lane < int(C)) v = dsmem_ld_f32(dsmem_map(smem_addr(&xchg.zhmax), uint32_t(lane)));
    v = warp_max(v);
    if (lane == 0) rs.zhmax = v;
  }
  __syncthreads();
  rc.zhmax = rs.zhmax;
  rc.thr = rs.zhmax + p.ln_tail_frac;

  // ---------------------------------------------------------------- sweep 4: head sums
  {
    float hp0 = 0.f, he0 = 0.f, tp0 = 0.f, ae0 = 0.f;
    if (finite) {
      for (int vi = tid; vi < nvec; vi += nthr) {
        const float4 z4 = reinterpret_cast<const float4*>(zst)[vi];
        const float4 q4 = reinterpret_cast<const float4*>(qst)[vi];
        const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
        const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pk = ex2_approx(fmaf(zz[e] * invT, kLog2e, -rc.ML)) * rc.inv_sum;
          const float zhs = fmaf(rc.etaT, qq[e] - pk, zz[e]) * invT;
          if (p.tail_mode == 0) {
            if (zhs >= rc.thr) {
              hp0 += pk;
              he0 += ex2_approx((zhs - rc.zhmax) * kLog2e);
            }
          } else {
            const float ek = ex2_approx((zhs - rc.zhmax) * kLog2e);
            ae0 += ek;
            if (zhs >= rc.thr) {
              hp0 += pk;
              he0 += ek;
            } else {
              tp0 += pk;
            }
          }
        }
      }
    }
    block_sum2(hp0, he0, xchg.head_p, xchg.head_e);
    if (p.tail_mode != 0) block_sum2(tp0, ae0, xchg.tail_p, xchg.all_e);
    if (tid == 0) xchg.err = s_err;
  }
  cluster_sync();  // #4

  // ---------------------------------------------------------------- row finalisation (CTA 0)
  DF Hp{0.0f, 0.0f}, He{0.0f, 0.0f}, Tp{0.0f, 0.0f}, Ae{0.0f, 0.0f};
  uint32_t err = 0;
  if (rank == 0 && warp == 0) {
    Hp = cluster_sum(xchg.head_p);
    He = cluster_sum(xchg.head_e);
    if (p.tail_mode != 0) {
      Tp = cluster_sum(xchg.tail_p);
      Ae = cluster_sum(xchg.all_e);
    }
    uint32_t e = (lane < int(C)) ? dsmem_ld_u32(dsmem_map(smem_addr(&xchg.err), uint32_t(lane))) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) e |= __shfl_xor_sync(0xffffffffu, e, o);
    err = e;
  }
  if (rank == 0 && tid == 0) {
    const float he = He.hi + He.lo;
    if (p.tail_mode == 0) {
      rc.head_scale = (he > 0.0f) ? (Hp.hi + Hp.lo) / he : 0.0f;
      rc.tail_scale = 1.0f;
    } else {
      // Z = tail p-mass + head phat-mass, phat = exp(zhat/T - max) / Ae:
      // tail p / Z, head exp(zhat/T - max) / (Ae Z) = exp(..) / (Ae Tp + He).
      const float tp = Tp.hi + Tp.lo, ae = Ae.hi + Ae.lo;
      const float z = tp + (ae > 0.0f ? he / ae : 0.0f);
      rc.tail_scale = (z > 0.0f) ? 1.0f / z : 0.0f;
      const float den = fmaf(ae, tp, he);
      rc.head_scale = (den > 0.0f) ? 1.0f / den : 0.0f;
    }
    uint32_t bits = 0;
    if (!finite) bits |= kBitNonfinite;
    if (err) bits |= kBitTimeout;
    if (pos < G) {
      const int d = p.draft_ids[size_t(req) * G + pos];
      if (d < 0 || d >= V) {
        bits |= kBitBadDraft;
      } else if (finite) {
        const uint32_t owner = uint32_t(d / p.n_slice);
        const int off = d - int(owner) * p.n_slice;
        const float zd = dsmem_ld_f32(dsmem_map(smem_addr(zst + off), owner));
        const float qd = dsmem_ld_f32(dsmem_map(smem_addr(qst + off), owner));
        float pd, zhsd, protd;
        rapid_entry(zd, qd, rc, pd, zhsd, protd);
        const Philox4 r4 = philox4x32_10(0u, uint32_t(pos), uint32_t(req), 0u + 4u * p.offset, p.seed_lo, p.seed_hi);
        const float u = uniform_from_word(r4.v[0]);
        if (u * qd < protd) bits |= kBitAccept;
      }
    }
    RapidRecord rec;
    rec.zs_max = M;
    rec.inv_sum = rc.inv_sum;
    rec.zhat_max = rc.zhmax;
    rec.head_scale = rc.head_scale;
    rec.tail_scale = rc.tail_scale;
    rec.bits = bits;
    rec.pad[0] = rec.pad[1] = 0;
    p.records[row] = rec;
    __threadfence();
    const uint32_t ticket = atomicAdd(&p.tickets[req], 1u);
    if (ticket == uint32_t(G)) {
      __threadfence();
      const volatile RapidRecord* recs = p.records + size_t(req) * R1;
      uint32_t any = 0;
      for (int i = 0; i < R1; ++i) any |= recs[i].bits;
      const uint32_t status = ((any & kBitNonfinite) ? 1u : 0u) | ((any & kBitBadDraft) ? 2u : 0u) |
                              ((any & kBitTimeout) ? 4u : 0u);
      if (status) {
        p.out_accept_len[req] = 0;
        for (int i = 0; i < R1; ++i) p.out_tokens[size_t(req) * R1 + i] = -1;
        p.out_req_status[req] = status;
        // The request's records are consumed: clear them (a call leaves the workspace zeroed).
        for (int i = 0; i < R1; ++i) p.records[size_t(req) * R1 + i] = RapidRecord{};
        p.tickets[req] = 0u;
      } else {
        int n = G;
        for (int i = 0; i < G; ++i)
          if (!(recs[i].bits & kBitAccept)) {
            n = i;
            break;
          }
        const float f0 = recs[n].zs_max, f1 = recs[n].inv_sum, f2 = recs[n].zhat_max, f3 = recs[n].head_scale;
        const float f4 = recs[n].tail_scale;
        for (int i = 0; i < R1; ++i) p.records[size_t(req) * R1 + i] = RapidRecord{};
        for (uint32_t q = 0; q < C; ++q) {
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.draw_row), q), uint32_t(n));
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.d_zs_max), q), __float_as_uint(f0));
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.d_inv_sum), q), __float_as_uint(f1));
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.d_zhat_max), q), __float_as_uint(f2));
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.d_head_scale), q), __float_as_uint(f3));
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.d_tail_scale), q), __float_as_uint(f4));
          dsmem_st_u32(dsmem_map(smem_addr(&xchg.draw_active), q), 1u);
        }
      }
    }
  }
  cluster_sync();  // #5: the draw broadcast is visible

  if (xchg.draw_active) {
    // ---------------------------------------------------------------- residual / bonus draw
    const int n = xchg.draw_row;
    const uint32_t stream = (n < G) ? 1u : 2u;
    RowConsts dc;
    dc.invT = invT;
    dc.etaT = p.eta * p.T;
    dc.ML = isfinite(xchg.d_zs_max) ? xchg.d_zs_max * kLog2e : 0.0f;
    dc.inv_sum = xchg.d_inv_sum;
    dc.zhmax = xchg.d_zhat_max;
    dc.thr = xchg.d_zhat_max + p.ln_tail_frac;
    dc.head_scale = xchg.d_head_scale;
    dc.tail_scale = xchg.d_tail_scale;
    const size_t nbase = (size_t(req) * R1 + n) * size_t(V);
    int winner = INT_MAX;
    for (int pass = 0; pass < 2 && winner == INT_MAX; ++pass) {
      // pass 0: residual (or protected target at the bonus position); pass 1: p, if the residual is all zero
      float bk = INFINITY;
      int bidx = INT_MAX;
      for (int vi = tid; vi < nvec; vi += nthr) {
        const int kb = v0 + vi * VEC;
        const Philox4 r4 =
            philox4x32_10(uint32_t(kb >> 2), uint32_t(n), uint32_t(req), stream + 4u * p.offset, p.seed_lo, p.seed_hi);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const int k = kb + e;
          if (k < v0 + len) {
            const float z = p.z[nbase + k];
            const float q = p.q[nbase + k];
            float pk, zhs, prot;
            rapid_entry(z, q, dc, pk, zhs, prot);
            float w;
            if (pass == 1) w = pk;
            else if (n < G) w = fmaxf(fmaxf(pk - prot, pk - q), 0.0f);
            else w = prot;
            if (w > 0.0f) {
              const float key = -logf(uniform_from_word(r4.v[e])) / w;
              if (key < bk) {
                bk = key;
                bidx = k;
              }
            }
          }
        }
      }
      warp_argmin(bk, bidx);
      if (lane == 0) {
        s_wf[warp] = bk;
        s_wi[warp] = bidx;
      }
      __syncthreads();
      if (warp == 0) {
        float v = lane < nwarps ? s_wf[lane] : INFINITY;
        int i = lane < nwarps ? s_wi[lane] : INT_MAX;
        warp_argmin(v, i);
        if (lane == 0) {
          xchg.race_key = v;
          xchg.race_idx = i;
        }
      }
      cluster_sync();  // #6 (per pass)
      float gv = INFINITY;
      int gi = INT_MAX;
      for (uint32_t q = 0; q < C; ++q)
        argmin_merge(gv, gi, dsmem_ld_f32(dsmem_map(smem_addr(&xchg.race_key), q)),
                     dsmem_ld_s32(dsmem_map(smem_addr(&xchg.race_idx), q)));
      winner = gi;
      cluster_sync();  // #7 (per pass): the exchange slots may be rewritten
    }
    if (rank == 0 && tid == 0) {
      int32_t* toks = p.out_tokens + size_t(req) * R1;
      const int32_t* dr = p.draft_ids + size_t(req) * G;
      for (int i = 0; i < R1; ++i) toks[i] = (i < n) ? dr[i] : (i == n ? (winner == INT_MAX ? 0 : winner) : -1);
      p.out_accept_len[req] = n;
      p.out_req_status[req] = 0u;
      p.tickets[req] = 0u;
    }
  }

  if (p.bulk && tid == 0 && s_err) {
    for (int c = 0; c < kNumChunks; ++c) {
      const int cv0 = c * chunk_vec;
      if (min(nvec, cv0 + chunk_vec) <= cv0) break;
      mbar_wait(smem_addr(&s_bar[c]), 0, kWaitPolls);
    }
  }
  cluster_sync();  // #8: shared memory stays alive until remote reads are done
}

int rapid_static_smem_bytes() {
  return int(sizeof(RapidXchg) + sizeof(RapidShared) + 32 * 4 + 32 * 4 + 32 * 2 * 4 + kNumChunks * 8 + 4 + 64);
}

cudaError_t launch_rapid(const RapidArgs& a, const LaunchPlan& plan, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(rapid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
  if (e != cudaSuccess) return e;
  if (plan.cluster > 8) {
    e = cudaFuncSetAttribute(rapid_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const int R = a.B * (a.G + 1);
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
  return cudaLaunchKernelEx(&cfg, rapid_kernel, a);
}

int rapid_max_active_clusters(const LaunchPlan& plan) {
  if (cudaFuncSetAttribute(rapid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem) != cudaSuccess)
    return 0;
  if (plan.cluster > 8 &&
      cudaFuncSetAttribute(rapid_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
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
  if (cudaOccupancyMaxActiveClusters(&n, rapid_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace asv
