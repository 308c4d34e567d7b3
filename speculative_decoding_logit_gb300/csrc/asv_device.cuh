// asv_device.cuh -- device-side building blocks shared by the verification kernels:
// inline-PTX wrappers for L2 cache policies, GPU-scope release/acquire, thread-block
// cluster barriers and distributed shared memory, the special-function unit's exp2/log2,
// bf16 unpacking, packed fp32 arithmetic, compensated sums, Philox and warp reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "asv_internal.h"

namespace asv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2f = 0.6931471805599453f;
constexpr double kLn2 = 0.69314718055994530942;

// Row record bits (workspace).
constexpr uint32_t kBitNonfinite = 1u;
constexpr uint32_t kBitBadDraft = 2u;
constexpr uint32_t kBitTimeout = 4u;
constexpr uint32_t kBitAccept = 8u;

// ------------------------------------------------------------------ checked build
// Built with -DASV_CHECKED, the kernels test every global and shared-memory index they form
// against the buffer it addresses.  A failed test is counted in the call's check log (two words at
// the end of the workspace: the count and the source line of the first failure) and the access is
// skipped -- nothing traps.  In the ordinary build the tests compile to nothing.
#ifdef ASV_CHECKED
__device__ __forceinline__ bool check_index(uint32_t* log, bool ok, int line) {
  if (!ok && log != nullptr) {
    if (atomicAdd(log, 1u) == 0u) atomicExch(log + 1, uint32_t(line));
  }
  return ok;
}
#define ASV_GUARD(args, cond) ::asv::check_index((args).check_log, bool(cond), __LINE__)
#else
#define ASV_GUARD(args, cond) true
#endif

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ L2 cache policies

// L2 policy that marks lines for early eviction (data read for the last time).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy that keeps lines cached in preference to others (data read again soon).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 cache policy); completes for the
// issuing thread at cp_async_wait_all.  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's committed copy groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ GPU-scope synchronisation
// Release/acquire operations at GPU scope for flags that CTAs of one launch exchange through
// global memory.

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// 16-byte load that is served by L2 (not a possibly stale L1 line).
__device__ __forceinline__ float4 ld_cg_f4(const void* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// ------------------------------------------------------------------ clusters / DSMEM

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Cluster barrier where only warp 0 has written data other CTAs read: warp 0 arrives with
// release semantics, the other warps relaxed; everyone waits with acquire semantics.
__device__ __forceinline__ void cluster_sync_w0(int warp) {
  if (warp == 0) cluster_arrive();
  else cluster_arrive_relaxed();
  cluster_wait();
}

// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ double dsmem_ld_f64(uint32_t a) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ int32_t dsmem_ld_s32(uint32_t a) {
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// ------------------------------------------------------------------ special-function unit

// 2^x and log2(x) on the special-function unit (approximate, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ element types

struct bf16_t {
  uint16_t bits;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------------ warp reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index): larger value wins; equal values -> lower index.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_merge(v, i, ov, oi);
  }
}

}  // namespace asv

namespace asv {

__device__ __forceinline__ void dsmem_st_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// ------------------------------------------------------------------ Philox4x32-10
// Counter-based generator of Salmon, Moraes, Dror and Shaw ("Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds; a round multiplies words 0 and 2 by the two round
// multipliers, XORs the high halves with words 1/3 and the key, and the key advances by the
// two Weyl increments before every round but the first.
struct Philox4 {
  uint32_t v[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                 uint32_t k1) {
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round) {
      k0 += kWeylA;
      k1 += kWeylB;
    }
    const uint32_t hiA = __umulhi(kMulA, c0), loA = kMulA * c0;
    const uint32_t hiB = __umulhi(kMulB, c2), loB = kMulB * c2;
    const uint32_t n0 = hiB ^ c1 ^ k0;
    const uint32_t n2 = hiA ^ c3 ^ k1;
    c0 = n0;
    c1 = loB;
    c2 = n2;
    c3 = loA;
  }
  Philox4 r;
  r.v[0] = c0;
  r.v[1] = c1;
  r.v[2] = c2;
  r.v[3] = c3;
  return r;
}

// Uniform in (0, 1) from a 32-bit word: ((w >> 9) + 0.5) * 2^-23, exact in fp32.
__device__ __forceinline__ float uniform_from_word(uint32_t w) {
  return (float(w >> 9) + 0.5f) * 1.1920928955078125e-7f;
}

}  // namespace asv

namespace asv {

// ------------------------------------------------------------------ packed arithmetic
// Two fp32 lanes per instruction (the sm_100 f32x2 forms, round to nearest) and bf16x2 maxima on
// raw bit patterns.  a - b is formed as fma(b, -1, a): one rounding, like a subtraction.

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }

// Lane-wise maximum of two bf16x2 words (exact; a NaN lane yields the other operand).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

}  // namespace asv

namespace asv {

// ------------------------------------------------------------------ compensated fp32 sums
// A value carried as an unevaluated sum hi + lo of two floats (Knuth's TwoSum keeps the
// rounding error of each addition), so partial sums cross warps and CTAs without fp64.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb) + (a.lo + b.lo);
  const float hi = s + e;
  return DF{hi, e - (hi - s)};
}


__device__ __forceinline__ void dsmem_st_f32(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// ln(x) for a positive finite float: x = 2^e * m with m in [0.75, 1.5), ln x = e ln2 + log1p(m - 1);
// m - 1 is exact and |log1p(m - 1)| < 0.41, so the absolute error stays near 6e-8.
__device__ __forceinline__ float ln_split(float x) {
  int e = int((__float_as_uint(x) >> 23) & 0xff) - 127;
  float m = __uint_as_float((__float_as_uint(x) & 0x007fffffu) | 0x3f800000u);  // [1, 2)
  if (m >= 1.5f) {
    m *= 0.5f;
    e += 1;
  }
  return fmaf(float(e), 0.693147182464599609375f, fmaf(float(e), -1.904654323148236e-09f, log1pf(m - 1.0f)));
}

}  // namespace asv
