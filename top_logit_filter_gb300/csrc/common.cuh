// Device helpers shared by the filter kernels: dtype traits and order keys,
// PTX wrappers for mbarriers, 1-D bulk (TMA) copies, thread-block-cluster
// barriers and distributed shared memory, and block-wide scans.
//
// Citations "[guide] §N" refer to the web page "CANN ops-nn 算子实战：
// ApplyTopKTopPWithSorted 的 top-k/top-p 采样过滤原理与 aclnn 调用指南" by
// its numbered sections.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "topkp.h"

namespace topkp {

constexpr int kThreads = 512;            // threads per CTA in every filter kernel
constexpr int kWarps = kThreads / 32;
constexpr int kL1Bits = 11;              // first radix digit: 2048 buckets
constexpr int kL1Bins = 1 << kL1Bits;
constexpr float kMassScaleF = 1099511627776.0f;  // 2^40 fixed-point units per unit of probability mass


// ------------------------------------------------------------------ dtypes
// -inf bit patterns of [guide] §6.3 (FLOAT16_NEG_INF, BF16_NEG_INF,
// FLOAT32_NEG_INF).
template <int DT> struct DType;
template <> struct DType<TOPKP_F32> {
  using raw = uint32_t;
  static constexpr int kKeyBits = 32;
  static constexpr raw kNegInf = 0xFF800000u;
  __device__ static __forceinline__ float to_float(raw b) { return __uint_as_float(b); }
  __device__ static __forceinline__ float round_to(float v) { return v; }
};
template <> struct DType<TOPKP_F16> {
  using raw = uint16_t;
  static constexpr int kKeyBits = 16;
  static constexpr raw kNegInf = 0xFC00u;
  __device__ static __forceinline__ float to_float(raw b) { return __half2float(__ushort_as_half(b)); }
  __device__ static __forceinline__ float round_to(float v) { return __half2float(__float2half_rn(v)); }
};
template <> struct DType<TOPKP_BF16> {
  using raw = uint16_t;
  static constexpr int kKeyBits = 16;
  static constexpr raw kNegInf = 0xFF80u;
  __device__ static __forceinline__ float to_float(raw b) { return __uint_as_float(((uint32_t)b) << 16); }
  __device__ static __forceinline__ float round_to(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
};

// Order key: an unsigned integer whose order is the float order of the
// value, with -0 and +0 mapped to the same key (the stable sort of
// [guide] §6.1 treats them as equal).  key = H + |x| for x >= 0 and
// H - |x| for x < 0, H = 2^(bits-1), on the magnitude bits.
template <int DT>
__device__ __forceinline__ uint32_t order_key(typename DType<DT>::raw b) {
  constexpr uint32_t H = 1u << (DType<DT>::kKeyBits - 1);
  const uint32_t u = (uint32_t)b;
  const uint32_t mag = u & (H - 1u);
  return (u & H) ? (H - mag) : (H + mag);
}

// Inverse of order_key (canonical +0 for the zero key).
template <int DT>
__device__ __forceinline__ typename DType<DT>::raw raw_of_key(uint32_t key) {
  constexpr uint32_t H = 1u << (DType<DT>::kKeyBits - 1);
  return (typename DType<DT>::raw)(key >= H ? (key - H) : (H | (H - key)));
}

template <int DT>
__device__ __forceinline__ float value_of_key(uint32_t key) {
  return DType<DT>::to_float(raw_of_key<DT>(key));
}

// Probability mass of one element, relative to the row maximum m, in 2^-40
// fixed point: exp(v - m) = 2^((v - m) log2 e), evaluated as one fused
// multiply-add and the hardware base-2 exponential (relative error about
// 2e-6 for |v - m| <= 40, far inside the 1e-5 tolerance on the cumulative
// probability).  Integer sums are exact and order-independent, which keeps
// the filter deterministic ([guide] §6.3: 默认确定性实现).  The function is
// the only source of masses, so equal values always get equal masses.
struct MassRef {
  float neg_m_log2e;
  __device__ explicit MassRef(float m) : neg_m_log2e(-m * 1.4426950408889634f) {}
};
__device__ __forceinline__ float mass_f32(float v, const MassRef& r) {
  const float t = fminf(fmaf(v, 1.4426950408889634f, r.neg_m_log2e), 0.0f);
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t));
  return e;
}
// mass_f32 of two values at once: one packed (f32x2) fused multiply-add and
// the same clamp and exponential per lane, so each lane equals mass_f32.
__device__ __forceinline__ float2 mass2_f32(float2 v, const MassRef& r) {
  unsigned long long xv, t;
  asm("mov.b64 %0, {%1, %2};" : "=l"(xv) : "f"(v.x), "f"(v.y));
  const unsigned long long s2 = 0x3fb8aa3b3fb8aa3bull;  // 1.4426950408889634f in both lanes
  unsigned long long b2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(b2) : "f"(r.neg_m_log2e));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(xv), "l"(s2), "l"(b2));
  float t0, t1, e0, e1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(t0), "=f"(t1) : "l"(t));
  t0 = fminf(t0, 0.0f);
  t1 = fminf(t1, 0.0f);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
  return make_float2(e0, e1);
}
// a + b lane by lane, one packed (f32x2) add
__device__ __forceinline__ float2 add2_f32(float2 a, float2 b) {
  unsigned long long x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  float r0, r1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(z));
  return make_float2(r0, r1);
}
// A finite float >= 0 below 2^63 rounded to the nearest integer, ties to
// even, with one fp32 add or one shift.  (The library conversion to a
// 64-bit integer runs on the FP64 pipe, which this GPU keeps very narrow.)
__host__ __device__ __forceinline__ uint32_t float_bits(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t b;
  memcpy(&b, &f, sizeof b);
  return b;
#endif
}
__host__ __device__ __forceinline__ unsigned long long f2ull_rn(float f) {
  // Below 2^23, adding 2^23 leaves the integer part in the mantissa, rounded
  // to nearest with ties to even by the fp32 add itself.  From 2^23 on, a
  // float is an integer: its mantissa shifted by the exponent.  (The
  // conversion instruction to 64 bits runs on the narrow FP64 pipe.)
  if (f < 8388608.0f) return (unsigned long long)(float_bits(f + 8388608.0f) - 0x4b000000u);
  const uint32_t b = float_bits(f);
  return (unsigned long long)((b & 0x7fffffu) | 0x800000u) << ((b >> 23) - 150u);
}
__device__ __forceinline__ unsigned long long mass_fixed(float v, const MassRef& r) {
  return f2ull_rn(mass_f32(v, r) * kMassScaleF);
}

// floor(thr * S) for thr in [0, 1], exactly, in integer operations: masked
// iff the cumulative mass is <= thr * S.
__host__ __device__ __forceinline__ unsigned long long mass_target(float thr, unsigned long long S) {
  if (!(thr > 0.0f)) return 0ull;
  if (thr >= 1.0f) return S;
  const uint32_t b = float_bits(thr);
  const uint32_t be = b >> 23;
  const uint32_t m = be ? ((b & 0x7fffffu) | 0x800000u) : (b & 0x7fffffu);
  const int sh = 150 - (int)(be ? be : 1u);     // thr = m * 2^-sh, sh >= 24
  const unsigned long long lo = S * (unsigned long long)m;
#ifdef __CUDA_ARCH__
  const unsigned long long hi = __umul64hi(S, (unsigned long long)m);
#else
  const unsigned long long hi = (unsigned long long)(((unsigned __int128)S * m) >> 64);
#endif
  if (sh >= 128) return 0ull;
  if (sh >= 64) return hi >> (sh - 64);
  return (lo >> sh) | (hi << (64 - sh));
}

// round_D(1 - p): ``1 - p`` on a p tensor of the logits dtype
// ([guide] §2 golden code and §3), clamped to [0, 1].
template <int DT>
__device__ __forceinline__ float top_p_threshold(const void* p, int64_t row) {
  const float pv = DType<DT>::to_float(reinterpret_cast<const typename DType<DT>::raw*>(p)[row]);
  float t = DType<DT>::round_to(1.0f - pv);
  t = fmaxf(t, 0.0f);
  return fminf(t, 1.0f);
}

// ------------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// 1-D bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from shared to global memory, in the current bulk group.
__device__ __forceinline__ void bulk_store_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of an mbarrier, giving up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policies and 16-byte global accesses that carry them.  Rows
// that the write pass reads again are loaded with evict_last; the final
// read and the output stores use evict_first.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_global_hint(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_global_hint(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

// 1-D bulk copy global -> shared with an L2 eviction policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier with release/acquire ordering of shared and global
// memory (all threads of every CTA in the cluster must execute it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of a cluster barrier, for a CTA that must stay resident
// until its peers have finished reading its shared memory.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ uint4 dsmem_ld_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long dsmem_ld_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// ------------------------------------------------------------ block scans
// Exclusive prefix sum over the CTA in thread order; *total gets the sum of
// all threads.  `ws` is kWarps words of shared scratch.  Contains
// __syncthreads(): every thread of the CTA must call it.
__device__ __forceinline__ unsigned long long block_exclusive_scan(unsigned long long v,
                                                                   unsigned long long* total,
                                                                   unsigned long long* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < kWarps ? ws[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) ws[lane] = w;
  }
  __syncthreads();
  const unsigned long long base = warp ? ws[warp - 1] : 0ull;
  *total = ws[kWarps - 1];
  __syncthreads();
  return base + x - v;
}

// Two exclusive prefix sums at once (one set of barriers): *ea / *eb get
// the prefixes of a / b, *ta / *tb their totals.  `ws` is 2 * kWarps words
// of shared scratch.  Contains __syncthreads().
__device__ __forceinline__ void block_exclusive_scan2(unsigned long long a, unsigned long long b,
                                                      unsigned long long* ea, unsigned long long* eb,
                                                      unsigned long long* ta, unsigned long long* tb,
                                                      unsigned long long* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = a, y = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long xu = __shfl_up_sync(0xffffffffu, x, o);
    const unsigned long long yu = __shfl_up_sync(0xffffffffu, y, o);
    if (lane >= o) {
      x += xu;
      y += yu;
    }
  }
  if (lane == 31) {
    ws[warp] = x;
    ws[kWarps + warp] = y;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long u = lane < kWarps ? ws[lane] : 0ull;
    unsigned long long w = lane < kWarps ? ws[kWarps + lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long uu = __shfl_up_sync(0xffffffffu, u, o);
      const unsigned long long wu = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) {
        u += uu;
        w += wu;
      }
    }
    if (lane < kWarps) {
      ws[lane] = u;
      ws[kWarps + lane] = w;
    }
  }
  __syncthreads();
  *ea = (warp ? ws[warp - 1] : 0ull) + x - a;
  *eb = (warp ? ws[kWarps + warp - 1] : 0ull) + y - b;
  *ta = ws[kWarps - 1];
  *tb = ws[2 * kWarps - 1];
  __syncthreads();
}

// Largest 64-bit value over the CTA (every thread gets it).  ws: kWarps
// words of shared scratch.  Contains __syncthreads().
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* ws) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // ws may still be read from an earlier call
  if (lane == 0) ws[warp] = v;
  __syncthreads();
  v = ws[lane < kWarps ? lane : 0];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// An fp32 score as an unsigned key of the same order (for packed maxima).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  const uint32_t fb = __float_as_uint(f);
  return (fb & 0x80000000u) ? ~fb : (fb | 0x80000000u);
}

__device__ __forceinline__ unsigned long long block_sum(unsigned long long v, unsigned long long* ws) {
  unsigned long long t;
  block_exclusive_scan(v, &t, ws);
  return t;
}

}  // namespace topkp
