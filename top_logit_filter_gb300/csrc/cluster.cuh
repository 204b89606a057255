// Collectives over the CTAs of one thread-block cluster that share a row.
//
// A row may be split over a cluster of cs CTAs (cs = 1, 2, 4 or 8), each
// owning a contiguous slice of it.  Every reduction the filter makes over the
// row (its maximum, histograms, mass tables, counts, tie ranks) then becomes
// a reduction over the cluster, through distributed shared memory.
//
// Rules of use, which keep every cluster barrier matched:
//   - every thread of every CTA of the cluster calls each collective at the
//     same point of the program: whether a collective runs at all may only
//     depend on values that are already identical in every CTA (the row's
//     parameters, or results of earlier collectives);
//   - the results are identical in every CTA;
//   - with cs == 1 the collectives return the CTA's own values and never
//     touch a cluster barrier or another CTA's memory;
//   - before it exits, every CTA of a cluster passes cluster_fence_exit(), so
//     none leaves while a peer may still read its shared memory.
#pragma once

#include "common.cuh"

namespace topkp {

struct Clu {
  int cs;         // CTAs per row
  uint32_t rank;  // this CTA's rank in the cluster
};

// Scalar exchange slots.  Two alternating sets: a value written for one
// exchange is never overwritten while a peer may still read it, because each
// exchange ends in a cluster barrier that every CTA must reach before any of
// them can start the exchange after the next.
struct ClSlots {
  unsigned long long v[2][4];
};

enum ClOp { kClSum, kClMax, kClMin, kClOr };

template <int OP>
__device__ __forceinline__ unsigned long long cl_combine(unsigned long long a, unsigned long long b) {
  if (OP == kClSum) return a + b;
  if (OP == kClMax) return a > b ? a : b;
  if (OP == kClMin) return a < b ? a : b;
  return a | b;
}

template <int OP>
__device__ __forceinline__ unsigned long long cl_identity() {
  return OP == kClMin ? ~0ull : 0ull;
}

// Reduces N CTA-uniform values over the cluster with OP, in place.
template <int OP, int N>
__device__ __forceinline__ void cl_reduce(const Clu& c, ClSlots& s, int& phase, unsigned long long (&v)[N]) {
  static_assert(N >= 1 && N <= 4, "at most four values per exchange");
  if (c.cs == 1) return;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) s.v[phase][i] = v[i];
  }
  cluster_sync_all();
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    unsigned long long x = cl_identity<OP>();
    if (lane < c.cs) x = dsmem_ld_u64(dsmem_addr(&s.v[phase][i], (uint32_t)lane));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) x = cl_combine<OP>(x, __shfl_xor_sync(0xffffffffu, x, o));
    v[i] = x;
  }
  phase ^= 1;
}

template <int OP>
__device__ __forceinline__ unsigned long long cl_reduce1(const Clu& c, ClSlots& s, int& phase, unsigned long long v) {
  unsigned long long a[1] = {v};
  cl_reduce<OP, 1>(c, s, phase, a);
  return a[0];
}

// Exclusive prefix over the cluster's ranks of N CTA-uniform counts: ex[i]
// gets the sum over the CTAs of lower rank, tot[i] the sum over all.
template <int N>
__device__ __forceinline__ void cl_prefix(const Clu& c, ClSlots& s, int& phase, const unsigned long long (&v)[N],
                                          unsigned long long (&ex)[N], unsigned long long (&tot)[N]) {
  if (c.cs == 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      ex[i] = 0;
      tot[i] = v[i];
    }
    return;
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) s.v[phase][i] = v[i];
  }
  cluster_sync_all();
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    unsigned long long x = 0;
    if (lane < c.cs) x = dsmem_ld_u64(dsmem_addr(&s.v[phase][i], (uint32_t)lane));
    const unsigned long long below = (uint32_t)lane < c.rank ? x : 0ull;
    unsigned long long e = below, t = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      e += __shfl_xor_sync(0xffffffffu, e, o);
      t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    ex[i] = e;
    tot[i] = t;
  }
  phase ^= 1;
}

// Sums a table of n 32-bit (W = uint32_t) or 64-bit (W = unsigned long long)
// counters, element by element, over the cluster: afterwards every CTA holds
// the cluster's sums in its own table.  The table starts 16-byte aligned and
// n * sizeof(W) is a multiple of 16; n * sizeof(W) / 16 <= NPT * kThreads.
// Two cluster barriers: one before the reads (every CTA's table is
// complete), one after them (no CTA overwrites its table while a peer still
// reads it).
template <typename W, int NPT>
__device__ __forceinline__ void cl_merge(const Clu& c, W* tab, int n) {
  if (c.cs == 1) return;
  const int nv = (int)((size_t)n * sizeof(W) / 16);
  uint4* t4 = reinterpret_cast<uint4*>(tab);
  cluster_sync_all();
  uint4 acc[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int i = j * kThreads + (int)threadIdx.x;
    acc[j] = make_uint4(0, 0, 0, 0);
    if (i < nv) {
      acc[j] = t4[i];
      for (int r = 1; r < c.cs; ++r) {
        const uint32_t peer = (c.rank + (uint32_t)r) % (uint32_t)c.cs;
        const uint4 y = dsmem_ld_v4(dsmem_addr(t4 + i, peer));
        if (sizeof(W) == 4) {
          acc[j].x += y.x;
          acc[j].y += y.y;
          acc[j].z += y.z;
          acc[j].w += y.w;
        } else {
          unsigned long long a0 = ((unsigned long long)acc[j].y << 32) | acc[j].x;
          unsigned long long a1 = ((unsigned long long)acc[j].w << 32) | acc[j].z;
          a0 += ((unsigned long long)y.y << 32) | y.x;
          a1 += ((unsigned long long)y.w << 32) | y.z;
          acc[j] = make_uint4((uint32_t)a0, (uint32_t)(a0 >> 32), (uint32_t)a1, (uint32_t)(a1 >> 32));
        }
      }
    }
  }
  cluster_sync_all();
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int i = j * kThreads + (int)threadIdx.x;
    if (i < nv) t4[i] = acc[j];
  }
  __syncthreads();
}

// A plain cluster barrier (release / acquire): with cl_sum_at, the CTAs
// read a big table through one barrier before the reads (every CTA's table
// is complete) and one after them (no CTA overwrites its table while a peer
// still reads it), without copying it.
__device__ __forceinline__ void cl_sync(const Clu& c) {
  if (c.cs > 1) cluster_sync_all();
}

// Entry i of a table of 32-bit counters, summed over the cluster (between
// two cl_sync calls).
__device__ __forceinline__ uint32_t cl_sum_at(const Clu& c, const uint32_t* local, int i) {
  uint32_t v = local[i];
  for (int r = 1; r < c.cs; ++r) v += dsmem_ld_u32(dsmem_addr(local + i, (c.rank + (uint32_t)r) % (uint32_t)c.cs));
  return v;
}

// Every CTA of the cluster calls this last: once it returns, no peer reads
// this CTA's shared memory any more, so the CTA may exit.
__device__ __forceinline__ void cluster_fence_exit(const Clu& c) {
  if (c.cs > 1) cluster_sync_all();
}

}  // namespace topkp
