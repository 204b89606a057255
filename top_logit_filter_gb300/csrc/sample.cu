// topkp_sample: min-p and the exponential-race sample on filtered rows.
//
// The steps are those of the page "aclnnTopKTopPSampleV2" (Formula / minP
// sampling; Formula / Subsequent processing, None and QSample modes), run on
// the filter's output, where every element is a logit or -inf.  With
// e(x) = exp(x - max) over the elements that are not -inf, the softmax
// probabilities are e / sum(e), and both decisions compare ratios of them:
//   - min-p removes x iff prob(x) < minP * prob(max), i.e. iff e(x) < minP
//     (minP >= 1: only the largest element, of equal largest values the one
//     with the largest index, stays);
//   - QSample takes the index of the largest prob(x) / (q + eps), i.e. of
//     the largest e(x) / (q + eps) among the kept elements; the None mode
//     takes the largest element.  Ties go to the largest index.
// So the normaliser is never formed, and both tests run on base-2 logarithms
// of those ratios (one fused multiply-add and one hardware log2 per element).
//
// Launch shape: one 512-thread CTA per row, like the filter.  Pass 1 reads
// the row once from HBM: it finds the largest element, lists the elements
// that are not -inf (with their positions) in shared memory while they fit,
// and copies the row to a separate output.  Pass 2 runs over that list --
// or, for rows with more survivors than the list holds, over the row again
// from L2 -- applies min-p (writing -inf where it removes an element) and
// reads q only at the kept elements.
#include "common.cuh"
#include "internal.h"

namespace topkp {

namespace {

// 16 bytes through the non-coherent path, not allocated in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int DT>
__device__ __forceinline__ typename DType<DT>::raw elem_of(const uint4& q, int j) {
  if (DType<DT>::kKeyBits == 16) {
    const uint32_t w = (j & 4) ? ((j & 2) ? q.w : q.z) : ((j & 2) ? q.y : q.x);
    return (typename DType<DT>::raw)((j & 1) ? (w >> 16) : (w & 0xffffu));
  }
  return (typename DType<DT>::raw)((j & 2) ? ((j & 1) ? q.w : q.z) : ((j & 1) ? q.y : q.x));
}

// The largest element of a 16-byte vector, as raw bits (packed maxima).
template <int DT>
__device__ __forceinline__ typename DType<DT>::raw vec_max_raw(const uint4& q);
template <>
__device__ __forceinline__ uint16_t vec_max_raw<TOPKP_BF16>(const uint4& q) {
  auto v2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); };
  const __nv_bfloat162 m = __hmax2(__hmax2(v2(q.x), v2(q.y)), __hmax2(v2(q.z), v2(q.w)));
  return __bfloat16_as_ushort(__hmax(__low2bfloat16(m), __high2bfloat16(m)));
}
template <>
__device__ __forceinline__ uint16_t vec_max_raw<TOPKP_F16>(const uint4& q) {
  auto v2 = [](uint32_t w) { return *reinterpret_cast<const __half2*>(&w); };
  const __half2 m = __hmax2(__hmax2(v2(q.x), v2(q.y)), __hmax2(v2(q.z), v2(q.w)));
  return __half_as_ushort(__hmax(__low2half(m), __high2half(m)));
}
template <>
__device__ __forceinline__ uint32_t vec_max_raw<TOPKP_F32>(const uint4& q) {
  return __float_as_uint(fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                               fmaxf(__uint_as_float(q.z), __uint_as_float(q.w))));
}

}  // namespace

constexpr int kLoads = 8;       // 16-byte vectors in flight per thread
constexpr int kListCap = 5120;  // elements that are not -inf listed per row (40 KB of shared memory)

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) sample_kernel(const SampleArgs a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  constexpr int VEC = 16 / sizeof(raw);
  __shared__ unsigned long long ws[kWarps];
  __shared__ uint32_t lpos[kListCap];
  __shared__ uint32_t lraw[kListCap];
  __shared__ uint32_t lcount;

  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t row = blockIdx.x;
  const int V = a.V;
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  raw* orow = a.out ? reinterpret_cast<raw*>(a.out) + row * a.ldo : nullptr;
  const float* qr = a.q ? a.q + row * a.ldq : nullptr;
  const bool in_place = orow != nullptr && reinterpret_cast<const void*>(orow) == reinterpret_cast<const void*>(xr);
  const bool copy_out = orow != nullptr && !in_place;

  // row geometry: unaligned head, whole 16-byte vectors, tail
  const uintptr_t xaddr = reinterpret_cast<uintptr_t>(xr);
  const int head = min(V, (int)(((16u - (uint32_t)(xaddr & 15u)) & 15u) / (uint32_t)sizeof(raw)));
  const int nvec = (V - head) / VEC;
  const int tail0 = head + nvec * VEC;
  const uint4* xv = reinterpret_cast<const uint4*>(xr + head);
  const bool vec_out = orow != nullptr && ((reinterpret_cast<uintptr_t>(orow) ^ xaddr) & 15u) == 0;
  const uint32_t kNegKey = order_key<DT>(D::kNegInf);
  const uint32_t NEG2 = VEC == 8 ? ((uint32_t)D::kNegInf | ((uint32_t)D::kNegInf << 16)) : (uint32_t)D::kNegInf;
  const uint4 kNegVec = make_uint4(NEG2, NEG2, NEG2, NEG2);
  const uint64_t pol_first = l2_policy_evict_first();

  if (tid == 0) lcount = 0;
  __syncthreads();

  // ---- pass 1 (from HBM): the largest key and the largest index holding
  // it (packed key << 32 | index, so one maximum orders both); the elements
  // that are not -inf, listed with their positions while they fit; and,
  // with a separate output, the row copied to it ----
  unsigned long long best = 0;
  auto see = [&](raw r, int i) {
    const unsigned long long c = ((unsigned long long)order_key<DT>(r) << 32) | (uint32_t)i;
    best = c > best ? c : best;
  };
  // lists the alive elements (bit j of bits) of the vector at e0; all lanes
  // of the warp call it together
  auto list_vec = [&](const uint4& q, int e0, uint32_t bits) {
    const uint32_t n = __popc(bits);
    if (!__any_sync(0xffffffffu, n != 0)) return;
    uint32_t incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    uint32_t base = 0;
    if (lane == 31) base = atomicAdd(&lcount, incl);
    base = __shfl_sync(0xffffffffu, base, 31) + incl - n;
    while (bits) {
      const int j = __ffs(bits) - 1;
      bits &= bits - 1u;
      const raw r = elem_of<DT>(q, j);
      if (base < (uint32_t)kListCap) {
        lpos[base] = (uint32_t)(e0 + j);
        lraw[base] = (uint32_t)r;
      }
      ++base;
    }
  };
  auto alive_bits = [&](const uint4& q) -> uint32_t {
    uint32_t bits = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) bits |= (elem_of<DT>(q, j) != D::kNegInf ? 1u : 0u) << j;
    return bits;
  };
  // the largest key of a vector (the -inf padding never exceeds a real element)
  auto vec_max_key = [&](const uint4& q) -> uint32_t { return order_key<DT>(vec_max_raw<DT>(q)); };
  for (int i = tid; i < head; i += kThreads) {
    const raw r = xr[i];
    if (copy_out) orow[i] = r;
    if (order_key<DT>(r) > kNegKey) {
      see(r, i);
      const uint32_t s = atomicAdd(&lcount, 1u);
      if (s < (uint32_t)kListCap) { lpos[s] = (uint32_t)i; lraw[s] = (uint32_t)r; }
    }
  }
  for (int i = tail0 + tid; i < V; i += kThreads) {
    const raw r = xr[i];
    if (copy_out) orow[i] = r;
    if (order_key<DT>(r) > kNegKey) {
      see(r, i);
      const uint32_t s = atomicAdd(&lcount, 1u);
      if (s < (uint32_t)kListCap) { lpos[s] = (uint32_t)i; lraw[s] = (uint32_t)r; }
    }
  }
  // kLoads vectors in flight per thread, all issued before any is used;
  // the loop bounds are warp-uniform, so whole warps take each step
  const int nsteps = (nvec + kThreads - 1 - (tid & ~31)) / kThreads;  // same for every lane of a warp
  for (int s0 = 0; s0 < nsteps; s0 += kLoads) {
    uint4 qv[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int v = (s0 + u) * kThreads + tid;
      qv[u] = v < nvec ? ld_stream_v4(xv + v) : kNegVec;
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      if (s0 + u >= nsteps) break;
      const int v = (s0 + u) * kThreads + tid;
      const int e0 = head + v * VEC;
      const uint4& q = qv[u];
      const bool masked = q.x == NEG2 && q.y == NEG2 && q.z == NEG2 && q.w == NEG2;
      if (!masked) {
        const uint32_t vk = vec_max_key(q);
        if (vk >= (uint32_t)(best >> 32)) {
#pragma unroll
          for (int j = 0; j < VEC; ++j) see(elem_of<DT>(q, j), e0 + j);
        }
      }
      // once the list is full (a dense row) nothing more is listed: the
      // second pass then reads the row again (warp-uniform test)
      if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t*>(&lcount), 0) <= (uint32_t)kListCap)
        list_vec(q, e0, masked ? 0u : alive_bits(q));
      if (copy_out && v < nvec) {
        if (vec_out) {
          st_global_hint(orow + e0, q, pol_first);
        } else {
#pragma unroll
          for (int j = 0; j < VEC; ++j) orow[e0 + j] = elem_of<DT>(q, j);
        }
      }
    }
  }
  best = block_max_u64(best, ws);  // (its barriers also publish the list)
  const uint32_t kmax = (uint32_t)(best >> 32);
  const int last = (int)(uint32_t)best;
  const uint32_t nlist = lcount;

  if (kmax <= kNegKey) {
    // no element that is not -inf (outside the contract): the copy stands
    if (a.token && tid == 0) a.token[row] = -1;
    return;
  }

  const float mpv = a.min_p ? a.min_p[row] : 0.0f;
  const bool minp_on = mpv > 0.0f;
  const bool only_last = mpv >= 1.0f;
  if (!qr && !(orow && minp_on)) {
    if (a.token && tid == 0) a.token[row] = last;
    return;
  }

  // ---- pass 2: min-p and the race, over the list (or, when the row held
  // more alive elements than the list, over the row again from L2).  The
  // output already holds the row, so only removed elements are written.
  // Both decisions run on base-2 logarithms of the ratios: with
  // t = (x - max) log2 e, min-p keeps t >= log2(minP) and the race takes the
  // largest t - log2(q + eps), which is the largest e(x) / (q + eps). ----
  if (only_last) {
    // one element stays: the token needs no race
    if (orow) {
      auto drop = [&](raw r, int i) {
        if (r != D::kNegInf && i != last) orow[i] = D::kNegInf;
      };
      if (nlist <= (uint32_t)kListCap) {
        for (uint32_t t = tid; t < nlist; t += kThreads) drop((raw)lraw[t], (int)lpos[t]);
      } else {
        for (int i = tid; i < V; i += kThreads) drop(xr[i], i);
      }
    }
    if (a.token && tid == 0) a.token[row] = last;
    return;
  }
  const float nml = -value_of_key<DT>(kmax) * 1.4426950408889634f;
  const float lmp = minp_on ? log2f(mpv) : -INFINITY;
  const float eps = a.eps;
  // this thread's leader of the race: score t - log2(q + eps) and index
  float bsc = -INFINITY;
  int bidx = -1;
  auto t_of = [&](raw r) -> float { return fmaf(D::to_float(r), 1.4426950408889634f, nml); };
  // the vector at e0 of a dense row with the elements of `drop` set to -inf:
  // one 16-byte store when the output is aligned like the row
  auto write_dropped = [&](int e0, const uint4& xin, uint32_t drop) {
    if (vec_out) {
      uint32_t w[4] = {xin.x, xin.y, xin.z, xin.w};
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        if ((drop >> j) & 1u) {
          if (VEC == 8) {
            const int sh = (j & 1) * 16;
            w[j >> 1] = (w[j >> 1] & ~(0xffffu << sh)) | ((uint32_t)D::kNegInf << sh);
          } else {
            w[j] = (uint32_t)D::kNegInf;
          }
        }
      }
      st_global_hint(orow + e0, make_uint4(w[0], w[1], w[2], w[3]), pol_first);
    } else {
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if ((drop >> j) & 1u) orow[e0 + j] = D::kNegInf;
    }
  };
  // a candidate at an index above every one this thread has seen: it wins
  // ties (equal scores go to the larger index)
  auto race_next = [&](float t, float qv, int i) {
    const float sc = t - __log2f(qv + eps);
    if (sc >= bsc) {
      bsc = sc;
      bidx = i;
    }
  };
  // a candidate in no particular order
  auto race_any = [&](float t, float qv, int i) {
    const float sc = t - __log2f(qv + eps);
    if (sc > bsc || (sc == bsc && i > bidx)) {
      bsc = sc;
      bidx = i;
    }
  };
  if (nlist <= (uint32_t)kListCap) {
    // the listed elements, four per thread at a time so their q loads overlap
    for (uint32_t t0 = tid; t0 < nlist; t0 += 4 * kThreads) {
      int pos[4];
      float t[4], qv[4];
      bool k[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t e = t0 + u * kThreads;
        k[u] = false;
        pos[u] = 0;
        t[u] = 0.0f;
        if (e < nlist) {
          pos[u] = (int)lpos[e];
          t[u] = t_of((raw)lraw[e]);
          k[u] = t[u] >= lmp;
          if (!k[u] && orow) orow[pos[u]] = D::kNegInf;
        }
        qv[u] = (k[u] && qr) ? __ldg(qr + pos[u]) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (k[u] && qr) race_any(t[u], qv[u], pos[u]);
    }
  } else {
    auto visit = [&](raw r, int i) {
      if (r == D::kNegInf) return;
      const float t = t_of(r);
      if (!(t >= lmp)) {
        if (orow) orow[i] = D::kNegInf;
      } else if (qr) {
        race_next(t, __ldg(qr + i), i);
      }
    };
    // in increasing index order per thread: the head, the vectors, the tail
    for (int i = tid; i < head; i += kThreads) visit(xr[i], i);
    // q of a whole vector in 16-byte loads when its row offset allows
    const bool qvec = qr != nullptr && ((reinterpret_cast<uintptr_t>(qr + head) & 15u) == 0);
    // Rows whose kept elements are not rare (at least one in 16 of the
    // listed ones, which are a sample of the row) read q with every vector,
    // both in flight together; the others read q only for vectors that hold
    // a kept element, after the vector has arrived.
    bool dense_q = false;
    if (qvec) {
      unsigned long long kept = 0;
      for (int t0 = tid; t0 < kListCap; t0 += kThreads) kept += t_of((raw)lraw[t0]) >= lmp ? 1u : 0u;
      dense_q = block_sum(kept, ws) * 16 >= (unsigned long long)kListCap;
    }
    if (dense_q) {
      constexpr int UQ = 2;
      for (int v0 = tid; v0 < nvec; v0 += kThreads * UQ) {
        uint4 xq[UQ];
        float4 qq[UQ][VEC / 4];
#pragma unroll
        for (int u = 0; u < UQ; ++u) {
          const int v = v0 + u * kThreads;
          xq[u] = v < nvec ? ld_global_hint(xv + v, pol_first) : kNegVec;
#pragma unroll
          for (int hq = 0; hq < VEC / 4; ++hq)
            qq[u][hq] = v < nvec ? __ldg(reinterpret_cast<const float4*>(qr + head + v * VEC) + hq)
                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < UQ; ++u) {
          const int v = v0 + u * kThreads;
          const int e0 = head + v * VEC;
          uint32_t drop = 0;
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            const raw r = elem_of<DT>(xq[u], j);
            if (r == D::kNegInf) continue;  // (also the padding past the row)
            const float tj = t_of(r);
            if (!(tj >= lmp)) {
              drop |= 1u << j;
            } else {
              const float4 f = qq[u][j >> 2];
              const float qj = (j & 3) == 0 ? f.x : (j & 3) == 1 ? f.y : (j & 3) == 2 ? f.z : f.w;
              race_next(tj, qj, e0 + j);
            }
          }
          if (drop && orow) write_dropped(e0, xq[u], drop);
        }
      }
    }
    constexpr int U2 = 4;
    for (int v0 = dense_q ? nvec : tid; v0 < nvec; v0 += kThreads * U2) {
      uint4 xq[U2];
#pragma unroll
      for (int u = 0; u < U2; ++u) {
        const int v = v0 + u * kThreads;
        xq[u] = v < nvec ? ld_global_hint(xv + v, pol_first) : kNegVec;
      }
#pragma unroll
      for (int u = 0; u < U2; ++u) {
        const int v = v0 + u * kThreads;
        const int e0 = head + v * VEC;
        uint32_t kb = 0, drop = 0;
        float t[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          const raw r = elem_of<DT>(xq[u], j);
          t[j] = t_of(r);
          if (r != D::kNegInf) {                 // never the -inf padding past the row
            if (t[j] >= lmp) kb |= 1u << j;
            else drop |= 1u << j;
          }
        }
        if (drop && orow) write_dropped(e0, xq[u], drop);
        if (qr && kb) {
          float qv[VEC];
          if (qvec) {
#pragma unroll
            for (int h = 0; h < VEC / 4; ++h) {
              const float4 f = __ldg(reinterpret_cast<const float4*>(qr + e0) + h);
              qv[4 * h] = f.x;
              qv[4 * h + 1] = f.y;
              qv[4 * h + 2] = f.z;
              qv[4 * h + 3] = f.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) qv[j] = ((kb >> j) & 1u) ? __ldg(qr + e0 + j) : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < VEC; ++j)
            if ((kb >> j) & 1u) race_next(t[j], qv[j], e0 + j);
        }
      }
    }
    for (int i = tail0 + tid; i < V; i += kThreads) visit(xr[i], i);
  }
  if (a.token) {
    if (qr) {
      // float order as unsigned order, then the larger index among equals
      const uint32_t key = float_order_key(bsc);
      unsigned long long race = bidx < 0 ? 0ull : (((unsigned long long)key << 32) | (uint32_t)bidx);
      race = block_max_u64(race, ws);
      if (tid == 0) a.token[row] = (int)(uint32_t)race;
    } else if (tid == 0) {
      a.token[row] = last;
    }
  }
}

template <int DT>
static cudaError_t launch_sample_dt(const SampleArgs& a, cudaStream_t s) {
  sample_kernel<DT><<<dim3((unsigned)a.B), dim3(kThreads), 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sample(topkp_dtype dt, const SampleArgs& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return launch_sample_dt<TOPKP_F32>(a, s);
    case TOPKP_F16: return launch_sample_dt<TOPKP_F16>(a, s);
    case TOPKP_BF16: return launch_sample_dt<TOPKP_BF16>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace topkp
