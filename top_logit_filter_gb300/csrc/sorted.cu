// topkp_apply_sorted: ApplyTopKTopPWithSorted ([guide] §3) -- rows arrive
// sorted ascending with their int32 source positions.
//
// With the order given, the cut is a sorted position J ([guide] §6.3: the
// optimised path locates the top-k boundary in the sorted row, accumulates
// the top-p boundary, then compares on the original logits):
//   * top-k: t = sorted[V-k]; J_k = first position holding t (ties survive);
//   * top-p: over the survivor tail [J_k, V), probability mass in 2^-40 fixed
//     point relative to the row maximum sorted[V-1]; J_p = first position
//     whose ascending cumulative mass exceeds round_D(1-p) * S, else V-1;
//   * everything at sorted positions >= J survives.
// Output.  When the survivors (sorted positions J..V-1) are at most an
// eighth of the row, the row is filled with -inf by coalesced vector stores
// and only the survivors are scattered through sorted_indices: two bytes
// per element plus the few survivors, and no tie handling, since the sorted
// order already is the stable order.  Otherwise, with logits: out[v] =
// logits[v] if logits[v] > T, -inf if below, and the elements tied with
// T = sorted[J] go through sorted_indices when the tie group straddles J
// (the page's CompareSelectOnLogits + ScatterBoundary); without logits:
// out[sorted_indices[j]] = j >= J ? sorted[j] : -inf.
//
// Launch shape: one cluster of `csize` CTAs per row.  Each CTA owns one chunk
// of the output and prefetches its logits chunk into shared memory with a
// bulk copy before the (latency-bound) boundary search, so the HBM read
// overlaps it.  The top-p tail is split over the cluster; partial sums and
// the boundary travel through distributed shared memory.
#include "common.cuh"
#include "internal.h"

namespace topkp {

static __device__ unsigned int g_device_error = 0;

struct __align__(16) SortedHdr {
  uint64_t mbar;
  unsigned long long ws[kWarps];
  unsigned long long part[16];   // per-rank tail mass, pushed by each rank
  int jcut;                      // top-p boundary, pushed by the owning rank
  int found;
};
static_assert(sizeof(SortedHdr) <= kSortedHdrBytes, "header too large");

// First position q <= p such that sv[q..p] are all equal to t (sv ascending,
// sv[p] == t).  Uniform across the CTA.
template <int DT>
__device__ int lower_bound_back(const typename DType<DT>::raw* sv, int p, float t) {
  int hi = p + 1;
  while (true) {
    const int lo = max(0, hi - kThreads);
    const int i = lo + (int)threadIdx.x;
    const bool less = i < hi && DType<DT>::to_float(sv[i]) < t;
    const int cnt = __syncthreads_count(less);
    if (cnt > 0 || lo == 0) return lo + cnt;
    hi = lo;
  }
}

// First position > p holding a value above t, or V.
template <int DT>
__device__ int upper_bound_fwd(const typename DType<DT>::raw* sv, int p, int V, float t) {
  int lo = p;
  while (true) {
    const int hi = min(V, lo + kThreads);
    const int i = lo + (int)threadIdx.x;
    const bool le = i < hi && DType<DT>::to_float(sv[i]) <= t;
    const int cnt = __syncthreads_count(le);
    if (cnt < hi - lo || hi == V) return lo + cnt;
    lo = hi;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) sorted_kernel(const SortedArgs a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  constexpr int VEC = 16 / sizeof(raw);

  extern __shared__ __align__(128) unsigned char smem[];
  SortedHdr& h = *reinterpret_cast<SortedHdr*>(smem);
  raw* stage = reinterpret_cast<raw*>(smem + kSortedHdrBytes);

  const int tid = threadIdx.x;
  const int C = a.csize;
  const uint32_t crank = C > 1 ? cluster_ctarank() : 0u;
  const int64_t row = blockIdx.x / C;
  const int V = a.V;
  const raw* sv = reinterpret_cast<const raw*>(a.sv) + row * (int64_t)V;
  const int32_t* si = a.si + row * (int64_t)V;
  const raw* lg = a.logits ? reinterpret_cast<const raw*>(a.logits) + row * (int64_t)V : nullptr;
  raw* o = reinterpret_cast<raw*>(a.out) + row * (int64_t)V;
  const int c0 = (int)min((int64_t)crank * a.chunk, (int64_t)V);
  const int c1 = (int)min((int64_t)c0 + a.chunk, (int64_t)V);
  const int n = c1 - c0;

  const int kv = a.k ? a.k[row] : 0;
  const bool topk = a.k != nullptr && kv >= 1 && kv <= V - 1;
  const bool topp = a.p != nullptr;

  // ---- prefetch this CTA's logits chunk (overlaps the boundary search),
  // unless top-k already promises few survivors (the logits go unread) ----
  const bool few_expected = topk && kv <= V / 8;
  const bool staged = lg != nullptr && a.aligned && !few_expected;
  const uint32_t bulk = staged ? ((uint32_t)n * (uint32_t)sizeof(raw)) & ~15u : 0u;
  if (tid == 0) {
    mbar_init(&h.mbar, 1);
    fence_mbar_init();
    h.found = 0;
  }
  __syncthreads();
  if (tid == 0 && bulk) {
    mbar_arrive_expect_tx(&h.mbar, bulk);
    bulk_g2s(stage, lg + c0, bulk, &h.mbar);
  }

  // fill this CTA's chunk with -inf: it needs no cut, so when top-k already
  // promises few survivors the stores drain while the cut is searched
  auto fill_chunk = [&]() {
    const uint32_t NEG2 = DType<DT>::kKeyBits == 16 ? ((uint32_t)D::kNegInf * 0x10001u) : (uint32_t)D::kNegInf;
    raw* oc = o + c0;
    const int head = ((uintptr_t)oc & 15u) ? min(n, (int)((16u - ((uintptr_t)oc & 15u)) / sizeof(raw))) : 0;
    for (int i = tid; i < head; i += kThreads) oc[i] = D::kNegInf;
    const int nv = (n - head) / VEC;
    uint4* ov = reinterpret_cast<uint4*>(oc + head);
    for (int i = tid; i < nv; i += kThreads) ov[i] = make_uint4(NEG2, NEG2, NEG2, NEG2);
    for (int i = head + nv * VEC + tid; i < n; i += kThreads) oc[i] = D::kNegInf;
  };
  if (few_expected) fill_chunk();

  // ---- top-k boundary ([guide] §2 steps 1-3) ----
  int jk = 0;
  if (topk) jk = lower_bound_back<DT>(sv, V - kv, D::to_float(sv[V - kv]));

  // ---- top-p boundary ([guide] §2 steps 4-7) ----
  int J = jk;
  if (topp) {
    const MassRef m(D::to_float(sv[V - 1]));
    const float thr = top_p_threshold<DT>(a.p, row);
    const int tail = V - jk;
    const int per_cta = (tail + C - 1) / C;
    const int a0 = jk + min(tail, (int)crank * per_cta);
    const int a1 = jk + min(tail, ((int)crank + 1) * per_cta);
    // Each thread sums a contiguous range of the tail in 16-byte loads: the
    // ranges are whole vectors from the first 16-byte aligned position ia
    // (thread 0 also takes [a0, ia), the last one the partial end).
    const int ia = min(a1, a0 + (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(sv + a0) & 15u)) & 15u) / sizeof(raw)));
    const int nvt = (a1 - ia) / VEC;                       // whole vectors from ia
    const int per_thr = (nvt + kThreads - 1) / kThreads;   // vectors per thread
    const int t0 = tid == 0 ? a0 : min(a1, ia + tid * per_thr * VEC);
    const int t1 = tid == kThreads - 1 ? a1 : min(a1, ia + (tid + 1) * per_thr * VEC);
    // mass of [s, e) (s on a vector boundary when it is >= ia), 4 vectors in flight
    auto range_mass = [&](int s, int e) -> unsigned long long {
      unsigned long long sum = 0;
      int j = s;
      for (; j < e && j < ia; ++j) sum += mass_fixed(D::to_float(sv[j]), m);
      for (; j + 4 * VEC <= e; j += 4 * VEC) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = __ldg(reinterpret_cast<const uint4*>(sv + j) + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const raw* r = reinterpret_cast<const raw*>(&q[u]);
#pragma unroll
          for (int i = 0; i < VEC; ++i) sum += mass_fixed(D::to_float(r[i]), m);
        }
      }
      for (; j + VEC <= e; j += VEC) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(sv + j));
        const raw* r = reinterpret_cast<const raw*>(&q);
#pragma unroll
        for (int i = 0; i < VEC; ++i) sum += mass_fixed(D::to_float(r[i]), m);
      }
      for (; j < e; ++j) sum += mass_fixed(D::to_float(sv[j]), m);
      return sum;
    };
    const unsigned long long mine = range_mass(t0, t1);
    const unsigned long long part = block_sum(mine, h.ws);
    if (tid == 0) {
      if (C > 1) {
        for (int r = 0; r < C; ++r) dsmem_st_u64(dsmem_addr(&h.part[crank], r), part);
      } else {
        h.part[0] = part;
      }
    }
    if (C > 1) cluster_sync_all(); else __syncthreads();
    unsigned long long S = 0, before = 0;
    for (int r = 0; r < C; ++r) {
      if (r < (int)crank) before += h.part[r];
      S += h.part[r];
    }
    const unsigned long long target = mass_target(thr, S);
    // the rank whose part holds the first cumulative mass above target
    if (before <= target && target < before + part) {
      unsigned long long tot;
      const unsigned long long ex = before + block_exclusive_scan(mine, &tot, h.ws);
      if (ex <= target && target < ex + mine) {
        unsigned long long cum = ex;
        for (int j = t0; j < t1; ++j) {
          cum += mass_fixed(D::to_float(sv[j]), m);
          if (cum > target) {
            if (C > 1) {
              for (int r = 0; r < C; ++r) {
                dsmem_st_u32(dsmem_addr(&h.jcut, r), (uint32_t)j);
                dsmem_st_u32(dsmem_addr(&h.found, r), 1u);
              }
            } else {
              h.jcut = j;
              h.found = 1;
            }
            break;
          }
        }
      }
    }
    if (C > 1) cluster_sync_all(); else __syncthreads();
    J = h.found ? h.jcut : V - 1;
  }

  // ---- write ([guide] §2 step 8) ----
  if (V - J <= V / 8) {
    // the chunk filled with -inf (unless done above), then the survivors
    if (bulk && !mbar_wait_bounded(&h.mbar, 0, a.timeout_ns)) atomicOr(&g_device_error, 1u);
    if (!few_expected) fill_chunk();
    if (C > 1) cluster_sync_all(); else __syncthreads();
    for (int j = J + (int)crank * kThreads + tid; j < V; j += C * kThreads) {
      const int v = si[j];
      if (v >= 0 && v < V) o[v] = sv[j];
    }
  } else if (lg != nullptr) {
    const float T = D::to_float(sv[J]);
    const bool any = topk || topp;
    const int lo_t = any ? lower_bound_back<DT>(sv, J, T) : J;
    const bool straddle = lo_t < J;
    bool ok = true;
    if (bulk) ok = mbar_wait_bounded(&h.mbar, 0, a.timeout_ns);
    if (!ok) atomicOr(&g_device_error, 1u);
    auto sel = [&](raw r) -> raw {
      if (!any) return r;
      const float x = D::to_float(r);
      return (x > T || (x == T && !straddle)) ? r : D::kNegInf;
    };
    if (ok) {
      if (staged) {
        for (int i = tid * VEC; i < n; i += kThreads * VEC) {
          if (i + VEC <= n) {
            uint4 v = *reinterpret_cast<const uint4*>(stage + i);
            raw* r = reinterpret_cast<raw*>(&v);
            bool skip = false;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
              if (straddle && D::to_float(r[j]) == T) skip = true;
              r[j] = sel(r[j]);
            }
            if (!skip) {
              *reinterpret_cast<uint4*>(o + c0 + i) = v;
            } else {
              const raw* src = stage + i;
#pragma unroll
              for (int j = 0; j < VEC; ++j)
                if (D::to_float(src[j]) != T) o[c0 + i + j] = r[j];
            }
          } else {
            for (int j = i; j < n; ++j) {
              const raw r = (uint32_t)j * sizeof(raw) < bulk ? stage[j] : lg[c0 + j];
              if (!(straddle && D::to_float(r) == T)) o[c0 + j] = sel(r);
            }
          }
        }
      } else {
        for (int i = tid; i < n; i += kThreads) {
          const raw r = lg[c0 + i];
          if (!(straddle && D::to_float(r) == T)) o[c0 + i] = sel(r);
        }
      }
      // ScatterBoundary: the tie group of T, through sorted_indices
      if (straddle) {
        const int hi_t = upper_bound_fwd<DT>(sv, J, V, T);
        for (int j = lo_t + (int)crank * kThreads + tid; j < hi_t; j += C * kThreads) {
          const int v = si[j];
          if (v >= 0 && v < V) o[v] = j >= J ? lg[v] : D::kNegInf;
        }
      }
    }
  } else {
    // scatter every sorted position of this chunk through sorted_indices
    for (int j = c0 + tid; j < c1; j += kThreads) {
      const int v = si[j];
      if (v >= 0 && v < V) o[v] = j >= J ? sv[j] : D::kNegInf;
    }
  }
}

template <int DT>
static cudaError_t launch_sorted_t(const SortedPlan& plan, const SortedArgs& a, cudaStream_t s) {
  auto kern = sorted_kernel<DT>;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * plan.csize), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = plan.csize > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_sorted(topkp_dtype dt, const SortedPlan& plan, const SortedArgs& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return launch_sorted_t<TOPKP_F32>(plan, a, s);
    case TOPKP_F16: return launch_sorted_t<TOPKP_F16>(plan, a, s);
    case TOPKP_BF16: return launch_sorted_t<TOPKP_BF16>(plan, a, s);
  }
  return cudaErrorInvalidValue;
}

// Reads and clears this translation unit's device error word.
cudaError_t sorted_take_device_error(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace topkp
