// topkp_apply: the fused top-k / top-p filter on raw logits, without a sort.
//
// What it computes is the eight-step formula of [guide] §2 (stable ascending
// sort, k-th-largest threshold, fp32 softmax over the survivors, ascending
// cumsum, mask C <= round_D(1-p) except the last position, scatter back).
// Instead of sorting, every row is reduced to one cut in the stable order:
// the sorted position J whose element has order key T and is the (r0+1)-th
// element equal to T in index order.  Everything at or after J survives:
//   keep(i) = key(i) > T  or  (key(i) == T and rank_among_ties(i) >= r0).
//
// Finding the cut is a radix select over order keys (11-bit first digit,
// then 5 bits for fp16/bf16, or 11 + 10 bits for fp32):
//   * top-k: descend on element counts to the key of the k-th largest;
//   * top-p: descend on probability mass (2^-40 fixed point, over the top-k
//     survivors) to the first key where the ascending cumulative mass exceeds
//     round_D(1-p) * S; the tie count r0 follows from the mass below that key.
//
// Launch shape: one thread-block cluster per row, `csize` CTAs, each owning a
// contiguous slice that is bulk-copied (TMA, cp.async.bulk) into shared memory
// once, so the row is read from HBM once and written once.  Histograms are
// combined across the cluster through distributed shared memory; all CTAs of
// a cluster take the same decisions from the same combined data.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace topkp {

static __device__ unsigned int g_device_error = 0;

struct __align__(16) ApplyHdr {
  uint64_t mbar[kApplyChunks];
  unsigned long long ws[kWarps];      // block-scan scratch
  unsigned long long sel_off;         // select result: mass/count outside the bin
  unsigned long long tie_in[16];      // tie counts pushed by each cluster rank
  int sel_bin;                        // select result: bin, -1 if none
  uint32_t maxkey;                    // local max key (read by peers)
  uint32_t failed;                    // local bounded-wait failure (read by peers)
  uint32_t g_maxkey;                  // cluster-wide max key
  uint32_t g_failed;                  // cluster-wide failure
  int idx_cut;                        // straddle: first kept tie, slice-local index
};
static_assert(sizeof(ApplyHdr) <= kApplyHdrBytes, "header too large");

// Radix digits: level 0 is the 11-bit first digit.
template <int KB> struct Levels;
template <> struct Levels<16> {
  static constexpr int n = 2;
  __device__ static constexpr int shift(int l) { return l == 0 ? 5 : 0; }
  __device__ static constexpr int bits(int l) { return l == 0 ? 11 : 5; }
};
template <> struct Levels<32> {
  static constexpr int n = 3;
  __device__ static constexpr int shift(int l) { return l == 0 ? 21 : (l == 1 ? 10 : 0); }
  __device__ static constexpr int bits(int l) { return l == 0 ? 11 : (l == 1 ? 11 : 10); }
};

__device__ __forceinline__ void csync(int C) {
  if (C > 1) cluster_sync_all();
  else __syncthreads();
}

// Sum of 4 consecutive u32 bins (thread t: bins 4t..4t+3) over the cluster.
__device__ __forceinline__ void combine_u32(const uint32_t* local, int nbins, int C, unsigned long long (&o)[4]) {
  o[0] = o[1] = o[2] = o[3] = 0;
  const int b0 = 4 * threadIdx.x;
  if (b0 >= nbins) return;
  if (C == 1) {
    const uint4 v = *reinterpret_cast<const uint4*>(local + b0);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    return;
  }
  for (int r = 0; r < C; ++r) {
    const uint4 v = dsmem_ld_v4(dsmem_addr(local + b0, r));
    o[0] += v.x; o[1] += v.y; o[2] += v.z; o[3] += v.w;
  }
}

__device__ __forceinline__ void combine_u64(const unsigned long long* local, int nbins, int C,
                                            unsigned long long (&o)[4]) {
  o[0] = o[1] = o[2] = o[3] = 0;
  const int b0 = 4 * threadIdx.x;
  if (b0 >= nbins) return;
  for (int r = 0; r < C; ++r) {
    uint4 v0, v1;
    if (C == 1) {
      v0 = *reinterpret_cast<const uint4*>(local + b0);
      v1 = *reinterpret_cast<const uint4*>(local + b0 + 2);
    } else {
      v0 = dsmem_ld_v4(dsmem_addr(local + b0, r));
      v1 = dsmem_ld_v4(dsmem_addr(local + b0 + 2, r));
    }
    o[0] += ((unsigned long long)v0.y << 32) | v0.x;
    o[1] += ((unsigned long long)v0.w << 32) | v0.z;
    o[2] += ((unsigned long long)v1.y << 32) | v1.x;
    o[3] += ((unsigned long long)v1.w << 32) | v1.z;
  }
}

// Bin holding the rank-th largest element (rank >= 1, counted from the top).
// Sets h.sel_bin and h.sel_off = number of elements in higher bins.
__device__ __forceinline__ void select_desc(const unsigned long long (&b)[4], unsigned long long rank, ApplyHdr& h) {
  if (threadIdx.x == 0) h.sel_bin = -1;
  unsigned long long tot;
  const unsigned long long s = b[0] + b[1] + b[2] + b[3];
  const unsigned long long ex = block_exclusive_scan(s, &tot, h.ws);
  const unsigned long long above = tot - ex - s;
  if (s != 0 && above < rank && rank <= above + s) {
    unsigned long long a2 = above;
#pragma unroll
    for (int j = 3; j >= 0; --j) {
      if (rank <= a2 + b[j]) {
        h.sel_bin = 4 * threadIdx.x + j;
        h.sel_off = a2;
        break;
      }
      a2 += b[j];
    }
  }
  __syncthreads();
}

// First bin whose ascending cumulative mass exceeds target.  Sets h.sel_bin
// (-1 if the total does not exceed target) and h.sel_off = mass below it.
__device__ __forceinline__ void select_asc(const unsigned long long (&b)[4], unsigned long long target, ApplyHdr& h) {
  if (threadIdx.x == 0) h.sel_bin = -1;
  unsigned long long tot;
  const unsigned long long s = b[0] + b[1] + b[2] + b[3];
  const unsigned long long ex = block_exclusive_scan(s, &tot, h.ws);
  if (ex <= target && target < ex + s) {
    unsigned long long below = ex;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (target < below + b[j]) {
        h.sel_bin = 4 * threadIdx.x + j;
        h.sel_off = below;
        break;
      }
      below += b[j];
    }
  }
  __syncthreads();
}

// Calls f(i, raw) for slice elements [e0, e1); e0 must be a multiple of the
// vector width.  Reads shared memory when the slice is staged, else global.
template <typename raw, bool STAGED, typename F>
__device__ __forceinline__ void for_each_elem(const raw* sl, const raw* xs, int e0, int e1, bool vec_ok, F&& f) {
  constexpr int VEC = 16 / sizeof(raw);
  if (STAGED || vec_ok) {
    const raw* src = STAGED ? sl : xs;
    for (int i = e0 + threadIdx.x * VEC; i < e1; i += kThreads * VEC) {
      if (i + VEC <= e1) {
        uint4 v = *reinterpret_cast<const uint4*>(src + i);
        const raw* r = reinterpret_cast<const raw*>(&v);
#pragma unroll
        for (int j = 0; j < VEC; ++j) f(i + j, r[j]);
      } else {
        for (int j = i; j < e1; ++j) f(j, src[j]);
      }
    }
  } else {
    for (int i = e0 + threadIdx.x; i < e1; i += kThreads) f(i, xs[i]);
  }
}

enum TieRule : int { kTiesKept = 0, kTiesMasked = 1, kTiesStraddle = 2 };

template <int DT, bool STAGED>
__global__ void __launch_bounds__(kThreads, 2) apply_kernel(const ApplyArgs a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  using L = Levels<D::kKeyBits>;
  constexpr int VEC = 16 / sizeof(raw);
  constexpr int SH1 = L::shift(0);

  extern __shared__ __align__(128) unsigned char smem[];
  ApplyHdr& h = *reinterpret_cast<ApplyHdr*>(smem);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kApplyHdrBytes);
  unsigned long long* mass = reinterpret_cast<unsigned long long*>(smem + kApplyHdrBytes + 2048 * 4);
  raw* sl = reinterpret_cast<raw*>(smem + kApplyFixedSmem);

  const int tid = threadIdx.x;
  const int C = a.csize;
  const uint32_t crank = C > 1 ? cluster_ctarank() : 0u;
  const int64_t row = blockIdx.x / C;
  const int64_t s0 = (int64_t)crank * a.slice;
  const int n = (int)max((int64_t)0, min((int64_t)a.slice, (int64_t)a.V - s0));
  const raw* xs = reinterpret_cast<const raw*>(a.x) + row * a.ldx + s0;
  raw* os = reinterpret_cast<raw*>(a.out) + row * a.ldo + s0;

  const int kv = a.k ? a.k[row] : 0;
  const bool topk = a.k != nullptr && kv >= 1 && kv <= a.V - 1;
  const bool topp = a.p != nullptr;

  // ---- phase 0: stage the slice (bulk copies in kApplyChunks pieces) ----
  const uint32_t nbytes = (uint32_t)n * (uint32_t)sizeof(raw);
  const uint32_t bulk = (STAGED && a.bulk_in) ? (nbytes & ~15u) : 0u;
  const uint32_t cbytes = ((bulk + kApplyChunks - 1) / kApplyChunks + 15u) & ~15u;
  if (tid == 0) {
    h.maxkey = 0;
    h.failed = 0;
    h.sel_bin = -1;
    for (int c = 0; c < kApplyChunks; ++c) mbar_init(&h.mbar[c], 1);
    fence_mbar_init();
  }
  for (int i = tid; i < kL1Bins; i += kThreads) hist[i] = 0;
  __syncthreads();
  if (STAGED) {
    if (tid == 0) {
      for (int c = 0; c < kApplyChunks; ++c) {
        const uint32_t off = c * cbytes;
        if (off >= bulk) break;
        const uint32_t len = min(cbytes, bulk - off);
        mbar_arrive_expect_tx(&h.mbar[c], len);
        bulk_g2s(reinterpret_cast<unsigned char*>(sl) + off, reinterpret_cast<const unsigned char*>(xs) + off, len,
                 &h.mbar[c]);
      }
    }
    for (int i = bulk / sizeof(raw) + tid; i < n; i += kThreads) sl[i] = xs[i];
    __syncthreads();
  }

  // ---- phase 1: first-digit counts and the maximum, chunk by chunk ----
  uint32_t kmax = 0;
  bool my_fail = false;
  auto count_l1 = [&](int, raw r) {
    const uint32_t key = order_key<DT>(r);
    atomicAdd(&hist[key >> SH1], 1u);
    kmax = max(kmax, key);
  };
  if (STAGED) {
    for (int c = 0; c < kApplyChunks; ++c) {
      const uint32_t off = c * cbytes;
      if (off >= bulk) break;
      const uint32_t len = min(cbytes, bulk - off);
      if (!mbar_wait_bounded(&h.mbar[c], 0, a.timeout_ns)) my_fail = true;
      for_each_elem<raw, true>(sl, xs, off / sizeof(raw), (off + len) / sizeof(raw), true, count_l1);
    }
    // elements after the last 16-byte boundary (loaded by plain loads)
    const int tail0 = bulk / sizeof(raw);
    for (int i = tail0 + tid; i < n; i += kThreads) count_l1(i, sl[i]);
  } else {
    for_each_elem<raw, false>(sl, xs, 0, n, a.bulk_in != 0, count_l1);
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((tid & 31) == 0) atomicMax(&h.maxkey, kmax);
  if (my_fail) {
    atomicOr(&h.failed, 1u);
    atomicOr(&g_device_error, 1u);
  }
  __syncthreads();

  // ---- phase 2: cluster-wide first-digit counts ----
  csync(C);
  unsigned long long cb[4];
  combine_u32(hist, kL1Bins, C, cb);
  if (tid == 0) {
    uint32_t gm = h.maxkey, gf = h.failed;
    for (int r = 0; r < C && C > 1; ++r) {
      gm = max(gm, dsmem_ld_u32(dsmem_addr(&h.maxkey, r)));
      gf |= dsmem_ld_u32(dsmem_addr(&h.failed, r));
    }
    h.g_maxkey = gm;
    h.g_failed = gf;
  }
  csync(C);  // peers are done reading hist / maxkey; hist may be reused
  const uint32_t gmax = h.g_maxkey;

  uint32_t T = 0;               // cut key
  unsigned long long r0 = 0;    // ties of T masked (in index order)
  bool cut_last = false;        // top-p keeps only the last sorted position
  uint32_t kkey = 0;            // key of the k-th largest

  // ---- top-k: descend on counts ([guide] §2 steps 1-3) ----
  if (topk) {
    select_desc(cb, (unsigned long long)kv, h);
    uint32_t prefix = (uint32_t)h.sel_bin;
    unsigned long long rank = (unsigned long long)kv - h.sel_off;
    for (int l = 1; l < L::n; ++l) {
      const int shp = L::shift(l - 1), sh = L::shift(l), nb = 1 << L::bits(l);
      for (int i = tid; i < nb; i += kThreads) hist[i] = 0;
      __syncthreads();
      for_each_elem<raw, STAGED>(sl, xs, 0, n, a.bulk_in != 0, [&](int, raw r) {
        const uint32_t key = order_key<DT>(r);
        if ((key >> shp) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
      });
      __syncthreads();
      csync(C);
      unsigned long long lb[4];
      combine_u32(hist, nb, C, lb);
      csync(C);
      select_desc(lb, rank, h);
      prefix = (prefix << L::bits(l)) | (uint32_t)h.sel_bin;
      rank -= h.sel_off;
    }
    kkey = prefix;
    T = kkey;
  }

  // ---- top-p: descend on probability mass ([guide] §2 steps 4-7) ----
  if (topp) {
    const float m = value_of_key<DT>(gmax);
    const uint32_t minkey = topk ? kkey : 0u;
    const float thr = top_p_threshold<DT>(a.p, row);
    for (int i = tid; i < kL1Bins; i += kThreads) mass[i] = 0;
    __syncthreads();
    for_each_elem<raw, STAGED>(sl, xs, 0, n, a.bulk_in != 0, [&](int, raw r) {
      const uint32_t key = order_key<DT>(r);
      if (key >= minkey) {
        const unsigned long long w = mass_fixed(D::to_float(r), m);
        if (w) atomicAdd(&mass[key >> SH1], w);
      }
    });
    __syncthreads();
    csync(C);
    unsigned long long mb[4];
    combine_u64(mass, kL1Bins, C, mb);
    csync(C);
    const unsigned long long S = block_sum(mb[0] + mb[1] + mb[2] + mb[3], h.ws);
    // masked iff cumulative mass <= thr * S  (integers: <= floor(thr * S))
    const unsigned long long target = (unsigned long long)floor((double)thr * (double)S);
    select_asc(mb, target, h);
    if (h.sel_bin < 0) {
      cut_last = true;
    } else {
      uint32_t prefix = (uint32_t)h.sel_bin;
      unsigned long long rem = target - h.sel_off;
      for (int l = 1; l < L::n; ++l) {
        const int shp = L::shift(l - 1), sh = L::shift(l), nb = 1 << L::bits(l);
        for (int i = tid; i < nb; i += kThreads) mass[i] = 0;
        __syncthreads();
        for_each_elem<raw, STAGED>(sl, xs, 0, n, a.bulk_in != 0, [&](int, raw r) {
          const uint32_t key = order_key<DT>(r);
          if (key >= minkey && (key >> shp) == prefix) {
            const unsigned long long w = mass_fixed(D::to_float(r), m);
            if (w) atomicAdd(&mass[(key >> sh) & (nb - 1)], w);
          }
        });
        __syncthreads();
        csync(C);
        unsigned long long lb[4];
        combine_u64(mass, nb, C, lb);
        csync(C);
        select_asc(lb, rem, h);
        prefix = (prefix << L::bits(l)) | (uint32_t)max(h.sel_bin, 0);
        rem -= h.sel_off;
      }
      T = prefix;
      const unsigned long long u = mass_fixed(value_of_key<DT>(T), m);
      r0 = u ? rem / u : 0ull;
    }
  }
  if (cut_last) T = gmax;

  // ---- ties of T in index order across the cluster ----
  int rule = kTiesKept;
  if (r0 > 0 || cut_last) {
    unsigned long long tc = 0;
    for_each_elem<raw, STAGED>(sl, xs, 0, n, a.bulk_in != 0, [&](int, raw r) { tc += (order_key<DT>(r) == T); });
    tc = block_sum(tc, h.ws);
    if (tid == 0) {
      if (C > 1) {
        for (int r = 0; r < C; ++r) dsmem_st_u64(dsmem_addr(&h.tie_in[crank], r), tc);
      } else {
        h.tie_in[0] = tc;
      }
    }
    csync(C);
    unsigned long long off = 0, tot = 0;
    for (int r = 0; r < C; ++r) {
      if (r < (int)crank) off += h.tie_in[r];
      tot += h.tie_in[r];
    }
    if (cut_last) r0 = tot - 1;
    const unsigned long long lm = r0 > off ? min(r0 - off, tc) : 0ull;  // my masked ties
    if (lm == 0) {
      rule = kTiesKept;
    } else if (lm == tc) {
      rule = kTiesMasked;
    } else {
      // straddle: slice-local index of my lm-th tie (0-based) in index order
      rule = kTiesStraddle;
      const int per = (n + kThreads - 1) / kThreads;
      const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
      unsigned long long cnt = 0;
      for (int i = i0; i < i1; ++i) cnt += (order_key<DT>(STAGED ? sl[i] : xs[i]) == T);
      unsigned long long tot2;
      const unsigned long long ex = block_exclusive_scan(cnt, &tot2, h.ws);
      if (ex <= lm && lm < ex + cnt) {
        unsigned long long seen = ex;
        for (int i = i0; i < i1; ++i) {
          if (order_key<DT>(STAGED ? sl[i] : xs[i]) == T) {
            if (seen == lm) {
              h.idx_cut = i;
              break;
            }
            ++seen;
          }
        }
      }
      __syncthreads();
    }
  }
  const int idx_cut = rule == kTiesStraddle ? h.idx_cut : 0;

  // ---- write: original element or -inf, in original order ([guide] §2 step 8) ----
  if (!h.g_failed) {
    auto keep = [&](int i, raw r) -> raw {
      const uint32_t key = order_key<DT>(r);
      bool kp = key > T;
      if (key == T) kp = (rule == kTiesKept) || (rule == kTiesStraddle && i >= idx_cut);
      return kp ? r : D::kNegInf;
    };
    if (a.vec_out && (STAGED || a.bulk_in)) {
      const raw* src = STAGED ? sl : xs;
      for (int i = tid * VEC; i < n; i += kThreads * VEC) {
        if (i + VEC <= n) {
          uint4 v = *reinterpret_cast<const uint4*>(src + i);
          raw* r = reinterpret_cast<raw*>(&v);
#pragma unroll
          for (int j = 0; j < VEC; ++j) r[j] = keep(i + j, r[j]);
          *reinterpret_cast<uint4*>(os + i) = v;
        } else {
          for (int j = i; j < n; ++j) os[j] = keep(j, src[j]);
        }
      }
    } else {
      for (int i = tid; i < n; i += kThreads) os[i] = keep(i, STAGED ? sl[i] : xs[i]);
    }
  }

  // a copy that timed out may still be in flight: wait (bounded) before the
  // shared memory is released
  if (STAGED && h.g_failed && tid == 0) {
    for (int c = 0; c < kApplyChunks; ++c) {
      if ((uint32_t)c * cbytes >= bulk) break;
      mbar_wait_bounded(&h.mbar[c], 0, a.timeout_ns);
    }
  }
}

template <int DT, bool STAGED>
static cudaError_t launch_one(const ApplyPlan& plan, const ApplyArgs& a, cudaStream_t s) {
  auto kern = apply_kernel<DT, STAGED>;
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

cudaError_t launch_apply(topkp_dtype dt, const ApplyPlan& plan, const ApplyArgs& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return plan.staged ? launch_one<TOPKP_F32, true>(plan, a, s) : launch_one<TOPKP_F32, false>(plan, a, s);
    case TOPKP_F16: return plan.staged ? launch_one<TOPKP_F16, true>(plan, a, s) : launch_one<TOPKP_F16, false>(plan, a, s);
    case TOPKP_BF16: return plan.staged ? launch_one<TOPKP_BF16, true>(plan, a, s) : launch_one<TOPKP_BF16, false>(plan, a, s);
  }
  return cudaErrorInvalidValue;
}

// Reads and clears this translation unit's device error word.
cudaError_t apply_take_device_error(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace topkp
