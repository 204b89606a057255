// topkp_sample_v2: the TopKTopPSampleV2 semantics of the page
// "aclnnTopKTopPSampleV2" (CANN community edition API reference; cited as
// [V2] by its headings Formula / TopK sampling, TopP sampling, minP
// sampling, Optional output, Subsequent processing, and Constraints).
//
// Per row, on the row ordered from the largest value down (equal values in
// increasing index): top-k keeps the first k positions; the probabilities
// are the softmax over the positions left (or the input values themselves
// when the input is not logits); top-p keeps a prefix by its cumulative
// probability; min-p keeps the positions whose probability reaches
// prob[0] * min_p; the sample picks the largest prob / (q + eps) among the
// kept prefix (q read by sorted position), or position 0 without q.
//
// Two kernels.  Rows whose top-k runs (k <= 1024 by the page's ks_max
// bound) never sort the whole row: a radix select with per-warp digit
// counts finds the k-th largest key T, one pass gathers exactly k elements
// (every key > T and the first ties of T in index order, ranked by the
// per-warp tie counts of the last digit), and a bitonic sort of those k
// entries in shared memory gives their order.  Rows whose top-k is skipped
// are sorted first by topkp_sort's kernel (descending, into the caller's
// workspace) and then walked in that order.  One 512-thread CTA per row;
// only CTA barriers, no waits.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace topkp {

namespace {

constexpr int kV2MaxK = 1024;  // top-k never keeps more ([V2] TopK sampling: ks_max <= 1024)

// Exclusive prefix sum of one double per thread over the CTA, in thread
// order; *total gets the sum.  ws: kWarps doubles of shared scratch.
__device__ __forceinline__ double block_scan_f64(double v, double* total, double* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  double before = 0.0, tot = 0.0;
  for (int w = 0; w < kWarps; ++w) {
    const double s = ws[w];
    before += w < warp ? s : 0.0;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

// Sum over the CTA in a fixed order (deterministic).
__device__ __forceinline__ double block_sum_f64(double v, double* ws) {
  double t;
  block_scan_f64(v, &t, ws);
  return t;
}

// Largest (value, then smallest position) over the CTA: returns the
// position, -1 if no thread holds one.  ws: kWarps doubles and ints.
__device__ __forceinline__ int block_argmax_first(double v, int pos, double* wsv, int* wsp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int op = __shfl_xor_sync(0xffffffffu, pos, o);
    if (op >= 0 && (pos < 0 || ov > v || (ov == v && op < pos))) {
      v = ov;
      pos = op;
    }
  }
  if (lane == 0) {
    wsv[warp] = v;
    wsp[warp] = pos;
  }
  __syncthreads();
  double bv = 0.0;
  int bp = -1;
  for (int w = 0; w < kWarps; ++w) {
    const double ov = wsv[w];
    const int op = wsp[w];
    if (op >= 0 && (bp < 0 || ov > bv || (ov == bv && op < bp))) {
      bv = ov;
      bp = op;
    }
  }
  __syncthreads();
  return bp;
}

struct V2Shared {
  unsigned long long list[kV2MaxK];      // (inverted key << 32 | index), sorted ascending
  float prob[kV2MaxK];
  uint32_t whist[kWarps][256];           // per-warp digit counts
  uint32_t bins[256];
  double wsd[kWarps];
  int wsi[kWarps];
  uint32_t ncol;
  int sel_digit;
  uint32_t sel_above;
};

// The stages after top-k on a prefix of n sorted positions whose fp32
// probabilities prob(j) the caller provides, identical for both kernels:
// the top-p prefix length (form: after a top-k stage, mass before j <= p;
// otherwise mass of j and after > fp32(1 - p)), the min-p prefix length,
// and the sampled position.  Every thread calls it.
struct V2Cut {
  int n_kept;
  int pick;         // sampled sorted position
  bool minp_ran;
};

template <typename ProbOf, typename QOf>
__device__ __forceinline__ V2Cut v2_cut(int n, bool after_topk, float p, float mp, bool has_q, ProbOf prob_of,
                                        QOf q_of, float eps, V2Shared& s) {
  const int tid = threadIdx.x;
  // contiguous per-thread segments of the n positions
  const int per = (n + kThreads - 1) / kThreads;
  const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
  double seg = 0.0;
  for (int j = j0; j < j1; ++j) seg += (double)prob_of(j);
  double total;
  const double before = block_scan_f64(seg, &total, s.wsd);
  // top-p: the kept positions form a prefix; count them
  int n_topp = n;
  if (p < 1.0f) {
    const double pd = (double)p;
    const double thr = (double)__fsub_rn(1.0f, p);
    int cnt = 0;
    double acc = before;
    for (int j = j0; j < j1; ++j) {
      const double pj = (double)prob_of(j);
      const bool keep = after_topk ? (acc <= pd) : (total - acc > thr);
      cnt += (keep || j == 0) ? 1 : 0;
      acc += pj;
    }
    n_topp = (int)block_sum_f64((double)cnt, s.wsd);
  }
  // min-p on the probabilities, which fall along the positions
  V2Cut c;
  c.minp_ran = mp > 0.0f;
  int n_kept = n_topp;
  if (c.minp_ran) {
    if (mp >= 1.0f) {
      n_kept = 1;
    } else {
      const double thd = (double)prob_of(0) * (double)mp;
      int cnt = 0;
      for (int j = j0; j < min(j1, n_topp); ++j) cnt += ((double)prob_of(j) >= thd || j == 0) ? 1 : 0;
      n_kept = (int)block_sum_f64((double)cnt, s.wsd);
    }
  }
  c.n_kept = max(1, n_kept);
  // the sample: the largest prob / (q + eps) over the kept prefix, first on ties
  c.pick = 0;
  if (has_q) {
    double best = -1.0;
    int bpos = -1;
    for (int j = j0; j < min(j1, c.n_kept); ++j) {
      const double r = (double)prob_of(j) / ((double)q_of(j) + (double)eps);
      if (bpos < 0 || r > best) {
        best = r;
        bpos = j;
      }
    }
    c.pick = block_argmax_first(best, bpos, s.wsd, s.wsi);
    if (c.pick < 0) c.pick = 0;
  }
  return c;
}

__device__ __forceinline__ bool v2_topk_runs(const V2Args& a, int64_t row) {
  if (a.k == nullptr) return false;
  const int kv = a.k[row];
  return kv >= 1 && kv <= min(a.V, a.ks_aligned);
}

// ---------------------------------------------------------------- top-k rows
template <int DT>
__global__ void __launch_bounds__(kThreads, 1) v2_topk_kernel(const V2Args a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  constexpr int KB = D::kKeyBits;
  constexpr uint32_t KMASK = (uint32_t)((1ull << KB) - 1ull);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V2Shared& s = *reinterpret_cast<V2Shared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  if (!v2_topk_runs(a, row)) return;
  const int V = a.V;
  const int k = a.k[row];
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  // warp w owns elements [w*per, (w+1)*per), lanes consecutive elements
  const int per = (V + kWarps - 1) / kWarps;
  const int wb = min(V, warp * per), we = min(V, wb + per);

  // ---- radix select of the k-th largest key, 8-bit digits from the top ----
  uint32_t prefix = 0;
  uint32_t rank = (uint32_t)k;  // rank of the wanted key among keys with this prefix, from the top
  for (int pass = 0; pass < KB / 8; ++pass) {
    const int sh = KB - 8 * (pass + 1);
    for (int i = tid; i < kWarps * 256; i += kThreads) (&s.whist[0][0])[i] = 0;
    __syncthreads();
    for (int i0 = wb; i0 < we; i0 += 32 * 8) {
      raw r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * 32 + lane;
        r[u] = i < we ? xr[i] : (raw)0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (i0 + u * 32 + lane < we) {
          const uint32_t key = order_key<DT>(r[u]);
          if (pass == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&s.whist[warp][(key >> sh) & 255u], 1u);
        }
      }
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t c = 0;
      for (int w = 0; w < kWarps; ++w) c += s.whist[w][tid];
      s.bins[tid] = c;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t above = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (above + s.bins[d] >= rank) break;
        above += s.bins[d];
      }
      s.sel_digit = d;
      s.sel_above = above;
    }
    __syncthreads();
    prefix = (prefix << 8) | (uint32_t)s.sel_digit;
    rank -= s.sel_above;
    __syncthreads();
  }
  const uint32_t T = prefix;
  // elements above T: k - rank; ties of T to keep: rank, the first in index order
  const uint32_t need_ties = rank;
  // ties of T in the warps before this one (the last pass counted them per warp)
  uint32_t tie_off = 0;
  for (int w = 0; w < warp; ++w) tie_off += s.whist[w][T & 255u];
  if (tid == 0) s.ncol = 0;
  for (int j = tid; j < kV2MaxK; j += kThreads) s.list[j] = ~0ull;  // padding sorts last
  __syncthreads();

  // ---- gather exactly k elements ----
  uint32_t seen = 0;
  for (int base = wb; base < we; base += 32) {
    const int i = base + lane;
    uint32_t key = 0;
    if (i < we) key = order_key<DT>(xr[i]);
    const bool gt = i < we && key > T;
    const bool eq = i < we && key == T;
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const uint32_t r = tie_off + seen + __popc(be & ((1u << lane) - 1u));
    seen += __popc(be);
    if (gt || (eq && r < need_ties)) {
      const uint32_t slot = atomicAdd(&s.ncol, 1u);
      if (slot < (uint32_t)kV2MaxK)
        s.list[slot] = ((unsigned long long)((~key) & KMASK) << 32) | (unsigned long long)(uint32_t)i;
    }
  }
  __syncthreads();

  // ---- bitonic sort of the 1024 entries, ascending ----
  for (int size = 2; size <= kV2MaxK; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < kV2MaxK / 2; t += kThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x0 = s.list[lo], x1 = s.list[hi];
        if ((x0 > x1) == up) {
          s.list[lo] = x1;
          s.list[hi] = x0;
        }
      }
      __syncthreads();
    }
  }

  // ---- probabilities of the k positions ----
  auto value_at = [&](int j) -> float {
    const uint32_t key = (~(uint32_t)(s.list[j] >> 32)) & KMASK;
    return value_of_key<DT>(key);
  };
  const float m = value_at(0);
  double part = 0.0;
  for (int j = tid; j < k; j += kThreads) {
    const float v = value_at(j);
    const float e = a.input_is_logits ? expf(v - m) : v;
    s.prob[j] = e;
    part += (double)e;
  }
  const double S = block_sum_f64(part, s.wsd);
  if (a.input_is_logits) {
    const float Sf = (float)S;
    for (int j = tid; j < k; j += kThreads) s.prob[j] = s.prob[j] / Sf;
  }
  __syncthreads();

  const float pv = a.p ? a.p[row] : 2.0f;
  const float mp = a.min_p ? a.min_p[row] : 0.0f;
  const float* qr = a.q ? a.q + row * a.ldq : nullptr;
  const V2Cut c = v2_cut(
      k, true, pv, mp, qr != nullptr, [&](int j) { return s.prob[j]; }, [&](int j) { return qr[j]; }, a.eps, s);
  auto index_at = [&](int j) -> int32_t { return (int32_t)(uint32_t)(s.list[j] & 0xffffffffull); };

  // ---- outputs ----
  if (a.token && tid == 0) a.token[row] = index_at(c.pick);
  if (a.select) {
    raw* orow = reinterpret_cast<raw*>(a.select) + row * a.ld_select;
    const raw def = a.input_is_logits ? D::kNegInf : (raw)0;
    for (int i = tid; i < V; i += kThreads) orow[i] = def;
    __syncthreads();
    for (int j = tid; j < c.n_kept; j += kThreads) {
      const int32_t ix = index_at(j);
      orow[ix] = xr[ix];
    }
  }
  if (a.logits_idx) {
    int32_t* li = a.logits_idx + row * (int64_t)V;
    for (int j = tid; j < V; j += kThreads) li[j] = j < k ? index_at(j) : -1;
  }
  if (a.sort_masked) {
    float* sm = a.sort_masked + row * (int64_t)V;
    const float fill = (c.minp_ran || !a.input_is_logits) ? 0.0f : -INFINITY;
    for (int j = tid; j < V; j += kThreads) sm[j] = j < c.n_kept ? s.prob[j] : fill;
  }
}

// ------------------------------------------------- rows with top-k skipped
// The row is already sorted (descending) in the workspace: sv / si.
template <int DT>
__global__ void __launch_bounds__(kThreads, 1) v2_sorted_kernel(const V2Args a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V2Shared& s = *reinterpret_cast<V2Shared*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  if (v2_topk_runs(a, row)) return;
  const int V = a.V;
  const raw* sv = reinterpret_cast<const raw*>(a.sv) + row * (int64_t)V;
  const int32_t* si = a.si + row * (int64_t)V;
  const float m = D::to_float(sv[0]);
  // probabilities: exp(x - m) / S, S summed in fp64 from fp32 terms
  double part = 0.0;
  for (int j = tid; j < V; j += kThreads) {
    const float v = D::to_float(sv[j]);
    part += (double)(a.input_is_logits ? expf(v - m) : v);
  }
  const double S = block_sum_f64(part, s.wsd);
  const float Sf = (float)S;
  auto prob_of = [&](int j) -> float {
    const float v = D::to_float(sv[j]);
    return a.input_is_logits ? expf(v - m) / Sf : v;
  };
  const float pv = a.p ? a.p[row] : 2.0f;
  const float mp = a.min_p ? a.min_p[row] : 0.0f;
  const float* qr = a.q ? a.q + row * a.ldq : nullptr;
  const V2Cut c = v2_cut(V, false, pv, mp, qr != nullptr, prob_of, [&](int j) { return qr[j]; }, a.eps, s);

  if (a.token && tid == 0) a.token[row] = si[c.pick];
  if (a.select) {
    const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
    raw* orow = reinterpret_cast<raw*>(a.select) + row * a.ld_select;
    const raw def = a.input_is_logits ? D::kNegInf : (raw)0;
    for (int i = tid; i < V; i += kThreads) orow[i] = def;
    __syncthreads();
    for (int j = tid; j < c.n_kept; j += kThreads) {
      const int32_t ix = si[j];
      if (ix >= 0 && ix < V) orow[ix] = xr[ix];
    }
  }
  if (a.logits_idx) {
    int32_t* li = a.logits_idx + row * (int64_t)V;
    for (int j = tid; j < V; j += kThreads) li[j] = si[j];
  }
  if (a.sort_masked) {
    float* sm = a.sort_masked + row * (int64_t)V;
    const float fill = (c.minp_ran || !a.input_is_logits) ? 0.0f : -INFINITY;
    for (int j = tid; j < V; j += kThreads) sm[j] = j < c.n_kept ? prob_of(j) : fill;
  }
}

template <int DT>
cudaError_t launch_v2_dt(const V2Args& a, cudaStream_t st) {
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(v2_topk_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(V2Shared));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(v2_sorted_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(V2Shared));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  v2_topk_kernel<DT><<<dim3((unsigned)a.B), dim3(kThreads), sizeof(V2Shared), st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.sv == nullptr) return e;
  v2_sorted_kernel<DT><<<dim3((unsigned)a.B), dim3(kThreads), sizeof(V2Shared), st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_v2(topkp_dtype dt, const V2Args& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return launch_v2_dt<TOPKP_F32>(a, s);
    case TOPKP_F16: return launch_v2_dt<TOPKP_F16>(a, s);
    case TOPKP_BF16: return launch_v2_dt<TOPKP_BF16>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace topkp
