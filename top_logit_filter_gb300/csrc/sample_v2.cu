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
constexpr int kV2Cand = 4096;  // candidates of the single-bound top-k (above: the radix select)
constexpr int kV2Bits = 12;    // bucket bits of the bound's histogram (4096 buckets)

// Element j of a 16-byte vector of raw values.
template <int DT>
__device__ __forceinline__ typename DType<DT>::raw v2_elem(const uint4& q, int j) {
  if (DType<DT>::kKeyBits == 16) {
    const uint32_t w = (j & 4) ? ((j & 2) ? q.w : q.z) : ((j & 2) ? q.y : q.x);
    return (typename DType<DT>::raw)((j & 1) ? (w >> 16) : (w & 0xffffu));
  }
  return (typename DType<DT>::raw)((j & 2) ? ((j & 1) ? q.w : q.z) : ((j & 1) ? q.y : q.x));
}

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
  unsigned long long cand[kV2Cand];      // candidates of the single-bound top-k
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

  // ---- single bound: the 16-byte vectors' maxima (and the unaligned head
  // and tail elements) counted in 4096 buckets from the top of the key;
  // the bucket holding the k-th largest of those is a lower bound L on the
  // k-th largest element (k disjoint units reach it).  One more pass lists
  // every element >= L, and a bitonic sort of the list gives the first k in
  // order.  Too few units or too many candidates: the radix select below. ----
  bool fast = false;
  {
    constexpr int VEC = 16 / (int)sizeof(raw);
    uint32_t* hist = &s.whist[0][0];  // 4096 buckets
    for (int i = tid; i < (1 << kV2Bits); i += kThreads) hist[i] = 0;
    if (tid == 0) {
      s.ncol = 0;
      s.sel_digit = -1;
    }
    __syncthreads();
    const uintptr_t xa = reinterpret_cast<uintptr_t>(xr);
    const int head = min(V, (int)(((16u - (uint32_t)(xa & 15u)) & 15u) / (uint32_t)sizeof(raw)));
    const int nvec = (V - head) / VEC;
    const int tail0 = head + nvec * VEC;
    const uint4* xv = reinterpret_cast<const uint4*>(xr + head);
    auto bucket_of = [&](uint32_t key) -> uint32_t { return key >> (KB - kV2Bits); };
    for (int v0 = tid; v0 < nvec; v0 += kThreads * 4) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * kThreads;
        q[u] = v < nvec ? xv[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v0 + u * kThreads < nvec) {
          uint32_t km = 0;
#pragma unroll
          for (int j = 0; j < VEC; ++j) km = max(km, order_key<DT>(v2_elem<DT>(q[u], j)));
          atomicAdd(&hist[bucket_of(km)], 1u);
        }
      }
    }
    for (int i = tid; i < head; i += kThreads) atomicAdd(&hist[bucket_of(order_key<DT>(xr[i]))], 1u);
    for (int i = tail0 + tid; i < V; i += kThreads) atomicAdd(&hist[bucket_of(order_key<DT>(xr[i]))], 1u);
    __syncthreads();
    // thread t holds buckets 8t .. 8t+7; the bucket where the count from the top reaches k
    constexpr int BPT = (1 << kV2Bits) / kThreads;
    unsigned long long c = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) c += hist[BPT * tid + j];
    unsigned long long tot;
    unsigned long long* wsu = reinterpret_cast<unsigned long long*>(s.wsd);
    const unsigned long long pre = block_exclusive_scan(c, &tot, wsu);
    const unsigned long long above = tot - pre - c;  // units in the buckets above this thread's
    if (above < (unsigned long long)k && (unsigned long long)k <= above + c) {
      unsigned long long acc = above;
      for (int j = BPT - 1; j >= 0; --j) {
        acc += hist[BPT * tid + j];
        if (acc >= (unsigned long long)k) {
          s.sel_digit = BPT * tid + j;
          break;
        }
      }
    }
    __syncthreads();
    const int lb = s.sel_digit;
    if (lb >= 0) {
      const uint32_t L = (uint32_t)lb << (KB - kV2Bits);
      auto take = [&](raw r, int i) {
        const uint32_t key = order_key<DT>(r);
        if (key >= L) {
          const uint32_t slot = atomicAdd(&s.ncol, 1u);
          if (slot < (uint32_t)kV2Cand)
            s.cand[slot] = ((unsigned long long)((~key) & KMASK) << 32) | (unsigned long long)(uint32_t)i;
        }
      };
      for (int v0 = tid; v0 < nvec; v0 += kThreads * 4) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * kThreads;
          q[u] = v < nvec ? xv[v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * kThreads;
          if (v < nvec) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) take(v2_elem<DT>(q[u], j), head + v * VEC + j);
          }
        }
      }
      for (int i = tid; i < head; i += kThreads) take(xr[i], i);
      for (int i = tail0 + tid; i < V; i += kThreads) take(xr[i], i);
      __syncthreads();
      const uint32_t n = s.ncol;
      fast = n >= (uint32_t)k && n <= (uint32_t)kV2Cand;
      if (fast) {
        int n2 = 2;
        while (n2 < (int)n) n2 <<= 1;
        for (int j = (int)n + tid; j < n2; j += kThreads) s.cand[j] = ~0ull;  // padding sorts last
        __syncthreads();
        for (int size = 2; size <= n2; size <<= 1) {
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t2 = tid; t2 < n2 / 2; t2 += kThreads) {
              const int lo = 2 * t2 - (t2 & (stride - 1));
              const int hi = lo + stride;
              const bool up = (lo & size) == 0;
              const unsigned long long x0 = s.cand[lo], x1 = s.cand[hi];
              if ((x0 > x1) == up) {
                s.cand[lo] = x1;
                s.cand[hi] = x0;
              }
            }
            __syncthreads();
          }
        }
        for (int j = tid; j < kV2MaxK; j += kThreads) s.list[j] = j < k ? s.cand[j] : ~0ull;
        __syncthreads();
      }
    }
  }

  if (!fast) {
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

  // ---- gather exactly k elements (eight loads per lane in flight, the
  // groups then taken in index order for the tie ranks) ----
  uint32_t seen = 0;
  for (int i0 = wb; i0 < we; i0 += 32 * 8) {
    raw rv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      rv[u] = i < we ? xr[i] : (raw)0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      const uint32_t key = i < we ? order_key<DT>(rv[u]) : 0u;
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
  }  // radix select

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
//
// A whole row is up to 2^20 positions, and this GPU's FP64 pipe runs at a
// sixty-fourth of the FP32 rate, so with logits the per-position work stays
// in fp32 and integers:
//   - S = sum of exp(x - max) as a fixed-point sum in units of 2^-43 (each
//     term rounded to the nearest unit; the sum's error, about 1e-11, is far
//     below the fp32 rounding of S that every probability uses);
//   - the top-p prefix from fixed-point prefix sums of the fp32
//     probabilities in units of 2^-63, found by three levels of search: the
//     warps' sixteenths of the row, the sixteenths of the one that holds the
//     cut, and one warp's walk through the last 1/256;
//   - min-p compares each fp32 probability with the smallest fp32 at or above
//     the fp64 threshold prob[0] * min_p, which decides exactly as the fp64
//     comparison does;
//   - the sample takes the largest fp32 ratio prob / (q + eps) first, and then
//     forms the fp64 ratio only for the positions whose fp32 ratio lies within
//     2^-20 of it: the fp32 ratio is within 2^-22 of the fp64 one, so the
//     fp64 maximum, first on ties, is among them.
// Rows of probabilities (input_is_logits false) take the general stages of
// v2_cut.

// Sum over this warp of a 64-bit value (every lane gets it).
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The fp32 value of a float_order_key.
__device__ __forceinline__ float float_of_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

constexpr float kExpUnit = 8796093022208.0f;        // 2^43: units of exp(x - max) per 1
constexpr float kProbUnit = 9223372036854775808.0f;  // 2^63: units of probability per 1

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) v2_sorted_kernel(const V2Args a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V2Shared& s = *reinterpret_cast<V2Shared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  if (v2_topk_runs(a, row)) return;
  const int V = a.V;
  const raw* sv = reinterpret_cast<const raw*>(a.sv) + row * (int64_t)V;
  const int32_t* si = a.si + row * (int64_t)V;
  const float m = D::to_float(sv[0]);
  const float pv = a.p ? a.p[row] : 2.0f;
  const float mp = a.min_p ? a.min_p[row] : 0.0f;
  const float* qr = a.q ? a.q + row * a.ldq : nullptr;
  unsigned long long* wsu = reinterpret_cast<unsigned long long*>(s.wsd);
  float Sf = 1.0f;
  V2Cut c;
  if (a.input_is_logits) {
    // ---- S, and the probabilities exp(x - m) / S in fp32 ----
    unsigned long long se = 0;
#pragma unroll 8
    for (int j = tid; j < V; j += kThreads) se += f2ull_rn(expf(D::to_float(sv[j]) - m) * kExpUnit);
    Sf = (float)((double)block_sum(se, wsu) * (1.0 / 8796093022208.0));
    auto prob_of = [&](int j) -> float { return expf(D::to_float(sv[j]) - m) / Sf; };
    auto units = [&](int j) -> unsigned long long { return f2ull_rn(prob_of(j) * kProbUnit); };

    // ---- top-p (mass of j and after > fp32(1 - p)): the first position
    // whose exclusive prefix reaches T - thr ends the kept prefix ----
    int n_topp = V;
    if (pv < 1.0f) {
      const float thr = __fsub_rn(1.0f, pv);
      const unsigned long long thr_u = thr >= 1.0f ? ~0ull : f2ull_rn(thr * kProbUnit);
      // level 1: the warps' sixteenths of the row
      const int w1 = ((V + kWarps - 1) / kWarps + 31) & ~31;
      const int a0 = min(V, warp * w1), a1 = min(V, a0 + w1);
      unsigned long long part = 0;
#pragma unroll 8
      for (int j = a0 + lane; j < a1; j += 32) part += units(j);
      part = warp_sum_u64(part);
      unsigned long long T;
      unsigned long long base = block_exclusive_scan(lane == 0 ? part : 0ull, &T, wsu);
      base = __shfl_sync(0xffffffffu, base, 0);
      const unsigned long long target = T > thr_u ? T - thr_u : 0ull;
      // the last range whose start lies below the target holds the first
      // position reaching it (or that position is the range's end)
      int lo = 0, hi = V;
      unsigned long long lo_base = 0;
      if (target > 0) {
        if (lane == 0) s.wsi[warp] = base < target ? 1 : 0;
        __syncthreads();
        int wl = 0;
        for (int w = 0; w < kWarps; ++w) wl = s.wsi[w] ? w : wl;
        __syncthreads();
        lo = min(V, wl * w1);
        hi = min(V, lo + w1);
        // the chosen range's start prefix, from the warp that owns it
        if (warp == wl && lane == 0) wsu[kWarps - 1] = base;
        __syncthreads();
        lo_base = wsu[kWarps - 1];
        __syncthreads();
        // level 2: sixteenths of that range
        const int w2 = ((hi - lo + kWarps - 1) / kWarps + 31) & ~31;
        const int b0 = min(hi, lo + warp * w2), b1 = min(hi, b0 + w2);
        unsigned long long part2 = 0;
#pragma unroll 4
        for (int j = b0 + lane; j < b1; j += 32) part2 += units(j);
        part2 = warp_sum_u64(part2);
        unsigned long long T2;
        unsigned long long base2 = block_exclusive_scan(lane == 0 ? part2 : 0ull, &T2, wsu);
        base2 = lo_base + __shfl_sync(0xffffffffu, base2, 0);
        if (lane == 0) s.wsi[warp] = (base2 < target && b0 < b1) || warp == 0 ? 1 : 0;
        __syncthreads();
        int wl2 = 0;
        for (int w = 0; w < kWarps; ++w) wl2 = s.wsi[w] ? w : wl2;
        __syncthreads();
        // level 3: one warp walks the chosen sixteenth, 32 positions at a time
        if (warp == wl2) {
          unsigned long long acc = base2;  // exclusive prefix at b0
          int found = b1;                  // no position in [b0, b1) reaches the target: the end
          for (int j0 = b0; j0 < b1; j0 += 32) {
            const int j = j0 + lane;
            const unsigned long long u = j < b1 ? units(j) : 0ull;
            unsigned long long incl = u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, j < b1 && acc + incl - u >= target);
            if (hit) {
              found = j0 + __ffs(hit) - 1;
              break;
            }
            acc += __shfl_sync(0xffffffffu, incl, 31);
          }
          if (lane == 0) s.wsi[0] = found;
        }
        __syncthreads();
        n_topp = s.wsi[0];
        __syncthreads();
      } else {
        n_topp = 0;  // no position after the first keeps more than thr
      }
      n_topp = max(1, n_topp);
    }

    // ---- min-p: prob >= prob[0] * min_p (fp64) is prob >= its fp32 ceiling ----
    c.minp_ran = mp > 0.0f;
    int n_kept = n_topp;
    if (c.minp_ran) {
      if (mp >= 1.0f) {
        n_kept = 1;
      } else {
        const float thd32 = __double2float_ru((double)prob_of(0) * (double)mp);
        unsigned long long cnt = 0;
#pragma unroll 8
        for (int j = tid; j < n_topp; j += kThreads) cnt += (prob_of(j) >= thd32 || j == 0) ? 1u : 0u;
        n_kept = (int)block_sum(cnt, wsu);
      }
    }
    c.n_kept = max(1, n_kept);

    // ---- the sample ----
    c.pick = 0;
    if (qr != nullptr) {
      const float eps32 = a.eps;
      uint32_t kmax = 0;
#pragma unroll 4
      for (int j = tid; j < c.n_kept; j += kThreads) kmax = max(kmax, float_order_key(prob_of(j) / (qr[j] + eps32)));
      const float r32max = float_of_order_key((uint32_t)block_max_u64(kmax, wsu));
      const float cut = r32max >= 0.0f ? r32max * (1.0f - 9.5367431640625e-7f) : r32max * (1.0f + 9.5367431640625e-7f);
      double best = -1.0;
      int bpos = -1;
      for (int j = tid; j < c.n_kept; j += kThreads) {
        const float pj = prob_of(j);
        const float qj = qr[j];
        if (pj / (qj + eps32) >= cut) {
          const double r = (double)pj / ((double)qj + (double)eps32);
          if (bpos < 0 || r > best) {
            best = r;
            bpos = j;
          }
        }
      }
      __syncthreads();  // every warp has read the maximum's scratch
      c.pick = block_argmax_first(best, bpos, s.wsd, s.wsi);
      if (c.pick < 0) c.pick = 0;
    }
  } else {
    // probabilities given: the general stages
    c = v2_cut(V, false, pv, mp, qr != nullptr, [&](int j) { return D::to_float(sv[j]); },
               [&](int j) { return qr[j]; }, a.eps, s);
  }
  auto prob_out = [&](int j) -> float {
    const float v = D::to_float(sv[j]);
    return a.input_is_logits ? expf(v - m) / Sf : v;
  };

  if (a.token && tid == 0) a.token[row] = si[c.pick];
  if (a.select) {
    const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
    raw* orow = reinterpret_cast<raw*>(a.select) + row * a.ld_select;
    const raw def = a.input_is_logits ? D::kNegInf : (raw)0;
#pragma unroll 8
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
    for (int j = tid; j < V; j += kThreads) sm[j] = j < c.n_kept ? prob_out(j) : fill;
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
