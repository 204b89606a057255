// topkp_apply: the fused top-k / top-p filter on raw logits, without a sort.
//
// What it computes is the eight-step formula of [guide] §2 (stable ascending
// sort, k-th-largest threshold, fp32 softmax over the survivors, ascending
// cumsum, mask C <= round_D(1-p) except the last position, scatter back).
// Instead of sorting, every row is reduced to one cut in the stable order:
// the element with order key T that is the (r0+1)-th element equal to T in
// index order.  Everything at or after it survives:
//   keep(i) = key(i) > T  or  (key(i) == T and rank_among_ties(i) >= r0).
//
// Launch shape: one 512-thread CTA per row, two CTAs per SM, so a decode
// batch of a few hundred rows runs as a single wave and every row's latency
// overlaps every other row's.  The row streams through a ring of four large
// shared-memory slots, each filled by one bulk copy (TMA, cp.async.bulk; few
// large copies keep the per-copy cost negligible), and warp w handles the
// w-th sixteenth of every slot.  The first pass reads HBM; the later passes
// read the same bytes again from L2, so HBM sees each logit read once and
// each output written once.
//
// Rows with top-k take the candidate path:
//   1. one packed max per 16-byte vector and a histogram of those vector
//      maxima over a 12-bit first digit;
//   2. the k-th largest vector maximum lower-bounds the row's k-th largest
//      element (k distinct elements reach it); its bucket floor L decides
//      candidacy.  A second pass tests every vector with one packed ">= L"
//      compare and each warp appends the few elements >= L to its own list;
//   3. the selection runs on the lists alone: the k-th largest key by counts,
//      then the top-p cut by probability mass (2^-40 fixed point; for 16-bit
//      dtypes an exact per-key histogram, so mass = count x exp(value - max)).

// Rows with top-p only (fp16 / bf16) take the window path:
//   1. phase 1 counts every element per first-digit bucket;
//   2. rigorous lower / upper bounds of every bucket's mass (count times the
//      mass of its smallest / largest value) bracket the top-p cut into a
//      window of buckets;
//   3. one pass computes every element's mass: the row total and the mass
//      below the window accumulate in registers (fp32 per 16-byte vector,
//      then 2^-40 fixed point), the window gets exact per-key counts; the
//      cut follows from count x mass per key.
// Everything else (fp32 top-p-only rows, candidate overflow, wide windows)
// takes the generic path: a radix descent over the whole row (11-bit first
// digit, then 5 bits for 16-bit keys or 11 + 10 for fp32).
//
// When the cut falls inside a run of equal values, the write pass ranks the
// ties in index order on the fly: per slot, a scan over the warps' tie
// counts, then a warp scan within each sixteenth.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace topkp {

static __device__ unsigned int g_device_error = 0;

constexpr int kBins = 4096;                  // candidate / window path first digit: 12 bits
constexpr int kSmallBins = 256;              // 8-bit digits over candidate lists
constexpr int kWinKeys = (int)(kApplyBigBytes / 4 / kApplyWarps);  // window keys per warp histogram
static_assert(kApplyWarps == kWarps, "one region per warp");

struct __align__(16) ApplyHdr {
  uint64_t full[kApplySlots];           // ring slot filled (bulk copy landed)
  uint64_t empty[kApplySlots];          // ring slot drained (one arrival per warp)
  unsigned long long ws[kWarps];        // block-scan scratch
  unsigned long long sel_off;           // select result: count/mass outside the bin
  unsigned long long small_mass[kSmallBins];
  uint32_t small_cnt[kSmallBins];
  uint32_t nseg[kApplyWarps];           // candidates in each warp's list
  uint32_t wtie[2][kApplyWarps];        // write pass: ties of T per warp sub-block, by chunk parity
  int sel_bin;                          // select result: bin, -1 if none
  uint32_t maxkey;                      // row max key
  uint32_t failed;                      // a bounded wait gave up
  uint32_t over;                        // a candidate list overflowed
};
static_assert(sizeof(ApplyHdr) <= kApplyHdrBytes, "header too large");

// Radix digits of the generic path: level 0 is an 11-bit first digit.
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

// ------------------------------------------------------- packed word ops
// A 16-byte vector is 4 words: 8 bf16/fp16 values (2 per word) or 4 fp32.
// Masks are all-ones in every lane (half or word) where the predicate holds.
template <int DT> struct Packed;
template <> struct Packed<TOPKP_BF16> {
  __device__ static __forceinline__ __nv_bfloat162 v2(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }
  __device__ static __forceinline__ uint32_t max_raw(uint4 q) {
    const __nv_bfloat162 m = __hmax2(__hmax2(v2(q.x), v2(q.y)), __hmax2(v2(q.z), v2(q.w)));
    const __nv_bfloat16 r = __hmax(__low2bfloat16(m), __high2bfloat16(m));
    return (uint32_t)__bfloat16_as_ushort(r);
  }
  __device__ static __forceinline__ uint32_t ge(uint32_t a, uint32_t b) { return __hge2_mask(v2(a), v2(b)); }
  __device__ static __forceinline__ uint32_t gt(uint32_t a, uint32_t b) { return __hgt2_mask(v2(a), v2(b)); }
  __device__ static __forceinline__ uint32_t eq(uint32_t a, uint32_t b) { return __heq2_mask(v2(a), v2(b)); }
  __device__ static __forceinline__ uint32_t splat(uint32_t raw) { return raw | (raw << 16); }
};
template <> struct Packed<TOPKP_F16> {
  __device__ static __forceinline__ __half2 v2(uint32_t w) { return *reinterpret_cast<__half2*>(&w); }
  __device__ static __forceinline__ uint32_t max_raw(uint4 q) {
    const __half2 m = __hmax2(__hmax2(v2(q.x), v2(q.y)), __hmax2(v2(q.z), v2(q.w)));
    const __half r = __hmax(__low2half(m), __high2half(m));
    return (uint32_t)__half_as_ushort(r);
  }
  __device__ static __forceinline__ uint32_t ge(uint32_t a, uint32_t b) { return __hge2_mask(v2(a), v2(b)); }
  __device__ static __forceinline__ uint32_t gt(uint32_t a, uint32_t b) { return __hgt2_mask(v2(a), v2(b)); }
  __device__ static __forceinline__ uint32_t eq(uint32_t a, uint32_t b) { return __heq2_mask(v2(a), v2(b)); }
  __device__ static __forceinline__ uint32_t splat(uint32_t raw) { return raw | (raw << 16); }
};
template <> struct Packed<TOPKP_F32> {
  __device__ static __forceinline__ uint32_t max_raw(uint4 q) {
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                                 fmaxf(__uint_as_float(q.z), __uint_as_float(q.w))));
  }
  __device__ static __forceinline__ uint32_t ge(uint32_t a, uint32_t b) {
    return __uint_as_float(a) >= __uint_as_float(b) ? 0xffffffffu : 0u;
  }
  __device__ static __forceinline__ uint32_t gt(uint32_t a, uint32_t b) {
    return __uint_as_float(a) > __uint_as_float(b) ? 0xffffffffu : 0u;
  }
  __device__ static __forceinline__ uint32_t eq(uint32_t a, uint32_t b) {
    return __uint_as_float(a) == __uint_as_float(b) ? 0xffffffffu : 0u;
  }
  __device__ static __forceinline__ uint32_t splat(uint32_t raw) { return raw; }
};

// One bit per element of a 16-byte vector from four per-word lane masks
// (bit j = element j), and back.
template <int KB>
__device__ __forceinline__ uint32_t mask_bits(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3) {
  if (KB == 16)
    return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
           ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
  return (m0 & 1u) | (m1 & 2u) | (m2 & 4u) | (m3 & 8u);
}
template <int KB>
__device__ __forceinline__ uint32_t bits_word_mask(uint32_t bits, int w) {
  if (KB == 16) return (((bits >> (2 * w)) & 1u) ? 0x0000ffffu : 0u) | (((bits >> (2 * w + 1)) & 1u) ? 0xffff0000u : 0u);
  return ((bits >> w) & 1u) ? 0xffffffffu : 0u;
}
// element j of a 16-byte vector
template <int DT>
__device__ __forceinline__ typename DType<DT>::raw vec_elem(const uint4& q, int j) {
  if (DType<DT>::kKeyBits == 16) {
    const uint32_t w = (j & 4) ? ((j & 2) ? q.w : q.z) : ((j & 2) ? q.y : q.x);
    return (typename DType<DT>::raw)((j & 1) ? (w >> 16) : (w & 0xffffu));
  }
  return (typename DType<DT>::raw)((j & 2) ? ((j & 1) ? q.w : q.z) : ((j & 1) ? q.y : q.x));
}

// --------------------------------------------------- block-wide selection
// Result of a block-wide bin selection, identical in every thread.
struct Sel {
  int bin;                   // selected bin, -1 if none
  unsigned long long off;    // count / mass outside the bin (above or below)
};

// Publishes the selection written into h by at most one thread: every thread
// copies it to registers, and h.sel_bin is reset behind a second barrier, so
// the next selection cannot overwrite it while a slow warp is still reading.
__device__ __forceinline__ Sel finish_select(ApplyHdr& h) {
  __syncthreads();
  const Sel r{h.sel_bin, h.sel_off};
  __syncthreads();
  if (threadIdx.x == 0) h.sel_bin = -1;
  return r;
}

// Bins per thread: thread t holds bins BPT*t .. BPT*t + BPT-1.
template <int BPT, typename B>
__device__ __forceinline__ void load_bins(const B* bins, int nbins, unsigned long long (&o)[BPT]) {
  const int b0 = BPT * threadIdx.x;
#pragma unroll
  for (int j = 0; j < BPT; ++j) o[j] = (b0 + j < nbins) ? (unsigned long long)bins[b0 + j] : 0ull;
}

// Bin holding the rank-th largest element (rank >= 1, counted from the top);
// off = number of elements in higher bins.  val(j) is the count of this
// thread's bin j (it may be called more than once).
template <int BPT, typename F>
__device__ __forceinline__ Sel select_desc_f(F&& val, unsigned long long rank, ApplyHdr& h) {
  unsigned long long s = 0, tot;
#pragma unroll
  for (int j = 0; j < BPT; ++j) s += val(j);
  const unsigned long long ex = block_exclusive_scan(s, &tot, h.ws);
  const unsigned long long above = tot - ex - s;
  if (s != 0 && above < rank && rank <= above + s) {
    unsigned long long a2 = above;
    for (int j = BPT - 1; j >= 0; --j) {
      const unsigned long long v = val(j);
      if (rank <= a2 + v) {
        h.sel_bin = BPT * threadIdx.x + j;
        h.sel_off = a2;
        break;
      }
      a2 += v;
    }
  }
  return finish_select(h);
}

// First bin whose ascending cumulative mass exceeds target (-1 if the total
// does not); off = mass below it.  val(j) is the mass of this thread's bin j.
template <int BPT, typename F>
__device__ __forceinline__ Sel select_asc_f(F&& val, unsigned long long target, ApplyHdr& h) {
  unsigned long long s = 0, tot;
#pragma unroll
  for (int j = 0; j < BPT; ++j) s += val(j);
  const unsigned long long ex = block_exclusive_scan(s, &tot, h.ws);
  if (ex <= target && target < ex + s) {
    unsigned long long below = ex;
    for (int j = 0; j < BPT; ++j) {
      const unsigned long long v = val(j);
      if (target < below + v) {
        h.sel_bin = BPT * threadIdx.x + j;
        h.sel_off = below;
        break;
      }
      below += v;
    }
  }
  return finish_select(h);
}

template <int BPT>
__device__ __forceinline__ Sel select_desc(const unsigned long long (&b)[BPT], unsigned long long rank, ApplyHdr& h) {
  return select_desc_f<BPT>([&](int j) { return b[j]; }, rank, h);
}

template <int BPT>
__device__ __forceinline__ Sel select_asc(const unsigned long long (&b)[BPT], unsigned long long target, ApplyHdr& h) {
  return select_asc_f<BPT>([&](int j) { return b[j]; }, target, h);
}

// Sum over the CTA of val(j) for every thread's BPT bins.
template <int BPT, typename F>
__device__ __forceinline__ unsigned long long block_sum_f(F&& val, unsigned long long* ws) {
  unsigned long long s = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) s += val(j);
  return block_sum(s, ws);
}

// masked iff cumulative mass <= thr * S (integers: <= floor(thr * S))
__device__ __forceinline__ unsigned long long mass_target(float thr, unsigned long long S) {
  return (unsigned long long)floor((double)thr * (double)S);
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

enum TieRule : int { kTiesKept = 0, kTiesMasked = 1, kTiesStraddle = 2, kKeepAll = 3 };

template <int DT>
using CandKey = typename std::conditional<DType<DT>::kKeyBits == 16, uint16_t, uint32_t>::type;

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) apply_kernel(const ApplyArgs a) {
  using D = DType<DT>;
  using P = Packed<DT>;
  using raw = typename D::raw;
  using L = Levels<D::kKeyBits>;
  using ckey = CandKey<DT>;
  constexpr int VEC = 16 / sizeof(raw);
  constexpr int KB = D::kKeyBits;
  constexpr int SHB = KB - 12;           // 12-bit first digit of the candidate / window paths
  constexpr int SH1 = L::shift(0);       // 11-bit first digit of the generic path
  constexpr int CAPW = (int)(kApplyBigBytes / sizeof(ckey)) / kApplyWarps;  // list entries per warp

  extern __shared__ __align__(128) unsigned char smem[];
  ApplyHdr& h = *reinterpret_cast<ApplyHdr*>(smem);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kApplyHdrBytes);
  unsigned char* big = smem + kApplyHdrBytes + kApplyHistBytes;
  unsigned char* ring = smem + kApplyFixedSmem;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int V = a.V;
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  raw* orow = reinterpret_cast<raw*>(a.out) + row * a.ldo;
  ckey* seg = reinterpret_cast<ckey*>(big) + warp * CAPW;
  uint32_t* whist = reinterpret_cast<uint32_t*>(big) + warp * kWinKeys;
  unsigned long long* mass = reinterpret_cast<unsigned long long*>(big);

  const int kv = a.k ? a.k[row] : 0;
  const bool topk = a.k != nullptr && kv >= 1 && kv <= V - 1;
  const bool topp = a.p != nullptr;
  const bool keepall = !topk && !topp;
  const bool window = !topk && topp && KB == 16;

  const uint64_t pol_last = l2_policy_evict_first();

  // ---- ring geometry ----
  const int CH = a.chunk;                         // bytes per slot
  const int CHE = CH / (int)sizeof(raw);          // elements per slot
  const int SUBV = CH / 16 / kApplyWarps;         // vectors per warp per slot
  const int nbytes = V * (int)sizeof(raw);
  const bool aligned = a.aligned != 0;
  const int nb16 = aligned ? (nbytes & ~15) : 0;  // bytes moved by bulk copies
  const int body = aligned ? nb16 / (int)sizeof(raw) : V;  // elements in whole chunks
  const int nch = (body * (int)sizeof(raw) + CH - 1) / CH;
  const bool has_tail = body < V;                 // aligned rows: the last < 16 bytes

  if (tid == 0) {
    h.maxkey = 0;
    h.failed = 0;
    h.over = 0;
    h.sel_bin = -1;
    for (int i = 0; i < kApplySlots; ++i) {
      mbar_init(&h.full[i], 1);
      mbar_init(&h.empty[i], kApplyWarps);
    }
    fence_mbar_init();
  }
  if (topk || window)
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
  __syncthreads();

  uint32_t used = 0;  // chunks consumed so far, all passes (CTA-uniform)
  bool my_fail = false;
  // thread 0: start the bulk copy of chunk c of the current pass (global chunk used + c)
  auto issue = [&](int c, bool last_use) {
    const uint32_t g = used + (uint32_t)c;
    const int slot = (int)(g % kApplySlots);
    if (g >= (uint32_t)kApplySlots &&
        !mbar_wait_bounded(&h.empty[slot], ((g / kApplySlots) - 1u) & 1u, a.timeout_ns))
      my_fail = true;
    const uint32_t bytes = (uint32_t)min(CH, nb16 - c * CH);
    mbar_arrive_expect_tx(&h.full[slot], bytes);
    const unsigned char* src = reinterpret_cast<const unsigned char*>(xr) + (size_t)c * CH;
    if (last_use) bulk_g2s_hint(ring + slot * CH, src, bytes, &h.full[slot], pol_last);
    else bulk_g2s(ring + slot * CH, src, bytes, &h.full[slot]);
  };
  // This warp's vectors of chunk c, in index order: f(e, q, nv) with q the
  // 16 bytes at row offsets e .. e+VEC-1, nv of them valid (0 on idle lanes).
  // The invalid elements of a partial vector hold -inf, which never exceeds
  // a valid element and has zero mass.  slot < 0: the tail after the last
  // whole chunk.  All lanes call f together.
  const uint32_t NEG2 = P::splat((uint32_t)D::kNegInf);
  auto warp_chunk = [&](int c, int slot, auto&& f) {
    if (slot < 0) {
      if (warp == 0) {
        uint4 q = make_uint4(NEG2, NEG2, NEG2, NEG2);
        raw* r = reinterpret_cast<raw*>(&q);
        int nv = 0;
        if (lane == 0) {
          nv = V - body;
#pragma unroll
          for (int j = 0; j < VEC; ++j)
            if (j < nv) r[j] = xr[body + j];
        }
        f(body, q, nv);
      }
      return;
    }
    const int valid = min(CHE, body - c * CHE);
    for (int s = 0; s < SUBV; s += 32) {
      const int v = warp * SUBV + s + lane;
      const int e = c * CHE + v * VEC;
      const int nv = max(0, min(VEC, valid - v * VEC));
      uint4 q = make_uint4(NEG2, NEG2, NEG2, NEG2);
      if (nv > 0) {
        if (aligned) {
          q = *reinterpret_cast<const uint4*>(ring + slot * CH + v * 16);
        } else {
          raw* r = reinterpret_cast<raw*>(&q);
#pragma unroll
          for (int j = 0; j < VEC; ++j)
            if (j < nv) r[j] = xr[e + j];
        }
      }
      f(e, q, nv);
    }
  };
  // One pass over the row: per_chunk(c, slot) runs on every thread for every
  // chunk (slot -1: the tail), in order.  last_use: the final read of the row.
  auto stream = [&](bool last_use, auto&& per_chunk) {
    if (aligned && tid == 0) {
      fence_proxy_async_shared();  // earlier reads of the slots precede the new copies
      for (int c = 0; c < min(nch, kApplySlots); ++c) issue(c, last_use);
    }
    for (int c = 0; c < nch; ++c) {
      const uint32_t g = used + (uint32_t)c;
      const int slot = (int)(g % kApplySlots);
      if (aligned && !mbar_wait_bounded(&h.full[slot], (g / kApplySlots) & 1u, a.timeout_ns)) my_fail = true;
      per_chunk(c, slot);
      __syncwarp();
      if (lane == 0) mbar_arrive(&h.empty[slot]);
      if (aligned && tid == 0 && c + kApplySlots < nch) {
        fence_proxy_async_shared();
        issue(c + kApplySlots, last_use);
      }
    }
    used += (uint32_t)nch;
    if (has_tail) per_chunk(nch, -1);
  };
  auto each_vec = [&](bool last_use, auto&& f) {
    stream(last_use, [&](int c, int slot) { warp_chunk(c, slot, f); });
  };
  auto each_elem = [&](auto&& g) {
    each_vec(false, [&](int, const uint4& q, int nv) {
      const raw* r = reinterpret_cast<const raw*>(&q);
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (j < nv) g(r[j]);
    });
  };

  // bit j set when element j (of nv) is >= the value whose lanes fill B2
  auto ge_bits = [&](const uint4& q, int nv, uint32_t B2) -> uint32_t {
    const uint32_t b = mask_bits<KB>(P::ge(q.x, B2), P::ge(q.y, B2), P::ge(q.z, B2), P::ge(q.w, B2));
    return b & ((1u << nv) - 1u);
  };
  auto eq_bits = [&](const uint4& q, int nv, uint32_t B2) -> uint32_t {
    const uint32_t b = mask_bits<KB>(P::eq(q.x, B2), P::eq(q.y, B2), P::eq(q.z, B2), P::eq(q.w, B2));
    return b & ((1u << nv) - 1u);
  };
  // key of the largest element of a vector with at least one valid element
  // (the -inf padding never wins)
  auto vmax_key = [&](const uint4& q) -> uint32_t { return order_key<DT>((raw)P::max_raw(q)); };
  // appends the elements flagged in bits to this warp's list (all lanes call it)
  uint32_t nseg = 0;  // warp-uniform
  auto append = [&](const uint4& q, uint32_t bits) {
    const uint32_t c = __popc(bits);
    if (!__any_sync(0xffffffffu, c != 0)) return;
    const uint32_t incl = warp_incl_scan(c);
    uint32_t slot = nseg + incl - c;
    while (bits) {
      const int j = __ffs(bits) - 1;
      bits &= bits - 1;
      if (slot < (uint32_t)CAPW) seg[slot] = (ckey)order_key<DT>(vec_elem<DT>(q, j));
      ++slot;
    }
    nseg += __shfl_sync(0xffffffffu, incl, 31);
  };

  // ---- pass A (from HBM): the row max, plus ----
  uint32_t kmax = 0;
  bool listed = false;   // top-k candidates collected during pass A
  uint32_t Lkey = 0;     // candidate bound
  if (topk) {
    // The first kApplySlots chunks stay resident until the k-th largest of
    // their vector maxima gives the candidate bound L; then every vector of
    // the row, those chunks included, is tested against L as it passes.
    const int npre = min(nch, kApplySlots);
    if (aligned && tid == 0)
      for (int c = 0; c < npre; ++c) issue(c, false);
    for (int c = 0; c < npre; ++c) {
      if (aligned && !mbar_wait_bounded(&h.full[c], 0u, a.timeout_ns)) my_fail = true;
      warp_chunk(c, c, [&](int, const uint4& q, int nv) {
        if (nv) {
          const uint32_t key = vmax_key(q);
          kmax = max(kmax, key);
          atomicAdd(&hist[key >> SHB], 1u);
        }
      });
    }
    __syncthreads();
    const int lb = select_desc_f<kBins / kThreads>(
        [&](int j) -> unsigned long long { return hist[(kBins / kThreads) * tid + j]; }, (unsigned long long)kv, h).bin;
    listed = lb >= 0;
    Lkey = listed ? (uint32_t)lb << SHB : 0u;
    const uint32_t L2 = P::splat((uint32_t)raw_of_key<DT>(Lkey));
    auto step_rest = [&](const uint4& q, int nv) {
      if (nv) {
        const uint32_t key = vmax_key(q);
        kmax = max(kmax, key);
        if (!listed) atomicAdd(&hist[key >> SHB], 1u);
      }
      if (listed) append(q, nv ? ge_bits(q, nv, L2) : 0u);
    };
    for (int c = 0; c < npre; ++c) {
      if (listed) warp_chunk(c, c, [&](int, const uint4& q, int nv) { append(q, nv ? ge_bits(q, nv, L2) : 0u); });
      __syncwarp();
      if (lane == 0) mbar_arrive(&h.empty[c]);
      if (aligned && tid == 0 && c + kApplySlots < nch) {
        fence_proxy_async_shared();
        issue(c + kApplySlots, false);
      }
    }
    for (int c = npre; c < nch; ++c) {
      const int slot = c % kApplySlots;
      if (aligned && !mbar_wait_bounded(&h.full[slot], (uint32_t)(c / kApplySlots) & 1u, a.timeout_ns))
        my_fail = true;
      warp_chunk(c, slot, [&](int, const uint4& q, int nv) { step_rest(q, nv); });
      __syncwarp();
      if (lane == 0) mbar_arrive(&h.empty[slot]);
      if (aligned && tid == 0 && c + kApplySlots < nch) {
        fence_proxy_async_shared();
        issue(c + kApplySlots, false);
      }
    }
    used = (uint32_t)nch;
    if (has_tail) warp_chunk(nch, -1, [&](int, const uint4& q, int nv) { step_rest(q, nv); });
  } else if (!keepall) {
    // the per-bucket counts of every element (window path)
    each_vec(false, [&](int, const uint4& q, int nv) {
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        if (j < nv) {
          const uint32_t key = order_key<DT>(vec_elem<DT>(q, j));
          kmax = max(kmax, key);
          if (window) atomicAdd(&hist[key >> SHB], 1u);
        }
      }
    });
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) atomicMax(&h.maxkey, kmax);
  __syncthreads();

  uint32_t T = 0;               // cut key
  unsigned long long r0 = 0;    // ties of T masked, in index order
  bool cut_last = false;        // top-p keeps only the last sorted position
  bool done = keepall;          // cut found
  const float thr = topp ? top_p_threshold<DT>(a.p, row) : 0.0f;
  const uint32_t gmax = h.maxkey;
  const MassRef mr(value_of_key<DT>(gmax));

  // ---------------------------------------------------- candidate path
  if (topk) {
    bool have = listed;
    if (!listed) {
      // k exceeds the resident vectors: bound from the whole row's vector
      // maxima, then pass B (from L2) collects the candidates
      const int lb = select_desc_f<kBins / kThreads>(
          [&](int j) -> unsigned long long { return hist[(kBins / kThreads) * tid + j]; }, (unsigned long long)kv, h).bin;
      if (lb >= 0) {
        Lkey = (uint32_t)lb << SHB;
        const uint32_t L2 = P::splat((uint32_t)raw_of_key<DT>(Lkey));
        each_vec(false, [&](int, const uint4& q, int nv) { append(q, nv ? ge_bits(q, nv, L2) : 0u); });
        have = true;
      }
    }
    if (have) {
      if (lane == 0) {
        h.nseg[warp] = min(nseg, (uint32_t)CAPW);
        if (nseg > (uint32_t)CAPW) h.over = 1;
      }
      __syncthreads();

      if (!h.over) {
        // ---- select on the lists (every element >= the k-th largest is listed) ----
        const int myn = (int)h.nseg[warp];
        auto each_own = [&](auto&& f) {
          for (int j = lane; j < myn; j += 32) f((uint32_t)seg[j]);
        };
        if (KB == 16 && gmax - Lkey < (uint32_t)kBins) {
          // exact per-key counts over [L, max]: a 16-bit key is a value
          for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
          __syncthreads();
          each_own([&](uint32_t key) { atomicAdd(&hist[key - Lkey], 1u); });
          __syncthreads();
          constexpr int BPT = kBins / kThreads;
          auto cnt = [&](int j) -> unsigned long long { return hist[BPT * tid + j]; };
          const int bk = select_desc_f<BPT>(cnt, (unsigned long long)kv, h).bin;
          T = Lkey + (uint32_t)bk;
          if (topp) {
            auto mb = [&](int j) -> unsigned long long {
              const int bin = BPT * tid + j;
              return (bin >= bk && hist[bin]) ? hist[bin] * mass_fixed(value_of_key<DT>(Lkey + bin), mr) : 0ull;
            };
            const unsigned long long S = block_sum_f<BPT>(mb, h.ws);
            const unsigned long long target = mass_target(thr, S);
            const Sel sp = select_asc_f<BPT>(mb, target, h);
            if (sp.bin < 0) {
              cut_last = true;
              r0 = hist[gmax - Lkey] - 1ull;
            } else {
              T = Lkey + (uint32_t)sp.bin;
              const unsigned long long u = mass_fixed(value_of_key<DT>(T), mr);
              r0 = u ? (target - sp.off) / u : 0ull;
            }
          }
        } else {
          // 8-bit radix digits over the list keys
          constexpr int NL = KB / 8;
          uint32_t prefix = 0;
          unsigned long long rank = (unsigned long long)kv;
          for (int l = 0; l < NL; ++l) {
            const int sh = KB - 8 * (l + 1);
            for (int i = tid; i < kSmallBins; i += kThreads) h.small_cnt[i] = 0;
            __syncthreads();
            each_own([&](uint32_t key) {
              if (l == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&h.small_cnt[(key >> sh) & 255u], 1u);
            });
            __syncthreads();
            unsigned long long cb[1];
            load_bins(h.small_cnt, kSmallBins, cb);
            const Sel sd = select_desc(cb, rank, h);
            prefix = (prefix << 8) | (uint32_t)max(sd.bin, 0);
            rank -= sd.off;
          }
          const uint32_t kkey = prefix;
          T = kkey;
          if (topp) {
            unsigned long long mine = 0;
            each_own([&](uint32_t key) {
              if (key >= kkey) mine += mass_fixed(value_of_key<DT>(key), mr);
            });
            const unsigned long long S = block_sum(mine, h.ws);
            unsigned long long rem = mass_target(thr, S);
            uint32_t pp = 0;
            for (int l = 0; l < NL && !cut_last; ++l) {
              const int sh = KB - 8 * (l + 1);
              for (int i = tid; i < kSmallBins; i += kThreads) h.small_mass[i] = 0;
              __syncthreads();
              each_own([&](uint32_t key) {
                if (key >= kkey && (l == 0 || (key >> (sh + 8)) == pp)) {
                  const unsigned long long w = mass_fixed(value_of_key<DT>(key), mr);
                  if (w) atomicAdd(&h.small_mass[(key >> sh) & 255u], w);
                }
              });
              __syncthreads();
              unsigned long long mb[1];
              load_bins(h.small_mass, kSmallBins, mb);
              const Sel sa = select_asc(mb, rem, h);
              if (sa.bin < 0) {
                cut_last = true;  // only possible at the first level
              } else {
                pp = (pp << 8) | (uint32_t)sa.bin;
                rem -= sa.off;
              }
            }
            if (cut_last) {
              uint32_t cm = 0;
              each_own([&](uint32_t key) { cm += (key == gmax); });
              r0 = block_sum(cm, h.ws) - 1ull;
            } else {
              T = pp;
              const unsigned long long u = mass_fixed(value_of_key<DT>(T), mr);
              r0 = u ? rem / u : 0ull;
            }
          }
        }
        if (cut_last) T = gmax;
        done = true;
      }
    }
  }

  // ------------------------------------------------------- window path
  if (window) {
    constexpr int BPT = kBins / kThreads;
    // rigorous bounds of each bucket's mass: counts times the mass of the
    // bucket's smallest / largest value, widened by 2^-20 and one unit
    auto lo = [&](int j) -> unsigned long long {
      const int b = BPT * tid + j;
      if (!hist[b]) return 0ull;
      const unsigned long long m0 = mass_fixed(value_of_key<DT>((uint32_t)b << SHB), mr);
      return hist[b] * (m0 - (m0 >> 20));
    };
    auto hi = [&](int j) -> unsigned long long {
      const int b = BPT * tid + j;
      if (!hist[b]) return 0ull;
      const unsigned long long m1 = mass_fixed(value_of_key<DT>(((uint32_t)b << SHB) | ((1u << SHB) - 1u)), mr);
      return hist[b] * (m1 + (m1 >> 20) + 1);
    };
    const unsigned long long SL = block_sum_f<BPT>(lo, h.ws), SU = block_sum_f<BPT>(hi, h.ws);
    const Sel s0 = select_asc_f<BPT>(hi, mass_target(thr, SL), h);
    const Sel s1 = select_asc_f<BPT>(lo, mass_target(thr, SU), h);
    int w0 = s0.bin < 0 ? kBins - 1 : s0.bin;
    int w1 = s1.bin < 0 ? kBins - 1 : s1.bin;
    if (thr >= 1.0f) w0 = w1 = (int)(gmax >> SHB);  // only the last position survives
    const int nwin = (w1 - w0 + 1) << SHB;
    if (w1 >= w0 && nwin <= kWinKeys) {
      // pass B (from L2): row mass and mass below the window (fp32 per
      // vector, then fixed point), per-key window counts per warp.  Window
      // membership is a float compare: key order is value order.
      const uint32_t wkey0 = (uint32_t)w0 << SHB;
      const float lo_f = value_of_key<DT>(wkey0);
      const float hi_f = value_of_key<DT>(((uint32_t)w1 << SHB) | ((1u << SHB) - 1u));
      for (int i = lane; i < kWinKeys; i += 32) whist[i] = 0;
      __syncwarp();
      unsigned long long s_mine = 0, b_mine = 0;
      each_vec(false, [&](int, const uint4& q, int nv) {
        float sv = 0.0f, bv = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          if (j < nv) {
            const raw rj = vec_elem<DT>(q, j);
            const float x = D::to_float(rj);
            const float ej = mass_f32(x, mr);
            sv += ej;
            if (x < lo_f) bv += ej;
            else if (x <= hi_f) atomicAdd(&whist[order_key<DT>(rj) - wkey0], 1u);
          }
        }
        s_mine += __float2ull_rn(sv * kMassScaleF);
        b_mine += __float2ull_rn(bv * kMassScaleF);
      });
      const unsigned long long S = block_sum(s_mine, h.ws);
      const unsigned long long below = block_sum(b_mine, h.ws);
      const unsigned long long target = mass_target(thr, S);
      if (target >= S) {
        // only the last sorted position survives: the last element equal to the max
        cut_last = true;
        T = gmax;
        uint32_t cm = 0;
        each_elem([&](raw r) { cm += (order_key<DT>(r) == gmax); });
        r0 = block_sum(cm, h.ws) - 1ull;
        done = true;
      } else if (target >= below) {
        // window keys, one per thread: counts summed over the warps
        unsigned long long wb[1] = {0};
        if (tid < nwin) {
          const uint32_t* allw = reinterpret_cast<const uint32_t*>(big);
          unsigned long long cw = 0;
          for (int w = 0; w < kApplyWarps; ++w) cw += allw[w * kWinKeys + tid];
          wb[0] = cw ? cw * mass_fixed(value_of_key<DT>(wkey0 + tid), mr) : 0ull;
        }
        const Sel sw2 = select_asc(wb, target - below, h);
        if (sw2.bin >= 0) {
          T = wkey0 + (uint32_t)sw2.bin;
          const unsigned long long u = mass_fixed(value_of_key<DT>(T), mr);
          r0 = u ? (target - below - sw2.off) / u : 0ull;
          done = true;
        }
      }
    }
  }

  // ------------------------------------------------------ generic path
  if (!done) {
    __syncthreads();
    uint32_t kkey = 0;
    cut_last = false;
    r0 = 0;
    if (topk) {
      for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
      __syncthreads();
      each_elem([&](raw r) { atomicAdd(&hist[order_key<DT>(r) >> SH1], 1u); });
      __syncthreads();
      unsigned long long cb[2048 / kThreads];
      load_bins(hist, 2048, cb);
      const Sel g0 = select_desc(cb, (unsigned long long)kv, h);
      uint32_t prefix = (uint32_t)max(g0.bin, 0);
      unsigned long long rank = (unsigned long long)kv - g0.off;
      for (int l = 1; l < L::n; ++l) {
        const int shp = L::shift(l - 1), sh = L::shift(l), nb = 1 << L::bits(l);
        for (int i = tid; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        each_elem([&](raw r) {
          const uint32_t key = order_key<DT>(r);
          if ((key >> shp) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
        });
        __syncthreads();
        unsigned long long lb2[2048 / kThreads];
        load_bins(hist, nb, lb2);
        const Sel gl = select_desc(lb2, rank, h);
        prefix = (prefix << L::bits(l)) | (uint32_t)max(gl.bin, 0);
        rank -= gl.off;
      }
      kkey = prefix;
      T = kkey;
    }
    if (topp) {
      const uint32_t minkey = topk ? kkey : 0u;
      for (int i = tid; i < 2048; i += kThreads) mass[i] = 0;
      __syncthreads();
      each_elem([&](raw r) {
        const uint32_t key = order_key<DT>(r);
        if (key >= minkey) {
          const unsigned long long w = mass_fixed(D::to_float(r), mr);
          if (w) atomicAdd(&mass[key >> SH1], w);
        }
      });
      __syncthreads();
      unsigned long long mb[2048 / kThreads];
      load_bins(mass, 2048, mb);
      unsigned long long part = 0;
#pragma unroll
      for (int j = 0; j < 2048 / kThreads; ++j) part += mb[j];
      const unsigned long long S = block_sum(part, h.ws);
      const unsigned long long target = mass_target(thr, S);
      const Sel gp = select_asc(mb, target, h);
      if (gp.bin < 0) {
        cut_last = true;
      } else {
        uint32_t prefix = (uint32_t)gp.bin;
        unsigned long long rem = target - gp.off;
        for (int l = 1; l < L::n; ++l) {
          const int shp = L::shift(l - 1), sh = L::shift(l), nb = 1 << L::bits(l);
          for (int i = tid; i < nb; i += kThreads) mass[i] = 0;
          __syncthreads();
          each_elem([&](raw r) {
            const uint32_t key = order_key<DT>(r);
            if (key >= minkey && (key >> shp) == prefix) {
              const unsigned long long w = mass_fixed(D::to_float(r), mr);
              if (w) atomicAdd(&mass[(key >> sh) & (nb - 1)], w);
            }
          });
          __syncthreads();
          unsigned long long lb2[2048 / kThreads];
          load_bins(mass, nb, lb2);
          const Sel gq = select_asc(lb2, rem, h);
          prefix = (prefix << L::bits(l)) | (uint32_t)max(gq.bin, 0);
          rem -= gq.off;
        }
        T = prefix;
        const unsigned long long u = mass_fixed(value_of_key<DT>(T), mr);
        r0 = u ? rem / u : 0ull;
      }
    }
    if (cut_last) {
      T = gmax;
      uint32_t cm = 0;
      each_elem([&](raw r) { cm += (order_key<DT>(r) == gmax); });
      r0 = block_sum(cm, h.ws) - 1ull;
    }
  }
  if (my_fail) atomicOr(&h.failed, 1u);
  __syncthreads();

  // ---- write pass: original element or -inf, in original order ([guide] §2 step 8) ----
  const bool skip_writes = h.failed != 0;
  const uint32_t T2 = P::splat((uint32_t)raw_of_key<DT>(T));
  const bool vec_store = a.vec_out != 0;
  auto put = [&](int e, const uint4& q, int nv) {
    if (skip_writes || my_fail || nv == 0) return;  // a timed-out slot holds stale data
    if (nv == VEC && vec_store) {
      st_global_hint(orow + e, q, pol_last);
    } else {
      const raw* r = reinterpret_cast<const raw*>(&q);
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (j < nv) orow[e + j] = r[j];
    }
  };
  const int wrule = keepall ? kKeepAll : (r0 == 0 ? kTiesKept : kTiesStraddle);
  if (wrule != kTiesStraddle) {
    each_vec(true, [&](int e, const uint4& qin, int nv) {
      uint4 q = qin;
      if (wrule == kTiesKept) {
        uint32_t* wv = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t mk = P::ge(wv[j], T2);
          wv[j] = (wv[j] & mk) | (NEG2 & ~mk);
        }
      }
      put(e, q, nv);
    });
  } else {
    // The cut falls inside the run of elements equal to T: the first r0 of
    // them, in index order, are masked.  Per chunk, a scan over the warps'
    // tie counts tells each warp whether its ties are all masked, all kept,
    // or (one warp of one chunk) split, which it resolves with warp scans.
    unsigned long long running = 0;  // ties in earlier chunks (CTA-uniform)
    stream(true, [&](int c, int slot) {
      uint32_t wc = 0;
      warp_chunk(c, slot, [&](int, const uint4& q, int nv) { wc += __popc(eq_bits(q, nv, T2)); });
      wc = __reduce_add_sync(0xffffffffu, wc);
      const int par = (c & 1);
      if (lane == 0) h.wtie[par][warp] = wc;
      __syncthreads();
      unsigned long long pre = running, tot = 0;
      for (int w = 0; w < kApplyWarps; ++w) {
        if (w < warp) pre += h.wtie[par][w];
        tot += h.wtie[par][w];
      }
      const int rl = (pre + wc <= r0) ? kTiesMasked : (pre >= r0 ? kTiesKept : kTiesStraddle);
      unsigned long long seen = pre;  // warp-uniform
      warp_chunk(c, slot, [&](int e, const uint4& qin, int nv) {
        uint4 q = qin;
        uint32_t keep_ties = 0;  // rl == kTiesStraddle: ties of this vector that stay
        if (rl == kTiesStraddle) {
          uint32_t tb = eq_bits(q, nv, T2);
          const uint32_t cnt = __popc(tb);
          const uint32_t incl = warp_incl_scan(cnt);
          unsigned long long rank = seen + incl - cnt;
          while (tb) {
            const int j = __ffs(tb) - 1;
            tb &= tb - 1;
            if (rank >= r0) keep_ties |= 1u << j;
            ++rank;
          }
          seen += __shfl_sync(0xffffffffu, incl, 31);
        }
        uint32_t* wv = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t mk;
          if (rl == kTiesKept) mk = P::ge(wv[j], T2);
          else if (rl == kTiesMasked) mk = P::gt(wv[j], T2);
          else mk = P::gt(wv[j], T2) | bits_word_mask<KB>(keep_ties, j);
          wv[j] = (wv[j] & mk) | (NEG2 & ~mk);
        }
        put(e, q, nv);
      });
      running += tot;
    });
  }
  if (my_fail) atomicOr(&g_device_error, 1u);
}

template <int DT>
static cudaError_t launch_one(const ApplyPlan& plan, const ApplyArgs& a, cudaStream_t s) {
  auto kern = apply_kernel<DT>;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  kern<<<dim3((unsigned)a.B), dim3(kThreads), plan.smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_apply(topkp_dtype dt, const ApplyPlan& plan, const ApplyArgs& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return launch_one<TOPKP_F32>(plan, a, s);
    case TOPKP_F16: return launch_one<TOPKP_F16>(plan, a, s);
    case TOPKP_BF16: return launch_one<TOPKP_BF16>(plan, a, s);
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
