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
// overlaps every other row's.  Warp w owns the w-th sixteenth of the row's
// 16-byte vectors (warp 0 also the unaligned head, the last warp the tail);
// its lanes read consecutive vectors straight into registers, several loads
// in flight per lane, so every warp load is one coalesced 512-byte access.
// The first pass reads HBM; later passes read the same bytes again from L2
// (the final one with an evict-first hint), so HBM sees each logit read once
// and each output written once.
//
// Rows with top-k take the candidate path:
//   1. pass A: one packed max per 16-byte vector, the row max, and a
//      histogram of the vector maxima over a 12-bit first digit;
//   2. the k-th largest vector maximum lower-bounds the row's k-th largest
//      element (k distinct elements reach it); its bucket floor L decides
//      candidacy.  Pass B tests every vector with one packed ">= L" compare
//      and appends the few elements >= L, with their positions, to its
//      warp's list.  For small k the first load group of every warp gives
//      the bound and pass A collects the candidates itself;
//   3. the selection runs on the lists alone: the k-th largest key by counts,
//      then the top-p cut by probability mass (2^-40 fixed point; for 16-bit
//      dtypes an exact per-key histogram, so mass = count x exp(value - max)).
// bf16 rows with top-p only take the mass-table path: pass A counts every
// element per key in a table of the keys that can carry mass (a few
// thousand), and the exact cut follows with one exponential per key.
// fp16 rows with top-p only (and bf16 rows whose keys do not fit) take the
// window path:
//   1. pass A counts every element per 12-bit bucket;
//   2. rigorous lower / upper bounds of every bucket's mass (count times the
//      mass of its smallest / largest value) bracket the top-p cut into a
//      window of buckets; each window bucket gets 16 per-key counters (only
//      the occupied ones when a window crossing zero spans too many);
//   3. pass B computes every element's mass: the row total and the mass
//      below the window accumulate in registers (each element's 2^-40
//      fixed-point mass, so every path sums the same integers), the few
//      elements inside the window are counted per key; the cut follows from
//      count x mass per key.
// Everything else (fp32 top-p-only rows, overflowing lists, windows with too
// many occupied buckets) takes the generic path: a radix descent over the
// whole row (11-bit first digit, then 5 bits for 16-bit keys or 11 + 10 for
// fp32).
//
// The write.  When the listed survivors are few, the row is filled with -inf
// and they are scattered to their positions (ties of T ranked by position),
// without reading the row again.  Otherwise a write pass re-reads the row:
// with per-warp tie counts of T from the lists, a warp whose ties are all
// masked or all kept applies one compare and only the warp where the cut
// falls ranks its ties with warp scans; without them, the ties are written
// as kept while every warp records their positions in index order, and the
// first r0 then become -inf.
#include <type_traits>

#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"

namespace topkp {

constexpr int kBins = 4096;                  // 12-bit first digit: candidate path, key-count buckets
constexpr int kSmallBins = 256;              // 8-bit digits over candidate lists
constexpr int kBPT = kBins / kThreads;       // 12-bit bins each thread scans
constexpr int kKeyBlocks = (int)(kApplyBigBytes / (16 * 4));  // 16-key count blocks of the window path
static_assert(kApplyAuxBytes >= (size_t)kKeyBlocks * (2 + 8), "block -> bucket map and block masses");
static_assert(kApplyAuxBytes >= (size_t)kThreads * 8, "per-thread partial masses of a split mass table");
static_assert(2 * kBins * 8 <= (int)kApplyBigBytes, "bucket mass bounds fit the big region");
constexpr uint32_t kNoBlock = 0xffffffffu;   // bucket without a count block
constexpr int kMassBins = (int)(kApplyBigBytes / 4);  // per-key counters of the bf16 mass-table path
constexpr int kTieRankMax = 1024;            // ties of the cut ranked by position for the scatter write
constexpr int kLoadsSimple = 8;              // vectors in flight per lane, light per-vector work
constexpr int kLoadsHeavy = 4;               // vectors in flight per lane, per-element work

struct __align__(16) ApplyHdr {
  // the small tables come first: cluster merges read them as 16-byte vectors
  unsigned long long small_mass[kSmallBins];
  uint32_t small_cnt[kSmallBins];
  unsigned long long ws[2 * kWarps];    // block-scan scratch (paired scans use both halves)
  unsigned long long sel_off;           // select result: count/mass outside the bin
  uint32_t nseg[kWarps];                // candidates in each warp's list
  uint32_t wtie[kWarps];                // ties of T in each warp's sixteenth of the row
  int sel_bin;                          // select result: bin, -1 if none
  uint32_t maxkey;                      // row max key
  uint32_t over;                        // a candidate list overflowed
  uint32_t fill;                        // write by a -inf fill plus a scatter of the listed survivors
  uint32_t ntie;                        // ties of T gathered for ranking
  uint32_t tie_cut;                     // position of the first kept tie of T
  int w0, w1;                           // window path: first / last bucket of the window
  uint32_t mt_a, mt_b, mt_floor, mt_k0;  // mass-table path: bin = a - mag (x < 0) or b + mag (x >= 0),
  int mt_qn;                             // mag clamped to >= floor; qn = bin of the negative floor;
  uint32_t mt_lump;                      // k0 = provisional max key; lump: floors hold zero-equal keys
  uint32_t slot;                         // block_first_true scratch
  ClSlots cx;                            // cluster exchange slots (rows split over a cluster)
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
  // both values of a word as floats (low half first)
  __device__ static __forceinline__ float2 unpack2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
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
  // both values of a word as floats (low half first)
  __device__ static __forceinline__ float2 unpack2(uint32_t w) { return __half22float2(*reinterpret_cast<__half2*>(&w)); }
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
  __device__ static __forceinline__ float2 unpack2(uint32_t w) { return make_float2(__uint_as_float(w), 0.0f); }
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

// Order keys of the two 16-bit values in a word, packed the same way (the
// order_key mapping, two lanes at once: neither lane carries into the other).
__device__ __forceinline__ uint32_t order_keys2(uint32_t w) {
  const uint32_t mag = w & 0x7fff7fffu;
  const uint32_t neg = (w >> 15) & 0x00010001u;
  const uint32_t m = (neg << 16) - neg;  // 0xffff in every negative lane
  return ((0x80008000u + mag) & ~m) | ((0x80008000u - mag) & m);
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



// Shared-memory slot of bin v in a table that thread t scans as the BPT
// consecutive bins BPT*t .. BPT*t+BPT-1 (BPT a power of two <= 32): the low
// bits are XORed with the bin's 32-word group, so the 32 lanes of a warp
// reading their j-th bins hit 32 different banks.  A bijection on every
// aligned run of BPT bins.
template <int BPT>
__device__ __forceinline__ uint32_t swz(uint32_t v) {
  static_assert(BPT >= 1 && BPT <= 32 && (BPT & (BPT - 1)) == 0, "BPT");
  return v ^ ((v >> 5) & (uint32_t)(BPT - 1));
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



// Smallest key in [lo, hi] where a predicate that is false then true over
// the keys holds (pred(hi) must hold), searched by the whole CTA: every
// round tests one evenly spaced key per thread.  `slot` is shared scratch.
template <typename Pred>
__device__ __forceinline__ uint32_t block_first_true(uint32_t lo, uint32_t hi, Pred pred, uint32_t* slot) {
  while (true) {
    const uint32_t span = hi - lo + 1;
    const uint32_t stride = (span + kThreads - 1) / kThreads;
    if (threadIdx.x == 0) *slot = hi;
    __syncthreads();
    const uint32_t key = lo + threadIdx.x * stride;
    if (key < hi && pred(key)) atomicMin(slot, key);
    __syncthreads();
    const uint32_t first = *slot;
    __syncthreads();
    if (stride == 1) return first;
    lo = first >= lo + stride - 1 ? first - (stride - 1) : lo;
    hi = first;
  }
}

// The top-p cut over n bins in ascending key order: bin i holds cnt(i)
// elements of key key_of(i), each of mass mass_fixed(value(key_of(i))).
// Bins below `first` are left out (top-k masked them).  Bins are spread
// evenly over the threads; one block scan gives the mass S and the target
// floor(thr * S), and the thread owning the bin where the ascending
// cumulative mass passes the target resolves the key and the masked ties.
// last: the target reaches S (only the last sorted position survives).
// Otherwise .bin is the cut key and .off the masked ties, or .bin = -1 when
// the cut falls in a bin that ok(i) rejects.
//
// For a table split over a cluster (every CTA counted its own slice into
// its own table, same layout), cnt reads this CTA's counts and cnt_all the
// cluster's; part (kThreads words of shared scratch) carries each thread's
// partial mass through one exchange, so only the walk to the cut reads the
// peers' tables.  For a table already summed over the cluster, cnt_all is
// cnt and part is null.
template <int DT, typename Cnt, typename CntAll, typename KeyOf, typename Ok>
__device__ __forceinline__ Sel mass_cut(int n, int first, Cnt cnt, CntAll cnt_all, KeyOf key_of, Ok ok,
                                        const MassRef& mr, float thr, ApplyHdr& h, bool* last, const Clu& cl,
                                        unsigned long long* part) {
  // an odd number of bins per thread: the lanes of a warp reading their
  // i-th bins then touch 32 different banks of a linear table
  const int bpt = ((n + kThreads - 1) / kThreads) | 1;
  const int b0 = min(n, (int)threadIdx.x * bpt), b1 = min(n, b0 + bpt);
  const int i0 = max(b0, first);
  // no branch on empty bins: the unrolled iterations overlap
  unsigned long long s = 0;
#pragma unroll 4
  for (int i = i0; i < b1; ++i)
    s += (unsigned long long)cnt(i) * mass_fixed(value_of_key<DT>(key_of(i)), mr);
  if (part != nullptr && cl.cs > 1) {
    part[threadIdx.x] = s;
    cl_merge<unsigned long long, 1>(cl, part, kThreads);
    s = part[threadIdx.x];
  }
  unsigned long long S;
  const unsigned long long ex = block_exclusive_scan(s, &S, h.ws);
  const unsigned long long target = mass_target(thr, S);
  *last = target >= S;
  if (*last) return Sel{-1, 0ull};
  // The warp of the one thread whose bins hold the target walks that
  // thread's bins 32 at a time: a scan over the lanes finds the bin where
  // the cumulative mass passes the target.
  const int lane = (int)threadIdx.x & 31;
  const unsigned own = __ballot_sync(0xffffffffu, ex <= target && target < ex + s);
  if (own) {
    const int src = __ffs(own) - 1;
    unsigned long long acc = __shfl_sync(0xffffffffu, ex, src);
    const int o0 = __shfl_sync(0xffffffffu, i0, src), o1 = __shfl_sync(0xffffffffu, b1, src);
    for (int base = o0; base < o1; base += 32) {
      const int i = base + lane;
      unsigned long long u = 0, mk = 0;
      if (i < o1) {
        u = mass_fixed(value_of_key<DT>(key_of(i)), mr);
        mk = (unsigned long long)cnt_all(i) * u;
      }
      unsigned long long incl = mk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned cross = __ballot_sync(0xffffffffu, i < o1 && target < acc + incl);
      if (cross) {
        if (lane == __ffs(cross) - 1 && ok(i)) {
          h.sel_bin = (int)key_of(i);
          h.sel_off = u ? (target - (acc + incl - mk)) / u : 0ull;
        }
        break;
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  return finish_select(h);
}

enum TieRule : int { kTiesKept = 0, kTiesMasked = 1, kTiesStraddle = 2, kKeepAll = 3 };

template <int DT>
using CandKey = typename std::conditional<DType<DT>::kKeyBits == 16, uint16_t, uint32_t>::type;

template <int N>
using Loads = std::integral_constant<int, N>;
// How a pass reads the row: through the non-coherent path, through L2 only,
// through the non-coherent path with an L2 evict-first hint (the one read of
// a row that is never read again), or (the final read of a row read more
// than once) with an L2 evict-first hint.
enum ReadKind { kReadNc, kReadCg, kReadNcFirst, kReadLast };
template <int R>
using ReadAs = std::integral_constant<int, R>;

// 16 bytes through the non-coherent path, not allocated in L1.  Only passes
// that end before the write pass starts use it, so even in place no CTA reads
// a logit it has already overwritten.
__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_nc_v4_hint(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// One row (cl.cs == 1) or one slice of a row split over a cluster.  The
// row's geometry and the state its steps share are members; each path of
// the selection and each write strategy is a method, run() calls them in
// order.  Every branch that leads to a cluster collective depends only on
// the row's parameters or on results of earlier collectives, so all CTAs of
// a cluster run the same collectives in the same order.
template <int DT>
struct RowFilter {
  using D = DType<DT>;
  using P = Packed<DT>;
  using raw = typename D::raw;
  using L = Levels<D::kKeyBits>;
  using ckey = CandKey<DT>;
  static constexpr int VEC = 16 / sizeof(raw);
  static constexpr int KB = D::kKeyBits;
  static constexpr int SHB = KB - 12;           // 12-bit first digit of the candidate / window paths
  static constexpr int SH1 = L::shift(0);       // 11-bit first digit of the generic path
  // list entries per warp: the raw value and its position in the row
  static constexpr int CAPW = (int)(kApplyBigBytes / (sizeof(ckey) + 4)) / kWarps / 2 * 2;

  // (a copy: a reference to the kernel's parameter block held in this object
  // made the compiler copy the block to local memory and spill registers)
  const ApplyArgs a;
  const int64_t row;
  const Clu cl;
  ApplyHdr& h;
  uint32_t* hist;
  unsigned char* aux;
  unsigned char* big;
  // window path: bucket -> count block, block -> bucket, block masses, counts
  uint32_t* block_of;
  uint16_t* bucket_of;
  unsigned long long* block_mass;
  uint32_t* kcount;
  int tid, lane, warp;
  int cph = 0;  // cluster exchange phase (cluster.cuh)
  int V;
  const raw* xr;
  raw* orow;  // nullptr: token only
  ckey* seg;
  uint32_t* segi;
  unsigned long long* mass;
  bool generic_only;
  int kv;
  bool topk, topp, keepall;
  float thr;
  // top-p alone with threshold 0 masks only elements of zero mass: the cut
  // follows from the row max, and pass A reads the max only
  bool p_zero, window, masstab, in_place;
  // row geometry: unaligned head, whole 16-byte vectors, tail; this CTA's
  // slice: vectors [cv0, cv1), plus the head (first CTA) and the tail (last
  // CTA); elements [e0, e1) of the row
  uintptr_t xaddr;
  int head, nvec, tail;
  const uint4* xv;
  int cv0, cv1, cn;
  bool own_head, own_tail;
  int e0, e1, per_warp, wb, we, nsteps;  // nsteps: warp-uniform
  bool vec_out;
  uint32_t NEG2;
  uint64_t pol_first;
  // single-pass top-k bound (see the constructor)
  int fv, rk;
  bool single;
  uint32_t Lkey = 0;  // candidate bound (candidate path)
  uint32_t gmax = 0;  // the row's max key
  bool early_fill = false;
  uint32_t T = 0;               // cut key
  unsigned long long r0 = 0;    // ties of T masked, in index order
  bool cut_last = false;        // top-p keeps only the last sorted position
  bool done = false;            // cut found
  bool have_wtie = false;       // h.wtie holds the ties of T per warp
  bool r0_known = true;         // cut_last: r0 already counted
  unsigned long long tie_off = 0;  // ties of T in the CTAs before this one (their slices come first)
  MassRef mr{0.0f};
  bool window_counted = false;  // the window path's bucket counts exist
  uint32_t T2 = 0;              // the cut's raw value in every lane

  __device__ __forceinline__ RowFilter(const ApplyArgs& a_, int64_t row_, const Clu& cl_, unsigned char* smem)
      : a(a_), row(row_), cl(cl_), h(*reinterpret_cast<ApplyHdr*>(smem)) {
    hist = reinterpret_cast<uint32_t*>(smem + kApplyHdrBytes);
    aux = smem + kApplyHdrBytes + kApplyHistBytes;
    big = aux + kApplyAuxBytes;
    block_of = hist;
    bucket_of = reinterpret_cast<uint16_t*>(aux);
    block_mass = reinterpret_cast<unsigned long long*>(aux + kKeyBlocks * 2);
    kcount = reinterpret_cast<uint32_t*>(big);
    tid = threadIdx.x;
    lane = tid & 31;
    warp = tid >> 5;
    V = a.V;
    xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
    orow = a.out ? reinterpret_cast<raw*>(a.out) + row * a.ldo : nullptr;
    seg = reinterpret_cast<ckey*>(big) + warp * CAPW;
    segi = reinterpret_cast<uint32_t*>(big + (size_t)kWarps * CAPW * sizeof(ckey)) + warp * CAPW;
    mass = reinterpret_cast<unsigned long long*>(big);
    generic_only = (a.force & kApplyForceGeneric) != 0;
    kv = a.k ? a.k[row] : 0;
    topk = a.k != nullptr && kv >= 1 && kv <= V - 1;
    topp = a.p != nullptr;
    keepall = !topk && !topp;
    thr = topp ? top_p_threshold<DT>(a.p, row) : 0.0f;
    p_zero = !topk && topp && !(thr > 0.0f) && !generic_only;
    window = !topk && topp && !p_zero && KB == 16 && !generic_only;
    masstab = window && DT == TOPKP_BF16;
    in_place = reinterpret_cast<const void*>(xr) == reinterpret_cast<const void*>(orow);
    xaddr = reinterpret_cast<uintptr_t>(xr);
    head = min(V, (int)(((16u - (uint32_t)(xaddr & 15u)) & 15u) / (uint32_t)sizeof(raw)));
    nvec = (V - head) / VEC;
    tail = V - head - nvec * VEC;
    xv = reinterpret_cast<const uint4*>(xr + head);
    cv0 = (int)((long long)nvec * cl.rank / cl.cs);
    cv1 = (int)((long long)nvec * (cl.rank + 1) / cl.cs);
    cn = cv1 - cv0;
    own_head = cl.rank == 0 && head > 0;
    own_tail = cl.rank == (uint32_t)cl.cs - 1u && tail > 0;
    e0 = cl.rank == 0 ? 0 : head + cv0 * VEC;
    e1 = cl.rank == (uint32_t)cl.cs - 1u ? V : head + cv1 * VEC;
    per_warp = (cn + kWarps - 1) / kWarps;
    wb = cv0 + min(cn, warp * per_warp);
    we = cv0 + min(cn, warp * per_warp + per_warp);
    nsteps = (we - wb + 31) / 32;
    vec_out = ((reinterpret_cast<uintptr_t>(orow) ^ xaddr) & 15u) == 0;
    NEG2 = P::splat((uint32_t)D::kNegInf);
    pol_first = l2_policy_evict_first();
    // Top-k: the first load group of every warp (fv vectors, a sample of the
    // row) bounds the candidates.  L is the bucket floor of the rk-th largest
    // vector maximum of the sample, rk = 2k x (sample share of the row), at
    // least 8: the row then holds about 2k elements >= L (rarely fewer than
    // k), which pass A lists, so the row is read once.  With rk = k (the sample is most of the row) L is a bound
    // by construction; otherwise it is checked after the pass: fewer than k
    // listed elements, or lists that overflow, restart the two-pass flow.
    // (the same in every CTA of a cluster: the smallest slice's first group)
    fv = min(nvec / cl.cs, kWarps * 32 * kLoadsHeavy);
    const long long rk_want = (2LL * kv * fv * VEC + V - 1) / V;
    rk = (int)min((long long)kv, max(8LL, rk_want));
    single = topk && !generic_only && rk <= fv && 8LL * kv <= (long long)kWarps * CAPW;
  }

  // the tables of the paths this row takes, cleared
  __device__ __forceinline__ void init_tables() {
    if (tid == 0) {
      h.maxkey = 0;
      h.over = 0;
      h.fill = 0;
      h.ntie = 0;
      h.tie_cut = 0;
      h.sel_bin = -1;
      h.w0 = kBins - 1;
      h.w1 = kBins - 1;
    }
    if (tid < kWarps) h.nseg[tid] = 0;
    if ((topk && !generic_only) || window)
      for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    if (masstab)
      for (int i = tid; i < kMassBins / 4; i += kThreads) reinterpret_cast<uint4*>(kcount)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
  }

  // One 16-byte vector of the row, read as the pass's load kind says.
  template <typename LC_>
  __device__ __forceinline__ uint4 load_vec(LC_ L_c, const uint4* a) {
    constexpr int L = decltype(L_c)::value;
    if constexpr (L == kReadLast) return ld_global_hint(a, pol_first);
    else if constexpr (L == kReadNcFirst) return ld_nc_v4_hint(a, pol_first);
    else if constexpr (L == kReadNc) return ld_nc_v4(a);
    else return __ldcg(a);
  }
  // n elements from row offset e0 as a vector, the rest -inf
  __device__ __forceinline__ uint4 load_partial(int ep, int n) {
    uint32_t w[4] = {NEG2, NEG2, NEG2, NEG2};
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      if (j < n) {
        const uint32_t b = (uint32_t)xr[ep + j];
        if (KB == 16) {
          const int sh = (j & 1) * 16;
          w[j >> 1] = (w[j >> 1] & ~(0xffffu << sh)) | (b << sh);
        } else {
          w[j] = b;
        }
      }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  // One pass over the row: f(e, q, nv) for this warp's vectors in index
  // order, q = the 16 bytes at row offsets e .. e+VEC-1 with nv of them valid
  // (-inf in the others, which never exceeds a valid element and has zero
  // mass; nv = 0 on idle lanes).  All lanes of a warp call f together.  U
  // vectors per lane are in flight, read as L_c (a ReadKind) says.
  template <typename UC_, typename LC_, typename F_>
  __device__ __forceinline__ void sweep(UC_ U_c, LC_ L_c, F_&& f) {
    constexpr int U = decltype(U_c)::value;
    if (warp == 0 && own_head) {
      const uint4 q = load_partial(0, lane == 0 ? head : 0);
      f(0, q, lane == 0 ? head : 0);
    }
    for (int s0 = 0; s0 < nsteps; s0 += U) {
      uint4 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = wb + (s0 + u) * 32 + lane;
        q[u] = make_uint4(NEG2, NEG2, NEG2, NEG2);
        if (v < we) q[u] = load_vec(L_c, xv + v);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (s0 + u < nsteps) {
          const int v = wb + (s0 + u) * 32 + lane;
          f(head + v * VEC, q[u], v < we ? VEC : 0);
        }
      }
    }
    if (warp == kWarps - 1 && own_tail) {
      const int et = head + nvec * VEC;
      const uint4 q = load_partial(et, lane == 0 ? tail : 0);
      f(et, q, lane == 0 ? tail : 0);
    }
  }
  // sweep() whose first load group (and the head / tail vectors) is read
  // before anything is processed; pre(q, head_vector, tail_vector) then runs
  // in every thread (it may synchronise the CTA), and f sees the row as in
  // sweep().
  template <typename UC_, typename LC_, typename PRE_, typename F_>
  __device__ __forceinline__ void sweep_pre(UC_ U_c, LC_ L_c, PRE_&& pre, F_&& f) {
    constexpr int U = decltype(U_c)::value;
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = wb + u * 32 + lane;
      q[u] = make_uint4(NEG2, NEG2, NEG2, NEG2);
      if (v < we) q[u] = load_vec(L_c, xv + v);
    }
    const uint4 hq = load_partial(0, (warp == 0 && lane == 0 && own_head) ? head : 0);
    const uint4 tq = load_partial(head + nvec * VEC, (warp == kWarps - 1 && lane == 0 && own_tail) ? tail : 0);
    pre(q, hq, tq);
    if (warp == 0 && own_head) f(0, hq, lane == 0 ? head : 0);
    // the next group's loads are in flight while this group is processed
    for (int s0 = 0; s0 < nsteps; s0 += U) {
      uint4 qn[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = wb + (s0 + U + u) * 32 + lane;
        qn[u] = make_uint4(NEG2, NEG2, NEG2, NEG2);
        if (v < we) qn[u] = load_vec(L_c, xv + v);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (s0 + u < nsteps) {
          const int v = wb + (s0 + u) * 32 + lane;
          f(head + v * VEC, q[u], v < we ? VEC : 0);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) q[u] = qn[u];
    }
    if (warp == kWarps - 1 && own_tail) f(head + nvec * VEC, tq, lane == 0 ? tail : 0);
  }
  template <typename G_>
  __device__ __forceinline__ void each_elem(G_&& g) {
    sweep(Loads<kLoadsHeavy>{}, ReadAs<kReadNc>{}, [&](int, const uint4& q, int nv) {
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (j < nv) g(vec_elem<DT>(q, j));
    });
  }

  // bit j set when element j (of nv) is >= / == the value whose lanes fill B2
  __device__ __forceinline__ uint32_t ge_bits(const uint4& q, int nv, uint32_t B2) {
    const uint32_t b = mask_bits<KB>(P::ge(q.x, B2), P::ge(q.y, B2), P::ge(q.z, B2), P::ge(q.w, B2));
    return b & ((1u << nv) - 1u);
  }
  __device__ __forceinline__ uint32_t eq_bits(const uint4& q, int nv, uint32_t B2) {
    const uint32_t b = mask_bits<KB>(P::eq(q.x, B2), P::eq(q.y, B2), P::eq(q.z, B2), P::eq(q.w, B2));
    return b & ((1u << nv) - 1u);
  }
  // key of the largest element of a vector with at least one valid element
  __device__ __forceinline__ uint32_t vmax_key(const uint4& q) { return order_key<DT>((raw)P::max_raw(q)); }

  // appends the elements of a vector that are >= the value filling the lanes
  // of L2 to this warp's list, with their positions
  __device__ __forceinline__ void append_ge(int e, const uint4& q, int nv, uint32_t L2) {
    if (nv != 0 && (P::ge(q.x, L2) | P::ge(q.y, L2) | P::ge(q.z, L2) | P::ge(q.w, L2)) != 0u) {
      uint32_t bits = ge_bits(q, nv, L2);
      uint32_t slot = atomicAdd(&h.nseg[warp], (uint32_t)__popc(bits));
      while (bits) {
        const int j = __ffs(bits) - 1;
        bits &= bits - 1;
        if (slot < (uint32_t)CAPW) {
          seg[slot] = (ckey)vec_elem<DT>(q, j);
          segi[slot] = (uint32_t)(e + j);
        }
        ++slot;
      }
    }
  }

  __device__ __forceinline__ void pass_a() {
    // ---- pass A (from HBM): the row max, plus the 12-bit first-digit
    // histogram of the vector maxima (candidate path) or of every element
    // (window path) ----
    uint32_t kmax = 0;
    if (single) {
      // the row's only read (unless the bound fails): evict-first in L2
      uint32_t L2 = 0;
      sweep_pre(
          Loads<kLoadsHeavy>{}, ReadAs<kReadNcFirst>{},
          [&](const uint4 (&q)[kLoadsHeavy], const uint4& hq, const uint4& tq) {
#pragma unroll
            for (int u = 0; u < kLoadsHeavy; ++u)
              if (wb + u * 32 + lane < we) atomicAdd(&hist[swz<kBPT>(vmax_key(q[u]) >> SHB)], 1u);
            if (warp == 0 && lane == 0 && own_head) atomicAdd(&hist[swz<kBPT>(vmax_key(hq) >> SHB)], 1u);
            if (warp == kWarps - 1 && lane == 0 && own_tail) atomicAdd(&hist[swz<kBPT>(vmax_key(tq) >> SHB)], 1u);
            __syncthreads();
            const int lb = select_desc_f<kBins / kThreads>(
                [&](int j) -> unsigned long long { return hist[swz<kBPT>(kBPT * tid + j)]; },
                (unsigned long long)rk, h).bin;
            // fewer than rk vectors in the groups: every element (the lists overflow)
            Lkey = lb > 0 ? (uint32_t)lb << SHB : order_key<DT>(D::kNegInf) + 1u;
            L2 = P::splat((uint32_t)raw_of_key<DT>(Lkey));
          },
          [&](int e, const uint4& q, int nv) {
            if (nv) kmax = max(kmax, vmax_key(q));
            append_ge(e, q, nv, L2);
          });
    } else if (topk && !generic_only) {
      sweep(Loads<kLoadsSimple>{}, ReadAs<kReadNc>{}, [&](int, const uint4& q, int nv) {
        if (nv) {
          const uint32_t key = vmax_key(q);
          kmax = max(kmax, key);
          atomicAdd(&hist[swz<kBPT>(key >> SHB)], 1u);
        }
      });
    } else if (masstab) {
      // A provisional max m0 (of every warp's first load group) fixes a table
      // in ascending key order that holds every key of non-zero mass for any
      // row max m >= m0.  It starts below m0 - 29.5 (mass 0 there for every m >=
      // m0).  A bf16 value of magnitude `mag` lands in bin a - mag (x < 0) or
      // b + mag (x >= 0) with mag first raised to a floor: when the range
      // crosses zero, magnitudes below 2^(e - 26) (e = exponent of m0 log2 e)
      // share the two floor bins -- for every m >= m0 > 0 the fused
      // multiply-add of mass_f32 rounds such x away, so their fp32 mass is
      // that of zero; otherwise the floor is the magnitude of m0 or of the
      // range's first key.  Bins outside the table (zero-mass negatives) are
      // skipped; a true max that needs a bin past the table, or values above
      // m0 merged by the floor, send the row to the window path.
      if constexpr (KB == 16) {
        uint32_t ta = 0, tb = 0, tfloor = 0;
        sweep_pre(
            Loads<kLoadsHeavy>{}, ReadAs<kReadCg>{},
            [&](const uint4 (&q)[kLoadsHeavy], const uint4& hq, const uint4& tq) {
              uint32_t km = max(vmax_key(hq), vmax_key(tq));
#pragma unroll
              for (int u = 0; u < kLoadsHeavy; ++u) km = max(km, vmax_key(q[u]));
              km = __reduce_max_sync(0xffffffffu, km);
              if (lane == 0) atomicMax(&h.maxkey, km);
              __syncthreads();
              // one table layout for the whole cluster: the largest first-group max
              const uint32_t k0 = (uint32_t)cl_reduce1<kClMax>(cl, h.cx, cph, h.maxkey);
              const float m0 = value_of_key<DT>(k0);
              constexpr uint32_t H = 1u << (KB - 1);
              const uint32_t kfin = order_key<DT>(D::kNegInf) + 1u;
              // first key: the bf16 at or below m0 - 29.5, one key lower still
              const uint32_t vb = __float_as_uint(m0 - 29.5f);
              const uint32_t r16 = (vb >> 16) + ((vb & 0x80000000u) && (vb & 0xffffu) ? 1u : 0u);
              const uint32_t klo = max(kfin, order_key<DT>((raw)r16) - 1u);
              uint32_t lump = 0, qn;
              if (klo < H) {
                const uint32_t mag_lo = H - klo;
                if (m0 > 0.0f) {
                  const int e = (int)((__float_as_uint(m0 * 1.4426950408889634f) >> 23) & 0xffu) - 127 - 26;
                  tfloor = e + 127 > 0 ? ((uint32_t)(e + 127) << 7) - 1u : 0u;  // largest magnitude below 2^e
                  lump = 1;
                } else {
                  tfloor = H - k0;  // magnitude of m0 (0 for m0 = 0)
                }
                ta = mag_lo;
                qn = mag_lo - tfloor;
              } else {
                tfloor = klo - H;  // positives only; the floor bin has zero mass
                ta = 0;            // every negative falls outside the table
                qn = 0xffffffffu;
              }
              // positives from the shared floor bin up (the negative floor bin when
              // the range crosses zero, else bin 0): both signs of a magnitude
              // at or below the floor -- and so -0 and +0 -- share one bin
              tb = (klo < H ? qn : 0u) - tfloor;
              if (tid == 0) {
                h.mt_a = ta;
                h.mt_b = tb;
                h.mt_floor = tfloor;
                h.mt_k0 = k0;
                h.mt_qn = (int)qn;
                h.mt_lump = lump;
              }
            },
            [&](int, const uint4& q, int nv) {
              if (nv) kmax = max(kmax, vmax_key(q));
              const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int j = 0; j < VEC; ++j) {
                const uint32_t v = (j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xffffu);
                const uint32_t mc = max(v & 0x7fffu, tfloor);
                const uint32_t bin = (v & 0x8000u) ? ta - mc : tb + mc;
                if (bin < (uint32_t)kMassBins) atomicAdd(&kcount[bin], 1u);  // never the -inf padding
              }
            });
      }
    } else if (window && DT != TOPKP_BF16) {
      if constexpr (KB == 16) {
        sweep(Loads<kLoadsHeavy>{}, ReadAs<kReadCg>{}, [&](int, const uint4& q, int nv) {
          if (nv) kmax = max(kmax, vmax_key(q));
          const uint32_t kp[4] = {order_keys2(q.x), order_keys2(q.y), order_keys2(q.z), order_keys2(q.w)};
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            const uint32_t key = (j & 1) ? (kp[j >> 1] >> 16) : (kp[j >> 1] & 0xffffu);
            if (j < nv) atomicAdd(&hist[swz<kBPT>(key >> SHB)], 1u);
          }
        });
      }
    } else if (!keepall || a.fused) {
      // the max alone (rows filtered by the max's threshold; and every row of
      // the fused sample, whose min-p and race are relative to the max)
      sweep(Loads<kLoadsSimple>{}, ReadAs<kReadNc>{}, [&](int, const uint4& q, int nv) {
        if (nv) kmax = max(kmax, vmax_key(q));
      });
    }
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) atomicMax(&h.maxkey, kmax);
    __syncthreads();
    gmax = (uint32_t)cl_reduce1<kClMax>(cl, h.cx, cph, h.maxkey);  // the row's max key
  }

  __device__ __forceinline__ void start_early_fill() {
    // Rows whose survivors number at most k <= V/8 end in the -inf fill and
    // scatter write (unless the cut's ties overflow the ranking).  Their fill
    // starts now, as bulk copies of a -inf block in shared memory (the window
    // path's region, unused by these rows) that run during the selection;
    // the write then waits for them and scatters the survivors.
    constexpr int kFillBlock = 8192;
    static_assert(kFillBlock <= (int)kApplyAuxBytes, "fill block fits the aux region");
    early_fill = topk && !generic_only && kv <= V / 8 && orow != nullptr &&
                            reinterpret_cast<const void*>(orow) != reinterpret_cast<const void*>(xr);
    if (early_fill) {
      uint4* negs = reinterpret_cast<uint4*>(aux);
      for (int i = tid; i < kFillBlock / 16; i += kThreads) negs[i] = make_uint4(NEG2, NEG2, NEG2, NEG2);
      fence_proxy_async_shared();
      __syncthreads();
      // this CTA's elements [e0, e1) of the output row
      raw* ob = orow + e0;
      const int n = e1 - e0;
      const uintptr_t oaddr = reinterpret_cast<uintptr_t>(ob);
      const int ohead = min(n, (int)(((16u - (uint32_t)(oaddr & 15u)) & 15u) / (uint32_t)sizeof(raw)));
      const int onv = (n - ohead) / VEC;
      for (int i = tid; i < ohead; i += kThreads) ob[i] = D::kNegInf;
      for (int i = ohead + onv * VEC + tid; i < n; i += kThreads) ob[i] = D::kNegInf;
      if (lane == 0) {
        // lane 0 of every warp issues every kWarps-th block
        unsigned char* dst = reinterpret_cast<unsigned char*>(ob + ohead);
        const long long body = (long long)onv * 16;
        for (long long off = (long long)warp * kFillBlock; off < body; off += (long long)kWarps * kFillBlock)
          bulk_store_s2g(dst + off, negs, (uint32_t)min(body - off, (long long)kFillBlock));
        bulk_commit_group();
      }
    }

  }

  __device__ __forceinline__ void candidate_path() {
    // ---------------------------------------------------- candidate path
    // Attempt 0 (single pass): every CTA listed its slice's elements >= its
    // own sampled bound L_r.  The union of the lists holds every element of
    // the row >= max_r L_r, so the k-th largest of the union is the row's as
    // soon as it is >= max_r L_r (always, with one CTA).  Otherwise, and for
    // rows without a sampled bound, attempt 1 takes one bound for the whole
    // cluster from the merged histogram of vector maxima and lists again.
    if (topk && !generic_only) {
      for (int attempt = single ? 0 : 1; attempt < 2 && !done; ++attempt) {
        bool listed = false;
        uint32_t Lmin = Lkey, Lmax = Lkey;  // smallest / largest bound of the cluster
        if (attempt == 0) {
          if (lane == 0 && h.nseg[warp] > (uint32_t)CAPW) {
            h.nseg[warp] = CAPW;
            h.over = 1;
          }
          __syncthreads();
          unsigned long long nl = 0;  // listed elements
          for (int w = 0; w < kWarps; ++w) nl += h.nseg[w];
          unsigned long long s2[2] = {(unsigned long long)h.over, nl};
          cl_reduce<kClSum, 2>(cl, h.cx, cph, s2);
          unsigned long long m2[2] = {(unsigned long long)Lkey, (unsigned long long)(0xffffffffu - Lkey)};
          cl_reduce<kClMax, 2>(cl, h.cx, cph, m2);
          Lmax = (uint32_t)m2[0];
          Lmin = 0xffffffffu - (uint32_t)m2[1];
          listed = s2[0] == 0 && s2[1] >= (unsigned long long)kv;
        } else {
          if (single) {
            // the sampled bounds were too loose (or too high): start over from
            // the slices' vector maxima
            __syncthreads();
            for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
            if (tid < kWarps) h.nseg[tid] = 0;
            if (tid == 0) h.over = 0;
            __syncthreads();
            sweep(Loads<kLoadsSimple>{}, ReadAs<kReadNc>{}, [&](int, const uint4& q, int nv) {
              if (nv) atomicAdd(&hist[swz<kBPT>(vmax_key(q) >> SHB)], 1u);
            });
            __syncthreads();
          }
          cl_merge<uint32_t, kBins / 4 / kThreads>(cl, hist, kBins);
          const int lb = select_desc_f<kBins / kThreads>(
              [&](int j) -> unsigned long long { return hist[swz<kBPT>(kBPT * tid + j)]; }, (unsigned long long)kv, h).bin;
          if (lb > 0) {
            // pass B (from L2): every element >= L joins its warp's list
            Lkey = Lmin = Lmax = (uint32_t)lb << SHB;
            const uint32_t L2 = P::splat((uint32_t)raw_of_key<DT>(Lkey));
            sweep(Loads<kLoadsSimple>{}, ReadAs<kReadNc>{}, [&](int e, const uint4& q, int nv) { append_ge(e, q, nv, L2); });
            __syncwarp();
            if (lane == 0 && h.nseg[warp] > (uint32_t)CAPW) {
              h.nseg[warp] = CAPW;
              h.over = 1;
            }
            __syncthreads();
            listed = cl_reduce1<kClSum>(cl, h.cx, cph, (unsigned long long)h.over) == 0;
          }
        }
        if (!listed) continue;
        // ---- select on the lists (every element >= the k-th largest is listed) ----
        T = 0;
        r0 = 0;
        cut_last = false;
        const int myn = (int)h.nseg[warp];
        auto each_own = [&](auto&& f) {
          for (int j = lane; j < myn; j += 32) f(order_key<DT>((raw)seg[j]));
        };
        if (KB == 16 && gmax - Lmin < (uint32_t)kBins) {
          // exact per-key counts over [Lmin, max]: a 16-bit key is a value
          for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
          __syncthreads();
          each_own([&](uint32_t key) { atomicAdd(&hist[swz<kBPT>(key - Lmin)], 1u); });
          __syncthreads();
          cl_merge<uint32_t, kBins / 4 / kThreads>(cl, hist, kBins);
          auto cnt = [&](int j) -> unsigned long long { return hist[swz<kBPT>(kBPT * tid + j)]; };
          const int bk = select_desc_f<kBPT>(cnt, (unsigned long long)kv, h).bin;
          T = Lmin + (uint32_t)bk;
          if (T < Lmax) continue;  // the lists may miss elements above the k-th largest
          if (topp) {
            bool last;
            auto hcnt = [&](int i) { return hist[swz<kBPT>(i)]; };
            const Sel sp = mass_cut<DT>(
                (int)(gmax - Lmin) + 1, bk, hcnt, hcnt, [&](int i) { return Lmin + (uint32_t)i; },
                [](int) { return true; }, mr, thr, h, &last, cl, nullptr);
            if (last) {
              cut_last = true;
              r0 = hist[swz<kBPT>(gmax - Lmin)] - 1ull;
            } else {
              T = (uint32_t)sp.bin;
              r0 = sp.off;
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
            cl_merge<uint32_t, 1>(cl, h.small_cnt, kSmallBins);
            unsigned long long cb[1];
            load_bins(h.small_cnt, kSmallBins, cb);
            const Sel sd = select_desc(cb, rank, h);
            prefix = (prefix << 8) | (uint32_t)max(sd.bin, 0);
            rank -= sd.off;
          }
          const uint32_t kkey = prefix;
          T = kkey;
          if (T < Lmax) continue;  // the lists may miss elements above the k-th largest
          if (topp) {
            unsigned long long mine = 0;
            each_own([&](uint32_t key) {
              if (key >= kkey) mine += mass_fixed(value_of_key<DT>(key), mr);
            });
            const unsigned long long S = cl_reduce1<kClSum>(cl, h.cx, cph, block_sum(mine, h.ws));
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
              cl_merge<unsigned long long, 1>(cl, h.small_mass, kSmallBins);
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
              r0 = cl_reduce1<kClSum>(cl, h.cx, cph, block_sum(cm, h.ws)) - 1ull;
            } else {
              T = pp;
              const unsigned long long u = mass_fixed(value_of_key<DT>(T), mr);
              r0 = u ? rem / u : 0ull;
            }
          }
        }
        if (cut_last) T = gmax;
        done = true;
        // ties of T per warp, from the lists (T >= L is listed)
        uint32_t ct = 0, cgt = 0;
        each_own([&](uint32_t key) {
          ct += (key == T);
          cgt += (key > T);
        });
        ct = __reduce_add_sync(0xffffffffu, ct);
        if (lane == 0) h.wtie[warp] = ct;
        have_wtie = true;
        // The survivors are listed with their positions: when they are few,
        // the write fills the row with -inf and scatters them, without a
        // second read of the row.  Ties of T are ranked by position: this
        // CTA's ties follow the tie_off ties of the CTAs before it.
        const unsigned long long ngt_mine = block_sum(cgt, h.ws);
        unsigned long long nt_mine = 0;
        for (int w = 0; w < kWarps; ++w) nt_mine += h.wtie[w];
        {
          const unsigned long long v2[2] = {nt_mine, ngt_mine};
          unsigned long long ex2[2], tot2[2];
          cl_prefix<2>(cl, h.cx, cph, v2, ex2, tot2);
          tie_off = ex2[0];
          const unsigned long long nties = tot2[0], ngt = tot2[1];
          const bool fill = ngt + (nties - r0) <= (unsigned long long)(V / 8) && (r0 == 0 || nties <= kTieRankMax);
          if (fill && r0 > 0) {
            // this CTA masks its first rl ties (all of them: tie_cut past every position)
            const unsigned long long rl = r0 > tie_off ? min(r0 - tie_off, nt_mine) : 0ull;
            uint32_t* tpos = hist;  // free again: positions of the ties of T
            for (int j = lane; j < myn; j += 32)
              if (order_key<DT>((raw)seg[j]) == T) tpos[atomicAdd(&h.ntie, 1u)] = segi[j];
            __syncthreads();
            const int nt = (int)h.ntie;
            if (rl == (unsigned long long)nt) {
              if (tid == 0) h.tie_cut = 0xffffffffu;
            } else {
              for (int t2 = tid; t2 < nt; t2 += kThreads) {
                const uint32_t mine = tpos[t2];
                int rank = 0;
                for (int u = 0; u < nt; ++u) rank += tpos[u] < mine;
                if (rank == (int)rl) h.tie_cut = mine;  // the first tie that stays
              }
            }
          }
          if (tid == 0) h.fill = fill ? 1u : 0u;
        }
      }
    }

  }

  __device__ __forceinline__ void mass_table_path() {
    // ------------------------------------------------------ mass-table path
    // bf16 rows with top-p only.  With 128 keys per binade, the keys whose
    // fixed-point mass is non-zero (value > max - 28.4) number a few thousand
    // once the keys around zero whose fp32 mass equals that of zero share one
    // bin.  One pass of per-key counts then gives the row mass, every
    // cumulative mass and the cut exactly; elements of zero mass are always
    // masked and never counted.  Rows whose range does not fit, or whose cut
    // falls among the zero-equal keys, take the window path.
    window_counted = !masstab;  // the window path's bucket counts exist
    if (masstab) {
      uint32_t* tab = kcount;
      cl_sync(cl);  // every CTA's table is complete: read the cluster's sums through cl_sum_at
      const uint32_t ta = h.mt_a, tb = h.mt_b, tfloor = h.mt_floor, k0 = h.mt_k0, lump = h.mt_lump;
      const int qn = h.mt_qn;
      constexpr uint32_t H = 1u << (KB - 1);
      // bin of the true max: past the table, or values above m0 merged into a
      // floor bin without the zero-equal guarantee, send the row to the window path
      const uint32_t graw = (uint32_t)raw_of_key<DT>(gmax);
      const uint32_t gbin = (graw & 0x8000u) ? ta - max(graw & 0x7fffu, tfloor) : tb + max(graw & 0x7fffu, tfloor);
      if (gbin < (uint32_t)kMassBins && (lump || qn < 0 || gmax == k0)) {
        // bin v holds key H - (a - v) up to the floor bin qn, key
        // H + (v - pbase + floor) above it (pbase: the floor bin, 0 when no
        // negative carries mass); a floor bin of several keys carries the mass
        // of zero and cannot hold the cut
        const int pbase = qn >= 0 ? qn : 0;
        auto key_of = [&](int v) -> uint32_t {
          return v <= qn ? H - (ta - (uint32_t)v) : H + ((uint32_t)(v - pbase) + tfloor);
        };
        const bool shared_floor = lump && tfloor > 0;
        bool last;
        const Sel sp = mass_cut<DT>(
            (int)gbin + 1, 0, [&](int v) { return tab[v]; }, [&](int v) { return cl_sum_at(cl, tab, v); }, key_of,
            [&](int v) { return !(shared_floor && v == qn); }, mr, thr, h, &last, cl,
            reinterpret_cast<unsigned long long*>(aux));
        if (last) {
          cut_last = true;
          T = gmax;
          r0_known = false;
          done = true;
        } else if (sp.bin >= 0) {
          T = (uint32_t)sp.bin;
          r0 = sp.off;
          done = true;
        }
      }
      cl_sync(cl);  // no peer reads this CTA's table any more
      if (!done) {
        // fall back to the window path: it needs the bucket counts
        __syncthreads();
        if constexpr (KB == 16) {
          sweep(Loads<kLoadsHeavy>{}, ReadAs<kReadCg>{}, [&](int, const uint4& q, int nv) {
            const uint32_t kp[4] = {order_keys2(q.x), order_keys2(q.y), order_keys2(q.z), order_keys2(q.w)};
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
              const uint32_t key = (j & 1) ? (kp[j >> 1] >> 16) : (kp[j >> 1] & 0xffffu);
              if (j < nv) atomicAdd(&hist[swz<kBPT>(key >> SHB)], 1u);
            }
          });
        }
        __syncthreads();
        window_counted = true;
      }
    }

  }

  __device__ __forceinline__ void window_path() {
    // ------------------------------------------------------- window path
    if (window && !done && window_counted) {
      constexpr int BPT = kBins / kThreads;  // thread t owns buckets BPT*t .. BPT*t+BPT-1
      cl_merge<uint32_t, kBins / 4 / kThreads>(cl, hist, kBins);
      unsigned long long* lo_m = reinterpret_cast<unsigned long long*>(big);  // [kBins]
      unsigned long long* hi_m = lo_m + kBins;                                // [kBins]
      // rigorous bounds of each bucket's mass: counts times the mass of the
      // bucket's smallest / largest value, widened by 2^-20 and one unit
      unsigned long long sl = 0, su = 0;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        const int b = BPT * tid + j;
        const uint32_t c = hist[swz<kBPT>(b)];
        unsigned long long lo = 0, hi = 0;
        if (c) {
          const unsigned long long m0 = mass_fixed(value_of_key<DT>((uint32_t)b << SHB), mr);
          const unsigned long long m1 = mass_fixed(value_of_key<DT>(((uint32_t)b << SHB) | ((1u << SHB) - 1u)), mr);
          lo = c * (m0 - (m0 >> 20));
          hi = c * (m1 + (m1 >> 20) + 1);
        }
        lo_m[b] = lo;
        hi_m[b] = hi;
        sl += lo;
        su += hi;
      }
      unsigned long long exl, exh, SL, SU;
      block_exclusive_scan2(sl, su, &exl, &exh, &SL, &SU, h.ws);
      // the cut's bucket lies between the first bucket whose upper-bound
      // cumulative mass passes the smallest possible target, and the first
      // whose lower-bound cumulative mass passes the largest possible one
      const unsigned long long tL = mass_target(thr, SL), tU = mass_target(thr, SU);
      if (exh <= tL && tL < exh + su) {
        unsigned long long acc = exh;
        for (int j = 0; j < BPT; ++j) {
          const int b = BPT * tid + j;
          if (tL < acc + hi_m[b]) {
            h.w0 = b;
            break;
          }
          acc += hi_m[b];
        }
      }
      if (exl <= tU && tU < exl + sl) {
        unsigned long long acc = exl;
        for (int j = 0; j < BPT; ++j) {
          const int b = BPT * tid + j;
          if (tU < acc + lo_m[b]) {
            h.w1 = b;
            break;
          }
          acc += lo_m[b];
        }
      }
      __syncthreads();
      int w0 = h.w0, w1 = h.w1;
      if (thr >= 1.0f) w0 = w1 = (int)(gmax >> SHB);  // only the last position survives
      // 16 per-key counters per window bucket: every bucket of the window in
      // order when they all fit (a counter's index is then key - first key of
      // the window), else only the occupied ones (a window that crosses zero
      // spans thousands of nearly empty buckets)
      const bool direct = w1 >= w0 && (w1 - w0 + 1) <= kKeyBlocks;
      // which of this thread's buckets get counters, decided before block_of
      // (which shares the counts' words) overwrites the counts
      uint32_t occ = 0, takes = 0;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        const int b = BPT * tid + j;
        const bool t = b >= w0 && b <= w1 && (direct || hist[swz<kBPT>(b)] != 0);
        takes |= (t ? 1u : 0u) << j;
        occ += t ? 1u : 0u;
      }
      unsigned long long nocc;
      uint32_t id = (uint32_t)block_exclusive_scan(occ, &nocc, h.ws);
      if (w1 >= w0 && nocc <= (unsigned long long)kKeyBlocks) {
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
          const int b = BPT * tid + j;
          if ((takes >> j) & 1u) {
            bucket_of[id] = (uint16_t)b;
            block_of[b] = id++;
          } else {
            block_of[b] = kNoBlock;
          }
        }
        uint4* kc4 = reinterpret_cast<uint4*>(kcount);
        for (int i = tid; i < (int)nocc * 4; i += kThreads) kc4[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        const uint32_t wkey0 = (uint32_t)w0 << SHB;
        const uint32_t nwin = (uint32_t)nocc * 16u;  // counters in use
        // pass B (from L2): row mass and mass below the window (every
        // element's fixed-point mass, so the sums equal those of the other
        // paths exactly), per-key counts inside the window.  Window membership
        // is a float compare: key order is value order.
        const float lo_f = value_of_key<DT>((uint32_t)w0 << SHB);
        unsigned long long s_mine = 0, b_mine = 0;
        const uint32_t LO2 = P::splat((uint32_t)raw_of_key<DT>((uint32_t)w0 << SHB));
        const uint32_t HI2 = P::splat((uint32_t)raw_of_key<DT>(((uint32_t)w1 << SHB) | ((1u << SHB) - 1u)));
        sweep(Loads<kLoadsHeavy>{}, ReadAs<kReadCg>{}, [&](int, const uint4& q, int nv) {
          // two values per word: one packed fma and two exponentials; the -inf
          // padding has zero mass, so no element mask is needed
          const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
          uint32_t wm[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 x = P::unpack2(wd[i]);
            const float2 e = mass2_f32(x, mr);
            const unsigned long long m0 = f2ull_rn(e.x * kMassScaleF), m1 = f2ull_rn(e.y * kMassScaleF);
            s_mine += m0 + m1;
            b_mine += (x.x < lo_f ? m0 : 0ull) + (x.y < lo_f ? m1 : 0ull);
            wm[i] = P::ge(wd[i], LO2) & ~P::gt(wd[i], HI2);
          }
          // the few elements inside the window: independent, predicated counts
          const uint32_t inwin = mask_bits<KB>(wm[0], wm[1], wm[2], wm[3]) & ((1u << nv) - 1u);
          if (inwin) {
            const uint32_t kp[4] = {order_keys2(wd[0]), order_keys2(wd[1]), order_keys2(wd[2]), order_keys2(wd[3])};
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
              if (inwin & (1u << j)) {
                const uint32_t key = (j & 1) ? (kp[j >> 1] >> 16) : (kp[j >> 1] & 0xffffu);
                const uint32_t ix = direct ? key - wkey0 : block_of[key >> SHB] * 16 + (key & 15u);
                if (ix < nwin) atomicAdd(&kcount[ix], 1u);  // always: key order is value order
              }
            }
          }
        });
        unsigned long long d0, d1, sb[2];
        block_exclusive_scan2(s_mine, b_mine, &d0, &d1, &sb[0], &sb[1], h.ws);
        cl_reduce<kClSum, 2>(cl, h.cx, cph, sb);  // (its barrier also completes every CTA's window counters)
        const unsigned long long S = sb[0], below = sb[1];
        const unsigned long long target = mass_target(thr, S);
        if (target >= S) {
          // only the last sorted position survives: the last element equal to the max
          cut_last = true;
          T = gmax;
          r0_known = false;
          done = true;
        } else if (target >= below) {
          // mass of every window key: one block per 16 lanes
          const uint32_t nblk = (uint32_t)nocc;
          for (uint32_t base = (uint32_t)warp * 2; base < nblk; base += 2 * kWarps) {
            const uint32_t blk = base + (uint32_t)(lane >> 4);
            unsigned long long m = 0;
            if (blk < nblk) {
              const uint32_t key = ((uint32_t)bucket_of[blk] << SHB) | (uint32_t)(lane & 15);
              const uint32_t c = cl_sum_at(cl, kcount, (int)(blk * 16 + (lane & 15)));
              if (c) m = (unsigned long long)c * mass_fixed(value_of_key<DT>(key), mr);
            }
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
            if (blk < nblk && (lane & 15) == 0) block_mass[blk] = m;
          }
          __syncthreads();
          unsigned long long mb[BPT], sm = 0, tot;
#pragma unroll
          for (int j = 0; j < BPT; ++j) {
            const uint32_t blk = block_of[BPT * tid + j];
            mb[j] = blk < (uint32_t)kKeyBlocks ? block_mass[blk] : 0ull;
            sm += mb[j];
          }
          const unsigned long long ex = block_exclusive_scan(sm, &tot, h.ws);
          const unsigned long long tw = target - below;  // mass of the window masked
          if (ex <= tw && tw < ex + sm) {
            unsigned long long acc = ex;
            for (int j = 0; j < BPT; ++j) {
              if (tw < acc + mb[j]) {
                const uint32_t b = (uint32_t)(BPT * tid + j);
                const int cb = (int)(block_of[b] * 16);
                for (int kk = 0; kk < 16; ++kk) {
                  const uint32_t c = cl_sum_at(cl, kcount, cb + kk);
                  if (!c) continue;
                  const uint32_t key = (b << SHB) | (uint32_t)kk;
                  const unsigned long long u = mass_fixed(value_of_key<DT>(key), mr);
                  const unsigned long long mk = (unsigned long long)c * u;
                  if (tw < acc + mk) {
                    h.sel_bin = (int)key;
                    h.sel_off = u ? (tw - acc) / u : 0ull;
                    break;
                  }
                  acc += mk;
                }
                break;
              }
              acc += mb[j];
            }
          }
          const Sel sp = finish_select(h);
          if (sp.bin >= 0) {
            T = (uint32_t)sp.bin;
            r0 = sp.off;
            done = true;
          }
        }
        cl_sync(cl);  // no peer reads this CTA's window counters any more
      }
    }

  }

  __device__ __forceinline__ void p_zero_path() {
    // ------------------------------------- top-p alone with threshold 0
    // Masked iff the cumulative mass is <= 0: exactly the elements of zero
    // fixed-point mass, the smallest values up to a key that the row max
    // alone fixes (mass grows with the key).  The first key of non-zero mass
    // is the cut, with every tie kept.  A row max that is not finite takes
    // the generic path.
    if (!done && p_zero && isfinite(value_of_key<DT>(gmax))) {
      T = block_first_true(order_key<DT>(D::kNegInf) + 1u, gmax,
                           [&](uint32_t key) { return mass_fixed(value_of_key<DT>(key), mr) > 0ull; }, &h.slot);
      r0 = 0;
      done = true;
    }

  }

  __device__ __forceinline__ void generic_path() {
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
        cl_merge<uint32_t, 2048 / 4 / kThreads>(cl, hist, 2048);
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
          cl_merge<uint32_t, 2048 / 4 / kThreads>(cl, hist, nb);
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
        cl_merge<unsigned long long, 2048 * 2 / 4 / kThreads>(cl, mass, 2048);
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
            cl_merge<unsigned long long, 2048 * 2 / 4 / kThreads>(cl, mass, nb);
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
        r0_known = false;
      }
    }

  }

  __device__ __forceinline__ void fused_sample() {
    // ---- fused sample: min-p and the exponential race on the survivors ----
    // The steps of the page aclnnTopKTopPSampleV2 (Formula / minP sampling,
    // Subsequent processing) on the filter's survivors, with the arithmetic of
    // topkp_sample: with t = (x - max) log2 e, min-p keeps t >= log2(min_p)
    // (min_p >= 1: the last sorted position alone); QSample takes the largest
    // t - log2(q + eps), ties to the larger index; without q the token is the
    // last sorted position (the largest value, of equals the largest index),
    // which every row keeps.  out, when given, holds the rows after min-p.
    const float mpv = a.min_p ? a.min_p[row] : 0.0f;
    const bool minp_on = mpv > 0.0f;
    const bool only_last = mpv >= 1.0f;
    const float* qr = a.q ? a.q + row * a.ldq : nullptr;
    const bool race_on = qr != nullptr && !only_last && a.token != nullptr;
    const float nml = -value_of_key<DT>(gmax) * 1.4426950408889634f;
    const float lmp = minp_on ? log2f(mpv) : -INFINITY;
    float bsc = -INFINITY;
    int bidx = -1;
    unsigned long long lastp = 0;  // largest (key << 32 | position): the last sorted position
    auto see_last = [&](raw r, int i) {
      const unsigned long long pk = ((unsigned long long)order_key<DT>(r) << 32) | (uint32_t)i;
      lastp = pk > lastp ? pk : lastp;
    };
    auto t_of = [&](raw r) -> float { return fmaf(D::to_float(r), 1.4426950408889634f, nml); };
    // one race candidate (score t - log2(q + eps), ties to the larger index)
    auto race = [&](float t, float qv, int i) {
      const float sc = t - __log2f(qv + a.eps);
      if (sc > bsc || (sc == bsc && i > bidx)) {
        bsc = sc;
        bidx = i;
      }
    };
    // a survivor of the filter: whether min-p keeps it, racing it if so
    auto keep_race = [&](raw r, int i) -> bool {
      const float t = t_of(r);
      if (!(t >= lmp)) return false;
      if (race_on) race(t, __ldg(qr + i), i);
      return true;
    };
    const int myn = h.fill ? (int)h.nseg[warp] : 0;
    const uint32_t tcut = h.tie_cut;
    auto listed_survivor = [&](int j) -> bool {
      const uint32_t key = order_key<DT>((raw)seg[j]);
      return key > T || (key == T && segi[j] >= tcut);
    };
    // this CTA's slice of the output row filled with -inf (rows whose
    // survivors are listed; the early fill did it already)
    auto fill_slice = [&]() {
      raw* ob = orow + e0;
      const int n = e1 - e0;
      const uintptr_t oaddr = reinterpret_cast<uintptr_t>(ob);
      const int ohead = min(n, (int)(((16u - (uint32_t)(oaddr & 15u)) & 15u) / (uint32_t)sizeof(raw)));
      const int onv = (n - ohead) / VEC;
      for (int i = tid; i < ohead; i += kThreads) ob[i] = D::kNegInf;
      uint4* ov = reinterpret_cast<uint4*>(ob + ohead);
      for (int i = tid; i < onv; i += kThreads) st_global_hint(ov + i, make_uint4(NEG2, NEG2, NEG2, NEG2), pol_first);
      for (int i = ohead + onv * VEC + tid; i < n; i += kThreads) ob[i] = D::kNegInf;
    };
    // the filter's keep rule per vector for rows that are not listed: the
    // per-warp tie counts of T, counted here when the cut did not provide them
    int rule = kKeepAll;
    unsigned long long seen = 0;
    if (!h.fill && !keepall) {
      if (!(r0_known && (r0 == 0 || have_wtie))) {
        uint32_t wn = 0;  // warp-uniform
        sweep(Loads<kLoadsSimple>{}, ReadAs<kReadCg>{}, [&](int, const uint4& q, int nv) {
          wn += __reduce_add_sync(0xffffffffu, (uint32_t)__popc(eq_bits(q, nv, T2)));
        });
        if (lane == 0) h.wtie[warp] = wn;
        __syncthreads();
        unsigned long long all_mine = 0;
        for (int w = 0; w < kWarps; ++w) all_mine += h.wtie[w];
        const unsigned long long v1[1] = {all_mine};
        unsigned long long ex1[1], tot1[1];
        cl_prefix<1>(cl, h.cx, cph, v1, ex1, tot1);
        tie_off = ex1[0];
        if (!r0_known) r0 = tot1[0] - 1ull;  // only the last sorted position survives
      }
      if (r0 == 0) {
        rule = kTiesKept;
      } else {
        unsigned long long pre = tie_off;
        for (int w = 0; w < warp; ++w) pre += h.wtie[w];
        const unsigned long long mine = h.wtie[warp];
        rule = (pre + mine <= r0) ? kTiesMasked : (pre >= r0 ? kTiesKept : kTiesStraddle);
        seen = pre;
      }
    }
    // bit j set when element j of the vector survives the filter
    auto survivor_bits = [&](const uint4& qin, int nv) -> uint32_t {
      uint32_t keep_ties = 0;
      if (rule == kTiesStraddle) {
        uint32_t tb = eq_bits(qin, nv, T2);
        const uint32_t cnt = __popc(tb);
        if (__any_sync(0xffffffffu, cnt != 0)) {
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
      }
      const uint32_t valid = (1u << nv) - 1u;
      if (rule == kKeepAll) return valid;
      uint32_t b;
      if (rule == kTiesKept) b = ge_bits(qin, nv, T2);
      else b = mask_bits<KB>(P::gt(qin.x, T2), P::gt(qin.y, T2), P::gt(qin.z, T2), P::gt(qin.w, T2)) | keep_ties;
      return b & valid;
    };
    // one vector written with the elements of `bits` kept, -inf elsewhere
    auto write_vec = [&](int e, const uint4& qin, int nv, uint32_t bits) {
      uint4 q = qin;
      q.x = (q.x & bits_word_mask<KB>(bits, 0)) | (NEG2 & ~bits_word_mask<KB>(bits, 0));
      q.y = (q.y & bits_word_mask<KB>(bits, 1)) | (NEG2 & ~bits_word_mask<KB>(bits, 1));
      q.z = (q.z & bits_word_mask<KB>(bits, 2)) | (NEG2 & ~bits_word_mask<KB>(bits, 2));
      q.w = (q.w & bits_word_mask<KB>(bits, 3)) | (NEG2 & ~bits_word_mask<KB>(bits, 3));
      if (nv == VEC && vec_out) {
        st_global_hint(orow + e, q, pol_first);
      } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
          if (j < nv) orow[e + j] = vec_elem<DT>(q, j);
      }
    };

    // A sweep that reads q with the row: x and the q of two vectors per lane
    // in flight together.  g(e, x, nv, qv, have_q) sees the vectors as in
    // sweep(); qv holds the vector's q when have_q (16-byte aligned q rows;
    // otherwise, and for the head and tail, g reads q itself).
    const bool q16 = race_on && ((reinterpret_cast<uintptr_t>(qr + head) & 15u) == 0);
    auto qsweep = [&](auto L_c, auto&& g) {
      float qnone[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) qnone[j] = 0.0f;
      if (warp == 0 && own_head) {
        const uint4 hq = load_partial(0, lane == 0 ? head : 0);
        g(0, hq, lane == 0 ? head : 0, qnone, false);
      }
      constexpr int UQ = 2;
      for (int s0 = 0; s0 < nsteps; s0 += UQ) {
        uint4 xq[UQ];
        float qv[UQ][VEC];
#pragma unroll
        for (int u = 0; u < UQ; ++u) {
          const int v = wb + (s0 + u) * 32 + lane;
          xq[u] = make_uint4(NEG2, NEG2, NEG2, NEG2);
          if (v < we) xq[u] = load_vec(L_c, xv + v);
#pragma unroll
          for (int hq = 0; hq < VEC / 4; ++hq) {
            float4 f = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (q16 && v < we) f = __ldg(reinterpret_cast<const float4*>(qr + head + v * VEC) + hq);
            qv[u][4 * hq] = f.x;
            qv[u][4 * hq + 1] = f.y;
            qv[u][4 * hq + 2] = f.z;
            qv[u][4 * hq + 3] = f.w;
          }
        }
#pragma unroll
        for (int u = 0; u < UQ; ++u) {
          if (s0 + u < nsteps) {
            const int v = wb + (s0 + u) * 32 + lane;
            g(head + v * VEC, xq[u], v < we ? VEC : 0, qv[u], q16);
          }
        }
      }
      if (warp == kWarps - 1 && own_tail) {
        const int et = head + nvec * VEC;
        const uint4 tq = load_partial(et, lane == 0 ? tail : 0);
        g(et, tq, lane == 0 ? tail : 0, qnone, false);
      }
    };
    // race the kept elements (bits) of one vector
    auto race_bits = [&](int e, const uint4& qin, uint32_t bits, const float (&qv)[VEC], bool have_q) {
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if ((bits >> j) & 1u) race(t_of(vec_elem<DT>(qin, j)), have_q ? qv[j] : __ldg(qr + e + j), e + j);
    };

    if (only_last) {
      // the last sorted position alone stays: find it, then write it
      if (h.fill) {
        for (int j = lane; j < myn; j += 32) see_last((raw)seg[j], (int)segi[j]);
      } else {
        sweep(Loads<kLoadsSimple>{}, ReadAs<kReadCg>{}, [&](int e, const uint4& q, int nv) {
#pragma unroll
          for (int j = 0; j < VEC; ++j)
            if (j < nv) see_last(vec_elem<DT>(q, j), e + j);
        });
      }
      lastp = cl_reduce1<kClMax>(cl, h.cx, cph, block_max_u64(lastp, h.ws));
      const int last = (int)(uint32_t)lastp;
      if (orow) {
        if (h.fill) {
          if (!early_fill) fill_slice();
          __syncthreads();
          for (int j = lane; j < myn; j += 32)
            if ((int)segi[j] == last) orow[last] = (raw)seg[j];
        } else {
          sweep(Loads<kLoadsSimple>{}, ReadAs<kReadLast>{}, [&](int e, const uint4& q, int nv) {
            if (nv == 0) return;
            const uint32_t bits = (last >= e && last < e + nv) ? 1u << (last - e) : 0u;
            write_vec(e, q, nv, bits);
          });
        }
      }
      if (a.token && tid == 0 && cl.rank == 0) a.token[row] = last;
      return;
    }

    if (h.fill) {
      if (orow && !early_fill) {
        fill_slice();
        __syncthreads();
      }
      // the listed survivors, four per lane at a time so their q loads overlap
      for (int j0 = lane; j0 < myn; j0 += 4 * 32) {
        float tq[4], qv[4];
        int pos[4];
        bool k[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * 32;
          k[u] = false;
          pos[u] = 0;
          tq[u] = 0.0f;
          if (j < myn && listed_survivor(j)) {
            const raw r = (raw)seg[j];
            pos[u] = (int)segi[j];
            see_last(r, pos[u]);
            tq[u] = t_of(r);
            k[u] = tq[u] >= lmp;
            if (k[u] && orow) orow[pos[u]] = r;
          }
          qv[u] = (k[u] && race_on) ? __ldg(qr + pos[u]) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (k[u] && race_on) race(tq[u], qv[u], pos[u]);
      }
    } else if (race_on) {
      // the survivors that min-p keeps race in the write sweep itself, which
      // reads q with the row (two vectors and their q in flight per lane)
      qsweep(ReadAs<kReadLast>{}, [&](int e, const uint4& qin, int nv, const float (&qv)[VEC], bool have_q) {
        const uint32_t sb = survivor_bits(qin, nv);
        uint32_t kb = 0;  // (min-p off still drops what is not >= -inf: a NaN)
#pragma unroll
        for (int j = 0; j < VEC; ++j)
          if (((sb >> j) & 1u) && t_of(vec_elem<DT>(qin, j)) >= lmp) kb |= 1u << j;
        race_bits(e, qin, kb, qv, have_q);
        if (nv != 0 && orow) write_vec(e, qin, nv, kb);
      });
    } else {
      // no race: the token is the last sorted position
      sweep(Loads<kLoadsSimple>{}, ReadAs<kReadLast>{}, [&](int e, const uint4& qin, int nv) {
        const uint32_t sb = survivor_bits(qin, nv);
        uint32_t kb = 0;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          if ((sb >> j) & 1u) {
            const raw r = vec_elem<DT>(qin, j);
            see_last(r, e + j);
            if (t_of(r) >= lmp) kb |= 1u << j;
          }
        }
        if (nv != 0 && orow) write_vec(e, qin, nv, kb);
      });
    }
    if (a.token) {
      unsigned long long pick;
      if (race_on) {
        pick = bidx < 0 ? 0ull : (((unsigned long long)float_order_key(bsc) << 32) | (uint32_t)bidx);
        pick = cl_reduce1<kClMax>(cl, h.cx, cph, block_max_u64(pick, h.ws));
      } else {
        pick = cl_reduce1<kClMax>(cl, h.cx, cph, block_max_u64(lastp, h.ws));
      }
      if (tid == 0 && cl.rank == 0) a.token[row] = (int)(uint32_t)pick;
    }

  }

  __device__ __forceinline__ void write_out() {
    // ---- write: the listed survivors over a -inf row ([guide] §2 step 8) ----
    if (h.fill) {
      if (!early_fill) {
        // this CTA's elements [e0, e1) of the output row
        raw* ob = orow + e0;
        const int n = e1 - e0;
        const uintptr_t oaddr = reinterpret_cast<uintptr_t>(ob);
        const int ohead = min(n, (int)(((16u - (uint32_t)(oaddr & 15u)) & 15u) / (uint32_t)sizeof(raw)));
        const int onv = (n - ohead) / VEC;
        for (int i = tid; i < ohead; i += kThreads) ob[i] = D::kNegInf;
        uint4* ov = reinterpret_cast<uint4*>(ob + ohead);
        for (int i = tid; i < onv; i += kThreads) st_global_hint(ov + i, make_uint4(NEG2, NEG2, NEG2, NEG2), pol_first);
        for (int i = ohead + onv * VEC + tid; i < n; i += kThreads) ob[i] = D::kNegInf;
        __syncthreads();
      }
      const int myn = (int)h.nseg[warp];
      const uint32_t tcut = h.tie_cut;
      for (int j = lane; j < myn; j += 32) {
        const raw r = (raw)seg[j];
        const uint32_t key = order_key<DT>(r);
        if (key > T || (key == T && segi[j] >= tcut)) orow[segi[j]] = r;
      }
      return;
    }

    // ---- write pass: original element or -inf, in original order ([guide] §2 step 8) ----
    // The rule per warp from the ties of T in the warps before it (h.wtie):
    // all masked, all kept, or the one warp where the cut falls ranks its ties.
    auto write_ranked = [&]() {
      int rule = kKeepAll;
      unsigned long long seen = 0;  // ties of T before this warp's next vector (straddling warp)
      if (!keepall) {
        if (r0 == 0) {
          rule = kTiesKept;
        } else {
          unsigned long long pre = tie_off;  // ties in the CTAs before this one come first
          for (int w = 0; w < warp; ++w) pre += h.wtie[w];
          const unsigned long long mine = h.wtie[warp];
          rule = (pre + mine <= r0) ? kTiesMasked : (pre >= r0 ? kTiesKept : kTiesStraddle);
          seen = pre;
        }
      }
      sweep(Loads<kLoadsSimple>{}, ReadAs<kReadLast>{}, [&](int e, const uint4& qin, int nv) {
        uint32_t keep_ties = 0;  // rule == kTiesStraddle: ties of this vector that stay
        if (rule == kTiesStraddle) {
          uint32_t tb = eq_bits(qin, nv, T2);
          const uint32_t cnt = __popc(tb);
          if (__any_sync(0xffffffffu, cnt != 0)) {
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
        }
        if (nv == 0) return;
        uint4 q = qin;
        if (rule != kKeepAll) {
          auto fix = [&](uint32_t w, int j) -> uint32_t {
            uint32_t mk;
            if (rule == kTiesKept) mk = P::ge(w, T2);
            else if (rule == kTiesMasked) mk = P::gt(w, T2);
            else mk = P::gt(w, T2) | bits_word_mask<KB>(keep_ties, j);
            return (w & mk) | (NEG2 & ~mk);
          };
          q.x = fix(q.x, 0);
          q.y = fix(q.y, 1);
          q.z = fix(q.z, 2);
          q.w = fix(q.w, 3);
        }
        if (nv == VEC && vec_out) {
          st_global_hint(orow + e, q, pol_first);
        } else {
    #pragma unroll
          for (int j = 0; j < VEC; ++j)
            if (j < nv) orow[e + j] = vec_elem<DT>(q, j);
        }
      });
    };
    const bool ranked = keepall || r0_known && (r0 == 0 || have_wtie);
    if (ranked) {
      write_ranked();
      return;
    }
    // Ties of T are written as kept while each warp records their positions,
    // in index order (lanes hold consecutive vectors, warps consecutive
    // sixteenths); the first r0 of them then become -inf.  Far too many ties
    // for the records: the counts are exact all the same, so the ranked write
    // runs again.
    constexpr int kTieCap = (int)(kApplyBigBytes / 4) / kWarps;
    uint32_t* tpos = reinterpret_cast<uint32_t*>(big) + warp * kTieCap;
    uint32_t wn = 0;  // warp-uniform
    sweep(Loads<kLoadsSimple>{}, ReadAs<kReadLast>{}, [&](int e, const uint4& qin, int nv) {
      // a packed equality test first: vectors holding a tie are rare
      const bool maybe = (P::eq(qin.x, T2) | P::eq(qin.y, T2) | P::eq(qin.z, T2) | P::eq(qin.w, T2)) != 0u;
      if (__any_sync(0xffffffffu, maybe)) {
        uint32_t tb = maybe ? eq_bits(qin, nv, T2) : 0u;
        const uint32_t cnt = __popc(tb);
        const uint32_t incl = warp_incl_scan(cnt);
        uint32_t slot = wn + incl - cnt;
        while (tb) {
          const int j = __ffs(tb) - 1;
          tb &= tb - 1;
          if (slot < (uint32_t)kTieCap) tpos[slot] = (uint32_t)(e + j);
          ++slot;
        }
        wn += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (nv == 0) return;
      uint4 q = qin;
      auto keep_ge = [&](uint32_t w) -> uint32_t {
        const uint32_t mk = P::ge(w, T2);
        return (w & mk) | (NEG2 & ~mk);
      };
      q.x = keep_ge(q.x);
      q.y = keep_ge(q.y);
      q.z = keep_ge(q.z);
      q.w = keep_ge(q.w);
      if (nv == VEC && vec_out) {
        st_global_hint(orow + e, q, pol_first);
      } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
          if (j < nv) orow[e + j] = vec_elem<DT>(q, j);
      }
    });
    if (lane == 0) h.wtie[warp] = wn;
    __syncthreads();
    unsigned long long all_mine = 0, pre = 0, overflow = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) pre += h.wtie[w];
      all_mine += h.wtie[w];
      overflow += h.wtie[w] > (uint32_t)kTieCap ? 1u : 0u;
    }
    unsigned long long all;
    {
      const unsigned long long v2[2] = {all_mine, overflow};
      unsigned long long ex2[2], tot2[2];
      cl_prefix<2>(cl, h.cx, cph, v2, ex2, tot2);
      tie_off = ex2[0];
      all = tot2[0];
      overflow = tot2[1];
    }
    pre += tie_off;
    if (!r0_known) r0 = all - 1ull;  // only the last sorted position survives: the last element equal to the max
    if (overflow) {
      write_ranked();
      return;
    }
    for (uint32_t j = lane; j < wn; j += 32)
      if (pre + j < r0) orow[tpos[j]] = D::kNegInf;
  }

  __device__ __forceinline__ void run() {
    if (keepall && in_place && !a.fused) return;  // nothing to filter, nothing to move
    init_tables();
    pass_a();
    start_early_fill();
    done = keepall;
    mr = MassRef(value_of_key<DT>(gmax));
    candidate_path();
    mass_table_path();
    window_path();
    p_zero_path();
    generic_path();
    T2 = P::splat((uint32_t)raw_of_key<DT>(T));
    __syncthreads();

    if (early_fill) {
      // the early fill has landed before any write of this row
      if (lane == 0) {
        bulk_wait_all();
        fence_proxy_async_global();
      }
      __syncthreads();
    }

    if (a.fused) {
      fused_sample();
      return;
    }
    write_out();
  }
};

template <int DT>
__device__ __forceinline__ void apply_row(const ApplyArgs& a, const int64_t row, const Clu& cl, unsigned char* smem) {
  RowFilter<DT> f(a, row, cl, smem);
  f.run();
}

// Mixed clusters: cluster c takes the c-th row without top-k while c < nd,
// the number of such rows (all CTAs of the cluster split it); after that,
// cluster c takes the rows with top-k numbered (c - nd) * cs + rank, one per
// CTA.  Rows of a kind are numbered in index order.  Returns -1 for a CTA
// whose number runs past its kind (it has no row).  The whole CTA calls
// this; scratch holds kWarps + 1 words of shared memory.
__device__ __forceinline__ int64_t mixed_row(const ApplyArgs& a, uint32_t rank, bool* split, uint32_t* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t c = blockIdx.x / (uint32_t)a.cs;
  auto dense = [&](int64_t r) -> bool {
    const int kv = a.k[r];
    return !(kv >= 1 && kv <= a.V - 1);
  };
  uint32_t n = 0;
  for (int64_t r = tid; r < a.B; r += kThreads) n += dense(r) ? 1u : 0u;
  n = __reduce_add_sync(0xffffffffu, n);
  if (lane == 0) scratch[warp] = n;
  if (tid == 0) scratch[kWarps] = 0xffffffffu;
  __syncthreads();
  int64_t nd = 0;
  for (int w = 0; w < kWarps; ++w) nd += scratch[w];
  __syncthreads();
  const bool want_dense = c < nd;
  const int64_t want = want_dense ? c : (c - nd) * a.cs + rank;
  *split = want_dense;
  int64_t seen = 0;  // rows of the wanted kind before this round
  for (int64_t base = 0; base < a.B && seen <= want; base += kThreads) {
    const int64_t r = base + tid;
    const bool m = r < a.B && dense(r) == want_dense;
    const uint32_t bal = __ballot_sync(0xffffffffu, m);
    if (lane == 0) scratch[warp] = (uint32_t)__popc(bal);
    __syncthreads();
    int64_t before = seen, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int64_t x = scratch[w];
      before += w < warp ? x : 0;
      tot += x;
    }
    if (m && before + __popc(bal & ((1u << lane) - 1u)) == want) scratch[kWarps] = (uint32_t)r;
    __syncthreads();
    seen += tot;
  }
  const uint32_t found = scratch[kWarps];
  __syncthreads();  // before the caller reuses the scratch
  return found == 0xffffffffu ? -1 : (int64_t)found;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) apply_kernel(const ApplyArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t rank = a.cs > 1 ? cluster_ctarank() : 0u;
  int64_t row = blockIdx.x / (uint32_t)a.cs;
  int cs = a.cs;
  if (a.mixed) {
    // a row with top-k reads itself once and runs on one CTA; a CTA without
    // a row leaves at once (no collective involves it)
    bool split = true;
    row = mixed_row(a, rank, &split, reinterpret_cast<uint32_t*>(smem));
    if (row < 0) return;
    if (!split) cs = 1;
  }
  // a CTA that filters a row alone owns all of it (rank 0 of a cluster of one)
  const Clu cl{cs, cs > 1 ? rank : 0u};
  apply_row<DT>(a, row, cl, smem);
  cluster_fence_exit(cl);
}

template <int DT>
static cudaError_t launch_one(const ApplyArgs& a, cudaStream_t s) {
  auto kern = apply_kernel<DT>;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kApplySmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kApplySmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cs > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_apply(topkp_dtype dt, const ApplyArgs& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return launch_one<TOPKP_F32>(a, s);
    case TOPKP_F16: return launch_one<TOPKP_F16>(a, s);
    case TOPKP_BF16: return launch_one<TOPKP_BF16>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace topkp
