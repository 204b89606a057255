// topkp_apply for short rows: one CTA holds the whole row on chip, so the row
// is read once and every step after the load runs in registers and shared
// memory, with a handful of block-wide steps and compact code.
//
// What it computes is the eight-step formula of [guide] §2, exactly as the
// main filter kernel (apply.cu) computes it: the same order keys, the same
// per-element masses in 2^-40 fixed point relative to the row maximum, the
// same integer sums, so both reach the same cut in the stable order and
// write the same bits.
//
// Two kernels:
//   * rows of at most 4096 elements (any dtype): the row is sorted in shared
//     memory by (order key, position), a bitonic sort, which is the stable
//     ascending sort of [guide] §2 step 1; the k-th largest is read off the
//     sorted row, the masses of the survivors are scanned in sorted order,
//     and position j is kept when its cumulative mass exceeds
//     floor(round_D(1 - p) x total) or it is the last position;
//   * 16-bit rows of at most 32768 elements: every thread keeps eight
//     16-byte vectors of the row in registers, and one table of per-key
//     counts (two 16-bit counters per word, 128 KB) gives every key's exact
//     mass as count x mass(key).  The top-k threshold and the top-p cut follow
//     from two block scans over the table in descending key order; ties of
//     the cut are ranked by position from per-vector tie counts.
#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"

namespace topkp {

namespace {

constexpr int kVecPerThread = kSmallTableMaxV / kThreads / 8;  // 16-byte vectors of 16-bit elements per thread
static_assert(kVecPerThread == 8, "table kernel layout");
constexpr int kTabWords = 65536 / 2;                            // two 16-bit key counters per word

struct SmallHdr {
  unsigned long long ws[2 * kWarps];  // block-scan scratch
  unsigned long long part;            // table kernel: survivors' mass in the block holding the top-k threshold
  uint32_t maxkey;
  uint32_t kkey;                      // top-k threshold key (0: none)
  uint32_t tkey;                      // cut key
  uint32_t r0;                        // ties of the cut key masked, in index order
  uint32_t kblock;                    // table kernel: block holding the top-k threshold
  uint32_t wblk;                      // table kernel: block the warp walk takes
  uint32_t here;                      // table kernel: this CTA holds the block the walk takes
  unsigned long long wabove;          // table kernel: count or mass above the walked block
  ClSlots cx;                         // table kernel: cluster exchange slots
};

// ------------------------------------------------------------ sort kernel
// Shared memory: the header, n (key << 32 | position) entries, the row's raw
// values and one keep flag per element.
constexpr size_t kSortEntOff = kSmallHdrBytes;
constexpr size_t kSortRowOff = kSortEntOff + (size_t)kSmallSortMaxV * 8;
constexpr size_t kSortFlagOff = kSortRowOff + (size_t)kSmallSortMaxV * 4;
static_assert(8 * kThreads == kSmallSortMaxV, "every position has a thread at eight per thread");
static_assert(sizeof(SmallHdr) <= kSmallHdrBytes, "header fits");

// One bitonic stage of stride S < E on the E positions a thread holds
// (positions tid*E + r).
template <int S, int E>
__device__ __forceinline__ void sort_stage_in_thread(unsigned long long (&v)[E], int tid, int size) {
#pragma unroll
  for (int r = 0; r < E; ++r) {
    if ((r & S) == 0) {
      const bool asc = ((tid * E + r) & size) == 0;
      const unsigned long long x = v[r], y = v[r + S];
      const bool swap = (x > y) == asc;
      v[r] = swap ? y : x;
      v[r + S] = swap ? x : y;
    }
  }
}

template <int DT, int E>
__global__ void __launch_bounds__(kThreads, 1) small_sort_kernel(const ApplyArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using D = DType<DT>;
  using raw = typename D::raw;
  SmallHdr& h = *reinterpret_cast<SmallHdr*>(smem);
  unsigned long long* ent = reinterpret_cast<unsigned long long*>(smem + kSortEntOff);
  raw* rowv = reinterpret_cast<raw*>(smem + kSortRowOff);
  uint8_t* keepf = smem + kSortFlagOff;

  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int V = a.V;
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  raw* orow = reinterpret_cast<raw*>(a.out) + row * a.ldo;
  const int kv = a.k ? a.k[row] : 0;
  const bool topk = a.k != nullptr && kv >= 1 && kv <= V - 1;
  const bool topp = a.p != nullptr;
  if (!topk && !topp) {  // nothing to filter: a copy, or nothing in place
    if (reinterpret_cast<const void*>(xr) != reinterpret_cast<const void*>(orow))
      for (int i = tid; i < V; i += kThreads) orow[i] = xr[i];
    return;
  }
  const float thr = topp ? top_p_threshold<DT>(a.p, row) : 0.0f;

  // thread t holds the entries of positions E t .. E t + E - 1 (before any
  // sort: the row's elements in index order; E = the padded row / 512, at
  // least 1); keep flags start cleared
  unsigned long long v[E];
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int i = tid * E + r;
    v[r] = ~0ull;  // above every element: the padding sorts last
    if (i < V) {
      const raw x = xr[i];
      rowv[i] = x;
      keepf[i] = 0;
      v[r] = ((unsigned long long)order_key<DT>(x) << 32) | (unsigned long long)i;
    }
  }
  // the largest entry: the max key and, of equal maxima, the largest
  // position -- the last sorted position, which always survives
  unsigned long long mx = 0;
#pragma unroll
  for (int r = 0; r < E; ++r)
    if (tid * E + r < V) mx = max(mx, v[r]);
  mx = block_max_u64(mx, h.ws);
  const uint32_t maxkey = (uint32_t)(mx >> 32);
  const int lastpos = (int)(uint32_t)mx;
  const MassRef mr(value_of_key<DT>(maxkey));

  // The k-th largest key by a radix select on 8-bit digits from the top (the
  // key at sorted position V - k; ties of it survive).  ent is free until a
  // sort needs it.
  auto kth_largest = [&](int k) -> uint32_t {
    uint32_t* hist = reinterpret_cast<uint32_t*>(ent);
    uint32_t prefix = 0;
    unsigned long long rank = (unsigned long long)k;
    for (int l = 0; l < D::kKeyBits / 8; ++l) {
      const int sh = D::kKeyBits - 8 * (l + 1);
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
#pragma unroll
      for (int r = 0; r < E; ++r) {
        if (tid * E + r < V) {
          const uint32_t key = (uint32_t)(v[r] >> 32);
          if (l == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&hist[(key >> sh) & 255u], 1u);
        }
      }
      __syncthreads();
      // thread t < 256 holds digit 255 - t: a scan in descending digit order
      const unsigned long long c = tid < 256 ? hist[255 - tid] : 0ull;
      unsigned long long tot;
      const unsigned long long above = block_exclusive_scan(c, &tot, h.ws);
      if (tid < 256 && above < rank && rank <= above + c) {
        h.kkey = (uint32_t)(255 - tid);
        h.wabove = above;
      }
      __syncthreads();
      prefix = (prefix << 8) | h.kkey;
      rank -= h.wabove;
      __syncthreads();
    }
    return prefix;
  };
  // bitonic sort of the first n entries (n a power of two), ascending:
  // (key, position) is the stable order.  A stage of stride s compares
  // position i with i ^ s, ascending where i & size is 0: within a thread
  // for s < E, between the lanes of a warp for s < 32 E, through shared
  // memory beyond.  Warps past n / E hold padding only and skip the stages.
  auto sort_n = [&](int n) {
    const bool live = (tid >> 5) * 32 * E < n;  // warp-uniform
    for (int size = 2; size <= n; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        if (stride >= 32 * E) {
#pragma unroll
          for (int r = 0; r < E; ++r) ent[tid * E + r] = v[r];
          __syncthreads();
          if (live) {
#pragma unroll
            for (int r = 0; r < E; ++r) {
              const int i = tid * E + r;
              const unsigned long long y = ent[i ^ stride];
              const bool keep_min = ((i & size) == 0) == ((i & stride) == 0);
              v[r] = keep_min ? min(v[r], y) : max(v[r], y);
            }
          }
          __syncthreads();
        } else if (live) {
          if (stride >= E) {
            const int lm = stride / E;  // partner lane distance
#pragma unroll
            for (int r = 0; r < E; ++r) {
              const int i = tid * E + r;
              const unsigned long long y = __shfl_xor_sync(0xffffffffu, v[r], lm);
              const bool keep_min = ((i & size) == 0) == ((i & stride) == 0);
              v[r] = keep_min ? min(v[r], y) : max(v[r], y);
            }
          } else {
            if constexpr (E >= 8) {
              if (stride == 4) sort_stage_in_thread<4, E>(v, tid, size);
            }
            if constexpr (E >= 4) {
              if (stride == 2) sort_stage_in_thread<2, E>(v, tid, size);
            }
            if constexpr (E >= 2) {
              if (stride == 1) sort_stage_in_thread<1, E>(v, tid, size);
            }
          }
        }
      }
    }
  };

  const uint32_t kkey = topk ? kth_largest(kv) : 0u;
  if (topp && thr >= 1.0f) {
    // masked wherever the cumulative mass is <= the whole mass: everything
    // but the last sorted position
    if (tid == 0) keepf[lastpos] = 1;
  } else if (!topp || (!(thr > 0.0f) && isfinite(value_of_key<DT>(maxkey)))) {
    // top-k alone, or top-p with threshold 0: masked where the cumulative
    // mass is <= 0, that is the elements of zero mass (mass grows with the
    // value), except the last sorted position; no order is needed
#pragma unroll
    for (int r = 0; r < E; ++r) {
      const int i = tid * E + r;
      if (i < V) {
        const uint32_t key = (uint32_t)(v[r] >> 32);
        const bool keep = key >= kkey && (!topp || mass_fixed(value_of_key<DT>(key), mr) > 0ull || i == lastpos);
        keepf[i] = keep ? 1 : 0;
      }
    }
  } else {
    // the cut needs the survivors in sorted order: with top-k only the
    // elements >= the k-th largest (every other one has zero mass and stays
    // masked), gathered to the first positions
    int nc = V;
    if (topk) {
      uint32_t c = 0;
#pragma unroll
      for (int r = 0; r < E; ++r)
        if (tid * E + r < V && (uint32_t)(v[r] >> 32) >= kkey) ++c;
      unsigned long long tot;
      uint32_t base = (uint32_t)block_exclusive_scan(c, &tot, h.ws);
#pragma unroll
      for (int r = 0; r < E; ++r)
        if (tid * E + r < V && (uint32_t)(v[r] >> 32) >= kkey) ent[base++] = v[r];
      __syncthreads();
      nc = (int)tot;
#pragma unroll
      for (int r = 0; r < E; ++r) v[r] = tid * E + r < nc ? ent[tid * E + r] : ~0ull;
      __syncthreads();
    }
    int n = 1;
    while (n < nc) n <<= 1;
    sort_n(n);
    unsigned long long m[E];
    unsigned long long mine = 0;
#pragma unroll
    for (int r = 0; r < E; ++r) {
      m[r] = 0;
      const int j = tid * E + r;
      if (j < nc) {
        const uint32_t key = (uint32_t)(v[r] >> 32);
        if (key >= kkey) m[r] = mass_fixed(value_of_key<DT>(key), mr);
        mine += m[r];
      }
    }
    unsigned long long S;
    unsigned long long acc = block_exclusive_scan(mine, &S, h.ws);
    const unsigned long long target = mass_target(thr, S);
#pragma unroll
    for (int r = 0; r < E; ++r) {
      const int j = tid * E + r;
      if (j < nc) {
        const uint32_t key = (uint32_t)(v[r] >> 32);
        acc += m[r];
        // masked when the cumulative mass is <= the threshold, except the last position
        const bool keep = key >= kkey && (acc > target || j == nc - 1);
        keepf[(uint32_t)v[r]] = keep ? 1 : 0;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < V; i += kThreads) orow[i] = keepf[i] ? rowv[i] : D::kNegInf;
}

// ----------------------------------------------------------- table kernel
constexpr size_t kTabOff = kSmallHdrBytes;
constexpr int kTabBuckets = 65536 / 16;                                      // 16-key buckets
constexpr size_t kBcntOff = kTabOff + (size_t)kTabWords * 4;                 // [kTabBuckets] counts
constexpr size_t kBmassOff = kBcntOff + (size_t)kTabBuckets * 4;             // [kTabBuckets] masses

template <int DT>
__device__ __forceinline__ uint32_t half_key(uint32_t w, int j) {
  return order_key<DT>((uint16_t)(j ? (w >> 16) : (w & 0xffffu)));
}

template <int DT, int CS>
__global__ void __launch_bounds__(kThreads, 1) small_table_kernel(const ApplyArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using D = DType<DT>;
  using raw = typename D::raw;
  static_assert(D::kKeyBits == 16, "16-bit keys");
  static_assert(CS == 1 || CS == 2, "one CTA per row, or a cluster of two");
  constexpr int VPT = kVecPerThread / CS;     // 16-byte vectors per thread
  constexpr int NBH = kTabBuckets / CS;        // buckets of this CTA's key range
  constexpr int BPB = NBH / kThreads;          // buckets per thread block of keys
  constexpr int KPB = BPB * 16;                // keys per block
  constexpr int KPL = KPB / 32;                // keys per lane in a warp walk
  SmallHdr& h = *reinterpret_cast<SmallHdr*>(smem);
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + kTabOff);

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  // a cluster of CS CTAs per row: CTA r holds the r-th part of the row's
  // elements and, for the scans, key range CS - 1 - r (the highest first)
  const uint32_t rank = CS > 1 ? cluster_ctarank() : 0u;
  const Clu cl{CS, rank};
  int cph = 0;
  const uint32_t peer = rank ^ 1u;
  const uint32_t half = (uint32_t)(CS - 1) - rank;
  const int64_t row = blockIdx.x / CS;
  const int V = a.V;
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  raw* orow = reinterpret_cast<raw*>(a.out) + row * a.ldo;
  const int kv = a.k ? a.k[row] : 0;
  const bool topk = a.k != nullptr && kv >= 1 && kv <= V - 1;
  const bool topp = a.p != nullptr;
  const bool in_place = reinterpret_cast<const void*>(xr) == reinterpret_cast<const void*>(orow);
  if (!topk && !topp) {  // (the same in every CTA of the cluster: nothing shared was touched)
    if (!in_place)
      for (int i = (int)rank * kThreads + tid; i < V; i += CS * kThreads) orow[i] = xr[i];
    return;
  }
  const float thr = topp ? top_p_threshold<DT>(a.p, row) : 0.0f;
  const bool xvec = (reinterpret_cast<uintptr_t>(xr) & 15u) == 0;
  const bool ovec = (reinterpret_cast<uintptr_t>(orow) & 15u) == 0;
  const uint32_t NEG2 = (uint32_t)D::kNegInf * 0x10001u;
  // this CTA's vector u: elements 8v .. 8v+7 with v = rank * VPT * kThreads + u * kThreads + tid
  auto elem0 = [&](int u) -> int { return (((int)rank * VPT + u) * kThreads + tid) * 8; };

  // ---- load ----
  uint4 q[VPT];
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int e = elem0(u);
    q[u] = make_uint4(NEG2, NEG2, NEG2, NEG2);
    if (e + 8 <= V && xvec) {
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(q[u].x), "=r"(q[u].y), "=r"(q[u].z), "=r"(q[u].w)
                   : "l"(xr + e));
    } else if (e < V) {
      uint32_t w[4] = {NEG2, NEG2, NEG2, NEG2};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e + j < V) {
          const int sh = (j & 1) * 16;
          w[j >> 1] = (w[j >> 1] & ~(0xffffu << sh)) | ((uint32_t)xr[e + j] << sh);
        }
      q[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  // the table is cleared while the loads are in flight
  for (int i = tid; i < kTabWords / 4; i += kThreads) reinterpret_cast<uint4*>(tab)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    h.maxkey = 0;
    h.kkey = 0;
    h.kblock = 0;
    h.wblk = 0;
    h.wabove = 0;
    h.part = 0;
    h.tkey = 0;
    h.r0 = 0;
    h.here = 0;
  }
  __syncthreads();

  // ---- per-key counts of this CTA's elements, and the row max ----
  uint32_t kmax = 0;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int e = elem0(u);
    const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (e + j < V) {
        const uint32_t key = half_key<DT>(wd[j >> 1], j & 1);
        kmax = max(kmax, key);
        atomicAdd(&tab[key >> 1], (key & 1u) ? 0x10000u : 1u);
      }
    }
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) atomicMax(&h.maxkey, kmax);
  __syncthreads();
  // (its cluster barrier also completes every CTA's table)
  const uint32_t maxkey = (uint32_t)cl_reduce1<kClMax>(cl, h.cx, cph, h.maxkey);
  const MassRef mr(value_of_key<DT>(maxkey));

  // the row's count of a key: this CTA's table plus the peer's (two 16-bit
  // counters per word; a count is at most 32768, so the halves never carry)
  auto word_at = [&](int i) -> uint32_t {
    uint32_t w = tab[i];
    if (CS > 1) w += dsmem_ld_u32(dsmem_addr(tab + i, peer));
    return w;
  };
  auto count_of = [&](uint32_t key) -> uint32_t {
    const uint32_t w = word_at((int)(key >> 1));
    return (key & 1u) ? (w >> 16) : (w & 0xffffu);
  };

  // ---- per 16-key bucket of this CTA's key range its count and (top-p)
  // its mass; thread t takes buckets t, t + 512, ... so that the dense key
  // ranges spread over all threads ----
  uint32_t* bcnt = reinterpret_cast<uint32_t*>(smem + kBcntOff);
  unsigned long long* bmass = reinterpret_cast<unsigned long long*>(smem + kBmassOff);
#pragma unroll 2
  for (int i = 0; i < BPB; ++i) {
    const int b = (int)half * NBH + i * kThreads + tid;
    uint4 wa = reinterpret_cast<const uint4*>(tab)[2 * b];
    uint4 wb = reinterpret_cast<const uint4*>(tab)[2 * b + 1];
    if (CS > 1) {
      const uint4 ra = dsmem_ld_v4(dsmem_addr(reinterpret_cast<const uint4*>(tab) + 2 * b, peer));
      const uint4 rb = dsmem_ld_v4(dsmem_addr(reinterpret_cast<const uint4*>(tab) + 2 * b + 1, peer));
      wa = make_uint4(wa.x + ra.x, wa.y + ra.y, wa.z + ra.z, wa.w + ra.w);
      wb = make_uint4(wb.x + rb.x, wb.y + rb.y, wb.z + rb.z, wb.w + rb.w);
    }
    const uint32_t ww[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    uint32_t c = 0;
    unsigned long long m = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      if (ww[w]) {
        const uint32_t c0 = ww[w] & 0xffffu, c1 = ww[w] >> 16;
        c += c0 + c1;
        if (topp) {
          const uint32_t key0 = (uint32_t)b * 16u + 2u * (uint32_t)w;
          if (c0) m += (unsigned long long)c0 * mass_fixed(value_of_key<DT>(key0), mr);
          if (c1) m += (unsigned long long)c1 * mass_fixed(value_of_key<DT>(key0 + 1u), mr);
        }
      }
    }
    bcnt[b] = c;
    bmass[b] = m;
  }
  __syncthreads();
  // ---- the table in descending key order: thread t owns the BPB buckets
  // of block gblk (the highest blocks in the lowest threads, and the CTAs
  // of lower rank hold the higher key ranges) ----
  const uint32_t gblk = half * (uint32_t)kThreads + (uint32_t)(kThreads - 1 - tid);
  uint32_t cnt = 0;
  unsigned long long mass = 0;
#pragma unroll
  for (int j = 0; j < BPB; ++j) {
    cnt += bcnt[gblk * BPB + j];
    mass += bmass[gblk * BPB + j];
  }
  // Warp 0 walks block b down from its largest key, starting `above` from
  // the top: the first key at which above + the counts (or masses, keys >=
  // lo only) so far reach `goal`.  Lane l takes keys b*KPB + KPB-1 - KPL*l - i.
  // Every lane gets the key and the sum before it.
  auto warp_walk = [&](uint32_t b, unsigned long long above, unsigned long long goal, bool by_mass, uint32_t lo,
                       unsigned long long* before) -> uint32_t {
    b %= (uint32_t)(kThreads * CS);  // a block of the table
    unsigned long long v[KPL], s = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const uint32_t key = b * KPB + (KPB - 1) - KPL * (uint32_t)lane - (uint32_t)i;
      const uint32_t c = key >= lo ? count_of(key) : 0u;
      v[i] = by_mass ? (c ? (unsigned long long)c * mass_fixed(value_of_key<DT>(key), mr) : 0ull) : c;
      s += v[i];
    }
    unsigned long long incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const bool here = above + incl - s < goal && goal <= above + incl;
    const int f = __ffs(__ballot_sync(0xffffffffu, here)) - 1;
    uint32_t key = 0;
    unsigned long long acc = above + incl - s;
    if (here) {
#pragma unroll
      for (int i = 0; i < KPL; ++i) {
        if (acc + v[i] >= goal) {
          key = b * KPB + (KPB - 1) - KPL * (uint32_t)lane - (uint32_t)i;
          break;
        }
        acc += v[i];
      }
    }
    *before = __shfl_sync(0xffffffffu, acc, f < 0 ? 0 : f);
    return __shfl_sync(0xffffffffu, key, f < 0 ? 0 : f);
  };
  // a result of the CTA that walked, stored in every CTA of the cluster
  auto put32 = [&](uint32_t* field, uint32_t v) {
    *field = v;
    if (CS > 1) dsmem_st_u32(dsmem_addr(field, peer), v);
  };
  auto put64 = [&](unsigned long long* field, unsigned long long v) {
    *field = v;
    if (CS > 1) dsmem_st_u64(dsmem_addr(field, peer), v);
  };
  // exclusive scan over the cluster in descending key order: the scan within
  // the CTA plus the totals of the CTAs of lower rank
  auto scan_desc = [&](unsigned long long v, unsigned long long* total) -> unsigned long long {
    unsigned long long tot;
    const unsigned long long ex = block_exclusive_scan(v, &tot, h.ws);
    const unsigned long long t1[1] = {tot};
    unsigned long long e1[1], a1[1];
    cl_prefix<1>(cl, h.cx, cph, t1, e1, a1);
    *total = a1[0];
    return e1[0] + ex;
  };

  // ---- top-k: the k-th largest key, from the counts above each block ----
  uint32_t kkey = 0;
  if (topk) {
    unsigned long long tot;
    const unsigned long long above = scan_desc(cnt, &tot);
    if (above < (unsigned long long)kv && (unsigned long long)kv <= above + cnt) {
      h.wblk = gblk;
      h.wabove = above;
      h.here = 1;
    }
    __syncthreads();
    if (h.here && warp == 0) {
      const uint32_t b = h.wblk;
      unsigned long long before;
      const uint32_t key = warp_walk(b, h.wabove, (unsigned long long)kv, false, 0u, &before);
      unsigned long long part = 0;  // mass of the block's keys >= the threshold
      if (topp) {
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          const uint32_t kk = b * KPB + (KPB - 1) - KPL * (uint32_t)lane - (uint32_t)i;
          const uint32_t c = kk >= key ? count_of(kk) : 0u;
          if (c) part += (unsigned long long)c * mass_fixed(value_of_key<DT>(kk), mr);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      }
      if (lane == 0) {
        put32(&h.kkey, key);
        put32(&h.kblock, b);
        put64(&h.part, part);
      }
    }
    cl_sync(cl);
    __syncthreads();
    kkey = h.kkey;
    if (tid == 0) h.here = 0;
    // survivors only: blocks below the threshold's block carry no mass, and
    // that block only its keys >= the threshold
    if (gblk < h.kblock) mass = 0;
    else if (gblk == h.kblock) mass = h.part;
  }

  // ---- top-p: the cut, walking down from the largest key; an element is
  // kept while the mass strictly above it is < R = S - floor(thr x S) ----
  uint32_t T = kkey, r0 = 0;
  if (topp) {
    unsigned long long S;
    const unsigned long long above = scan_desc(mass, &S);
    const unsigned long long R = S - mass_target(thr, S);
    if (R != 0 && above < R && R <= above + mass) {
      h.wblk = gblk;
      h.wabove = above;
      h.here = 1;
    }
    __syncthreads();
    if (R == 0) {
      // only the last sorted position survives: the last element equal to the max
      T = maxkey;
      r0 = count_of(maxkey) - 1u;
    } else {
      if (h.here && warp == 0) {
        unsigned long long base;
        const uint32_t key = warp_walk(h.wblk, h.wabove, R, true, kkey, &base);
        if (lane == 0) {
          const unsigned long long u = mass_fixed(value_of_key<DT>(key), mr);
          // the (R - base) / u rounded up ties of largest positions stay
          const uint32_t c = count_of(key);
          const unsigned long long keep = u ? (R - base + u - 1) / u : (unsigned long long)c;
          put32(&h.tkey, key);
          put32(&h.r0, c - (uint32_t)min(keep, (unsigned long long)c));
        }
      }
      cl_sync(cl);
      __syncthreads();
      T = h.tkey;
      r0 = h.r0;
    }
  }

  // ---- ties of T ranked by position: index order is (CTA, u, thread, element) ----
  uint32_t tie_before[VPT];
#pragma unroll
  for (int u = 0; u < VPT; ++u) tie_before[u] = 0;
  if (r0 > 0) {
    uint32_t tc[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int e = elem0(u);
      const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
      tc[u] = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e + j < V && half_key<DT>(wd[j >> 1], j & 1) == T) ++tc[u];
    }
    // four 16-bit lanes per word: at most 8 x kThreads ties per vector round
    unsigned long long pa = 0, pb = 0;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      if (u < 4) pa |= (unsigned long long)tc[u] << (16 * u);
      else pb |= (unsigned long long)tc[u] << (16 * (u - 4));
    }
    unsigned long long ea, eb, ta, tb;
    block_exclusive_scan2(pa, pb, &ea, &eb, &ta, &tb, h.ws);
    uint32_t rounds = 0;  // ties in the earlier vector rounds of this CTA
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const unsigned long long ex = u < 4 ? ea : eb, tot = u < 4 ? ta : tb;
      const int sh = 16 * (u & 3);
      tie_before[u] = rounds + (uint32_t)((ex >> sh) & 0xffffu);
      rounds += (uint32_t)((tot >> sh) & 0xffffu);
    }
    // the CTAs before this one hold the earlier elements of the row
    const unsigned long long t1[1] = {rounds};
    unsigned long long e1[1], a1[1];
    cl_prefix<1>(cl, h.cx, cph, t1, e1, a1);
#pragma unroll
    for (int u = 0; u < VPT; ++u) tie_before[u] += (uint32_t)e1[0];
  }

  // ---- write: the element, or -inf, in original order ([guide] §2 step 8) ----
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int e = elem0(u);
    if (e >= V) continue;
    const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
    uint32_t o[4];
    uint32_t rnk = tie_before[u];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = (j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xffffu);
      const uint32_t key = order_key<DT>((uint16_t)b);
      bool keep = key > T;
      if (key == T) {
        keep = rnk >= r0;
        ++rnk;
      }
      const uint32_t ob = keep ? b : (uint32_t)D::kNegInf;
      if (j & 1) o[j >> 1] |= ob << 16;
      else o[j >> 1] = ob;
    }
    if (e + 8 <= V && ovec) {
      *reinterpret_cast<uint4*>(orow + e) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e + j < V) orow[e + j] = (raw)((j & 1) ? (o[j >> 1] >> 16) : (o[j >> 1] & 0xffffu));
    }
  }
  cluster_fence_exit(cl);  // no peer reads this CTA's table or header any more
}

template <typename K>
cudaError_t launch_small(K kern, size_t smem, const ApplyArgs& a, cudaStream_t s, int* configured_dev) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (*configured_dev != dev) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    *configured_dev = dev;
  }
  kern<<<(unsigned)a.B, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_sort_path(const ApplyArgs& a, cudaStream_t s) {
  // positions per thread: the padded row over 512 threads
  static thread_local int dev[4] = {-1, -1, -1, -1};
  if (a.V > 2048) return launch_small(small_sort_kernel<DT, 8>, kSmallSortSmem, a, s, &dev[3]);
  if (a.V > 1024) return launch_small(small_sort_kernel<DT, 4>, kSmallSortSmem, a, s, &dev[2]);
  if (a.V > 512) return launch_small(small_sort_kernel<DT, 2>, kSmallSortSmem, a, s, &dev[1]);
  return launch_small(small_sort_kernel<DT, 1>, kSmallSortSmem, a, s, &dev[0]);
}

template <int DT>
cudaError_t launch_table_path(const ApplyArgs& a, int cs, cudaStream_t s) {
  static thread_local int dev[2] = {-1, -1};
  if (cs == 1) return launch_small(small_table_kernel<DT, 1>, kSmallTableSmem, a, s, &dev[0]);
  // a cluster of two CTAs per row
  auto kern = small_table_kernel<DT, 2>;
  int d = 0;
  cudaGetDevice(&d);
  if (dev[1] != d) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallTableSmem);
    if (e != cudaSuccess) return e;
    dev[1] = d;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmallTableSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

static_assert(kSortFlagOff + kSmallSortMaxV <= kSmallSortSmem, "sort kernel shared memory");
static_assert(kBmassOff + (size_t)kTabBuckets * 8 <= kSmallTableSmem, "table kernel shared memory");

cudaError_t launch_apply_small(topkp_dtype dt, const ApplyArgs& a, int table_cs, cudaStream_t s) {
  if (a.V <= kSmallSortMaxV) {
    switch (dt) {
      case TOPKP_F32: return launch_sort_path<TOPKP_F32>(a, s);
      case TOPKP_F16: return launch_sort_path<TOPKP_F16>(a, s);
      case TOPKP_BF16: return launch_sort_path<TOPKP_BF16>(a, s);
    }
    return cudaErrorInvalidValue;
  }
  switch (dt) {
    case TOPKP_F16: return launch_table_path<TOPKP_F16>(a, table_cs, s);
    case TOPKP_BF16: return launch_table_path<TOPKP_BF16>(a, table_cs, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace topkp
