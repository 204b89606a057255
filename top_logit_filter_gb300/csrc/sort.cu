// topkp_sort: the stable ascending sort of every row that comes before
// ApplyTopKTopPWithSorted in the aclnn call chain ([guide] §6.1: l0op::Sort
// with descending = false, stable = true).  Output: sorted_value (the raw
// bits, -0 and +0 included, in ascending order, equal values in increasing
// original index) and sorted_indices (int32 original positions).
//
// A least-significant-digit radix sort per row on the order keys of
// common.cuh (-0 and +0 share a key, so they stay in index order), one
// 8-bit digit per pass: 2 passes for 16-bit keys, 4 for fp32.  Passes
// alternate between the caller's workspace and the outputs so that the last
// one writes the outputs.  Every pass:
//   1. counts the row's digits (256 bins) and scans them into bucket bases;
//   2. walks the row in index order, 512 elements per tile (one per
//      thread); a warp finds the lanes holding the same digit with eight
//      ballots, the warps' per-digit counts are scanned in warp order, and
//      a running count per digit carries the earlier tiles, so every element
//      lands at base + earlier tiles + earlier warps + earlier lanes: a
//      stable counting sort on the digit.
// One 512-thread CTA per row; only shared-memory barriers, no waits.
#include "common.cuh"
#include "internal.h"

namespace topkp {

namespace {

constexpr int kDigits = 256;

// Exclusive scan of v over the first 256 threads (every thread calls it);
// returns the scan in threads 0..255.
__device__ __forceinline__ uint32_t scan256(uint32_t v, uint32_t* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (tid < kDigits && lane == 31) tmp[warp] = incl;
  __syncthreads();
  uint32_t off = 0;
  if (tid < kDigits)
    for (int w = 0; w < warp; ++w) off += tmp[w];
  __syncthreads();
  return off + incl - v;
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) sort_kernel(const SortArgs a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  constexpr int P = D::kKeyBits / 8;  // digit passes
  __shared__ uint32_t hist[kDigits];
  __shared__ uint32_t base[kDigits];
  __shared__ uint32_t running[kDigits];
  __shared__ uint32_t wcount[kWarps][kDigits];
  __shared__ uint32_t woff[kWarps][kDigits];
  __shared__ uint32_t tmp[kWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int V = a.V;
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  raw* out_v = reinterpret_cast<raw*>(a.sorted_value) + row * (int64_t)V;
  int32_t* out_i = a.sorted_indices + row * (int64_t)V;
  raw* ws_v = reinterpret_cast<raw*>(a.ws_value) + row * (int64_t)V;
  int32_t* ws_i = a.ws_index + row * (int64_t)V;
  const uint32_t lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < kWarps * kDigits; i += kThreads) (&wcount[0][0])[i] = 0;

  for (int pass = 0; pass < P; ++pass) {
    const int shift = 8 * pass;
    // the last pass writes the outputs; earlier ones alternate with the workspace
    const bool to_out = ((P - 1 - pass) & 1) == 0;
    raw* dv = to_out ? out_v : ws_v;
    int32_t* di = to_out ? out_i : ws_i;
    const raw* sv = pass == 0 ? xr : (to_out ? ws_v : out_v);
    const int32_t* si = to_out ? ws_i : out_i;  // unused in pass 0
    auto digit_of = [&](raw r) -> uint32_t { return (order_key<DT>(r) >> shift) & 255u; };

    // ---- 1. digit counts and bucket bases ----
    if (tid < kDigits) hist[tid] = 0;
    __syncthreads();
    for (int i = tid; i < V; i += kThreads) atomicAdd(&hist[digit_of(sv[i])], 1u);
    __syncthreads();
    const uint32_t hv = tid < kDigits ? hist[tid] : 0u;
    const uint32_t ex = scan256(hv, tmp);
    if (tid < kDigits) {
      base[tid] = ex;
      running[tid] = 0;
    }
    __syncthreads();

    // ---- 2. stable scatter, one element per thread per tile ----
    for (int t0 = 0; t0 < V; t0 += kThreads) {
      const int i = t0 + tid;
      const bool valid = i < V;
      raw r = 0;
      int32_t ix = 0;
      uint32_t d = 0;
      if (valid) {
        r = sv[i];
        ix = pass == 0 ? i : si[i];
        d = digit_of(r);
      }
      // lanes holding the same digit
      uint32_t peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t m = __ballot_sync(0xffffffffu, (d >> b) & 1u);
        peers &= ((d >> b) & 1u) ? m : ~m;
      }
      const uint32_t lower = __popc(peers & lt_mask);
      if (valid && lower == 0) wcount[warp][d] = __popc(peers);
      __syncthreads();
      if (tid < kDigits) {
        uint32_t acc = running[tid];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const uint32_t c = wcount[w][tid];
          woff[w][tid] = acc;
          acc += c;
          wcount[w][tid] = 0;
        }
        running[tid] = acc;
      }
      __syncthreads();
      if (valid) {
        const uint32_t pos = base[d] + woff[warp][d] + lower;
        if (pos < (uint32_t)V) {
          dv[pos] = r;
          di[pos] = ix;
        }
      }
    }
    __syncthreads();  // this pass's writes before the next pass reads them
  }
}

template <int DT>
static cudaError_t launch_sort_dt(const SortArgs& a, cudaStream_t s) {
  sort_kernel<DT><<<dim3((unsigned)a.B), dim3(kThreads), 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sort(topkp_dtype dt, const SortArgs& a, cudaStream_t s) {
  switch (dt) {
    case TOPKP_F32: return launch_sort_dt<TOPKP_F32>(a, s);
    case TOPKP_F16: return launch_sort_dt<TOPKP_F16>(a, s);
    case TOPKP_BF16: return launch_sort_dt<TOPKP_BF16>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace topkp
