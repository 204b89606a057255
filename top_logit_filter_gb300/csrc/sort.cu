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
#include <cstdio>
#include <mutex>

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
  if (a.skip_k != nullptr) {
    const int kv = a.skip_k[row];
    if (kv >= 1 && kv <= a.skip_kmax) return;  // a row the caller does not need sorted
  }
  // descending: the keys inverted, so the stable ascending order of the
  // inverted keys is the largest value first with ties in index order
  const uint32_t kinv = a.descending ? (uint32_t)((1ull << D::kKeyBits) - 1ull) : 0u;
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
    auto digit_of = [&](raw r) -> uint32_t { return ((order_key<DT>(r) ^ kinv) >> shift) & 255u; };

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

// ------------------------------------------------- sort without allocation
// topkp_sort_static: the same sort with its scratch in this library's own
// device memory.  Some callers cannot allocate device memory at the moment
// they sort: code that runs inside a memory pool it does not own, a plugin
// handed only the tensors it works on, or a host that has already reserved
// the GPU's memory for other work.  For them the scratch lives in one static
// device array that a GPU reserves when it loads this file's module (under
// CUDA's default lazy loading: at the first sort call on that device) and
// holds until the process exits.  Every call uses the same array, so calls that overlap
// on the GPU (other streams, other host threads) race on it; the sort
// overwrites all of the scratch it reads, so nothing needs clearing between
// calls.
namespace topkp {

constexpr size_t kStaticSortScratch = 16u << 20;  // bytes: the largest workspace this entry point serves
static __device__ __align__(256) unsigned char g_sort_scratch[kStaticSortScratch];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};
}  // namespace

}  // namespace topkp

extern "C" topkp_status topkp_sort_static(const void* logits, int64_t B, int64_t V, int64_t ld_logits,
                                          topkp_dtype dtype, void* sorted_value, int32_t* sorted_indices,
                                          void* stream) {
  using namespace topkp;
  report_launches(0);
  char msg[256];
  const int es = dtype == TOPKP_F32 ? 4 : ((dtype == TOPKP_F16 || dtype == TOPKP_BF16) ? 2 : 0);
  if (!es) {
    snprintf(msg, sizeof msg, "topkp_sort_static: unknown dtype %d", (int)dtype);
    return report_error(TOPKP_ERR_PARAM_INVALID, msg);
  }
  if (B < 0 || V < 0 || V > TOPKP_MAX_V) {
    snprintf(msg, sizeof msg, "topkp_sort_static: bad shape B=%lld V=%lld", (long long)B, (long long)V);
    return report_error(TOPKP_ERR_PARAM_INVALID, msg);
  }
  if (B == 0 || V == 0) return TOPKP_SUCCESS;
  const size_t need = topkp_sort_workspace_size(B, V, dtype);
  if (need > kStaticSortScratch) {
    snprintf(msg, sizeof msg,
             "topkp_sort_static: B=%lld x V=%lld needs %zu bytes of scratch, above its fixed %zu; use topkp_sort "
             "with a workspace", (long long)B, (long long)V, need, kStaticSortScratch);
    return report_error(TOPKP_ERR_PARAM_INVALID, msg);
  }
  if (!logits || !sorted_value || !sorted_indices)
    return report_error(TOPKP_ERR_PARAM_NULLPTR, "topkp_sort_static: logits or an output is NULL");
  if (ld_logits < V) return report_error(TOPKP_ERR_PARAM_INVALID, "topkp_sort_static: row stride below V");
  if ((uintptr_t)logits % es || (uintptr_t)sorted_value % es || (uintptr_t)sorted_indices % 4)
    return report_error(TOPKP_ERR_PARAM_INVALID, "topkp_sort_static: a pointer is not aligned to its element size");
  const size_t n = (size_t)B * (size_t)V;
  const uintptr_t x0 = (uintptr_t)logits, x1 = x0 + (size_t)((B - 1) * ld_logits + V) * es;
  const uintptr_t v0 = (uintptr_t)sorted_value, v1 = v0 + n * es;
  const uintptr_t i0 = (uintptr_t)sorted_indices, i1 = i0 + n * 4;
  if ((v0 < x1 && x0 < v1) || (i0 < x1 && x0 < i1) || (v0 < i1 && i0 < v1))
    return report_error(TOPKP_ERR_PARAM_INVALID, "topkp_sort_static: outputs and logits must not overlap");

  // set-up, once per device, with that device current: the scratch array's
  // device address (the symbol's host-side name is not one)
  int dev = -1;
  if (device_sms(&dev) <= 0 || dev < 0 || dev >= 64)
    return report_error(TOPKP_ERR_LAUNCH, "topkp_sort_static: no usable CUDA device");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      // loads this module on the device if it is not loaded yet, which
      // reserves the array: that can fail for want of memory
      const cudaError_t e = cudaGetSymbolAddress(&p, g_sort_scratch);
      if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        snprintf(msg, sizeof msg,
                 "topkp_sort_static: device %d is out of memory: loading the sort reserves its %zu-byte static "
                 "scratch", dev, kStaticSortScratch);
        return report_error(TOPKP_ERR_NO_MEMORY, msg);
      }
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        snprintf(msg, sizeof msg, "topkp_sort_static: cannot find the scratch array on device %d (%s)", dev,
                 cudaGetErrorString(e));
        return report_error(TOPKP_ERR_LAUNCH, msg);
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }

  SortArgs a = {};
  a.x = logits;
  a.sorted_value = sorted_value;
  a.sorted_indices = sorted_indices;
  a.ws_index = reinterpret_cast<int32_t*>(scratch);
  a.ws_value = static_cast<char*>(scratch) + (n * 4 + 255) / 256 * 256;
  a.ldx = ld_logits;
  a.B = B;  // B * V fits the scratch, so B is far below the grid limit
  a.V = (int32_t)V;
  const cudaError_t e = launch_sort(dtype, a, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(msg, sizeof msg, "topkp_sort_static: launch failed (%s)", cudaGetErrorString(e));
    return report_error(TOPKP_ERR_LAUNCH, msg);
  }
  report_launches(1);
  return TOPKP_SUCCESS;
}
