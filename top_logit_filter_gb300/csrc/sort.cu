// topkp_sort: the stable ascending sort of every row that comes before
// ApplyTopKTopPWithSorted in the aclnn call chain ([guide] §6.1: l0op::Sort
// with descending = false, stable = true).  Output: sorted_value (the raw
// bits, -0 and +0 included, in ascending order, equal values in increasing
// original index) and sorted_indices (int32 original positions).
//
// A least-significant-digit radix sort per row on the order keys of
// common.cuh (-0 and +0 share a key, so they stay in index order), 8-bit
// digits: 2 passes for 16-bit keys, 4 for fp32.  One 512-thread CTA per
// row, or (small batches) a thread-block cluster of up to eight, described
// at the kernel.  The row is read once to count every pass's digits (P
// histograms of 256 bins, scanned into bucket bases).  Then every pass walks its source in
// index order, 4096 elements per tile (eight per thread; warp w holds
// elements w*256 .. w*256+255 of the tile, lanes consecutive): a warp ranks
// each element among the earlier equal digits of its warp (one match_any finds
// the lanes with its digit) and a per-warp running count per digit; the warps'
// counts are scanned in warp order per digit, and a running count per digit
// carries the earlier tiles, so every element lands at base + earlier tiles
// + earlier warps + its rank in the warp: a stable counting sort on the
// digit.  Passes alternate between the caller's workspace and the outputs
// so that the last one writes the outputs.  Only CTA and cluster barriers,
// no waits; every scatter position is checked against V.
#include <cstdio>
#include <mutex>

#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"

namespace topkp {

namespace {

constexpr int kDigits = 256;
constexpr int kPer = 8;                        // elements per thread per tile
constexpr int kTile = kThreads * kPer;         // 4096
constexpr int kWarpSpan = 32 * kPer;           // 256 consecutive elements per warp per tile

struct SortShared {
  uint32_t base[4][kDigits];                   // bucket bases of every pass
  uint32_t running[kDigits];                   // elements of earlier tiles per digit
  uint32_t lstart[kDigits];                    // where a digit's elements start in the staged tile
  uint32_t gstart[kDigits];                    // where they go in the destination
  uint32_t wcnt[kWarps][kDigits];              // this tile's count per warp and digit
  uint32_t woff[kWarps][kDigits];              // where a warp's elements of a digit start in the stage
  uint32_t tmp[kWarps];
  uint32_t stage_v[kTile];                     // the tile ordered by digit (raw bits)
  int32_t stage_i[kTile];                      // and the elements' original indices
};

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

// A row may also run on a thread-block cluster of CS CTAs, each owning a
// contiguous slice of every pass's source: before each pass the CTAs count
// that pass's digits in their slices and read one another's counts through
// distributed shared memory, so each knows where its run of every digit
// starts (the runs of the slices before it come first, which keeps the sort
// stable); after each pass a fence and a cluster barrier make the pass's
// writes visible to the whole cluster.  Few rows then still fill the GPU.
template <int DT, int CS>
__global__ void __launch_bounds__(kThreads, 2) sort_kernel(const SortArgs a) {
  using D = DType<DT>;
  using raw = typename D::raw;
  constexpr int P = D::kKeyBits / 8;  // digit passes
  extern __shared__ __align__(16) unsigned char sort_smem[];
  SortShared& s = *reinterpret_cast<SortShared*>(sort_smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = CS > 1 ? cluster_ctarank() : 0u;
  const int64_t row = blockIdx.x / CS;
  const int V = a.V;
  if (a.skip_k != nullptr) {
    const int kv = a.skip_k[row];
    if (kv >= 1 && kv <= a.skip_kmax) return;  // a row the caller does not need sorted (the whole cluster leaves)
  }
  // this CTA's slice [s0, s1) of every pass's source
  const int chunk = (V + CS - 1) / CS;
  const int s0 = min(V, (int)rank * chunk), s1 = min(V, s0 + chunk);
  // descending: the keys inverted, so the stable ascending order of the
  // inverted keys is the largest value first with ties in index order
  const uint32_t kinv = a.descending ? (uint32_t)((1ull << D::kKeyBits) - 1ull) : 0u;
  const raw* xr = reinterpret_cast<const raw*>(a.x) + row * a.ldx;
  raw* out_v = reinterpret_cast<raw*>(a.sorted_value) + row * (int64_t)V;
  int32_t* out_i = a.sorted_indices + row * (int64_t)V;
  raw* ws_v = reinterpret_cast<raw*>(a.ws_value) + row * (int64_t)V;
  int32_t* ws_i = a.ws_index + row * (int64_t)V;
  const uint32_t lt_mask = (1u << lane) - 1u;
  auto key_of = [&](raw r) -> uint32_t { return order_key<DT>(r) ^ kinv; };

  // ---- every pass's digit counts from one read, scanned into bucket bases
  // (one CTA per row; a cluster counts each pass's source before the pass) ----
  for (int i = tid; i < 4 * kDigits; i += kThreads) (&s.base[0][0])[i] = 0;
  for (int i = tid; i < kWarps * kDigits; i += kThreads) (&s.wcnt[0][0])[i] = 0;
  __syncthreads();
  for (int i0 = 0; CS == 1 && i0 < V; i0 += kTile) {
    raw r[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + u * kThreads + tid;
      r[u] = i < V ? xr[i] : (raw)0;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      if (i0 + u * kThreads + tid < V) {
        const uint32_t key = key_of(r[u]);
#pragma unroll
        for (int p = 0; p < P; ++p) atomicAdd(&s.base[p][(key >> (8 * p)) & 255u], 1u);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const uint32_t hv = tid < kDigits ? s.base[p][tid] : 0u;
    const uint32_t ex = scan256(hv, s.tmp);
    if (tid < kDigits) s.base[p][tid] = ex;
  }
  __syncthreads();
  // a cluster's later passes read what other SMs wrote in this launch:
  // through L2 only, never a stale L1 line
  auto ld_val = [&](const raw* p, int i, int pass) -> raw { return (pass == 0 || CS == 1) ? p[i] : __ldcg(p + i); };

  for (int pass = 0; pass < P; ++pass) {
    const int shift = 8 * pass;
    // the last pass writes the outputs; earlier ones alternate with the workspace
    const bool to_out = ((P - 1 - pass) & 1) == 0;
    raw* dv = to_out ? out_v : ws_v;
    int32_t* di = to_out ? out_i : ws_i;
    const raw* sv = pass == 0 ? xr : (to_out ? ws_v : out_v);
    const int32_t* si = to_out ? ws_i : out_i;  // unused in pass 0
    if constexpr (CS > 1) {
      // this pass's digit counts in this CTA's slice of the source, and the
      // cluster's: a digit's run starts after the smaller digits' runs of the
      // whole row and this digit's runs of the slices before this one
      uint32_t* cnt = s.gstart;  // free until the tiles
      if (tid < kDigits) cnt[tid] = 0;
      __syncthreads();
      for (int i0 = s0; i0 < s1; i0 += kThreads * kPer) {
        raw r[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int i = i0 + u * kThreads + tid;
          r[u] = i < s1 ? ld_val(sv, i, pass) : (raw)0;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u)
          if (i0 + u * kThreads + tid < s1) atomicAdd(&cnt[(key_of(r[u]) >> shift) & 255u], 1u);
      }
      __syncthreads();
      cluster_sync_all();  // every CTA's counts are complete
      uint32_t tot = 0, before = 0;
      if (tid < kDigits) {
        for (int r2 = 0; r2 < CS; ++r2) {
          const uint32_t c = dsmem_ld_u32(dsmem_addr(cnt + tid, (uint32_t)r2));
          tot += c;
          before += (uint32_t)r2 < rank ? c : 0u;
        }
      }
      const uint32_t ex = scan256(tot, s.tmp);
      cluster_sync_all();  // no peer reads these counts any more
      if (tid < kDigits) s.base[pass][tid] = ex + before;
    }
    if (tid < kDigits) s.running[tid] = 0;
    __syncthreads();

    for (int t0 = s0; t0 < s1; t0 += kTile) {
      raw r[kPer];
      int32_t ix[kPer];
      uint32_t d[kPer], rk[kPer];
      const int wbase = t0 + warp * kWarpSpan;
      {
        // the next tile into L2 while this one is processed: values, then positions
        const int n0 = t0 + kTile;
        const int nv = min(kTile, s1 - n0);
        if (nv > 0) {
          const int vlines = (nv * (int)sizeof(raw) + 127) / 128;
          const int ilines = pass == 0 ? 0 : (nv * 4 + 127) / 128;
          if (tid < vlines) asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(sv + n0) + tid * 128));
          else if (tid < vlines + ilines)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(si + n0) + (tid - vlines) * 128));
        }
      }
      // every load of the tile in flight before any is used
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = wbase + u * 32 + lane;
        r[u] = 0;
        ix[u] = 0;
        if (i < s1) {
          r[u] = ld_val(sv, i, pass);
          ix[u] = pass == 0 ? i : (CS == 1 ? si[i] : __ldcg(si + i));
        }
      }
      // ---- rank every element among the earlier equal digits of its warp ----
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const bool valid = wbase + u * 32 + lane < s1;
        d[u] = valid ? (key_of(r[u]) >> shift) & 255u : 256u;  // 256: invalid lanes match only each other
        const uint32_t peers = __match_any_sync(0xffffffffu, d[u]);  // the lanes holding the same digit
        const uint32_t before = valid ? s.wcnt[warp][d[u]] : 0u;
        rk[u] = before + __popc(peers & lt_mask);
        __syncwarp();
        if (valid && (peers & lt_mask) == 0) s.wcnt[warp][d[u]] = before + __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      // ---- the tile's count per digit, scanned: where each digit's run
      // starts in the staged tile and in the destination ----
      uint32_t tc = 0;
      if (tid < kDigits) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tc += s.wcnt[w][tid];
      }
      const uint32_t ls = scan256(tc, s.tmp);
      if (tid < kDigits) {
        uint32_t acc = ls;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const uint32_t c = s.wcnt[w][tid];
          s.woff[w][tid] = acc;
          acc += c;
          s.wcnt[w][tid] = 0;
        }
        s.lstart[tid] = ls;
        s.gstart[tid] = s.base[pass][tid] + s.running[tid];
        s.running[tid] += tc;
      }
      __syncthreads();
      // ---- the tile staged in shared memory in digit order (stable) ----
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if (d[u] < 256u) {
          const uint32_t L = s.woff[warp][d[u]] + rk[u];
          s.stage_v[L] = (uint32_t)r[u];
          s.stage_i[L] = ix[u];
        }
      }
      __syncthreads();
      // ---- each digit's run written to consecutive destination positions ----
      const int tn = min(kTile, s1 - t0);
      for (int L = tid; L < tn; L += kThreads) {
        const raw rv = (raw)s.stage_v[L];
        const uint32_t dd = (key_of(rv) >> shift) & 255u;
        const uint32_t pos = s.gstart[dd] + ((uint32_t)L - s.lstart[dd]);
        if (pos < (uint32_t)V) {
          dv[pos] = rv;
          di[pos] = s.stage_i[L];
        }
      }
      __syncthreads();  // the stage is free for the next tile
    }
    if constexpr (CS > 1) {
      __threadfence();
      cluster_sync_all();  // this pass's writes, by every CTA, before the next pass reads them
    } else {
      __syncthreads();  // this pass's writes before the next pass reads them
    }
  }
}

template <int DT, int CS>
static cudaError_t launch_sort_cs(const SortArgs& a, cudaStream_t s) {
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    const cudaError_t e =
        cudaFuncSetAttribute(sort_kernel<DT, CS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SortShared));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * CS));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(SortShared);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CS > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, sort_kernel<DT, CS>, a);
}

template <int DT>
static cudaError_t launch_sort_dt(const SortArgs& a, cudaStream_t s) {
  switch (a.cs) {
    case 2: return launch_sort_cs<DT, 2>(a, s);
    case 4: return launch_sort_cs<DT, 4>(a, s);
    case 8: return launch_sort_cs<DT, 8>(a, s);
    default: return launch_sort_cs<DT, 1>(a, s);
  }
}

int sort_cluster_size(int64_t B, int num_sms) {
  int cs = 1;
  while (cs < 8 && B * (int64_t)(2 * cs) <= 2LL * num_sms) cs *= 2;
  return cs;
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
  const int sms = device_sms(&dev);
  if (sms <= 0 || dev < 0 || dev >= 64)
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
  a.B = B;  // B * V fits the scratch, so B * 8 is far below the grid limit
  a.V = (int32_t)V;
  a.cs = sort_cluster_size(B, sms);
  const cudaError_t e = launch_sort(dtype, a, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(msg, sizeof msg, "topkp_sort_static: launch failed (%s)", cudaGetErrorString(e));
    return report_error(TOPKP_ERR_LAUNCH, msg);
  }
  report_launches(1);
  return TOPKP_SUCCESS;
}
