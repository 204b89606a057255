// Host/device interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "topkp.h"

namespace topkp {

// ---------------------------------------------------------------- apply
// One CTA filters one row.  The row streams through a ring of kApplySlots
// chunk-sized slots in shared memory, filled by single large bulk copies:
// once from HBM, then again from L2 for the later passes.  Warp w handles
// the w-th sixteenth of every chunk.
struct ApplyArgs {
  const void* x;          // logits [B, ldx]
  void* out;              // out [B, ldo]
  const void* p;          // [B] dtype or nullptr
  const int32_t* k;       // [B] or nullptr
  int64_t ldx, ldo;       // row strides, elements
  int64_t B;
  int32_t V;
  int32_t chunk;          // bytes per ring slot (multiple of 8 KB)
  int32_t aligned;        // rows of x are 16-byte aligned: bulk copies / vector loads
  int32_t vec_out;        // rows of out are 16-byte aligned: vector stores
  uint64_t timeout_ns;    // limit of every bounded wait
};

struct ApplyPlan {
  int chunk = 16384;
  int ctas_per_sm = 2;
  size_t smem = 0;        // dynamic shared memory per CTA
};

// Shared memory of one apply CTA: header (mbarriers, small histograms), a
// 4096-bin histogram, a 24 KB region for the per-warp candidate lists (or
// per-warp window counts, or generic-path mass bins), then the ring.
constexpr int kApplyWarps = 16;
constexpr int kApplySlots = 4;
constexpr size_t kApplyHdrBytes = 4096;
constexpr size_t kApplyHistBytes = 4096 * 4;
constexpr size_t kApplyBigBytes = 24576;
constexpr size_t kApplyFixedSmem = kApplyHdrBytes + kApplyHistBytes + kApplyBigBytes;

inline size_t apply_smem_bytes(int chunk) { return kApplyFixedSmem + (size_t)kApplySlots * chunk; }

cudaError_t launch_apply(topkp_dtype dt, const ApplyPlan& plan, const ApplyArgs& a, cudaStream_t s);

// Chooses the ring slot size and CTAs per SM for a problem on a device with
// `num_sms` SMs and `l2_bytes` of L2.
ApplyPlan plan_apply(int64_t B, int64_t V, int esize, int num_sms, int64_t l2_bytes, const char* force);

// --------------------------------------------------------------- sorted
struct SortedArgs {
  const void* sv;          // sorted_value [B, V]
  const int32_t* si;       // sorted_indices [B, V]
  const void* logits;      // [B, V] or nullptr
  void* out;               // [B, V]
  const void* p;           // [B] or nullptr
  const int32_t* k;        // [B] or nullptr
  int64_t B;
  int32_t V;
  int32_t chunk;           // output elements per CTA
  int32_t csize;           // CTAs per row (= cluster size)
  int32_t aligned;         // logits / out rows 16-byte aligned
  uint64_t timeout_ns;
};

constexpr size_t kSortedHdrBytes = 512;

struct SortedPlan {
  int csize = 1;
  int chunk = 0;
  size_t smem = 0;
};

SortedPlan plan_sorted(int64_t B, int64_t V, int esize, int num_sms, bool with_logits, const char* force);
cudaError_t launch_sorted(topkp_dtype dt, const SortedPlan& plan, const SortedArgs& a, cudaStream_t s);

// Each kernel translation unit keeps a device error word (bit 0: a bounded
// wait gave up); these read and clear it (synchronous).
cudaError_t apply_take_device_error(unsigned int* out);
cudaError_t sorted_take_device_error(unsigned int* out);

}  // namespace topkp
