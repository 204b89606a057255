// Host/device interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/topkp.h"

namespace topkp {

// ---------------------------------------------------------------- apply
// One row of logits is split into `csize` contiguous slices of `slice`
// elements; the CTAs of one thread-block cluster take one slice each and
// cooperate through distributed shared memory.
struct ApplyArgs {
  const void* x;          // logits [B, ldx]
  void* out;              // out [B, ldo]
  const void* p;          // [B] dtype or nullptr
  const int32_t* k;       // [B] or nullptr
  int64_t ldx, ldo;       // row strides, elements
  int64_t B;
  int32_t V;
  int32_t slice;          // elements per CTA (multiple of 16)
  int32_t csize;          // CTAs per row (= cluster size)
  int32_t bulk_in;        // rows of x are 16-byte aligned: bulk copies / vector loads
  int32_t vec_out;        // rows of out are 16-byte aligned: vector stores
  int32_t pad_;
  uint64_t timeout_ns;    // limit of every bounded wait
};

struct ApplyPlan {
  int csize = 1;
  int slice = 0;
  bool staged = true;
  size_t smem = 0;        // dynamic shared memory per CTA
};

constexpr int kApplyChunks = 4;       // bulk copies (and mbarriers) per slice
constexpr size_t kApplyHdrBytes = 512;
constexpr size_t kApplyFixedSmem = kApplyHdrBytes + 2048 * 4 + 2048 * 8;

inline size_t apply_smem_bytes(int slice, int esize, bool staged) {
  return kApplyFixedSmem + (staged ? ((size_t)slice * esize + 127) / 128 * 128 : 0);
}

cudaError_t launch_apply(topkp_dtype dt, const ApplyPlan& plan, const ApplyArgs& a, cudaStream_t s);

// Chooses csize / slice / staging for a problem; `num_sms` of the device.
ApplyPlan plan_apply(int64_t B, int64_t V, int esize, int num_sms, const char* force);

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
