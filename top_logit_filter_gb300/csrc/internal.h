// Host/device interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "topkp.h"

namespace topkp {

// ---------------------------------------------------------------- apply
// A cluster of cs CTAs filters one row (cs = 1: one CTA, no cluster); each
// CTA owns a contiguous slice of the row's 16-byte vectors, and warp w of a
// CTA the w-th sixteenth of its slice, read straight into registers: once
// from HBM, then again from L2 for the later passes.  Every reduction over
// the row goes through the cluster's distributed shared memory.
struct ApplyArgs {
  const void* x;          // logits [B, ldx]
  void* out;              // out [B, ldo]
  const void* p;          // [B] dtype or nullptr
  const int32_t* k;       // [B] or nullptr
  int64_t ldx, ldo;       // row strides, elements
  int64_t B;
  int32_t V;
  int32_t cs;             // CTAs per cluster (1, 2, 4 or 8)
  int32_t mixed;          // clusters take one row without top-k, or cs rows with top-k (one per CTA)
  int32_t force;          // kApplyForce* bits (testing: route rows to one path)
  // fused sample (topkp_apply_sample): min-p and the exponential race on the
  // filter's survivors; out may then be nullptr (token only)
  int32_t fused;
  const float* min_p;     // [B] or nullptr
  const float* q;         // [B, ldq] or nullptr
  int64_t ldq;
  float eps;
  int32_t* token;         // [B] or nullptr
};

// Every row that needs a cut takes the generic radix path.
constexpr int32_t kApplyForceGeneric = 1;

// Shared memory of one apply CTA: header (small histograms, scan scratch,
// cluster exchange slots), a 4096-entry table (bucket histogram, or bucket
// -> count block), a 10 KB auxiliary region (count block -> bucket, block
// masses), and a 64 KB region for the per-key count blocks (or the per-warp
// candidate lists, or the generic path's mass bins).
constexpr size_t kApplyHdrBytes = 4096;
constexpr size_t kApplyHistBytes = 4096 * 4;
constexpr size_t kApplyAuxBytes = 1024 * 2 + 1024 * 8;
constexpr size_t kApplyBigBytes = 65536;
constexpr size_t kApplySmem = kApplyHdrBytes + kApplyHistBytes + kApplyAuxBytes + kApplyBigBytes;

// Launch plan of topkp_apply for a batch of B rows of length V on num_sms
// SMs (two CTAs per SM).  Rows without top-k (top-p alone, or a copy) read
// themselves twice; rows with top-k read themselves once.  Without k every
// row is split over a cluster of cs CTAs while the split batch still runs as
// one resident wave and every slice keeps at least kApplyMinSlice elements.
// With k the clusters are mixed: a cluster takes one row without top-k,
// split over its cs CTAs, or cs rows with top-k, one per CTA; the rows
// without top-k come first.  cs is sized for up to one such row in
// kApplyDenseShare.  force (testing) may name a plan: "cN" splits every row
// over N CTAs, "mN" makes mixed clusters of N (N = 1, 2, 4, 8), alone or
// after "generic,".
constexpr int64_t kApplyMinSlice = 4096;
constexpr int64_t kApplyDenseShare = 8;
struct ApplyPlan {
  int cs = 1;
  int mixed = 0;
  int force_bits = 0;
};
ApplyPlan plan_apply(int64_t B, int64_t V, bool has_k, int num_sms, const char* force);

cudaError_t launch_apply(topkp_dtype dt, const ApplyArgs& a, cudaStream_t s);

// Short rows (small.cu): the whole row stays on chip.  Rows of at most
// kSmallSortMaxV elements (any dtype) are sorted in shared memory, one CTA
// per row; 16-bit rows of at most kSmallTableMaxV elements stay in registers
// and are counted per key, on one CTA per row or a cluster of table_cs = 2
// (while two CTAs per row still fit one per SM).  Same results as
// launch_apply, bit for bit; no fused sample.
constexpr int kSmallSortMaxV = 4096;
constexpr int kSmallTableMaxV = 32768;
constexpr size_t kSmallHdrBytes = 512;
constexpr size_t kSmallSortSmem = kSmallHdrBytes + (size_t)kSmallSortMaxV * (8 + 4 + 1);
constexpr size_t kSmallTableSmem = kSmallHdrBytes + 65536 * 2 + 4096 * (4 + 8);
// Whether a row shape takes the short-row kernels.
inline bool small_rows(topkp_dtype dt, int64_t V) {
  return V <= kSmallSortMaxV || (dt != TOPKP_F32 && V <= kSmallTableMaxV);
}
cudaError_t launch_apply_small(topkp_dtype dt, const ApplyArgs& a, int table_cs, cudaStream_t s);

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

// --------------------------------------------------------------- sample
// One CTA per filtered row: the largest element (pass 1, from HBM), then
// min-p and the exponential race over the row again (pass 2, from L2).
struct SampleArgs {
  const void* x;           // filtered [B, ldx]
  void* out;               // [B, ldo] or nullptr
  const float* min_p;      // [B] or nullptr
  const float* q;          // [B, ldq] or nullptr
  int32_t* token;          // [B] or nullptr
  int64_t ldx, ldo, ldq;
  int64_t B;
  int32_t V;
  float eps;
};

cudaError_t launch_sample(topkp_dtype dt, const SampleArgs& a, cudaStream_t s);

// ----------------------------------------------------------------- sort
// One CTA per row: a stable least-significant-digit radix sort, 8-bit
// digits, ping-ponging between the workspace and the outputs.
struct SortArgs {
  const void* x;            // logits [B, ldx]
  void* sorted_value;       // [B, V] contiguous
  int32_t* sorted_indices;  // [B, V] contiguous
  void* ws_value;           // [B, V] workspace, dtype
  int32_t* ws_index;        // [B, V] workspace, int32
  int64_t ldx;
  int64_t B;
  int32_t V;
  int32_t descending;       // largest first (equal values still in increasing index)
  const int32_t* skip_k;    // [B] or nullptr: rows with 1 <= skip_k[row] <= skip_kmax are not sorted
  int32_t skip_kmax;
  int32_t cs;               // CTAs per row (a thread-block cluster): 1, 2, 4 or 8
};

// CTAs per row of the sort for a batch of B rows on num_sms SMs: the
// largest of 1, 2, 4, 8 that keeps the batch within one wave of two CTAs
// per SM.
int sort_cluster_size(int64_t B, int num_sms);

cudaError_t launch_sort(topkp_dtype dt, const SortArgs& a, cudaStream_t s);

// --------------------------------------------------------- sample (V2)
// The TopKTopPSampleV2 semantics: rows whose top-k runs (1 <= k <=
// min(V, ks_aligned)) are filtered by one CTA each without a full sort;
// the other rows come sorted (descending) in sv / si.
struct V2Args {
  const void* x;            // logits [B, ldx]
  int64_t ldx;
  const int32_t* k;         // [B] or nullptr
  const float* p;           // [B] or nullptr
  const float* min_p;       // [B] or nullptr
  const float* q;           // [B, ldq] or nullptr
  int64_t ldq;
  float eps;
  int32_t ks_aligned;       // ks_max rounded up to a multiple of 8
  int32_t input_is_logits;
  void* select;             // [B, ld_select] dtype or nullptr
  int64_t ld_select;
  int32_t* token;           // [B] or nullptr
  int32_t* logits_idx;      // [B, V] or nullptr
  float* sort_masked;       // [B, V] or nullptr
  const void* sv;           // [B, V] sorted values (rows whose top-k is skipped)
  const int32_t* si;        // [B, V] their original indices
  int64_t B;
  int32_t V;
};

cudaError_t launch_v2(topkp_dtype dt, const V2Args& a, cudaStream_t s);

// Error and launch reporting for entry points outside api.cu (the thread's
// last error string, the last launch count), and the current device's SM
// count (-1 without a usable device).
topkp_status report_error(topkp_status code, const char* msg);
void report_launches(int n);
int device_sms(int* dev);

// The sorted-path translation unit keeps a device error word (bit 0: a
// bounded wait gave up); this reads and clears it (synchronous).
cudaError_t sorted_take_device_error(unsigned int* out);

}  // namespace topkp
