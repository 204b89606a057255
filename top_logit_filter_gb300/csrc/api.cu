// C ABI of libtopkp.so: argument checks (host only, no device sync), launch
// planning and launches.  The checks follow the order of the page's
// CheckParams ([guide] §5.3): null pointers, then dtypes, then shapes.
#include <cstdarg>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "internal.h"

namespace topkp {
namespace {

thread_local std::string g_last_error;
thread_local int g_last_launches = 0;

topkp_status fail(topkp_status code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
topkp_status fail(topkp_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int esize_of(topkp_dtype dt) {
  switch (dt) {
    case TOPKP_F32: return 4;
    case TOPKP_F16: return 2;
    case TOPKP_BF16: return 2;
  }
  return 0;
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + bn && b0 < a0 + an;
}

// Streaming multiprocessor count of the current device (cached per device).
int current_sms(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev]) {
    *dev_out = dev;
    return cache[dev];
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  *dev_out = dev;
  return sms;
}

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s for any single bounded wait
constexpr int64_t kV2MaxV = 1LL << 20;          // [V2] Constraints: 0 < vocSize <= 2^20

}  // namespace

// For entry points defined in other translation units.
topkp_status report_error(topkp_status code, const char* msg) {
  g_last_error = msg;
  return code;
}
void report_launches(int n) { g_last_launches = n; }
int device_sms(int* dev) { return current_sms(dev); }

// ------------------------------------------------------------------ planners
ApplyPlan plan_apply(int64_t B, int64_t V, bool has_k, int num_sms, const char* force) {
  ApplyPlan pl;
  int cs = 0;
  if (force && *force) {
    const char* f = force;
    if (strncmp(f, "generic", 7) == 0) {
      pl.force_bits |= kApplyForceGeneric;
      f += 7;
      if (*f == ',') ++f;
    }
    if (*f == 'c' || *f == 'm') {
      pl.mixed = *f == 'm';
      cs = atoi(f + 1);
    }
    if (cs != 1 && cs != 2 && cs != 4 && cs != 8) {
      cs = 0;
      pl.mixed = 0;
    }
  }
  if (cs == 0) {
    // one resident wave: two CTAs per SM
    const int64_t slots = 2LL * num_sms;
    cs = 1;
    if (!has_k) {
      while (cs < 8 && B * cs * 2 <= slots && V / (2 * cs) >= kApplyMinSlice) cs *= 2;
    } else {
      // mixed clusters of 2c CTAs: the dense rows take 2c CTAs each, the
      // others one, and clusters are filled
      const int64_t dense = (B + kApplyDenseShare - 1) / kApplyDenseShare;
      while (cs < 8 && dense * 2 * cs + (B - dense) + 2 * cs <= slots && V / (2 * cs) >= kApplyMinSlice) cs *= 2;
      pl.mixed = cs > 1;
    }
  }
  if (!has_k) pl.mixed = 0;  // every row is dense: plain clusters
  pl.cs = cs;
  return pl;
}

static int slice_for(int64_t V, int C) {
  const int64_t s = (V + C - 1) / C;
  return (int)((s + 15) / 16 * 16);
}

SortedPlan plan_sorted(int64_t B, int64_t V, int esize, int num_sms, bool with_logits, const char* force) {
  SortedPlan p;
  int c = 0;
  if (force && *force) sscanf(force, "%d", &c);
  if (c <= 0) {
    // one CTA per row; rows split over a cluster only when there are too
    // few rows to give every SM two CTAs (the write of a row with few
    // survivors is a fill plus a short scatter, so a CTA per row keeps the
    // latency-bound boundary search to one per row)
    c = 1;
    while (c < 8 && B * c < 2LL * num_sms && V / (c + 1) >= 2048) ++c;
  }
  if (c > 8) c = 8;
  while (c > 1 && (int64_t)(c - 1) * slice_for(V, c) >= V) --c;
  p.csize = c;
  p.chunk = slice_for(V, c);
  p.smem = kSortedHdrBytes + (with_logits ? ((size_t)p.chunk * esize + 127) / 128 * 128 : 0);
  if (p.smem > 227 * 1024) {  // very long rows: no staging
    p.smem = kSortedHdrBytes;
  }
  return p;
}

}  // namespace topkp

using namespace topkp;

extern "C" {

const char* topkp_last_error_string(void) { return g_last_error.c_str(); }

int topkp_last_launch_count(void) { return g_last_launches; }

}  // extern "C"

namespace {

// topkp_apply and topkp_apply_sample: the same checks and launch; the fused
// call adds min-p and the sample, and may leave out NULL (token only).
topkp_status apply_impl(const char* fn, const void* logits, int64_t B, int64_t V, int64_t ld_logits,
                        topkp_dtype dtype, const void* p, const int32_t* k, bool fused, const float* min_p,
                        const float* q, int64_t ldq, float eps, void* out, int64_t ld_out, int32_t* token,
                        void* stream) {
  g_last_launches = 0;
  if (!p && !k) return fail(TOPKP_ERR_PARAM_NULLPTR, "%s: p and k are both NULL (at least one is required)", fn);
  if (fused && !out && !token) return fail(TOPKP_ERR_PARAM_NULLPTR, "%s: out and token are both NULL", fn);
  const int es = esize_of(dtype);
  if (!es) return fail(TOPKP_ERR_PARAM_INVALID, "%s: unknown dtype %d", fn, (int)dtype);
  if (B < 0 || V < 0) return fail(TOPKP_ERR_PARAM_INVALID, "%s: negative shape B=%lld V=%lld", fn, (long long)B, (long long)V);
  if (V > TOPKP_MAX_V)
    return fail(TOPKP_ERR_PARAM_INVALID, "%s: V=%lld exceeds the maximum %lld", fn, (long long)V, (long long)TOPKP_MAX_V);
  if (fused && !(eps >= 0.0f)) return fail(TOPKP_ERR_PARAM_INVALID, "%s: eps must be >= 0", fn);
  if (B == 0 || V == 0) return TOPKP_SUCCESS;
  if (!logits) return fail(TOPKP_ERR_PARAM_NULLPTR, "%s: logits is NULL", fn);
  if (!out && !fused) return fail(TOPKP_ERR_PARAM_NULLPTR, "%s: out is NULL", fn);
  if (ld_logits < V || (out && ld_out < V) || (q && ldq < V))
    return fail(TOPKP_ERR_PARAM_INVALID, "%s: row stride below V (ld_logits=%lld ld_out=%lld V=%lld)", fn,
                (long long)ld_logits, (long long)ld_out, (long long)V);
  if ((uintptr_t)logits % es || (out && (uintptr_t)out % es) || (p && (uintptr_t)p % es) || (k && (uintptr_t)k % 4) ||
      (min_p && (uintptr_t)min_p % 4) || (q && (uintptr_t)q % 4) || (token && (uintptr_t)token % 4))
    return fail(TOPKP_ERR_PARAM_INVALID, "%s: a pointer is not aligned to its element size", fn);
  const size_t xbytes = (size_t)((B - 1) * ld_logits + V) * es;
  const size_t obytes = out ? (size_t)((B - 1) * ld_out + V) * es : 0;
  const size_t qbytes = q ? (size_t)((B - 1) * ldq + V) * 4 : 0;
  const bool in_place = (logits == out && ld_logits == ld_out);
  if (out && !in_place && overlaps(logits, xbytes, out, obytes))
    return fail(TOPKP_ERR_PARAM_INVALID, "%s: out partially overlaps logits", fn);
  if (overlaps(p, (size_t)B * es, out, obytes) || overlaps(k, (size_t)B * 4, out, obytes) ||
      overlaps(min_p, (size_t)B * 4, out, obytes) || overlaps(q, qbytes, out, obytes))
    return fail(TOPKP_ERR_PARAM_INVALID, "%s: out overlaps another argument", fn);
  if (token && (overlaps(token, (size_t)B * 4, logits, xbytes) || overlaps(token, (size_t)B * 4, out, obytes) ||
                overlaps(token, (size_t)B * 4, p, (size_t)B * es) || overlaps(token, (size_t)B * 4, k, (size_t)B * 4) ||
                overlaps(token, (size_t)B * 4, min_p, (size_t)B * 4) || overlaps(token, (size_t)B * 4, q, qbytes)))
    return fail(TOPKP_ERR_PARAM_INVALID, "%s: token overlaps another argument", fn);

  int dev = 0;
  const int sms = current_sms(&dev);
  if (sms <= 0) return fail(TOPKP_ERR_LAUNCH, "%s: no usable CUDA device", fn);
  ApplyArgs a = {};
  a.x = logits;
  a.out = out;
  a.p = p;
  a.k = k;
  a.ldx = ld_logits;
  a.ldo = out ? ld_out : V;
  a.V = (int32_t)V;
  // Short rows take the on-chip kernels (small.cu) unless a plan of the main
  // kernel is forced; "small" forces them wherever the shape allows, "small1"
  // / "small2" with one CTA / a cluster of two per 16-bit row counted per key.
  const char* force = getenv("TOPKP_FORCE_PLAN");
  const bool small = !fused && small_rows(dtype, V) && (!force || !*force || strncmp(force, "small", 5) == 0);
  int table_cs = 2 * B <= (int64_t)sms ? 2 : 1;  // one CTA per SM: two per row while the batch fits
  if (force && strcmp(force, "small1") == 0) table_cs = 1;
  if (force && strcmp(force, "small2") == 0) table_cs = 2;
  const ApplyPlan plan = small ? ApplyPlan{} : plan_apply(B, V, k != nullptr, sms, force);
  a.cs = plan.cs;
  a.mixed = plan.mixed;
  a.force = plan.force_bits;
  a.fused = fused ? 1 : 0;
  a.min_p = min_p;
  a.q = q;
  a.ldq = q ? ldq : V;
  a.eps = eps;
  a.token = token;
  // cs CTAs per row; grid.x must stay below 2^31
  const int64_t max_rows = INT_MAX / (small ? 2 : a.cs);
  int launches = 0;
  for (int64_t r0 = 0; r0 < B; r0 += max_rows) {
    const int64_t nb = B - r0 < max_rows ? B - r0 : max_rows;
    ApplyArgs ai = a;
    ai.B = nb;
    ai.x = (const char*)logits + r0 * ld_logits * es;
    ai.out = out ? (char*)out + r0 * ld_out * es : nullptr;
    ai.p = p ? (const char*)p + r0 * es : nullptr;
    ai.k = k ? k + r0 : nullptr;
    ai.min_p = min_p ? min_p + r0 : nullptr;
    ai.q = q ? q + r0 * ldq : nullptr;
    ai.token = token ? token + r0 : nullptr;
    const cudaError_t e = small ? launch_apply_small(dtype, ai, table_cs, (cudaStream_t)stream)
                                : launch_apply(dtype, ai, (cudaStream_t)stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(TOPKP_ERR_LAUNCH, "%s: launch failed (%s; %s, cs=%d)", fn, cudaGetErrorString(e),
                  small ? "short-row kernel" : "main kernel", a.cs);
    }
    ++launches;
  }
  g_last_launches = launches;
  return TOPKP_SUCCESS;
}

}  // namespace

extern "C" {

topkp_status topkp_apply(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                         const void* p, const int32_t* k, void* out, int64_t ld_out, void* stream) {
  return apply_impl("topkp_apply", logits, B, V, ld_logits, dtype, p, k, false, nullptr, nullptr, 0, 0.0f, out,
                    ld_out, nullptr, stream);
}

topkp_status topkp_apply_sample(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                                const void* p, const int32_t* k, const float* min_p, const float* q, int64_t ldq,
                                float eps, void* out, int64_t ld_out, int32_t* token, void* stream) {
  return apply_impl("topkp_apply_sample", logits, B, V, ld_logits, dtype, p, k, true, min_p, q, ldq, eps, out,
                    ld_out, token, stream);
}

topkp_status topkp_apply_sorted(const void* sorted_value, const int32_t* sorted_indices, int64_t B, int64_t V,
                                topkp_dtype dtype, const void* p, const int32_t* k, const void* logits, void* out,
                                void* stream) {
  g_last_launches = 0;
  if (!p && !k)
    return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_apply_sorted: p and k are both NULL (at least one is required)");
  const int es = esize_of(dtype);
  if (!es) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_apply_sorted: unknown dtype %d", (int)dtype);
  if (B < 0 || V < 0)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_apply_sorted: negative shape B=%lld V=%lld", (long long)B, (long long)V);
  if (V > TOPKP_MAX_V)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_apply_sorted: V=%lld exceeds the maximum %lld", (long long)V,
                (long long)TOPKP_MAX_V);
  if (B == 0 || V == 0) return TOPKP_SUCCESS;
  if (!sorted_value) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_apply_sorted: sorted_value is NULL");
  if (!sorted_indices) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_apply_sorted: sorted_indices is NULL");
  if (!out) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_apply_sorted: out is NULL");
  const size_t n = (size_t)(B * V);
  if (overlaps(out, n * es, sorted_value, n * es) || overlaps(out, n * es, sorted_indices, n * 4) ||
      overlaps(out, n * es, logits, n * es) || overlaps(out, n * es, p, (size_t)B * es) ||
      overlaps(out, n * es, k, (size_t)B * 4))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_apply_sorted: out overlaps an input");

  int dev = 0;
  const int sms = current_sms(&dev);
  if (sms <= 0) return fail(TOPKP_ERR_LAUNCH, "topkp_apply_sorted: no usable CUDA device");
  const SortedPlan plan = plan_sorted(B, V, es, sms, logits != nullptr, getenv("TOPKP_FORCE_SORTED_PLAN"));

  SortedArgs a = {};
  a.sv = sorted_value;
  a.si = sorted_indices;
  a.logits = logits;
  a.out = out;
  a.p = p;
  a.k = k;
  a.V = (int32_t)V;
  a.chunk = plan.chunk;
  a.csize = plan.csize;
  a.aligned = logits && plan.smem > kSortedHdrBytes && ((uintptr_t)logits % 16 == 0) && ((uintptr_t)out % 16 == 0) &&
              ((V * es) % 16 == 0);
  a.timeout_ns = kTimeoutNs;
  const int64_t max_rows = (INT_MAX / plan.csize);
  int launches = 0;
  for (int64_t r0 = 0; r0 < B; r0 += max_rows) {
    const int64_t nb = B - r0 < max_rows ? B - r0 : max_rows;
    SortedArgs ai = a;
    ai.B = nb;
    ai.sv = (const char*)sorted_value + r0 * V * es;
    ai.si = sorted_indices + r0 * V;
    ai.logits = logits ? (const char*)logits + r0 * V * es : nullptr;
    ai.out = (char*)out + r0 * V * es;
    ai.p = p ? (const char*)p + r0 * es : nullptr;
    ai.k = k ? k + r0 : nullptr;
    const cudaError_t e = launch_sorted(dtype, plan, ai, (cudaStream_t)stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(TOPKP_ERR_LAUNCH, "topkp_apply_sorted: launch failed (%s; csize=%d chunk=%d smem=%zu)",
                  cudaGetErrorString(e), plan.csize, plan.chunk, plan.smem);
    }
    ++launches;
  }
  g_last_launches = launches;
  return TOPKP_SUCCESS;
}

topkp_status topkp_sample(const void* filtered, int64_t B, int64_t V, int64_t ld, topkp_dtype dtype,
                          const float* min_p, const float* q, int64_t ldq, float eps,
                          void* out, int64_t ld_out, int32_t* token, void* stream) {
  g_last_launches = 0;
  if (!out && !token) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sample: out and token are both NULL");
  const int es = esize_of(dtype);
  if (!es) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: unknown dtype %d", (int)dtype);
  if (B < 0 || V < 0) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: negative shape B=%lld V=%lld", (long long)B, (long long)V);
  if (V > TOPKP_MAX_V)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: V=%lld exceeds the maximum %lld", (long long)V, (long long)TOPKP_MAX_V);
  if (B == 0 || V == 0) return TOPKP_SUCCESS;
  if (!filtered) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sample: filtered is NULL");
  if (ld < V || (out && ld_out < V) || (q && ldq < V))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: row stride below V (ld=%lld ld_out=%lld ldq=%lld V=%lld)",
                (long long)ld, (long long)ld_out, (long long)ldq, (long long)V);
  if (!(eps >= 0.0f)) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: eps must be >= 0");
  if ((uintptr_t)filtered % es || (out && (uintptr_t)out % es) || (min_p && (uintptr_t)min_p % 4) ||
      (q && (uintptr_t)q % 4) || (token && (uintptr_t)token % 4))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: a pointer is not aligned to its element size");
  const size_t xbytes = (size_t)((B - 1) * ld + V) * es;
  const size_t obytes = out ? (size_t)((B - 1) * ld_out + V) * es : 0;
  const size_t qbytes = q ? (size_t)((B - 1) * ldq + V) * 4 : 0;
  const bool in_place = out == filtered && ld_out == ld;
  if (out && !in_place && overlaps(filtered, xbytes, out, obytes))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: out partially overlaps filtered");
  if (overlaps(out, obytes, q, qbytes) || overlaps(out, obytes, min_p, (size_t)B * 4) ||
      overlaps(out, obytes, token, (size_t)B * 4) || overlaps(token, (size_t)B * 4, filtered, xbytes) ||
      overlaps(token, (size_t)B * 4, q, qbytes) || overlaps(token, (size_t)B * 4, min_p, (size_t)B * 4))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample: an output overlaps another argument");

  int dev = 0;
  if (current_sms(&dev) <= 0) return fail(TOPKP_ERR_LAUNCH, "topkp_sample: no usable CUDA device");

  SampleArgs a = {};
  a.x = filtered;
  a.out = out;
  a.min_p = min_p;
  a.q = q;
  a.token = token;
  a.ldx = ld;
  a.ldo = ld_out;
  a.ldq = ldq;
  a.V = (int32_t)V;
  a.eps = eps;
  const int64_t max_rows = INT_MAX;
  int launches = 0;
  for (int64_t r0 = 0; r0 < B; r0 += max_rows) {
    const int64_t nb = B - r0 < max_rows ? B - r0 : max_rows;
    SampleArgs ai = a;
    ai.B = nb;
    ai.x = (const char*)filtered + r0 * ld * es;
    ai.out = out ? (char*)out + r0 * ld_out * es : nullptr;
    ai.min_p = min_p ? min_p + r0 : nullptr;
    ai.q = q ? q + r0 * ldq : nullptr;
    ai.token = token ? token + r0 : nullptr;
    const cudaError_t e = launch_sample(dtype, ai, (cudaStream_t)stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(TOPKP_ERR_LAUNCH, "topkp_sample: launch failed (%s)", cudaGetErrorString(e));
    }
    ++launches;
  }
  g_last_launches = launches;
  return TOPKP_SUCCESS;
}

size_t topkp_sort_workspace_size(int64_t B, int64_t V, topkp_dtype dtype) {
  const int es = esize_of(dtype);
  if (!es || B <= 0 || V <= 0 || V > TOPKP_MAX_V) return 0;
  // int32 indices first (4-byte aligned), then the values, 256-byte aligned
  const size_t n = (size_t)B * (size_t)V;
  return (n * 4 + 255) / 256 * 256 + (n * es + 255) / 256 * 256;
}

topkp_status topkp_sort(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                        void* sorted_value, int32_t* sorted_indices, void* workspace, size_t workspace_bytes,
                        void* stream) {
  g_last_launches = 0;
  const int es = esize_of(dtype);
  if (!es) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: unknown dtype %d", (int)dtype);
  if (B < 0 || V < 0) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: negative shape B=%lld V=%lld", (long long)B, (long long)V);
  if (V > TOPKP_MAX_V)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: V=%lld exceeds the maximum %lld", (long long)V, (long long)TOPKP_MAX_V);
  if (B == 0 || V == 0) return TOPKP_SUCCESS;
  if (!logits) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sort: logits is NULL");
  if (!sorted_value || !sorted_indices) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sort: an output is NULL");
  if (!workspace) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sort: workspace is NULL");
  if (ld_logits < V)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: row stride %lld below V=%lld", (long long)ld_logits, (long long)V);
  const size_t need = topkp_sort_workspace_size(B, V, dtype);
  if (workspace_bytes < need)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if ((uintptr_t)logits % es || (uintptr_t)sorted_value % es || (uintptr_t)sorted_indices % 4 ||
      (uintptr_t)workspace % 256)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: a pointer is not aligned (elements; workspace 256 bytes)");
  const size_t n = (size_t)B * (size_t)V;
  const size_t xbytes = (size_t)((B - 1) * ld_logits + V) * es;
  if (overlaps(sorted_value, n * es, logits, xbytes) || overlaps(sorted_indices, n * 4, logits, xbytes) ||
      overlaps(sorted_value, n * es, sorted_indices, n * 4) || overlaps(workspace, need, logits, xbytes) ||
      overlaps(workspace, need, sorted_value, n * es) || overlaps(workspace, need, sorted_indices, n * 4))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sort: outputs, workspace and logits must not overlap");

  int dev = 0;
  const int sms = current_sms(&dev);
  if (sms <= 0) return fail(TOPKP_ERR_LAUNCH, "topkp_sort: no usable CUDA device");

  SortArgs a = {};
  a.x = logits;
  a.sorted_value = sorted_value;
  a.sorted_indices = sorted_indices;
  a.ws_index = reinterpret_cast<int32_t*>(workspace);
  a.ws_value = (char*)workspace + (n * 4 + 255) / 256 * 256;
  a.ldx = ld_logits;
  a.V = (int32_t)V;
  a.cs = sort_cluster_size(B, sms);
  const int64_t max_rows = INT_MAX / a.cs;
  int launches = 0;
  for (int64_t r0 = 0; r0 < B; r0 += max_rows) {
    const int64_t nb = B - r0 < max_rows ? B - r0 : max_rows;
    SortArgs ai = a;
    ai.B = nb;
    ai.x = (const char*)logits + r0 * ld_logits * es;
    ai.sorted_value = (char*)sorted_value + r0 * V * es;
    ai.sorted_indices = sorted_indices + r0 * V;
    ai.ws_value = (char*)a.ws_value + r0 * V * es;
    ai.ws_index = a.ws_index + r0 * V;
    const cudaError_t e = launch_sort(dtype, ai, (cudaStream_t)stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(TOPKP_ERR_LAUNCH, "topkp_sort: launch failed (%s)", cudaGetErrorString(e));
    }
    ++launches;
  }
  g_last_launches = launches;
  return TOPKP_SUCCESS;
}

size_t topkp_sample_v2_workspace_size(int64_t B, int64_t V, topkp_dtype dtype) {
  const int es = esize_of(dtype);
  if (!es || B <= 0 || V <= 0 || V > kV2MaxV) return 0;
  const size_t n = (size_t)B * (size_t)V;
  return (n * es + 255) / 256 * 256 + (n * 4 + 255) / 256 * 256 + topkp_sort_workspace_size(B, V, dtype);
}

topkp_status topkp_sample_v2(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                             const int32_t* top_k, const float* top_p, const float* min_p, const float* q,
                             int64_t ldq, float eps, int32_t ks_max, int32_t input_is_logits, void* select,
                             int64_t ld_select, int32_t* token, int32_t* logits_idx, float* sort_masked,
                             void* workspace, size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  const int es = esize_of(dtype);
  if (!es) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: unknown dtype %d", (int)dtype);
  if (B < 0 || V < 0 || V > kV2MaxV)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: bad shape B=%lld V=%lld (0 <= V <= 2^20)", (long long)B,
                (long long)V);
  if (ks_max < 1 || ks_max > 1024)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: ks_max=%d outside [1, 1024]", (int)ks_max);
  if (!(eps >= 0.0f)) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: eps must be >= 0");
  if (!select && !token && !logits_idx && !sort_masked)
    return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sample_v2: no output given");
  if (B == 0 || V == 0) return TOPKP_SUCCESS;
  if (!logits) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sample_v2: logits is NULL");
  if (!workspace) return fail(TOPKP_ERR_PARAM_NULLPTR, "topkp_sample_v2: workspace is NULL");
  if (ld_logits < V || (select && ld_select < V) || (q && ldq < V))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: a row stride is below V");
  const size_t need = topkp_sample_v2_workspace_size(B, V, dtype);
  if (workspace_bytes < need)
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if ((uintptr_t)logits % es || (select && (uintptr_t)select % es) || (uintptr_t)workspace % 256 ||
      (top_k && (uintptr_t)top_k % 4) || (top_p && (uintptr_t)top_p % 4) || (min_p && (uintptr_t)min_p % 4) ||
      (q && (uintptr_t)q % 4) || (token && (uintptr_t)token % 4) || (logits_idx && (uintptr_t)logits_idx % 4) ||
      (sort_masked && (uintptr_t)sort_masked % 4))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: a pointer is not aligned (elements; workspace 256 bytes)");
  const size_t n = (size_t)B * (size_t)V;
  const size_t xb = (size_t)((B - 1) * ld_logits + V) * es;
  const size_t sb = select ? (size_t)((B - 1) * ld_select + V) * es : 0;
  const size_t qb = q ? (size_t)((B - 1) * ldq + V) * 4 : 0;
  const void* outs[4] = {select, token, logits_idx, sort_masked};
  const size_t osz[4] = {sb, (size_t)B * 4, n * 4, n * 4};
  const void* ins[6] = {logits, top_k, top_p, min_p, q, workspace};
  const size_t isz[6] = {xb, (size_t)B * 4, (size_t)B * 4, (size_t)B * 4, qb, need};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 6; ++j)
      if (outs[i] && overlaps(outs[i], osz[i], ins[j], isz[j]))
        return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: an output overlaps an input or the workspace");
    for (int j = i + 1; j < 4; ++j)
      if (outs[i] && outs[j] && overlaps(outs[i], osz[i], outs[j], osz[j]))
        return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: two outputs overlap");
  }
  if (overlaps(workspace, need, logits, xb) || overlaps(workspace, need, q, qb))
    return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: the workspace overlaps an input");
  int dev = 0;
  if (current_sms(&dev) <= 0) return fail(TOPKP_ERR_LAUNCH, "topkp_sample_v2: no usable CUDA device");
  if (B > INT_MAX) return fail(TOPKP_ERR_PARAM_INVALID, "topkp_sample_v2: B above 2^31 - 1");

  // workspace: sorted values, their indices, then the sort's own scratch
  char* w = (char*)workspace;
  void* sv = w;
  int32_t* si = reinterpret_cast<int32_t*>(w + (n * es + 255) / 256 * 256);
  char* scratch = w + (n * es + 255) / 256 * 256 + (n * 4 + 255) / 256 * 256;
  const int ks_aligned = (ks_max + 7) / 8 * 8 > 1024 ? 1024 : (ks_max + 7) / 8 * 8;

  // 1. the rows whose top-k is skipped, sorted from the largest value down
  SortArgs sa = {};
  sa.x = logits;
  sa.sorted_value = sv;
  sa.sorted_indices = si;
  sa.ws_index = reinterpret_cast<int32_t*>(scratch);
  sa.ws_value = scratch + (n * 4 + 255) / 256 * 256;
  sa.ldx = ld_logits;
  sa.B = B;
  sa.V = (int32_t)V;
  sa.descending = 1;
  sa.skip_k = top_k;
  sa.skip_kmax = (int32_t)(V < ks_aligned ? V : ks_aligned);
  // few rows skip top-k, so each is sorted by a cluster of eight CTAs (the
  // clusters of the other rows leave at once)
  sa.cs = B <= INT_MAX / 8 ? 8 : 1;
  cudaError_t e = launch_sort(dtype, sa, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TOPKP_ERR_LAUNCH, "topkp_sample_v2: sort launch failed (%s)", cudaGetErrorString(e));
  }
  // 2. the filter stages and the sample
  V2Args a = {};
  a.x = logits;
  a.ldx = ld_logits;
  a.k = top_k;
  a.p = top_p;
  a.min_p = min_p;
  a.q = q;
  a.ldq = ldq;
  a.eps = eps;
  a.ks_aligned = ks_aligned;
  a.input_is_logits = input_is_logits ? 1 : 0;
  a.select = select;
  a.ld_select = ld_select;
  a.token = token;
  a.logits_idx = logits_idx;
  a.sort_masked = sort_masked;
  a.sv = sv;
  a.si = si;
  a.B = B;
  a.V = (int32_t)V;
  e = launch_v2(dtype, a, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TOPKP_ERR_LAUNCH, "topkp_sample_v2: launch failed (%s)", cudaGetErrorString(e));
  }
  g_last_launches = 3;
  return TOPKP_SUCCESS;
}

topkp_status topkp_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TOPKP_ERR_LAUNCH, "topkp_device_status: stream error: %s", cudaGetErrorString(e));
  }
  unsigned int w = 0;
  e = sorted_take_device_error(&w);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TOPKP_ERR_LAUNCH, "topkp_device_status: cannot read the device error word: %s", cudaGetErrorString(e));
  }
  if (w) return fail(TOPKP_ERR_DEVICE_TIMEOUT, "topkp_device_status: a kernel gave up a bounded wait");
  return TOPKP_SUCCESS;
}

}  // extern "C"
