/* Plain C99 client of include/topkp.h: every entry point links, and the
 * argument checks answer with the documented status codes before any device
 * work.  Built and run by tests/test_abi_c.py (no GPU needed). */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "topkp.h"

static int failures = 0;

static void expect(const char* what, topkp_status got, topkp_status want) {
  if (got != want) {
    printf("FAIL %s: status %d, want %d (%s)\n", what, got, want, topkp_last_error_string());
    ++failures;
  }
}

int main(void) {
  /* never dereferenced: each call below is rejected by its argument checks */
  void* fake = (void*)(uintptr_t)(1u << 20);
  const int32_t* fake_k = (const int32_t*)((uintptr_t)(1u << 20) + 4096);
  void* fake_out = (void*)((uintptr_t)(1u << 20) + 8192);
  int32_t* fake_tok = (int32_t*)((uintptr_t)(1u << 20) + 12288);

  expect("apply, p and k NULL", topkp_apply(fake, 2, 8, 8, TOPKP_BF16, NULL, NULL, fake_out, 8, NULL),
         TOPKP_ERR_PARAM_NULLPTR);
  if (strstr(topkp_last_error_string(), "NULL") == NULL) {
    printf("FAIL: error string does not name the NULL argument: %s\n", topkp_last_error_string());
    ++failures;
  }
  expect("apply, bad dtype", topkp_apply(fake, 2, 8, 8, (topkp_dtype)9, NULL, fake_k, fake_out, 8, NULL),
         TOPKP_ERR_PARAM_INVALID);
  expect("apply, stride below V", topkp_apply(fake, 2, 8, 7, TOPKP_F32, NULL, fake_k, fake_out, 8, NULL),
         TOPKP_ERR_PARAM_INVALID);
  expect("apply, empty batch", topkp_apply(fake, 0, 8, 8, TOPKP_F16, NULL, fake_k, fake_out, 8, NULL),
         TOPKP_SUCCESS);
  expect("apply_sorted, NULL indices",
         topkp_apply_sorted(fake, NULL, 2, 8, TOPKP_BF16, NULL, fake_k, NULL, fake_out, NULL),
         TOPKP_ERR_PARAM_NULLPTR);
  expect("sample, no output",
         topkp_sample(fake, 2, 8, 8, TOPKP_BF16, NULL, NULL, 8, 1e-10f, NULL, 8, NULL, NULL),
         TOPKP_ERR_PARAM_NULLPTR);
  expect("sample, negative eps",
         topkp_sample(fake, 2, 8, 8, TOPKP_BF16, NULL, NULL, 8, -1.0f, NULL, 8, fake_tok, NULL),
         TOPKP_ERR_PARAM_INVALID);
  expect("sample, empty rows",
         topkp_sample(fake, 2, 0, 8, TOPKP_BF16, NULL, NULL, 8, 1e-10f, NULL, 8, fake_tok, NULL),
         TOPKP_SUCCESS);
  if (topkp_sort_workspace_size(2, 8, TOPKP_BF16) != 512u) {
    printf("FAIL: sort workspace size for 2 x 8 bf16 is %zu, want 512\n", topkp_sort_workspace_size(2, 8, TOPKP_BF16));
    ++failures;
  }
  expect("sort, workspace too small",
         topkp_sort(fake, 2, 8, 8, TOPKP_BF16, fake_out, fake_tok, (void*)((uintptr_t)(1u << 20) + 16384), 100, NULL),
         TOPKP_ERR_PARAM_INVALID);
  expect("sort_static, above its scratch",
         topkp_sort_static(fake, 64, 152064, 152064, TOPKP_BF16, fake_out, fake_tok, NULL), TOPKP_ERR_PARAM_INVALID);
  if (topkp_last_launch_count() != 0) {
    printf("FAIL: launches counted for an empty problem\n");
    ++failures;
  }
  /* topkp_sample_v2: checks before any device work */
  {
    int32_t* fake_idx = (int32_t*)((uintptr_t)(1u << 20) + 16384);
    expect("sample_v2, ks_max 0",
           topkp_sample_v2(fake, 2, 8, 8, TOPKP_BF16, fake_k, NULL, NULL, NULL, 8, 0.0f, 0, 1, NULL, 8, fake_tok,
                           NULL, NULL, fake_out, 1u << 20, NULL),
           TOPKP_ERR_PARAM_INVALID);
    expect("sample_v2, ks_max 1025",
           topkp_sample_v2(fake, 2, 8, 8, TOPKP_BF16, fake_k, NULL, NULL, NULL, 8, 0.0f, 1025, 1, NULL, 8, fake_tok,
                           NULL, NULL, fake_out, 1u << 20, NULL),
           TOPKP_ERR_PARAM_INVALID);
    expect("sample_v2, no output",
           topkp_sample_v2(fake, 2, 8, 8, TOPKP_BF16, fake_k, NULL, NULL, NULL, 8, 0.0f, 64, 1, NULL, 8, NULL, NULL,
                           NULL, fake_out, 1u << 20, NULL),
           TOPKP_ERR_PARAM_NULLPTR);
    expect("sample_v2, V above 2^20",
           topkp_sample_v2(fake, 2, (1 << 20) + 1, (1 << 20) + 1, TOPKP_F32, NULL, NULL, NULL, NULL, 8, 0.0f, 64, 1,
                           NULL, 8, fake_tok, NULL, NULL, fake_out, 1u << 20, NULL),
           TOPKP_ERR_PARAM_INVALID);
    expect("sample_v2, workspace too small",
           topkp_sample_v2(fake, 2, 8, 8, TOPKP_BF16, fake_k, NULL, NULL, NULL, 8, 0.0f, 64, 1, NULL, 8, fake_tok,
                           fake_idx, NULL, fake_out, 16, NULL),
           TOPKP_ERR_PARAM_INVALID);
    expect("sample_v2, empty batch",
           topkp_sample_v2(NULL, 0, 8, 8, TOPKP_BF16, NULL, NULL, NULL, NULL, 8, 0.0f, 64, 1, NULL, 8, fake_tok, NULL,
                           NULL, NULL, 0, NULL),
           TOPKP_SUCCESS);
    if (topkp_sample_v2_workspace_size(2, 8, TOPKP_BF16) == 0) {
      printf("FAIL: sample_v2 workspace size is 0\n");
      ++failures;
    }
  }
  if (failures == 0) printf("abi ok\n");
  return failures == 0 ? 0 : 1;
}
