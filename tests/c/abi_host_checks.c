/* A plain C caller of libwqmm.so: includes the public header, links the
 * library and exercises the host-side argument checks of several entry
 * points (none of these calls reaches the GPU).  Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "wqmm.h"

static int failures = 0;

static void expect(const char* what, int got, int want) {
  if (got != want) {
    printf("FAIL %s: got %d (%s), want %d\n", what, got, wqmm_status_string(got), want);
    ++failures;
  }
}

int main(void) {
  /* 16-byte aligned, never dereferenced: every call below is rejected (or
   * returns for an empty output) before any device access. */
  void* fake = (void*)(uintptr_t)0x10000;
  void* odd = (void*)(uintptr_t)0x10001;

  expect("version", wqmm_version(), 100);
  expect("status string", strcmp(wqmm_status_string(WQMM_ERR_MISALIGNED), "WQMM_ERR_MISALIGNED"), 0);

  expect("fp4 odd K", fp4_weight_matmul(fake, fake, fake, fake, NULL, fake, 4, 16, 31, 16,
                                        WQMM_BF16, NULL), WQMM_ERR_INVALID_ARG);
  expect("fp4 block size", fp4_weight_matmul(fake, fake, fake, fake, NULL, fake, 4, 16, 32, 24,
                                             WQMM_BF16, NULL), WQMM_ERR_UNSUPPORTED);
  expect("fp4 misaligned A", fp4_weight_matmul(odd, fake, fake, fake, NULL, fake, 4, 16, 32, 16,
                                               WQMM_BF16, NULL), WQMM_ERR_MISALIGNED);
  expect("fp4 empty", fp4_weight_matmul(NULL, fake, fake, fake, NULL, NULL, 0, 16, 32, 16,
                                        WQMM_BF16, NULL), WQMM_OK);
  expect("fp8 null scale", fp8_weight_matmul(fake, fake, NULL, NULL, fake, 4, 16, 32, 128,
                                             WQMM_FP16, NULL), WQMM_ERR_INVALID_ARG);
  expect("dequant odd K", fp4_dequantize(fake, fake, fake, fake, 4, 33, 16, WQMM_BF16, NULL),
         WQMM_ERR_INVALID_ARG);
  expect("workspace bytes", (int)fp8_w8a8_workspace_bytes(9, 32), 9 * 32 * 2);
  expect("noalloc over limit",
         fp8_weight_matmul_w8a8_noalloc(fake, fake, fake, fake, NULL, fake,
                                        (int64_t)(WQMM_NOALLOC_SCRATCH_BYTES / (2 * 4096)) + 1, 64,
                                        4096, 128, WQMM_BF16, NULL),
         WQMM_ERR_UNSUPPORTED);
  expect("fp4 x fp4 K", fp4_fp4_matmul(fake, fake, fake, fake, fake, NULL, fake, 16, 32, 48,
                                       WQMM_BF16, NULL), WQMM_ERR_UNSUPPORTED);
  expect("actq odd K", fp4_quantize_activation(fake, fake, fake, 4, 33, WQMM_BF16, NULL),
         WQMM_ERR_INVALID_ARG);
  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
