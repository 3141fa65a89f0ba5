/*
 * A plain C99 caller of librmsnorm.so, built against include/rmsnorm.h by
 * tests/test_c_abi.py: the header compiles as C (no C++ types or
 * keywords leak into it) and the library's host-side argument checks answer
 * a C program without a GPU.  Every call here fails validation or is the
 * empty batch, so no pointer below is ever dereferenced and nothing is
 * launched.  Prints "ok" and exits 0 when every expectation holds.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "rmsnorm.h"

static int failures = 0;

#define EXPECT(cond)                                              \
  do {                                                            \
    if (!(cond)) {                                                \
      fprintf(stderr, "c_abi_check.c:%d: %s\n", __LINE__, #cond); \
      ++failures;                                                 \
    }                                                             \
  } while (0)

/* Fake device addresses 16 MiB apart, never dereferenced. */
static void* fake(unsigned k) { return (void*)(uintptr_t)((uintptr_t)k << 24); }

int main(void) {
  void* x = fake(1);
  void* g = fake(2);
  void* y = fake(3);
  float* r = (float*)fake(4);
  void* dy = fake(5);
  void* dx = fake(6);
  float* dg = (float*)fake(7);
  void* ws = fake(8);
  int i, j;

  /* forward: each bad argument alone is rejected before any CUDA call */
  EXPECT(rms_fwd(NULL, g, y, r, 4, 8, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, NULL, y, r, 4, 8, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, NULL, r, 4, 8, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, y, NULL, 4, 8, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, y, r, -1, 8, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, y, r, 4, 0, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, y, r, 4, 8, -1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, y, r, 4, 8, 1e-6f, (rms_dtype)5, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd(x, g, y, r, 4, 8, 1e-6f, RMS_BF16, 2, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd_ex(x, g, y, r, 4, 8, 1e-6f, RMS_BF16, 0, (rms_path)5, NULL) ==
         RMS_ERR_INVALID_ARG);
  /* outputs may not overlap inputs: y starting 16 bytes into x */
  EXPECT(rms_fwd(x, g, (char*)x + 16, r, 4, 8, 1e-6f, RMS_BF16, 0, NULL) == RMS_ERR_INVALID_ARG);
  /* an empty batch is a no-op, pointers unused */
  EXPECT(rms_fwd(NULL, NULL, NULL, NULL, 0, 8, 1e-6f, RMS_F32, 0, NULL) == RMS_OK);

  /* backward */
  EXPECT(rms_bwd(dy, x, g, r, dx, dg, NULL, 4, 8, RMS_BF16, 0, 0, NULL) == RMS_ERR_WORKSPACE);
  EXPECT(rms_bwd(dy, x, g, r, dx, NULL, ws, 4, 8, RMS_BF16, 0, 0, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_bwd(dy, x, g, r, dx, dg, ws, 4, 8, RMS_BF16, 0, 2, NULL) == RMS_ERR_INVALID_ARG);
  /* in place: dx must be NULL or dy itself */
  EXPECT(rms_bwd(dy, x, g, r, dx, dg, ws, 4, 8, RMS_BF16, 0, 1, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_bwd_ex(dy, x, g, r, dx, dg, ws, (size_t)1 << 30, 4, 8, (rms_dtype)5, 0, 0,
                    RMS_PATH_AUTO, NULL) == RMS_ERR_INVALID_ARG);

  /* the other entry points share the checks */
  EXPECT(ln_fwd(NULL, g, NULL, y, r, r + 64, 4, 8, 1e-5f, RMS_F16, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd_quant(x, g, NULL, r, r + 64, 4, 8, 1e-6f, RMS_BF16, 0, NULL) ==
         RMS_ERR_INVALID_ARG);
  EXPECT(rms_fwd_quant_ex(x, g, (uint8_t*)y, r, r + 64, 4, 8, 1e-6f, RMS_BF16, 0,
                          RMS_PATH_STAGED, NULL) == RMS_ERR_UNSUPPORTED);
  EXPECT(rms_fwd_add(x, NULL, g, y, dy, r, 4, 8, 1e-6f, RMS_BF16, 0, NULL) ==
         RMS_ERR_INVALID_ARG);

  /* the weight-type cast of dgamma: null, size, dtype and overlap checks */
  EXPECT(rms_dgamma_cast(NULL, y, 8, RMS_BF16, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_dgamma_cast(dg, NULL, 8, RMS_BF16, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_dgamma_cast(dg, y, 0, RMS_BF16, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_dgamma_cast(dg, y, 8, (rms_dtype)5, NULL) == RMS_ERR_INVALID_ARG);
  EXPECT(rms_dgamma_cast(dg, (char*)dg + 8, 8, RMS_BF16, NULL) == RMS_ERR_INVALID_ARG);

  /* sizes of nothing need no device */
  EXPECT(rms_bwd_workspace_size(0, 8) == 0);
  EXPECT(rms_bwd_workspace_size(4, 0) == 0);

  /* every status has its own static description */
  for (i = 0; i <= RMS_ERR_TIMEOUT; ++i) {
    const char* a = rms_status_string((rms_status)i);
    EXPECT(a != NULL && a[0] != '\0');
    for (j = 0; j < i; ++j) EXPECT(strcmp(a, rms_status_string((rms_status)j)) != 0);
  }

  /* process-wide settings round-trip */
  {
    const int64_t prev = rms_set_wait_limit(123);
    EXPECT(rms_set_wait_limit(prev) == 123);
  }

  if (failures) {
    fprintf(stderr, "%d expectation(s) failed\n", failures);
    return 1;
  }
  printf("ok\n");
  return 0;
}
