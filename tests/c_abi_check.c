/*
 * c_abi_check.c -- a plain C11 client of libgdn.so, built against include/gdn.h alone (the
 * hooks of include/gdn_debug.h exist only in the test build, libgdn_test.so).  It calls only paths that end in host-side validation or pure host
 * arithmetic (no CUDA call is reached), so it runs without a GPU; tests/test_abi.py compiles it
 * with gcc -std=c11 -Wall -Wextra -Werror and expects it to print "ok".
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn.h"

#define EXPECT(expr, want)                                                                       \
  do {                                                                                           \
    const gdn_status got_ = (expr);                                                              \
    if (got_ != (want)) {                                                                        \
      fprintf(stderr, "line %d: %s returned %s, expected %s (%s)\n", __LINE__, #expr,           \
              gdn_status_string(got_), gdn_status_string(want), gdn_last_error_message());      \
      return 1;                                                                                  \
    }                                                                                            \
  } while (0)

int main(void) {
  const gdn_geometry geo = {16, 48, 128, 128, 4};
  const gdn_geometry kda = {64, 64, 128, 128, 4};
  const gdn_geometry uneven = {16, 40, 128, 128, 4}; /* Hv not a multiple of Hk */
  const gdn_geometry narrow = {16, 48, 64, 128, 4};  /* Dk other than 128 */
  /* 16-byte aligned and 2-byte aligned addresses that are never dereferenced */
  void* fake = (void*)(uintptr_t)0x10000;
  void* odd = (void*)(uintptr_t)0x10002;

  if (strncmp(gdn_version(), "gdn-gb300", 9) != 0) return 1;
  if (strcmp(gdn_status_string(GDN_ERR_MISALIGNED), "GDN_ERR_MISALIGNED") != 0) return 1;

  /* geometry and size checks */
  EXPECT(gdn_conv1d_prefill(&uneven, fake, fake, fake, 1, 4, NULL, NULL, fake, NULL), GDN_ERR_UNSUPPORTED_GEOMETRY);
  EXPECT(gdn_conv1d_prefill(&narrow, fake, fake, fake, 1, 4, NULL, NULL, fake, NULL), GDN_ERR_UNSUPPORTED_GEOMETRY);
  EXPECT(gdn_conv1d_prefill(&geo, fake, fake, fake, 0, 4, NULL, NULL, fake, NULL), GDN_ERR_INVALID_ARGUMENT);
  EXPECT(gdn_chunk_prefill(&geo, fake, fake, fake, fake, -1, 16, 0.088f, 1e-6f, NULL, NULL, NULL, NULL, 1e-6f,
                           fake, NULL, 0, NULL),
         GDN_ERR_INVALID_ARGUMENT);
  EXPECT(gdn_gated_rmsnorm(&geo, fake, fake, fake, 1e-6f, fake, -1, NULL), GDN_ERR_INVALID_ARGUMENT);
  EXPECT(gdn_gates(&geo, fake, fake, fake, fake, fake, fake, -1, NULL), GDN_ERR_INVALID_ARGUMENT);

  /* alignment */
  EXPECT(gdn_decode_step(&geo, odd, fake, fake, fake, fake, fake, fake, fake, 0.088f, 1e-6f, 1e-6f, fake, 4, NULL),
         GDN_ERR_MISALIGNED);
  EXPECT(gdn_kda_decode_step(&kda, fake, fake, fake, odd, -1.0f, fake, fake, fake, fake, 0.088f, 1e-6f, 1e-6f, fake,
                             4, NULL),
         GDN_ERR_MISALIGNED);

  /* argument values */
  EXPECT(gdn_kda_recurrence(&kda, fake, fake, NAN, fake, fake, 2, 8, 0.088f, 1e-6f, NULL, NULL, NULL, NULL, 1e-6f,
                            fake, NULL),
         GDN_ERR_INVALID_ARGUMENT);
  EXPECT(gdn_verify(&geo, fake, fake, fake, fake, fake, fake, fake, fake, 0.088f, 1e-6f, 1e-6f, fake, 4, 18, fake,
                    1u << 30, NULL),
         GDN_ERR_INVALID_ARGUMENT);
  EXPECT(gdn_verify_commit(&geo, fake, fake, (size_t)1 << 30, fake, fake, 4, 0, NULL), GDN_ERR_INVALID_ARGUMENT);
  EXPECT(gdn_verify_commit(&geo, fake, fake, 100, fake, fake, 4, 8, NULL), GDN_ERR_WORKSPACE);

  /* empty calls launch nothing and succeed */
  EXPECT(gdn_decode_step(&geo, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0.088f, 1e-6f, 1e-6f, NULL, 0, NULL),
         GDN_OK);
  EXPECT(gdn_kda_recurrence(&kda, NULL, NULL, -INFINITY, NULL, NULL, 0, 0, 0.088f, 1e-6f, NULL, NULL, NULL, NULL,
                            1e-6f, NULL, NULL),
         GDN_OK);

  EXPECT(gdn_kda_chunk_prefill(&kda, NULL, NULL, -INFINITY, NULL, NULL, 0, 0, 0.088f, 1e-6f, NULL, NULL, NULL,
                               NULL, 1e-6f, NULL, NULL, 0, NULL),
         GDN_OK);
  EXPECT(gdn_kda_chunk_prefill(&kda, fake, fake, -1.0f, fake, fake, 2, 8, 0.088f, 1e-6f, NULL, NULL, NULL, NULL,
                               1e-6f, fake, NULL, 0, NULL),
         GDN_ERR_WORKSPACE);

  EXPECT(gdn_kda_prefill(&kda, NULL, NULL, NULL, 0, 0, NULL, NULL, NULL, NULL, -INFINITY, NULL, 0.088f, 1e-6f, NULL,
                         NULL, NULL, NULL, 1e-6f, NULL, NULL, 0, NULL),
         GDN_OK);

  /* sizes computed on the host */
  if (gdn_verify_stash_size(&geo, 256, 8) != (size_t)256 * 8 * 53440) return 1;
  if (gdn_verify_stash_size(&geo, 1, 18) != 0) return 1;
  if (gdn_chunk_prefill_workspace_size(&geo, 4, 16384) == 0) return 1;
  if (gdn_chunk_prefill_min_workspace_size(&geo, 4, 16384) == 0) return 1;
  if (gdn_kda_chunk_prefill_workspace_size(&kda, 4, 16384) != (size_t)256 + 256 + 256 + (size_t)259 * 64 * 108032)
    return 1;

  printf("ok\n");
  return 0;
}
