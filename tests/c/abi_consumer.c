/* A plain C99 consumer of include/prism.h, built and run by tests/test_c_consumer.py
 * against libprism.so.  It exercises only the host-side parts of the ABI (sizes, plans,
 * argument checks), so it runs without a GPU; it fails with a message and exit code 1 on
 * the first unexpected answer. */
#include <stdio.h>
#include <string.h>

#include "prism.h"

static int fails = 0;
#define EXPECT(cond)                                                  \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "line %d: expected %s\n", __LINE__, #cond);     \
      ++fails;                                                        \
    }                                                                 \
  } while (0)

int main(void) {
  /* long-context shapes: 1 x 65536 tokens, 32 heads of 128, L = 4, w = 4, chunk 64 */
  prism_dims d;
  memset(&d, 0, sizeof d);
  d.B = 1; d.T = 65536; d.H = 32; d.d_k = 128; d.d_v = 128;
  d.conv_width = 4; d.L = 4; d.chunk = 64; d.dtype = PRISM_BF16; d.flags = 0;

  const size_t ws = prism_workspace_bytes(&d);
  EXPECT(ws > 0 && ws % 256 == 0);
  size_t offs[PRISM_WS_COUNT];
  EXPECT(prism_workspace_layout(&d, offs, PRISM_WS_COUNT) == PRISM_OK);
  EXPECT(offs[PRISM_WS_STATUS] == 0);
  EXPECT(prism_backward_workspace_bytes(&d) > 0);

  /* refused dims answer before anything touches a device */
  prism_dims bad = d;
  bad.chunk = 48;
  EXPECT(prism_workspace_bytes(&bad) == 0);
  bad = d;
  bad.d_v = 64;
  EXPECT(prism_workspace_layout(&bad, offs, PRISM_WS_COUNT) == PRISM_ERR_UNSUPPORTED);
  EXPECT(prism_forward(&d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                       NULL, NULL, 0, NULL) == PRISM_ERR_INVALID_ARG);
  int status = -1;
  EXPECT(prism_device_status(&d, NULL, ws, &status, NULL) == PRISM_ERR_WORKSPACE);
  EXPECT(prism_device_status(&d, (void*)0x100000, ws, NULL, NULL) == PRISM_ERR_INVALID_ARG);
  EXPECT(status == -1);

  /* the host-to-host entry: 8 token segments of 8192 tokens with the default minimum */
  int n = 0, bounds[PRISM_HOST_MAX_PIECES + 1];
  EXPECT(prism_host_plan(&d, 8, (size_t)32 << 20, &n, bounds) == PRISM_OK);
  EXPECT(n == 8 && bounds[0] == 0 && bounds[1] == 8192 && bounds[8] == 65536);
  EXPECT(prism_host_arena_bytes(&d, 8, (size_t)32 << 20) > 0);
  EXPECT(prism_host_arena_bytes(&d, PRISM_HOST_MAX_PIECES + 1, 0) == 0);

  for (int code = PRISM_OK; code <= PRISM_ERR_SCRATCH_LIMIT; ++code)
    EXPECT(prism_strerror(code) != NULL && prism_strerror(code)[0] != '\0');

  if (fails) return 1;
  printf("ok\n");
  return 0;
}
