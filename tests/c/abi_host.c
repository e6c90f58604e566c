/* Plain C99 client of the library's C ABI (host-only calls, no GPU needed): the header compiles
 * as C, the library links and loads, the size queries answer, and calls with bad arguments are
 * rejected before anything is launched. Pointers below are never dereferenced. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe_gb300.h"

static int failures = 0;
#define EXPECT(cond)                                                   \
  do {                                                                 \
    if (!(cond)) {                                                     \
      fprintf(stderr, "line %d: expectation failed: %s\n", __LINE__, #cond); \
      ++failures;                                                      \
    }                                                                  \
  } while (0)

int main(void) {
  moe_dims full = {2048, 256, 8, 512, 512, 64};
  moe_dims bad = full;
  moe_layer layer;
  void* fake = (void*)(uintptr_t)(1u << 20); /* 128-byte aligned, never dereferenced */
  size_t ws16;

  EXPECT(moe_packed_bytes(&full) == (size_t)257 * 1769472u);
  EXPECT(moe_tile_rows() == 192);
  ws16 = moe_workspace_bytes(&full, 16);
  EXPECT(ws16 > 0);
  EXPECT(moe_workspace_bytes(&full, 4096) > ws16);
  EXPECT(moe_workspace_bytes(&full, 0) == 0);
  bad.group = 32;
  EXPECT(moe_packed_bytes(&bad) == 0 && moe_workspace_bytes(&bad, 16) == 0);
  EXPECT(strlen(moe_status_string(MOE_ERR_WORKSPACE_TOO_SMALL)) > 0);

  memset(&layer, 0, sizeof layer);
  layer.dims = full;
  layer.router_w = (const uint16_t*)fake;
  layer.packed = fake;
  EXPECT(moe_prefill(&layer, NULL, 16, (uint16_t*)fake, NULL, fake, ws16, NULL) == MOE_ERR_INVALID_ARG);
  EXPECT(moe_prefill(&layer, (const uint16_t*)fake, 70000, (uint16_t*)fake, NULL, fake, ws16, NULL) ==
         MOE_ERR_UNSUPPORTED_SHAPE);
  EXPECT(moe_prefill(&layer, (const uint16_t*)fake, 16, (uint16_t*)fake, NULL, fake, ws16 - 1, NULL) ==
         MOE_ERR_WORKSPACE_TOO_SMALL);
  EXPECT(moe_decode(&layer, (const uint16_t*)((char*)fake + 8), (uint16_t*)fake, NULL, fake, ws16, NULL) ==
         MOE_ERR_MISALIGNED);
  EXPECT(moe_prefill_chunked(&layer, (const uint16_t*)fake, 100000, (uint16_t*)fake, 0, fake, ws16, NULL) ==
         MOE_ERR_INVALID_ARG);
  EXPECT(moe_route(&layer, NULL, NULL, 16, NULL, fake, ws16, NULL) == MOE_ERR_INVALID_ARG);
  layer.dims.group = 128;
  EXPECT(moe_decode(&layer, (const uint16_t*)fake, (uint16_t*)fake, NULL, fake, ws16, NULL) ==
         MOE_ERR_UNSUPPORTED_SHAPE);

  if (failures) return 1;
  printf("c abi ok\n");
  return 0;
}
