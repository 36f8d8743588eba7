/* A plain C11 client of include/gmlp.h: compiles without any C++ or CUDA
 * header, links libgmlp.so, and exercises the calls that need no GPU (layout
 * queries, size queries, host-side argument checks and the error text).
 * Prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "gmlp.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      printf("FAILED line %d: %s\n", __LINE__, #cond);           \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  CHECK(strstr(gmlp_version(), "sm_103a") != NULL);
  CHECK(gmlp_colwise_tokens(513, 4) == 128 * (5 + 4));
  CHECK(gmlp_colwise_tokens(-1, 4) == 0);
  CHECK(gmlp_tiled_scales_bytes(512, 4, 8) == (size_t)(4 + 4) * 128 * 8);

  /* GEMM_TILED: row 64 of splits {64, 65} opens the second group's first tile */
  const int64_t splits[2] = {64, 65};
  CHECK(gmlp_query_layout(GMLP_LAYOUT_TILED_SCALE, splits, 2, 4, 64, 0) == 512);
  CHECK(gmlp_query_layout(GMLP_LAYOUT_TILED_SCALE, splits, 2, 4, 33, 2) == (33 % 32) * 16 + (33 / 32) * 4 + 2);
  CHECK(gmlp_query_layout(GMLP_LAYOUT_TILED_SCALE, splits, 2, 4, 129, 0) == -1);
  CHECK(gmlp_query_layout(GMLP_LAYOUT_COLWISE_CODE, splits, 2, 256, 65, 3) == (1 * 256 + 3) * 128 + 1);
  CHECK(gmlp_query_layout(9, splits, 2, 4, 0, 0) == -1);

  /* argument checks return a status before anything is launched */
  gmlp_recipe rec;
  memset(&rec, 0, sizeof(rec));
  rec.format = GMLP_MXFP8;
  rec.scale_layout = GMLP_SCALES_GEMM_TILED;
  CHECK(gmlp_forward(NULL, 128, 256, 256, NULL, 1, NULL, NULL, NULL, GMLP_ACT_SWIGLU, &rec, NULL, NULL, NULL, 0,
                     NULL) == GMLP_ERR_INVALID_ARG);
  CHECK(strstr(gmlp_last_error(), "split_sizes") != NULL);
  CHECK(gmlp_group_quantize(NULL, 128, 100, (const int64_t*)(uintptr_t)4096, 1, &rec, NULL, NULL, NULL, NULL,
                            NULL) == GMLP_ERR_INVALID_DIMS);
  rec.format = 7;
  CHECK(gmlp_group_hadamard_amax(NULL, 0, 128, (const int64_t*)(uintptr_t)4096, 0, 0, NULL, NULL, NULL) ==
        GMLP_ERR_INVALID_DIMS);
  printf("ok\n");
  return 0;
}
