/* A plain C99 program that uses libmxq through include/mxq.h alone: the
 * header must compile as C and every call below must link and behave as
 * documented without a GPU (queries, and argument errors that return before
 * anything is launched).  Pointers are fake device addresses that are never
 * dereferenced.  Exit status 0 when every expectation holds. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "mxq.h"

static int failures = 0;

#define EXPECT(cond)                                                         \
  do {                                                                       \
    if (!(cond)) {                                                           \
      fprintf(stderr, "%s:%d: expected %s\n", __FILE__, __LINE__, #cond);    \
      failures++;                                                            \
    }                                                                        \
  } while (0)

int main(void) {
  void* p = (void*)(uintptr_t)0x100000; /* 16-byte aligned */
  void* u = (void*)(uintptr_t)0x100008; /* misaligned */
  int st;

  EXPECT(mxq_version() == 100);
  EXPECT(mxq_arch_supported(10, 3) == 1);
  EXPECT(mxq_arch_supported(10, 0) == 0);
  EXPECT(strcmp(mxq_status_string(MXQ_ERR_WORKSPACE), "MXQ_ERR_WORKSPACE") == 0);

  st = mxq_inv_rope_group_quant(NULL, 4, 1, 256, 0, NULL, NULL, NULL, 0, 0, p, p, NULL, NULL);
  EXPECT(st == MXQ_ERR_NULL);
  EXPECT(strlen(mxq_last_error()) > 0);
  st = mxq_inv_rope_group_quant(u, 4, 1, 256, 0, NULL, NULL, NULL, 0, 0, p, p, NULL, NULL);
  EXPECT(st == MXQ_ERR_ALIGN);
  st = mxq_inv_rope_group_quant(NULL, 0, 1, 256, 0, NULL, NULL, NULL, 0, 0, NULL, NULL, NULL, NULL);
  EXPECT(st == MXQ_OK); /* T == 0 is a no-op */

  /* 1 MiB of prepared scales for W [8, 1024, 4096]: 8 x 32 groups x 8 row blocks x 512 B */
  EXPECT(mxq_weight_scale_bytes(8, 1024, 4096) == (size_t)8 * 32 * 8 * 512);
  st = mxq_prepare_weight_scales(p, 8, 1024, 4100, p, NULL);
  EXPECT(st == MXQ_ERR_SHAPE);

  EXPECT(mxq_bmm_workspace_bytes(8192, 8, 1024, 4096) == 0);
  st = mxq_bmm_a8w8(p, p, p, p, p, 4, 1, 120, 256, NULL, 0, NULL);
  EXPECT(st == MXQ_ERR_SHAPE);
  st = mxq_bmm_a8w8(p, p, p, p, p, 4, 1, 128, 65536 + 16, NULL, 0, NULL);
  EXPECT(st == MXQ_ERR_UNSUPPORTED);

  EXPECT(mxq_linear_workspace_bytes(8, 5120, 576) == 0);
  st = mxq_linear(p, p, p, p, 100, 5120, 576, NULL, 0, NULL);
  EXPECT(st == MXQ_ERR_WORKSPACE);

  EXPECT(mxq_wo_a_workspace_bytes(32, 8, 4096, 1024) == 0);
  EXPECT(mxq_wo_a_workspace_bytes(33, 8, 4096, 1024) == (size_t)33 * 8 * 4096 + 33 * 8 * 32);
  st = mxq_wo_a(p, p, p, p, 32, 16, p, p, p, 8192, 8, 4096, 1024, 64, NULL, NULL, 0, NULL);
  EXPECT(st == MXQ_ERR_WORKSPACE);
  st = mxq_wo_a(p, p, p, p, 36, 16, p, p, p, 4, 8, 4096, 1024, 64, NULL, NULL, 0, NULL);
  EXPECT(st == MXQ_ERR_ALIGN); /* cos/sin row stride % 8 */

  st = mxq_dequant_bf16(p, p, p, 0, 16, 128, NULL);
  EXPECT(st == MXQ_OK); /* B == 0 is a no-op */
  st = mxq_dequant_bf16(p, p, p, 1, 16, 120, NULL);
  EXPECT(st == MXQ_ERR_SHAPE);
  st = mxq_scales_f32_to_e8m0(p, -1, p, NULL, NULL);
  EXPECT(st == MXQ_ERR_SHAPE);

  st = mxq_linear_noalloc(p, p, p, p, 1 << 20, 5120, 576, NULL);
  EXPECT(st == MXQ_ERR_WORKSPACE); /* beyond the fixed scratch */

  st = mxq_linear_noalloc(p, p, p, u, 100, 5120, 576, NULL);
  EXPECT(st == MXQ_ERR_ALIGN); /* every rule checked before anything is enqueued */
  st = mxq_linear_noalloc(p, p, p, p, 1, 5120, 131072, NULL);
  EXPECT(st == MXQ_ERR_UNSUPPORTED);

  /* KV insert: an E4M3 cache needs its per-tensor scale; a BF16 cache does not. */
  st = mxq_rope_kv_insert(p, p, 4, 2, 512, p, 512, p, p, p, 32, 16, 64, p, p, 8, MXQ_CACHE_E4M3,
                          NULL, NULL, NULL);
  EXPECT(st == MXQ_ERR_NULL);
  st = mxq_rope_kv_insert(p, p, 4, 2, 512, p, 520, p, p, p, 32, 16, 64, p, p, 8, MXQ_CACHE_BF16,
                          NULL, NULL, NULL);
  EXPECT(st == MXQ_ERR_SHAPE);
  EXPECT(MXQ_DEVERR_SLOT == 4);

  printf("%d failures\n", failures);
  return failures ? 1 : 0;
}
