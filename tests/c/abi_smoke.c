/* Calls the library through its C header alone: a C11 program, no CUDA headers
 * and no Python.  Needs no GPU: every call below fails a host-side check or
 * only computes a size, and the process checks the returned values. */
#include <stdio.h>
#include <string.h>

#include "gqa_attn.h"

#define EXPECT(cond)                                                \
  do {                                                              \
    if (!(cond)) {                                                  \
      fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
      return 1;                                                     \
    }                                                               \
  } while (0)

int main(void) {
  EXPECT(gqa_version() >= 100);
  EXPECT(strcmp(gqa_status_str(GQA_OK), "GQA_OK") == 0);
  EXPECT(strcmp(gqa_status_str(GQA_ERR_UNSUPPORTED), "GQA_ERR_UNSUPPORTED") == 0);
  EXPECT(strcmp(gqa_status_str(99), "GQA_ERR_UNKNOWN") == 0);

  /* sizes: ceil(32768 / 19) rounded up to the 64-token tile */
  EXPECT(gqa_attn_decode_split_chunk(32768, 19) == 1728);
  const size_t ml = (size_t)2 * 64 * 38 * 8, off = (ml + 255) / 256 * 256;
  EXPECT(gqa_attn_decode_workspace_bytes(2, 64, 128, 38) == off + (size_t)2 * 64 * 38 * 128 * 4);
  EXPECT(gqa_attn_decode_workspace_bytes(2, 64, 128, 1) == 0);

  /* host-side argument checks: nothing is launched, nothing is touched */
  gqa_stream_t s = NULL;
  EXPECT(gqa_attn_decode(NULL, NULL, NULL, NULL, 1, 64, 8, 2, 128, 0.1f, 1, NULL, NULL, NULL, s) ==
         GQA_ERR_INVALID_ARG);
  EXPECT(gqa_attn_decode_combine(NULL, 1, 8, 128, 2, NULL, NULL, s) == GQA_ERR_INVALID_ARG);
  EXPECT(gqa_attn_prefill_causal(NULL, NULL, NULL, 1, 128, 8, 2, 128, 0.1f, NULL, NULL, s) ==
         GQA_ERR_INVALID_ARG);
  printf("abi_smoke: ok (version %d)\n", gqa_version());
  return 0;
}
