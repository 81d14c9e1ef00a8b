/* Plain C99 use of the library's C ABI: the header compiles as C, every call links, and
 * argument validation answers without a device (nothing here is ever launched). */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "attn.h"

static int failures = 0;

static void expect(const char* what, attn_status_t got, attn_status_t want) {
  if (got != want) {
    printf("FAIL %s: got %d (%s), want %d\n", what, (int)got, attn_status_string(got), (int)want);
    ++failures;
  }
}

int main(void) {
  /* 16-byte aligned fake device addresses: never dereferenced, validation fails first */
  void* a = (void*)(uintptr_t)0x7F0000000000ull;
  void* o = (void*)(uintptr_t)0x7F0000100000ull;
  void* mis = (void*)(uintptr_t)0x7F0000000008ull;
  if (attn_version() < 200) {
    printf("FAIL attn_version\n");
    ++failures;
  }
  if (strcmp(attn_status_string(ATTN_OK), attn_status_string(ATTN_ERR_INVALID_ARG)) == 0) {
    printf("FAIL status strings\n");
    ++failures;
  }
  expect("rope_apply null", rope_apply(NULL, o, ATTN_BF16, 1, 1, 1, 64, 0, 1e4f, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("prefill misaligned",
         attn_prefill(a, a, a, mis, NULL, ATTN_BF16, 1.f, 1.f, 1.f, 1, 4, 1, 128, 64, 1, 0.f, 1,
                      1e4f, 0, NULL, 0, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("prefill head dim",
         attn_prefill(a, a, a, o, NULL, ATTN_BF16, 1.f, 1.f, 1.f, 1, 4, 1, 128, 96, 1, 0.f, 1,
                      1e4f, 0, NULL, 0, NULL),
         ATTN_ERR_UNSUPPORTED);
  expect("chunk lengths",
         attn_prefill_chunk(a, a, a, o, NULL, ATTN_BF16, 1.f, 1.f, 1.f, 1, 4, 1, 64, 32, 64, 64,
                            0.f, 1, 1e4f, 0, NULL, 0, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("decode groups",
         attn_decode(a, a, a, (const int32_t*)o, 2048, o, NULL, ATTN_BF16, 1, 30, 8, 128, 0.f, 1,
                     1e4f, o, 1u << 20, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("append no workspace",
         attn_decode_append(a, a, a, a, a, (int32_t*)o, 2048, o, NULL, ATTN_BF16, 1, 32, 8, 128,
                            0.f, 1, 1e4f, NULL, 0, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("latent heads",
         attn_decode_latent(a, a, (const int32_t*)o, 2048, o, NULL, ATTN_BF16, 1, 17, 0.f, 1,
                            1e4f, o, 1u << 20, NULL),
         ATTN_ERR_UNSUPPORTED);
  expect("rope style range",
         rope_apply_style(a, o, ATTN_BF16, 1, 1, 1, 64, 0, 1e4f, (attn_rope_style_t)4, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("interleaved flag without a mode",
         attn_prefill(a, a, a, o, NULL, ATTN_BF16, 1.f, 1.f, 1.f, 1, 4, 1, 128, 64, 1, 0.f,
                      ATTN_ROPE_FLAG_INTERLEAVED, 1e4f, 0, NULL, 0, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("interleaved fused form",
         attn_prefill(a, a, a, o, NULL, ATTN_BF16, 1.f, 1.f, 1.f, 1, 4, 1, 128, 64, 1, 0.f,
                      2 | ATTN_ROPE_FLAG_INTERLEAVED, 1e4f, 0, NULL, 0, NULL),
         ATTN_ERR_UNSUPPORTED);
  expect("backward fp8",
         attn_prefill_backward(a, a, a, a, (const float*)o, a, o, o, o, ATTN_FP8_E5M2, 1, 4, 1,
                               128, 64, 1, 0.f, o, 1u << 30, NULL),
         ATTN_ERR_UNSUPPORTED);
  expect("backward workspace",
         attn_prefill_backward(a, a, a, a, (const float*)o, a, o, o, o, ATTN_BF16, 1, 4, 1, 128,
                               64, 1, 0.f, o, 16, NULL),
         ATTN_ERR_WORKSPACE);
  if (attn_prefill_backward_workspace_size(1, 4, 128, 64) == 0) {
    printf("FAIL backward workspace size\n");
    ++failures;
  }
  expect("split hook range", attn_set_decode_splits(-1), ATTN_ERR_INVALID_ARG);
  expect("backward path range", attn_set_backward_path(3), ATTN_ERR_INVALID_ARG);
  expect("backward path default", attn_set_backward_path(0), ATTN_OK);
  expect("prefill rotation workspace missing",
         attn_prefill(a, a, a, o, NULL, ATTN_BF16, 1.f, 1.f, 1.f, 4, 32, 8, 16384, 128, 1, 0.f, 1,
                      1e4f, 0, NULL, 0, NULL),
         ATTN_ERR_WORKSPACE);
  if (attn_prefill_workspace_size(4, 32, 8, 16384, 128, ATTN_BF16, 1) !=
      (size_t)(4 + 1) * 32 * 16384 * 128 * 2) {
    printf("FAIL prefill workspace size\n");
    ++failures;
  }
  if (attn_prefill_chunk_workspace_size(1, 4, 32, 64, ATTN_FP8_E5M2, 1) != 0) {
    printf("FAIL chunk workspace size (fp8 rotates in the kernel)\n");
    ++failures;
  }
  if (attn_decode_workspace_size(1, 30, 8, 128, 2048) != 0) {
    printf("FAIL workspace size of an invalid shape\n");
    ++failures;
  }
  printf(failures ? "abi_check: %d failures\n" : "abi_check: ok\n", failures);
  return failures ? 1 : 0;
}
