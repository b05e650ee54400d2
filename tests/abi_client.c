/* A plain C11 client of include/moe_fp8.h, built and run by tests/test_abi_c.py on the host.
 * It checks that the header is valid C, that the library links from C, and that host-side
 * validation answers before any launch. No GPU is touched: every call below returns from
 * validation, and the pointers are 16-byte-aligned stand-ins that are never dereferenced.
 * Output: one "name value" line per check. */
#include <stdint.h>
#include <stdio.h>

#include "moe_fp8.h"

int main(void) {
  const moe_fp8_shape_t s = {2048, 768, 128, 8, 16};
  const moe_fp8_shape_t bad_e = {2048, 768, 100, 8, 16};
  const moe_fp8_shape_t bad_h = {2176, 768, 128, 8, 16}; /* 17 x 128: not a multiple of 256 */
  void* p = (void*)(uintptr_t)0x10000;
  const float* mis = (const float*)(uintptr_t)0x10004;
  const cudaStream_t st = (cudaStream_t)0;
  const size_t need = moe_fp8_workspace_bytes(&s);

  printf("version %s\n", moe_fp8_version());
  printf("ws_bytes %zu\n", need);
  printf("ws_bytes_bad_e %zu\n", moe_fp8_workspace_bytes(&bad_e));
  printf("ws_bytes_bad_h %zu\n", moe_fp8_workspace_bytes(&bad_h));
  printf("forward_ok_m0 %d\n", (int)moe_fp8_forward(p, p, p, 0, p, p, p, p, p, p, need, &s, st));
  printf("forward_null_hidden %d\n", (int)moe_fp8_forward(NULL, p, p, 4, p, p, p, p, p, p, need, &s, st));
  printf("forward_m_above_max %d\n", (int)moe_fp8_forward(p, p, p, 17, p, p, p, p, p, p, need, &s, st));
  printf("forward_small_ws %d\n", (int)moe_fp8_forward(p, p, p, 4, p, p, p, p, p, p, need - 1, &s, st));
  printf("forward_bad_shape %d\n", (int)moe_fp8_forward(p, p, p, 4, p, p, p, p, p, p, need, &bad_h, st));
  printf("route_ok_m0 %d\n", (int)moe_route(p, p, NULL, 0, &s, 1, p, p, st));
  printf("route_misaligned_bias %d\n", (int)moe_route(p, p, mis, 1, &s, 1, p, p, st));
  printf("route_bad_shape %d\n", (int)moe_route(p, p, NULL, 1, &bad_e, 1, p, p, st));
  printf("read_status_null %d\n", (int)moe_fp8_read_status(NULL, p, st));
  return 0;
}
