// Host-side cases of the self-check predicates of ptx.cuh (the conditions the
// checked build tests before each TMA copy and TMEM access).  Prints one
// line "name value" per case; tests/test_selfcheck.py compares them with the
// expected values.
#include <cstdio>
#include "../transformer_scaled_dot_sdpa_gb300/csrc/ptx.cuh"
using namespace gb300;
int main() {
  // innermost TMA coordinate x: x * element size on a 16-byte boundary
  printf("coord_bf16_0 %d\n", tma_inner_coord_ok(0, 2));
  printf("coord_bf16_64 %d\n", tma_inner_coord_ok(64, 2));
  printf("coord_bf16_8 %d\n", tma_inner_coord_ok(8, 2));
  printf("coord_bf16_4 %d\n", tma_inner_coord_ok(4, 2));
  printf("coord_bf16_neg8 %d\n", tma_inner_coord_ok(-8, 2));
  printf("coord_bf16_neg3 %d\n", tma_inner_coord_ok(-3, 2));
  printf("coord_f32_4 %d\n", tma_inner_coord_ok(4, 4));
  printf("coord_f32_2 %d\n", tma_inner_coord_ok(2, 4));
  printf("coord_u8_16 %d\n", tma_inner_coord_ok(16, 1));
  printf("coord_u8_8 %d\n", tma_inner_coord_ok(8, 1));
  // 128-byte-swizzled tiles start on 1024 bytes
  printf("tile_0 %d\n", swizzled_tile_ok(0u));
  printf("tile_16384 %d\n", swizzled_tile_ok(16384u));
  printf("tile_512 %d\n", swizzled_tile_ok(512u));
  printf("tile_1040 %d\n", swizzled_tile_ok(1040u));
  // TMEM: lane field 32 * (warp % 4), columns within 512
  const unsigned lane64 = 64u << 16;
  printf("tmem_w2_col0 %d\n", tmem_warp_access_ok(lane64 + 0u, 32u, 2u));
  printf("tmem_w6_col480 %d\n", tmem_warp_access_ok(lane64 + 480u, 32u, 6u));
  printf("tmem_w6_col481 %d\n", tmem_warp_access_ok(lane64 + 481u, 32u, 6u));
  printf("tmem_w1_lane64 %d\n", tmem_warp_access_ok(lane64, 32u, 1u));
  printf("tmem_w0_lane0_col256 %d\n", tmem_warp_access_ok(256u, 32u, 0u));
  return 0;
}
