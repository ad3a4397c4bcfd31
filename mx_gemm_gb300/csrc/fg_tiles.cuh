// Output-tile walk and bf16 packing shared by the large-M kernels.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

namespace fg {

// Tiles are walked in groups of `group_n` weight tiles; inside a group the
// weight tile index runs fastest, so the CTAs resident at one time share a
// band of weights (kept in L2) and a few row blocks of A.
struct TileCoord {
  int m, n;
};

__device__ __forceinline__ TileCoord tile_coord(int t, int tiles_m, int tiles_n, int group_n) {
  const int per_group = group_n * tiles_m;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int gn = min(group_n, tiles_n - g * group_n);
  TileCoord c;
  c.m = r / gn;
  c.n = g * group_n + (r - c.m * gn);
  return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace fg
