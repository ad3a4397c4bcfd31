// Output-tile walk and bf16 packing shared by the large-M kernels.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

namespace fg {

// Tiles are walked in groups of kGroupN weight tiles; inside a group the A row
// block index runs fastest, so the CTAs resident at one time share a band of
// weights (kept in L2) and a few A row blocks.
constexpr int kGroupN = 16;

struct TileCoord {
  int m, n;
};

__device__ __forceinline__ TileCoord tile_coord(int t, int tiles_m, int tiles_n) {
  const int per_group = kGroupN * tiles_m;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int gn = min(kGroupN, tiles_n - g * kGroupN);
  TileCoord c;
  c.m = r / gn;
  c.n = g * kGroupN + (r - c.m * gn);
  return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace fg
