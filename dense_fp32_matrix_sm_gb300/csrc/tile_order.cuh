// tile_order.cuh -- the grouped (L2-aware) order in which persistent CTAs
// walk output tiles: consecutive tile ids cover group_m tile-rows of one
// tile-column before moving to the next column, so CTAs running at the same
// time share A and B tiles in L2 ("Writing a Fast Matmul in CUDA, Step by
// Step", "What cuBLAS and CUTLASS add": threadblock rasterization).
#pragma once

namespace sgemm {

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& tm, int& tn) {
  const int per_group = group_m * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * group_m;
  const int rows = min(tiles_m - first_m, group_m);
  const int in_group = tile - group * per_group;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

}  // namespace sgemm
