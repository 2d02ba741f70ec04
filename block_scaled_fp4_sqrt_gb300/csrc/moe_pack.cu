// Layout conversions done outside the hot loop: expert weights repacked at handle creation into
// tile-contiguous codes and scale atoms, and caller-provided activation scales turned into the
// per-tile atoms the grouped GEMMs copy into tensor memory.
#include <algorithm>

#include "moe_device.cuh"

namespace moe {

namespace {

// canonical [rows, d/32] scale bytes -> per-tile atoms [tile, d/128, 512]
__global__ void rows_sf_to_atoms_kernel(const uint8_t* __restrict__ a_s_rows, const RowTile* __restrict__ tiles,
                                        const int32_t* __restrict__ n_tiles, int d, int max_tiles,
                                        uint8_t* __restrict__ atoms) {
  const int nt = min(*n_tiles, max_tiles);
  const int groups = d / kKGroup;
  for (int ti = blockIdx.x; ti < nt; ti += gridDim.x) {
    const RowTile rt = tiles[ti];
    for (int idx = threadIdx.x; idx < rt.nrows * groups; idx += blockDim.x) {
      const int n = idx / groups, grp = idx - n * groups;
      const uint32_t word = *reinterpret_cast<const uint32_t*>(a_s_rows + (size_t)(rt.row0 + n) * (d / 32) + grp * 4);
      *reinterpret_cast<uint32_t*>(atoms + ((size_t)ti * groups + grp) * kSfAtomBytes + (n & 31) * 16 +
                                   ((n >> 5) & 3) * 4) = word;
    }
  }
}

// the inverse: per-tile atoms [tile, K/128, 512] -> canonical [rows, K/32] scale bytes
__global__ void atoms_to_rows_sf_kernel(const uint8_t* __restrict__ atoms, const RowTile* __restrict__ tiles,
                                        const int32_t* __restrict__ n_tiles, int K, int max_tiles,
                                        uint8_t* __restrict__ rows_sf) {
  const int nt = min(*n_tiles, max_tiles);
  const int groups = K / kKGroup;
  for (int ti = blockIdx.x; ti < nt; ti += gridDim.x) {
    const RowTile rt = tiles[ti];
    for (int idx = threadIdx.x; idx < rt.nrows * groups; idx += blockDim.x) {
      const int n = idx / groups, grp = idx - n * groups;
      const uint32_t word = *reinterpret_cast<const uint32_t*>(atoms + ((size_t)ti * groups + grp) * kSfAtomBytes +
                                                               (n & 31) * 16 + ((n >> 5) & 3) * 4);
      *reinterpret_cast<uint32_t*>(rows_sf + (size_t)(rt.row0 + n) * (K / 32) + grp * 4) = word;
    }
  }
}

// Output tile and row inside its 256-row slab of canonical weight row `row` (see launch_pack_weights).
__device__ __forceinline__ void slab_of_row(int row, int rows, int mode, int* tile, int* rr) {
  if (mode == 0) {
    const int f = rows / 2;
    const bool up = row >= f;
    const int fr = up ? row - f : row;
    *tile = fr >> 7;
    *rr = (up ? 128 : 0) + (fr & 127);
  } else {
    *tile = row >> 8;
    *rr = row & 255;
  }
}

// codes [n, rows, K/2] -> packed [n, K/128, rows/256, 256, 64]; one 16-byte chunk per thread step.  The
// K group is outside the output tile so that CTAs working on neighbouring output tiles of one expert
// read neighbouring 16 KB blocks at the same time.
__global__ void pack_weights_kernel(const uint8_t* __restrict__ src, int n, int rows, int K, int mode,
                                    uint8_t* __restrict__ dst) {
  const int KG = K / kKGroup, MT = rows / 256;
  const size_t total = (size_t)n * rows * (K / 2) / 16;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int c16 = (int)(i & 3);
    const int rr = (int)((i >> 2) & 255);
    const size_t rest = i >> 10;  // (e * KG + kg) * MT + mt
    const int mt = (int)(rest % MT);
    const size_t ekg = rest / MT;
    const int kg = (int)(ekg % KG);
    const size_t e = ekg / KG;
    int row;
    if (mode == 0) row = rr < 128 ? mt * 128 + rr : rows / 2 + mt * 128 + (rr - 128);
    else row = mt * 256 + rr;
    const uint4 v = *reinterpret_cast<const uint4*>(src + (e * rows + row) * (size_t)(K / 2) + kg * 64 + c16 * 16);
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
}

// scales [n, rows, K/32] -> atoms [n, K/128, rows/256, 2, 512]
__global__ void pack_weight_sf_kernel(const uint8_t* __restrict__ s, int n, int rows, int K, int mode,
                                      uint8_t* __restrict__ atoms) {
  const int groups = K / kKGroup, MT = rows / 256;
  const size_t total = (size_t)n * rows * groups;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int grp = (int)(i % groups);
    const size_t er = i / groups;  // e * rows + r
    const int r = (int)(er % rows);
    const size_t e = er / rows;
    int tile, rr;
    slab_of_row(r, rows, mode, &tile, &rr);
    const int half = rr >> 7, lr = rr & 127;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(s + er * (K / 32) + grp * 4);
    const size_t blk = (((e * groups + grp) * MT + tile) * 2 + half);
    *reinterpret_cast<uint32_t*>(atoms + blk * kSfAtomBytes + (lr & 31) * 16 + (lr >> 5) * 4) = word;
  }
}

}  // namespace

cudaError_t launch_rows_sf_to_atoms(const uint8_t* a_s_rows, const RowTile* tiles, const int32_t* n_tiles, int d,
                                    int max_tiles, uint8_t* atoms, cudaStream_t s) {
  rows_sf_to_atoms_kernel<<<296, 256, 0, s>>>(a_s_rows, tiles, n_tiles, d, max_tiles, atoms);
  return cudaGetLastError();
}

cudaError_t launch_atoms_to_rows_sf(const uint8_t* atoms, const RowTile* tiles, const int32_t* n_tiles, int K,
                                    int max_tiles, uint8_t* rows_sf, cudaStream_t s) {
  atoms_to_rows_sf_kernel<<<296, 256, 0, s>>>(atoms, tiles, n_tiles, K, max_tiles, rows_sf);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const uint8_t* codes, int n, int rows, int K, int mode, uint8_t* packed,
                                cudaStream_t s) {
  const size_t total = (size_t)n * rows * (K / 2) / 16;
  const int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 32);
  pack_weights_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(codes, n, rows, K, mode, packed);
  return cudaGetLastError();
}

cudaError_t launch_pack_weight_sf(const uint8_t* sc, int n, int rows, int K, int mode, uint8_t* atoms,
                                  cudaStream_t s) {
  const size_t total = (size_t)n * rows * (K / kKGroup);
  const int blocks = (int)std::min<size_t>((total + 255) / 256, 4096);
  pack_weight_sf_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(sc, n, rows, K, mode, atoms);
  return cudaGetLastError();
}

}  // namespace moe
