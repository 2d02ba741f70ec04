// Token <-> expert dispatch and combine (the single-GPU form of the pypto page's "dispatch /
// combine" around expert_routed / expert_shared, "MoE and output stages"):
//
//  * histogram:  per 32-token chunk, how many (token, slot) pairs go to each expert group;
//  * scan:       exclusive sums over chunks (per group) and over groups -> counts, offsets and a
//                device-side list of row tiles for the grouped GEMMs (no host round trip);
//  * gather:     MXFP8 quantisation of each token row (E4M3, one E8M0 scale per 32 along d) and
//                its copy to every expert row it is routed to, expert-major with tokens ascending
//                inside an expert (deterministic: a token's rank comes from a warp ballot over
//                the lower tokens of its chunk plus the chunk's exclusive base, no atomics);
//  * combine:    out[t] = sum_j Yr[inv_pos[t, j]] + Yr[R + t] in fp32, in the fixed order j = 0..k-1
//                then the shared row, rounded once to bf16 (the weighted-sum epilogue; the routing
//                weight was applied in the down GEMM).
#include <algorithm>

#include "moe_device.cuh"

namespace moe {

namespace {

__device__ __forceinline__ int clamp_id(int e, int E, int* status) {
  if (e < 0 || e >= E) {
    set_status(status, DEV_BAD_EXPERT_ID);
    return 0;
  }
  return e;
}

// one warp per 32-token chunk; chunk_hist[c][g] = number of (t, j) in chunk c with ids[t, j] = g
__global__ void histogram_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int G, int n_chunks,
                                 int32_t* __restrict__ chunk_hist, int* status) {
  extern __shared__ int sh_hist[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * (blockDim.x >> 5) + warp;
  int* h = sh_hist + warp * G;
  for (int g = lane; g < G; g += 32) h[g] = 0;
  __syncwarp();
  if (chunk < n_chunks) {
    const int t = chunk * 32 + lane;
    if (t < T)
      for (int j = 0; j < k; ++j) atomicAdd(&h[clamp_id(ids[(size_t)t * k + j], E, status)], 1);
  }
  __syncwarp();
  if (chunk < n_chunks)
    for (int g = lane; g < G; g += 32) chunk_hist[(size_t)chunk * G + g] = h[g];
}

// Build row tiles of at most bn rows per group from (offsets, per-group tile offsets).
__device__ void write_tiles(const int* s_off, const int* s_cnt, const int* s_toff, int G, int bn, int max_tiles,
                            RowTile* tiles) {
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int cnt = s_cnt[g];
    for (int i = 0; i * bn < cnt; ++i) {
      const int idx = s_toff[g] + i;
      if (idx < max_tiles) {
        RowTile rt;
        rt.group = g;
        rt.row0 = s_off[g] + i * bn;
        rt.nrows = min(bn, cnt - i * bn);
        rt.pad = 0;
        tiles[idx] = rt;
      }
    }
  }
}

__device__ void serial_group_scan(const int* s_cnt, int* s_off, int* s_toff, int G, int bn, int max_tiles,
                                  int32_t* offsets, int32_t* tile_off, int32_t* n_tiles, int* status) {
  if (threadIdx.x == 0) {
    int off = 0, toff = 0;
    for (int g = 0; g < G; ++g) {
      s_off[g] = off;
      s_toff[g] = toff;
      offsets[g] = off;
      tile_off[g] = toff;
      off += s_cnt[g];
      toff += (s_cnt[g] + bn - 1) / bn;
    }
    offsets[G] = off;
    tile_off[G] = toff;
    if (toff > max_tiles) set_status(status, DEV_BAD_WORK);
    *n_tiles = min(toff, max_tiles);
  }
}

constexpr int kMaxGroups = 2048;

// Single block.  Column scans of chunk_hist (in place, exclusive) -> counts; group scans -> offsets
// and tile offsets; then the tile list.  The shared group (index E when has_shared) holds all T rows.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ chunk_hist, int n_chunks, int T, int E,
                                                    int G, int has_shared, int bn, int max_tiles,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ tile_off, int32_t* __restrict__ n_tiles,
                                                    RowTile* __restrict__ tiles, int* status) {
  __shared__ int s_cnt[kMaxGroups], s_off[kMaxGroups], s_toff[kMaxGroups];
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int run = 0;
    if (has_shared && g == E) {
      run = T;
    } else {
      int c = 0;
      for (; c + 8 <= n_chunks; c += 8) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = chunk_hist[(size_t)(c + i) * G + g];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          chunk_hist[(size_t)(c + i) * G + g] = run;
          run += v[i];
        }
      }
      for (; c < n_chunks; ++c) {
        const int v = chunk_hist[(size_t)c * G + g];
        chunk_hist[(size_t)c * G + g] = run;
        run += v;
      }
    }
    counts[g] = run;
    s_cnt[g] = run;
  }
  __syncthreads();
  serial_group_scan(s_cnt, s_off, s_toff, G, bn, max_tiles, offsets, tile_off, n_tiles, status);
  __syncthreads();
  write_tiles(s_off, s_cnt, s_toff, G, bn, max_tiles, tiles);
}

// Tiles for caller-given group offsets (moe_expert_ffn).  offsets[G] must equal n_rows; offsets
// NULL means one group holding all n_rows rows.
__global__ void __launch_bounds__(1024) tiles_from_offsets_kernel(const int32_t* __restrict__ offsets, int G,
                                                                  int n_rows, int bn, int max_tiles,
                                                                  int32_t* __restrict__ tile_off,
                                                                  int32_t* __restrict__ n_tiles,
                                                                  RowTile* __restrict__ tiles, int* status) {
  __shared__ int s_cnt[kMaxGroups], s_off[kMaxGroups], s_toff[kMaxGroups];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = offsets && (offsets[0] != 0 || offsets[G] != n_rows) ? 1 : 0;
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int c = offsets ? offsets[g + 1] - offsets[g] : n_rows;
    if (c < 0) {
      bad = 1;
      c = 0;
    }
    s_cnt[g] = c;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      set_status(status, DEV_BAD_WORK);
      *n_tiles = 0;
    }
    return;
  }
  if (threadIdx.x == 0) {
    int toff = 0;
    for (int g = 0; g < G; ++g) {
      s_off[g] = offsets ? offsets[g] : 0;
      s_toff[g] = toff;
      tile_off[g] = toff;
      toff += (s_cnt[g] + bn - 1) / bn;
    }
    tile_off[G] = toff;
    if (toff > max_tiles) set_status(status, DEV_BAD_WORK);
    *n_tiles = min(toff, max_tiles);
  }
  __syncthreads();
  write_tiles(s_off, s_cnt, s_toff, G, bn, max_tiles, tiles);
}

// One warp per token.  Lane l quantises the 128-element groups l, l+32, ...: four MXFP8 blocks
// each, so the four scale bytes of a group form one 32-bit word, which is exactly one word of a
// scale atom (bytes = 32-element blocks of one 128-element K group).
__global__ void __launch_bounds__(256) gather_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ ids, const float* __restrict__ wts,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_off,
    int T, int d, int k, int E, int G, int has_shared, int bn, uint8_t* __restrict__ a_q,
    uint8_t* __restrict__ a_sf_atoms, uint8_t* __restrict__ a_s_rows, int32_t* __restrict__ perm_tok,
    int32_t* __restrict__ inv_pos, float* __restrict__ row_w) {
  constexpr int kMaxDst = 17;  // top-k <= 16, plus the shared row
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int chunk = t >> 5, t0 = chunk * 32;
  // destinations: routed rows, then the shared row
  int dst_row[kMaxDst], dst_tile[kMaxDst], dst_n[kMaxDst];
  int n_dst = 0;
  const int tl = t0 + lane;  // lane's token for the rank ballots
  for (int j = 0; j < k; ++j) {
    const int e = clamp_id(ids[(size_t)t * k + j], E, nullptr);
    bool hit = false;
    if (tl < t)
      for (int jj = 0; jj < k; ++jj) hit |= clamp_id(ids[(size_t)tl * k + jj], E, nullptr) == e;
    const int rank = __popc(__ballot_sync(0xFFFFFFFFu, hit));
    const int local = chunk_base[(size_t)chunk * G + e] + rank;
    const int row = offsets[e] + local;
    dst_row[n_dst] = row;
    dst_tile[n_dst] = tile_off[e] + local / bn;
    dst_n[n_dst] = local % bn;
    ++n_dst;
    if (lane == 0) {
      perm_tok[row] = t;
      inv_pos[(size_t)t * k + j] = row;
      if (row_w) row_w[row] = wts ? wts[(size_t)t * k + j] : 1.0f;
    }
  }
  if (has_shared) {
    const int row = offsets[E] + t;
    dst_row[n_dst] = row;
    dst_tile[n_dst] = tile_off[E] + t / bn;
    dst_n[n_dst] = t % bn;
    ++n_dst;
    if (lane == 0) {
      perm_tok[row] = t;
      if (row_w) row_w[row] = 1.0f;
    }
  }
  const int n_groups = d / kKGroup;
  const int kg_total = n_groups;
  for (int grp = lane; grp < n_groups; grp += 32) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + grp * kKGroup);
    uint32_t packed[32];  // 128 E4M3 codes
    uint32_t sword = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float v[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 raw = __ldg(src + b * 4 + c);
        const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[c * 8 + i] = __bfloat162float(hv[i]);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const int se = mxfp8_block_exp(amax);
      const float mul = exp2_neg_int(se);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = e4m3x2(v[4 * i] * mul, v[4 * i + 1] * mul);
        const uint32_t hi = e4m3x2(v[4 * i + 2] * mul, v[4 * i + 3] * mul);
        packed[b * 8 + i] = lo | (hi << 16);
      }
      sword |= (uint32_t)(se + 127) << (8 * b);
    }
    for (int q = 0; q < n_dst; ++q) {
      uint4* dst = reinterpret_cast<uint4*>(a_q + (size_t)dst_row[q] * d + grp * kKGroup);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      if (a_sf_atoms) {
        const int n = dst_n[q];
        uint32_t* w = reinterpret_cast<uint32_t*>(a_sf_atoms + ((size_t)dst_tile[q] * kg_total + grp) * kSfAtomBytes +
                                                  (n & 31) * 16 + ((n >> 5) & 3) * 4);
        *w = sword;
      }
      if (a_s_rows) *reinterpret_cast<uint32_t*>(a_s_rows + (size_t)dst_row[q] * (d / 32) + grp * 4) = sword;
    }
  }
}

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

// codes [n, rows, K/2] -> packed [n, rows/256, K/128, 256, 64]; one 16-byte chunk per thread step
__global__ void pack_weights_kernel(const uint8_t* __restrict__ src, int n, int rows, int K, int mode,
                                    uint8_t* __restrict__ dst) {
  const int KG = K / kKGroup, MT = rows / 256;
  const size_t total = (size_t)n * rows * (K / 2) / 16;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int c16 = (int)(i & 3);
    const int rr = (int)((i >> 2) & 255);
    const size_t rest = i >> 10;  // (e * MT + mt) * KG + kg
    const int kg = (int)(rest % KG);
    const size_t emt = rest / KG;
    const int mt = (int)(emt % MT);
    const size_t e = emt / MT;
    int row;
    if (mode == 0) row = rr < 128 ? mt * 128 + rr : rows / 2 + mt * 128 + (rr - 128);
    else row = mt * 256 + rr;
    const uint4 v = *reinterpret_cast<const uint4*>(src + (e * rows + row) * (size_t)(K / 2) + kg * 64 + c16 * 16);
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
}

// scales [n, rows, K/32] -> atoms [n, rows/256, K/128, 2, 512]
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
    const size_t blk = (((e * MT + tile) * groups + grp) * 2 + half);
    *reinterpret_cast<uint32_t*>(atoms + blk * kSfAtomBytes + (lr & 31) * 16 + (lr >> 5) * 4) = word;
  }
}

// out[t, c] = bf16( sum_j Yr[inv_pos[t, j], c] + Yr[R + t, c] ), fp32 rows, 8 columns per thread
__global__ void combine_kernel(const float* __restrict__ y_rows, const int32_t* __restrict__ inv_pos, int T, int d,
                               int k, int R, int has_shared, __nv_bfloat16* __restrict__ out) {
  const int vec_per_row = d / 8;
  const size_t total = (size_t)T * vec_per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / vec_per_row), c8 = (int)(i % vec_per_row);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    auto add_row = [&](int r) {
      const float4* src = reinterpret_cast<const float4*>(y_rows + (size_t)r * d) + 2 * c8;
      const float4 a = __ldg(src), b = __ldg(src + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    };
    for (int j = 0; j < k; ++j) add_row(__ldg(&inv_pos[(size_t)t * k + j]));
    if (has_shared) add_row(R + t);
    uint4 o;
    __nv_bfloat16* ov = reinterpret_cast<__nv_bfloat16*>(&o);
#pragma unroll
    for (int q = 0; q < 8; ++q) ov[q] = __float2bfloat16_rn(acc[q]);
    reinterpret_cast<uint4*>(out + (size_t)t * d)[c8] = o;
  }
}

}  // namespace

cudaError_t launch_histogram(const int32_t* ids, int T, int k, int E, int G, int32_t* chunk_hist, int* status,
                             cudaStream_t s) {
  const int n_chunks = (T + 31) / 32;
  const int warps = 8;
  const int blocks = (n_chunks + warps - 1) / warps;
  histogram_kernel<<<blocks, warps * 32, (size_t)warps * G * sizeof(int), s>>>(ids, T, k, E, G, n_chunks, chunk_hist,
                                                                               status);
  return cudaGetLastError();
}

cudaError_t launch_scan(int32_t* chunk_hist, int n_chunks, int T, int E, int G, int has_shared, int bn, int max_tiles,
                        int32_t* counts, int32_t* offsets, int32_t* tile_off, int32_t* n_tiles, RowTile* tiles,
                        int* status, cudaStream_t s) {
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  scan_kernel<<<1, 1024, 0, s>>>(chunk_hist, n_chunks, T, E, G, has_shared, bn, max_tiles, counts, offsets, tile_off,
                                 n_tiles, tiles, status);
  return cudaGetLastError();
}

cudaError_t launch_tiles_from_offsets(const int32_t* offsets, int G, int n_rows, int bn, int max_tiles,
                                      int32_t* tile_off, int32_t* n_tiles, RowTile* tiles, int* status,
                                      cudaStream_t s) {
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  tiles_from_offsets_kernel<<<1, 1024, 0, s>>>(offsets, G, n_rows, bn, max_tiles, tile_off, n_tiles, tiles, status);
  return cudaGetLastError();
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* ids, const float* wts, const int32_t* chunk_hist,
                          const int32_t* offsets, const int32_t* tile_off, int T, int d, int k, int E, int G,
                          int has_shared, int bn, uint8_t* a_q, uint8_t* a_sf_atoms, uint8_t* a_s_rows,
                          int32_t* perm_tok, int32_t* inv_pos, float* row_w, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (T * 32 + threads - 1) / threads;
  gather_kernel<<<blocks, threads, 0, s>>>(x, ids, wts, chunk_hist, offsets, tile_off, T, d, k, E, G, has_shared, bn,
                                           a_q, a_sf_atoms, a_s_rows, perm_tok, inv_pos, row_w);
  return cudaGetLastError();
}

cudaError_t launch_rows_sf_to_atoms(const uint8_t* a_s_rows, const RowTile* tiles, const int32_t* n_tiles, int d,
                                    int max_tiles, uint8_t* atoms, cudaStream_t s) {
  rows_sf_to_atoms_kernel<<<296, 256, 0, s>>>(a_s_rows, tiles, n_tiles, d, max_tiles, atoms);
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

cudaError_t launch_combine(const float* y_rows, const int32_t* inv_pos, int T, int d, int k, int R,
                           int has_shared, __nv_bfloat16* out, cudaStream_t s) {
  const size_t total = (size_t)T * (d / 8);
  int blocks = (int)((total + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  combine_kernel<<<blocks, 256, 0, s>>>(y_rows, inv_pos, T, d, k, R, has_shared, out);
  return cudaGetLastError();
}

}  // namespace moe
