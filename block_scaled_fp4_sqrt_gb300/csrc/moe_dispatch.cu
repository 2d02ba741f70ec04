// Token <-> expert dispatch and combine (the single-GPU form of the pypto page's "dispatch /
// combine" around expert_routed / expert_shared, "MoE and output stages"):
//
//  * histogram:  per 32-token chunk, how many (token, slot) pairs go to each expert group (a warp vote,
//                match.any + popc, per routing slot);
//  * scans:      per group, exclusive sums over its chunks (one block per group); over groups, row
//                offsets, tile offsets and a device-side list of row tiles for the grouped GEMMs (one
//                block, warp-shuffle scans; no host round trip);
//  * gather:     MXFP8 quantisation of each token row (E4M3, one E8M0 scale per 32 along d) and its
//                copy to every expert row it is routed to, expert-major with tokens ascending inside an
//                expert (deterministic: a token's rank comes from a warp ballot over the lower tokens of
//                its chunk plus the chunk's exclusive base, no atomics);
//  * combine:    out[t] = sum_j Yr[inv_pos[t, j]] + Yr[R + t] in fp32, in the fixed order j = 0..k-1
//                then the shared row, rounded once to bf16 (the weighted-sum epilogue; the routing
//                weight was applied in the down GEMM).
#include "moe_device.cuh"

namespace moe {

namespace {

constexpr int kMaxGroups = 2048;

__device__ __forceinline__ int clamp_id(int e, int E, int* status) {
  if (e < 0 || e >= E) {
    set_status(status, DEV_BAD_EXPERT_ID);
    return 0;
  }
  return e;
}

// One warp per 32-token chunk; chunk_hist[g][c] = number of (t, j) in chunk c with ids[t, j] = g.
// Warp-vote histogram: for each routing slot j, match.any gives every lane the set of lanes whose token
// chose the same expert, and the lowest lane of each set adds the set's population count.  Within one
// slot the adding lanes hold distinct experts, so the warp's private histogram needs no atomics.
__global__ void histogram_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int G, int n_chunks,
                                 int32_t* __restrict__ chunk_hist, int* status) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sh_hist[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * (blockDim.x >> 5) + warp;
  int* h = sh_hist + warp * G;
  for (int g = lane; g < G; g += 32) h[g] = 0;
  __syncwarp();
  if (chunk < n_chunks) {
    const int t = chunk * 32 + lane;
    for (int j = 0; j < k; ++j) {
      const int e = t < T ? clamp_id(ids[(size_t)t * k + j], E, status) : -1;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
      if (e >= 0 && (peers & ((1u << lane) - 1u)) == 0u) h[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncwarp();
  if (chunk < n_chunks)
    for (int g = lane; g < G; g += 32) chunk_hist[(size_t)g * n_chunks + chunk] = h[g];
}

// Exclusive scan of one int per thread over the block (blockDim.x a multiple of 32, at most 1024);
// returns the thread's exclusive prefix and the block total in *total.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += o;
    }
    warp_sums[lane] = w;  // inclusive prefix of the warp totals
  }
  __syncthreads();
  const int before = warp ? warp_sums[warp - 1] : 0;
  *total = warp_sums[nwarps - 1];
  __syncthreads();
  return before + incl - v;
}

// One block per group: the group's chunk counts (chunk_hist[g][*]) become exclusive bases in place, and
// its total goes to counts[g].  The shared group (index E when has_shared) holds all T rows.
__global__ void __launch_bounds__(256) colscan_kernel(int32_t* __restrict__ chunk_hist, int n_chunks, int T, int E,
                                                      int has_shared, int32_t* __restrict__ counts) {
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.x;
  if (has_shared && g == E) {
    if (threadIdx.x == 0) counts[g] = T;
    return;
  }
  int32_t* row = chunk_hist + (size_t)g * n_chunks;
  int carry = 0;
  for (int base = 0; base < n_chunks; base += blockDim.x) {
    const int c = base + threadIdx.x;
    const int v = c < n_chunks ? row[c] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, &tot);
    if (c < n_chunks) row[c] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) counts[g] = carry;
}

// Single block: per-group row counts (from counts, from caller offsets, or one group of n_rows) ->
// offsets [G+1] (if requested), tile offsets [G+1], and the list of row tiles of at most bn rows.  With
// pad_pairs every non-empty group gets an even number of tiles (the last one, if added, holds no rows).
__global__ void __launch_bounds__(1024) groupscan_kernel(const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets_in, int G, int n_rows,
                                                         int bn, int max_tiles, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ tile_off,
                                                         int32_t* __restrict__ n_tiles, RowTile* __restrict__ tiles,
                                                         int* status, int pad_pairs) {
  __shared__ int s_cnt[kMaxGroups], s_off[kMaxGroups], s_toff[kMaxGroups];
  __shared__ int bad;
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) bad = (offsets_in && (offsets_in[0] != 0 || offsets_in[G] != n_rows)) ? 1 : 0;
  __syncthreads();
  int carry_r = 0, carry_t = 0;
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    int c = 0;
    if (g < G) {
      if (offsets_in) {
        c = offsets_in[g + 1] - offsets_in[g];
        if (c < 0) {
          bad = 1;
          c = 0;
        }
      } else {
        c = counts ? counts[g] : n_rows;
      }
    }
    int tot_r, tot_t;
    int nt = (c + bn - 1) / bn;
    if (pad_pairs) nt += nt & 1;
    const int ex_r = block_exclusive_scan(c, &tot_r);
    const int ex_t = block_exclusive_scan(nt, &tot_t);
    if (g < G) {
      s_cnt[g] = c;
      s_off[g] = offsets_in ? offsets_in[g] : carry_r + ex_r;
      s_toff[g] = carry_t + ex_t;
      if (offsets) offsets[g] = carry_r + ex_r;
      tile_off[g] = carry_t + ex_t;
    }
    carry_r += tot_r;
    carry_t += tot_t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (offsets) offsets[G] = carry_r;
    tile_off[G] = carry_t;
    if (bad) {
      set_status(status, DEV_BAD_WORK);
      *n_tiles = 0;
    } else {
      if (carry_t > max_tiles) set_status(status, DEV_BAD_WORK);
      *n_tiles = min(carry_t, max_tiles);
    }
  }
  __syncthreads();
  if (bad) return;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int cnt = s_cnt[g];
    int nt = (cnt + bn - 1) / bn;
    if (pad_pairs) nt += nt & 1;
    for (int i = 0; i < nt; ++i) {
      const int idx = s_toff[g] + i;
      if (idx < max_tiles) {
        RowTile rt;
        rt.group = g;
        rt.row0 = s_off[g] + i * bn;
        rt.nrows = max(0, min(bn, cnt - i * bn));
        rt.pad = 0;
        tiles[idx] = rt;
      }
    }
  }
}

// One block per token, one thread per 32-element MXFP8 block.
//  * The token's x row is loaded first: nothing about it depends on the routing.
//  * The ids of the token's 32-token chunk go to shared memory; warp 0 takes one ballot per routing
//    slot j (rank of the token among the lower tokens of its chunk that chose the same expert), and
//    lanes 0..k-1 then look up their expert's chunk base and offsets at the same time, so the block
//    waits for one round of dependent loads instead of k.  The destinations (k routed rows and the
//    shared row) are published in shared memory.
//  * Each warp quantises 32 MX blocks (1 KB of E4M3) and stores them to every destination row with two
//    instructions of 512 contiguous bytes (lane l stores 16-byte chunk l of each half, moved there by
//    shuffles); four consecutive threads (one 128-element K group) pack their scale bytes into one
//    32-bit word, which is one word of a scale atom.
//  * FP4 (the MXFP4-activation variant): the warp's 32 blocks are 512 bytes of packed E2M1 codes, and
//    lane l's 16 bytes are chunk l of them: one store per destination row, no shuffles.
template <bool FP4>
__global__ void __launch_bounds__(128) gather_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ ids, const float* __restrict__ wts,
    const int32_t* __restrict__ chunk_base, int n_chunks, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ tile_off, int T, int d, int k, int E, int has_shared, int bn,
    uint8_t* __restrict__ a_q, uint8_t* __restrict__ a_sf_atoms, uint8_t* __restrict__ a_s_rows,
    int32_t* __restrict__ perm_tok, int32_t* __restrict__ inv_pos, float* __restrict__ row_w) {
  constexpr int kMaxDst = 17;  // top-k <= 16, plus the shared row
  __shared__ int s_ids[32 * 16];
  __shared__ int s_row[kMaxDst], s_tile[kMaxDst], s_n[kMaxDst];
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = d / 32;
  const int n_dst = k + (has_shared ? 1 : 0);
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const int chunk = t >> 5, tc = t & 31;
    // 1. this thread's first MX block of the row (the loop below loads the rest, if d > 32 * threads)
    uint4 raw[4];
    {
      const int b = threadIdx.x;
      if (b < nb) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + b * 32);
#pragma unroll
        for (int c = 0; c < 4; ++c) raw[c] = __ldg(src + c);
      }
    }
    // 2. the chunk's ids
    for (int i = threadIdx.x; i < 32 * k; i += blockDim.x) {
      const int tt = (chunk << 5) + i / k;
      s_ids[i] = tt < T ? clamp_id(__ldg(&ids[(size_t)(chunk << 5) * k + i]), E, nullptr) : -1;
    }
    __syncthreads();
    // 3. destinations
    if (warp == 0) {
      int my_ids[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) my_ids[jj] = jj < k ? s_ids[lane * k + jj] : -2;
      int my_e = 0, my_rank = 0;
      for (int j = 0; j < k; ++j) {
        const int e = s_ids[tc * k + j];
        bool hit = false;
        if (lane < tc) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) hit |= my_ids[jj] == e;
        }
        const int rank = __popc(__ballot_sync(0xFFFFFFFFu, hit));
        if (lane == j) {
          my_e = e;
          my_rank = rank;
        }
      }
      if (lane < k) {
        const int local = chunk_base[(size_t)my_e * n_chunks + chunk] + my_rank;
        const int row = offsets[my_e] + local;
        s_row[lane] = row;
        s_tile[lane] = tile_off[my_e] + local / bn;
        s_n[lane] = local % bn;
        perm_tok[row] = t;
        inv_pos[(size_t)t * k + lane] = row;
        if (row_w) row_w[row] = wts ? wts[(size_t)t * k + lane] : 1.0f;
      } else if (lane == k && has_shared) {
        const int row = offsets[E] + t;
        s_row[lane] = row;
        s_tile[lane] = tile_off[E] + t / bn;
        s_n[lane] = t % bn;
        perm_tok[row] = t;
        if (row_w) row_w[row] = 1.0f;
      }
    }
    __syncthreads();
    // 4. quantise and store
    for (int b0 = 0; b0 < nb; b0 += blockDim.x) {
      const int b = b0 + threadIdx.x;
      const bool on = b < nb;
      if (b0 > 0 && on) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + b * 32);
#pragma unroll
        for (int c = 0; c < 4; ++c) raw[c] = __ldg(src + c);
      }
      uint32_t packed[8];
      uint32_t byte = 0;
      if (on) {
        float v[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[c * 8 + i] = __bfloat162float(hv[i]);
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const int se = FP4 ? mxfp4_block_exp(amax) : mxfp8_block_exp(amax);
        const float mul = exp2_neg_int(se);
        if (FP4) {
          const uint4 c = e2m1_block(v, mul);
          packed[0] = c.x;
          packed[1] = c.y;
          packed[2] = c.z;
          packed[3] = c.w;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t lo = e4m3x2(v[4 * i] * mul, v[4 * i + 1] * mul);
            const uint32_t hi = e4m3x2(v[4 * i + 2] * mul, v[4 * i + 3] * mul);
            packed[i] = lo | (hi << 16);
          }
        }
        byte = (uint32_t)(se + 127);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) packed[i] = 0u;
      }
      uint32_t word = byte;
      word |= __shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8;
      word |= __shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16;
      word |= __shfl_down_sync(0xFFFFFFFFu, byte, 3) << 24;
      // the warp's 32 MX blocks are 64 chunks of 16 bytes; half h of the stores is chunks 32h .. 32h+31,
      // and chunk c is half (c & 1) of MX block c / 2, i.e. of lane c / 2 of this warp
      const int wb0 = b - lane;  // the warp's first MX block
      uint4 outv[2];
#pragma unroll
      for (int h = 0; h < (FP4 ? 0 : 2); ++h) {
        const int src_lane = 16 * h + (lane >> 1);
        uint32_t w4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = __shfl_sync(0xFFFFFFFFu, packed[j], src_lane);
          const uint32_t hi = __shfl_sync(0xFFFFFFFFu, packed[4 + j], src_lane);
          w4[j] = (lane & 1) ? hi : lo;
        }
        outv[h] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      const int grp = b >> 2;
      for (int q = 0; q < n_dst; ++q) {
        const int row = s_row[q];
        if (FP4) {
          if (on) reinterpret_cast<uint4*>(a_q + (size_t)row * (d / 2))[b] =
              make_uint4(packed[0], packed[1], packed[2], packed[3]);
        } else {
          uint8_t* rowp = a_q + (size_t)row * d;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int blk = wb0 + 16 * h + (lane >> 1);  // MX block whose half this lane stores
            if (blk < nb) reinterpret_cast<uint4*>(rowp + (size_t)blk * 32)[lane & 1] = outv[h];
          }
        }
        if (on && (b & 3) == 0) {
          if (a_sf_atoms) {
            const int n = s_n[q];
            *reinterpret_cast<uint32_t*>(a_sf_atoms + ((size_t)s_tile[q] * (d / kKGroup) + grp) * kSfAtomBytes +
                                         (n & 31) * 16 + ((n >> 5) & 3) * 4) = word;
          }
          if (a_s_rows) *reinterpret_cast<uint32_t*>(a_s_rows + (size_t)row * nb + b) = word;
        }
      }
    }
    __syncthreads();  // s_ids and the destinations are rewritten by the next token
  }
}

// out[t, c] = bf16( sum_j Yr[inv_pos[t, j], c] + Yr[R + t, c] ) in fp32; the rows are scaled fp16 (ExpertRows:
// value * 2^(byte - 127), one byte per 32 columns), exact in fp32.  A block takes one token at a time and
// a thread 16 columns of it: two 16-byte loads and one scale byte per row, all rows' loads in flight at
// once (the combine streams the rows from HBM, so bytes in flight per thread set its speed).
// F32OUT writes the same fp32 sum without the final rounding (the test hook moe_testing_read_y32).
template <bool F32OUT>
__global__ void __launch_bounds__(256, 2) combine_kernel(ExpertRows y_rows, const int32_t* __restrict__ inv_pos, int T,
                                                      int d, int k, int R, int has_shared,
                                                      const __nv_bfloat16* residual, void* out_) {
  pdl_trigger();
  pdl_wait();
  const int vec_per_row = d / 16, nb = d / 32;
  const __half* __restrict__ yv = y_rows.val;
  const uint8_t* __restrict__ ye = y_rows.exp;
  const int n = k + (has_shared ? 1 : 0);
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) {
      float acc[16];
      if (residual) {  // a residual stream enters first: out = bf16(x + sum of the rows); out may alias it
        const uint4* rp = reinterpret_cast<const uint4*>(residual + (size_t)t * d) + 2 * c;
        const uint4 r0 = rp[0], r1 = rp[1];
        const __nv_bfloat16* h0 = reinterpret_cast<const __nv_bfloat16*>(&r0);
        const __nv_bfloat16* h1 = reinterpret_cast<const __nv_bfloat16*>(&r1);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[q] = __bfloat162float(h0[q]);
          acc[8 + q] = __bfloat162float(h1[q]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = 0.f;
      }
      auto add = [&](uint4 v, float sc, int o) {
        const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(h2[q]);
          acc[o + 2 * q] += f.x * sc;
          acc[o + 2 * q + 1] += f.y * sc;
        }
      };
      if (n <= 8) {
        // all row indices, then all row loads, then the sum in slot order
        int rows[8];
        uint4 va[8], vb[8];
        uint32_t e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          rows[j] = j < k ? __ldg(&inv_pos[(size_t)t * k + j]) : (j == k && has_shared ? R + t : -1);
        const uint4* yv4 = reinterpret_cast<const uint4*>(yv) + 2 * c;
        const uint8_t* yec = ye + (c >> 1);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (rows[j] >= 0) {  // 32-bit offsets: rows * d / 8 stays below 2^32 for every workspace size
            const uint32_t o = (uint32_t)rows[j] * (uint32_t)(d / 8);
            va[j] = __ldg(yv4 + o);
            vb[j] = __ldg(yv4 + o + 1);
            e[j] = __ldg(yec + (uint32_t)rows[j] * (uint32_t)nb);
          }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (rows[j] >= 0) {
            const float sc = row16_scale(e[j]);
            add(va[j], sc, 0);
            add(vb[j], sc, 8);
          }
      } else {
        auto add_row = [&](int r) {
          const uint4* p = reinterpret_cast<const uint4*>(yv + (size_t)r * d) + 2 * c;
          const float sc = row16_scale(__ldg(ye + (size_t)r * nb + (c >> 1)));
          add(__ldg(p), sc, 0);
          add(__ldg(p + 1), sc, 8);
        };
        for (int j = 0; j < k; ++j) add_row(__ldg(&inv_pos[(size_t)t * k + j]));
        if (has_shared) add_row(R + t);
      }
      if (F32OUT) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out_) + (size_t)t * d) + 4 * c;
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
      } else {
        uint4 o[2];
        __nv_bfloat16* ov = reinterpret_cast<__nv_bfloat16*>(o);
#pragma unroll
        for (int q = 0; q < 16; ++q) ov[q] = __float2bfloat16_rn(acc[q]);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_) + (size_t)t * d) + 2 * c;
        dst[0] = o[0];
        dst[1] = o[1];
      }
    }
  }
}

}  // namespace

cudaError_t launch_histogram(const int32_t* ids, int T, int k, int E, int G, int32_t* chunk_hist, int* status,
                             cudaStream_t s) {
  const int n_chunks = (T + 31) / 32;
  const int warps = 8;
  const int blocks = (n_chunks + warps - 1) / warps;
  return launch_pdl(histogram_kernel, dim3(blocks), dim3(warps * 32), (size_t)warps * G * sizeof(int), s, ids, T, k, E,
                    G, n_chunks, chunk_hist, status);
}

cudaError_t launch_scan(int32_t* chunk_hist, int n_chunks, int T, int E, int G, int has_shared, int bn, int max_tiles,
                        int32_t* counts, int32_t* offsets, int32_t* tile_off, int32_t* n_tiles, RowTile* tiles,
                        int* status, cudaStream_t s, int pad_pairs) {
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  const int threads = n_chunks >= 256 ? 256 : ((n_chunks + 31) / 32) * 32;
  cudaError_t e = launch_pdl(colscan_kernel, dim3(G), dim3(threads), 0, s, chunk_hist, n_chunks, T, E, has_shared,
                             counts);
  if (e != cudaSuccess) return e;
  return launch_pdl(groupscan_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)counts, (const int32_t*)nullptr, G, 0,
                    bn, max_tiles, offsets, tile_off, n_tiles, tiles, status, pad_pairs);
}

cudaError_t launch_tiles_from_offsets(const int32_t* offsets, int G, int n_rows, int bn, int max_tiles,
                                      int32_t* tile_off, int32_t* n_tiles, RowTile* tiles, int* status,
                                      cudaStream_t s, int pad_pairs) {
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  return launch_pdl(groupscan_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)nullptr, offsets, G, n_rows, bn,
                    max_tiles, (int32_t*)nullptr, tile_off, n_tiles, tiles, status, pad_pairs);
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* ids, const float* wts, const int32_t* chunk_hist,
                          const int32_t* offsets, const int32_t* tile_off, int T, int d, int k, int E, int G,
                          int has_shared, int bn, uint8_t* a_q, uint8_t* a_sf_atoms, uint8_t* a_s_rows,
                          int32_t* perm_tok, int32_t* inv_pos, float* row_w, int act_fp4, cudaStream_t s) {
  (void)G;
  const int n_chunks = (T + 31) / 32;
  const int nb = d / 32;
  const int threads = nb >= 128 ? 128 : ((nb + 31) / 32) * 32;
  const int blocks = T < 152 * 16 ? T : 152 * 16;
  if (act_fp4)
    return launch_pdl(gather_kernel<true>, dim3(blocks), dim3(threads), 0, s, x, ids, wts, chunk_hist, n_chunks,
                      offsets, tile_off, T, d, k, E, has_shared, bn, a_q, a_sf_atoms, a_s_rows, perm_tok, inv_pos,
                      row_w);
  return launch_pdl(gather_kernel<false>, dim3(blocks), dim3(threads), 0, s, x, ids, wts, chunk_hist, n_chunks,
                    offsets, tile_off, T, d, k, E, has_shared, bn, a_q, a_sf_atoms, a_s_rows, perm_tok, inv_pos, row_w);
}

cudaError_t launch_combine(ExpertRows y_rows, const int32_t* inv_pos, int T, int d, int k, int R,
                           int has_shared, const __nv_bfloat16* residual, __nv_bfloat16* out, cudaStream_t s,
                           float* out_f32) {
  if ((uint64_t)(R + (has_shared ? T : 0)) * (uint64_t)(d / 8) >= (1ull << 32)) return cudaErrorInvalidValue;
  const int vec_per_row = d / 16;
  const int threads = vec_per_row >= 256 ? 256 : ((vec_per_row + 31) / 32) * 32;
  int blocks = T < 152 * 8 ? T : 152 * 8;
  if (blocks < 1) blocks = 1;
  if (out_f32)
    return launch_pdl(combine_kernel<true>, dim3(blocks), dim3(threads), 0, s, y_rows, inv_pos, T, d, k, R,
                      has_shared, residual, static_cast<void*>(out_f32));
  return launch_pdl(combine_kernel<false>, dim3(blocks), dim3(threads), 0, s, y_rows, inv_pos, T, d, k, R,
                    has_shared, residual, static_cast<void*>(out));
}

}  // namespace moe
