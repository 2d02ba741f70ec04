// The dispatch state of a batch written by one CTA from its routing alone -- what the histogram and the
// two scan kernels compute (moe_dispatch.cu), for batches small enough that the last CTA of the routing
// kernel does it sooner than three more launches would.  The permutation it describes is the same: rows
// expert-major, tokens ascending inside an expert (the single-GPU dispatch of the pypto page's "MoE and
// output stages"), then one shared row per token.
#pragma once

#include "moe_device.cuh"

namespace moe {

// Where the state goes (all device memory of the workspace).
struct DispatchOut {
  int G, has_shared, bn, max_tiles;
  int pad_pairs;        // every non-empty group gets an even number of tiles (the CTA-pair GEMMs)
  int32_t* chunk_base;  // [G][n_chunks] exclusive base of each 32-token chunk's rows inside its group
  int32_t* counts;      // [G]
  int32_t* offsets;     // [G + 1]
  int32_t* tile_off;    // [G + 1]
  int32_t* n_tiles;     // [1]
  RowTile* tiles;       // [max_tiles]
};

// Batches the writer takes: at most 32 chunks of 32 rows, so that one warp lane holds one chunk.
constexpr int kDispatchStateMaxT = 1024;

// Shared-memory ints the writer needs for a batch of T rows.
__host__ __device__ constexpr int dispatch_state_smem_ints(int G, int T) { return G * ((T + 31) / 32) + 3 * G + 2 + 64; }

// Exclusive prefix of (a, b) over the CTA's threads (blockDim.x a multiple of 32, at most 1024); totals in
// *ta, *tb.  wsum: 64 ints of shared scratch.  Every thread of the CTA calls it.
__device__ __forceinline__ void block_scan2(int a, int b, int* ea, int* eb, int* ta, int* tb, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int oa = __shfl_up_sync(0xFFFFFFFFu, ia, off), ob = __shfl_up_sync(0xFFFFFFFFu, ib, off);
    if (lane >= off) {
      ia += oa;
      ib += ob;
    }
  }
  if (lane == 31) {
    wsum[warp] = ia;
    wsum[32 + warp] = ib;
  }
  __syncthreads();
  int ba = 0, bb = 0, sa = 0, sb = 0;
  for (int q = 0; q < nw; ++q) {
    const int xa = wsum[q], xb = wsum[32 + q];
    if (q < warp) {
      ba += xa;
      bb += xb;
    }
    sa += xa;
    sb += xb;
  }
  *ea = ba + ia - a;
  *eb = bb + ib - b;
  *ta = sa;
  *tb = sb;
  __syncthreads();  // wsum is reused by the next call
}

// Called by every thread of one CTA, after the routing ids [T, k] (device memory, written by this kernel's
// CTAs, made visible by the caller's fences) are final; T <= kDispatchStateMaxT.
// smem: dispatch_state_smem_ints(G, T) ints.  Every phase spreads over all the CTA's threads: the histogram
// takes the ids in one coalesced pass into shared-memory atomics, a warp scans the chunks of one or more
// groups at a time, and each tile entry is written by its own thread.
__device__ inline void write_dispatch_state(const int32_t* ids, int T, int k, int E, const DispatchOut& o, int* smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int G = o.G, n_chunks = (T + 31) / 32;
  int* h = smem;                // [n_chunks][G] rows of each group in each chunk
  int* cnt = h + G * n_chunks;  // [G]
  int* roff = cnt + G;          // [G + 1] row offsets
  int* toff = roff + G + 1;     // [G + 1] tile offsets
  int* wsum = toff + G + 1;     // [64]
  for (int i = threadIdx.x; i < G * n_chunks; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int rows_per_chunk = 32 * k;
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    int e = __ldcg(&ids[i]);
    if (e < 0 || e >= E) e = 0;  // an id outside [0, E) counts as expert 0, as the gather places it
    atomicAdd(&h[(i / rows_per_chunk) * G + e], 1);
  }
  __syncthreads();
  // per group: exclusive bases over its chunks and its row count (the shared group holds all T rows and
  // needs no bases).  A warp takes 32 / W groups at once, W = n_chunks rounded up to a power of two, and
  // scans each group's chunks inside its own W-lane segment.
  int W = 1;
  while (W < n_chunks) W <<= 1;
  const int per_warp = 32 / W, c = lane & (W - 1);
  for (int g0 = warp * per_warp; g0 < G; g0 += nw * per_warp) {
    const int g = g0 + lane / W;
    const bool live = g < G && !(o.has_shared && g == E);
    const int v = live && c < n_chunks ? h[c * G + g] : 0;
    int incl = v;
    for (int off = 1; off < W; off <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, incl, off, W);
      if (c >= off) incl += u;
    }
    const int total = __shfl_sync(0xFFFFFFFFu, incl, W - 1, W);
    if (live && c < n_chunks) o.chunk_base[(size_t)g * n_chunks + c] = incl - v;
    if (g < G && c == 0) {
      const int n = live ? total : T;
      cnt[g] = n;
      o.counts[g] = n;
    }
  }
  __syncthreads();
  // over groups: row offsets and tile offsets
  int carry_r = 0, carry_t = 0;
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    const int n = g < G ? cnt[g] : 0;
    int nt = (n + o.bn - 1) / o.bn;
    if (o.pad_pairs) nt += nt & 1;
    int er, et, tr, tt;
    block_scan2(n, nt, &er, &et, &tr, &tt, wsum);
    if (g < G) {
      roff[g] = carry_r + er;
      toff[g] = carry_t + et;
      o.offsets[g] = carry_r + er;
      o.tile_off[g] = carry_t + et;
    }
    carry_r += tr;
    carry_t += tt;
  }
  if (threadIdx.x == 0) {
    roff[G] = carry_r;
    toff[G] = carry_t;
    o.offsets[G] = carry_r;
    o.tile_off[G] = carry_t;
    *o.n_tiles = min(carry_t, o.max_tiles);
  }
  __syncthreads();
  // the tile list: tile i belongs to the last group whose tile offset is <= i
  const int n_t = min(carry_t, o.max_tiles);
  for (int i = threadIdx.x; i < n_t; i += blockDim.x) {
    int lo = 0, hi = G;  // toff[lo] <= i < toff[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (toff[mid] <= i) lo = mid;
      else hi = mid;
    }
    const int q = i - toff[lo];
    RowTile rt;
    rt.group = lo;
    rt.row0 = roff[lo] + q * o.bn;
    rt.nrows = max(0, min(o.bn, cnt[lo] - q * o.bn));
    rt.pad = 0;
    o.tiles[i] = rt;
  }
}

}  // namespace moe
