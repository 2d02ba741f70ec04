// Checkpoint ingest: arrays of 17-byte MXFP4 blocks (one E8M0 scale byte, then 16 bytes holding 32 E2M1
// codes) -> the canonical codes and scales that moe_experts_create takes.  The model card's "Conversion
// to the .fst container" stores experts as such blocks; the TensorSharp page ("Getting a drafter") says
// the checkpoint's layout is GGUF's MXFP4 "up to nibble order".  Two nibble orders are read:
//   paired (MOE_MX_NIBBLES_PAIRED): byte i holds elements 2i (low nibble) and 2i+1 (high nibble) --
//                                   the canonical order, so only the scale moves out;
//   split  (MOE_MX_NIBBLES_SPLIT):  byte i holds elements i (low nibble) and i+16 (high nibble).
// A [rows x K] matrix stored as rows * K/32 blocks in row-major order unpacks to codes [rows][K/2] and
// scales [rows][K/32].
#include "moe_device.cuh"

namespace moe {

namespace {

// one thread per block; blocks sit at a 17-byte stride, so they are read byte by byte
__global__ void mx_blocks_unpack_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, int split,
                                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  pdl_trigger();
  pdl_wait();
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < n_blocks; b += (int64_t)gridDim.x * blockDim.x) {
    const uint8_t* src = blocks + b * 17;
    uint8_t q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = src[1 + i];
    uint32_t out[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * w + j;  // output byte: elements 2i, 2i+1
        uint32_t lo, hi;
        if (split) {
          const int e0 = 2 * i, e1 = 2 * i + 1;  // element e lives in byte e % 16, high nibble if e >= 16
          lo = e0 < 16 ? (q[e0] & 0xFu) : (q[e0 - 16] >> 4);
          hi = e1 < 16 ? (q[e1] & 0xFu) : (q[e1 - 16] >> 4);
        } else {
          lo = q[i] & 0xFu;
          hi = q[i] >> 4;
        }
        v |= (lo | (hi << 4)) << (8 * j);
      }
      out[w] = v;
    }
    uint8_t* dst = codes + b * 16;
    if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = (uint8_t)(out[i >> 2] >> (8 * (i & 3)));
    }
    scales[b] = src[0];
  }
}

}  // namespace

}  // namespace moe

extern "C" MOE_API moe_status_t moe_mx_blocks_unpack(const uint8_t* blocks, int64_t n_blocks, int32_t nibble_order,
                                                     uint8_t* codes, uint8_t* scales, moe_stream_t stream) {
  if (n_blocks < 0) {
    moe::set_last_error("n_blocks is negative");
    return MOE_ERR_INVALID_ARG;
  }
  if (n_blocks == 0) return MOE_OK;
  if (!blocks || !codes || !scales) {
    moe::set_last_error("a buffer is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (nibble_order != MOE_MX_NIBBLES_PAIRED && nibble_order != MOE_MX_NIBBLES_SPLIT) {
    moe::set_last_error("unknown nibble order");
    return MOE_ERR_INVALID_ARG;
  }
  const int64_t want = (n_blocks + 255) / 256;
  const int grid = (int)(want < 152 * 32 ? want : 152 * 32);
  const cudaError_t e =
      moe::launch_pdl(moe::mx_blocks_unpack_kernel, dim3(grid), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                      blocks, n_blocks, nibble_order == MOE_MX_NIBBLES_SPLIT ? 1 : 0, codes, scales);
  if (e != cudaSuccess) {
    moe::set_last_error(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
