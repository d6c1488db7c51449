// k_repack.cu -- weights -> MMA-ready tiles (run once at layer creation).
//
// Input: the Q8_0 layout of the Q8_0 lm_head re-quantiser (gemma4/model.rs): per row,
// cols/32 blocks of 34 bytes = fp16 scale d (little endian) + 32 int8 q.  The 34-byte
// stride is not 16-byte aligned, so the decode GEMV could not use 128-bit loads on it.
// Output (values untouched, only moved): one 544-byte tile per 16 rows x 32 columns,
//   bytes [0, 512): lane l = 4g + t owns bytes [16l, 16l+16): word 0 = row g, word 1 =
//     row g+8 for columns {2t, 2t+1, 2t+8, 2t+9} of the block's first 16 columns;
//     words 2, 3 the same for columns 16 + {...}.  Each byte stores q + 128 (so the GEMV
//     converts it to fp16 without a sign step).
//   bytes [512, 544): 8 half2, entry g = (d[row g], d[row g + 8]).
#include "hfa_common.cuh"
#include "hfa_internal.h"

namespace hfa {

// Tile (row group r, block b) of a matrix with R_total row groups lands at index
// ((b / nbs) * R_total + rg) * nbs + b % nbs, rg = row_group0 + r * rg_stride: the row
// groups of one k-split of nbs blocks are then one contiguous byte range, which the
// persistent kernels copy in bulk (rg_stride 2 interleaves two matrices' row groups).
__global__ void repack_q8_0_split_kernel(const uint8_t* __restrict__ src, int rows, int cols,
                                         uint8_t* __restrict__ dst, int row_group0, int rg_stride,
                                         int R_total, int nbs) {
  const int nb = cols / 32;
  const long long n = (long long)(rows / 16) * nb * 32;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(idx & 31);
    const long long tile = idx >> 5;
    const int b = (int)(tile % nb);
    const int r = (int)(tile / nb);
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* row_g = src + (size_t)(16 * r + g) * nb * 34 + (size_t)b * 34;
    const uint8_t* row_g8 = row_g + (size_t)8 * nb * 34;
    uint32_t w[4];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint8_t* rp = half ? row_g8 : row_g;
        const int c0 = 16 * ks + 2 * t;
        const int cs[4] = {c0, c0 + 1, c0 + 8, c0 + 9};
        uint32_t v = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) v |= (uint32_t)((uint8_t)(rp[2 + cs[e]] + 128u)) << (8 * e);
        w[2 * ks + half] = v;
      }
    }
    const long long out_tile =
        ((long long)(b / nbs) * R_total + (row_group0 + (long long)r * rg_stride)) * nbs + (b % nbs);
    uint8_t* tp = dst + out_tile * kQ8TileBytes;
    reinterpret_cast<uint4*>(tp)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
    if (t == 0) {
      __half dg = __ushort_as_half((unsigned short)(row_g[0] | (row_g[1] << 8)));
      __half dg8 = __ushort_as_half((unsigned short)(row_g8[0] | (row_g8[1] << 8)));
      reinterpret_cast<__half2*>(tp + 512)[g] = __halves2half2(dg, dg8);
    }
  }
}

cudaError_t launch_repack_q8_0_split(const uint8_t* src, int rows, int cols, uint8_t* dst,
                                     int row_group0, int R_total, int nbs, cudaStream_t s,
                                     int rg_stride) {
  long long n = (long long)(rows / 16) * (cols / 32) * 32;
  int threads = 256;
  long long blocks = (n + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;
  repack_q8_0_split_kernel<<<(int)blocks, threads, 0, s>>>(src, rows, cols, dst, row_group0,
                                                           rg_stride, R_total, nbs);
  return cudaGetLastError();
}

// bf16 matrix [rows, K] (rows 0 .. n0-1 from s0, the next n1 from s1, the rest from
// s2) -> the shared-memory image of the verify GEMM's A stages: tile (m, c) of 128 rows x
// 64 columns is 16 KB at ((m * K / 64) + c) * 16 KB, row r of the tile at r * 128 bytes,
// its 16-byte group j at position j XOR (r mod 8) -- the 128-byte swizzle the tensor-core
// descriptors read.  The row tiles of one matrix stream as one contiguous range each.
__global__ void repack_bf16_tiles_kernel(const __nv_bfloat16* __restrict__ s0, int n0,
                                         const __nv_bfloat16* __restrict__ s1, int n1,
                                         const __nv_bfloat16* __restrict__ s2, int rows, int K,
                                         uint8_t* __restrict__ dst) {
  const int g8 = K / 8;  // 16-byte groups per row
  const long long n = (long long)rows * g8;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n;
       u += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(u / g8), j8 = (int)(u - (long long)row * g8);
    const __nv_bfloat16* src = row < n0        ? s0 + (size_t)row * K
                               : row < n0 + n1 ? s1 + (size_t)(row - n0) * K
                                               : s2 + (size_t)(row - n0 - n1) * K;
    const uint4 v = *reinterpret_cast<const uint4*>(src + j8 * 8);
    const int m = row >> 7, r = row & 127, c = j8 >> 3, j = j8 & 7;
    const size_t off = (((size_t)m * (K / 64) + c) * 128 + r) * 128 + ((j ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(dst + off) = v;
  }
}

cudaError_t launch_repack_bf16_tiles(const __nv_bfloat16* s0, int n0, const __nv_bfloat16* s1,
                                     int n1, const __nv_bfloat16* s2, int rows, int K,
                                     uint8_t* dst, cudaStream_t s) {
  const long long n = (long long)rows * (K / 8);
  long long blocks = (n + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  repack_bf16_tiles_kernel<<<(int)blocks, 256, 0, s>>>(s0, n0, s1, n1, s2, rows, K, dst);
  return cudaGetLastError();
}

}  // namespace hfa
