// k_gemv.cu -- dequantising Q8_0 GEMV for the decode step.
//
// Two modes share one kernel body:
//  * kModeQKV  (pre-attention norm + QKV projection + per-head norm + RoPE + KV append):
//    gemma4/gpu_full_attn.rs, encode_one_layer: "Pre-attention norm", "QKV projections",
//    "Fused per-head RMS norm + RoPE on Q and K", "GPU V norm" and the dense KV copy.
//  * kModeOProj (o_proj + residual): encode_one_layer "O-proj"; the residual
//    connection of dflash/forward.rs (dispatch_dflash_residual_add, h = x + attn).
//
// Work split.  The weight matrix is a sequence of 16x32 tiles (row group r, k-block b)
// ordered (k-split s, r, b).  Each CTA takes a contiguous range of that sequence and each
// warp a contiguous sub-range, so every warp streams the same number of tiles (+-1).
// One 16-byte load per lane brings a whole tile; two m16n8k16 fp16 MMAs per tile and
// per batch tile multiply it with the activations.  Activations enter as fp16 hi + lo
// pairs (columns 2j and 2j+1 of the MMA's N dimension), which keeps about 22 bits of the
// fp32 value; int8 -> fp16 is exact, and the per-block fp16 scale multiplies the fp32
// partial products of each block.
//
// Completion.  Partial sums go to an fp32 accumulator with red.add; each warp then adds
// the number of tiles it finished to a per-head (QKV) or per-row-group (o_proj) ticket.
// The warp whose tiles complete a head / row group reads the sums back, resets them to
// zero and runs the epilogue for it.  No warp ever waits for another.
#include "hfa_common.cuh"
#include "hfa_finish.cuh"
#include "hfa_internal.h"

namespace hfa {

constexpr int kChunk = 8;        // tiles in flight per lane (16 B weights + 4 B scales each)
constexpr int kItemsPerCta = 8;  // warps per CTA, one work item each

template <int NT, int MODE>
__device__ __forceinline__ void flush_item(const GemvArgs& a, float (&acc)[NT][4], int r,
                                           int ntiles, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int R16 = a.R * 16;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int b = nt * 4 + t;
    if (b < a.batch) {
      red_add_f32(a.acc + (size_t)b * R16 + r * 16 + g, acc[nt][0] + acc[nt][1]);
      red_add_f32(a.acc + (size_t)b * R16 + r * 16 + g + 8, acc[nt][2] + acc[nt][3]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  }
  __syncwarp();
  int done = 0;
  int key = MODE == kModeQKV ? (r * 16) / a.hd : r;
  int need = MODE == kModeQKV ? (a.hd / 16) * a.nb : a.nb;
  if (lane == 0) done = (atom_add_acq_rel(a.ticket + key, ntiles) + ntiles == need);
  done = __shfl_sync(0xffffffffu, done, 0);
  __syncwarp();
  if (done) {
    if (lane == 0) a.ticket[key] = 0;
    if (MODE == kModeQKV) {
      if (a.hd == 64) finish_head<64>(a, key, lane);
      else if (a.hd == 128) finish_head<128>(a, key, lane);
      else finish_head<256>(a, key, lane);
    } else {
      finish_rowgroup(a, key, lane);
    }
  }
}

// One tile: convert the 16 biased bytes of this lane into the A registers of two k16
// MMAs, multiply with every batch tile of the activation, scale by the block's d.
template <int NT>
__device__ __forceinline__ void tile_mma(float (&acc)[NT][4], const uint4 w, uint32_t dbits,
                                         const uint4* xrow) {
  uint32_t A0[4], A1[4];
  A0[0] = u8x2_to_h2(w.x, kSelLo);
  A0[1] = u8x2_to_h2(w.y, kSelLo);
  A0[2] = u8x2_to_h2(w.x, kSelHi);
  A0[3] = u8x2_to_h2(w.y, kSelHi);
  A1[0] = u8x2_to_h2(w.z, kSelLo);
  A1[1] = u8x2_to_h2(w.w, kSelLo);
  A1[2] = u8x2_to_h2(w.z, kSelHi);
  A1[3] = u8x2_to_h2(w.w, kSelHi);
  const __half2 d2 = *reinterpret_cast<const __half2*>(&dbits);
  const float dg = __low2float(d2), dg8 = __high2float(d2);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4 xb = xrow[nt * 32];
    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16(tmp, A0, xb.x, xb.y);
    mma_f16(tmp, A1, xb.z, xb.w);
    acc[nt][0] = fmaf(tmp[0], dg, acc[nt][0]);
    acc[nt][1] = fmaf(tmp[1], dg, acc[nt][1]);
    acc[nt][2] = fmaf(tmp[2], dg8, acc[nt][2]);
    acc[nt][3] = fmaf(tmp[3], dg8, acc[nt][3]);
  }
}

// Work item = (k-split s, row group r): the nbs consecutive tiles of 16 rows x (nbs x 32)
// columns, one warp per item, CTAs of kItemsPerCta consecutive items (s-major).  The
// first kChunk tiles are loaded before anything else; the kernel's prologue (input
// norm statistics, activation operand of the CTA's k-range) hides their latency.
template <int NT, int MODE>
__global__ void __launch_bounds__(kItemsPerCta * 32, NT >= 4 ? 2 : 3)
    gemv_q8_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint4 xf[];  // [blocks of this CTA][NT][32 lanes]
  __shared__ float s_inv[16];
  __shared__ float s_ss[16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int items = a.S * a.R;
  const int item0 = blockIdx.x * kItemsPerCta;
  const int nitems = items - item0 < kItemsPerCta ? items - item0 : kItemsPerCta;
  const int s_first = item0 / a.R, s_last = (item0 + nitems - 1) / a.R;
  const int blk0 = s_first * a.nbs;
  const int nblk = (s_last - s_first + 1) * a.nbs;
  const bool active = warp < nitems;
  const int item = active ? item0 + warp : item0;
  const int s = item / a.R, r = item - s * a.R;
  const uint8_t* wbase = a.wq + ((size_t)r * a.nb + (size_t)s * a.nbs) * 512 + lane * 16;
  const __half2* dbase = a.wd + ((size_t)r * a.nb + (size_t)s * a.nbs) * 8 + g;

  // weights never depend on an earlier kernel: start their first chunk now
  uint4 wv[kChunk];
  uint32_t dv[kChunk];
  if (active) {
#pragma unroll
    for (int u = 0; u < kChunk; ++u)
      if (u < a.nbs) {
        wv[u] = ldg_stream_v4(wbase + (size_t)u * 512);
        dv[u] = ldg_stream_u32(dbase + (size_t)u * 8);
      }
    if (lane == 0 && a.nbs > kChunk) {
      prefetch_bulk_l2(wbase + (size_t)kChunk * 512, (uint32_t)(a.nbs - kChunk) * 512u);
    }
  }
  pdl_wait();

  if (MODE == kModeQKV) {
    // input RMSNorm statistics of every batch row (full rows, fp32): all threads share
    // the 8-column groups of all rows, partial sums meet in shared memory
    if (threadIdx.x < 16) s_ss[threadIdx.x] = 0.f;
    __syncthreads();
    const int gpr = a.cols / 8;  // groups per row
    const int ngroups = a.batch * gpr;
    for (int e0 = threadIdx.x; e0 < ngroups; e0 += 4 * blockDim.x) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * blockDim.x;
        if (e < ngroups)
          raw[u] = *reinterpret_cast<const uint4*>(a.x + (size_t)(e / gpr) * a.cols + (e % gpr) * 8);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * blockDim.x;
        if (e < ngroups) {
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
          float ss = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            ss += f.x * f.x + f.y * f.y;
          }
          if (gpr % 32 == 0) {
            // a warp's 32 consecutive groups lie in one row: one shared atomic per warp
            ss = warp_sum(ss);
            if ((threadIdx.x & 31) == 0) atomicAdd(&s_ss[e / gpr], ss);
          } else {
            atomicAdd(&s_ss[e / gpr], ss);
          }
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < a.batch) s_inv[threadIdx.x] = rsqrtf(s_ss[threadIdx.x] / a.cols + a.eps);
    __syncthreads();
  }

  // activation operand registers for the blocks this CTA touches: one thread turns 8
  // consecutive activations of one batch row into the hi and lo words of 4 lanes
  {
    uint32_t* xw = reinterpret_cast<uint32_t*>(xf);
    const int groups = nblk * 4;  // 8-column groups per batch row
    for (int e = threadIdx.x; e < NT * 4 * groups; e += blockDim.x) {
      const int b = e / groups, gi = e - b * groups;
      const int jb = gi >> 2, c = gi & 3;         // block, 8-column group in the block
      const int k = (blk0 + jb) * 32 + c * 8;
      float v[8];
      if (b < a.batch) {
        if (MODE == kModeQKV) {
          const uint4 raw = *reinterpret_cast<const uint4*>(a.x + (size_t)b * a.cols + k);
          const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.w_in + k));
          const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.w_in + k + 4));
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
          const float wv8[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          const float inv = s_inv[b];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x * inv * wv8[2 * i];
            v[2 * i + 1] = f.y * inv * wv8[2 * i + 1];
          }
        } else {
          const float4 f0 = *reinterpret_cast<const float4*>(a.xin + (size_t)b * a.cols + k);
          const float4 f1 = *reinterpret_cast<const float4*>(a.xin + (size_t)b * a.cols + k + 4);
          v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
          v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
      // columns 8c .. 8c+7 of the block: k-step ks = c / 2, register half hf = c % 2;
      // lane t holds the pair (2t, 2t+1); lanes g = 2(b%4) (hi) and 2(b%4)+1 (lo)
      const int ks = c >> 1, hf = c & 1, nt = b >> 2, gh = 2 * (b & 3);
      const int word = 2 * ks + hf;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        __half h0, l0, h1, l1;
        split_f16(v[2 * t], h0, l0);
        split_f16(v[2 * t + 1], h1, l1);
        const int base = ((jb * NT + nt) * 32) * 4 + word;
        xw[base + (gh * 4 + t) * 4] = pack_h2(h0, h1);
        xw[base + ((gh + 1) * 4 + t) * 4] = pack_h2(l0, l1);
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  if (!active) return;

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  const uint4* xrow = xf + (size_t)((s * a.nbs - blk0) * NT) * 32 + lane;

  if (a.nbs % kChunk == 0) {
    for (int c = 0; c < a.nbs; c += kChunk) {
      if (c > 0) {
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
          wv[u] = ldg_stream_v4(wbase + (size_t)(c + u) * 512);
          dv[u] = ldg_stream_u32(dbase + (size_t)(c + u) * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < kChunk; ++u) tile_mma<NT>(acc, wv[u], dv[u], xrow + (c + u) * NT * 32);
    }
  } else {
    for (int c = 0; c < a.nbs; c += kChunk) {
      if (c > 0) {
#pragma unroll
        for (int u = 0; u < kChunk; ++u)
          if (c + u < a.nbs) {
            wv[u] = ldg_stream_v4(wbase + (size_t)(c + u) * 512);
            dv[u] = ldg_stream_u32(dbase + (size_t)(c + u) * 8);
          }
      }
#pragma unroll
      for (int u = 0; u < kChunk; ++u)
        if (c + u < a.nbs) tile_mma<NT>(acc, wv[u], dv[u], xrow + (c + u) * NT * 32);
    }
  }
  flush_item<NT, MODE>(a, acc, r, a.nbs, lane);
}

int gemv_ntiles(int batch) { return batch <= 4 ? 1 : (batch <= 8 ? 2 : 4); }

int gemv_items_per_cta() { return kItemsPerCta; }

size_t gemv_smem_bytes(int batch, int blocks_per_cta_max) {
  return (size_t)blocks_per_cta_max * gemv_ntiles(batch) * 32 * sizeof(uint4);
}

template <int NT, int MODE>
static cudaError_t launch_t(const GemvArgs& a, int grid, int threads, size_t smem, bool pdl,
                            cudaStream_t s) {
  auto kern = gemv_q8_kernel<NT, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_gemv(int mode, const GemvArgs& a, int grid, int threads, size_t smem,
                        bool pdl, cudaStream_t s) {
  const int nt = gemv_ntiles(a.batch);
  if (mode == kModeQKV) {
    if (nt == 1) return launch_t<1, kModeQKV>(a, grid, threads, smem, pdl, s);
    if (nt == 2) return launch_t<2, kModeQKV>(a, grid, threads, smem, pdl, s);
    return launch_t<4, kModeQKV>(a, grid, threads, smem, pdl, s);
  }
  if (nt == 1) return launch_t<1, kModeOProj>(a, grid, threads, smem, pdl, s);
  if (nt == 2) return launch_t<2, kModeOProj>(a, grid, threads, smem, pdl, s);
  return launch_t<4, kModeOProj>(a, grid, threads, smem, pdl, s);
}

}  // namespace hfa
