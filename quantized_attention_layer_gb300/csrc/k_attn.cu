// k_attn.cu -- split-K GQA flash-decode over the bf16 KV cache.
//
// gemma4/gpu_full_attn.rs, encode_one_layer, "Dense flash_attn_vec": a single query
// per head attends to the cached keys of its KV head (num_heads / num_kv_heads query
// heads per KV head), mask "causal" over the populated ring slots or a sliding window
// over a linear buffer, scale 1.0 and an optional softcap (FlashAttnVecParams); the
// kernel runs as a main pass over key chunks plus a reduce pass.  The softcap is
// tanh(s / cap) * cap (dflash/forward.rs, softcap section).
//
// GB300 design.  One CTA = (sequence, KV head, key chunk).  A producer warp streams
// K and V tiles of T keys with 2-D TMA (128-byte swizzle) into a ring of NS shared
// stages guarded by mbarriers; consumer warps each take 16 keys of every stage.  All
// query heads of the group share one m16n8k16 MMA: rows 0..G-1 hold the bf16 "hi"
// part of each query, rows 8..8+G-1 the bf16 "lo" remainder, so S = Q K^T keeps about
// 16 bits of the fp32 query.  Softmax weights are split the same way for O += P V.
// The online softmax runs in base-2 units (log2 e folded into the query).  Each CTA
// writes (m, l, O) for its chunk; the last CTA of a (sequence, KV head) -- found with an
// atomic ticket, no waiting -- merges the chunks with log-sum-exp weights.
#include "hfa_common.cuh"
#include "hfa_internal.h"

namespace hfa {

constexpr int kKeysPerWarp = 16;
constexpr int kStages = 3;

// One CTA per SM streams 3 stages of ~64 KB (K + V); consumer warps take 16 keys each.
template <int HD>
struct AttnCfg {
  static constexpr int NC = HD >= 256 ? 4 : 8;       // consumer warps
  static constexpr int T = NC * kKeysPerWarp;         // keys per stage
  static constexpr int BOXES = HD / 64;               // 64-element (128 B) TMA boxes per row
  static constexpr int TILE_BYTES = T * HD * 2;       // one of K or V
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int KS = HD / 16;                  // k16 steps of S = Q K^T
  static constexpr int NTO = HD / 8;                  // n8 tiles of O
  static constexpr int QF_BYTES = KS * 32 * 16;
  static constexpr int RS = HD + 4;                   // record stride: O[HD], m, l, pad
  // the cross-warp merge reuses the stage buffers after the last stage
  static constexpr int RED_BYTES = NC * 8 * RS * 4;
  static constexpr size_t SMEM = 1024 + (size_t)kStages * STAGE_BYTES + QF_BYTES + 256;
  static_assert(RED_BYTES <= kStages * STAGE_BYTES, "merge area must fit in the stages");
};

// byte offset of (row, 16-byte chunk) inside a TMA tile written with 128-byte swizzle:
// box j = chunk / 8 holds dims [64 j, 64 j + 64); inside a 128-byte row the chunk index
// is XORed with (row mod 8).
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  const int box = chunk >> 3, c = chunk & 7;
  return (uint32_t)(box * (AttnCfg<HD>::T * 128) + row * 128 + ((c ^ (row & 7)) << 4));
}

template <int HD>
__global__ void __launch_bounds__(288)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const AttnArgs a) {
  using Cfg = AttnCfg<HD>;
  constexpr int T = Cfg::T;
  constexpr int kNC = Cfg::NC;
  constexpr int RS = Cfg::RS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* stages = smem;
  uint4* qf = reinterpret_cast<uint4*>(smem + kStages * Cfg::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * Cfg::STAGE_BYTES + Cfg::QF_BYTES);
  uint64_t* empty = full + kStages;
  int* s_flags = reinterpret_cast<int*>(empty + kStages);  // [0] abort, [1] issued, [2] last

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.nh / a.nkv;
  const int unit = blockIdx.x / a.splits, split = blockIdx.x - unit * a.splits;
  const int b = unit / a.nkv, kvh = unit - b * a.nkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNC);
    }
    s_flags[0] = 0;
    s_flags[1] = 0;
    fence_barrier_init();
  }
  if (warp == kNC && lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  __syncthreads();
  pdl_wait();  // q and the appended K/V row come from the previous kernel

  // visible slot range [lo, hi] of this sequence
  const int P = a.seq_pos[b];
  int lo, hi;
  if (a.ring) {
    lo = 0;
    hi = P < a.C - 1 ? P : a.C - 1;
  } else {
    lo = a.sliding ? (P - a.window + 1 > 0 ? P - a.window + 1 : 0) : 0;
    hi = P;
  }
  const bool bad = P < 0 || (!a.ring && P >= a.C);
  const int k_begin = lo + split * a.chunk;
  int k_end = k_begin + a.chunk;
  if (k_end > hi + 1) k_end = hi + 1;
  const int nkeys = bad ? 0 : (k_end > k_begin ? k_end - k_begin : 0);
  const int ntiles = (nkeys + T - 1) / T;
  const int row0 = unit * a.C + k_begin;  // TMA row of the first key of this chunk

  float* part = a.part + ((size_t)unit * a.splits + split) * 8 * RS;

  if (warp == kNC) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        if (i >= kStages) {
          if (!mbar_wait(&empty[st], ((i / kStages) - 1) & 1, a.err, &s_flags[0])) {
            atomicExch(&s_flags[0], 1);
            break;
          }
        }
        if (*(volatile int*)&s_flags[0]) break;
        uint8_t* kt = stages + st * Cfg::STAGE_BYTES;
        uint8_t* vt = kt + Cfg::TILE_BYTES;
        mbar_arrive_expect_tx(&full[st], Cfg::STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < Cfg::BOXES; ++j) {
          tma_load_2d(kt + j * T * 128, &tmk, &full[st], 64 * j, row0 + i * T);
          tma_load_2d(vt + j * T * 128, &tmv, &full[st], 64 * j, row0 + i * T);
        }
        issued = i + 1;
      }
      s_flags[1] = issued;
    }
  } else {
    // ------------------------------------------------------------- consumers
    // query fragments: A operand rows 0..G-1 = hi(q * qscale), rows 8..8+G-1 = lo
    for (int ks = warp; ks < Cfg::KS; ks += kNC) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (g < G) {
        const float* q = a.q + ((size_t)b * a.nh + kvh * G + g) * HD + ks * 16 + 2 * t;
        __nv_bfloat16 h[4], l[4];
        split_bf16(q[0] * a.qscale, h[0], l[0]);
        split_bf16(q[1] * a.qscale, h[1], l[1]);
        split_bf16(q[8] * a.qscale, h[2], l[2]);
        split_bf16(q[9] * a.qscale, h[3], l[3]);
        w[0] = pack_bf2(h[0], h[1]);
        w[1] = pack_bf2(l[0], l[1]);
        w[2] = pack_bf2(h[2], h[3]);
        w[3] = pack_bf2(l[2], l[3]);
      }
      qf[ks * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kNC * 32));

    float m = -INFINITY, l = 0.f;
    float o[Cfg::NTO][4];
#pragma unroll
    for (int i = 0; i < Cfg::NTO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    const uint32_t stage_base = smem_u32(stages);
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % kStages;
      if (*(volatile int*)&s_flags[0]) break;
      if (!mbar_wait(&full[st], (i / kStages) & 1, a.err, &s_flags[0])) {
        atomicExch(&s_flags[0], 1);
        break;
      }
      const uint32_t kb = stage_base + st * Cfg::STAGE_BYTES;
      const uint32_t vb = kb + Cfg::TILE_BYTES;
      const int krow = warp * kKeysPerWarp;

      // S = Q K^T for 16 keys: two n8 tiles
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < Cfg::KS; ++ks) {
        const uint4 qa = qf[ks * 32 + lane];
        const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
        const int mrow = krow + ((lane >> 4) << 3) + (lane & 7);
        const int mchunk = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kb + swz<HD>(mrow, mchunk), b0, b1, b2, b3);
        mma_bf16(s0, A, b0, b1);
        mma_bf16(s1, A, b2, b3);
      }
      // logits of head g for keys krow + {2t, 2t+1, 8+2t, 9+2t} (hi row + lo row)
      float sv[4] = {s0[0] + s0[2], s0[1] + s0[3], s1[0] + s1[2], s1[1] + s1[3]};
      const int kidx0 = k_begin + i * T + krow + 2 * t;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kidx0 + (e & 1) + ((e >> 1) << 3);
        float s = sv[e];
        if (a.cap_log2 != 0.f) s = a.cap_log2 * tanhf(s);
        sv[e] = key < k_end ? s : -INFINITY;
      }
      float mloc = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
      const float m_new = fmaxf(m, mloc);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float corr = exp2f(m - m_use);
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = exp2f(sv[e] - m_use);
      l = l * corr + (p[0] + p[1]) + (p[2] + p[3]);
      m = m_new;
#pragma unroll
      for (int nt = 0; nt < Cfg::NTO; ++nt) {
        o[nt][0] *= corr;
        o[nt][1] *= corr;
        o[nt][2] *= corr;
        o[nt][3] *= corr;
      }
      // P as the A operand: row g = hi(p), row g + 8 = lo(p); k = the 16 keys
      uint32_t PA[4];
      {
        __nv_bfloat16 h[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16(p[e], h[e], lw[e]);
        PA[0] = pack_bf2(h[0], h[1]);
        PA[1] = pack_bf2(lw[0], lw[1]);
        PA[2] = pack_bf2(h[2], h[3]);
        PA[3] = pack_bf2(lw[2], lw[3]);
      }
      // O += P V over HD/8 n8 tiles, two per ldmatrix.x4.trans
#pragma unroll
      for (int np = 0; np < Cfg::NTO / 2; ++np) {
        const int mrow = krow + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int mchunk = np * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vb + swz<HD>(mrow, mchunk), b0, b1, b2, b3);
        mma_bf16(o[2 * np], PA, b0, b1);
        mma_bf16(o[2 * np + 1], PA, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);

    // ------------------------------------------------- merge the consumer warps
    // every stage has been consumed (or the CTA aborted): reuse the stage buffers
    asm volatile("bar.sync 1, %0;" ::"n"(kNC * 32));
    float* red = reinterpret_cast<float*>(stages);  // [warp][8][RS]
    float* mine = red + warp * 8 * RS;
    if (g < G) {
      if (t == 0) {
        mine[g * RS + HD] = m;
        mine[g * RS + HD + 1] = l;
      }
#pragma unroll
      for (int nt = 0; nt < Cfg::NTO; ++nt) {
        mine[g * RS + nt * 8 + 2 * t] = o[nt][0] + o[nt][2];
        mine[g * RS + nt * 8 + 2 * t + 1] = o[nt][1] + o[nt][3];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kNC * 32));
    for (int e = threadIdx.x; e < G * (HD + 2); e += kNC * 32) {
      const int h = e / (HD + 2), d = e - h * (HD + 2);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kNC; ++w) M = fmaxf(M, red[(w * 8 + h) * RS + HD]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float acc = 0.f;
      if (d == HD) {
        acc = M;
      } else {
#pragma unroll
        for (int w = 0; w < kNC; ++w)
          acc += exp2f(red[(w * 8 + h) * RS + HD] - Mu) * red[(w * 8 + h) * RS + d];
      }
      part[h * RS + d] = acc;
    }
  }

  // drain: every TMA this CTA issued has landed before the CTA may exit
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = s_flags[1];
    for (int st = 0; st < kStages && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / kStages) * kStages;
      mbar_wait(&full[st], (last / kStages) & 1, a.err);
    }
  }

  // ------------------------------------------------- last chunk merges the unit
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(a.ticket + unit, 1);
    s_flags[2] = (old == a.splits - 1);
  }
  __syncthreads();
  if (!s_flags[2]) return;
  __threadfence();
  if (threadIdx.x == 0) a.ticket[unit] = 0;
  const float* up = a.part + (size_t)unit * a.splits * 8 * RS;
  // weight of chunk s for head h: 2^(m_s - M) / sum_s' 2^(m_s' - M) l_s'
  float* wsm = reinterpret_cast<float*>(stages);  // [8][splits]
  const int nwarps = blockDim.x >> 5;
  for (int h = warp; h < G; h += nwarps) {
    float M = -INFINITY;
    for (int sp = lane; sp < a.splits; sp += 32)
      M = fmaxf(M, ld_cg_f32(up + (sp * 8 + h) * RS + HD));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mu = M == -INFINITY ? 0.f : M;
    float den = 0.f;
    for (int sp = lane; sp < a.splits; sp += 32) {
      const float* ps = up + (sp * 8 + h) * RS;
      const float f = exp2f(ld_cg_f32(ps + HD) - Mu);
      wsm[h * a.splits + sp] = f;
      den += f * ld_cg_f32(ps + HD + 1);
    }
    den = warp_sum(den);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __syncwarp();
    for (int sp = lane; sp < a.splits; sp += 32) wsm[h * a.splits + sp] *= inv;
  }
  __syncthreads();
  // o[h][d] = sum_s w[h][s] O_s[h][d]: warps stride over chunks, lanes over float4
  // columns, every load of a warp independent; partial sums meet in shared memory
  float* osum = wsm + 8 * a.splits;  // [nwarps][G * HD]
  constexpr int Q4 = HD / 4;
  const int ncol = G * Q4;
  for (int c = lane; c < ncol; c += 32) {
    const int h = c / Q4, d4 = c - h * Q4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int sp = warp;
    for (; sp + nwarps < a.splits; sp += 2 * nwarps) {
      const float4 v0 = __ldcg(reinterpret_cast<const float4*>(up + (sp * 8 + h) * RS) + d4);
      const float4 v1 =
          __ldcg(reinterpret_cast<const float4*>(up + ((sp + nwarps) * 8 + h) * RS) + d4);
      const float w0 = wsm[h * a.splits + sp], w1 = wsm[h * a.splits + sp + nwarps];
      acc.x += w0 * v0.x + w1 * v1.x;
      acc.y += w0 * v0.y + w1 * v1.y;
      acc.z += w0 * v0.z + w1 * v1.z;
      acc.w += w0 * v0.w + w1 * v1.w;
    }
    if (sp < a.splits) {
      const float4 v0 = __ldcg(reinterpret_cast<const float4*>(up + (sp * 8 + h) * RS) + d4);
      const float w0 = wsm[h * a.splits + sp];
      acc.x += w0 * v0.x;
      acc.y += w0 * v0.y;
      acc.z += w0 * v0.z;
      acc.w += w0 * v0.w;
    }
    reinterpret_cast<float4*>(osum + warp * G * HD)[c] = acc;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < ncol; c += blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(osum)[c];
    for (int w = 1; w < nwarps; ++w) {
      const float4 v = reinterpret_cast<const float4*>(osum + w * G * HD)[c];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int h = c / Q4, d4 = c - h * Q4;
    reinterpret_cast<float4*>(a.o + ((size_t)b * a.nh + kvh * G + h) * HD)[d4] = acc;
  }
}

int attn_keys_per_stage(int hd) {
  return hd == 64 ? AttnCfg<64>::T : (hd == 128 ? AttnCfg<128>::T : AttnCfg<256>::T);
}
int attn_threads(int hd) { return (attn_keys_per_stage(hd) / kKeysPerWarp + 1) * 32; }
int attn_record_floats(int hd) { return 8 * (hd + 4); }
size_t attn_smem_bytes(int hd) {
  if (hd == 64) return AttnCfg<64>::SMEM;
  if (hd == 128) return AttnCfg<128>::SMEM;
  return AttnCfg<256>::SMEM;
}

template <int HD>
static cudaError_t launch_hd(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid, bool pdl, cudaStream_t s) {
  auto kern = attn_decode_kernel<HD>;
  const size_t smem = AttnCfg<HD>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((AttnCfg<HD>::NC + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

cudaError_t launch_attn(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        int grid, bool pdl, cudaStream_t s) {
  if (a.hd == 64) return launch_hd<64>(a, tk, tv, grid, pdl, s);
  if (a.hd == 128) return launch_hd<128>(a, tk, tv, grid, pdl, s);
  return launch_hd<256>(a, tk, tv, grid, pdl, s);
}

}  // namespace hfa
