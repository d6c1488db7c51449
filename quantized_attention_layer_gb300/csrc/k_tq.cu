// k_tq.cu -- the quantised (TurboQuant) KV cache: codebook, encode on append, and the
// flash-decode attention that reads the codes.
//
// gemma4/gpu_full_attn.rs, encode_one_layer: the Hadamard-quantize KV encode
// (hadamard_quantize_kv, hadamard_quantize_kv_hb: sign pre-multiply, normalised FWHT, a
// norm per 256-dim block, Lloyd-Max codes packed as 4-bit nibbles or one byte per value),
// the TQ attention (flash_attn_vec_tq, flash_attn_vec_tq_hb: the query pre-rotated the
// same way, scores and the weighted sum of V taken in the rotated domain, the output
// sign-undone by fwht_sign_undo), and the hybrid layout (K stored raw, V coded;
// flash_attn_vec_hybrid).  gemma4/model.rs gives the buffers: codes [nkv, capacity,
// hd * bits / 8] and f32 norms [nkv, capacity, hd / 256] per layer.
//
// The pages name the codebooks but do not print them: the codebook is the Lloyd-Max
// quantiser of N(0, 1), computed here on the host when a format is created.  Blocks are
// min(hd, 256) dims; a block's norm is the RMS of its rotated values, which are coded
// as value / norm with the nearest centroid (a value on a cell boundary takes the upper
// cell); 4-bit codes put element 2j in the low nibble of byte j.
//
// GB300 design.  The encode is tiny (a few rows per step) and takes its decisions in
// double precision: one warp per row, the FWHT butterflies across lanes by shuffles and
// within a lane over its registers, the block norm by a warp reduction, the cell by a
// binary search over the boundaries.  The attention is a split-K flash-decode whose work
// per key is a table lookup and a few multiply-adds per element: CUDA cores in fp32, one
// key per thread for the scores (the query read from shared memory as a broadcast), one
// dimension per thread for the weighted sum (the codes of a key row read coalesced), the
// online softmax per 256-key tile, and the chunks combined by the last CTA of each
// (sequence, KV head), which also undoes the rotation.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "hfa_common.cuh"
#include "hfa_internal.h"
#include "hfa_tq.cuh"

struct hfa_tq {
  int hd, bits, sbits, levels, blocks, code_bytes, device;  // sbits: bits stored per code
  float* centroids = nullptr;  // device [levels]
  double* bounds = nullptr;    // device [levels - 1]: the interior cell boundaries, ascending
  float* signs = nullptr;      // device [hd]: +-1
  std::vector<float> centroids_host;
};

namespace hfa {
namespace {

// ------------------------------------------------------------------ codebook (host)
double std_normal_tail(double x) { return 0.5 * erfc(x * 0.70710678118654752440); }
double std_normal_pdf(double x) {
  return std::isinf(x) ? 0.0 : 0.39894228040143267794 * exp(-0.5 * x * x);
}

// Lloyd-Max quantiser of N(0, 1) with `levels` (even) outputs, symmetric about 0.  Works on
// the positive half: thresholds t_0 = 0 < t_1 < ... < t_K = +inf (K = levels / 2), each
// t_i the midpoint of the outputs beside it, each output y_i the mean of N(0, 1) on
// [t_i, t_{i+1}], alternated until no output moves by more than 1e-14.
void lloyd_max_positive_half(int levels, std::vector<double>& cent, std::vector<double>& bnd) {
  const int K = levels / 2;
  std::vector<double> y(K), t(K + 1);
  for (int i = 0; i < K; ++i) y[i] = 3.0 * (i + 0.5) / K;  // any ascending start converges
  t[0] = 0.0;
  t[K] = INFINITY;
  for (int round = 0; round < 2000000; ++round) {
    for (int i = 1; i < K; ++i) t[i] = 0.5 * (y[i - 1] + y[i]);
    double moved = 0.0;
    for (int i = 0; i < K; ++i) {
      const double p = std_normal_tail(t[i]) - std_normal_tail(t[i + 1]);
      const double mean = (std_normal_pdf(t[i]) - std_normal_pdf(t[i + 1])) / p;
      moved = fmax(moved, fabs(mean - y[i]));
      y[i] = mean;
    }
    if (moved <= 1e-14) break;
  }
  for (int i = 1; i < K; ++i) t[i] = 0.5 * (y[i - 1] + y[i]);
  cent.assign(levels, 0.0);
  bnd.assign(levels - 1, 0.0);
  for (int i = 0; i < K; ++i) {
    cent[K + i] = y[i];
    cent[K - 1 - i] = -y[i];
  }
  for (int i = 0; i < K; ++i) {  // interior boundaries: -t_{K-1} .. -t_1, 0, t_1 .. t_{K-1}
    bnd[K - 1 + i] = t[i];
    bnd[K - 1 - i] = -t[i];
  }
}

// one computed codebook per code width, shared by every format of the process
struct Codebook {
  std::vector<double> cent, bnd;
};
std::mutex g_cb_mu;
Codebook g_cb[9];

const Codebook& codebook(int bits) {
  std::lock_guard<std::mutex> lock(g_cb_mu);
  Codebook& cb = g_cb[bits];
  if (cb.cent.empty()) lloyd_max_positive_half(1 << bits, cb.cent, cb.bnd);
  return cb;
}

constexpr int kTqThreads = 256;  // attention CTA: 8 warps; a tile is 256 keys
constexpr int kTqMaxG = 8;
constexpr int kTqMaxSplits = 256;  // the merge's weight table: kTqMaxG * 256 floats

// ------------------------------------------------------------------ encode (device)
struct TqAppendArgs {
  const float* x;        // [rows, hd], rows = B * nkv
  const int* seq_pos;    // [B]
  const double* bounds;  // [levels - 1]
  const float* signs;    // [hd]
  uint8_t* codes;        // [B, nkv, C, code_bytes]
  float* norms;          // [B, nkv, C, blocks]
  unsigned* err;         // nullable: bit 1 = a position outside the cache reached the kernel
  int rows, nkv, C, ring, levels;
};

// One warp per row: element i = lane + 32 j of the row sits in register j of lane `lane`.
template <int HD, int BITS>
__global__ void __launch_bounds__(128) tq_append_kernel(const TqAppendArgs a) {
  constexpr int J = HD / 32;
  constexpr int B = HD < 256 ? HD : 256;  // dims per block
  constexpr int JB = B / 32;              // registers per block
  constexpr int NB = HD / B;
  __shared__ double s_bnd[255];
  for (int i = threadIdx.x; i < a.levels - 1; i += blockDim.x) s_bnd[i] = a.bounds[i];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  if (row >= a.rows) return;
  const int b = row / a.nkv;
  const int P = a.seq_pos[b];
  if (P < 0 || (!a.ring && P >= a.C)) {
    if (lane == 0 && a.err) atomicOr(a.err, 2u);
    return;
  }
  const int slot = a.ring ? P % a.C : P;
  double u[J];
#pragma unroll
  for (int j = 0; j < J; ++j)
    u[j] = (double)a.x[(size_t)row * HD + lane + 32 * j] * (double)a.signs[lane + 32 * j];
  // butterflies of stride h in the order 1, 2, 4, ..., B/2 (each block on its own)
#pragma unroll
  for (int h = 1; h < 32 && h < B; h <<= 1) {
    const bool upper = lane & h;  // this lane holds x[i + h] of its pair
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const double other = __shfl_xor_sync(0xffffffffu, u[j], h);
      u[j] = upper ? other - u[j] : u[j] + other;
    }
  }
#pragma unroll
  for (int hj = 1; hj < JB; hj <<= 1) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      if (!(j & hj)) {
        const double a0 = u[j], a1 = u[j + hj];
        u[j] = a0 + a1;
        u[j + hj] = a0 - a1;
      }
    }
  }
  const double scale = 1.0 / sqrt((double)B);
#pragma unroll
  for (int j = 0; j < J; ++j) u[j] *= scale;
  const size_t at = ((size_t)row * a.C + slot);
#pragma unroll
  for (int k = 0; k < NB; ++k) {
    double ss = 0.0;
#pragma unroll
    for (int j = k * JB; j < (k + 1) * JB; ++j) ss += u[j] * u[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const double norm = sqrt(ss / B);
    if (lane == 0) a.norms[at * NB + k] = (float)norm;
#pragma unroll
    for (int j = k * JB; j < (k + 1) * JB; ++j) {
      const double e = norm > 0.0 ? u[j] / norm : 0.0;
      // the cell: the number of interior boundaries <= e
      int lo = 0, hi = a.levels - 1;  // answer in [lo, hi]
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;  // is boundary `mid` <= e ?
        if (s_bnd[mid] <= e) lo = mid + 1;
        else hi = mid;
      }
      const int code = lo;
      const int i = lane + 32 * j;
      if (BITS == 8) {
        a.codes[at * HD + i] = (uint8_t)code;
      } else {
        const int hi_code = __shfl_down_sync(0xffffffffu, code, 1);
        if (!(lane & 1)) a.codes[at * (HD / 2) + i / 2] = (uint8_t)(code | (hi_code << 4));
      }
    }
  }
}

// ------------------------------------------------------------------ attention (device)


template <int HD>
struct TqCfg {
  static constexpr int BLK = HD < 256 ? HD : 256;
  static constexpr int NB = HD / BLK;
  static constexpr int RS = HD + 4;
  // phase 2: four dimensions per thread, HD / 4 threads per key row, NKS key subsets
  static constexpr int TPR = HD / 4;
  static constexpr int NKS = kTqThreads / TPR;
};

// GM: the most query heads per KV head this instantiation handles (G rounded up to 2, 4, 8)
template <int HD, int BITS, bool KRAW, int GM>
struct TqSmem {
  static constexpr int LEVELS = 1 << BITS;
  static constexpr int NB = TqCfg<HD>::NB;
  // the centroid table with one copy per bank (entry c of lane l at c * 32 + l), so the
  // lookups of a warp never collide; the queries; the per-tile scores / weights; V norms
  static constexpr size_t TAB = (size_t)LEVELS * 32 * 4;
  static constexpr size_t Q = (size_t)GM * HD * 4;
  static constexpr size_t PB = (size_t)kTqMaxG * kTqThreads * 4;
  static constexpr size_t VN = (size_t)kTqThreads * NB * 4;
  static constexpr size_t BYTES = TAB + Q + PB + VN + 3 * kTqMaxG * 4 + 16;
};

template <int HD, int BITS, bool KRAW, int GM>
__global__ void __launch_bounds__(kTqThreads) tq_attn_kernel(const TqAttnArgs a) {
  using Cfg = TqCfg<HD>;
  using SM = TqSmem<HD, BITS, KRAW, GM>;
  constexpr int RS = Cfg::RS;
  constexpr int NB = Cfg::NB;
  constexpr int BLK = Cfg::BLK;
  constexpr int CB = HD * BITS / 8;  // code bytes of a row
  constexpr int NKS = Cfg::NKS;
  constexpr int TPR = Cfg::TPR;
  constexpr int LEVELS = 1 << BITS;
  extern __shared__ __align__(16) uint8_t tq_smem[];
  float* s_tab = reinterpret_cast<float*>(tq_smem);
  float* s_q = reinterpret_cast<float*>(tq_smem + SM::TAB);   // [GM][HD]
  float* s_p = reinterpret_cast<float*>(tq_smem + SM::TAB + SM::Q);  // [8][256]
  float* s_vn = reinterpret_cast<float*>(tq_smem + SM::TAB + SM::Q + SM::PB);  // [256][NB]
  float* s_corr = reinterpret_cast<float*>(tq_smem + SM::TAB + SM::Q + SM::PB + SM::VN);
  float* s_m = s_corr + kTqMaxG;
  float* s_l = s_m + kTqMaxG;
  int* s_last = reinterpret_cast<int*>(s_l + kTqMaxG);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.nh / a.nkv;  // <= GM
  const int unit = blockIdx.x / a.splits, split = blockIdx.x - unit * a.splits;
  const int b = unit / a.nkv, kvh = unit - b * a.nkv;
  // the table has room for 2^BITS levels; a byte-coded format may use fewer (5, 6 bits).
  // Each centroid is loaded once (into the score area), then copied to its 32 bank slots.
  for (int c = tid; c < LEVELS; c += kTqThreads) s_p[c] = c < a.levels ? a.centroids[c] : 0.f;
  __syncthreads();
  for (int i = tid; i < LEVELS * 32; i += kTqThreads) s_tab[i] = s_p[i >> 5];
  for (int e = tid; e < GM * HD; e += kTqThreads) {
    const int h = e / HD, i = e - h * HD;
    const float qv = h < G ? a.q[((size_t)b * a.nh + kvh * G + h) * HD + i] * a.qscale : 0.f;
    s_q[h * HD + i] = KRAW ? qv : qv * a.signs[i];
  }
  if (tid < kTqMaxG) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  __syncthreads();
  if (!KRAW)  // the query in the keys' rotated domain
    tq_fwht_rows(s_q, GM, HD, BLK, HD, tid, kTqThreads, []() { __syncthreads(); });

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
  if (bad && tid == 0 && split == 0 && a.err) atomicOr(a.err, 2u);
  const int k_begin = lo + split * a.chunk;
  int k_end = k_begin + a.chunk;
  if (k_end > hi + 1) k_end = hi + 1;
  if (bad) k_end = k_begin;
  const size_t row0 = (size_t)unit * a.C;  // cache row of slot 0 of this unit

  // phase 2 accumulators: dims 4 (tid % TPR) .. + 3 for every query head
  const int ks = tid / TPR, d0 = 4 * (tid - ks * TPR);
  float acc[4][GM];
#pragma unroll
  for (int d = 0; d < 4; ++d)
#pragma unroll
    for (int h = 0; h < GM; ++h) acc[d][h] = 0.f;

  for (int t0 = k_begin; t0 < k_end; t0 += kTqThreads) {
    // ---- phase 1: one key per thread, its score for every query head (every lane reads
    // the same query element at a time: a broadcast); eight 16-byte loads in flight
    {
      const int key = t0 + tid;
      float sc[GM];
#pragma unroll
      for (int h = 0; h < GM; ++h) sc[h] = 0.f;
      if (key < k_end) {
        const size_t r = row0 + key;
        if (KRAW) {
          const uint4* kr = reinterpret_cast<const uint4*>(a.k_raw + r * HD);
          for (int c0 = 0; c0 < HD / 8; c0 += 8) {
            uint4 w8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w8[u] = __ldg(kr + c0 + u);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const __nv_bfloat162* kp = reinterpret_cast<const __nv_bfloat162*>(&w8[u]);
              float kv[8];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(kp[e]);
                kv[2 * e] = f.x;
                kv[2 * e + 1] = f.y;
              }
              const int i0 = (c0 + u) * 8;
#pragma unroll
              for (int h = 0; h < GM; ++h) {
                const float4 qa = *reinterpret_cast<const float4*>(s_q + h * HD + i0);
                const float4 qb = *reinterpret_cast<const float4*>(s_q + h * HD + i0 + 4);
                sc[h] += qa.x * kv[0] + qa.y * kv[1] + qa.z * kv[2] + qa.w * kv[3] +
                         qb.x * kv[4] + qb.y * kv[5] + qb.z * kv[6] + qb.w * kv[7];
              }
            }
          }
        } else {
          const uint4* kc = reinterpret_cast<const uint4*>(a.k_codes + r * CB);
          constexpr int VPC = 128 / BITS;        // values per 16-byte chunk
          constexpr int CPB = BLK / VPC;         // chunks per block
          constexpr int CG = CPB < 8 ? CPB : 8;  // chunks loaded together
#pragma unroll
          for (int k = 0; k < NB; ++k) {
            float part[GM];
#pragma unroll
            for (int h = 0; h < GM; ++h) part[h] = 0.f;
            for (int c0 = k * CPB; c0 < (k + 1) * CPB; c0 += CG) {
              uint4 w8[CG];
#pragma unroll
              for (int u = 0; u < CG; ++u) w8[u] = __ldg(kc + c0 + u);
#pragma unroll
              for (int u = 0; u < CG; ++u) {
                const uint32_t ws[4] = {w8[u].x, w8[u].y, w8[u].z, w8[u].w};
#pragma unroll
                for (int q4 = 0; q4 < VPC / 4; ++q4) {
                  float kv[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int vi = q4 * 4 + e;
                    const uint32_t word = ws[vi / (32 / BITS)];
                    const int code = (word >> ((vi % (32 / BITS)) * BITS)) & (LEVELS - 1);
                    kv[e] = s_tab[code * 32 + lane];
                  }
                  const int i0 = (c0 + u) * VPC + q4 * 4;
#pragma unroll
                  for (int h = 0; h < GM; ++h) {
                    const float4 qa = *reinterpret_cast<const float4*>(s_q + h * HD + i0);
                    part[h] += qa.x * kv[0] + qa.y * kv[1] + qa.z * kv[2] + qa.w * kv[3];
                  }
                }
              }
            }
            const float kn = __ldg(a.k_norms + r * NB + k);
#pragma unroll
            for (int h = 0; h < GM; ++h) sc[h] += part[h] * kn;
          }
        }
#pragma unroll
        for (int k = 0; k < NB; ++k) s_vn[tid * NB + k] = __ldg(a.v_norms + r * NB + k);
      }
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h < G) {
          float sv = sc[h];
          if (a.cap_log2 != 0.f) sv = a.cap_log2 * tanhf(sv);
          s_p[h * kTqThreads + tid] = key < k_end ? sv : -INFINITY;
        }
      }
    }
    __syncthreads();
    // ---- online softmax over the tile, one warp per query head
    for (int h = warp; h < G; h += kTqThreads / 32) {
      float* ph = s_p + h * kTqThreads;
      float mx = -INFINITY;
      for (int j = lane; j < kTqThreads; j += 32) mx = fmaxf(mx, ph[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = s_m[h];
      const float m_new = fmaxf(m_old, mx);
      const float mu = m_new == -INFINITY ? 0.f : m_new;
      float sum = 0.f;
      for (int j = lane; j < kTqThreads; j += 32) {
        const float p = exp2f(ph[j] - mu);
        ph[j] = p;
        sum += p;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float corr = exp2f(m_old - mu);
        s_corr[h] = corr;
        s_l[h] = s_l[h] * corr + sum;
        s_m[h] = m_new;
      }
    }
    __syncthreads();
    // ---- phase 2: four dimensions per thread, the keys of its subset (four keys' codes
    // loaded together); the weighted sum of the decoded values in the rotated domain
    {
      float corr[GM];
#pragma unroll
      for (int h = 0; h < GM; ++h) corr[h] = h < G ? s_corr[h] : 0.f;
#pragma unroll
      for (int d = 0; d < 4; ++d)
#pragma unroll
        for (int h = 0; h < GM; ++h) acc[d][h] *= corr[h];
      const int nk = k_end - t0 < kTqThreads ? k_end - t0 : kTqThreads;
      const int blk = d0 / BLK;
      for (int j0 = ks; j0 < nk; j0 += 4 * NKS) {
        uint32_t cw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * NKS;
          const size_t r = row0 + t0 + (j < nk ? j : j0);  // in range
          if (BITS == 8)
            cw[u] = __ldg(reinterpret_cast<const uint32_t*>(a.v_codes + r * CB + d0));
          else
            cw[u] = __ldg(reinterpret_cast<const uint16_t*>(a.v_codes + r * CB + d0 / 2));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * NKS;
          if (j < nk) {
            const float vn = s_vn[j * NB + blk];
            float val[4];
#pragma unroll
            for (int d = 0; d < 4; ++d) val[d] = s_tab[((cw[u] >> (d * BITS)) & (LEVELS - 1)) * 32 + lane] * vn;
#pragma unroll
            for (int h = 0; h < GM; ++h) {
              const float p = s_p[h * kTqThreads + j];
#pragma unroll
              for (int d = 0; d < 4; ++d) acc[d][h] = fmaf(p, val[d], acc[d][h]);
            }
          }
        }
      }
    }
    __syncthreads();
  }

  // ---- the chunk's record: the key subsets added in order, then m and l
  float* rec = a.part + ((size_t)unit * a.splits + split) * 8 * RS;
  {
    // [NKS][GM][HD] floats = 4 * 256 * GM: the query area (8 HD floats) holds it for
    // HD >= 4 * 32 GM / 8..., the score area (8 * 256) always does for GM <= 2; use whichever
    // fits, else two halves through the score area
    float* red = s_p;
    static_assert(NKS * HD == 4 * kTqThreads, "four dims per thread");
    constexpr int HALF = GM * 4 * kTqThreads <= kTqMaxG * kTqThreads ? GM : kTqMaxG / 4;
    for (int h0 = 0; h0 < GM; h0 += HALF) {
#pragma unroll
      for (int d = 0; d < 4; ++d)
#pragma unroll
        for (int h = 0; h < GM; ++h)
          if (h >= h0 && h < h0 + HALF) red[((h - h0) * NKS + ks) * HD + d0 + d] = acc[d][h];
      __syncthreads();
      for (int e = tid; e < HALF * HD; e += kTqThreads) {
        const int hh = e / HD, i = e - hh * HD;
        float sum = 0.f;
        for (int k2 = 0; k2 < NKS; ++k2) sum += red[(hh * NKS + k2) * HD + i];
        if (h0 + hh < G) rec[(h0 + hh) * RS + i] = sum;
      }
      __syncthreads();
    }
    if (tid < G) {
      rec[tid * RS + HD] = s_m[tid];
      rec[tid * RS + HD + 1] = s_l[tid];
    }
  }

  // ---- the last chunk of the unit merges the records and undoes the rotation
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(a.ticket + unit, 1) == a.splits - 1;
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  if (tid == 0) a.ticket[unit] = 0;
  const float* up = a.part + (size_t)unit * a.splits * 8 * RS;
  tq_merge_records<HD, kTqThreads>(up, a.splits, G, s_p, s_q, a.signs, a.o + ((size_t)b * a.nh + kvh * G) * HD);
}

template <int HD, int BITS>
cudaError_t launch_append_t(const TqAppendArgs& a, cudaStream_t s) {
  tq_append_kernel<HD, BITS><<<(a.rows + 3) / 4, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <int HD, int BITS, bool KRAW, int GM>
cudaError_t launch_gm(const TqAttnArgs& a, int grid, cudaStream_t s) {
  auto kern = tq_attn_kernel<HD, BITS, KRAW, GM>;
  const size_t smem = TqSmem<HD, BITS, KRAW, GM>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTqThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int HD, int BITS, bool KRAW>
cudaError_t launch_attn_t(const TqAttnArgs& a, int grid, cudaStream_t s) {
  const int G = a.nh / a.nkv;
  if (G <= 2) return launch_gm<HD, BITS, KRAW, 2>(a, grid, s);
  if (G <= 4) return launch_gm<HD, BITS, KRAW, 4>(a, grid, s);
  return launch_gm<HD, BITS, KRAW, 8>(a, grid, s);
}

template <int HD>
cudaError_t launch_attn_hd(const TqAttnArgs& a, int bits, bool kraw, int grid, cudaStream_t s) {
  if (bits == 8)
    return kraw ? launch_attn_t<HD, 8, true>(a, grid, s) : launch_attn_t<HD, 8, false>(a, grid, s);
  return kraw ? launch_attn_t<HD, 4, true>(a, grid, s) : launch_attn_t<HD, 4, false>(a, grid, s);
}

thread_local char g_tq_error[256];
hfa_status tq_fail(hfa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_tq_error, sizeof g_tq_error, fmt, ap);
  va_end(ap);
  set_thread_error(g_tq_error);
  return st;
}

bool aligned(const void* p, size_t n) { return ((uintptr_t)p % n) == 0; }

}  // namespace
}  // namespace hfa

using namespace hfa;

extern "C" hfa_status hfa_tq_create(int head_dim, int bits, const int8_t* signs, hfa_tq** out) {
  if (!out) return tq_fail(HFA_EINVAL, "out is NULL");
  *out = nullptr;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256 && head_dim != 512)
    return tq_fail(HFA_EUNSUPPORTED, "head_dim=%d (supported: 64, 128, 256, 512)", head_dim);
  if (bits != 4 && bits != 5 && bits != 6 && bits != 8)
    return tq_fail(HFA_EUNSUPPORTED, "bits=%d (supported: 4, 5, 6, 8)", bits);
  if (!signs) return tq_fail(HFA_EINVAL, "signs is NULL");
  for (int i = 0; i < head_dim; ++i)
    if (signs[i] != 1 && signs[i] != -1) return tq_fail(HFA_EINVAL, "signs[%d]=%d is not +-1", i, signs[i]);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tq_fail(HFA_EDEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  const Codebook& cb = codebook(bits);
  hfa_tq* t = new hfa_tq();
  t->hd = head_dim;
  t->bits = bits;
  t->levels = 1 << bits;
  t->blocks = head_dim / (head_dim < 256 ? head_dim : 256);
  t->sbits = bits == 4 ? 4 : 8;  // 5- and 6-bit codes are stored one per byte
  t->code_bytes = head_dim * t->sbits / 8;
  t->device = dev;
  t->centroids_host.assign(cb.cent.begin(), cb.cent.end());
  std::vector<float> sg(head_dim);
  for (int i = 0; i < head_dim; ++i) sg[i] = (float)signs[i];
  e = cudaMalloc(&t->centroids, t->levels * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&t->bounds, (t->levels - 1) * sizeof(double));
  if (e == cudaSuccess) e = cudaMalloc(&t->signs, head_dim * sizeof(float));
  if (e == cudaSuccess)
    e = cudaMemcpy(t->centroids, t->centroids_host.data(), t->levels * sizeof(float),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(t->bounds, cb.bnd.data(), (t->levels - 1) * sizeof(double), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(t->signs, sg.data(), head_dim * sizeof(float), cudaMemcpyHostToDevice);
  // a copy from pageable memory may return before its DMA lands, and the attention reads
  // the centroids before its programmatic-dependency wait: the tables are complete first
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(t->centroids);
    cudaFree(t->bounds);
    cudaFree(t->signs);
    delete t;
    return tq_fail(HFA_ENOMEM, "format tables: %s", cudaGetErrorString(e));
  }
  *out = t;
  return HFA_OK;
}

extern "C" hfa_status hfa_tq_destroy(hfa_tq* t) {
  if (!t) return HFA_EINVAL;
  cudaDeviceSynchronize();
  cudaFree(t->centroids);
  cudaFree(t->bounds);
  cudaFree(t->signs);
  delete t;
  return HFA_OK;
}

extern "C" int hfa_tq_code_bytes(const hfa_tq* t) { return t ? t->code_bytes : 0; }
extern "C" int hfa_tq_blocks(const hfa_tq* t) { return t ? t->blocks : 0; }

extern "C" int hfa_tq_codebook(const hfa_tq* t, float* centroids, int n) {
  if (!t) return 0;
  for (int i = 0; i < n && i < t->levels; ++i) centroids[i] = t->centroids_host[i];
  return t->levels;
}

extern "C" hfa_status hfa_tq_append(const hfa_tq* t, void* stream, const float* x,
                                    const int32_t* pos_dev, const int32_t* pos_host, int batch,
                                    int nkv, int capacity, int ring, uint8_t* codes,
                                    float* norms) {
  if (!t) return tq_fail(HFA_EINVAL, "format is NULL");
  if (!x || !pos_dev || !pos_host || !codes || !norms) return tq_fail(HFA_EINVAL, "a pointer is NULL");
  if (batch < 1 || nkv < 1 || capacity < 1 || capacity >= (1 << 24) || batch > 4096 || nkv > 4096)
    return tq_fail(HFA_EINVAL, "batch=%d, nkv=%d, capacity=%d", batch, nkv, capacity);
  if (!aligned(x, 16) || !aligned(norms, 4))
    return tq_fail(HFA_EINVAL, "x must be 16-byte aligned, norms 4-byte aligned");
  for (int b = 0; b < batch; ++b) {
    const int P = pos_host[b];
    if (P < 0 || (!ring && P >= capacity))
      return tq_fail(HFA_ERANGE, "seq_pos[%d]=%d outside the cache (capacity %d)", b, P, capacity);
  }
  TqAppendArgs a{};
  a.x = x;
  a.seq_pos = pos_dev;
  a.bounds = t->bounds;
  a.signs = t->signs;
  a.codes = codes;
  a.norms = norms;
  a.err = nullptr;
  a.rows = batch * nkv;
  a.nkv = nkv;
  a.C = capacity;
  a.ring = ring ? 1 : 0;
  a.levels = t->levels;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  switch (t->hd * 16 + t->sbits) {
    case 64 * 16 + 4: e = launch_append_t<64, 4>(a, s); break;
    case 64 * 16 + 8: e = launch_append_t<64, 8>(a, s); break;
    case 128 * 16 + 4: e = launch_append_t<128, 4>(a, s); break;
    case 128 * 16 + 8: e = launch_append_t<128, 8>(a, s); break;
    case 256 * 16 + 4: e = launch_append_t<256, 4>(a, s); break;
    case 256 * 16 + 8: e = launch_append_t<256, 8>(a, s); break;
    case 512 * 16 + 4: e = launch_append_t<512, 4>(a, s); break;
    default: e = launch_append_t<512, 8>(a, s); break;
  }
  if (e != cudaSuccess) return tq_fail(HFA_ECUDA, "encode launch: %s", cudaGetErrorString(e));
  return HFA_OK;
}

namespace {
// workspace: [status word, tickets [units], group tickets [units][16], 256-byte aligned]
// [records [units][splits][8][hd + 4]][group folds [units][16][8][hd + 4]]
constexpr int kTqGroups = 16;
size_t tq_ws_head(int units) { return ((size_t)(1 + units + units * kTqGroups) * 4 + 255) / 256 * 256; }
size_t tq_ws_folds(int units, int hd) { return (size_t)units * kTqGroups * 8 * (hd + 4) * sizeof(float); }
// splits per group of the two-level merge: one group (a single merge) while one CTA reads
// at most 64 KB of records (the second ticket round would cost more than it saves); else
// about sqrt(splits), so that each level reads a few records
int tq_group(int S, int G, int hd) {
  if (S <= 4 || (size_t)S * G * (hd + 4) * sizeof(float) <= 65536) return S;
  int g = 1;
  while (g * g < S) ++g;
  return g;
}
int tq_splits(int units, int max_keys, int sms) {
  int S = (8 * sms + units - 1) / units;  // many CTAs: the per-key work is latency-bound
  if (S > kTqMaxSplits) S = kTqMaxSplits;
  const int tiles = (max_keys + kTqThreads - 1) / kTqThreads;
  if (S > tiles) S = tiles;
  if (S < 1) S = 1;
  return S;
}
// the tensor-core kernel: one CTA per SM, chunks a multiple of its stage
int tq_mma_splits(int units, int max_keys, int sms, int hd) {
  int S = sms / units;
  if (S > kTqMaxSplits) S = kTqMaxSplits;
  const int T = tq_mma_keys_per_stage(hd);
  const int tiles = (max_keys + T - 1) / T;
  if (S > tiles) S = tiles;
  if (S < 1) S = 1;
  return S;
}
int tq_mma_chunk(int max_keys, int S, int hd) {
  const int T = tq_mma_keys_per_stage(hd);
  const int c = (max_keys + S - 1) / S;
  return (c + T - 1) / T * T;
}
// either kernel's record count fits: the workspace does not depend on the code width
int tq_ws_splits(int units, int max_keys, int sms, int hd) {
  const int a = tq_splits(units, max_keys, sms);
  const int b = tq_mma_splits(units, max_keys, sms, hd);
  return a > b ? a : b;
}
int visible(const hfa_attn_desc* d, int P) {
  const bool ring = d->flags & HFA_F_RING;
  if (ring) return (P < d->kv_capacity - 1 ? P : d->kv_capacity - 1) + 1;
  const int lo = d->layer_type == HFA_SLIDING ? (P - d->window + 1 > 0 ? P - d->window + 1 : 0) : 0;
  return P - lo + 1;
}
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}
}  // namespace

extern "C" size_t hfa_attention_tq_workspace_bytes(const hfa_attn_desc* d, int batch, int max_keys) {
  if (!d || batch < 1 || max_keys < 1 || d->num_kv_heads < 1) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int units = batch * d->num_kv_heads;
  const int S = tq_ws_splits(units, max_keys, sms, d->head_dim);
  return tq_ws_head(units) + (size_t)units * S * 8 * (d->head_dim + 4) * sizeof(float) +
         tq_ws_folds(units, d->head_dim);
}

extern "C" hfa_status hfa_attention_decode_tq(const hfa_attn_desc* d, const hfa_tq* t, void* stream,
                                              const float* q, const int32_t* pos_dev,
                                              const int32_t* pos_host, int batch,
                                              const uint8_t* k_codes, const float* k_norms,
                                              const void* k_raw, const uint8_t* v_codes,
                                              const float* v_norms, void* ws, size_t ws_bytes,
                                              float* o) {
  if (!d || !t) return tq_fail(HFA_EINVAL, "desc or format is NULL");
  const int nh = d->num_heads, nkv = d->num_kv_heads, hd = d->head_dim;
  if (nh <= 0 || nkv <= 0 || nh % nkv) return tq_fail(HFA_EINVAL, "num_heads=%d, num_kv_heads=%d", nh, nkv);
  if (nh / nkv > kTqMaxG) return tq_fail(HFA_EUNSUPPORTED, "GQA group %d > %d", nh / nkv, kTqMaxG);
  if (hd != t->hd) return tq_fail(HFA_EINVAL, "head_dim=%d, the format is for %d", hd, t->hd);
  if (d->layer_type != HFA_SLIDING && d->layer_type != HFA_FULL)
    return tq_fail(HFA_EINVAL, "layer_type=%d", d->layer_type);
  if (d->layer_type == HFA_SLIDING && d->window <= 0) return tq_fail(HFA_EINVAL, "window=%d", d->window);
  if (d->kv_capacity <= 0 || d->kv_capacity >= (1 << 24))
    return tq_fail(HFA_EINVAL, "kv_capacity=%d outside [1, 2^24)", d->kv_capacity);
  if (d->flags & ~HFA_F_RING) return tq_fail(HFA_EINVAL, "flags 0x%x", d->flags);
  const bool ring = d->flags & HFA_F_RING;
  if (ring && (d->layer_type != HFA_SLIDING || d->kv_capacity != d->window))
    return tq_fail(HFA_EINVAL, "a ring cache needs a sliding layer with kv_capacity == window");
  if (!(d->attn_scale > 0.f) || !(d->softcap >= 0.f)) return tq_fail(HFA_EINVAL, "attn_scale, softcap");
  const bool kraw = k_codes == nullptr;
  if (!q || !pos_dev || !pos_host || !v_codes || !v_norms || !ws || !o ||
      (kraw ? !k_raw : !k_norms))
    return tq_fail(HFA_EINVAL, "a pointer argument is NULL");
  if (batch < 1 || batch > 4096) return tq_fail(HFA_EINVAL, "batch=%d", batch);
  if (!aligned(q, 16) || !aligned(ws, 16) || !aligned(o, 16) || !aligned(k_codes, 16) ||
      !aligned(v_codes, 16) || !aligned(k_raw, 16) || !aligned(k_norms, 4) || !aligned(v_norms, 4))
    return tq_fail(HFA_EINVAL, "q, o, the workspace and the code arrays must be 16-byte aligned");
  int max_keys = 0;
  for (int b = 0; b < batch; ++b) {
    const int P = pos_host[b];
    if (P < 0 || (!ring && P >= d->kv_capacity))
      return tq_fail(HFA_ERANGE, "seq_pos[%d]=%d outside the cache (capacity %d)", b, P, d->kv_capacity);
    const int n = visible(d, P);
    if (n > max_keys) max_keys = n;
  }
  const int sms = sm_count();
  if (sms <= 0) return tq_fail(HFA_EDEVICE, "no CUDA device");
  const int units = batch * nkv;
  if ((long long)units * d->kv_capacity >= (1ll << 40)) return tq_fail(HFA_EUNSUPPORTED, "cache too large");
  const int Sws = tq_ws_splits(units, max_keys, sms, hd);
  const size_t need = tq_ws_head(units) + (size_t)units * Sws * 8 * (hd + 4) * sizeof(float) +
                      tq_ws_folds(units, hd);
  if (ws_bytes < need) return tq_fail(HFA_EINVAL, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  // the tensor-core kernel (every head dim; raw keys up to 256; TMA rows are 32-bit)
  const bool mma = tq_mma_supported(hd, t->sbits, kraw) && (long long)units * d->kv_capacity < (1ll << 31);
  int S, chunk;
  if (mma) {
    S = tq_mma_splits(units, max_keys, sms, hd);
    chunk = tq_mma_chunk(max_keys, S, hd);
    S = (max_keys + chunk - 1) / chunk;  // no chunk starts past the longest sequence
  } else {
    S = tq_splits(units, max_keys, sms);
    chunk = (max_keys + S - 1) / S;
    chunk = (chunk + kTqThreads - 1) / kTqThreads * kTqThreads;
  }
  TqAttnArgs a{};
  a.q = q;
  a.seq_pos = pos_dev;
  a.k_codes = k_codes;
  a.k_norms = k_norms;
  a.k_raw = (const __nv_bfloat16*)k_raw;
  a.v_codes = v_codes;
  a.v_norms = v_norms;
  a.centroids = t->centroids;
  a.signs = t->signs;
  a.err = (unsigned*)ws;
  a.ticket = (int*)ws + 1;
  a.ticket1 = (int*)ws + 1 + units;
  a.part = (float*)((char*)ws + tq_ws_head(units));
  a.part1 = a.part + (size_t)units * Sws * 8 * (hd + 4);
  a.group = tq_group(S, nh / nkv, hd);
  a.o = o;
  a.B = batch;
  a.nh = nh;
  a.nkv = nkv;
  a.C = d->kv_capacity;
  a.sliding = d->layer_type == HFA_SLIDING;
  a.window = d->window;
  a.ring = ring ? 1 : 0;
  a.levels = t->levels;
  a.splits = S;
  a.chunk = chunk;
  const float log2e = 1.4426950408889634f;
  if (d->softcap > 0.f) {
    a.qscale = d->attn_scale / d->softcap;
    a.cap_log2 = d->softcap * log2e;
  } else {
    a.qscale = d->attn_scale * log2e;
    a.cap_log2 = 0.f;
  }
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  const int grid = units * S;
  if (mma) {
    CUtensorMap tk, tv;
    const long long rows = (long long)units * d->kv_capacity;
    const int T = tq_mma_keys_per_stage(hd);
    const int box = t->code_bytes < 128 ? t->code_bytes : 128;
    const hfa_status mk = kraw ? hfa_encode_kv_map(&tk, const_cast<void*>(k_raw), (int)rows, hd, T)
                               : hfa_encode_u8_map(&tk, k_codes, rows, t->code_bytes, box, T);
    if (mk != HFA_OK || hfa_encode_u8_map(&tv, v_codes, rows, t->code_bytes, box, T) != HFA_OK)
      return tq_fail(HFA_EINVAL, "cannot describe the code arrays to the TMA unit");
    e = launch_tq_attn_mma(a, tk, tv, hd, t->sbits, kraw, grid, s);
    if (e != cudaSuccess) return tq_fail(HFA_ECUDA, "attention launch: %s", cudaGetErrorString(e));
    return HFA_OK;
  }
  if (hd == 64) e = launch_attn_hd<64>(a, t->sbits, kraw, grid, s);
  else if (hd == 128) e = launch_attn_hd<128>(a, t->sbits, kraw, grid, s);
  else if (hd == 256) e = launch_attn_hd<256>(a, t->sbits, kraw, grid, s);
  else e = launch_attn_hd<512>(a, t->sbits, kraw, grid, s);
  if (e != cudaSuccess) return tq_fail(HFA_ECUDA, "attention launch: %s", cudaGetErrorString(e));
  return HFA_OK;
}
