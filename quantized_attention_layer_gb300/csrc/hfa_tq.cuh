// hfa_tq.cuh -- pieces shared by the two flash-decode kernels over the quantised
// (TurboQuant) KV cache (k_tq.cu: CUDA cores, every head dim; k_tq_mma.cu: tensor cores):
// the normalised FWHT of rows in shared memory, and the last CTA's merge of the chunk
// records followed by the inverse rotation.
//
// gemma4/gpu_full_attn.rs, encode_one_layer: the query is rotated like the keys (sign
// pre-multiply, normalised FWHT per 256-dim block), scores and the weighted sum of V are
// taken in the rotated domain, and the output is rotated back (fwht_sign_undo).
#pragma once

#include "hfa_common.cuh"

namespace hfa {

// Normalised FWHT (blocks of n <= 256 values) of `count` rows of `row_len` floats, `stride`
// apart, by threads tid = 0 .. nthr-1 that all call it with the same arguments; the
// butterflies in the order 1, 2, 4, ... (each a + b, a - b), then the 1/sqrt(n) scale.
// `sync` is the barrier of those threads.
template <typename Sync>
__device__ __forceinline__ void tq_fwht_rows(float* v, int count, int stride, int n, int row_len,
                                             int tid, int nthr, Sync sync) {
  for (int h = 1; h < n; h <<= 1) {
    const int pairs = count * (row_len / 2);
    for (int p = tid; p < pairs; p += nthr) {
      const int r = p / (row_len / 2), k = p - r * (row_len / 2);
      // k-th pair of the row: block base + index with bit h clear
      const int blk = k / (n / 2), kk = k - blk * (n / 2);
      const int i = blk * n + (kk / h) * 2 * h + (kk % h);
      float* x = v + r * stride;
      const float a0 = x[i], a1 = x[i + h];
      x[i] = a0 + a1;
      x[i + h] = a0 - a1;
    }
    sync();
  }
  const float sc = rsqrtf((float)n);
  for (int e = tid; e < count * row_len; e += nthr) {
    const int r = e / row_len, i = e - r * row_len;
    v[r * stride + i] *= sc;
  }
  sync();
}

// Normalised FWHT of one block of N (32..256) floats at v by one warp, in registers: lane
// l holds elements l R .. l R + R - 1 (R = N / 32); butterflies 1 .. R / 2 inside the
// lane, then R .. N / 2 across lanes by shuffles (the lane whose bit is set takes
// partner - own, the other own + partner), the same additions in the same order as
// tq_fwht_rows.
template <int N>
__device__ __forceinline__ void tq_fwht_warp(float* v, int lane) {
  constexpr int R = N / 32;
  static_assert(R >= 1 && N <= 256, "32 .. 256 values per block");
  float x[R];
#pragma unroll
  for (int j = 0; j < R; ++j) x[j] = v[lane * R + j];
#pragma unroll
  for (int h = 1; h < R; h <<= 1)
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (!(j & h)) {
        const float a0 = x[j], a1 = x[j + h];
        x[j] = a0 + a1;
        x[j + h] = a0 - a1;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, x[j], m);
      x[j] = (lane & m) ? p - x[j] : x[j] + p;
    }
  const float sc = rsqrtf((float)N);
#pragma unroll
  for (int j = 0; j < R; ++j) v[lane * R + j] = x[j] * sc;
}

// Columns of chunk records ([n][8][HD + 4]: O, m, l; column c = head c / (HD / 4), dims
// 4 (c mod (HD / 4)) ..): the thread's columns are c = tid + k nthr (k < CPT).  A batch is
// four records' values of all of them, loaded together; batches are added in record order.
template <int HD, int CPT>
__device__ __forceinline__ void tq_load_columns(const float* up, int n, int sp0, int G,
                                                float4 (&v)[CPT][4], int tid, int nthr) {
  constexpr int RS = HD + 4, Q4 = HD / 4;
  const int ncol = G * Q4;
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = tid + k * nthr < ncol ? tid + k * nthr : ncol - 1;  // in range
    const int h = c / Q4, d4 = c - h * Q4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int sp = sp0 + u < n ? sp0 + u : n - 1;  // in range
      v[k][u] = __ldcg(reinterpret_cast<const float4*>(up + (sp * 8 + h) * RS) + d4);
    }
  }
}
template <int HD, int CPT>
__device__ __forceinline__ void tq_add_columns(const float4 (&v)[CPT][4], int n, int sp0, int G,
                                               const float* wsm, float4 (&acc)[CPT], int tid,
                                               int nthr) {
  constexpr int Q4 = HD / 4;
  const int ncol = G * Q4;
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = tid + k * nthr;
    if (c < ncol) {
      const int h = c / Q4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (sp0 + u < n) {
          const float w = wsm[h * n + sp0 + u];
          acc[k].x = fmaf(w, v[k][u].x, acc[k].x);
          acc[k].y = fmaf(w, v[k][u].y, acc[k].y);
          acc[k].z = fmaf(w, v[k][u].z, acc[k].z);
          acc[k].w = fmaf(w, v[k][u].w, acc[k].w);
        }
      }
    }
  }
}

// The per-head weights of n records: wsm[h n + sp] = 2^(m_sp - M) (times `norm` ? 1 / den :
// 1), M = max m_sp, den = sum 2^(m_sp - M) l_sp; every m and l of a head loaded in one
// round (up to 256 records).  One warp per head; returns nothing, writes M and den through
// the callback of the head's lane 0.
template <int HD, typename OnHead>
__device__ __forceinline__ void tq_record_weights(const float* up, int n, int G, float* wsm,
                                                  bool norm, OnHead on_head) {
  constexpr int RS = HD + 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  for (int h = warp; h < G; h += nw) {
    float mv[8], lv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int sp = lane + 32 * k;
      mv[k] = sp < n ? __ldcg(up + (sp * 8 + h) * RS + HD) : -INFINITY;
      lv[k] = sp < n ? __ldcg(up + (sp * 8 + h) * RS + HD + 1) : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < 8; ++k) M = fmaxf(M, mv[k]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mu = M == -INFINITY ? 0.f : M;
    float f[8], den = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      f[k] = exp2f(mv[k] - Mu);
      den += f[k] * lv[k];
    }
    den = warp_sum(den);
    const float inv = norm ? (den > 0.f ? 1.f / den : 0.f) : 1.f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (lane + 32 * k < n) wsm[h * n + lane + 32 * k] = f[k] * inv;
    if (lane == 0) on_head(h, M, den);
  }
}

// Folds n chunk records at `up` ([n][8][HD + 4]: O, m, l) into one record at `dst` of the
// same form: m = max m_s, l = sum 2^(m_s - m) l_s, O = sum 2^(m_s - m) O_s (not normalised,
// so folds compose), the records added in order.  Every thread of the CTA (NTHR of them)
// calls it; wsm holds G x n floats of shared memory.  The first records' columns are in
// flight while the weights are formed.
template <int HD, int NTHR>
__device__ void tq_fold_records(const float* up, int n, int G, float* wsm, float* dst) {
  constexpr int RS = HD + 4, Q4 = HD / 4, CPT = (8 * Q4 + NTHR - 1) / NTHR;
  const int tid = threadIdx.x, nthr = blockDim.x;
  float4 v[CPT][4];
  tq_load_columns<HD, CPT>(up, n, 0, G, v, tid, nthr);
  tq_record_weights<HD>(up, n, G, wsm, false, [&](int h, float M, float den) {
    dst[h * RS + HD] = M;
    dst[h * RS + HD + 1] = den;
  });
  __syncthreads();
  float4 acc[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  tq_add_columns<HD, CPT>(v, n, 0, G, wsm, acc, tid, nthr);
  for (int sp0 = 4; sp0 < n; sp0 += 4) {
    tq_load_columns<HD, CPT>(up, n, sp0, G, v, tid, nthr);
    tq_add_columns<HD, CPT>(v, n, sp0, G, wsm, acc, tid, nthr);
  }
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = tid + k * nthr;
    if (c < G * Q4) reinterpret_cast<float4*>(dst + (c / Q4) * RS)[c % Q4] = acc[k];
  }
}

// The last CTA of a (sequence, KV head): the chunk records at `up` ([splits][8][HD + 4]:
// O in the rotated domain, then m and l in base-2 units) combined with the weights
// 2^(m_s - M) / sum_s' 2^(m_s' - M) l_s', the chunks added in order, then rotated back
// (the normalised FWHT is its own inverse; then the signs) into o ([G][HD]).  wsm holds
// G x splits floats and s_o G x HD floats of shared memory; every thread of the CTA (NTHR
// of them) calls it.
template <int HD, int NTHR>
__device__ void tq_merge_records(const float* up, int splits, int G, float* wsm, float* s_o,
                                 const float* signs, float* o) {
  constexpr int BLK = HD < 256 ? HD : 256;
  constexpr int Q4 = HD / 4, CPT = (8 * Q4 + NTHR - 1) / NTHR;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
  float4 v[CPT][4];
  tq_load_columns<HD, CPT>(up, splits, 0, G, v, tid, nthr);
  tq_record_weights<HD>(up, splits, G, wsm, true, [](int, float, float) {});
  __syncthreads();
  // o[h][i] = sum_s w[h][s] O_s[h][i], the chunks added in order
  float4 acc[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  tq_add_columns<HD, CPT>(v, splits, 0, G, wsm, acc, tid, nthr);
  for (int sp0 = 4; sp0 < splits; sp0 += 4) {
    tq_load_columns<HD, CPT>(up, splits, sp0, G, v, tid, nthr);
    tq_add_columns<HD, CPT>(v, splits, sp0, G, wsm, acc, tid, nthr);
  }
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = tid + k * nthr;
    if (c < G * Q4) reinterpret_cast<float4*>(s_o)[c] = acc[k];
  }
  __syncthreads();
  for (int r = warp; r < G * (HD / BLK); r += nw) tq_fwht_warp<BLK>(s_o + r * BLK, lane);
  __syncthreads();
  for (int e = tid; e < G * HD; e += nthr) {
    const int h = e / HD, i = e - h * HD;
    o[h * HD + i] = s_o[h * HD + i] * signs[i];
  }
}

}  // namespace hfa
