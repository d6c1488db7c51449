// hfa_finish.cuh -- epilogues that run once a head (QKV) or a row group (o_proj) of a
// projection is complete: per-head RMSNorm, NeoX RoPE and the bf16 KV append
// (gemma4/gpu_full_attn.rs, encode_one_layer: fused per-head norm + RoPE, GPU V norm,
// dense KV copy), and the residual add (dflash/forward.rs, dispatch_dflash_residual_add).
#pragma once
#include "hfa_common.cuh"
#include "hfa_internal.h"

namespace hfa {

// Cosine and sine of phi = P * theta^(-2i/hd) with phi reduced exactly enough in fp32:
// u = P * g with g = theta^(-2i/hd) / (2 pi) held as an fp32 (hi, lo) pair; the product
// P * hi is split into its rounded value and exact error (fma), the integer part is
// dropped, and sincospi of twice the fractional turn gives the rotation.
__device__ __forceinline__ void rope_cs(int P, float2 gpair, float& c, float& s) {
  const float Pf = (float)P;
  const float p1 = Pf * gpair.x;
  const float e1 = fmaf(Pf, gpair.x, -p1);
  const float k = rintf(p1);
  const float r = (p1 - k) + (e1 + Pf * gpair.y);
  sincospif(2.0f * r, &s, &c);
}

// Epilogue of one token row b of one attention head (QKV mode): v holds rows
// [hh*hd, hh*hd + hd) of the QKV output for that token, lane + 32 j in v[j].
// Used by the verify-block GEMM once the k-split partial sums are added.
template <int HD>
static __device__ __forceinline__ void finish_head_row(const GemvArgs& a, int hh, int b, float (&v)[HD / 32],
                                       int lane) {
  constexpr int J = HD / 32;   // values per lane; pairs (j, j + J/2) are RoPE partners
  const int kind = hh < a.nh ? 0 : (hh < a.nh + a.nkv ? 1 : 2);  // q, k, v
  if (kind == 0 && a.kv_only) return;
  const int seq = a.rows_are_tokens ? 0 : b;
  const int P = a.rows_are_tokens ? a.base_pos + b : a.seq_pos[b];
  if (kind == 1 && a.k_eq_v && P >= 0 && (a.ring || P < a.C)) {
    // no V projection: V is the raw K, RMS-normalised per head with unit weight
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) ss += v[j] * v[j];
    const float inv = rsqrtf(warp_sum(ss) / HD + a.eps);
    const int kvh = hh - a.nh;
    const int slot = a.ring ? P % a.C : P;
    __nv_bfloat16* dst = a.v_cache + (((size_t)seq * a.nkv + kvh) * a.C + slot) * HD;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      dst[lane + 32 * j] = __float2bfloat16_rn(v[j] * inv);
      if (a.v_tap) a.v_tap[((size_t)b * a.nkv + kvh) * HD + lane + 32 * j] = v[j] * inv;
    }
  }
  if (kind < 2 || a.v_unit_norm) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) ss += v[j] * v[j];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / HD + a.eps);
    const float* w = kind == 0 ? a.w_q : a.w_k;  // a valid address for v too (unused)
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float wj = w[lane + 32 * j];
      v[j] *= inv * (kind < 2 ? wj : 1.0f);
    }
  }
  if (kind < 2) {
#pragma unroll
    for (int j = 0; j < J / 2; ++j) {
      float c, s;
      rope_cs(P, a.rope_g[lane + 32 * j], c, s);
      const float x0 = v[j], x1 = v[j + J / 2];
      v[j] = x0 * c - x1 * s;
      v[j + J / 2] = x0 * s + x1 * c;
    }
  }
  if (kind == 0) {
    float* q = a.q_out + ((size_t)b * a.nh + hh) * HD;
#pragma unroll
    for (int j = 0; j < J; ++j) q[lane + 32 * j] = v[j];
    if (HD == 128 && a.qx) {
      // the tensor-core operand of the verify attention: query row qr = b G + hh % G of
      // KV head hh / G, scaled, bf16 hi in row qr and lo in row qr + 64, dims in two
      // 64-wide boxes, 16-byte chunk c of row r at (c XOR (r % 8))
      const int qr = b * a.G + hh % a.G;
      uint8_t* img = a.qx + (size_t)(hh / a.G) * 32768;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int d = lane + 32 * j;
        __nv_bfloat16 h, lo;
        split_bf16(v[j] * a.qscale, h, lo);
        const int box = d >> 6, c = (d & 63) >> 3, e = d & 7;
        const int rh = qr, rl = qr + 64;
        *reinterpret_cast<__nv_bfloat16*>(img + box * 16384 + rh * 128 + ((c ^ (rh & 7)) << 4) + 2 * e) = h;
        *reinterpret_cast<__nv_bfloat16*>(img + box * 16384 + rl * 128 + ((c ^ (rl & 7)) << 4) + 2 * e) = lo;
      }
    }
  } else {
    const int kvh = kind == 1 ? hh - a.nh : hh - a.nh - a.nkv;
    if (P < 0 || (!a.ring && P >= a.C)) {
      if (lane == 0) atomicOr(a.err, kErrBadPosition);
      return;
    }
    const int slot = a.ring ? P % a.C : P;
    __nv_bfloat16* cache = kind == 1 ? a.k_cache : a.v_cache;
    __nv_bfloat16* dst = cache + (((size_t)seq * a.nkv + kvh) * a.C + slot) * HD;
    float* tap = kind == 1 ? a.k_tap : a.v_tap;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      dst[lane + 32 * j] = __float2bfloat16_rn(v[j]);
      if (tap) tap[((size_t)b * a.nkv + kvh) * HD + lane + 32 * j] = v[j];
    }
  }
}

// Epilogue of one output (o_proj mode): token row b, output feature `row`, projection
// value y: out = bf16(x + y), or y kept in y_post for the post-attention norm pass (which
// needs the whole row's mean of y^2 first).
static __device__ __forceinline__ void finish_row_item(const GemvArgs& a, int b, int row,
                                                       float y) {
  const size_t off = (size_t)b * a.R * 16 + row;
  if (a.y_post) {
    a.y_post[off] = y;
    return;
  }
  const float o = __bfloat162float(a.x[off]) + y;
  a.out[off] = __float2bfloat16_rn(o);
  if (a.out_tap) a.out_tap[off] = o;
}

}  // namespace hfa
