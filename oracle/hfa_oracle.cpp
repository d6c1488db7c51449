// hfa_oracle.cpp -- plain fp64 CPU oracle for the decode step and the verify block of
// one Gemma-style attention layer.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the CPU-baseline
// leg of the benchmark; never by the CUDA library.  No blocking, fusion or reordering
// beyond what each definition states; OpenMP only spreads independent rows / heads
// over cores.  Page references ([P1], [P2], [P3]) are spelled out in hfa_oracle.h.
#include "hfa_oracle.h"

#include <cmath>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// ---------------------------------------------------------------- scalar formats

double orc_bf16_to_f64(uint16_t b) {
  // bf16 is the top half of an IEEE binary32 pattern: exact in double.
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t orc_f64_to_bf16(double v) {
  // Round directly from double to bf16 (1 sign, 8 exponent, 7 fraction bits),
  // nearest, ties to even.  No detour through binary32 (that would round twice).
  if (std::isnan(v)) return 0x7FC0;
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return sign | 0x7F80;
  int e;
  std::frexp(a, &e);        // a in [2^(e-1), 2^e)
  int E = e - 1;            // a = 1.f * 2^E
  if (E < -126) E = -126;   // below the normal range: fixed quantum 2^-133
  double quantum = std::ldexp(1.0, E - 7);
  double r = std::nearbyint(a / quantum);  // default rounding mode: ties to even
  if (r >= 256.0) { E += 1; r = 128.0; }
  uint32_t bits;
  if (r >= 128.0) {
    int biased = E + 127;
    if (biased >= 255) return sign | 0x7F80;
    bits = ((uint32_t)biased << 7) | ((uint32_t)r - 128u);
  } else {
    bits = (uint32_t)r;  // subnormal
  }
  return (uint16_t)(sign | bits);
}

double orc_f16_to_f64(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = std::ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = std::ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

// ---------------------------------------------------------------- Q8_0 and matvec

void orc_q8_0_dequant_row(const uint8_t* row_blocks, int cols, double* out) {
  int nb = cols / 32;
  for (int b = 0; b < nb; ++b) {
    const uint8_t* blk = row_blocks + (size_t)b * 34;
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));  // little endian
    double d = orc_f16_to_f64(dbits);
    for (int i = 0; i < 32; ++i) out[b * 32 + i] = d * (double)(int8_t)blk[2 + i];
  }
}

void orc_q8_0_matvec(const uint8_t* blocks, int rows, int cols, const double* x, double* y) {
  size_t row_bytes = (size_t)(cols / 32) * 34;
#pragma omp parallel
  {
    std::vector<double> w(cols);
#pragma omp for schedule(static)
    for (int r = 0; r < rows; ++r) {
      orc_q8_0_dequant_row(blocks + (size_t)r * row_bytes, cols, w.data());
      double acc = 0.0;
      for (int c = 0; c < cols; ++c) acc += w[c] * x[c];
      y[r] = acc;
    }
  }
}

void orc_q8_0_matvec_blockwise(const uint8_t* blocks, int rows, int cols, const double* x,
                               double* y) {
  size_t row_bytes = (size_t)(cols / 32) * 34;
  int nb = cols / 32;
  for (int r = 0; r < rows; ++r) {
    double acc = 0.0;
    for (int b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (size_t)r * row_bytes + (size_t)b * 34;
      double d = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
      double s = 0.0;
      for (int i = 0; i < 32; ++i) s += (double)(int8_t)blk[2 + i] * x[b * 32 + i];
      acc += d * s;
    }
    y[r] = acc;
  }
}

void orc_bf16_matvec(const uint16_t* w, int rows, int cols, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    double acc = 0.0;
    const uint16_t* row = w + (size_t)r * cols;
    for (int c = 0; c < cols; ++c) acc += orc_bf16_to_f64(row[c]) * x[c];
    y[r] = acc;
  }
}

static void matvec(const orc_desc* d, const void* w, int rows, int cols, const double* x,
                   double* y) {
  if (d->weights_bf16) orc_bf16_matvec((const uint16_t*)w, rows, cols, x, y);
  else orc_q8_0_matvec((const uint8_t*)w, rows, cols, x, y);
}

// ---------------------------------------------------------------- norms and RoPE

void orc_rmsnorm(const double* x, const float* w, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / std::sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (w ? (double)w[i] : 1.0);
}

void orc_rope_neox(double* u, int hd, double pos, double theta) {
  orc_rope_neox_ff(u, hd, pos, theta, nullptr);
}

void orc_rope_neox_ff(double* u, int hd, double pos, double theta, const float* ff) {
  int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = std::pow(theta, -2.0 * i / hd);
    double phi = pos * inv_freq;
    if (ff) phi /= (double)ff[i];  // frequency factor of the pair (global layers)
    double c = std::cos(phi), s = std::sin(phi);
    double a = u[i], b = u[i + half];
    u[i] = a * c - b * s;
    u[i + half] = a * s + b * c;
  }
}

// ---------------------------------------------------------------- slots, visibility

long orc_kv_slot(long pos, long capacity, int ring) { return ring ? pos % capacity : pos; }

int orc_key_visible(long p, long P, int sliding, long window) {
  if (p < 0 || p > P) return 0;
  if (sliding && p <= P - window) return 0;
  return 1;
}

long orc_slot_position(long slot, long P, long capacity, int ring) {
  if (slot < 0 || slot >= capacity) return -1;
  if (!ring) return slot <= P ? slot : -1;
  if (slot > P) return -1;
  return P - ((P - slot) % capacity);
}

// ---------------------------------------------------------------- attention

void orc_attend(const double* q, const uint16_t* k_rows, const uint16_t* v_rows, int hd,
                const long* rows, long n, double scale, double softcap, double* weights,
                double* o) {
  std::vector<double> s(n > 0 ? n : 1);
  double m = -INFINITY;
  for (long j = 0; j < n; ++j) {
    const uint16_t* kr = k_rows + (size_t)rows[j] * hd;
    double dot = 0.0;
    for (int i = 0; i < hd; ++i) dot += q[i] * orc_bf16_to_f64(kr[i]);
    double sj = scale * dot;
    if (softcap > 0.0) sj = softcap * std::tanh(sj / softcap);
    s[j] = sj;
    if (sj > m) m = sj;
  }
  double l = 0.0;
  for (long j = 0; j < n; ++j) { s[j] = std::exp(s[j] - m); l += s[j]; }
  for (int i = 0; i < hd; ++i) o[i] = 0.0;
  for (long j = 0; j < n; ++j) {
    double p = s[j] / l;
    if (weights) weights[j] = p;
    const uint16_t* vr = v_rows + (size_t)rows[j] * hd;
    for (int i = 0; i < hd; ++i) o[i] += p * orc_bf16_to_f64(vr[i]);
  }
}

// ---------------------------------------------------------------- layer pieces

static int check_desc(const orc_desc* d) {
  if (!d || d->hidden <= 0 || d->num_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0)
    return -1;
  if (d->hidden % 32 || d->num_heads % d->num_kv_heads || d->head_dim % 2) return -1;
  if (d->kv_capacity <= 0) return -1;
  if (d->layer_type == 0 && d->window <= 0) return -1;
  return 0;
}

// Steps 1-4 for one token: input RMSNorm, Q/K/V projections, per-head norms, RoPE.
static void project_token(const orc_desc* d, const void* wq, const void* wk, const void* wv,
                          const float* w_in, const float* w_q, const float* w_k,
                          const uint16_t* x_row, long P, double* q, double* k, double* v) {
  int H = d->hidden, nh = d->num_heads, nkv = d->num_kv_heads, hd = d->head_dim;
  std::vector<double> xd(H), n(H);
  for (int i = 0; i < H; ++i) xd[i] = orc_bf16_to_f64(x_row[i]);
  orc_rmsnorm(xd.data(), w_in, H, d->eps, n.data());                 // [P1] pre-attn norm
  matvec(d, wq, nh * hd, H, n.data(), q);                            // [P1] QKV projections
  matvec(d, wk, nkv * hd, H, n.data(), k);
  if (d->k_eq_v)                                  // [P2] no v_proj: V comes from the raw K
    std::memcpy(v, k, (size_t)nkv * hd * sizeof(double));
  else
    matvec(d, wv, nkv * hd, H, n.data(), v);
  std::vector<double> t(hd);
  for (int h = 0; h < nh; ++h) {                                     // [P1] q_norm + RoPE
    orc_rmsnorm(q + h * hd, w_q, hd, d->eps, t.data());
    std::memcpy(q + h * hd, t.data(), hd * sizeof(double));
    orc_rope_neox_ff(q + h * hd, hd, (double)P, d->rope_theta, d->rope_freq_factors);
  }
  for (int h = 0; h < nkv; ++h) {                                    // [P1] k_norm + RoPE
    orc_rmsnorm(k + h * hd, w_k, hd, d->eps, t.data());
    std::memcpy(k + h * hd, t.data(), hd * sizeof(double));
    orc_rope_neox_ff(k + h * hd, hd, (double)P, d->rope_theta, d->rope_freq_factors);
    if (d->v_unit_norm || d->k_eq_v) {                               // [P1] GPU V norm
      orc_rmsnorm(v + h * hd, nullptr, hd, d->eps, t.data());
      std::memcpy(v + h * hd, t.data(), hd * sizeof(double));
    }
  }
}

// Step 5: append k, v (rounded to bf16) at the slot of position P.
static void append_kv(const orc_desc* d, uint16_t* kc, uint16_t* vc, long P, const double* k,
                      const double* v) {
  int nkv = d->num_kv_heads, hd = d->head_dim;
  long C = d->kv_capacity;
  long slot = orc_kv_slot(P, C, d->ring);
  for (int h = 0; h < nkv; ++h)
    for (int i = 0; i < hd; ++i) {
      size_t off = ((size_t)h * C + slot) * hd + i;
      kc[off] = orc_f64_to_bf16(k[h * hd + i]);
      vc[off] = orc_f64_to_bf16(v[h * hd + i]);
    }
}

// Step 6 for all query heads of one token at position P; P_written is the last
// position appended (it decides what a ring slot holds).
static void attend_token(const orc_desc* d, const uint16_t* kc, const uint16_t* vc, long P,
                         long P_written, const double* q, double* o) {
  int nh = d->num_heads, nkv = d->num_kv_heads, hd = d->head_dim, g = nh / nkv;
  long C = d->kv_capacity;
  std::vector<long> rows;
  rows.reserve(C);
  for (long s = 0; s < C; ++s) {
    long p = orc_slot_position(s, P_written, C, d->ring);
    if (p >= 0 && orc_key_visible(p, P, d->layer_type == 0, d->window)) rows.push_back(s);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < nh; ++h) {
    int kvh = h / g;
    const uint16_t* kb = kc + (size_t)kvh * C * hd;
    const uint16_t* vb = vc + (size_t)kvh * C * hd;
    orc_attend(q + h * hd, kb, vb, hd, rows.data(), (long)rows.size(), d->attn_scale,
               d->softcap, nullptr, o + h * hd);
  }
}

// Steps 7-8: o_proj and the residual add.
static void output_token(const orc_desc* d, const void* wo, const uint16_t* x_row,
                         const double* o, double* out, uint16_t* out_bf16) {
  int H = d->hidden;
  std::vector<double> y(H);
  matvec(d, wo, H, d->num_heads * d->head_dim, o, y.data());  // [P1] O-proj
  if (d->w_post) {                              // [P1] fused post-attention norm + add
    std::vector<double> t(H);
    orc_rmsnorm(y.data(), d->w_post, H, d->eps, t.data());
    y = t;
  }
  for (int i = 0; i < H; ++i) {                                 // [P3] residual add
    double r = orc_bf16_to_f64(x_row[i]) + y[i];
    if (out) out[i] = r;
    if (out_bf16) out_bf16[i] = orc_f64_to_bf16(r);
  }
}

int orc_decode_step(const orc_desc* d, const void* wq, const void* wk, const void* wv,
                    const void* wo, const float* w_in, const float* w_q, const float* w_k,
                    const uint16_t* x, const int32_t* seq_pos, int B, uint16_t* k_cache,
                    uint16_t* v_cache, double* q_out, double* k_out, double* v_out,
                    double* attn_out, double* out, uint16_t* out_bf16) {
  if (check_desc(d) || B <= 0 || !x || !seq_pos || !k_cache || !v_cache) return -1;
  int H = d->hidden, nh = d->num_heads, nkv = d->num_kv_heads, hd = d->head_dim;
  long C = d->kv_capacity;
  for (int b = 0; b < B; ++b) {
    if (seq_pos[b] < 0) return -1;
    if (!d->ring && seq_pos[b] >= C) return -1;
  }
  std::vector<double> q(nh * hd), k(nkv * hd), v(nkv * hd), o(nh * hd);
  for (int b = 0; b < B; ++b) {
    long P = seq_pos[b];
    const uint16_t* xr = x + (size_t)b * H;
    uint16_t* kc = k_cache + (size_t)b * nkv * C * hd;
    uint16_t* vc = v_cache + (size_t)b * nkv * C * hd;
    project_token(d, wq, wk, wv, w_in, w_q, w_k, xr, P, q.data(), k.data(), v.data());
    append_kv(d, kc, vc, P, k.data(), v.data());
    attend_token(d, kc, vc, P, P, q.data(), o.data());
    output_token(d, wo, xr, o.data(), out ? out + (size_t)b * H : nullptr,
                 out_bf16 ? out_bf16 + (size_t)b * H : nullptr);
    if (q_out) std::memcpy(q_out + (size_t)b * nh * hd, q.data(), nh * hd * sizeof(double));
    if (k_out) std::memcpy(k_out + (size_t)b * nkv * hd, k.data(), nkv * hd * sizeof(double));
    if (v_out) std::memcpy(v_out + (size_t)b * nkv * hd, v.data(), nkv * hd * sizeof(double));
    if (attn_out)
      std::memcpy(attn_out + (size_t)b * nh * hd, o.data(), nh * hd * sizeof(double));
  }
  return 0;
}

int orc_verify_block(const orc_desc* d, const void* wq, const void* wk, const void* wv,
                     const void* wo, const float* w_in, const float* w_q, const float* w_k,
                     const uint16_t* x, int L, int base_pos, uint16_t* k_cache,
                     uint16_t* v_cache, double* q_out, double* k_out, double* v_out,
                     double* attn_out, double* out, uint16_t* out_bf16) {
  if (check_desc(d) || L <= 0 || base_pos < 0 || !x || !k_cache || !v_cache) return -1;
  if (d->ring) return -1;  // a ring would overwrite keys earlier rows of the block still see
  int H = d->hidden, nh = d->num_heads, nkv = d->num_kv_heads, hd = d->head_dim;
  long last = (long)base_pos + L - 1;
  if (last >= d->kv_capacity) return -1;
  std::vector<double> q((size_t)L * nh * hd), k((size_t)L * nkv * hd), v((size_t)L * nkv * hd),
      o((size_t)L * nh * hd);
  for (int i = 0; i < L; ++i)
    project_token(d, wq, wk, wv, w_in, w_q, w_k, x + (size_t)i * H, base_pos + i,
                  &q[(size_t)i * nh * hd], &k[(size_t)i * nkv * hd], &v[(size_t)i * nkv * hd]);
  for (int i = 0; i < L; ++i)
    append_kv(d, k_cache, v_cache, base_pos + i, &k[(size_t)i * nkv * hd],
              &v[(size_t)i * nkv * hd]);
  // row i sees positions <= base_pos + i (causal), or the whole block on a full layer of
  // a bidirectional block [P3]
  const bool bidir = d->block_bidir && d->layer_type == 1;
  for (int i = 0; i < L; ++i)
    attend_token(d, k_cache, v_cache, bidir ? last : base_pos + i, last,
                 &q[(size_t)i * nh * hd], &o[(size_t)i * nh * hd]);
  for (int i = 0; i < L; ++i)
    output_token(d, wo, x + (size_t)i * H, &o[(size_t)i * nh * hd],
                 out ? out + (size_t)i * H : nullptr,
                 out_bf16 ? out_bf16 + (size_t)i * H : nullptr);
  if (q_out) std::memcpy(q_out, q.data(), q.size() * sizeof(double));
  if (k_out) std::memcpy(k_out, k.data(), k.size() * sizeof(double));
  if (v_out) std::memcpy(v_out, v.data(), v.size() * sizeof(double));
  if (attn_out) std::memcpy(attn_out, o.data(), o.size() * sizeof(double));
  return 0;
}

int orc_ctx_append(const orc_desc* d, const void* wk, const void* wv, const float* w_k,
                   const uint16_t* x_ctx, int S, int base_pos, uint16_t* k_cache,
                   uint16_t* v_cache, double* k_out, double* v_out) {
  if (check_desc(d) || S <= 0 || base_pos < 0 || !x_ctx || !k_cache || !v_cache) return -1;
  if (d->ring || (long)base_pos + S > d->kv_capacity) return -1;
  int H = d->hidden, nkv = d->num_kv_heads, hd = d->head_dim;
  std::vector<double> n(H), k((size_t)nkv * hd), v((size_t)nkv * hd), t(hd);
  for (int r = 0; r < S; ++r) {
    const long P = base_pos + r;
    for (int i = 0; i < H; ++i) n[i] = orc_bf16_to_f64(x_ctx[(size_t)r * H + i]);  // no norm
    matvec(d, wk, nkv * hd, H, n.data(), k.data());                             // [P3] k_proj
    if (d->k_eq_v) std::memcpy(v.data(), k.data(), k.size() * sizeof(double));
    else matvec(d, wv, nkv * hd, H, n.data(), v.data());                        // [P3] v_proj
    for (int h = 0; h < nkv; ++h) {
      orc_rmsnorm(&k[(size_t)h * hd], w_k, hd, d->eps, t.data());               // k_norm
      std::memcpy(&k[(size_t)h * hd], t.data(), hd * sizeof(double));
      orc_rope_neox_ff(&k[(size_t)h * hd], hd, (double)P, d->rope_theta, d->rope_freq_factors);
      if (d->v_unit_norm || d->k_eq_v) {
        orc_rmsnorm(&v[(size_t)h * hd], nullptr, hd, d->eps, t.data());
        std::memcpy(&v[(size_t)h * hd], t.data(), hd * sizeof(double));
      }
    }
    append_kv(d, k_cache, v_cache, P, k.data(), v.data());
    if (k_out) std::memcpy(k_out + (size_t)r * nkv * hd, k.data(), k.size() * sizeof(double));
    if (v_out) std::memcpy(v_out + (size_t)r * nkv * hd, v.data(), v.size() * sizeof(double));
  }
  return 0;
}

double orc_gelu_tanh(double x) {
  const double c = std::sqrt(2.0 / M_PI);
  return 0.5 * x * (1.0 + std::tanh(c * (x + 0.044715 * x * x * x)));
}

int orc_ffn_step(int H, int I, double eps, const uint8_t* wg, const uint8_t* wu,
                 const uint8_t* wd, const float* w_pre, const float* w_post,
                 const float* scalar, int scalar_len, const uint16_t* h, int B, double* a_out,
                 double* out, uint16_t* out_bf16) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32 || B <= 0 || !wg || !wu || !wd || !w_pre ||
      !w_post || !scalar || (scalar_len != 1 && scalar_len != H) || !h)
    return -1;
  std::vector<double> x(H), n(H), g(I), u(I), a(I), d(H);
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < H; ++i) x[i] = orc_bf16_to_f64(h[(size_t)b * H + i]);
    orc_rmsnorm(x.data(), w_pre, H, eps, n.data());            // [P1] pre-FF norm
    orc_q8_0_matvec(wg, I, H, n.data(), g.data());             // [P1] dense gate
    orc_q8_0_matvec(wu, I, H, n.data(), u.data());             // [P1] dense up
    for (int i = 0; i < I; ++i) a[i] = orc_gelu_tanh(g[i]) * u[i];  // [P1] fused_gelu_mul
    orc_q8_0_matvec(wd, H, I, a.data(), d.data());             // [P1] dense down
    std::vector<double> dn(H);
    orc_rmsnorm(d.data(), w_post, H, eps, dn.data());          // [P1] post-FF norm
    for (int i = 0; i < H; ++i) {                              // [P1] end of layer
      const double r = (x[i] + dn[i]) * (double)scalar[scalar_len == 1 ? 0 : i];
      if (out) out[(size_t)b * H + i] = r;
      if (out_bf16) out_bf16[(size_t)b * H + i] = orc_f64_to_bf16(r);
    }
    if (a_out) std::memcpy(a_out + (size_t)b * I, a.data(), I * sizeof(double));
  }
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

}  // extern "C"
