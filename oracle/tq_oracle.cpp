// tq_oracle.cpp -- plain fp64 CPU oracle of the quantised (TurboQuant) KV cache.
//
// TEST INFRASTRUCTURE ONLY (see tq_oracle.h for the sources and the readings).  Every
// function is the plain definition, in double precision, in the order the pages give:
// sign pre-multiply, normalised FWHT, block norm, nearest Lloyd-Max centroid.
#include "tq_oracle.h"

#include <cmath>
#include <vector>

extern "C" double orc_bf16_to_f64(uint16_t b);

namespace {

const double kInvSqrt2 = 0.70710678118654752440;
const double kInvSqrt2Pi = 0.39894228040143267794;

double pdf(double x) { return std::isinf(x) ? 0.0 : kInvSqrt2Pi * std::exp(-0.5 * x * x); }
// x * pdf(x), 0 at +-inf
double xpdf(double x) { return std::isinf(x) ? 0.0 : x * pdf(x); }

// P(a < X < b) for X ~ N(0, 1), from erfc on the side that keeps its precision
double mass(double a, double b) {
  if (a >= 0.0) return 0.5 * (std::erfc(a * kInvSqrt2) - std::erfc(b * kInvSqrt2));
  if (b <= 0.0) return 0.5 * (std::erfc(-b * kInvSqrt2) - std::erfc(-a * kInvSqrt2));
  return 1.0 - 0.5 * std::erfc(-a * kInvSqrt2) - 0.5 * std::erfc(b * kInvSqrt2);
}

// quantile of N(0, 1) by bisection on the CDF (initial centroids only)
double quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    if (mass(-INFINITY, mid) < p) lo = mid;
    else hi = mid;
  }
  return 0.5 * (lo + hi);
}

int block_dims(int hd) { return hd < 256 ? hd : 256; }

// index of the cell of e: the largest i with boundaries[i] <= e (boundaries[0] = -inf)
int cell_of(double e, const double* boundaries, int levels) {
  int c = 0;
  for (int i = 1; i < levels; ++i)
    if (e >= boundaries[i]) c = i;
  return c;
}

}  // namespace

extern "C" {

int orc_lloyd_max_normal(int levels, double* c, double* b) {
  for (int i = levels / 2; i < levels; ++i) {
    c[i] = quantile((i + 0.5) / levels);
    c[levels - 1 - i] = -c[i];
  }
  b[0] = -INFINITY;
  b[levels] = INFINITY;
  int rounds = 0;
  for (; rounds < 2000000; ++rounds) {
    for (int i = 1; i < levels; ++i) b[i] = 0.5 * (c[i - 1] + c[i]);  // nearest neighbour
    double moved = 0.0;
    for (int i = levels / 2; i < levels; ++i) {  // centroid: E[X | b_i < X < b_{i+1}]
      const double m = (pdf(b[i]) - pdf(b[i + 1])) / mass(b[i], b[i + 1]);
      moved = std::fmax(moved, std::fabs(m - c[i]));
      c[i] = m;
      c[levels - 1 - i] = -m;  // N(0, 1) is symmetric: so is its quantiser
    }
    if (moved < 1e-13) break;
  }
  for (int i = 1; i < levels; ++i) b[i] = 0.5 * (c[i - 1] + c[i]);
  return rounds + 1;
}

double orc_lloyd_max_mse(int levels, const double* c, const double* b) {
  // on [a, b]: int x^2 phi = P + a phi(a) - b phi(b), int x phi = phi(a) - phi(b), int phi = P
  double mse = 0.0;
  for (int i = 0; i < levels; ++i) {
    const double lo = b[i], hi = b[i + 1];
    const double P = mass(lo, hi);
    const double m1 = pdf(lo) - pdf(hi);
    const double m2 = P + xpdf(lo) - xpdf(hi);
    mse += m2 - 2.0 * c[i] * m1 + c[i] * c[i] * P;
  }
  return mse;
}

void orc_fwht(double* x, int n) {
  for (int h = 1; h < n; h *= 2)
    for (int i = 0; i < n; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        const double a = x[j], bb = x[j + h];
        x[j] = a + bb;
        x[j + h] = a - bb;
      }
  const double s = 1.0 / std::sqrt((double)n);
  for (int i = 0; i < n; ++i) x[i] *= s;
}

void orc_tq_rotate(double* x, int hd, const int8_t* signs) {
  const int B = block_dims(hd);
  for (int i = 0; i < hd; ++i) x[i] *= (double)signs[i];  // sign pre-multiply
  for (int k = 0; k < hd; k += B) orc_fwht(x + k, B);       // normalised FWHT per block
}

void orc_tq_unrotate(double* x, int hd, const int8_t* signs) {
  const int B = block_dims(hd);
  for (int k = 0; k < hd; k += B) orc_fwht(x + k, B);       // the FWHT is its own inverse
  for (int i = 0; i < hd; ++i) x[i] *= (double)signs[i];  // sign undo
}

// 4-bit codes two to a byte; 5-, 6- and 8-bit codes one to a byte (the byte-packed form)
int orc_tq_code_bytes(int hd, int bits) { return bits == 4 ? hd / 2 : hd; }
int orc_tq_blocks(int hd) { return hd / block_dims(hd); }

void orc_tq_encode_row(const double* x, int hd, const int8_t* signs, int bits,
                       const double* boundaries, uint8_t* codes, float* norms) {
  const int B = block_dims(hd), levels = 1 << bits;
  std::vector<double> u(x, x + hd);
  orc_tq_rotate(u.data(), hd, signs);
  std::vector<int> code(hd);
  for (int k = 0; k < hd; k += B) {
    double ss = 0.0;
    for (int i = k; i < k + B; ++i) ss += u[i] * u[i];
    const double norm = std::sqrt(ss / B);
    norms[k / B] = (float)norm;
    for (int i = k; i < k + B; ++i)
      code[i] = cell_of(norm > 0.0 ? u[i] / norm : 0.0, boundaries, levels);
  }
  if (bits != 4) {
    for (int i = 0; i < hd; ++i) codes[i] = (uint8_t)code[i];
  } else {
    for (int j = 0; j < hd / 2; ++j) codes[j] = (uint8_t)(code[2 * j] | (code[2 * j + 1] << 4));
  }
}

void orc_tq_decode_row(const uint8_t* codes, const float* norms, int hd, int bits,
                       const double* centroids, double* u) {
  const int B = block_dims(hd);
  for (int i = 0; i < hd; ++i) {
    const int c = bits != 4 ? codes[i] : ((codes[i / 2] >> (4 * (i & 1))) & 15);
    u[i] = centroids[c] * (double)norms[i / B];
  }
}

void orc_attend_tq(const double* q, int hd, int bits, const int8_t* signs,
                   const double* centroids, const uint8_t* k_codes, const float* k_norms,
                   const uint16_t* k_bf16, const uint8_t* v_codes, const float* v_norms,
                   const long* rows, long n, double scale, double softcap, double* o) {
  const int cb = orc_tq_code_bytes(hd, bits), nb = orc_tq_blocks(hd);
  std::vector<double> qr(q, q + hd), kv(hd), s(n > 0 ? n : 1);
  orc_tq_rotate(qr.data(), hd, signs);  // Q pre-rotated like the coded keys
  double m = -INFINITY;
  for (long j = 0; j < n; ++j) {
    double dot = 0.0;
    if (k_codes) {
      orc_tq_decode_row(k_codes + (size_t)rows[j] * cb, k_norms + (size_t)rows[j] * nb, hd,
                        bits, centroids, kv.data());
      for (int i = 0; i < hd; ++i) dot += qr[i] * kv[i];
    } else {  // hybrid: raw keys, raw query
      for (int i = 0; i < hd; ++i) dot += q[i] * orc_bf16_to_f64(k_bf16[(size_t)rows[j] * hd + i]);
    }
    double sj = scale * dot;
    if (softcap > 0.0) sj = softcap * std::tanh(sj / softcap);
    s[j] = sj;
    if (sj > m) m = sj;
  }
  double l = 0.0;
  for (long j = 0; j < n; ++j) {
    s[j] = std::exp(s[j] - m);
    l += s[j];
  }
  for (int i = 0; i < hd; ++i) o[i] = 0.0;
  for (long j = 0; j < n; ++j) {
    orc_tq_decode_row(v_codes + (size_t)rows[j] * cb, v_norms + (size_t)rows[j] * nb, hd, bits,
                      centroids, kv.data());
    const double p = s[j] / l;
    for (int i = 0; i < hd; ++i) o[i] += p * kv[i];
  }
  orc_tq_unrotate(o, hd, signs);  // the weighted sum back out of the rotated domain
}

}  // extern "C"
