// k_ffn.cu -- the dense feed-forward half of the layer as one persistent kernel (sm_103a).
//
// gemma4/gpu_full_attn.rs, encode_one_layer: the dense MLP (pre-feed-forward RMSNorm,
// gate and up projections, fused_gelu_mul, down projection) and the end of the layer
// (RMSNorm of the down output with post_feedforward_layernorm, residual add, layer_scalar):
//   n = h (.) w_pre / rms(h);  a = gelu(Wg n) (.) (Wu n);  d = Wd a;
//   out = (h + d (.) w_post / rms(d)) (.) s,
// gelu(x) = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), rms(v) = sqrt(mean(v^2) + eps).
//
// One CTA per SM, launched cooperatively so that every CTA is resident while the CTAs
// poll one another's partial sums.  Three phases:
//   1  [Wg; Wu] times h (.) w_pre.  The row groups (16 rows) of Wg and Wu are interleaved
//      (gate r, up r) and cut into k-splits; a ring stage holds whole row groups of one
//      k-split, the consumer warps share its tiles (a row group's tiles split evenly over
//      the warps that own it) and add their sums through shared memory.  The partial sums
//      go out tagged with the step number (no grid barrier).  1/rms(h) is a per-row factor,
//      applied in phase 2.
//   2  Wd times a.  The operand of a k-split is formed from the phase-1 partial sums of its
//      columns: g, u summed over the k-splits and times 1/rms(h), a = gelu(g) u.
//   3  the end of the layer: d summed over the phase-2 k-splits, sum(d^2) per row exchanged
//      between the CTAs that share the row (tagged), out = (h + d w_post / rms(d)) s.
// A producer warp streams every weight tile of both phases through a ring of shared-memory
// stages with 1-D bulk copies: a stage is reloaded as soon as every consumer warp has read
// its tiles, phase 2's stages included -- they depend on nothing of the step, so HBM keeps
// streaming while the consumers wait for the phase-1 sums.  The ring fill starts once the
// activations of the first operand are in, whose loads would otherwise queue behind it.
//
// The GEMV is latency-bound on the warp MMA, so there are 16 consumer warps (8 with four
// batch tiles, whose registers allow no more) and each runs two tiles' MMAs interleaved.
// The warps that share a row group of a stage add their sums through shared memory (one
// of two buffers, alternating) behind a named barrier of their own, each warp storing a
// share of the results: no barrier spans the CTA within a phase.
//
// Every wait is bounded in wall time; a CTA that gives up sets an error bit, skips its
// remaining work (every barrier is still passed) and drains its copies in flight.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "hfa_common.cuh"
#include "hfa_gemv.cuh"
#include "hfa_internal.h"

namespace hfa {
namespace ffn {

constexpr int kStageBytes = 49152;
constexpr int kSmallBytes = 1024;
constexpr int kMaxBatch = 16;
constexpr int kMaxS1 = 16;  // k-splits of phase 1 (read per phase-2 operand)
constexpr int kMaxS2 = 32;  // k-splits of phase 2 (read per output)
constexpr int kMaxGrid = 256;
constexpr int kMaxOutputsPerCta = 2048;  // phase 3 keeps d of its outputs in the sums area

// Instrumentation (hfa_ffn_set_stamps): thread 0 of each CTA (the producer's lane 0 for
// kStampIssued) records %globaltimer at these points of every step.
enum {
  kStampEntry = 0,  // barriers initialised
  kStampWait,       // the previous kernel has completed
  kStampOp1,        // first phase-1 operand built
  kStampFirst,      // first stage computed (warp 0)
  kStampPh1,        // last phase-1 stage stored
  kStampOp2,        // first phase-2 operand built (phase-1 sums of its columns in)
  kStampPh2,        // last phase-2 stage stored
  kStampD,          // d of this CTA's outputs summed
  kStampNorm,       // 1/rms(d) of its rows known
  kStampExit,       // outputs written
  kStampIssued,     // producer: last stage issued
  kStampArrived = 11,  // [8]: stages 0..7 computed (warp 0: its wait and its tiles)
  kStampIssue = 19,    // [8]: producer: loads kStages..kStages+7 issued (their slot free)
  kStampSlots = 32,
};
#define FFN_STAMP(a, k)                                                        \
  do {                                                                         \
    if ((a).stamps) (a).stamps[blockIdx.x * kStampSlots + (k)] = globaltimer_ns(); \
  } while (0)

// GEMV operand bytes (nbs x NT x 512) the kernel for `nt` batch tiles holds
__host__ __device__ constexpr int op_bytes(int nt) { return nt == 1 ? 24576 : (nt == 2 ? 16384 : 49152); }

template <int NT>
struct Cfg {
  static constexpr int kCW = NT == 4 ? 8 : 16;  // consumer warps
  static constexpr int kConsumers = kCW * 32;
  static constexpr int kThreads = kConsumers + 32;  // + the producer warp
  static constexpr int kStages = NT == 4 ? 3 : 4;
  static constexpr int kOpBytes = op_bytes(NT);
  static constexpr int kRedHalf = kCW * NT * 32 * 2 * 4;  // warp sums of one stage
  static constexpr int kRedBytes = 2 * kRedHalf;
  static constexpr size_t kSmem =
      1024 + (size_t)kStages * kStageBytes + kOpBytes + kRedBytes + kSmallBytes;
  static_assert(kMaxOutputsPerCta * 4 <= kRedBytes, "phase-3 outputs in the sums area");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

// Named barriers: 1 all consumers, 2 consumers + producer (first activations in),
// 3 + j the consumer warps of row group j of a stage.
template <int NT>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(Cfg<NT>::kConsumers) : "memory");
}
__device__ __forceinline__ void group_sync(int j, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(3 + j), "r"(threads) : "memory");
}

// balanced partition of n items over P parts (n < 2^24, P <= kMaxGrid)
__device__ __forceinline__ int part_begin(int c, int n, int P) {
  return (int)((unsigned)c * (unsigned)n / (unsigned)P);
}
__device__ __forceinline__ int part_of(int t, int n, int P) {
  return (int)(((unsigned)(t + 1) * (unsigned)P - 1u) / (unsigned)n);
}

struct StageGeo {
  int s, rg0, nrg;
  size_t off;
  uint32_t bytes;
};
// ring stage k of a phase: k-split s, row groups [rg0, rg0 + nrg), its bytes in the stream
__device__ __forceinline__ StageGeo stage_geo(const FfnPhase& p, int k) {
  const int nps = (p.R + p.rgs - 1) / p.rgs;
  StageGeo g;
  g.s = k / nps;
  g.rg0 = (k - g.s * nps) * p.rgs;
  g.nrg = p.R - g.rg0 < p.rgs ? p.R - g.rg0 : p.rgs;
  g.off = ((size_t)g.s * p.R + g.rg0) * p.nbs * kQ8TileBytes;
  g.bytes = (uint32_t)(g.nrg * p.nbs * kQ8TileBytes);
  return g;
}

// x/2 (1 + tanh z) written as x / (1 + e^(-2z)), z = sqrt(2/pi) (x + 0.044715 x^3); for
// x -> -inf the exponential overflows to +inf and the quotient is -0.
__device__ __forceinline__ float gelu_tanh(float x) {
  const float z = 0.7978845608028654f * fmaf(0.044715f * x, x * x, x);
  return x / (1.f + __expf(-2.f * z));
}

// Gives up a poll: records the timeout and stops the CTA's remaining work.
__device__ __forceinline__ bool poll_expired(uint64_t t0, unsigned* err, volatile int* abort) {
  if (*abort) return true;
  if (globaltimer_ns() - t0 > kWaitLimitNs) {
    atomicOr(err, kErrWaitTimeout);
    *abort = 1;
    return true;
  }
  return false;
}

// Largest |v| of batch row b over a warp whose 32 consecutive items cover at most three
// consecutive rows (every row has at least 16 items): one warp reduction per row, one
// shared atomic per row and warp.
__device__ __forceinline__ void warp_row_max(unsigned* s_max, int b, unsigned m, int lane) {
  const int b0 = __shfl_sync(0xffffffffu, b, 0);
  const int b1 = __shfl_sync(0xffffffffu, b, 31);
#pragma unroll
  for (int d = 0; d < 3; ++d) {
    const unsigned r = __reduce_max_sync(0xffffffffu, b == b0 + d ? m : 0u);
    if (lane == 0 && b0 + d <= b1 && r) atomicMax(&s_max[b0 + d], r);
  }
}

// The operand words hold f32 values (hi word: column cc, lo word: column cc + 1); this
// pass scales each batch row by the power of two of its largest |value| and splits it
// into fp16 hi + lo.  The words of batch columns past B are left as they are: the MMA
// keeps columns apart, and the sums of those columns are never read.  s_inv gets the
// scales' inverse.  The (row, pair) items are independent: one flat loop over all of them.
template <int NT>
__device__ void finish_operand(uint32_t* op, const unsigned* s_max, float* s_inv, int B,
                               int pairs) {
  constexpr int C = Cfg<NT>::kConsumers;
  const int tid = threadIdx.x, total = B * pairs;
#pragma unroll 4
  for (int e = tid; e < total; e += C) {
    const int b = e / pairs, p = e - b * pairs;
    const float sc = exp2i(scale_exp(s_max[b]));
    const int wd = operand_word<NT>(2 * p, b);
    __half h0, l0, h1, l1;
    split_f16(__uint_as_float(op[wd]) * sc, h0, l0);
    split_f16(__uint_as_float(op[wd + 16]) * sc, h1, l1);
    op[wd] = pack_h2(h0, h1);
    op[wd + 16] = pack_h2(l0, l1);
  }
  if (tid < B) s_inv[tid] = exp2i(-scale_exp(s_max[tid]));
  consumer_sync<NT>();
}

// Phase-1 operand of k-split s: v = h (.) w_pre over the split's columns.  With `signal`,
// the consumers release the producer (barrier 2) once all their activations are in: loads
// issued behind the ring's bulk copies wait for them, so none is left for after the release.
template <int NT>
__device__ void build_op1(const FfnArgs& a, int s, uint32_t* op, unsigned* s_max, float* s_inv,
                          bool signal) {
  constexpr int C = Cfg<NT>::kConsumers;
  constexpr int L = NT == 4 ? 12 : 4;  // pairs per thread and round (the 16-row operand in one)
  const int tid = threadIdx.x, lane = tid & 31;
  const int ncols = a.p1.nbs * 32, c0 = s * ncols, pairs = ncols / 2, total = a.B * pairs;
  if (tid < kMaxBatch) s_max[tid] = 0u;
  consumer_sync<NT>();
  for (int base = 0; base < total; base += L * C) {
    float2 hv[L], wv[L];
#pragma unroll
    for (int k = 0; k < L; ++k) {  // every load of the round first
      const int e = base + k * C + tid, ee = e < total ? e : total - 1;
      const int b = ee / pairs, col = c0 + 2 * (ee - b * pairs);
      hv[k] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a.h + (size_t)b * a.H + col));
      wv[k] = __ldg(reinterpret_cast<const float2*>(a.w_pre + col));
    }
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const int e = base + k * C + tid, ee = e < total ? e : total - 1;
      const int b = ee / pairs, cc = 2 * (ee - b * pairs);
      const float v0 = hv[k].x * wv[k].x, v1 = hv[k].y * wv[k].y;
      if (e < total) {
        const int wd = operand_word<NT>(cc, b);
        op[wd] = __float_as_uint(v0);
        op[wd + 16] = __float_as_uint(v1);
      }
      warp_row_max(s_max, b, e < total ? __float_as_uint(fmaxf(fabsf(v0), fabsf(v1))) : 0u, lane);
    }
  }
  if (signal)  // the values are used: their loads have completed
    asm volatile("bar.arrive 2, %0;" ::"n"(Cfg<NT>::kThreads) : "memory");
  consumer_sync<NT>();
  finish_operand<NT>(op, s_max, s_inv, a.B, pairs);
}

// Phase-2 operand of k-split s: for each column x of the split, g and u = the phase-1
// partial sums added in k-split order, times 1/rms(h); a = gelu(g) u (written to the tap
// by the one CTA that loads the split's first stage).  Each thread polls two column pairs
// in PS k-splits at once (16-byte loads of g and u pairs), every load of a round issued
// before the first tag is checked: the rounds are L2 round trips one after another.
template <int NT>
__device__ void build_op2(const FfnArgs& a, int s, uint32_t* op, unsigned* s_max, float* s_inv,
                          const float* s_hinv, bool tap, uint32_t tag, volatile int* abort) {
  constexpr int C = Cfg<NT>::kConsumers;
  const int tid = threadIdx.x, lane = tid & 31;
  const int ncols = a.p2.nbs * 32, c0 = s * ncols, pairs = ncols / 2, total = a.B * pairs;
  constexpr int PS = NT == 4 ? 4 : 2;
  const size_t sstride = (size_t)a.B * 2 * a.I;
  if (tid < kMaxBatch) s_max[tid] = 0u;
  consumer_sync<NT>();
  for (int base = 0; base < total; base += 2 * C) {
    float g[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, u[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    const unsigned long long* src[2];
    int bb[2], cc[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = base + k * C + tid, ee = e < total ? e : total - 1;
      bb[k] = ee / pairs;
      cc[k] = 2 * (ee - bb[k] * pairs);
      src[k] = a.part1 + (size_t)bb[k] * 2 * a.I + c0 + cc[k];
    }
    for (int s0 = 0; s0 < a.p1.S; s0 += PS) {
      unsigned long long w[2][PS][4];
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        bool ready = true;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int i = 0; i < PS; ++i) {
            // entries b * 2I + c0 + cc (+ I) of a split: even indices, 16-byte aligned
            const int sx = s0 + i < a.p1.S ? s0 + i : a.p1.S - 1;
            const unsigned long long* p = src[k] + sx * sstride;
            ld_tagged2(p, w[k][i][0], w[k][i][1]);
            ld_tagged2(p + a.I, w[k][i][2], w[k][i][3]);
          }
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int i = 0; i < PS; ++i)
#pragma unroll
            for (int m = 0; m < 4; ++m) ready = ready && (uint32_t)(w[k][i][m] >> 32) == tag;
        if (ready || poll_expired(t0, a.err, abort)) break;
        __nanosleep(32);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < PS; ++i)
          if (s0 + i < a.p1.S) {
            g[k][0] += tagged_value(w[k][i][0]);
            g[k][1] += tagged_value(w[k][i][1]);
            u[k][0] += tagged_value(w[k][i][2]);
            u[k][1] += tagged_value(w[k][i][3]);
          }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = base + k * C + tid;
      const float hinv = s_hinv[bb[k]];
      const float a0 = gelu_tanh(g[k][0] * hinv) * (u[k][0] * hinv);
      const float a1 = gelu_tanh(g[k][1] * hinv) * (u[k][1] * hinv);
      if (e < total) {
        if (tap) {
          a.a_tap[(size_t)bb[k] * a.I + c0 + cc[k]] = a0;
          a.a_tap[(size_t)bb[k] * a.I + c0 + cc[k] + 1] = a1;
        }
        const int wd = operand_word<NT>(cc[k], bb[k]);
        op[wd] = __float_as_uint(a0);
        op[wd + 16] = __float_as_uint(a1);
      }
      warp_row_max(s_max, bb[k], e < total ? __float_as_uint(fmaxf(fabsf(a0), fabsf(a1))) : 0u,
                   lane);
    }
  }
  consumer_sync<NT>();
  finish_operand<NT>(op, s_max, s_inv, a.B, pairs);
}

// 1/rms(h) of every batch row: one warp per row, 16-byte loads, the warp tree.
template <int NT>
__device__ void h_inv_rms(const FfnArgs& a, float* s_hinv, int warp, int lane) {
  for (int b = warp; b < a.B; b += Cfg<NT>::kCW) {
    const uint4* row = reinterpret_cast<const uint4*>(a.h + (size_t)b * a.H);
    float ss = 0.f;
    for (int i = lane; i < a.H / 8; i += 32) {
      const uint4 u = row[i];
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(p[k]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) s_hinv[b] = rsqrtf(ss / a.H + a.eps);
  }
}

template <int NT>
__global__ void __launch_bounds__(Cfg<NT>::kThreads, 1) ffn_kernel(const __grid_constant__ FfnArgs a) {
  using K = Cfg<NT>;
  constexpr int kCW = K::kCW, kConsumers = K::kConsumers, kStages = K::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* ring = smem;
  uint32_t* op = reinterpret_cast<uint32_t*>(smem + kStages * kStageBytes);
  float* red = reinterpret_cast<float*>(smem + kStages * kStageBytes + K::kOpBytes);
  uint8_t* small = smem + kStages * kStageBytes + K::kOpBytes + K::kRedBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(small);
  uint64_t* empty = full + kStages;
  volatile int* s_abort = reinterpret_cast<volatile int*>(small + 64);
  uint32_t* s_tag = reinterpret_cast<uint32_t*>(small + 68);
  unsigned* s_max = reinterpret_cast<unsigned*>(small + 128);  // [16]
  float* s_inv = reinterpret_cast<float*>(small + 192);        // [16] operand scale undo
  float* s_hinv = reinterpret_cast<float*>(small + 256);       // [16] 1/rms(h)
  float* s_dinv = reinterpret_cast<float*>(small + 320);       // [2] 1/rms(d)
  float* wred = reinterpret_cast<float*>(small + 384);         // [16 warps][2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, nctas = gridDim.x;
  if (blockDim.x != K::kThreads) return;  // the host always launches kThreads
  const int k10 = part_begin(c, a.p1.stages, nctas), k11 = part_begin(c + 1, a.p1.stages, nctas);
  const int k20 = part_begin(c, a.p2.stages, nctas), k21 = part_begin(c + 1, a.p2.stages, nctas);
  const int n1 = k11 - k10, nld = n1 + (k21 - k20);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) FFN_STAMP(a, kStampEntry);
  // Programmatic dependent launch: the next kernel may be scheduled now; nothing is read
  // before the previous kernel has completed.
  pdl_launch_dependents();
  pdl_wait();
  if (tid == 0) {
    // the step's number: every CTA of a launch reads the counter before its own increment
    // and after every increment of the launches before it
    const unsigned long long v = ld_acquire_u64(a.ctr);
    *s_tag = (uint32_t)(v / (unsigned long long)nctas) + 1u;  // 0 marks "never written"
    red_release_add_u64(a.ctr, 1ull);
    FFN_STAMP(a, kStampWait);
  }
  __syncthreads();
  const uint32_t tag = *s_tag;

  if (warp == kCW) {
    // ================================================================ producer
    // the first operand's activations go out before the ring fill (barrier 2)
    if (n1 > 0) asm volatile("bar.sync 2, %0;" ::"n"(K::kThreads) : "memory");
    if (lane == 0) {
      int i = 0;
      for (; i < nld; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) - 1) & 1, a.err, s_abort)) {
          *s_abort = 1;
          break;
        }
        const StageGeo g = i < n1 ? stage_geo(a.p1, k10 + i) : stage_geo(a.p2, k20 + i - n1);
        mbar_arrive_expect_tx(&full[st], g.bytes);
        bulk_load(ring + st * kStageBytes, (i < n1 ? a.p1.w : a.p2.w) + g.off, g.bytes, &full[st]);
        if (i >= kStages && i - kStages < 8) FFN_STAMP(a, kStampIssue + i - kStages);
      }
      FFN_STAMP(a, kStampIssued);
      // every copy in flight lands before the CTA exits (the last use of each slot)
      for (int j = i > kStages ? i - kStages : 0; j < i; ++j)
        mbar_wait(&full[j % kStages], (j / kStages) & 1, a.err);
    }
    return;
  }

  // ================================================================== consumers
  int cur = -1;  // operand held: phase-2 k-splits are numbered from 65536
  bool have_hinv = false;
  const int nps2 = (a.p2.R + a.p2.rgs - 1) / a.p2.rgs;
  for (int i = 0; i < nld; ++i) {
    const bool ph1 = i < n1;
    const FfnPhase& P = ph1 ? a.p1 : a.p2;
    const StageGeo g = ph1 ? stage_geo(a.p1, k10 + i) : stage_geo(a.p2, k20 + i - n1);
    const int key = (ph1 ? 0 : 65536) + g.s;
    if (key != cur) {
      if (!ph1 && !have_hinv) {
        h_inv_rms<NT>(a, s_hinv, warp, lane);
        have_hinv = true;
      }
      consumer_sync<NT>();  // the previous operand is no longer read; s_hinv is visible
      if (ph1) {
        build_op1<NT>(a, g.s, op, s_max, s_inv, i == 0);
        if (tid == 0 && i == 0) FFN_STAMP(a, kStampOp1);
      } else {
        const int first = g.s * nps2;  // the split's first stage
        const bool tap = a.a_tap && first >= k20 && first < k21;
        build_op2<NT>(a, g.s, op, s_max, s_inv, s_hinv, tap, tag, s_abort);
        if (tid == 0 && i == n1) FFN_STAMP(a, kStampOp2);
      }
      cur = key;
    }
    const int st = i % kStages;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int wpr = kCW / P.rgs;  // warps per row group
    const int j = warp / wpr, qw = warp - j * wpr;
    if (mbar_wait(&full[st], (i / kStages) & 1, a.err, s_abort) && !*s_abort) {
      if (j < g.nrg) {
        const int t0 = qw * P.nbs / wpr, t1 = (qw + 1) * P.nbs / wpr;
        const uint32_t tp = smem_u32(ring + st * kStageBytes) + (uint32_t)(j * P.nbs * kQ8TileBytes);
        const uint32_t fr = smem_u32(op) + lane * 16;
        const uint32_t dl = 512 + (lane >> 2) * 4;
        int t = t0;
#pragma unroll 2
        for (; t + 1 < t1; t += 2) {
          const uint32_t pa = tp + t * kQ8TileBytes, pb = pa + kQ8TileBytes;
          q8_tile2_mma<NT>(acc, lds128(pa + lane * 16), lds32(pa + dl), fr + t * NT * 512,
                           lds128(pb + lane * 16), lds32(pb + dl), fr + (t + 1) * NT * 512);
        }
        if (t < t1) {
          const uint32_t pa = tp + t * kQ8TileBytes;
          q8_tile_mma<NT>(acc, lds128(pa + lane * 16), lds32(pa + dl), fr + t * NT * 512);
        }
      }
    } else {
      *s_abort = 1;
    }
    if (tid == 0 && i < 8) FFN_STAMP(a, kStampArrived + i);
    if (tid == 0 && i == 0) FFN_STAMP(a, kStampFirst);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the slot
    if (j < g.nrg) {
      // the row group's sums: its warps' parts through shared memory (the buffer of this
      // stage's parity: a group writes it again two of its stages later, after its barrier
      // of the stage in between, which every warp of the group passes after its reads)
      float* rb = red + (i & 1) * (K::kRedHalf / 4);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float2 v;
        v.x = acc[nt][0] + acc[nt][1];  // row g, batch 4 nt + t (hi + lo columns)
        v.y = acc[nt][2] + acc[nt][3];  // row g + 8
        reinterpret_cast<float2*>(rb)[(warp * NT + nt) * 32 + lane] = v;
      }
      group_sync(j, wpr * 32);
      // outputs (b, row) of the group spread over its warps: output e -> warp e % wpr
      const int rg = g.rg0 + j;
      for (int e = lane * wpr + qw; e < a.B * 16; e += 32 * wpr) {
        const int b = e >> 4, row = e & 15;
        const int nt = b >> 2, src_lane = (row & 7) * 4 + (b & 3), half = row >> 3;
        const float* rp = rb + ((j * wpr * NT + nt) * 32 + src_lane) * 2 + half;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w)
          if (w < wpr) v += rp[w * NT * 64];
        v *= s_inv[b];
        unsigned long long* dst =
            ph1 ? a.part1 + ((size_t)g.s * a.B + b) * (2 * (size_t)a.I) + (rg & 1) * (size_t)a.I +
                      (rg >> 1) * 16 + row
                : a.part2 + ((size_t)g.s * a.B + b) * a.H + rg * 16 + row;
        st_tagged(dst, v, tag);
      }
    }
    if (tid == 0 && i == n1 - 1) FFN_STAMP(a, kStampPh1);
    if (tid == 0 && i == nld - 1) FFN_STAMP(a, kStampPh2);
  }

  // ================================================================== phase 3
  consumer_sync<NT>();  // every stage's sums are read: the sums area holds d from here
  const int N = a.B * a.H;
  const int e0 = part_begin(c, N, nctas), e1 = part_begin(c + 1, N, nctas);
  const int b_lo = e0 < e1 ? e0 / a.H : 0;
  const int split_e = (b_lo + 1) * a.H;  // first output of the second row
  const size_t s2stride = (size_t)a.B * a.H;
  float ps0 = 0.f, ps1 = 0.f;
  for (int e = e0 + tid; e < e1; e += kConsumers) {
    float d = 0.f;
    // the k-splits' entries polled P3 at a time (more with four batch tiles, whose plans
    // have more splits and whose threads have the registers)
    constexpr int P3 = NT == 4 ? 24 : 8;
    for (int s0 = 0; s0 < a.p2.S; s0 += P3) {
      unsigned long long w[P3];
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        bool ready = true;
#pragma unroll
        for (int k = 0; k < P3; ++k) {
          const int sx = s0 + k < a.p2.S ? s0 + k : a.p2.S - 1;
          w[k] = ld_tagged(a.part2 + sx * s2stride + e);
        }
#pragma unroll
        for (int k = 0; k < P3; ++k) ready = ready && (uint32_t)(w[k] >> 32) == tag;
        if (ready || poll_expired(t0, a.err, s_abort)) break;
        __nanosleep(32);
      }
#pragma unroll
      for (int k = 0; k < P3; ++k)
        if (s0 + k < a.p2.S) d += tagged_value(w[k]);
    }
    red[e - e0] = d;
    if (e < split_e) ps0 = fmaf(d, d, ps0);
    else ps1 = fmaf(d, d, ps1);
  }
  {
    const float t0 = warp_sum(ps0), t1 = warp_sum(ps1);
    if (lane == 0) {
      wred[warp * 2] = t0;
      wred[warp * 2 + 1] = t1;
    }
  }
  consumer_sync<NT>();
  if (tid == 0) FFN_STAMP(a, kStampD);
  if (tid < 2 && e0 < e1 && b_lo + tid <= (e1 - 1) / a.H) {
    float t = 0.f;
    for (int w = 0; w < kCW; ++w) t += wred[w * 2 + tid];
    st_tagged(a.post_part + 2 * c + tid, t, tag);
  }
  // the parts of every CTA that shares a row with this one, added in CTA order
  float* gath = reinterpret_cast<float*>(op);  // the operand is no longer needed
  if (e0 < e1) {
    for (int r = 0; r < 2 && b_lo + r <= (e1 - 1) / a.H; ++r) {
      const int b = b_lo + r;
      const int cf = part_of(b * a.H, N, nctas), cl = part_of((b + 1) * a.H - 1, N, nctas);
      for (int cc = cf + tid; cc <= cl; cc += kConsumers) {
        const int beg = part_begin(cc, N, nctas);
        float v = 0.f;  // a CTA without outputs adds nothing
        if (beg < part_begin(cc + 1, N, nctas)) {
          const int slot = b - beg / a.H;
          const uint64_t t0 = globaltimer_ns();
          unsigned long long w;
          for (;;) {
            w = ld_tagged(a.post_part + 2 * cc + slot);
            if ((uint32_t)(w >> 32) == tag || poll_expired(t0, a.err, s_abort)) break;
            __nanosleep(32);
          }
          v = tagged_value(w);
        }
        gath[cc - cf] = v;
      }
      consumer_sync<NT>();
      if (tid == 0) {
        float t = 0.f;
        for (int cc = cf; cc <= cl; ++cc) t += gath[cc - cf];
        s_dinv[r] = rsqrtf(t / a.H + a.eps);
      }
      consumer_sync<NT>();
    }
  }
  if (tid == 0) FFN_STAMP(a, kStampNorm);
  for (int e = e0 + tid; e < e1; e += kConsumers) {
    const int second = e >= split_e ? 1 : 0;
    const int i = e - (b_lo + second) * a.H;
    const float hv = __bfloat162float(a.h[e]);
    const float sc = a.scalar[a.scalar_len == 1 ? 0 : i];
    const float r = (hv + red[e - e0] * a.w_post[i] * s_dinv[second]) * sc;
    a.out[e] = __float2bfloat16_rn(r);
    if (a.out_f32) a.out_f32[e] = r;
  }
  if (tid == 0) FFN_STAMP(a, kStampExit);
}

}  // namespace ffn

int ffn_max_outputs_per_cta() { return ffn::kMaxOutputsPerCta; }

// largest k-split (blocks) whose operand every kernel up to nt_max batch tiles holds
static int max_blocks_per_split(int nt_max) {
  int m = 1 << 30;
  for (int nt = 1; nt <= nt_max; nt *= 2) {
    const int v = ffn::op_bytes(nt) / (nt * 512);
    m = v < m ? v : m;
  }
  return m;
}

bool ffn_plan_fits(const FfnPhase& p, int nt) {
  return p.nbs * nt * 512 <= ffn::op_bytes(nt) &&
         (long long)p.rgs * p.nbs * kQ8TileBytes <= ffn::kStageBytes;
}

bool plan_ffn_phase(FfnPhase* p, int R, int nb, bool pairs, int nt_max, int grid) {
  // cost: the bytes of the busiest CTA, plus a charge per stage (its barrier and
  // reduction) and per k-split (phase 1's splits are all read by every phase-2 operand)
  long long best = -1;
  const int maxS = pairs ? ffn::kMaxS1 : ffn::kMaxS2;
  for (int S = 1; S <= nb && S <= maxS; ++S) {
    if (nb % S) continue;
    const int nbs = nb / S;
    if (nbs > max_blocks_per_split(nt_max)) continue;
    for (int rgs = 1; rgs <= 8; rgs *= 2) {
      if (pairs && (rgs & 1)) continue;
      const long long sb = (long long)rgs * nbs * kQ8TileBytes;
      if (sb > ffn::kStageBytes) continue;
      const long long stages = (long long)S * ((R + rgs - 1) / rgs);
      const long long per = (stages + grid - 1) / grid;
      const long long cost = per * (sb + 4096) + S * (pairs ? 4096 : 512);
      if (best < 0 || cost < best) {
        best = cost;
        p->R = R;
        p->nbs = nbs;
        p->S = S;
        p->rgs = rgs;
        p->stages = (int)stages;
      }
    }
  }
  return best >= 0;
}

namespace {
template <int NT>
struct FfnOptIn {
  static unsigned long long mask;
};
template <int NT>
unsigned long long FfnOptIn<NT>::mask = 0ull;

template <int NT>
cudaError_t launch_ffn_t(const FfnArgs& a, int grid, cudaStream_t s) {
  using K = ffn::Cfg<NT>;
  auto kern = ffn::ffn_kernel<NT>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  unsigned long long* opted_in = &FfnOptIn<NT>::mask;
  if (!bit || !(__atomic_load_n(opted_in, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K::kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(opted_in, bit, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(K::kThreads);
  cfg.dynamicSmemBytes = K::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a);
}
}  // namespace

cudaError_t launch_ffn(const FfnArgs& a, int grid, cudaStream_t s) {
  if (a.B <= 4) return launch_ffn_t<1>(a, grid, s);
  if (a.B <= 8) return launch_ffn_t<2>(a, grid, s);
  return launch_ffn_t<4>(a, grid, s);
}

}  // namespace hfa

// ====================================================================== C ABI
using namespace hfa;

struct hfa_ffn {
  hfa_ffn_desc d;
  int device = 0;
  int grid = 0;
  int nt_max = 1;
  FfnPhase p1{}, p2{};
  uint8_t* w1 = nullptr;  // [Wg; Wu] tiles, row groups interleaved
  uint8_t* w2 = nullptr;  // Wd tiles
  float* w_pre = nullptr;
  float* w_post = nullptr;
  float* scalar = nullptr;
  unsigned long long* part1 = nullptr;
  unsigned long long* part2 = nullptr;
  unsigned long long* post_part = nullptr;
  unsigned long long* ctr = nullptr;
  unsigned* err = nullptr;
  unsigned long long* stamps = nullptr;
  char msg[256] = {0};
};

static thread_local char g_ffn_error[256];

static hfa_status ffn_fail(hfa_ffn* F, hfa_status st, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (F) snprintf(F->msg, sizeof F->msg, "%s", buf);
  snprintf(g_ffn_error, sizeof g_ffn_error, "%s", buf);
  set_thread_error(g_ffn_error);
  return st;
}

static void ffn_free(hfa_ffn* F) {
  if (!F) return;
  cudaFree(F->w1);
  cudaFree(F->w2);
  cudaFree(F->w_pre);
  cudaFree(F->w_post);
  cudaFree(F->scalar);
  cudaFree(F->part1);
  cudaFree(F->part2);
  cudaFree(F->post_part);
  cudaFree(F->ctr);
  cudaFree(F->err);
  delete F;
}

static bool is_sm103(int dev) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
  return major == 10 && minor == 3;
}

extern "C" hfa_status hfa_ffn_create(const hfa_ffn_desc* d, const void* w_gate, const void* w_up,
                                     const void* w_down, const float* w_pre, const float* w_post,
                                     const float* scalar, void* stream, hfa_ffn** out) {
  if (!out) return ffn_fail(nullptr, HFA_EINVAL, "out is NULL");
  *out = nullptr;
  if (!d) return ffn_fail(nullptr, HFA_EINVAL, "desc is NULL");
  const int H = d->hidden, I = d->intermediate;
  if (H <= 0 || I <= 0 || H % 32 || I % 32)
    return ffn_fail(nullptr, HFA_EINVAL, "hidden=%d, intermediate=%d: positive multiples of 32 "
                    "(whole Q8_0 blocks) required", H, I);
  if (d->scalar_len != 1 && d->scalar_len != H)
    return ffn_fail(nullptr, HFA_EINVAL, "scalar_len=%d (1 or hidden)", d->scalar_len);
  if (d->max_batch < 1 || d->max_batch > ffn::kMaxBatch)
    return ffn_fail(nullptr, HFA_EUNSUPPORTED, "max_batch=%d (1..%d)", d->max_batch, ffn::kMaxBatch);
  if (!(d->eps >= 0.f)) return ffn_fail(nullptr, HFA_EINVAL, "eps must be >= 0");
  if (!w_gate || !w_up || !w_down || !w_pre || !w_post || !scalar)
    return ffn_fail(nullptr, HFA_EINVAL, "a weight pointer is NULL");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ffn_fail(nullptr, HFA_EDEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  if (!is_sm103(dev)) return ffn_fail(nullptr, HFA_EDEVICE, "device %d is not sm_103", dev);
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms < ffn::kMaxGrid ? sms : ffn::kMaxGrid;
  if (grid <= d->max_batch)
    return ffn_fail(nullptr, HFA_EUNSUPPORTED, "%d SMs for batches of %d", grid, d->max_batch);
  if ((long long)d->max_batch * H > (long long)grid * ffn_max_outputs_per_cta())
    return ffn_fail(nullptr, HFA_EUNSUPPORTED, "max_batch * hidden = %lld outputs over %d CTAs",
                    (long long)d->max_batch * H, grid);
  if ((long long)d->max_batch * H >= (1ll << 24) || 2ll * I / 16 * (H / 32) >= (1ll << 24))
    return ffn_fail(nullptr, HFA_EUNSUPPORTED, "shape too large");
  hfa_ffn* F = new hfa_ffn();
  F->d = *d;
  F->device = dev;
  F->grid = grid;
  F->nt_max = d->max_batch <= 4 ? 1 : (d->max_batch <= 8 ? 2 : 4);
  if (!plan_ffn_phase(&F->p1, 2 * I / 16, H / 32, true, F->nt_max, grid) ||
      !plan_ffn_phase(&F->p2, H / 16, I / 32, false, F->nt_max, grid)) {
    ffn_free(F);
    return ffn_fail(nullptr, HFA_EUNSUPPORTED, "no GEMV plan for hidden=%d, intermediate=%d, "
                    "max_batch=%d", H, I, d->max_batch);
  }
  cudaStream_t s = (cudaStream_t)stream;
  const size_t b1 = (size_t)2 * I / 16 * (H / 32) * kQ8TileBytes;
  const size_t b2 = (size_t)H / 16 * (I / 32) * kQ8TileBytes;
  const int B = d->max_batch;
  e = cudaMalloc(&F->w1, b1);
  if (e == cudaSuccess) e = cudaMalloc(&F->w2, b2);
  if (e == cudaSuccess) e = cudaMalloc(&F->w_pre, H * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&F->w_post, H * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&F->scalar, d->scalar_len * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&F->part1, (size_t)F->p1.S * B * 2 * I * 8);
  if (e == cudaSuccess) e = cudaMalloc(&F->part2, (size_t)F->p2.S * B * H * 8);
  if (e == cudaSuccess) e = cudaMalloc(&F->post_part, (size_t)grid * 2 * 8);
  if (e == cudaSuccess) e = cudaMalloc(&F->ctr, 8);
  if (e == cudaSuccess) e = cudaMalloc(&F->err, 4);
  if (e != cudaSuccess) {
    ffn_free(F);
    return ffn_fail(nullptr, HFA_ENOMEM, "device allocation: %s", cudaGetErrorString(e));
  }
  F->p1.w = F->w1;
  F->p2.w = F->w2;
  e = launch_repack_q8_0_split((const uint8_t*)w_gate, I, H, F->w1, 0, F->p1.R, F->p1.nbs, s, 2);
  if (e == cudaSuccess)
    e = launch_repack_q8_0_split((const uint8_t*)w_up, I, H, F->w1, 1, F->p1.R, F->p1.nbs, s, 2);
  if (e == cudaSuccess)
    e = launch_repack_q8_0_split((const uint8_t*)w_down, H, I, F->w2, 0, F->p2.R, F->p2.nbs, s, 1);
  if (e == cudaSuccess) e = cudaMemcpyAsync(F->w_pre, w_pre, H * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(F->w_post, w_post, H * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(F->scalar, scalar, d->scalar_len * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->part1, 0, (size_t)F->p1.S * B * 2 * I * 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->part2, 0, (size_t)F->p2.S * B * H * 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->post_part, 0, (size_t)grid * 2 * 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->ctr, 0, 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->err, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    ffn_free(F);
    return ffn_fail(nullptr, HFA_ECUDA, "create: %s", cudaGetErrorString(e));
  }
  *out = F;
  return HFA_OK;
}

extern "C" hfa_status hfa_ffn_destroy(hfa_ffn* F) {
  if (!F) return HFA_EINVAL;
  ffn_free(F);
  return HFA_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

extern "C" hfa_status hfa_ffn_step(hfa_ffn* F, void* stream, const void* h, int batch, void* out,
                                   float* out_f32, float* a_tap) {
  if (!F) return ffn_fail(nullptr, HFA_EINVAL, "ffn is NULL");
  if (batch < 1 || batch > F->d.max_batch)
    return ffn_fail(F, HFA_EINVAL, "batch=%d outside 1..max_batch=%d", batch, F->d.max_batch);
  if (!h || !out) return ffn_fail(F, HFA_EINVAL, "h or out is NULL");
  if (!aligned16(h) || !aligned16(out) || (out_f32 && !aligned16(out_f32)) ||
      (a_tap && !aligned16(a_tap)))
    return ffn_fail(F, HFA_EINVAL, "device buffers must be 16-byte aligned");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != F->device)
    return ffn_fail(F, HFA_EDEVICE, "current device is not the one the FFN was created on");
  FfnArgs a{};
  a.p1 = F->p1;
  a.p2 = F->p2;
  a.h = (const __nv_bfloat16*)h;
  a.w_pre = F->w_pre;
  a.w_post = F->w_post;
  a.scalar = F->scalar;
  a.scalar_len = F->d.scalar_len;
  a.part1 = F->part1;
  a.part2 = F->part2;
  a.post_part = F->post_part;
  a.ctr = F->ctr;
  a.err = F->err;
  a.out = (__nv_bfloat16*)out;
  a.out_f32 = out_f32;
  a.a_tap = a_tap;
  a.stamps = F->stamps;
  a.B = batch;
  a.H = F->d.hidden;
  a.I = F->d.intermediate;
  a.eps = F->d.eps;
  const int nt = batch <= 4 ? 1 : (batch <= 8 ? 2 : 4);
  if (!ffn_plan_fits(F->p1, nt) || !ffn_plan_fits(F->p2, nt))
    return ffn_fail(F, HFA_EUNSUPPORTED, "the plan does not fit the kernel for batch %d", batch);
  const cudaError_t e = launch_ffn(a, F->grid, (cudaStream_t)stream);
  if (e != cudaSuccess) return ffn_fail(F, HFA_ECUDA, "FFN launch: %s", cudaGetErrorString(e));
  return HFA_OK;
}

extern "C" hfa_status hfa_ffn_set_stamps(hfa_ffn* F, unsigned long long* stamps) {
  if (!F) return ffn_fail(nullptr, HFA_EINVAL, "ffn is NULL");
  F->stamps = stamps;
  return HFA_OK;
}

extern "C" int hfa_ffn_stamp_rows(const hfa_ffn* F) { return F ? F->grid : 0; }

extern "C" hfa_status hfa_ffn_check_status(hfa_ffn* F, void* stream) {
  if (!F) return ffn_fail(nullptr, HFA_EINVAL, "ffn is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  unsigned v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, F->err, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return ffn_fail(F, HFA_ECUDA, "read status: %s", cudaGetErrorString(e));
  if (v == 0) return HFA_OK;
  // a step that gave up leaves the step count and the partial sums behind: all restart
  const int B = F->d.max_batch, H = F->d.hidden, I = F->d.intermediate;
  e = cudaMemsetAsync(F->err, 0, 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->ctr, 0, 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->part1, 0, (size_t)F->p1.S * B * 2 * I * 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->part2, 0, (size_t)F->p2.S * B * H * 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(F->post_part, 0, (size_t)F->grid * 2 * 8, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return ffn_fail(F, HFA_ECUDA, "reset: %s", cudaGetErrorString(e));
  return ffn_fail(F, HFA_EDEVICE, "device status 0x%x:%s", v,
                  (v & kErrWaitTimeout) ? " a bounded wait gave up" : "");
}

extern "C" const char* hfa_ffn_last_error(const hfa_ffn* F) { return F ? F->msg : g_ffn_error; }

extern "C" int hfa_ffn_plan_info(const hfa_ffn* F, int n, int* v) {
  if (!F || !v) return -1;
  const int vals[] = {F->grid, F->nt_max, F->p1.S, F->p1.nbs, F->p1.rgs, F->p1.stages,
                      F->p2.S, F->p2.nbs, F->p2.rgs, F->p2.stages};
  const int m = (int)(sizeof vals / sizeof vals[0]);
  for (int i = 0; i < n && i < m; ++i) v[i] = vals[i];
  return m;
}
