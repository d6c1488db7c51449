// k_step.cuh -- the decode step of one attention layer as one persistent kernel.
//
// One CTA per SM, launched cooperatively so that every CTA is resident and the CTAs may
// wait for one another at two grid barriers.  Three phases:
//   A  QKV projection of x (.) w_in with the Q8_0 matrix [Wq; Wk; Wv]
//      (gemma4/gpu_full_attn.rs, encode_one_layer: "Pre-attention norm", "QKV
//      projections").  The input norm's 1/rms(x) is a per-row factor, so it is applied
//      after the projection (phase B), and the projection never waits for it.
//   B  per (sequence, KV head) unit: q_norm / k_norm, NeoX RoPE and the bf16 KV append
//      ("Fused per-head RMS norm + RoPE on Q and K", "GPU V norm", dense KV copy), then
//      the GQA flash-decode over the unit's visible keys ("Dense flash_attn_vec",
//      FlashAttnVecParams; softcap of dflash/forward.rs).  The key tiles of all units are
//      dealt out evenly over the CTAs; every CTA writes one (m, l, O) record per unit it
//      touched.
//   C  o_proj and the residual ("O-proj"; dflash/forward.rs residual add).  The records
//      of phase B are combined with log-sum-exp weights while the GEMV operand is built,
//      so the split-K attention needs no combine pass of its own.
// Data movement: one producer warp streams everything the CTA reads in bulk -- the weight
// tiles of phase A, the K/V tiles of phase B, the weight tiles of phase C -- through one
// ring of shared-memory stages, in that order and as far ahead as the ring allows.  No
// load waits for a result of the step except the K/V tile holding the slot appended in
// this step: the producer issues it after the append has been written.
//
// Every wait (mbarrier, grid barrier) is bounded in wall time; a CTA that gives up sets
// an error bit, stops loading and computing, still passes every later barrier so that
// the others are not held, and drains its copies in flight before it exits.
#pragma once
#include "hfa_common.cuh"
#include "hfa_finish.cuh"
#include "hfa_gemv.cuh"
#include "hfa_internal.h"

namespace hfa {
namespace step {

constexpr int kCW = 8;                    // consumer warps
constexpr int kConsumers = kCW * 32;
constexpr int kThreads = kConsumers + 32; // + the producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 65536;
constexpr int kUnionBytes = 33792;        // GEMV operand / query rows / merge area
constexpr int kSmallBytes = 1024;         // barriers, flags, per-row values
constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kUnionBytes + kSmallBytes;
constexpr int kKeysPerWarp = 16;
constexpr int kMaxBatch = 16;
// K/V tiles prefetched into L2 during phase A, and the most K/V tiles brought into the ring
// before the queries of the first unit are formed (0: no limit).  With one batch tile the
// head epilogue's loads of the QKV partial sums would otherwise queue behind the ring fill;
// with more batch tiles phase A is long enough that the fill is over before they are issued.
template <int NT> struct Fill {
  static constexpr int kEarlyTiles = NT == 1 ? 3 : 2;
  static constexpr int kBeforeQueries = NT == 1 ? 2 : 0;
};
constexpr uint32_t kSuccChunk = 16384;    // next layer's weights: L2 prefetch chunk ...
constexpr unsigned kSuccPauseNs = 400;    // ... and the pause after each

// Instrumentation (hfa_set_step_stamps): with a stamp buffer set, thread 0 of each CTA and
// the producer's lane 0 record %globaltimer at these points of every step.
enum {
  kStampEntry = 0,   // CTA start, barriers initialised
  kStampOperand,     // phase A operand built (activations loaded)
  kStampGemvA,       // phase A GEMV done
  kStampAttn,        // first key tile's queries ready
  kStampStream,      // last key tile consumed
  kStampRecords,     // attention records written
  kStampBarrier,     // grid barrier passed
  kStampMerge,       // o_proj operand merged
  kStampGemvC,       // o_proj GEMV done
  kStampExit,        // residual written
  kStampProdA,       // producer: first QKV copy issued
  kStampProdKV,      // producer: last key tile issued
  kStampProdC,       // producer: o_proj copies issued
  kStampWait,        // the wait for the previous kernel on the stream returned
  kStampSlots = 16
};
#define HFA_STAMP(a, k) \
  do { if ((a).stamps) (a).stamps[blockIdx.x * kStampSlots + (k)] = globaltimer_ns(); } while (0)

// per batch row: position, visible slots [lo, hi], key tiles, tile of the new slot, slot
enum { kGeoP = 0, kGeoLo, kGeoHi, kGeoNt, kGeoTn, kGeoSlot, kGeoPre, kGeoInts = 8 };

// Attention tile shape: NC key groups of 16 keys per tile; with HD = 256 the 8 consumer
// warps pair up on a key group (both form S = Q K^T, each accumulates half of O's dims),
// which halves the O registers of a warp; with HD = 512 four warps share a key group (a
// 32-key tile of K and V is then one 64 KB stage).
template <int HD>
struct Attn {
  static constexpr int NC = HD >= 512 ? 2 : (HD >= 256 ? 4 : 8);  // key groups of a tile
  static constexpr int DSPLIT = kCW / NC;             // warps per key group
  static constexpr int T = NC * kKeysPerWarp;         // keys per tile
  static constexpr int BOXES = HD / 64;               // 128-byte TMA boxes per row
  static constexpr int TILE_BYTES = T * HD * 2;       // one of K, V
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int KS = HD / 16;
  static constexpr int NTO = HD / 8;                  // n8 tiles of O
  static constexpr int NTW = NTO / DSPLIT;            // n8 tiles of O per warp
  static constexpr int RS = HD + 4;                   // record: O[HD], m, l, pad
  static constexpr int QS_OFF = KS * 32 * 16 > 8192 ? KS * 32 * 16 : 8192;  // query rows (f32)
  static_assert(STAGE_BYTES <= kStageBytes, "a K/V tile must fit a stage");
  static_assert(NC * DSPLIT == kCW, "every consumer warp takes part");
  static_assert(NC * 8 * RS * 4 <= kUnionBytes, "merge area must fit the union");
  static_assert(KS * 32 * 16 <= QS_OFF && QS_OFF + 8 * HD * 4 <= kUnionBytes, "query rows");
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Balanced partition of n items over P parts: part c owns [begin(c), begin(c + 1)).
// 32-bit products: the host keeps every partitioned count below 2^24 (key tiles, B x H
// outputs, row groups) and the grid at most 256 CTAs.
__device__ __forceinline__ int part_begin(int c, int n, int P) {
  return (int)((unsigned)c * (unsigned)n / (unsigned)P);
}
// the part that owns item t (0 <= t < n): the largest c with begin(c) <= t
__device__ __forceinline__ int part_of(int t, int n, int P) {
  return (int)(((unsigned)(t + 1) * (unsigned)P - 1u) / (unsigned)n);
}

// Rows of a split-K GEMV owned by CTA c: the CTAs are dealt out over the k-splits, and
// the CTAs of one split share its row groups evenly.
struct Slice {
  int s, r0, r1;
  bool first;  // first CTA of its split
};
__device__ __forceinline__ Slice gemv_slice(const StepGemv& g, int c, int nctas) {
  Slice sl;
  sl.s = part_of(c, nctas, g.S);
  const int c0 = part_begin(sl.s, nctas, g.S), c1 = part_begin(sl.s + 1, nctas, g.S);
  sl.r0 = part_begin(c - c0, g.R, c1 - c0);
  sl.r1 = part_begin(c - c0 + 1, g.R, c1 - c0);
  sl.first = c == c0;
  return sl;
}

// Units (sequence b, KV head kvh) in order u = b * nkv + kvh; unit u holds nt_b key tiles.
// Calls f(b, kvh, lt0, lt1) for the part [lt0, lt1) of each unit inside the global tile
// range [t0, t1).
template <typename F>
__device__ __forceinline__ void for_each_segment(const int* geo, int B, int nkv, int t0, int t1,
                                                 F&& f) {
  int base = 0;
  for (int b = 0; b < B && base < t1; ++b) {
    const int nt = geo[b * kGeoInts + kGeoNt];
    const int span = nt * nkv;
    if (nt > 0 && base + span > t0) {
      const int kv0 = t0 > base ? (t0 - base) / nt : 0;
      for (int kvh = kv0; kvh < nkv; ++kvh) {
        const int ub = base + kvh * nt;
        if (ub >= t1) break;
        const int lt0 = t0 > ub ? t0 - ub : 0;
        const int lt1 = (t1 < ub + nt ? t1 : ub + nt) - ub;
        if (lt1 > lt0) f(b, kvh, lt0, lt1);
      }
    }
    base += span;
  }
}
// i-th tile of a segment in load order: the tile holding the new slot (tn, if inside
// [lt0, lt1)) goes last, so that its late load does not hold up the others.
__device__ __forceinline__ int seg_tile(int i, int lt0, int lt1, int tn) {
  if (tn < lt0 || tn >= lt1) return lt0 + i;
  if (i < tn - lt0) return lt0 + i;
  if (i < lt1 - lt0 - 1) return lt0 + i + 1;
  return tn;
}

// Grid barrier of the consumer warps (the producer runs ahead and never joins), once a
// step, before the attention records are merged.  The arrival counter only grows: the
// barrier of a step completes when it reaches base + grid, base = grid * (steps before
// this one), which every CTA reads off the counter at its start (the count is then inside
// [base, base + grid)); the same number tags the step's partial sums, which the readers
// poll instead of waiting at barriers of their own.
// Arrival is one release reduction (no round trip); a CTA that has given up arrives
// without waiting, so the count stays exact.
// Split in two so that a CTA can do work of its own between its arrival and the wait.
__device__ __forceinline__ void grid_arrive(unsigned long long* gbar) {
  consumer_sync();
  if (threadIdx.x == 0) red_release_add_u64(gbar, 1ull);
}
__device__ __forceinline__ void grid_wait(const unsigned long long* gbar, unsigned long long target,
                                          unsigned* err, volatile int* abort) {
  if (threadIdx.x == 0 && !*abort) {
    const uint64_t t0 = globaltimer_ns();
    while ((long long)(ld_acquire_u64(gbar) - target) < 0) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, kErrWaitTimeout);
        *abort = 1;
        break;
      }
    }
  }
  consumer_sync();
}

// ------------------------------------------------------------------ GEMV pieces
// Phase A operand: v = x (.) w_in over the columns of k-split s, for every batch row,
// scaled per row by a power of two (exact; undone in the flush) and split into fp16
// hi + lo.
template <int NT>
__device__ void build_x_operand(const StepArgs& a, int s, uint32_t* xw, unsigned* s_max,
                                float* s_inv, unsigned long long arrivals0,
                                unsigned long long* s_gbase, uint32_t* s_tag) {
  const int tid = threadIdx.x;
  const int nbs = a.qkv.nbs;
  const int groups = nbs * 4;  // 8-column groups per batch row
  const int total = NT * 4 * groups;
  // every load first (x rows and w_in of all NT groups of this thread), then the math
  uint4 raw[NT];
  float4 w0[NT], w1[NT];
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    const int e = tid + k * kConsumers;
    const int b = e / groups, gi = e - b * groups;
    const bool live = e < total && b < a.B;
    // addresses stay in range for the lanes without a live group
    const int bx = live ? b : 0;
    const int col = s * nbs * 32 + (live ? gi : 0) * 8;
    raw[k] = *reinterpret_cast<const uint4*>(a.x + (size_t)bx * a.H + col);
    w0[k] = __ldg(reinterpret_cast<const float4*>(a.w_in + col));
    w1[k] = __ldg(reinterpret_cast<const float4*>(a.w_in + col + 4));
  }
  float v[NT][8];
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    const int e = tid + k * kConsumers;
    const int b = e / groups;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[k][i] = 0.f;
    if (e < total && b < a.B) {
      const float wv[8] = {w0[k].x, w0[k].y, w0[k].z, w0[k].w, w1[k].x, w1[k].y, w1[k].z, w1[k].w};
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[k][2 * i] = f.x * wv[2 * i];
        v[k][2 * i + 1] = f.y * wv[2 * i + 1];
        mx = fmaxf(mx, fmaxf(fabsf(v[k][2 * i]), fabsf(v[k][2 * i + 1])));
      }
      atomicMax(&s_max[b], __float_as_uint(mx));
    }
  }
  // the activations are in registers: the producer may start the weight stream
  asm volatile("bar.arrive 3, %0;" ::"n"(kThreads) : "memory");
  if (tid == 0) {
    // this step's number: one grid barrier a step, counted since the layer was created
    *s_gbase = arrivals0 / gridDim.x * gridDim.x;     // used by thread 0 only
    *s_tag = (uint32_t)(arrivals0 / gridDim.x) + 1u;  // 0 marks "never written"
  }
  consumer_sync();
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    const int e = tid + k * kConsumers;
    if (e < total) {
      const int b = e / groups, gi = e - b * groups;
      const float sc = b < a.B ? exp2i(scale_exp(s_max[b])) : 1.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        __half h0, l0, h1, l1;
        split_f16(v[k][2 * t] * sc, h0, l0);
        split_f16(v[k][2 * t + 1] * sc, h1, l1);
        const int w = operand_word<NT>(gi * 8 + 2 * t, b);
        xw[w] = pack_h2(h0, h1);
        xw[w + 16] = pack_h2(l0, l1);
      }
    }
  }
  if (tid < a.B) s_inv[tid] = exp2i(-scale_exp(s_max[tid]));
  consumer_sync();
}

// sum(x^2) of one input row over its H columns, by one warp in a fixed order: 16-byte
// loads strided over the lanes (16 in flight per lane), then the warp tree.
__device__ __forceinline__ float row_sumsq(const __nv_bfloat16* x, int H, int lane) {
  const uint4* xr = reinterpret_cast<const uint4*>(x);
  const int n = H / 8;
  float acc = 0.f;
  for (int i0 = 0; i0 < n; i0 += 32 * 16) {
    uint4 u[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int i = i0 + k * 32 + lane;
      u[k] = xr[i < n ? i : n - 1];  // in range; lanes past the row add nothing
      if (i >= n) u[k] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        acc = fmaf(f.x, f.x, acc);
        acc = fmaf(f.y, f.y, acc);
      }
    }
  }
  return warp_sum(acc);
}

// Residual epilogue: CTA c finishes its share [i0, i1) of the B x H outputs,
// out = bf16(x + sum over the o_proj k-splits), the splits added in order 0, 1, ..., S - 1.
// A round covers kPer * per outputs (per = 256 / S): thread (k, sp) loads split sp of
// outputs k, k + per, ... (all in flight together; again, after a short pause, until every
// tag is this step's) into shared memory, then one thread per output adds its S partial
// sums.  No grid barrier: each partial sum carries its step tag.
static __device__ void finish_outputs(const StepArgs& a, int c, int nctas, float* red,
                                      uint32_t tag, volatile int* abort) {
  constexpr int kPer = 8;
  const int S = a.o.S;  // <= grid <= 256
  const int n = a.B * a.H;
  const int i0 = part_begin(c, n, nctas), i1 = part_begin(c + 1, n, nctas);
  const size_t split_stride = (size_t)a.B * a.H;
  const int tid = threadIdx.x;
  const int per = kConsumers / S, k = tid / S, sp = tid - k * S;
  // outputs of a round: at most 2 per thread, so that the residual inputs of a thread's
  // outputs (tid, tid + 256) are loaded ahead of the wait
  const int nu = kPer < 2 * kConsumers / per ? kPer : 2 * kConsumers / per;
  const int round = nu * per;
  const unsigned long long* ys = a.y_part + sp * split_stride;
#pragma unroll 1
  for (int base = i0; base < i1; base += round) {
    float xo[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = base + tid + j * kConsumers;
      xo[j] = __bfloat162float(a.x[i < i1 ? i : i1 - 1]);
    }
    if (k < per) {
      unsigned long long w[kPer];
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        bool ready = true;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int i = u < nu ? base + u * per + k : i1;
          w[u] = ld_tagged(ys + (i < i1 ? i : i1 - 1));
          ready = ready && (uint32_t)(w[u] >> 32) == tag;
        }
        if (ready) break;
        if (*abort || globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.err, kErrWaitTimeout);
          *abort = 1;
          break;
        }
        __nanosleep(64);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u)
        if (u < nu) red[(u * per + k) * S + sp] = tagged_value(w[u]);
    }
    consumer_sync();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int o = tid + j * kConsumers;
      if (o < round && base + o < i1) {
        const int i = base + o;
        float y = 0.f;
#pragma unroll 1
        for (int t = 0; t < S; ++t) y += red[o * S + t];
        const float r = xo[j] + y;
        a.out[i] = __float2bfloat16_rn(r);
        if (a.out_tap) a.out_tap[i] = r;
      }
    }
    consumer_sync();
  }
}

// Post-attention RMSNorm variant of the residual epilogue: out = x + y * w_post * r_b,
// r_b = 1 / sqrt(mean over the row b of y^2 + eps).  A CTA's share [i0, i1) of the B x H
// outputs spans at most two batch rows (share <= H).  The CTA sums its splits into y (kept
// in `ybuf`, shared memory), publishes sum(y^2) of its part of each row (tagged, slot 0 for
// its first row, 1 for the second), then adds up, in CTA order, the parts of the CTAs that
// share each of its rows, and writes its outputs.
static __device__ __forceinline__ void finish_outputs_post(const StepArgs& a, int c, int nctas,
                                                        float* red, float* ybuf, uint32_t tag,
                                                        volatile int* abort) {
  const int S = a.o.S;
  const int n = a.B * a.H;
  const int i0 = part_begin(c, n, nctas), i1 = part_begin(c + 1, n, nctas);
  const size_t split_stride = (size_t)a.B * a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = kConsumers / S, k = tid / S, sp = tid - k * S;
  const int round = per;  // one output per (k, all splits) per round
  const unsigned long long* ys = a.y_part + sp * split_stride;
  float* wred = red + kConsumers * 8;  // [8 warps][2]
  float* s_inv = wred + 16;            // [2]
  const int b_lo = i0 < i1 ? i0 / a.H : 0;
  float ps0 = 0.f, ps1 = 0.f;  // this thread's part of sum(y^2) of rows b_lo, b_lo + 1
  const int split_i = (b_lo + 1) * a.H;  // first output of the second row
#pragma unroll 1
  for (int base = i0; base < i1; base += round) {
    if (k < per) {
      const int i = base + k;
      const uint64_t t0 = globaltimer_ns();
      unsigned long long w;
      for (;;) {
        w = ld_tagged(ys + (i < i1 ? i : i1 - 1));
        if ((uint32_t)(w >> 32) == tag) break;
        if (*abort || globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.err, kErrWaitTimeout);
          *abort = 1;
          break;
        }
        __nanosleep(64);
      }
      red[k * S + sp] = tagged_value(w);
    }
    consumer_sync();
    if (tid < round && base + tid < i1) {
      const int i = base + tid;
      float y = 0.f;
#pragma unroll 1
      for (int t = 0; t < S; ++t) y += red[tid * S + t];
      ybuf[i - i0] = y;
      if (i < split_i) ps0 += y * y;
      else ps1 += y * y;
    }
    consumer_sync();
  }
  // this CTA's parts of sum(y^2): warp trees, then the warps in order
  {
    const float t0 = warp_sum(ps0), t1 = warp_sum(ps1);
    if (lane == 0) {
      wred[warp * 2] = t0;
      wred[warp * 2 + 1] = t1;
    }
  }
  consumer_sync();
  if (tid < 2 && i0 < i1 && b_lo + tid <= (i1 - 1) / a.H) {
    float t = 0.f;
    for (int w = 0; w < kCW; ++w) t += wred[w * 2 + tid];
    st_tagged(a.post_part + 2 * c + tid, t, tag);
  }
  // the parts of every CTA that shares a row with this one, added in CTA order
  if (i0 < i1) {
#pragma unroll 1
    for (int r = 0; r < 2 && b_lo + r <= (i1 - 1) / a.H; ++r) {
      const int b = b_lo + r;
      const int cf = part_of(b * a.H, n, nctas), cl = part_of((b + 1) * a.H - 1, n, nctas);
#pragma unroll 1
      for (int cc = cf + tid; cc <= cl; cc += kConsumers) {
        const int beg = part_begin(cc, n, nctas);
        if (beg == part_begin(cc + 1, n, nctas)) {  // a CTA without outputs adds nothing
          red[cc - cf] = 0.f;
          continue;
        }
        const int slot = b - beg / a.H;
        const uint64_t t0 = globaltimer_ns();
        unsigned long long w;
        for (;;) {
          w = ld_tagged(a.post_part + 2 * cc + slot);
          if ((uint32_t)(w >> 32) == tag) break;
          if (*abort || globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.err, kErrWaitTimeout);
            *abort = 1;
            break;
          }
          __nanosleep(64);
        }
        red[cc - cf] = tagged_value(w);
      }
      consumer_sync();
      if (tid == 0) {
        float t = 0.f;
        for (int cc = cf; cc <= cl; ++cc) t += red[cc - cf];
        s_inv[r] = rsqrtf(t / a.H + a.eps);
      }
      consumer_sync();
    }
  }
#pragma unroll 1
  for (int i = i0 + tid; i < i1; i += kConsumers) {
    const bool second = i >= split_i;
    const int col = second ? i - split_i : i - b_lo * a.H;
    const float r = __bfloat162float(a.x[i]) + ybuf[i - i0] * a.w_post[col] * s_inv[second ? 1 : 0];
    a.out[i] = __float2bfloat16_rn(r);
    if (a.out_tap) a.out_tap[i] = r;
  }
}

// The work items of one ring stage (n_items items of nbs tiles, row groups r_first ..),
// one whole item per warp at a time.  The partial sums of rows [16 r, 16 r + 16) over an
// item's tiles are stored (no atomics, tagged with the step) into the k-split's slice of
// `part`, times the batch row's factor `scale` (nullable: 1).  One out-of-line copy serves both GEMVs, so
// the o_proj phase runs code the QKV phase already brought into the instruction cache;
// the stage and the operand fragments come as shared-window addresses (ld.shared).
template <int NT, int UNR = 4>
__device__ __noinline__ void gemv_stage(const StepGemv& gm, int B, unsigned long long* part,
                                        int s, uint32_t stage, int n_items, int r_first,
                                        uint32_t frag, const float* scale, uint32_t tag, int warp,
                                        int lane) {
  const int nbs = gm.nbs;
  const int g = lane >> 2, t = lane & 3;
  const int R16 = gm.R * 16;
  unsigned long long* dst = part + (size_t)s * B * R16;
  for (int item = warp; item < n_items; item += kCW) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint32_t tp = stage + (uint32_t)(item * nbs * kQ8TileBytes);
    const uint32_t fr = frag + lane * 16;
#pragma unroll UNR
    for (int i = 0; i < nbs; ++i) {
      const uint4 w = lds128(tp + i * kQ8TileBytes + lane * 16);
      const uint32_t d = lds32(tp + i * kQ8TileBytes + 512 + g * 4);
      q8_tile_mma<NT>(acc, w, d, fr + i * NT * 512);
    }
    const int r = r_first + item;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int b = nt * 4 + t;
      if (b < B) {
        const float f = scale ? scale[b] : 1.f;
        st_tagged(dst + (size_t)b * R16 + r * 16 + g, (acc[nt][0] + acc[nt][1]) * f, tag);
        st_tagged(dst + (size_t)b * R16 + r * 16 + g + 8, (acc[nt][2] + acc[nt][3]) * f, tag);
      }
    }
  }
}

// ------------------------------------------------------------------ attention pieces
// byte offset of (row, 16-byte chunk) in a TMA tile written with the 128-byte swizzle
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  const int box = chunk >> 3, c = chunk & 7;
  return (uint32_t)(box * (Attn<HD>::T * 128) + row * 128 + ((c ^ (row & 7)) << 4));
}

// One head of unit (b, kvh): job < G query head kvh * G + job, G the key, G + 1 the value
// (with k_eq_v there is no value job: the key job writes V = unit RMSNorm of the raw K).
// Raw projection * 1/rms(x), per-head RMSNorm (q, k; v with the unit-norm flag), RoPE
// (q, k); queries go to q_s, the key and value row to the cache slot (bf16, RNE).
// the RoPE rotation of one pair, out of line: one copy of the sin/cos code serves all
static __device__ __noinline__ float2 rope_rotate(int P, float2 g, float x0, float x1) {
  float c, s;
  rope_cs(P, g, c, s);
  return make_float2(x0 * c - x1 * s, x0 * s + x1 * c);
}

template <int HD>
__device__ void head_job(const StepArgs& a, const int* geo, int b, int kvh, int job, int G,
                         float xss, float* q_s, bool tap_q, uint32_t tag, volatile int* abort,
                         int lane) {
  constexpr int J = HD / 32;
  const int rows = a.qkv.R * 16;  // q, k and (without k_eq_v) v heads
  const int kind = job < G ? 0 : (job == G ? 1 : 2);
  const int row0 = kind == 0 ? (kvh * G + job) * HD
                             : (kind == 1 ? (a.nh + kvh) * HD : (a.nh + a.nkv + kvh) * HD);
  // the projection: partial sums of the k-splits added in a fixed order, every load of a
  // group of kSG splits issued before the first add, and issued again (after a short
  // pause) until every one carries this step's tag: no grid barrier orders them
  constexpr int kSG = HD >= 512 ? 2 : 8;  // J values of kSG splits per load round
  const unsigned long long* src = a.qkv_part + (size_t)b * rows + row0 + lane;
  const size_t split_stride = (size_t)a.B * rows;
  // the per-head norm weight and the RoPE angles are constants: loaded before the wait for
  // the partial sums, so that no dependent global load follows it
  float wn[J];
  float2 rg[J / 2];
  {
    const float* w = kind == 0 ? a.w_q : a.w_k;  // a valid address for v too (unused)
#pragma unroll
    for (int j = 0; j < J; ++j) wn[j] = __ldg(w + lane + 32 * j);
#pragma unroll
    for (int j = 0; j < J / 2; ++j) rg[j] = __ldg(a.rope_g + lane + 32 * j);
  }
  float v[J];
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] = 0.f;
  const uint64_t t_start = globaltimer_ns();
  for (int s0 = 0; s0 < a.qkv.S; s0 += kSG) {
    float t[kSG][J];
    for (;;) {
      bool ready = true;
#pragma unroll
      for (int i = 0; i < kSG; ++i) {
        const int s = s0 + i < a.qkv.S ? s0 + i : a.qkv.S - 1;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const unsigned long long w = ld_tagged(src + s * split_stride + 32 * j);
          ready = ready && (uint32_t)(w >> 32) == tag;
          t[i][j] = tagged_value(w);
        }
      }
      if (ready) break;
      if (*abort || globaltimer_ns() - t_start > kWaitLimitNs) {
        atomicOr(a.err, kErrWaitTimeout);
        *abort = 1;
        break;
      }
      __nanosleep(32);
    }
#pragma unroll
    for (int i = 0; i < kSG; ++i)
      if (s0 + i < a.qkv.S) {
#pragma unroll
        for (int j = 0; j < J; ++j) v[j] += t[i][j];
      }
  }
  // input RMSNorm factor 1/rms(x) of the row, applied to the projection (linear)
  const float xinv = rsqrtf(xss / a.H + a.eps);
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] *= xinv;
  const int slot = geo[b * kGeoInts + kGeoSlot];
  if (kind == 1 && a.k_eq_v) {
    // no V projection: V is the raw K, RMS-normalised per head with unit weight
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) ss += v[j] * v[j];
    const float inv = rsqrtf(warp_sum(ss) / HD + a.eps);
    __nv_bfloat16* dst = a.v_cache + (((size_t)b * a.nkv + kvh) * a.C + slot) * HD;
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
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] *= inv * (kind < 2 ? wn[j] : 1.0f);
  }
  if (kind < 2) {
    const int P = geo[b * kGeoInts + kGeoP];
#pragma unroll
    for (int j = 0; j < J / 2; ++j) {
      const float2 r = rope_rotate(P, rg[j], v[j], v[j + J / 2]);
      v[j] = r.x;
      v[j + J / 2] = r.y;
    }
  }
  if (kind == 0) {
#pragma unroll
    for (int j = 0; j < J; ++j) q_s[job * HD + lane + 32 * j] = v[j];
    if (tap_q) {
      float* qt = a.q_tap + ((size_t)b * a.nh + kvh * G + job) * HD;
#pragma unroll
      for (int j = 0; j < J; ++j) qt[lane + 32 * j] = v[j];
    }
  } else {
    __nv_bfloat16* dst =
        (kind == 1 ? a.k_cache : a.v_cache) + (((size_t)b * a.nkv + kvh) * a.C + slot) * HD;
    float* tap = kind == 1 ? a.k_tap : a.v_tap;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      dst[lane + 32 * j] = __float2bfloat16_rn(v[j]);
      if (tap) tap[((size_t)b * a.nkv + kvh) * HD + lane + 32 * j] = v[j];
    }
    // the row is read next by a TMA load (async proxy) of this CTA
    fence_proxy_async_global();
  }
}

// One K/V tile: S = Q K^T for the 16 keys of key group kg (queries of the group as bf16
// hi rows 0..G-1 and lo rows 8..8+G-1), online softmax in base 2, O += P V with P split
// hi/lo, for the n8 tiles of O of dim part dh.
template <int HD>
__device__ __forceinline__ void attn_tile(uint32_t kb, const uint4* qf, int key0, int k_end,
                                          float cap_log2, float& m, float& l,
                                          float (&o)[Attn<HD>::NTW][4], int kg, int dh,
                                          int lane) {
  using AC = Attn<HD>;
  const uint32_t vb = kb + AC::TILE_BYTES;
  const int krow = kg * kKeysPerWarp;
  const int t = lane & 3;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < AC::KS; ++ks) {
    const uint4 qa = qf[ks * 32 + lane];
    const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
    const int mrow = krow + ((lane >> 4) << 3) + (lane & 7);
    const int mchunk = ks * 2 + ((lane >> 3) & 1);
    uint32_t b0, b1, b2, b3;
    ldmatrix_x4(kb + swz<HD>(mrow, mchunk), b0, b1, b2, b3);
    mma_bf16(s0, A, b0, b1);
    mma_bf16(s1, A, b2, b3);
  }
  float sv[4] = {s0[0] + s0[2], s0[1] + s0[3], s1[0] + s1[2], s1[1] + s1[3]};
  const int kidx0 = key0 + krow + 2 * t;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int key = kidx0 + (e & 1) + ((e >> 1) << 3);
    float s = sv[e];
    if (cap_log2 != 0.f) s = cap_log2 * tanhf(s);
    sv[e] = key < k_end ? s : -INFINITY;
  }
  float mloc = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
  const float m_new = fmaxf(m, mloc);
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float corr = ex2_approx(m - m_use);
  float p[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) p[e] = ex2_approx(sv[e] - m_use);
  l = l * corr + (p[0] + p[1]) + (p[2] + p[3]);
  m = m_new;
#pragma unroll
  for (int nt = 0; nt < AC::NTW; ++nt) {
    o[nt][0] *= corr;
    o[nt][1] *= corr;
    o[nt][2] *= corr;
    o[nt][3] *= corr;
  }
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
#pragma unroll
  for (int np = 0; np < AC::NTW / 2; ++np) {
    const int mrow = krow + (((lane >> 3) & 1) << 3) + (lane & 7);
    const int mchunk = (dh * (AC::NTW / 2) + np) * 2 + (lane >> 4);
    uint32_t b0, b1, b2, b3;
    ldmatrix_x4_trans(vb + swz<HD>(mrow, mchunk), b0, b1, b2, b3);
    mma_bf16(o[2 * np], PA, b0, b1);
    mma_bf16(o[2 * np + 1], PA, b2, b3);
  }
}

// The o_proj operand of k-split s, merged from the attention records after the second
// grid barrier by every CTA that multiplies that split (each merges what it needs; no
// CTA waits on another's merge).  For batch row b and columns d .. d + 3 of query head h,
// over the records r of h's unit (one per CTA that attended over its key tiles):
//   o = sum_r 2^(m_r - M) O_r / sum_r 2^(m_r - M) l_r,   M = max_r m_r,
// stored as fp16 hi + lo in MMA fragment order.  The first CTA of the split also writes o
// as the fp32 attention output.  A job is a column quad of one batch row.  With at most
// 256 jobs, RL = 256 / jobs (a power of two) lanes share a job, lane k taking records
// k, k + RL, ..., and their partial (M, den, acc) combine over a fixed butterfly; with
// more jobs, a thread takes JG of them at a time.  Each lane keeps the loads of RU records
// of each of its jobs in flight together.
// units[b * nk + kvh - kvh0] = first record slot | record count << 16 (build_unit_table).
template <int HD, int NT, int JG, int RU>
__device__ void merge_jobs(const StepArgs& a, int G, int s, bool write_attn, uint32_t* xw,
                           const unsigned* units, int nk, int kvh0) {
  using AC = Attn<HD>;
  const int nq = a.o.nbs * 8;  // column quads of the split (<= 128)
  const int jobs = a.B * nq;
  int RL = 1;
  while (JG == 1 && RL < 32 && jobs * RL * 2 <= kConsumers) RL *= 2;
  const int sub = threadIdx.x & (RL - 1);
  const int jstep = kConsumers / RL;
  // JG == 1: one pass for every thread (jobs <= jstep), so that all lanes of a warp reach
  // the butterfly's shuffles
  const int npass = JG == 1 ? 1 : (jobs + JG * jstep - 1) / (JG * jstep);
  for (int pass = 0; pass < npass; ++pass) {
    const int j0 = threadIdx.x / RL + pass * JG * jstep;
    const float* row[JG];
    int cnt[JG], dd[JG], maxc = 0;
#pragma unroll
    for (int g = 0; g < JG; ++g) {
      const int j = j0 + g * jstep;
      const int jj = j < jobs ? j : 0;  // a job past the end reads job 0's table (unused)
      const int b = jj / nq, col = s * 4 * nq + 4 * (jj - b * nq);
      const int hq = col / HD, kvh = hq / G;
      dd[g] = col % HD;
      const unsigned u = units[b * nk + kvh - kvh0];
      const int n = j < jobs ? (int)(u >> 16) : 0;
      cnt[g] = n > sub ? (n - sub + RL - 1) / RL : 0;  // this lane's records
      maxc = cnt[g] > maxc ? cnt[g] : maxc;
      row[g] = a.rec + ((size_t)(u & 0xffffu) * 8 + (hq - kvh * G)) * AC::RS +
               (size_t)sub * 8 * AC::RS;
    }
    float M[JG], den[JG];
    float4 acc[JG];
#pragma unroll
    for (int g = 0; g < JG; ++g) {
      M[g] = -INFINITY;
      den[g] = 0.f;
      acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 1
    for (int r0 = 0; r0 < maxc; r0 += RU) {
      float2 ml[JG][RU];
      float4 v[JG][RU];
#pragma unroll
      for (int g = 0; g < JG; ++g) {
        const int last = cnt[g] > 0 ? cnt[g] - 1 : 0;
#pragma unroll
        for (int i = 0; i < RU; ++i) {
          // clamped to a record of the lane (in range); slots past its count weigh 0
          const float* q = row[g] + min(r0 + i, last) * (RL * 8 * AC::RS);
          ml[g][i] = __ldcg(reinterpret_cast<const float2*>(q + HD));
          v[g][i] = __ldcg(reinterpret_cast<const float4*>(q + dd[g]));
        }
      }
#pragma unroll
      for (int g = 0; g < JG; ++g) {
        float Mc = M[g];
#pragma unroll
        for (int i = 0; i < RU; ++i) {
          if (r0 + i >= cnt[g]) {  // weight 0, and nothing of a record outside the run
            ml[g][i] = make_float2(-INFINITY, 0.f);
            v[g][i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          Mc = fmaxf(Mc, ml[g][i].x);
        }
        const float Mu = Mc == -INFINITY ? 0.f : Mc;
        const float f = ex2_approx(M[g] - Mu);  // rescales what earlier chunks summed
        den[g] *= f;
        acc[g].x *= f;
        acc[g].y *= f;
        acc[g].z *= f;
        acc[g].w *= f;
#pragma unroll
        for (int i = 0; i < RU; ++i) {
          const float w = ex2_approx(ml[g][i].x - Mu);
          den[g] = fmaf(w, ml[g][i].y, den[g]);
          acc[g].x = fmaf(w, v[g][i].x, acc[g].x);
          acc[g].y = fmaf(w, v[g][i].y, acc[g].y);
          acc[g].z = fmaf(w, v[g][i].z, acc[g].z);
          acc[g].w = fmaf(w, v[g][i].w, acc[g].w);
        }
        M[g] = Mc;
      }
    }
    // the lanes of a job: butterfly over their partial states (a fixed order)
    for (int o = 1; o < RL; o <<= 1) {
      const float Mo = __shfl_xor_sync(0xffffffffu, M[0], o);
      const float Mn = fmaxf(M[0], Mo);
      const float Mu = Mn == -INFINITY ? 0.f : Mn;
      const float fa = ex2_approx(M[0] - Mu), fb = ex2_approx(Mo - Mu);
      den[0] = den[0] * fa + __shfl_xor_sync(0xffffffffu, den[0], o) * fb;
      acc[0].x = acc[0].x * fa + __shfl_xor_sync(0xffffffffu, acc[0].x, o) * fb;
      acc[0].y = acc[0].y * fa + __shfl_xor_sync(0xffffffffu, acc[0].y, o) * fb;
      acc[0].z = acc[0].z * fa + __shfl_xor_sync(0xffffffffu, acc[0].z, o) * fb;
      acc[0].w = acc[0].w * fa + __shfl_xor_sync(0xffffffffu, acc[0].w, o) * fb;
      M[0] = Mn;
    }
#pragma unroll
    for (int g = 0; g < JG; ++g) {
      const int j = j0 + g * jstep;
      if (j < jobs && sub == 0) {
        const int b = j / nq, cq = 4 * (j - b * nq);
        const float inv = den[g] > 0.f ? rcp_approx(den[g]) : 0.f;
        const float4 o = make_float4(acc[g].x * inv, acc[g].y * inv, acc[g].z * inv, acc[g].w * inv);
        if (write_attn)
          *reinterpret_cast<float4*>(a.o_attn + (size_t)b * a.nh * HD + s * 4 * nq + cq) = o;
        __half h0, l0, h1, l1;
        split_f16(o.x, h0, l0);
        split_f16(o.y, h1, l1);
        int w = operand_word<NT>(cq, b);
        xw[w] = pack_h2(h0, h1);
        xw[w + 16] = pack_h2(l0, l1);
        split_f16(o.z, h0, l0);
        split_f16(o.w, h1, l1);
        w = operand_word<NT>(cq + 2, b);
        xw[w] = pack_h2(h0, h1);
        xw[w + 16] = pack_h2(l0, l1);
      }
    }
  }
}

constexpr int kOperandBytes = 16 * 4 * 512;  // o_proj operand: nbs <= 16 blocks, NT <= 4
static_assert(kOperandBytes + kMaxBatch * 9 * 4 <= kUnionBytes, "unit table after the operand");

// The record runs of the units whose query heads own the o_proj split s's columns
// [s W, s W + W) (at most 9 KV heads): units[b * nk + kvh - kvh0] = first record slot |
// record count << 16.  Depends on the geometry only, so it is built while the CTA waits
// at the second grid barrier.  The host keeps the grid-wide key-tile count below 2^24 and
// the grid at most 256 CTAs: the CTA that owns tile t, ((t + 1) P - 1) / Nt, is exact in
// 32-bit arithmetic.
template <int HD>
__device__ __forceinline__ void build_unit_table(const StepArgs& a, const int* geo, int Nt, int G,
                                                 int s, unsigned* units) {
  const int W = a.o.nbs * 32;
  const int kvh0 = s * W / HD / G, nk = (s * W + W - 1) / HD / G - kvh0 + 1;
  const int tid = threadIdx.x;
  if (tid < a.B * nk) {
    const int b = tid / nk, kvh = kvh0 + tid - b * nk;
    const int nt = geo[b * kGeoInts + kGeoNt];
    const int pre = geo[b * kGeoInts + kGeoPre] + kvh * nt;  // the unit's first tile
    const unsigned P = gridDim.x;
    const int first = nt > 0 ? (int)(((unsigned)(pre + 1) * P - 1u) / (unsigned)Nt) : 0;
    const int last = nt > 0 ? (int)(((unsigned)(pre + nt) * P - 1u) / (unsigned)Nt) : -1;
    // the record of CTA first + r for unit u sits in slot first + r + u
    units[tid] = (unsigned)(first + b * a.nkv + kvh) | ((unsigned)(last - first + 1) << 16);
  }
}

// Builds the o_proj operand of k-split s in xw (the union) from the records.  Batch slots
// past B are left as they are: their MMA columns never reach a stored output.
template <int HD, int NT>
__device__ __forceinline__ void merge_operand(const StepArgs& a, int G, int s, bool write_attn,
                                              uint32_t* xw) {
  const int W = a.o.nbs * 32;
  const int kvh0 = s * W / HD / G, nk = (s * W + W - 1) / HD / G - kvh0 + 1;
  const unsigned* units =
      reinterpret_cast<const unsigned*>(reinterpret_cast<const uint8_t*>(xw) + kOperandBytes);
  // up to 256 column quads: lanes share a job's records; more: several jobs per thread
  if (a.B * W / 4 <= kConsumers)
    merge_jobs<HD, NT, 1, 10>(a, G, s, write_attn, xw, units, nk, kvh0);
  else
    merge_jobs<HD, NT, 4, 3>(a, G, s, write_attn, xw, units, nk, kvh0);
}

// ------------------------------------------------------------------ the load schedule
// A CTA's loads in order: the stages of its QKV slice (phase A), its K/V tiles (phase B),
// the stages of its o_proj slice (phase C).  Load j can also be prefetched into L2 by
// its byte ranges: the first kEarlyTiles K/V tiles go to L2 while phase A still holds the
// ring, so HBM keeps streaming through the phase A tail and the grid barrier.  Deeper
// prefetching only lengthens the queues that the step's latency-bound parts (barriers,
// the head epilogue, the record merge) wait in, and thrashes L2 on long contexts.
struct Schedule {
  Slice sa, so;
  int nA, nB, nC;
  int t0, t1;  // global key tiles [t0, t1)
};

__device__ __forceinline__ int gemv_loads(const StepGemv& g, const Slice& sl) {
  return (sl.r1 - sl.r0 + g.ips - 1) / g.ips;
}

template <int HD>
__device__ void prefetch_load(const StepArgs& a, const Schedule& sc, const int* geo, int j) {
  using AC = Attn<HD>;
  if (j < sc.nA || j >= sc.nA + sc.nB) {
    const bool in_a = j < sc.nA;
    const StepGemv& g = in_a ? a.qkv : a.o;
    const Slice& sl = in_a ? sc.sa : sc.so;
    const int r = sl.r0 + (in_a ? j : j - sc.nA - sc.nB) * g.ips;
    const int n = g.ips < sl.r1 - r ? g.ips : sl.r1 - r;
    prefetch_bulk_l2(g.w + ((size_t)sl.s * g.R + r) * g.nbs * kQ8TileBytes,
                     (uint32_t)(n * g.nbs * kQ8TileBytes));
    return;
  }
  int t = sc.t0 + (j - sc.nA);  // global tile -> (b, kvh, tile)
  for (int b = 0; b < a.B; ++b) {
    const int nt = geo[b * kGeoInts + kGeoNt];
    if (t < nt * a.nkv) {
      const int kvh = t / nt, lt = t - kvh * nt;
      const long long row = (long long)(b * a.nkv + kvh) * a.C + geo[b * kGeoInts + kGeoLo] +
                            (long long)lt * AC::T;
      long long nrow = AC::T;
      if (row + nrow > a.cache_rows) nrow = a.cache_rows - row;  // last tile of the cache
      if (nrow > 0) {
        const uint32_t bytes = (uint32_t)(nrow * HD * 2);
        prefetch_bulk_l2(a.k_cache + row * HD, bytes);
        prefetch_bulk_l2(a.v_cache + row * HD, bytes);
      }
      return;
    }
    t -= nt * a.nkv;
  }
}

// ------------------------------------------------------------------ the kernel
template <int HD, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    step_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const __grid_constant__ StepArgs a) {
  using AC = Attn<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* uni = smem + kStages * kStageBytes;
  uint8_t* small = uni + kUnionBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(small);
  uint64_t* empty = full + kStages;
  uint64_t* append_bar = empty + kStages;
  uint64_t* next_bar = append_bar + 1;  // consumers passed the grid barrier
  uint64_t* arrived_bar = reinterpret_cast<uint64_t*>(small + 88);  // ... arrived at it
  uint64_t* stall_bar = reinterpret_cast<uint64_t*>(small + 288);  // test hook: never completes
  uint64_t* polled_bar = reinterpret_cast<uint64_t*>(small + 296);  // first queries formed
  volatile int* s_abort = reinterpret_cast<volatile int*>(small + 64);
  int* s_issued = reinterpret_cast<int*>(small + 68);
  uint32_t* s_tag = reinterpret_cast<uint32_t*>(small + 72);  // this step's partial-sum tag
  unsigned long long* s_gbase = reinterpret_cast<unsigned long long*>(small + 80);
  unsigned* s_max = reinterpret_cast<unsigned*>(small + 96);
  float* s_xss = reinterpret_cast<float*>(small + 160);  // sum(x^2) per batch row
  float* s_inv = reinterpret_cast<float*>(small + 224);  // [16]: 2^-scale per batch row
  int* geo = reinterpret_cast<int*>(small + 512);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, nctas = gridDim.x;
  if (blockDim.x != kThreads) return;  // the launch always uses kThreads (B <= 16 is checked
                                       // on the host)

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    mbar_init(append_bar, 1);
    mbar_init(next_bar, 1);
    mbar_init(arrived_bar, 1);
    mbar_init(stall_bar, 1);
    mbar_init(polled_bar, 1);
    *s_abort = 0;
    *s_issued = 0;
    fence_barrier_init();
  }
  if (tid < kMaxBatch) s_max[tid] = 0u;
  __syncthreads();
  if (tid == 0) HFA_STAMP(a, kStampEntry);
  // Programmatic dependent launch: the next kernel on the stream may be scheduled now (its
  // CTAs take over the SMs as these exit).  Nothing this kernel reads or writes in global
  // memory is touched before the wait for the previous kernel, except what no kernel
  // writes: the weights, loaded here into the first ring stages with a single batch tile
  // (with more, the activation loads would queue behind them).
  constexpr bool early_qkv = NT == 1;
  {
    pdl_launch_dependents();
    if (early_qkv && warp == kCW && lane == 0) {
      const Slice sa0 = gemv_slice(a.qkv, c, nctas);
      const int nA0 = (sa0.r1 - sa0.r0 + a.qkv.ips - 1) / a.qkv.ips;
      for (int k = 0; k < nA0 && k < kStages; ++k) {
        const int r = sa0.r0 + k * a.qkv.ips;
        const int n = a.qkv.ips < sa0.r1 - r ? a.qkv.ips : sa0.r1 - r;
        const uint32_t bytes = (uint32_t)(n * a.qkv.nbs * kQ8TileBytes);
        mbar_arrive_expect_tx(&full[k], bytes);
        bulk_load(ring + k * kStageBytes, a.qkv.w + ((size_t)sa0.s * a.qkv.R + r) * a.qkv.nbs * kQ8TileBytes,
                  bytes, &full[k]);
      }
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
    }
    pdl_wait();
    if (tid == 0) HFA_STAMP(a, kStampWait);
  }

  const int G = a.nh / a.nkv;
  if (warp == kCW) {
    // ============================================================== producer
    Schedule sc;
    sc.sa = gemv_slice(a.qkv, c, nctas);
    sc.so = gemv_slice(a.o, c, nctas);
    sc.nA = gemv_loads(a.qkv, sc.sa);
    sc.nC = gemv_loads(a.o, sc.so);
    uint32_t q = 0;
    bool ok = true;
    auto acquire = [&](uint32_t bytes) -> int {
      const int st = (int)(q % kStages);
      if (q >= (uint32_t)kStages &&
          !mbar_wait(&empty[st], ((q / kStages) - 1) & 1, a.err, s_abort)) {
        *s_abort = 1;
        return -1;
      }
      if (*s_abort) return -1;
      mbar_arrive_expect_tx(&full[st], bytes);
      return st;
    };
    auto issue_gemv = [&](const StepGemv& g, const Slice& sl, int k) {
      const int r = sl.r0 + k * g.ips;
      const int n = g.ips < sl.r1 - r ? g.ips : sl.r1 - r;
      const uint32_t bytes = (uint32_t)(n * g.nbs * kQ8TileBytes);
      const int st = acquire(bytes);
      if (st < 0) {
        ok = false;
        return;
      }
      bulk_load(ring + st * kStageBytes, g.w + ((size_t)sl.s * g.R + r) * g.nbs * kQ8TileBytes,
                bytes, &full[st]);
      ++q;
    };
    // phase A depends on nothing of this step; its copies go out as soon as the consumers
    // hold their activations (barrier 3), whose loads would otherwise queue behind them
    asm volatile("bar.sync 3, %0;" ::"n"(kThreads) : "memory");
    if (lane == 0) {
      if (early_qkv) {
        q = (uint32_t)(sc.nA < kStages ? sc.nA : kStages);  // issued before the wait
      } else {
        for (int k = 0; k < sc.nA && k < kStages && ok; ++k) issue_gemv(a.qkv, sc.sa, k);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
      }
      HFA_STAMP(a, kStampProdA);
    }
    __syncwarp();
    // visible slots and key tiles of each sequence, for both sides (consumers read them
    // after barrier 2)
    int span = 0;  // key tiles of this lane's sequence over all KV heads
    if (lane < a.B) {
      const int b = lane < a.B ? lane : 0;  // in range even where the test is folded away
      const int P = a.seq_pos[b];
      const bool bad = P < 0 || (!a.ring && P >= a.C);
      int lo, hi, slot;
      if (a.ring) {
        lo = 0;
        hi = P < a.C - 1 ? P : a.C - 1;
        slot = bad ? 0 : P % a.C;
      } else {
        lo = a.sliding ? (P - a.window + 1 > 0 ? P - a.window + 1 : 0) : 0;
        hi = P;
        slot = P;
      }
      int* gb = geo + b * kGeoInts;
      gb[kGeoP] = P;
      gb[kGeoLo] = lo;
      gb[kGeoHi] = hi;
      gb[kGeoNt] = bad ? 0 : (hi - lo + 1 + AC::T - 1) / AC::T;
      gb[kGeoTn] = bad ? -1 : (slot - lo) / AC::T;
      gb[kGeoSlot] = slot;
      span = gb[kGeoNt] * a.nkv;
      if (bad && c == 0) atomicOr(a.err, kErrBadPosition);
    }
    int incl = span;  // inclusive prefix over the sequences
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < a.B) geo[lane * kGeoInts + kGeoPre] = incl - span;
    __syncwarp();
    {
      int Nt = 0;
      for (int b = 0; b < a.B; ++b) Nt += geo[b * kGeoInts + kGeoNt] * a.nkv;
      sc.t0 = Nt > 0 ? part_begin(c, Nt, nctas) : 0;
      sc.t1 = Nt > 0 ? part_begin(c + 1, Nt, nctas) : 0;
      sc.nB = sc.t1 - sc.t0;
    }
    if (lane == 0)
      for (int j = 0; j < Fill<NT>::kEarlyTiles && j < sc.nB; ++j)
        prefetch_load<HD>(a, sc, geo, sc.nA + j);
    // while the consumers run phase A: sum(x^2) of the input rows whose key tiles this CTA
    // attends over (the input norm's statistic, read in phase B)
    {
      int base = 0;
      for (int b = 0; b < a.B; ++b) {
        const int span_b = geo[b * kGeoInts + kGeoNt] * a.nkv;
        if (span_b > 0 && base < sc.t1 && base + span_b > sc.t0) {
          const float ss = row_sumsq(a.x + (size_t)b * a.H, a.H, lane);
          if (lane == 0) s_xss[b] = ss;
        }
        base += span_b;
      }
    }
    __syncwarp();
    asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");  // geometry, statistics
    if (lane == 0) {
      uint32_t n_app = 0;  // appends waited for (one per unit whose new slot is here)
      const uint64_t kv_policy = l2_policy_evict_first();  // the cache is read once a step
      for (int k = (int)q; k < sc.nA && ok; ++k) issue_gemv(a.qkv, sc.sa, k);
      int kv_issued = 0;  // K/V tiles issued so far (for the fill limit)
      for_each_segment(geo, a.B, a.nkv, sc.t0, sc.t1, [&](int b, int kvh, int lt0, int lt1) {
        const int lo = geo[b * kGeoInts + kGeoLo], tn = geo[b * kGeoInts + kGeoTn];
        const bool owner = tn >= lt0 && tn < lt1;
        const int row_base = (b * a.nkv + kvh) * a.C + lo;
        for (int i = 0; ok && i < lt1 - lt0; ++i) {
          const int lt = seg_tile(i, lt0, lt1, owner ? tn : -1);
          if (owner && lt == tn) {
            // the slot appended in this step: its row is written by this CTA's consumers
            if (!mbar_wait(append_bar, n_app & 1, a.err, s_abort)) {
              *s_abort = 1;
              ok = false;
              break;
            }
            ++n_app;
          }
          if (Fill<NT>::kBeforeQueries > 0 && kv_issued == Fill<NT>::kBeforeQueries &&
              !mbar_wait(polled_bar, 0, a.err, s_abort)) {
            ok = false;
            break;
          }
          ++kv_issued;
          const int st = acquire(AC::STAGE_BYTES);
          if (st < 0) {
            ok = false;
            break;
          }
          uint8_t* kt = ring + st * kStageBytes;
          uint8_t* vt = kt + AC::TILE_BYTES;
          const int row = row_base + lt * AC::T;
#pragma unroll
          for (int j = 0; j < AC::BOXES; ++j) {
            tma_load_2d_hint(kt + j * AC::T * 128, &tmk, &full[st], 64 * j, row, kv_policy);
            tma_load_2d_hint(vt + j * AC::T * 128, &tmv, &full[st], 64 * j, row, kv_policy);
          }
          ++q;
        }
      });
      // the o_proj slice goes out once the consumers have arrived at the grid barrier: the
      // arrival's release waits for this SM's copies in flight, so they come after it
      HFA_STAMP(a, kStampProdKV);
      if (sc.nC > 0 && ok && !mbar_wait(arrived_bar, 0, a.err, s_abort)) ok = false;
      for (int k = 0; k < sc.nC && ok; ++k) issue_gemv(a.o, sc.so, k);
      HFA_STAMP(a, kStampProdC);
      *s_issued = (int)q;
      // the layer that runs next: its first loads (this CTA's QKV slice, same shape) go to
      // L2 once the attention is over, while the o_proj phase leaves HBM idle; paced, so
      // that the latency-bound tail of this step does not queue behind them
      if (a.next_qkv_w && ok && mbar_wait(next_bar, 0, a.err, s_abort)) {
        const uint8_t* src =
            a.next_qkv_w + ((size_t)sc.sa.s * a.qkv.R + sc.sa.r0) * a.qkv.nbs * kQ8TileBytes;
        const size_t bytes = (size_t)(sc.sa.r1 - sc.sa.r0) * a.qkv.nbs * kQ8TileBytes;
        for (size_t off = 0; off < bytes; off += kSuccChunk) {
          prefetch_bulk_l2(src + off, (uint32_t)(bytes - off < kSuccChunk ? bytes - off : kSuccChunk));
          __nanosleep(kSuccPauseNs);
        }
      }
    }
  } else {
    // ============================================================== consumers
    // the barrier count at the start numbers this step (read now, used after phase A)
    const unsigned long long arrivals0 = tid == 0 ? ldcg_pinned64(a.gbar) : 0ull;
    uint32_t q = 0;
    auto wait_stage = [&]() -> int {
      const int st = (int)(q % kStages);
      const bool ok = mbar_wait(&full[st], (q / kStages) & 1, a.err, s_abort);
      if (!ok) *s_abort = 1;
      return ok ? st : -1;
    };
    auto release_stage = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[q % kStages]);
      ++q;
    };

    // ---------------------------------------------------------- A: QKV
    {
      const Slice sl = gemv_slice(a.qkv, c, nctas);
      build_x_operand<NT>(a, sl.s, reinterpret_cast<uint32_t*>(uni), s_max, s_inv, arrivals0,
                          s_gbase, s_tag);
      if (tid == 0) HFA_STAMP(a, kStampOperand);
      const uint32_t tag = *s_tag;
      // test hook of the failure path: a bounded wait that runs out
      if (a.stall && c == 0 && !mbar_wait(stall_bar, 0, a.err, s_abort)) *s_abort = 1;
      for (int r = sl.r0; r < sl.r1; r += a.qkv.ips) {
        const int n = a.qkv.ips < sl.r1 - r ? a.qkv.ips : sl.r1 - r;
        const int st = wait_stage();
        if (st >= 0)
          gemv_stage<NT>(a.qkv, a.B, a.qkv_part, sl.s, smem_u32(ring + st * kStageBytes), n, r,
                         smem_u32(uni), s_inv, tag, warp, lane);
        release_stage();
      }
    }
    if (tid == 0) HFA_STAMP(a, kStampGemvA);
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");  // geometry, statistics
    int Nt = 0;
    for (int b = 0; b < a.B; ++b) Nt += geo[b * kGeoInts + kGeoNt] * a.nkv;
    const int t0 = Nt > 0 ? part_begin(c, Nt, nctas) : 0;
    const int t1 = Nt > 0 ? part_begin(c + 1, Nt, nctas) : 0;

    // ---------------------------------------------------------- B: attention
    {
      uint4* qf = reinterpret_cast<uint4*>(uni);
      float* q_s = reinterpret_cast<float*>(uni + AC::QS_OFF);
      float* red = reinterpret_cast<float*>(uni);  // [key group][8][RS] after the last tile
      const uint32_t ring_base = smem_u32(ring);
      bool first_segment = true;  // stamps: queries of the CTA's first segment ready
      for_each_segment(geo, a.B, a.nkv, t0, t1, [&](int b, int kvh, int lt0, int lt1) {
        const int* gb = geo + b * kGeoInts;
        const int lo = gb[kGeoLo], hi = gb[kGeoHi], tn = gb[kGeoTn];
        const bool owner = tn >= lt0 && tn < lt1;
        const int unit = b * a.nkv + kvh;
        const int njobs = G + (owner ? (a.k_eq_v ? 1 : 2) : 0);  // q heads, k, v
        for (int job = warp; job < njobs; job += kCW)
          head_job<HD>(a, geo, b, kvh, job, G, s_xss[b], q_s, lt0 == 0 && a.q_tap != nullptr,
                       *s_tag, s_abort, lane);
        consumer_sync();
        if (tid == 0 && first_segment) mbar_arrive(polled_bar);
        if (owner && tid == 0) mbar_arrive(append_bar);
        // query fragments: rows 0..G-1 = hi(q * qscale), rows 8..8+G-1 = lo
        {
          const int g = lane >> 2, t = lane & 3;
          for (int ks = warp; ks < AC::KS; ks += kCW) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (g < G) {
              const float* qr = q_s + g * HD + ks * 16 + 2 * t;
              __nv_bfloat16 h[4], l[4];
              split_bf16(qr[0] * a.qscale, h[0], l[0]);
              split_bf16(qr[1] * a.qscale, h[1], l[1]);
              split_bf16(qr[8] * a.qscale, h[2], l[2]);
              split_bf16(qr[9] * a.qscale, h[3], l[3]);
              w[0] = pack_bf2(h[0], h[1]);
              w[1] = pack_bf2(l[0], l[1]);
              w[2] = pack_bf2(h[2], h[3]);
              w[3] = pack_bf2(l[2], l[3]);
            }
            qf[ks * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        consumer_sync();
        if (tid == 0 && first_segment) HFA_STAMP(a, kStampAttn);
        first_segment = false;
        const int kg = warp % AC::NC, dh = warp / AC::NC;  // key group, dim part
        float m = -INFINITY, l = 0.f;
        float o[AC::NTW][4];
#pragma unroll
        for (int i = 0; i < AC::NTW; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        for (int i = 0; i < lt1 - lt0; ++i) {
          const int lt = seg_tile(i, lt0, lt1, owner ? tn : -1);
          const int st = wait_stage();
          if (st >= 0)
            attn_tile<HD>(ring_base + st * kStageBytes, qf, lo + lt * AC::T, hi + 1, a.cap_log2,
                          m, l, o, kg, dh, lane);
          release_stage();
        }
        if (tid == 0) HFA_STAMP(a, kStampStream);
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        // combine the warps of this CTA into the unit's record of this CTA
        consumer_sync();
        {
          const int g = lane >> 2, t = lane & 3;
          float* mine = red + kg * 8 * AC::RS;
          if (g < G) {
            if (t == 0 && dh == 0) {
              mine[g * AC::RS + HD] = m;
              mine[g * AC::RS + HD + 1] = l;
            }
#pragma unroll
            for (int nt = 0; nt < AC::NTW; ++nt) {
              const int d = (dh * AC::NTW + nt) * 8 + 2 * t;
              mine[g * AC::RS + d] = o[nt][0] + o[nt][2];
              mine[g * AC::RS + d + 1] = o[nt][1] + o[nt][3];
            }
          }
        }
        consumer_sync();
        float* rec = a.rec + (size_t)(c + unit) * 8 * AC::RS;
        for (int e = tid; e < G * (HD + 2); e += kConsumers) {
          const int h = e / (HD + 2), d = e - h * (HD + 2);
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < AC::NC; ++w) M = fmaxf(M, red[(w * 8 + h) * AC::RS + HD]);
          const float Mu = M == -INFINITY ? 0.f : M;
          float acc = 0.f;
          if (d == HD) {
            acc = M;
          } else {
#pragma unroll
            for (int w = 0; w < AC::NC; ++w)
              acc += ex2_approx(red[(w * 8 + h) * AC::RS + HD] - Mu) * red[(w * 8 + h) * AC::RS + d];
          }
          rec[h * AC::RS + d] = acc;
        }
        consumer_sync();  // the next segment's queries overwrite the merge area
      });
      // A CTA without tiles (fewer tiles than CTAs) that sits inside a unit's run of
      // CTAs -- its position t0 is a tile of the unit other than the first -- leaves a
      // zero-weight record there, so that the unit's records fill one run of slots.
      int tin = t0, bin = 0;
      if (t0 == t1 && t0 < Nt)
        while (tin >= geo[bin * kGeoInts + kGeoNt] * a.nkv)
          tin -= geo[bin++ * kGeoInts + kGeoNt] * a.nkv;
      if (t0 == t1 && t0 < Nt && tin % geo[bin * kGeoInts + kGeoNt] != 0) {
        const int b = bin;
        const int kvh = tin / geo[b * kGeoInts + kGeoNt];
        float* rec = a.rec + (size_t)(c + b * a.nkv + kvh) * 8 * AC::RS;
        for (int e = tid; e < 8 * AC::RS; e += kConsumers) {
          const int d = e % AC::RS;
          rec[e] = d == HD ? -INFINITY : 0.f;
        }
      }
    }
    const Slice sl = gemv_slice(a.o, c, nctas);
    if (tid == 0) HFA_STAMP(a, kStampRecords);
    grid_arrive(a.gbar);
    if (tid == 0) mbar_arrive(arrived_bar);
    build_unit_table<HD>(a, geo, Nt, G, sl.s,
                         reinterpret_cast<unsigned*>(uni + kOperandBytes));  // while waiting
    grid_wait(a.gbar, *s_gbase + (unsigned long long)nctas, a.err, s_abort);
    if (tid == 0) HFA_STAMP(a, kStampBarrier);
    if (a.next_qkv_w && tid == 0) mbar_arrive(next_bar);

    // ---------------------------------------------------------- C: o_proj + residual
    {
      merge_operand<HD, NT>(a, G, sl.s, sl.first, reinterpret_cast<uint32_t*>(uni));
      consumer_sync();
      if (tid == 0) HFA_STAMP(a, kStampMerge);
      for (int r = sl.r0; r < sl.r1; r += a.o.ips) {
        const int n = a.o.ips < sl.r1 - r ? a.o.ips : sl.r1 - r;
        const int st = wait_stage();
        if (st >= 0)
          gemv_stage<NT>(a.o, a.B, a.y_part, sl.s, smem_u32(ring + st * kStageBytes), n, r,
                         smem_u32(uni), nullptr, *s_tag, warp, lane);
        release_stage();
      }
    }
    consumer_sync();  // the union (operand) is free for the epilogue
    if (tid == 0) HFA_STAMP(a, kStampGemvC);
    if (a.w_post)
      finish_outputs_post(a, c, nctas, reinterpret_cast<float*>(uni),
                          reinterpret_cast<float*>(ring), *s_tag, s_abort);
    else
      finish_outputs(a, c, nctas, reinterpret_cast<float*>(uni), *s_tag, s_abort);
    if (tid == 0) HFA_STAMP(a, kStampExit);
  }

  // drain: after a give-up, copies may still be landing in the ring
  __syncthreads();
  if (tid == 0 && *s_abort) {
    const int issued = *s_issued;
    for (int st = 0; st < kStages && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / kStages) * kStages;
      mbar_wait(&full[st], (last / kStages) & 1, a.err);
    }
  }
}

}  // namespace step
namespace {
// devices on which a kernel instantiation has its shared-memory opt-in (internal linkage:
// a function-local static of a template would be merged across every loaded library)
template <int HD, int NT>
struct StepOptIn {
  static unsigned long long mask;
};
template <int HD, int NT>
unsigned long long StepOptIn<HD, NT>::mask = 0ull;
}  // namespace
namespace step {

template <int HD, int NT>
cudaError_t launch_step_t(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                          int grid, cudaStream_t s) {
  auto kern = step_kernel<HD, NT>;
  // the shared-memory opt-in, once per device (devices 0..63; beyond, every launch)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  unsigned long long* opted_in = &StepOptIn<HD, NT>::mask;
  if (!bit || !(__atomic_load_n(opted_in, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(opted_in, bit, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

template <int HD>
cudaError_t launch_step_hd(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           int grid, cudaStream_t s) {
  const int nt = a.B <= 4 ? 1 : (a.B <= 8 ? 2 : 4);
  if (nt == 1) return launch_step_t<HD, 1>(a, tk, tv, grid, s);
  if (nt == 2) return launch_step_t<HD, 2>(a, tk, tv, grid, s);
  return launch_step_t<HD, 4>(a, tk, tv, grid, s);
}

}  // namespace step
}  // namespace hfa
