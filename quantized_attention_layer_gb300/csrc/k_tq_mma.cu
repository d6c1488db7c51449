// k_tq_mma.cu -- flash-decode over the quantised (TurboQuant) KV cache on the tensor cores:
// head dims 64, 128, 256 and 512 (one norm block per 256 dims), codes of 4 bits (two per
// byte) or one byte per code, K coded or stored raw in bf16 (the hybrid layout, up to hd
// 256).
//
// gemma4/gpu_full_attn.rs, encode_one_layer: the TQ attention (flash_attn_vec_tq,
// flash_attn_vec_tq_hb, flash_attn_vec_hybrid): each score is the rotated query against
// the key's centroids times the key's block norm, the output the softmax-weighted sum of
// the value centroids times the value norms, both in the rotated domain; the output is
// rotated back at the end.  This is the arithmetic of the CUDA-core kernel in k_tq.cu,
// mapped onto mma.sync.
//
// GB300 design.  One CTA = (sequence, KV head, key chunk), one per SM.  A producer warp
// streams stages of T keys: the K and V code tiles by 2-D TMA (byte rows, swizzled at the
// box width, so the consumers' 32-bit reads of eight rows never share a bank) and the
// norms by 4-byte cp.async (a chunk may start at any key), all completing on the stage's
// mbarrier.  Consumer warps take 16 keys of each stage.  Centroids are decoded through a
// table in shared memory (one copy per bank: entry c of lane l at word 32 c + l) holding
// each centroid as bf16 hi + lo; two table words give a pair of MMA operand registers by
// one byte permute each.  All query heads of the group share one m16n8k16 MMA: rows
// 0..G-1 hold hi(q), rows 8..8+G-1 lo(q), against B = hi(c) and B = lo(c), so the scores
// keep about 16 bits of both operands; P times the V norm is split the same way for
// O += P V.  A 32-bit code read gives four (8-bit) or eight (4-bit) adjacent dims of one
// key, and the MMA's k index (scores) and n index (O) walk the dims in that order: the
// query fragments and the output columns follow the same permutation, so every code is
// read once and nothing is transposed.
#include "hfa_common.cuh"
#include "hfa_internal.h"
#include "hfa_tq.cuh"

namespace hfa {
namespace {

constexpr int kTqmMaxStages = 4;
constexpr int kTqmSmemBudget = 225280;  // stages + tables + query areas, bytes
constexpr int kTqmMaxSplits = 256;      // the merge's weight table: 8 x 256 floats
constexpr int kTqmMaxGroups = 16;       // groups of the two-level merge (16 x 16 >= 256)

template <int HD, int SBITS, bool KRAW>
struct TqmCfg {
  // consumer warps; with the producer 3 warps per scheduler (hd <= 128).  A key group of
  // 16 keys belongs to QW warps, each decoding DPW of its dims (at hd 512 four warps of 128
  // dims: the output accumulators of one warp stay at 64 registers)
  static constexpr int NC = HD >= 512 ? 8 : (HD >= 256 ? 4 : 11);
  static constexpr int QW = HD >= 512 ? 4 : 1;  // warps per key group
  static constexpr int KG = NC / QW;            // key groups of a stage
  static constexpr int DPW = HD / QW;           // dims per warp
  static constexpr int BLK = HD < 256 ? HD : 256;  // norm block
  static constexpr int NB = HD / BLK;              // norm blocks per row
  static constexpr int T = KG * 16;                // keys per stage
  static constexpr int CB = HD * SBITS / 8;         // code bytes of a row
  static constexpr int BOXW = CB < 128 ? CB : 128;  // bytes of a TMA box row
  static constexpr int NBOX = CB / BOXW;
  static constexpr int SWM = BOXW == 128 ? 7 : (BOXW == 64 ? 3 : 1);  // swizzled row bits
  static constexpr int KTILE = KRAW ? T * HD * 2 : T * CB;
  static constexpr int VTILE = T * CB;
  // f32 [T][NB] K norms (coded K), then [T][NB] V norms
  static constexpr int NORM_OFF = KTILE + VTILE;
  static constexpr int NNORM = KRAW ? 1 : 2;
  static constexpr int STAGE = (KTILE + VTILE + NNORM * T * NB * 4 + 1023) / 1024 * 1024;
  // the table: 8-bit codes one word per code (bf16 hi | lo << 16); 4-bit codes one 64-bit
  // entry per byte, i.e. per pair of codes (hi pair, lo pair); both one copy per bank
  static constexpr int LEV = 1 << SBITS;  // code levels
  static constexpr int ENT = 256;
  static constexpr int EB = SBITS == 8 ? 4 : 8;  // entry bytes
  static constexpr int TAB = ENT * 32 * EB;
  static constexpr int KS = HD / 16;    // k16 steps of S = Q K^T
  static constexpr int KSW = DPW / 16;  // the steps of one warp
  static constexpr int NTO = DPW / 8;   // n8 tiles of one warp's O
  static constexpr int RS = HD + 4;   // record: O[HD], m, l, pad
  static constexpr int QF = KS * 32 * 16;
  static constexpr int SQ = 8 * HD * 4;  // the rotated queries (f32), later the merged O
  // the key groups' partial scores: [2 stage parities][KG][QW][32 lanes] float4, then the
  // warps' stage flags [2][KG][QW] int
  static constexpr int XFL = 2 * KG * QW * 32 * 16;
  static constexpr int XCH = QW > 1 ? XFL + (2 * KG * QW * 4 + 15) / 16 * 16 : 0;
  static constexpr int FIXED = TAB + QF + SQ + XCH + 256;
  static_assert(LEV * 4 <= QF, "the code words fit in the fragment area");
  static constexpr int NS0 = (kTqmSmemBudget - FIXED) / STAGE;
  static constexpr int NS = NS0 < kTqmMaxStages ? NS0 : kTqmMaxStages;
  static constexpr size_t SMEM = 1024 + (size_t)NS * STAGE + FIXED;
  static constexpr int THREADS = (NC + 1) * 32;
  static_assert(NS >= 2, "two stages at least");
  static_assert(KG * 8 * RS * 4 <= NS * STAGE, "the groups' records fit in the stages");
  static_assert(QW == 1 || !KRAW, "raw keys: one warp per key group");
  static_assert(DPW % (SBITS == 8 ? 32 : 64) == 0 && BLK % DPW == 0,
                "a warp's dims: whole code groups inside one norm block");
  static_assert(8 * kTqmMaxSplits * 4 <= NS * STAGE, "the merge weights fit in the stages");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// shared address of byte `byte` (a multiple of 4) of key row `row` in a code tile: boxes of
// BOXW bytes x T rows one after another, each written by TMA with the swizzle of its width
// (the 16-byte chunk index XOR the row bits above the 128-byte line)
template <class Cfg>
__device__ __forceinline__ uint32_t code_addr(uint32_t tile, int row, int byte) {
  const int box = byte / Cfg::BOXW, bb = byte - box * Cfg::BOXW;
  const uint32_t lin = (uint32_t)(row * Cfg::BOXW + bb);
  return tile + (uint32_t)(box * (Cfg::T * Cfg::BOXW)) + (lin ^ (((lin >> 7) & Cfg::SWM) << 4));
}

// raw bf16 K tile (hybrid layout): boxes of 64 dims (128 B) x T rows, 128-byte swizzle
template <class Cfg>
__device__ __forceinline__ uint32_t raw_addr(uint32_t tile, int row, int chunk) {
  const int box = chunk >> 3, c = chunk & 7;
  return tile + (uint32_t)(box * (Cfg::T * 128) + row * 128 + ((c ^ (row & 7)) << 4));
}

// The dim that k index (2t + e) (hh = 0) or (2t + 8 + e) (hh = 1) of k16 step ks stands
// for.  Coded K: the code word a lane reads holds adjacent dims (4 per 8-bit word, 8 per
// 4-bit word); raw K: the natural order, as ldmatrix delivers it.
template <int SBITS, bool KRAW>
__device__ __forceinline__ int qdim(int ks, int t, int hh, int e) {
  if (KRAW) return 16 * ks + 2 * t + 8 * hh + e;
  if (SBITS == 8) return 16 * ks + 4 * t + 2 * hh + e;
  return 32 * (ks >> 1) + 8 * t + 4 * (ks & 1) + 2 * hh + e;
}

// the table word (bf16 hi | lo << 16) of code c for this lane
__device__ __forceinline__ uint32_t tab_ld(uint32_t tab_lane, uint32_t c) {
  return lds32(tab_lane + (c << 7));
}
// the table word of byte j of w (an 8-bit code): the byte moved down by one permute
__device__ __forceinline__ uint32_t tab_ld8(uint32_t tab_lane, uint32_t w, int j) {
  return tab_ld(tab_lane, __byte_perm(w, 0u, 0x4440u | (uint32_t)j));
}
// the 4-bit table entry of byte j of w (two codes: the low nibble first) for this lane:
// .x = (hi, hi), .y = (lo, lo); entries 256 bytes apart
__device__ __forceinline__ uint2 pair_ld(uint32_t tab_lane8, uint32_t w, int j) {
  const uint32_t off = __byte_perm(w, 0u, 0x4404u | ((uint32_t)j << 4));  // byte j << 8
  uint2 v;
  asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(tab_lane8 + off));
  return v;
}
// operand registers of two adjacent k (or two keys) from their table words
__device__ __forceinline__ uint32_t hi_pair(uint32_t e0, uint32_t e1) {
  return __byte_perm(e0, e1, 0x5410);
}
__device__ __forceinline__ uint32_t lo_pair(uint32_t e0, uint32_t e1) {
  return __byte_perm(e0, e1, 0x7632);
}

// S += [hi(q); lo(q)] (hi(c) + lo(c)) for one k16 step of 8-bit codes: bytes 0, 1 of w are
// k = 2t, 2t + 1 (b0), bytes 2, 3 are k = 2t + 8, 2t + 9 (b1) (hi and lo terms in separate
// accumulators: two dependency chains of half the length)
__device__ __forceinline__ void score_step8(float (&sh)[4], float (&sl)[4], const uint32_t (&A)[4],
                                            uint32_t tab, uint32_t w) {
  const uint32_t e0 = tab_ld8(tab, w, 0), e1 = tab_ld8(tab, w, 1);
  const uint32_t e2 = tab_ld8(tab, w, 2), e3 = tab_ld8(tab, w, 3);
  mma_bf16(sh, A, hi_pair(e0, e1), hi_pair(e2, e3));
  mma_bf16(sl, A, lo_pair(e0, e1), lo_pair(e2, e3));
}

// O_tile += [hi(p); lo(p)] (hi(v) + lo(v)) for 8-bit codes: byte j of the words of keys 2t,
// 2t + 1 (b0) and 2t + 8, 2t + 9 (b1) is the lane's column of n8 tile j
__device__ __forceinline__ void pv_tile8(float (&o)[4], const uint32_t (&PA)[4], uint32_t tab,
                                         uint32_t wA, uint32_t wB, uint32_t wC, uint32_t wD, int j) {
  const uint32_t eA = tab_ld8(tab, wA, j), eB = tab_ld8(tab, wB, j);
  const uint32_t eC = tab_ld8(tab, wC, j), eD = tab_ld8(tab, wD, j);
  mma_bf16(o, PA, hi_pair(eA, eB), hi_pair(eC, eD));
  mma_bf16(o, PA, lo_pair(eA, eB), lo_pair(eC, eD));
}

__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// the mbarrier gets this thread's arrival once its earlier cp.async copies have landed
// (counted in the barrier's expected arrivals)
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

template <int NT>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

template <int HD, int SBITS, bool KRAW>
__global__ void __launch_bounds__(TqmCfg<HD, SBITS, KRAW>::THREADS, 1)
    tq_attn_mma_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const TqAttnArgs a) {
  using Cfg = TqmCfg<HD, SBITS, KRAW>;
  constexpr int NC = Cfg::NC, T = Cfg::T, NS = Cfg::NS, RS = Cfg::RS;
  constexpr int NCT = NC * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* stages = smem;
  uint32_t* s_tab = reinterpret_cast<uint32_t*>(smem + NS * Cfg::STAGE);
  uint4* qf = reinterpret_cast<uint4*>(smem + NS * Cfg::STAGE + Cfg::TAB);
  float* s_q = reinterpret_cast<float*>(smem + NS * Cfg::STAGE + Cfg::TAB + Cfg::QF);
  float4* s_x = reinterpret_cast<float4*>(smem + NS * Cfg::STAGE + Cfg::TAB + Cfg::QF + Cfg::SQ);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * Cfg::STAGE + Cfg::TAB + Cfg::QF +
                                               Cfg::SQ + Cfg::XCH);
  uint64_t* empty = full + NS;
  int* s_flags = reinterpret_cast<int*>(empty + NS);  // [0] abort, [1] issued, [2] last

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.nh / a.nkv;
  const int unit = blockIdx.x / a.splits, split = blockIdx.x - unit * a.splits;
  const int b = unit / a.nkv, kvh = unit - b * a.nkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1 + 32);  // the TMA issue + the producer lanes' norm copies
      mbar_init(&empty[i], NC);
    }
    s_flags[0] = 0;
    s_flags[1] = 0;
    fence_barrier_init();
  }
  if (warp == NC && lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp < NC) {
    // the decode table (the format's centroids never change: read before the dependency
    // wait); each centroid loaded once, then copied to its bank slots
    uint32_t* s_cw = reinterpret_cast<uint32_t*>(qf);
    for (int c = threadIdx.x; c < Cfg::LEV; c += NCT) {
      const float f = c < a.levels ? __ldg(a.centroids + c) : 0.f;
      __nv_bfloat16 h, l;
      split_bf16(f, h, l);
      s_cw[c] = pack_bf2(h, l);
    }
    consumer_bar<NCT>();
    if (SBITS == 8) {
      for (int i = threadIdx.x; i < 256 * 32; i += NCT) s_tab[i] = s_cw[i >> 5];
    } else {
      for (int i = threadIdx.x; i < 256 * 32; i += NCT) {
        const uint32_t v = (uint32_t)(i >> 5);
        const uint32_t e0 = s_cw[v & 15u], e1 = s_cw[v >> 4];
        reinterpret_cast<uint2*>(s_tab)[i] = make_uint2(hi_pair(e0, e1), lo_pair(e0, e1));
      }
    }
  }
  __syncthreads();  // the table is written; the code words are no longer read
  // Programmatic dependent launch: q and the codes come from earlier kernels
  pdl_wait();

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
  if (bad && threadIdx.x == 0 && split == 0 && a.err) atomicOr(a.err, 2u);
  const int k_begin = lo + split * a.chunk;
  int k_end = k_begin + a.chunk;
  if (k_end > hi + 1) k_end = hi + 1;
  const int nkeys = bad ? 0 : (k_end > k_begin ? k_end - k_begin : 0);
  const int ntiles = (nkeys + T - 1) / T;
  const int row0 = unit * a.C + k_begin;  // TMA row of the chunk's first key

  float* part = a.part + ((size_t)unit * a.splits + split) * 8 * RS;

  if (warp == NC) {
    // ------------------------------------------------------------- producer
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NS;
      if (i >= NS && !mbar_wait(&empty[st], ((i / NS) - 1) & 1, a.err, &s_flags[0])) {
        atomicExch(&s_flags[0], 1);
        break;
      }
      if (*(volatile int*)&s_flags[0]) break;
      uint8_t* sb = stages + st * Cfg::STAGE;
      const int y = row0 + i * T;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[st], Cfg::KTILE + Cfg::VTILE);
        if (KRAW) {
#pragma unroll
          for (int j = 0; j < HD / 64; ++j) tma_load_2d(sb + j * T * 128, &tmk, &full[st], 64 * j, y);
        } else {
#pragma unroll
          for (int j = 0; j < Cfg::NBOX; ++j)
            tma_load_2d(sb + j * T * Cfg::BOXW, &tmk, &full[st], j * Cfg::BOXW, y);
        }
#pragma unroll
        for (int j = 0; j < Cfg::NBOX; ++j)
          tma_load_2d(sb + Cfg::KTILE + j * T * Cfg::BOXW, &tmv, &full[st], j * Cfg::BOXW, y);
      }
      // the norms of the stage's keys (past the chunk: its last key, never used)
      float* nd = reinterpret_cast<float*>(sb + Cfg::NORM_OFF);
      const int kb0 = k_begin + i * T;
      constexpr int NB = Cfg::NB;
      for (int e = lane; e < T * NB; e += 32) {
        const int j = e / NB, bk = e - j * NB;
        const int key = kb0 + j < k_end ? kb0 + j : k_end - 1;
        const size_t r = ((size_t)unit * a.C + key) * NB + bk;
        if (!KRAW) cp_async_4(nd + e, a.k_norms + r);
        cp_async_4(nd + (KRAW ? 0 : T * NB) + e, a.v_norms + r);
      }
      cp_async_arrive_noinc(&full[st]);
      issued = i + 1;
    }
    if (lane == 0) s_flags[1] = issued;
  } else {
    // ------------------------------------------------------------- consumers
    const int ctid = threadIdx.x;
    auto csync = []() { consumer_bar<NCT>(); };
    {
      // the queries (scaled, and sign-multiplied for coded keys): 16-byte loads, all of a
      // thread's in flight at once
      constexpr int Q4 = HD / 4, QN = (8 * Q4 + NCT - 1) / NCT;
      float4 qv[QN], sg[QN];
#pragma unroll
      for (int k = 0; k < QN; ++k) {
        const int e = ctid + k * NCT, ee = e < 8 * Q4 ? e : 8 * Q4 - 1;
        const int h = ee / Q4, i4 = ee - h * Q4;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        qv[k] = h < G ? __ldg(reinterpret_cast<const float4*>(a.q + ((size_t)b * a.nh + kvh * G + h) * HD) + i4) : z;
        sg[k] = KRAW ? make_float4(1.f, 1.f, 1.f, 1.f) : __ldg(reinterpret_cast<const float4*>(a.signs) + i4);
      }
#pragma unroll
      for (int k = 0; k < QN; ++k) {
        const int e = ctid + k * NCT;
        if (e < 8 * Q4) {
          float4 r;
          r.x = qv[k].x * a.qscale;
          r.y = qv[k].y * a.qscale;
          r.z = qv[k].z * a.qscale;
          r.w = qv[k].w * a.qscale;
          if (!KRAW) {
            r.x *= sg[k].x;
            r.y *= sg[k].y;
            r.z *= sg[k].z;
            r.w *= sg[k].w;
          }
          reinterpret_cast<float4*>(s_q)[e] = r;
        }
      }
    }
    csync();
    if (!KRAW) {  // the query in the keys' rotated domain: one warp per head
      for (int r = warp; r < G * Cfg::NB; r += NC) tq_fwht_warp<Cfg::BLK>(s_q + r * Cfg::BLK, lane);
      csync();
    }
    // query fragments: A rows 0..G-1 = hi(q), rows 8..8+G-1 = lo(q), k in the codes' order
    for (int ks = warp; ks < Cfg::KS; ks += NC) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (g < G) {
        __nv_bfloat16 h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          split_bf16(s_q[g * HD + qdim<SBITS, KRAW>(ks, t, k >> 1, k & 1)], h[k], l[k]);
        w[0] = pack_bf2(h[0], h[1]);
        w[1] = pack_bf2(l[0], l[1]);
        w[2] = pack_bf2(h[2], h[3]);
        w[3] = pack_bf2(l[2], l[3]);
      }
      qf[ks * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    csync();

    float m = -INFINITY, l = 0.f;
    float o[Cfg::NTO][4];
#pragma unroll
    for (int i = 0; i < Cfg::NTO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const uint32_t tab = smem_u32(s_tab) + lane * Cfg::EB;
    const uint32_t stage_base = smem_u32(stages);
    const int kgp = warp / Cfg::QW, qd = warp - kgp * Cfg::QW;  // key group, dim quarter
    const int krow = kgp * 16;
    constexpr int NB = Cfg::NB, DPW = Cfg::DPW;
    const int blkw = qd * DPW / Cfg::BLK;  // the norm block of the warp's dims

    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NS;
      // a warp of a key group with partners leaves the loop only together with them, after
      // the group's barrier of the stage (a warp left alone at that barrier would wait for
      // ever); a failed wait still marks the stage bad
      bool ok = !*(volatile int*)&s_flags[0];
      if (ok && !mbar_wait(&full[st], (i / NS) & 1, a.err, &s_flags[0])) {
        atomicExch(&s_flags[0], 1);
        ok = false;
      }
      if (Cfg::QW == 1 && !ok) break;
      const uint32_t kb = stage_base + st * Cfg::STAGE;
      const uint32_t vb = kb + Cfg::KTILE;
      const float* nrm = reinterpret_cast<const float*>(stages + st * Cfg::STAGE + Cfg::NORM_OFF);

      // S = Q K^T for 16 keys: n8 tiles of keys krow + g (s0) and krow + 8 + g (s1)
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};  // lo(c) terms
      if constexpr (KRAW) {
#pragma unroll
        for (int ks = 0; ks < Cfg::KS; ++ks) {
          const uint4 qa = qf[ks * 32 + lane];
          const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
          const int mrow = krow + ((lane >> 4) << 3) + (lane & 7);
          const int mchunk = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(raw_addr<Cfg>(kb, mrow, mchunk), b0, b1, b2, b3);
          mma_bf16(s0, A, b0, b1);
          mma_bf16(s1, A, b2, b3);
        }
      } else if constexpr (SBITS == 8) {
#pragma unroll
        for (int kw = 0; kw < Cfg::KSW; ++kw) {
          const int ks = qd * Cfg::KSW + kw;
          const uint32_t w0 = lds32(code_addr<Cfg>(kb, krow + g, 16 * ks + 4 * t));
          const uint32_t w1 = lds32(code_addr<Cfg>(kb, krow + 8 + g, 16 * ks + 4 * t));
          const uint4 qa = qf[ks * 32 + lane];
          const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
          score_step8(s0, u0, A, tab, w0);
          score_step8(s1, u1, A, tab, w1);
        }
      } else {
        // byte j of a code word = the codes of k = 2t, 2t + 1 (j even) or 2t + 8, 2t + 9
        // (j odd) of k16 step 2 mw + j / 2: one table entry gives both operand words
#pragma unroll
        for (int mx = 0; mx < DPW / 32; ++mx) {
          const int mw = qd * (DPW / 32) + mx;
          const uint32_t w0 = lds32(code_addr<Cfg>(kb, krow + g, 16 * mw + 4 * t));
          const uint32_t w1 = lds32(code_addr<Cfg>(kb, krow + 8 + g, 16 * mw + 4 * t));
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint4 qa = qf[(2 * mw + half) * 32 + lane];
            const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
            const uint2 a0 = pair_ld(tab, w0, 2 * half), a1 = pair_ld(tab, w0, 2 * half + 1);
            const uint2 c0 = pair_ld(tab, w1, 2 * half), c1 = pair_ld(tab, w1, 2 * half + 1);
            mma_bf16(s0, A, a0.x, a1.x);
            mma_bf16(u0, A, a0.y, a1.y);
            mma_bf16(s1, A, c0.x, c1.x);
            mma_bf16(u1, A, c0.y, c1.y);
          }
        }
      }
      // logits of head g for local keys krow + {2t, 2t+1, 8+2t, 9+2t} (hi row + lo row),
      // times the keys' norms
      float sv[4] = {(s0[0] + s0[2]) + (u0[0] + u0[2]), (s0[1] + s0[3]) + (u0[1] + u0[3]),
                     (s1[0] + s1[2]) + (u1[0] + u1[2]), (s1[1] + s1[3]) + (u1[1] + u1[3])};
      const int kl0 = krow + 2 * t;
      const int kidx0 = k_begin + i * T + kl0;
      bool valid[4];
#pragma unroll
      if constexpr (Cfg::QW > 1) {
        // the key group's warps hold the partial sums of their dims: exchange them (the
        // buffer of this stage's parity: a warp writes it again two stages later, after the
        // group's barrier of the stage between), then add each norm block's parts
        int* s_ok = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(s_x) + Cfg::XFL);
        const int xs = ((i & 1) * Cfg::KG + kgp) * Cfg::QW;
        s_x[(xs + qd) * 32 + lane] = make_float4(sv[0], sv[1], sv[2], sv[3]);
        if (lane == 0) s_ok[xs + qd] = ok ? 1 : 0;
        asm volatile("bar.sync %0, %1;" ::"r"(2 + kgp), "n"(Cfg::QW * 32) : "memory");
        bool all_ok = true;
#pragma unroll
        for (int q = 0; q < Cfg::QW; ++q) all_ok = all_ok && s_ok[xs + q] != 0;
        if (!all_ok) break;  // the same decision in every warp of the group
        float blk[NB][4];
#pragma unroll
        for (int bk = 0; bk < NB; ++bk) blk[bk][0] = blk[bk][1] = blk[bk][2] = blk[bk][3] = 0.f;
#pragma unroll
        for (int q = 0; q < Cfg::QW; ++q) {
          const float4 x = s_x[(((i & 1) * Cfg::KG + kgp) * Cfg::QW + q) * 32 + lane];
          const int bk = q * DPW / Cfg::BLK;
          blk[bk][0] += x.x;
          blk[bk][1] += x.y;
          blk[bk][2] += x.z;
          blk[bk][3] += x.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dk = (e & 1) + ((e >> 1) << 3);
          float sc = 0.f;
#pragma unroll
          for (int bk = 0; bk < NB; ++bk) sc += blk[bk][e] * nrm[(kl0 + dk) * NB + bk];
          sv[e] = sc;
        }
      }
      for (int e = 0; e < 4; ++e) {
        const int dk = (e & 1) + ((e >> 1) << 3);
        float s = sv[e];
        if (!KRAW && Cfg::QW == 1) s *= nrm[kl0 + dk];
        if (a.cap_log2 != 0.f) s = a.cap_log2 * tanhf(s);
        valid[e] = kidx0 + dk < k_end;
        sv[e] = valid[e] ? s : -INFINITY;
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
      if (__any_sync(0xffffffffu, corr != 1.f)) {  // most tiles leave every head's max
#pragma unroll
        for (int nt = 0; nt < Cfg::NTO; ++nt) {
          o[nt][0] *= corr;
          o[nt][1] *= corr;
          o[nt][2] *= corr;
          o[nt][3] *= corr;
        }
      }
      // P times the V norms as the A operand: row g = hi, row g + 8 = lo; k = the 16 keys
      uint32_t PA[4];
      {
        __nv_bfloat16 h[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dk = (e & 1) + ((e >> 1) << 3);
          const float pv = valid[e] ? p[e] * nrm[(KRAW ? 0 : T * NB) + (kl0 + dk) * NB + blkw] : 0.f;
          split_bf16(pv, h[e], lw[e]);
        }
        PA[0] = pack_bf2(h[0], h[1]);
        PA[1] = pack_bf2(lw[0], lw[1]);
        PA[2] = pack_bf2(h[2], h[3]);
        PA[3] = pack_bf2(lw[2], lw[3]);
      }
      // O += P V: the lane reads keys 2t, 2t+1, 2t+8, 2t+9 at the 4 (8 for 4-bit) adjacent
      // dims of its column; n8 tile j of a group holds the dims base + (4 or 8) col + j
      if constexpr (SBITS == 8) {
#pragma unroll
        for (int gx = 0; gx < DPW / 32; ++gx) {
          const int grp = qd * (DPW / 32) + gx;
          const int byte = grp * 32 + 4 * g;
          const uint32_t wA = lds32(code_addr<Cfg>(vb, krow + 2 * t, byte));
          const uint32_t wB = lds32(code_addr<Cfg>(vb, krow + 2 * t + 1, byte));
          const uint32_t wC = lds32(code_addr<Cfg>(vb, krow + 2 * t + 8, byte));
          const uint32_t wD = lds32(code_addr<Cfg>(vb, krow + 2 * t + 9, byte));
#pragma unroll
          for (int j = 0; j < 4; ++j) pv_tile8(o[gx * 4 + j], PA, tab, wA, wB, wC, wD, j);
        }
      } else {
#pragma unroll
        for (int gx = 0; gx < DPW / 64; ++gx) {
          const int grp = qd * (DPW / 64) + gx;
          const int byte = grp * 32 + 4 * g;
          const uint32_t wA = lds32(code_addr<Cfg>(vb, krow + 2 * t, byte));
          const uint32_t wB = lds32(code_addr<Cfg>(vb, krow + 2 * t + 1, byte));
          const uint32_t wC = lds32(code_addr<Cfg>(vb, krow + 2 * t + 8, byte));
          const uint32_t wD = lds32(code_addr<Cfg>(vb, krow + 2 * t + 9, byte));
          // byte k of xe / xo: the codes of dim 2k / 2k + 1 (of the lane's eight) for keys
          // 2t (low nibble) and 2t + 1; ye / yo the same for keys 2t + 8, 2t + 9
          const uint32_t xe = (wA & 0x0f0f0f0fu) | ((wB << 4) & 0xf0f0f0f0u);
          const uint32_t xo = ((wA >> 4) & 0x0f0f0f0fu) | (wB & 0xf0f0f0f0u);
          const uint32_t ye = (wC & 0x0f0f0f0fu) | ((wD << 4) & 0xf0f0f0f0u);
          const uint32_t yo = ((wC >> 4) & 0x0f0f0f0fu) | (wD & 0xf0f0f0f0u);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint2 b0 = pair_ld(tab, (j & 1) ? xo : xe, j >> 1);
            const uint2 b1 = pair_ld(tab, (j & 1) ? yo : ye, j >> 1);
            mma_bf16(o[gx * 8 + j], PA, b0.x, b1.x);
            mma_bf16(o[gx * 8 + j], PA, b0.y, b1.y);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);

    // ------------------------------------------------- merge the consumer warps
    // every stage has been consumed (or the CTA aborted): reuse the stage buffers
    csync();
    float* red = reinterpret_cast<float*>(stages);  // [key group][8][RS]
    float* mine = red + kgp * 8 * RS;
    if (g < G) {
      if (t == 0 && qd == 0) {
        mine[g * RS + HD] = m;
        mine[g * RS + HD + 1] = l;
      }
#pragma unroll
      for (int nt = 0; nt < Cfg::NTO; ++nt) {
        // columns 2t, 2t + 1 of tile nt: the dims of the permuted order
        int d0, d1;
        if (SBITS == 8) {
          d0 = qd * DPW + (nt >> 2) * 32 + 8 * t + (nt & 3);
          d1 = d0 + 4;
        } else {
          d0 = qd * DPW + (nt >> 3) * 64 + 16 * t + (nt & 7);
          d1 = d0 + 8;
        }
        mine[g * RS + d0] = o[nt][0] + o[nt][2];
        mine[g * RS + d1] = o[nt][1] + o[nt][3];
      }
    }
    csync();
    // per head: the key groups' weights 2^(m_w - M) into the records' pad words, m and l
    // of the CTA's record
    for (int h = ctid; h < G; h += NCT) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < Cfg::KG; ++w) M = fmaxf(M, red[(w * 8 + h) * RS + HD]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < Cfg::KG; ++w) {
        const float f = exp2f(red[(w * 8 + h) * RS + HD] - Mu);
        red[(w * 8 + h) * RS + HD + 2] = f;
        lsum += f * red[(w * 8 + h) * RS + HD + 1];
      }
      part[h * RS + HD] = M;
      part[h * RS + HD + 1] = lsum;
    }
    csync();
    // O = sum_w f_w O_w, the groups in order, four dims a thread
    constexpr int Q4 = HD / 4;
    for (int e = ctid; e < G * Q4; e += NCT) {
      const int h = e / Q4, d4 = e - h * Q4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < Cfg::KG; ++w) {
        const float f = red[(w * 8 + h) * RS + HD + 2];
        const float4 x = reinterpret_cast<const float4*>(red + (w * 8 + h) * RS)[d4];
        acc.x += f * x.x;
        acc.y += f * x.y;
        acc.z += f * x.z;
        acc.w += f * x.w;
      }
      reinterpret_cast<float4*>(part + h * RS)[d4] = acc;
    }
  }

  // drain: every copy this CTA issued has landed before it may exit or reuse the stages
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = s_flags[1];
    for (int st = 0; st < NS && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / NS) * NS;
      mbar_wait(&full[st], (last / NS) & 1, a.err);
    }
  }

  // ------------------------------------------------- the merge, in two levels
  // the last chunk of each group folds the group's records; the last group of the unit
  // merges the folds and rotates back (with one group, it merges the chunks themselves)
  const int ng = (a.splits + a.group - 1) / a.group;
  const int grp = split / a.group, g0 = grp * a.group;
  const int gn = a.splits - g0 < a.group ? a.splits - g0 : a.group;
  float* wsm = reinterpret_cast<float*>(stages);
  __threadfence();
  __syncthreads();
  if (ng > 1) {
    int* t1 = a.ticket1 + unit * kTqmMaxGroups + grp;
    if (threadIdx.x == 0) s_flags[2] = atomicAdd(t1, 1) == gn - 1;
    __syncthreads();
    if (!s_flags[2]) return;
    __threadfence();
    if (threadIdx.x == 0) *t1 = 0;
    tq_fold_records<HD, Cfg::THREADS>(a.part + ((size_t)unit * a.splits + g0) * 8 * RS, gn, G, wsm,
                        a.part1 + ((size_t)unit * kTqmMaxGroups + grp) * 8 * RS);
    __threadfence();
    __syncthreads();
  }
  // the unit's ticket counts the folds (two levels) or the chunks (one)
  const int arrivals = ng > 1 ? ng : a.splits;
  if (threadIdx.x == 0) s_flags[2] = atomicAdd(a.ticket + unit, 1) == arrivals - 1;
  __syncthreads();
  if (!s_flags[2]) return;
  __threadfence();
  if (threadIdx.x == 0) a.ticket[unit] = 0;
  const float* up = ng > 1 ? a.part1 + (size_t)unit * kTqmMaxGroups * 8 * RS
                           : a.part + (size_t)unit * a.splits * 8 * RS;
  tq_merge_records<HD, Cfg::THREADS>(up, ng > 1 ? ng : a.splits, G, wsm, s_q, a.signs,
                       a.o + ((size_t)b * a.nh + kvh * G) * HD);
}

template <int HD, int SBITS, bool KRAW>
cudaError_t launch_t(const TqAttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                     cudaStream_t s) {
  using Cfg = TqmCfg<HD, SBITS, KRAW>;
  auto kern = tq_attn_mma_kernel<HD, SBITS, KRAW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Cfg::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

template <int HD>
cudaError_t launch_hd(const TqAttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                      int sbits, bool kraw, int grid, cudaStream_t s) {
  if (sbits == 8)
    return kraw ? launch_t<HD, 8, true>(a, tk, tv, grid, s) : launch_t<HD, 8, false>(a, tk, tv, grid, s);
  return kraw ? launch_t<HD, 4, true>(a, tk, tv, grid, s) : launch_t<HD, 4, false>(a, tk, tv, grid, s);
}

}  // namespace

bool tq_mma_supported(int hd, int sbits, bool kraw) {
  return (hd == 64 || hd == 128 || hd == 256 || (hd == 512 && !kraw)) && (sbits == 4 || sbits == 8);
}
int tq_mma_keys_per_stage(int hd) { return hd >= 512 ? 32 : (hd >= 256 ? 64 : 176); }
int tq_mma_threads(int hd) { return hd >= 512 ? 288 : (tq_mma_keys_per_stage(hd) / 16 + 1) * 32; }

cudaError_t launch_tq_attn_mma(const TqAttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                               int hd, int sbits, bool kraw, int grid, cudaStream_t s) {
  if (a.splits > kTqmMaxSplits || a.group < 1 ||
      (a.splits + a.group - 1) / a.group > kTqmMaxGroups)
    return cudaErrorInvalidValue;
  if (hd == 64) return launch_hd<64>(a, tk, tv, sbits, kraw, grid, s);
  if (hd == 128) return launch_hd<128>(a, tk, tv, sbits, kraw, grid, s);
  if (hd == 256) return launch_hd<256>(a, tk, tv, sbits, kraw, grid, s);
  if (kraw) return cudaErrorInvalidValue;  // raw keys at hd 512: the CUDA-core kernel
  return sbits == 8 ? launch_t<512, 8, false>(a, tk, tv, grid, s)
                    : launch_t<512, 4, false>(a, tk, tv, grid, s);
}

}  // namespace hfa
