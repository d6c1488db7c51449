// k_verify.cu -- the multi-token verify block of one layer (L <= 16 tokens, batch 1).
//
// gemma4/model.rs names the dense tree-verify entry of the full layer; the block form is
// the one dflash/forward.rs builds for its drafter: input norm and projections of all L
// rows, per-head norms, RoPE at positions base .. base+L-1, all L K/V rows appended to
// the cache, attention of every row over the cache (causal inside the block), o_proj,
// residual.  With bf16 weights the projections are dense contractions [L, H] x [H, N]:
//
//  * verify_gemm_kernel (tcgen05): swap-AB -- the weight rows are the MMA's M = 128, the
//    activations its N = 32 (16 tokens x fp32 split into bf16 hi and lo, so the product
//    keeps ~16 bits of the activation), K in 64-element stages.  A producer thread
//    streams 128x64 weight tiles -- repacked at layer creation into the 128-byte-swizzled
//    shared-memory image, so each is one 16 KB bulk copy -- with the matching 4 KB
//    activation chunk into a 10-stage ring; one thread issues tcgen05.mma into a 128x32
//    fp32 TMEM accumulator and releases stages with tcgen05.commit.  The k-splits of a
//    row tile add their partial sums through global memory as tagged entries (QKV: one
//    cooperative launch, a CTA on every SM) or, in a cluster, through distributed shared
//    memory (o_proj); then the head epilogue (norms, RoPE, KV append; the query also as the
//    attention's operand image) or the residual epilogue runs on the complete rows.
//  * attn_verify_tc_kernel (head_dim 128, tcgen05): one CTA per (KV head, key chunk);
//    S = Qx K^T and O += Px Vt on the tensor cores with TMEM accumulators, the online
//    softmax of each query split over the four threads that hold its two TMEM rows.
//  * attn_verify_kernel (head_dim 64, 256; mma.sync): one CTA per (KV head, key chunk); a
//    TMA producer warp streams K and V tiles, each consumer warp owns 8 query rows (bf16
//    hi/lo in MMA rows g and g + 8) and takes every 64-key stage in one online-softmax
//    update, with the causal / window mask of its rows.
//  * attn_verify_hy_kernel (head_dim 512): the scores on mma.sync with each warp's query
//    fragments in registers, O += P V on tcgen05 into a 512-column TMEM accumulator.
//    The attention kernels write one (O, m, l) record per query row and CTA.
//  * attn_verify_merge_kernel: the records of a KV head's chunks combined, a few query
//    rows per CTA, into the f32 output and the o_proj activation operand.
#include <cooperative_groups.h>
#include <stdio.h>

#include "hfa_common.cuh"
#include "hfa_finish.cuh"
#include "hfa_gemv.cuh"
#include "hfa_internal.h"
#include "hfa_verify.h"

namespace hfa {

// ------------------------------------------------------------------ GEMM (tcgen05)
// Writes columns [8e, 8e + 8) of activation row t into the operand: bf16 hi in row t,
// bf16 lo in row 16 + t of chunk e / 8, 16-byte group (e % 8) XOR (row % 8).
__device__ __forceinline__ void store_bop_group(uint8_t* bops, int t, int e, const float (&v)[8]) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat16 h0, l0, h1, l1;
    split_bf16(v[2 * i], h0, l0);
    split_bf16(v[2 * i + 1], h1, l1);
    hw[i] = pack_bf2(h0, h1);
    lw[i] = pack_bf2(l0, l1);
  }
  uint8_t* chunk = bops + (size_t)(e >> 3) * (32 * 128);
  const int c16 = e & 7, rh = t, rl = 16 + t;
  *reinterpret_cast<uint4*>(chunk + rh * 128 + ((c16 ^ (rh & 7)) << 4)) =
      make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(chunk + rl * 128 + ((c16 ^ (rl & 7)) << 4)) =
      make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

constexpr int kVM = 128;         // weight rows per CTA = MMA M
constexpr int kVN = 32;          // MMA N: 16 tokens x (hi, lo)
constexpr int kVK = 64;          // K elements per stage (one 128-byte swizzled row)
constexpr int kVStages = 10;     // ring depth: 200 KB of copies in flight per SM
constexpr int kAStageBytes = kVM * kVK * 2;  // 16 KB weight tile
constexpr int kBChunkBytes = kVN * kVK * 2;  // 4 KB activation chunk
constexpr int kVStageBytes = kAStageBytes + kBChunkBytes;
constexpr int kVTableBytes = 3 * 512 * 4;  // QKV epilogue: w_q, w_k, RoPE table (hd <= 512)
constexpr size_t kVGemmSmem = 1024 + (size_t)kVStages * kVStageBytes + 256 + kVTableBytes;

struct VGemmArgs {
  GemvArgs g;        // epilogue arguments (norms, RoPE, caches, residual, ...)
  const uint8_t* wt;    // weights as 16 KB tiles [rows / 128][K / 64] (launch_repack_bf16_tiles)
  const uint8_t* bops;  // activation operand, [K / 64 chunks][32 rows][128 B], swizzled
  int rows;          // output features
  int K;             // input features
  int chunks;        // K / 64
  int splits;        // k-splits per row tile
  int tpc;           // row tiles per cluster: hd / 128 for QKV heads wider than a tile, else 1
  int tile_base;     // first row tile (the context rows start at the key rows' tile)
  // With gpart set, the k-splits add their partial sums through global memory instead of a
  // cluster: CTA i stores [16 tokens][128 rows] f32 as 8-byte entries (value | launch tag)
  // at gpart + i * 2048, and the CTAs of a group (the tpc x splits consecutive CTAs that a
  // cluster would hold) poll one another's entries.  gctr counts launches x grid (the tags).
  // The GEMMs that share gpart keep apart tag spaces (tag_lane 0 or 1: tags 2 n + 2 +
  // tag_lane for the n-th launch), so no launch can take an entry another GEMM left.
  unsigned long long* gpart;
  unsigned long long* gctr;
  uint32_t tag_lane;
};

// Activation operand of the verify GEMMs, built once per call: row t of the block
// (t < L; zero rows otherwise), normalised by its input RMSNorm (QKV mode), split into
// bf16 hi (operand row t) and lo (row 16 + t), written chunk by chunk (64 columns,
// 32 rows of 128 B) in the 128-byte swizzled order the tensor cores read.
// One CTA per operand row pair t.
__global__ void __launch_bounds__(256) verify_prep_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const float* __restrict__ w_in,
                                                         float eps, int L, int K,
                                                         uint8_t* __restrict__ bops) {
  __shared__ float s_red[8];
  const int t = blockIdx.x;
  const int ngroups = K / 8;
  if (t < L)  // the input row into L2 while the previous kernel finishes
    for (int e = threadIdx.x; e < K / 64; e += blockDim.x) prefetch_l2(x + (size_t)t * K + e * 64);
  pdl_wait();
  float inv = 0.f;
  if (t < L) {
    float ss = 0.f;
    for (int e = threadIdx.x; e < ngroups; e += blockDim.x) {
      const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)t * K + e * 8);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        ss += f.x * f.x + f.y * f.y;
      }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_red[w];
    inv = w_in ? rsqrtf(tot / K + eps) : 1.f;  // context rows (w_in NULL): no input norm
  }
  for (int e = threadIdx.x; e < ngroups; e += blockDim.x) {
    float v[8];
    if (t < L) {
      const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)t * K + e * 8);
      const float4 one = make_float4(1.f, 1.f, 1.f, 1.f);
      const float4 w0 = w_in ? __ldg(reinterpret_cast<const float4*>(w_in + e * 8)) : one;
      const float4 w1 = w_in ? __ldg(reinterpret_cast<const float4*>(w_in + e * 8 + 4)) : one;
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x * inv * wv[2 * i];
        v[2 * i + 1] = f.y * inv * wv[2 * i + 1];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    store_bop_group(bops, t, e, v);
  }
  pdl_launch_dependents();
}

template <int MODE>
__global__ void __launch_bounds__(128, 1) verify_gemm_kernel(const VGemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* ring = smem;  // stage i: weight tile (16 KB), then activation chunk (4 KB)
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kVStages * kVStageBytes);
  uint64_t* empty = full + kVStages;
  uint64_t* done = empty + kVStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  uint32_t* s_tag = s_tmem + 1;                                  // global reduction: this launch's tag
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 2);
  float* s_tab = reinterpret_cast<float*>(ring + kVStages * kVStageBytes + 256);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = a.tile_base + blockIdx.x / a.splits, sp = blockIdx.x % a.splits;
  const int c0 = a.chunks * sp / a.splits, c1 = a.chunks * (sp + 1) / a.splits;
  const int nch = c1 - c0;
  const int m0 = mt * kVM;
  const int L = a.g.batch;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&full[i], 2);  // one arrival with the weight copy, one with the activation's
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kVN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // the weights never depend on an earlier kernel: fill the ring's weight tiles right
  // away.  The CTA's tiles (m, c0 .. c1 - 1) are one contiguous range, 16 KB a stage;
  // the activation chunks (laid out in shared-memory order by verify_prep_kernel or
  // the attention merge) follow once the previous kernel has finished.
  const uint8_t* wsrc = a.wt + ((size_t)mt * a.chunks + c0) * kAStageBytes;
  const uint8_t* bsrc = a.bops + (size_t)c0 * kBChunkBytes;
  const int npre = nch < kVStages ? nch : kVStages;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < npre; ++i) {
      mbar_arrive_expect_tx(&full[i], kAStageBytes);
      bulk_load(ring + i * kVStageBytes, wsrc + (size_t)i * kAStageBytes, kAStageBytes, &full[i]);
    }
  }
  if (warp == 2) {
    // the lines the epilogue reads (the residual in o_proj mode, the norm weights and
    // RoPE table in QKV mode) into L2, where the weight stream would have left them cold
    if (MODE == kModeOProj) {
      const int R16 = a.g.R * 16;
      for (int q = lane; q < 4 * L; q += 32)
        prefetch_l2(a.g.x + (size_t)(q >> 2) * R16 + m0 + (q & 3) * 32);
    } else {
      // the epilogue's tables into shared memory: w_q, w_k (hd floats each), then the
      // RoPE table (hd / 2 float2); written by this warp, read after the __syncthreads
      // that precedes the epilogue
      const int hd = a.g.hd;
      const float* rg = reinterpret_cast<const float*>(a.g.rope_g);
      for (int i = lane; i < hd; i += 32) {
        s_tab[i] = a.g.w_q[i];
        s_tab[hd + i] = a.g.w_k[i];
        s_tab[2 * hd + i] = rg[i];
      }
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  if (a.gpart && threadIdx.x == 0) {
    // the launch's number: every CTA reads the counter before its own increment and after
    // every increment of the launches before it
    const unsigned long long n = ld_acquire_u64(a.gctr);
    // 0 marks "never written"
    *s_tag = 2u * ((uint32_t)(n / (unsigned long long)gridDim.x) + 1u) + a.tag_lane;
    *s_abort = 0;
    red_release_add_u64(a.gctr, 1ull);
  }

  if (warp == 0 && lane == 0) {
    // ---- producer
    for (int i = 0; i < npre; ++i) {
      mbar_arrive_expect_tx(&full[i], kBChunkBytes);
      bulk_load(ring + i * kVStageBytes + kAStageBytes, bsrc + (size_t)i * kBChunkBytes,
                kBChunkBytes, &full[i]);
    }
    for (int i = npre; i < nch; ++i) {
      const int st = i % kVStages;
      if (!mbar_wait(&empty[st], ((i / kVStages) - 1) & 1, a.g.err)) break;
      uint8_t* stage = ring + st * kVStageBytes;
      mbar_arrive_expect_tx(&full[st], kAStageBytes);
      bulk_load(stage, wsrc + (size_t)i * kAStageBytes, kAStageBytes, &full[st]);
      mbar_arrive_expect_tx(&full[st], kBChunkBytes);
      bulk_load(stage + kAStageBytes, bsrc + (size_t)i * kBChunkBytes, kBChunkBytes, &full[st]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kVM, kVN);
    for (int i = 0; i < nch; ++i) {
      const int st = i % kVStages;
      if (!mbar_wait(&full[st], (i / kVStages) & 1, a.g.err)) break;
      tc_fence_after();
      const uint32_t abase = smem_u32(ring + st * kVStageBytes);
      const uint32_t bbase = abase + kAStageBytes;
#pragma unroll
      for (int kk = 0; kk < kVK / 16; ++kk)
        tc_mma_f16(tmem, smem_desc_sw128(abase + kk * 32), smem_desc_sw128(bbase + kk * 32),
                   idesc, (i | kk) != 0);
      tc_commit(&empty[st]);
    }
    tc_commit(done);
  }
  __syncwarp();
  // ---- epilogue: accumulator rows 32w..32w+31, columns 0..15 hi, 16..31 lo.  The CTA's
  // partial sums go to its own shared memory (the ring is drained: every copy has been
  // consumed by the MMAs that `done` waited for) as [16 tokens][128 rows] f32.
  // agreed across the warp: the tcgen05 loads below are .sync.aligned, and a wait that runs
  // out near its limit could end differently on different lanes
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, a.g.err));
  tc_fence_after();
  float* psum = reinterpret_cast<float*>(ring);
  {
    float hi[16], lo[16];
    if (ok) {
      const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
      tmem_ld_32x32b_x16(taddr, hi);
      tmem_ld_32x32b_x16(taddr + 16, lo);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) psum[t * kVM + 32 * warp + lane] = ok ? hi[t] + lo[t] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kVN);

  // ---- k-split reduction.  The group is the a.splits CTAs of a.tpc consecutive row tiles
  // (rank = tile-in-group * splits + split): a cluster reading distributed shared memory, or
  // (gpart set) CTAs polling one another's tagged entries in global memory.  Each output is
  // summed over the splits in rank order, so the result does not depend on timing.
  namespace cg = cooperative_groups;
  GemvArgs g = a.g;
  if (MODE == kModeQKV) {
    g.w_q = s_tab;
    g.w_k = s_tab + a.g.hd;
    g.rope_g = reinterpret_cast<const float2*>(s_tab + 2 * a.g.hd);
  }
  const int S = a.splits;
  const int cs = S * a.tpc;
  int rank;
  uint32_t tag = 0;
  if (a.gpart) {
    rank = (int)(blockIdx.x % (unsigned)cs);
    tag = *s_tag;
    unsigned long long* mine = a.gpart + (size_t)blockIdx.x * (16 * kVM);
    for (int i = threadIdx.x; i < 16 * kVM; i += blockDim.x) st_tagged(mine + i, psum[i], tag);
  } else {
    rank = (int)cg::this_cluster().block_rank();
    cg::this_cluster().sync();  // every CTA's partial sums are visible
  }
  const unsigned long long* gbase =
      a.gpart ? a.gpart + (size_t)(blockIdx.x - rank) * (16 * kVM) : nullptr;
  // output (row r of the group's rows, token t) summed over the splits
  auto split_sum = [&](int r, int t) -> float {
    float acc = 0.f;
    if (a.gpart) {
      const unsigned long long* p = gbase + (size_t)((r >> 7) * S) * (16 * kVM) + t * kVM + (r & 127);
      for (int c0 = 0; c0 < S; c0 += 4) {
        unsigned long long w[4];
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
          bool ready = true;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[i] = ld_tagged(p + (size_t)(c0 + i < S ? c0 + i : S - 1) * (16 * kVM));
            ready = ready && (uint32_t)(w[i] >> 32) == tag;
          }
          if (ready || *s_abort) break;
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.g.err, kErrWaitTimeout);
            *s_abort = 1;
            break;
          }
          __nanosleep(32);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (c0 + i < S) acc += tagged_value(w[i]);
      }
    } else {
      cg::cluster_group cluster = cg::this_cluster();
      for (int c = 0; c < S; ++c)
        acc += cluster.map_shared_rank(psum, (r >> 7) * S + c)[t * kVM + (r & 127)];
    }
    return acc;
  };
  // rows rb + 32 j (j < nj <= 8) of token t: with gpart, every row's entries polled in one
  // round (one L2 round trip for all of them, not one per row); the splits added in rank
  // order as split_sum does
  auto split_sum_rows = [&](int rb, int t, int nj, float (&v)[8]) {
    if (!a.gpart) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < nj) v[j] = split_sum(rb + 32 * j, t);
      return;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
    for (int c0 = 0; c0 < S; c0 += 4) {
      unsigned long long w[8][4];
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < nj) {
            const int r = rb + 32 * j;
            const unsigned long long* p =
                gbase + (size_t)((r >> 7) * S) * (16 * kVM) + t * kVM + (r & 127);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w[j][i] = ld_tagged(p + (size_t)(c0 + i < S ? c0 + i : S - 1) * (16 * kVM));
          }
        }
        bool ready = true;
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (j < nj) ready = ready && (uint32_t)(w[j][i] >> 32) == tag;
        if (ready || *s_abort) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.g.err, kErrWaitTimeout);
          *s_abort = 1;
          break;
        }
        __nanosleep(32);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (j < nj && c0 + i < S) v[j] += tagged_value(w[j][i]);
    }
  };
  if (MODE == kModeQKV) {
    // items (head, token) of the group's rows, one warp each
    const int hd = a.g.hd;
    const int tile0 = m0 / kVM - (rank / S);  // first row tile of the group
    const int rows0 = tile0 * kVM;
    const int nheads = a.tpc * kVM / hd;
    const int nitems = nheads * L;
    for (int it = rank * 4 + warp; it < nitems; it += cs * 4) {
      const int hl = it / L, t = it - hl * L;
      const int hh = rows0 / hd + hl;
      float u[8];
      split_sum_rows(hl * hd + lane, t, hd < 256 ? hd / 32 : 8, u);
      if (hd == 64) {
        float v[2] = {u[0], u[1]};
        finish_head_row<64>(g, hh, t, v, lane);
      } else if (hd == 128) {
        float v[4] = {u[0], u[1], u[2], u[3]};
        finish_head_row<128>(g, hh, t, v, lane);
      } else if (hd == 256) {
        finish_head_row<256>(g, hh, t, u, lane);
      } else if (hd == 512) {  // the head's second 256 rows in a second polling round
        float u2[8];
        split_sum_rows(hl * hd + 256 + lane, t, 8, u2);
        float v[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[j] = u[j];
          v[8 + j] = u2[j];
        }
        finish_head_row<512>(g, hh, t, v, lane);
      }
    }
  } else {
    // items (token, row) of the tile, a contiguous range per rank
    const int n = L * kVM;
    const int i0 = n * rank / S, i1 = n * (rank + 1) / S;
    for (int i = i0 + (int)threadIdx.x; i < i1; i += blockDim.x) {
      const float y = split_sum(i & 127, i >> 7);
      finish_row_item(g, i >> 7, m0 + (i & 127), y);
    }
  }
  if (!a.gpart) cg::this_cluster().sync();  // no CTA leaves while another reads its shared memory
}

// ------------------------------------------------------------------ block attention
constexpr int kVT = 64;  // keys per stage

struct VAttnArgs {
  const float* q;  // [L, nh, hd]
  int L, nh, nkv, G, C, base, sliding, window;
  int bidir;       // every row sees the whole block (full layers of the drafter)
  float qscale, cap_log2;
  int splits, chunk, klo, khi;  // keys [klo, khi] are read by some row
  float* part;                  // [nkv][splits][64 rows][hd + 4]: O[hd], m, l, pad
  uint8_t* bops;                // o_proj activation operand (see store_bop_group)
  const uint8_t* qx;            // head_dim 128: the scaled q as an MMA operand image per KV head
  float* o;                     // [L, nh, hd]
  unsigned* err;
};

template <int HD>
struct VACfg {
  static constexpr int NS = HD >= 256 ? 2 : 3;  // stages (shared memory budget)
  static constexpr int TILE = kVT * HD * 2;
  static constexpr int STAGE = 2 * TILE;
  static constexpr int KS = HD / 16;
  static constexpr int NTO = HD / 8;
  static constexpr int KB = HD >= 256 ? 16 : 64;  // keys per online-softmax update (registers)
  static constexpr size_t SMEM = 1024 + (size_t)NS * STAGE + 8 * KS * 32 * 16 + 256;
};


template <int HD>
__global__ void __launch_bounds__(288) attn_verify_kernel(const __grid_constant__ CUtensorMap tmk,
                                                          const __grid_constant__ CUtensorMap tmv,
                                                          const VAttnArgs a) {
  using Cfg = VACfg<HD>;
  constexpr int NS = Cfg::NS;
  constexpr int KB = Cfg::KB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* stages = smem;
  uint4* qf = reinterpret_cast<uint4*>(smem + NS * Cfg::STAGE);  // [warp][KS][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * Cfg::STAGE + 8 * Cfg::KS * 512);
  uint64_t* empty = full + NS;
  int* s_flags = reinterpret_cast<int*>(empty + NS);

  const int nc = (blockDim.x >> 5) - 1;  // consumer warps, 8 query rows each
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = blockIdx.x / a.splits, split = blockIdx.x - kvh * a.splits;
  const int NQ = a.L * a.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nc);
    }
    s_flags[0] = 0;
    s_flags[1] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int k_begin = a.klo + split * a.chunk;
  int k_end = k_begin + a.chunk;
  if (k_end > a.khi + 1) k_end = a.khi + 1;
  const int nkeys = k_end > k_begin ? k_end - k_begin : 0;
  const int ntiles = (nkeys + kVT - 1) / kVT;
  const int row0 = kvh * a.C + k_begin;
  constexpr int RS = HD + 4;
  float* part = a.part + ((size_t)kvh * a.splits + split) * 64 * RS;

  if (warp == nc) {
    if (lane == 0) {
      // keys before the block's first position are not written by the QKV kernel: the
      // first stages of such keys are requested before waiting for it
      int issued = 0;
      bool waited = false;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (!waited && (i >= NS || k_begin + (i + 1) * kVT > a.base)) {
          pdl_wait();
          waited = true;
        }
        if (i >= NS && !mbar_wait(&empty[st], ((i / NS) - 1) & 1, a.err, &s_flags[0])) {
          atomicExch(&s_flags[0], 1);
          break;
        }
        if (*(volatile int*)&s_flags[0]) break;
        uint8_t* kt = stages + st * Cfg::STAGE;
        mbar_arrive_expect_tx(&full[st], Cfg::STAGE);
#pragma unroll
        for (int j = 0; j < HD / 64; ++j) {
          tma_load_2d(kt + j * kVT * 128, &tmk, &full[st], 64 * j, row0 + i * kVT);
          tma_load_2d(kt + Cfg::TILE + j * kVT * 128, &tmv, &full[st], 64 * j, row0 + i * kVT);
        }
        issued = i + 1;
      }
      if (!waited) pdl_wait();
      s_flags[1] = issued;
    }
    pdl_launch_dependents();
  } else {
    pdl_wait();
    pdl_launch_dependents();
    // query rows of this warp: q = 8 warp + g  ->  token q / G, head kvh G + q % G
    const int qrow = 8 * warp + g;
    const bool qvalid = qrow < NQ;
    const int tok = qvalid ? qrow / a.G : 0;
    const int limit = a.bidir ? a.base + a.L - 1 : a.base + tok;  // last visible position
    uint4* myq = qf + warp * Cfg::KS * 32;
    for (int ks = 0; ks < Cfg::KS; ++ks) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (qvalid) {
        const float* q =
            a.q + ((size_t)tok * a.nh + kvh * a.G + qrow % a.G) * HD + ks * 16 + 2 * t;
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
      myq[ks * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncwarp();
    float m = -INFINITY, l = 0.f;
    float o[Cfg::NTO][4];
#pragma unroll
    for (int i = 0; i < Cfg::NTO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const uint32_t stage_base = smem_u32(stages);
    // A K or V stage holds HD / 64 boxes of 64 keys x 128 bytes: 16-byte chunk c of key
    // row r sits at (c / 8) * 8 KB + r * 128 + ((c % 8) XOR (r % 8)) * 16.  The lane parts
    // of the ldmatrix addresses (the compile-time row and chunk terms split off): the K
    // fragments read row 16 kg + (lane / 16) 8 + lane % 8,
    // chunk 2 ks + (lane / 8) % 2; the V fragments row 16 kk + ((lane / 8) % 2) 8 + lane % 8,
    // chunk 2 np + lane / 16.  Rows are multiples of 8 apart, so row % 8 = lane % 8 and the
    // XOR term depends on the chunk only through (chunk % 8) / 2: four offsets per operand.
    uint32_t swk[4], swv[4];
    {
      const int l7 = lane & 7;
      const int xk = ((lane >> 3) & 1) ^ l7, xv = (lane >> 4) ^ l7;
      const uint32_t rk = (uint32_t)((((lane >> 4) << 3) + l7) * 128);
      const uint32_t rv = (uint32_t)(((((lane >> 3) & 1) << 3) + l7) * 128);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        swk[j] = rk + (uint32_t)(((2 * j) ^ xk) << 4);
        swv[j] = rv + (uint32_t)(((2 * j) ^ xv) << 4);
      }
    }
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NS;
      if (*(volatile int*)&s_flags[0]) break;
      if (!mbar_wait(&full[st], (i / NS) & 1, a.err, &s_flags[0])) {
        atomicExch(&s_flags[0], 1);
        break;
      }
      const uint32_t kb0 = stage_base + st * Cfg::STAGE;
      const uint32_t vb0 = kb0 + Cfg::TILE;
#pragma unroll 1
      for (int hb = 0; hb < kVT; hb += KB) {
      const int key_lo = k_begin + i * kVT + hb, key_hi = key_lo + KB - 1;
      if (key_lo >= k_end) break;
      // scores of KB keys, KB / 8 independent accumulator chains: n-tile j holds keys
      // 8j .. 8j + 7, rows g (q hi) and g + 8 (q lo)
      float s[KB / 8][4];
#pragma unroll
      for (int j = 0; j < KB / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < Cfg::KS; ++ks) {
        const uint4 qa = myq[ks * 32 + lane];
        const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
#pragma unroll
        for (int kg = 0; kg < KB / 16; ++kg) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb0 + swk[ks & 3] + (uint32_t)((ks >> 2) * (kVT * 128) + (hb + kg * 16) * 128),
                      b0, b1, b2, b3);
          mma_bf16(s[2 * kg], A, b0, b1);
          mma_bf16(s[2 * kg + 1], A, b2, b3);
        }
      }
      // this lane's KB / 4 scores: keys key_lo + 8 (e / 2) + 2 t + e % 2
      constexpr int NE = KB / 4;
      float sc[NE];
#pragma unroll
      for (int j = 0; j < KB / 8; ++j) {
        sc[2 * j] = s[j][0] + s[j][2];
        sc[2 * j + 1] = s[j][1] + s[j][3];
      }
      if (a.cap_log2 != 0.f) {
#pragma unroll
        for (int e = 0; e < NE; ++e) sc[e] = a.cap_log2 * tanhf(sc[e]);
      }
      // keys past the chunk, after this row's position or before its window: masked
      if (!(key_hi < k_end && key_hi <= limit && (!a.sliding || key_lo > limit - a.window))) {
#pragma unroll
        for (int e = 0; e < NE; ++e) {
          const int key = key_lo + 8 * (e >> 1) + 2 * t + (e & 1);
          const bool vis = key < k_end && key <= limit && (!a.sliding || key > limit - a.window);
          if (!vis) sc[e] = -INFINITY;
        }
      }
      float mloc = sc[0];
#pragma unroll
      for (int e = 1; e < NE; ++e) mloc = fmaxf(mloc, sc[e]);
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
      const float m_new = fmaxf(m, mloc);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float corr = ex2_approx(m - m_use);
      m = m_new;
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        sc[e] = ex2_approx(sc[e] - m_use);
        psum += sc[e];
      }
      l = l * corr + psum;
      if (__any_sync(0xffffffffu, corr != 1.f)) {  // else every factor is exactly 1
#pragma unroll
        for (int nt = 0; nt < Cfg::NTO; ++nt) {
          o[nt][0] *= corr;
          o[nt][1] *= corr;
          o[nt][2] *= corr;
          o[nt][3] *= corr;
        }
      }
      // O += P V in 16-key steps; P (hi in rows g, lo in rows g + 8) is the A operand.
      // Rows of the last stage past the chunk may hold any bits (a NaN times a zero
      // weight is NaN): their V elements are zeroed in the fragments.
      const bool tail = key_hi >= k_end;
#pragma unroll
      for (int kk = 0; kk < KB / 16; ++kk) {
        uint32_t PA[4];
        {
          __nv_bfloat16 h[4], lw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16(sc[4 * kk + e], h[e], lw[e]);
          PA[0] = pack_bf2(h[0], h[1]);
          PA[1] = pack_bf2(lw[0], lw[1]);
          PA[2] = pack_bf2(h[2], h[3]);
          PA[3] = pack_bf2(lw[2], lw[3]);
        }
        const int kv0 = key_lo + kk * 16 + 2 * t;
        const uint32_t mlo = (kv0 < k_end ? 0xffffu : 0u) | (kv0 + 1 < k_end ? 0xffff0000u : 0u);
        const uint32_t mhi = (kv0 + 8 < k_end ? 0xffffu : 0u) | (kv0 + 9 < k_end ? 0xffff0000u : 0u);
#pragma unroll
        for (int np = 0; np < Cfg::NTO / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(
              vb0 + swv[np & 3] + (uint32_t)((np >> 2) * (kVT * 128) + (hb + kk * 16) * 128),
              b0, b1, b2, b3);
          if (tail) {
            b0 &= mlo;
            b2 &= mlo;
            b1 &= mhi;
            b3 &= mhi;
          }
          mma_bf16(o[2 * np], PA, b0, b1);
          mma_bf16(o[2 * np + 1], PA, b2, b3);
        }
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (qvalid) {
      float* pr = part + (size_t)qrow * RS;
      if (t == 0) *reinterpret_cast<float2*>(pr + HD) = make_float2(m, l);
#pragma unroll
      for (int nt = 0; nt < Cfg::NTO; ++nt)
        *reinterpret_cast<float2*>(pr + nt * 8 + 2 * t) =
            make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = s_flags[1];
    for (int st = 0; st < NS && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / NS) * NS;
      mbar_wait(&full[st], (last / NS) & 1, a.err);
    }
  }
}

// ------------------------------------------------------------------ block attention (tcgen05)
// The same records as attn_verify_kernel, for head_dim 128, with both products on the
// 5th-generation tensor cores.  Per CTA (KV head, key chunk) and 64-key stage i:
//   S_i = Qx K^T   M = 128 rows (queries 0..63 as bf16 hi, then the same queries as lo),
//                  N = 64 keys, K = 128: the score of query q is S[q] + S[q + 64];
//                  two TMEM buffers, so S_{i+1} is computed while stage i's softmax runs;
//   O  += Px Vt    M = 128 rows (P hi for rows 0..63, P lo for 64..127), N = 128 dims,
//                  K = 64 keys, accumulated in TMEM; Vt is the stage's V transposed in
//                  shared memory.  Px and Vt are double-buffered, so the next stage's
//                  softmax does not wait for this MMA.  Query q's O is O[q] + O[q + 64].
// Eight consumer warps: warps w and w + 4 share TMEM lane quadrant w (rows 32w .. 32w+31),
// one per half of the columns.  The four threads of query q (rows q and q + 64, two
// column halves) split the stage's keys 16 each, exchanging score parts and maxima through
// shared memory, and each writes P (hi and lo) for its keys; the warps also transpose V
// (ldmatrix + stmatrix.trans, keys past the chunk zeroed).  When a query's running
// maximum moves, its O rows are rescaled in TMEM before the next O += P V.  One thread of
// warp 8 streams K/V stages with TMA and issues the MMAs.
namespace vtc {
constexpr int NS = 3;                          // K/V stages of 64 keys
constexpr int STAGE = 2 * kVT * 128 * 2;       // K (2 boxes) + V (2 boxes): 32 KB
constexpr int QX_OFF = NS * STAGE;             // Qx: 2 boxes x 128 rows x 128 B
constexpr int PX_OFF = QX_OFF + 32768;         // Px [2]: 128 rows x 128 B each
constexpr int VT_OFF = PX_OFF + 32768;         // Vt [2]: 128 rows (dims) x 128 B (64 keys)
constexpr int SL_OFF = VT_OFF + 32768;         // score parts f32 [64][64]
constexpr int MX_OFF = SL_OFF + 16384;         // stage maxima (then partial sums) f32 [64][4]
constexpr int BAR_OFF = MX_OFF + 1024;
constexpr size_t SMEM = 1024 + BAR_OFF + 256;
constexpr int THREADS = 288;                 // 8 consumer warps + the producer warp
constexpr int NCW = 8;
}  // namespace vtc

__global__ void __launch_bounds__(vtc::THREADS, 1)
    attn_verify_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const VAttnArgs a) {
  using namespace vtc;
  constexpr int HD = 128;
  constexpr int RS = HD + 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // [NS]
  uint64_t* s_bar = full + NS;    // [2] S of stage i in TMEM buffer i % 2
  uint64_t* p_bar = s_bar + 2;    // Px, Vt written and O rescaled (one arrival per warp)
  uint64_t* pv_bar = p_bar + 1;   // [2] O += P V of stage i done: Px, Vt buffer i % 2 free
  uint64_t* qx_bar = pv_bar + 2;  // Qx landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(qx_bar + 1);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);
  int* s_issued = s_abort + 1;
  float* mx_s = reinterpret_cast<float*>(smem + MX_OFF);
  float4* slo = reinterpret_cast<float4*>(smem + SL_OFF);  // [64 queries][16] swizzled

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.x / a.splits, split = blockIdx.x - kvh * a.splits;
  const int NQ = a.L * a.G;
  const int k_begin = a.klo + split * a.chunk;
  int k_end = k_begin + a.chunk;
  if (k_end > a.khi + 1) k_end = a.khi + 1;
  const int nkeys = k_end > k_begin ? k_end - k_begin : 0;
  const int ntiles = (nkeys + kVT - 1) / kVT;
  const int row0 = kvh * a.C + k_begin;
  const uint32_t sbase = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    mbar_init(p_bar, NCW);
    mbar_init(&pv_bar[0], 1);
    mbar_init(&pv_bar[1], 1);
    mbar_init(qx_bar, 1);
    *s_abort = 0;
    *s_issued = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, 256);  // S in columns [0, 64) and [64, 128), O in [128, 256)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tO = tmem + 128;

  if (warp == NCW) {
    if (lane == 0) {
      // ---- producer and MMA issuer
      auto issue = [&](int i) {
        uint8_t* st = smem + (i % NS) * STAGE;
        mbar_arrive_expect_tx(&full[i % NS], STAGE);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          tma_load_2d(st + j * kVT * 128, &tmk, &full[i % NS], 64 * j, row0 + i * kVT);
          tma_load_2d(st + 2 * kVT * 128 + j * kVT * 128, &tmv, &full[i % NS], 64 * j,
                      row0 + i * kVT);
        }
      };
      constexpr uint32_t idS = idesc_bf16_f32(128, 64), idPV = idesc_bf16_f32(128, 128);
      auto mma_s = [&](int i) {  // S_i into buffer i % 2 (its stage has landed)
        const uint32_t kb = sbase + (i % NS) * STAGE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + (i & 1) * 64,
                     smem_desc_sw128(sbase + QX_OFF + (kk >> 2) * 16384 + (kk & 3) * 32),
                     smem_desc_sw128(kb + (kk >> 2) * 8192 + (kk & 3) * 32), idS, kk != 0);
        tc_commit(&s_bar[i & 1]);
      };
      // keys before the block's first position are not written by the QKV kernel
      int n0 = 0;
      for (; n0 < NS && n0 < ntiles && k_begin + (n0 + 1) * kVT <= a.base; ++n0) issue(n0);
      pdl_wait();
      for (; n0 < NS && n0 < ntiles; ++n0) issue(n0);
      int issued = n0;
      // the queries, written by the QKV kernel's head epilogue in operand form
      mbar_arrive_expect_tx(qx_bar, 32768);
      bulk_load(smem + QX_OFF, a.qx + (size_t)kvh * 32768, 32768, qx_bar);
      bool ok = mbar_wait(qx_bar, 0, a.err, s_abort);
      if (ok && ntiles > 0) {
        ok = mbar_wait(&full[0], 0, a.err, s_abort);
        tc_fence_after();
        if (ok) mma_s(0);
      }
      for (int i = 0; ok && i < ntiles; ++i) {
        if (i + 1 < ntiles) {  // the next scores while this stage's softmax runs
          if (!mbar_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1, a.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_s(i + 1);
        }
        if (!mbar_wait(p_bar, i & 1, a.err, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pb = (uint32_t)(i & 1) * 16384;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16(tO, smem_desc_sw128(sbase + PX_OFF + pb + kk * 32),
                     smem_desc_sw128(sbase + VT_OFF + pb + kk * 32), idPV, (i | kk) != 0);
        tc_commit(&pv_bar[i & 1]);
        if (i + NS < ntiles) {  // K went into S_i, V into Vt: the stage is free
          issue(i + NS);
          ++issued;
        }
      }
      if (!ok) *(volatile int*)s_abort = 1;
      *s_issued = issued;
    } else {
      pdl_wait();
    }
    pdl_launch_dependents();
  } else {
    pdl_wait();
    pdl_launch_dependents();
    // consumer warp w: TMEM lane quadrant w % 4 (row r), column half hf = w / 4
    const int hf = warp >> 2;
    const int r = 32 * (warp & 3) + lane;  // TMEM lane / operand row
    const int q = r & 63;                  // query of the row
    const int lo = r >= 64 ? 1 : 0;        // row holds the lo part
    const bool qvalid = q < NQ;
    const int tok = qvalid ? q / a.G : 0;
    const int limit = a.bidir ? a.base + a.L - 1 : a.base + tok;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int part = 2 * hf + lo;          // this thread's 16 keys of the stage: 16 part ..
    float m = -INFINITY, l = 0.f;
    // every consumer runs every stage's named barriers, also after a give-up (a bounded
    // wait that runs out sets the abort flag; later waits return at once), so no thread is
    // left at a barrier the others skipped; the result is agreed across the warp, as what
    // follows are .sync.aligned instructions
    bool dead = false;
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
      if (!dead && !mbar_wait(bar, parity, a.err, s_abort)) {
        dead = true;
        *(volatile int*)s_abort = 1;
      }
      dead = !__all_sync(0xffffffffu, !dead);
      return !dead;
    };
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NS;
      const int key_lo = k_begin + i * kVT;
      // the four threads of query q (rows q and q + 64, column halves 0 and 1) hold its
      // scores' hi or lo part for 32 keys; each takes 16 of them, swapping the other 16
      // with its partner row through shared memory
      float sv[32];
      if (wait_ok(&s_bar[i & 1], (i >> 1) & 1)) {
        tc_fence_after();
        uint32_t t[2][16];
        tmem_ld16_nowait(tmem + (i & 1) * 64 + lane_off + 32 * hf, t[0]);
        tmem_ld16_nowait(tmem + (i & 1) * 64 + lane_off + 32 * hf + 16, t[1]);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          sv[e] = __uint_as_float(t[0][e]);
          sv[16 + e] = __uint_as_float(t[1][e]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = 0.f;
      }
      // Px, Vt buffer i % 2 is free once O += P V of stage i - 2 is done (the S barrier
      // does not cover MMAs issued after S)
      const uint32_t pb = (uint32_t)(i & 1) * 16384;
      if (i >= 2) wait_ok(&pv_bar[i & 1], ((i - 2) >> 1) & 1);
      float sc[16], give[16];  // (selected with fixed indices: no local memory)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        sc[c] = lo ? sv[16 + c] : sv[c];
        give[c] = lo ? sv[c] : sv[16 + c];
      }
      // keys 32 hf + 16 (1 - lo) .. go to the partner row, in float4 slot (key / 4)
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int kc = 8 * hf + 4 * (1 - lo) + c4;
        slo[q * 16 + (kc ^ (q & 15))] =
            make_float4(give[4 * c4], give[4 * c4 + 1], give[4 * c4 + 2], give[4 * c4 + 3]);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // score parts out
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int kc = 4 * part + c4;
        const float4 v = slo[q * 16 + (kc ^ (q & 15))];
        sc[4 * c4] += v.x;
        sc[4 * c4 + 1] += v.y;
        sc[4 * c4 + 2] += v.z;
        sc[4 * c4 + 3] += v.w;
      }
      if (a.cap_log2 != 0.f) {
#pragma unroll
        for (int c = 0; c < 16; ++c) sc[c] = a.cap_log2 * tanhf(sc[c]);
      }
      const int klo = key_lo + 16 * part;  // first key of this thread's part
      if (!(klo + 15 < k_end && klo + 15 <= limit && (!a.sliding || klo > limit - a.window))) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int key = klo + c;
          const bool vis = key < k_end && key <= limit && (!a.sliding || key > limit - a.window);
          if (!vis) sc[c] = -INFINITY;
        }
      }
      float mx[4] = {sc[0], sc[1], sc[2], sc[3]};  // four independent chains
#pragma unroll
      for (int c = 4; c < 16; ++c) mx[c & 3] = fmaxf(mx[c & 3], sc[c]);
      mx_s[4 * q + part] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      asm volatile("bar.sync 1, 256;" ::: "memory");  // maxima out
      const float4 mq = *reinterpret_cast<const float4*>(mx_s + 4 * q);
      const float m_new = fmaxf(m, fmaxf(fmaxf(mq.x, mq.y), fmaxf(mq.z, mq.w)));
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float corr = ex2_approx(m - m_use);
      m = m_new;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {  // P hi (row q) and lo (row q + 64) of the part
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2_approx(sc[8 * c8 + 2 * e] - m_use);
          const float p1 = ex2_approx(sc[8 * c8 + 2 * e + 1] - m_use);
          ps[e] += p0 + p1;
          __nv_bfloat16 h0, l0, h1, l1;
          split_bf16(p0, h0, l0);
          split_bf16(p1, h1, l1);
          hw[e] = pack_bf2(h0, h1);
          lw[e] = pack_bf2(l0, l1);
        }
        const int chunk = 2 * part + c8;
        const uint32_t sw = (uint32_t)((chunk ^ (q & 7)) << 4);
        *reinterpret_cast<uint4*>(smem + PX_OFF + pb + q * 128 + sw) =
            make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(smem + PX_OFF + pb + (q + 64) * 128 + sw) =
            make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      l = l * corr + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      // the transposed V of the stage, an eighth per warp: 8 key blocks x 16 dim blocks
      // of 8x8, one x4 taking 4 dim blocks of a key block
      {
        const bool vin = wait_ok(&full[st], (i / NS) & 1);
        const uint32_t vb = sbase + st * STAGE + 2 * kVT * 128;
        for (int blk = warp; vin && blk < 32; blk += NCW) {
          const int ka = blk >> 2, b0 = (blk & 3) * 4;  // key block, first dim block
          const int mj = lane >> 3, j = lane & 7;        // matrix, row within it
          const int bb = b0 + mj;                        // this lane's dim block
          const int key = 8 * ka + j;
          const uint32_t src = vb + (bb >> 3) * 8192 + key * 128 + (((bb & 7) ^ (key & 7)) << 4);
          uint32_t v0, v1, v2, v3;
          ldmatrix_x4(src, v0, v1, v2, v3);
          if (key_lo + 8 * ka + (lane >> 2) >= k_end) v0 = v1 = v2 = v3 = 0u;  // held key
          const int dim = 8 * bb + j;
          const uint32_t dst = sbase + VT_OFF + pb + dim * 128 + ((ka ^ (dim & 7)) << 4);
          stmatrix_x4_trans(dst, v0, v1, v2, v3);
        }
      }
      fence_proxy_async_smem();
      // O rows of a query whose maximum moved are rescaled before O += P V of this stage,
      // once the previous one is done (stage 0's MMA overwrites: nothing to scale); each
      // thread its row's column half, by the correction it computed itself (the four
      // threads of a query hold the same maxima); each warp then reports its P and Vt
      // writes and its rescale on p_bar
      const float cr = corr;
      if (i > 0 && !dead && __any_sync(0xffffffffu, cr != 1.f) &&
          wait_ok(&pv_bar[(i - 1) & 1], ((i - 1) >> 1) & 1)) {
        tc_fence_after();
        uint32_t t[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16_nowait(tO + lane_off + 64 * hf + 16 * c, t[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 16; ++e) t[c][e] = __float_as_uint(__uint_as_float(t[c][e]) * cr);
          tmem_st16(tO + lane_off + 64 * hf + 16 * c, t[c]);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_bar);
    }
    // O: wait for the last O += P V; each thread loads its row's column half, and the two
    // parts of each query are added through shared memory (the ring is idle)
    float o[64];
    if (ntiles > 0 && wait_ok(&pv_bar[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) {
      tc_fence_after();
      uint32_t t[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld16_nowait(tO + lane_off + 64 * hf + 16 * c, t[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) o[16 * c + e] = __uint_as_float(t[c][e]);
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) o[j] = 0.f;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    mx_s[4 * q + part] = l;  // the four partial sums of the query
    float4* ox = reinterpret_cast<float4*>(smem);  // [64 queries][32] swizzled
    if (lo) {
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const int k4 = 16 * hf + c4;
        ox[q * 32 + (k4 ^ (q & 31))] = make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (!lo && qvalid && !*(volatile int*)s_abort) {
      float* pr = a.part + ((size_t)kvh * a.splits + split) * 64 * RS + (size_t)q * RS;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const int k4 = 16 * hf + c4;
        const float4 v = ox[q * 32 + (k4 ^ (q & 31))];
        *reinterpret_cast<float4*>(pr + 4 * k4) =
            make_float4(o[4 * c4] + v.x, o[4 * c4 + 1] + v.y, o[4 * c4 + 2] + v.z, o[4 * c4 + 3] + v.w);
      }
      if (hf == 0) {
        const float4 lq = *reinterpret_cast<const float4*>(mx_s + 4 * q);
        *reinterpret_cast<float2*>(pr + HD) = make_float2(m, (lq.x + lq.y) + (lq.z + lq.w));
      }
    }
  }
  // drain: copies may still be landing after a give-up; then TMEM back
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = *s_issued;
    for (int st = 0; st < NS && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / NS) * NS;
      mbar_wait(&full[st], (last / NS) & 1, a.err);
    }
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ block attention at hd 512
// The records of attn_verify_kernel for 512-wide heads, one CTA per (KV head, key chunk),
// over 32-key stages:
//   scores on mma.sync: each consumer warp keeps its 8 query rows (bf16 hi in MMA rows g,
//     lo in g + 8) as A fragments in registers for all 512 dims, so shared memory carries
//     only the K tile to the scores;
//   O += Px V on tcgen05 into a 128 x 512 f32 TMEM accumulator (rows 0..63 take P hi,
//     64..127 P lo; query q's output is O[q] + O[q + 64]): per 16 keys two N = 256 MMAs,
//     V read in place from its stage as an MN-major operand (keys along K, dims along N).
// A row's reference maximum moves only when a stage's maximum passes it by more than
// kRefSlack (log2 units), so P <= 2^kRefSlack and the O rows in TMEM are rescaled only
// then; the record holds the reference as m and l = sum 2^(s - m).  One thread of warp 8
// streams K and V with TMA and issues the MMAs; K and V stages have barriers of their own:
// K of tile i + 2 loads once the scores have read tile i, V once its MMAs are done.
namespace vhy {
constexpr int HD = 512;
constexpr int VT = 32;                       // keys per stage
constexpr int TILE = VT * HD * 2;            // one K or V stage: 8 boxes of 32 keys x 128 B
constexpr int K_OFF = 0;                     // K stages [2]
constexpr int V_OFF = 2 * TILE;              // V stages [2]
constexpr int PX_OFF = 4 * TILE;             // Px [2]: 128 rows x 128 B, keys 0..31
constexpr int AUX_OFF = PX_OFF + 2 * 16384;  // corrections [2][64], flags [2][8], m [64], l [64]
constexpr int BAR_OFF = AUX_OFF + 2048;
constexpr size_t SMEM = 1024 + BAR_OFF + 256;
constexpr int THREADS = 288;                 // 8 consumer warps + the producer warp
constexpr int NCW = 8;
constexpr float kRefSlack = 8.f;
}  // namespace vhy

__global__ void __launch_bounds__(vhy::THREADS, 1)
    attn_verify_hy_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const VAttnArgs a) {
  using namespace vhy;
  constexpr int RS = HD + 4;
  constexpr int KS = HD / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // [2] K stage landed
  uint64_t* vfull = kfull + 2;   // [2] V stage landed
  uint64_t* p_bar = vfull + 2;   // Px written, rows rescaled, K read (one arrival per warp)
  uint64_t* pv_bar = p_bar + 1;  // [2] O += P V of stage i done (Px buffer, V stage i % 2 free)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(pv_bar + 2);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);
  int* s_kiss = s_abort + 1;  // K tiles requested
  int* s_viss = s_abort + 2;  // V tiles requested
  float* s_corr = reinterpret_cast<float*>(smem + AUX_OFF);      // [2][64] by stage parity
  int* s_need = reinterpret_cast<int*>(smem + AUX_OFF + 512);    // [2][8] by stage parity
  float* s_m = reinterpret_cast<float*>(smem + AUX_OFF + 1024);  // [64]
  float* s_l = s_m + 64;                                         // [64]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.x / a.splits, split = blockIdx.x - kvh * a.splits;
  const int NQ = a.L * a.G;
  const int k_begin = a.klo + split * a.chunk;
  int k_end = k_begin + a.chunk;
  if (k_end > a.khi + 1) k_end = a.khi + 1;
  const int nkeys = k_end > k_begin ? k_end - k_begin : 0;
  const int ntiles = (nkeys + VT - 1) / VT;
  const int row0 = kvh * a.C + k_begin;
  const uint32_t sbase = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&pv_bar[i], 1);
    }
    mbar_init(p_bar, NCW);
    *s_abort = 0;
    *s_kiss = 0;
    *s_viss = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, 512);  // O: 128 lanes x 512 f32 columns
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == NCW) {
    if (lane == 0) {
      // ---- producer and MMA issuer
      auto load_k = [&](int i) {
        uint8_t* st = smem + K_OFF + (i & 1) * TILE;
        mbar_arrive_expect_tx(&kfull[i & 1], TILE);
#pragma unroll
        for (int j = 0; j < HD / 64; ++j)
          tma_load_2d(st + j * VT * 128, &tmk, &kfull[i & 1], 64 * j, row0 + i * VT);
      };
      auto load_v = [&](int i) {
        uint8_t* st = smem + V_OFF + (i & 1) * TILE;
        mbar_arrive_expect_tx(&vfull[i & 1], TILE);
#pragma unroll
        for (int j = 0; j < HD / 64; ++j)
          tma_load_2d(st + j * VT * 128, &tmv, &vfull[i & 1], 64 * j, row0 + i * VT);
      };
      // keys before the block's first position are not written by the QKV kernel
      int n0 = 0;
      for (; n0 < 2 && n0 < ntiles && k_begin + (n0 + 1) * VT <= a.base; ++n0) {
        load_k(n0);
        load_v(n0);
      }
      pdl_wait();
      for (; n0 < 2 && n0 < ntiles; ++n0) {
        load_k(n0);
        load_v(n0);
      }
      int kiss = n0, viss = n0, pv_issued = 0;
      constexpr uint32_t idPV = idesc_bf16_f32_bmn(128, 256);
      bool ok = true;
      for (int i = 0; ok && i < ntiles; ++i) {
        if (!mbar_wait(p_bar, i & 1, a.err, s_abort) ||
            !mbar_wait(&vfull[i & 1], (i >> 1) & 1, a.err, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t px = sbase + PX_OFF + (uint32_t)(i & 1) * 16384;
        const uint32_t vb = sbase + V_OFF + (uint32_t)(i & 1) * TILE;
#pragma unroll
        for (int h = 0; h < 2; ++h)      // output dims 256 h .. 256 h + 255: V boxes 4 h ..
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)  // keys 16 kk .. 16 kk + 15
            tc_mma_f16(tmem + 256 * h, smem_desc_sw128(px + kk * 32),
                       smem_desc_sw128_mn(vb + h * 4 * (VT * 128) + kk * 2048, VT * 128), idPV,
                       (i | kk) != 0);
        tc_commit(&pv_bar[i & 1]);
        pv_issued = i + 1;
        if (i + 2 < ntiles) {
          load_k(i + 2);  // the scores have read K of stage i (p_bar)
          ++kiss;
          if (!mbar_wait(&pv_bar[i & 1], (i >> 1) & 1, a.err, s_abort)) {
            ok = false;
            break;
          }
          load_v(i + 2);  // the MMAs have read V of stage i
          ++viss;
        }
      }
      if (!ok) *(volatile int*)s_abort = 1;
      // the MMAs complete in order: the last one's commit covers all of them
      if (pv_issued > 0) mbar_wait(&pv_bar[(pv_issued - 1) & 1], ((pv_issued - 1) >> 1) & 1, a.err);
      *s_kiss = kiss;
      *s_viss = viss;
    } else {
      pdl_wait();
    }
    pdl_launch_dependents();
  } else {
    pdl_wait();
    pdl_launch_dependents();
    const int g = lane >> 2, t = lane & 3;
    const int qrow = 8 * warp + g;  // query of this lane's score rows
    const bool qvalid = qrow < NQ;
    const int tok = qvalid ? qrow / a.G : 0;
    const int limit = a.bidir ? a.base + a.L - 1 : a.base + tok;  // last visible position
    // the query as A fragments of every 16-dim k-step (scaled; hi in row g, lo in row g + 8)
    uint32_t qa[KS][4];
    {
      const float* q = a.q + ((size_t)tok * a.nh + kvh * a.G + qrow % a.G) * HD + 2 * t;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
        if (qvalid) {
          const float2 v0 = *reinterpret_cast<const float2*>(q + ks * 16);
          const float2 v1 = *reinterpret_cast<const float2*>(q + ks * 16 + 8);
          __nv_bfloat16 h[4], lw[4];
          split_bf16(v0.x * a.qscale, h[0], lw[0]);
          split_bf16(v0.y * a.qscale, h[1], lw[1]);
          split_bf16(v1.x * a.qscale, h[2], lw[2]);
          split_bf16(v1.y * a.qscale, h[3], lw[3]);
          qa[ks][0] = pack_bf2(h[0], h[1]);
          qa[ks][1] = pack_bf2(lw[0], lw[1]);
          qa[ks][2] = pack_bf2(h[2], h[3]);
          qa[ks][3] = pack_bf2(lw[2], lw[3]);
        }
      }
    }
    // ldmatrix lane offsets of the K fragments (row 16 hb + (lane / 16) 8 + lane % 8,
    // 16-byte chunk 2 ks + (lane / 8) % 2 of its box, swizzled by row % 8 = lane % 8)
    uint32_t swk[4];
    {
      const int l7 = lane & 7;
      const int xk = ((lane >> 3) & 1) ^ l7;
      const uint32_t rk = (uint32_t)((((lane >> 4) << 3) + l7) * 128);
#pragma unroll
      for (int j = 0; j < 4; ++j) swk[j] = rk + (uint32_t)(((2 * j) ^ xk) << 4);
    }
    float m_ref = -INFINITY, l = 0.f;
    // every consumer runs every stage's named barriers, also after a give-up (a bounded
    // wait that runs out sets the abort flag; later waits return at once); the result is
    // agreed across the warp, as the tcgen05 loads and stores are .sync.aligned
    bool dead = false;
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
      if (!dead && !mbar_wait(bar, parity, a.err, s_abort)) {
        dead = true;
        *(volatile int*)s_abort = 1;
      }
      dead = !__all_sync(0xffffffffu, !dead);
      return !dead;
    };
    // this warp's TMEM rows (lane quadrant warp % 4) and column half (warp / 4)
    const int r_t = 32 * (warp & 3) + lane;
    const int q_t = r_t & 63;
    const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256 * (warp >> 2);
    for (int i = 0; i < ntiles; ++i) {
      const int key0 = k_begin + i * VT;
      float p[2][4];  // 16-key half hb: keys 16 hb + 8 (e / 2) + 2 t + e % 2
      float mloc = -INFINITY;
      if (wait_ok(&kfull[i & 1], (i >> 1) & 1)) {
        const uint32_t kb = sbase + K_OFF + (uint32_t)(i & 1) * TILE;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float s[2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kb + swk[ks & 3] + (uint32_t)((ks >> 2) * (VT * 128) + hb * 16 * 128), b0,
                        b1, b2, b3);
            mma_bf16(s[0], qa[ks], b0, b1);
            mma_bf16(s[1], qa[ks], b2, b3);
          }
          float sc[4] = {s[0][0] + s[0][2], s[0][1] + s[0][3], s[1][0] + s[1][2],
                         s[1][1] + s[1][3]};
          if (a.cap_log2 != 0.f) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[e] = a.cap_log2 * tanhf(sc[e]);
          }
          // keys past the chunk, after this row's position or before its window: masked
          const int klo = key0 + 16 * hb;
          if (!(klo + 15 < k_end && klo + 15 <= limit && (!a.sliding || klo > limit - a.window))) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = klo + 8 * (e >> 1) + 2 * t + (e & 1);
              const bool vis = key < k_end && key <= limit && (!a.sliding || key > limit - a.window);
              if (!vis) sc[e] = -INFINITY;
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            p[hb][e] = sc[e];
            mloc = fmaxf(mloc, sc[e]);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) p[0][e] = p[1][e] = -INFINITY;
      }
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
      // the reference moves only past the slack (from -inf: the O rows are exactly zero)
      float corr = 1.f;
      if (mloc > m_ref + kRefSlack) {
        if (m_ref != -INFINITY) corr = ex2_approx(m_ref - mloc);
        m_ref = mloc;
      }
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      float psum = 0.f;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          p[hb][e] = ex2_approx(p[hb][e] - m_use);
          psum += p[hb][e];
        }
      l = l * corr + psum;
      // P hi in row qrow, lo in row qrow + 64 of Px buffer i % 2 (its previous MMA, stage
      // i - 2, was waited for at the end of stage i - 1): key pair (8 c + 2 t, + 1) is the
      // t-th word of 16-byte chunk c, stored at chunk c XOR (row % 8)
      uint8_t* px = smem + PX_OFF + (i & 1) * 16384;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          __nv_bfloat16 h0, l0, h1, l1;
          split_bf16(p[hb][2 * j], h0, l0);
          split_bf16(p[hb][2 * j + 1], h1, l1);
          const int c = 2 * hb + j;
          const int off = (qrow & 7) * 128 + ((c ^ (qrow & 7)) << 4) + 4 * t;
          *reinterpret_cast<uint32_t*>(px + (qrow >> 3) * 1024 + off) = pack_bf2(h0, h1);
          *reinterpret_cast<uint32_t*>(px + ((qrow + 64) >> 3) * 1024 + off) = pack_bf2(l0, l1);
        }
      // the last tile's V rows past the chunk may hold any bits (a NaN times a zero weight
      // is NaN): zeroed before the MMA reads them
      if (i == ntiles - 1 && key0 + VT > k_end && wait_ok(&vfull[i & 1], (i >> 1) & 1)) {
        const int nv = k_end - key0, nr = VT - nv;
        uint8_t* vt = smem + V_OFF + (i & 1) * TILE;
        for (int z = threadIdx.x; z < nr * 8 * 8; z += NCW * 32) {
          const int box = z / (nr * 8), rem = z - box * (nr * 8);
          *reinterpret_cast<uint4*>(vt + box * (VT * 128) + (nv + (rem >> 3)) * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      const int b = i & 1;
      if (t == 0) s_corr[b * 64 + qrow] = corr;
      const bool need = __any_sync(0xffffffffu, corr != 1.f);
      if (lane == 0) s_need[b * 8 + warp] = need ? 1 : 0;
      fence_proxy_async_smem();
      // O += P V of stage i - 1 is done before this stage's p_bar phase can complete (so the
      // MMA thread has taken the previous phase), and before rows are rescaled
      const bool prev = i == 0 || wait_ok(&pv_bar[(i - 1) & 1], ((i - 1) >> 1) & 1);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      bool any = false;
#pragma unroll
      for (int w = 0; w < NCW; ++w) any = any || s_need[b * 8 + w] != 0;
      if (i > 0 && any && prev) {
        const float cr = s_corr[b * 64 + q_t];
        if (__any_sync(0xffffffffu, cr != 1.f)) {
          tc_fence_after();
          // 16 columns a round: the query fragments stay live in registers meanwhile
#pragma unroll 1
          for (int c0 = 0; c0 < 256; c0 += 16) {
            uint32_t tv[16];
            tmem_ld16_nowait(t_row + c0, tv);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) tv[e] = __float_as_uint(__uint_as_float(tv[e]) * cr);
            tmem_st16(t_row + c0, tv);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_bar);
    }
    // m and l of each query row (its four lanes hold the same reference; l summed)
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (t == 0) {
      s_m[qrow] = m_ref;
      s_l[qrow] = l;
    }
    // O: the last O += P V done; the rows q + 64 (P lo) are added to rows q through shared
    // memory (the K and V stages are idle: every copy has been consumed)
    const bool have = ntiles > 0 && wait_ok(&pv_bar[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1);
    tc_fence_after();
    asm volatile("bar.sync 1, 256;" ::: "memory");
    // every condition around a tcgen05 load or store is agreed across the warp (they are
    // .sync.aligned); the abort flag can change while the lanes read it
    const bool live = __all_sync(0xffffffffu, have && !*(volatile int*)s_abort);
    const bool lo = r_t >= 64;
    const int hf = warp >> 2;
    float4* ox = reinterpret_cast<float4*>(smem);  // [64 queries][128 float4], swizzled
    if (lo && live) {
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 64) {
        uint32_t tv[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16_nowait(t_row + c0 + 16 * c, tv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int k4 = (256 * hf + c0) / 4 + c;
          ox[q_t * 128 + (k4 ^ (q_t & 7))] =
              make_float4(__uint_as_float(tv[c >> 2][4 * (c & 3)]),
                          __uint_as_float(tv[c >> 2][4 * (c & 3) + 1]),
                          __uint_as_float(tv[c >> 2][4 * (c & 3) + 2]),
                          __uint_as_float(tv[c >> 2][4 * (c & 3) + 3]));
        }
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (!lo) {  // a whole warp: its TMEM loads run on every lane, valid query row or not
      const bool ok_all = __all_sync(0xffffffffu, !*(volatile int*)s_abort);  // every lane
      const bool store = q_t < NQ && ok_all;
      float* pr = a.part + ((size_t)kvh * a.splits + split) * 64 * RS + (size_t)q_t * RS;
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 64) {
        uint32_t tv[4][16];
        if (live) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16_nowait(t_row + c0 + 16 * c, tv[c]);
          tmem_wait_ld();
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int k4 = (256 * hf + c0) / 4 + c;
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (live) {
            const float4 v = ox[q_t * 128 + (k4 ^ (q_t & 7))];
            o = make_float4(__uint_as_float(tv[c >> 2][4 * (c & 3)]) + v.x,
                            __uint_as_float(tv[c >> 2][4 * (c & 3) + 1]) + v.y,
                            __uint_as_float(tv[c >> 2][4 * (c & 3) + 2]) + v.z,
                            __uint_as_float(tv[c >> 2][4 * (c & 3) + 3]) + v.w);
          }
          if (store) *reinterpret_cast<float4*>(pr + 4 * k4) = o;
        }
      }
      if (store && hf == 0) *reinterpret_cast<float2*>(pr + HD) = make_float2(s_m[q_t], s_l[q_t]);
    }
  }
  // drain: copies may still be landing after a give-up; then TMEM back
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int kiss = *s_kiss, viss = *s_viss;
    for (int st = 0; st < 2; ++st) {
      if (st < kiss) mbar_wait(&kfull[st], (((st + ((kiss - 1 - st) / 2) * 2)) >> 1) & 1, a.err);
      if (st < viss) mbar_wait(&vfull[st], (((st + ((viss - 1 - st) / 2) * 2)) >> 1) & 1, a.err);
    }
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Combination of the block attention's split records, one CTA per RPW = 256 / HD query
// rows of one KV head (one row at HD 512; the lanes of a row own CPL = 8 output columns
// each, 16 at HD 512):
//   M = max_s m_s,  w_s = 2^(m_s - M),  o = sum_s w_s O_s / sum_s w_s l_s.
// The (m, l) pairs go through shared memory; the four warps each sum a quarter of the
// splits (their records loaded in the same round as the pairs) and the partial sums are
// added in warp order, so the result does not depend on timing.  The output is written twice: f32 o, and the o_proj GEMM's activation operand.
template <int HD>
__global__ void __launch_bounds__(128) attn_verify_merge_kernel(const VAttnArgs a) {
  constexpr int CPL = HD <= 256 ? 8 : HD / 32;  // output columns per lane
  constexpr int NV = CPL / 4;                   // float4 of a record per lane
  constexpr int LPR = HD / CPL;                 // lanes per query row
  constexpr int RPW = 32 / LPR;                 // query rows per CTA
  constexpr int RS = HD + 4;
  __shared__ float4 s_acc[4][32][NV];
  extern __shared__ float2 s_ml[];  // [RPW][splits]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y;
  const int NQ = a.L * a.G;
  const int S = a.splits;
  const int sub = lane / LPR, d8 = lane - sub * LPR;
  const int r = blockIdx.x * RPW + sub;
  const int rr = r < NQ ? r : NQ - 1;
  const float* up = a.part + (size_t)kvh * S * 64 * RS;
  pdl_wait();
  pdl_launch_dependents();
  // every load in one round: the (m, l) pairs into shared memory, and this warp's first
  // MB records (splits warp, warp + 4, ...) into registers
  constexpr int MB = 24 / NV;
  for (int it = threadIdx.x; it < RPW * S; it += blockDim.x) {
    const int row = it / S, sp = it - row * S;
    const int qr = blockIdx.x * RPW + row < NQ ? blockIdx.x * RPW + row : NQ - 1;
    s_ml[it] = __ldcg(reinterpret_cast<const float2*>(up + ((size_t)sp * 64 + qr) * RS + HD));
  }
  const float* base = up + (size_t)rr * RS + CPL * d8;
  float4 v[NV * MB];
#pragma unroll
  for (int j = 0; j < MB; ++j) {
    const int sp = warp + 4 * j;
    if (sp < S) {
      const float4* src = reinterpret_cast<const float4*>(base + (size_t)sp * 64 * RS);
#pragma unroll
      for (int u = 0; u < NV; ++u) v[NV * j + u] = __ldcg(src + u);
    }
  }
  __syncthreads();
  const float2* ml = s_ml + sub * S;
  float M = -INFINITY;
  for (int sp = d8; sp < S; sp += LPR) M = fmaxf(M, ml[sp].x);
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float Mu = M == -INFINITY ? 0.f : M;
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int sp0 = warp;; sp0 += 4 * MB) {
#pragma unroll
    for (int j = 0; j < MB; ++j) {
      const int sp = sp0 + 4 * j;
      if (sp < S) {
        const float w = ex2_approx(ml[sp].x - Mu);
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          acc[4 * u] += w * v[NV * j + u].x;
          acc[4 * u + 1] += w * v[NV * j + u].y;
          acc[4 * u + 2] += w * v[NV * j + u].z;
          acc[4 * u + 3] += w * v[NV * j + u].w;
        }
      }
    }
    if (sp0 + 4 * MB >= S) break;
#pragma unroll
    for (int j = 0; j < MB; ++j) {  // more than 4 MB splits: the next batch
      const int sp = sp0 + 4 * MB + 4 * j;
      if (sp < S) {
        const float4* src = reinterpret_cast<const float4*>(base + (size_t)sp * 64 * RS);
#pragma unroll
        for (int u = 0; u < NV; ++u) v[NV * j + u] = __ldcg(src + u);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < NV; ++u)
    s_acc[warp][lane][u] = make_float4(acc[4 * u], acc[4 * u + 1], acc[4 * u + 2], acc[4 * u + 3]);
  __syncthreads();
  if (warp != 0) return;
  float den = 0.f;
  for (int q = d8; q < S; q += LPR) den += ex2_approx(ml[q].x - Mu) * ml[q].y;
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float out[CPL];
#pragma unroll
  for (int h = 0; h < NV; ++h) {
    float4 t0 = s_acc[0][lane][h];
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      const float4 tw = s_acc[w][lane][h];
      t0.x += tw.x; t0.y += tw.y; t0.z += tw.z; t0.w += tw.w;
    }
    out[4 * h] = t0.x * inv;
    out[4 * h + 1] = t0.y * inv;
    out[4 * h + 2] = t0.z * inv;
    out[4 * h + 3] = t0.w * inv;
  }
  if (r >= NQ) return;
  const int tok = r / a.G, h = kvh * a.G + r % a.G;
  float4* dst = reinterpret_cast<float4*>(a.o + ((size_t)tok * a.nh + h) * HD) + NV * d8;
#pragma unroll
  for (int u = 0; u < NV; ++u)
    dst[u] = make_float4(out[4 * u], out[4 * u + 1], out[4 * u + 2], out[4 * u + 3]);
  // the same values as the o_proj GEMM's activation operand (columns h * HD + CPL d8 ..)
#pragma unroll
  for (int gq = 0; gq < CPL / 8; ++gq) {
    float o8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o8[i] = out[8 * gq + i];
    store_bop_group(a.bops, tok, (h * HD + CPL * d8) / 8 + gq, o8);
  }
}

// Post-attention RMSNorm of the verify block, one CTA per token row: sum(y^2) in a fixed
// order (thread strides, warp trees, warps in order), then out = bf16(x + y w r).
__global__ void __launch_bounds__(256) post_norm_rows_kernel(const float* __restrict__ y,
                                                             const __nv_bfloat16* __restrict__ x,
                                                             const float* __restrict__ w, int H,
                                                             float eps, __nv_bfloat16* out,
                                                             float* out_tap) {
  __shared__ float s_w[8];
  const int row = blockIdx.x, tid = threadIdx.x;
  const float* yr = y + (size_t)row * H;
  float ss = 0.f;
  for (int i = tid; i < H; i += 256) ss += yr[i] * yr[i];
  ss = warp_sum(ss);
  if ((tid & 31) == 0) s_w[tid >> 5] = ss;
  __syncthreads();
  float t = 0.f;
  for (int k = 0; k < 8; ++k) t += s_w[k];
  const float r = rsqrtf(t / H + eps);
  for (int i = tid; i < H; i += 256) {
    const float o = __bfloat162float(x[(size_t)row * H + i]) + yr[i] * w[i] * r;
    out[(size_t)row * H + i] = __float2bfloat16_rn(o);
    if (out_tap) out_tap[(size_t)row * H + i] = o;
  }
}

// ------------------------------------------------------------------ host side
struct VerifyState {
  float* part = nullptr;        // [max(SMs, nkv)][64][hd + 4]
  float* y_post = nullptr;      // [16][H]: o_proj output kept for the post-attention norm
  uint8_t* bq = nullptr;        // QKV activation operand [H / 64][32][128 B]
  uint8_t* bo = nullptr;        // o_proj activation operand [nh hd / 64][32][128 B]
  uint8_t* qx = nullptr;        // head_dim 128: attention query operand [nkv][32 KB]
  size_t part_records = 0;
  int max_clusters[9] = {};     // co-resident GEMM clusters of n CTAs (index n)
  // the QKV GEMMs' k-split partial sums through global memory (no cluster): tagged
  // entries [CTA][16 tokens][128 rows], and one launch counter for the block's QKV GEMM
  // and one for the context rows' (different grids)
  unsigned long long* gpart = nullptr;
  unsigned long long* gctr = nullptr;  // [2]
  size_t gpart_entries = 0;
};

static char g_verify_error[256];
const char* verify_error() { return g_verify_error; }

hfa_status verify_create(const hfa_layer_desc& d, int num_sms, VerifyState** out) {
  *out = nullptr;
  if (!(d.flags & HFA_F_WEIGHTS_BF16)) {
    *out = new VerifyState();  // a Q8_0 layer has no verify block: nothing to allocate
    return HFA_OK;
  }
  const int rows_qkv = qkv_rows(d);
  if (rows_qkv % kVM || d.hidden % kVM || d.hidden % kVK || (d.num_heads * d.head_dim) % kVK) {
    snprintf(g_verify_error, sizeof g_verify_error,
             "verify GEMM needs projection sizes that are multiples of 128");
    return HFA_EUNSUPPORTED;
  }
  VerifyState* v = new VerifyState();
  const int nkv = d.num_kv_heads;
  v->part_records = (size_t)(num_sms > nkv ? num_sms : nkv);
  cudaError_t e = cudaMalloc(&v->part, v->part_records * 64 * (d.head_dim + 4) * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&v->bq, (size_t)(d.hidden / kVK) * kBChunkBytes);
  if (e == cudaSuccess)
    e = cudaMalloc(&v->bo, (size_t)(d.num_heads * d.head_dim / kVK) * kBChunkBytes);
  if (e == cudaSuccess)
    e = cudaMemset(v->bo, 0, (size_t)(d.num_heads * d.head_dim / kVK) * kBChunkBytes);
  if (e == cudaSuccess && d.head_dim == 128) {  // rows past L * G stay zero
    e = cudaMalloc(&v->qx, (size_t)nkv * 32768);
    if (e == cudaSuccess) e = cudaMemset(v->qx, 0, (size_t)nkv * 32768);
  }
  if (e == cudaSuccess) e = cudaMalloc(&v->y_post, (size_t)16 * d.hidden * sizeof(float));
  v->gpart_entries = (size_t)num_sms * 16 * kVM;  // at most one CTA per SM (cooperative)
  if (e == cudaSuccess) e = cudaMalloc(&v->gpart, v->gpart_entries * 8);
  if (e == cudaSuccess) e = cudaMemset(v->gpart, 0, v->gpart_entries * 8);
  if (e == cudaSuccess) e = cudaMalloc(&v->gctr, 2 * 8);
  if (e == cudaSuccess) e = cudaMemset(v->gctr, 0, 2 * 8);
  if (e != cudaSuccess) {
    snprintf(g_verify_error, sizeof g_verify_error, "%s", cudaGetErrorString(e));
    verify_free(v);
    return HFA_ENOMEM;
  }
  // how many GEMM clusters of each size fit on the GPU at once (GPCs hold different
  // numbers of SMs, so this is not num_sms / n)
  e = cudaFuncSetAttribute(verify_gemm_kernel<kModeQKV>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVGemmSmem);
  v->max_clusters[1] = num_sms;
  for (int n = 2; n <= 8 && e == cudaSuccess; ++n) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kVGemmSmem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)n;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&v->max_clusters[n], verify_gemm_kernel<kModeQKV>, &cfg);
  }
  if (e != cudaSuccess) {
    snprintf(g_verify_error, sizeof g_verify_error, "cluster occupancy: %s",
             cudaGetErrorString(e));
    verify_free(v);
    return HFA_ECUDA;
  }
  *out = v;
  return HFA_OK;
}

void verify_free(VerifyState* v) {
  if (!v) return;
  cudaFree(v->part);
  cudaFree(v->y_post);
  cudaFree(v->bq);
  cudaFree(v->bo);
  cudaFree(v->qx);
  cudaFree(v->gpart);
  cudaFree(v->gctr);
  delete v;
}

hfa_status verify_reset(VerifyState* v, cudaStream_t s) {
  if (!v || !v->gpart) return HFA_OK;
  cudaError_t e = cudaMemsetAsync(v->gpart, 0, v->gpart_entries * 8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(v->gctr, 0, 2 * 8, s);
  return e == cudaSuccess ? HFA_OK : HFA_ECUDA;
}

template <typename Kern, typename... Args>
static cudaError_t launch_ex3(Kern kern, dim3 grid, int threads, size_t smem, bool pdl,
                              cudaStream_t s, int cluster, bool coop, Args... args) {
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (coop) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na++].val.cooperative = 1;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na++].val.programmaticStreamSerializationAllowed = 1;
  }
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na++].val.clusterDim.z = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern, typename... Args>
static cudaError_t launch_ex2(Kern kern, dim3 grid, int threads, size_t smem, bool pdl,
                              cudaStream_t s, int cluster, Args... args) {
  return launch_ex3(kern, grid, threads, smem, pdl, s, cluster, false, args...);
}

template <typename Kern, typename... Args>
static cudaError_t launch_ex(Kern kern, int grid, int threads, size_t smem, bool pdl,
                             cudaStream_t s, Args... args) {
  return launch_ex2(kern, dim3(grid), threads, smem, pdl, s, 1, args...);
}

// k-splits per row tile: the SMs shared out over the tiles, with every cluster of
// tpc tiles x splits CTAs (at most 8, reducing through distributed shared memory)
// resident at once -- max_clusters[n] is how many clusters of n CTAs the GPU holds.
static int gemm_splits(int tiles, int chunks, int num_sms, int tpc, const int* max_clusters) {
  int S = num_sms / tiles;
  if (S > 8 / tpc) S = 8 / tpc;
  if (S > chunks) S = chunks;
  while (S > 1 && tiles / tpc > max_clusters[S * tpc]) --S;
  if (S < 1) S = 1;
  return S;
}

// k-splits per row tile when the splits add through global memory: the SMs shared out over
// the tiles (one CTA per SM, all resident: a cooperative launch), at most 8
static int gemm_splits_flat(int tiles, int chunks, int num_sms, int tpc) {
  int S = num_sms / tiles;
  if (S > 8 / tpc) S = 8 / tpc;
  if (S > chunks) S = chunks;
  return S < 1 ? 1 : S;
}

hfa_status verify_ctx_append(VerifyState* v, const VerifyCall& c, char* msg, int n) {
  const hfa_layer_desc& d = *c.d;
  const int H = d.hidden, nh = d.num_heads, nkv = d.num_kv_heads, hd = d.head_dim;
  const int rows_qkv = qkv_rows(d);
  if (!(d.flags & HFA_F_WEIGHTS_BF16) || !v->part) {
    snprintf(msg, n, "context rows need the bf16 (verify) weights");
    return HFA_EUNSUPPORTED;
  }
  cudaStream_t s = c.stream;
  const bool pdl = c.timer == nullptr;
  auto tb = [&](const char* nm) { if (c.timer) c.timer->begin(s, nm); };
  auto te = [&]() { if (c.timer) c.timer->end(s); };
  // (0) the rows as they are (w_in NULL: no input norm), bf16 hi/lo operand
  tb("ctx_prep");
  cudaError_t e = launch_ex(verify_prep_kernel, 16, 256, 0, pdl, s, c.x, (const float*)nullptr,
                            d.eps, c.L, H, v->bq);
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "context prep launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }
  // (1) the K and V rows only: row tiles from the one holding the first key row
  VGemmArgs qa{};
  qa.bops = v->bq;
  qa.wt = reinterpret_cast<const uint8_t*>(c.wqkv);
  qa.g.batch = c.L;
  qa.g.x = c.x;
  qa.g.eps = d.eps;
  qa.g.R = rows_qkv / 16;
  qa.g.err = c.err;
  qa.g.nh = nh;
  qa.g.nkv = nkv;
  qa.g.hd = hd;
  qa.g.C = d.kv_capacity;
  qa.g.w_q = c.w_q;
  qa.g.w_k = c.w_k;
  qa.g.rope_g = c.rope_g;
  qa.g.v_unit_norm = (d.flags & HFA_F_V_UNIT_NORM) ? 1 : 0;
  qa.g.k_eq_v = (d.flags & HFA_F_K_EQ_V) ? 1 : 0;
  qa.g.kv_only = 1;
  qa.g.q_out = c.q_f32;
  qa.g.G = nh / nkv;
  qa.g.k_cache = c.k_cache;
  qa.g.v_cache = c.v_cache;
  qa.g.k_tap = c.k_tap;
  qa.g.v_tap = c.v_tap;
  qa.g.rows_are_tokens = 1;
  qa.g.base_pos = c.base_pos;
  qa.rows = rows_qkv;
  qa.K = H;
  qa.chunks = H / kVK;
  qa.tpc = hd > kVM ? hd / kVM : 1;
  qa.tile_base = (nh * hd / kVM) / qa.tpc * qa.tpc;  // aligned to the clusters of a head
  const int ktiles = rows_qkv / kVM - qa.tile_base;
  // the k-splits add through global memory when every row tile can have a CTA resident,
  // else through clusters
  const bool flat = ktiles <= c.num_sms;
  qa.splits = flat ? gemm_splits_flat(ktiles, qa.chunks, c.num_sms, qa.tpc)
                   : gemm_splits(ktiles, qa.chunks, c.num_sms, qa.tpc, v->max_clusters);
  qa.gpart = flat ? v->gpart : nullptr;
  qa.gctr = v->gctr + 1;
  qa.tag_lane = 1;  // odd tags: the block's QKV GEMM uses the same gpart with even ones
  tb("ctx_kv_gemm");
  e = launch_ex3(verify_gemm_kernel<kModeQKV>, dim3(ktiles * qa.splits), 128, kVGemmSmem, pdl, s,
                 flat ? 1 : qa.splits * qa.tpc, flat, qa);
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "context K/V launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }
  return HFA_OK;
}

hfa_status verify_run(VerifyState* v, const VerifyCall& c, char* msg, int n) {
  const hfa_layer_desc& d = *c.d;
  const int H = d.hidden, nh = d.num_heads, nkv = d.num_kv_heads, hd = d.head_dim;
  const int G = nh / nkv;
  const int rows_qkv = qkv_rows(d);
  if (!(d.flags & HFA_F_WEIGHTS_BF16) || !v->part) {
    snprintf(msg, n, "verify is built for bf16 weights");
    return HFA_EUNSUPPORTED;
  }
  if (c.L * G > 64) {
    snprintf(msg, n, "L * (num_heads / num_kv_heads) = %d > 64 query rows per KV head", c.L * G);
    return HFA_EUNSUPPORTED;
  }

  const int VT = hd == 512 ? vhy::VT : kVT;  // keys per attention stage
  CUtensorMap tk, tv;
  if (hfa_encode_kv_map(&tk, c.k_cache, nkv * d.kv_capacity, hd, VT) != HFA_OK ||
      hfa_encode_kv_map(&tv, c.v_cache, nkv * d.kv_capacity, hd, VT) != HFA_OK) {
    snprintf(msg, n, "cannot describe the KV cache to the TMA unit");
    return HFA_EINVAL;
  }
  cudaStream_t s = c.stream;
  cudaError_t e;
  const bool pdl = c.timer == nullptr;
  auto tb = [&](const char* nm) { if (c.timer) c.timer->begin(s, nm); };
  auto te = [&]() { if (c.timer) c.timer->end(s); };

  // (0) activation operand of the QKV projection: input RMSNorm, bf16 hi/lo split
  tb("verify_prep");
  e = launch_ex(verify_prep_kernel, 16, 256, 0, pdl, s, c.x, c.w_in, d.eps, c.L, H, v->bq);
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "verify prep launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }

  // (1) QKV projection + per-head norms + RoPE + append of all L rows
  VGemmArgs qa{};
  qa.bops = v->bq;
  qa.wt = reinterpret_cast<const uint8_t*>(c.wqkv);
  qa.g.batch = c.L;
  qa.g.x = c.x;
  qa.g.w_in = c.w_in;
  qa.g.eps = d.eps;
  qa.g.R = rows_qkv / 16;
  qa.g.err = c.err;
  qa.g.nh = nh;
  qa.g.nkv = nkv;
  qa.g.hd = hd;
  qa.g.C = d.kv_capacity;
  qa.g.ring = 0;
  qa.g.w_q = c.w_q;
  qa.g.w_k = c.w_k;
  qa.g.rope_g = c.rope_g;
  qa.g.v_unit_norm = (d.flags & HFA_F_V_UNIT_NORM) ? 1 : 0;
  qa.g.k_eq_v = (d.flags & HFA_F_K_EQ_V) ? 1 : 0;
  qa.g.q_out = c.q_f32;
  qa.g.qx = v->qx;  // head_dim 128 only (else null)
  qa.g.qscale = d.softcap > 0.f ? d.attn_scale / d.softcap : d.attn_scale * 1.4426950408889634f;
  qa.g.G = G;
  qa.g.k_cache = c.k_cache;
  qa.g.v_cache = c.v_cache;
  qa.g.k_tap = c.k_tap;
  qa.g.v_tap = c.v_tap;
  qa.g.rows_are_tokens = 1;
  qa.g.base_pos = c.base_pos;
  qa.rows = rows_qkv;
  qa.K = H;
  qa.chunks = H / kVK;
  const int qtiles = rows_qkv / kVM;
  qa.tpc = hd > kVM ? hd / kVM : 1;
  const bool flat = qtiles <= c.num_sms;  // as for the context rows
  qa.splits = flat ? gemm_splits_flat(qtiles, qa.chunks, c.num_sms, qa.tpc)
                   : gemm_splits(qtiles, qa.chunks, c.num_sms, qa.tpc, v->max_clusters);
  qa.gpart = flat ? v->gpart : nullptr;
  qa.gctr = v->gctr;
  tb("verify_qkv_gemm");
  e = launch_ex3(verify_gemm_kernel<kModeQKV>, dim3(qtiles * qa.splits), 128, kVGemmSmem, pdl, s,
                 flat ? 1 : qa.splits * qa.tpc, flat, qa);
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "verify QKV launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }

  // (2) block attention
  VAttnArgs aa{};
  aa.q = c.q_f32;
  aa.L = c.L;
  aa.nh = nh;
  aa.nkv = nkv;
  aa.G = G;
  aa.C = d.kv_capacity;
  aa.base = c.base_pos;
  aa.sliding = d.layer_type == HFA_SLIDING;
  aa.bidir = c.bidir && d.layer_type == HFA_FULL;
  aa.window = d.window;
  const float log2e = 1.4426950408889634f;
  if (d.softcap > 0.f) {
    aa.qscale = d.attn_scale / d.softcap;
    aa.cap_log2 = d.softcap * log2e;
  } else {
    aa.qscale = d.attn_scale * log2e;
    aa.cap_log2 = 0.f;
  }
  aa.klo = aa.sliding ? (c.base_pos - d.window + 1 > 0 ? c.base_pos - d.window + 1 : 0) : 0;
  aa.khi = c.base_pos + c.L - 1;
  const int nkeys = aa.khi - aa.klo + 1;
  int S = c.num_sms / nkv;
  const int max_tiles = (nkeys + VT - 1) / VT;
  if (S > max_tiles) S = max_tiles;
  if ((size_t)S * nkv > v->part_records) S = (int)(v->part_records / nkv);
  if (S < 1) S = 1;
  int chunk = (nkeys + S - 1) / S;
  chunk = (chunk + VT - 1) / VT * VT;
  S = (nkeys + chunk - 1) / chunk;
  aa.splits = S;
  aa.chunk = chunk;
  aa.part = v->part;
  aa.bops = v->bo;
  aa.qx = v->qx;
  aa.o = c.o_f32;
  aa.err = c.err;
  const int nq_warps = (c.L * G + 7) / 8;
  const int athreads = (nq_warps + 1) * 32;
  tb("verify_attention");
  if (hd == 64)
    e = launch_ex(attn_verify_kernel<64>, nkv * S, athreads, VACfg<64>::SMEM, pdl, s, tk, tv, aa);
  else if (hd == 128)  // both products on the tensor cores (TMEM accumulators)
    e = launch_ex(attn_verify_tc_kernel, nkv * S, vtc::THREADS, vtc::SMEM, pdl, s, tk, tv, aa);
  else if (hd == 256)
    e = launch_ex(attn_verify_kernel<256>, nkv * S, athreads, VACfg<256>::SMEM, pdl, s, tk, tv,
                  aa);
  else if (hd == 512)  // scores on mma.sync, O in TMEM (tcgen05)
    e = launch_ex(attn_verify_hy_kernel, nkv * S, vhy::THREADS, vhy::SMEM, pdl, s, tk, tv, aa);
  else
    e = cudaErrorInvalidValue;  // every kernel is sized for its head dim: none other is launched
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "verify attention launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }
  // (2b) combination of the split records
  const int rpw = hd <= 256 ? 256 / hd : 1;  // query rows per merge CTA
  const size_t msmem = (size_t)rpw * S * sizeof(float2);
  const int mgrid = (c.L * G + rpw - 1) / rpw;
  tb("verify_attn_merge");
  if (hd == 64)
    e = launch_ex2(attn_verify_merge_kernel<64>, dim3(mgrid, nkv), 128, msmem, pdl, s, 1, aa);
  else if (hd == 128)
    e = launch_ex2(attn_verify_merge_kernel<128>, dim3(mgrid, nkv), 128, msmem, pdl, s, 1, aa);
  else if (hd == 256)
    e = launch_ex2(attn_verify_merge_kernel<256>, dim3(mgrid, nkv), 128, msmem, pdl, s, 1, aa);
  else if (hd == 512)
    e = launch_ex2(attn_verify_merge_kernel<512>, dim3(mgrid, nkv), 128, msmem, pdl, s, 1, aa);
  else
    e = cudaErrorInvalidValue;
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "verify attention merge launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }

  // (3) o_proj + residual
  VGemmArgs oa{};
  oa.bops = v->bo;
  oa.wt = reinterpret_cast<const uint8_t*>(c.wo);
  oa.g.batch = c.L;
  oa.g.x = c.x;
  oa.g.xin = c.o_f32;
  oa.g.R = H / 16;
  oa.g.err = c.err;
  oa.g.out = c.out;
  oa.g.out_tap = c.out_tap;
  oa.g.y_post = c.w_post ? v->y_post : nullptr;
  oa.rows = H;
  oa.K = nh * hd;
  oa.chunks = oa.K / kVK;
  const int otiles = H / kVM;
  oa.tpc = 1;
  oa.splits = gemm_splits(otiles, oa.chunks, c.num_sms, 1, v->max_clusters);
  tb("verify_oproj_gemm");
  e = launch_ex2(verify_gemm_kernel<kModeOProj>, dim3(otiles * oa.splits), 128, kVGemmSmem, pdl,
                 s, oa.splits, oa);
  te();
  if (e != cudaSuccess) {
    snprintf(msg, n, "verify o_proj launch: %s", cudaGetErrorString(e));
    return HFA_ECUDA;
  }
  if (c.w_post) {
    // (4) post-attention norm: out = x + y * w_post / sqrt(mean(y^2) + eps), one CTA a row
    tb("verify_post_norm");
    post_norm_rows_kernel<<<c.L, 256, 0, s>>>(v->y_post, c.x, c.w_post, d.hidden, d.eps, c.out,
                                              c.out_tap);
    e = cudaGetLastError();
    te();
    if (e != cudaSuccess) {
      snprintf(msg, n, "verify post-norm launch: %s", cudaGetErrorString(e));
      return HFA_ECUDA;
    }
  }
  return HFA_OK;
}

}  // namespace hfa
