// hfa_internal.h -- host-side declarations shared by the libhfa translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/hfa.h"

namespace hfa {

// Rows of the concatenated QKV projection: q, k and (without k_eq_v) v heads.
inline int qkv_rows(const hfa_layer_desc& d) {
  const int kv = (d.flags & HFA_F_K_EQ_V) ? 1 : 2;
  return (d.num_heads + kv * d.num_kv_heads) * d.head_dim;
}

// Epilogue arguments of the verify-block GEMMs (per-head norm + RoPE + KV append, and
// the residual), shared with the finishers of hfa_finish.cuh.
struct GemvArgs {
  int R;             // row groups of 16
  int batch;
  const __nv_bfloat16* x;  // QKV: layer input bf16 [B, cols]; OPROJ: residual bf16 [B, R*16]
  const float* w_in;       // QKV: input RMSNorm weight [cols]
  const float* xin;        // OPROJ: attention output f32 [B, cols]
  float eps;
  unsigned* err;
  // QKV finisher
  int nh, nkv, hd, C, ring;
  const float* w_q;
  const float* w_k;
  const float2* rope_g;    // [hd/2] (hi, lo) of theta^(-2i/hd) / (2 pi)
  const int* seq_pos;      // [B]
  int v_unit_norm;
  int k_eq_v;              // the key finisher also writes V = unit RMSNorm of the raw K
  int kv_only;             // rows of query heads are skipped (context rows: K and V only)
  float* q_out;            // f32 [B, nh, hd]
  uint8_t* qx;             // nullable: the scaled q as the verify attention's tensor-core
                           // operand, [nkv][2 boxes][128 rows][128 B] (see finish_head_row)
  float qscale;            // scale folded into qx
  int G;                   // query heads per KV head
  __nv_bfloat16* k_cache;  // [B, nkv, C, hd]
  __nv_bfloat16* v_cache;
  float* k_tap;            // nullable f32 [B, nkv, hd]
  float* v_tap;
  // OPROJ finisher
  __nv_bfloat16* out;      // bf16 [B, R*16]
  float* out_tap;          // nullable f32 [B, R*16]
  float* y_post;           // nullable f32 [B, R*16]: y kept for the post-attention norm pass
  // verify rows: row b of the GEMV is token b of sequence 0 at position base_pos + b
  int rows_are_tokens;
  int base_pos;
};

struct AttnArgs {
  const float* q;      // f32 [B*Lq, nh, hd]
  const int* seq_pos;  // [B]
  int B, nh, nkv, hd, C;
  int sliding, window, ring;
  float qscale;        // folded into q: scale*log2(e) (no softcap) or scale/softcap
  float cap_log2;      // softcap*log2(e), 0 = no softcap
  int splits;          // S per (sequence, kv head)
  int chunk;           // keys per split
  float* part;         // [B*nkv][S][8][hd + 4]: O[hd], m, l, pad
  int* ticket;         // [B*nkv]
  float* o;            // f32 [B, nh, hd]
  unsigned* err;
};

enum GemvMode { kModeQKV = 0, kModeOProj = 1 };

// One Q8_0 projection in the layout of the persistent decode-step kernel: 16 x 32 tiles
// of 544 bytes (512 bytes of biased int8 in MMA operand order, then 8 half2 scales),
// ordered (k-split s, row group r, block bb) so that the row groups one CTA owns in one
// k-split are a single contiguous byte range.
constexpr int kQ8TileBytes = 544;
struct StepGemv {
  const uint8_t* w;  // [S][R][nbs] tiles
  int R;             // row groups of 16 rows
  int nb;            // 32-column blocks per row
  int nbs;           // blocks per k-split
  int S;             // k-splits (nb / nbs), at most the grid size
  int ips;           // work items (nbs tiles each) per ring stage
};

// Arguments of the persistent decode-step kernel (one CTA per SM, cooperative launch).
struct StepArgs {
  StepGemv qkv, o;
  const __nv_bfloat16* x;  // layer input bf16 [B, H]
  const float* w_in;       // input RMSNorm weight [H]
  const float* w_q;        // per-head norm weights [hd]
  const float* w_k;
  const float2* rope_g;    // [hd/2] (hi, lo) of theta^(-2i/hd) / (2 pi)
  const int* seq_pos;      // [B]
  __nv_bfloat16* k_cache;  // [B, nkv, C, hd]
  __nv_bfloat16* v_cache;
  unsigned long long* qkv_part;  // [qkv.S][B][(nh + 2 nkv) hd]: f32 bits | step tag << 32
  float* rec;              // f32 [(grid + B nkv)][8][hd + 4]: (O, m, l) per key range
  unsigned long long* y_part;    // [o.S][B][H]: f32 bits | step tag << 32
  float* o_attn;           // f32 [B, nh, hd]: attention output (combined records)
  unsigned long long* gbar;  // grid barrier arrivals: only grows, one per CTA per step, so
                             // it also numbers the steps (graph replays included)
  unsigned* err;
  float* q_tap;            // nullable f32 [B, nh, hd] (q after RoPE)
  float* k_tap;            // nullable f32 [B, nkv, hd]
  float* v_tap;
  float* out_tap;          // nullable f32 [B, H]
  __nv_bfloat16* out;      // bf16 [B, H]
  const uint8_t* next_qkv_w;  // nullable: QKV tiles (same layout) of the layer that runs next
  int stall;               // test hook: CTA 0's consumers wait on a barrier nothing completes
  const float* w_post;     // nullable f32 [H]: post-attention RMSNorm of the o_proj output
  unsigned long long* post_part;  // [grid][2] tagged partial sum(y^2) (with w_post)
  unsigned long long* stamps;  // nullable [grid][16]: %globaltimer at fixed points (see kStamp*)
  int B, H, nh, nkv, C, sliding, window, ring, v_unit_norm;
  int k_eq_v;              // no V rows: the K job also writes V = unit RMSNorm of raw K
  long long cache_rows;    // B * nkv * C: rows of the [rows, hd] view of each cache
  float eps;
  float qscale;            // scale * log2(e), or scale / softcap with a softcap
  float cap_log2;          // softcap * log2(e), 0 = no softcap
};

// One GEMV of the persistent FFN kernel: Q8_0 tiles in the order [k-split][row group]
// [block] (see launch_repack_q8_0_split), streamed in ring stages of `rgs` row groups of
// one k-split.
struct FfnPhase {
  const uint8_t* w;  // tiles
  int R;             // row groups of 16 rows (phase 1: gate and up interleaved, 2 I / 16)
  int nbs;           // blocks (tiles) per k-split
  int S;             // k-splits
  int rgs;           // row groups per ring stage: 1, 2, 4 or 8 (even in phase 1)
  int stages;        // S * ceil(R / rgs)
};

// Arguments of the persistent FFN kernel (one CTA per SM, cooperative launch).
struct FfnArgs {
  FfnPhase p1, p2;               // [Wg; Wu] (interleaved row groups) and Wd
  const __nv_bfloat16* h;        // bf16 [B, H]: the FFN input and the residual
  const float* w_pre;            // f32 [H]: pre-FF RMSNorm weight
  const float* w_post;           // f32 [H]: post-FF RMSNorm weight
  const float* scalar;           // f32 [scalar_len]: the layer scalar
  int scalar_len;                // 1 or H
  unsigned long long* part1;     // [p1.S][B][2 I]: gate rows, then up rows (tagged f32)
  unsigned long long* part2;     // [p2.S][B][H] (tagged f32)
  unsigned long long* post_part; // [grid][2]: tagged partial sum(d^2)
  unsigned long long* ctr;       // launches x grid: numbers the steps (tags)
  unsigned* err;
  __nv_bfloat16* out;            // bf16 [B, H]
  float* out_f32;                // nullable f32 [B, H]
  float* a_tap;                  // nullable f32 [B, I]: GELU(gate) * up
  unsigned long long* stamps;    // nullable [grid][16]: %globaltimer at fixed points
  int B, H, I;
  float eps;
};

// Optional per-launch event timing (the layer's hfa_set_kernel_timing); begin/end
// bracket one kernel launch on `s`.
struct LaunchTimer {
  virtual void begin(cudaStream_t s, const char* name) = 0;
  virtual void end(cudaStream_t s) = 0;
  virtual ~LaunchTimer() {}
};

// message returned by hfa_last_error(NULL) on this thread
void set_thread_error(const char* msg);

cudaError_t launch_repack_q8_0_split(const uint8_t* src, int rows, int cols, uint8_t* dst,
                                     int row_group0, int R_total, int nbs, cudaStream_t s,
                                     int rg_stride = 1);
// bf16 [rows, K] (rows from s0, then s1, then s2) -> 128 x 64 tiles of 16 KB in the
// 128-byte-swizzled order of the verify GEMM's shared-memory stages
cudaError_t launch_repack_bf16_tiles(const __nv_bfloat16* s0, int n0, const __nv_bfloat16* s1,
                                     int n1, const __nv_bfloat16* s2, int rows, int K,
                                     uint8_t* dst, cudaStream_t s);
// the decode step: grid = one CTA per SM (cooperative), ntiles = gemv batch tiles
cudaError_t launch_step(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hd,
                        int grid, cudaStream_t s);
size_t step_smem_bytes();
int step_keys_per_tile(int hd);  // keys of one K/V tile of the decode-step kernel
size_t step_stage_bytes();
int step_threads();
int step_batch_tiles(int batch);

// the FFN step: grid = one CTA per SM (cooperative); the plan of one GEMV phase for
// batches up to 4 * nt_max rows, false when no plan fits the kernel's buffers
bool plan_ffn_phase(FfnPhase* p, int R, int nb, bool pairs, int nt_max, int grid);
bool ffn_plan_fits(const FfnPhase& p, int nt);  // the kernel for nt batch tiles holds it
cudaError_t launch_ffn(const FfnArgs& a, int grid, cudaStream_t s);
int ffn_max_outputs_per_cta();  // B * H / grid must not exceed it

cudaError_t launch_attn(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        int grid, bool pdl, cudaStream_t s);

// flash-decode over the quantised KV cache (k_tq.cu, k_tq_mma.cu)
struct TqAttnArgs {
  const float* q;         // [B, nh, hd] after norm and RoPE
  const int* seq_pos;     // [B]
  const uint8_t* k_codes;  // [B, nkv, C, code_bytes], or NULL (hybrid: raw bf16 keys)
  const float* k_norms;   // [B, nkv, C, blocks]
  const __nv_bfloat16* k_raw;  // hybrid: [B, nkv, C, hd]
  const uint8_t* v_codes;
  const float* v_norms;
  const float* centroids;  // [levels]
  const float* signs;      // [hd]
  float* part;             // [units * splits][8][hd + 4]: O (rotated), m, l
  int* ticket;             // [units]
  // two-level merge (tensor-core kernel): the chunks of a unit form groups of `group`; the
  // last CTA of a group folds its records into part1 [units][16][8][hd + 4] (ticket1
  // [units][16]), the last of those folds the groups'
  float* part1;
  int* ticket1;
  int group;
  float* o;                // [B, nh, hd]
  unsigned* err;
  int B, nh, nkv, C, sliding, window, ring, levels;
  int splits, chunk;       // key chunks per unit, keys per chunk
  float qscale;            // scale * log2 e, or scale / softcap
  float cap_log2;          // softcap * log2 e, 0 = none
};
// the tensor-core kernel: head dims 64, 128, 256 and 512, codes of 4 or 8 stored bits, K
// coded or raw bf16 (kraw, up to hd 256); tk / tv describe the K and V arrays as 2-D TMA
// views; one CTA of tq_mma_threads(hd) per SM, chunks of any length
bool tq_mma_supported(int hd, int sbits, bool kraw);
int tq_mma_keys_per_stage(int hd);
int tq_mma_threads(int hd);
cudaError_t launch_tq_attn_mma(const TqAttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                               int hd, int sbits, bool kraw, int grid, cudaStream_t s);
int attn_keys_per_stage(int hd);
size_t attn_smem_bytes(int hd);
int attn_threads(int hd);
int attn_record_floats(int hd);  // floats of one chunk record (8 heads x (hd + 4))

}  // namespace hfa

// 2-D views of a cache for the TMA unit (hfa_api.cu): bf16 [rows, hd] in boxes of 64 x
// box_rows with 128-byte swizzle; bytes [rows, row_bytes] in boxes of box_bytes x box_rows
// (box_bytes 32, 64 or 128, the swizzle of the same width)
hfa_status hfa_encode_kv_map(CUtensorMap* map, void* base, int rows, int hd, int box_rows);
hfa_status hfa_encode_u8_map(CUtensorMap* map, const void* base, long long rows, int row_bytes,
                             int box_bytes, int box_rows);
