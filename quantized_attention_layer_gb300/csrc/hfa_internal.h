// hfa_internal.h -- host-side declarations shared by the libhfa translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/hfa.h"

namespace hfa {

// Repacked Q8_0 matrix: 16-row x 32-column tiles of 512 bytes, laid out so that one
// 16-byte load per lane gives that lane's operand registers of two m16n8k16 MMAs.
struct Q8Tiles {
  uint8_t* q = nullptr;  // [rows/16][cols/32][32 lanes][16 B], bytes hold q + 128
  __half2* d = nullptr;  // [rows/16][cols/32][8]: (d[row g], d[row g + 8])
  int rows = 0, cols = 0;
};

// Arguments of the dequantising GEMV kernels (both modes).
struct GemvArgs {
  const uint8_t* wq;
  const __half2* wd;
  int R;             // row groups of 16
  int nb;            // 32-column blocks per row
  int S;             // k splits
  int nbs;           // blocks per split (nb / S): the tiles of one work item
  long long tiles;   // S * R * nbs
  int batch;
  int cols;
  const __nv_bfloat16* x;  // QKV: layer input bf16 [B, cols]; OPROJ: residual bf16 [B, R*16]
  const float* w_in;       // QKV: input RMSNorm weight [cols]
  const float* xin;        // OPROJ: attention output f32 [B, cols]
  float eps;
  float* acc;              // f32 [B, R*16], zero between launches
  int* ticket;             // QKV: per head; OPROJ: per row group
  unsigned* err;
  // QKV finisher
  int nh, nkv, hd, C, ring;
  const float* w_q;
  const float* w_k;
  const float2* rope_g;    // [hd/2] (hi, lo) of theta^(-2i/hd) / (2 pi)
  const int* seq_pos;      // [B]
  int v_unit_norm;
  float* q_out;            // f32 [B, nh, hd]
  __nv_bfloat16* k_cache;  // [B, nkv, C, hd]
  __nv_bfloat16* v_cache;
  float* k_tap;            // nullable f32 [B, nkv, hd]
  float* v_tap;
  // OPROJ finisher
  __nv_bfloat16* out;      // bf16 [B, R*16]
  float* out_tap;          // nullable f32 [B, R*16]
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

// Optional per-launch event timing (the layer's hfa_set_kernel_timing); begin/end
// bracket one kernel launch on `s`.
struct LaunchTimer {
  virtual void begin(cudaStream_t s, const char* name) = 0;
  virtual void end(cudaStream_t s) = 0;
  virtual ~LaunchTimer() {}
};

// message returned by hfa_last_error(NULL) on this thread
void set_thread_error(const char* msg);

// TMA descriptor of a row-major bf16 matrix [rows, inner] with boxes of
// box_inner x box_rows and the 128-byte swizzle (box_inner * 2 must be 128)
bool encode_bf16_2d(CUtensorMap* map, void* base, int inner, int rows, int box_inner,
                    int box_rows);

cudaError_t launch_repack_q8_0(const uint8_t* src, int rows, int cols, Q8Tiles* dst,
                               size_t row_offset_rows, cudaStream_t s);
cudaError_t launch_gemv(int mode, const GemvArgs& a, int grid, int threads, size_t smem,
                        bool pdl, cudaStream_t s);
size_t gemv_smem_bytes(int batch, int blocks_per_cta_max);
int gemv_ntiles(int batch);
int gemv_items_per_cta();

cudaError_t launch_attn(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        int grid, bool pdl, cudaStream_t s);
int attn_keys_per_stage(int hd);
size_t attn_smem_bytes(int hd);
int attn_threads(int hd);
int attn_record_floats(int hd);  // floats of one chunk record (8 heads x (hd + 4))

}  // namespace hfa
