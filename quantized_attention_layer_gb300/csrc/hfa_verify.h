// hfa_verify.h -- the multi-token verify block (host interface between hfa_api.cu and
// the verify kernels).
#pragma once
#include <cuda_runtime.h>

#include "hfa_internal.h"

namespace hfa {

struct VerifyState;

struct VerifyCall {
  const hfa_layer_desc* d;
  cudaStream_t stream;
  const __nv_bfloat16* x;  // [L, H]
  int L;
  int base_pos;
  __nv_bfloat16* k_cache;  // [1, nkv, C, hd]
  __nv_bfloat16* v_cache;
  __nv_bfloat16* out;      // [L, H]
  const __nv_bfloat16* wqkv;  // [qkv_rows(d), H]: q, k and (without k_eq_v) v rows, as
                              // 128 x 64 tiles (launch_repack_bf16_tiles)
  const __nv_bfloat16* wo;    // [H, nh hd], as 128 x 64 tiles
  const float* w_in;
  const float* w_q;
  const float* w_k;
  const float2* rope_g;
  float* q_f32;   // [L, nh, hd]
  float* o_f32;   // [L, nh, hd]
  float* k_tap;   // nullable [L, nkv, hd]
  float* v_tap;
  float* out_tap; // nullable [L, H]
  const float* w_post;  // nullable [H]: out = x + RMSNorm(y) * w_post
  unsigned* err;
  int num_sms;
  LaunchTimer* timer;  // nullable; when set, launches are timed and not PDL-chained
  int bidir;           // full layer: every row sees the whole block (the drafter's blocks)
};

hfa_status verify_create(const hfa_layer_desc& d, int num_sms, VerifyState** out);
void verify_free(VerifyState* v);
// after a device error: the QKV GEMMs' launch counters and tagged partial sums restart
hfa_status verify_reset(VerifyState* v, cudaStream_t s);
const char* verify_error();
hfa_status verify_run(VerifyState* v, const VerifyCall& c, char* msg, int msg_len);
// the drafter's context rows: c.x holds c.L rows, projected by Wk and Wv only (no input
// norm), k_norm + RoPE, appended at c.base_pos ..; q, attention and o_proj are not run
hfa_status verify_ctx_append(VerifyState* v, const VerifyCall& c, char* msg, int msg_len);

}  // namespace hfa
