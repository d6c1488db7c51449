/*
 * hfa_oracle.h -- plain, slow, fp64 CPU oracle for one Gemma-style attention block.
 *
 * TEST INFRASTRUCTURE ONLY.  This oracle exists to check the CUDA library.  Only the
 * test suite, the smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or helper with the CUDA library, and the library
 * never calls it.
 *
 * Every step is the plain definition, accumulated in double precision from the exact
 * input values (bf16 -> double, Q8_0 -> (double)fp16(d) * q).  Sources, by page:
 *   [P1] hf2q docs.rs page "src/inference/models/gemma4/gpu_full_attn.rs",
 *        function encode_one_layer (the per-layer decode encoder);
 *   [P2] hf2q docs.rs page "src/inference/models/gemma4/model.rs";
 *   [P3] hf2q docs.rs page "src/inference/spec_decode/dflash/forward.rs".
 *
 * Parity pins: every function below is pinned by a CPU test against a closed form,
 * an invariant, brute force or a library routine (see tests/test_oracle_*.py).
 * The whole-layer outputs have no printed values on the pages to compare with.
 */
#ifndef HFA_ORACLE_H
#define HFA_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int hidden, num_heads, num_kv_heads, head_dim;
  int layer_type;      /* 0 = sliding window, 1 = full (global) attention */
  int window;          /* sliding window W: keys with P-W < p <= P are visible */
  double eps;          /* RMSNorm epsilon (input norm and per-head norms) */
  double rope_theta;   /* RoPE base */
  double attn_scale;   /* logit scale (1.0 on the Gemma decode path) */
  double softcap;      /* 0 = off; else s -> cap * tanh(s / cap) */
  int kv_capacity;     /* slots per (sequence, kv head) */
  int ring;            /* 1: slot = pos % capacity; 0: slot = pos */
  int v_unit_norm;     /* 1: V is RMS-normalised per head with unit weight */
  int weights_bf16;    /* 0: Q/K/V/O are Q8_0 blocks; 1: dense bf16 [out, in] */
  /* Gemma decode variants [P1 fused head norm + RoPE with freq factors on global layers,
   * GPU V norm, fused post-attention norm + residual add; P2 v_proj None when k_eq_v,
   * rope_freqs.weight, post_attention_norm.weight]: */
  int k_eq_v;                      /* 1: no V projection; V = unit RMSNorm of the raw K */
  const float* rope_freq_factors;  /* NULL, or [hd/2]: phi_i = pos * theta^(-2i/hd) / f_i */
  const float* w_post;             /* NULL, or [hidden]: out = x + RMSNorm(y) * w_post */
  /* [P3 dispatch_dflash_decoder_layer_attention: bidirectional within the block on full
   * layers, causal + window on sliding ones]: 1 = every row of a verify block sees the
   * whole block on a full layer */
  int block_bidir;
} orc_desc;

/* ---- scalar formats ---- */
double orc_bf16_to_f64(uint16_t b);
uint16_t orc_f64_to_bf16(double v);          /* round to nearest, ties to even */
double orc_f16_to_f64(uint16_t h);           /* IEEE binary16, subnormals included */

/* ---- Q8_0 blocks [P2, Q8_0 lm_head re-quantiser]: per 32 values, 2-byte LE fp16
 *      scale d followed by 32 int8 q; value = d * q ---- */
void orc_q8_0_dequant_row(const uint8_t* row_blocks, int cols, double* out);
/* y = W x, W given as Q8_0 rows: each row is dequantised densely, then dotted. */
void orc_q8_0_matvec(const uint8_t* blocks, int rows, int cols, const double* x, double* y);
/* same product, block by block: y_r = sum_b d_rb * sum_i q_rbi x_{32b+i} */
void orc_q8_0_matvec_blockwise(const uint8_t* blocks, int rows, int cols, const double* x,
                               double* y);
/* y = W x with dense bf16 W [rows, cols] */
void orc_bf16_matvec(const uint16_t* w, int rows, int cols, const double* x, double* y);

/* ---- RMSNorm [P1 pre-attention norm; P3 dispatch_dflash_head_norm]:
 *      y = x * w / sqrt(mean(x^2) + eps); w == NULL means unit weight ---- */
void orc_rmsnorm(const double* x, const float* w, int n, double eps, double* y);

/* ---- RoPE, NeoX pairing (i, i + hd/2) [P1 fused head norm + RoPE (half_rope = hd/2);
 *      P3 dispatch_dflash_rope]: phi_i = pos * theta^(-2i/hd) ---- */
void orc_rope_neox(double* u, int hd, double pos, double theta);
/* the same with per-pair frequency factors (NULL: none): phi_i = pos * theta^(-2i/hd) / f_i */
void orc_rope_neox_ff(double* u, int hd, double pos, double theta, const float* ff);

/* ---- KV slots and visibility [P1 dense decode SDPA: write_slot and kv_seq_len] ---- */
long orc_kv_slot(long pos, long capacity, int ring);
/* key at logical position p is visible to the query at position P */
int orc_key_visible(long p, long P, int sliding, long window);
/* logical position held by a slot after position P was appended, -1 if none */
long orc_slot_position(long slot, long P, long capacity, int ring);

/* ---- attention of one query over an explicit list of cache rows (bf16) ----
 * s_j = scale * q.K_j; optional softcap; p = softmax(s); o = sum_j p_j V_j.
 * weights (nullable) receives p_j. */
void orc_attend(const double* q, const uint16_t* k_rows, const uint16_t* v_rows, int hd,
                const long* rows, long n, double scale, double softcap, double* weights,
                double* o);

/* ---- the decode step for B independent sequences ----
 * x bf16 [B, H]; seq_pos int32 [B]; caches bf16 [B, nkv, C, hd] updated in place.
 * Outputs (each nullable): q [B, nh, hd] after norm+RoPE; k, v [B, nkv, hd] before
 * rounding to bf16; attn [B, nh, hd]; out [B, H] (double) and out_bf16 [B, H].
 * Returns 0, or -1 on invalid arguments. */
int orc_decode_step(const orc_desc* d, const void* wq, const void* wk, const void* wv,
                    const void* wo, const float* w_in, const float* w_q, const float* w_k,
                    const uint16_t* x, const int32_t* seq_pos, int B, uint16_t* k_cache,
                    uint16_t* v_cache, double* q_out, double* k_out, double* v_out,
                    double* attn_out, double* out, uint16_t* out_bf16);

/* ---- the multi-token verify block (one sequence) ----
 * L tokens at positions base_pos .. base_pos+L-1.  All L K/V rows are appended first;
 * row i then attends causally to positions <= base_pos + i (within the window when
 * sliding).  Shapes as in orc_decode_step with B replaced by L for x/q/k/v/attn/out;
 * the caches are [1, nkv, C, hd]. */
int orc_verify_block(const orc_desc* d, const void* wq, const void* wk, const void* wv,
                     const void* wo, const float* w_in, const float* w_q, const float* w_k,
                     const uint16_t* x, int L, int base_pos, uint16_t* k_cache,
                     uint16_t* v_cache, double* q_out, double* k_out, double* v_out,
                     double* attn_out, double* out, uint16_t* out_bf16);

/* ---- the drafter's context rows [P3 dispatch_dflash_decoder_layer_attention]: S rows
 * x_ctx bf16 [S, H] (already normalised by the model: no input RMSNorm) projected by Wk
 * and Wv only, k_norm + RoPE on k at positions base_pos .. base_pos+S-1, V as in the decode
 * step (unit-normed with v_unit_norm or k_eq_v, the raw K with k_eq_v), appended as bf16.
 * k_out, v_out (nullable) [S, nkv, hd] before rounding.  Returns 0, -1 on bad arguments. */
int orc_ctx_append(const orc_desc* d, const void* wk, const void* wv, const float* w_k,
                   const uint16_t* x_ctx, int S, int base_pos, uint16_t* k_cache,
                   uint16_t* v_cache, double* k_out, double* v_out);

/* ---- the dense FFN half of the layer [P1 encode_one_layer, groups B8-B11 and the
 * end-of-layer norm: pre-FF RMSNorm, dense gate and up projections, fused_gelu_mul, the
 * down projection, the post-FF RMSNorm added to the residual, the layer scalar]:
 *   n = h * w_pre / sqrt(mean(h^2) + eps);  a = gelu(Wg n) * (Wu n);  d = Wd a;
 *   out = (h + d * w_post / sqrt(mean(d^2) + eps)) * s,
 * gelu(x) = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), s the layer scalar (one value,
 * or one per channel when scalar_len == H).  Wg, Wu Q8_0 [I, H]; Wd Q8_0 [H, I];
 * h bf16 [B, H].  Outputs (nullable): a [B, I], out [B, H] and its bf16 rounding. */
double orc_gelu_tanh(double x);
int orc_ffn_step(int H, int I, double eps, const uint8_t* wg, const uint8_t* wu,
                 const uint8_t* wd, const float* w_pre, const float* w_post,
                 const float* scalar, int scalar_len, const uint16_t* h, int B, double* a_out,
                 double* out, uint16_t* out_bf16);

/* number of OpenMP threads the oracle uses (1 when built without OpenMP) */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
