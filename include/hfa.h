/*
 * hfa.h -- C ABI of libhfa: the single-token decode step and the multi-token verify
 * block of one Gemma-style attention layer on an NVIDIA GB300 (sm_103a), attention over
 * a quantised KV cache, and the layer's dense feed-forward half.
 *
 * Sources of the operation (hf2q documentation pages):
 *   "gemma4/gpu_full_attn.rs", encode_one_layer: the per-layer decode encoder --
 *     pre-attention norm, the Q/K/V projections (dispatch_qmatmul), the fused per-head
 *     norm + RoPE, the GPU V norm, the dense KV copy, dense flash_attn_vec (main +
 *     reduce) and the O projection.  FlashAttnVecParams gives the attention
 *     parameters: num_heads, num_kv_heads, head_dim, kv_seq_len, kv_capacity, scale,
 *     mask_type, sliding_window, softcap.
 *   "gemma4/model.rs": the Q8_0 block format (Q8_0 lm_head re-quantiser), the dense
 *     KV buffer layout [n_kv_heads, capacity, head_dim] with sliding layers as rings
 *     of capacity = sliding window, and the dense tree-verify entry point.
 *   "gemma4/gpu_full_attn.rs", encode_one_layer, the dense MLP and the end of the
 *     layer: pre- and post-feed-forward RMSNorm, gate/up/down projections, GELU(gate) *
 *     up, the residual add and the layer scalar (hfa_ffn_*).
 *   "spec_decode/dflash/forward.rs": per-head RMSNorm over rows = L * n_heads, NeoX
 *     RoPE with a position offset, the logit softcap tanh(s / cap) * cap, the residual
 *     add, and SDPA of an L-row block over the cache (all rows of the block appended).
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are CUDA device pointers on the current device; pointers
 *     named *_host are host pointers.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream).  Work is enqueued on `stream` and returns before it completes,
 *     unless the entry point says otherwise.
 *   - All argument checks run on the host before anything is launched; a rejected
 *     call launches nothing and touches no device memory.  The reason is available
 *     from hfa_last_error().
 *   - No entry point allocates device memory except the create functions
 *     (hfa_layer_create, hfa_tq_create, hfa_ffn_create).
 *   - bf16 = IEEE bfloat16 bit pattern (uint16), row-major, densely packed.
 */
#ifndef HFA_H
#define HFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hfa_layer hfa_layer; /* opaque; owned by the library */

typedef enum {
  HFA_OK = 0,
  HFA_EINVAL = -1,       /* bad argument: null pointer, shape, flag combination */
  HFA_ERANGE = -2,       /* a position outside the cache or the layer's limits */
  HFA_ENOMEM = -3,       /* device allocation failed (the create functions only) */
  HFA_ECUDA = -4,        /* a CUDA call failed; hfa_last_error has the CUDA message */
  HFA_EUNSUPPORTED = -5, /* valid request this library does not implement */
  HFA_EDEVICE = -6,      /* no usable sm_103 device, or a device-side check failed */
} hfa_status;

typedef enum { HFA_SLIDING = 0, HFA_FULL = 1 } hfa_layer_type;

/* flags */
#define HFA_F_V_UNIT_NORM 0x1u  /* V gets a per-head RMSNorm with unit weight (GPU V norm) */
#define HFA_F_WEIGHTS_BF16 0x2u /* Q/K/V/O are dense bf16 [out, in] instead of Q8_0 */
#define HFA_F_RING 0x4u         /* sliding ring buffer: slot = pos % kv_capacity */
#define HFA_F_DEBUG_TAPS 0x8u   /* keep fp32 copies of q, k, v, attention and output */
#define HFA_F_K_EQ_V 0x10u      /* no V projection: V = per-head unit RMSNorm of the raw K
                                   (Gemma global layers; model.rs, v_proj None when k_eq_v) */
#define HFA_F_BLOCK_BIDIR 0x20u /* verify blocks of a FULL layer attend bidirectionally
                                   within the block (the drafter's full-attention layers,
                                   dflash/forward.rs); sliding layers stay causal */

typedef struct {
  int hidden;       /* H: a multiple of 32 (whole Q8_0 blocks; HFA_EINVAL otherwise);
                       multiples of 64 are supported (HFA_EUNSUPPORTED otherwise) */
  int num_heads;    /* query heads nh */
  int num_kv_heads; /* key/value heads nkv; nh % nkv == 0 and nh / nkv <= 8 */
  int head_dim;     /* hd in {64, 128, 256, 512}; 512 is the global layers' width */
  int layer_type;   /* hfa_layer_type */
  int window;       /* sliding window W (keys with P-W < p <= P visible); SLIDING only */
  float eps;        /* RMSNorm epsilon of the input norm and the per-head norms */
  float rope_theta; /* RoPE base; NeoX pairing (i, i + hd/2), phi_i = P * theta^(-2i/hd) */
  float attn_scale; /* logit scale; 1.0 on the Gemma decode path */
  float softcap;    /* 0 = off; else logits s -> softcap * tanh(s / softcap) */
  int kv_capacity;  /* C: slots per (sequence, kv head); a ring needs C == window */
  int max_batch;    /* largest batch a decode step may pass (sizes the scratch) */
  int max_verify_len; /* largest L of hfa_verify_block; 0 = verify not used */
  unsigned flags;   /* HFA_F_* */
} hfa_layer_desc;

/*
 * Create a layer.  Weights are read from device memory and copied (Q8_0: re-laid out
 * for coalesced loads; the values are untouched) into library-owned memory, so the
 * caller may free them when the call returns.  The call synchronises `stream`.
 *
 *   wq_dev [nh*hd, H], wk_dev [nkv*hd, H], wv_dev [nkv*hd, H], wo_dev [H, nh*hd]
 *     (wv_dev is ignored, and may be NULL, with HFA_F_K_EQ_V):
 *     Q8_0: rows of H/32 (resp. nh*hd/32) blocks of 34 bytes -- fp16 scale d (little
 *     endian) then 32 int8 q, value = d * q (Q8_0 lm_head re-quantiser, model.rs).
 *     With HFA_F_WEIGHTS_BF16: dense bf16, row-major [out, in].
 *   w_in_dev f32 [H], w_q_dev f32 [hd], w_k_dev f32 [hd]: RMSNorm weights, used as
 *     y = x * w / sqrt(mean(x^2) + eps).
 * Errors: HFA_EINVAL (shape, flags), HFA_EUNSUPPORTED (a shape this library does not
 * cover), HFA_EDEVICE (no sm_103 device), HFA_ENOMEM, HFA_ECUDA.  *out is NULL on
 * error.
 */
hfa_status hfa_layer_create(const hfa_layer_desc* desc, const void* wq_dev, const void* wk_dev,
                            const void* wv_dev, const void* wo_dev, const float* w_in_dev,
                            const float* w_q_dev, const float* w_k_dev, void* stream,
                            hfa_layer** out);

/*
 * One decode step for `batch` independent sequences (encode_one_layer, attention half):
 *   n = RMSNorm(x) ; [q;k;v] = W n ; q,k = per-head RMSNorm + RoPE at seq_pos ;
 *   append bf16(k), bf16(v) at slot seq_pos (linear) or seq_pos % C (ring) ;
 *   o = softmax(scale * q K^T [softcap] [window mask]) V over the visible keys ;
 *   out = x + Wo o   (x + RMSNorm(Wo o) * w_post with hfa_set_post_norm).
 *
 *   x_dev        bf16 [batch, H]
 *   seq_pos_dev  int32 [batch], device copy read by the kernels
 *   seq_pos_host int32 [batch], host copy of the same values, used for validation
 *   k_cache_dev, v_cache_dev  bf16 [batch, nkv, C, hd]; one slot per sequence and
 *                kv head is written in place, every other slot is only read
 *   out_dev      bf16 [batch, H]
 * Linear caches need 0 <= seq_pos < C (HFA_ERANGE otherwise).  Requires Q8_0 weights.
 * The cache must hold the earlier positions of each sequence: positions
 * max(0, P-W+1) .. P-1 (sliding) or 0 .. P-1 (full).
 * The step is one cooperative launch of at most one CTA per SM (one per SM unless the
 * layer's largest step has less work: a tiny layer runs on a few); it fails with HFA_ECUDA when the
 * device cannot hold that grid at once (e.g. SMs taken by another context).  It is
 * launched with programmatic dependent launch: it may start while the previous kernel on
 * `stream` finishes, reads nothing but the layer's own weights until that kernel has
 * completed, and lets the next kernel on `stream` start the same way.  Steps on
 * one layer handle must not overlap on the GPU (they share the layer's scratch).
 */
hfa_status hfa_decode_step(hfa_layer* layer, void* stream, const void* x_dev,
                           const int32_t* seq_pos_dev, const int32_t* seq_pos_host, int batch,
                           void* k_cache_dev, void* v_cache_dev, void* out_dev);

/*
 * The same decode step taking its per-step input and output in host memory:
 * copies x_host and seq_pos_host to library staging buffers on `stream`, runs the
 * step, copies the result back to out_host and synchronises `stream` before
 * returning.  x_host bf16 [batch, H], out_host bf16 [batch, H] (pinned memory gives
 * asynchronous copies; pageable memory works but is slower).  The caches stay in
 * device memory.
 */
hfa_status hfa_decode_step_host(hfa_layer* layer, void* stream, const void* x_host,
                                const int32_t* seq_pos_host, int batch, void* k_cache_dev,
                                void* v_cache_dev, void* out_host);

/*
 * Multi-token verify block, one sequence (the dense tree-verify entry of model.rs;
 * the block form of forward.rs): L tokens at positions base_pos .. base_pos+L-1.
 * All L K/V rows are appended; row i attends to cache positions <= base_pos + i
 * (and within the window when sliding).  Accepting or rolling back the appended rows
 * is the caller's business.
 *   x_dev bf16 [L, H]; k_cache_dev, v_cache_dev bf16 [1, nkv, C, hd]; out_dev bf16 [L, H].
 * Needs a linear cache with base_pos + L <= C and 1 <= L <= max_verify_len.
 * Errors: HFA_EINVAL for NULL or unaligned (16-byte) pointers, for L outside
 * [1, max_verify_len] or a layer made with max_verify_len = 0; HFA_ERANGE for positions
 * past the cache; HFA_EUNSUPPORTED for a ring cache, a Q8_0 layer (the block runs on
 * bf16 weights, HFA_F_WEIGHTS_BF16) or L * (nh / nkv) > 64 query rows per KV head.  At
 * create, max_verify_len > 16 and projection sizes that are not multiples of 128 rows
 * are HFA_EUNSUPPORTED, and so is a cache of nkv * kv_capacity + 256 >= 2^31 rows (the
 * kernels address it in 32-bit rows).  The post-attention norm, RoPE frequency factors and
 * HFA_F_K_EQ_V apply as in the decode step.
 */
hfa_status hfa_verify_block(hfa_layer* layer, void* stream, const void* x_dev, int L,
                            int base_pos, void* k_cache_dev, void* v_cache_dev, void* out_dev);

/*
 * The drafter's context rows (spec_decode/dflash/forward.rs,
 * dispatch_dflash_decoder_layer_attention: k_ctx, v_ctx and their cache append): S rows
 * x_ctx_dev bf16 [S, H], already normalised by the drafter model (no input RMSNorm here),
 * projected by Wk and Wv only, k_norm and RoPE at positions base_pos .. base_pos+S-1, V as
 * in the block (unit-normed with HFA_F_V_UNIT_NORM or HFA_F_K_EQ_V), appended as bf16 at
 * those slots.  A drafter step is this call followed by hfa_verify_block of the L block
 * rows at base_pos + S (their K/V land past the committed context, in the slack the
 * caller does not commit), on a layer with HFA_F_BLOCK_BIDIR if it is a full layer, and
 * attn_scale 1/sqrt(hd).  Needs a bf16-weight layer (as hfa_verify_block) and
 * 1 <= S <= max_verify_len, base_pos + S <= kv_capacity.
 * Errors: HFA_EINVAL, HFA_ERANGE, HFA_EUNSUPPORTED (ring cache, Q8_0 layer), HFA_ECUDA.
 */
hfa_status hfa_ctx_append(hfa_layer* layer, void* stream, const void* x_ctx_dev, int S,
                          int base_pos, void* k_cache_dev, void* v_cache_dev);

/*
 * The attention step alone ("Dense flash_attn_vec" of encode_one_layer), for callers
 * that compute q themselves: split-K GQA flash-decode of one query per head over the
 * visible keys of a bf16 cache, optional softcap, log-sum-exp merge of the chunks.
 *   q_dev        f32 [batch, nh, hd]: queries after norm and RoPE (scale not applied)
 *   seq_pos_dev / seq_pos_host  int32 [batch]: the query positions (as in the decode step)
 *   k_cache_dev, v_cache_dev    bf16 [batch, nkv, C, hd], read only
 *   workspace_dev  device scratch of at least hfa_attention_workspace_bytes(desc, batch)
 *                  bytes, 16-byte aligned, all zero before its first use; each call leaves
 *                  it ready for the next (its counters return to zero).  Word 0 is a
 *                  device status word: non-zero means a bounded wait gave up (bit 0) or a
 *                  position was refused (bit 1).  Calls sharing a workspace must not
 *                  overlap on the GPU.
 *   o_dev        f32 [batch, nh, hd]
 * Errors come back as for hfa_layer_create (message via hfa_last_error(NULL)).
 */
typedef struct {
  int num_heads, num_kv_heads, head_dim; /* as in hfa_layer_desc */
  int layer_type, window, kv_capacity;
  float attn_scale, softcap;
  unsigned flags; /* HFA_F_RING or 0 */
} hfa_attn_desc;

size_t hfa_attention_workspace_bytes(const hfa_attn_desc* desc, int batch);
hfa_status hfa_attention_decode(const hfa_attn_desc* desc, void* stream, const float* q_dev,
                                const int32_t* seq_pos_dev, const int32_t* seq_pos_host,
                                int batch, const void* k_cache_dev, const void* v_cache_dev,
                                void* workspace_dev, size_t workspace_bytes, float* o_dev);

/*
 * hfa_attention_decode without a workspace argument, for callers that cannot allocate
 * device memory where they run attention (an engine that fixes all device memory at
 * start-up, a plugin whose host owns the allocator, code that must not let
 * cudaMalloc/cudaFree synchronise the device).  No counterpart on the documentation
 * pages: an interface addition of this library.
 * Its scratch is a file-scope device array of 4 MiB that every GPU loading the library
 * holds until exit.  Arguments and results are those of hfa_attention_decode; a batch
 * whose scratch (hfa_attention_workspace_bytes) exceeds 4 MiB is rejected with
 * HFA_ERANGE.  The first call on each device looks up the array's address (make it
 * before any stream capture).  Each call clears the array's counters on `stream`; all
 * calls share the array, so calls that overlap on the GPU race and must not be issued.
 * Neither device-side condition that hfa_attention_decode records in its status word (a
 * bounded wait that gave up, a position refused on the device, e.g. seq_pos_dev
 * disagreeing with seq_pos_host) is reported by this variant: the next call clears the
 * word, and the output of such a call is wrong without notice.  Callers that need that
 * check use hfa_attention_decode and read word 0 of their workspace.  The cached address
 * belongs to the device's context: after cudaDeviceReset (or any reset of the primary
 * context) this entry point must not be called again in the process.  Allocates nothing.
 */
hfa_status hfa_attention_decode_noalloc(const hfa_attn_desc* desc, void* stream,
                                        const float* q_dev, const int32_t* seq_pos_dev,
                                        const int32_t* seq_pos_host, int batch,
                                        const void* k_cache_dev, const void* v_cache_dev,
                                        float* o_dev);

/*
 * Quantised KV cache (TurboQuant): gpu_full_attn.rs, encode_one_layer -- the
 * Hadamard-quantize KV encode (sign pre-multiply, normalised FWHT, a norm per 256-dim
 * block, Lloyd-Max codes packed as 4-bit nibbles or, at 5, 6 and 8 bits, one byte per
 * value), the attention
 * over codes (the query pre-rotated, the output sign-undone) and the hybrid layout (raw
 * keys, coded values); model.rs, the cache buffers.
 * A format fixes head_dim, the code width and the sign pre-multiply.  Rows are coded in
 * blocks of B = min(head_dim, 256) values: u = H (s . x) / sqrt(B) (H the Sylvester
 * Hadamard matrix), norm = sqrt(mean(u^2)) stored as f32, and each u_i / norm coded by the
 * cell of the Lloyd-Max quantiser of N(0, 1) with 2^bits levels that holds it (a value on
 * a boundary takes the upper cell; the library computes the quantiser when the format is
 * created).  bits 5, 6, 8: one byte per value; bits 4: value 2j in the low nibble of byte
 * j, 2j+1 in the high nibble.  A coded value decodes to centroid[code] * norm (rotated).
 *   head_dim in {64, 128, 256, 512}; bits in {4, 5, 6, 8};
 *   signs_host int8 [head_dim], each +1 or -1, copied.
 * Synchronises the device: the format's tables are in device memory when it returns (the
 * attention reads them before waiting for the kernels that precede it).
 * Errors: HFA_EINVAL, HFA_EUNSUPPORTED, HFA_EDEVICE, HFA_ENOMEM.
 */
typedef struct hfa_tq hfa_tq;
hfa_status hfa_tq_create(int head_dim, int bits, const int8_t* signs_host, hfa_tq** out);
hfa_status hfa_tq_destroy(hfa_tq* fmt);
int hfa_tq_code_bytes(const hfa_tq* fmt); /* bytes of one row's codes: head_dim / 2 at 4 bits,
                                             head_dim at 5, 6 and 8 bits */
int hfa_tq_blocks(const hfa_tq* fmt);     /* norms per row: head_dim / B */
/* copies up to n centroids (ascending) to centroids_host; returns the level count */
int hfa_tq_codebook(const hfa_tq* fmt, float* centroids_host, int n);

/*
 * The KV append of a coded cache: row (b, h) of x_dev f32 [batch, nkv, head_dim] is coded
 * into slot seq_pos[b] (linear) or seq_pos[b] % capacity (ring) of codes_dev
 * [batch, nkv, capacity, code_bytes] and norms_dev f32 [batch, nkv, capacity, blocks];
 * every other slot is left as it is.  The decisions (the norm, the cells) are taken in
 * double precision from the f32 inputs.  x_dev 16-byte aligned.
 * Errors: HFA_EINVAL, HFA_ERANGE (a position outside a linear cache), HFA_ECUDA.
 */
hfa_status hfa_tq_append(const hfa_tq* fmt, void* stream, const float* x_dev,
                         const int32_t* seq_pos_dev, const int32_t* seq_pos_host, int batch,
                         int nkv, int capacity, int ring, uint8_t* codes_dev, float* norms_dev);

/*
 * Attention over a coded cache: as hfa_attention_decode (same descriptor, positions, masks,
 * scale and softcap), with the keys given by k_codes_dev / k_norms_dev in the format, or,
 * when k_codes_dev is NULL, by raw bf16 keys k_raw_dev [batch, nkv, capacity, head_dim]
 * (the hybrid layout), and the values always coded (v_codes_dev, v_norms_dev).  Scores
 * with coded keys use the rotated query (the rotation is orthogonal, so they equal q . k
 * over the decoded keys); the weighted sum of the decoded values is rotated back.
 *   workspace_dev  at least hfa_attention_tq_workspace_bytes(desc, batch, max_keys)
 *                  bytes, max_keys the most visible keys of any sequence of the call,
 *                  16-byte aligned, zero before its first use; each call leaves it ready
 *                  for the next.  Calls sharing a workspace must not overlap on the GPU.
 * fmt->head_dim must equal desc->head_dim.  q, o, the workspace and the code arrays
 * 16-byte aligned.  Errors as hfa_attention_decode (message via hfa_last_error(NULL)).
 */
size_t hfa_attention_tq_workspace_bytes(const hfa_attn_desc* desc, int batch, int max_keys);
hfa_status hfa_attention_decode_tq(const hfa_attn_desc* desc, const hfa_tq* fmt, void* stream,
                                   const float* q_dev, const int32_t* seq_pos_dev,
                                   const int32_t* seq_pos_host, int batch,
                                   const uint8_t* k_codes_dev, const float* k_norms_dev,
                                   const void* k_raw_dev, const uint8_t* v_codes_dev,
                                   const float* v_norms_dev, void* workspace_dev,
                                   size_t workspace_bytes, float* o_dev);

/*
 * ---- The dense feed-forward half of a layer (gemma4/gpu_full_attn.rs, encode_one_layer:
 * the dense MLP -- pre-feed-forward RMSNorm, gate and up projections, fused_gelu_mul,
 * down projection -- and the end of the layer: RMSNorm of the down output with
 * post_feedforward_layernorm, residual add, layer_scalar).  For each batch row h:
 *   n = h * w_pre / sqrt(mean(h^2) + eps) ;  a = gelu(Wg n) * (Wu n) ;  d = Wd a ;
 *   out = (h + d * w_post / sqrt(mean(d^2) + eps)) * s,
 * gelu(x) = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) (the tanh form; the pages name
 * the fused kernel without printing its formula), s the layer scalar: one value or one
 * per channel.  The MoE branch of the pages' 26B model is not part of this object.
 */
typedef struct hfa_ffn hfa_ffn; /* opaque; owned by the library */
typedef struct {
  int hidden;       /* H: a positive multiple of 32 (HFA_EINVAL otherwise) */
  int intermediate; /* I: a positive multiple of 32 (HFA_EINVAL otherwise) */
  float eps;        /* RMSNorm epsilon of both norms, >= 0 */
  int scalar_len;   /* 1 (one layer scalar) or H (one per channel) */
  int max_batch;    /* largest batch of hfa_ffn_step, 1..16; sizes the scratch and the
                       weights' tile order (HFA_EUNSUPPORTED outside) */
} hfa_ffn_desc;

/*
 * Create the FFN half.  Weights are read from device memory and copied (Q8_0 re-laid out
 * in MMA tiles; the values are untouched) into library-owned memory; the caller may free
 * them when the call returns.  Synchronises `stream`; allocates (the only FFN call that
 * does).
 *   w_gate_dev, w_up_dev  Q8_0 [I, H] (rows of H/32 blocks of 34 bytes: fp16 scale d,
 *                         little endian, then 32 int8 q; value = d * q)
 *   w_down_dev            Q8_0 [H, I]
 *   w_pre_dev, w_post_dev f32 [H];  scalar_dev f32 [scalar_len]
 * Errors: HFA_EINVAL (shape, NULL pointer), HFA_EUNSUPPORTED (max_batch, a shape the
 * kernel's buffers cannot plan), HFA_EDEVICE (no sm_103 device), HFA_ENOMEM, HFA_ECUDA.
 * Messages via hfa_ffn_last_error(NULL).  *out is NULL on error.
 */
hfa_status hfa_ffn_create(const hfa_ffn_desc* desc, const void* w_gate_dev, const void* w_up_dev,
                          const void* w_down_dev, const float* w_pre_dev, const float* w_post_dev,
                          const float* scalar_dev, void* stream, hfa_ffn** out);
hfa_status hfa_ffn_destroy(hfa_ffn* ffn);

/*
 * One FFN step for `batch` rows (1..max_batch), one cooperative launch of one CTA per SM
 * with programmatic dependent launch (as hfa_decode_step: only the weights are read
 * before the previous kernel on `stream` has completed).  Steps on one object must not
 * overlap on the GPU (they share its scratch).
 *   h_dev        bf16 [batch, H]: the FFN input, also the residual (the attention half's
 *                output)
 *   out_dev      bf16 [batch, H]: the layer output, round to nearest even
 *   out_f32_dev  nullable f32 [batch, H]: the same before rounding
 *   a_dev        nullable f32 [batch, I]: gelu(gate) * up, for tests
 * Every buffer 16-byte aligned (HFA_EINVAL otherwise).  Errors: HFA_EINVAL, HFA_EDEVICE
 * (another current device), HFA_ECUDA (launch; e.g. the SMs cannot all hold a CTA).
 */
hfa_status hfa_ffn_step(hfa_ffn* ffn, void* stream, const void* h_dev, int batch, void* out_dev,
                        float* out_f32_dev, float* a_dev);
/* Reads (synchronising `stream`) and clears the device error word: HFA_OK, or HFA_EDEVICE
 * when a bounded wait of an earlier step gave up (its outputs are then invalid; the step
 * count and partial sums restart). */
hfa_status hfa_ffn_check_status(hfa_ffn* ffn, void* stream);
const char* hfa_ffn_last_error(const hfa_ffn* ffn); /* NULL: this thread's last create error */
/* Instrumentation (no counterpart on the pages): with a buffer set, every later step writes
 * per CTA c the GPU's nanosecond timer into stamps_dev[c * 32 + k], k = 0 entry, 1 the
 * previous kernel completed, 2 first gate/up operand built, 3 first stage computed, 4 last
 * gate/up stage stored, 5 first down operand built, 6 last down stage stored, 7 down sums
 * of the CTA's outputs added, 8 post-FF norm known, 9 exit, 10 last weight stage issued,
 * 11..18 ring stages 0..7 arrived, 19..26 loads 4..11 issued (slots a CTA does not reach
 * keep their old value).  The buffer (int64 [rows][32], rows = hfa_ffn_stamp_rows) must
 * stay valid while set; NULL clears.  Results are unchanged. */
hfa_status hfa_ffn_set_stamps(hfa_ffn* ffn, unsigned long long* stamps_dev);
int hfa_ffn_stamp_rows(const hfa_ffn* ffn);
/* the work plan: grid, batch tiles, then (k-splits, blocks per split, row groups per
 * stage, stages) of the gate/up and of the down projection; returns the count (10) */
int hfa_ffn_plan_info(const hfa_ffn* ffn, int n, int* values);

/*
 * Successor hint for decoding through a stack of layers (no counterpart on the pages,
 * which run one layer at a time).  Once set, each decode step of `layer` prefetches into
 * L2, during its last phase (o_proj and residual, when HBM is otherwise idle), the Q8_0
 * QKV weights that the next decode step of `next` reads first.  Results are unchanged.
 *   next  a layer of the same shape (hidden, heads, kv heads, head dim) with Q8_0
 *         weights, or NULL to clear the hint.  It must stay alive while it is set: destroy
 *         or re-point `layer`'s hint before destroying `next`.
 * Errors: HFA_EINVAL (shapes differ, bf16 weights, NULL layer).
 */
hfa_status hfa_set_successor(hfa_layer* layer, const hfa_layer* next);

/*
 * Instrumentation of the decode step (no counterpart on the pages): with a buffer set,
 * every later decode step of `layer` writes, per CTA c (at most one per SM), the GPU's
 * nanosecond timer (%globaltimer) at fixed points into stamps_dev[c * 16 + k]:
 *   k = 0 CTA start, 1 activations loaded, 2 QKV projection done, 3 first queries ready,
 *   4 last key tile consumed, 5 attention records written, 6 grid barrier passed,
 *   7 o_proj operand merged, 8 o_proj done, 9 residual written (CTA end);
 *   10 first QKV copy issued, 11 last key tile issued, 12 o_proj copies issued,
 *   13 the wait for the previous kernel on the stream returned.
 * Slots 14 and 15 are unused.  A step may start (slot 0) while the previous kernel on the
 * stream is still finishing (programmatic dependent launch); from slot 13 on it runs alone.
 * max over c of slot 9 minus min over c of slot 13 is the kernel's own duration.  Results
 * are unchanged; the stores cost a few instructions.
 *   stamps_dev  u64 device buffer of hfa_step_stamp_rows(layer) * 16 entries, 8-byte
 *               aligned, owned by the caller; NULL turns the stamps off.
 * Errors: HFA_EINVAL (NULL layer, misaligned buffer).
 */
hfa_status hfa_set_step_stamps(hfa_layer* layer, unsigned long long* stamps_dev);
int hfa_step_stamp_rows(const hfa_layer* layer); /* CTAs of a step: rows of the stamp buffer */

/*
 * Test hook for the failure path: in the next decode step of `layer`, the consumer warps
 * of CTA 0 wait on an mbarrier that nothing completes.  The wait gives up after its bound
 * (about 1 s of the GPU clock), the step's other waits give up in turn, and the step ends
 * with its error word set: hfa_check_device_status then reports HFA_EDEVICE ("a bounded
 * wait gave up") and resets the step kernel's state.  No fault, trap or unbounded wait is
 * involved; the outputs of that one step are undefined.  Errors: HFA_EINVAL (NULL layer).
 */
hfa_status hfa_debug_stall_next_step(hfa_layer* layer);

/*
 * RoPE frequency factors of a global layer (gpu_full_attn.rs passes them to the fused
 * head norm + RoPE of full layers; model.rs loads rope_freqs.weight): each pair's angle
 * becomes phi_i = P * theta^(-2i/hd) / f_i, for decode steps and verify blocks alike.
 *   factors_host  f32 [hd/2] in host memory, each finite and > 0; NULL restores
 *                 phi_i = P * theta^(-2i/hd).
 * Enqueued on `stream` (the table is updated in stream order).  Errors: HFA_EINVAL.
 */
hfa_status hfa_set_rope_freq_factors(hfa_layer* layer, const float* factors_host, void* stream);

/*
 * Post-attention RMSNorm (gpu_full_attn.rs, fused post-attention norm + residual add):
 * the output becomes out = x + y * w_post / sqrt(mean(y^2) + eps), y = Wo o, for decode
 * steps and verify blocks.
 *   w_post_dev  f32 [H] in device memory, copied (the caller may free it); NULL turns the
 *               norm off again.
 * Enqueued on `stream`.  Errors: HFA_EINVAL, HFA_ENOMEM, HFA_ECUDA.
 */
hfa_status hfa_set_post_norm(hfa_layer* layer, const float* w_post_dev, void* stream);

/*
 * Copy of the library-owned weight tiles, for checking the re-layout done at create
 * (the values are moved, never changed).  `which` selects the buffer:
 *   0  Q8_0 [Wq; Wk; Wv] tiles, 1  Q8_0 Wo tiles: 544-byte tiles of 16 rows x 32 columns
 *      ordered (k-split s, row group r, block bb), a k-split being nbs consecutive
 *      32-column blocks, nbs the largest divisor of the row's block count up to 16.
 *      Tile bytes [0, 512): lane l = 4g + t holds four little-endian words at 16 l:
 *      word 2 ks + h = row g + 8 h, columns 16 ks + {2t, 2t+1, 2t+8, 2t+9} (byte e of the
 *      word for the e-th of those columns), each byte q + 128; bytes [512, 544): eight
 *      (fp16 d of row g, fp16 d of row g + 8) pairs, g = 0..7.
 *   2  bf16 [Wq; Wk; Wv] tiles, 3  bf16 Wo tiles (HFA_F_WEIGHTS_BF16 layers): 16 KB tiles
 *      of 128 rows x 64 columns, tile (m, c) at (m * K / 64 + c) * 16 KB, row r at
 *      r * 128 bytes, its 16-byte group j at (j XOR (r mod 8)) * 16.
 * hfa_weight_tile_bytes returns the size of the selected buffer (0: the layer has none).
 * hfa_debug_weight_tiles copies it to dst_dev (at least that many bytes) on `stream`.
 * Errors: HFA_EINVAL (NULL layer or pointer, a buffer the layer does not have, dst too
 * small), HFA_ECUDA.
 */
size_t hfa_weight_tile_bytes(const hfa_layer* layer, int which);
hfa_status hfa_debug_weight_tiles(hfa_layer* layer, int which, void* dst_dev, size_t dst_bytes,
                                  void* stream);

/* Release the layer and its device memory (synchronises the device first). */
hfa_status hfa_destroy(hfa_layer* layer);

/* Last error message of `layer`; with NULL, the last error of a create on this thread. */
const char* hfa_last_error(const hfa_layer* layer);

/*
 * Copies of the fp32 intermediate values of the last step, for layers created with
 * HFA_F_DEBUG_TAPS (HFA_EINVAL otherwise).  Device pointers, each nullable:
 *   q [rows, nh, hd] after norm + RoPE;  k, v [rows, nkv, hd] before the bf16 rounding;
 *   attn [rows, nh, hd];  out [rows, H] before the bf16 rounding;
 * rows = the batch of the last decode step, or L of the last verify block.
 * Enqueued on `stream`.
 */
hfa_status hfa_debug_taps(hfa_layer* layer, void* stream, float* q_dev, float* k_dev,
                          float* v_dev, float* attn_dev, float* out_dev);

/*
 * Device-side status of earlier steps: bounded waits that gave up, or positions the
 * kernels refused.  Synchronises `stream`; returns HFA_OK, or HFA_EDEVICE with the
 * reason in hfa_last_error, and clears the record (and, after a give-up, resets the
 * step kernel's grid-barrier counter and clears its step-tagged partial sums, so that
 * later steps start clean).
 */
hfa_status hfa_check_device_status(hfa_layer* layer, void* stream);

/*
 * Per-kernel timing: when enabled, the library records CUDA events around each of
 * its kernels on the launching stream.  hfa_kernel_times synchronises and returns,
 * for up to `n` kernel slots, the summed milliseconds and the launch count since the
 * last call, and each slot's name (static strings).  Returns the number of slots.
 */
int hfa_set_kernel_timing(hfa_layer* layer, int enable);
int hfa_kernel_times(hfa_layer* layer, int n, const char** names, float* total_ms,
                     int* launches);

/* Launch plan details (for logs and the benchmark): fills up to n ints:
 * [0] key tiles of the last step (all sequences and kv heads), [1] keys per tile,
 * [2] step grid, [3] step grid, [4] SM count. */
int hfa_plan_info(const hfa_layer* layer, int n, int* values);

#ifdef __cplusplus
}
#endif
#endif /* HFA_H */
