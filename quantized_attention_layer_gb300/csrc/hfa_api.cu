// hfa_api.cu -- the C ABI of libhfa (declared in include/hfa.h).
//
// Host side only: argument validation (before any launch), ownership of the repacked
// weights and of the per-layer scratch, launch plans, and the kernel launches of one
// decode step: one persistent kernel (k_step.cuh) that runs the QKV projection, the
// per-head norms, RoPE and KV append, the split-K flash-decode and the o_proj GEMV with
// the residual.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <string>
#include <vector>

#include "hfa_common.cuh"
#include "hfa_internal.h"
#include "hfa_verify.h"

using namespace hfa;

static thread_local char g_create_error[512];

void hfa::set_thread_error(const char* msg) { snprintf(g_create_error, sizeof g_create_error, "%s", msg); }

struct KernelTimer {
  const char* name;
  cudaEvent_t start, stop;
};

struct hfa_layer;
static void timer_begin(hfa_layer* L, cudaStream_t s, const char* name, KernelTimer* t);
static void timer_end(hfa_layer* L, cudaStream_t s, KernelTimer* t);

// adapter that lets the verify kernels record into the layer's timing slots
struct LayerTimer : hfa::LaunchTimer {
  hfa_layer* L = nullptr;
  KernelTimer t{};
  void begin(cudaStream_t s, const char* name) override { timer_begin(L, s, name, &t); }
  void end(cudaStream_t s) override { timer_end(L, s, &t); }
};

struct hfa_layer {
  hfa_layer_desc d{};
  int device = 0;
  int num_sms = 0;
  int grid = 0;  // CTAs of a decode step: fixed per layer (the step tags count launches x grid)
  int G = 0;
  int rows_qkv = 0;
  int max_rows = 0;
  // weights: Q8_0 tiles in the decode-step layout
  uint8_t* wqkv_t = nullptr;
  uint8_t* wo_t = nullptr;
  StepGemv g_qkv{}, g_o{};
  const uint8_t* successor_qkv = nullptr;  // QKV tiles of the layer that runs next
  unsigned long long* stamps = nullptr;     // caller's [SMs][16] timer stamps, or NULL
  int stall_next = 0;  // test hook (hfa_debug_stall_next_step), one step
  __nv_bfloat16* wqkv_bf16 = nullptr;  // verify path: [(nh + 2 nkv) hd, H] as 128 x 64 tiles
  __nv_bfloat16* wo_bf16 = nullptr;    // [H, nh hd] as 128 x 64 tiles
  float* w_in = nullptr;
  float* w_q = nullptr;
  float* w_k = nullptr;
  float2* rope_g = nullptr;
  std::vector<float2> rope_host;  // source of the last table upload (stream-ordered)
  float* w_post = nullptr;        // post-attention RMSNorm weight [H] (allocated on first use)
  bool w_post_on = false;         // the norm is applied
  unsigned long long* post_part = nullptr;  // [grid][2] tagged partial sum(y^2) per CTA
  // scratch
  unsigned long long* qkv_part = nullptr;  // tagged partial sums (value | step << 32)
  float* q_f32 = nullptr;
  float* attn_rec = nullptr;
  float* o_f32 = nullptr;
  unsigned long long* y_part = nullptr;
  unsigned long long* gbar = nullptr;
  float* k_tap = nullptr;
  float* v_tap = nullptr;
  float* out_tap = nullptr;
  unsigned* err = nullptr;
  __nv_bfloat16* x_stage = nullptr;
  int* pos_stage = nullptr;
  __nv_bfloat16* out_stage = nullptr;
  hfa::VerifyState* verify = nullptr;
  // tensor maps of the caches of the last call
  const void* tm_k_ptr = nullptr;
  const void* tm_v_ptr = nullptr;
  int tm_rows = 0;
  CUtensorMap tm_k{}, tm_v{};
  // plan of the last call
  int last_splits = 0, last_gemv_grid = 0, last_attn_grid = 0;  // tiles, grids
  int last_rows = 0;
  // timing
  bool timing = false;
  std::vector<KernelTimer> pending;
  std::vector<cudaEvent_t> event_pool;
  std::vector<std::string> slot_names;
  std::vector<float> slot_ms;
  std::vector<int> slot_count;
  std::vector<void*> allocations;
  char last_error[512] = {0};
};

// ------------------------------------------------------------------ error helpers
static hfa_status fail(hfa_layer* L, hfa_status st, const char* fmt, ...) {
  char* buf = L ? L->last_error : g_create_error;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, 512, fmt, ap);
  va_end(ap);
  return st;
}
static hfa_status cuda_fail(hfa_layer* L, cudaError_t e, const char* what) {
  return fail(L, HFA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}
#define CK(L, expr, what)                           \
  do {                                              \
    cudaError_t _e = (expr);                        \
    if (_e != cudaSuccess) return cuda_fail(L, _e, what); \
  } while (0)

template <typename T>
static cudaError_t lalloc(hfa_layer* L, T** p, size_t count) {
  *p = nullptr;
  if (count == 0) return cudaSuccess;
  cudaError_t e = cudaMalloc((void**)p, count * sizeof(T));
  if (e == cudaSuccess) L->allocations.push_back((void*)*p);
  return e;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// 2-D bf16 view [rows, hd] of a cache, boxes of 64 x box_rows with 128-byte swizzle.
hfa_status hfa_encode_kv_map(CUtensorMap* map, void* base, int rows, int hd, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return HFA_EDEVICE;
  cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HFA_OK : HFA_EINVAL;
}

hfa_status hfa_encode_u8_map(CUtensorMap* map, const void* base, long long rows, int row_bytes,
                             int box_bytes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return HFA_EDEVICE;
  if (box_bytes != 32 && box_bytes != 64 && box_bytes != 128) return HFA_EINVAL;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HFA_OK : HFA_EINVAL;
}

// ------------------------------------------------------------------ timing
static void timer_begin(hfa_layer* L, cudaStream_t s, const char* name, KernelTimer* t) {
  t->name = name;
  t->start = t->stop = nullptr;
  if (!L->timing) return;
  for (int i = 0; i < 2; ++i) {
    cudaEvent_t e;
    if (!L->event_pool.empty()) {
      e = L->event_pool.back();
      L->event_pool.pop_back();
    } else if (cudaEventCreate(&e) != cudaSuccess) {
      return;
    }
    (i == 0 ? t->start : t->stop) = e;
  }
  cudaEventRecord(t->start, s);
}
static void timer_end(hfa_layer* L, cudaStream_t s, KernelTimer* t) {
  if (!L->timing || !t->start) return;
  cudaEventRecord(t->stop, s);
  L->pending.push_back(*t);
}

// ------------------------------------------------------------------ validation
static bool is_pow2_hd(int hd) { return hd == 64 || hd == 128 || hd == 256; }
// the decode step also covers the 512-wide heads of the pages' global layers
static bool step_hd(int hd) { return is_pow2_hd(hd) || hd == 512; }

static hfa_status validate_desc(const hfa_layer_desc* d) {
  if (!d) return fail(nullptr, HFA_EINVAL, "desc is NULL");
  if (d->hidden <= 0 || d->hidden % 32 || d->hidden > 65536)
    return fail(nullptr, HFA_EINVAL, "hidden=%d must be a positive multiple of 32, at most 65536",
                d->hidden);
  if (d->hidden % 64)  // a valid Q8_0 row length (whole 32-value blocks) not covered here
    return fail(nullptr, HFA_EUNSUPPORTED, "hidden=%d: only multiples of 64 are supported",
                d->hidden);
  if (d->num_heads <= 0 || d->num_kv_heads <= 0 || d->num_heads % d->num_kv_heads)
    return fail(nullptr, HFA_EINVAL, "num_heads=%d must be a positive multiple of num_kv_heads=%d",
                d->num_heads, d->num_kv_heads);
  if (d->num_heads / d->num_kv_heads > 8)
    return fail(nullptr, HFA_EUNSUPPORTED, "GQA group %d > 8", d->num_heads / d->num_kv_heads);
  if (!step_hd(d->head_dim))
    return fail(nullptr, HFA_EUNSUPPORTED, "head_dim=%d (supported: 64, 128, 256, 512)",
                d->head_dim);
  if (d->layer_type != HFA_SLIDING && d->layer_type != HFA_FULL)
    return fail(nullptr, HFA_EINVAL, "layer_type=%d", d->layer_type);
  if (d->layer_type == HFA_SLIDING && d->window <= 0)
    return fail(nullptr, HFA_EINVAL, "sliding layer needs window > 0");
  if (d->kv_capacity <= 0 || d->kv_capacity >= (1 << 24))
    return fail(nullptr, HFA_EINVAL, "kv_capacity=%d outside [1, 2^24)", d->kv_capacity);
  if ((d->flags & HFA_F_RING) && (d->layer_type != HFA_SLIDING || d->kv_capacity != d->window))
    return fail(nullptr, HFA_EINVAL, "a ring cache needs a sliding layer with kv_capacity == window");
  if (d->max_batch < 1 || d->max_batch > 16)
    return fail(nullptr, HFA_EUNSUPPORTED, "max_batch=%d outside [1, 16]", d->max_batch);
  if (d->max_verify_len < 0 || d->max_verify_len > 16)
    return fail(nullptr, HFA_EUNSUPPORTED, "max_verify_len=%d outside [0, 16]", d->max_verify_len);
  // the verify kernels address each cache as [nkv * C, hd] rows with 32-bit TMA rows
  if (d->max_verify_len > 0 && (long long)d->num_kv_heads * d->kv_capacity + 256 >= (1ll << 31))
    return fail(nullptr, HFA_EUNSUPPORTED, "verify: cache too large for 32-bit TMA rows");
  if (!(d->eps >= 0.f) || !(d->rope_theta > 0.f) || !(d->attn_scale > 0.f) || !(d->softcap >= 0.f))
    return fail(nullptr, HFA_EINVAL, "eps, rope_theta, attn_scale, softcap out of range");
  if (d->flags & ~(HFA_F_V_UNIT_NORM | HFA_F_WEIGHTS_BF16 | HFA_F_RING | HFA_F_DEBUG_TAPS |
                   HFA_F_K_EQ_V | HFA_F_BLOCK_BIDIR))
    return fail(nullptr, HFA_EINVAL, "unknown flags 0x%x", d->flags);
  return HFA_OK;
}

// Split-K shape of a decode-step GEMV: k-splits of nbs 32-column blocks, nbs the largest
// divisor of the block count up to 16 (512 columns), and as many nbs-tile work items per
// 64 KiB ring stage as fit.
static int step_grid(const hfa_layer_desc& d, const StepGemv& qkv, const StepGemv& o, int sms);

static void plan_step_gemv(StepGemv* g, int rows, int cols) {
  g->R = rows / 16;
  g->nb = cols / 32;
  g->nbs = 1;
  for (int d = 16; d >= 1; --d)
    if (g->nb % d == 0) {
      g->nbs = d;
      break;
    }
  g->S = g->nb / g->nbs;
  g->ips = (int)(step_stage_bytes() / ((size_t)g->nbs * kQ8TileBytes));
  g->w = nullptr;
}

// RoPE table: theta^(-2i/hd) / (2 pi) / f_i in double (f_i = 1 without frequency factors),
// stored as an fp32 (hi, lo) pair per pair i; the kernels reduce P * g exactly enough.
// The host copy lives in the layer, so that the asynchronous upload can read it later.
static cudaError_t upload_rope_table(hfa_layer* L, const float* ff, cudaStream_t s) {
  const int hd = L->d.head_dim;
  L->rope_host.resize(hd / 2);
  for (int i = 0; i < hd / 2; ++i) {
    double v = pow((double)L->d.rope_theta, -2.0 * i / hd) / (2.0 * M_PI);
    if (ff) v /= (double)ff[i];
    const float hi = (float)v;
    L->rope_host[i] = make_float2(hi, (float)(v - (double)hi));
  }
  return cudaMemcpyAsync(L->rope_g, L->rope_host.data(), (size_t)hd / 2 * sizeof(float2),
                         cudaMemcpyHostToDevice, s);
}

// ------------------------------------------------------------------ create / destroy
static void free_layer(hfa_layer* L) {
  if (!L) return;
  if (L->verify) hfa::verify_free(L->verify);
  for (void* p : L->allocations) cudaFree(p);
  for (auto& t : L->pending) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  for (auto e : L->event_pool) cudaEventDestroy(e);
  delete L;
}

extern "C" hfa_status hfa_layer_create(const hfa_layer_desc* desc, const void* wq, const void* wk,
                                       const void* wv, const void* wo, const float* w_in,
                                       const float* w_q, const float* w_k, void* stream,
                                       hfa_layer** out) {
  if (!out) return fail(nullptr, HFA_EINVAL, "out is NULL");
  *out = nullptr;
  hfa_status st = validate_desc(desc);
  if (st != HFA_OK) return st;
  if (!wq || !wk || (!wv && !(desc->flags & HFA_F_K_EQ_V)) || !wo || !w_in || !w_q || !w_k)
    return fail(nullptr, HFA_EINVAL, "a weight pointer is NULL");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(nullptr, HFA_EDEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return fail(nullptr, HFA_EDEVICE, "%s", cudaGetErrorString(e));
  if (prop.major != 10 || prop.minor != 3)
    return fail(nullptr, HFA_EDEVICE, "device %s is sm_%d%d; libhfa is built for sm_103a only",
                prop.name, prop.major, prop.minor);
  if (!encode_fn()) return fail(nullptr, HFA_EDEVICE, "cuTensorMapEncodeTiled unavailable");
  if (prop.multiProcessorCount > 256)  // the step kernel's partitions: 32-bit products
    return fail(nullptr, HFA_EUNSUPPORTED, "%d SMs: at most 256 supported",
                prop.multiProcessorCount);

  hfa_layer* L = new hfa_layer();
  L->d = *desc;
  L->device = dev;
  L->num_sms = prop.multiProcessorCount;
  const hfa_layer_desc& d = L->d;
  const int H = d.hidden, nh = d.num_heads, nkv = d.num_kv_heads, hd = d.head_dim;
  L->G = nh / nkv;
  L->rows_qkv = qkv_rows(d);  // no V rows with k_eq_v
  L->max_rows = d.max_batch > d.max_verify_len ? d.max_batch : d.max_verify_len;
  const int MR = L->max_rows;
  cudaStream_t s = (cudaStream_t)stream;
  const bool bf16w = d.flags & HFA_F_WEIGHTS_BF16;

#define LA(ptr, n)                                                        \
  do {                                                                    \
    cudaError_t _e = lalloc(L, &(ptr), (size_t)(n));                      \
    if (_e != cudaSuccess) {                                              \
      snprintf(g_create_error, 512, "cudaMalloc: %s", cudaGetErrorString(_e)); \
      free_layer(L);                                                      \
      return HFA_ENOMEM;                                                  \
    }                                                                     \
  } while (0)
#define LC(expr, what)                                                    \
  do {                                                                    \
    cudaError_t _e = (expr);                                              \
    if (_e != cudaSuccess) {                                              \
      snprintf(g_create_error, 512, "%s: %s", what, cudaGetErrorString(_e)); \
      free_layer(L);                                                      \
      return HFA_ECUDA;                                                   \
    }                                                                     \
  } while (0)

  if (!bf16w) {
    plan_step_gemv(&L->g_qkv, L->rows_qkv, H);
    plan_step_gemv(&L->g_o, H, nh * hd);
    if (L->g_qkv.S > L->num_sms || L->g_o.S > L->num_sms) {
      snprintf(g_create_error, 512, "hidden=%d / nh*hd=%d need more k-splits than the %d SMs",
               H, nh * hd, L->num_sms);
      delete L;
      return HFA_EUNSUPPORTED;
    }
    const int Rq = L->rows_qkv / 16;
    L->grid = step_grid(*desc, L->g_qkv, L->g_o, L->num_sms);
    LA(L->wqkv_t, (size_t)Rq * L->g_qkv.nb * kQ8TileBytes);
    LA(L->wo_t, (size_t)(H / 16) * L->g_o.nb * kQ8TileBytes);
    L->g_qkv.w = L->wqkv_t;
    L->g_o.w = L->wo_t;
    const int nbq = L->g_qkv.nbs, nbo = L->g_o.nbs;
    LC(launch_repack_q8_0_split((const uint8_t*)wq, nh * hd, H, L->wqkv_t, 0, Rq, nbq, s),
       "repack wq");
    LC(launch_repack_q8_0_split((const uint8_t*)wk, nkv * hd, H, L->wqkv_t, nh * hd / 16, Rq, nbq,
                                s),
       "repack wk");
    if (!(d.flags & HFA_F_K_EQ_V))
      LC(launch_repack_q8_0_split((const uint8_t*)wv, nkv * hd, H, L->wqkv_t,
                                  (nh + nkv) * hd / 16, Rq, nbq, s),
         "repack wv");
    LC(launch_repack_q8_0_split((const uint8_t*)wo, H, nh * hd, L->wo_t, 0, H / 16, nbo, s),
       "repack wo");
  } else {
    LA(L->wqkv_bf16, (size_t)L->rows_qkv * H);
    LA(L->wo_bf16, (size_t)H * nh * hd);
    if (L->rows_qkv % 128 == 0 && H % 128 == 0 && H % 64 == 0 && (nh * hd) % 64 == 0) {
      const bool kv1 = d.flags & HFA_F_K_EQ_V;
      LC(launch_repack_bf16_tiles((const __nv_bfloat16*)wq, nh * hd, (const __nv_bfloat16*)wk,
                                  kv1 ? L->rows_qkv - nh * hd : nkv * hd,
                                  (const __nv_bfloat16*)(kv1 ? wk : wv), L->rows_qkv, H,
                                  (uint8_t*)L->wqkv_bf16, s),
         "repack wqkv");
      LC(launch_repack_bf16_tiles((const __nv_bfloat16*)wo, H, (const __nv_bfloat16*)wo, 0,
                                  (const __nv_bfloat16*)wo, H, nh * hd, (uint8_t*)L->wo_bf16, s),
         "repack wo");
    }
  }
  LA(L->w_in, H);
  LA(L->w_q, hd);
  LA(L->w_k, hd);
  LC(cudaMemcpyAsync(L->w_in, w_in, H * 4, cudaMemcpyDeviceToDevice, s), "copy w_in");
  LC(cudaMemcpyAsync(L->w_q, w_q, hd * 4, cudaMemcpyDeviceToDevice, s), "copy w_q");
  LC(cudaMemcpyAsync(L->w_k, w_k, hd * 4, cudaMemcpyDeviceToDevice, s), "copy w_k");
  LA(L->rope_g, hd / 2);
  LC(upload_rope_table(L, nullptr, s), "copy rope table");
  LC(cudaStreamSynchronize(s), "create sync");
  // scratch
  const int units = d.max_batch * nkv;
  if (!bf16w) {
    LA(L->qkv_part, (size_t)L->g_qkv.S * d.max_batch * L->rows_qkv);
    LA(L->y_part, (size_t)L->g_o.S * d.max_batch * H);
  }
  LA(L->q_f32, (size_t)MR * nh * hd);
  // one (m, l, O) record per (CTA, unit) pair of the step kernel: ids c + u are unique
  LA(L->attn_rec, (size_t)(L->num_sms + units) * attn_record_floats(hd));
  LA(L->gbar, 1);
  LA(L->o_f32, (size_t)MR * nh * hd);
  LA(L->err, 1);
  LA(L->x_stage, (size_t)d.max_batch * H);
  LA(L->pos_stage, d.max_batch);
  LA(L->out_stage, (size_t)d.max_batch * H);
  if (d.flags & HFA_F_DEBUG_TAPS) {
    LA(L->k_tap, (size_t)MR * nkv * hd);
    LA(L->v_tap, (size_t)MR * nkv * hd);
    LA(L->out_tap, (size_t)MR * H);
  }
  LC(cudaMemsetAsync(L->gbar, 0, 8, s), "memset");
  if (!bf16w) {  // tag 0 never matches a step (tags start at 1)
    LC(cudaMemsetAsync(L->qkv_part, 0, (size_t)L->g_qkv.S * d.max_batch * L->rows_qkv * 8, s),
       "memset");
    LC(cudaMemsetAsync(L->y_part, 0, (size_t)L->g_o.S * d.max_batch * H * 8, s), "memset");
  }
  LC(cudaMemsetAsync(L->err, 0, 4, s), "memset");
  if (d.max_verify_len > 0) {
    hfa_status vs = hfa::verify_create(L->d, L->num_sms, &L->verify);
    if (vs != HFA_OK) {
      snprintf(g_create_error, 512, "verify scratch: %s", hfa::verify_error());
      free_layer(L);
      return vs;
    }
  }
  LC(cudaStreamSynchronize(s), "create sync");
  *out = L;
  return HFA_OK;
#undef LA
#undef LC
}

extern "C" hfa_status hfa_set_successor(hfa_layer* L, const hfa_layer* next) {
  if (!L) return HFA_EINVAL;
  if (!next) {
    L->successor_qkv = nullptr;
    return HFA_OK;
  }
  const hfa_layer_desc &a = L->d, &b = next->d;
  if (!L->wqkv_t || !next->wqkv_t)
    return fail(L, HFA_EINVAL, "the successor hint needs Q8_0 weights on both layers");
  if (a.hidden != b.hidden || a.num_heads != b.num_heads || a.num_kv_heads != b.num_kv_heads ||
      a.head_dim != b.head_dim || next->device != L->device)
    return fail(L, HFA_EINVAL, "the successor must have the same shape, on the same device");
  L->successor_qkv = next->wqkv_t;
  return HFA_OK;
}

extern "C" hfa_status hfa_set_rope_freq_factors(hfa_layer* L, const float* ff, void* stream) {
  if (!L) return HFA_EINVAL;
  const int hd = L->d.head_dim;
  if (ff)
    for (int i = 0; i < hd / 2; ++i)
      if (!(ff[i] > 0.f) || !isfinite(ff[i]))
        return fail(L, HFA_EINVAL, "frequency factor %d is %g (need finite and > 0)", i,
                    (double)ff[i]);
  cudaStream_t s = (cudaStream_t)stream;
  CK(L, upload_rope_table(L, ff, s), "copy rope table");
  return HFA_OK;
}

extern "C" hfa_status hfa_set_post_norm(hfa_layer* L, const float* w_post, void* stream) {
  if (!L) return HFA_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  if (!w_post) {
    L->w_post_on = false;
    return HFA_OK;
  }
  if (!L->w_post) {
    cudaError_t e = cudaMalloc(&L->w_post, (size_t)L->d.hidden * sizeof(float));
    if (e == cudaSuccess) L->allocations.push_back(L->w_post);
    else L->w_post = nullptr;
    if (e == cudaSuccess) {
      e = cudaMalloc(&L->post_part, (size_t)L->num_sms * 2 * sizeof(unsigned long long));
      if (e == cudaSuccess) L->allocations.push_back(L->post_part);
      else L->post_part = nullptr;
    }
    if (e != cudaSuccess) return fail(L, HFA_ENOMEM, "cudaMalloc: %s", cudaGetErrorString(e));
    CK(L, cudaMemsetAsync(L->post_part, 0, (size_t)L->num_sms * 2 * 8, s), "memset");
  }
  CK(L, cudaMemcpyAsync(L->w_post, w_post, (size_t)L->d.hidden * sizeof(float),
                        cudaMemcpyDeviceToDevice, s), "copy w_post");
  L->w_post_on = true;
  return HFA_OK;
}

extern "C" hfa_status hfa_set_step_stamps(hfa_layer* L, unsigned long long* stamps) {
  if (!L) return HFA_EINVAL;
  if (stamps && ((uintptr_t)stamps & 7))
    return fail(L, HFA_EINVAL, "the stamp buffer must be 8-byte aligned");
  L->stamps = stamps;
  return HFA_OK;
}

extern "C" int hfa_step_stamp_rows(const hfa_layer* L) { return L ? L->grid : 0; }

static size_t weight_tile_bytes(const hfa_layer* L, int which, const void** src) {
  *src = nullptr;
  if (!L) return 0;
  const hfa_layer_desc& d = L->d;
  const int H = d.hidden, qo = d.num_heads * d.head_dim;
  switch (which) {
    case 0:
      *src = L->wqkv_t;
      return L->wqkv_t ? (size_t)(L->rows_qkv / 16) * L->g_qkv.nb * kQ8TileBytes : 0;
    case 1:
      *src = L->wo_t;
      return L->wo_t ? (size_t)(H / 16) * L->g_o.nb * kQ8TileBytes : 0;
    case 2:
      *src = L->wqkv_bf16;
      return L->wqkv_bf16 ? (size_t)L->rows_qkv * H * 2 : 0;
    case 3:
      *src = L->wo_bf16;
      return L->wo_bf16 ? (size_t)H * qo * 2 : 0;
    default:
      return 0;
  }
}

extern "C" size_t hfa_weight_tile_bytes(const hfa_layer* L, int which) {
  const void* src;
  return weight_tile_bytes(L, which, &src);
}

extern "C" hfa_status hfa_debug_weight_tiles(hfa_layer* L, int which, void* dst, size_t dst_bytes,
                                             void* stream) {
  if (!L) return HFA_EINVAL;
  const void* src;
  const size_t n = weight_tile_bytes(L, which, &src);
  if (!n || !src) return fail(L, HFA_EINVAL, "the layer has no weight buffer %d", which);
  if (!dst || dst_bytes < n)
    return fail(L, HFA_EINVAL, "destination of %zu bytes, %zu needed", dst_bytes, n);
  CK(L, cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, (cudaStream_t)stream),
     "copy weight tiles");
  return HFA_OK;
}

extern "C" hfa_status hfa_debug_stall_next_step(hfa_layer* L) {
  if (!L) return HFA_EINVAL;
  L->stall_next = 1;
  return HFA_OK;
}

extern "C" hfa_status hfa_destroy(hfa_layer* L) {
  if (!L) return HFA_EINVAL;
  cudaDeviceSynchronize();
  free_layer(L);
  return HFA_OK;
}

extern "C" const char* hfa_last_error(const hfa_layer* L) {
  return L ? L->last_error : g_create_error;
}

// ------------------------------------------------------------------ decode step
static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

static hfa_status ensure_maps(hfa_layer* L, void* kc, void* vc, int rows) {
  if (L->tm_k_ptr == kc && L->tm_v_ptr == vc && L->tm_rows == rows) return HFA_OK;
  const int T = step_keys_per_tile(L->d.head_dim);
  if (hfa_encode_kv_map(&L->tm_k, kc, rows, L->d.head_dim, T) != HFA_OK ||
      hfa_encode_kv_map(&L->tm_v, vc, rows, L->d.head_dim, T) != HFA_OK)
    return fail(L, HFA_EINVAL, "cannot describe the KV cache to the TMA unit");
  L->tm_k_ptr = kc;
  L->tm_v_ptr = vc;
  L->tm_rows = rows;
  return HFA_OK;
}

// Split-K plan of the flash-decode launch: as many chunks per (sequence, KV head) as
// fill every SM once (two CTAs per SM when the stages fit twice), chunks a multiple of
// the stage length.
static void fill_attn(AttnArgs& aa, int nh, int nkv, int hd, int C, int layer_type, int window,
                      bool ring, float scale, float softcap, int batch, int max_keys, int num_sms,
                      int max_splits, int* S_out) {
  const int T = attn_keys_per_stage(hd);
  const int units = batch * nkv;
  const int per_sm = attn_smem_bytes(hd) <= 113 * 1024 ? 2 : 1;
  int S = (num_sms * per_sm) / units;
  const int max_tiles = (max_keys + T - 1) / T;
  if (S > max_tiles) S = max_tiles;
  if (S > max_splits) S = max_splits;
  if (S < 1) S = 1;
  int chunk = (max_keys + S - 1) / S;
  chunk = (chunk + T - 1) / T * T;
  S = (max_keys + chunk - 1) / chunk;
  aa.B = batch;
  aa.nh = nh;
  aa.nkv = nkv;
  aa.hd = hd;
  aa.C = C;
  aa.sliding = layer_type == HFA_SLIDING;
  aa.window = window;
  aa.ring = ring;
  const float log2e = 1.4426950408889634f;
  if (softcap > 0.f) {
    aa.qscale = scale / softcap;
    aa.cap_log2 = softcap * log2e;
  } else {
    aa.qscale = scale * log2e;
    aa.cap_log2 = 0.f;
  }
  aa.splits = S;
  aa.chunk = chunk;
  *S_out = S;
}

// CTAs of a layer's decode step: one per SM, or fewer for a layer whose largest step has
// less work than SMs (the QKV and o_proj row groups two to a CTA, and the key tiles of the
// most visible keys at max_batch), never fewer than the GEMVs' k-splits.  Fixed per layer:
// the step tags are launches x grid.
static int step_grid(const hfa_layer_desc& d, const StepGemv& qkv, const StepGemv& o, int sms) {
  const int T = step_keys_per_tile(d.head_dim);
  const bool ring = d.flags & HFA_F_RING;
  const int vis = (d.layer_type == HFA_SLIDING && !ring && d.window < d.kv_capacity) ? d.window
                                                                                     : d.kv_capacity;
  const long long tiles = (long long)d.max_batch * d.num_kv_heads * ((vis + T - 1) / T + 1);
  long long work = tiles;
  if ((qkv.R + 1) / 2 > work) work = (qkv.R + 1) / 2;
  if ((o.R + 1) / 2 > work) work = (o.R + 1) / 2;
  if (work > d.hidden) work = d.hidden;  // every CTA keeps outputs of a batch-1 step
  const int lo = qkv.S > o.S ? qkv.S : o.S;
  return (int)(work > sms ? sms : (work < lo ? lo : work));
}

static int visible_keys(const hfa_layer_desc& d, int P) {
  const bool ring = d.flags & HFA_F_RING;
  if (ring) return (P < d.kv_capacity - 1 ? P : d.kv_capacity - 1) + 1;
  int lo = d.layer_type == HFA_SLIDING ? (P - d.window + 1 > 0 ? P - d.window + 1 : 0) : 0;
  return P - lo + 1;
}

extern "C" hfa_status hfa_decode_step(hfa_layer* L, void* stream, const void* x,
                                      const int32_t* pos_dev, const int32_t* pos_host,
                                      int batch, void* kc, void* vc, void* out) {
  if (!L) return HFA_EINVAL;
  const hfa_layer_desc& d = L->d;
  if (d.flags & HFA_F_WEIGHTS_BF16)
    return fail(L, HFA_EUNSUPPORTED, "the decode step needs Q8_0 weights");
  if (!x || !pos_dev || !pos_host || !kc || !vc || !out)
    return fail(L, HFA_EINVAL, "a pointer argument is NULL");
  if (batch < 1 || batch > d.max_batch)
    return fail(L, HFA_EINVAL, "batch=%d outside [1, max_batch=%d]", batch, d.max_batch);
  if (!aligned16(x) || !aligned16(kc) || !aligned16(vc) || !aligned16(out))
    return fail(L, HFA_EINVAL, "x, caches and out must be 16-byte aligned");
  const bool ring = d.flags & HFA_F_RING;
  int max_keys = 0;
  for (int b = 0; b < batch; ++b) {
    const int P = pos_host[b];
    if (P < 0 || (!ring && P >= d.kv_capacity) || P >= (1 << 24))
      return fail(L, HFA_ERANGE, "seq_pos[%d]=%d outside the cache (capacity %d%s)", b, P,
                  d.kv_capacity, ring ? ", ring" : "");
    const int n = visible_keys(d, P);
    if (n > max_keys) max_keys = n;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int nkv = d.num_kv_heads, hd = d.head_dim;
  const long long rows = (long long)batch * nkv * d.kv_capacity;
  if (rows + 256 >= (1ll << 31))
    return fail(L, HFA_EUNSUPPORTED, "cache too large for 32-bit TMA rows");
  // the step kernel's key-tile partition in 32-bit arithmetic
  if (rows / step_keys_per_tile(hd) + (long long)batch * nkv >= (1ll << 24))
    return fail(L, HFA_EUNSUPPORTED, "cache too large: 2^24 key tiles or more");
  hfa_status st = ensure_maps(L, kc, vc, (int)rows);
  if (st != HFA_OK) return st;

  const bool taps = d.flags & HFA_F_DEBUG_TAPS;
  StepArgs sa{};
  sa.qkv = L->g_qkv;
  sa.o = L->g_o;
  sa.x = (const __nv_bfloat16*)x;
  sa.w_in = L->w_in;
  sa.w_q = L->w_q;
  sa.w_k = L->w_k;
  sa.rope_g = L->rope_g;
  sa.seq_pos = pos_dev;
  sa.k_cache = (__nv_bfloat16*)kc;
  sa.v_cache = (__nv_bfloat16*)vc;
  sa.qkv_part = L->qkv_part;
  sa.rec = L->attn_rec;
  sa.y_part = L->y_part;
  sa.gbar = L->gbar;
  sa.o_attn = L->o_f32;  // also the attention tap
  sa.err = L->err;
  sa.q_tap = taps ? L->q_f32 : nullptr;
  sa.k_tap = L->k_tap;
  sa.v_tap = L->v_tap;
  sa.out_tap = L->out_tap;
  sa.out = (__nv_bfloat16*)out;
  sa.next_qkv_w = L->successor_qkv;
  sa.stall = L->stall_next;
  sa.w_post = L->w_post_on ? L->w_post : nullptr;
  sa.post_part = L->post_part;
  sa.stamps = L->stamps;
  sa.k_eq_v = (d.flags & HFA_F_K_EQ_V) ? 1 : 0;
  L->stall_next = 0;
  sa.B = batch;
  sa.H = d.hidden;
  sa.nh = d.num_heads;
  sa.nkv = nkv;
  sa.C = d.kv_capacity;
  sa.cache_rows = rows;
  sa.sliding = d.layer_type == HFA_SLIDING;
  sa.window = d.window;
  sa.ring = ring ? 1 : 0;
  sa.v_unit_norm = (d.flags & HFA_F_V_UNIT_NORM) ? 1 : 0;
  sa.eps = d.eps;
  const float log2e = 1.4426950408889634f;
  if (d.softcap > 0.f) {
    sa.qscale = d.attn_scale / d.softcap;
    sa.cap_log2 = d.softcap * log2e;
  } else {
    sa.qscale = d.attn_scale * log2e;
    sa.cap_log2 = 0.f;
  }
  const int T = step_keys_per_tile(hd);
  int tiles = 0;
  for (int b = 0; b < batch; ++b) tiles += (visible_keys(d, pos_host[b]) + T - 1) / T * nkv;
  L->last_splits = tiles;
  L->last_gemv_grid = L->grid;
  L->last_attn_grid = L->grid;
  KernelTimer t;
  timer_begin(L, s, "decode_step", &t);
  cudaError_t e = launch_step(sa, L->tm_k, L->tm_v, hd, L->grid, s);
  timer_end(L, s, &t);
  if (e != cudaSuccess) return cuda_fail(L, e, "decode-step kernel launch");
  L->last_rows = batch;
  return HFA_OK;
}

// ------------------------------------------------------------------ attention alone
static hfa_status validate_attn_desc(const hfa_attn_desc* d) {
  if (!d) return fail(nullptr, HFA_EINVAL, "desc is NULL");
  if (d->num_heads <= 0 || d->num_kv_heads <= 0 || d->num_heads % d->num_kv_heads)
    return fail(nullptr, HFA_EINVAL, "num_heads=%d must be a positive multiple of num_kv_heads=%d",
                d->num_heads, d->num_kv_heads);
  if (d->num_heads / d->num_kv_heads > 8)
    return fail(nullptr, HFA_EUNSUPPORTED, "GQA group %d > 8", d->num_heads / d->num_kv_heads);
  if (!is_pow2_hd(d->head_dim))
    return fail(nullptr, HFA_EUNSUPPORTED, "head_dim=%d (supported: 64, 128, 256)", d->head_dim);
  if (d->layer_type != HFA_SLIDING && d->layer_type != HFA_FULL)
    return fail(nullptr, HFA_EINVAL, "layer_type=%d", d->layer_type);
  if (d->layer_type == HFA_SLIDING && d->window <= 0)
    return fail(nullptr, HFA_EINVAL, "sliding layer needs window > 0");
  if (d->kv_capacity <= 0 || d->kv_capacity >= (1 << 24))
    return fail(nullptr, HFA_EINVAL, "kv_capacity=%d outside [1, 2^24)", d->kv_capacity);
  if (d->flags & ~HFA_F_RING) return fail(nullptr, HFA_EINVAL, "flags 0x%x", d->flags);
  if ((d->flags & HFA_F_RING) && (d->layer_type != HFA_SLIDING || d->kv_capacity != d->window))
    return fail(nullptr, HFA_EINVAL, "a ring cache needs a sliding layer with kv_capacity == window");
  if (!(d->attn_scale > 0.f) || !(d->softcap >= 0.f))
    return fail(nullptr, HFA_EINVAL, "attn_scale, softcap out of range");
  return HFA_OK;
}

static int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// workspace: [status word + tickets, 256-byte aligned][one (m, l, O) record per chunk].
// The plan gives S = floor(slots / units) chunks per unit (at least 1), so units * S
// never exceeds max(slots, units) with slots = 2 * SMs.
static size_t attn_ws_head_bytes(int units) { return ((size_t)(units + 1) * 4 + 255) / 256 * 256; }
static size_t attn_ws_bytes(int units, int slots, int hd) {
  const size_t chunks = (size_t)(units > slots ? units : slots);
  return attn_ws_head_bytes(units) + chunks * attn_record_floats(hd) * 4;
}

extern "C" size_t hfa_attention_workspace_bytes(const hfa_attn_desc* d, int batch) {
  if (validate_attn_desc(d) != HFA_OK || batch < 1) return 0;
  const int sms = current_sm_count();
  if (sms <= 0) return 0;
  return attn_ws_bytes(batch * d->num_kv_heads, 2 * sms, d->head_dim);
}

extern "C" hfa_status hfa_attention_decode(const hfa_attn_desc* d, void* stream, const float* q,
                                           const int32_t* pos_dev, const int32_t* pos_host,
                                           int batch, const void* kc, const void* vc, void* ws,
                                           size_t ws_bytes, float* o) {
  hfa_status st = validate_attn_desc(d);
  if (st != HFA_OK) return st;
  if (!q || !pos_dev || !pos_host || !kc || !vc || !ws || !o)
    return fail(nullptr, HFA_EINVAL, "a pointer argument is NULL");
  if (batch < 1 || batch > 4096) return fail(nullptr, HFA_EINVAL, "batch=%d", batch);
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(ws) || !aligned16(o))
    return fail(nullptr, HFA_EINVAL, "q, caches, workspace and o must be 16-byte aligned");
  const bool ring = d->flags & HFA_F_RING;
  hfa_layer_desc ld{};
  ld.layer_type = d->layer_type;
  ld.window = d->window;
  ld.kv_capacity = d->kv_capacity;
  ld.flags = d->flags;
  int max_keys = 0;
  for (int b = 0; b < batch; ++b) {
    const int P = pos_host[b];
    if (P < 0 || (!ring && P >= d->kv_capacity) || P >= (1 << 24))
      return fail(nullptr, HFA_ERANGE, "seq_pos[%d]=%d outside the cache (capacity %d)", b, P,
                  d->kv_capacity);
    const int n = visible_keys(ld, P);
    if (n > max_keys) max_keys = n;
  }
  const int sms = current_sm_count();
  if (sms <= 0) return fail(nullptr, HFA_EDEVICE, "no CUDA device");
  const int units = batch * d->num_kv_heads;
  const size_t need = attn_ws_bytes(units, 2 * sms, d->head_dim);
  if (ws_bytes < need)
    return fail(nullptr, HFA_EINVAL, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  const long long rows = (long long)units * d->kv_capacity;
  if (rows + 256 >= (1ll << 31)) return fail(nullptr, HFA_EUNSUPPORTED, "cache too large");
  CUtensorMap tk, tv;
  const int T = attn_keys_per_stage(d->head_dim);
  if (hfa_encode_kv_map(&tk, (void*)kc, (int)rows, d->head_dim, T) != HFA_OK ||
      hfa_encode_kv_map(&tv, (void*)vc, (int)rows, d->head_dim, T) != HFA_OK)
    return fail(nullptr, HFA_EINVAL, "cannot describe the KV cache to the TMA unit");
  AttnArgs aa{};
  int S = 0;
  fill_attn(aa, d->num_heads, d->num_kv_heads, d->head_dim, d->kv_capacity, d->layer_type,
            d->window, ring, d->attn_scale, d->softcap, batch, max_keys, sms, 2 * sms, &S);
  aa.q = q;
  aa.seq_pos = pos_dev;
  aa.err = (unsigned*)ws;
  aa.ticket = (int*)ws + 1;
  aa.part = (float*)((char*)ws + attn_ws_head_bytes(units));
  aa.o = o;
  cudaError_t e = launch_attn(aa, tk, tv, units * S, false, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "attention kernel launch");
  return HFA_OK;
}

extern "C" hfa_status hfa_decode_step_host(hfa_layer* L, void* stream, const void* x_host,
                                           const int32_t* pos_host, int batch, void* kc,
                                           void* vc, void* out_host) {
  if (!L) return HFA_EINVAL;
  if (!x_host || !pos_host || !out_host) return fail(L, HFA_EINVAL, "a host pointer is NULL");
  if (batch < 1 || batch > L->d.max_batch)
    return fail(L, HFA_EINVAL, "batch=%d outside [1, max_batch=%d]", batch, L->d.max_batch);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t xb = (size_t)batch * L->d.hidden * 2;
  CK(L, cudaMemcpyAsync(L->x_stage, x_host, xb, cudaMemcpyHostToDevice, s), "copy x in");
  CK(L, cudaMemcpyAsync(L->pos_stage, pos_host, batch * 4, cudaMemcpyHostToDevice, s),
     "copy seq_pos in");
  hfa_status st = hfa_decode_step(L, stream, L->x_stage, L->pos_stage, pos_host, batch, kc, vc,
                                  L->out_stage);
  if (st != HFA_OK) return st;
  CK(L, cudaMemcpyAsync(out_host, L->out_stage, xb, cudaMemcpyDeviceToHost, s), "copy out");
  CK(L, cudaStreamSynchronize(s), "sync");
  return HFA_OK;
}

// ------------------------------------------------------------------ verify block
extern "C" hfa_status hfa_verify_block(hfa_layer* L, void* stream, const void* x, int Lt,
                                       int base_pos, void* kc, void* vc, void* out) {
  if (!L) return HFA_EINVAL;
  const hfa_layer_desc& d = L->d;
  if (d.max_verify_len <= 0 || !L->verify)
    return fail(L, HFA_EINVAL, "layer created with max_verify_len = 0");
  if (!x || !kc || !vc || !out) return fail(L, HFA_EINVAL, "a pointer argument is NULL");
  if (Lt < 1 || Lt > d.max_verify_len)
    return fail(L, HFA_EINVAL, "L=%d outside [1, max_verify_len=%d]", Lt, d.max_verify_len);
  if (d.flags & HFA_F_RING) return fail(L, HFA_EUNSUPPORTED, "verify needs a linear cache");
  if (base_pos < 0 || (long long)base_pos + Lt > d.kv_capacity)
    return fail(L, HFA_ERANGE, "positions %d..%d outside the cache (capacity %d)", base_pos,
                base_pos + Lt - 1, d.kv_capacity);
  if (!aligned16(x) || !aligned16(kc) || !aligned16(vc) || !aligned16(out))
    return fail(L, HFA_EINVAL, "x, caches and out must be 16-byte aligned");
  if (!(d.flags & HFA_F_WEIGHTS_BF16))
    return fail(L, HFA_EUNSUPPORTED, "verify is built for bf16 weights");
  if ((long long)d.num_kv_heads * d.kv_capacity + 256 >= (1ll << 31))
    return fail(L, HFA_EUNSUPPORTED, "cache too large for 32-bit TMA rows");
  hfa::VerifyCall c{};
  c.d = &L->d;
  c.stream = (cudaStream_t)stream;
  c.x = (const __nv_bfloat16*)x;
  c.L = Lt;
  c.base_pos = base_pos;
  c.k_cache = (__nv_bfloat16*)kc;
  c.v_cache = (__nv_bfloat16*)vc;
  c.out = (__nv_bfloat16*)out;
  c.wqkv = L->wqkv_bf16;
  c.wo = L->wo_bf16;
  c.w_in = L->w_in;
  c.w_q = L->w_q;
  c.w_k = L->w_k;
  c.rope_g = L->rope_g;
  c.q_f32 = L->q_f32;
  c.o_f32 = L->o_f32;
  c.w_post = L->w_post_on ? L->w_post : nullptr;
  c.k_tap = L->k_tap;
  c.v_tap = L->v_tap;
  c.out_tap = L->out_tap;
  c.err = L->err;
  c.num_sms = L->num_sms;
  c.bidir = (d.flags & HFA_F_BLOCK_BIDIR) ? 1 : 0;
  LayerTimer lt;
  lt.L = L;
  c.timer = L->timing ? &lt : nullptr;
  char msg[256] = {0};
  hfa_status st = hfa::verify_run(L->verify, c, msg, sizeof msg);
  if (st != HFA_OK) return fail(L, st, "%s", msg);
  L->last_rows = Lt;
  return HFA_OK;
}

extern "C" hfa_status hfa_ctx_append(hfa_layer* L, void* stream, const void* x, int S, int base_pos,
                                     void* kc, void* vc) {
  if (!L) return HFA_EINVAL;
  const hfa_layer_desc& d = L->d;
  if (d.max_verify_len <= 0 || !L->verify)
    return fail(L, HFA_EINVAL, "layer created with max_verify_len = 0");
  if (!x || !kc || !vc) return fail(L, HFA_EINVAL, "a pointer argument is NULL");
  if (S < 1 || S > d.max_verify_len)
    return fail(L, HFA_EINVAL, "S=%d outside [1, max_verify_len=%d]", S, d.max_verify_len);
  if (d.flags & HFA_F_RING) return fail(L, HFA_EUNSUPPORTED, "context rows need a linear cache");
  if (base_pos < 0 || (long long)base_pos + S > d.kv_capacity)
    return fail(L, HFA_ERANGE, "positions %d..%d outside the cache (capacity %d)", base_pos,
                base_pos + S - 1, d.kv_capacity);
  if (!aligned16(x) || !aligned16(kc) || !aligned16(vc))
    return fail(L, HFA_EINVAL, "x_ctx and the caches must be 16-byte aligned");
  if (!(d.flags & HFA_F_WEIGHTS_BF16))
    return fail(L, HFA_EUNSUPPORTED, "context rows need bf16 weights");
  hfa::VerifyCall c{};
  c.d = &L->d;
  c.stream = (cudaStream_t)stream;
  c.x = (const __nv_bfloat16*)x;
  c.L = S;
  c.base_pos = base_pos;
  c.k_cache = (__nv_bfloat16*)kc;
  c.v_cache = (__nv_bfloat16*)vc;
  c.wqkv = L->wqkv_bf16;
  c.w_q = L->w_q;
  c.w_k = L->w_k;
  c.rope_g = L->rope_g;
  c.q_f32 = L->q_f32;
  c.k_tap = L->k_tap;
  c.v_tap = L->v_tap;
  c.err = L->err;
  c.num_sms = L->num_sms;
  LayerTimer lt;
  lt.L = L;
  c.timer = L->timing ? &lt : nullptr;
  char msg[256] = {0};
  hfa_status st = hfa::verify_ctx_append(L->verify, c, msg, sizeof msg);
  if (st != HFA_OK) return fail(L, st, "%s", msg);
  L->last_rows = S;
  return HFA_OK;
}

// ------------------------------------------------------------------ debug / status
extern "C" hfa_status hfa_debug_taps(hfa_layer* L, void* stream, float* q, float* k, float* v,
                                     float* attn, float* out) {
  if (!L) return HFA_EINVAL;
  if (!(L->d.flags & HFA_F_DEBUG_TAPS))
    return fail(L, HFA_EINVAL, "layer created without HFA_F_DEBUG_TAPS");
  if (L->last_rows == 0) return fail(L, HFA_EINVAL, "no step has run yet");
  cudaStream_t s = (cudaStream_t)stream;
  const size_t r = L->last_rows, nh = L->d.num_heads, nkv = L->d.num_kv_heads,
               hd = L->d.head_dim, H = L->d.hidden;
  auto cp = [&](float* dst, const float* src, size_t n) -> cudaError_t {
    return dst ? cudaMemcpyAsync(dst, src, n * 4, cudaMemcpyDeviceToDevice, s) : cudaSuccess;
  };
  CK(L, cp(q, L->q_f32, r * nh * hd), "tap q");
  CK(L, cp(k, L->k_tap, r * nkv * hd), "tap k");
  CK(L, cp(v, L->v_tap, r * nkv * hd), "tap v");
  CK(L, cp(attn, L->o_f32, r * nh * hd), "tap attn");
  CK(L, cp(out, L->out_tap, r * H), "tap out");
  return HFA_OK;
}

extern "C" hfa_status hfa_check_device_status(hfa_layer* L, void* stream) {
  if (!L) return HFA_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned v = 0;
  CK(L, cudaMemcpyAsync(&v, L->err, 4, cudaMemcpyDeviceToHost, s), "read status");
  CK(L, cudaStreamSynchronize(s), "sync");
  if (v == 0) return HFA_OK;
  CK(L, cudaMemsetAsync(L->err, 0, 4, s), "clear status");
  // a step that gave up may have left the grid barrier mid-count; the step numbers start
  // again, so the tagged partial sums of earlier steps are cleared with it
  CK(L, cudaMemsetAsync(L->gbar, 0, 8, s), "reset grid barrier");
  if (L->qkv_part)
    CK(L, cudaMemsetAsync(L->qkv_part, 0,
                          (size_t)L->g_qkv.S * L->d.max_batch * L->rows_qkv * 8, s), "reset");
  if (L->y_part)
    CK(L, cudaMemsetAsync(L->y_part, 0, (size_t)L->g_o.S * L->d.max_batch * L->d.hidden * 8, s),
       "reset");
  if (L->post_part)
    CK(L, cudaMemsetAsync(L->post_part, 0, (size_t)L->num_sms * 2 * 8, s), "reset");
  if (L->verify && hfa::verify_reset(L->verify, s) != HFA_OK)
    return fail(L, HFA_ECUDA, "reset of the verify partial sums failed");
  CK(L, cudaStreamSynchronize(s), "sync");
  return fail(L, HFA_EDEVICE, "device status 0x%x:%s%s%s", v,
              (v & kErrWaitTimeout) ? " a bounded wait gave up;" : "",
              (v & kErrBadPosition) ? " a position outside the cache was skipped;" : "",
              (v & kErrBadPlan) ? " inconsistent launch plan;" : "");
}

extern "C" int hfa_set_kernel_timing(hfa_layer* L, int enable) {
  if (!L) return -1;
  L->timing = enable != 0;
  return 0;
}

extern "C" int hfa_kernel_times(hfa_layer* L, int n, const char** names, float* total_ms,
                                int* launches) {
  if (!L) return -1;
  for (auto& t : L->pending) {
    cudaEventSynchronize(t.stop);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, t.start, t.stop);
    size_t i = 0;
    for (; i < L->slot_names.size(); ++i)
      if (L->slot_names[i] == t.name) break;
    if (i == L->slot_names.size()) {
      L->slot_names.push_back(t.name);
      L->slot_ms.push_back(0.f);
      L->slot_count.push_back(0);
    }
    L->slot_ms[i] += ms;
    L->slot_count[i] += 1;
    L->event_pool.push_back(t.start);
    L->event_pool.push_back(t.stop);
  }
  L->pending.clear();
  static const char* kNames[] = {"decode_step",       "flash_decode",      "verify_prep",
                                 "verify_qkv_gemm",   "verify_attention",  "verify_attn_merge",
                                 "verify_oproj_gemm", "verify_post_norm"};
  int k = 0;
  for (size_t i = 0; i < L->slot_names.size() && k < n; ++i, ++k) {
    const char* nm = "?";
    for (const char* c : kNames)
      if (L->slot_names[i] == c) nm = c;
    if (names) names[k] = nm;
    if (total_ms) total_ms[k] = L->slot_ms[i];
    if (launches) launches[k] = L->slot_count[i];
  }
  L->slot_names.clear();
  L->slot_ms.clear();
  L->slot_count.clear();
  return k;
}

extern "C" int hfa_plan_info(const hfa_layer* L, int n, int* v) {
  if (!L || !v) return -1;
  const int vals[5] = {L->last_splits, step_keys_per_tile(L->d.head_dim), L->last_gemv_grid,
                       L->last_attn_grid, L->num_sms};
  int k = n < 5 ? n : 5;
  for (int i = 0; i < k; ++i) v[i] = vals[i];
  return k;
}
