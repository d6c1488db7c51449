// hfa_api.cu -- the C ABI of libhfa (declared in include/hfa.h).
//
// Host side only: argument validation (before any launch), ownership of the repacked
// weights and of the per-layer scratch, launch plans, and the kernel launches of one
// decode step: (1) input RMSNorm + QKV GEMV + per-head norm + RoPE + KV append,
// (2) split-K flash-decode with the chunk merge, (3) o_proj GEMV + residual.
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
  int G = 0;
  int rows_qkv = 0;
  int max_rows = 0;
  // weights
  Q8Tiles wqkv, wo;
  __nv_bfloat16* wqkv_bf16 = nullptr;  // verify path: [(nh + 2 nkv) hd, H]
  __nv_bfloat16* wo_bf16 = nullptr;    // [H, nh hd]
  float* w_in = nullptr;
  float* w_q = nullptr;
  float* w_k = nullptr;
  float2* rope_g = nullptr;
  // scratch
  float* qkv_acc = nullptr;
  int* head_ticket = nullptr;
  float* q_f32 = nullptr;
  float* attn_part = nullptr;
  int* attn_ticket = nullptr;
  float* o_f32 = nullptr;
  float* y_acc = nullptr;
  int* row_ticket = nullptr;
  float* k_tap = nullptr;
  float* v_tap = nullptr;
  float* out_tap = nullptr;
  unsigned* err = nullptr;
  __nv_bfloat16* x_stage = nullptr;
  int* pos_stage = nullptr;
  __nv_bfloat16* out_stage = nullptr;
  int max_splits = 0;
  hfa::VerifyState* verify = nullptr;
  // tensor maps of the caches of the last call
  const void* tm_k_ptr = nullptr;
  const void* tm_v_ptr = nullptr;
  int tm_rows = 0;
  CUtensorMap tm_k{}, tm_v{};
  // plan of the last call
  int last_splits = 0, last_gemv_grid = 0, last_attn_grid = 0;
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

bool hfa::encode_bf16_2d(CUtensorMap* map, void* base, int inner, int rows, int box_inner,
                         int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

static hfa_status validate_desc(const hfa_layer_desc* d) {
  if (!d) return fail(nullptr, HFA_EINVAL, "desc is NULL");
  if (d->hidden <= 0 || d->hidden % 64)
    return fail(nullptr, HFA_EINVAL, "hidden=%d must be a positive multiple of 64", d->hidden);
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
  if ((d->flags & HFA_F_RING) && (d->layer_type != HFA_SLIDING || d->kv_capacity != d->window))
    return fail(nullptr, HFA_EINVAL, "a ring cache needs a sliding layer with kv_capacity == window");
  if (d->max_batch < 1 || d->max_batch > 16)
    return fail(nullptr, HFA_EUNSUPPORTED, "max_batch=%d outside [1, 16]", d->max_batch);
  if (d->max_verify_len < 0 || d->max_verify_len > 16)
    return fail(nullptr, HFA_EUNSUPPORTED, "max_verify_len=%d outside [0, 16]", d->max_verify_len);
  if (!(d->eps >= 0.f) || !(d->rope_theta > 0.f) || !(d->attn_scale > 0.f) || !(d->softcap >= 0.f))
    return fail(nullptr, HFA_EINVAL, "eps, rope_theta, attn_scale, softcap out of range");
  if (d->flags & ~(HFA_F_V_UNIT_NORM | HFA_F_WEIGHTS_BF16 | HFA_F_RING | HFA_F_DEBUG_TAPS))
    return fail(nullptr, HFA_EINVAL, "unknown flags 0x%x", d->flags);
  return HFA_OK;
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
  if (!wq || !wk || !wv || !wo || !w_in || !w_q || !w_k)
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

  hfa_layer* L = new hfa_layer();
  L->d = *desc;
  L->device = dev;
  L->num_sms = prop.multiProcessorCount;
  const hfa_layer_desc& d = L->d;
  const int H = d.hidden, nh = d.num_heads, nkv = d.num_kv_heads, hd = d.head_dim;
  L->G = nh / nkv;
  L->rows_qkv = (nh + 2 * nkv) * hd;
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
    L->wqkv.rows = L->rows_qkv;
    L->wqkv.cols = H;
    LA(L->wqkv.q, (size_t)L->rows_qkv * H);
    LA(L->wqkv.d, (size_t)L->rows_qkv / 16 * (H / 32) * 8);
    L->wo.rows = H;
    L->wo.cols = nh * hd;
    LA(L->wo.q, (size_t)H * nh * hd);
    LA(L->wo.d, (size_t)H / 16 * (nh * hd / 32) * 8);
    LC(launch_repack_q8_0((const uint8_t*)wq, nh * hd, H, &L->wqkv, 0, s), "repack wq");
    LC(launch_repack_q8_0((const uint8_t*)wk, nkv * hd, H, &L->wqkv, nh * hd, s), "repack wk");
    LC(launch_repack_q8_0((const uint8_t*)wv, nkv * hd, H, &L->wqkv, (nh + nkv) * hd, s),
       "repack wv");
    LC(launch_repack_q8_0((const uint8_t*)wo, H, nh * hd, &L->wo, 0, s), "repack wo");
  } else {
    LA(L->wqkv_bf16, (size_t)L->rows_qkv * H);
    LA(L->wo_bf16, (size_t)H * nh * hd);
    const size_t qb = (size_t)nh * hd * H * 2, kb = (size_t)nkv * hd * H * 2;
    LC(cudaMemcpyAsync(L->wqkv_bf16, wq, qb, cudaMemcpyDeviceToDevice, s), "copy wq");
    LC(cudaMemcpyAsync((char*)L->wqkv_bf16 + qb, wk, kb, cudaMemcpyDeviceToDevice, s), "copy wk");
    LC(cudaMemcpyAsync((char*)L->wqkv_bf16 + qb + kb, wv, kb, cudaMemcpyDeviceToDevice, s),
       "copy wv");
    LC(cudaMemcpyAsync(L->wo_bf16, wo, (size_t)H * nh * hd * 2, cudaMemcpyDeviceToDevice, s),
       "copy wo");
  }
  LA(L->w_in, H);
  LA(L->w_q, hd);
  LA(L->w_k, hd);
  LC(cudaMemcpyAsync(L->w_in, w_in, H * 4, cudaMemcpyDeviceToDevice, s), "copy w_in");
  LC(cudaMemcpyAsync(L->w_q, w_q, hd * 4, cudaMemcpyDeviceToDevice, s), "copy w_q");
  LC(cudaMemcpyAsync(L->w_k, w_k, hd * 4, cudaMemcpyDeviceToDevice, s), "copy w_k");
  {
    // theta^(-2i/hd) / (2 pi) in double, stored as an fp32 (hi, lo) pair
    std::vector<float2> g(hd / 2);
    for (int i = 0; i < hd / 2; ++i) {
      double v = pow((double)d.rope_theta, -2.0 * i / hd) / (2.0 * M_PI);
      float hi = (float)v;
      g[i] = make_float2(hi, (float)(v - (double)hi));
    }
    LA(L->rope_g, hd / 2);
    LC(cudaMemcpyAsync(L->rope_g, g.data(), g.size() * sizeof(float2), cudaMemcpyHostToDevice, s),
       "copy rope table");
    LC(cudaStreamSynchronize(s), "create sync");
  }
  // scratch
  L->max_splits = 2 * L->num_sms;
  const int units = d.max_batch * nkv;
  LA(L->qkv_acc, (size_t)MR * L->rows_qkv);
  LA(L->head_ticket, nh + 2 * nkv);
  LA(L->q_f32, (size_t)MR * nh * hd);
  // one (m, l, O) record per attention chunk: units * splits <= max(2 SMs, units)
  LA(L->attn_part, (size_t)(units > L->max_splits ? units : L->max_splits) * attn_record_floats(hd));
  LA(L->attn_ticket, units);
  LA(L->o_f32, (size_t)MR * nh * hd);
  LA(L->y_acc, (size_t)MR * H);
  LA(L->row_ticket, H / 16);
  LA(L->err, 1);
  LA(L->x_stage, (size_t)d.max_batch * H);
  LA(L->pos_stage, d.max_batch);
  LA(L->out_stage, (size_t)d.max_batch * H);
  if (d.flags & HFA_F_DEBUG_TAPS) {
    LA(L->k_tap, (size_t)MR * nkv * hd);
    LA(L->v_tap, (size_t)MR * nkv * hd);
    LA(L->out_tap, (size_t)MR * H);
  }
  for (void* p : L->allocations) {
    (void)p;
  }
  LC(cudaMemsetAsync(L->qkv_acc, 0, (size_t)MR * L->rows_qkv * 4, s), "memset");
  LC(cudaMemsetAsync(L->head_ticket, 0, (nh + 2 * nkv) * 4, s), "memset");
  LC(cudaMemsetAsync(L->attn_ticket, 0, units * 4, s), "memset");
  LC(cudaMemsetAsync(L->y_acc, 0, (size_t)MR * H * 4, s), "memset");
  LC(cudaMemsetAsync(L->row_ticket, 0, H / 16 * 4, s), "memset");
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

static void fill_gemv_common(hfa_layer* L, GemvArgs& a, const Q8Tiles& w, int batch) {
  a.wq = w.q;
  a.wd = w.d;
  a.R = w.rows / 16;
  a.nb = w.cols / 32;
  a.batch = batch;
  a.cols = w.cols;
  a.err = L->err;
}

// k-split and grid of one GEMV: every warp streams the same number of tiles; the
// activation operand of the (at most two) k-splits a CTA touches must fit in shared memory.
// Work items of the GEMV: (k-split, row group) pairs of nbs tiles, one warp each, CTAs
// of gemv_items_per_cta() consecutive items.  nbs = 16 blocks (512 columns) where the row
// allows it, doubled while that leaves more than three CTAs per SM.
static void plan_gemv(hfa_layer* L, GemvArgs& a, int* grid, int* threads, size_t* smem) {
  const int ipc = gemv_items_per_cta();
  int nbs = a.nb % 16 == 0 ? 16 : (a.nb % 8 == 0 ? 8 : a.nb);
  const long long resident = (gemv_ntiles(a.batch) >= 4 ? 2LL : 3LL) * L->num_sms;  // CTAs
  while (a.nb % (2 * nbs) == 0 && (long long)(a.nb / nbs) * a.R / ipc > resident) nbs *= 2;
  a.S = a.nb / nbs;
  a.nbs = nbs;
  a.tiles = (long long)a.S * a.R * a.nbs;
  const int items = a.S * a.R;
  // k-splits one CTA's ipc consecutive items can span (one when R is a multiple of ipc)
  int spans = a.R % ipc == 0 ? 1 : (ipc - 1) / a.R + 2;
  if (spans > a.S) spans = a.S;
  const int blocks_max = spans * nbs;
  *smem = gemv_smem_bytes(a.batch, blocks_max);
  *threads = ipc * 32;
  *grid = (items + ipc - 1) / ipc;
}

static hfa_status launch_qkv(hfa_layer* L, cudaStream_t s, const void* x, const int* pos_dev,
                             int rows, bool tokens, void* kc, void* vc) {
  GemvArgs a{};
  fill_gemv_common(L, a, L->wqkv, rows);
  a.x = (const __nv_bfloat16*)x;
  a.w_in = L->w_in;
  a.eps = L->d.eps;
  a.acc = L->qkv_acc;
  a.ticket = L->head_ticket;
  a.nh = L->d.num_heads;
  a.nkv = L->d.num_kv_heads;
  a.hd = L->d.head_dim;
  a.C = L->d.kv_capacity;
  a.ring = (L->d.flags & HFA_F_RING) ? 1 : 0;
  a.w_q = L->w_q;
  a.w_k = L->w_k;
  a.rope_g = L->rope_g;
  a.seq_pos = pos_dev;
  a.v_unit_norm = (L->d.flags & HFA_F_V_UNIT_NORM) ? 1 : 0;
  a.q_out = L->q_f32;
  a.k_cache = (__nv_bfloat16*)kc;
  a.v_cache = (__nv_bfloat16*)vc;
  a.k_tap = L->k_tap;
  a.v_tap = L->v_tap;
  a.rows_are_tokens = tokens ? 1 : 0;
  int grid, threads;
  size_t smem;
  plan_gemv(L, a, &grid, &threads, &smem);
  L->last_gemv_grid = grid;
  KernelTimer t;
  timer_begin(L, s, "qkv_norm_rope_append", &t);
  cudaError_t e = launch_gemv(kModeQKV, a, grid, threads, smem, !L->timing, s);
  timer_end(L, s, &t);
  if (e != cudaSuccess) return cuda_fail(L, e, "qkv kernel launch");
  return HFA_OK;
}

static hfa_status launch_oproj(hfa_layer* L, cudaStream_t s, const void* x, int rows,
                               void* out) {
  GemvArgs a{};
  fill_gemv_common(L, a, L->wo, rows);
  a.x = (const __nv_bfloat16*)x;
  a.xin = L->o_f32;
  a.acc = L->y_acc;
  a.ticket = L->row_ticket;
  a.out = (__nv_bfloat16*)out;
  a.out_tap = L->out_tap;
  int grid, threads;
  size_t smem;
  plan_gemv(L, a, &grid, &threads, &smem);
  KernelTimer t;
  timer_begin(L, s, "oproj_residual", &t);
  cudaError_t e = launch_gemv(kModeOProj, a, grid, threads, smem, !L->timing, s);
  timer_end(L, s, &t);
  if (e != cudaSuccess) return cuda_fail(L, e, "o_proj kernel launch");
  return HFA_OK;
}

static hfa_status ensure_maps(hfa_layer* L, void* kc, void* vc, int rows) {
  if (L->tm_k_ptr == kc && L->tm_v_ptr == vc && L->tm_rows == rows) return HFA_OK;
  const int T = attn_keys_per_stage(L->d.head_dim);
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
  if (rows >= (1ll << 31)) return fail(L, HFA_EUNSUPPORTED, "cache too large for 32-bit TMA rows");
  hfa_status st = ensure_maps(L, kc, vc, (int)rows);
  if (st != HFA_OK) return st;

  // (1) input norm + QKV + per-head norm + RoPE + append
  st = launch_qkv(L, s, x, pos_dev, batch, false, kc, vc);
  if (st != HFA_OK) return st;

  // (2) attention
  AttnArgs aa{};
  int S = 0;
  fill_attn(aa, d.num_heads, nkv, hd, d.kv_capacity, d.layer_type, d.window, ring, d.attn_scale,
            d.softcap, batch, max_keys, L->num_sms, L->max_splits, &S);
  aa.q = L->q_f32;
  aa.seq_pos = pos_dev;
  aa.part = L->attn_part;
  aa.ticket = L->attn_ticket;
  aa.o = L->o_f32;
  aa.err = L->err;
  const int units = batch * nkv;
  L->last_splits = S;
  L->last_attn_grid = units * S;
  {
    KernelTimer t;
    timer_begin(L, s, "flash_decode", &t);
    cudaError_t e = launch_attn(aa, L->tm_k, L->tm_v, units * S, !L->timing, s);
    timer_end(L, s, &t);
    if (e != cudaSuccess) return cuda_fail(L, e, "attention kernel launch");
  }

  // (3) o_proj + residual
  st = launch_oproj(L, s, x, batch, out);
  if (st != HFA_OK) return st;
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
  if (rows >= (1ll << 31)) return fail(nullptr, HFA_EUNSUPPORTED, "cache too large");
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
  c.k_tap = L->k_tap;
  c.v_tap = L->v_tap;
  c.out_tap = L->out_tap;
  c.err = L->err;
  c.num_sms = L->num_sms;
  LayerTimer lt;
  lt.L = L;
  c.timer = L->timing ? &lt : nullptr;
  char msg[256] = {0};
  hfa_status st = hfa::verify_run(L->verify, c, msg, sizeof msg);
  if (st != HFA_OK) return fail(L, st, "%s", msg);
  L->last_rows = Lt;
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
  static const char* kNames[] = {"qkv_norm_rope_append", "flash_decode", "oproj_residual",
                                 "verify_prep", "verify_qkv_gemm", "verify_norm_rope_append", "verify_attention",
                                 "verify_oproj_gemm", "verify_residual"};
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
  const int vals[5] = {L->last_splits, attn_keys_per_stage(L->d.head_dim), L->last_gemv_grid,
                       L->last_attn_grid, L->num_sms};
  int k = n < 5 ? n : 5;
  for (int i = 0; i < k; ++i) v[i] = vals[i];
  return k;
}
