// C ABI of the library (include/llama_block.h): argument validation, workspace planning,
// RoPE frequency set-up, tensor-map encoding and kernel dispatch.  Nothing here allocates
// device memory, synchronises a stream (except llama_get_device_status) or touches the host
// copy of any tensor.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.h"

namespace llama {

// ------------------------------------------------------------------ device status word
__device__ unsigned g_device_status;

unsigned* status_ptr() {
  static unsigned* cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<unsigned*>(p);
  }
  return cached[dev];
}

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// ------------------------------------------------------------------ launch profiling
namespace prof {
struct Rec { const char* name; int a, b; };
static std::mutex mu;
static bool on = false;
static std::vector<cudaEvent_t> pool;
static size_t next = 0;
static std::vector<Rec> recs;
static int open_a = -1;
static const char* open_name = nullptr;

static int take() {
  if (next == pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
    pool.push_back(e);
  }
  return (int)next++;
}
static void begin(const char* name, cudaStream_t st) {
  if (!on) return;
  std::lock_guard<std::mutex> g(mu);
  open_a = take();
  open_name = name;
  if (open_a >= 0) cudaEventRecord(pool[open_a], st);
}
static void end(cudaStream_t st) {
  if (!on) return;
  std::lock_guard<std::mutex> g(mu);
  if (open_a < 0) return;
  const int b = take();
  if (b < 0) return;
  cudaEventRecord(pool[b], st);
  recs.push_back({open_name, open_a, b});
  open_a = -1;
}
}  // namespace prof

// ------------------------------------------------------------------ programmatic dependent launch
static thread_local bool t_pdl = false;
void set_pdl(bool on) { t_pdl = on; }
bool pdl_enabled() { return t_pdl; }

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_4d_u8(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                       const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t s[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t e[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool encode_tmap_4d_bf16(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                         const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t s[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t e[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// ------------------------------------------------------------------ helpers
namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline size_t esize(int dtype) { return dtype == LLAMA_F32 ? 4 : 2; }
inline size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

constexpr int64_t kMaxPos = (int64_t)1 << 24;

int check_dtype(int dtype) { return (dtype == LLAMA_F32 || dtype == LLAMA_BF16) ? LLAMA_OK : LLAMA_ERR_UNSUPPORTED; }

// Common shape checks; `need` selects which fields must be positive.
enum : unsigned { NEED_ROWS = 1, NEED_D = 2, NEED_HEADS = 4, NEED_FF = 8 };
int check_dims(const llama_dims* d, unsigned need) {
  if (!d) return LLAMA_ERR_INVALID_ARG;
  if (d->B < 0 || d->S < 0 || d->d_model < 0 || d->n_q < 0 || d->n_kv < 0 || d->head_dim < 0 || d->d_ff < 0)
    return LLAMA_ERR_INVALID_ARG;
  if ((need & NEED_D) && d->d_model <= 0) return LLAMA_ERR_INVALID_ARG;
  if (need & NEED_HEADS) {
    if (d->n_q <= 0 || d->n_kv <= 0 || d->head_dim <= 0 || d->n_q % d->n_kv != 0) return LLAMA_ERR_INVALID_ARG;
    if (d->head_dim % 2 != 0) return LLAMA_ERR_INVALID_ARG;
    if (d->head_dim > 2 * kMaxRopePairs) return LLAMA_ERR_UNSUPPORTED;
    if (!(d->theta_base > 0.0) || !std::isfinite(d->theta_base)) return LLAMA_ERR_INVALID_ARG;
  }
  if ((need & NEED_FF) && d->d_ff <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!(d->eps >= 0.0) || !std::isfinite(d->eps)) return LLAMA_ERR_INVALID_ARG;
  const int64_t big = (int64_t)1 << 31;
  if (d->B * d->S >= big || d->d_model >= big || d->d_ff >= big) return LLAMA_ERR_UNSUPPORTED;
  return LLAMA_OK;
}

// theta_k = theta_base^(-2k/head_dim), split into two floats (hi = fl(theta_k)).
void rope_freqs(const llama_dims* d, RopeFreq* out) {
  const int half = (int)(d->head_dim / 2);
  for (int k = 0; k < half; ++k) {
    const double th = std::pow(d->theta_base, -2.0 * (double)k / (double)d->head_dim);
    const float hi = (float)th;
    out[k].hi = hi;
    out[k].lo = (float)(th - (double)hi);
  }
}

int launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA;
}

// GEMM dispatch: tcgen05 for the bf16 shapes it supports, CUDA cores otherwise.
int run_gemm(const GemmDesc& g, const char* role, cudaStream_t st) {
  static const char* const tc_names[] = {"gemm_tc_store", "gemm_tc_resid", "gemm_tc_swiglu", "gemm_tc_qkv",
                                         "gemm_tc_atomic"};
  static const char* const simt_names[] = {"gemm_simt_store", "gemm_simt_resid", "gemm_simt_swiglu",
                                           "gemm_simt_qkv", "gemm_simt_atomic"};
  const bool tc = gemm_tc_supported(g);
  prof::begin(role ? role : (tc ? tc_names[g.epi.kind] : simt_names[g.epi.kind]), st);
  if (tc) {
    unsigned* status = status_ptr();
    if (!status) return LLAMA_ERR_CUDA;
    const int rc = gemm_tc2_supported(g) ? launch_gemm_tc2(g, status, st) : launch_gemm_tc(g, num_sms(), status, st);
    if (rc != 0) return LLAMA_ERR_CUDA;
  } else {
    if (launch_gemm_simt(g, st) != 0) return LLAMA_ERR_CUDA;
  }
  prof::end(st);
  return launch_status();
}

int run_attention(const AttnDesc& a, cudaStream_t st) {
  if (a.k_scale) {   // 8-bit cache: the tensor-core decode kernel is the only path
    if (!decode_attn8_supported(a)) return LLAMA_ERR_UNSUPPORTED;
    if (!a.ws || a.ws_bytes < decode_attn_ws_bytes(a)) return LLAMA_ERR_WORKSPACE;
    unsigned* status = status_ptr();
    if (!status) return LLAMA_ERR_CUDA;
    prof::begin("attn_decode_kv8", st);
    if (launch_decode_attn8(a, a.ws, num_sms(), status, st) != 0) return LLAMA_ERR_CUDA;
    prof::end(st);
    return launch_status();
  }
  if (a.block_table && !(decode_attn_supported(a) && a.ws && a.ws_bytes >= decode_attn_ws_bytes(a)))
    return LLAMA_ERR_UNSUPPORTED;   // a paged cache is read by the split-K decode kernel only
  if (decode_attn_supported(a) && a.ws && a.ws_bytes >= decode_attn_ws_bytes(a)) {
    unsigned* status = status_ptr();
    if (!status) return LLAMA_ERR_CUDA;
    prof::begin("attn_decode_tc", st);
    if (launch_decode_attn(a, a.ws, num_sms(), status, st) != 0) return LLAMA_ERR_CUDA;
    prof::end(st);
    return launch_status();
  }
  const bool tc = attn_tc_supported(a);
  prof::begin(tc ? "attn_tc" : "attn_simt", st);
  if (tc) {
    unsigned* status = status_ptr();
    if (!status) return LLAMA_ERR_CUDA;
    if (launch_attn_tc(a, num_sms(), status, st) != 0) return LLAMA_ERR_CUDA;
  } else {
    if (launch_attn_simt(a, st) != 0) return LLAMA_ERR_CUDA;
  }
  prof::end(st);
  return launch_status();
}

int run_rmsnorm(int dtype, int x_f32, int y_f32, const void* x, const void* g, void* y, int64_t rows, int64_t d,
                float eps, cudaStream_t st, float* rs_out = nullptr) {
  prof::begin("rmsnorm", st);
  if (launch_rmsnorm(dtype, x_f32, y_f32, x, g, y, rs_out, rows, d, eps, st) != 0) return LLAMA_ERR_UNSUPPORTED;
  prof::end(st);
  return launch_status();
}

Epi make_epi(int kind, int out_f32, void* out, int64_t ldo) {
  Epi e;
  memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.out_f32 = out_f32;
  e.out = out;
  e.ldo = ldo;
  e.S = 1;
  return e;
}

GemmDesc make_gemm(int dtype, int64_t M, const void* A, int64_t K) {
  GemmDesc g;
  memset(&g, 0, sizeof(g));
  g.M = M;
  g.K = K;
  g.dtype = dtype;
  g.A = A;
  g.lda = K;
  return g;
}

// Workspace carving: fixed-order, 256-byte aligned slices.
struct Carver {
  char* base;
  size_t off = 0;
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += round256(bytes);
    return p;
  }
};

// Scratch the attention call needs when a one-token step runs on the split-K decode kernel,
// sized for a cache of kv_capacity positions.
size_t attn_scratch_bytes(const llama_dims* d, int dtype, int64_t kv_capacity) {
  if (d->S != 1 || kv_capacity < 1) return 0;
  AttnDesc a;
  memset(&a, 0, sizeof(a));
  a.dtype = dtype; a.B = d->B; a.S = 1; a.n_q = d->n_q; a.n_kv = d->n_kv; a.hd = d->head_dim;
  a.pos0 = kv_capacity - 1;
  return (dtype == LLAMA_BF16 && d->head_dim == 128) ? decode_attn_ws_bytes(a) : 0;
}

struct BlockWs {
  void *u, *q, *o, *h, *m, *k, *v;
  float *rs1, *rs2;   // per-row RMSNorm factors of the attention and FFN norms
  float* ss;          // [T, d_model / 256] sums of squares of h per 256-column tile (fused FFN norm)
  float2* rope_tab;   // [S, hd/2] (cos, sin) of the call's positions
  void* attn;         // split-K attention scratch (one-token steps)
  size_t attn_bytes;
  size_t bytes;
};

BlockWs plan_block(const llama_dims* d, int dtype, bool own_kv, void* base, int64_t kv_capacity = 0) {
  const size_t es = esize(dtype);
  const size_t T = (size_t)(d->B * d->S);
  Carver c{static_cast<char*>(base)};
  BlockWs w;
  w.u = c.take(T * d->d_model * es);
  w.q = c.take(T * d->n_q * d->head_dim * es);
  w.o = c.take(T * d->n_q * d->head_dim * es);
  w.h = c.take(T * d->d_model * 4);     // residual stream after attention, kept in fp32
  w.m = c.take(T * d->d_ff * es);
  w.k = own_kv ? c.take(T * d->n_kv * d->head_dim * es) : nullptr;
  w.v = own_kv ? c.take(T * d->n_kv * d->head_dim * es) : nullptr;
  w.rs1 = static_cast<float*>(c.take(T * 4));
  w.rs2 = static_cast<float*>(c.take(T * 4));
  w.ss = static_cast<float*>(c.take(T * (size_t)((d->d_model + 127) / 128) * 4));
  w.rope_tab = static_cast<float2*>(c.take((size_t)d->S * (d->head_dim / 2) * sizeof(float2)));
  w.attn_bytes = attn_scratch_bytes(d, dtype, own_kv ? d->S : kv_capacity);
  w.attn = w.attn_bytes ? c.take(w.attn_bytes) : nullptr;
  w.bytes = c.off;
  return w;
}

struct DecodeWs {
  void *xres, *u, *q, *o, *m;
  float *rs1, *rs2;
  void* attn;
  size_t attn_bytes;
  size_t bytes;
};

DecodeWs plan_decode(const llama_dims* d, int dtype, void* base, int64_t kv_capacity) {
  const size_t es = esize(dtype);
  const size_t T = (size_t)d->B;
  Carver c{static_cast<char*>(base)};
  DecodeWs w;
  w.xres = c.take(T * d->d_model * 4);
  w.u = c.take(T * d->d_model * es);
  w.q = c.take(T * d->n_q * d->head_dim * es);
  w.o = c.take(T * d->n_q * d->head_dim * es);
  w.m = c.take(T * d->d_ff * es);
  w.rs1 = static_cast<float*>(c.take(T * 4));
  w.rs2 = static_cast<float*>(c.take(T * 4));
  w.attn_bytes = attn_scratch_bytes(d, dtype, kv_capacity);
  w.attn = w.attn_bytes ? c.take(w.attn_bytes) : nullptr;
  w.bytes = c.off;
  return w;
}

// The Q/K/V projection with RoPE on Q and K and the K/V write into [B, cap, n_kv*hd] caches.
int run_qkv(const llama_dims* d, int dtype, const llama_block_weights* w, const void* u, const float* row_scale,
            void* q, void* kc, void* vc, int64_t cap, int64_t pos0, cudaStream_t st, float2* rope_tab = nullptr,
            bool tab_ready = false) {
  const int64_t T = d->B * d->S, hq = d->n_q * d->head_dim, hkv = d->n_kv * d->head_dim;
  GemmDesc g = make_gemm(dtype, T, u, d->d_model);
  g.nseg = 3;
  g.B[0] = w->wq; g.nB[0] = hq;
  g.B[1] = w->wk; g.nB[1] = hkv;
  g.B[2] = w->wv; g.nB[2] = hkv;
  g.N = hq + 2 * hkv;
  g.epi = make_epi(EPI_QKV, dtype == LLAMA_F32, q, hq);
  g.epi.k_out = kc;
  g.epi.v_out = vc;
  g.epi.nq_cols = hq;
  g.epi.nkv_cols = hkv;
  g.epi.S = d->S;
  g.epi.cap = cap;
  g.epi.pos0 = pos0;
  g.epi.hd = (int)d->head_dim;
  g.epi.row_scale = row_scale;
  rope_freqs(d, g.epi.freq);
  if (rope_tab && !tab_ready) {   // one (cos, sin) per position and frequency, shared by every head
    prof::begin("rope_table", st);
    if (launch_rope_table(rope_tab, d->S, (int)d->head_dim, pos0, g.epi.freq, st) != 0) return LLAMA_ERR_CUDA;
    prof::end(st);
  }
  g.epi.rope_tab = rope_tab;
  return run_gemm(g, nullptr, st);
}

// out = resid + A W^T  (W [N, K])
GemmDesc linear_resid_desc(int dtype, int64_t M, const void* A, int64_t K, const void* W, int64_t N,
                           const void* resid, int resid_f32, void* out, int out_f32) {
  GemmDesc g = make_gemm(dtype, M, A, K);
  g.nseg = 1;
  g.B[0] = W; g.nB[0] = N;
  g.N = N;
  g.epi = make_epi(resid ? EPI_RESID : EPI_STORE, out_f32, out, N);
  g.epi.resid = resid;
  g.epi.resid_f32 = resid_f32;
  g.epi.ldr = N;
  return g;
}

int run_linear_resid(int dtype, int64_t M, const void* A, int64_t K, const void* W, int64_t N, const void* resid,
                     int resid_f32, void* out, int out_f32, cudaStream_t st) {
  return run_gemm(linear_resid_desc(dtype, M, A, K, W, N, resid, resid_f32, out, out_f32), nullptr, st);
}

GemmDesc gate_up_desc(int dtype, int64_t M, const void* A, int64_t K, const void* wg, const void* wu, int64_t dff,
                      void* m, const float* row_scale) {
  GemmDesc g = make_gemm(dtype, M, A, K);
  g.nseg = 2;
  g.B[0] = wg; g.nB[0] = dff;
  g.B[1] = wu; g.nB[1] = dff;
  g.N = 2 * dff;
  g.epi = make_epi(EPI_SWIGLU, dtype == LLAMA_F32, m, dff);
  g.epi.row_scale = row_scale;
  return g;
}

AttnDesc make_attn(const llama_dims* d, int dtype, const void* q, const void* k, const void* v, void* o, int64_t cap,
                   int64_t pos0) {
  AttnDesc a;
  memset(&a, 0, sizeof(a));
  a.dtype = dtype;
  a.q = q; a.k = k; a.v = v; a.o = o;
  a.B = d->B; a.S = d->S; a.n_q = d->n_q; a.n_kv = d->n_kv; a.hd = d->head_dim;
  a.cap = cap;
  a.pos0 = pos0;
  a.scale = (float)(1.0 / std::sqrt((double)d->head_dim));
  return a;
}

bool block_weights_ok(const llama_block_weights* w) {
  if (!w) return false;
  const void* ps[9] = {w->attn_norm_g, w->wq, w->wk, w->wv, w->wo, w->ffn_norm_g, w->w_gate, w->w_up, w->w_down};
  for (const void* p : ps)
    if (!p) return false;
  return true;
}
bool block_weights_aligned(const llama_block_weights* w) {
  const void* ps[9] = {w->attn_norm_g, w->wq, w->wk, w->wv, w->wo, w->ffn_norm_g, w->w_gate, w->w_up, w->w_down};
  for (const void* p : ps)
    if (!aligned16(p)) return false;
  return true;
}

// One block on already-validated arguments (shared by block_forward and the decode stack).
// x/y: dtype rows unless x_f32 (decode residual stream in fp32, updated in place: y == x).
// x_f32: x is fp32; y is fp32 when x_f32 or y_f32 is set (the residual stream of a stack).
int block_body(const llama_dims* d, int dtype, const llama_block_weights* w, const void* x, int x_f32, void* y,
               int64_t pos0, void* kc, void* vc, int64_t cap, const BlockWs& ws, cudaStream_t st, int y_f32 = 0) {
  const int64_t T = d->B * d->S, D = d->d_model, hq = d->n_q * d->head_dim;
  const int f32 = dtype == LLAMA_F32;
  const float eps = (float)d->eps;
  int rc;
  // RMSNorm(x; g_attn) = rs1 * (x * g_attn): the GEMM takes a = x * g_attn (exact in bf16 when the
  // gain is one) and multiplies its fp32 accumulator by rs1[row] before RoPE.
  // bf16 rows: the norm and the RoPE table of the call's positions in one launch
  const bool fused_tab = !x_f32 && !f32 && ws.rope_tab &&
                         rmsnorm_rope_table_ok(x, w->attn_norm_g, ws.u, T, D, d->S, (int)d->head_dim);
  if (fused_tab) {
    RopeFreq freq[kMaxRopePairs];
    rope_freqs(d, freq);
    prof::begin("rmsnorm", st);
    // the block's first kernel goes out without programmatic launch: what precedes it in the stream
    // may be a wait on another stream (a copy of x), which it must not overlap
    const bool pdl = pdl_enabled();
    set_pdl(false);
    const int lrc = launch_rmsnorm_rope_table(x, w->attn_norm_g, ws.u, ws.rs1, T, D, eps, ws.rope_tab, d->S,
                                              (int)d->head_dim, pos0, freq, st);
    set_pdl(pdl);
    if (lrc != 0) return LLAMA_ERR_UNSUPPORTED;
    prof::end(st);
    if ((rc = launch_status()) != LLAMA_OK) return rc;
  } else if ((rc = run_rmsnorm(dtype, x_f32 || f32, f32, x, w->attn_norm_g, ws.u, T, D, eps, st, ws.rs1)) !=
             LLAMA_OK) {
    return rc;
  }
  // q, k, v with RoPE; k, v written into the cache at pos0..pos0+S-1
  if ((rc = run_qkv(d, dtype, w, ws.u, ws.rs1, ws.q, kc, vc, cap, pos0, st, ws.rope_tab, fused_tab)) != LLAMA_OK)
    return rc;
  // o = causal GQA attention
  AttnDesc a = make_attn(d, dtype, ws.q, kc, vc, ws.o, cap, pos0);
  a.ws = ws.attn;
  a.ws_bytes = ws.attn_bytes;
  if ((rc = run_attention(a, st)) != LLAMA_OK) return rc;
  // h = x + o W_O^T, kept in fp32; an fp32 y holds it (the down projection then adds in place)
  y_f32 = y_f32 || x_f32 || f32;
  void* h = y_f32 ? y : ws.h;
  GemmDesc go = linear_resid_desc(dtype, T, ws.o, hq, w->wo, D, x, x_f32 || f32, h, 1);
  // m = SiLU(w W_gate^T) * (w W_up^T), w = RMSNorm(h; g_ffn) in the same split form (reuses u)
  GemmDesc gu = gate_up_desc(dtype, T, ws.u, D, w->w_gate, w->w_up, d->d_ff, ws.m, ws.rs2);
  // On the SM-pair GEMMs the norm needs no kernel of its own: the O projection's epilogue writes
  // h * g_ffn and the sums of squares of h per 128 columns, and the gate/up epilogue turns
  // the row's sums into its factor.
  const bool fuse = ws.ss && D % 256 == 0 && gemm_tc_supported(go) && gemm_tc2_supported(go) &&
                    gemm_tc_supported(gu) && gemm_tc2_supported(gu);
  if (fuse) {
    go.epi.norm_u = ws.u;
    go.epi.norm_g = w->ffn_norm_g;
    go.epi.ss_out = ws.ss;
    go.epi.ss_n = (int)(D / 128);
    gu.epi.row_scale = nullptr;
    gu.epi.ss_in = ws.ss;
    gu.epi.ss_n = (int)(D / 128);
    gu.epi.ss_inv_d = 1.0f / (float)D;
    gu.epi.ss_eps = eps;
  }
  if ((rc = run_gemm(go, nullptr, st)) != LLAMA_OK) return rc;
  if (!fuse && (rc = run_rmsnorm(dtype, 1, f32, h, w->ffn_norm_g, ws.u, T, D, eps, st, ws.rs2)) != LLAMA_OK)
    return rc;
  if ((rc = run_gemm(gu, nullptr, st)) != LLAMA_OK) return rc;
  // y = h + m W_down^T
  return run_linear_resid(dtype, T, ws.m, d->d_ff, w->w_down, D, h, 1, y, y_f32, st);
}

// ------------------------------------------------------------------------------------------
// Decode stack on the tensor cores.  Every projection is a weight-streaming GEMM over B <= 128
// token rows: 128-column tiles split along K into ~kDecodeUnits work units write fp32 partials,
// and a finisher reduces them and applies what follows (row scale, RoPE and the KV write,
// SiLU*mul, the residual add and the next RMSNorm).  GEMM inputs are passed as bf16 hi + lo
// parts (two MMAs per k-step into one accumulator): the weights are still read once, and the
// activations keep ~16 mantissa bits, which holds the 32-layer drift of a bf16-only data flow.
// ------------------------------------------------------------------------------------------
// K splits of a weight-streaming projection with fixed units (128-column tile, K range): the count
// (1..16) that minimises the k-blocks the busiest SM streams when the units are dealt out over
// the 152 SMs of the part; ties go to fewer splits (fewer partials for the finisher).  The 8B QKV
// projection (48 tiles x 64 k-blocks) gets 3 splits: 22 k-blocks on the busiest SM against an
// even share of 20.2 (7 splits, 336 units, would give 30).
constexpr int64_t kDecodeSms = 152;

int decode_splits(int64_t n_cols, int64_t K) {
  const int64_t tiles = (n_cols + 127) / 128;
  const int64_t nkb = (K + 63) / 64;
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int want = 1; want <= 16; ++want) {
    const int sp = gemm_skinny_splits(K, want);
    const int64_t kbps = (nkb + sp - 1) / sp;
    const int64_t cost = ((tiles * sp + kDecodeSms - 1) / kDecodeSms) * kbps;
    if (cost < best_cost) { best_cost = cost; best = sp; }
  }
  return best;
}

bool decode_tc_path(const llama_dims* d, int dtype) {
  if (dtype != LLAMA_BF16 || d->B > 128 || d->head_dim != 128 || d->d_model > 8192) return false;
  const int64_t hq = d->n_q * d->head_dim, hkv = d->n_kv * d->head_dim;
  if (d->d_model % 128 || hq % 128 || hkv % 128 || d->d_ff % 128) return false;
  const int64_t r = d->n_q / d->n_kv;
  return r == 1 || r == 2 || r == 4 || r == 8 || r == 16;
}

struct DecodeTcWs {
  float* xres;
  void* act;          // stacked GEMM input [2 Mp, width]: hi rows 0..B-1, lo rows Mp..Mp+B-1
  int64_t mp;
  void* q;
  float *rs1, *rs2, *part;
  void* attn;
  size_t attn_bytes, bytes;
  int s_qkv, s_o, s_gu, s_down;
};

DecodeTcWs plan_decode_tc(const llama_dims* d, void* base, int64_t kv_capacity) {
  const size_t Bn = (size_t)d->B;
  const int64_t hq = d->n_q * d->head_dim, hkv = d->n_kv * d->head_dim;
  DecodeTcWs w;
  w.s_qkv = decode_splits(hq + 2 * hkv, d->d_model);
  w.s_o = decode_splits(d->d_model, hq);
  w.s_gu = decode_splits(2 * d->d_ff, d->d_model);
  w.s_down = decode_splits(d->d_model, d->d_ff);
  const size_t act = (size_t)std::max(std::max(d->d_model, hq), d->d_ff);
  w.mp = skinny_mp(d->B);
  const size_t part = std::max((size_t)w.s_qkv * (hq + 2 * hkv), (size_t)w.s_gu * 2 * d->d_ff);
  Carver c{static_cast<char*>(base)};
  w.xres = static_cast<float*>(c.take(Bn * d->d_model * 4));
  w.act = c.take((size_t)(2 * w.mp) * act * 2);
  w.q = c.take(Bn * hq * 2);
  w.rs1 = static_cast<float*>(c.take(Bn * 4));
  w.rs2 = static_cast<float*>(c.take(Bn * 4));
  w.part = static_cast<float*>(c.take(Bn * part * 4));
  w.attn_bytes = attn_scratch_bytes(d, LLAMA_BF16, kv_capacity);
  w.attn = c.take(w.attn_bytes);
  w.bytes = c.off;
  return w;
}

// out = (X_hi + X_lo) W^T on the weight-streaming GEMM: fp32 split-K partials (mode 0), added
// into out (mode 1), or stored with the row scale (mode 2).
int run_skinny(const char* role, int64_t M, const void* x2, int64_t K, const void* const* W, const int64_t* n_rows,
               int nseg, int splits, int mode, float* out, int64_t ldo, const float* row_scale, cudaStream_t st) {
  SkinnyDesc g;
  memset(&g, 0, sizeof(g));
  g.M = M;
  g.K = K;
  g.X2 = x2;
  g.nseg = nseg;
  for (int s = 0; s < nseg; ++s) { g.W[s] = W[s]; g.nW[s] = n_rows[s]; }
  g.k_splits = splits;
  g.mode = mode;
  g.out = out;
  g.ldo = ldo;
  g.row_scale = row_scale;
  unsigned* status = status_ptr();
  if (!status) return LLAMA_ERR_CUDA;
  prof::begin(role, st);
  if (launch_gemm_skinny(g, num_sms(), status, st) != 0) return LLAMA_ERR_UNSUPPORTED;
  prof::end(st);
  return launch_status();
}

int run_fin(const char* role, int launch_rc, cudaStream_t st) {
  (void)role;
  if (launch_rc != 0) return LLAMA_ERR_CUDA;
  return launch_status();
}

// kv_scales: null for a bf16 cache; for an 8-bit cache, [n_layers][2 (K, V)][n_kv] fp32 scales.
// Where the decode step's K/V live: a dense cache [L, B, cap, n_kv, hd] with every sequence at
// position t, or (block_table set) a paged pool [L, n_pages, 128, n_kv, hd] with per-sequence
// positions seq_pos (t is then their upper bound).
struct PagedCache {
  const int* block_table = nullptr;
  const int* seq_pos = nullptr;
  int64_t max_pages = 0, n_pages = 0;
};

int decode_stack_tc(const llama_dims* d, int n_layers, const llama_block_weights* layers, const void* final_g,
                    const void* w_lm, int64_t vocab, const void* x_emb, void* k_cache, void* v_cache, int64_t cap,
                    int64_t t_cache, float* logits, const DecodeTcWs& w, const float* kv_scales, cudaStream_t st,
                    const PagedCache& pc = PagedCache()) {
  const int B = (int)d->B, D = (int)d->d_model;
  const int64_t hq = d->n_q * d->head_dim, hkv = d->n_kv * d->head_dim;
  const float eps = (float)d->eps;
  const bool paged = pc.block_table != nullptr;
  const size_t layer_cache = (size_t)((paged ? pc.n_pages * 128 : d->B * cap) * hkv) * (kv_scales ? 1 : 2);
  RopeFreq freq[kMaxRopePairs];
  rope_freqs(d, freq);
  int rc;
  for (int l = 0; l < n_layers; ++l) {
    const llama_block_weights& lw = layers[l];
    void* kc = static_cast<char*>(k_cache) + l * layer_cache;
    void* vc = static_cast<char*>(v_cache) + l * layer_cache;
    const float* ks = kv_scales ? kv_scales + (size_t)l * 2 * d->n_kv : nullptr;
    const float* vs = kv_scales ? ks + d->n_kv : nullptr;
    // (layer 0: x = embedding rows) a = x * g_attn (hi, lo); rs1
    prof::begin("fin_norm", st);
    rc = launch_fin_norm(w.xres, l == 0 ? x_emb : nullptr, nullptr, 0, lw.attn_norm_g, w.act,
                         static_cast<char*>(w.act) + w.mp * D * 2, w.rs1, B, D, eps, st);
    prof::end(st);
    if ((rc = run_fin("fin_norm", rc, st)) != LLAMA_OK) return rc;
    // Q/K/V partials
    const void* wqkv[3] = {lw.wq, lw.wk, lw.wv};
    const int64_t nqkv[3] = {hq, hkv, hkv};
    if ((rc = run_skinny("gemm_tc_dec_qkv", B, w.act, D, wqkv, nqkv, 3, w.s_qkv, 0, w.part, hq + 2 * hkv, nullptr,
                         st)) != LLAMA_OK)
      return rc;
    prof::begin("fin_qkv", st);
    rc = launch_fin_qkv(w.part, w.s_qkv, w.rs1, w.q, kc, vc, B, (int)hq, (int)hkv, (int)d->head_dim, cap, t_cache, freq,
                        ks, vs, pc.block_table, (int)pc.max_pages, pc.seq_pos, pc.n_pages, st);
    prof::end(st);
    if ((rc = run_fin("fin_qkv", rc, st)) != LLAMA_OK) return rc;
    // attention over t_cache + 1 keys; o as hi + lo into the activation buffers
    AttnDesc a = make_attn(d, LLAMA_BF16, w.q, kc, vc, w.act, cap, t_cache);
    a.o_lo = static_cast<char*>(w.act) + w.mp * hq * 2;
    a.ws = w.attn;
    a.ws_bytes = w.attn_bytes;
    a.k_scale = ks;
    a.v_scale = vs;
    a.block_table = pc.block_table;
    a.seq_pos = pc.seq_pos;
    a.max_pages = pc.max_pages;
    a.n_pages = pc.n_pages;
    if ((rc = run_attention(a, st)) != LLAMA_OK) return rc;
    // h = x + o W_O^T: the split-K partials are added straight into the fp32 residual stream
    const void* wo[1] = {lw.wo};
    const int64_t no[1] = {D};
    if ((rc = run_skinny("gemm_tc_dec_o", B, w.act, hq, wo, no, 1, w.s_o, 1, w.xres, D, nullptr, st)) != LLAMA_OK)
      return rc;
    // a2 = h * g_ffn (hi, lo); rs2
    prof::begin("fin_norm", st);
    rc = launch_fin_norm(w.xres, nullptr, nullptr, 0, lw.ffn_norm_g, w.act, static_cast<char*>(w.act) + w.mp * D * 2,
                         w.rs2, B, D, eps, st);
    prof::end(st);
    if ((rc = run_fin("fin_norm", rc, st)) != LLAMA_OK) return rc;
    // gate | up partials; m = SiLU(rs2 gate) * (rs2 up) (hi, lo)
    const void* wgu[2] = {lw.w_gate, lw.w_up};
    const int64_t ngu[2] = {d->d_ff, d->d_ff};
    if ((rc = run_skinny("gemm_tc_dec_gateup", B, w.act, D, wgu, ngu, 2, w.s_gu, 0, w.part, 2 * d->d_ff, nullptr,
                         st)) != LLAMA_OK)
      return rc;
    prof::begin("fin_swiglu", st);
    rc = launch_fin_swiglu(w.part, w.s_gu, w.rs2, w.act, static_cast<char*>(w.act) + w.mp * d->d_ff * 2, B,
                           (int)d->d_ff, st);
    prof::end(st);
    if ((rc = run_fin("fin_swiglu", rc, st)) != LLAMA_OK) return rc;
    // y = h + m W_down^T, added into the residual stream the same way
    const void* wd[1] = {lw.w_down};
    const int64_t nd[1] = {D};
    if ((rc = run_skinny("gemm_tc_dec_down", B, w.act, d->d_ff, wd, nd, 1, w.s_down, 1, w.xres, D, nullptr, st)) !=
        LLAMA_OK)
      return rc;
  }
  // final RMSNorm in split form, then the LM head with the row scale in its epilogue
  prof::begin("fin_norm", st);
  rc = launch_fin_norm(w.xres, nullptr, nullptr, 0, final_g, w.act, static_cast<char*>(w.act) + w.mp * D * 2, w.rs1,
                       B, D, eps, st);
  prof::end(st);
  if ((rc = run_fin("fin_norm", rc, st)) != LLAMA_OK) return rc;
  const void* wl[1] = {w_lm};
  const int64_t nl[1] = {vocab};
  if (vocab % 128 == 0)
    return run_skinny("gemm_tc_lm_head", B, w.act, D, wl, nl, 1, 1, 2, logits, vocab, w.rs1, st);
  // a vocabulary that is not a multiple of 128 rows: generic GEMM on the hi part with the row scale
  GemmDesc g = make_gemm(LLAMA_BF16, B, w.act, D);
  g.nseg = 1; g.B[0] = w_lm; g.nB[0] = vocab; g.N = vocab;
  g.epi = make_epi(EPI_STORE, 1, logits, vocab);
  g.epi.row_scale = w.rs1;
  return run_gemm(g, "gemm_lm_head", st);
}

}  // namespace
LLAMA_DEFINE_BOUNDS_READER(api)

}  // namespace llama

using namespace llama;

extern "C" {

int llama_build_info(void) { return kBoundsChecks ? LLAMA_BUILD_BOUNDS_CHECKS : 0; }

const char* llama_status_string(int status) {
  switch (status) {
    case LLAMA_OK: return "ok";
    case LLAMA_ERR_INVALID_ARG: return "invalid argument";
    case LLAMA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LLAMA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case LLAMA_ERR_WORKSPACE: return "workspace missing or too small";
    case LLAMA_ERR_CUDA: return "CUDA error";
    case LLAMA_ERR_TIMEOUT: return "device wait timed out";
    case LLAMA_ERR_BOUNDS: return "device index outside its tensor (bounds-checking build)";
    default: return "unknown status";
  }
}

int llama_profile_enable(int on) {
  std::lock_guard<std::mutex> g(prof::mu);
  prof::on = on != 0;
  return LLAMA_OK;
}

int llama_profile_read(int max_kinds, const char** names, int* launches, double* total_ms, int* n_kinds) {
  if (!n_kinds || max_kinds < 0 || (max_kinds > 0 && (!names || !launches || !total_ms))) return LLAMA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return LLAMA_ERR_CUDA;
  std::lock_guard<std::mutex> g(prof::mu);
  int n = 0;
  for (const prof::Rec& r : prof::recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, prof::pool[r.a], prof::pool[r.b]) != cudaSuccess) return LLAMA_ERR_CUDA;
    int i = 0;
    while (i < n && std::strcmp(names[i], r.name) != 0) ++i;
    if (i == n) {
      if (n == max_kinds) continue;
      names[n] = r.name; launches[n] = 0; total_ms[n] = 0.0; ++n;
    }
    launches[i] += 1;
    total_ms[i] += ms;
  }
  prof::recs.clear();
  prof::next = 0;
  *n_kinds = n;
  return LLAMA_OK;
}

int llama_get_device_status(int* out, void* stream) {
  if (!out) return LLAMA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return LLAMA_ERR_CUDA;
  unsigned* p = status_ptr();
  if (!p) return LLAMA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return LLAMA_ERR_CUDA;
  }
  unsigned bounds = 0;
  if (kBoundsChecks)
    bounds = bounds_read_clear_api() | bounds_read_clear_kernels_simt() | bounds_read_clear_gemm_tc() |
             bounds_read_clear_gemm_tc2() | bounds_read_clear_gemm_skinny() | bounds_read_clear_attn_tc() |
             bounds_read_clear_decode_attn() | bounds_read_clear_decode_attn8() | bounds_read_clear_decode_fin() |
             bounds_read_clear_sample() | bounds_read_clear_selftest();
  *out = (v & STATUS_TIMEOUT) ? LLAMA_ERR_TIMEOUT
         : bounds             ? LLAMA_ERR_BOUNDS
         : (v & STATUS_BAD_TOKEN) ? LLAMA_ERR_INVALID_ARG
                                  : LLAMA_OK;
  return LLAMA_OK;
}

int llama_sample(const float* logits, int64_t B, int64_t vocab, int64_t ld, float temperature, int64_t top_k,
                 float top_p, const float* u, int32_t* tokens, void* stream) {
  if (B < 0 || vocab < 1 || vocab > (int64_t(1) << 30) || ld < vocab || B > INT32_MAX) return LLAMA_ERR_INVALID_ARG;
  if (std::isnan(temperature) || std::isnan(top_p)) return LLAMA_ERR_INVALID_ARG;
  if (B == 0) return LLAMA_OK;
  if (!logits || !u || !tokens) return LLAMA_ERR_INVALID_ARG;
  if ((uintptr_t)logits % 4 || (uintptr_t)u % 4 || (uintptr_t)tokens % 4) return LLAMA_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  prof::begin("sample", st);
  const int rc = launch_sample(logits, B, vocab, ld, temperature, top_k, top_p, u, tokens, st);
  prof::end(st);
  return rc ? LLAMA_ERR_CUDA : launch_status();
}

int llama_embed(int dtype, const void* table, int64_t vocab, int64_t d_model, const int32_t* tokens, int64_t n,
                void* x, void* stream) {
  int rc;
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  if (vocab < 1 || d_model < 1 || n < 0 || n > INT32_MAX || vocab > INT32_MAX) return LLAMA_ERR_INVALID_ARG;
  if (n == 0) return LLAMA_OK;
  if (!table || !tokens || !x) return LLAMA_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  if (!status) return LLAMA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  prof::begin("embed", st);
  rc = launch_embed(dtype, table, vocab, d_model, tokens, n, x, status, st);
  prof::end(st);
  return rc ? LLAMA_ERR_CUDA : launch_status();
}

size_t llama_workspace_bytes(int op, const llama_dims* d, int dtype, int n_layers, int64_t vocab,
                             int64_t kv_capacity) {
  (void)n_layers; (void)vocab;
  if (!d || check_dtype(dtype) != LLAMA_OK) return 0;
  const size_t es = esize(dtype);
  switch (op) {
    case LLAMA_OP_SWIGLU_FFN: return round256((size_t)(d->B * d->S * d->d_ff) * es);
    case LLAMA_OP_GQA_ATTENTION: return attn_scratch_bytes(d, dtype, kv_capacity);
    case LLAMA_OP_BLOCK_FORWARD: return plan_block(d, dtype, kv_capacity <= 0, nullptr, kv_capacity).bytes;
    case LLAMA_OP_STACK_DECODE_STEP:
      return decode_tc_path(d, dtype) ? plan_decode_tc(d, nullptr, kv_capacity).bytes
                                      : plan_decode(d, dtype, nullptr, kv_capacity).bytes;
    default: return 0;
  }
}

int llama_rmsnorm(const llama_dims* d, int dtype, const void* x, const void* g, void* y, void* stream) {
  int rc;
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  if ((rc = check_dims(d, NEED_D)) != LLAMA_OK) return rc;
  const int64_t rows = d->B * d->S;
  if (rows == 0) return LLAMA_OK;
  if (!x || !g || !y) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(g) || !aligned16(y)) return LLAMA_ERR_ALIGNMENT;
  const int f32 = dtype == LLAMA_F32;
  return run_rmsnorm(dtype, f32, f32, x, g, y, rows, d->d_model, (float)d->eps, static_cast<cudaStream_t>(stream));
}

int llama_rope(const llama_dims* d, int dtype, void* q, void* k, int64_t pos0, void* stream) {
  int rc;
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  if ((rc = check_dims(d, NEED_HEADS)) != LLAMA_OK) return rc;
  if (pos0 < 0 || pos0 + d->S > kMaxPos) return LLAMA_ERR_INVALID_ARG;
  if (d->B * d->S == 0 || (!q && !k)) return LLAMA_OK;
  if ((q && !aligned16(q)) || (k && !aligned16(k))) return LLAMA_ERR_ALIGNMENT;
  RopeFreq f[kMaxRopePairs];
  rope_freqs(d, f);
  if (launch_rope(dtype, q, k, d->B, d->S, q ? d->n_q : 0, k ? d->n_kv : 0, (int)d->head_dim, pos0, f,
                  static_cast<cudaStream_t>(stream)) != 0)
    return LLAMA_ERR_CUDA;
  return launch_status();
}

int llama_gqa_attention(const llama_dims* d, int dtype, const void* q, const void* k, const void* v,
                        int64_t kv_capacity, int64_t pos0, void* o, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  if ((rc = check_dims(d, NEED_HEADS)) != LLAMA_OK) return rc;
  if (pos0 < 0 || kv_capacity < 0 || pos0 + d->S > kv_capacity || pos0 + d->S > kMaxPos) return LLAMA_ERR_INVALID_ARG;
  if (d->B * d->S == 0) return LLAMA_OK;
  if (!q || !k || !v || !o) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LLAMA_ERR_ALIGNMENT;
  if (ws_bytes > 0 && (!ws || !aligned16(ws))) return ws ? LLAMA_ERR_ALIGNMENT : LLAMA_ERR_WORKSPACE;
  if (ws_bytes < attn_scratch_bytes(d, dtype, pos0 + d->S)) return LLAMA_ERR_WORKSPACE;
  AttnDesc a = make_attn(d, dtype, q, k, v, o, kv_capacity, pos0);
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  return run_attention(a, static_cast<cudaStream_t>(stream));
}

int llama_swiglu_ffn(const llama_dims* d, int dtype, const void* x, const void* w_gate, const void* w_up,
                     const void* w_down, void* y, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  if ((rc = check_dims(d, NEED_D | NEED_FF)) != LLAMA_OK) return rc;
  const int64_t T = d->B * d->S;
  if (T == 0) return LLAMA_OK;
  if (!x || !w_gate || !w_up || !w_down || !y || x == y) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(y))
    return LLAMA_ERR_ALIGNMENT;
  const size_t need = llama_workspace_bytes(LLAMA_OP_SWIGLU_FFN, d, dtype, 0, 0, 0);
  if (!ws || ws_bytes < need) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = run_gemm(gate_up_desc(dtype, T, x, d->d_model, w_gate, w_up, d->d_ff, ws, nullptr), nullptr, st)) != LLAMA_OK)
    return rc;
  return run_linear_resid(dtype, T, ws, d->d_ff, w_down, d->d_model, nullptr, 0, y, dtype == LLAMA_F32, st);
}

int llama_block_forward(const llama_dims* d, int dtype_flags, const llama_block_weights* w, const void* x, void* y,
                        int64_t pos0, void* k_cache, void* v_cache, int64_t cache_capacity, void* ws, size_t ws_bytes,
                        void* stream) {
  int rc;
  const int dtype = dtype_flags & ~(LLAMA_X_F32 | LLAMA_Y_F32);
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  const int x_f32 = (dtype_flags & LLAMA_X_F32) ? 1 : 0, y_f32 = (dtype_flags & LLAMA_Y_F32) ? 1 : 0;
  if ((rc = check_dims(d, NEED_D | NEED_HEADS | NEED_FF)) != LLAMA_OK) return rc;
  if (!block_weights_ok(w) || !x || !y || x == y) return LLAMA_ERR_INVALID_ARG;
  const bool own_kv = !k_cache && !v_cache;
  if (!own_kv && (!k_cache || !v_cache)) return LLAMA_ERR_INVALID_ARG;
  if (own_kv) {
    if (pos0 != 0) return LLAMA_ERR_INVALID_ARG;
    cache_capacity = d->S;
  }
  if (pos0 < 0 || pos0 + d->S > cache_capacity || pos0 + d->S > kMaxPos) return LLAMA_ERR_INVALID_ARG;
  if (d->B * d->S == 0) return LLAMA_OK;
  if (!aligned16(x) || !aligned16(y) || !block_weights_aligned(w) || (k_cache && !aligned16(k_cache)) ||
      (v_cache && !aligned16(v_cache)))
    return LLAMA_ERR_ALIGNMENT;
  const size_t need = plan_block(d, dtype, own_kv, nullptr, cache_capacity).bytes;
  if (!ws || ws_bytes < need) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  BlockWs b = plan_block(d, dtype, own_kv, ws, cache_capacity);
  void* kc = own_kv ? b.k : k_cache;
  void* vc = own_kv ? b.v : v_cache;
  // the block's kernels that are made for it (the fused norm, the SM-pair GEMMs, the prefill
  // attention) go out with programmatic dependent launch: each one's set-up overlaps its
  // predecessor's tail, and each waits in griddepcontrol.wait before touching its inputs
  set_pdl(true);
  const int body_rc = block_body(d, dtype, w, x, x_f32, y, pos0, kc, vc, cache_capacity, b, static_cast<cudaStream_t>(stream),
                                 y_f32);
  set_pdl(false);
  return body_rc;
}

int llama_stack_decode_step(const llama_dims* d, int dtype, int n_layers, const llama_block_weights* layers,
                            const void* final_g, const void* w_lm, int64_t vocab, const void* x_emb, void* k_cache,
                            void* v_cache, int64_t cache_capacity, int64_t t_cache, float* logits, void* ws,
                            size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_dtype(dtype)) != LLAMA_OK) return rc;
  if ((rc = check_dims(d, NEED_D | NEED_HEADS | NEED_FF)) != LLAMA_OK) return rc;
  if (d->S != 1 || n_layers <= 0 || vocab <= 0 || !layers || !final_g || !w_lm || !x_emb || !k_cache || !v_cache ||
      !logits)
    return LLAMA_ERR_INVALID_ARG;
  if (t_cache < 0 || t_cache + 1 > cache_capacity || t_cache + 1 > kMaxPos) return LLAMA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!block_weights_ok(&layers[l])) return LLAMA_ERR_INVALID_ARG;
  if (d->B == 0) return LLAMA_OK;
  for (int l = 0; l < n_layers; ++l)
    if (!block_weights_aligned(&layers[l])) return LLAMA_ERR_ALIGNMENT;
  if (!aligned16(final_g) || !aligned16(w_lm) || !aligned16(x_emb) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(logits))
    return LLAMA_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (decode_tc_path(d, dtype)) {
    const size_t need_tc = plan_decode_tc(d, nullptr, cache_capacity).bytes;
    if (!ws || ws_bytes < need_tc) return LLAMA_ERR_WORKSPACE;
    if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
    // the decode chain's kernels may overlap their predecessors' tails (each waits for its inputs)
    set_pdl(true);
    const int rc_tc = decode_stack_tc(d, n_layers, layers, final_g, w_lm, vocab, x_emb, k_cache, v_cache, cache_capacity,
                                      t_cache, logits, plan_decode_tc(d, ws, cache_capacity), nullptr, st);
    set_pdl(false);
    return rc_tc;
  }
  const size_t need = plan_decode(d, dtype, nullptr, cache_capacity).bytes;
  if (!ws || ws_bytes < need) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  DecodeWs dw = plan_decode(d, dtype, ws, cache_capacity);
  const int64_t Bn = d->B, D = d->d_model;
  const size_t es = esize(dtype);
  // fp32 residual stream <- embedding rows
  if (dtype == LLAMA_F32) {
    if (cudaMemcpyAsync(dw.xres, x_emb, (size_t)(Bn * D) * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return LLAMA_ERR_CUDA;
  } else if (launch_widen_bf16(x_emb, static_cast<float*>(dw.xres), Bn * D, st) != 0) {
    return LLAMA_ERR_CUDA;
  }
  const size_t layer_cache = (size_t)(Bn * cache_capacity * d->n_kv * d->head_dim) * es;
  BlockWs b;
  b.u = dw.u; b.q = dw.q; b.o = dw.o; b.h = nullptr; b.m = dw.m; b.k = nullptr; b.v = nullptr; b.bytes = 0;
  b.rs1 = dw.rs1; b.rs2 = dw.rs2;
  b.ss = nullptr;         // the SM-pair GEMMs (and the fused norm) need at least 256 rows
  b.rope_tab = nullptr;   // one position per step: computed in the epilogue
  b.attn = dw.attn; b.attn_bytes = dw.attn_bytes;
  for (int l = 0; l < n_layers; ++l) {
    void* kc = static_cast<char*>(k_cache) + l * layer_cache;
    void* vc = static_cast<char*>(v_cache) + l * layer_cache;
    if ((rc = block_body(d, dtype, &layers[l], dw.xres, 1, dw.xres, t_cache, kc, vc, cache_capacity, b, st)) !=
        LLAMA_OK)
      return rc;
  }
  // z = RMSNorm(x; g_final); logits = z W_lm^T (fp32)
  if ((rc = run_rmsnorm(dtype, 1, dtype == LLAMA_F32, dw.xres, final_g, dw.u, Bn, D, (float)d->eps, st)) != LLAMA_OK)
    return rc;
  return run_linear_resid(dtype, Bn, dw.u, D, w_lm, vocab, nullptr, 0, logits, 1, st);
}

int llama_stack_decode_step_kv8(const llama_dims* d, int n_layers, const llama_block_weights* layers,
                                const void* final_g, const void* w_lm, int64_t vocab, const void* x_emb,
                                void* k_cache, void* v_cache, const float* kv_scales, int64_t cache_capacity,
                                int64_t t_cache, float* logits, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_dims(d, NEED_D | NEED_HEADS | NEED_FF)) != LLAMA_OK) return rc;
  if (d->S != 1 || n_layers <= 0 || vocab <= 0 || !layers || !final_g || !w_lm || !x_emb || !k_cache || !v_cache ||
      !kv_scales || !logits)
    return LLAMA_ERR_INVALID_ARG;
  if (t_cache < 0 || t_cache + 1 > cache_capacity || t_cache + 1 > kMaxPos) return LLAMA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!block_weights_ok(&layers[l])) return LLAMA_ERR_INVALID_ARG;
  if (!decode_tc_path(d, LLAMA_BF16)) return LLAMA_ERR_UNSUPPORTED;
  if (d->B == 0) return LLAMA_OK;
  for (int l = 0; l < n_layers; ++l)
    if (!block_weights_aligned(&layers[l])) return LLAMA_ERR_ALIGNMENT;
  if (!aligned16(final_g) || !aligned16(w_lm) || !aligned16(x_emb) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(logits) || ((uintptr_t)kv_scales & 3))
    return LLAMA_ERR_ALIGNMENT;
  const size_t need = plan_decode_tc(d, nullptr, cache_capacity).bytes;
  if (!ws || ws_bytes < need) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  set_pdl(true);
  rc = decode_stack_tc(d, n_layers, layers, final_g, w_lm, vocab, x_emb, k_cache, v_cache, cache_capacity, t_cache,
                       logits, plan_decode_tc(d, ws, cache_capacity), kv_scales, st);
  set_pdl(false);
  return rc;
}

int llama_stack_decode_step_paged(const llama_dims* d, int n_layers, const llama_block_weights* layers,
                                  const void* final_g, const void* w_lm, int64_t vocab, const void* x_emb,
                                  void* k_pool, void* v_pool, int64_t n_pages, const int32_t* block_table,
                                  int64_t max_pages, const int32_t* seq_pos, int64_t max_pos, float* logits, void* ws,
                                  size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_dims(d, NEED_D | NEED_HEADS | NEED_FF)) != LLAMA_OK) return rc;
  if (d->S != 1 || n_layers <= 0 || vocab <= 0 || !layers || !final_g || !w_lm || !x_emb || !k_pool || !v_pool ||
      !block_table || !seq_pos || !logits)
    return LLAMA_ERR_INVALID_ARG;
  if (n_pages < 1 || max_pages < 1 || max_pos < 0 || max_pos + 1 > max_pages * 128 || max_pos + 1 > kMaxPos ||
      n_pages > INT32_MAX || max_pages > INT32_MAX)
    return LLAMA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!block_weights_ok(&layers[l])) return LLAMA_ERR_INVALID_ARG;
  if (!decode_tc_path(d, LLAMA_BF16)) return LLAMA_ERR_UNSUPPORTED;
  if (d->B == 0) return LLAMA_OK;
  for (int l = 0; l < n_layers; ++l)
    if (!block_weights_aligned(&layers[l])) return LLAMA_ERR_ALIGNMENT;
  if (!aligned16(final_g) || !aligned16(w_lm) || !aligned16(x_emb) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(logits) || ((uintptr_t)block_table & 3) || ((uintptr_t)seq_pos & 3))
    return LLAMA_ERR_ALIGNMENT;
  const size_t need = plan_decode_tc(d, nullptr, max_pos + 1).bytes;
  if (!ws || ws_bytes < need) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  PagedCache pc;
  pc.block_table = block_table;
  pc.seq_pos = seq_pos;
  pc.max_pages = max_pages;
  pc.n_pages = n_pages;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  set_pdl(true);
  rc = decode_stack_tc(d, n_layers, layers, final_g, w_lm, vocab, x_emb, k_pool, v_pool, max_pos + 1, max_pos, logits,
                       plan_decode_tc(d, ws, max_pos + 1), nullptr, st, pc);
  set_pdl(false);
  return rc;
}

int llama_gqa_attention_decode_paged(const llama_dims* d, const void* q, const void* k_pool, const void* v_pool,
                                     int64_t n_pages, const int32_t* block_table, int64_t max_pages,
                                     const int32_t* seq_pos, int64_t max_pos, void* o, void* ws, size_t ws_bytes,
                                     void* stream) {
  int rc;
  if ((rc = check_dims(d, NEED_HEADS)) != LLAMA_OK) return rc;
  if (d->S != 1 || n_pages < 1 || max_pages < 1 || max_pos < 0 || max_pos + 1 > max_pages * 128 ||
      max_pos + 1 > kMaxPos || n_pages > INT32_MAX || max_pages > INT32_MAX)
    return LLAMA_ERR_INVALID_ARG;
  if (d->B == 0) return LLAMA_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_pos || !o) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) || ((uintptr_t)block_table & 3) ||
      ((uintptr_t)seq_pos & 3))
    return LLAMA_ERR_ALIGNMENT;
  AttnDesc a = make_attn(d, LLAMA_BF16, q, k_pool, v_pool, o, max_pos + 1, max_pos);
  a.block_table = block_table;
  a.seq_pos = seq_pos;
  a.max_pages = max_pages;
  a.n_pages = n_pages;
  if (!decode_attn_supported(a)) return LLAMA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < decode_attn_ws_bytes(a)) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  return run_attention(a, static_cast<cudaStream_t>(stream));
}

int llama_gqa_attention_decode_kv8(const llama_dims* d, const void* q, const void* k, const void* v,
                                   const float* k_scale, const float* v_scale, int64_t kv_capacity, int64_t pos0,
                                   void* o, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_dims(d, NEED_HEADS)) != LLAMA_OK) return rc;
  if (d->S != 1 || pos0 < 0 || kv_capacity < 0 || pos0 + 1 > kv_capacity || pos0 + 1 > kMaxPos)
    return LLAMA_ERR_INVALID_ARG;
  if (d->B == 0) return LLAMA_OK;
  if (!q || !k || !v || !o || !k_scale || !v_scale) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || ((uintptr_t)k_scale & 3) ||
      ((uintptr_t)v_scale & 3))
    return LLAMA_ERR_ALIGNMENT;
  AttnDesc a = make_attn(d, LLAMA_BF16, q, k, v, o, kv_capacity, pos0);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  if (!decode_attn8_supported(a)) return LLAMA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < decode_attn_ws_bytes(a)) return LLAMA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LLAMA_ERR_ALIGNMENT;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  return run_attention(a, static_cast<cudaStream_t>(stream));
}

int llama_kv_quantize(const void* x, int64_t n_tokens, int64_t n_kv, int64_t head_dim, const float* scale,
                      void* codes, void* stream) {
  if (n_tokens < 0 || n_kv < 1 || head_dim < 8 || head_dim % 8) return LLAMA_ERR_INVALID_ARG;
  if (n_tokens == 0) return LLAMA_OK;
  if (!x || !scale || !codes) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || ((uintptr_t)codes & 7) || ((uintptr_t)scale & 3)) return LLAMA_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  prof::begin("kv_quantize", st);
  const int rc = launch_kv_quantize(x, scale, codes, n_tokens * n_kv * head_dim, (int)n_kv, (int)head_dim, st);
  prof::end(st);
  return rc ? LLAMA_ERR_CUDA : launch_status();
}

}  // extern "C"
