// Internal interface between the C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <utility>

#include "common.cuh"

namespace llama {

constexpr int kMaxRopePairs = 128;   // head_dim <= 256

// Bounds words of the translation units (see LLAMA_DEFINE_BOUNDS_READER in common.cuh).
unsigned bounds_read_clear_api();
unsigned bounds_read_clear_kernels_simt();
unsigned bounds_read_clear_gemm_tc();
unsigned bounds_read_clear_gemm_tc2();
unsigned bounds_read_clear_gemm_skinny();
unsigned bounds_read_clear_attn_tc();
unsigned bounds_read_clear_decode_attn();
unsigned bounds_read_clear_decode_attn8();
unsigned bounds_read_clear_decode_fin();
unsigned bounds_read_clear_sample();
unsigned bounds_read_clear_selftest();

// What a GEMM does with its fp32 result D[r, c] (r < M, c < N).
enum EpiKind : int {
  EPI_STORE = 0,   // out[r, c] = D
  EPI_RESID = 1,   // out[r, c] = resid[r, c] + D           (out may alias resid)
  EPI_SWIGLU = 2,  // out[r, j] = SiLU(D_gate[r, j]) * D_up[r, j]; B = (gate, up)
  EPI_QKV = 3,     // columns [0,nq) -> RoPE -> q; [nq, nq+nkv) -> RoPE -> k cache; rest -> v cache
  EPI_ATOMIC = 4,  // out[r, c] += D  (fp32 out; partial sums of a split K range)
};

struct Epi {
  int kind;
  int out_f32;          // 1: out is float32, 0: bf16
  const float* row_scale;  // when set, D[r, :] is first multiplied by row_scale[r]
  void* out;            // STORE/RESID/SWIGLU/ATOMIC: [M, ldo]; QKV: q [M, nq_cols]
  int64_t ldo;
  const void* resid;
  int resid_f32;
  int64_t ldr;
  // EPI_QKV: token r = b*S + s sits at position pos0 + s; its K/V row in the caches
  // [B, cap, nkv_cols] is b*cap + pos0 + s.
  void* k_out;
  void* v_out;
  int64_t nq_cols, nkv_cols;
  int64_t S, cap, pos0;
  int hd;
  const float2* rope_tab;   // optional [S, hd/2] (cos, sin) for positions pos0 .. pos0+S-1
  RopeFreq freq[kMaxRopePairs];
  // RMSNorm of the GEMM's output, split across two GEMMs (SM-pair kernel only):
  //   EPI_RESID with norm_u: also writes norm_u[r, c] = bf16(h[r, c] * norm_g[c]) (ld ldo) and the
  //   sum of squares of h over each 128-column half of a 256-column tile to ss_out[r * ss_n + half];
  //   any kind with ss_in: the row factor is rsqrt(sum_j ss_in[r * ss_n + j] * ss_inv_d + ss_eps).
  void* norm_u;
  const void* norm_g;   // bf16 [N]
  float* ss_out;
  const float* ss_in;
  int ss_n;
  float ss_inv_d, ss_eps;
  // extents for the bounds checks of -DLLAMA_DEBUG builds, set by the GEMM launchers
  // (epi_set_extents): rows of D, and rows of `out` (k_splits * M for split-K partials)
  int64_t M, out_rows;
};
inline void epi_set_extents(Epi& e, int64_t M, int64_t out_rows) {
  e.M = M;
  e.out_rows = out_rows;
}

// D[M, N] = A[M, K] * B[N, K]^T with B the row-concatenation of nseg segments
// (the returned split count can be lower than asked: see launch_gemm_tc)
// (for EPI_SWIGLU: B[0] = W_gate, B[1] = W_up, N = 2 * d_ff, output width d_ff).
struct GemmDesc {
  int64_t M, N, K;
  int dtype;            // LLAMA_F32 or LLAMA_BF16, for A and B
  const void* A;
  const void* A_lo;     // optional low bf16 part of A (A = A + A_lo), same layout; tcgen05 path only
  int64_t lda;          // elements
  int k_splits;         // > 1: fp32 partial sums of K ranges to out[split * M + r, c] (EPI_STORE only)
  int narrow;           // 1: 128-column tiles (more tiles for skinny M)
  const void* B[3];
  int64_t nB[3];        // rows of each segment
  int nseg;
  Epi epi;
};

struct AttnDesc {
  int dtype;
  const void* q;        // [B, S, n_q, hd]
  const void* k;        // [B, cap, n_kv, hd]
  const void* v;
  void* o;              // [B, S, n_q, hd]
  void* o_lo;           // decode kernel only, optional: low bf16 part of o
  int64_t B, S, n_q, n_kv, hd, cap, pos0;
  float scale;          // 1/sqrt(hd)
  void* ws;             // scratch for the split-K decode kernel (may be null)
  size_t ws_bytes;
  const float* k_scale; // 8-bit cache: k and v hold E4M3 codes, x = code * scale[kv head]
  const float* v_scale;
  const int* block_table;   // decode kernel, paged cache: k/v are pools [n_pages, 128, n_kv, hd]
  const int* seq_pos;       //   per-sequence new-token positions (pos0 = their upper bound)
  int64_t max_pages, n_pages;
};

// rows x d RMSNorm; x_f32/y_f32 give the element types of x and y, g has type `dtype`.
// rs_out == nullptr: y = x * rs * g.  Otherwise y = x * g and rs_out[row] = rs (split form).
int launch_rmsnorm(int dtype, int x_f32, int y_f32, const void* x, const void* g, void* y, float* rs_out,
                   int64_t rows, int64_t d, float eps, cudaStream_t st);
int launch_rope(int dtype, void* q, void* k, int64_t B, int64_t S, int64_t n_q, int64_t n_kv, int hd,
                int64_t pos0, const RopeFreq* freq, cudaStream_t st);
int launch_gemm_simt(const GemmDesc& g, cudaStream_t st);
int launch_attn_simt(const AttnDesc& a, cudaStream_t st);
int launch_widen_bf16(const void* src, float* dst, int64_t n, cudaStream_t st);
// tab[s, k] = (cos, sin)((pos0 + s) * theta_k) for s < S, k < hd/2.
int launch_rope_table(float2* tab, int64_t S, int hd, int64_t pos0, const RopeFreq* freq, cudaStream_t st);
// Both of the above in one launch, for bf16 rows in the split form (rs_out set) whose width takes
// the register path (16-byte aligned, d % 8 == 0, d <= 4096); returns -1 (nothing launched) otherwise.
bool rmsnorm_rope_table_ok(const void* x, const void* g, const void* y, int64_t rows, int64_t d, int64_t S, int hd);
int launch_rmsnorm_rope_table(const void* x, const void* g, void* y, float* rs, int64_t rows, int64_t d, float eps,
                              float2* tab, int64_t S, int hd, int64_t pos0, const RopeFreq* freq, cudaStream_t st);

// tensor-core paths (bf16 only)
bool gemm_tc_supported(const GemmDesc& g);
int launch_gemm_tc(const GemmDesc& g, int num_sms, unsigned* status, cudaStream_t st);
// Weight-streaming GEMM for M <= 128 token rows (decode): out = (X_hi + X_lo) W^T with the token
// rows stacked in X2 = [hi rows 0..M-1 | lo rows Mp..Mp+M-1], Mp = skinny_mp(M).
struct SkinnyDesc {
  int64_t M, K;
  const void* X2;
  const void* W[3];
  int64_t nW[3];          // rows of each weight segment (multiples of 128)
  int nseg;
  int k_splits;
  int mode;               // 0: fp32 partials out[split*M + c, n]; 1: atomic add out[c, n]; 2: store (x row_scale)
  float* out;
  int64_t ldo;
  const float* row_scale;
};
inline int64_t skinny_mp(int64_t M) { return M <= 64 ? 64 : 128; }
int launch_gemm_skinny(const SkinnyDesc& g, int num_sms, unsigned* status, cudaStream_t st);
int gemm_skinny_splits(int64_t K, int requested);

// The SM-pair (cta_group::2) version for large M: 256 x 256 tiles, no dual A / split K.
bool gemm_tc2_supported(const GemmDesc& g);
int launch_gemm_tc2(const GemmDesc& g, unsigned* status, cudaStream_t st);
// The number of K splits launch_gemm_tc uses for a requested count.
int gemm_tc_effective_splits(int64_t K, int requested);
bool attn_tc_supported(const AttnDesc& a);
bool decode_attn_supported(const AttnDesc& a);
size_t decode_attn_ws_bytes(const AttnDesc& a);   // for kv_len = pos0 + 1
int launch_decode_attn(const AttnDesc& a, void* ws, int num_sms, unsigned* status, cudaStream_t st);
void decode_attn_plan(int64_t kv_len, int& kv_tiles, int& chunk_tiles, int& n_chunks);
int launch_decode_combine(const float* part_o, const float* part_ml, void* o, void* o_lo, int64_t B, int64_t n_q,
                          int n_chunks, cudaStream_t st);
// decode_attn8.cu: the same over an 8-bit (E4M3) cache with per-head scales; same workspace size
bool decode_attn8_supported(const AttnDesc& a);
int launch_decode_attn8(const AttnDesc& a, void* ws, int num_sms, unsigned* status, cudaStream_t st);
// codes[i] = E4M3(fl32(x[i]) / scale[head of i]) for n bf16 elements laid out [.., n_kv, hd]
int launch_kv_quantize(const void* x, const float* scale, void* codes, int64_t n, int n_kv, int hd, cudaStream_t st);
int launch_attn_tc(const AttnDesc& a, int num_sms, unsigned* status, cudaStream_t st);

// Decode-step finishers (decode_fin.cu): split-K reductions fused with what follows each GEMM.
int launch_fin_norm(float* x, const void* init_bf16, const float* part, int n_split, const void* g, void* a_hi,
                    void* a_lo, float* rs, int B, int d, float eps, cudaStream_t st);
int launch_fin_qkv(const float* part, int n_split, const float* rs, void* q, void* kc, void* vc, int B, int nq_cols,
                   int nkv_cols, int hd, int64_t cap, int64_t t, const RopeFreq* freq, const float* k_scale,
                   const float* v_scale, const int* block_table, int max_pages, const int* seq_pos,
                   int64_t n_pages, cudaStream_t st);
int launch_fin_swiglu(const float* part, int n_split, const float* rs, void* m_hi, void* m_lo, int B, int dff,
                      cudaStream_t st);

// Kernels of the decode chain are launched with programmatic stream serialization (they may
// begin while their predecessor drains; see pdl_trigger / pdl_wait) while this is on.
void set_pdl(bool on);
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (pdl_enabled()) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// sample.cu: next-token choice (one CTA per row) and the embedding lookup
int launch_sample(const float* logits, int64_t B, int64_t V, int64_t ld, float temperature, int64_t top_k,
                  float top_p, const float* u, int* tokens, cudaStream_t st);
int launch_embed(int dtype, const void* table, int64_t V, int64_t d, const int* tokens, int64_t n, void* x,
                 unsigned* status, cudaStream_t st);

// The current device's status word (device address) and SM count.
unsigned* status_ptr();
int num_sms();

// tensor-map encoding (driver entry point resolved through the runtime)
bool encode_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
bool encode_tmap_4d_u8(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                       const uint32_t* box);
bool encode_tmap_4d_bf16(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                         const uint32_t* box);
bool encode_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

}  // namespace llama
