// kernels.h -- launchers of the TSP block kernels (one definition per .cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "tsp.h"

namespace tsp {

// rowwise.cu
tsp_status launch_zigzag_permute(const void* src, void* dst, int64_t S, int D, int64_t row_bytes,
                                 int inverse, cudaStream_t st);
// Element types of internal buffers.
enum { TY_F32 = 0, TY_BF16 = 1, TY_F16 = 2 };

// dtype TSP_F32: everything fp32.  dtype TSP_BF16: g is bf16; (u, out) is one
// of (fp32, fp16), (bf16, fp16), (bf16, bf16).
tsp_status launch_rmsnorm_fwd(const void* u, int u_ty, const void* g, void* out, int out_ty,
                              float* rstd, int64_t rows, int n, float eps, int dtype,
                              cudaStream_t st);
int rmsnorm_bwd_blocks(int64_t rows);
// du = rstd (dout g - nrm mean(dout g nrm)), nrm = u rstd; out = resid + du, where
// resid is resid_f32 (fp32) or resid_t (storage dtype), exactly one non-NULL;
// dg = sum over rows of dout * nrm (dg_part: rmsnorm_bwd_blocks(rows) x n fp32 scratch).
// dtype TSP_BF16: g and resid_t are bf16; (u, out_t) is (fp32, fp16) or (bf16, bf16).
tsp_status launch_rmsnorm_bwd(const float* dout, const void* u, int u_ty, const void* g,
                              const float* rstd, const float* resid_f32, const void* resid_t,
                              float* out_f32, void* out_t, int out_ty, float* dg, float* dg_part,
                              int64_t rows, int n, int dtype, cudaStream_t st);
tsp_status launch_convert_bf16_f16(const void* src, void* dst, int64_t n, cudaStream_t st);
tsp_status launch_convert_f32_f16(const float* src, void* dst, int64_t n, cudaStream_t st);
// rotary embedding: table[row][j] = (cos, sin) of pos(row) * base^(-2j/dh), j < dh/2,
// pos(row) the global position of zigzag row `row`; then rotate the Q (cols
// [0, d)) and K (cols [d, 2d)) blocks of a [S, ld] buffer of type ty in place
tsp_status launch_rope_table(float2* table, int64_t S, int D, int dh, float base, cudaStream_t st);
// (Q: H heads at column 0; K: Hkv heads at column d)
tsp_status launch_rope(void* qkv, int ty, int64_t S, int ld, int d, int H, int Hkv, int dh,
                       const float2* table, int inverse, cudaStream_t st);
// up to kMaxConvert conversions (n[k] elements each, multiples of 8) in one launch
constexpr int kMaxConvert = 8;
tsp_status launch_convert_bf16_f16_many(const void* const* src, void* const* dst, const int64_t* n,
                                        int count, cudaStream_t st);
tsp_status launch_swiglu_f32(const float* AB, float* G, int64_t rows, int I, cudaStream_t st);
tsp_status launch_swiglu_bwd_f32(const float* dG, const float* AB, float* dAB, int64_t rows, int I,
                                 cudaStream_t st);
tsp_status launch_pack_attn_shards(const void* wq, const void* wk, const void* wv, const void* wo,
                                   void* dst, int d, int D, int dtype, cudaStream_t st);
tsp_status launch_pack_mlp_shards(const void* w1, const void* w3, const void* w2, void* dst, int d,
                                  int I, int D, int dtype, cudaStream_t st);

// simt_f32.cu
tsp_status launch_gemm_f32(int M, int N, int K, const float* A, int64_t sam, int64_t sak,
                           const float* B, int64_t sbn, int64_t sbk, float* C, int64_t ldc,
                           const float* R, int64_t ldr, int acc, cudaStream_t st);
// QKV: [S, d + 2*Hkv*dh] (Q | K | V); query head h reads K/V head h / (H / Hkv)
tsp_status launch_attn_f32_fwd(const float* QKV, int64_t S, int H, int Hkv, int dh, int D, float* O,
                               float* LSE, cudaStream_t st);
tsp_status launch_attn_f32_bwd(const float* QKV, const float* O, const float* dO, const float* LSE,
                               float* delta, float* dQKV, int64_t S, int H, int Hkv, int dh, int D,
                               cudaStream_t st);

// attn_fwd.cu
tsp_status launch_attn_fwd_f16(const void* qkv, void* o, float* lse, int64_t S, int H, int Hkv, int dh,
                                int D, cudaStream_t st);
// one virtual rank r's query rows (multi-head, H heads of width dh): q [2c, ldq]
// its own rows (head h at column h*dh), kv [S, ldkv] the gathered K|V in zigzag
// row order (K head h at h*dh, V at H*dh + h*dh); o [2c, ldo], lse [H, 2c].
// When the rank's blocks alone would fill too few SMs the key range is split
// into chunks merged by log-sum-exp: part_o / part_lse, fp32 scratch of
// H * n_items_max * 256 * (dh + 1) floats (attn_rank_split_plan), then hold
// the chunks' partials (null when the plan has no split).
tsp_status launch_attn_fwd_rank_f16(const void* q, int64_t ldq, const void* kv, int64_t ldkv,
                                    void* o, int64_t ldo, float* lse, float* part_o,
                                    float* part_lse, int64_t S, int H, int dh, int D, int r,
                                    cudaStream_t st);
// lc = key tiles per chunk (0: no split) and the bound on one head's chunks
void attn_rank_split_plan(int64_t S, int D, int H, int* lc, int* n_items_max);

// attn_bwd.cu (delta: 2 x H x S fp32 scratch, -Delta then -LSE*log2(e))
tsp_status launch_attn_bwd_f16(const void* qkv, const void* o, const void* dO, const float* lse,
                                float* delta, float* dq_acc, void* dqkv, int64_t S, int H, int Hkv, int dh,
                                int D, cudaStream_t st);
// One rank's query rows (2c rows: Q, O, dO [2c, Hk*dh] fp16, LSE [Hk][2c]) of
// Hk heads against the gathered K|V [S, 2*Hk*dh] (zigzag row order): dQ
// [2c, Hk*dh] fp16, and dK|dV [S, 2*Hk*dh] fp16 for every key (the rank's
// queries' share; zero where none reaches).  delta: 2*Hk*2c fp32 scratch,
// dq_acc: 2c*Hk*dh fp32 scratch.
tsp_status launch_attn_bwd_rank_f16(const void* q, const void* kv, const void* o, const void* dO,
                                    const float* lse, float* delta, float* dq_acc, void* dq,
                                    void* dkv, int64_t S, int Hk, int dh, int D, int r,
                                    cudaStream_t st);

// decode.cu: inference decode against the zigzag KV cache
enum { GEMV_STORE = 0, GEMV_RES = 1, GEMV_SWIGLU = 2, GEMV_QKV = 3 };
struct Gemv {
  int epi = GEMV_STORE;
  int dtype = TSP_BF16;        // TSP_BF16: W bf16, x fp16; TSP_F32: W and x fp32
  const void* x = nullptr;     // [T, K], row stride ldx elements
  int64_t ldx = 0;
  const void* w[3] = {nullptr, nullptr, nullptr};   // weight segments [rows[s], K], stacked
  int rows[3] = {0, 0, 0};     // (GEMV_SWIGLU: w[0] = W1, w[1] = W3, both rows[0] rows)
  int nseg = 1;
  int K = 0, T = 0;
  void* out = nullptr;         // [T, N], row stride ldo elements, type out_ty
  int64_t ldo = 0;
  int out_ty = TY_F16;
  const void* res = nullptr;   // GEMV_RES: out = x W^T + res (type res_ty, stride ldr)
  int64_t ldr = 0;
  int res_ty = TY_F32;
  // GEMV_QKV (segments W_Q, W_K, W_V): rows computed in pairs (j, j + dh/2) of
  // one head; the first qk_heads heads (Q and K) are rotated at positions
  // pos0 + t when rope_base > 0; columns >= d (K | V) are also written to the
  // cache rows pos0 + t (row stride ldkv)
  int dh = 0, qk_heads = 0, d = 0;
  float rope_base = 0.f;
  int64_t pos0 = 0;
  void* kv = nullptr;
  int64_t ldkv = 0;
  int64_t kv_rows = 0;         // rows of the cache (bound of the appended rows)
  const char* name = "gemv";
};
tsp_status launch_gemv(const Gemv& g, cudaStream_t st);
// partial attention of the T new query rows over the cache rows, one split of
// cache rows per CTA, then the log-sum-exp merge of the splits into O [T, d]
struct DecodeAttn {
  int dtype = TSP_BF16;        // cache / q / O element type: fp16 (TSP_BF16) or fp32
  const void* q = nullptr;     // [T, ldq], query head h at column h*dh
  int64_t ldq = 0;
  const void* kv = nullptr;    // cache rows [K | V], row stride 2*Hkv*dh
  void* o = nullptr;           // [T, d]
  float* part_o = nullptr;     // [nsplit][H][T][dh]
  float2* part_ml = nullptr;   // [nsplit][H][T] (max, sum) in log2 units
  int64_t S = 0, n_cached = 0; // prompt rows (zigzag), rows cached before this call
  int D = 1, T = 1, H = 1, Hkv = 1, dh = 0;
};
int64_t decode_splits(int64_t S, int D, int64_t n_rows);
tsp_status launch_decode_attn(const DecodeAttn& a, cudaStream_t st);

// api.cu: TSP_OK if the configuration is valid (the entry points' common check)
tsp_status cfg_status(const tsp_cfg* cfg);

// api.cu: the block forward and backward with the residual stream's element
// type chosen per call (the C entry points pass the cfg dtype; the stack keeps
// the stream between layers in fp32).  In a bf16 configuration x_f32 / y_f32 /
// dy_f32 select fp32 for x, y and dy; in an fp32 configuration everything is
// fp32 and the flags are ignored.  prep (nullable): fp16 weight copies made
// by tsp_block_weights_prepare (bf16 only), used instead of converting the
// weights in the call.  Arguments are checked as by tsp_block_fwd /
// tsp_block_bwd (and their _prepared forms).
tsp_status block_fwd_checked(const tsp_cfg* cfg, const void* x_z, bool x_f32, const tsp_attn_w* aw,
                             const tsp_mlp_w* mw, const void* prep, void* y_z, bool y_f32,
                             void* saved, void* ws, size_t ws_bytes, cudaStream_t st);
tsp_status block_bwd_checked(const tsp_cfg* cfg, const void* x_z, bool x_f32, const void* dy_z,
                             bool dy_f32, const void* saved, const tsp_attn_w* aw,
                             const tsp_mlp_w* mw, const void* prep, float* dx_z,
                             float* const* grads, void* ws, size_t ws_bytes, cudaStream_t st);

}  // namespace tsp
