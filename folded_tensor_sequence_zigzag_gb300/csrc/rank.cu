// rank.cu -- one rank's steps of the TSP forward schedule (per-rank calls).
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), section 2,
// "Runtime schedules".  Attention layers: the packed W_Q/W_K/W_V/W_O shards
// are broadcast one after another; every rank projects its own tokens with
// the shard it has just received, the K/V of the sequence is all-gathered,
// and every rank runs FlashAttention for its zigzag rows.  Gated-MLP layers:
// the W_1/W_2/W_3 shards travel around a ring and every rank accumulates its
// partial outputs locally, with no all-reduce.
//
// Each call here is what rank r computes between two exchanges of that
// schedule, on its own 2c rows (chunk r, then chunk 2D-1-r):
//   tsp_rank_attn_project  broadcast step k: a_r = rms(x_r) (at k = 0), then
//                          the rank's Q and its K|V of the heads in shard k;
//   (the caller all-gathers the ranks' K|V of shard k)
//   tsp_rank_attn_heads    attention of the rank's rows for shard k's heads
//                          against the gathered K|V, and the W_O shard added
//                          onto the fp32 residual rows;
//   tsp_rank_mlp_step      ring step t with the shard the rank holds,
//                          (r - t) mod D: G = silu(b W_1^T) * (b W_3^T),
//                          y += G W_2^T (b = rms(h) at t = 0).
// With head-aligned shards (D divides H) shard k carries whole heads, so the
// attention of a broadcast step needs only that shard's K/V: the layer
// streams shard by shard, each shard's weights used once.  The kernels are
// the block's own (tcgen05 GEMM, the zigzag attention in its one-rank mode).
#include <cstring>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"

namespace tsp {
namespace {

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
cudaStream_t S_(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int64_t bound(int64_t k, int64_t n, int D) { return k * n / D; }   // shard boundary floor(k n / D)

// per-rank workspace: pieces kept from one call to the next of the same rank
struct RankWs {
  void *a, *shard, *q, *o, *b, *g;
  float* lse;
  // backward: rstd of both norms, dy and dh in fp16, the MLP shard's A|B and
  // dA|dB, dO and dQ of the attention shard, and fp32 scratch
  float *rstd1, *rstd2, *delta, *dq_acc, *dg_part;
  void *dy16, *dh16, *ab, *dab, *dO, *dq;
  float *part_o, *part_lse;   // the attention's chunk partials (split plan; may be empty)
  size_t bytes;
};

RankWs rank_layout(const tsp_cfg* c, uint8_t* base) {
  const size_t rows = (size_t)(c->S / c->D), d = (size_t)c->d;
  const size_t maxC = (size_t)((c->d + c->D - 1) / c->D), maxI = (size_t)((c->inter + c->D - 1) / c->D);
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off += up256(bytes);
    return p;
  };
  RankWs W;
  W.a = take(rows * d * 2);                                       // rms(x_r), fp16
  W.shard = take(std::max(4 * maxC, 3 * maxI) * d * 2);           // the received shard, fp16
  W.q = take(rows * maxC * 2);                                    // Q of shard k's heads
  W.o = take(rows * maxC * 2);                                    // O of shard k's heads
  W.lse = (float*)take(maxC / (size_t)c->dh * rows * 4);
  W.b = take(rows * d * 2);                                       // rms(h_r), fp16
  W.g = take(rows * maxI * 2);                                    // G of the held MLP shard
  W.rstd1 = (float*)take(rows * 4);
  W.rstd2 = (float*)take(rows * 4);
  W.dy16 = take(rows * d * 2);
  W.dh16 = take(rows * d * 2);
  W.ab = take(rows * 2 * maxI * 2);                               // A | B of the held shard
  W.dab = take(rows * 2 * maxI * 2);                              // dA | dB
  W.dO = take(rows * maxC * 2);
  W.dq = take(rows * maxC * 2);
  W.delta = (float*)take(2 * (maxC / (size_t)c->dh) * rows * 4);  // -Delta and -LSE*log2(e)
  W.dq_acc = (float*)take(rows * maxC * 4);
  W.dg_part = (float*)take((size_t)rmsnorm_bwd_blocks((int64_t)rows) * d * 4);
  int lc = 0, n_items = 0;
  attn_rank_split_plan(c->S, c->D, (int)(maxC / (size_t)c->dh), &lc, &n_items);
  const size_t part_rows = maxC / (size_t)c->dh * (size_t)n_items * 256;
  W.part_o = lc ? (float*)take(part_rows * (size_t)c->dh * 4) : nullptr;
  W.part_lse = lc ? (float*)take(part_rows * 4) : nullptr;
  W.bytes = off;
  return W;
}

// shapes the per-rank calls take: the bf16 tensor-core path, the pages' block
// (multi-head attention, no rotary embedding), head-aligned shards of at least
// two heads, MLP shards a multiple of 32 wide
tsp_status check_rank_cfg(const tsp_cfg* c) {
  tsp_status r = cfg_status(c);
  if (r != TSP_OK) return r;
  if (c->dtype != TSP_BF16) return TSP_ERR_UNSUPPORTED;
  if ((c->Hkv != 0 && c->Hkv != c->H) || c->rope_base > 0.f) return TSP_ERR_UNSUPPORTED;
  if (c->dh != 128 || c->H % c->D != 0 || (c->H / c->D) < 2) return TSP_ERR_UNSUPPORTED;
  if ((c->S / (2 * c->D)) % 256 != 0 || c->d % 256 != 0) return TSP_ERR_UNSUPPORTED;
  if (c->inter % c->D != 0 || (c->inter / c->D) % 32 != 0) return TSP_ERR_UNSUPPORTED;
  return TSP_OK;
}

tsp_status check_ws(const tsp_cfg* c, void* ws, size_t ws_bytes) {
  if (!al16(ws) || ws_bytes < rank_layout(c, nullptr).bytes) return TSP_ERR_INVALID_ARG;
  return TSP_OK;
}

}  // namespace
}  // namespace tsp

using namespace tsp;

extern "C" {

size_t tsp_rank_workspace_bytes(const tsp_cfg* cfg) {
  if (check_rank_cfg(cfg) != TSP_OK) return 0;
  return rank_layout(cfg, nullptr).bytes;
}

tsp_status tsp_pack_mlp_shards(const tsp_cfg* cfg, const tsp_mlp_w* w, void* dst, void* stream) {
  tsp_status r = cfg_status(cfg);
  if (r != TSP_OK) return r;
  if (!w || !w->w1 || !w->w3 || !w->w2 || !dst) return TSP_ERR_INVALID_ARG;
  return launch_pack_mlp_shards(w->w1, w->w3, w->w2, dst, cfg->d, cfg->inter, cfg->D, cfg->dtype,
                                S_(stream));
}

tsp_status tsp_rank_attn_project(const tsp_cfg* cfg, int32_t r, int32_t k, const void* x_r,
                                 const void* g_attn, const void* shard_k, void* kv_k, void* ws,
                                 size_t ws_bytes, void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D || k < 0 || k >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(x_r) || !al16(g_attn) || !al16(shard_k) || !al16(kv_k)) return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  const int d = cfg->d;
  const int Ck = (int)(bound(k + 1, d, cfg->D) - bound(k, d, cfg->D));
  if (k == 0 && (st = launch_rmsnorm_fwd(x_r, TY_BF16, g_attn, W.a, TY_F16, nullptr, rows, d,
                                         cfg->eps, cfg->dtype, s)) != TSP_OK)
    return st;
  // the received shard (Q, K, V rows, then W_O^T rows) in the fp16 operand type
  if ((st = launch_convert_bf16_f16(shard_k, W.shard, (int64_t)4 * Ck * d, s)) != TSP_OK) return st;
  if (Ck % 256 == 0) {
    // one GEMM over the shard's Q, K and V rows: Q of the shard's heads for
    // the rank's rows into the workspace, K | V (the rank's part of the
    // all-gather) into kv_k
    TcGemm g;
    g.M = (int)rows; g.N = 3 * Ck; g.K = d;
    g.A[0] = W.a; g.lda[0] = d; g.kseg_len[0] = d;
    g.B[0] = W.shard; g.ldb[0] = d;
    g.epi = EPI_STORE; g.out_type = OUT_F16; g.out = W.q; g.ldo = Ck;
    g.n_split = Ck; g.out2 = kv_k; g.ldo2 = 2 * Ck; g.name = "rank_gemm_qkv";
    return gemm_tc(g, s);
  }
  TcGemm q;   // Q of the shard's heads for the rank's rows
  q.M = (int)rows; q.N = Ck; q.K = d;
  q.A[0] = W.a; q.lda[0] = d; q.kseg_len[0] = d;
  q.B[0] = W.shard; q.ldb[0] = d;
  q.epi = EPI_STORE; q.out_type = OUT_F16; q.out = W.q; q.ldo = Ck; q.name = "rank_gemm_q";
  if ((st = gemm_tc(q, s)) != TSP_OK) return st;
  TcGemm kv;  // K | V of the shard's heads: the rank's part of the all-gather
  kv.M = (int)rows; kv.N = 2 * Ck; kv.K = d;
  kv.A[0] = W.a; kv.lda[0] = d; kv.kseg_len[0] = d;
  kv.B[0] = (const uint8_t*)W.shard + (size_t)Ck * d * 2; kv.ldb[0] = d;
  kv.epi = EPI_STORE; kv.out_type = OUT_F16; kv.out = kv_k; kv.ldo = 2 * Ck; kv.name = "rank_gemm_kv";
  return gemm_tc(kv, s);
}

tsp_status tsp_rank_attn_heads(const tsp_cfg* cfg, int32_t r, int32_t k, const void* x_r,
                               const void* kv_all_k, float* h_r, void* ws, size_t ws_bytes,
                               void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D || k < 0 || k >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(x_r) || !al16(kv_all_k) || !al16(h_r)) return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  const int d = cfg->d;
  const int Ck = (int)(bound(k + 1, d, cfg->D) - bound(k, d, cfg->D));
  if ((st = launch_attn_fwd_rank_f16(W.q, Ck, kv_all_k, 2 * (int64_t)Ck, W.o, Ck, W.lse, W.part_o,
                                     W.part_lse, cfg->S,
                                     Ck / cfg->dh, cfg->dh, cfg->D, r, s)) != TSP_OK)
    return st;
  // h_r (+)= O_k W_O[:, C_k]^T; W_O[:, C_k]^T sits in the shard as [C_k, d]
  // rows: the B operand read MN-major.  Step 0 adds the residual x_r.
  TcGemm o;
  o.M = (int)rows; o.N = d; o.K = Ck;
  o.A[0] = W.o; o.lda[0] = Ck; o.kseg_len[0] = Ck;
  o.b_mn = true; o.B[0] = (const uint8_t*)W.shard + (size_t)3 * Ck * d * 2; o.ldb[0] = d;
  o.epi = EPI_RES; o.res = k == 0 ? x_r : (const void*)h_r; o.res_f32 = k != 0; o.ldr = d;
  o.out = h_r; o.out_type = OUT_F32; o.ldo = d; o.name = "rank_gemm_oproj";
  return gemm_tc(o, s);
}

tsp_status tsp_rank_mlp_step(const tsp_cfg* cfg, int32_t r, int32_t t, const float* h_r,
                             const void* g_mlp, const void* shard, float* y_r, void* y_out,
                             void* ws, size_t ws_bytes, void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D || t < 0 || t >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(h_r) || !al16(g_mlp) || !al16(shard) || !al16(y_r)) return TSP_ERR_INVALID_ARG;
  if (y_out && !al16(y_out)) return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  const int d = cfg->d, I = cfg->inter, D = cfg->D;
  const int sh = ((r - t) % D + D) % D;   // the shard rank r holds at ring step t
  const int Is = (int)(bound(sh + 1, I, D) - bound(sh, I, D));
  if (t == 0 && (st = launch_rmsnorm_fwd(h_r, TY_F32, g_mlp, W.b, TY_F16, nullptr, rows, d,
                                         cfg->eps, cfg->dtype, s)) != TSP_OK)
    return st;
  if ((st = launch_convert_bf16_f16(shard, W.shard, (int64_t)3 * Is * d, s)) != TSP_OK) return st;
  TcGemm g;   // G = silu(b W_1[I_s]^T) * (b W_3[I_s]^T)
  g.M = (int)rows; g.N = Is; g.K = d;
  g.A[0] = W.b; g.lda[0] = d; g.kseg_len[0] = d;
  g.B[0] = W.shard; g.B[1] = (const uint8_t*)W.shard + (size_t)Is * d * 2;
  g.ldb[0] = g.ldb[1] = d;
  g.paired = true; g.epi = EPI_SWIGLU; g.out = W.g; g.ldo = Is; g.name = "rank_gemm_w13_swiglu";
  if ((st = gemm_tc(g, s)) != TSP_OK) return st;
  // y (+)= G W_2[:, I_s]^T; W_2[:, I_s]^T sits in the shard as [I_s, d] rows
  // (B read MN-major).  Step 0 adds the residual h_r; the last step may write
  // the result in the API dtype instead of y_r.
  TcGemm o;
  o.M = (int)rows; o.N = d; o.K = Is;
  o.A[0] = W.g; o.lda[0] = Is; o.kseg_len[0] = Is;
  o.b_mn = true; o.B[0] = (const uint8_t*)W.shard + (size_t)2 * Is * d * 2; o.ldb[0] = d;
  o.epi = EPI_RES; o.res = t == 0 ? h_r : y_r; o.res_f32 = true; o.ldr = d;
  const bool last = t == D - 1 && y_out;
  o.out = last ? y_out : (void*)y_r; o.out_type = last ? OUT_BF16 : OUT_F32; o.ldo = d;
  o.name = "rank_gemm_w2";
  return gemm_tc(o, s);
}

// ---------------------------------------------------------------------------
// The backward of the schedule (reading R17): the same shards in reverse.
// ---------------------------------------------------------------------------

tsp_status tsp_rank_mlp_bwd_step(const tsp_cfg* cfg, int32_t r, int32_t t, const float* h_r,
                                 const void* g_mlp, const void* shard, const void* dy_r,
                                 float* grad, float* db_r, void* ws, size_t ws_bytes,
                                 void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D || t < 0 || t >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(h_r) || !al16(g_mlp) || !al16(shard) || !al16(dy_r) || !al16(grad) || !al16(db_r))
    return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  const int d = cfg->d, I = cfg->inter, D = cfg->D;
  const int sh = ((r - t) % D + D) % D;   // the shard rank r holds at ring step t
  const int Is = (int)(bound(sh + 1, I, D) - bound(sh, I, D));
  const size_t e = 2;
  if (t == 0) {
    if ((st = launch_rmsnorm_fwd(h_r, TY_F32, g_mlp, W.b, TY_F16, W.rstd2, rows, d, cfg->eps,
                                 cfg->dtype, s)) != TSP_OK)
      return st;
    if ((st = launch_convert_bf16_f16(dy_r, W.dy16, rows * d, s)) != TSP_OK) return st;
  }
  if ((st = launch_convert_bf16_f16(shard, W.shard, (int64_t)3 * Is * d, s)) != TSP_OK) return st;
  const uint8_t* w1s = (const uint8_t*)W.shard;
  const uint8_t* w2t = w1s + (size_t)2 * Is * d * e;   // W_2[:, I_s]^T, [I_s, d]
  {   // G and the pre-activations A | B of the held shard (recomputed)
    TcGemm g;
    g.M = (int)rows; g.N = Is; g.K = d;
    g.A[0] = W.b; g.lda[0] = d; g.kseg_len[0] = d;
    g.B[0] = w1s; g.B[1] = w1s + (size_t)Is * d * e; g.ldb[0] = g.ldb[1] = d;
    g.paired = true; g.epi = EPI_SWIGLU; g.out = W.g; g.ldo = Is;
    g.out2 = W.ab; g.ldo2 = 2 * (int64_t)Is;
    g.out3 = (uint8_t*)W.ab + (size_t)Is * e; g.ldo3 = 2 * (int64_t)Is;
    g.name = "rank_gemm_w13_recompute";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
  }
  {   // dG = dy W_2[:, I_s] -> dA | dB through the SwiGLU derivative
    TcGemm g;
    g.M = (int)rows; g.N = Is; g.K = d;
    g.A[0] = W.dy16; g.lda[0] = d; g.kseg_len[0] = d;
    g.B[0] = w2t; g.ldb[0] = d;
    g.epi = EPI_SWIGLU_BWD; g.e1 = W.ab; g.e2 = (const uint8_t*)W.ab + (size_t)Is * e;
    g.lde = 2 * (int64_t)Is;
    g.out = W.dab; g.ldo = 2 * (int64_t)Is;
    g.out2 = (uint8_t*)W.dab + (size_t)Is * e; g.ldo2 = 2 * (int64_t)Is;
    g.name = "rank_gemm_dgrad_w2_swiglu";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
  }
  {   // db (+)= [dA | dB] [W_1[I_s]; W_3[I_s]]
    TcGemm g;
    g.M = (int)rows; g.N = d; g.K = 2 * Is;
    g.A[0] = W.dab; g.lda[0] = 2 * Is; g.kseg_len[0] = 2 * Is;
    g.b_mn = true; g.B[0] = w1s; g.ldb[0] = d;
    if (t == 0) {
      g.epi = EPI_F32;
    } else {
      g.epi = EPI_RES; g.res = db_r; g.res_f32 = true; g.ldr = d; g.out_type = OUT_F32;
    }
    g.out = db_r; g.ldo = d; g.name = "rank_gemm_dgrad_w13";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
  }
  {   // the shard's gradient (+)= this rank's rows: [dA | dB]^T b, then G^T dy
    TcGemm g;
    g.M = 2 * Is; g.N = d; g.K = (int)rows;
    g.a_mn = true; g.A[0] = W.dab; g.lda[0] = 2 * Is; g.kseg_len[0] = (int)rows;
    g.b_mn = true; g.B[0] = W.b; g.ldb[0] = d;
    g.epi = EPI_RES; g.res = grad; g.res_f32 = true; g.ldr = d; g.out_type = OUT_F32;
    g.out = grad; g.ldo = d; g.name = "rank_gemm_wgrad_w13";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
    TcGemm g2;
    float* g2out = grad + (size_t)2 * Is * d;
    g2.M = Is; g2.N = d; g2.K = (int)rows;
    g2.a_mn = true; g2.A[0] = W.g; g2.lda[0] = Is; g2.kseg_len[0] = (int)rows;
    g2.b_mn = true; g2.B[0] = W.dy16; g2.ldb[0] = d;
    g2.epi = EPI_RES; g2.res = g2out; g2.res_f32 = true; g2.ldr = d; g2.out_type = OUT_F32;
    g2.out = g2out; g2.ldo = d; g2.name = "rank_gemm_wgrad_w2";
    return gemm_tc(g2, s);
  }
}

tsp_status tsp_rank_mlp_bwd_finish(const tsp_cfg* cfg, int32_t r, const float* h_r,
                                   const void* g_mlp, const float* db_r, const void* dy_r,
                                   float* dh_r, float* dg_mlp, void* ws, size_t ws_bytes,
                                   void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(h_r) || !al16(g_mlp) || !al16(db_r) || !al16(dy_r) || !al16(dh_r) || !al16(dg_mlp))
    return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  const int64_t rows = cfg->S / cfg->D;
  // dh = dy + RMSNorm_2 backward of db (fp32, and fp16 for the attention GEMMs)
  return launch_rmsnorm_bwd(db_r, h_r, TY_F32, g_mlp, W.rstd2, nullptr, dy_r, dh_r, W.dh16, TY_F16,
                            dg_mlp, W.dg_part, rows, cfg->d, cfg->dtype, S_(stream));
}

tsp_status tsp_rank_attn_bwd_heads(const tsp_cfg* cfg, int32_t r, int32_t k,
                                   const void* kv_all_k, float* grad_k, void* dkv_k, void* ws,
                                   size_t ws_bytes, void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D || k < 0 || k >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(kv_all_k) || !al16(grad_k) || !al16(dkv_k)) return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  const int d = cfg->d;
  const int Ck = (int)(bound(k + 1, d, cfg->D) - bound(k, d, cfg->D));
  const size_t e = 2;
  // O and LSE of the rank's rows for shard k's heads (recomputed)
  if ((st = launch_attn_fwd_rank_f16(W.q, Ck, kv_all_k, 2 * (int64_t)Ck, W.o, Ck, W.lse, W.part_o,
                                     W.part_lse, cfg->S,
                                     Ck / cfg->dh, cfg->dh, cfg->D, r, s)) != TSP_OK)
    return st;
  const uint8_t* wot = (const uint8_t*)W.shard + (size_t)3 * Ck * d * e;   // W_O[:, C_k]^T
  {   // dO = dh W_O[:, C_k]
    TcGemm g;
    g.M = (int)rows; g.N = Ck; g.K = d;
    g.A[0] = W.dh16; g.lda[0] = d; g.kseg_len[0] = d;
    g.B[0] = wot; g.ldb[0] = d;
    g.epi = EPI_STORE; g.out_type = OUT_F16; g.out = W.dO; g.ldo = Ck; g.name = "rank_gemm_dgrad_wo";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
  }
  {   // this rank's part of the gradient of W_O[:, C_k]^T: O^T dh
    TcGemm g;
    g.M = Ck; g.N = d; g.K = (int)rows;
    g.a_mn = true; g.A[0] = W.o; g.lda[0] = Ck; g.kseg_len[0] = (int)rows;
    g.b_mn = true; g.B[0] = W.dh16; g.ldb[0] = d;
    g.epi = EPI_F32; g.out = grad_k + (size_t)3 * Ck * d; g.ldo = d; g.name = "rank_gemm_wgrad_wo";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
  }
  // the rank's query rows back-propagated: dQ (kept), dK | dV of every key
  return launch_attn_bwd_rank_f16(W.q, kv_all_k, W.o, W.dO, W.lse, W.delta, W.dq_acc, W.dq, dkv_k,
                                  cfg->S, Ck / cfg->dh, cfg->dh, cfg->D, r, s);
}

tsp_status tsp_rank_attn_bwd_weights(const tsp_cfg* cfg, int32_t r, int32_t k,
                                     const void* dkv_own, float* grad_k, float* da_r, void* ws,
                                     size_t ws_bytes, void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D || k < 0 || k >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(dkv_own) || !al16(grad_k) || !al16(da_r)) return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  const int d = cfg->d;
  const int Ck = (int)(bound(k + 1, d, cfg->D) - bound(k, d, cfg->D));
  const size_t e = 2;
  {   // this rank's part of the gradients of W_Q[C_k], then W_K[C_k] | W_V[C_k]
    TcGemm g;
    g.M = Ck; g.N = d; g.K = (int)rows;
    g.a_mn = true; g.A[0] = W.dq; g.lda[0] = Ck; g.kseg_len[0] = (int)rows;
    g.b_mn = true; g.B[0] = W.a; g.ldb[0] = d;
    g.epi = EPI_F32; g.out = grad_k; g.ldo = d; g.name = "rank_gemm_wgrad_q";
    if ((st = gemm_tc(g, s)) != TSP_OK) return st;
    TcGemm g2;
    g2.M = 2 * Ck; g2.N = d; g2.K = (int)rows;
    g2.a_mn = true; g2.A[0] = dkv_own; g2.lda[0] = 2 * Ck; g2.kseg_len[0] = (int)rows;
    g2.b_mn = true; g2.B[0] = W.a; g2.ldb[0] = d;
    g2.epi = EPI_F32; g2.out = grad_k + (size_t)Ck * d; g2.ldo = d; g2.name = "rank_gemm_wgrad_kv";
    if ((st = gemm_tc(g2, s)) != TSP_OK) return st;
  }
  // da (+)= dQ W_Q[C_k] + [dK | dV] [W_K[C_k]; W_V[C_k]]: two K segments
  TcGemm g;
  g.M = (int)rows; g.N = d; g.K = 3 * Ck; g.nks = 2;
  g.A[0] = W.dq; g.lda[0] = Ck; g.kseg_len[0] = Ck;
  g.A[1] = dkv_own; g.lda[1] = 2 * Ck; g.kseg_len[1] = 2 * Ck;
  g.b_mn = true; g.B[0] = W.shard; g.B[1] = (const uint8_t*)W.shard + (size_t)Ck * d * e;
  g.ldb[0] = g.ldb[1] = d;
  if (k == 0) {
    g.epi = EPI_F32;
  } else {
    g.epi = EPI_RES; g.res = da_r; g.res_f32 = true; g.ldr = d; g.out_type = OUT_F32;
  }
  g.out = da_r; g.ldo = d; g.name = "rank_gemm_dgrad_qkv";
  return gemm_tc(g, s);
}

tsp_status tsp_rank_attn_bwd_finish(const tsp_cfg* cfg, int32_t r, const void* x_r,
                                    const void* g_attn, const float* da_r, const float* dh_r,
                                    float* dx_r, float* dg_attn, void* ws, size_t ws_bytes,
                                    void* stream) {
  tsp_status st = check_rank_cfg(cfg);
  if (st != TSP_OK) return st;
  if (r < 0 || r >= cfg->D) return TSP_ERR_INVALID_ARG;
  if (!al16(x_r) || !al16(g_attn) || !al16(da_r) || !al16(dh_r) || !al16(dx_r) || !al16(dg_attn))
    return TSP_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != TSP_OK) return st;
  const RankWs W = rank_layout(cfg, (uint8_t*)ws);
  cudaStream_t s = S_(stream);
  const int64_t rows = cfg->S / cfg->D;
  // rstd of the first norm (the forward kept only its output)
  if ((st = launch_rmsnorm_fwd(x_r, TY_BF16, g_attn, W.a, TY_F16, W.rstd1, rows, cfg->d, cfg->eps,
                               cfg->dtype, s)) != TSP_OK)
    return st;
  // dx = dh + RMSNorm_1 backward of da
  return launch_rmsnorm_bwd(da_r, x_r, TY_BF16, g_attn, W.rstd1, dh_r, nullptr, dx_r, nullptr,
                            TY_BF16, dg_attn, W.dg_part, rows, cfg->d, cfg->dtype, s);
}

}  // extern "C"
