// stack.cu -- a stack of L TSP blocks (the multi-layer model the fold is
// applied to) and the per-virtual-rank memory account of the fold.
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), sections 1-3:
// every rank holds 1/D of the parameters and 1/D of the tokens of every
// layer, and the fold is the only layout of the compared ones that cuts both
// weight and activation memory by D without D^2 devices.  The stack here is
// the plain composition y = B_{L-1}(... B_0(x)); each block is tsp_block_fwd /
// tsp_block_bwd with its own weights, so every step still runs in the block's
// kernels.
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace tsp {
namespace {

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }
size_t elt_of(const tsp_cfg* c) { return c->dtype == TSP_BF16 ? 2 : 4; }
size_t act_bytes(const tsp_cfg* c) { return up256((size_t)c->S * c->d * elt_of(c)); }
bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

// per-layer slot of the training record: the layer's input, then the block's
// saved activations
size_t layer_slot(const tsp_cfg* c) { return act_bytes(c) + up256(tsp_saved_bytes(c)); }

}  // namespace
}  // namespace tsp

using namespace tsp;

extern "C" {

size_t tsp_stack_saved_bytes(const tsp_cfg* cfg, int32_t L) {
  if (L < 1 || tsp_saved_bytes(cfg) == 0) return 0;
  return (size_t)L * layer_slot(cfg);
}

size_t tsp_stack_workspace_bytes(const tsp_cfg* cfg, int32_t L, int32_t op) {
  if (L < 1) return 0;
  const size_t w = tsp_workspace_bytes(cfg, op);
  if (w == 0) return 0;
  if (op == TSP_OP_BLOCK_FWD) return up256(w) + 2 * act_bytes(cfg);   // + ping-pong layer outputs
  if (op == TSP_OP_BLOCK_BWD)                                         // + fp32 dx, dy in cfg dtype
    return up256(w) + up256((size_t)cfg->S * cfg->d * 4) + act_bytes(cfg);
  return 0;
}

tsp_status tsp_stack_fwd(const tsp_cfg* cfg, int32_t L, const void* x_z, const tsp_attn_w* aw,
                         const tsp_mlp_w* mw, void* y_z, void* saved, void* ws, size_t ws_bytes,
                         void* stream) {
  if (L < 1 || !aw || !mw || !al16(x_z) || !al16(y_z) || !al16(ws)) return TSP_ERR_INVALID_ARG;
  const size_t need = tsp_stack_workspace_bytes(cfg, L, TSP_OP_BLOCK_FWD);
  if (need == 0 || ws_bytes < need) return TSP_ERR_INVALID_ARG;
  if (saved && !al16(saved)) return TSP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t blk_ws = up256(tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD));
  const size_t nbytes = (size_t)cfg->S * cfg->d * elt_of(cfg);
  uint8_t* w = (uint8_t*)ws;
  tsp_status r = TSP_OK;
  if (saved) {
    // training: layer l's input sits at the head of its slot, so the backward
    // has every layer's input; each layer writes the next layer's input slot
    const size_t slot = layer_slot(cfg), ab = act_bytes(cfg);
    uint8_t* sv = (uint8_t*)saved;
    if (cudaMemcpyAsync(sv, x_z, nbytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return TSP_ERR_CUDA;
    for (int l = 0; l < L && r == TSP_OK; ++l) {
      uint8_t* in = sv + (size_t)l * slot;
      void* out = l == L - 1 ? y_z : (void*)(sv + (size_t)(l + 1) * slot);
      r = tsp_block_fwd(cfg, in, &aw[l], &mw[l], out, in + ab, w, blk_ws, stream);
    }
    return r;
  }
  uint8_t* buf[2] = {w + blk_ws, w + blk_ws + act_bytes(cfg)};
  for (int l = 0; l < L && r == TSP_OK; ++l) {
    const void* in = l == 0 ? x_z : buf[(l - 1) & 1];
    void* out = l == L - 1 ? y_z : buf[l & 1];
    r = tsp_block_fwd(cfg, in, &aw[l], &mw[l], out, nullptr, w, blk_ws, stream);
  }
  return r;
}

tsp_status tsp_stack_bwd(const tsp_cfg* cfg, int32_t L, const void* dy_z, const void* saved,
                         const tsp_attn_w* aw, const tsp_mlp_w* mw, float* dx_z,
                         float* const* grads, void* ws, size_t ws_bytes, void* stream) {
  if (L < 1 || !aw || !mw || !grads || !al16(dy_z) || !al16(saved) || !al16(dx_z) || !al16(ws))
    return TSP_ERR_INVALID_ARG;
  const size_t need = tsp_stack_workspace_bytes(cfg, L, TSP_OP_BLOCK_BWD);
  if (need == 0 || ws_bytes < need) return TSP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t blk_ws = up256(tsp_workspace_bytes(cfg, TSP_OP_BLOCK_BWD));
  const size_t slot = layer_slot(cfg), ab = act_bytes(cfg);
  const int64_t n = cfg->S * (int64_t)cfg->d;
  uint8_t* w = (uint8_t*)ws;
  float* dxbuf = (float*)(w + blk_ws);
  uint8_t* dybuf = w + blk_ws + up256((size_t)n * 4);
  const uint8_t* sv = (const uint8_t*)saved;
  for (int l = L - 1; l >= 0; --l) {
    const uint8_t* in = sv + (size_t)l * slot;
    const void* dy = l == L - 1 ? dy_z : (const void*)dybuf;
    float* dx = l == 0 ? dx_z : dxbuf;
    float* const* G = grads + 9 * (size_t)l;
    tsp_status r = tsp_block_bwd(cfg, in, dy, in + ab, &aw[l], &mw[l], dx, G[0], G[1], G[2], G[3],
                                 G[4], G[5], G[6], G[7], G[8], w, blk_ws, stream);
    if (r != TSP_OK) return r;
    if (l > 0) {
      // the gradient handed to the layer below is in the storage dtype, as
      // the block's dy input is
      if (cfg->dtype == TSP_BF16) {
        if ((r = launch_convert_f32_bf16(dxbuf, dybuf, n, st)) != TSP_OK) return r;
      } else if (cudaMemcpyAsync(dybuf, dxbuf, (size_t)n * 4, cudaMemcpyDeviceToDevice, st) !=
                 cudaSuccess) {
        return TSP_ERR_CUDA;
      }
    }
  }
  return TSP_OK;
}

tsp_status tsp_rank_memory(const tsp_cfg* cfg, int32_t L, int32_t training, int32_t scheme,
                           tsp_rank_mem* out) {
  if (!out || L < 1 || scheme < TSP_MEM_TSP || scheme > TSP_MEM_TP_SP) return TSP_ERR_INVALID_ARG;
  const size_t saved = tsp_saved_bytes(cfg);
  if (saved == 0) return TSP_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  const double D = cfg->D, S = (double)cfg->S, d = cfg->d, I = cfg->inter;
  const double e = (double)elt_of(cfg);
  // K/V width: Hkv heads of dh (Hkv = H without grouped-query attention)
  const double dkv = (cfg->Hkv > 0 ? (double)cfg->Hkv : (double)cfg->H) * cfg->dh;
  // weights of one layer: W_Q, W_O (d x d), W_K, W_V (dkv x d), W_1, W_3, W_2 and both gains
  const double W = ((2.0 * d * d + 2.0 * d * dkv + 3.0 * d * I) + 2.0 * d) * e;
  // activations one layer keeps per token for its backward: the block's
  // saved buffer plus the layer input (inference: the largest single layer's
  // forward workspace, which is all freed before the next layer)
  const double A_tok = training ? ((double)saved + (double)act_bytes(cfg)) / S
                                : (double)tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD) / S;
  const double A = (training ? L : 1) * A_tok * S;   // whole sequence
  double w_share = 1.0, a_share = 1.0;
  switch (scheme) {
    case TSP_MEM_TSP: w_share = 1.0 / D; a_share = 1.0 / D; out->devices = D; break;
    case TSP_MEM_DP: w_share = 1.0; a_share = 1.0; out->devices = D; break;   // D replicas
    case TSP_MEM_TP: w_share = 1.0 / D; a_share = 1.0; out->devices = D; break;
    case TSP_MEM_SP: w_share = 1.0; a_share = 1.0 / D; out->devices = D; break;
    case TSP_MEM_TP_SP: w_share = 1.0 / D; a_share = 1.0 / D; out->devices = D * D; break;
  }
  out->weights = L * W * w_share;
  out->activations = A * a_share;
  // the fold's transients (one layer at a time): one broadcast attention
  // shard plus the gathered K/V of the whole sequence, or one MLP ring shard
  if (scheme == TSP_MEM_TSP) {
    const double attn = (2.0 * d * d + 2.0 * d * dkv) / D * e + 2.0 * S * dkv * e;
    const double mlp = 3.0 * d * I / D * e;
    out->transient = attn > mlp ? attn : mlp;
  }
  out->total = out->weights + out->activations + out->transient;
  return TSP_OK;
}

}  // extern "C"
