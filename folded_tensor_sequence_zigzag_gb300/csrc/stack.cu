// stack.cu -- a stack of L TSP blocks (the multi-layer model the fold is
// applied to) and the per-virtual-rank memory account of the fold.
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), sections 1-3:
// every rank holds 1/D of the parameters and 1/D of the tokens of every
// layer, and the fold is the only layout of the compared ones that cuts both
// weight and activation memory by D without D^2 devices.  The stack here is
// the plain composition y = B_{L-1}(... B_0(x)); each block is the block
// forward / backward of tsp_block_fwd / tsp_block_bwd with its own weights, so
// every step still runs in the block's kernels.  The residual stream between
// layers stays in fp32, as it does inside a block (h): layer outputs and the
// gradient handed down to the layer below are fp32; only x and y (cfg dtype)
// and dx (fp32) are the stack's own input and outputs.
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace tsp {
namespace {

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }
size_t elt_of(const tsp_cfg* c) { return c->dtype == TSP_BF16 ? 2 : 4; }
// one layer's input or output between layers: the residual stream, kept in
// fp32 across the whole stack as it is inside the block (only the stack's own
// input x and output y are in the cfg dtype)
size_t stream_bytes(const tsp_cfg* c) { return up256((size_t)c->S * c->d * 4); }
bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

// per-layer slot of the training record: the layer's input, then the block's
// saved activations.  Layer 0's input is the caller's x (cfg dtype); the
// others are fp32.
size_t layer_slot(const tsp_cfg* c) { return stream_bytes(c) + up256(tsp_saved_bytes(c)); }

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
  const int base = op & ~TSP_OP_PREPARED;
  if (base != TSP_OP_BLOCK_FWD && base != TSP_OP_BLOCK_BWD) return 0;
  const size_t w = tsp_workspace_bytes(cfg, op);
  if (w == 0) return 0;
  // + two fp32 stream buffers: ping-pong layer outputs (forward) or the
  // gradient handed down between layers (backward)
  return up256(w) + 2 * stream_bytes(cfg);
}

}  // extern "C"

namespace tsp {
namespace {

// prep: nullable host array of L prepared weight buffers
tsp_status stack_fwd(const tsp_cfg* cfg, int32_t L, const void* x_z, const void* const* prep,
                     const tsp_attn_w* aw, const tsp_mlp_w* mw, void* y_z, void* saved, void* ws,
                     size_t ws_bytes, void* stream) {
  if (L < 1 || !aw || !mw || !al16(x_z) || !al16(y_z) || !al16(ws)) return TSP_ERR_INVALID_ARG;
  const int pf = prep ? TSP_OP_PREPARED : 0;
  const size_t need = tsp_stack_workspace_bytes(cfg, L, TSP_OP_BLOCK_FWD | pf);
  if (need == 0 || ws_bytes < need) return TSP_ERR_INVALID_ARG;
  if (saved && !al16(saved)) return TSP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t blk_ws = up256(tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD | pf));
  uint8_t* w = (uint8_t*)ws;
  tsp_status r = TSP_OK;
  if (saved) {
    // training: layer l's input sits at the head of its slot, so the backward
    // has every layer's input; each layer writes the next layer's input slot
    const size_t slot = layer_slot(cfg), sb = stream_bytes(cfg);
    const size_t xbytes = (size_t)cfg->S * cfg->d * elt_of(cfg);
    uint8_t* sv = (uint8_t*)saved;
    if (cudaMemcpyAsync(sv, x_z, xbytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return TSP_ERR_CUDA;
    for (int l = 0; l < L && r == TSP_OK; ++l) {
      uint8_t* in = sv + (size_t)l * slot;
      const bool last = l == L - 1;
      void* out = last ? y_z : (void*)(sv + (size_t)(l + 1) * slot);
      r = block_fwd_checked(cfg, in, l > 0, &aw[l], &mw[l], prep ? prep[l] : nullptr, out, !last,
                            in + sb, w, blk_ws, st);
    }
    return r;
  }
  uint8_t* buf[2] = {w + blk_ws, w + blk_ws + stream_bytes(cfg)};
  for (int l = 0; l < L && r == TSP_OK; ++l) {
    const bool last = l == L - 1;
    const void* in = l == 0 ? x_z : buf[(l - 1) & 1];
    void* out = last ? y_z : buf[l & 1];
    r = block_fwd_checked(cfg, in, l > 0, &aw[l], &mw[l], prep ? prep[l] : nullptr, out, !last,
                          nullptr, w, blk_ws, st);
  }
  return r;
}

tsp_status stack_bwd(const tsp_cfg* cfg, int32_t L, const void* dy_z, const void* saved,
                     const void* const* prep, const tsp_attn_w* aw, const tsp_mlp_w* mw,
                     float* dx_z, float* const* grads, void* ws, size_t ws_bytes, void* stream) {
  if (L < 1 || !aw || !mw || !grads || !al16(dy_z) || !al16(saved) || !al16(dx_z) || !al16(ws))
    return TSP_ERR_INVALID_ARG;
  const int pf = prep ? TSP_OP_PREPARED : 0;
  const size_t need = tsp_stack_workspace_bytes(cfg, L, TSP_OP_BLOCK_BWD | pf);
  if (need == 0 || ws_bytes < need) return TSP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t blk_ws = up256(tsp_workspace_bytes(cfg, TSP_OP_BLOCK_BWD | pf));
  const size_t slot = layer_slot(cfg), sb = stream_bytes(cfg);
  uint8_t* w = (uint8_t*)ws;
  // the gradient of layer l's input is the upstream gradient of layer l - 1:
  // fp32, ping-ponged between two buffers
  float* gbuf[2] = {(float*)(w + blk_ws), (float*)(w + blk_ws + sb)};
  const uint8_t* sv = (const uint8_t*)saved;
  for (int l = L - 1; l >= 0; --l) {
    const uint8_t* in = sv + (size_t)l * slot;
    const bool top = l == L - 1;
    const void* dy = top ? dy_z : (const void*)gbuf[(l + 1) & 1];
    float* dx = l == 0 ? dx_z : gbuf[l & 1];
    tsp_status r = block_bwd_checked(cfg, in, l > 0, dy, !top, in + sb, &aw[l], &mw[l],
                                     prep ? prep[l] : nullptr, dx, grads + 9 * (size_t)l, w,
                                     blk_ws, st);
    if (r != TSP_OK) return r;
  }
  return TSP_OK;
}

}  // namespace
}  // namespace tsp

extern "C" {

tsp_status tsp_stack_fwd(const tsp_cfg* cfg, int32_t L, const void* x_z, const tsp_attn_w* aw,
                         const tsp_mlp_w* mw, void* y_z, void* saved, void* ws, size_t ws_bytes,
                         void* stream) {
  return stack_fwd(cfg, L, x_z, nullptr, aw, mw, y_z, saved, ws, ws_bytes, stream);
}

tsp_status tsp_stack_fwd_prepared(const tsp_cfg* cfg, int32_t L, const void* x_z,
                                  const void* const* prep, const tsp_attn_w* aw,
                                  const tsp_mlp_w* mw, void* y_z, void* saved, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!prep) return TSP_ERR_INVALID_ARG;
  return stack_fwd(cfg, L, x_z, prep, aw, mw, y_z, saved, ws, ws_bytes, stream);
}

tsp_status tsp_stack_bwd(const tsp_cfg* cfg, int32_t L, const void* dy_z, const void* saved,
                         const tsp_attn_w* aw, const tsp_mlp_w* mw, float* dx_z,
                         float* const* grads, void* ws, size_t ws_bytes, void* stream) {
  return stack_bwd(cfg, L, dy_z, saved, nullptr, aw, mw, dx_z, grads, ws, ws_bytes, stream);
}

tsp_status tsp_stack_bwd_prepared(const tsp_cfg* cfg, int32_t L, const void* dy_z,
                                  const void* saved, const void* const* prep,
                                  const tsp_attn_w* aw, const tsp_mlp_w* mw, float* dx_z,
                                  float* const* grads, void* ws, size_t ws_bytes, void* stream) {
  if (!prep) return TSP_ERR_INVALID_ARG;
  return stack_bwd(cfg, L, dy_z, saved, prep, aw, mw, dx_z, grads, ws, ws_bytes, stream);
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
  // saved buffer plus the layer input, a slot of the fp32 residual stream
  // (inference: the largest single layer's forward workspace, which is all
  // freed before the next layer)
  const double A_tok = training ? ((double)saved + (double)stream_bytes(cfg)) / S
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
