/*
 * tsp.h -- C ABI of the TSP-folded transformer block for one GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * Source page: "Folding Tensor and Sequence Parallelism for Memory-Efficient
 * Transformer Training & Inference" (gist.science summary), section 2
 * ("Methodology: TSP").  Under TSP every one of D ranks holds 1/D of the
 * parameters and 1/D of the tokens ("Unified sharding").  Attention layers
 * walk the packed W_Q/W_K/W_V/W_O shards (one rank broadcasts its shard per
 * step), project every rank's own tokens, all-gather K/V over the sequence
 * and run FlashAttention on zigzag-partitioned causal rows ("Runtime
 * schedules", attention bullet).  Gated-MLP layers rotate W_1/W_2/W_3 shards
 * around a ring; every rank accumulates its partial outputs locally, so no
 * all-reduce is needed ("Runtime schedules", gated-MLP bullet).
 *
 * Here the D ranks are VIRTUAL ranks on one GPU: rank r's tokens are rows
 * [r*2c, (r+1)*2c) of one rank-major "zigzag" buffer, the gathered K/V is the
 * same buffer, and a weight shard is a column range of the unsharded weight.
 * The block is pre-norm:
 *     a = rms(x; g_attn),  Q|K|V = a [W_Q|W_K|W_V]^T,  O = causal MHA(Q,K,V),
 *     h = x + O W_O^T,     b = rms(h; g_mlp),
 *     y = h + (silu(b W_1^T) * (b W_3^T)) W_2^T
 * with rms(u; g) = u / sqrt(mean(u^2) + eps) * g, scale 1/sqrt(dh), causal
 * mask j <= i with the diagonal included, no biases, no positional encoding.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers unless a comment says otherwise; the caller
 *    allocates and owns every buffer.  The library never allocates device
 *    memory: scratch comes from the caller's workspace (tsp_workspace_bytes).
 *  - Matrices are row-major.  Weights use the nn.Linear convention
 *    [out, in]: W_Q, W_K, W_V, W_O are [d, d]; W_1, W_3 are [inter, d];
 *    W_2 is [d, inter]; gains are [d].
 *  - Activations (x_z, h_z, y_z, dy_z, dx_z) are in zigzag rank-major order:
 *    [D][2][c][d] with c = S/(2D); rank r's slot 0 holds global chunk r and
 *    slot 1 holds chunk 2D-1-r, positions ascending inside a chunk.
 *    tsp_zigzag_permute converts from/to global token order.
 *  - dtype TSP_BF16: activations, weights and gains are bf16; accumulation,
 *    softmax and norms run in fp32.  TSP_F32: everything fp32 (exact fp32
 *    SIMT path, meant for small shapes).  Weight/gain gradients are always
 *    fp32 and are OVERWRITTEN (not accumulated into).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous on that stream; outputs are ready when the stream
 *    reaches the call.
 *  - Errors a host can detect (bad sizes, NULL or misaligned pointers, short
 *    workspace, shapes the bf16 kernels do not take) are returned at once and
 *    nothing is launched.  Launch failures return TSP_ERR_CUDA.  Errors the
 *    device detects set a sticky device status word read by
 *    tsp_device_status; kernels never trap.  They are: a pipeline wait that
 *    exceeded its time limit (TSP_ERR_TIMEOUT), and, in the bf16
 *    configuration, a value that the tensor-core path holds in fp16 -- the
 *    weights, the normalised activations, Q/K/V, G, the SwiGLU
 *    pre-activations, the upstream gradient and the backward's fp16
 *    operands -- that is not finite or too large for fp16 (|v| >= 65520,
 *    which fp16 rounds to infinity): TSP_ERR_RANGE.  The result of such a
 *    call is not valid.  (Magnitudes below 6.1e-5 are kept as fp16
 *    subnormals with fewer significant bits; that is not reported.)  The
 *    checked build (libtsp_check.so, compiled with TSP_CHECK) also tests the
 *    global indices the kernels compute -- zigzag rows, shard and segment
 *    indices, tile rows, cache rows, partial slots -- before each access and
 *    skips an access that fails, recording TSP_ERR_BOUNDS; the normal build
 *    carries none of these tests.
 *    While the word holds an error, the tensor-core kernels return without
 *    doing their work, until tsp_device_status(stream, 1) clears it.
 *  - All pointers must be 16-byte aligned; row strides are dense.
 */
#ifndef TSP_H_
#define TSP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TSP_OK = 0,
  TSP_ERR_INVALID_ARG = 1,   /* bad size, NULL or misaligned pointer, short buffer */
  TSP_ERR_UNSUPPORTED = 2,   /* valid shape that the selected kernels do not take */
  TSP_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed               */
  TSP_ERR_TIMEOUT = 4,       /* a device pipeline wait exceeded its time limit     */
  TSP_ERR_RANGE = 5,         /* a value the bf16 path holds in fp16 was out of fp16 range */
  TSP_ERR_BOUNDS = 6         /* checked build only: a computed index failed its bounds check */
} tsp_status;

typedef enum { TSP_F32 = 0, TSP_BF16 = 1 } tsp_dtype;

/* Block configuration.  Causal attention always.
 *   S      tokens (multiple of 2D)
 *   d      d_model;  H heads;  dh = d / H (must equal d / H)
 *   inter  SwiGLU intermediate size
 *   D      virtual ranks, 1..64
 *   eps    RMSNorm epsilon
 *   dtype  tsp_dtype
 * bf16 kernels additionally need: d % 256 == 0, inter % 128 == 0, and for
 * attention dh == 128 and c = S/(2D) a multiple of 256.  Other valid shapes
 * return TSP_ERR_UNSUPPORTED in bf16 (there is no silent fallback). */
typedef struct {
  int64_t S;
  int32_t d, H, dh, inter, D;
  float eps;
  int32_t dtype;
  /* Rotary position embedding of Q and K (not on the pages; a variant):
   * 0 = none (the pages' block); > 0 = the rotate-half rotation with
   * frequencies rope_base^(-2j/dh), j < dh/2, at each token's global
   * position (the zigzag layout only moves rows).  Needs an even dh. */
  float rope_base;
  /* K/V heads (grouped-query attention, a variant; not on the pages):
   * 0 or H = multi-head attention; otherwise a divisor of H, and the H/Hkv
   * query heads h = g*(H/Hkv) .. (g+1)*(H/Hkv)-1 share K/V head g.  W_K and
   * W_V are then [Hkv*dh, d].  The bf16 kernels need Hkv*dh % 256 == 0. */
  int32_t Hkv;
  /* Sequence tiling of the gated MLP in the training step (TiledMLP-style;
   * a variant, not on the pages): 0 = off; otherwise the rows per tile, a
   * multiple of 128 that divides the 2c rows of a virtual rank.  The
   * training forward then runs the MLP one tile at a time and keeps neither
   * G nor the pre-activations for the backward, which recomputes them tile
   * by tile from the saved normalised input, so the MLP's [S, inter]-sized
   * buffers shrink to [tile, inter].  bf16 only (TSP_ERR_UNSUPPORTED for
   * fp32). */
  int32_t mlp_tile;
} tsp_cfg;

/* Attention-half weights: wq, wo [d, d]; wk, wv [Hkv*dh, d] ([d, d] for
 * multi-head attention); g_attn [d]. */
typedef struct {
  const void *wq, *wk, *wv, *wo, *g_attn;
} tsp_attn_w;

/* Gated-MLP weights: w1, w3 [inter, d]; w2 [d, inter]; g_mlp [d] or NULL
 * (NULL: no RMSNorm, b = h).  add_residual: 1 -> y = h + MLP(b), 0 -> y = MLP(b). */
typedef struct {
  const void *w1, *w3, *w2, *g_mlp;
  int32_t add_residual;
} tsp_mlp_w;

/* Workspace queries (op selects the entry point).  TSP_OP_BLOCK_FWD_TRAIN:
 * the block forward with a `saved` buffer (activations go there; the
 * workspace holds the weight copies and, with mlp_tile, one MLP tile).
 * OR TSP_OP_PREPARED into TSP_OP_BLOCK_FWD, TSP_OP_BLOCK_BWD or
 * TSP_OP_BLOCK_FWD_TRAIN for the _prepared entry points, whose workspace
 * holds no weight copies (other ops with the flag: 0). */
enum { TSP_OP_ATTN_FWD = 0, TSP_OP_MLP_FWD = 1, TSP_OP_BLOCK_FWD = 2, TSP_OP_BLOCK_BWD = 3,
       TSP_OP_BLOCK_FWD_TRAIN = 4, TSP_OP_PREPARED = 16 };

/* Zigzag causal partitioning (section 2, attention bullet: "zigzag
 * partitioning balances the causal attention work").  Bit-exact row copy.
 *   inverse = 0: src in global order [S][row_bytes] -> dst zigzag rank-major;
 *   inverse = 1: zigzag rank-major -> global order.
 * row_bytes: bytes per token row (e.g. d * sizeof(element)); any value > 0,
 * multiples of 16 take the vectorised path.  src and dst must not overlap.
 * Errors: TSP_ERR_INVALID_ARG if S <= 0, D not in 1..64, S % (2D) != 0,
 * row_bytes <= 0 or a NULL pointer. */
tsp_status tsp_zigzag_permute(const void* src, void* dst, int64_t S, int32_t D,
                              int64_t row_bytes, int32_t inverse, void* stream);

/* Row-wise RMSNorm (pre-norm of both halves of the block; the pages give no
 * formula, the plain reading is the one above).  u, out: [rows, n] of the
 * cfg dtype; g: [n] of the cfg dtype; rstd (nullable): [rows] fp32 receives
 * 1/sqrt(mean(u^2)+eps).  dtype: tsp_dtype. */
tsp_status tsp_rmsnorm_fwd(const void* u, const void* g, void* out, float* rstd,
                           int64_t rows, int32_t n, float eps, int32_t dtype, void* stream);

/* Bytes of caller workspace an entry point needs for cfg (0 if cfg invalid). */
size_t tsp_workspace_bytes(const tsp_cfg* cfg, int32_t op);

/* Bytes of the activation buffer tsp_block_fwd fills for tsp_block_bwd. */
size_t tsp_saved_bytes(const tsp_cfg* cfg);

/* Attention half of the block (section 2, attention bullet): for shard
 * k = 0..D-1 every virtual rank projects its rows with the W_Q/W_K/W_V
 * columns of shard k; K/V of all ranks form the gathered context; each rank's
 * zigzag rows attend causally to it; each rank accumulates O[:,C_k] W_O[:,C_k]^T
 * over k in fp32 onto its residual rows:  h_z = x_z + Attn(rms(x_z)) W_O^T.
 * x_z, h_z: [S, d] zigzag.  ws: tsp_workspace_bytes(cfg, TSP_OP_ATTN_FWD). */
tsp_status tsp_attn_block_fwd(const tsp_cfg* cfg, const void* x_z, const tsp_attn_w* w,
                              void* h_z, void* ws, size_t ws_bytes, void* stream);

/* Gated-MLP half (section 2, gated-MLP bullet): shard I_k of W_1/W_3 (rows)
 * and W_2 (columns); virtual rank r takes shard (r - t) mod D at ring step t
 * and accumulates G[:,I_k] W_2[:,I_k]^T in fp32 on its own rows.
 *   y_z = [h_z +] (silu(b W_1^T) * (b W_3^T)) W_2^T, b = rms(h_z; g_mlp) or h_z.
 * h_z, y_z: [S, d] zigzag.  ws: tsp_workspace_bytes(cfg, TSP_OP_MLP_FWD). */
tsp_status tsp_gated_mlp_fwd(const tsp_cfg* cfg, const void* h_z, const tsp_mlp_w* w,
                             void* y_z, void* ws, size_t ws_bytes, void* stream);

/* Size of the device scratch that tsp_gated_mlp_fwd_noalloc works in: 32 MiB.
 * Every GPU that loads this library holds it until the process exits. */
#define TSP_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Gated-MLP half without a caller workspace.  The pages have no counterpart
 * for this entry point: it exists for callers that cannot allocate device
 * memory at the point of the call -- for example a plugin whose execute hook
 * runs inside an inference engine that has already planned every byte of
 * device memory (an extra allocation could fail or break that plan), or a
 * latency-critical loop that cannot afford the device-wide synchronisation a
 * cudaMalloc/cudaFree may imply.  It computes exactly what tsp_gated_mlp_fwd
 * computes, with the same arguments minus (ws, ws_bytes); its scratch (the
 * normalised input, G, and the fp16 weight copies) lives in one fixed
 * TSP_NOALLOC_SCRATCH_BYTES array compiled into the library.  It allocates
 * nothing.
 *  - Limit: if tsp_workspace_bytes(cfg, TSP_OP_MLP_FWD) exceeds
 *    TSP_NOALLOC_SCRATCH_BYTES it returns TSP_ERR_INVALID_ARG and launches
 *    nothing (other argument errors as for tsp_gated_mlp_fwd).
 *  - The first call on a device looks up the array's device address with that
 *    device current (cudaGetSymbolAddress; TSP_ERR_CUDA if that fails).  Make
 *    that first call before any stream capture.
 *  - Every call shares the one array, which keeps the previous call's
 *    contents; no part of it needs to start at zero (each call writes every
 *    byte it reads).  Calls that overlap on the GPU (other streams, other host
 *    threads) race on it: order them on one stream or synchronise them. */
tsp_status tsp_gated_mlp_fwd_noalloc(const tsp_cfg* cfg, const void* h_z, const tsp_mlp_w* w,
                                     void* y_z, void* stream);

/* Whole block forward: y_z = MLP-half(Attention-half(x_z)).  mlp_w->g_mlp
 * must be non-NULL and add_residual 1 (pre-norm block).  saved (nullable):
 * tsp_saved_bytes(cfg) bytes that receive the activations tsp_block_bwd
 * needs; NULL for inference.  ws: tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD)
 * for inference, tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD_TRAIN) (or more)
 * with `saved`. */
tsp_status tsp_block_fwd(const tsp_cfg* cfg, const void* x_z, const tsp_attn_w* aw,
                         const tsp_mlp_w* mw, void* y_z, void* saved,
                         void* ws, size_t ws_bytes, void* stream);

/* Whole block backward of L = sum(dy * y).  Inputs: x_z and dy_z ([S, d]
 * zigzag, cfg dtype), saved (filled by tsp_block_fwd with the same cfg,
 * weights and x_z).  Outputs, all fp32: dx_z ([S, d] zigzag -- the gradient
 * of the residual stream, kept in fp32 like the stream itself: at early
 * positions, which every later query attends, it reaches ~10x its RMS, where
 * a bf16 result would lose more than the bf16 path's error budget to its own
 * rounding) and the gradients dwq, dwo [d, d], dwk, dwv [Hkv*dh, d], dw1, dw3 [inter, d],
 * dw2 [d, inter], dg_attn, dg_mlp [d] -- each the sum over the D virtual
 * ranks' token rows (the reduction TSP performs toward the shard owners).
 * ws: tsp_workspace_bytes(cfg, TSP_OP_BLOCK_BWD). */
tsp_status tsp_block_bwd(const tsp_cfg* cfg, const void* x_z, const void* dy_z,
                         const void* saved, const tsp_attn_w* aw, const tsp_mlp_w* mw,
                         float* dx_z, float* dwq, float* dwk, float* dwv, float* dwo,
                         float* dw1, float* dw3, float* dw2, float* dg_attn, float* dg_mlp,
                         void* ws, size_t ws_bytes, void* stream);

/* ---- Weights converted once (not on the pages: an implementation choice) ----
 * The bf16 path's tensor-core operands are fp16 (10-bit mantissa), so every
 * whole-block call first converts the bf16 weight matrices it reads into fp16
 * copies in its workspace (4 bytes of traffic per weight element, every
 * call).  A caller whose weights stay the same across calls -- inference, or
 * the forward and backward of one training step between two optimizer
 * updates -- converts them once into a buffer it owns and passes that
 * instead.
 * tsp_block_weights_bytes: bytes of one block's fp16 copies (W_Q, W_K, W_V,
 *   W_O, W_1, W_3, W_2, 256-byte aligned pieces); 0 for TSP_F32 (which reads
 *   the weights as they are) or an invalid cfg.
 * tsp_block_weights_prepare: writes them into prep (16-byte aligned, that
 *   many bytes).  A weight that fp16 cannot hold sets TSP_ERR_RANGE in the
 *   device status word.  The copies are valid until the caller changes the
 *   weights; they are not tracked.  TSP_F32: nothing to do, TSP_OK.
 * tsp_block_fwd_prepared / tsp_block_bwd_prepared: tsp_block_fwd /
 *   tsp_block_bwd reading the weight matrices from prep (bf16: required; the
 *   matrix pointers in aw, mw may then be NULL, the gains and add_residual
 *   are still read from them; TSP_F32: prep is ignored).  Workspace:
 *   tsp_workspace_bytes(cfg, op | TSP_OP_PREPARED). */
size_t tsp_block_weights_bytes(const tsp_cfg* cfg);
tsp_status tsp_block_weights_prepare(const tsp_cfg* cfg, const tsp_attn_w* aw, const tsp_mlp_w* mw,
                                     void* prep, void* stream);
tsp_status tsp_block_fwd_prepared(const tsp_cfg* cfg, const void* x_z, const void* prep,
                                  const tsp_attn_w* aw, const tsp_mlp_w* mw, void* y_z, void* saved,
                                  void* ws, size_t ws_bytes, void* stream);
tsp_status tsp_block_bwd_prepared(const tsp_cfg* cfg, const void* x_z, const void* dy_z,
                                  const void* saved, const void* prep, const tsp_attn_w* aw,
                                  const tsp_mlp_w* mw, float* dx_z, float* dwq, float* dwk,
                                  float* dwv, float* dwo, float* dw1, float* dw3, float* dw2,
                                  float* dg_attn, float* dg_mlp, void* ws, size_t ws_bytes,
                                  void* stream);

/* ---- Inference: prefill, then decode against the zigzag KV cache ----
 * (section 2, attention bullet: each rank holds the K/V of its own zigzag
 * rows; the pages' title names inference, their schedules describe the
 * full-sequence pass, which is the prefill.)
 *
 * KV cache: kv_rows_cap rows of [K (Hkv*dh) | V (Hkv*dh)], row-major, in the
 * internal element type (fp16 for TSP_BF16, fp32 for TSP_F32), K after the
 * rotary embedding when cfg->rope_base > 0.  Rows [0, S) hold the prompt in
 * zigzag row order (row i is the token at global position zz_pos(i); virtual
 * rank r owns rows [r*2c, (r+1)*2c), c = S/(2D)); rows [S, n) hold decoded
 * tokens, row = position.  The caller owns it.
 *
 * tsp_kv_cache_bytes: bytes of a cache of kv_rows_cap rows (0 if invalid).
 * tsp_block_prefill: tsp_block_fwd(x_z -> y_z, inference) over the S prompt
 *   tokens, then their K and V into cache rows [0, S).  ws as for
 *   tsp_block_fwd (tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD)).
 * tsp_block_decode: T (1..TSP_DECODE_MAX_T) new tokens at positions
 *   n_cached .. n_cached+T-1, where n_cached (S <= n_cached <=
 *   kv_rows_cap - T) rows are already in the cache.  x, y: [T, d] in
 *   position order (cfg dtype).  Appends the new tokens' K/V at rows
 *   n_cached.., then each new token attends to every cached row at or
 *   before its position: per virtual rank over the zigzag rows it owns,
 *   merged by log-sum-exp.  y equals rows n_cached.. of the block forward
 *   over the whole sequence.  Reads the weights directly (no converted
 *   copies).  ws: tsp_decode_workspace_bytes(cfg, T, kv_rows_cap).
 * Errors: TSP_ERR_INVALID_ARG for NULL/misaligned pointers, T out of range,
 *   n_cached out of range, a short workspace or cache; TSP_ERR_UNSUPPORTED
 *   for shapes the decode kernels do not take (head width dh other than 64
 *   or 128 in bf16, or 16, 32 or 64 in fp32; d or inter not a multiple of 8
 *   (bf16) / 4 (fp32); T * max(d, inter) elements above 200 KB of shared
 *   memory). */
#define TSP_DECODE_MAX_T 8
size_t tsp_kv_cache_bytes(const tsp_cfg* cfg, int64_t kv_rows_cap);
size_t tsp_decode_workspace_bytes(const tsp_cfg* cfg, int32_t T, int64_t kv_rows_cap);
tsp_status tsp_block_prefill(const tsp_cfg* cfg, const void* x_z, const tsp_attn_w* aw,
                             const tsp_mlp_w* mw, void* y_z, void* kv, int64_t kv_rows_cap,
                             void* ws, size_t ws_bytes, void* stream);
tsp_status tsp_block_decode(const tsp_cfg* cfg, const void* x, int32_t T, int64_t n_cached,
                            const tsp_attn_w* aw, const tsp_mlp_w* mw, void* y, void* kv,
                            int64_t kv_rows_cap, void* ws, size_t ws_bytes, void* stream);

/* ---- Stack of L blocks (the multi-layer model the fold is applied to) ----
 * y = B_{L-1}(... B_0(x)), B_l = the block above with weights aw[l], mw[l];
 * every layer runs the block's forward / backward, so the kernels are the
 * block's.  The residual stream between layers stays in fp32, as it does
 * inside a block: each layer's output, and in the backward the gradient each
 * layer hands to the one below, are fp32 (no rounding to the cfg dtype
 * between layers).  aw, mw: host arrays of L weight sets (each as for
 * tsp_block_fwd).
 *
 * tsp_stack_saved_bytes: training record of L layers (each layer's input,
 *   in an fp32-sized slot, plus its block's saved activations); 0 if cfg is
 *   invalid or L < 1.
 * tsp_stack_workspace_bytes: op = TSP_OP_BLOCK_FWD (forward, with or without
 *   the training record) or TSP_OP_BLOCK_BWD; 0 if invalid.
 * tsp_stack_fwd: x_z, y_z [S, d] zigzag (cfg dtype); saved = NULL for
 *   inference or tsp_stack_saved_bytes(cfg, L) bytes for training.
 * tsp_stack_bwd: backward of L = sum(dy * y) through the stack.  dy_z [S, d]
 *   (cfg dtype), saved as filled by tsp_stack_fwd, dx_z [S, d] fp32 out.
 *   grads: host array of 9*L fp32 device pointers, layer l at 9*l in the
 *   order dwq, dwk, dwv, dwo, dw1, dw3, dw2, dg_attn, dg_mlp (each sized as
 *   for tsp_block_bwd, overwritten).  The gradient between layers is fp32.
 * Errors: TSP_ERR_INVALID_ARG for L < 1, NULL or misaligned pointers or a
 *   short workspace; otherwise as for the block calls, stopping at the first
 *   failing layer. */
size_t tsp_stack_saved_bytes(const tsp_cfg* cfg, int32_t L);
size_t tsp_stack_workspace_bytes(const tsp_cfg* cfg, int32_t L, int32_t op);
tsp_status tsp_stack_fwd(const tsp_cfg* cfg, int32_t L, const void* x_z, const tsp_attn_w* aw,
                         const tsp_mlp_w* mw, void* y_z, void* saved, void* ws,
                         size_t ws_bytes, void* stream);
tsp_status tsp_stack_bwd(const tsp_cfg* cfg, int32_t L, const void* dy_z, const void* saved,
                         const tsp_attn_w* aw, const tsp_mlp_w* mw, float* dx_z,
                         float* const* grads, void* ws, size_t ws_bytes, void* stream);
/* The same with every layer's weights converted once (see
 * tsp_block_weights_prepare): prep is a host array of L device pointers,
 * layer l's fp16 copies at prep[l].  Workspace: tsp_stack_workspace_bytes(cfg,
 * L, op | TSP_OP_PREPARED). */
tsp_status tsp_stack_fwd_prepared(const tsp_cfg* cfg, int32_t L, const void* x_z,
                                  const void* const* prep, const tsp_attn_w* aw,
                                  const tsp_mlp_w* mw, void* y_z, void* saved, void* ws,
                                  size_t ws_bytes, void* stream);
tsp_status tsp_stack_bwd_prepared(const tsp_cfg* cfg, int32_t L, const void* dy_z,
                                  const void* saved, const void* const* prep,
                                  const tsp_attn_w* aw, const tsp_mlp_w* mw, float* dx_z,
                                  float* const* grads, void* ws, size_t ws_bytes, void* stream);

/* ---- Per-rank memory account (sections 1-3: the fold cuts both weight and
 * activation memory per rank by D; TP cuts only weights, SP only
 * activations, TP+SP both but on D^2 devices, DP neither).  Bytes one rank
 * holds for an L-layer stack of cfg's block at cfg->S tokens and degree
 * cfg->D:
 *   weights      L layers' parameters (cfg dtype) times the scheme's share;
 *   activations  training: L x (block saved buffer + layer input), i.e. the
 *                tsp_stack_saved_bytes record, times the scheme's token
 *                share; inference: one layer's forward workspace;
 *   transient    TSP only: the larger of one broadcast attention shard plus
 *                the gathered K and V of all S tokens, and one MLP ring shard;
 *   devices      devices the scheme occupies (D, or D*D for TP+SP).
 * Shares come from the same buffer plan the kernels use.  Host-only; no GPU. */
enum { TSP_MEM_TSP = 0, TSP_MEM_DP = 1, TSP_MEM_TP = 2, TSP_MEM_SP = 3, TSP_MEM_TP_SP = 4 };
typedef struct {
  double weights, activations, transient, total, devices;
} tsp_rank_mem;
tsp_status tsp_rank_memory(const tsp_cfg* cfg, int32_t L, int32_t training, int32_t scheme,
                           tsp_rank_mem* out);

/* Packed shard layout, what one broadcast step of the attention schedule
 * carries ("packed W_Q, W_K, W_V, W_O"): for shard k (columns C_k of width
 * d/D, boundaries floor(k*d/D)) writes [W_Q[C_k,:]; W_K[C_k,:]; W_V[C_k,:];
 * W_O[:,C_k]^T] as a [4*|C_k|, d] block; shards follow each other in dst.
 * Elements of the cfg dtype; dst holds 4*d*d elements.  The forward kernels
 * read the unsharded weights directly and do not need this.  Multi-head
 * attention only (TSP_ERR_UNSUPPORTED with grouped K/V heads). */
tsp_status tsp_pack_attn_shards(const tsp_cfg* cfg, const tsp_attn_w* w, void* dst, void* stream);

/* Packed MLP shards, what one step of the ring schedule hands on (section 2,
 * gated-MLP bullet: W_1, W_2, W_3 shards rotate around the ranks): shard k
 * (rows I_k of W_1 and W_3, boundaries floor(k*inter/D)) is written as
 * [W_1[I_k,:]; W_3[I_k,:]; W_2[:,I_k]^T], a [3*|I_k|, d] block; shards
 * follow each other in dst (3*inter*d elements of the cfg dtype). */
tsp_status tsp_pack_mlp_shards(const tsp_cfg* cfg, const tsp_mlp_w* w, void* dst, void* stream);

/* ---- One rank's steps of the forward schedule (section 2, "Runtime
 * schedules") ----
 * Where the other entry points run all D ranks at once on one GPU, these
 * compute what one rank r computes between two exchanges of the schedule,
 * from the data that rank holds; the caller moves the data between ranks.
 * A forward of the block is, for every rank r:
 *   for k = 0..D-1 (attention shard k broadcast by its owner):
 *     tsp_rank_attn_project(r, k, x_r, g_attn, shard_k, kv_k[r])
 *     all-gather: kv_all_k = kv_k[0] ; kv_k[1] ; ... ; kv_k[D-1] (rows stacked)
 *     tsp_rank_attn_heads(r, k, x_r, kv_all_k, h_r)
 *   for t = 0..D-1 (MLP shard (r - t) mod D received from rank r - 1):
 *     tsp_rank_mlp_step(r, t, h_r, g_mlp, mlp_shard_{(r-t) mod D}, y_r, y_out_r)
 * Shards are head-aligned (D divides H), so broadcast step k carries whole
 * heads and its attention needs only that shard's K/V: every shard's weights
 * are used once, while they are held.
 * Buffers (rows = 2c = S/D, rank r's zigzag rows, chunk r then chunk 2D-1-r):
 *   x_r      [2c, d] cfg dtype: the rank's input rows;
 *   shard_k  [4*|C_k|, d] cfg dtype: block k of tsp_pack_attn_shards;
 *   kv_k     [2c, 2*|C_k|] fp16: the rank's K | V of shard k's heads (out);
 *   kv_all_k [S, 2*|C_k|] fp16: every rank's kv_k, rank q's at rows q*2c;
 *   h_r      [2c, d] fp32: residual stream after the attention half
 *            (written at k = 0 as x_r + ..., accumulated at k > 0);
 *   mlp shard [3*|I_s|, d] cfg dtype: block s of tsp_pack_mlp_shards;
 *   y_r      [2c, d] fp32: MLP accumulator (t = 0 starts from h_r);
 *   y_out_r  [2c, d] cfg dtype (nullable): at t = D-1 the block output goes
 *            here instead of y_r;
 *   ws       tsp_rank_workspace_bytes(cfg) bytes, one per rank, passed to
 *            all of that rank's calls of the layer in the order above (it
 *            keeps the normalised rows, the received shard and Q between
 *            calls; at short sequences, where a rank's 256-row blocks would
 *            fill too few SMs, it also holds the attention's per-chunk
 *            partial outputs: the key range is split into chunks whose
 *            results are merged by their log-sum-exp).
 * Shapes: TSP_BF16, multi-head attention without rotary embedding, dh = 128,
 * D divides H with H/D >= 2, c a multiple of 256, d a multiple of 256,
 * inter a multiple of 32*D; otherwise TSP_ERR_UNSUPPORTED (and
 * tsp_rank_workspace_bytes returns 0).  Errors as for the block calls. */
size_t tsp_rank_workspace_bytes(const tsp_cfg* cfg);
tsp_status tsp_rank_attn_project(const tsp_cfg* cfg, int32_t r, int32_t k, const void* x_r,
                                 const void* g_attn, const void* shard_k, void* kv_k, void* ws,
                                 size_t ws_bytes, void* stream);
tsp_status tsp_rank_attn_heads(const tsp_cfg* cfg, int32_t r, int32_t k, const void* x_r,
                               const void* kv_all_k, float* h_r, void* ws, size_t ws_bytes,
                               void* stream);
tsp_status tsp_rank_mlp_step(const tsp_cfg* cfg, int32_t r, int32_t t, const float* h_r,
                             const void* g_mlp, const void* shard, float* y_r, void* y_out,
                             void* ws, size_t ws_bytes, void* stream);

/* ---- The backward of the per-rank schedule ----------------------------------
 * The pages describe the forward only; the backward moves the same shards in
 * reverse (same page, section 2, read as follows).  Per block, after the
 * forward calls above ran for rank r with the same `ws`:
 *
 *   for t = 0 .. D-1:   (the ring again; the shard's gradient travels with it)
 *     tsp_rank_mlp_bwd_step(r, t, h_r, g_mlp, mlp_shard_{(r-t) mod D}, dy_r, grad, db_r)
 *     pass (shard, grad) to rank r+1       (D passes: the last one home)
 *   tsp_rank_mlp_bwd_finish(r, h_r, g_mlp, db_r, dy_r -> dh_r, dg_mlp part)
 *   for k = 0 .. D-1:   (the attention shards broadcast again)
 *     tsp_rank_attn_project(r, k, x_r, g_attn, attn_shard_k -> kv_k)   (as forward)
 *     all-gather kv_k -> kv_all_k
 *     tsp_rank_attn_bwd_heads(r, k, kv_all_k -> grad_k[W_O part], dkv_k)
 *     reduce-scatter the ranks' dkv_k -> dkv_own_r (own rows, summed)
 *     tsp_rank_attn_bwd_weights(r, k, dkv_own_r -> grad_k[Q|K|V parts], da_r)
 *     reduce grad_k to its owner, rank k
 *   tsp_rank_attn_bwd_finish(r, x_r, g_attn, da_r, dh_r -> dx_r, dg_attn part)
 *   all-reduce the gain gradients
 *
 * Shapes and layouts (rows = 2c, Ck / Is the shard widths, fp32 unless noted):
 *   dy_r [rows, d] bf16;  db_r, dh_r, da_r, dx_r [rows, d];
 *   grad (MLP shard gradient, packed like the shard) [3*Is, d]: rows 0..Is-1
 *     dW_1[I_s], then dW_3[I_s], then dW_2[:, I_s]^T; ACCUMULATED into (the
 *     first holder's buffer must be zero);  db_r written at t = 0, then
 *     accumulated;
 *   grad_k (attention shard gradient, packed like the shard) [4*Ck, d]:
 *     dW_Q[C_k], dW_K[C_k], dW_V[C_k], dW_O[:, C_k]^T, this rank's rows' part,
 *     OVERWRITTEN (the W_O part by ..._heads, the rest by ..._weights);
 *   dkv_k [S, 2*Ck] fp16, zigzag row order: dK | dV of every key from this
 *     rank's queries (zero where none reaches);  dkv_own_r [rows, 2*Ck]
 *     fp16: the sum over all ranks of their dkv_k at rank r's rows;
 *   da_r written at k = 0, then accumulated;  dg_mlp, dg_attn [d]: this
 *     rank's part (sum over ranks for the gain gradient).
 * Errors as for the forward per-rank calls. */
tsp_status tsp_rank_mlp_bwd_step(const tsp_cfg* cfg, int32_t r, int32_t t, const float* h_r,
                                 const void* g_mlp, const void* shard, const void* dy_r,
                                 float* grad, float* db_r, void* ws, size_t ws_bytes,
                                 void* stream);
tsp_status tsp_rank_mlp_bwd_finish(const tsp_cfg* cfg, int32_t r, const float* h_r,
                                   const void* g_mlp, const float* db_r, const void* dy_r,
                                   float* dh_r, float* dg_mlp, void* ws, size_t ws_bytes,
                                   void* stream);
tsp_status tsp_rank_attn_bwd_heads(const tsp_cfg* cfg, int32_t r, int32_t k,
                                   const void* kv_all_k, float* grad_k, void* dkv_k, void* ws,
                                   size_t ws_bytes, void* stream);
tsp_status tsp_rank_attn_bwd_weights(const tsp_cfg* cfg, int32_t r, int32_t k,
                                     const void* dkv_own, float* grad_k, float* da_r, void* ws,
                                     size_t ws_bytes, void* stream);
tsp_status tsp_rank_attn_bwd_finish(const tsp_cfg* cfg, int32_t r, const void* x_r,
                                    const void* g_attn, const float* da_r, const float* dh_r,
                                    float* dx_r, float* dg_attn, void* ws, size_t ws_bytes,
                                    void* stream);

/* Reads (and with reset != 0 clears) the sticky device status word.  Waits
 * for `stream` to finish.  Returns TSP_OK or the first device error seen
 * (TSP_ERR_TIMEOUT or TSP_ERR_RANGE). */
tsp_status tsp_device_status(void* stream, int32_t reset);

/* Static string for a status code. */
const char* tsp_strerror(tsp_status s);

/* Number of SMs the kernels size their persistent grids for (current device,
 * queried on first use; 0 if no device). */
int32_t tsp_num_sms(void);

/* Launch accounting (not on the pages: measurement plumbing).
 * tsp_profile_enable(1) clears the record and starts bracketing every later
 * launch site with CUDA events on its stream; (0) stops.  tsp_profile_report
 * waits for the recorded events and writes one line per launch-site label,
 * "label<TAB>kernels<TAB>total_ms<NL>", into buf (host memory, `bytes` long,
 * NUL-terminated); returns the number of lines, or -1 if buf is too small or
 * an event failed.  tsp_launch_count: kernels launched by the library since
 * it was loaded. */
void tsp_profile_enable(int32_t on);
int32_t tsp_profile_report(char* buf, int64_t bytes);
int64_t tsp_launch_count(void);

/* Failure-detection test knob (not on the pages): the next n tensor-core GEMM
 * launches each leave one pipeline stage of their first CTA unfilled, so that
 * CTA's bounded wait runs out (after TSP_WAIT_LIMIT_MS, an environment
 * variable read once, default 4000) and the call reports TSP_ERR_TIMEOUT
 * through tsp_device_status -- without a fault or a hang.  n <= 0 turns it
 * off.  Never needed in normal use. */
void tsp_debug_skip_stage(int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* TSP_H_ */
