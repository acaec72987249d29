// api.cu -- the C ABI (include/tsp.h): argument checks, workspace layout and
// the launch sequence of the TSP-folded block on one stream.
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), section 2.
// The D ranks are virtual: rank r's tokens are rows [r*2c, (r+1)*2c) of the
// zigzag buffer, a weight shard is a column range of the unsharded weight,
// and every collective of the real schedule becomes a layout fact:
//   broadcast of shard k  -> the GEMM's N (or K) range is segmented by shard;
//   K/V all-gather        -> all ranks' K/V already sit in one buffer;
//   MLP ring              -> the W_2 GEMM's K loop runs in ring order per rank;
//   weight-grad reduction -> the wgrad GEMMs' K loop (tokens) runs over every
//                            rank's rows into one fp32 accumulator.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"

namespace tsp {

__device__ int g_status_word = 0;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return dev;
}

namespace {
std::atomic<int> g_debug_skip{0};
}  // namespace

bool take_debug_skip() {
  int n = g_debug_skip.load(std::memory_order_relaxed);
  while (n > 0 && !g_debug_skip.compare_exchange_weak(n, n - 1)) {
  }
  return n > 0;
}

int* status_word() {
  static int* ptr[kMaxDevices] = {nullptr};
  const int dev = current_device();
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess) ptr[dev] = (int*)p;
  }
  return ptr[dev];
}

int num_sms() {
  static int n[kMaxDevices] = {0};
  const int dev = current_device();
  if (n[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) v = 0;
    n[dev] = v > 0 ? v : 1;
  }
  return n[dev];
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = getenv("TSP_WAIT_LIMIT_MS");  // debug knob; default 4 s per wait
    uint64_t ms = 4000;
    if (e && atoll(e) > 0) ms = (uint64_t)atoll(e);
    return ms * 1000000ull;
  }();
  return v;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
}  // namespace

bool tma_map_f16(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld,
                 int box_outer) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_outer};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Launch accounting: every kernel launch site is wrapped in a Prof scope that
// counts its kernels and, while profiling is on, brackets them with CUDA
// events recorded on the launch stream.
// ---------------------------------------------------------------------------
namespace {
std::atomic<long long> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfRec {
  const char* name;
  int kernels;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

Prof::Prof(const char* name, cudaStream_t st, int kernels) : name_(name), kernels_(kernels), st_(st) {
  g_launches.fetch_add(kernels);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  on_ = true;
  a_ = pool_event();
  b_ = pool_event();
  cudaEventRecord(a_, st_);
}

Prof::~Prof() {
  if (!on_) return;
  cudaEventRecord(b_, st_);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.push_back(ProfRec{name_, kernels_, a_, b_});
}

namespace {

bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// K/V heads, the width of K (and of V), and the row length of the Q|K|V buffer
int kv_heads(const tsp_cfg* c) { return c->Hkv > 0 ? c->Hkv : c->H; }
int64_t kv_dim(const tsp_cfg* c) { return (int64_t)kv_heads(c) * c->dh; }
int64_t qkv_ld(const tsp_cfg* c) { return c->d + 2 * kv_dim(c); }

tsp_status check_cfg(const tsp_cfg* c) {
  if (!c) return TSP_ERR_INVALID_ARG;
  if (c->S <= 0 || c->D < 1 || c->D > 64 || c->S % (2 * (int64_t)c->D) != 0)
    return TSP_ERR_INVALID_ARG;
  if (c->d <= 0 || c->H <= 0 || c->d % c->H != 0 || c->dh != c->d / c->H) return TSP_ERR_INVALID_ARG;
  if (c->inter <= 0 || c->d < c->D || c->inter < c->D) return TSP_ERR_INVALID_ARG;
  if (c->dtype != TSP_F32 && c->dtype != TSP_BF16) return TSP_ERR_INVALID_ARG;
  if (!(c->eps >= 0.f)) return TSP_ERR_INVALID_ARG;
  if (!(c->rope_base >= 0.f) || (c->rope_base > 0.f && c->dh % 2 != 0)) return TSP_ERR_INVALID_ARG;
  if (c->Hkv < 0 || (c->Hkv > 0 && c->H % c->Hkv != 0)) return TSP_ERR_INVALID_ARG;
  if (kv_dim(c) < c->D) return TSP_ERR_INVALID_ARG;
  if (c->mlp_tile < 0) return TSP_ERR_INVALID_ARG;
  if (c->mlp_tile > 0) {
    if (c->mlp_tile % 128 != 0 || (c->S / c->D) % c->mlp_tile != 0) return TSP_ERR_INVALID_ARG;
    if (c->dtype != TSP_BF16) return TSP_ERR_UNSUPPORTED;
  }
  if (c->S > (int64_t)1 << 31) return TSP_ERR_UNSUPPORTED;
  if (c->dtype == TSP_F32 && c->dh > 128) return TSP_ERR_UNSUPPORTED;
  return TSP_OK;
}

tsp_status check_bf16_mlp(const tsp_cfg* c) {
  if (c->dtype != TSP_BF16) return TSP_OK;
  if (c->d % 256 != 0 || c->inter % 128 != 0) return TSP_ERR_UNSUPPORTED;
  return TSP_OK;
}
tsp_status check_bf16_attn(const tsp_cfg* c) {
  if (c->dtype != TSP_BF16) return TSP_OK;
  if (c->d % 256 != 0 || c->dh != 128 || (c->S / (2 * c->D)) % 256 != 0) return TSP_ERR_UNSUPPORTED;
  if (kv_dim(c) % 256 != 0) return TSP_ERR_UNSUPPORTED;
  return TSP_OK;
}

// Activation buffers of the forward pass (the "saved" set of the backward).
struct Acts {
  float *rstd1, *rstd2, *lse;
  void *a, *qkv, *o, *h, *b, *ab, *g;
  float2* rope;   // (cos, sin) per zigzag row and frequency, when cfg->rope_base > 0
  size_t bytes;
};

enum { PART_ATTN = 1, PART_MLP = 2, PART_AB = 4, PART_NO_G = 8 };

Acts acts_layout(const tsp_cfg* c, int parts, uint8_t* base) {
  const size_t e = c->dtype == TSP_BF16 ? 2 : 4;
  const size_t S = (size_t)c->S, d = (size_t)c->d, I = (size_t)c->inter, H = (size_t)c->H;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off += up256(bytes);
    return p;
  };
  Acts A;
  memset(&A, 0, sizeof(A));
  if (parts & PART_ATTN) {
    A.rstd1 = (float*)take(S * 4);
    A.lse = (float*)take(H * S * 4);
    A.a = take(S * d * e);
    A.qkv = take(S * (size_t)qkv_ld(c) * e);
    A.o = take(S * d * e);
    if (c->rope_base > 0.f) A.rope = (float2*)take(S * (size_t)(c->dh / 2) * sizeof(float2));
  }
  if (parts & PART_MLP) {
    A.rstd2 = (float*)take(S * 4);
    A.h = (parts & PART_ATTN) ? take(S * d * 4) : nullptr;  // fp32 residual stream
    A.b = take(S * d * e);
    if (!(parts & PART_NO_G)) A.g = take(S * I * e);
    if (parts & PART_AB) A.ab = take(S * 2 * I * e);
  }
  A.bytes = off;
  return A;
}

int fwd_parts(const tsp_cfg* c, bool training) {
  // with MLP tiling the training record keeps neither G nor A|B (the
  // backward recomputes them tile by tile from b)
  if (training && c->mlp_tile > 0) return PART_ATTN | PART_MLP | PART_NO_G;
  // the fp32 path builds G from A|B, so it always keeps them
  return PART_ATTN | PART_MLP | ((training || c->dtype == TSP_F32) ? PART_AB : 0);
}

// bytes of one MLP tile's G (fp16) in the training forward's workspace
size_t mlp_tile_g_bytes(const tsp_cfg* c) {
  return c->mlp_tile > 0 ? up256((size_t)c->mlp_tile * c->inter * 2) : 0;
}

struct BwdWs {
  void *dab, *dg_f32, *db, *dh_f32, *dh_t, *dO, *dqkv, *da, *dy16;
  void *gt, *abt;   // MLP tiling: one tile's recomputed G and A|B
  float *delta, *dq_acc, *dg_part;
  size_t bytes;
};

BwdWs bwd_layout(const tsp_cfg* c, uint8_t* base) {
  const size_t e = c->dtype == TSP_BF16 ? 2 : 4;
  const size_t S = (size_t)c->S, d = (size_t)c->d, I = (size_t)c->inter, H = (size_t)c->H;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off += up256(bytes);
    return p;
  };
  BwdWs W;
  memset(&W, 0, sizeof(W));
  const size_t mrows = c->mlp_tile > 0 ? (size_t)c->mlp_tile : S;   // rows of the MLP buffers
  W.dab = take(mrows * 2 * I * e);
  if (c->mlp_tile > 0) {
    W.gt = take(mrows * I * e);
    W.abt = take(mrows * 2 * I * e);
  }
  if (c->dtype == TSP_F32) W.dg_f32 = take(S * I * 4);
  W.db = take(S * d * 4);
  W.dh_f32 = take(S * d * 4);
  if (c->dtype == TSP_BF16) W.dh_t = take(S * d * e);
  W.dO = take(S * d * e);
  W.dqkv = take(S * (size_t)qkv_ld(c) * e);
  W.da = take(S * d * 4);
  W.delta = (float*)take(2 * H * S * 4);   // Delta [H, S], then (bf16 path) LSE*log2(e) - 8
  if (c->dtype == TSP_BF16) W.dq_acc = (float*)take(S * d * 4);
  W.dg_part = (float*)take((size_t)rmsnorm_bwd_blocks(c->S) * d * 4);
  if (c->dtype == TSP_BF16) W.dy16 = take(S * d * 2);
  W.bytes = off;
  return W;
}

// fp16 copies of the bf16 weights (the internal tensor-core operand type);
// refreshed from the caller's weights on every call.
struct WCache {
  void *wq, *wk, *wv, *wo, *w1, *w3, *w2;
  size_t bytes;
};

enum { WC_ATTN = 1, WC_MLP = 2 };

WCache wcache_layout(const tsp_cfg* c, int which, uint8_t* base) {
  WCache W;
  memset(&W, 0, sizeof(W));
  if (c->dtype != TSP_BF16) return W;
  const size_t d = (size_t)c->d, I = (size_t)c->inter;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off += up256(bytes);
    return p;
  };
  if (which & WC_ATTN) {
    const size_t dk = (size_t)kv_dim(c);
    W.wq = take(d * d * 2);
    W.wk = take(dk * d * 2);
    W.wv = take(dk * d * 2);
    W.wo = take(d * d * 2);
  }
  if (which & WC_MLP) {
    W.w1 = take(I * d * 2);
    W.w3 = take(I * d * 2);
    W.w2 = take(d * I * 2);
  }
  W.bytes = off;
  return W;
}

tsp_status fill_wcache(const tsp_cfg* c, const WCache& W, const tsp_attn_w* aw, const tsp_mlp_w* mw,
                       cudaStream_t st) {
  const int64_t dd = (int64_t)c->d * c->d, Id = (int64_t)c->inter * c->d;
  const void* src[kMaxConvert];
  void* dst[kMaxConvert];
  int64_t n[kMaxConvert];
  int k = 0;
  auto add = [&](const void* s_, void* d_, int64_t n_) {
    src[k] = s_;
    dst[k] = d_;
    n[k] = n_;
    ++k;
  };
  if (W.wq) {
    const int64_t kd = kv_dim(c) * c->d;
    add(aw->wq, W.wq, dd);
    add(aw->wk, W.wk, kd);
    add(aw->wv, W.wv, kd);
    add(aw->wo, W.wo, dd);
  }
  if (W.w1) {
    add(mw->w1, W.w1, Id);
    add(mw->w3, W.w3, Id);
    add(mw->w2, W.w2, Id);
  }
  return k == 0 ? TSP_OK : launch_convert_bf16_f16_many(src, dst, n, k, st);
}

cudaStream_t S_(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Rotary embedding of the Q and K column blocks of an [S, d + 2*Hkv*dh] Q|K|V buffer
// (inverse = 1: the transposed rotation, which maps gradients of the rotated
// Q, K back to gradients of the projections).  The forward fills the table of
// (cos, sin) per zigzag row first; the backward reuses the saved one.
tsp_status rope_qk(const tsp_cfg* c, const Acts& A, void* qkv, int ty, int inverse,
                   cudaStream_t st) {
  if (c->rope_base <= 0.f) return TSP_OK;
  tsp_status r;
  if (!inverse &&
      (r = launch_rope_table(A.rope, c->S, c->D, c->dh, c->rope_base, st)) != TSP_OK)
    return r;
  return launch_rope(qkv, ty, c->S, (int)qkv_ld(c), c->d, c->H, kv_heads(c), c->dh, A.rope,
                     inverse, st);
}

// ----------------------------------------------------------------------------
// Forward halves
// ----------------------------------------------------------------------------

// x_f32: the input x is fp32 (a residual stream kept in fp32) instead of the cfg dtype.
// h_f32: write h in fp32 (the block's residual stream) instead of the cfg dtype.
// WC: fp16 weight copies (bf16 configuration; filled by the caller of this function).
tsp_status attn_half(const tsp_cfg* c, const void* x, bool x_f32, const tsp_attn_w* w,
                     const WCache& WC, void* h, bool h_f32, const Acts& A, cudaStream_t st) {
  const int64_t S = c->S;
  const int d = c->d, D = c->D;
  const int x_ty = (c->dtype == TSP_BF16 && !x_f32) ? TY_BF16 : TY_F32;
  tsp_status r = launch_rmsnorm_fwd(x, x_ty, w->g_attn, A.a,
                                    c->dtype == TSP_BF16 ? TY_F16 : TY_F32, A.rstd1, S, d, c->eps,
                                    c->dtype, st);
  if (r != TSP_OK) return r;
  if (c->dtype == TSP_BF16) {
    // Q|K|V: the N range is split into the W_Q, W_K, W_V segments; within a
    // segment the N tiles are the column shards C_k streamed one after another.
    const int64_t ld = qkv_ld(c), dk = kv_dim(c);
    if (dk == d) {
      TcGemm g;
      g.M = (int)S; g.N = 3 * d; g.K = d;
      g.A[0] = A.a; g.lda[0] = d; g.kseg_len[0] = d;
      g.B[0] = WC.wq; g.B[1] = WC.wk; g.B[2] = WC.wv;
      g.ldb[0] = g.ldb[1] = g.ldb[2] = d;
      g.nseg_n = d; g.name = "gemm_qkv";
      g.epi = EPI_STORE; g.out_type = OUT_F16; g.out = A.qkv; g.ldo = ld;
      if ((r = gemm_tc(g, st)) != TSP_OK) return r;
    } else {
      // grouped K/V heads: Q (d columns), then K|V (2 x kv_dim columns)
      TcGemm q;
      q.M = (int)S; q.N = d; q.K = d;
      q.A[0] = A.a; q.lda[0] = d; q.kseg_len[0] = d;
      q.B[0] = WC.wq; q.ldb[0] = d; q.name = "gemm_q";
      q.epi = EPI_STORE; q.out_type = OUT_F16; q.out = A.qkv; q.ldo = ld;
      if ((r = gemm_tc(q, st)) != TSP_OK) return r;
      TcGemm kv;
      kv.M = (int)S; kv.N = (int)(2 * dk); kv.K = d;
      kv.A[0] = A.a; kv.lda[0] = d; kv.kseg_len[0] = d;
      kv.B[0] = WC.wk; kv.B[1] = WC.wv; kv.ldb[0] = kv.ldb[1] = d;
      kv.nseg_n = (int)dk; kv.name = "gemm_kv";
      kv.epi = EPI_STORE; kv.out_type = OUT_F16; kv.out = (uint8_t*)A.qkv + (size_t)d * 2;
      kv.ldo = ld;
      if ((r = gemm_tc(kv, st)) != TSP_OK) return r;
    }
    if ((r = rope_qk(c, A, A.qkv, TY_F16, 0, st)) != TSP_OK) return r;
    if ((r = launch_attn_fwd_f16(A.qkv, A.o, A.lse, S, c->H, kv_heads(c), c->dh, D, st)) != TSP_OK)
      return r;
    // W_O: split-K over the shards C_k (k = 0..D-1, broadcast order), fp32
    // accumulation in TMEM, residual x added in the epilogue.
    TcGemm o;
    o.M = (int)S; o.N = d; o.K = d;
    o.A[0] = A.o; o.lda[0] = d; o.kseg_len[0] = d;
    o.B[0] = WC.wo; o.ldb[0] = d;
    o.epi = EPI_RES; o.res = x; o.ldr = d; o.res_f32 = x_f32; o.name = "gemm_oproj";
    o.out = h; o.ldo = d; o.out_type = h_f32 ? OUT_F32 : OUT_BF16;
    return gemm_tc(o, st);
  }
  // exact fp32 path: literal shard loop
  const float* a = (const float*)A.a;
  float* qkv = (float*)A.qkv;
  const int ld = (int)qkv_ld(c), dk = (int)kv_dim(c);
  const float* W3[3] = {(const float*)w->wq, (const float*)w->wk, (const float*)w->wv};
  const int width[3] = {d, dk, dk}, col0[3] = {0, d, d + dk};
  for (int k = 0; k < D; ++k) {
    for (int j = 0; j < 3; ++j) {
      const int n = width[j];
      const int lo = (int)((int64_t)k * n / D), hi = (int)((int64_t)(k + 1) * n / D);
      r = launch_gemm_f32((int)S, hi - lo, d, a, d, 1, W3[j] + (int64_t)lo * d, d, 1,
                          qkv + col0[j] + lo, ld, nullptr, 0, 0, st);
      if (r != TSP_OK) return r;
    }
  }
  if ((r = rope_qk(c, A, qkv, TY_F32, 0, st)) != TSP_OK) return r;
  if ((r = launch_attn_f32_fwd(qkv, S, c->H, kv_heads(c), c->dh, D, (float*)A.o, A.lse, st)) !=
      TSP_OK)
    return r;
  for (int k = 0; k < D; ++k) {
    const int lo = (int)((int64_t)k * d / D), hi = (int)((int64_t)(k + 1) * d / D);
    r = launch_gemm_f32((int)S, d, hi - lo, (const float*)A.o + lo, d, 1, (const float*)w->wo + lo,
                        d, 1, (float*)h, d, k == 0 ? (const float*)x : nullptr, d, k > 0, st);
    if (r != TSP_OK) return r;
  }
  return TSP_OK;
}

// hin_f32: the input h is fp32 (the block's residual stream), else the cfg dtype.
// y_f32: write y in fp32 instead of the cfg dtype (bf16 configuration).
// g_tile (training with cfg->mlp_tile): the MLP runs one row tile at a time
// with G in this [mlp_tile, inter] buffer, and keeps no G or A|B.
tsp_status mlp_half(const tsp_cfg* c, const void* hin, bool hin_f32, const tsp_mlp_w* w,
                    const WCache& WC, void* y, bool y_f32, const Acts& A, cudaStream_t st,
                    void* g_tile = nullptr) {
  const int64_t S = c->S;
  const int d = c->d, I = c->inter, D = c->D;
  const int64_t rows_per_rank = S / D;
  tsp_status r;
  const void* b = hin;
  const bool bf = c->dtype == TSP_BF16;
  if (w->g_mlp) {
    if ((r = launch_rmsnorm_fwd(hin, bf ? (hin_f32 ? TY_F32 : TY_BF16) : TY_F32, w->g_mlp, A.b,
                                bf ? TY_F16 : TY_F32, A.rstd2, S, d, c->eps, c->dtype, st)) !=
        TSP_OK)
      return r;
    b = A.b;
  } else if (bf) {
    // no norm: the GEMM operand is h itself, in the internal fp16 type
    if (hin_f32) return TSP_ERR_UNSUPPORTED;
    if ((r = launch_convert_bf16_f16(hin, A.b, S * d, st)) != TSP_OK) return r;
    b = A.b;
  }
  if (bf && g_tile) {
    // sequence tiles (each inside one virtual rank's rows): the same two
    // GEMMs as below on M = mlp_tile rows, G living only for its tile
    const int64_t tile = c->mlp_tile;
    for (int64_t t0 = 0; t0 < S; t0 += tile) {
      TcGemm g;
      g.M = (int)tile; g.N = I; g.K = d;
      g.A[0] = (const uint8_t*)b + (size_t)t0 * d * 2; g.lda[0] = d; g.kseg_len[0] = d;
      g.B[0] = WC.w1; g.B[1] = WC.w3; g.ldb[0] = g.ldb[1] = d;
      g.paired = true; g.name = "gemm_w13_swiglu";
      g.epi = EPI_SWIGLU; g.out = g_tile; g.ldo = I;
      if ((r = gemm_tc(g, st)) != TSP_OK) return r;
      TcGemm o;
      o.M = (int)tile; o.N = d; o.K = I;
      o.A[0] = g_tile; o.lda[0] = I; o.kseg_len[0] = I;
      o.B[0] = WC.w2; o.ldb[0] = I;
      o.rot_rows = (int)tile; o.rot_r0 = (int)(t0 / rows_per_rank); o.rot_D = D;
      o.name = "gemm_w2";
      o.out = (uint8_t*)y + (size_t)t0 * d * (y_f32 ? 4 : 2); o.ldo = d;
      o.out_type = y_f32 ? OUT_F32 : OUT_BF16;
      if (w->add_residual) {
        o.epi = EPI_RES; o.res = (const uint8_t*)hin + (size_t)t0 * d * (hin_f32 ? 4 : 2);
        o.ldr = d; o.res_f32 = hin_f32;
      } else {
        o.epi = EPI_STORE;
      }
      if ((r = gemm_tc(o, st)) != TSP_OK) return r;
    }
    return TSP_OK;
  }
  if (bf) {
    // W_1|W_3: one 256-wide B tile = 128 rows of W_1 and the same 128 rows of
    // W_3 (split-N over the I_k shards); SiLU(.)*gate fused in the epilogue.
    TcGemm g;
    g.M = (int)S; g.N = I; g.K = d;
    g.A[0] = b; g.lda[0] = d; g.kseg_len[0] = d;
    g.B[0] = WC.w1; g.B[1] = WC.w3; g.ldb[0] = g.ldb[1] = d;
    g.paired = true; g.name = "gemm_w13_swiglu";
    g.epi = EPI_SWIGLU; g.out = A.g; g.ldo = I;
    if (A.ab) {
      g.out2 = A.ab; g.ldo2 = 2 * (int64_t)I;
      g.out3 = (uint8_t*)A.ab + (size_t)I * 2; g.ldo3 = 2 * (int64_t)I;
    }
    if ((r = gemm_tc(g, st)) != TSP_OK) return r;
    // W_2: K = I walked shard by shard in ring order (r - t) mod D for the
    // virtual rank r owning the row tile; residual fused.
    TcGemm o;
    o.M = (int)S; o.N = d; o.K = I;
    o.A[0] = A.g; o.lda[0] = I; o.kseg_len[0] = I;
    o.B[0] = WC.w2; o.ldb[0] = I;
    o.rot_rows = (int)rows_per_rank; o.rot_D = D; o.name = "gemm_w2";
    o.out = y; o.ldo = d; o.out_type = y_f32 ? OUT_F32 : OUT_BF16;
    if (w->add_residual) {
      o.epi = EPI_RES; o.res = hin; o.ldr = d; o.res_f32 = hin_f32;
    } else {
      o.epi = EPI_STORE;
    }
    return gemm_tc(o, st);
  }
  const float* bin = (const float*)b;
  float* ab = (float*)A.ab;
  for (int k = 0; k < D; ++k) {
    const int lo = (int)((int64_t)k * I / D), hi = (int)((int64_t)(k + 1) * I / D);
    if ((r = launch_gemm_f32((int)S, hi - lo, d, bin, d, 1, (const float*)w->w1 + (int64_t)lo * d, d,
                             1, ab + lo, 2 * I, nullptr, 0, 0, st)) != TSP_OK)
      return r;
    if ((r = launch_gemm_f32((int)S, hi - lo, d, bin, d, 1, (const float*)w->w3 + (int64_t)lo * d, d,
                             1, ab + I + lo, 2 * I, nullptr, 0, 0, st)) != TSP_OK)
      return r;
  }
  if ((r = launch_swiglu_f32(ab, (float*)A.g, S, I, st)) != TSP_OK) return r;
  // ring: virtual rank rr takes shard (rr - t) mod D at step t
  for (int rr = 0; rr < D; ++rr) {
    const int64_t r0 = rr * rows_per_rank;
    for (int t = 0; t < D; ++t) {
      const int k = ((rr - t) % D + D) % D;
      const int lo = (int)((int64_t)k * I / D), hi = (int)((int64_t)(k + 1) * I / D);
      const float* res = (t == 0 && w->add_residual) ? (const float*)hin + r0 * d : nullptr;
      r = launch_gemm_f32((int)rows_per_rank, d, hi - lo, (const float*)A.g + r0 * I + lo, I, 1,
                          (const float*)w->w2 + lo, I, 1, (float*)y + r0 * d, d, res, d, t > 0, st);
      if (r != TSP_OK) return r;
    }
  }
  return TSP_OK;
}

// mats = false: the weight matrices are not read (their fp16 copies come
// prepared), only the gains
tsp_status check_attn_w(const tsp_attn_w* w, bool mats = true) {
  if (!w || !al16(w->g_attn)) return TSP_ERR_INVALID_ARG;
  if (mats && (!al16(w->wq) || !al16(w->wk) || !al16(w->wv) || !al16(w->wo)))
    return TSP_ERR_INVALID_ARG;
  return TSP_OK;
}
tsp_status check_mlp_w(const tsp_mlp_w* w, bool need_norm, bool mats = true) {
  if (!w || (mats && (!al16(w->w1) || !al16(w->w3) || !al16(w->w2)))) return TSP_ERR_INVALID_ARG;
  if (w->g_mlp && !al16(w->g_mlp)) return TSP_ERR_INVALID_ARG;
  if (need_norm && (!w->g_mlp || !w->add_residual)) return TSP_ERR_INVALID_ARG;
  return TSP_OK;
}

// ----------------------------------------------------------------------------
// Decode workspace: the T new tokens' activations and the attention splits'
// partial results (sized for a cache of `cap` rows).
// ----------------------------------------------------------------------------
struct DecWs {
  void *a, *qkv, *o, *g;   // a: the normalised rows (both norms in turn)
  float *h, *rstd, *part_o;
  float2* part_ml;
  size_t bytes;
};

DecWs decode_layout(const tsp_cfg* c, int T, int64_t cap, uint8_t* base) {
  const size_t e = c->dtype == TSP_BF16 ? 2 : 4;   // fp16 / fp32 internal element
  const size_t d = (size_t)c->d, I = (size_t)c->inter, H = (size_t)c->H, dh = (size_t)c->dh;
  DecWs W;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off += up256(bytes);
    return p;
  };
  W.a = take(T * d * e);
  W.rstd = (float*)take(T * 4);
  W.qkv = take(T * (size_t)qkv_ld(c) * e);
  W.o = take(T * d * e);
  W.g = take(T * I * e);
  W.h = (float*)take(T * d * 4);
  const size_t nsplit = (size_t)decode_splits(c->S, c->D, cap);
  W.part_o = (float*)take(nsplit * H * T * dh * 4);
  W.part_ml = (float2*)take(nsplit * H * T * sizeof(float2));
  W.bytes = off;
  return W;
}

tsp_status decode_impl(const tsp_cfg* c, const void* x, int T, int64_t n_cached,
                       const tsp_attn_w* aw, const tsp_mlp_w* mw, void* y, void* kv,
                       int64_t kv_rows, const DecWs& W, cudaStream_t st) {
  const bool bf = c->dtype == TSP_BF16;
  const int io_ty = bf ? TY_BF16 : TY_F32, ct = bf ? TY_F16 : TY_F32;
  const int d = c->d, I = c->inter, dk = (int)kv_dim(c);
  const int64_t ld = qkv_ld(c);
  tsp_status r;
  // a = rms(x; g_attn)
  if ((r = launch_rmsnorm_fwd(x, io_ty, aw->g_attn, W.a, ct, W.rstd, T, d, c->eps, c->dtype,
                              st)) != TSP_OK)
    return r;
  // q | k | v = a [W_Q; W_K; W_V]^T, Q and K rotated at their positions,
  // K | V also appended to the cache rows n_cached ..
  {
    Gemv g;
    g.epi = GEMV_QKV; g.dtype = c->dtype; g.x = W.a; g.ldx = d;
    g.w[0] = aw->wq; g.w[1] = aw->wk; g.w[2] = aw->wv;
    g.rows[0] = d; g.rows[1] = dk; g.rows[2] = dk; g.nseg = 3;
    g.K = d; g.T = T; g.out = W.qkv; g.ldo = ld; g.out_ty = ct;
    g.dh = c->dh; g.qk_heads = c->H + kv_heads(c); g.d = d; g.rope_base = c->rope_base;
    g.pos0 = n_cached; g.kv = kv; g.ldkv = 2 * dk; g.kv_rows = kv_rows; g.name = "gemv_qkv";
    if ((r = launch_gemv(g, st)) != TSP_OK) return r;
  }
  {
    DecodeAttn a;
    a.dtype = c->dtype; a.q = W.qkv; a.ldq = ld; a.kv = kv; a.o = W.o;
    a.part_o = W.part_o; a.part_ml = W.part_ml;
    a.S = c->S; a.n_cached = n_cached; a.D = c->D; a.T = T;
    a.H = c->H; a.Hkv = kv_heads(c); a.dh = c->dh;
    if ((r = launch_decode_attn(a, st)) != TSP_OK) return r;
  }
  // h = x + O W_O^T (fp32)
  {
    Gemv g;
    g.epi = GEMV_RES; g.dtype = c->dtype; g.x = W.o; g.ldx = d;
    g.w[0] = aw->wo; g.rows[0] = d; g.nseg = 1; g.K = d; g.T = T;
    g.out = W.h; g.ldo = d; g.out_ty = TY_F32; g.res = x; g.ldr = d; g.res_ty = io_ty;
    g.name = "gemv_oproj";
    if ((r = launch_gemv(g, st)) != TSP_OK) return r;
  }
  // G = silu(b W_1^T) * (b W_3^T), b = rms(h; g_mlp)
  if ((r = launch_rmsnorm_fwd(W.h, TY_F32, mw->g_mlp, W.a, ct, W.rstd, T, d, c->eps, c->dtype,
                              st)) != TSP_OK)
    return r;
  {
    Gemv g;
    g.epi = GEMV_SWIGLU; g.dtype = c->dtype; g.x = W.a; g.ldx = d;
    g.w[0] = mw->w1; g.w[1] = mw->w3; g.rows[0] = g.rows[1] = I; g.nseg = 2;
    g.K = d; g.T = T; g.out = W.g; g.ldo = I; g.out_ty = ct; g.name = "gemv_w13_swiglu";
    if ((r = launch_gemv(g, st)) != TSP_OK) return r;
  }
  // y = h + G W_2^T
  Gemv g;
  g.epi = GEMV_RES; g.dtype = c->dtype; g.x = W.g; g.ldx = I;
  g.w[0] = mw->w2; g.rows[0] = d; g.nseg = 1; g.K = I; g.T = T;
  g.out = y; g.ldo = d; g.out_ty = io_ty; g.res = W.h; g.ldr = d; g.res_ty = TY_F32;
  g.name = "gemv_w2";
  return launch_gemv(g, st);
}

}  // namespace

// ----------------------------------------------------------------------------
// Backward (defined below the C entry points' helpers)
// ----------------------------------------------------------------------------
tsp_status block_bwd_impl(const tsp_cfg* c, const void* x, bool x_f32, const void* dy,
                          bool dy_f32, const void* saved, const tsp_attn_w* aw,
                          const tsp_mlp_w* mw, const void* prep, float* dx, float* dwq,
                          float* dwk, float* dwv, float* dwo, float* dw1, float* dw3, float* dw2,
                          float* dg_attn, float* dg_mlp, void* ws, cudaStream_t st);


tsp_status cfg_status(const tsp_cfg* cfg) { return check_cfg(cfg); }

tsp_status block_fwd_checked(const tsp_cfg* cfg, const void* x_z, bool x_f32, const tsp_attn_w* aw,
                             const tsp_mlp_w* mw, const void* prep, void* y_z, bool y_f32,
                             void* saved, void* ws, size_t ws_bytes, cudaStream_t st) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  // bf16 with prepared fp16 copies: the matrices themselves are not read
  const bool use_prep = prep != nullptr && cfg->dtype == TSP_BF16;
  if (prep && !al16(prep)) return TSP_ERR_INVALID_ARG;
  if ((r = check_attn_w(aw, !use_prep)) != TSP_OK) return r;
  if ((r = check_mlp_w(mw, true, !use_prep)) != TSP_OK) return r;
  if (!al16(x_z) || !al16(y_z)) return TSP_ERR_INVALID_ARG;
  if ((r = check_bf16_attn(cfg)) != TSP_OK) return r;
  if ((r = check_bf16_mlp(cfg)) != TSP_OK) return r;
  const bool training = saved != nullptr;
  const int parts = fwd_parts(cfg, training);
  const size_t nwc = use_prep ? 0 : wcache_layout(cfg, WC_ATTN | WC_MLP, nullptr).bytes;
  const int prep_flag = use_prep ? TSP_OP_PREPARED : 0;
  const size_t ntile = training ? mlp_tile_g_bytes(cfg) : 0;
  uint8_t *abase, *wbase;
  if (training) {
    // activations go to `saved`; the workspace holds the fp16 weight copies
    // (and, with MLP tiling, one tile's G)
    if (!al16(saved)) return TSP_ERR_INVALID_ARG;
    if (nwc + ntile > 0 && (!al16(ws) || ws_bytes < nwc + ntile)) return TSP_ERR_INVALID_ARG;
    abase = (uint8_t*)saved;
    wbase = (uint8_t*)ws;
  } else {
    if (!al16(ws) || ws_bytes < tsp_workspace_bytes(cfg, TSP_OP_BLOCK_FWD | prep_flag))
      return TSP_ERR_INVALID_ARG;
    abase = (uint8_t*)ws;
    wbase = (uint8_t*)ws + acts_layout(cfg, parts, nullptr).bytes;
  }
  const Acts A = acts_layout(cfg, parts, abase);
  const WCache WC = wcache_layout(cfg, WC_ATTN | WC_MLP, use_prep ? (uint8_t*)prep : wbase);
  if (!use_prep && (r = fill_wcache(cfg, WC, aw, mw, st)) != TSP_OK) return r;
  if ((r = attn_half(cfg, x_z, x_f32, aw, WC, A.h, true, A, st)) != TSP_OK) return r;
  return mlp_half(cfg, A.h, true, mw, WC, y_z, y_f32, A, st, ntile ? wbase + nwc : nullptr);
}

tsp_status block_bwd_checked(const tsp_cfg* cfg, const void* x_z, bool x_f32, const void* dy_z,
                             bool dy_f32, const void* saved, const tsp_attn_w* aw,
                             const tsp_mlp_w* mw, const void* prep, float* dx_z,
                             float* const* grads, void* ws, size_t ws_bytes, cudaStream_t st) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  const bool use_prep = prep != nullptr && cfg->dtype == TSP_BF16;
  if (prep && !al16(prep)) return TSP_ERR_INVALID_ARG;
  if ((r = check_attn_w(aw, !use_prep)) != TSP_OK) return r;
  if ((r = check_mlp_w(mw, true, !use_prep)) != TSP_OK) return r;
  if (!al16(x_z) || !al16(dy_z) || !al16(saved) || !al16(dx_z) || !grads) return TSP_ERR_INVALID_ARG;
  for (int k = 0; k < 9; ++k)
    if (!al16(grads[k])) return TSP_ERR_INVALID_ARG;
  if ((r = check_bf16_attn(cfg)) != TSP_OK) return r;
  if ((r = check_bf16_mlp(cfg)) != TSP_OK) return r;
  if (!al16(ws) ||
      ws_bytes < tsp_workspace_bytes(cfg, TSP_OP_BLOCK_BWD | (use_prep ? TSP_OP_PREPARED : 0)))
    return TSP_ERR_INVALID_ARG;
  const bool bf = cfg->dtype == TSP_BF16;
  return block_bwd_impl(cfg, x_z, bf && x_f32, dy_z, bf && dy_f32, saved, aw, mw,
                        use_prep ? prep : nullptr, dx_z, grads[0], grads[1], grads[2], grads[3],
                        grads[4], grads[5], grads[6], grads[7], grads[8], ws, st);
}

}  // namespace tsp

using namespace tsp;

extern "C" {

const char* tsp_strerror(tsp_status s) {
  switch (s) {
    case TSP_OK: return "ok";
    case TSP_ERR_INVALID_ARG: return "invalid argument";
    case TSP_ERR_UNSUPPORTED: return "shape not supported by the selected kernels";
    case TSP_ERR_CUDA: return "CUDA runtime error";
    case TSP_ERR_TIMEOUT: return "device pipeline wait exceeded its time limit";
    case TSP_ERR_RANGE: return "a value held in fp16 inside the bf16 path was out of fp16 range";
    case TSP_ERR_BOUNDS: return "a computed index failed its bounds check (checked build)";
  }
  return "unknown status";
}

int32_t tsp_num_sms(void) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) return 0;
  return num_sms();
}

tsp_status tsp_zigzag_permute(const void* src, void* dst, int64_t S, int32_t D, int64_t row_bytes,
                              int32_t inverse, void* stream) {
  if (!src || !dst || S <= 0 || D < 1 || D > 64 || S % (2 * (int64_t)D) != 0 || row_bytes <= 0)
    return TSP_ERR_INVALID_ARG;
  return launch_zigzag_permute(src, dst, S, D, row_bytes, inverse, S_(stream));
}

tsp_status tsp_rmsnorm_fwd(const void* u, const void* g, void* out, float* rstd, int64_t rows,
                           int32_t n, float eps, int32_t dtype, void* stream) {
  if (!u || !g || !out || rows <= 0 || n <= 0 || (dtype != TSP_F32 && dtype != TSP_BF16) ||
      !(eps >= 0.f))
    return TSP_ERR_INVALID_ARG;
  const int ty = dtype == TSP_BF16 ? TY_BF16 : TY_F32;
  return launch_rmsnorm_fwd(u, ty, g, out, ty, rstd, rows, n, eps, dtype, S_(stream));
}

size_t tsp_workspace_bytes(const tsp_cfg* cfg, int32_t op) {
  if (check_cfg(cfg) != TSP_OK) return 0;
  if (op & TSP_OP_PREPARED) {
    // the whole-block calls with prepared fp16 weight copies: no copies in the workspace
    const int base = op & ~TSP_OP_PREPARED;
    const size_t nwc = wcache_layout(cfg, WC_ATTN | WC_MLP, nullptr).bytes;
    if (base != TSP_OP_BLOCK_FWD && base != TSP_OP_BLOCK_BWD && base != TSP_OP_BLOCK_FWD_TRAIN)
      return 0;
    const size_t full = tsp_workspace_bytes(cfg, base);
    return std::max<size_t>(256, full - nwc);
  }
  switch (op) {
    case TSP_OP_ATTN_FWD:
      return acts_layout(cfg, PART_ATTN, nullptr).bytes + wcache_layout(cfg, WC_ATTN, nullptr).bytes;
    case TSP_OP_MLP_FWD:
      return acts_layout(cfg, PART_MLP | (cfg->dtype == TSP_F32 ? PART_AB : 0), nullptr).bytes +
             wcache_layout(cfg, WC_MLP, nullptr).bytes;
    case TSP_OP_BLOCK_FWD:
      return acts_layout(cfg, fwd_parts(cfg, false), nullptr).bytes +
             wcache_layout(cfg, WC_ATTN | WC_MLP, nullptr).bytes;
    case TSP_OP_BLOCK_BWD:
      return bwd_layout(cfg, nullptr).bytes + wcache_layout(cfg, WC_ATTN | WC_MLP, nullptr).bytes;
    case TSP_OP_BLOCK_FWD_TRAIN:
      return std::max<size_t>(256, wcache_layout(cfg, WC_ATTN | WC_MLP, nullptr).bytes +
                                       mlp_tile_g_bytes(cfg));
  }
  return 0;
}

size_t tsp_saved_bytes(const tsp_cfg* cfg) {
  if (check_cfg(cfg) != TSP_OK) return 0;
  return acts_layout(cfg, fwd_parts(cfg, true), nullptr).bytes;
}

tsp_status tsp_attn_block_fwd(const tsp_cfg* cfg, const void* x_z, const tsp_attn_w* w, void* h_z,
                              void* ws, size_t ws_bytes, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if ((r = check_attn_w(w)) != TSP_OK) return r;
  if (!al16(x_z) || !al16(h_z)) return TSP_ERR_INVALID_ARG;
  if ((r = check_bf16_attn(cfg)) != TSP_OK) return r;
  const size_t na = acts_layout(cfg, PART_ATTN, nullptr).bytes;
  if (!al16(ws) || ws_bytes < tsp_workspace_bytes(cfg, TSP_OP_ATTN_FWD)) return TSP_ERR_INVALID_ARG;
  const Acts A = acts_layout(cfg, PART_ATTN, (uint8_t*)ws);
  const WCache WC = wcache_layout(cfg, WC_ATTN, (uint8_t*)ws + na);
  cudaStream_t st = S_(stream);
  if ((r = fill_wcache(cfg, WC, w, nullptr, st)) != TSP_OK) return r;
  return attn_half(cfg, x_z, false, w, WC, h_z, false, A, st);
}

tsp_status tsp_gated_mlp_fwd(const tsp_cfg* cfg, const void* h_z, const tsp_mlp_w* w, void* y_z,
                             void* ws, size_t ws_bytes, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if ((r = check_mlp_w(w, false)) != TSP_OK) return r;
  if (!al16(h_z) || !al16(y_z)) return TSP_ERR_INVALID_ARG;
  if ((r = check_bf16_mlp(cfg)) != TSP_OK) return r;
  const int parts = PART_MLP | (cfg->dtype == TSP_F32 ? PART_AB : 0);
  const size_t na = acts_layout(cfg, parts, nullptr).bytes;
  if (!al16(ws) || ws_bytes < tsp_workspace_bytes(cfg, TSP_OP_MLP_FWD)) return TSP_ERR_INVALID_ARG;
  const Acts A = acts_layout(cfg, parts, (uint8_t*)ws);
  const WCache WC = wcache_layout(cfg, WC_MLP, (uint8_t*)ws + na);
  cudaStream_t st = S_(stream);
  if ((r = fill_wcache(cfg, WC, nullptr, w, st)) != TSP_OK) return r;
  return mlp_half(cfg, h_z, false, w, WC, y_z, false, A, st);
}

tsp_status tsp_block_fwd(const tsp_cfg* cfg, const void* x_z, const tsp_attn_w* aw,
                         const tsp_mlp_w* mw, void* y_z, void* saved, void* ws, size_t ws_bytes,
                         void* stream) {
  return block_fwd_checked(cfg, x_z, false, aw, mw, nullptr, y_z, false, saved, ws, ws_bytes,
                           S_(stream));
}

size_t tsp_block_weights_bytes(const tsp_cfg* cfg) {
  if (check_cfg(cfg) != TSP_OK || cfg->dtype != TSP_BF16) return 0;
  return wcache_layout(cfg, WC_ATTN | WC_MLP, nullptr).bytes;
}

tsp_status tsp_block_weights_prepare(const tsp_cfg* cfg, const tsp_attn_w* aw, const tsp_mlp_w* mw,
                                     void* prep, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if ((r = check_attn_w(aw)) != TSP_OK) return r;
  if ((r = check_mlp_w(mw, false)) != TSP_OK) return r;
  if (cfg->dtype != TSP_BF16) return TSP_OK;   // the fp32 path reads the weights as they are
  if (!al16(prep)) return TSP_ERR_INVALID_ARG;
  return fill_wcache(cfg, wcache_layout(cfg, WC_ATTN | WC_MLP, (uint8_t*)prep), aw, mw, S_(stream));
}

tsp_status tsp_block_fwd_prepared(const tsp_cfg* cfg, const void* x_z, const void* prep,
                                  const tsp_attn_w* aw, const tsp_mlp_w* mw, void* y_z, void* saved,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (cfg && cfg->dtype == TSP_BF16 && !prep) return TSP_ERR_INVALID_ARG;
  return block_fwd_checked(cfg, x_z, false, aw, mw, prep, y_z, false, saved, ws, ws_bytes,
                           S_(stream));
}

tsp_status tsp_block_bwd_prepared(const tsp_cfg* cfg, const void* x_z, const void* dy_z,
                                  const void* saved, const void* prep, const tsp_attn_w* aw,
                                  const tsp_mlp_w* mw, float* dx_z, float* dwq, float* dwk,
                                  float* dwv, float* dwo, float* dw1, float* dw3, float* dw2,
                                  float* dg_attn, float* dg_mlp, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (cfg && cfg->dtype == TSP_BF16 && !prep) return TSP_ERR_INVALID_ARG;
  float* const grads[9] = {dwq, dwk, dwv, dwo, dw1, dw3, dw2, dg_attn, dg_mlp};
  return block_bwd_checked(cfg, x_z, false, dy_z, false, saved, aw, mw, prep, dx_z, grads, ws,
                           ws_bytes, S_(stream));
}

tsp_status tsp_block_bwd(const tsp_cfg* cfg, const void* x_z, const void* dy_z, const void* saved,
                         const tsp_attn_w* aw, const tsp_mlp_w* mw, float* dx_z, float* dwq,
                         float* dwk, float* dwv, float* dwo, float* dw1, float* dw3, float* dw2,
                         float* dg_attn, float* dg_mlp, void* ws, size_t ws_bytes, void* stream) {
  float* const grads[9] = {dwq, dwk, dwv, dwo, dw1, dw3, dw2, dg_attn, dg_mlp};
  return block_bwd_checked(cfg, x_z, false, dy_z, false, saved, aw, mw, nullptr, dx_z, grads, ws,
                           ws_bytes, S_(stream));
}

size_t tsp_kv_cache_bytes(const tsp_cfg* cfg, int64_t kv_rows_cap) {
  if (check_cfg(cfg) != TSP_OK || kv_rows_cap < cfg->S) return 0;
  const size_t e = cfg->dtype == TSP_BF16 ? 2 : 4;
  return (size_t)kv_rows_cap * 2 * (size_t)kv_dim(cfg) * e;
}

size_t tsp_decode_workspace_bytes(const tsp_cfg* cfg, int32_t T, int64_t kv_rows_cap) {
  if (check_cfg(cfg) != TSP_OK || T < 1 || T > TSP_DECODE_MAX_T || kv_rows_cap < cfg->S + T)
    return 0;
  return decode_layout(cfg, T, kv_rows_cap, nullptr).bytes;
}

tsp_status tsp_block_prefill(const tsp_cfg* cfg, const void* x_z, const tsp_attn_w* aw,
                             const tsp_mlp_w* mw, void* y_z, void* kv, int64_t kv_rows_cap,
                             void* ws, size_t ws_bytes, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if (!al16(kv) || kv_rows_cap < cfg->S) return TSP_ERR_INVALID_ARG;
  if ((r = tsp_block_fwd(cfg, x_z, aw, mw, y_z, nullptr, ws, ws_bytes, stream)) != TSP_OK) return r;
  // the prompt's K (rotated) and V, still in the forward's Q|K|V buffer
  const Acts A = acts_layout(cfg, fwd_parts(cfg, false), (uint8_t*)ws);
  const size_t e = cfg->dtype == TSP_BF16 ? 2 : 4;
  const size_t dk = (size_t)kv_dim(cfg);
  TSP_CUDA_TRY(cudaMemcpy2DAsync(kv, 2 * dk * e, (const uint8_t*)A.qkv + (size_t)cfg->d * e,
                                 (size_t)qkv_ld(cfg) * e, 2 * dk * e, (size_t)cfg->S,
                                 cudaMemcpyDeviceToDevice, S_(stream)));
  return TSP_OK;
}

tsp_status tsp_block_decode(const tsp_cfg* cfg, const void* x, int32_t T, int64_t n_cached,
                            const tsp_attn_w* aw, const tsp_mlp_w* mw, void* y, void* kv,
                            int64_t kv_rows_cap, void* ws, size_t ws_bytes, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if ((r = check_attn_w(aw)) != TSP_OK) return r;
  if ((r = check_mlp_w(mw, true)) != TSP_OK) return r;
  if (T < 1 || T > TSP_DECODE_MAX_T) return TSP_ERR_INVALID_ARG;
  if (n_cached < cfg->S || n_cached + T > kv_rows_cap) return TSP_ERR_INVALID_ARG;
  if (!al16(x) || !al16(y) || !al16(kv)) return TSP_ERR_INVALID_ARG;
  if (!al16(ws) || ws_bytes < tsp_decode_workspace_bytes(cfg, T, kv_rows_cap))
    return TSP_ERR_INVALID_ARG;
  const DecWs W = decode_layout(cfg, T, kv_rows_cap, (uint8_t*)ws);
  return decode_impl(cfg, x, T, n_cached, aw, mw, y, kv, kv_rows_cap, W, S_(stream));
}

tsp_status tsp_pack_attn_shards(const tsp_cfg* cfg, const tsp_attn_w* w, void* dst, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if (!w || !w->wq || !w->wk || !w->wv || !w->wo || !dst) return TSP_ERR_INVALID_ARG;
  if (kv_dim(cfg) != cfg->d) return TSP_ERR_UNSUPPORTED;   // the packed layout is for MHA
  return launch_pack_attn_shards(w->wq, w->wk, w->wv, w->wo, dst, cfg->d, cfg->D, cfg->dtype,
                                 S_(stream));
}

void tsp_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  g_prof_on = on != 0;
}

int32_t tsp_profile_report(char* buf, int64_t bytes) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  std::map<std::string, std::pair<long long, double>> agg;
  for (auto& r : g_prof) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -1;
    auto& e = agg[r.name];
    e.first += r.kernels;
    e.second += ms;
  }
  std::string out;
  for (auto& kv : agg) {
    char line[256];
    snprintf(line, sizeof(line), "%s\t%lld\t%.6f\n", kv.first.c_str(), kv.second.first,
             kv.second.second);
    out += line;
  }
  if (!buf || bytes <= (int64_t)out.size()) return -1;
  memcpy(buf, out.c_str(), out.size() + 1);
  return (int32_t)agg.size();
}

int64_t tsp_launch_count(void) { return g_launches.load(); }

void tsp_debug_skip_stage(int32_t n) { g_debug_skip.store(n > 0 ? n : 0); }

tsp_status tsp_device_status(void* stream, int32_t reset) {
  int* p = status_word();
  if (!p) return TSP_ERR_CUDA;
  int v = 0;
  if (cudaStreamSynchronize(S_(stream)) != cudaSuccess) return TSP_ERR_CUDA;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TSP_ERR_CUDA;
  if (reset) {
    const int z = 0;
    if (cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return TSP_ERR_CUDA;
  }
  return (tsp_status)v;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Backward of the block
// ----------------------------------------------------------------------------
namespace tsp {

tsp_status block_bwd_impl(const tsp_cfg* c, const void* x, bool x_f32, const void* dy,
                          bool dy_f32, const void* saved, const tsp_attn_w* aw,
                          const tsp_mlp_w* mw, const void* prep, float* dx, float* dwq,
                          float* dwk, float* dwv, float* dwo, float* dw1, float* dw3, float* dw2,
                          float* dg_attn, float* dg_mlp, void* ws, cudaStream_t st) {
  const int64_t S = c->S;
  const int d = c->d, I = c->inter, D = c->D, H = c->H, dh = c->dh;
  const Acts A = acts_layout(c, fwd_parts(c, true), (uint8_t*)saved);
  const BwdWs W = bwd_layout(c, (uint8_t*)ws);
  tsp_status r;
  if (c->dtype == TSP_BF16) {
    const size_t e = 2;
    // the fp16 weight copies: prepared by the caller, or converted here
    const WCache WC = wcache_layout(c, WC_ATTN | WC_MLP, prep ? (uint8_t*)prep : (uint8_t*)ws + W.bytes);
    if (!prep && (r = fill_wcache(c, WC, aw, mw, st)) != TSP_OK) return r;
    // the upstream gradient in the internal fp16 operand type
    r = dy_f32 ? launch_convert_f32_f16((const float*)dy, W.dy16, S * d, st)
               : launch_convert_bf16_f16(dy, W.dy16, S * d, st);
    if (r != TSP_OK) return r;
    // MLP backward, over the whole sequence or (cfg->mlp_tile) one row tile at
    // a time; weight gradients sum over the tiles in fp32 (each tile lies in
    // one virtual rank's rows, so this is still the sum over the ranks' rows)
    const bool tiled = c->mlp_tile > 0;
    const int64_t tile = tiled ? c->mlp_tile : S;
    for (int64_t t0 = 0; t0 < S; t0 += tile) {
      const bool first = t0 == 0;
      const void* ab = A.ab;
      const void* gg = A.g;
      const uint8_t* b_t = (const uint8_t*)A.b + (size_t)t0 * d * e;
      const uint8_t* dy_t = (const uint8_t*)W.dy16 + (size_t)t0 * d * e;
      if (tiled) {
        // recompute the tile's G and A|B from the saved b
        TcGemm g;
        g.M = (int)tile; g.N = I; g.K = d;
        g.A[0] = b_t; g.lda[0] = d; g.kseg_len[0] = d;
        g.B[0] = WC.w1; g.B[1] = WC.w3; g.ldb[0] = g.ldb[1] = d;
        g.paired = true; g.name = "gemm_w13_recompute";
        g.epi = EPI_SWIGLU; g.out = W.gt; g.ldo = I;
        g.out2 = W.abt; g.ldo2 = 2 * (int64_t)I;
        g.out3 = (uint8_t*)W.abt + (size_t)I * e; g.ldo3 = 2 * (int64_t)I;
        if ((r = gemm_tc(g, st)) != TSP_OK) return r;
        ab = W.abt;
        gg = W.gt;
      }
      // dA|dB = SwiGLU'(dG), dG = dy W_2   (B operand W_2 read MN-major)
      {
        TcGemm g;
        g.M = (int)tile; g.N = I; g.K = d;
        g.A[0] = dy_t; g.lda[0] = d; g.kseg_len[0] = d;
        g.b_mn = true; g.B[0] = WC.w2; g.ldb[0] = I;
        g.epi = EPI_SWIGLU_BWD; g.name = "gemm_dgrad_w2_swiglu";
        g.e1 = ab; g.e2 = (const uint8_t*)ab + (size_t)I * e; g.lde = 2 * (int64_t)I;
        g.out = W.dab; g.ldo = 2 * (int64_t)I;
        g.out2 = (uint8_t*)W.dab + (size_t)I * e; g.ldo2 = 2 * (int64_t)I;
        if ((r = gemm_tc(g, st)) != TSP_OK) return r;
      }
      // a weight gradient of this tile: written by the first, added by the rest
      auto wgrad_epi = [&](TcGemm& g, float* out, int64_t ldo) {
        g.out = out; g.ldo = ldo;
        if (first) {
          g.epi = EPI_F32;
        } else {
          g.epi = EPI_RES; g.res = out; g.ldr = ldo; g.res_f32 = true; g.out_type = OUT_F32;
        }
      };
      // dW_2 = dy^T G: K = tokens, i.e. every virtual rank's rows summed in fp32
      {
        TcGemm g;
        g.M = d; g.N = I; g.K = (int)tile;
        g.a_mn = true; g.A[0] = dy_t; g.lda[0] = d; g.kseg_len[0] = (int)tile;
        g.b_mn = true; g.B[0] = gg; g.ldb[0] = I;
        g.name = "gemm_wgrad_w2";
        wgrad_epi(g, dw2, I);
        if ((r = gemm_tc(g, st)) != TSP_OK) return r;
      }
      if (!tiled) {
        // dW_1 | dW_3 = [dA | dB]^T b (one launch, rows split between the outputs)
        TcGemm g;
        g.M = 2 * I; g.N = d; g.K = (int)S;
        g.a_mn = true; g.A[0] = W.dab; g.lda[0] = 2 * (int64_t)I; g.kseg_len[0] = (int)S;
        g.b_mn = true; g.B[0] = A.b; g.ldb[0] = d;
        g.epi = EPI_F32; g.ldo = d; g.m_seg = I; g.name = "gemm_wgrad_w13";
        g.outs[0] = dw1; g.outs[1] = dw3;
        if ((r = gemm_tc(g, st)) != TSP_OK) return r;
      } else {
        for (int part = 0; part < 2; ++part) {   // dW_1 from dA, dW_3 from dB
          TcGemm g;
          g.M = I; g.N = d; g.K = (int)tile;
          g.a_mn = true; g.A[0] = (const uint8_t*)W.dab + (size_t)part * I * e;
          g.lda[0] = 2 * (int64_t)I; g.kseg_len[0] = (int)tile;
          g.b_mn = true; g.B[0] = b_t; g.ldb[0] = d;
          g.name = "gemm_wgrad_w13";
          wgrad_epi(g, part == 0 ? dw1 : dw3, d);
          if ((r = gemm_tc(g, st)) != TSP_OK) return r;
        }
      }
      // db = dA W_1 + dB W_3 (two K segments), fp32
      {
        TcGemm g;
        g.M = (int)tile; g.N = d; g.K = 2 * I;
        g.nks = 2;
        g.A[0] = W.dab; g.A[1] = (uint8_t*)W.dab + (size_t)I * e;
        g.lda[0] = g.lda[1] = 2 * (int64_t)I;
        g.kseg_len[0] = g.kseg_len[1] = I;
        g.b_mn = true; g.B[0] = WC.w1; g.B[1] = WC.w3; g.ldb[0] = g.ldb[1] = d;
        g.epi = EPI_F32; g.out = (float*)W.db + (size_t)t0 * d; g.ldo = d;
        g.name = "gemm_dgrad_w13";
        if ((r = gemm_tc(g, st)) != TSP_OK) return r;
      }
    }
    // dh = dy + RMSNorm_2'(db)   (fp32, plus an fp16 copy for the GEMMs)
    if ((r = launch_rmsnorm_bwd((const float*)W.db, A.h, TY_F32, mw->g_mlp, A.rstd2,
                                dy_f32 ? (const float*)dy : nullptr, dy_f32 ? nullptr : dy,
                                (float*)W.dh_f32, W.dh_t, TY_F16, dg_mlp, W.dg_part, S, d,
                                c->dtype, st)) != TSP_OK)
      return r;
    // dW_O = dh^T O
    {
      TcGemm g;
      g.M = d; g.N = d; g.K = (int)S;
      g.a_mn = true; g.A[0] = W.dh_t; g.lda[0] = d; g.kseg_len[0] = (int)S;
      g.b_mn = true; g.B[0] = A.o; g.ldb[0] = d;
      g.epi = EPI_F32; g.out = dwo; g.ldo = d; g.name = "gemm_wgrad_wo";
      if ((r = gemm_tc(g, st)) != TSP_OK) return r;
    }
    // dO = dh W_O
    {
      TcGemm g;
      g.M = (int)S; g.N = d; g.K = d;
      g.A[0] = W.dh_t; g.lda[0] = d; g.kseg_len[0] = d;
      g.b_mn = true; g.B[0] = WC.wo; g.ldb[0] = d;
      g.epi = EPI_STORE; g.out_type = OUT_F16; g.out = W.dO; g.ldo = d; g.name = "gemm_dgrad_wo";
      if ((r = gemm_tc(g, st)) != TSP_OK) return r;
    }
    if ((r = launch_attn_bwd_f16(A.qkv, A.o, W.dO, A.lse, W.delta, W.dq_acc, W.dqkv, S, H,
                                 kv_heads(c), dh, D, st)) != TSP_OK)
      return r;
    // gradients of the rotated Q, K -> gradients of the projections
    if ((r = rope_qk(c, A, W.dqkv, TY_F16, 1, st)) != TSP_OK) return r;
    // dW_Q | dW_K | dW_V = [dQ | dK | dV]^T a
    const int64_t ld = qkv_ld(c), dk = kv_dim(c);
    if (dk == d) {
      TcGemm g;
      g.M = 3 * d; g.N = d; g.K = (int)S;
      g.a_mn = true; g.A[0] = W.dqkv; g.lda[0] = ld; g.kseg_len[0] = (int)S;
      g.b_mn = true; g.B[0] = A.a; g.ldb[0] = d;
      g.epi = EPI_F32; g.ldo = d; g.m_seg = d; g.name = "gemm_wgrad_qkv";
      g.outs[0] = dwq; g.outs[1] = dwk; g.outs[2] = dwv;
      if ((r = gemm_tc(g, st)) != TSP_OK) return r;
    } else {
      TcGemm q;
      q.M = d; q.N = d; q.K = (int)S;
      q.a_mn = true; q.A[0] = W.dqkv; q.lda[0] = ld; q.kseg_len[0] = (int)S;
      q.b_mn = true; q.B[0] = A.a; q.ldb[0] = d;
      q.epi = EPI_F32; q.out = dwq; q.ldo = d; q.name = "gemm_wgrad_q";
      if ((r = gemm_tc(q, st)) != TSP_OK) return r;
      TcGemm kv;
      kv.M = (int)(2 * dk); kv.N = d; kv.K = (int)S;
      kv.a_mn = true; kv.A[0] = (uint8_t*)W.dqkv + (size_t)d * e; kv.lda[0] = ld;
      kv.kseg_len[0] = (int)S;
      kv.b_mn = true; kv.B[0] = A.a; kv.ldb[0] = d;
      kv.epi = EPI_F32; kv.ldo = d; kv.m_seg = dk; kv.name = "gemm_wgrad_kv";
      kv.outs[0] = dwk; kv.outs[1] = dwv;
      if ((r = gemm_tc(kv, st)) != TSP_OK) return r;
    }
    // da = dQ W_Q + dK W_K + dV W_V (three K segments), fp32
    {
      TcGemm g;
      g.M = (int)S; g.N = d; g.K = (int)ld;
      g.nks = 3;
      const void* ws3[3] = {WC.wq, WC.wk, WC.wv};
      const int64_t seg[3] = {d, dk, dk}, col[3] = {0, d, d + dk};
      for (int j = 0; j < 3; ++j) {
        g.A[j] = (uint8_t*)W.dqkv + (size_t)col[j] * e;
        g.lda[j] = ld;
        g.kseg_len[j] = (int)seg[j];
        g.B[j] = ws3[j];
        g.ldb[j] = d;
      }
      g.b_mn = true;
      g.epi = EPI_F32; g.out = W.da; g.ldo = d; g.name = "gemm_dgrad_qkv";
      if ((r = gemm_tc(g, st)) != TSP_OK) return r;
    }
    // dx = dh + RMSNorm_1'(da), fp32
    return launch_rmsnorm_bwd((const float*)W.da, x, x_f32 ? TY_F32 : TY_BF16, aw->g_attn, A.rstd1,
                              (const float*)W.dh_f32, nullptr, dx, nullptr,
                              x_f32 ? TY_F16 : TY_BF16, dg_attn, W.dg_part, S, d, c->dtype, st);
  }

  // ------------------------------------------------------------ exact fp32
  const int64_t R = S / D;  // rows per virtual rank
  const float* dyf = (const float*)dy;
  const float* ab = (const float*)A.ab;
  float* dab = (float*)W.dab;
  float* dG = (float*)W.dg_f32;
  if ((r = launch_gemm_f32((int)S, I, d, dyf, d, 1, (const float*)mw->w2, 1, I, dG, I, nullptr, 0,
                           0, st)) != TSP_OK)
    return r;
  if ((r = launch_swiglu_bwd_f32(dG, ab, dab, S, I, st)) != TSP_OK) return r;
  for (int rr = 0; rr < D; ++rr) {  // weight grads: sum over the virtual ranks' rows
    const int64_t r0 = rr * R;
    if ((r = launch_gemm_f32(d, I, (int)R, dyf + r0 * d, 1, d, (const float*)A.g + r0 * I, 1, I,
                             dw2, I, nullptr, 0, rr > 0, st)) != TSP_OK)
      return r;
    if ((r = launch_gemm_f32(I, d, (int)R, dab + r0 * 2 * I, 1, 2 * I, (const float*)A.b + r0 * d,
                             1, d, dw1, d, nullptr, 0, rr > 0, st)) != TSP_OK)
      return r;
    if ((r = launch_gemm_f32(I, d, (int)R, dab + r0 * 2 * I + I, 1, 2 * I,
                             (const float*)A.b + r0 * d, 1, d, dw3, d, nullptr, 0, rr > 0, st)) !=
        TSP_OK)
      return r;
  }
  float* db = (float*)W.db;
  if ((r = launch_gemm_f32((int)S, d, I, dab, 2 * I, 1, (const float*)mw->w1, 1, d, db, d, nullptr,
                           0, 0, st)) != TSP_OK)
    return r;
  if ((r = launch_gemm_f32((int)S, d, I, dab + I, 2 * I, 1, (const float*)mw->w3, 1, d, db, d,
                           nullptr, 0, 1, st)) != TSP_OK)
    return r;
  float* dhf = (float*)W.dh_f32;
  if ((r = launch_rmsnorm_bwd(db, A.h, TY_F32, mw->g_mlp, A.rstd2, dyf, nullptr, dhf, nullptr,
                              TY_F32, dg_mlp, W.dg_part, S, d, c->dtype, st)) != TSP_OK)
    return r;
  for (int rr = 0; rr < D; ++rr) {
    const int64_t r0 = rr * R;
    if ((r = launch_gemm_f32(d, d, (int)R, dhf + r0 * d, 1, d, (const float*)A.o + r0 * d, 1, d, dwo,
                             d, nullptr, 0, rr > 0, st)) != TSP_OK)
      return r;
  }
  float* dO = (float*)W.dO;
  if ((r = launch_gemm_f32((int)S, d, d, dhf, d, 1, (const float*)aw->wo, 1, d, dO, d, nullptr, 0, 0,
                           st)) != TSP_OK)
    return r;
  float* dqkv = (float*)W.dqkv;
  if ((r = launch_attn_f32_bwd((const float*)A.qkv, (const float*)A.o, dO, A.lse, W.delta, dqkv, S,
                               H, kv_heads(c), dh, D, st)) != TSP_OK)
    return r;
  if ((r = rope_qk(c, A, dqkv, TY_F32, 1, st)) != TSP_OK) return r;
  float* dws[3] = {dwq, dwk, dwv};
  const float* wts[3] = {(const float*)aw->wq, (const float*)aw->wk, (const float*)aw->wv};
  const int ld = (int)qkv_ld(c), dk = (int)kv_dim(c);
  const int width[3] = {d, dk, dk}, col0[3] = {0, d, d + dk};
  for (int j = 0; j < 3; ++j) {
    for (int rr = 0; rr < D; ++rr) {
      const int64_t r0 = rr * R;
      if ((r = launch_gemm_f32(width[j], d, (int)R, dqkv + r0 * ld + col0[j], 1, ld,
                               (const float*)A.a + r0 * d, 1, d, dws[j], d, nullptr, 0, rr > 0,
                               st)) != TSP_OK)
        return r;
    }
  }
  float* da = (float*)W.da;
  for (int j = 0; j < 3; ++j) {
    if ((r = launch_gemm_f32((int)S, d, width[j], dqkv + col0[j], ld, 1, wts[j], 1, d, da, d,
                             nullptr, 0, j > 0, st)) != TSP_OK)
      return r;
  }
  return launch_rmsnorm_bwd(da, x, TY_F32, aw->g_attn, A.rstd1, dhf, nullptr, dx, nullptr,
                            TY_F32, dg_attn, W.dg_part, S, d, c->dtype, st);
}

}  // namespace tsp

// ----------------------------------------------------------------------------
// Gated-MLP forward for callers that cannot allocate: the scratch is this
// fixed device array instead of a caller workspace.
// ----------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[TSP_NOALLOC_SCRATCH_BYTES];

namespace tsp {
namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.  (In host code the array's name is
// only a host-side stand-in, never a device pointer.)
tsp_status noalloc_scratch(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TSP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return TSP_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = (uint8_t*)g_noalloc_addr[dev];
  return TSP_OK;
}
}  // namespace
}  // namespace tsp

extern "C" tsp_status tsp_gated_mlp_fwd_noalloc(const tsp_cfg* cfg, const void* h_z,
                                                const tsp_mlp_w* w, void* y_z, void* stream) {
  tsp_status r = check_cfg(cfg);
  if (r != TSP_OK) return r;
  if ((r = check_mlp_w(w, false)) != TSP_OK) return r;
  if (!al16(h_z) || !al16(y_z)) return TSP_ERR_INVALID_ARG;
  if ((r = check_bf16_mlp(cfg)) != TSP_OK) return r;
  const size_t need = tsp_workspace_bytes(cfg, TSP_OP_MLP_FWD);
  if (need == 0 || need > (size_t)TSP_NOALLOC_SCRATCH_BYTES) return TSP_ERR_INVALID_ARG;
  uint8_t* scratch = nullptr;
  if ((r = noalloc_scratch(&scratch)) != TSP_OK) return r;
  const int parts = PART_MLP | (cfg->dtype == TSP_F32 ? PART_AB : 0);
  const size_t na = acts_layout(cfg, parts, nullptr).bytes;
  const Acts A = acts_layout(cfg, parts, scratch);
  const WCache WC = wcache_layout(cfg, WC_MLP, scratch + na);
  cudaStream_t st = S_(stream);
  if ((r = fill_wcache(cfg, WC, nullptr, w, st)) != TSP_OK) return r;
  return mlp_half(cfg, h_z, false, w, WC, y_z, false, A, st);
}
