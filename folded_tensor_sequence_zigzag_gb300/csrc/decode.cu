// decode.cu -- inference decode of the TSP-folded block against the zigzag KV cache.
//
// "Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
// Training & Inference", section 2 ("Runtime schedules", attention bullet):
// every rank keeps the K/V of its own zigzag rows.  A decode step of T new
// tokens is HBM-bound: it streams every weight once (a few hundred MB for the
// 7B-shaped block) and the cached K/V of the whole sequence, against only
// 2*T flops per weight.  So its kernels are plain SIMT streaming kernels
// sized for bandwidth, not tensor-core GEMMs:
//
//  * gemv_kernel: y[T, N] = x[T, K] W[N, K]^T with fused epilogues (store,
//    + residual, SiLU(W1 x) * (W3 x), and for Q|K|V the rotary embedding of
//    Q and K plus the append of K|V to the cache).  A warp streams groups of
//    NR output rows, walking K with 16-byte non-allocating loads (four in
//    flight per row); x sits in shared memory.
//  * attention of the new tokens over the cache, in splits of 128 cache rows.
//    The splits never straddle a virtual rank's 2c zigzag rows, so each
//    rank's partial attention over the K/V it owns is formed where that K/V
//    lives (the decode counterpart of the prefill's K/V all-gather); the
//    decoded tokens' own rows, appended after the prompt, form the last
//    splits.  Three kernels:
//    - decode_attn_stream_kernel (fp16 cache, at most 4 query rows per K/V
//      head): one wave of CTAs, each walking a slice of the splits with its
//      warps' rows staged by cp.async three splits deep, the dot products on
//      the tensor cores (mma.sync) and an online softmax;
//    - decode_attn_mma_kernel (fp16 cache, more query rows): a CTA per
//      (K/V head, split), the head group's query rows all in that CTA, so
//      every cache row is read once;
//    - decode_attn_kernel (fp32 cache): a lane per key, K read to registers,
//      V staged by cp.async; the query rows of a K/V head group are split
//      over a few CTAs when the heads and splits alone give too few.
//  * decode_combine_kernel: merges the splits' (max, sum, unnormalised O) by
//    their log-sum-exp into O [T, d].
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace tsp {
namespace {

constexpr int kGemvWarps = 8;
constexpr int kRopeMaxHalf = 64;   // rotary pairs per head the fused Q|K|V epilogue takes (dh <= 128)
constexpr int kAttnWarps = 4;
constexpr int kSplitRows = 32 * kAttnWarps;   // cache rows per attention CTA (a lane per row)
constexpr int kQB = 4;                        // query rows per compute pass

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16 bytes of weights -> floats
template <typename WT> struct WVec;
template <> struct WVec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void cvt(uint4 v, float (&w)[8]) {
    w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
  }
};
template <> struct WVec<float> {
  static constexpr int N = 4;
  __device__ static void cvt(uint4 v, float (&w)[4]) {
    w[0] = __uint_as_float(v.x); w[1] = __uint_as_float(v.y);
    w[2] = __uint_as_float(v.z); w[3] = __uint_as_float(v.w);
  }
};
// 16 bytes of activations (the same element count as WVec) -> floats
template <typename XT> struct XVec;
template <> struct XVec<__half> {
  __device__ static void cvt(uint4 v, float (&x)[8]) {
    x[0] = f16_lo(v.x); x[1] = f16_hi(v.x); x[2] = f16_lo(v.y); x[3] = f16_hi(v.y);
    x[4] = f16_lo(v.z); x[5] = f16_hi(v.z); x[6] = f16_lo(v.w); x[7] = f16_hi(v.w);
  }
};
template <> struct XVec<float> {
  __device__ static void cvt(uint4 v, float (&x)[4]) { WVec<float>::cvt(v, x); }
};

__device__ __forceinline__ float load_any(const void* p, int64_t i, int ty) {
  if (ty == TY_F32) return reinterpret_cast<const float*>(p)[i];
  if (ty == TY_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}
__device__ __forceinline__ void store_any(void* p, int64_t i, int ty, float v) {
  if (ty == TY_F32)
    reinterpret_cast<float*>(p)[i] = v;
  else if (ty == TY_BF16)
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
}

// store_any, recording in `bad` an fp16 value out of fp16 range
__device__ __forceinline__ void store_chk(void* p, int64_t i, int ty, float v, bool& bad) {
  if (ty == TY_F16) bad |= f16_bad(v);
  store_any(p, i, ty, v);
}

struct GemvArgs {
  const void* x;
  int64_t ldx;
  const void* w[3];
  int seg_end[3];   // cumulative rows
  int nseg, N, K, T;
  void* out;
  int64_t ldo;
  int out_ty;
  const void* res;
  int64_t ldr;
  int res_ty;
  // GEMV_QKV: head width, Q+K head count, K|V column start, rotary
  // frequencies and the position of token 0; the cache rows pos0.. receive
  // the K|V columns
  int dh, qk_heads, d, rope;
  int64_t pos0;
  void* kv;
  int64_t ldkv;
  int* status;   // sticky device status word (TSP_ERR_RANGE)
  int64_t kv_rows;   // rows of the cache (the appended rows must fall inside)
  double freq[kRopeMaxHalf];   // base^(-2j/dh), formed on the host in fp64
};

// Output rows n0 .. n0+NR-1 of one warp (GEMV_SWIGLU: outputs n0.., each
// from row n of W1 and row n of W3).
template <typename WT, typename XT, int EPI, int NR>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int VEC = WVec<WT>::N;
  constexpr bool PAIRED = EPI == GEMV_SWIGLU || EPI == GEMV_QKV;
  constexpr int NW = PAIRED ? 2 * NR : NR;   // weight rows per warp
  extern __shared__ __align__(16) uint8_t smem_raw[];
  XT* xs = reinterpret_cast<XT*>(smem_raw);
  const int T = a.T, K = a.K;
  // x [T, K] -> shared memory (16-byte pieces)
  {
    const int per_row = K * (int)sizeof(XT) / 16;
    for (int i = threadIdx.x; i < T * per_row; i += blockDim.x) {
      const int t = i / per_row, v = i - t * per_row;
      const uint4 val = *reinterpret_cast<const uint4*>(
          reinterpret_cast<const uint8_t*>(a.x) + ((int64_t)t * a.ldx * (int64_t)sizeof(XT)) + v * 16);
      reinterpret_cast<uint4*>(xs + (int64_t)t * K)[v] = val;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool bad = false;   // an fp16 output out of range
  // row groups are dealt out grid-stride: every warp streams several groups
  for (int grp = blockIdx.x * kGemvWarps + warp; grp * NR < a.N; grp += gridDim.x * kGemvWarps) {
    const int n0 = grp * NR;
    const WT* rp[NW];
    bool ok[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      int n;
      const WT* base;
      if (EPI == GEMV_SWIGLU) {
        n = n0 + (i >> 1);
        base = reinterpret_cast<const WT*>(a.w[i & 1]);
        ok[i] = n < a.N;
      } else if (EPI == GEMV_QKV) {
        // output pair n0 + (i >> 1) = (head hh, j < dh/2): rows hh*dh + j and + dh/2
        const int half = a.dh >> 1;
        const int pi = n0 + (i >> 1), hh = pi / half, j = pi - hh * half;
        n = hh * a.dh + j + (i & 1) * half;
        ok[i] = pi < a.N;
        int s = 0, lo = 0;
        while (s + 1 < a.nseg && n >= a.seg_end[s]) lo = a.seg_end[s++];
        base = reinterpret_cast<const WT*>(a.w[s]);
        n -= lo;
      } else {
        n = n0 + i;
        ok[i] = n < a.N;
        int s = 0, lo = 0;
        while (s + 1 < a.nseg && n >= a.seg_end[s]) lo = a.seg_end[s++];
        base = reinterpret_cast<const WT*>(a.w[s]);
        n -= lo;
      }
      rp[i] = base + (int64_t)(ok[i] ? n : 0) * K;
    }
    float acc[NW][TSP_DECODE_MAX_T];
#pragma unroll
    for (int i = 0; i < NW; ++i)
#pragma unroll
      for (int t = 0; t < TSP_DECODE_MAX_T; ++t) acc[i][t] = 0.f;
    // U 16-byte loads per weight row are issued before any of them is used,
    // so every warp keeps U * NW * 512 bytes in flight
    constexpr int U = 4, STEP = 32 * VEC;
    auto fma_piece = [&](const uint4 (&wv)[NW], int k) {
      float w[NW][VEC];
#pragma unroll
      for (int i = 0; i < NW; ++i) WVec<WT>::cvt(wv[i], w[i]);
#pragma unroll
      for (int t = 0; t < TSP_DECODE_MAX_T; ++t) {
        if (t < T) {
          float xv[VEC];
          XVec<XT>::cvt(*reinterpret_cast<const uint4*>(xs + (int64_t)t * K + k), xv);
#pragma unroll
          for (int i = 0; i < NW; ++i)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[i][t] = fmaf(w[i][e], xv[e], acc[i][t]);
        }
      }
    };
    int k = lane * VEC;
    for (; k + (U - 1) * STEP < K; k += U * STEP) {
      uint4 wv[U][NW];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < NW; ++i)
          wv[u][i] = ok[i] ? ld_stream(rp[i] + k + u * STEP) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < U; ++u) fma_piece(wv[u], k + u * STEP);
    }
    for (; k < K; k += STEP) {
      uint4 wv[NW];
#pragma unroll
      for (int i = 0; i < NW; ++i) wv[i] = ok[i] ? ld_stream(rp[i] + k) : make_uint4(0u, 0u, 0u, 0u);
      fma_piece(wv, k);
    }
#pragma unroll
    for (int i = 0; i < NW; ++i)
#pragma unroll
      for (int t = 0; t < TSP_DECODE_MAX_T; ++t)
        if (t < T) acc[i][t] = warp_sum(acc[i][t]);
    if (lane == 0) {
      if (EPI == GEMV_QKV) {
        const int half = a.dh >> 1;
#pragma unroll
        for (int jp = 0; jp < NR; ++jp) {
          const int pi = n0 + jp;
          if (pi >= a.N) continue;
          const int hh = pi / half, j = pi - hh * half;
          const int n1 = hh * a.dh + j, n2 = n1 + half;
          const bool rot = a.rope && hh < a.qk_heads;
          // the angle in fp64, reduced modulo 2 pi before the fp32 sine and
          // cosine (an fp32 angle is off by ~0.06 rad at 1M positions)
          const double f = rot ? a.freq[j] : 0.0;
#pragma unroll
          for (int t = 0; t < TSP_DECODE_MAX_T; ++t) {
            if (t >= T) continue;
            float v1 = acc[2 * jp][t], v2 = acc[2 * jp + 1][t];
            if (rot) {
              const double ang = (double)(a.pos0 + t) * f;
              const double two_pi = 6.283185307179586476925287;
              float sv, cv;
              sincosf((float)(ang - two_pi * rint(ang / two_pi)), &sv, &cv);
              const float r1 = v1 * cv - v2 * sv, r2 = v1 * sv + v2 * cv;
              v1 = r1;
              v2 = r2;
            }
            store_chk(a.out, (int64_t)t * a.ldo + n1, a.out_ty, v1, bad);
            store_chk(a.out, (int64_t)t * a.ldo + n2, a.out_ty, v2, bad);
            if (n1 >= a.d &&   // K or V: also the cache row of this token
                TSP_INB(a.pos0 + t >= 0 && a.pos0 + t < a.kv_rows, a.status)) {
              store_chk(a.kv, (a.pos0 + t) * a.ldkv + (n1 - a.d), a.out_ty, v1, bad);
              store_chk(a.kv, (a.pos0 + t) * a.ldkv + (n2 - a.d), a.out_ty, v2, bad);
            }
          }
        }
      } else if (EPI == GEMV_SWIGLU) {
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const int n = n0 + j;
          if (n >= a.N) continue;
#pragma unroll
          for (int t = 0; t < TSP_DECODE_MAX_T; ++t) {
            if (t >= T) continue;
            const float g1 = acc[2 * j][t], g3 = acc[2 * j + 1][t];
            store_chk(a.out, (int64_t)t * a.ldo + n, a.out_ty, g1 * sigmoidf_(g1) * g3, bad);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          const int n = n0 + i;
          if (n >= a.N) continue;
#pragma unroll
          for (int t = 0; t < TSP_DECODE_MAX_T; ++t) {
            if (t >= T) continue;
            float v = acc[i][t];
            if (EPI == GEMV_RES) v += load_any(a.res, (int64_t)t * a.ldr + n, a.res_ty);
            store_chk(a.out, (int64_t)t * a.ldo + n, a.out_ty, v, bad);
          }
        }
      }
    }
  }
  if (bad) report_status(a.status, (int)TSP_ERR_RANGE);
}

template <typename WT, typename XT, int EPI, int NR>
tsp_status gemv_launch(const GemvArgs& ga, const char* name, cudaStream_t st) {
  const size_t smem = (size_t)ga.T * ga.K * sizeof(XT);
  // the dynamic shared memory size this instantiation allows, per device
  static size_t attr[kMaxDevices] = {};
  const int dev = current_device();
  if (smem > 48 * 1024 && smem > attr[dev]) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(gemv_kernel<WT, XT, EPI, NR>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr[dev] = smem;
  }
  const int per_cta = kGemvWarps * NR;
  // a few CTAs per SM, each warp looping over row groups (no partial last wave)
  const int grid = (int)std::min<int64_t>((ga.N + per_cta - 1) / per_cta, 4 * (int64_t)num_sms());
  Prof prof(name, st);
  gemv_kernel<WT, XT, EPI, NR><<<grid, kGemvWarps * 32, smem, st>>>(ga);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

template <typename WT, typename XT, int EPI>
tsp_status gemv_nr(const GemvArgs& ga, const char* name, cudaStream_t st) {
  // two rows a warp halve the shared-memory reads of x per weight byte once
  // several tokens share each weight
  return ga.T > 2 ? gemv_launch<WT, XT, EPI, 2>(ga, name, st)
                  : gemv_launch<WT, XT, EPI, 1>(ga, name, st);
}

template <typename WT, typename XT>
tsp_status gemv_epi(const GemvArgs& ga, int epi, const char* name, cudaStream_t st) {
  switch (epi) {
    case GEMV_QKV: return gemv_nr<WT, XT, GEMV_QKV>(ga, name, st);
    case GEMV_STORE: return gemv_nr<WT, XT, GEMV_STORE>(ga, name, st);
    case GEMV_RES: return gemv_nr<WT, XT, GEMV_RES>(ga, name, st);
    case GEMV_SWIGLU: return gemv_nr<WT, XT, GEMV_SWIGLU>(ga, name, st);
  }
  return TSP_ERR_INVALID_ARG;
}

// ----------------------------------------------------------------------------
// Attention of the new tokens over the cache
// ----------------------------------------------------------------------------

struct AttnArgs {
  CUtensorMap tm;        // streaming kernel: the cache [n_total, ldkv], box {64, 32}, 128B swizzle
  const void* q;
  int64_t ldq;
  const void* kv;
  int64_t ldkv;          // 2 * dkv
  float* part_o;
  float2* part_ml;
  int64_t S, c, n_cached, n_total;
  int D, spr, nsplit, T, H, G, dkv;   // spr: splits per rank
  int nz, qpc;   // query-row groups per (K/V head, split); query rows per group
  int nslice;    // streaming kernel: CTAs per K/V head, each over a slice of the splits
  float scale_log2;
  int* status;   // sticky device status word (checked build: TSP_ERR_BOUNDS)
  uint64_t limit_ns;   // bound of one wait (streaming kernel)
};

// cache rows [r0, r1) of split `s`: splits 0 .. D*spr-1 cut each rank's 2c
// zigzag rows into pieces of kSplitRows; the rest cut the decoded rows [S, n_total).
__device__ __forceinline__ void split_rows(const AttnArgs& a, int s, int64_t& r0, int64_t& r1) {
  const int prompt_splits = a.D * a.spr;
  if (s < prompt_splits) {
    const int r = s / a.spr, j = s - r * a.spr;
    const int64_t rank0 = (int64_t)r * 2 * a.c, rank1 = rank0 + 2 * a.c;
    r0 = rank0 + (int64_t)j * kSplitRows;
    r1 = min(r0 + kSplitRows, rank1);
  } else {
    r0 = a.S + (int64_t)(s - prompt_splits) * kSplitRows;
    r1 = min(r0 + kSplitRows, a.n_total);
  }
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// V elements one lane holds for one key: VPL of type CT
template <typename CT, int VPL> struct VReg;
template <> struct VReg<float, 2> {
  float2 r;
  __device__ void load(const float* p) { r = *reinterpret_cast<const float2*>(p); }
  __device__ void zero() { r = make_float2(0.f, 0.f); }
  __device__ void get(float (&v)[2]) const { v[0] = r.x; v[1] = r.y; }
};
template <> struct VReg<float, 1> {
  float r;
  __device__ void load(const float* p) { r = *p; }
  __device__ void zero() { r = 0.f; }
  __device__ void get(float (&v)[1]) const { v[0] = r; }
};

// CTA = (K/V head g, split s of <= 128 cache rows, query group z); warp w
// takes rows r0 + 32w .. r0 + 32w + 31.  Every lane issues its K pieces and
// its V columns of the warp's 32 keys before any arithmetic, so a warp has
// 16 KB of loads in flight, all coalesced: a K row is read by LPR lanes
// (16 bytes each) and its dot products reduced across them; a V row by the
// whole warp.  No shared-memory staging of K/V; the warps' partial softmax
// results are merged in shared memory.
template <typename CT, int DH>
__global__ void __launch_bounds__(kAttnWarps * 32, 4) decode_attn_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int E = 16 / sizeof(CT);          // elements per 16-byte piece
  constexpr int LPR = DH / E;                 // lanes per K row (a piece each)
  constexpr int RPI = 32 / LPR;               // K rows per warp-wide load
  constexpr int KIT = LPR;                    // loads covering the warp's 32 rows
  constexpr int VPL = DH >= 32 ? DH / 32 : 1; // V columns per lane
  constexpr int VLANES = DH / VPL;            // lanes holding V columns
  __shared__ __align__(16) float qs[kQB][DH];
  __shared__ __align__(16) float pw[kAttnWarps][kQB][32];
  __shared__ __align__(16) float ro[kAttnWarps][kQB][DH];
  __shared__ __align__(16) CT vs[kAttnWarps][32][DH];   // each warp's V rows (cp.async)
  __shared__ float2 rml[kAttnWarps][kQB];

  // the nz CTAs of one (K/V head, split) are neighbours in x: they run
  // together and share the K/V rows through L2
  const int g = blockIdx.x / a.nz, z = blockIdx.x - g * a.nz, s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t r0, r1;
  split_rows(a, s, r0, r1);
  const bool rows_in = TSP_INB(r0 >= 0 && r0 <= r1 && r1 <= a.n_total, a.status);
  const int64_t wr0 = r0 + warp * 32;
  const bool wactive = rows_in && wr0 < r1;
  const int64_t kr = wr0 + lane;              // this lane's key row
  const bool kin = rows_in && kr < r1;
  const CT* base = reinterpret_cast<const CT*>(a.kv) + (int64_t)g * DH;

  const int kl = lane % LPR, kh = lane / LPR;   // piece and row of this lane in a K load
  uint4 kreg[KIT];
  if (wactive) {
#pragma unroll
    for (int it = 0; it < KIT; ++it) {
      const int64_t row = wr0 + it * RPI + kh;
      kreg[it] = ld_nc16(base + (row < r1 ? row : r0) * a.ldkv + kl * E);
    }
    // V rows -> this warp's shared-memory slice without holding registers;
    // rows past the split read as zeros (their p is 0)
    for (int i = lane; i < 32 * LPR; i += 32) {
      const int k = i / LPR, pc = i - k * LPR;
      const bool in = wr0 + k < r1;
      cp_async16(smem_u32(&vs[warp][k][pc * E]), base + (in ? wr0 + k : r0) * a.ldkv + a.dkv + pc * E,
                 in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  bool v_ready = false;

  // query rows of this K/V head: qr = (head g*G + gi, token t), gi = qr / T;
  // this CTA takes rows [z*qpc, min(QR, (z+1)*qpc))
  const int QR = min(a.G * a.T, (z + 1) * a.qpc);
  for (int qb = z * a.qpc; qb < QR; qb += kQB) {
    const int nq = min(kQB, QR - qb);
    for (int idx = threadIdx.x; idx < kQB * DH; idx += kAttnWarps * 32) {
      const int i = idx / DH, j = idx - i * DH;
      float v = 0.f;
      if (i < nq) {
        const int qr = qb + i, gi = qr / a.T, t = qr - gi * a.T;
        v = to_f(reinterpret_cast<const CT*>(a.q)[(int64_t)t * a.ldq + (g * a.G + gi) * DH + j]);
      }
      qs[i][j] = v;
    }
    __syncthreads();
    if (wactive) {
      // sc[i] = q_i . K[row wr0 + lane]: per load, partial dot products over
      // each row's LPR lanes, reduced, then handed to the lane that owns the row
      float sc[kQB];
#pragma unroll
      for (int i = 0; i < kQB; ++i) sc[i] = 0.f;
#pragma unroll
      for (int i = 0; i < kQB; ++i) {
        if (i < nq) {
          float qv[E];
#pragma unroll
          for (int e = 0; e < E; ++e) qv[e] = qs[i][kl * E + e];
#pragma unroll
          for (int it = 0; it < KIT; ++it) {
            float kf[E];
            if constexpr (sizeof(CT) == 2) {
              XVec<__half>::cvt(kreg[it], *reinterpret_cast<float(*)[8]>(kf));
            } else {
              XVec<float>::cvt(kreg[it], *reinterpret_cast<float(*)[4]>(kf));
            }
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) part = fmaf(qv[e], kf[e], part);
#pragma unroll
            for (int off = LPR / 2; off >= 1; off >>= 1)
              part += __shfl_xor_sync(0xffffffffu, part, off);
            // row it*RPI + h sits in lanes h*LPR ..; lane j owns row j
            const float v = __shfl_sync(0xffffffffu, part, (lane % RPI) * LPR);
            if (lane / RPI == it) sc[i] = v;
          }
        }
      }
      // softmax pieces over the warp's 32 keys
#pragma unroll
      for (int i = 0; i < kQB; ++i) {
        if (i < nq) {
          const int t = (qb + i) % a.T;
          // prompt rows precede every new token; a new row is visible to the
          // tokens at or after its own position
          const bool vis = kin && (kr < a.S || kr <= a.n_cached + t);
          const float x = vis ? sc[i] * a.scale_log2 : -INFINITY;
          const float m = warp_max(x);
          const float p = m == -INFINITY ? 0.f : exp2f(x - m);
          const float l = warp_sum(p);
          pw[warp][i][lane] = p;
          if (lane == 0) rml[warp][i] = make_float2(m, l);
        }
      }
      if (!v_ready) {   // this lane's V copies, then the whole warp's, are in place
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        v_ready = true;
      }
      __syncwarp();
      // O piece = P V over the warp's keys: lane = V columns
      float o[kQB][VPL];
#pragma unroll
      for (int i = 0; i < kQB; ++i)
#pragma unroll
        for (int v = 0; v < VPL; ++v) o[i][v] = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 32; k4 += 4) {
        float vf[4][VPL];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          VReg<CT, VPL> vr;
          if (lane < VLANES)
            vr.load(&vs[warp][k4 + kk][lane * VPL]);
          else
            vr.zero();
          vr.get(vf[kk]);
        }
#pragma unroll
        for (int i = 0; i < kQB; ++i) {
          if (i < nq) {
            const float4 p4 = *reinterpret_cast<const float4*>(&pw[warp][i][k4]);
            const float pk[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int v = 0; v < VPL; ++v) o[i][v] = fmaf(pk[kk], vf[kk][v], o[i][v]);
          }
        }
      }
      if (lane < VLANES) {
#pragma unroll
        for (int i = 0; i < kQB; ++i)
          if (i < nq)
#pragma unroll
            for (int v = 0; v < VPL; ++v) ro[warp][i][lane * VPL + v] = o[i][v];
      }
    } else if (lane < kQB) {
      rml[warp][lane] = make_float2(-INFINITY, 0.f);   // no rows: no contribution
    }
    __syncthreads();
    // merge the warps: M = max m_w, O = sum 2^(m_w - M) o_w, L likewise
    for (int idx = threadIdx.x; idx < nq * DH; idx += kAttnWarps * 32) {
      const int i = idx / DH, j = idx - i * DH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, rml[w][i].x);
      float O = 0.f, L = 0.f;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float2 ml = rml[w][i];
        const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
        O = fmaf(sc, ml.x == -INFINITY ? 0.f : ro[w][i][j], O);
        L = fmaf(sc, ml.y, L);
      }
      const int qr = qb + i, gi = qr / a.T, t = qr - gi * a.T;
      const int64_t slot = ((int64_t)s * a.H + g * a.G + gi) * a.T + t;
      if (!TSP_INB(slot >= 0 && slot < (int64_t)a.nsplit * a.H * a.T, a.status)) continue;
      a.part_o[slot * DH + j] = O;
      if (j == 0) a.part_ml[slot] = make_float2(M, L);
    }
    __syncthreads();
  }
}

// ---- the fp16 kernel: dot products and P V on the tensor cores (mma.sync) ----
//
// CTA = (K/V head g, split s of <= 128 cache rows, query group z), warp w takes
// rows 32w .. 32w+31 as above.  The warp stages its K and V rows in its
// shared-memory slice by cp.async (the 16-byte pieces of row r swizzled by
// r mod 8, so the 8x8 matrix loads hit distinct banks without padding, and
// three CTAs fit an SM), then for each pass of up to kQB query rows (the
// MMA's other rows read one shared zero row) computes S = Q K^T over its 32 keys
// with m16n8k16 MMAs (fp16 in, fp32 accumulate), the softmax pieces on the
// accumulator fragments, and O = P V with P taken straight from those
// fragments as the A operand.  A cache row costs a few tensor-core
// instructions instead of the scalar dot products and lane shuffles of the
// fp32 kernel, so the CTA's time is its loads.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A B + C, m16n8k16, A row-major fp16, B column-major fp16, fp32 C/D
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int DH>
struct MmaSmem {
  static constexpr int RB = DH * 2;                       // bytes per staged row
  static constexpr int WARP_BYTES = 2 * 32 * RB;          // a warp's K rows, then its V rows
  static constexpr int Q_BYTES = (kQB + 1) * RB;          // kQB query rows and a zero row
  static constexpr int BYTES = kAttnWarps * WARP_BYTES + Q_BYTES;
  // byte offset of 16-byte piece `c` of staged row `r`
  static __device__ __forceinline__ uint32_t at(int r, int c) {
    return (uint32_t)(r * RB + ((c ^ (r & 7)) << 4));
  }
};

template <int DH>
__global__ void __launch_bounds__(kAttnWarps * 32, 3) decode_attn_mma_kernel(const __grid_constant__ AttnArgs a) {
  using L = MmaSmem<DH>;
  constexpr int CPR = DH * 2 / 16;              // 16-byte pieces per K (or V) row
  constexpr int NT = DH / 8;                    // n8 tiles of O (dh)
  extern __shared__ __align__(16) uint8_t mma_smem[];
  __shared__ __align__(16) float ro[kAttnWarps][kQB][DH];
  __shared__ float2 rml[kAttnWarps][kQB];

  const int g = blockIdx.x / a.nz, z = blockIdx.x - g * a.nz, s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;      // MMA fragment row group and thread in it
  int64_t r0, r1;
  split_rows(a, s, r0, r1);
  const bool rows_in = TSP_INB(r0 >= 0 && r0 <= r1 && r1 <= a.n_total, a.status);
  const int64_t wr0 = r0 + warp * 32;
  const bool wactive = rows_in && wr0 < r1;
  const __half* base = reinterpret_cast<const __half*>(a.kv) + (int64_t)g * DH;
  const uint32_t ks = smem_u32(mma_smem) + (uint32_t)(warp * L::WARP_BYTES);   // K rows
  const uint32_t vs = ks + 32 * L::RB;                                          // V rows
  const uint32_t qsm = smem_u32(mma_smem) + (uint32_t)(kAttnWarps * L::WARP_BYTES);
  __half* qh = reinterpret_cast<__half*>(mma_smem + kAttnWarps * L::WARP_BYTES);

  if (wactive) {
    // K and V rows of the warp -> its slice; rows past the split read as zeros
    for (int i = lane; i < 2 * 32 * CPR; i += 32) {
      const int kv = i / (32 * CPR), k = (i / CPR) & 31, pc = i % CPR;
      const bool in = wr0 + k < r1;
      cp_async16(ks + (uint32_t)(kv * 32 * L::RB) + L::at(k, pc),
                 base + (in ? wr0 + k : r0) * a.ldkv + kv * a.dkv + pc * 8, in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  bool kv_ready = false;

  const int QR = min(a.G * a.T, (z + 1) * a.qpc);
  for (int qb = z * a.qpc; qb < QR; qb += kQB) {
    const int nq = min(kQB, QR - qb);
    // query rows qb .. qb+nq-1 into staged rows 0..nq-1; rows nq..kQB are zero
    // (row kQB stands in for the MMA's rows kQB..15)
    for (int idx = threadIdx.x; idx < (kQB + 1) * (DH / 8); idx += kAttnWarps * 32) {
      const int i = idx / (DH / 8), pc = idx - i * (DH / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (i < nq) {
        const int qr = qb + i, gi = qr / a.T, t = qr - gi * a.T;
        v = *reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(a.q) +
                                            (int64_t)t * a.ldq + (g * a.G + gi) * DH + pc * 8);
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(qh) + L::at(i, pc)) = v;
    }
    __syncthreads();
    if (wactive) {
      if (!kv_ready) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();
        kv_ready = true;
      }
      // S[16 query rows x 32 keys] = Q K^T: four n8 tiles of keys, DH/16 k-steps
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        uint32_t qa[4];
        const int qrow = (lane & 15) < kQB ? (lane & 15) : kQB;
        ldsm_x4(qsm + L::at(qrow, 2 * kk + (lane >> 4)), qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
        for (int nt = 0; nt < 4; nt += 2) {
          // matrices: (keys nt*8.., dh lo), (nt*8.., dh hi), ((nt+1)*8.., lo), ((nt+1)*8.., hi)
          const int m = lane >> 3;
          const uint32_t addr = ks + L::at((nt + (m >> 1)) * 8 + (lane & 7), 2 * kk + (m & 1));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma16816(sc[nt], qa, b0, b1);
          mma16816(sc[nt + 1], qa, b2, b3);
        }
      }
      // softmax pieces of rows gq (sc[.][0..1]) over the warp's keys nt*8 + 2 tq + {0, 1};
      // rows gq + 8 (sc[.][2..3]) are padding
      const int t_row = (qb + gq) % a.T;
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t kr = wr0 + nt * 8 + 2 * tq + e;
          // prompt rows precede every new token; a new row is visible to the
          // tokens at or after its own position
          const bool vis = kr < r1 && (kr < a.S || kr <= a.n_cached + t_row);
          sc[nt][e] = vis ? sc[nt][e] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[nt][e]);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      float l = 0.f;
      uint32_t pa[2][4];   // P as the A operand of P V: k-steps of 16 keys
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float p0 = mx == -INFINITY ? 0.f : exp2f(sc[nt][0] - mx);
        const float p1 = mx == -INFINITY ? 0.f : exp2f(sc[nt][1] - mx);
        l += p0 + p1;
        pa[nt >> 1][(nt & 1) * 2] = pack_f16(p0, p1);   // rows gq: a0 (keys lo) / a2 (keys hi)
        pa[nt >> 1][(nt & 1) * 2 + 1] = 0u;             // rows gq + 8: padding
      }
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      // O[16 x DH] = P V: V read transposed (k = keys, n = dh)
      float o[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
          // matrices: (keys kk*16 + 0..7, dh nt*8..), (keys +8..15, nt), (0..7, nt+1), (8..15, nt+1)
          const int m = lane >> 3;
          const uint32_t addr = vs + L::at(kk * 16 + (m & 1) * 8 + (lane & 7), nt + (m >> 1));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma16816(o[nt], pa[kk], b0, b1);
          mma16816(o[nt + 1], pa[kk], b2, b3);
        }
      }
      if (gq < nq) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          *reinterpret_cast<float2*>(&ro[warp][gq][nt * 8 + 2 * tq]) = make_float2(o[nt][0], o[nt][1]);
        if (tq == 0) rml[warp][gq] = make_float2(mx, l);
      }
    } else if (lane < kQB) {
      rml[warp][lane] = make_float2(-INFINITY, 0.f);   // no rows: no contribution
    }
    __syncthreads();
    // merge the warps: M = max m_w, O = sum 2^(m_w - M) o_w, L likewise
    for (int idx = threadIdx.x; idx < nq * DH; idx += kAttnWarps * 32) {
      const int i = idx / DH, j = idx - i * DH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, rml[w][i].x);
      float O = 0.f, L2 = 0.f;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float2 ml = rml[w][i];
        const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
        O = fmaf(sc, ml.x == -INFINITY ? 0.f : ro[w][i][j], O);
        L2 = fmaf(sc, ml.y, L2);
      }
      const int qr = qb + i, gi = qr / a.T, t = qr - gi * a.T;
      const int64_t slot = ((int64_t)s * a.H + g * a.G + gi) * a.T + t;
      if (!TSP_INB(slot >= 0 && slot < (int64_t)a.nsplit * a.H * a.T, a.status)) continue;
      a.part_o[slot * DH + j] = O;
      if (j == 0) a.part_ml[slot] = make_float2(M, L2);
    }
    __syncthreads();
  }
}

// Streaming variant for at most kQB query rows per K/V head (one decoded
// token, or a few with grouped heads): the grid is one wave, nslice CTAs per
// K/V head (a CTA an SM), and CTA p walks the splits
// [p*nsplit/nslice, (p+1)*nsplit/nslice).  Each warp takes its 32 rows of
// every split in turn through a ring of kStreamStages shared-memory stages
// that one lane fills with tensor copies (TMA: 64-column boxes of 32 rows,
// 128-byte swizzle, an mbarrier a stage), kStreamStages - 1 splits ahead of
// the one its MMAs work on, and keeps a running (max, sum, O) per query row
// -- the online softmax of the flash-attention forward.  The cache streams
// without CTAs starting and ending in waves, and a warp spends no issue slots
// on copy addresses.  Every CTA writes one partial per query row; the combine
// kernel merges the nslice partials.
constexpr int kStreamStages = 3;
template <int DH>
struct StreamSmem {
  static constexpr int BOX_BYTES = 32 * 128;                  // 32 rows x 64 fp16 columns
  static constexpr int KV_BYTES = (DH / 64) * BOX_BYTES;      // a warp's K (or V) rows
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;            // K boxes, then V boxes
  static constexpr int WARP_BYTES = kStreamStages * STAGE_BYTES;
  static constexpr int OFF_Q = kAttnWarps * WARP_BYTES;       // staged query rows (MmaSmem layout)
  static constexpr int OFF_BAR = OFF_Q + MmaSmem<DH>::Q_BYTES;
  static constexpr int BYTES = OFF_BAR + kAttnWarps * kStreamStages * 8 + 1024;  // + alignment
  // byte offset of 16-byte piece c (of DH/8) of staged row r in a K or V part
  static __device__ __forceinline__ uint32_t at(int r, int c) {
    return (uint32_t)((c >> 3) * BOX_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }
};

// Waits for phase `parity` of a stage's barrier for at most limit_ns; on
// time-out records TSP_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, int* status,
                                           uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) {
      report_timeout(status);
      return false;
    }
  }
  return true;
}

template <int DH>
__global__ void __launch_bounds__(kAttnWarps * 32, 1)
    decode_attn_stream_kernel(const __grid_constant__ AttnArgs a) {
  using L = MmaSmem<DH>;
  using SL = StreamSmem<DH>;
  constexpr int NT = DH / 8;                    // n8 tiles of O (dh)
  extern __shared__ __align__(16) uint8_t mma_smem[];
  __shared__ __align__(16) float ro[kAttnWarps][kQB][DH];
  __shared__ float2 rml[kAttnWarps][kQB];

  const int g = blockIdx.x, p = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;      // MMA fragment row group and thread in it
  const int s_lo = (int)((int64_t)p * a.nsplit / a.nslice);
  const int s_hi = (int)((int64_t)(p + 1) * a.nsplit / a.nslice);
  const int nq = a.G * a.T;                     // <= kQB (host-checked)
  // the 128-byte swizzle repeats every 1024 bytes: boxes start on that boundary
  const uint32_t raw = smem_u32(mma_smem);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = mma_smem + (sbase - raw);
  const uint32_t wsm = sbase + (uint32_t)(warp * SL::WARP_BYTES);
  const uint32_t qsm = sbase + (uint32_t)SL::OFF_Q;
  const uint32_t wbar = sbase + (uint32_t)SL::OFF_BAR + (uint32_t)(warp * kStreamStages * 8);
  if (lane == 0) {
    for (int st = 0; st < kStreamStages; ++st) mbar_init(wbar + 8u * st, 1);
    fence_barrier_init();
  }
  __syncwarp();

  // split cursors: (s, rank, piece) walked forward one split at a time, so
  // the rows of a split cost no division; a warp with no rows in a split
  // neither loads nor waits for it
  struct Cur {
    int s, r, j;
  };
  auto start = [&](int s) {
    Cur c{s, a.D, 0};
    if (s < a.D * a.spr) {
      c.r = s / a.spr;
      c.j = s - c.r * a.spr;
    }
    return c;
  };
  auto next = [&](Cur& c) {
    ++c.s;
    if (c.r < a.D && ++c.j == a.spr) {
      c.j = 0;
      ++c.r;
    }
  };
  auto rows_of = [&](const Cur& c, int64_t& r0, int64_t& r1) -> bool {
    if (c.r < a.D) {
      const int64_t rank0 = (int64_t)c.r * 2 * a.c;
      r0 = rank0 + (int64_t)c.j * kSplitRows;
      r1 = min(r0 + kSplitRows, rank0 + 2 * a.c);
    } else {
      r0 = a.S + (int64_t)(c.s - a.D * a.spr) * kSplitRows;
      r1 = min(r0 + kSplitRows, a.n_total);
    }
    return c.s < s_hi && TSP_INB(r0 >= 0 && r0 <= r1 && r1 <= a.n_total, a.status) &&
           r0 + warp * 32 < r1;
  };
  uint32_t pending = 0;   // bit st: stage st has a fill not yet waited for
  auto load = [&](const Cur& c, int stage) {
    int64_t r0, r1;
    if (!rows_of(c, r0, r1)) return;
    pending |= 1u << stage;
    if (lane != 0) return;
    const uint32_t dst = wsm + (uint32_t)(stage * SL::STAGE_BYTES), bar = wbar + 8u * stage;
    const int y = (int)(r0 + warp * 32);        // rows past the cache read as zeros
    mbar_arrive_expect_tx(bar, (uint32_t)SL::STAGE_BYTES);
#pragma unroll
    for (int kv = 0; kv < 2; ++kv)
#pragma unroll
      for (int b = 0; b < DH / 64; ++b)
        tma_load_2d(dst + (uint32_t)(kv * SL::KV_BYTES + b * SL::BOX_BYTES), &a.tm,
                    kv * a.dkv + g * DH + b * 64, y, bar);
  };
  Cur cl = start(s_lo);   // next split to load
#pragma unroll
  for (int i = 0; i < kStreamStages - 1; ++i) {
    load(cl, i);
    next(cl);
  }

  // the query rows into staged rows 0..nq-1; rows nq..kQB are zero (row kQB
  // stands in for the MMA's rows kQB..15)
  uint8_t* qh = gbase + SL::OFF_Q;
  for (int idx = threadIdx.x; idx < (kQB + 1) * (DH / 8); idx += kAttnWarps * 32) {
    const int i = idx / (DH / 8), pc = idx - i * (DH / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (i < nq) {
      const int gi = i / a.T, t = i - gi * a.T;
      v = *reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(a.q) +
                                          (int64_t)t * a.ldq + (g * a.G + gi) * DH + pc * 8);
    }
    *reinterpret_cast<uint4*>(qh + L::at(i, pc)) = v;
  }
  __syncthreads();
  // the query fragments (A operand of S = Q K^T), the same for every split
  uint32_t qa[DH / 16][4];
  {
    const int qrow = (lane & 15) < kQB ? (lane & 15) : kQB;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk)
      ldsm_x4(qsm + L::at(qrow, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  const int t_row = gq % a.T;                   // token of fragment row gq (rows >= nq unused)
  const int64_t new_lim = a.n_cached + t_row + 1;   // decoded rows row gq may see: below this
  float m_run = -INFINITY, l_run = 0.f;         // row gq's running max (log2 units) and sum
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  uint32_t phase = 0;     // bit st: parity of stage st's next fill
  bool ok = true;         // false after a timed-out wait (warp-uniform)

  Cur cc = start(s_lo);   // split consumed
  for (int it = 0; cc.s < s_hi; ++it, next(cc)) {
    if (ok) {
      load(cl, (it + kStreamStages - 1) % kStreamStages);
      next(cl);
    }
    int64_t r0, r1;
    if (!rows_of(cc, r0, r1)) continue;         // warp-uniform
    const int st = it % kStreamStages;
    if (ok) {
      ok = __all_sync(0xffffffffu, stage_wait(wbar + 8u * st, (phase >> st) & 1u, a.status,
                                              a.limit_ns));
      if (ok) {
        phase ^= 1u << st;
        pending &= ~(1u << st);
      }
    }
    if (!ok) continue;
    const int64_t wr0 = r0 + warp * 32;
    // keys wr0 + k with k < vis_n are visible to row gq: prompt rows below r1;
    // decoded rows also at or before the row's own position
    const int64_t lim = r0 >= a.S ? min(r1, new_lim) : r1;
    const int vis_n = (int)max((int64_t)0, min((int64_t)32, lim - wr0));
    const uint32_t ks = wsm + (uint32_t)(st * SL::STAGE_BYTES);
    const uint32_t vs = ks + (uint32_t)SL::KV_BYTES;
    // S[16 query rows x 32 keys] = Q K^T: four n8 tiles of keys, DH/16 k-steps
    float sc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
      for (int nt = 0; nt < 4; nt += 2) {
        const int m = lane >> 3;
        const uint32_t addr = ks + SL::at((nt + (m >> 1)) * 8 + (lane & 7), 2 * kk + (m & 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma16816(sc[nt], qa[kk], b0, b1);
        mma16816(sc[nt + 1], qa[kk], b2, b3);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[nt][e] = nt * 8 + 2 * tq + e < vis_n ? sc[nt][e] * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sc[nt][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    // the earlier rows' share 2^(m_run - m_new); nothing seen yet -> O and l are 0
    const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
    float l = 0.f;
    uint32_t pa[2][4];   // P as the A operand of P V: k-steps of 16 keys
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = m_new == -INFINITY ? 0.f : exp2f(sc[nt][0] - m_new);
      const float p1 = m_new == -INFINITY ? 0.f : exp2f(sc[nt][1] - m_new);
      l += p0 + p1;
      pa[nt >> 1][(nt & 1) * 2] = pack_f16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = 0u;
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l_run = fmaf(l_run, alpha, l);
    m_run = m_new;
    if (__any_sync(0xffffffffu, alpha != 1.f)) {   // O rescaled only when a max grew
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] *= alpha;
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        const int m = lane >> 3;
        const uint32_t addr = vs + SL::at(kk * 16 + (m & 1) * 8 + (lane & 7), nt + (m >> 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma16816(o[nt], pa[kk], b0, b1);
        mma16816(o[nt + 1], pa[kk], b2, b3);
      }
    }
    __syncwarp();   // the stage just read is refilled by a later iteration's load
  }
  // after a wait ran out (the status word carries the error and the merge
  // below still runs), wait -- bounded again -- for the copies in flight
#pragma unroll
  for (int st = 0; st < kStreamStages; ++st)
    if (pending & (1u << st)) (void)stage_wait(wbar + 8u * st, (phase >> st) & 1u, a.status, a.limit_ns);

  if (gq < nq) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float2*>(&ro[warp][gq][nt * 8 + 2 * tq]) = make_float2(o[nt][0], o[nt][1]);
    if (tq == 0) rml[warp][gq] = make_float2(m_run, l_run);
  }
  __syncthreads();
  // merge the warps: M = max m_w, O = sum 2^(m_w - M) o_w, L likewise
  for (int idx = threadIdx.x; idx < nq * DH; idx += kAttnWarps * 32) {
    const int i = idx / DH, j = idx - i * DH;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, rml[w][i].x);
    float O = 0.f, L2 = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float2 ml = rml[w][i];
      const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
      O = fmaf(sc, ml.x == -INFINITY ? 0.f : ro[w][i][j], O);
      L2 = fmaf(sc, ml.y, L2);
    }
    const int gi = i / a.T, t = i - gi * a.T;
    const int64_t slot = ((int64_t)p * a.H + g * a.G + gi) * a.T + t;
    if (!TSP_INB(slot >= 0 && slot < (int64_t)a.nslice * a.H * a.T, a.status)) continue;
    a.part_o[slot * DH + j] = O;
    if (j == 0) a.part_ml[slot] = make_float2(M, L2);
  }
}

// CTA per (head, token): the maxima first (lane-parallel loads), then warp w
// adds splits w, w + 8, ... with no branch between its loads; the warps merge
// in shared memory:  O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
constexpr int kCombineWarps = 8;
template <typename CT>
__global__ void __launch_bounds__(kCombineWarps * 32)
    decode_combine_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                          CT* __restrict__ o, int nsplit, int H, int T, int dh) {
  __shared__ float acc_s[kCombineWarps][128];
  __shared__ float red[kCombineWarps];
  const int ht = blockIdx.x, h = ht / T, t = ht - h * T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int s = threadIdx.x; s < nsplit; s += kCombineWarps * 32)
    M = fmaxf(M, part_ml[((int64_t)s * H + h) * T + t].x);
  M = warp_max(M);
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, red[w]);
  __syncthreads();   // red is reused for the sums below
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
#pragma unroll 8
  for (int s = warp; s < nsplit; s += kCombineWarps) {
    const int64_t idx = ((int64_t)s * H + h) * T + t;
    const float2 ml = part_ml[idx];
    const float* po = part_o + idx * dh;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = lane + 32 * i < dh ? po[lane + 32 * i] : 0.f;
    // a split with no visible row (m = -inf) adds nothing
    const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
    L = fmaf(sc, ml.y, L);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf(sc, v[i], acc[i]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc_s[warp][lane + 32 * i] = acc[i];
  if (lane == 0) red[warp] = L;
  __syncthreads();
  if (threadIdx.x < dh) {
    float sum = 0.f, lt = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      sum += acc_s[w][threadIdx.x];
      lt += red[w];
    }
    o[(int64_t)t * H * dh + h * dh + threadIdx.x] = from_f<CT>(sum / lt);
  }
}

template <int DH>
tsp_status decode_attn_mma(const AttnArgs& aa, cudaStream_t st) {
  const size_t smem = MmaSmem<DH>::BYTES;
  static bool attr[kMaxDevices] = {};   // the attribute holds for one device
  const int dev = current_device();
  if (!attr[dev]) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(decode_attn_mma_kernel<DH>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr[dev] = true;
  }
  Prof prof("decode_attn", st);
  // the K/V head varies fastest: CTAs running together read whole cache rows
  dim3 grid((unsigned)(aa.H / aa.G * aa.nz), (unsigned)aa.nsplit);
  decode_attn_mma_kernel<DH><<<grid, kAttnWarps * 32, smem, st>>>(aa);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

template <int DH>
tsp_status decode_attn_stream(const AttnArgs& aa, cudaStream_t st) {
  const size_t smem = StreamSmem<DH>::BYTES;
  static bool attr[kMaxDevices] = {};   // the attribute holds for one device
  const int dev = current_device();
  if (!attr[dev]) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(decode_attn_stream_kernel<DH>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr[dev] = true;
  }
  Prof prof("decode_attn", st);
  dim3 grid((unsigned)(aa.H / aa.G), (unsigned)aa.nslice);
  decode_attn_stream_kernel<DH><<<grid, kAttnWarps * 32, smem, st>>>(aa);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

template <typename CT, int DH>
tsp_status decode_attn_t(const AttnArgs& aa, cudaStream_t st) {
  Prof prof("decode_attn", st);
  // the K/V head varies fastest: CTAs running together read whole cache rows
  dim3 grid((unsigned)(aa.H / aa.G * aa.nz), (unsigned)aa.nsplit);
  decode_attn_kernel<CT, DH><<<grid, kAttnWarps * 32, 0, st>>>(aa);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace

tsp_status launch_gemv(const Gemv& g, cudaStream_t st) {
  if (g.T < 1 || g.T > TSP_DECODE_MAX_T || g.K <= 0 || g.nseg < 1 || g.nseg > 3)
    return TSP_ERR_INVALID_ARG;
  const bool bf = g.dtype == TSP_BF16;
  const int xsz = bf ? 2 : 4;
  // 16-byte pieces of every weight row and every x row
  if ((g.K * xsz) % 16 != 0) return TSP_ERR_UNSUPPORTED;
  if ((g.ldx * xsz) % 16 != 0 || ((uintptr_t)g.x & 15u)) return TSP_ERR_UNSUPPORTED;
  if ((size_t)g.T * g.K * xsz > 200 * 1024) return TSP_ERR_UNSUPPORTED;
  GemvArgs ga;
  memset(&ga, 0, sizeof(ga));
  ga.status = status_word();
  ga.x = g.x;
  ga.ldx = g.ldx;
  int n = 0;
  const int nseg = g.epi == GEMV_SWIGLU ? 2 : g.nseg;
  for (int s = 0; s < nseg; ++s) {
    if (!g.w[s] || ((uintptr_t)g.w[s] & 15u)) return TSP_ERR_INVALID_ARG;
    ga.w[s] = g.w[s];
    n += g.epi == GEMV_SWIGLU ? 0 : g.rows[s];
    ga.seg_end[s] = n;
  }
  ga.nseg = nseg;
  ga.N = g.epi == GEMV_SWIGLU ? g.rows[0] : g.epi == GEMV_QKV ? n / 2 : n;
  if (g.epi == GEMV_QKV && (g.dh < 2 || g.dh % 2 != 0 || n % g.dh != 0)) return TSP_ERR_INVALID_ARG;
  ga.dh = g.dh;
  ga.qk_heads = g.qk_heads;
  ga.d = g.d;
  ga.pos0 = g.pos0;
  if (g.epi == GEMV_QKV && g.rope_base > 0.f) {
    if (g.dh / 2 > kRopeMaxHalf) return TSP_ERR_UNSUPPORTED;
    ga.rope = 1;
    for (int j = 0; j < g.dh / 2; ++j)
      ga.freq[j] = std::pow((double)g.rope_base, -2.0 * j / (double)g.dh);
  }
  ga.kv = g.kv;
  ga.ldkv = g.ldkv;
  ga.kv_rows = g.kv_rows;
  ga.K = g.K;
  ga.T = g.T;
  ga.out = g.out;
  ga.ldo = g.ldo;
  ga.out_ty = g.out_ty;
  ga.res = g.res;
  ga.ldr = g.ldr;
  ga.res_ty = g.res_ty;
  if (ga.N <= 0) return TSP_ERR_INVALID_ARG;
  return bf ? gemv_epi<__nv_bfloat16, __half>(ga, g.epi, g.name, st)
            : gemv_epi<float, float>(ga, g.epi, g.name, st);
}

int64_t decode_splits(int64_t S, int D, int64_t n_rows) {
  const int64_t c2 = S / D;   // 2c rows per virtual rank
  const int64_t spr = (c2 + kSplitRows - 1) / kSplitRows;
  return D * spr + (n_rows - S + kSplitRows - 1) / kSplitRows;
}

tsp_status launch_decode_attn(const DecodeAttn& d, cudaStream_t st) {
  if (d.T < 1 || d.T > TSP_DECODE_MAX_T || d.Hkv < 1 || d.H % d.Hkv != 0) return TSP_ERR_INVALID_ARG;
  if (((uintptr_t)d.kv & 15u) || ((uintptr_t)d.q & 15u)) return TSP_ERR_INVALID_ARG;
  AttnArgs aa;
  memset(&aa, 0, sizeof(aa));
  aa.q = d.q;
  aa.ldq = d.ldq;
  aa.kv = d.kv;
  aa.dkv = d.Hkv * d.dh;
  aa.ldkv = 2 * (int64_t)aa.dkv;
  aa.part_o = d.part_o;
  aa.part_ml = d.part_ml;
  aa.S = d.S;
  aa.D = d.D;
  aa.c = d.S / (2 * d.D);
  aa.n_cached = d.n_cached;
  aa.n_total = d.n_cached + d.T;
  aa.status = status_word();
  aa.spr = (int)((2 * aa.c + kSplitRows - 1) / kSplitRows);
  aa.nsplit = (int)decode_splits(d.S, d.D, aa.n_total);
  aa.T = d.T;
  aa.H = d.H;
  aa.G = d.H / d.Hkv;
  aa.scale_log2 = 1.4426950408889634f / sqrtf((float)d.dh);
  // query-row groups.  The fp16 kernel (dot products on the tensor cores)
  // serves all G*T query rows of a K/V head in one CTA, so every cache row is
  // read once.  The fp32 kernel's scalar arithmetic grows with the rows, so
  // it splits them over enough CTAs for ~4 waves of 3 per SM when the K/V
  // heads and splits alone give fewer (grouped K/V heads, short caches).
  {
    const int QR = aa.G * aa.T;
    int nz = 1;
    if (d.dtype != TSP_BF16) {
      const int64_t base_ctas = (int64_t)d.Hkv * aa.nsplit;
      const int64_t want = 12 * (int64_t)num_sms();
      nz = (int)std::min<int64_t>(QR, std::max<int64_t>(1, (want + base_ctas - 1) / base_ctas));
    }
    aa.qpc = (QR + nz - 1) / nz;
    aa.nz = (QR + aa.qpc - 1) / aa.qpc;
  }
  tsp_status r = TSP_ERR_UNSUPPORTED;
  int n_part = aa.nsplit;   // partials per query row the combine kernel merges
  if (d.dtype == TSP_BF16) {
    // a few query rows per K/V head (one token; grouped heads): one wave of
    // streaming CTAs, each over a slice of the splits, when the K/V heads
    // leave room for at least two slices a head
    const int sms = num_sms();
    if (aa.G * aa.T <= kQB && 2 * d.Hkv <= sms && (d.dh == 128 || d.dh == 64)) {
      aa.nslice = std::min(aa.nsplit, sms / d.Hkv);
      aa.limit_ns = wait_limit_ns();
      n_part = aa.nslice;
      // x of every box (a multiple of 64 columns) is 16-byte aligned; the
      // row extent n_total makes rows past the cache read as zeros
      if (!tma_map_f16(&aa.tm, d.kv, aa.ldkv, aa.n_total, aa.ldkv, 32)) return TSP_ERR_CUDA;
      r = d.dh == 128 ? decode_attn_stream<128>(aa, st) : decode_attn_stream<64>(aa, st);
    } else if (d.dh == 128) {
      r = decode_attn_mma<128>(aa, st);
    } else if (d.dh == 64) {
      r = decode_attn_mma<64>(aa, st);
    }
  } else {
    if (d.dh == 64) r = decode_attn_t<float, 64>(aa, st);
    else if (d.dh == 32) r = decode_attn_t<float, 32>(aa, st);
    else if (d.dh == 16) r = decode_attn_t<float, 16>(aa, st);
  }
  if (r != TSP_OK) return r;
  Prof prof("decode_combine", st);
  const int blocks = d.H * d.T;   // a CTA per (head, token)
  if (d.dtype == TSP_BF16)
    decode_combine_kernel<__half><<<blocks, kCombineWarps * 32, 0, st>>>(
        aa.part_o, aa.part_ml, (__half*)d.o, n_part, d.H, d.T, d.dh);
  else
    decode_combine_kernel<float><<<blocks, kCombineWarps * 32, 0, st>>>(
        aa.part_o, aa.part_ml, (float*)d.o, aa.nsplit, d.H, d.T, d.dh);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
