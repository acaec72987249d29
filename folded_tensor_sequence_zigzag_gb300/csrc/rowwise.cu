// rowwise.cu -- HBM-bound kernels: zigzag gather/scatter and RMSNorm fwd/bwd.
//
// Zigzag causal partitioning: "Folding Tensor and Sequence Parallelism for
// Memory-Efficient Transformer Training & Inference" (gist.science summary),
// section 2, attention-layer schedule (zigzag partitioning balances causal
// attention).  Rank r owns chunks r and 2D-1-r of the 2D equal chunks.
// RMSNorm: the pages give no formula; the plain reading of a pre-norm block,
// rms(u; g) = u / sqrt(mean(u^2) + eps) * g with fp32 arithmetic.
#include <cmath>
#include <cstring>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace tsp {

// ---------------------------------------------------------------------------
// K1: zigzag permute.  One CTA row at a time (grid-stride over rows), 16-byte
// vectors when the row length allows it, 4-way unrolled for memory-level
// parallelism.  Bit-exact copy.
// ---------------------------------------------------------------------------
template <typename V>
__global__ void __launch_bounds__(256) zigzag_permute_kernel(const V* __restrict__ src,
                                                             V* __restrict__ dst, int64_t S,
                                                             int64_t c, int D, int64_t vpr,
                                                             int inverse, int* status) {
  for (int64_t row = blockIdx.x; row < S; row += gridDim.x) {
    // forward: dst zigzag row <- src global row pos(row)
    // inverse: dst global row <- src zigzag row row_of_pos(row)
    const int64_t srow = inverse ? zz_row_of_pos(row, c, D) : zz_pos_of_row(row, c, D);
    if (!TSP_INB(srow >= 0 && srow < S, status)) continue;
    const V* s = src + srow * vpr;
    V* d = dst + row * vpr;
    int64_t v = threadIdx.x;
    for (; v + 3 * blockDim.x < vpr; v += 4 * blockDim.x) {
      V a0 = s[v], a1 = s[v + blockDim.x], a2 = s[v + 2 * blockDim.x], a3 = s[v + 3 * blockDim.x];
      d[v] = a0;
      d[v + blockDim.x] = a1;
      d[v + 2 * blockDim.x] = a2;
      d[v + 3 * blockDim.x] = a3;
    }
    for (; v < vpr; v += blockDim.x) d[v] = s[v];
  }
}

tsp_status launch_zigzag_permute(const void* src, void* dst, int64_t S, int D, int64_t row_bytes,
                                 int inverse, cudaStream_t st) {
  const int64_t c = S / (2 * D);
  const int grid = (int)std::min<int64_t>(S, (int64_t)num_sms() * 8);
  Prof prof(inverse ? "zigzag_unpermute" : "zigzag_permute", st);
  if (row_bytes % 16 == 0) {
    zigzag_permute_kernel<uint4><<<grid, 256, 0, st>>>((const uint4*)src, (uint4*)dst, S, c, D,
                                                       row_bytes / 16, inverse, status_word());
  } else if (row_bytes % 4 == 0) {
    zigzag_permute_kernel<uint32_t><<<grid, 256, 0, st>>>((const uint32_t*)src, (uint32_t*)dst, S,
                                                          c, D, row_bytes / 4, inverse, status_word());
  } else {
    zigzag_permute_kernel<uint8_t><<<grid, 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, S, c,
                                                         D, row_bytes, inverse, status_word());
  }
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// ---------------------------------------------------------------------------
// K2: RMSNorm forward.  One warp per row; the row stays in registers (UPL
// units of 8 elements per lane), so u is read once and out written once.
// Input and output types may differ (the block's fp32 residual stream h is
// normalised into the bf16 GEMM operand b).
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f) {
  if constexpr (sizeof(T) == 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = lo2<T>(w[i]);
      f[2 * i + 1] = hi2<T>(w[i]);
    }
  } else {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float* f) {
  if constexpr (sizeof(T) == 2) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack2<T>(f[0], f[1]), pack2<T>(f[2], f[3]),
                                              pack2<T>(f[4], f[5]), pack2<T>(f[6], f[7]));
  } else {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

template <typename Tin, typename Tg, typename T, int UPL>
__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(const Tin* __restrict__ u,
                                                          const Tg* __restrict__ g,
                                                          T* __restrict__ out,
                                                          float* __restrict__ rstd_out,
                                                          int64_t rows, int n, float eps,
                                                          int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  bool bad = false;   // an fp16 output out of range
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int nu = n >> 3;  // 8-element units per row
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const Tin* src = u + row * n;
    float v[UPL][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < UPL; ++i) {
      const int idx = lane + 32 * i;
      if (idx < nu) {
        load8(src + idx * 8, v[i]);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[i][e], v[i][e], ss);
      }
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)n + eps);
    if (lane == 0 && rstd_out) rstd_out[row] = r;
    T* dst = out + row * n;
#pragma unroll
    for (int i = 0; i < UPL; ++i) {
      const int idx = lane + 32 * i;
      if (idx < nu) {
        float gf[8];
        load8(g + idx * 8, gf);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][e] = v[i][e] * r * gf[e];
        if constexpr (std::is_same<T, __half>::value) bad |= f16_bad_n<8>(v[i]);
        store8(dst + idx * 8, v[i]);
      }
    }
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

// Row-per-CTA variant for n % 512 == 0, n <= 16384: n/16 threads, 16 elements
// (two 8-element units) per thread, the row sum reduced through shared memory
// with one barrier per row (double-buffered partials).  Few registers, so many
// CTAs share an SM and many rows are in flight: the warp-per-row kernel above
// holds a whole row per warp in registers and runs latency-bound.
template <typename Tin, typename Tg, typename T>
__global__ void __launch_bounds__(1024) rmsnorm_fwd_cta_kernel(const Tin* __restrict__ u,
                                                               const Tg* __restrict__ g,
                                                               T* __restrict__ out,
                                                               float* __restrict__ rstd_out,
                                                               int64_t rows, int n, float eps,
                                                               int* __restrict__ status) {
  __shared__ float part[2][32];
  bool bad = false;   // an fp16 output out of range
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = blockDim.x >> 5;
  const int c0 = t * 8, c1 = (t + blockDim.x) * 8;   // this thread's two units
  float gf0[8], gf1[8];
  load8(g + c0, gf0);
  load8(g + c1, gf1);
  int it = 0;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
    const Tin* src = u + row * n;
    float v0[8], v1[8];
    load8(src + c0, v0);
    load8(src + c1, v1);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v0[e], v0[e], fmaf(v1[e], v1[e], ss));
    ss = warp_sum(ss);
    if (lane == 0) part[it & 1][warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nw; ++w) tot += part[it & 1][w];
    const float r = rsqrtf(tot / (float)n + eps);
    if (t == 0 && rstd_out) rstd_out[row] = r;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v0[e] = v0[e] * r * gf0[e];
      v1[e] = v1[e] * r * gf1[e];
    }
    T* dst = out + row * n;
    if constexpr (std::is_same<T, __half>::value) bad |= f16_bad_n<8>(v0) | f16_bad_n<8>(v1);
    store8(dst + c0, v0);
    store8(dst + c1, v1);
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

// Scalar fallback for rows whose length is not a multiple of 8 (or unaligned).
template <typename Tin, typename Tg, typename T>
__global__ void rmsnorm_fwd_scalar_kernel(const Tin* __restrict__ u, const Tg* __restrict__ g,
                                          T* __restrict__ out, float* __restrict__ rstd_out,
                                          int64_t rows, int n, float eps, int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  bool bad = false;   // an fp16 output out of range
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    float ss = 0.f;
    for (int i = lane; i < n; i += 32) {
      float f = to_f(u[row * n + i]);
      ss = fmaf(f, f, ss);
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)n + eps);
    if (lane == 0 && rstd_out) rstd_out[row] = r;
    for (int i = lane; i < n; i += 32) {
      const float o = to_f(u[row * n + i]) * r * to_f(g[i]);
      if constexpr (std::is_same<T, __half>::value) bad |= f16_bad(o);
      out[row * n + i] = from_f<T>(o);
    }
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

template <typename Tin, typename Tg, typename T>
static tsp_status rmsnorm_fwd_t(const Tin* u, const Tg* g, T* out, float* rstd, int64_t rows, int n,
                                float eps, cudaStream_t st) {
  const int64_t want = (rows + 7) / 8;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * 8));
  const bool vec_ok = (n % 8 == 0) && ((uintptr_t)u % 16 == 0) && ((uintptr_t)g % 16 == 0) &&
                      ((uintptr_t)out % 16 == 0);
  const int nu = n / 8;
  int* status = status_word();
  Prof prof("rmsnorm_fwd", st);
  if (vec_ok && n % 512 == 0 && n <= 16384) {
    const int threads = n / 16;
    const int per_sm = std::max(1, 2048 / threads);
    const int grid2 = (int)std::max<int64_t>(1, std::min<int64_t>(rows, (int64_t)num_sms() * per_sm));
    rmsnorm_fwd_cta_kernel<Tin, Tg, T><<<grid2, threads, 0, st>>>(u, g, out, rstd, rows, n, eps, status);
  } else if (vec_ok && nu <= 32)
    rmsnorm_fwd_kernel<Tin, Tg, T, 1><<<grid, 256, 0, st>>>(u, g, out, rstd, rows, n, eps, status);
  else if (vec_ok && nu <= 128)
    rmsnorm_fwd_kernel<Tin, Tg, T, 4><<<grid, 256, 0, st>>>(u, g, out, rstd, rows, n, eps, status);
  else if (vec_ok && nu <= 512)
    rmsnorm_fwd_kernel<Tin, Tg, T, 16><<<grid, 256, 0, st>>>(u, g, out, rstd, rows, n, eps, status);
  else
    rmsnorm_fwd_scalar_kernel<Tin, Tg, T><<<grid, 256, 0, st>>>(u, g, out, rstd, rows, n, eps, status);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

tsp_status launch_rmsnorm_fwd(const void* u, int u_ty, const void* g, void* out, int out_ty,
                              float* rstd, int64_t rows, int n, float eps, int dtype,
                              cudaStream_t st) {
  typedef __nv_bfloat16 bf;
  if (dtype != TSP_BF16)
    return rmsnorm_fwd_t((const float*)u, (const float*)g, (float*)out, rstd, rows, n, eps, st);
  const bf* gb = (const bf*)g;
  if (u_ty == TY_F32 && out_ty == TY_F16)
    return rmsnorm_fwd_t((const float*)u, gb, (ct_t*)out, rstd, rows, n, eps, st);
  if (u_ty == TY_BF16 && out_ty == TY_F16)
    return rmsnorm_fwd_t((const bf*)u, gb, (ct_t*)out, rstd, rows, n, eps, st);
  if (u_ty == TY_BF16 && out_ty == TY_BF16)
    return rmsnorm_fwd_t((const bf*)u, gb, (bf*)out, rstd, rows, n, eps, st);
  return TSP_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------------------
// K8: RMSNorm backward fused with the residual-gradient add.
//   nrm = u * rstd;  gd = dout * g
//   du  = rstd * (gd - nrm * mean(gd * nrm))
//   res_out = resid + du          (fp32 and/or storage-dtype copies)
//   dg_part[block] = sum over the block's rows of dout * nrm
// dout is fp32; u is of type Tu (the fp32 residual stream or the storage
// dtype); g, resid_t and out_t are of the storage dtype T.
// One warp per row (strided loop over columns); the gain gradient of a CTA is
// gathered in shared memory and written as one partial row, summed by
// rowsum_partials_kernel.
// ---------------------------------------------------------------------------
template <typename Tu, typename T, typename Tr, typename To>
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(
    const float* __restrict__ dout, const Tu* __restrict__ u, const T* __restrict__ g,
    const float* __restrict__ rstd, const float* __restrict__ resid_f32,
    const Tr* __restrict__ resid_t, float* __restrict__ out_f32, To* __restrict__ out_t,
    float* __restrict__ dg_part, int64_t rows, int n) {
  extern __shared__ float s_dg[];
  for (int i = threadIdx.x; i < n; i += blockDim.x) s_dg[i] = 0.f;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const float r = rstd[row];
    const float* dr = dout + row * n;
    const Tu* ur = u + row * n;
    float dot = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float nrm = to_f(ur[i]) * r;
      const float dv = dr[i];
      dot = fmaf(dv * to_f(g[i]), nrm, dot);
      atomicAdd(&s_dg[i], dv * nrm);
    }
    dot = warp_sum(dot) / (float)n;
    for (int i = lane; i < n; i += 32) {
      const float nrm = to_f(ur[i]) * r;
      const float du = r * (dr[i] * to_f(g[i]) - nrm * dot);
      const float o = (resid_f32 ? resid_f32[row * n + i] : to_f(resid_t[row * n + i])) + du;
      if (out_f32) out_f32[row * n + i] = o;
      if (out_t) out_t[row * n + i] = from_f<To>(o);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) dg_part[(int64_t)blockIdx.x * n + i] = s_dg[i];
}

int rmsnorm_bwd_blocks(int64_t rows) {
  return (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 2));
}

// Fast path of K8 for n = 1024*K: 256 threads a CTA, thread t owns the
// columns k*1024 + 4t .. +3 (k < K) of every row the CTA visits, so its share
// of the gain gradient stays in registers and every load is a 16-byte (fp32)
// or 8-byte (16-bit) vector.  Rows are read once; the row dot product is
// reduced across the CTA with one barrier per row (double-buffered partials).
template <typename T> __device__ __forceinline__ float4 load4(const T* p);
template <> __device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
template <> __device__ __forceinline__ float4 load4<__half>(const __half* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
template <typename T> __device__ __forceinline__ void store4(T* p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&a);
  o.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = o;
}
template <> __device__ __forceinline__ void store4<__half>(__half* p, float4 v) {
  const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&a);
  o.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = o;
}
__device__ __forceinline__ float f4(const float4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

template <int K, typename Tu, typename T, typename Tr, typename To>
__global__ void __launch_bounds__(256) rmsnorm_bwd_vec_kernel(
    const float* __restrict__ dout, const Tu* __restrict__ u, const T* __restrict__ g,
    const float* __restrict__ rstd, const float* __restrict__ resid_f32,
    const Tr* __restrict__ resid_t, float* __restrict__ out_f32, To* __restrict__ out_t,
    float* __restrict__ dg_part, int64_t rows) {
  constexpr int n = 1024 * K;
  __shared__ float red[2][8];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float4 gv[K], dg[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    gv[k] = load4(g + k * 1024 + 4 * t);
    dg[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  int it = 0;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
    const float r = rstd[row];
    const int64_t base = row * n + 4 * t;
    float4 dv[K], nv[K];
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      dv[k] = load4(dout + base + k * 1024);
      nv[k] = load4(u + base + k * 1024);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      nv[k] = make_float4(nv[k].x * r, nv[k].y * r, nv[k].z * r, nv[k].w * r);
      dot = fmaf(dv[k].x * gv[k].x, nv[k].x, dot);
      dot = fmaf(dv[k].y * gv[k].y, nv[k].y, dot);
      dot = fmaf(dv[k].z * gv[k].z, nv[k].z, dot);
      dot = fmaf(dv[k].w * gv[k].w, nv[k].w, dot);
      dg[k].x = fmaf(dv[k].x, nv[k].x, dg[k].x);
      dg[k].y = fmaf(dv[k].y, nv[k].y, dg[k].y);
      dg[k].z = fmaf(dv[k].z, nv[k].z, dg[k].z);
      dg[k].w = fmaf(dv[k].w, nv[k].w, dg[k].w);
    }
    dot = warp_sum(dot);
    if (lane == 0) red[it & 1][warp] = dot;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[it & 1][w];
    tot *= 1.f / (float)n;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float4 res = resid_f32 ? load4(resid_f32 + base + k * 1024)
                                   : load4(resid_t + base + k * 1024);
      float4 o;
      o.x = res.x + r * (dv[k].x * gv[k].x - nv[k].x * tot);
      o.y = res.y + r * (dv[k].y * gv[k].y - nv[k].y * tot);
      o.z = res.z + r * (dv[k].z * gv[k].z - nv[k].z * tot);
      o.w = res.w + r * (dv[k].w * gv[k].w - nv[k].w * tot);
      if (out_f32) store4(out_f32 + base + k * 1024, o);
      if (out_t) store4(out_t + base + k * 1024, o);
    }
  }
  float* part = dg_part + (int64_t)blockIdx.x * n + 4 * t;
#pragma unroll
  for (int k = 0; k < K; ++k) store4(part + k * 1024, dg[k]);
}

// out[i] = sum_b part[b][i], b in a fixed order: 32 columns a CTA, the
// partial rows split 8 ways and combined in shared memory (deterministic).
__global__ void __launch_bounds__(256) rowsum_partials_kernel(const float* __restrict__ part,
                                                              float* __restrict__ out, int nb,
                                                              int n) {
  __shared__ float acc[8][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int i = blockIdx.x * 32 + tx;
  float s = 0.f;
  if (i < n)
    for (int b = ty; b < nb; b += 8) s += part[(int64_t)b * n + i];
  acc[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && i < n) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) o += acc[w][tx];
    out[i] = o;
  }
}

template <typename Tu, typename T, typename Tr, typename To>
static tsp_status rmsnorm_bwd_t(const float* dout, const Tu* u, const T* g, const float* rstd,
                                const float* resid_f32, const Tr* resid_t, float* out_f32, To* out_t,
                                float* dg, float* dg_part, int64_t rows, int n, cudaStream_t st) {
  const int grid = rmsnorm_bwd_blocks(rows);
  Prof prof("rmsnorm_bwd", st, 2);
  auto al16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  const bool vec = n % 1024 == 0 && (n / 1024 == 1 || n / 1024 == 2 || n / 1024 == 4 ||
                                     n / 1024 == 8) &&
                   al16(dout) && al16(u) && al16(g) && al16(resid_f32) && al16(resid_t) &&
                   al16(out_f32) && al16(out_t) && al16(dg_part);
  if (vec) {
#define TSP_RMSB_VEC(K)                                                                     \
  rmsnorm_bwd_vec_kernel<K, Tu, T, Tr, To><<<grid, 256, 0, st>>>(dout, u, g, rstd, resid_f32, \
                                                                 resid_t, out_f32, out_t,     \
                                                                 dg_part, rows)
    switch (n / 1024) {
      case 1: TSP_RMSB_VEC(1); break;
      case 2: TSP_RMSB_VEC(2); break;
      case 4: TSP_RMSB_VEC(4); break;
      default: TSP_RMSB_VEC(8); break;
    }
#undef TSP_RMSB_VEC
  } else {
    const size_t sm = (size_t)n * sizeof(float);
    if (sm > 48 * 1024)
      TSP_CUDA_TRY(cudaFuncSetAttribute(rmsnorm_bwd_kernel<Tu, T, Tr, To>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
    rmsnorm_bwd_kernel<Tu, T, Tr, To><<<grid, 256, sm, st>>>(dout, u, g, rstd, resid_f32, resid_t,
                                                             out_f32, out_t, dg_part, rows, n);
  }
  TSP_CUDA_TRY(cudaGetLastError());
  rowsum_partials_kernel<<<(n + 31) / 32, 256, 0, st>>>(dg_part, dg, grid, n);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

tsp_status launch_rmsnorm_bwd(const float* dout, const void* u, int u_ty, const void* g,
                              const float* rstd, const float* resid_f32, const void* resid_t,
                              float* out_f32, void* out_t, int out_ty, float* dg, float* dg_part,
                              int64_t rows, int n, int dtype, cudaStream_t st) {
  typedef __nv_bfloat16 bf;
  if (dtype != TSP_BF16)
    return rmsnorm_bwd_t(dout, (const float*)u, (const float*)g, rstd, resid_f32,
                         (const float*)resid_t, out_f32, (float*)out_t, dg, dg_part, rows, n, st);
  const bf* gb = (const bf*)g;
  // MLP norm: u = h (fp32 residual stream), resid = dy (bf16), out = dh (fp32) + fp16 copy
  if (u_ty == TY_F32 && out_ty == TY_F16)
    return rmsnorm_bwd_t(dout, (const float*)u, gb, rstd, resid_f32, (const bf*)resid_t, out_f32,
                         (ct_t*)out_t, dg, dg_part, rows, n, st);
  // attention norm: u = x (bf16), resid = dh (fp32), out = dx (bf16)
  if (u_ty == TY_BF16 && out_ty == TY_BF16)
    return rmsnorm_bwd_t(dout, (const bf*)u, gb, rstd, resid_f32, (const bf*)resid_t, out_f32,
                         (bf*)out_t, dg, dg_part, rows, n, st);
  return TSP_ERR_UNSUPPORTED;
}

// Eight bf16 values -> fp16 (exact whenever in range); `bad` collects values
// fp16 cannot hold.
__device__ __forceinline__ uint4 cvt8_bf16_f16(const uint4 v, bool& bad) {
  float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
  bad |= f16_bad_n<8>(f);
  return make_uint4(pack_f16(f[0], f[1]), pack_f16(f[2], f[3]), pack_f16(f[4], f[5]),
                    pack_f16(f[6], f[7]));
}

// bf16 -> fp16, 8 elements per thread-iteration (n % 8 == 0, 16-byte aligned)
__global__ void convert_bf16_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                        int64_t n8, int* __restrict__ status) {
  bool bad = false;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8;
       t += (int64_t)gridDim.x * blockDim.x)
    dst[t] = cvt8_bf16_f16(src[t], bad);
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

tsp_status launch_convert_bf16_f16(const void* src, void* dst, int64_t n, cudaStream_t st) {
  if (n % 8 != 0 || ((uintptr_t)src & 15u) || ((uintptr_t)dst & 15u)) return TSP_ERR_UNSUPPORTED;
  Prof prof("convert_bf16_f16", st);
  const int64_t n8 = n / 8;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n8 + 255) / 256, (int64_t)num_sms() * 8));
  convert_bf16_f16_kernel<<<grid, 256, 0, st>>>((const uint4*)src, (uint4*)dst, n8, status_word());
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// Several bf16 -> fp16 conversions in one launch: the buffers are laid end to
// end in one index space of 8-element units; a thread walks its grid-stride
// indices upward, so its buffer index only moves forward.
struct ConvertList {
  const uint4* src[kMaxConvert];
  uint4* dst[kMaxConvert];
  int64_t end8[kMaxConvert];   // exclusive prefix ends, in 8-element units
  int count;
};

__global__ void convert_bf16_f16_many_kernel(const __grid_constant__ ConvertList L,
                                             int* __restrict__ status) {
  const int64_t total = L.end8[L.count - 1];
  int seg = 0;
  bool bad = false;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    while (t >= L.end8[seg]) ++seg;
    const int64_t i = t - (seg > 0 ? L.end8[seg - 1] : 0);
    L.dst[seg][i] = cvt8_bf16_f16(L.src[seg][i], bad);
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

tsp_status launch_convert_bf16_f16_many(const void* const* src, void* const* dst, const int64_t* n,
                                        int count, cudaStream_t st) {
  if (count < 1 || count > kMaxConvert) return TSP_ERR_INVALID_ARG;
  ConvertList L;
  memset(&L, 0, sizeof(L));
  int64_t acc = 0;
  for (int k = 0; k < count; ++k) {
    if (n[k] % 8 != 0 || ((uintptr_t)src[k] & 15u) || ((uintptr_t)dst[k] & 15u))
      return TSP_ERR_UNSUPPORTED;
    L.src[k] = (const uint4*)src[k];
    L.dst[k] = (uint4*)dst[k];
    acc += n[k] / 8;
    L.end8[k] = acc;
  }
  L.count = count;
  if (acc == 0) return TSP_OK;
  Prof prof("convert_bf16_f16", st);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((acc + 255) / 256, (int64_t)num_sms() * 8));
  convert_bf16_f16_many_kernel<<<grid, 256, 0, st>>>(L, status_word());
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// fp32 -> fp16 (round to nearest), 8 elements per thread-iteration
__global__ void convert_f32_f16_kernel(const float4* __restrict__ src, uint4* __restrict__ dst,
                                       int64_t n8, int* __restrict__ status) {
  bool bad = false;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8;
       t += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = src[2 * t], b = src[2 * t + 1];
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    bad |= f16_bad_n<8>(f);
    dst[t] = make_uint4(pack_f16(a.x, a.y), pack_f16(a.z, a.w), pack_f16(b.x, b.y),
                        pack_f16(b.z, b.w));
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

tsp_status launch_convert_f32_f16(const float* src, void* dst, int64_t n, cudaStream_t st) {
  if (n % 8 != 0 || ((uintptr_t)src & 15u) || ((uintptr_t)dst & 15u)) return TSP_ERR_UNSUPPORTED;
  Prof prof("convert_f32_f16", st);
  const int64_t n8 = n / 8;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n8 + 255) / 256, (int64_t)num_sms() * 8));
  convert_f32_f16_kernel<<<grid, 256, 0, st>>>((const float4*)src, (uint4*)dst, n8, status_word());
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// ---------------------------------------------------------------------------
// Rotary position embedding (a variant; the pages' block has none).
// Rotate-half form: within each head, element j < dh/2 pairs with j + dh/2 and
// the pair turns by the angle pos * f_j, f_j = base^(-2j/dh).  The angle is
// formed and reduced modulo 2*pi in fp64 (at a million positions an fp32
// product would be off by a twentieth of a radian); sin and cos of the
// reduced angle are taken in fp32.  The frequencies come from the host in
// fp64.
// ---------------------------------------------------------------------------
constexpr int kRopeMaxHalf = 128;
struct RopeFreq {
  double f[kRopeMaxHalf];
};

// row `row` holds zigzag position zz_pos_of_row(row)
__global__ void rope_table_kernel(float2* __restrict__ tab, int64_t S, int64_t c, int D, int half,
                                  const __grid_constant__ RopeFreq F) {
  const int64_t total = S * half;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = t / half;
    const int j = (int)(t - row * half);
    const double ang = (double)zz_pos_of_row(row, c, D) * F.f[j];
    const double two_pi = 6.283185307179586476925287;
    const double red = ang - two_pi * rint(ang / two_pi);
    float sv, cv;
    sincosf((float)red, &sv, &cv);
    tab[t] = make_float2(cv, sv);
  }
}

tsp_status launch_rope_table(float2* table, int64_t S, int D, int dh, float base, cudaStream_t st) {
  const int half = dh / 2;
  if (!table || half < 1 || half > kRopeMaxHalf || D < 1) return TSP_ERR_UNSUPPORTED;
  RopeFreq F;
  for (int j = 0; j < half; ++j) F.f[j] = std::pow((double)base, -2.0 * j / (double)dh);
  Prof prof("rope_table", st);
  const int64_t total = S * half;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms() * 8));
  rope_table_kernel<<<grid, 256, 0, st>>>(table, S, S / (2 * D), D, half, F);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// one thread = one (row, head of Q or K, pair j); consecutive threads take
// consecutive j of one head, so both halves of a head are read coalesced.
// Heads 0..H-1 are Q's (column 0), heads H..H+Hkv-1 are K's (column d).
template <typename T>
__global__ void rope_kernel(T* __restrict__ qkv, int64_t S, int ld, int d, int H, int Hkv,
                            int half, const float2* __restrict__ tab, float sgn,
                            int* __restrict__ status) {
  const int64_t per_row = (int64_t)(H + Hkv) * half;
  const int64_t total = S * per_row;
  bool bad = false;   // an fp16 output out of range
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = t / per_row;
    const int rem = (int)(t - row * per_row);
    const int hh = rem / half, j = rem - hh * half;
    const int64_t col = hh < H ? (int64_t)hh * 2 * half : d + (int64_t)(hh - H) * 2 * half;
    T* p = qkv + row * ld + col + j;
    const float2 cs = tab[row * half + j];
    const float s = sgn * cs.y;
    const float x1 = to_f(p[0]), x2 = to_f(p[half]);
    const float y1 = x1 * cs.x - x2 * s, y2 = x1 * s + x2 * cs.x;
    if constexpr (std::is_same<T, __half>::value) bad |= f16_bad(y1) | f16_bad(y2);
    p[0] = from_f<T>(y1);
    p[half] = from_f<T>(y2);
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

tsp_status launch_rope(void* qkv, int ty, int64_t S, int ld, int d, int H, int Hkv, int dh,
                       const float2* table, int inverse, cudaStream_t st) {
  const int half = dh / 2;
  if (!qkv || !table || half < 1) return TSP_ERR_INVALID_ARG;
  Prof prof("rope", st);
  const int64_t total = S * (int64_t)(H + Hkv) * half;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms() * 8));
  const float sgn = inverse ? -1.f : 1.f;
  if (ty == TY_F16)
    rope_kernel<__half><<<grid, 256, 0, st>>>((__half*)qkv, S, ld, d, H, Hkv, half, table, sgn,
                                              status_word());
  else if (ty == TY_F32)
    rope_kernel<float><<<grid, 256, 0, st>>>((float*)qkv, S, ld, d, H, Hkv, half, table, sgn,
                                             status_word());
  else
    return TSP_ERR_UNSUPPORTED;
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// ---------------------------------------------------------------------------
// Elementwise helpers of the exact-fp32 path.
// ---------------------------------------------------------------------------

// G = silu(A) * B, with A = AB[:, :I] and B = AB[:, I:]  (row stride 2I)
__global__ void swiglu_f32_kernel(const float* __restrict__ AB, float* __restrict__ G, int64_t rows,
                                  int I) {
  const int64_t total = rows * I;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / I;
    const int i = (int)(t - r * I);
    const float a = AB[r * 2 * I + i], b = AB[r * 2 * I + I + i];
    G[t] = a * sigmoidf_(a) * b;
  }
}

// dA = dG * B * s(A) * (1 + A (1 - s(A))),  dB = dG * silu(A)   (into dAB [rows, 2I])
__global__ void swiglu_bwd_f32_kernel(const float* __restrict__ dG, const float* __restrict__ AB,
                                      float* __restrict__ dAB, int64_t rows, int I) {
  const int64_t total = rows * I;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / I;
    const int i = (int)(t - r * I);
    const float a = AB[r * 2 * I + i], b = AB[r * 2 * I + I + i];
    const float s = sigmoidf_(a);
    const float dg = dG[t];
    dAB[r * 2 * I + i] = dg * b * s * (1.f + a * (1.f - s));
    dAB[r * 2 * I + I + i] = dg * a * s;
  }
}

tsp_status launch_swiglu_f32(const float* AB, float* G, int64_t rows, int I, cudaStream_t st) {
  Prof prof("swiglu_f32", st);
  swiglu_f32_kernel<<<num_sms() * 4, 256, 0, st>>>(AB, G, rows, I);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}
tsp_status launch_swiglu_bwd_f32(const float* dG, const float* AB, float* dAB, int64_t rows, int I,
                                 cudaStream_t st) {
  Prof prof("swiglu_bwd_f32", st);
  swiglu_bwd_f32_kernel<<<num_sms() * 4, 256, 0, st>>>(dG, AB, dAB, rows, I);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// Pack the attention shards: shard k -> [W_Q[C_k,:]; W_K[C_k,:]; W_V[C_k,:]; W_O[:,C_k]^T].
template <typename T>
__global__ void pack_attn_shards_kernel(const T* __restrict__ wq, const T* __restrict__ wk,
                                        const T* __restrict__ wv, const T* __restrict__ wo,
                                        T* __restrict__ dst, int d, int D) {
  const int64_t total = (int64_t)4 * d * d;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t orow = t / d;  // row of dst
    const int col = (int)(t - orow * d);
    // find shard k with 4*lo(k) <= orow < 4*lo(k+1)
    int k = (int)((orow / 4) * D / d);
    while (k > 0 && 4 * ((int64_t)k * d / D) > orow) --k;
    while (k + 1 < D && 4 * ((int64_t)(k + 1) * d / D) <= orow) ++k;
    const int64_t lo = (int64_t)k * d / D, w = (int64_t)(k + 1) * d / D - lo;
    const int64_t rr = orow - 4 * lo;
    const int part = (int)(rr / w);
    const int64_t ci = lo + (rr - part * w);
    T v;
    if (part == 0) v = wq[ci * d + col];
    else if (part == 1) v = wk[ci * d + col];
    else if (part == 2) v = wv[ci * d + col];
    else v = wo[(int64_t)col * d + ci];
    dst[t] = v;
  }
}

// Packed MLP shards, what one step of the ring hands on: shard k (rows I_k of
// W_1 and W_3, boundaries floor(k*I/D)) is [W_1[I_k,:]; W_3[I_k,:]; W_2[:,I_k]^T],
// a [3*|I_k|, d] block; shards follow each other.
template <typename T>
__global__ void pack_mlp_shards_kernel(const T* __restrict__ w1, const T* __restrict__ w3,
                                       const T* __restrict__ w2, T* __restrict__ dst, int d, int I,
                                       int D) {
  const int64_t total = (int64_t)3 * I * d;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t orow = t / d;  // row of dst
    const int col = (int)(t - orow * d);
    // shard k with 3*lo(k) <= orow < 3*lo(k+1)
    int k = (int)((orow / 3) * D / I);
    while (k > 0 && 3 * ((int64_t)k * I / D) > orow) --k;
    while (k + 1 < D && 3 * ((int64_t)(k + 1) * I / D) <= orow) ++k;
    const int64_t lo = (int64_t)k * I / D, w = (int64_t)(k + 1) * I / D - lo;
    const int64_t rr = orow - 3 * lo;
    const int part = (int)(rr / w);
    const int64_t ii = lo + (rr - part * w);
    T v;
    if (part == 0) v = w1[ii * d + col];
    else if (part == 1) v = w3[ii * d + col];
    else v = w2[(int64_t)col * I + ii];
    dst[t] = v;
  }
}

tsp_status launch_pack_mlp_shards(const void* w1, const void* w3, const void* w2, void* dst, int d,
                                  int I, int D, int dtype, cudaStream_t st) {
  Prof prof("pack_mlp_shards", st);
  if (dtype == TSP_BF16)
    pack_mlp_shards_kernel<__nv_bfloat16><<<num_sms() * 4, 256, 0, st>>>(
        (const __nv_bfloat16*)w1, (const __nv_bfloat16*)w3, (const __nv_bfloat16*)w2,
        (__nv_bfloat16*)dst, d, I, D);
  else
    pack_mlp_shards_kernel<float><<<num_sms() * 4, 256, 0, st>>>(
        (const float*)w1, (const float*)w3, (const float*)w2, (float*)dst, d, I, D);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

tsp_status launch_pack_attn_shards(const void* wq, const void* wk, const void* wv, const void* wo,
                                   void* dst, int d, int D, int dtype, cudaStream_t st) {
  Prof prof("pack_attn_shards", st);
  if (dtype == TSP_BF16)
    pack_attn_shards_kernel<__nv_bfloat16><<<num_sms() * 4, 256, 0, st>>>(
        (const __nv_bfloat16*)wq, (const __nv_bfloat16*)wk, (const __nv_bfloat16*)wv,
        (const __nv_bfloat16*)wo, (__nv_bfloat16*)dst, d, D);
  else
    pack_attn_shards_kernel<float><<<num_sms() * 4, 256, 0, st>>>(
        (const float*)wq, (const float*)wk, (const float*)wv, (const float*)wo, (float*)dst, d, D);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
