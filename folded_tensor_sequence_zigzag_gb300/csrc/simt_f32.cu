// simt_f32.cu -- exact-fp32 CUDA-core path of the block (small shapes).
//
// tcgen05 has no true-fp32 kind and TF32 cannot hold a 1e-4 absolute error,
// so the fp32 configuration runs on FFMA: a strided tiled GEMM and
// warp-per-row causal attention forward/backward over the zigzag layout.
// Source of the schedule: "Folding Tensor and Sequence Parallelism for
// Memory-Efficient Transformer Training & Inference" (gist.science summary),
// section 2; the host code in api.cu walks the shard loops.
#include "common.cuh"
#include "kernels.h"

namespace tsp {

// ---------------------------------------------------------------------------
// C[m*ldc+n] = (acc ? C : 0) + (R ? R[m*ldr+n] : 0) + sum_k A(m,k) B(n,k)
// A(m,k) = A[m*sam + k*sak], B(n,k) = B[n*sbn + k*sbk].  64x64 tile, BK 16,
// 256 threads x (4x4) outputs.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gemm_f32_kernel(int M, int N, int K, const float* __restrict__ A,
                                                       int64_t sam, int64_t sak,
                                                       const float* __restrict__ B, int64_t sbn,
                                                       int64_t sbk, float* C, int64_t ldc,
                                                       const float* R, int64_t ldr, int acc) {
  __shared__ float sA[16][65];
  __shared__ float sB[16][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float c[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = i / 64, mm = i % 64;
      const int m = m0 + mm, n = n0 + mm, k = k0 + kk;
      sA[kk][mm] = (m < M && k < K) ? A[(int64_t)m * sam + (int64_t)k * sak] : 0.f;
      sB[kk][mm] = (n < N && k < K) ? B[(int64_t)n * sbn + (int64_t)k * sbk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = sA[kk][ty + 16 * i];
        b[i] = sB[kk][tx + 16 * i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) c[i][j] = fmaf(a[i], b[j], c[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      float v = c[i][j];
      if (R) v += R[(int64_t)m * ldr + n];
      if (acc) v += C[(int64_t)m * ldc + n];
      C[(int64_t)m * ldc + n] = v;
    }
  }
}

tsp_status launch_gemm_f32(int M, int N, int K, const float* A, int64_t sam, int64_t sak,
                           const float* B, int64_t sbn, int64_t sbk, float* C, int64_t ldc,
                           const float* R, int64_t ldr, int acc, cudaStream_t st) {
  if (M <= 0 || N <= 0) return TSP_OK;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  Prof prof("gemm_f32", st);
  gemm_f32_kernel<<<grid, 256, 0, st>>>(M, N, K, A, sam, sak, B, sbn, sbk, C, ldc, R, ldr, acc);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

// ---------------------------------------------------------------------------
// Causal attention, one warp per (zigzag query row, head).  Keys are visited
// in global position order 0..pos(i); key position p lives at buffer row
// zz_row_of_pos(p).  Online softmax with expf (fp32).
//   Q, K, V: row stride ld (elements), head h at columns h*dh.
//   O: [S, ldo]; LSE: [H, S] (zigzag row order), natural log.
// ---------------------------------------------------------------------------
constexpr int kMaxDhPerLane = 4;  // dh <= 128

__global__ void attn_f32_fwd_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                    const float* __restrict__ V, int64_t ld, float* __restrict__ O,
                                    int64_t ldo, float* __restrict__ LSE, int64_t S, int H, int dh,
                                    int64_t c, int D, float scale, int G) {
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= S * H) return;
  const int64_t b = gw / H;
  const int h = (int)(gw - b * H);
  const int hk = h / G;   // K/V head of query head h
  const int64_t p = zz_pos_of_row(b, c, D);
  float q[kMaxDhPerLane], o[kMaxDhPerLane];
#pragma unroll
  for (int j = 0; j < kMaxDhPerLane; ++j) {
    const int col = lane + 32 * j;
    q[j] = col < dh ? Q[b * ld + h * dh + col] : 0.f;
    o[j] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int64_t kp = 0; kp <= p; ++kp) {
    const int64_t kb = zz_row_of_pos(kp, c, D);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxDhPerLane; ++j) {
      const int col = lane + 32 * j;
      if (col < dh) s = fmaf(q[j], K[kb * ld + hk * dh + col], s);
    }
    s = warp_sum(s) * scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);
    const float e = expf(s - mn);
    l = l * corr + e;
#pragma unroll
    for (int j = 0; j < kMaxDhPerLane; ++j) {
      const int col = lane + 32 * j;
      if (col < dh) o[j] = o[j] * corr + e * V[kb * ld + hk * dh + col];
    }
    m = mn;
  }
#pragma unroll
  for (int j = 0; j < kMaxDhPerLane; ++j) {
    const int col = lane + 32 * j;
    if (col < dh) O[b * ldo + h * dh + col] = o[j] / l;
  }
  if (lane == 0) LSE[(int64_t)h * S + b] = m + logf(l);
}

// Delta[h][i] = sum_c dO[i][h*dh+c] * O[i][h*dh+c]
__global__ void attn_f32_delta_kernel(const float* __restrict__ O, const float* __restrict__ dO,
                                      int64_t ld, float* __restrict__ delta, int64_t S, int H,
                                      int dh) {
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= S * H) return;
  const int64_t b = gw / H;
  const int h = (int)(gw - b * H);
  float s = 0.f;
  for (int col = lane; col < dh; col += 32) s += O[b * ld + h * dh + col] * dO[b * ld + h * dh + col];
  s = warp_sum(s);
  if (lane == 0) delta[(int64_t)h * S + b] = s;
}

// dQ_i = scale * sum_{pos(j)<=pos(i)} P_ij (dO_i.V_j - Delta_i) K_j, P_ij = exp(s_ij - LSE_i)
__global__ void attn_f32_dq_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                   const float* __restrict__ V, int64_t ld,
                                   const float* __restrict__ dO, int64_t lddo,
                                   const float* __restrict__ LSE, const float* __restrict__ delta,
                                   float* __restrict__ dQ, int64_t lddq, int64_t S, int H, int dh,
                                   int64_t c, int D, float scale, int G) {
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= S * H) return;
  const int64_t b = gw / H;
  const int h = (int)(gw - b * H);
  const int hk = h / G;
  const int64_t p = zz_pos_of_row(b, c, D);
  float q[kMaxDhPerLane], g[kMaxDhPerLane], dq[kMaxDhPerLane];
#pragma unroll
  for (int j = 0; j < kMaxDhPerLane; ++j) {
    const int col = lane + 32 * j;
    q[j] = col < dh ? Q[b * ld + h * dh + col] : 0.f;
    g[j] = col < dh ? dO[b * lddo + h * dh + col] : 0.f;
    dq[j] = 0.f;
  }
  const float lse = LSE[(int64_t)h * S + b], dl = delta[(int64_t)h * S + b];
  for (int64_t kp = 0; kp <= p; ++kp) {
    const int64_t kb = zz_row_of_pos(kp, c, D);
    float s = 0.f, dp = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxDhPerLane; ++j) {
      const int col = lane + 32 * j;
      if (col < dh) {
        s = fmaf(q[j], K[kb * ld + hk * dh + col], s);
        dp = fmaf(g[j], V[kb * ld + hk * dh + col], dp);
      }
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    const float P = expf(s * scale - lse);
    const float ds = P * (dp - dl) * scale;
#pragma unroll
    for (int j = 0; j < kMaxDhPerLane; ++j) {
      const int col = lane + 32 * j;
      if (col < dh) dq[j] = fmaf(ds, K[kb * ld + hk * dh + col], dq[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxDhPerLane; ++j) {
    const int col = lane + 32 * j;
    if (col < dh) dQ[b * lddq + h * dh + col] = dq[j];
  }
}

// dV_j = sum_{pos(i)>=pos(j)} P_ij dO_i ;  dK_j = scale * sum P_ij (dO_i.V_j - Delta_i) Q_i
__global__ void attn_f32_dkdv_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                     const float* __restrict__ V, int64_t ld,
                                     const float* __restrict__ dO, int64_t lddo,
                                     const float* __restrict__ LSE,
                                     const float* __restrict__ delta, float* __restrict__ dK,
                                     float* __restrict__ dV, int64_t lddkv, int64_t S, int H, int dh,
                                     int64_t c, int D, float scale, int G) {
  // one warp per (key row, K/V head); the G query heads of the group add up
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int Hk = H / G;
  if (gw >= S * Hk) return;
  const int64_t kb = gw / Hk;
  const int hk = (int)(gw - kb * Hk);
  const int64_t kpos = zz_pos_of_row(kb, c, D);
  float k[kMaxDhPerLane], v[kMaxDhPerLane], dk[kMaxDhPerLane], dv[kMaxDhPerLane];
#pragma unroll
  for (int j = 0; j < kMaxDhPerLane; ++j) {
    const int col = lane + 32 * j;
    k[j] = col < dh ? K[kb * ld + hk * dh + col] : 0.f;
    v[j] = col < dh ? V[kb * ld + hk * dh + col] : 0.f;
    dk[j] = dv[j] = 0.f;
  }
  for (int gi = 0; gi < G; ++gi) {
    const int h = hk * G + gi;
    for (int64_t qp = kpos; qp < S; ++qp) {
      const int64_t qb = zz_row_of_pos(qp, c, D);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxDhPerLane; ++j) {
        const int col = lane + 32 * j;
        if (col < dh) {
          s = fmaf(Q[qb * ld + h * dh + col], k[j], s);
          dp = fmaf(dO[qb * lddo + h * dh + col], v[j], dp);
        }
      }
      s = warp_sum(s);
      dp = warp_sum(dp);
      const float P = expf(s * scale - LSE[(int64_t)h * S + qb]);
      const float ds = P * (dp - delta[(int64_t)h * S + qb]) * scale;
#pragma unroll
      for (int j = 0; j < kMaxDhPerLane; ++j) {
        const int col = lane + 32 * j;
        if (col < dh) {
          dv[j] = fmaf(P, dO[qb * lddo + h * dh + col], dv[j]);
          dk[j] = fmaf(ds, Q[qb * ld + h * dh + col], dk[j]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxDhPerLane; ++j) {
    const int col = lane + 32 * j;
    if (col < dh) {
      dK[kb * lddkv + hk * dh + col] = dk[j];
      dV[kb * lddkv + hk * dh + col] = dv[j];
    }
  }
}

static int warp_grid(int64_t warps) { return (int)((warps * 32 + 255) / 256); }

tsp_status launch_attn_f32_fwd(const float* QKV, int64_t S, int H, int Hkv, int dh, int D, float* O,
                               float* LSE, cudaStream_t st) {
  const int d = H * dh, dk = Hkv * dh;
  const int64_t ld = d + 2 * (int64_t)dk;
  const int64_t c = S / (2 * D);
  Prof prof("attn_f32_fwd", st);
  attn_f32_fwd_kernel<<<warp_grid(S * H), 256, 0, st>>>(QKV, QKV + d, QKV + d + dk, ld, O, d, LSE,
                                                         S, H, dh, c, D, 1.0f / sqrtf((float)dh),
                                                         H / Hkv);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

tsp_status launch_attn_f32_bwd(const float* QKV, const float* O, const float* dO, const float* LSE,
                               float* delta, float* dQKV, int64_t S, int H, int Hkv, int dh, int D,
                               cudaStream_t st) {
  const int d = H * dh, dk = Hkv * dh;
  const int64_t ld = d + 2 * (int64_t)dk;
  const int64_t c = S / (2 * D);
  const float scale = 1.0f / sqrtf((float)dh);
  Prof prof("attn_f32_bwd", st, 3);
  attn_f32_delta_kernel<<<warp_grid(S * H), 256, 0, st>>>(O, dO, d, delta, S, H, dh);
  TSP_CUDA_TRY(cudaGetLastError());
  attn_f32_dq_kernel<<<warp_grid(S * H), 256, 0, st>>>(QKV, QKV + d, QKV + d + dk, ld, dO, d, LSE,
                                                        delta, dQKV, ld, S, H, dh, c, D, scale,
                                                        H / Hkv);
  TSP_CUDA_TRY(cudaGetLastError());
  attn_f32_dkdv_kernel<<<warp_grid(S * Hkv), 256, 0, st>>>(
      QKV, QKV + d, QKV + d + dk, ld, dO, d, LSE, delta, dQKV + d, dQKV + d + dk, ld, S, H, dh, c,
      D, scale, H / Hkv);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
