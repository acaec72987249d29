// attn_bwd.cu -- causal flash-attention backward over the zigzag layout (fp16
// tensor-core operands, fp32 accumulation).
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), section 2: the
// attention layer runs FlashAttention over the gathered K/V with zigzag
// partitioning balancing the causal work; this is the gradient of that step.
// With P_ij = exp(s_ij - LSE_i) (recomputed from the saved LSE):
//   dV_j = sum_i P_ij dO_i,   dP_ij = dO_i . V_j,   Delta_i = dO_i . O_i,
//   dS_ij = P_ij (dP_ij - Delta_i),
//   dQ_i = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i.
//
// Work unit = one CTA = (head, virtual rank r, key tile t of 128 keys): it
// owns key tile t of chunk r and the mirrored tile of chunk 2D-1-r, and walks
// the 64-row query tiles at positions >= the key tile.  The two causal query
// ranges add up to S + 128 rows for every (r, t), so CTAs are balanced.
// Per CTA: 8 warps, warp w owns keys 16w..16w+15 of the tile and keeps its
// dK, dV accumulators in registers; S^T and dP^T are computed key-major on
// mma.sync m16n8k16; dS goes through shared memory for dQ, which is
// accumulated in fp32 with vector atomics and converted to fp16 at the end.
#include "common.cuh"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BC = 128, BR = 64, DH = 128, NTHR = 256;
constexpr int ROWB = DH * 2;                 // 256 bytes per row
constexpr int SK_BYTES = BC * ROWB;          // 32 KB
constexpr int SQ_BYTES = BR * ROWB;          // 16 KB
constexpr int SDS_BYTES = BR * BC * 2;       // 16 KB
constexpr int OFF_K = 0, OFF_V = SK_BYTES, OFF_Q = 2 * SK_BYTES;   // Q[2], dO[2] follow
constexpr int OFF_DO = OFF_Q + 2 * SQ_BYTES;
constexpr int OFF_DS = OFF_DO + 2 * SQ_BYTES;
constexpr int OFF_L = OFF_DS + SDS_BYTES;    // float L[2][64], Dl[2][64]
constexpr int SMEM = OFF_L + 4 * BR * 4;
constexpr float kOperandScale = 256.f;            // P, dS scaling into fp16's normal range
constexpr float kOperandUnscale = 1.f / 256.f;

__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * ROWB + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void load_rows(uint32_t sdst, const ct_t* g, int64_t ld,
                                          int nrows) {
  for (int i = threadIdx.x; i < nrows * 16; i += NTHR) {
    const int row = i >> 4, ch = i & 15;
    cp_async16(sdst + swz(row, ch * 8), g + (int64_t)row * ld + ch * 8);
  }
}

struct BwdArgs {
  const ct_t* qkv;  // [S, 3d]
  const ct_t* dO;   // [S, d]
  const float* lse;          // [H, S] natural log
  const float* delta;        // [H, S]
  float* dq_acc;             // [S, d] fp32, zeroed
  ct_t* dqkv;       // [S, 3d]: dK, dV written here
  int64_t S, c;
  int D, d, n_kt;            // n_kt = c / 128
  float scale, scale_log2;
};

__device__ void key_tile(const BwdArgs& a, int h, int64_t k0, uint8_t* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ld = 3 * (int64_t)a.d;
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + OFF_K, sV = s0 + OFF_V, sDS = s0 + OFF_DS;
  float* sL = reinterpret_cast<float*>(smem + OFF_L);   // [2][64]
  float* sDl = sL + 2 * BR;                             // [2][64]
  const int64_t krow0 = zz_row_of_pos(k0, a.c, a.D);
  const ct_t* kg = a.qkv + krow0 * ld + a.d + h * DH;
  const int nq = (int)((a.S - k0) / BR);

  auto load_q = [&](int j, int b) {
    const int64_t q0 = k0 + (int64_t)j * BR;
    const int64_t qrow = zz_row_of_pos(q0, a.c, a.D);
    load_rows(s0 + OFF_Q + b * SQ_BYTES, a.qkv + qrow * ld + h * DH, ld, BR);
    load_rows(s0 + OFF_DO + b * SQ_BYTES, a.dO + qrow * a.d + h * DH, a.d, BR);
    if (threadIdx.x < BR) {
      cp_async4(smem_u32(sL + b * BR + threadIdx.x), a.lse + (int64_t)h * a.S + qrow + threadIdx.x);
    } else if (threadIdx.x < 2 * BR) {
      const int t = threadIdx.x - BR;
      cp_async4(smem_u32(sDl + b * BR + t), a.delta + (int64_t)h * a.S + qrow + t);
    }
  };
  load_rows(sK, kg, ld, BC);
  load_rows(sV, kg + a.d, ld, BC);
  load_q(0, 0);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  float dk[16][4], dv[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;
  const int64_t kw0 = k0 + warp * 16;
  const int64_t kp_lo = kw0 + (lane >> 2), kp_hi = kp_lo + 8;
  const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;  // A-fragment row (key)
  constexpr float LOG2E = 1.4426950408889634f;

  for (int j = 0; j < nq; ++j) {
    const int b = j & 1;
    if (j + 1 < nq) load_q(j + 1, b ^ 1);
    cp_async_commit();
    const uint32_t sQ = s0 + OFF_Q + b * SQ_BYTES, sdO = s0 + OFF_DO + b * SQ_BYTES;
    const float* L = sL + b * BR;
    const float* Dl = sDl + b * BR;
    const int64_t q0 = k0 + (int64_t)j * BR;
    const bool active = q0 + BR - 1 >= kw0;
    if (active) {
      float st[8][4], dp[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[i][e] = dp[i][e] = 0.f;
      // S^T = K Q^T and dP^T = V dO^T  (16 keys x 64 queries)
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t ka[4], va[4];
        const int col = ks * 16 + (lane >> 4) * 8;
        ldsm_x4(sK + swz(arow, col), ka[0], ka[1], ka[2], ka[3]);
        ldsm_x4(sV + swz(arow, col), va[0], va[1], va[2], va[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          const int q = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int bc = ks * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(sQ + swz(q, bc), b0, b1, b2, b3);
          mma_f16(st[2 * np], ka, b0, b1);
          mma_f16(st[2 * np + 1], ka, b2, b3);
          ldsm_x4(sdO + swz(q, bc), b0, b1, b2, b3);
          mma_f16(dp[2 * np], va, b0, b1);
          mma_f16(dp[2 * np + 1], va, b2, b3);
        }
      }
      // P^T and dS^T in place (st -> P, dp -> dS)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ql = i * 8 + (lane & 3) * 2 + e;
          const int64_t qp = q0 + ql;
          const float l2 = L[ql] * LOG2E, dl = Dl[ql];
          float p0 = exp2f(st[i][e] * a.scale_log2 - l2);
          float p1 = exp2f(st[i][2 + e] * a.scale_log2 - l2);
          if (kp_lo > qp) p0 = 0.f;
          if (kp_hi > qp) p1 = 0.f;
          st[i][e] = p0;
          st[i][2 + e] = p1;
          dp[i][e] = p0 * (dp[i][e] - dl);
          dp[i][2 + e] = p1 * (dp[i][2 + e] - dl);
        }
      }
      // dV += P^T dO ; dK += dS^T Q   (k-dimension = 64 queries).  P and dS
      // enter the fp16 MMAs scaled by 2^8 so that small probabilities stay in
      // fp16's normal range; the accumulators are scaled back at the end.
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          st[i][e] *= kOperandScale;
          dp[i][e] *= kOperandScale;
        }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t pa[4] = {pack_f16(st[2 * ks][0], st[2 * ks][1]),
                                pack_f16(st[2 * ks][2], st[2 * ks][3]),
                                pack_f16(st[2 * ks + 1][0], st[2 * ks + 1][1]),
                                pack_f16(st[2 * ks + 1][2], st[2 * ks + 1][3])};
        const uint32_t da[4] = {pack_f16(dp[2 * ks][0], dp[2 * ks][1]),
                                pack_f16(dp[2 * ks][2], dp[2 * ks][3]),
                                pack_f16(dp[2 * ks + 1][0], dp[2 * ks + 1][1]),
                                pack_f16(dp[2 * ks + 1][2], dp[2 * ks + 1][3])};
        const int q = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int dpi = 0; dpi < 8; ++dpi) {
          uint32_t b0, b1, b2, b3;
          const int col = dpi * 16 + (lane >> 4) * 8;
          ldsm_x4_t(sdO + swz(q, col), b0, b1, b2, b3);
          mma_f16(dv[2 * dpi], pa, b0, b1);
          mma_f16(dv[2 * dpi + 1], pa, b2, b3);
          ldsm_x4_t(sQ + swz(q, col), b0, b1, b2, b3);
          mma_f16(dk[2 * dpi], da, b0, b1);
          mma_f16(dk[2 * dpi + 1], da, b2, b3);
        }
      }
      // dS (query-major) into shared memory for dQ
      ct_t* ds = reinterpret_cast<ct_t*>(smem + OFF_DS);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ql = i * 8 + (lane & 3) * 2 + e;
          const int kl = warp * 16 + (lane >> 2);
          ds[swz(ql, kl) >> 1] = __float2half_rn(dp[i][e]);
          ds[swz(ql, kl + 8) >> 1] = __float2half_rn(dp[i][2 + e]);
        }
      }
    } else {
      ct_t* ds = reinterpret_cast<ct_t*>(smem + OFF_DS);
      for (int i = lane; i < BR * 16; i += 32) {
        const int ql = i >> 4, kl = warp * 16 + (i & 15);
        ds[swz(ql, kl) >> 1] = __float2half_rn(0.f);
      }
    }
    __syncthreads();
    // dQ partial = dS K: warp -> 16 queries x 64 dh columns
    {
      const int qw = (warp & 3) * 16, cw = (warp >> 2) * 64;
      float acc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      const int qa = qw + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {   // 128 keys
        uint32_t af[4];
        ldsm_x4(sDS + swz(qa, ks * 16 + (lane >> 4) * 8), af[0], af[1], af[2], af[3]);
        const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int dpi = 0; dpi < 4; ++dpi) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sK + swz(key, cw + dpi * 16 + (lane >> 4) * 8), b0, b1, b2, b3);
          mma_f16(acc[2 * dpi], af, b0, b1);
          mma_f16(acc[2 * dpi + 1], af, b2, b3);
        }
      }
      const int64_t qrow = zz_row_of_pos(q0, a.c, a.D) + qw + (lane >> 2);
      float* dst_lo = a.dq_acc + qrow * a.d + h * DH + cw + (lane & 3) * 2;
      float* dst_hi = dst_lo + 8 * (int64_t)a.d;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float sc = a.scale * kOperandUnscale;
        atomicAdd(reinterpret_cast<float2*>(dst_lo + i * 8), make_float2(acc[i][0] * sc, acc[i][1] * sc));
        atomicAdd(reinterpret_cast<float2*>(dst_hi + i * 8), make_float2(acc[i][2] * sc, acc[i][3] * sc));
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }
  // dK (scaled), dV -> fp16 rows of the key tile
  const int64_t row_lo = krow0 + warp * 16 + (lane >> 2), row_hi = row_lo + 8;
  ct_t* dk_lo = a.dqkv + row_lo * ld + a.d + h * DH;
  ct_t* dk_hi = a.dqkv + row_hi * ld + a.d + h * DH;
  const float skk = a.scale * kOperandUnscale;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
    *reinterpret_cast<uint32_t*>(dk_lo + col) = pack_f16(dk[i][0] * skk, dk[i][1] * skk);
    *reinterpret_cast<uint32_t*>(dk_hi + col) = pack_f16(dk[i][2] * skk, dk[i][3] * skk);
    *reinterpret_cast<uint32_t*>(dk_lo + a.d + col) =
        pack_f16(dv[i][0] * kOperandUnscale, dv[i][1] * kOperandUnscale);
    *reinterpret_cast<uint32_t*>(dk_hi + a.d + col) =
        pack_f16(dv[i][2] * kOperandUnscale, dv[i][3] * kOperandUnscale);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(NTHR, 1) attn_bwd_zigzag_kernel(const BwdArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int h = blockIdx.y;
  const int pair = blockIdx.x;
  const int r = pair / a.n_kt, t = pair - r * a.n_kt;
  const int64_t kA = (int64_t)r * a.c + (int64_t)t * BC;
  const int64_t kB = (int64_t)(2 * a.D - 1 - r) * a.c + (int64_t)(a.n_kt - 1 - t) * BC;
  key_tile(a, h, kA, smem);   // long query range first
  key_tile(a, h, kB, smem);
}

// Delta[h][row] = dO[row, head h] . O[row, head h]  (warp per row and head)
__global__ void attn_delta_kernel(const ct_t* __restrict__ o,
                                  const ct_t* __restrict__ dO, float* __restrict__ delta,
                                  int64_t S, int H, int d) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < S * H; w += nw) {
    const int64_t row = w / H;
    const int h = (int)(w - row * H);
    const uint2 ov = *reinterpret_cast<const uint2*>(o + row * d + h * DH + lane * 4);
    const uint2 gv = *reinterpret_cast<const uint2*>(dO + row * d + h * DH + lane * 4);
    float s = f16_lo(ov.x) * f16_lo(gv.x) + f16_hi(ov.x) * f16_hi(gv.x) +
              f16_lo(ov.y) * f16_lo(gv.y) + f16_hi(ov.y) * f16_hi(gv.y);
    s = warp_sum(s);
    if (lane == 0) delta[(int64_t)h * S + row] = s;
  }
}

// dQKV[:, 0:d] = fp16(dq_acc)
__global__ void dq_convert_kernel(const float* __restrict__ acc, ct_t* __restrict__ dqkv,
                                  int64_t S, int d) {
  const int64_t total4 = S * d / 4;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total4;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = t * 4;
    const int64_t row = e / d;
    const int col = (int)(e - row * d);
    const float4 v = reinterpret_cast<const float4*>(acc)[t];
    uint2 o;
    o.x = pack_f16(v.x, v.y);
    o.y = pack_f16(v.z, v.w);
    *reinterpret_cast<uint2*>(dqkv + row * 3 * (int64_t)d + col) = o;
  }
}

}  // namespace

tsp_status launch_attn_bwd_f16(const void* qkv, const void* o, const void* dO, const float* lse,
                                float* delta, float* dq_acc, void* dqkv, int64_t S, int H, int dh,
                                int D, cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BC != 0) return TSP_ERR_UNSUPPORTED;
  const int d = H * dh;
  {
  Prof prof("attn_bwd_prep", st);
  attn_delta_kernel<<<num_sms() * 8, 256, 0, st>>>((const ct_t*)o,
                                                   (const ct_t*)dO, delta, S, H, d);
  TSP_CUDA_TRY(cudaGetLastError());
  TSP_CUDA_TRY(cudaMemsetAsync(dq_acc, 0, (size_t)S * d * sizeof(float), st));
  }
  BwdArgs a;
  a.qkv = (const ct_t*)qkv;
  a.dO = (const ct_t*)dO;
  a.lse = lse;
  a.delta = delta;
  a.dq_acc = dq_acc;
  a.dqkv = (ct_t*)dqkv;
  a.S = S;
  a.c = c;
  a.D = D;
  a.d = d;
  a.n_kt = (int)(c / BC);
  a.scale = 1.0f / sqrtf((float)dh);
  a.scale_log2 = 1.4426950408889634f * a.scale;
  static bool attr = false;
  if (!attr) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_zigzag_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    attr = true;
  }
  dim3 grid((unsigned)(D * a.n_kt), (unsigned)H);
  {
    Prof prof("attn_bwd", st);
    attn_bwd_zigzag_kernel<<<grid, NTHR, SMEM, st>>>(a);
    TSP_CUDA_TRY(cudaGetLastError());
  }
  Prof prof("attn_bwd_dq_convert", st);
  dq_convert_kernel<<<num_sms() * 8, 256, 0, st>>>(dq_acc, (ct_t*)dqkv, S, d);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
