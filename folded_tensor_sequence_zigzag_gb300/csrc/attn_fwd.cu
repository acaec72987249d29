// attn_fwd.cu -- causal flash-attention forward over the zigzag layout (fp16
// tensor-core operands, fp32 softmax and accumulation).
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), section 2,
// attention-layer schedule: after the K/V all-gather every rank runs
// FlashAttention for its own tokens, and zigzag partitioning keeps the causal
// work of the ranks equal.  On one GPU the gathered K/V is the zigzag buffer
// itself: key position p is read from buffer row zz_row_of_pos(p).
//
// Work unit = one CTA = (head h, virtual rank r, q-tile t): it processes the
// 128 query rows of tile t in chunk r AND the mirrored tile n-1-t of chunk
// 2D-1-r (n = c/128 tiles per chunk).  Their causal key ranges add up to
// S + 128 keys for every (r, t), so every CTA carries the same work.
// Key tiles past a query tile's last row are never visited; only the two
// 64-key tiles on the diagonal are masked element-wise.
//
// Inner loop (per warp: 16 query rows, dh = 128; per CTA: 8 warps, 128 rows):
// S = Q K^T on mma.sync m16n8k16 fp16 -> fp32, online softmax in the log2
// domain with exp2f, O += P V with P re-packed from the accumulator
// registers.  K/V tiles (64 keys) are double-buffered with cp.async.
#include "common.cuh"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BQ = 128, BKV = 64, DH = 128, NTHR = 256;
constexpr int TILE_ROW_BYTES = DH * 2;  // 256
constexpr int SQ_BYTES = BQ * TILE_ROW_BYTES;
constexpr int SKV_BYTES = BKV * TILE_ROW_BYTES;
constexpr int SMEM = SQ_BYTES + 4 * SKV_BYTES;  // Q + 2 x (K, V)

// byte offset of (row, col) in a [rows][128] 16-bit tile, 16-byte chunks XOR-swizzled by row
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * TILE_ROW_BYTES + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
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

// rows [0, nrows) x 128 16-bit columns from global (row stride ld elements) into a swizzled tile
__device__ __forceinline__ void load_tile(uint32_t sdst, const ct_t* g, int64_t ld,
                                          int nrows) {
  for (int i = threadIdx.x; i < nrows * 16; i += NTHR) {
    const int row = i >> 4, ch = i & 15;
    cp_async16(sdst + swz(row, ch * 8), g + (int64_t)row * ld + ch * 8);
  }
}

struct AttnArgs {
  const ct_t* qkv;  // [S, 3d]
  ct_t* o;          // [S, d]
  float* lse;                // [H, S]
  int64_t S;
  int64_t c;
  int D, H, d, n_tiles;      // n_tiles = c / 128
  float scale_log2;          // log2(e) / sqrt(dh)
};

__device__ void attend_tile(const AttnArgs& a, int h, int64_t p0, uint8_t* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ld = 3 * (int64_t)a.d;
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + SQ_BYTES;
  // buffer b: K at sK0 + b*2*SKV, V at +SKV
  const int64_t qrow0 = zz_row_of_pos(p0, a.c, a.D);
  const ct_t* qg = a.qkv + qrow0 * ld + h * DH;
  const int nt = (int)((p0 + BQ) / BKV);

  auto kv_src = [&](int j) {
    const int64_t k0 = (int64_t)j * BKV;
    return a.qkv + zz_row_of_pos(k0, a.c, a.D) * ld + a.d + h * DH;
  };
  load_tile(sQ, qg, ld, BQ);
  {
    const ct_t* ks = kv_src(0);
    load_tile(sK0, ks, ld, BKV);
    load_tile(sK0 + SKV_BYTES, ks + a.d, ld, BKV);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  // Q fragments for this warp's 16 rows, 8 k-steps over dh
  uint32_t qf[8][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int col = ks * 16 + (lane >> 4) * 8;
      ldsm_x4(sQ + swz(r, col), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  const int64_t wq0 = p0 + warp * 16;                 // first query position of this warp
  const int64_t q_lo = wq0 + (lane >> 2), q_hi = q_lo + 8;

  for (int j = 0; j < nt; ++j) {
    const uint32_t sK = sK0 + (uint32_t)(j & 1) * 2 * SKV_BYTES;
    const uint32_t sV = sK + SKV_BYTES;
    if (j + 1 < nt) {
      const uint32_t nK = sK0 + (uint32_t)((j + 1) & 1) * 2 * SKV_BYTES;
      const ct_t* ks = kv_src(j + 1);
      load_tile(nK, ks, ld, BKV);
      load_tile(nK + SKV_BYTES, ks + a.d, ld, BKV);
    }
    cp_async_commit();
    const int64_t k0 = (int64_t)j * BKV;
    if (k0 <= wq0 + 15) {
      float s[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int col = ks * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(sK + swz(key, col), b0, b1, b2, b3);
          mma_f16(s[2 * np], qf[ks], b0, b1);
          mma_f16(s[2 * np + 1], qf[ks], b2, b3);
        }
      }
      const bool diag = k0 + BKV - 1 > wq0;
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v0 = s[i][e] * a.scale_log2, v1 = s[i][2 + e] * a.scale_log2;
          if (diag) {
            const int64_t kp = k0 + i * 8 + (lane & 3) * 2 + e;
            if (kp > q_lo) v0 = -INFINITY;
            if (kp > q_hi) v1 = -INFINITY;
          }
          s[i][e] = v0;
          s[i][2 + e] = v1;
          mx_lo = fmaxf(mx_lo, v0);
          mx_hi = fmaxf(mx_hi, v1);
        }
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float c_lo = exp2f(m_lo - mn_lo), c_hi = exp2f(m_hi - mn_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      float sum_lo = 0.f, sum_hi = 0.f;
      uint32_t pf[4][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p0v = exp2f(s[i][0] - mn_lo), p1v = exp2f(s[i][1] - mn_lo);
        const float p2v = exp2f(s[i][2] - mn_hi), p3v = exp2f(s[i][3] - mn_hi);
        sum_lo += p0v + p1v;
        sum_hi += p2v + p3v;
        // C fragment of n-tile i -> A fragment of k-step i/2
        pf[i >> 1][(i & 1) * 2 + 0] = pack_f16(p0v, p1v);
        pf[i >> 1][(i & 1) * 2 + 1] = pack_f16(p2v, p3v);
      }
      l_lo = l_lo * c_lo + sum_lo;
      l_hi = l_hi * c_hi + sum_hi;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= c_lo;
        o[i][1] *= c_lo;
        o[i][2] *= c_hi;
        o[i][3] *= c_hi;
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        // A fragment order: (rows lo, k 0-7), (rows hi, k 0-7), (rows lo, k 8-15), (rows hi, k 8-15)
        const uint32_t af[4] = {pf[ks][0], pf[ks][1], pf[ks][2], pf[ks][3]};
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          uint32_t b0, b1, b2, b3;
          const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = dp * 16 + (lane >> 4) * 8;
          ldsm_x4_t(sV + swz(key, col), b0, b1, b2, b3);
          mma_f16(o[2 * dp], af, b0, b1);
          mma_f16(o[2 * dp + 1], af, b2, b3);
        }
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }
  // finalize: full row sums across the quad
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float inv_lo = 1.f / l_lo, inv_hi = 1.f / l_hi;
  const int64_t row_lo = qrow0 + warp * 16 + (lane >> 2), row_hi = row_lo + 8;
  ct_t* out_lo = a.o + row_lo * a.d + h * DH;
  ct_t* out_hi = a.o + row_hi * a.d + h * DH;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
    *reinterpret_cast<uint32_t*>(out_lo + col) = pack_f16(o[i][0] * inv_lo, o[i][1] * inv_lo);
    *reinterpret_cast<uint32_t*>(out_hi + col) = pack_f16(o[i][2] * inv_hi, o[i][3] * inv_hi);
  }
  if ((lane & 3) == 0) {
    constexpr float LN2 = 0.69314718055994530942f;
    a.lse[(int64_t)h * a.S + row_lo] = (m_lo + log2f(l_lo)) * LN2;
    a.lse[(int64_t)h * a.S + row_hi] = (m_hi + log2f(l_hi)) * LN2;
  }
  __syncthreads();  // smem is reused by the next tile
}

__global__ void __launch_bounds__(NTHR, 1) attn_fwd_zigzag_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int h = blockIdx.y;
  const int pair = blockIdx.x;          // r * n_tiles + t
  const int r = pair / a.n_tiles, t = pair - r * a.n_tiles;
  const int64_t pA = (int64_t)r * a.c + (int64_t)t * BQ;                                  // chunk r
  const int64_t pB = (int64_t)(2 * a.D - 1 - r) * a.c + (int64_t)(a.n_tiles - 1 - t) * BQ;  // mirror
  attend_tile(a, h, pB, smem);
  attend_tile(a, h, pA, smem);
}

}  // namespace

int attn_fwd_smem_bytes() { return SMEM; }

tsp_status launch_attn_fwd_f16(const void* qkv, void* o, float* lse, int64_t S, int H, int dh,
                                int D, cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BQ != 0) return TSP_ERR_UNSUPPORTED;
  AttnArgs a;
  a.qkv = (const ct_t*)qkv;
  a.o = (ct_t*)o;
  a.lse = lse;
  a.S = S;
  a.c = c;
  a.D = D;
  a.H = H;
  a.d = H * dh;
  a.n_tiles = (int)(c / BQ);
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  static bool attr = false;
  if (!attr) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_zigzag_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    attr = true;
  }
  dim3 grid((unsigned)(D * a.n_tiles), (unsigned)H);
  Prof prof("attn_fwd", st);
  attn_fwd_zigzag_kernel<<<grid, NTHR, SMEM, st>>>(a);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
