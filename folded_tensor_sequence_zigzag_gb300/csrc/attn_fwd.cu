// attn_fwd.cu -- causal flash-attention forward over the zigzag layout on the
// 5th-generation tensor cores (tcgen05.mma kind::f16, fp16 operands, fp32
// accumulators in TMEM, softmax in fp32).
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), section 2,
// attention-layer schedule: after the K/V all-gather every rank runs
// FlashAttention for its own tokens, and zigzag partitioning keeps the causal
// work of the ranks equal.  On one GPU the gathered K/V is the zigzag buffer
// itself: key position p is read from buffer row zz_row_of_pos(p).
//
// Work unit = one CTA = (head h, virtual rank r, q-tile t): the 128 query rows
// of tile t in chunk r AND the mirrored tile n-1-t of chunk 2D-1-r
// (n = c/128).  Their causal key ranges add up to S + 128 keys for every
// (r, t), so every CTA carries the same work.  Key tiles past a query tile's
// last row are never visited; only the diagonal 128-key tile is masked.
//
// Per KV tile j (128 keys), warp-specialised:
//   warp 8   TMA producer: Q once per q-tile, K_j and V_j into a 2-stage ring
//            (128-byte swizzle; Q, K, V are column boxes of the Q|K|V buffer);
//   warp 9   TMEM allocator + MMA issuer: S_j = Q K_j^T into one of two
//            128-column TMEM buffers (issued one tile ahead), then
//            O += P_j V_j into a 128-column TMEM accumulator, with V read
//            MN-major (dh contiguous) straight from the buffer;
//   warps 0-7 softmax: query row = TMEM lane; warps w and w+4 share 32 rows,
//            each thread owning 64 of the 128 key columns (the row max is
//            exchanged through shared memory); p = 2^(s*scale*log2e - m) with
//            one FFMA + MUFU ex2 per score, written as fp16 into swizzled
//            shared memory (the A operand of the PV MMA).
// The running max m is only raised (and O rescaled in TMEM) when a warp's
// row max grows by more than 2^8 -- the result O/l is exact either way and
// p stays below 256.  All mbarrier waits are bounded (TSP_ERR_TIMEOUT).
#include <cstring>
#include <memory>

#include "common.cuh"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BQ = 128, BKV = 128, DH = 128;
constexpr int NSOFT = 256;                 // 8 softmax warps: two threads per query row
constexpr int NTHR = NSOFT + 64;           // + producer warp + MMA warp
constexpr int WARP_PROD = 8, WARP_MMA = 9;
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128x128 fp16 tile (two 64-column boxes)
constexpr int BOX_BYTES = TILE_BYTES / 2;  // 128 rows x 64 columns
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;        // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;    // 2 stages
constexpr int OFF_P = OFF_V + 2 * TILE_BYTES;    // 1 buffer
constexpr int OFF_X = OFF_P + TILE_BYTES;        // row-max exchange [2][2][128] + row-sum [2][128]
constexpr int OFF_BAR = OFF_X + 3 * 1024;
constexpr int SMEM = OFF_BAR + 256 + 1024;       // + 1 KB alignment slack
constexpr uint32_t TMEM_COLS = 512;              // S0 | S1 | O | (unused)
constexpr uint32_t TM_S = 0, TM_O = 256;
constexpr float RESCALE_LOG2 = 8.0f;             // lazy-rescale threshold (log2 units)

// Named barrier over the softmax warps that also ANDs a predicate: every
// participant leaves with the same verdict, so a loop exit taken on a failed
// (timed-out) wait is uniform and nobody is left at a barrier.
__device__ __forceinline__ bool softmax_bar_and(bool pred) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"(pred ? 1u : 0u), "r"(NSOFT)
      : "memory");
  return res != 0;
}

struct TcAttnArgs {
  CUtensorMap tm;       // Q|K|V buffer [S rows, 3d cols] fp16, box {64, 128}, 128B swizzle
  ct_t* o;              // [S, d]
  float* lse;           // [H, S]
  int64_t S, c;
  int D, d, n_tiles;    // n_tiles = c / 128
  float scale_log2;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

__global__ void __launch_bounds__(NTHR, 1) attn_fwd_tc_kernel(const __grid_constant__ TcAttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + OFF_BAR;
  // barrier map (8 bytes each)
  const uint32_t q_full = bars + 0;
  auto k_full = [&](int s) { return bars + 8u * (1 + s); };
  auto v_full = [&](int s) { return bars + 8u * (3 + s); };
  auto kv_empty = [&](int s) { return bars + 8u * (5 + s); };
  auto s_full = [&](int b) { return bars + 8u * (7 + b); };
  const uint32_t p_full = bars + 8u * 9;
  const uint32_t p_free = bars + 8u * 10;
  const uint32_t o_final = bars + 8u * 13;
  const uint32_t drain_bar = bars + 8u * 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_BAR + 168);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int pair = blockIdx.x;
  const int r = pair / a.n_tiles, t = pair - r * a.n_tiles;
  int64_t p0s[2];
  p0s[0] = (int64_t)(2 * a.D - 1 - r) * a.c + (int64_t)(a.n_tiles - 1 - t) * BQ;  // mirror tile
  p0s[1] = (int64_t)r * a.c + (int64_t)t * BQ;                                      // own tile

  // a device error recorded earlier (sticky until the host resets it) skips the work
  if (*(volatile int*)a.status != 0) return;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(kv_empty(s), 1);
      mbar_init(s_full(s), 1);
    }
    mbar_init(p_full, NSOFT);
    mbar_init(p_free, 1);
    mbar_init(o_final, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == WARP_PROD && lane == 0) tma_prefetch_desc(&a.tm);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint32_t it = 0;          // KV tiles processed by this CTA so far (both q-tiles)
  uint32_t k_issued = 0;    // producer: K/V stages issued
  uint32_t q_issued = 0;    // producer: Q tiles issued
  for (int tile = 0; tile < 2; ++tile) {
    const int64_t p0 = p0s[tile];
    const int n = (int)(p0 / BKV) + 1;
    const int64_t qrow0 = zz_row_of_pos(p0, a.c, a.D);
    if (warp == WARP_PROD) {
      // ------------------------------------------------------------ producer
      if (lane == 0 && !*abort_flag) {
        mbar_arrive_expect_tx(q_full, TILE_BYTES);
        tma_load_2d(base + OFF_Q, &a.tm, h * DH, (int)qrow0, q_full);
        tma_load_2d(base + OFF_Q + BOX_BYTES, &a.tm, h * DH + 64, (int)qrow0, q_full);
        ++q_issued;
        for (int j = 0; j < n; ++j) {
          const uint32_t cur = it + j, st = cur & 1u;
          if (!mbar_wait(kv_empty(st), ((cur >> 1) & 1u) ^ 1u, a.status, abort_flag, a.limit_ns))
            break;
          const int krow = (int)zz_row_of_pos((int64_t)j * BKV, a.c, a.D);
          const uint32_t sk = base + OFF_K + st * TILE_BYTES, sv = base + OFF_V + st * TILE_BYTES;
          mbar_arrive_expect_tx(k_full(st), TILE_BYTES);
          tma_load_2d(sk, &a.tm, a.d + h * DH, krow, k_full(st));
          tma_load_2d(sk + BOX_BYTES, &a.tm, a.d + h * DH + 64, krow, k_full(st));
          mbar_arrive_expect_tx(v_full(st), TILE_BYTES);
          tma_load_2d(sv, &a.tm, 2 * a.d + h * DH, krow, v_full(st));
          tma_load_2d(sv + BOX_BYTES, &a.tm, 2 * a.d + h * DH + 64, krow, v_full(st));
          ++k_issued;
        }
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && !*abort_flag) {
        constexpr uint32_t idesc_s = idesc_f16_f32(BQ, BKV, false, false, false);
        constexpr uint32_t idesc_o = idesc_f16_f32(BQ, DH, false, true, false);
        bool ok = mbar_wait(q_full, (uint32_t)tile & 1u, a.status, abort_flag, a.limit_ns);
        auto issue_s = [&](uint32_t cur) -> bool {
          const uint32_t st = cur & 1u;
          if (!mbar_wait(k_full(st), (cur >> 1) & 1u, a.status, abort_flag, a.limit_ns)) return false;
          tc_fence_after();
          const uint32_t sq = base + OFF_Q, sk = base + OFF_K + st * TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            umma_f16_ss(tmem + TM_S + st * 128, sdesc_sw128(sq + off, 16, 1024),
                        sdesc_sw128(sk + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full(st));
          return true;
        };
        if (ok) ok = issue_s(it);
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t cur = it + j, b = cur & 1u;
          if (j + 1 < n && !(ok = issue_s(cur + 1))) break;
          if (!mbar_wait(p_full, cur & 1u, a.status, abort_flag, a.limit_ns) ||
              !mbar_wait(v_full(b), (cur >> 1) & 1u, a.status, abort_flag, a.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sp = base + OFF_P, sv = base + OFF_V + b * TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            const uint32_t poff = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            umma_f16_ss(tmem + TM_O, sdesc_sw128(sp + poff, 16, 1024),
                        sdesc_sw128(sv + kk * 2048, BOX_BYTES, 1024), idesc_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(kv_empty(b));
          umma_commit(p_free);
        }
        if (ok) {
          umma_commit(o_final);
        } else {
          umma_commit(drain_bar);
          drain_wait(drain_bar, 0, a.limit_ns);
        }
      }
    } else {
      // ------------------------------------------------------------ softmax
      const int quarter = warp & 3, half = warp >> 2;
      const int row = quarter * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
      float* xmax = reinterpret_cast<float*>(gbase + OFF_X);  // [2 parity][2 half][128 rows]
      float* lsum = xmax + 512;                               // [2 half][128 rows]
      uint8_t* prow = gbase + OFF_P + half * BOX_BYTES + (row >> 3) * 1024 + (row & 7) * 128;
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t cur = it + j, b = cur & 1u;
        bool okl = ok && mbar_wait(s_full(b), (cur >> 1) & 1u, a.status, abort_flag, a.limit_ns);
        okl = __all_sync(0xffffffffu, okl);
        uint32_t sr[2][32];
        float mxp = -INFINITY;
        if (okl) {
          tc_fence_after();
          tmem_ld32(lane_base + TM_S + b * 128 + half * 64, sr[0]);
          tmem_ld32(lane_base + TM_S + b * 128 + half * 64 + 32, sr[1]);
          tmem_wait_ld();
          if (j == n - 1) {  // diagonal tile: key index > query index is masked
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (half * 64 + q * 32 + e > row) sr[q][e] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e) mxp = fmaxf(mxp, __uint_as_float(sr[q][e]));
          xmax[b * 256 + half * 128 + row] = mxp;
        }
        ok = softmax_bar_and(okl);
        if (!ok) break;
        const float mx = fmaxf(mxp, xmax[b * 256 + (1 - half) * 128 + row]) * a.scale_log2;
        // lazy rescale, decided per warp (TMEM access is warp-collective); the
        // two warps of a row pair see the same maxima and decide alike
        const bool mine = mx > m_used + RESCALE_LOG2;
        const bool resc = __any_sync(0xffffffffu, mine);
        float alpha = 1.f;
        if (resc) {
          const float m_new = mine ? mx : m_used;
          alpha = ex2_approx(m_used - m_new);   // 0 on the first tile, 1 if unchanged
          l *= alpha;
          m_used = m_new;
        }
        // PV(cur-1) must have finished before P is overwritten or O rescaled
        if (cur >= 1) {
          bool wok = mbar_wait(p_free, (cur - 1) & 1u, a.status, abort_flag, a.limit_ns);
          if (!__all_sync(0xffffffffu, wok)) {
            ok = false;
            continue;  // the next vote (or the epilogue's) takes everyone out
          }
          tc_fence_after();
        }
        if (resc && j > 0) {
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {
            uint32_t ov[32];
            tmem_ld32(lane_base + TM_O + half * 64 + q * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(lane_base + TM_O + half * 64 + q * 32, ov);
          }
          tmem_wait_st();
        }
        const float neg_m = -m_used;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0v = ex2_approx(fmaf(__uint_as_float(sr[q][e]), a.scale_log2, neg_m));
            const float p1v = ex2_approx(fmaf(__uint_as_float(sr[q][e + 1]), a.scale_log2, neg_m));
            sum += p0v + p1v;
            pk[e >> 1] = pack_f16(p0v, p1v);
          }
          // keys half*64 + q*32 .. +31 -> 16-byte chunks 4q .. 4q+3 of box `half`
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int chunk = q * 4 + c;
            *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
        }
        l += sum;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      // epilogue: O / l -> fp16 rows, LSE
      bool eok = ok && mbar_wait(o_final, (uint32_t)tile & 1u, a.status, abort_flag, a.limit_ns);
      eok = __all_sync(0xffffffffu, eok);
      if (eok) lsum[half * 128 + row] = l;
      eok = softmax_bar_and(eok);
      if (eok) {
        tc_fence_after();
        const float l_tot = l + lsum[(1 - half) * 128 + row];
        const float inv = 1.f / l_tot;
        ct_t* orow = a.o + (qrow0 + row) * (int64_t)a.d + h * DH + half * 64;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          uint32_t ov[32];
          tmem_ld32(lane_base + TM_O + half * 64 + q * 32, ov);
          tmem_wait_ld();
          uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(
                pack_f16(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv),
                pack_f16(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv),
                pack_f16(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv),
                pack_f16(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv));
        }
        if (half == 0) {
          constexpr float LN2 = 0.69314718055994530942f;
          a.lse[(int64_t)h * a.S + qrow0 + row] = (m_used + __log2f(l_tot)) * LN2;
        }
      }
      tc_fence_before();
    }
    it += (uint32_t)n;
    __syncthreads();  // Q, O and the barriers' phases are reused by the next q-tile
    tc_fence_after();
  }
  // drain: copies the producer issued that nobody consumed (abort path only)
  if (warp == WARP_PROD && lane == 0 && *abort_flag) {
    const uint32_t n_out = k_issued < 2u ? k_issued : 2u;
    for (uint32_t jj = k_issued - n_out; jj < k_issued; ++jj) {
      drain_wait(k_full(jj & 1u), (jj >> 1) & 1u, a.limit_ns);
      drain_wait(v_full(jj & 1u), (jj >> 1) & 1u, a.limit_ns);
    }
    if (q_issued > 0) drain_wait(q_full, (q_issued - 1) & 1u, a.limit_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_attn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

tsp_status launch_attn_fwd_f16(const void* qkv, void* o, float* lse, int64_t S, int H, int dh,
                               int D, cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BQ != 0) return TSP_ERR_UNSUPPORTED;
  if (S > (int64_t)INT32_MAX) return TSP_ERR_UNSUPPORTED;
  const int d = H * dh;
  if (((uintptr_t)qkv & 15u) || ((3 * d * 2) % 16)) return TSP_ERR_INVALID_ARG;
  TcAttnArgs* a = new TcAttnArgs();
  std::unique_ptr<TcAttnArgs> guard(a);
  memset(a, 0, sizeof(TcAttnArgs));
  EncodeTiledFn fn = encode_fn_attn();
  if (!fn) return TSP_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)(3 * d), (cuuint64_t)S};
  const cuuint64_t strides[1] = {(cuuint64_t)(3 * d * 2)};
  const cuuint32_t box[2] = {64u, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  if (fn(&a->tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(qkv), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TSP_ERR_CUDA;
  a->o = (ct_t*)o;
  a->lse = lse;
  a->S = S;
  a->c = c;
  a->D = D;
  a->d = d;
  a->n_tiles = (int)(c / BQ);
  a->scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  a->status = status_word();
  a->limit_ns = wait_limit_ns();
  static bool attr = false;
  if (!attr) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    attr = true;
  }
  dim3 grid((unsigned)(D * a->n_tiles), (unsigned)H);
  Prof prof("attn_fwd", st);
  attn_fwd_tc_kernel<<<grid, NTHR, SMEM, st>>>(*a);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
