// attn_bwd.cu -- causal flash-attention backward over the zigzag layout on the
// 5th-generation tensor cores (tcgen05.mma kind::f16, fp16 operands, fp32
// accumulators in TMEM).
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
// Work unit = one CTA = (head, virtual rank r, key tile t of 128 keys): key
// tile t of chunk r and the mirrored tile of chunk 2D-1-r, each walking the
// 64-row query tiles at positions >= the tile; the two query ranges add up to
// S + 128 rows for every (r, t), so CTAs are balanced.  Per query tile:
//   warp 12  TMA producer: K, V once per key tile; Q_i, dO_i (+ LSE_i, Delta_i
//            by bulk copy) into a 3-stage ring;
//   warp 13  MMA issuer: S^T = K Q_i^T and dP^T = V dO_i^T (M = 128 keys,
//            N = 64 queries) for tile i+1 as soon as tile i's were read; then
//            dV += P^T dO_i, dK += dS^T Q_i (TMEM accumulators across every
//            query tile) and dQ_i^T = K^T dS^T (M = 128 dh, N = 64 queries);
//   warps 0-7 (key = TMEM lane; warps w and w+4 share 32 keys, each thread
//            owning 32 of the 64 query columns): P = 2^(s*scale*log2e - LSE*log2e),
//            dS = P (dP - Delta), both written as fp16 (scaled by 2^8 to keep
//            small probabilities in fp16's normal range) into swizzled smem,
//            which serves as the K-major A operand of dV/dK and, unchanged, as
//            the MN-major B operand of dQ^T; at the end dK, dV -> fp16 rows;
//   warps 8-11 (thread = dh = TMEM lane): drain dQ_i^T from TMEM into the fp32
//            dQ accumulator with warp-coalesced atomics.
// All mbarrier waits are bounded (TSP_ERR_TIMEOUT) and every loop exit is
// uniform across the threads that share a barrier.
#include <cstring>
#include <memory>

#include "common.cuh"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BC = 128, BR = 64, DH = 128;
constexpr int NSOFT = 256;                 // 8 warps: two threads per key row
constexpr int NTHR = NSOFT + 128 + 64;     // + 4 dQ-drain warps + producer + MMA
constexpr int WARP_PROD = 12, WARP_MMA = 13;   // warps 8-11 drain dQ
constexpr int KT_BYTES = BC * DH * 2;      // 32 KB: 128 keys x 128 dh
constexpr int QT_BYTES = BR * DH * 2;      // 16 KB: 64 queries x 128 dh
constexpr int PT_BYTES = BC * BR * 2;      // 16 KB: 128 keys x 64 queries
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KT_BYTES;
constexpr int QSTAGES = 3;                        // Q/dO ring depth (covers TMA latency)
constexpr int OFF_Q = OFF_V + KT_BYTES;            // QSTAGES stages
constexpr int OFF_DO = OFF_Q + QSTAGES * QT_BYTES; // QSTAGES stages
constexpr int OFF_P = OFF_DO + QSTAGES * QT_BYTES; // 2 buffers
constexpr int OFF_DS = OFF_P + 2 * PT_BYTES;       // 2 buffers
constexpr int OFF_L = OFF_DS + 2 * PT_BYTES;       // [QSTAGES][LSE 64 | Delta 64] floats
constexpr int OFF_BAR = OFF_L + QSTAGES * 2 * BR * 4;
constexpr int SMEM = OFF_BAR + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_DQ = 128, TM_DV = 256, TM_DK = 384;
constexpr float kOperandScale = 256.f;           // P, dS scaling into fp16's normal range
constexpr float kOperandUnscale = 1.f / 256.f;

struct TcBwdArgs {
  CUtensorMap tm_qkv;   // Q|K|V [S, 3d] fp16, box {64, 64}, 128B swizzle
  CUtensorMap tm_do;    // dO [S, d] fp16, box {64, 64}, 128B swizzle
  const float* lse;     // [H, S]
  const float* delta;   // [H, S]
  float* dq_acc;        // [S, d] fp32, zeroed
  ct_t* dqkv;           // [S, 3d]: dK, dV written here
  int64_t S, c;
  int D, d, n_kt;       // n_kt = c / 128
  float scale, scale_log2;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// Named barrier of the P/dS warps (id 1, 256 threads) or of the dQ warps
// (id 2, 128 threads) that ANDs a predicate: a loop exit taken on a failed
// (timed-out) wait is the same for all of them.
__device__ __forceinline__ bool group_bar_and(int id, int nthreads, bool pred) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return res != 0;
}

__global__ void __launch_bounds__(NTHR, 1) attn_bwd_tc_kernel(const __grid_constant__ TcBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + OFF_BAR;
  const uint32_t kv_full = bars;
  auto qd_full = [&](uint32_t s) { return bars + 8u * (1 + s); };       // 1..3
  auto qd_empty = [&](uint32_t s) { return bars + 8u * (4 + s); };      // 4..6
  const uint32_t s_full = bars + 8u * 7;
  const uint32_t s_free = bars + 8u * 8;
  auto p_full = [&](uint32_t b) { return bars + 8u * (9 + b); };
  auto p_free = [&](uint32_t b) { return bars + 8u * (11 + b); };
  const uint32_t dq_full = bars + 8u * 13;
  const uint32_t dq_empty = bars + 8u * 14;
  const uint32_t kv_done = bars + 8u * 15;
  const uint32_t drain_bar = bars + 8u * 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_BAR + 168);

  if (*(volatile int*)a.status != 0) return;  // an earlier device error skips the work

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int pair = blockIdx.x;
  const int r = pair / a.n_kt, t = pair - r * a.n_kt;
  int64_t k0s[2];
  k0s[0] = (int64_t)r * a.c + (int64_t)t * BC;                                      // long range
  k0s[1] = (int64_t)(2 * a.D - 1 - r) * a.c + (int64_t)(a.n_kt - 1 - t) * BC;      // mirror

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < QSTAGES; ++s) {
      mbar_init(qd_full(s), 1);
      mbar_init(qd_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(p_full(b), NSOFT);
      mbar_init(p_free(b), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, NSOFT);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(kv_done, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == WARP_PROD && lane == 0) {
    tma_prefetch_desc(&a.tm_qkv);
    tma_prefetch_desc(&a.tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  float* sLD = reinterpret_cast<float*>(gbase + OFF_L);  // [stage][LSE 64 | Delta 64]
  // Q/dO ring position of query tile `cur` (CTA-wide counter)
  auto qst = [](uint32_t cur) { return cur % QSTAGES; };
  auto qph = [](uint32_t cur) { return (cur / QSTAGES) & 1u; };

  uint32_t it = 0;        // query tiles processed by this CTA so far
  uint32_t q_issued = 0, kv_issued = 0;
  for (int tile = 0; tile < 2; ++tile) {
    const int64_t k0 = k0s[tile];
    const int nq = (int)((a.S - k0) / BR);
    const int64_t krow0 = zz_row_of_pos(k0, a.c, a.D);
    if (warp == WARP_PROD) {
      // ------------------------------------------------------------ producer
      if (lane == 0 && !*abort_flag) {
        mbar_arrive_expect_tx(kv_full, 2 * KT_BYTES);
#pragma unroll
        for (int jh = 0; jh < 2; ++jh)
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            const uint32_t off = jh * (KT_BYTES / 2) + rh * (KT_BYTES / 4);
            tma_load_2d(base + OFF_K + off, &a.tm_qkv, a.d + h * DH + 64 * jh,
                        (int)(krow0 + 64 * rh), kv_full);
            tma_load_2d(base + OFF_V + off, &a.tm_qkv, 2 * a.d + h * DH + 64 * jh,
                        (int)(krow0 + 64 * rh), kv_full);
          }
        ++kv_issued;
        for (int j = 0; j < nq; ++j) {
          const uint32_t cur = it + j, st = qst(cur);
          if (!mbar_wait(qd_empty(st), qph(cur) ^ 1u, a.status, abort_flag, a.limit_ns))
            break;
          const int64_t qrow = zz_row_of_pos(k0 + (int64_t)j * BR, a.c, a.D);
          const uint32_t fb = qd_full(st);
          mbar_arrive_expect_tx(fb, 2 * QT_BYTES + 2 * BR * 4);
#pragma unroll
          for (int jh = 0; jh < 2; ++jh) {
            tma_load_2d(base + OFF_Q + st * QT_BYTES + jh * (QT_BYTES / 2), &a.tm_qkv,
                        h * DH + 64 * jh, (int)qrow, fb);
            tma_load_2d(base + OFF_DO + st * QT_BYTES + jh * (QT_BYTES / 2), &a.tm_do,
                        h * DH + 64 * jh, (int)qrow, fb);
          }
          const uint32_t sl = smem_u32(sLD + st * 2 * BR);
          bulk_load(sl, a.lse + (int64_t)h * a.S + qrow, BR * 4, fb);
          bulk_load(sl + BR * 4, a.delta + (int64_t)h * a.S + qrow, BR * 4, fb);
          ++q_issued;
        }
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && !*abort_flag) {
        constexpr uint32_t id_s = idesc_f16_f32(BC, BR, false, false, false);   // S^T, dP^T
        constexpr uint32_t id_kv = idesc_f16_f32(BC, DH, false, true, false);   // dV, dK
        constexpr uint32_t id_q = idesc_f16_f32(DH, BR, true, true, false);     // dQ^T
        bool ok = mbar_wait(kv_full, (uint32_t)tile & 1u, a.status, abort_flag, a.limit_ns);
        // base descriptors, computed once: the issue loops only add constants
        const uint64_t dK_k = sdesc_sw128(base + OFF_K, 16, 1024);            // K, K-major
        const uint64_t dV_k = sdesc_sw128(base + OFF_V, 16, 1024);            // V, K-major
        const uint64_t dK_mn = sdesc_sw128(base + OFF_K, KT_BYTES / 2, 1024); // K^T, MN-major
        const uint64_t dQ_k = sdesc_sw128(base + OFF_Q, 16, 1024);            // Q stages, K-major
        const uint64_t dDO_k = sdesc_sw128(base + OFF_DO, 16, 1024);          // dO stages, K-major
        const uint64_t dQ_mn = sdesc_sw128(base + OFF_Q, QT_BYTES / 2, 1024); // Q stages, MN-major
        const uint64_t dDO_mn = sdesc_sw128(base + OFF_DO, QT_BYTES / 2, 1024);
        const uint64_t dP_k = sdesc_sw128(base + OFF_P, 16, 1024);            // P^T buffers
        const uint64_t dDS_k = sdesc_sw128(base + OFF_DS, 16, 1024);          // dS^T buffers
        const uint64_t dDS_mn = sdesc_sw128(base + OFF_DS, PT_BYTES, 1024);   // dS, MN-major
        auto issue_s = [&](uint32_t cur) -> bool {
          const uint32_t st = qst(cur);
          if (!mbar_wait(qd_full(st), qph(cur), a.status, abort_flag, a.limit_ns))
            return false;
          if (cur >= 1 && !mbar_wait(s_free, (cur - 1) & 1u, a.status, abort_flag, a.limit_ns))
            return false;
          tc_fence_after();
          const uint64_t bq = sdesc_add(dQ_k, st * QT_BYTES), bdo = sdesc_add(dDO_k, st * QT_BYTES);
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * (KT_BYTES / 2) + (kk & 3) * 32;
            const uint32_t boff = (kk >> 2) * (QT_BYTES / 2) + (kk & 3) * 32;
            umma_f16_ss_hot(tmem + TM_S, sdesc_add(dK_k, aoff), sdesc_add(bq, boff), id_s,
                            kk > 0 ? 1u : 0u);
            umma_f16_ss_hot(tmem + TM_DP, sdesc_add(dV_k, aoff), sdesc_add(bdo, boff), id_s,
                            kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
          return true;
        };
        if (ok) ok = issue_s(it);
        for (int j = 0; j < nq && ok; ++j) {
          const uint32_t cur = it + j, st = qst(cur), pb = cur & 1u;
          if (j + 1 < nq && !(ok = issue_s(cur + 1))) break;
          if (!mbar_wait(p_full(pb), (cur >> 1) & 1u, a.status, abort_flag, a.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ap = sdesc_add(dP_k, pb * PT_BYTES), ads = sdesc_add(dDS_k, pb * PT_BYTES);
          const uint64_t bdo = sdesc_add(dDO_mn, st * QT_BYTES), bq = sdesc_add(dQ_mn, st * QT_BYTES);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < BR / 16; ++kk) {
            const uint32_t acc = kk > 0 ? 1u : acc0;
            umma_f16_ss_hot(tmem + TM_DV, sdesc_add(ap, kk * 32), sdesc_add(bdo, kk * 2048), id_kv,
                            acc);
            umma_f16_ss_hot(tmem + TM_DK, sdesc_add(ads, kk * 32), sdesc_add(bq, kk * 2048), id_kv,
                            acc);
          }
          umma_commit(qd_empty(st));
          if (cur >= 1 && !mbar_wait(dq_empty, (cur - 1) & 1u, a.status, abort_flag, a.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bds = sdesc_add(dDS_mn, pb * PT_BYTES);
#pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            umma_f16_ss_hot(tmem + TM_DQ, sdesc_add(dK_mn, kk * 2048), sdesc_add(bds, kk * 2048),
                            id_q, kk > 0 ? 1u : 0u);
          umma_commit(dq_full);
          umma_commit(p_free(pb));
        }
        if (ok) {
          umma_commit(kv_done);
        } else {
          umma_commit(drain_bar);
          drain_wait(drain_bar, 0, a.limit_ns);
        }
      }
    } else if (warp < 8) {
      // ------------------------------------------------------------ P, dS (thread = key)
      const int quarter = warp & 3, half = warp >> 2;
      const int row = quarter * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
      const int64_t kp = k0 + row;
      constexpr float LOG2E = 1.4426950408889634f;
      bool ok = true;
      for (int j = 0; j < nq; ++j) {
        const uint32_t cur = it + j, st = qst(cur), pb = cur & 1u;
        bool okl = ok && mbar_wait(s_full, cur & 1u, a.status, abort_flag, a.limit_ns);
        okl = okl && mbar_wait(qd_full(st), qph(cur), a.status, abort_flag, a.limit_ns);
        // buffer pb was last read by the MMAs of query tile cur-2
        if (okl && cur >= 2)
          okl = mbar_wait(p_free(pb), ((cur - 2) >> 1) & 1u, a.status, abort_flag, a.limit_ns);
        ok = group_bar_and(1, NSOFT, okl);
        if (!ok) break;
        uint32_t sv[32], dv[32];
        tc_fence_after();
        tmem_ld32(lane_base + TM_S + half * 32, sv);
        tmem_ld32(lane_base + TM_DP + half * 32, dv);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free);
        const float* L = sLD + st * 2 * BR;
        const float* Dl = L + BR;
        const int64_t q0 = k0 + (int64_t)j * BR;
        const bool diag = q0 < k0 + BC;
        uint8_t* prow = gbase + OFF_P + pb * PT_BYTES + (row >> 3) * 1024 + (row & 7) * 128;
        uint8_t* drow = gbase + OFF_DS + pb * PT_BYTES + (row >> 3) * 1024 + (row & 7) * 128;
        // this thread's 32 query columns, 8 at a time (LSE, Delta read as float4)
        const float neg_l_scale = -LOG2E;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int qb = half * 32 + c * 8;
          const float4 l0 = *reinterpret_cast<const float4*>(L + qb);
          const float4 l1 = *reinterpret_cast<const float4*>(L + qb + 4);
          const float4 d0 = *reinterpret_cast<const float4*>(Dl + qb);
          const float4 d1 = *reinterpret_cast<const float4*>(Dl + qb + 4);
          const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
          const float dlv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
          uint32_t pk[4], dk[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float pp[2], dd[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int x = c * 8 + e + u;
              float p = ex2_approx(fmaf(__uint_as_float(sv[x]), a.scale_log2, lv[e + u] * neg_l_scale));
              if (diag && kp > q0 + qb + e + u) p = 0.f;
              pp[u] = p * kOperandScale;
              dd[u] = pp[u] * (__uint_as_float(dv[x]) - dlv[e + u]);
            }
            pk[e >> 1] = pack_f16(pp[0], pp[1]);
            dk[e >> 1] = pack_f16(dd[0], dd[1]);
          }
          const int chunk = half * 4 + c;
          const uint32_t off = (uint32_t)((chunk ^ (row & 7)) << 4);
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(drow + off) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(p_full(pb));
      }
      // dK, dV of this key tile -> fp16 rows
      bool eok = ok && mbar_wait(kv_done, (uint32_t)tile & 1u, a.status, abort_flag, a.limit_ns);
      eok = __all_sync(0xffffffffu, eok);
      if (eok) {
        tc_fence_after();
        ct_t* dkrow = a.dqkv + (krow0 + row) * 3 * (int64_t)a.d + a.d + h * DH;
        const float skk = a.scale * kOperandUnscale;
        {
          const int part = half;   // warps 0-3 write dK, warps 4-7 write dV
          const float mul = part == 0 ? skk : kOperandUnscale;
          ct_t* out = dkrow + part * a.d;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            tmem_ld32(lane_base + (part == 0 ? TM_DK : TM_DV) + q * 32, v);
            tmem_wait_ld();
            uint4* dst = reinterpret_cast<uint4*>(out + q * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c] = make_uint4(
                  pack_f16(__uint_as_float(v[8 * c]) * mul, __uint_as_float(v[8 * c + 1]) * mul),
                  pack_f16(__uint_as_float(v[8 * c + 2]) * mul, __uint_as_float(v[8 * c + 3]) * mul),
                  pack_f16(__uint_as_float(v[8 * c + 4]) * mul, __uint_as_float(v[8 * c + 5]) * mul),
                  pack_f16(__uint_as_float(v[8 * c + 6]) * mul, __uint_as_float(v[8 * c + 7]) * mul));
          }
        }
      }
      tc_fence_before();
    } else {
      // ------------------------------------------------------------ dQ drain (thread = dh)
      const int quarter = warp & 3;
      const int dh = quarter * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
      const float sc = a.scale * kOperandUnscale;
      bool ok = true;
      for (int j = 0; j < nq; ++j) {
        const uint32_t cur = it + j;
        bool okl = ok && mbar_wait(dq_full, cur & 1u, a.status, abort_flag, a.limit_ns);
        ok = group_bar_and(2, 128, okl);
        if (!ok) break;
        uint32_t v[2][32];
        tc_fence_after();
        tmem_ld32(lane_base + TM_DQ, v[0]);
        tmem_ld32(lane_base + TM_DQ + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(dq_empty);
        const int64_t qrow = zz_row_of_pos(k0 + (int64_t)j * BR, a.c, a.D);
        float* dst = a.dq_acc + qrow * a.d + h * DH + dh;
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            atomicAdd(dst + (int64_t)(q * 32 + e) * a.d, __uint_as_float(v[q][e]) * sc);
      }
      tc_fence_before();
    }
    it += (uint32_t)nq;
    __syncthreads();   // K/V tiles, TMEM accumulators and barrier phases move on
    tc_fence_after();
  }
  if (warp == WARP_PROD && lane == 0 && *abort_flag) {
    const uint32_t n_out = q_issued < (uint32_t)QSTAGES ? q_issued : (uint32_t)QSTAGES;
    for (uint32_t jj = q_issued - n_out; jj < q_issued; ++jj)
      drain_wait(qd_full(qst(jj)), qph(jj), a.limit_ns);
    if (kv_issued > 0) drain_wait(kv_full, (kv_issued - 1) & 1u, a.limit_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Delta[h][row] = dO[row, head h] . O[row, head h]  (warp per row and head)
__global__ void attn_delta_kernel(const ct_t* __restrict__ o, const ct_t* __restrict__ dO,
                                  float* __restrict__ delta, int64_t S, int H, int d) {
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_bwd() {
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

// Row-major fp16 [rows, cols] with box {64 columns, 64 rows}, 128-byte swizzle.
bool map_2d(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows) {
  EncodeTiledFn fn = encode_fn_bwd();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  const cuuint32_t box[2] = {64u, 64u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

tsp_status launch_attn_bwd_f16(const void* qkv, const void* o, const void* dO, const float* lse,
                               float* delta, float* dq_acc, void* dqkv, int64_t S, int H, int dh,
                               int D, cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BC != 0 || S > (int64_t)INT32_MAX) return TSP_ERR_UNSUPPORTED;
  const int d = H * dh;
  if (((uintptr_t)qkv & 15u) || ((uintptr_t)dO & 15u) || ((uintptr_t)lse & 15u) ||
      ((uintptr_t)delta & 15u) || (S * 4) % 16 != 0)
    return TSP_ERR_INVALID_ARG;
  {
    Prof prof("attn_bwd_prep", st);
    attn_delta_kernel<<<num_sms() * 8, 256, 0, st>>>((const ct_t*)o, (const ct_t*)dO, delta, S, H,
                                                     d);
    TSP_CUDA_TRY(cudaGetLastError());
    TSP_CUDA_TRY(cudaMemsetAsync(dq_acc, 0, (size_t)S * d * sizeof(float), st));
  }
  TcBwdArgs* a = new TcBwdArgs();
  std::unique_ptr<TcBwdArgs> guard(a);
  memset(a, 0, sizeof(TcBwdArgs));
  if (!map_2d(&a->tm_qkv, qkv, 3 * (int64_t)d, S) || !map_2d(&a->tm_do, dO, d, S))
    return TSP_ERR_CUDA;
  a->lse = lse;
  a->delta = delta;
  a->dq_acc = dq_acc;
  a->dqkv = (ct_t*)dqkv;
  a->S = S;
  a->c = c;
  a->D = D;
  a->d = d;
  a->n_kt = (int)(c / BC);
  a->scale = 1.0f / sqrtf((float)dh);
  a->scale_log2 = 1.4426950408889634f * a->scale;
  a->status = status_word();
  a->limit_ns = wait_limit_ns();
  static bool attr = false;
  if (!attr) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    attr = true;
  }
  dim3 grid((unsigned)(D * a->n_kt), (unsigned)H);
  {
    Prof prof("attn_bwd", st);
    attn_bwd_tc_kernel<<<grid, NTHR, SMEM, st>>>(*a);
    TSP_CUDA_TRY(cudaGetLastError());
  }
  Prof prof("attn_bwd_dq_convert", st);
  dq_convert_kernel<<<num_sms() * 8, 256, 0, st>>>(dq_acc, (ct_t*)dqkv, S, d);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
