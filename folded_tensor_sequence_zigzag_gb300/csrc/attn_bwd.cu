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
// 128-row query tiles at positions >= the tile; the two query ranges add up to
// S + 128 rows for every (r, t), so CTAs are balanced.  Every MMA is
// M = 128, N = 128 (an N = 64 MMA costs three quarters of an N = 128 one).
//
// Tensor memory (512 columns) is time-shared per query tile c:
//   cols   0..127  S^T(c) = K Q_c^T, then dQ^T(c) = K^T dS^T(c);
//   cols 128..255  dP^T(c) = V dO_c^T; the P/dS warps overwrite it with
//                  P^T(c) as fp16 pairs (each thread only over columns it has
//                  read), the A operand of dV;
//   cols 256..511  dV, dK accumulated over all query tiles of the key tile.
// One issue burst per query tile, in tensor-core order
//   dK(c) | dQ^T(c) | dV(c) | dP^T(c+1) | S^T(c+1)
// (dP^T(c+1) follows dV(c), which read P^T(c) from the same columns; S^T(c+1)
// waits until the dQ drain has read dQ^T(c), which the three MMA groups in
// between leave time for).  All MMAs of a tile are issued while the FFMA-heavy
// P/dS warps wait: a tcgen05.mma issue needs scheduler slots that those warps
// would otherwise take.
//   warps 0-7  P/dS: thread = key = TMEM lane, warps w and w+4 share 32 keys
//              and take 64 query columns each: P = 2^(s*scale*log2e - L2)
//              with L2 = LSE*log2e precomputed per query, two probabilities a
//              MUFU operation (fp16 pairs), scaled by 2^8 (which keeps small
//              probabilities in fp16's normal range), dS = P (dP - Delta)
//              at the same scale; P^T into TMEM, dS^T into swizzled shared memory (the
//              K-major A operand of dK and the MN-major B operand of dQ^T);
//              at the end of a key tile dK (warps 0-3), dV (4-7) -> fp16 rows;
//   warps 8-11 dQ drain (thread = dh = TMEM lane): dQ^T(c) into the fp32 dQ
//              accumulator with warp-coalesced reductions, paced;
//   warp 12    TMA producer: K, V once per key tile; Q_c, dO_c (+ LSE_c,
//              Delta_c by bulk copy) through a 2-stage ring;
//   warp 13    TMEM allocator + MMA issuer.
// All mbarrier waits are bounded (TSP_ERR_TIMEOUT); TMEM accesses and loop
// exits are warp-uniform.
#include <cstring>
#include <memory>

#include "common.cuh"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BC = 128, BR = 128, DH = 128;
constexpr int NTHR = 512;                  // P/dS x8, dQ drain x4, producer, MMA, 2 idle
// Register split (setmaxnreg): the dQ drain holds a whole dQ^T row of 128 fp32
// values, so its warpgroup takes REG_DRAIN registers a thread from the
// producer/MMA warpgroup; the P/dS warpgroups keep the launch count.  The host
// checks the sum against the launch allocation before every launch.
constexpr int REG_CTRL = 96, REG_DRAIN = 160;
constexpr int WARP_DRAIN = 8, WARP_PROD = 12, WARP_MMA = 13;
constexpr int TILE_BYTES = 128 * 128 * 2;  // 32 KB: 128 rows x 128 fp16
constexpr int BOX_BYTES = TILE_BYTES / 2;  // 128 rows x 64 columns (one TMA box)
constexpr int QSTAGES = 2;                 // Q/dO ring depth
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + TILE_BYTES;
constexpr int OFF_Q = OFF_V + TILE_BYTES;               // QSTAGES stages
constexpr int OFF_DO = OFF_Q + QSTAGES * TILE_BYTES;    // QSTAGES stages
constexpr int OFF_DS = OFF_DO + QSTAGES * TILE_BYTES;   // dS^T, one buffer
constexpr int OFF_L = OFF_DS + TILE_BYTES;              // [stage][LSE 128 | Delta 128] floats
constexpr int OFF_BAR = OFF_L + QSTAGES * 2 * BR * 4;
constexpr int SMEM = OFF_BAR + 256;        // the dynamic base must be 1024-byte aligned
static_assert(SMEM <= 232448, "shared memory above the per-block limit");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_SQ = 0, TM_DPP = 128, TM_DV = 256, TM_DK = 384;
constexpr float kOperandUnscale = 1.f / 256.f;   // P, dS carry 2^8 (fp16's normal range)
// mbarrier indices
constexpr int B_KV = 0, B_QFULL = 1, B_QEMPTY = B_QFULL + QSTAGES, B_DP = B_QEMPTY + QSTAGES,
              B_P = B_DP + 1 /* two: query halves A and B */, B_DQF = B_P + 2, B_DQE = B_DQF + 1,
              B_KVDONE = B_DQE + 1, B_DRAIN = B_KVDONE + 1, N_BARS = B_DRAIN + 1;
static_assert(N_BARS * 8 <= 160, "barriers overlap the TMEM slot");

// Fp16 operands through 128-byte-swizzled maps (box {64, 128}).  The query
// side (Q, dO, LSE, Delta, dQ) is indexed by query row = zigzag row - q_row_off;
// the batched call passes the whole sequence (q_row_off 0), the one-rank call
// its own 2c rows (q_row_off = r * 2c).
struct TcBwdArgs {
  CUtensorMap tm_q;     // Q: query head h at columns q_col0 + h*dh
  CUtensorMap tm_kv;    // K at columns kv_col0 + g*dh, V at kv_col0 + dkv + g*dh; all S rows
  CUtensorMap tm_do;    // dO: query head h at columns h*dh
  const float* lse2;    // [H][lse_ld]: -LSE * log2(e)
  const float* delta;   // [H][lse_ld]: -Delta
  float* dq_acc;        // [query head][query rows][dh] fp32 (head-major), zeroed
  ct_t* out;            // dK at (zigzag row, out_col0 + g*dh), dV out_dkv columns further
  int64_t S, c, out_ld, q_row_off, q_rows, lse_ld;
  int q_col0, kv_col0, out_col0, out_dkv;
  int D, n_kt;          // n_kt = c / 128
  int G, dkv;           // query heads per K/V head; K/V width Hkv*dh
  int rank;             // one-rank call: the rank whose query rows are back-propagated
  float scale, scale_log2;
  int* status;
  uint64_t limit_ns;
};

// The query tiles a key tile at position k0 meets, per query head: every tile
// from k0 on (batched), or the one rank's tiles from k0 on -- the rest of its
// chunk r, then the rest of its chunk 2D-1-r (RANK).
struct QTiles {
  int nqh;              // per query head
  int nA;               // RANK: tiles from chunk r
  int64_t a0, b0;       // RANK: first positions in chunks r and 2D-1-r
};
template <bool RANK>
__device__ __forceinline__ QTiles qtiles(const TcBwdArgs& a, int64_t k0) {
  QTiles q;
  if (!RANK) {
    q.nqh = (int)((a.S - k0) / BR);
    q.nA = 0; q.a0 = q.b0 = 0;
    return q;
  }
  const int64_t ca = (int64_t)a.rank * a.c, cb = (int64_t)(2 * a.D - 1 - a.rank) * a.c;
  q.a0 = k0 > ca ? k0 : ca;
  q.b0 = k0 > cb ? k0 : cb;
  q.nA = q.a0 < ca + a.c ? (int)((ca + a.c - q.a0) / BR) : 0;
  const int nB = q.b0 < cb + a.c ? (int)((cb + a.c - q.b0) / BR) : 0;
  q.nqh = q.nA + nB;
  return q;
}
// position of query tile jj (0 .. nqh-1) of one head
template <bool RANK>
__device__ __forceinline__ int64_t qpos(const QTiles& q, int64_t k0, int jj) {
  if (!RANK) return k0 + (int64_t)jj * BR;
  return jj < q.nA ? q.a0 + (int64_t)jj * BR : q.b0 + (int64_t)(jj - q.nA) * BR;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// barrier `id` over `nthreads` threads (whole warps), independent of barrier 0
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// 2^8 P and 2^8 dS of 32 consecutive queries of one key, as fp16 pairs.
// P = 2^(s*scale*log2e - LSE*log2e): the exponents (<= 0) are rounded to fp16
// pairs and one MUFU operation gives both probabilities (fp16 resolves the
// exponents of the large probabilities to 2^-11 or better); 2^8 P is exact
// from there and keeps small probabilities in fp16's normal range;
// dS = 2^8 P * (dP - Delta) with dP - Delta in fp32 first.  MASK: queries
// before the key (x < kx) get P = 0 through an exponent of -inf.
template <bool MASK>
__device__ __forceinline__ void p_ds_32(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                        const float* L, const float* Dl, float scale_log2, int kx,
                                        uint32_t (&pk)[16], uint32_t (&dk)[16]) {
  const uint32_t k256 = 0x5C005C00u;   // (256, 256) in fp16
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {
    const float4 l0 = *reinterpret_cast<const float4*>(L + c8 * 8);
    const float4 l1 = *reinterpret_cast<const float4*>(L + c8 * 8 + 4);
    const float4 d0 = *reinterpret_cast<const float4*>(Dl + c8 * 8);
    const float4 d1 = *reinterpret_cast<const float4*>(Dl + c8 * 8 + 4);
    const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
    const float dlv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int x = c8 * 8 + e;
      // L and Delta arrive negated, so both pairs are one .f32x2 operation each
      float2 xx = ffma2(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])),
                        make_float2(scale_log2, scale_log2), make_float2(lv[e], lv[e + 1]));
      if (MASK) {
        if (kx > x) xx.x = -INFINITY;
        if (kx > x + 1) xx.y = -INFINITY;
      }
      const uint32_t p2 = hmul2_u32(ex2_approx_f16x2(pack_f16(xx.x, xx.y)), k256);
      const float2 gg = fadd2(make_float2(__uint_as_float(dv[x]), __uint_as_float(dv[x + 1])),
                              make_float2(dlv[e], dlv[e + 1]));
      const uint32_t g2 = pack_f16(gg.x, gg.y);
      pk[x >> 1] = p2;
      dk[x >> 1] = hmul2_u32(p2, g2);
    }
  }
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// GROUPED = false: one query head per K/V head (G = 1), the loops' group
// arithmetic folded away at compile time.  RANK: one rank's query rows
// against every key tile (one key tile per CTA, blockIdx.x = its index; a
// key tile no query of the rank reaches is skipped, its output rows having
// been zeroed by the caller).
template <bool GROUPED, bool RANK>
__global__ void __launch_bounds__(NTHR, 1) attn_bwd_tc_kernel(const __grid_constant__ TcBwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* gbase = smem_raw;
  const uint32_t bars = base + OFF_BAR;
  const uint32_t kv_full = bars + 8u * B_KV;
  auto qd_full = [&](uint32_t s) { return bars + 8u * (B_QFULL + s); };
  auto qd_empty = [&](uint32_t s) { return bars + 8u * (B_QEMPTY + s); };
  const uint32_t dp_full = bars + 8u * B_DP;     // S^T(c), dP^T(c) and all earlier MMAs done
  // P^T(c) in TMEM and dS^T(c) in shared memory for query half X (queries 64X .. 64X+63)
  auto p_full = [&](int X) { return bars + 8u * (B_P + X); };
  const uint32_t dq_full = bars + 8u * B_DQF;
  const uint32_t dq_empty = bars + 8u * B_DQE;
  const uint32_t kv_done = bars + 8u * B_KVDONE;
  const uint32_t drain_bar = bars + 8u * B_DRAIN;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_BAR + 168);

  // an earlier device error skips the work; thread 0 alone reads the word and
  // the barrier hands every thread the same answer, so the CTA leaves whole
  // or not at all (the word can change while the CTA starts)
  if (__syncthreads_or(threadIdx.x == 0 && *(volatile int*)a.status != 0)) return;
  // the 128-byte-swizzled tiles need a 1024-byte aligned base; the layout has
  // no slack to realign it
  if (base & 1023u) {
    if (threadIdx.x == 0) report_status(a.status, (int)TSP_ERR_UNSUPPORTED);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // one CTA per (K/V head g, key-tile pair); its query iterations run over the
  // G query heads of the group, head-major, so dK and dV add up in TMEM
  const int g = blockIdx.y;
  const int G = GROUPED ? a.G : 1;
  const int pair = blockIdx.x;
  const int r = pair / a.n_kt, t = pair - r * a.n_kt;
  constexpr int NTILE = RANK ? 1 : 2;   // key tiles per CTA
  int64_t k0s[2];
  if (RANK) {
    k0s[0] = (int64_t)blockIdx.x * BC;
    k0s[1] = 0;
  } else {
    k0s[0] = (int64_t)r * a.c + (int64_t)t * BC;                                    // long range
    k0s[1] = (int64_t)(2 * a.D - 1 - r) * a.c + (int64_t)(a.n_kt - 1 - t) * BC;    // mirror
  }

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < QSTAGES; ++s) {
      mbar_init(qd_full(s), 1);
      mbar_init(qd_empty(s), 1);
    }
    mbar_init(dp_full, 1);
    mbar_init(p_full(0), 256);
    mbar_init(p_full(1), 256);
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
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_kv);
    tma_prefetch_desc(&a.tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  float* sLD = reinterpret_cast<float*>(gbase + OFF_L);  // [stage][LSE 128 | Delta 128]
  // Q/dO ring position of query tile `cur` (CTA-wide counter)
  auto qst = [](uint32_t cur) { return cur % QSTAGES; };
  auto qph = [](uint32_t cur) { return (cur / QSTAGES) & 1u; };

  // Each role runs its own loop over the two key tiles, so the register limit
  // that setmaxnreg sets covers all code of that role.
  uint32_t it = 0;        // query tiles processed by this CTA so far (one copy per role)
  auto tile_sync = [&]() {  // K/V tiles, TMEM accumulators and barrier phases move on
    tc_fence_before();
    named_bar_sync(1, NTHR);
    tc_fence_after();
  };
  if (warp >= WARP_PROD) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(REG_CTRL));
    uint32_t q_issued = 0, kv_issued = 0;
    for (int tile = 0; tile < NTILE; ++tile) {
      const int64_t k0 = k0s[tile];
      const QTiles qt = qtiles<RANK>(a, k0);
      const int nqh = qt.nqh;                  // query tiles per head
      const int nq = nqh * G;                  // query iterations of this key tile
      if (RANK && nq == 0) continue;           // every role skips it alike
      const int64_t krow0 = zz_row_of_pos(k0, a.c, a.D);
      if (warp == WARP_PROD) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !*abort_flag) {
          (void)TSP_INB(krow0 >= 0 && krow0 + BC <= a.S, a.status);   // tensor copies: report only
          mbar_arrive_expect_tx(kv_full, 2 * TILE_BYTES);
#pragma unroll
          for (int jh = 0; jh < 2; ++jh) {
            tma_load_2d(base + OFF_K + jh * BOX_BYTES, &a.tm_kv, a.kv_col0 + g * DH + 64 * jh, (int)krow0,
                        kv_full);
            tma_load_2d(base + OFF_V + jh * BOX_BYTES, &a.tm_kv, a.kv_col0 + a.dkv + g * DH + 64 * jh,
                        (int)krow0, kv_full);
          }
          ++kv_issued;
          for (int j = 0; j < nq; ++j) {
            const uint32_t cur = it + j, st = qst(cur);
            if (!mbar_wait(qd_empty(st), qph(cur) ^ 1u, a.status, abort_flag, a.limit_ns)) break;
            const int gi = GROUPED ? j / nqh : 0, jj = j - gi * nqh;
            const int h = g * G + gi;
            int64_t qrow = zz_row_of_pos32((int)qpos<RANK>(qt, k0, jj), (int)a.c, a.D) - a.q_row_off;
            // a failed check reads row 0 instead: the copy still lands, so the
            // pipeline's byte counts hold
            if (!TSP_INB(qrow >= 0 && qrow + BR <= a.q_rows, a.status)) qrow = 0;
            const uint32_t fb = qd_full(st);
            mbar_arrive_expect_tx(fb, 2 * TILE_BYTES + 2 * BR * 4);
#pragma unroll
            for (int jh = 0; jh < 2; ++jh) {
              tma_load_2d(base + OFF_Q + st * TILE_BYTES + jh * BOX_BYTES, &a.tm_q,
                          a.q_col0 + h * DH + 64 * jh, (int)qrow, fb);
              tma_load_2d(base + OFF_DO + st * TILE_BYTES + jh * BOX_BYTES, &a.tm_do,
                          h * DH + 64 * jh, (int)qrow, fb);
            }
            const uint32_t sl = smem_u32(sLD + st * 2 * BR);
            bulk_load(sl, a.lse2 + (int64_t)h * a.lse_ld + qrow, BR * 4, fb);
            bulk_load(sl + BR * 4, a.delta + (int64_t)h * a.lse_ld + qrow, BR * 4, fb);
            ++q_issued;
          }
        }
      } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort_flag) {
          constexpr uint32_t id_f = idesc_f16_f32(128, 128, false, false, false);  // S^T, dP^T
          constexpr uint32_t id_kv = idesc_f16_f32(128, 128, false, true, false);  // dV, dK
          constexpr uint32_t id_q64 = idesc_f16_f32(128, 64, true, true, false);   // dQ^T half
          // base descriptors, computed once: the issue loops only add constants
          const uint64_t dK_k = sdesc_sw128(base + OFF_K, 16, 1024);           // K, K-major
          const uint64_t dV_k = sdesc_sw128(base + OFF_V, 16, 1024);           // V, K-major
          const uint64_t dK_mn = sdesc_sw128(base + OFF_K, BOX_BYTES, 1024);   // K^T, MN-major
          const uint64_t dQ_k = sdesc_sw128(base + OFF_Q, 16, 1024);           // Q stages
          const uint64_t dDO_k = sdesc_sw128(base + OFF_DO, 16, 1024);         // dO stages
          const uint64_t dQ_mn = sdesc_sw128(base + OFF_Q, BOX_BYTES, 1024);
          const uint64_t dDO_mn = sdesc_sw128(base + OFF_DO, BOX_BYTES, 1024);
          const uint64_t dDS_k = sdesc_sw128(base + OFF_DS, 16, 1024);         // dS^T, K-major
          const uint64_t dDS_mn = sdesc_sw128(base + OFF_DS, BOX_BYTES, 1024); // dS^T, MN-major
          bool ok = mbar_wait(kv_full, (uint32_t)tile & 1u, a.status, abort_flag, a.limit_ns);
          // S^T(cur) = K Q^T or dP^T(cur) = V dO^T: M = 128 keys, N = 128 queries, K = dh
          auto issue_sdp = [&](uint32_t d_tmem, uint64_t a0, uint64_t b0) {
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
              umma_f16_ss_hot(tmem + d_tmem, sdesc_add(a0, off), sdesc_add(b0, off), id_f,
                              kk > 0 ? 1u : 0u);
            }
          };
          if (ok) ok = mbar_wait(qd_full(qst(it)), qph(it), a.status, abort_flag, a.limit_ns);
          if (ok) {
            tc_fence_after();
            const uint32_t so = qst(it) * TILE_BYTES;
            issue_sdp(TM_SQ, dK_k, sdesc_add(dQ_k, so));
            issue_sdp(TM_DPP, dV_k, sdesc_add(dDO_k, so));
            umma_commit(dp_full);
          }
          for (int j = 0; j < nq && ok; ++j) {
            const uint32_t cur = it + j, so = qst(cur) * TILE_BYTES;
            const uint64_t bdo = sdesc_add(dDO_mn, so), bq = sdesc_add(dQ_mn, so);
            const uint32_t acc0 = j > 0 ? 1u : 0u;
            // The query tile in two halves X = A, B (queries 64X .. 64X+63): the
            // MMAs of half A run while the P/dS warps work on half B.
#pragma unroll
            for (int X = 0; X < 2; ++X) {
              if (!(ok = mbar_wait(p_full(X), cur & 1u, a.status, abort_flag, a.limit_ns))) break;
              tc_fence_after();
              // dK += dS^T Q over the half's queries: M = 128 keys, N = 128 dh, K = 64
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const int kk = 4 * X + k4;
                umma_f16_ss_hot(tmem + TM_DK, sdesc_add(dDS_k, X * BOX_BYTES + k4 * 32),
                                sdesc_add(bq, kk * 2048), id_kv, kk > 0 ? 1u : acc0);
              }
              // dQ^T of the half = K^T dS^T: M = 128 dh, N = 64 queries, K = 128 keys,
              // into S^T's columns of the same queries (the half has read them)
#pragma unroll
              for (int kk = 0; kk < BC / 16; ++kk)
                umma_f16_ss_hot(tmem + TM_SQ + 64 * X, sdesc_add(dK_mn, kk * 2048),
                                sdesc_add(dDS_mn, X * BOX_BYTES + kk * 2048), id_q64,
                                kk > 0 ? 1u : 0u);
              if (X == 1) umma_commit(dq_full);
              // dV += P^T dO over the half (A = P^T from TMEM: queries 16kk .. 16kk+15
              // at column 32 (kk / 2) + 8 (kk % 2))
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const int kk = 4 * X + k4;
                umma_f16_ts_hot(tmem + TM_DV, tmem + TM_DPP + 32 * (kk >> 1) + 8 * (kk & 1),
                                sdesc_add(bdo, kk * 2048), id_kv, kk > 0 ? 1u : acc0);
              }
            }
            if (!ok) break;
            umma_commit(qd_empty(qst(cur)));
            if (j + 1 < nq) {
              const uint32_t nx = cur + 1, so1 = qst(nx) * TILE_BYTES;
              if (!(ok = mbar_wait(qd_full(qst(nx)), qph(nx), a.status, abort_flag, a.limit_ns)))
                break;
              tc_fence_after();
              issue_sdp(TM_DPP, dV_k, sdesc_add(dDO_k, so1));
              // S^T(cur+1) reuses the dQ^T columns once the drain has read them
              if (!(ok = mbar_wait(dq_empty, cur & 1u, a.status, abort_flag, a.limit_ns))) break;
              tc_fence_after();
              issue_sdp(TM_SQ, dK_k, sdesc_add(dQ_k, so1));
              umma_commit(dp_full);
            }
          }
          if (ok) {
            umma_commit(kv_done);
          } else {
            umma_commit(drain_bar);
            drain_wait(drain_bar, 0, a.limit_ns);
          }
        }
      }
      it += (uint32_t)nq;
      tile_sync();
    }
    if (warp == WARP_PROD && lane == 0 && *abort_flag) {
      const uint32_t n_out = q_issued < (uint32_t)QSTAGES ? q_issued : (uint32_t)QSTAGES;
      for (uint32_t jj = q_issued - n_out; jj < q_issued; ++jj)
        drain_wait(qd_full(qst(jj)), qph(jj), a.limit_ns);
      if (kv_issued > 0) drain_wait(kv_full, (kv_issued - 1) & 1u, a.limit_ns);
    }
  } else if (warp >= WARP_DRAIN) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(REG_DRAIN));
    for (int tile = 0; tile < NTILE; ++tile) {
      const int64_t k0 = k0s[tile];
      const QTiles qt = qtiles<RANK>(a, k0);
      const int nqh = qt.nqh;
      const int nq = nqh * G;
      if (RANK && nq == 0) continue;
      {
        // ------------------------------------------------------------ dQ drain (thread = dh)
        // all 128 query columns are read before the TMEM columns are released, so
        // S^T(cur+1) never waits for the atomics (which take ~2700 clocks a tile:
        // 64 KB at the ~24 bytes a clock an SM gets for global reductions)
        const int quarter = warp & 3;
        const int dh = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        bool ok = true;
        for (int j = 0; j < nq; ++j) {
          const uint32_t cur = it + j;
          const bool okl = ok && mbar_wait(dq_full, cur & 1u, a.status, abort_flag, a.limit_ns);
          if (!(ok = __all_sync(0xffffffffu, okl))) break;
          tc_fence_after();
          uint32_t v[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(lane_base + TM_SQ + q * 32, v[q]);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(dq_empty);   // dQ^T(cur) read: its columns may take S^T(cur+1)
          const int gi = GROUPED ? j / nqh : 0, jj = j - gi * nqh;
          const int64_t qrow =
              zz_row_of_pos32((int)qpos<RANK>(qt, k0, jj), (int)a.c, a.D) - a.q_row_off;
          const bool q_in = TSP_INB(qrow >= 0 && qrow + BR <= a.q_rows, a.status);
          // head-major accumulator: the tile's 128 query rows of this head are
          // DH floats apart, so every reduction's address is dst plus a
          // constant (no per-reduction address arithmetic in the drain, whose
          // warps share the MMA issuer's schedulers)
          float* dst = a.dq_acc + ((int64_t)(g * G + gi) * a.q_rows + qrow) * DH + dh;
          // dQ^T leaves unscaled (scale * 2^-8 is applied once per element by
          // dq_convert_kernel): a multiply per reduction would take issue slots
          // from the schedulers the MMA-issuing thread shares.
          // The reductions leave in 8 groups of 16 with a short sleep between
          // them: at ~24 bytes a clock an SM's reductions drain slower than the
          // warps issue them, and a full queue holds up the P/dS warps' shared
          // memory loads and stores behind it (the tile took ~8% longer with
          // the reductions issued in one burst).  The sleeps must stay well
          // inside a tile's time (~2.5 us): at 8 x 400 ns the drain became the
          // bottleneck (+55%); 150 and 250 ns time alike.
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (q_in) atomicAdd(dst + (q * 32 + h2 * 16 + e) * DH,
                                    __uint_as_float(v[q][h2 * 16 + e]));
              __nanosleep(150);
            }
          }
        }
        tc_fence_before();
      }
      it += (uint32_t)nq;
      tile_sync();
    }
  } else {
    for (int tile = 0; tile < NTILE; ++tile) {
      const int64_t k0 = k0s[tile];
      const QTiles qt = qtiles<RANK>(a, k0);
      const int nqh = qt.nqh;
      const int nq = nqh * G;
      if (RANK && nq == 0) continue;
      const int64_t krow0 = zz_row_of_pos(k0, a.c, a.D);
      {
        // ------------------------------------------------------------ P, dS (thread = key)
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        uint8_t* drow = gbase + OFF_DS + (row >> 3) * 1024 + (row & 7) * 128;
        bool ok = true;
        for (int j = 0; j < nq; ++j) {
          const uint32_t cur = it + j, st = qst(cur);
          bool okl = ok && mbar_wait(dp_full, cur & 1u, a.status, abort_flag, a.limit_ns);
          okl = okl && mbar_wait(qd_full(st), qph(cur), a.status, abort_flag, a.limit_ns);
          if (!(ok = __all_sync(0xffffffffu, okl))) break;
          tc_fence_after();
          const float* L = sLD + st * 2 * BR;
          const float* Dl = L + BR;
          // query tile == key tile (the first of each head): key index > query index is masked
          const bool diag = RANK ? qpos<RANK>(qt, k0, j) == k0 : (GROUPED ? j % nqh == 0 : j == 0);
          // query half X (queries 64X .. 64X+63) by all eight warps, A then B:
          // warps w and w+4 share a key and take 32 queries of the half each
#pragma unroll
          for (int X = 0; X < 2; ++X) {
            const int qb = X * 64 + half * 32;     // this thread's 32 query columns
            uint32_t sv[32], dv[32];
            tmem_ld32(lane_base + TM_SQ + qb, sv);
            tmem_ld32(lane_base + TM_DPP + qb, dv);
            tmem_wait_ld();
            uint32_t pk[16], dk[16];
            if (diag)
              p_ds_32<true>(sv, dv, L + qb, Dl + qb, a.scale_log2, row - qb, pk, dk);
            else
              p_ds_32<false>(sv, dv, L + qb, Dl + qb, a.scale_log2, row - qb, pk, dk);
            // P^T over dP^T columns this thread has read: queries qb .. qb+31 ->
            // columns qb .. qb+15 (query chunk kk at 32 (kk / 2) + 8 (kk % 2))
            tmem_st16(lane_base + TM_DPP + qb, pk);
            // dS^T row `row`, queries qb.. -> box X, 16-byte chunks 4*half .. 4*half+3
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int chunk = half * 4 + c;
              *reinterpret_cast<uint4*>(drow + X * BOX_BYTES + ((chunk ^ (row & 7)) << 4)) =
                  make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full(X));
          }
        }
        // dK, dV of this key tile -> fp16 rows
        bool eok = ok && mbar_wait(kv_done, (uint32_t)tile & 1u, a.status, abort_flag, a.limit_ns);
        if (__all_sync(0xffffffffu, eok)) {
          tc_fence_after();
          const bool k_in = TSP_INB(krow0 >= 0 && krow0 + row < a.S, a.status);
          ct_t* dkrow = a.out + (krow0 + row) * a.out_ld + a.out_col0 + g * DH;
          const float mul = half == 0 ? a.scale * kOperandUnscale : kOperandUnscale;
          ct_t* out = dkrow + half * a.out_dkv;   // warps 0-3 write dK, warps 4-7 write dV
          // (a dS beyond fp16 range makes dK and dQ non-finite, so the checks
          // of the dK, dV rows here and of dQ in dq_convert_kernel cover it)
          bool bad = false;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            tmem_ld32(lane_base + (half == 0 ? TM_DK : TM_DV) + q * 32, v);
            tmem_wait_ld();
            float f[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * mul;
            bad |= f16_bad_n<32>(f);
            uint4* dst = reinterpret_cast<uint4*>(out + q * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (k_in) dst[c] = make_uint4(pack_f16(f[8 * c], f[8 * c + 1]), pack_f16(f[8 * c + 2], f[8 * c + 3]),
                                  pack_f16(f[8 * c + 4], f[8 * c + 5]),
                                  pack_f16(f[8 * c + 6], f[8 * c + 7]));
          }
          if (bad) report_status(a.status, (int)TSP_ERR_RANGE);
        }
        tc_fence_before();
      }
      it += (uint32_t)nq;
      tile_sync();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Delta[h][row] = dO[row, head h] . O[row, head h] and
// L2[h][row] = LSE[h][row] * log2(e) (the exponent offset of P)
// (warp per row and head)
__global__ void attn_delta_kernel(const ct_t* __restrict__ o, const ct_t* __restrict__ dO,
                                  const float* __restrict__ lse, float* __restrict__ delta,
                                  float* __restrict__ lse2, int64_t S, int H, int d) {
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
    if (lane == 0) {
      // both negated: the P/dS warps add them (x = s * scale log2e - L2,
      // dP - Delta) with two-lane fp32 operations that take no negation
      delta[(int64_t)h * S + row] = -s;
      lse2[(int64_t)h * S + row] = -lse[(int64_t)h * S + row] * 1.4426950408889634f;
    }
  }
}

// dQKV[:, 0:d] = fp16(dq_acc); dQKV rows are ld elements apart
// dQ = mul * acc (mul = softmax scale * 2^-8: the accumulator holds the dQ^T
// MMA outputs unscaled), acc head-major [d / DH][S][DH] -> fp16 rows of
// stride ld, head h at columns h*DH
__global__ void dq_convert_kernel(const float* __restrict__ acc, ct_t* __restrict__ dqkv,
                                  int64_t S, int d, int64_t ld, float mul,
                                  int* __restrict__ status) {
  const int64_t total4 = S * d / 4;
  bool bad = false;   // an fp16 output out of range
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total4;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = t * 4;
    const int64_t row = e / d;
    const int col = (int)(e - row * d);
    const int hh = col / DH, j = col - hh * DH;
    float4 v = *reinterpret_cast<const float4*>(acc + ((int64_t)hh * S + row) * DH + j);
    v.x *= mul;
    v.y *= mul;
    v.z *= mul;
    v.w *= mul;
    bad |= f16_bad(v.x) | f16_bad(v.y) | f16_bad(v.z) | f16_bad(v.w);
    uint2 o;
    o.x = pack_f16(v.x, v.y);
    o.y = pack_f16(v.z, v.w);
    *reinterpret_cast<uint2*>(dqkv + row * ld + col) = o;
  }
  if (bad) report_status(status, (int)TSP_ERR_RANGE);
}

// Row-major fp16 [rows, cols] with box {64 columns, 128 rows}, 128-byte swizzle.
bool map_2d(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows) {
  return tma_map_f16(m, ptr, cols, rows, cols, 128);
}

}  // namespace

namespace {

// The backward kernel with its shared-memory attribute (once per device) and
// the register-split check; grid (key-tile units, K/V heads).
template <bool GROUPED, bool RANK>
tsp_status launch_bwd_kernel(const TcBwdArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = attn_bwd_tc_kernel<GROUPED, RANK>;
  static bool attr[kMaxDevices] = {};   // the attribute holds for one device
  static int launch_regs = 0;
  const int dev = current_device();
  if (!attr[dev]) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    cudaFuncAttributes fa;
    TSP_CUDA_TRY(cudaFuncGetAttributes(&fa, kern));
    launch_regs = fa.numRegs;
    attr[dev] = true;
  }
  // setmaxnreg.inc would wait forever if the split exceeded the launch allocation
  const int64_t lr = launch_regs;
  if (lr * NTHR < lr * 256 + 128 * (REG_DRAIN + REG_CTRL)) return TSP_ERR_UNSUPPORTED;
  Prof prof(RANK ? "rank_attn_bwd" : "attn_bwd", st);
  kern<<<grid, NTHR, SMEM, st>>>(a);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace

tsp_status launch_attn_bwd_f16(const void* qkv, const void* o, const void* dO, const float* lse,
                               float* delta, float* dq_acc, void* dqkv, int64_t S, int H, int Hkv,
                               int dh, int D, cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BC != 0 || S > (int64_t)INT32_MAX) return TSP_ERR_UNSUPPORTED;
  if (S % 4 != 0) return TSP_ERR_UNSUPPORTED;
  if (Hkv < 1 || H % Hkv != 0) return TSP_ERR_INVALID_ARG;
  const int d = H * dh, dkv = Hkv * dh;
  const int64_t ld = d + 2 * (int64_t)dkv;
  if (((uintptr_t)qkv & 15u) || ((uintptr_t)dO & 15u) || ((uintptr_t)lse & 15u) ||
      ((uintptr_t)delta & 15u) || (S * 4) % 16 != 0)
    return TSP_ERR_INVALID_ARG;
  {
    Prof prof("attn_bwd_prep", st);
    attn_delta_kernel<<<num_sms() * 8, 256, 0, st>>>((const ct_t*)o, (const ct_t*)dO, lse, delta,
                                                     delta + (int64_t)H * S, S, H, d);
    TSP_CUDA_TRY(cudaGetLastError());
    TSP_CUDA_TRY(cudaMemsetAsync(dq_acc, 0, (size_t)S * d * sizeof(float), st));
  }
  TcBwdArgs* a = new TcBwdArgs();
  std::unique_ptr<TcBwdArgs> guard(a);
  memset(a, 0, sizeof(TcBwdArgs));
  if (!map_2d(&a->tm_q, qkv, ld, S) || !map_2d(&a->tm_do, dO, d, S)) return TSP_ERR_CUDA;
  a->tm_kv = a->tm_q;
  a->q_col0 = 0;
  a->kv_col0 = d;
  a->lse2 = delta + (int64_t)H * S;
  a->delta = delta;
  a->dq_acc = dq_acc;
  a->out = (ct_t*)dqkv;
  a->out_ld = ld;
  a->out_col0 = d;
  a->out_dkv = dkv;
  a->S = S;
  a->c = c;
  a->D = D;
  a->q_row_off = 0;
  a->q_rows = S;
  a->lse_ld = S;
  a->G = H / Hkv;
  a->dkv = dkv;
  a->n_kt = (int)(c / BC);
  a->rank = -1;
  a->scale = 1.0f / sqrtf((float)dh);
  a->scale_log2 = 1.4426950408889634f * a->scale;
  a->status = status_word();
  a->limit_ns = wait_limit_ns();
  const dim3 grid((unsigned)(D * a->n_kt), (unsigned)Hkv);
  const tsp_status r = Hkv != H ? launch_bwd_kernel<true, false>(*a, grid, st)
                                : launch_bwd_kernel<false, false>(*a, grid, st);
  if (r != TSP_OK) return r;
  Prof prof("attn_bwd_dq_convert", st);
  dq_convert_kernel<<<num_sms() * 8, 256, 0, st>>>(dq_acc, (ct_t*)dqkv, S, d, ld,
                                                    a->scale * kOperandUnscale, a->status);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

tsp_status launch_attn_bwd_rank_f16(const void* q, const void* kv, const void* o, const void* dO,
                                    const float* lse, float* delta, float* dq_acc, void* dq,
                                    void* dkv, int64_t S, int Hk, int dh, int D, int r,
                                    cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D), rows = 2 * c;
  if (c % BC != 0 || S > (int64_t)INT32_MAX || r < 0 || r >= D) return TSP_ERR_UNSUPPORTED;
  const int Ck = Hk * dh;
  const void* ptrs[9] = {q, kv, o, dO, lse, delta, dq_acc, dq, dkv};
  for (const void* p : ptrs)
    if (!p || ((uintptr_t)p & 15u)) return TSP_ERR_INVALID_ARG;
  {
    Prof prof("rank_attn_bwd_prep", st);
    attn_delta_kernel<<<num_sms() * 8, 256, 0, st>>>((const ct_t*)o, (const ct_t*)dO, lse, delta,
                                                     delta + (int64_t)Hk * rows, rows, Hk, Ck);
    TSP_CUDA_TRY(cudaGetLastError());
    TSP_CUDA_TRY(cudaMemsetAsync(dq_acc, 0, (size_t)rows * Ck * sizeof(float), st));
    // key tiles none of the rank's queries reach keep these zeros
    TSP_CUDA_TRY(cudaMemsetAsync(dkv, 0, (size_t)S * 2 * Ck * sizeof(ct_t), st));
  }
  TcBwdArgs* a = new TcBwdArgs();
  std::unique_ptr<TcBwdArgs> guard(a);
  memset(a, 0, sizeof(TcBwdArgs));
  if (!map_2d(&a->tm_q, q, Ck, rows) || !map_2d(&a->tm_kv, kv, 2 * (int64_t)Ck, S) ||
      !map_2d(&a->tm_do, dO, Ck, rows))
    return TSP_ERR_CUDA;
  a->q_col0 = 0;
  a->kv_col0 = 0;
  a->lse2 = delta + (int64_t)Hk * rows;
  a->delta = delta;
  a->dq_acc = dq_acc;
  a->out = (ct_t*)dkv;
  a->out_ld = 2 * Ck;
  a->out_col0 = 0;
  a->out_dkv = Ck;
  a->S = S;
  a->c = c;
  a->D = D;
  a->q_row_off = (int64_t)r * rows;
  a->q_rows = rows;
  a->lse_ld = rows;
  a->G = 1;
  a->dkv = Ck;
  a->n_kt = (int)(c / BC);
  a->rank = r;
  a->scale = 1.0f / sqrtf((float)dh);
  a->scale_log2 = 1.4426950408889634f * a->scale;
  a->status = status_word();
  a->limit_ns = wait_limit_ns();
  const tsp_status res = launch_bwd_kernel<false, true>(*a, dim3((unsigned)(S / BC), (unsigned)Hk), st);
  if (res != TSP_OK) return res;
  Prof prof("rank_attn_bwd_dq_convert", st);
  dq_convert_kernel<<<num_sms() * 8, 256, 0, st>>>(dq_acc, (ct_t*)dq, rows, Ck, Ck,
                                                    a->scale * kOperandUnscale, a->status);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

}  // namespace tsp
