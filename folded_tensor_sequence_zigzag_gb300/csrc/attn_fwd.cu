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
// Work unit = one CTA = (head h, virtual rank r, 256-row block t): block t of
// chunk r AND the mirrored block nb-1-t of chunk 2D-1-r (nb = c/256).  The
// causal key ranges of the two blocks add up to the same count for every
// (r, t), so every CTA carries the same work.  Key tiles past a query tile's
// last row are never visited; only the diagonal 128-key tile is masked.
//
// A block is two 128-row query tiles, A = rows [p0, p0+128) and
// B = rows [p0+128, p0+256), that share every K/V tile (B needs one more, its
// own diagonal).  Ping-pong: while the softmax warps of one tile turn their
// 128x128 scores into probabilities, the tensor core runs the other tile's
// MMAs, so the MUFU/FMA work of the softmax hides behind tcgen05 work.
//   warps 8-11 (one warpgroup, registers handed to the softmax warpgroups):
//   warp 8   TMA producer: Q_A, Q_B once per block; K_j, V_j through a 4-slot
//            ring of 128x128 fp16 tiles (128-byte swizzle, column boxes of
//            the Q|K|V buffer);
//   warp 9   TMEM allocator + MMA issuer, in the order
//            S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//            with S_X = Q_X K_j^T into a 128-column TMEM buffer per tile and
//            O_X += P_X V_j into a 128-column TMEM accumulator per tile
//            (V read MN-major, dh contiguous, straight from the buffer);
//   warps 0-3 / 4-7  softmax of tile A / B: thread = query row = TMEM lane;
//            p = 2^(s*scale*log2e - m) with one FFMA + MUFU ex2 per score,
//            written as fp16 pairs into TMEM over the scores just read: PV
//            takes P as its A operand from tensor memory.
// Shared memory feeds the tensor core at about 128 bytes a clock per SM,
// which an M=128, N=128 MMA with both operands in shared memory uses up on
// its own; with P in TMEM, PV reads only V there, and no P store competes
// with the operand reads.
// The running max m is only raised (and O rescaled in TMEM) when a warp's row
// max grows by more than 2^8; O/l is exact either way and p stays below 256.
// All mbarrier waits are bounded (TSP_ERR_TIMEOUT); loop exits are
// warp-uniform (TMEM access is warp-collective).
#include <cstring>
#include <memory>

#include "common.cuh"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BQ = 128, BKV = 128, DH = 128, BLOCK = 2 * BQ;
constexpr int NTHR = 384;                  // 8 softmax warps + producer + MMA + 2 idle
// Register split (setmaxnreg): each softmax thread keeps a full 128-score row
// in registers, so the two softmax warpgroups take REG_SOFT registers a
// thread and the producer/MMA warpgroup gives its share back.  The sum must
// stay within the block's launch allocation (NTHR x registers at launch);
// the host checks that before every launch.
constexpr int REG_SOFT = 208, REG_CTRL = 64;
constexpr int REG_TOTAL = 2 * 128 * REG_SOFT + 128 * REG_CTRL;
constexpr int WARP_PROD = 8, WARP_MMA = 9;
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128x128 fp16 tile (two 64-column boxes)
constexpr int BOX_BYTES = TILE_BYTES / 2;  // 128 rows x 64 columns
constexpr int NSLOT = 4;                   // K/V ring: K_0 V_0 K_1 V_1 ... in 4 slots
constexpr int OFF_Q = 0;                         // Q_A, Q_B
constexpr int OFF_KV = OFF_Q + 2 * TILE_BYTES;   // ring slots
constexpr int OFF_BAR = OFF_KV + NSLOT * TILE_BYTES;
// mbarrier indices
constexpr int B_QFULL = 0, B_SFULL = 1, B_SEMPTY = B_SFULL + NSLOT, B_S = B_SEMPTY + NSLOT,
              B_P = B_S + 2, B_O = B_P + 2, B_DRAIN = B_O + 2, N_BARS = B_DRAIN + 1;
static_assert(N_BARS * 8 <= 160, "barriers overlap the TMEM slot");
constexpr int SMEM = OFF_BAR + 256 + 1024;       // + 1 KB alignment slack
constexpr uint32_t TMEM_COLS = 512;              // S_A | S_B | O_A | O_B
constexpr float RESCALE_LOG2 = 8.0f;             // lazy-rescale threshold (log2 units)

struct TcAttnArgs {
  // K/V: rows in zigzag order over all S positions, K of K/V head g at columns
  // kv_col0 + g*dh, V at kv_col0 + dkv + g*dh (fp16, box {64, 128}, 128B swizzle)
  CUtensorMap tm;
  // Q: query head h at columns q_col0 + h*dh of the rows of zigzag row
  // index - q_row_off (the whole Q|K|V buffer, or one rank's own rows)
  CUtensorMap tm_q;
  ct_t* o;              // O row (zigzag row index - o_row_off), row stride ldo
  float* lse;           // [H][lse_ld] at (zigzag row index - o_row_off)
  int64_t S, c, q_row_off, o_row_off, ldo, lse_ld;
  int D, d, n_blocks;   // n_blocks = c / 256
  int rank0;            // virtual rank of blockIdx.x / n_blocks == 0
  int q_col0, kv_col0;
  int G, dkv;           // query heads per K/V head; K/V width Hkv*dh
  float scale_log2;
  int* status;
  uint64_t limit_ns;
  // one-rank split mode (split_lc > 0): a CTA per chunk of split_lc key tiles
  // of one of the rank's 256-row blocks (the last chunk takes the block's last
  // two tiles, its diagonals), writing O / l in fp32 and log2-sum-exp to the
  // partials [H][n_items][256][DH] and [H][n_items][256] that
  // attn_split_merge_kernel merges
  int split_lc, n_items;
  float* part_o;
  float* part_lse;
};

// The work of blockIdx.x = `pair`, item `blk` of the CTA: the block's first
// query position p0 and its key tiles [j0, j1) of the block's nB = p0/128 + 2
// (tile A reads [j0, min(j1, nB - 1)), its diagonal tile nB - 2; tile B reads
// up to its own diagonal nB - 1).  Without a split: block `blk` of the
// mirrored pair `pair` (blk 0 in chunk 2D-1-r, blk 1 in chunk r), every tile.
struct Item {
  int64_t p0;
  int j0, j1;
};
// blocks of one rank in split mode: b < nb are chunk r's blocks in order,
// b >= nb chunk 2D-1-r's, mirrored (b = nb + t has block nb-1-t)
__device__ __forceinline__ int64_t split_block_p0(const TcAttnArgs& a, int b) {
  const int nb = a.n_blocks;
  return b < nb ? (int64_t)a.rank0 * a.c + (int64_t)b * BLOCK
                : (int64_t)(2 * a.D - 1 - a.rank0) * a.c + (int64_t)(2 * nb - 1 - b) * BLOCK;
}
// chunks of a block with nB key tiles: split_lc tiles each, the last one up
// to split_lc + 1 (never fewer than the two diagonal tiles)
__device__ __forceinline__ int split_chunks(int nB, int lc) { return (nB - 2) / lc + 1; }

__device__ __forceinline__ Item item_of(const TcAttnArgs& a, int pair, int blk) {
  Item it;
  if (a.split_lc == 0) {
    const int rl = pair / a.n_blocks, t = pair - rl * a.n_blocks;
    const int r = a.rank0 + rl;
    it.p0 = blk == 0 ? (int64_t)(2 * a.D - 1 - r) * a.c + (int64_t)(a.n_blocks - 1 - t) * BLOCK
                     : (int64_t)r * a.c + (int64_t)t * BLOCK;
    it.j0 = 0;
    it.j1 = (int)(it.p0 / BKV) + 2;
    return it;
  }
  int rem = pair;
  for (int b = 0; b < 2 * a.n_blocks; ++b) {
    const int64_t pb = split_block_p0(a, b);
    const int nB = (int)(pb / BKV) + 2;
    const int nch = split_chunks(nB, a.split_lc);
    if (rem < nch) {
      it.p0 = pb;
      it.j0 = rem * a.split_lc;
      it.j1 = rem == nch - 1 ? nB : it.j0 + a.split_lc;
      return it;
    }
    rem -= nch;
  }
  it.p0 = 0;
  it.j0 = it.j1 = 0;   // past the last item: no work
  return it;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// barrier `id` over `nthreads` threads (whole warps), independent of barrier 0
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

__global__ void __launch_bounds__(NTHR, 1) attn_fwd_tc_kernel(const __grid_constant__ TcAttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + OFF_BAR;
  const uint32_t q_full = bars + 8u * B_QFULL;
  auto slot_full = [&](uint32_t s) { return bars + 8u * (B_SFULL + s); };
  auto slot_empty = [&](uint32_t s) { return bars + 8u * (B_SEMPTY + s); };
  auto s_full = [&](int x) { return bars + 8u * (B_S + x); };
  auto p_full = [&](int x) { return bars + 8u * (B_P + x); };
  auto o_done = [&](int x) { return bars + 8u * (B_O + x); };
  const uint32_t drain_bar = bars + 8u * B_DRAIN;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_BAR + 168);

  // an earlier device error skips the work; thread 0 alone reads the word and
  // the barrier hands every thread the same answer, so the CTA leaves whole
  // or not at all (the word can change while the CTA starts)
  if (__syncthreads_or(threadIdx.x == 0 && *(volatile int*)a.status != 0)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int kcol = a.kv_col0 + (h / a.G) * DH;   // K columns of this head's K/V head; V at + dkv
  const int pair = blockIdx.x;
  const int n_it = a.split_lc ? 1 : 2;   // items (blocks, or chunks of one) of this CTA
  // a split-mode CTA past the last chunk has nothing to do (every thread
  // computes the same answer before any barrier or TMEM is set up)
  if (a.split_lc && item_of(a, pair, 0).j1 == 0) return;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), 128);
      mbar_init(o_done(x), 1);
    }
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
    tma_prefetch_desc(&a.tm);
    tma_prefetch_desc(&a.tm_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Each role runs its own loop over the two blocks, so the register limit
  // that setmaxnreg sets covers all code of that role.
  auto block_sync = [&]() {  // Q, O, P and the TMEM buffers move on to the next block
    tc_fence_before();
    named_bar_sync(1, NTHR);
    tc_fence_after();
  };
  if (warp >= WARP_PROD) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(REG_CTRL));
    uint32_t n_loads = 0;          // producer: ring loads issued (K and V tiles)
    uint32_t n_cons = 0;           // MMA: ring loads consumed
    uint32_t cnt_a = 0, cnt_b = 0; // MMA: PV rounds of tile A / tile B so far
    uint32_t q_issued = 0;
    for (int blk = 0; blk < n_it; ++blk) {
      const Item itm = item_of(a, pair, blk);
      const int64_t p0 = itm.p0;
      const int nA = (int)(p0 / BKV) + 1;     // KV tiles of tile A (last one diagonal)
      const int j0 = itm.j0, j1 = itm.j1;     // this item's tiles; tile B's last is nA
      const int64_t qrow0 = zz_row_of_pos(p0, a.c, a.D);   // 256 rows, contiguous
      if (warp == WARP_PROD) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !*abort_flag) {
          mbar_arrive_expect_tx(q_full, 2 * TILE_BYTES);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int qr = (int)(qrow0 - a.q_row_off + x * BQ);
            // a tensor copy reads the fill value past its map, so the check reports only
            (void)TSP_INB(qr >= 0 && qr + BQ <= a.lse_ld, a.status);
            tma_load_2d(base + OFF_Q + x * TILE_BYTES, &a.tm_q, a.q_col0 + h * DH, qr, q_full);
            tma_load_2d(base + OFF_Q + x * TILE_BYTES + BOX_BYTES, &a.tm_q, a.q_col0 + h * DH + 64,
                        qr, q_full);
          }
          ++q_issued;
          bool ok = true;
          for (int j = j0; j < j1 && ok; ++j) {
            const int krow = zz_row_of_pos32(j * BKV, (int)a.c, a.D);
            (void)TSP_INB(krow >= 0 && krow + BKV <= a.S, a.status);
#pragma unroll 1
            for (int kv = 0; kv < 2; ++kv) {   // K_j then V_j
              const uint32_t n = n_loads, s = n % NSLOT;
              if (!mbar_wait(slot_empty(s), ((n / NSLOT) & 1u) ^ 1u, a.status, abort_flag,
                             a.limit_ns)) {
                ok = false;
                break;
              }
              const uint32_t dst = base + OFF_KV + s * TILE_BYTES;
              const int col = kcol + kv * a.dkv;
              mbar_arrive_expect_tx(slot_full(s), TILE_BYTES);
              tma_load_2d(dst, &a.tm, col, krow, slot_full(s));
              tma_load_2d(dst + BOX_BYTES, &a.tm, col + 64, krow, slot_full(s));
              ++n_loads;
            }
          }
        }
      } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort_flag) {
          constexpr uint32_t idesc_s = idesc_f16_f32(BQ, BKV, false, false, false);
          constexpr uint32_t idesc_o = idesc_f16_f32(BQ, DH, false, true, false);
          bool ok = mbar_wait(q_full, (uint32_t)blk & 1u, a.status, abort_flag, a.limit_ns);
          // the ring slot of the next load in order, once it is filled
          // (its slot is n_cons % NSLOT before the call)
          auto take = [&]() -> bool {
            const uint32_t n = n_cons++;
            if (!mbar_wait(slot_full(n % NSLOT), (n / NSLOT) & 1u, a.status, abort_flag, a.limit_ns))
              return false;
            tc_fence_after();
            return true;
          };
          // base descriptors, computed once: the issue loops only add constants
          const uint64_t dq0 = sdesc_sw128(base + OFF_Q, 16, 1024);     // Q, K-major
          const uint64_t dk0 = sdesc_sw128(base + OFF_KV, 16, 1024);    // K, K-major
          const uint64_t dv0 = sdesc_sw128(base + OFF_KV, BOX_BYTES, 1024);   // V, MN-major
          auto mma_s = [&](int x, uint32_t kslot) {
            const uint64_t da = sdesc_add(dq0, x * TILE_BYTES);
            const uint64_t db = sdesc_add(dk0, kslot * TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
              umma_f16_ss_hot(tmem + x * 128, sdesc_add(da, off), sdesc_add(db, off), idesc_s,
                              kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full(x));
          };
          auto mma_pv = [&](int x, uint32_t vslot, bool first) -> bool {
            const uint32_t cx = x == 0 ? cnt_a : cnt_b;
            if (!mbar_wait(p_full(x), cx & 1u, a.status, abort_flag, a.limit_ns)) return false;
            tc_fence_after();
            // P_x sits in TMEM (the first 64 columns of S_x, fp16 pairs): A from
            // tensor memory, only V is read from shared memory
            const uint32_t ta = tmem + x * 128;
            const uint64_t db = sdesc_add(dv0, vslot * TILE_BYTES);
            const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
              umma_f16_ts_hot(tmem + 256 + x * 128, ta + kk * 8, sdesc_add(db, kk * 2048), idesc_o,
                              kk > 0 ? 1u : acc0);
            umma_commit(o_done(x));
            if (x == 0) ++cnt_a; else ++cnt_b;
            return true;
          };
          uint32_t kslot = 0, vslot = 0;
          kslot = n_cons % NSLOT;
          if (ok && (ok = take())) {
            mma_s(0, kslot);
            mma_s(1, kslot);
            umma_commit(slot_empty(kslot));
          }
          for (int j = j0; j < j1 && ok; ++j) {
            vslot = n_cons % NSLOT;
            if (!(ok = take())) break;
            uint32_t kn = 0;
            const bool next_k = j + 1 < j1;
            if (j < nA) {
              if (!(ok = mma_pv(0, vslot, j == j0))) break;
              if (next_k) {
                kn = n_cons % NSLOT;
                if (!(ok = take())) break;
                if (j + 1 < nA) mma_s(0, kn);
              }
            } else if (next_k) {
              kn = n_cons % NSLOT;
              if (!(ok = take())) break;
            }
            if (!(ok = mma_pv(1, vslot, j == j0))) break;
            umma_commit(slot_empty(vslot));
            if (next_k) {
              mma_s(1, kn);
              umma_commit(slot_empty(kn));
            }
          }
          if (!ok) {
            umma_commit(drain_bar);
            drain_wait(drain_bar, 0, a.limit_ns);
          }
        }
      }
      block_sync();
    }
    // drain: copies the producer issued that nobody consumed (abort path only)
    if (warp == WARP_PROD && lane == 0 && *abort_flag) {
      const uint32_t n_out = n_loads < (uint32_t)NSLOT ? n_loads : (uint32_t)NSLOT;
      for (uint32_t n = n_loads - n_out; n < n_loads; ++n)
        drain_wait(slot_full(n % NSLOT), (n / NSLOT) & 1u, a.limit_ns);
      if (q_issued > 0) drain_wait(q_full, (q_issued - 1) & 1u, a.limit_ns);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(REG_SOFT));
    uint32_t rounds = 0;           // rounds (S, P, PV) of this thread's tile so far
    for (int blk = 0; blk < n_it; ++blk) {
      const Item itm = item_of(a, pair, blk);
      const int64_t p0 = itm.p0;
      const int nA = (int)(p0 / BKV) + 1;     // KV tiles of tile A (last one diagonal)
      const int nB = nA + 1;                  // tile B has one more, its own diagonal
      const int64_t qrow0 = zz_row_of_pos(p0, a.c, a.D);   // 256 rows, contiguous
      {
        // ------------------------------------------------------------ softmax of tile x
        const int x = warp >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int nX = x == 0 ? nA : nB;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t tm_s = lane_base + x * 128, tm_o = lane_base + 256 + x * 128;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        const int jx1 = min(itm.j1, nX);
        for (int j = itm.j0; j < jx1; ++j) {
          const uint32_t c_now = rounds;
          bool okl = mbar_wait(s_full(x), c_now & 1u, a.status, abort_flag, a.limit_ns);
          if (!__all_sync(0xffffffffu, okl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sr[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tm_s + q * 32, sr[q]);
          tmem_wait_ld();
          if (j == nX - 1) {  // diagonal tile: key index > query index is masked
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (q * 32 + e > row) sr[q][e] = __float_as_uint(-INFINITY);
          }
          // row max over 16 independent partial maxima (short dependency
          // chains), three scores an instruction: 72 max instructions a row
          // instead of 127
          auto S_ = [&](int i) { return __uint_as_float(sr[i >> 5][i & 31]); };
          float mp[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) mp[k] = fmax3f(S_(k), S_(k + 16), S_(k + 32));
#pragma unroll
          for (int k = 0; k < 16; ++k) {   // scores 48 + k + 16 i, i = 0..4
            mp[k] = fmax3f(mp[k], S_(48 + k), S_(64 + k));
            mp[k] = fmax3f(mp[k], S_(80 + k), S_(96 + k));
            mp[k] = fmaxf(mp[k], S_(112 + k));
          }
#pragma unroll
          for (int k = 0; k < 5; ++k) mp[k] = fmax3f(mp[k], mp[k + 5], mp[k + 10]);
          mp[0] = fmax3f(mp[0], mp[1], mp[15]);
          mp[2] = fmax3f(mp[2], mp[3], mp[4]);
          const float mx = fmaxf(mp[0], mp[2]) * a.scale_log2;
          const bool mine = mx > m_used + RESCALE_LOG2;
          const bool resc = __any_sync(0xffffffffu, mine);
          float alpha = 1.f;
          if (resc) {
            const float m_new = mine ? mx : m_used;
            alpha = ex2_approx(m_used - m_new);   // 0 on the first tile, 1 if unchanged
            l *= alpha;
            m_used = m_new;
          }
          // probabilities first (fp16 pairs), so the scores' registers are free
          // before O is touched
          // the exponent in fp32, rounded to fp16 pairs; 2^x of both halves in
          // one MUFU operation, which is already the fp16 P the PV MMA takes
          const float neg_m = -m_used;
          uint32_t ps[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};   // partial row sums (fp16 pairs)
          uint32_t pk[2][32];   // column i of P_x holds keys 2i (low half) and 2i+1
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 xx =
                  ffma2(make_float2(__uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1])),
                        make_float2(a.scale_log2, a.scale_log2), make_float2(neg_m, neg_m));
              const uint32_t p2 = ex2_approx_f16x2(pack_f16(xx.x, xx.y));
              pk[q >> 1][(q & 1) * 16 + (e >> 1)] = p2;
              ps[(e >> 1) & 7] = hadd2_u32(ps[(e >> 1) & 7], p2);   // 8 terms a partial
            }
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) sum += f16_lo(ps[k]) + f16_hi(ps[k]);
          // PV_x(j-1) must have finished before P_x is overwritten or O_x rescaled
          if (j > itm.j0) {
            okl = mbar_wait(o_done(x), (c_now - 1) & 1u, a.status, abort_flag, a.limit_ns);
            if (!__all_sync(0xffffffffu, okl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (resc) {
#pragma unroll 1
              for (int q = 0; q < 4; ++q) {
                uint32_t ov[32];
                tmem_ld32(tm_o + q * 32, ov);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                tmem_st32(tm_o + q * 32, ov);
              }
              tmem_wait_st();
            }
          }
          // P_x into TMEM over the scores just read (columns 0..63 of S_x); the
          // next S_x MMA is issued after PV_x, which reads P_x first
          tmem_st32(tm_s, pk[0]);
          tmem_st32(tm_s + 32, pk[1]);
          tmem_wait_st();
          l += sum;
          tc_fence_before();
          mbar_arrive(p_full(x));
          rounds = c_now + 1;
        }
        // epilogue: O / l -> fp16 rows, LSE (after the last PV of this tile)
        const bool eok =
            ok && mbar_wait(o_done(x), (rounds - 1) & 1u, a.status, abort_flag, a.limit_ns);
        if (__all_sync(0xffffffffu, eok) && a.split_lc) {
          // split mode: this chunk's O / l (fp32) and log2 of its sum
          tc_fence_after();
          const float inv = 1.f / l;
          const int64_t prow = ((int64_t)h * a.n_items + pair) * BLOCK + x * BQ + row;
          const bool p_in = TSP_INB(pair < a.n_items, a.status);
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow * DH);
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t ov[32];
            tmem_ld32(tm_o + q * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              if (p_in) dst[q * 8 + c] = make_float4(
                  __uint_as_float(ov[4 * c + 0]) * inv, __uint_as_float(ov[4 * c + 1]) * inv,
                  __uint_as_float(ov[4 * c + 2]) * inv, __uint_as_float(ov[4 * c + 3]) * inv);
          }
          if (p_in) a.part_lse[prow] = m_used + __log2f(l);
        } else if (__all_sync(0xffffffffu, eok)) {
          tc_fence_after();
          const float inv = 1.f / l;
          const int64_t orow_i = qrow0 - a.o_row_off + x * BQ + row;
          const bool o_in = TSP_INB(orow_i >= 0 && orow_i < a.lse_ld, a.status);
          ct_t* orow = a.o + orow_i * a.ldo + h * DH;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t ov[32];
            tmem_ld32(tm_o + q * 32, ov);
            tmem_wait_ld();
            uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (o_in) dst[c] = make_uint4(
                  pack_f16(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv),
                  pack_f16(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv),
                  pack_f16(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv),
                  pack_f16(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv));
          }
          constexpr float LN2 = 0.69314718055994530942f;
          if (o_in) a.lse[(int64_t)h * a.lse_ld + orow_i] = (m_used + __log2f(l)) * LN2;
        }
        tc_fence_before();
          }
      block_sync();
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

// Split mode: merges the chunks of every query row of the rank by their
// log-sum-exp, O = sum 2^(s_i - M) O_i / sum 2^(s_i - M) with s_i = log2 of
// chunk i's sum and M = max s_i, and LSE = (M + log2 sum) ln 2.  A warp per
// (rank-local row, head); each lane holds four of the DH columns.
__global__ void __launch_bounds__(256) attn_split_merge_kernel(const __grid_constant__ TcAttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rr = (int64_t)blockIdx.x * 8 + warp;   // rank-local row: chunk r, then 2D-1-r
  const int h = blockIdx.y;
  if (rr >= 2 * a.c) return;
  const int nb = a.n_blocks;
  const int64_t within = rr < a.c ? rr : rr - a.c;
  const int k = (int)(within / BLOCK), i = (int)(within - (int64_t)k * BLOCK);
  const int b = rr < a.c ? k : 2 * nb - 1 - k;       // the row's block (split_block_p0 order)
  int first = 0;                                      // its first chunk
  for (int bb = 0; bb < b; ++bb)
    first += split_chunks((int)(split_block_p0(a, bb) / BKV) + 2, a.split_lc);
  const int64_t p0 = split_block_p0(a, b);
  const int nch = split_chunks((int)(p0 / BKV) + 2, a.split_lc);
  const int64_t orow = zz_row_of_pos(p0, a.c, a.D) - a.o_row_off + i;
  if (!TSP_INB(first + nch <= a.n_items && orow >= 0 && orow < a.lse_ld, a.status)) return;
  const int64_t base = ((int64_t)h * a.n_items + first) * BLOCK + i;
  float M = -INFINITY;
  for (int s = 0; s < nch; ++s) M = fmaxf(M, a.part_lse[base + (int64_t)s * BLOCK]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  for (int s = 0; s < nch; ++s) {
    const int64_t pr = base + (int64_t)s * BLOCK;
    const float w = exp2f(a.part_lse[pr] - M);
    const float4 v = reinterpret_cast<const float4*>(a.part_o + pr * DH)[lane];
    L += w;
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  const float inv = 1.f / L;
  *reinterpret_cast<uint2*>(a.o + orow * a.ldo + h * DH + lane * 4) =
      make_uint2(pack_f16(acc.x * inv, acc.y * inv), pack_f16(acc.z * inv, acc.w * inv));
  constexpr float LN2 = 0.69314718055994530942f;
  if (lane == 0) a.lse[(int64_t)h * a.lse_ld + orow] = (M + __log2f(L)) * LN2;
}

}  // namespace

// The one-rank split plan for a launch of H heads: no split while the rank's
// 256-row block pairs and heads give at least kSplitBelow CTAs (half of the
// 152 SMs); else chunks of lc key tiles, lc sized for about kSplitCtas CTAs
// (one wave: 304 CTAs took 1% longer, their extra partials costing the merge
// more than the finer chunks saved; 456 took 3% longer).
// n_items_max bounds the chunks of one head over the rank's blocks for every
// rank: with T the key tiles of a rank's blocks (the same for every rank:
// mirrored blocks' counts add up to a constant), sum (nB_b - 2) / lc + 1 is at
// most T / lc + 2 nb.
void attn_rank_split_plan(int64_t S, int D, int H, int* lc, int* n_items_max) {
  constexpr int kSplitBelow = 76, kSplitCtas = 152;
  const int64_t c = S / (2 * D), nb = c / BLOCK;
  *lc = 0;
  *n_items_max = 0;
  if (nb < 1 || nb * H >= kSplitBelow) return;
  const int64_t T = nb * (((2 * (int64_t)D - 1) * c + (nb - 1) * BLOCK) / BKV + 4);
  const int64_t l = std::max<int64_t>(2, (T * H + kSplitCtas - 1) / kSplitCtas);
  *lc = (int)l;
  *n_items_max = (int)(T / l + 2 * nb);
}

namespace {

// fp16 [rows, cols] row-major, box {64 columns, 128 rows}, 128-byte swizzle
bool attn_map(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows) {
  return tma_map_f16(m, ptr, cols, rows, cols, 128);
}

// a: maps, pointers and offsets filled in; the common fields, checks and launch
tsp_status attn_launch(TcAttnArgs* a, int64_t S, int H, int Hkv, int dh, int D, int nranks,
                       cudaStream_t st) {
  a->S = S;
  a->c = S / (2 * D);
  a->D = D;
  a->d = H * dh;
  a->G = H / Hkv;
  a->dkv = Hkv * dh;
  a->n_blocks = (int)(a->c / BLOCK);
  a->scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  a->status = status_word();
  a->limit_ns = wait_limit_ns();
  static bool attr[kMaxDevices] = {};   // the attribute holds for one device
  static int launch_regs = 0;
  const int dev = current_device();
  if (!attr[dev]) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    cudaFuncAttributes fa;
    TSP_CUDA_TRY(cudaFuncGetAttributes(&fa, attn_fwd_tc_kernel));
    launch_regs = fa.numRegs;
    attr[dev] = true;
  }
  // setmaxnreg.inc would wait forever if the split exceeded the launch allocation
  if ((int64_t)launch_regs * NTHR < (int64_t)REG_TOTAL) return TSP_ERR_UNSUPPORTED;
  dim3 grid((unsigned)(a->split_lc ? a->n_items : nranks * a->n_blocks), (unsigned)H);
  {
    Prof prof("attn_fwd", st);
    attn_fwd_tc_kernel<<<grid, NTHR, SMEM, st>>>(*a);
    TSP_CUDA_TRY(cudaGetLastError());
  }
  if (a->split_lc) {
    Prof prof("attn_split_merge", st);
    dim3 mgrid((unsigned)((2 * a->c + 7) / 8), (unsigned)H);
    attn_split_merge_kernel<<<mgrid, 256, 0, st>>>(*a);
    TSP_CUDA_TRY(cudaGetLastError());
  }
  return TSP_OK;
}

}  // namespace

tsp_status launch_attn_fwd_f16(const void* qkv, void* o, float* lse, int64_t S, int H, int Hkv,
                               int dh, int D, cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BLOCK != 0) return TSP_ERR_UNSUPPORTED;
  if (S > (int64_t)INT32_MAX) return TSP_ERR_UNSUPPORTED;
  if (Hkv < 1 || H % Hkv != 0) return TSP_ERR_INVALID_ARG;
  const int d = H * dh, dkv = Hkv * dh;
  const int64_t ld = d + 2 * (int64_t)dkv;
  if (((uintptr_t)qkv & 15u) || ((ld * 2) % 16)) return TSP_ERR_INVALID_ARG;
  TcAttnArgs* a = new TcAttnArgs();
  std::unique_ptr<TcAttnArgs> guard(a);
  memset(a, 0, sizeof(TcAttnArgs));
  // Q, K and V all in the one Q|K|V buffer: Q at column 0, K at d, V at d + dkv
  if (!attn_map(&a->tm, qkv, ld, S)) return TSP_ERR_CUDA;
  a->tm_q = a->tm;
  a->kv_col0 = d;
  a->o = (ct_t*)o;
  a->ldo = d;
  a->lse = lse;
  a->lse_ld = S;
  return attn_launch(a, S, H, Hkv, dh, D, D, st);
}

tsp_status launch_attn_fwd_rank_f16(const void* q, int64_t ldq, const void* kv, int64_t ldkv,
                                    void* o, int64_t ldo, float* lse, float* part_o,
                                    float* part_lse, int64_t S, int H, int dh, int D, int r,
                                    cudaStream_t st) {
  if (dh != DH) return TSP_ERR_UNSUPPORTED;
  const int64_t c = S / (2 * D);
  if (c % BLOCK != 0 || S > (int64_t)INT32_MAX) return TSP_ERR_UNSUPPORTED;
  if (r < 0 || r >= D || H < 1) return TSP_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15u) || ((uintptr_t)kv & 15u) || ((ldq * 2) % 16) || ((ldkv * 2) % 16) ||
      ldq < (int64_t)H * dh || ldkv < 2 * (int64_t)H * dh)
    return TSP_ERR_INVALID_ARG;
  TcAttnArgs* a = new TcAttnArgs();
  std::unique_ptr<TcAttnArgs> guard(a);
  memset(a, 0, sizeof(TcAttnArgs));
  // the rank's own 2c rows of Q; the gathered K|V of all S rows (K at 0, V at H*dh)
  if (!attn_map(&a->tm_q, q, ldq, 2 * c) || !attn_map(&a->tm, kv, ldkv, S)) return TSP_ERR_CUDA;
  a->q_row_off = a->o_row_off = (int64_t)r * 2 * c;
  a->rank0 = r;
  a->o = (ct_t*)o;
  a->ldo = ldo;
  a->lse = lse;
  a->lse_ld = 2 * c;
  int lc = 0, n_max = 0;
  attn_rank_split_plan(S, D, H, &lc, &n_max);
  if (lc > 0) {
    // this rank's chunk count (at most the plan's bound, which sized the partials)
    const int nb = (int)(c / BLOCK);
    int n = 0;
    for (int b = 0; b < 2 * nb; ++b) {
      const int64_t pb = b < nb ? (int64_t)r * c + (int64_t)b * BLOCK
                                : (int64_t)(2 * D - 1 - r) * c + (int64_t)(2 * nb - 1 - b) * BLOCK;
      n += (int)((pb / BKV + 2 - 2) / lc + 1);
    }
    if (n > n_max || !part_o || !part_lse || ((uintptr_t)part_o & 15u))
      return TSP_ERR_INVALID_ARG;
    a->split_lc = lc;
    a->n_items = n;
    a->part_o = part_o;
    a->part_lse = part_lse;
  }
  return attn_launch(a, S, H, H, dh, D, 1, st);
}

}  // namespace tsp
