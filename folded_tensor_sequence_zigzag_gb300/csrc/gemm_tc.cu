// gemm_tc.cu -- shard-streamed projection GEMMs on the 5th-generation tensor
// cores (tcgen05.mma kind::f16, bf16 operands, fp32 accumulators in TMEM).
//
// Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference" (gist.science summary), section 2:
//  * attention layers: the packed W_Q/W_K/W_V/W_O shards are broadcast one at
//    a time and every rank projects its own tokens with the current shard --
//    here the N range of the Q|K|V GEMM is segmented by shard (split-N), and
//    the W_O projection sums the shards' partial outputs (split-K) in fp32;
//  * gated-MLP layers: the W_1/W_3/W_2 shards travel around a ring and every
//    rank accumulates its partial output locally (no all-reduce) -- here the
//    W_2 GEMM walks its K range shard by shard in the ring order of the
//    virtual rank that owns the row tile, (r - t) mod D at step t, with the
//    running sum kept in the fp32 TMEM accumulator.
//
// Kernel structure (one CTA per SM, persistent over output tiles):
// Operands are fp16 (the block's internal tensor-core type, see common.cuh).
//   warps 0-3  epilogue: tcgen05.ld the 128x256 fp32 accumulator (one TMEM
//              lane = one output row per thread), fused epilogue, stores;
//   warp 4     TMA producer: 4-stage ring of A (128x64) + B (256x64) tiles
//              in 128-byte-swizzled shared memory;
//   warp 5     TMEM allocator + single-thread tcgen05.mma issuer.
// Two 256-column accumulators (512 TMEM columns) let the epilogue of tile i
// overlap the main loop of tile i+1.  Every mbarrier wait is bounded; a wait
// that runs out records TSP_ERR_TIMEOUT, drains the CTA's copies and MMAs,
// frees TMEM and returns.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <memory>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"

namespace tsp {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;

struct KParams {
  CUtensorMap ta[3];
  CUtensorMap tb[3];
  int M, N, K;
  int nkb;
  int nks;
  int kseg_kb[4];
  int nseg_n;
  int rot_rows, rot_D, rot_r0;
  int tiles_m, tiles_n, group_m, group_n;   // tile order: see slab_order()
  int n_tile;  // output columns per tile (256, or 128 for the paired SwiGLU tile)
  void* out;
  int64_t ldo;
  void* out2;
  int64_t ldo2;
  void* out3;
  int64_t ldo3;
  const void* res;
  int64_t ldr;
  int res_f32, out_type;
  const void* e1;
  const void* e2;
  int64_t lde;
  int64_t m_seg;
  void* outs[3];
  int n_split;   // EPI_STORE: columns from here on go to out2
  int* status;
  uint64_t limit_ns;
  int debug_skip;  // failure-detection test: CTA 0 never loads its first stage
  int shard_kb[65];
};

// Output tile of tile index t.  The output is walked in slabs: group_m
// M-tiles across every N-tile (group_n == 0), or group_n N-tiles across every
// M-tile; inside a slab the slab's own dimension varies fastest, so the tiles
// that run at the same time on the persistent CTAs share the slab's operand
// tiles and every wave touches all of them.
__device__ __forceinline__ void tile_of(const KParams& p, int t, int& mb, int& nb) {
  if (p.group_n > 0) {
    const int per_group = p.group_n * p.tiles_m;
    const int g = t / per_group;
    const int first = g * p.group_n;
    const int gs = min(p.tiles_n - first, p.group_n);
    const int r = t - g * per_group;
    nb = first + r % gs;
    mb = r / gs;
    return;
  }
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int gs = min(p.tiles_m - first, p.group_m);
  const int r = t - g * per_group;
  mb = first + r % gs;
  nb = r / gs;
}

__device__ __forceinline__ int kseg_of(const KParams& p, int kb) {
  int s = 0;
  while (s + 1 < p.nks && kb >= p.kseg_kb[s + 1]) ++s;
  return s;
}

// Waits that ignore the abort flag (used only to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

template <typename T>
__device__ __forceinline__ void store16x32(T* dst, const float* f) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d4[q] = make_uint4(pack2<T>(f[8 * q + 0], f[8 * q + 1]), pack2<T>(f[8 * q + 2], f[8 * q + 3]),
                       pack2<T>(f[8 * q + 4], f[8 * q + 5]), pack2<T>(f[8 * q + 6], f[8 * q + 7]));
}
template <typename T>
__device__ __forceinline__ void load16x32(const T* src, float* f) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = s4[q];
    f[8 * q + 0] = lo2<T>(v.x); f[8 * q + 1] = hi2<T>(v.x);
    f[8 * q + 2] = lo2<T>(v.y); f[8 * q + 3] = hi2<T>(v.y);
    f[8 * q + 4] = lo2<T>(v.z); f[8 * q + 5] = hi2<T>(v.z);
    f[8 * q + 6] = lo2<T>(v.w); f[8 * q + 7] = hi2<T>(v.w);
  }
}
__device__ __forceinline__ void store_f32x32(float* dst, const float* f) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d4[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
}
// out_type: OUT_F16 (internal operand), OUT_BF16 (API output), OUT_F32
__device__ __forceinline__ void store_any32(void* base, int64_t off, const float* f, int out_type) {
  if (out_type == OUT_F32) store_f32x32((float*)base + off, f);
  else if (out_type == OUT_BF16) store16x32((__nv_bfloat16*)base + off, f);
  else store16x32((ct_t*)base + off, f);
}

template <int EPI, bool A_MN, bool B_MN, bool PAIRED>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_tc_kernel(const __grid_constant__ KParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + STAGES * STAGE_BYTES;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bars + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bars + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + STAGES * STAGE_BYTES + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + STAGES * STAGE_BYTES + 136);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // a device error recorded earlier (sticky until the host resets it) skips the
  // work; thread 0 alone reads the word and the barrier hands every thread the
  // same answer, so the CTA leaves whole or not at all
  if (__syncthreads_or(threadIdx.x == 0 && *(volatile int*)p.status != 0)) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    for (int i = 0; i < p.nks; ++i) {
      tma_prefetch_desc(&p.ta[i]);
      tma_prefetch_desc(&p.tb[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = p.tiles_m * p.tiles_n;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_of(p, t, mb, nb);
        const int m0 = mb * BM, n0 = nb * p.n_tile;
        int rank = 0;
        if (p.rot_D > 0) rank = min(p.rot_r0 + m0 / p.rot_rows, p.rot_D - 1);
        int step = 0, sh = rank, kb = p.rot_D > 0 ? p.shard_kb[rank] : 0;
        for (int i = 0; i < p.nkb; ++i) {
          if (p.rot_D > 0) {
            while (kb >= p.shard_kb[sh + 1]) {
              if (!TSP_INB(step + 1 < p.rot_D, p.status)) break;   // shard table exhausted
              ++step;
              sh = (rank - step + p.rot_D) % p.rot_D;
              kb = p.shard_kb[sh];
            }
          } else {
            kb = i;
          }
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status, abort_flag, p.limit_ns)) {
            ok = false;
            break;
          }
          if (p.debug_skip && blockIdx.x == 0 && issued == 0 && i == 0) {
            // test knob: this stage is never filled, so the MMA's wait on it runs out
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            ++kb;
            continue;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const int seg = kseg_of(p, kb);
          const int kloc = (kb - p.kseg_kb[seg]) * BK;
          // A tile
          if (!A_MN) {
            tma_load_2d(sa, &p.ta[seg], kloc, m0, fb);
          } else {
            tma_load_2d(sa, &p.ta[seg], m0, kloc, fb);
            tma_load_2d(sa + 8192, &p.ta[seg], m0 + 64, kloc, fb);
          }
          // B tile
          if (PAIRED) {
            tma_load_2d(sb, &p.tb[0], kloc, n0, fb);
            tma_load_2d(sb + B_BYTES / 2, &p.tb[1], kloc, n0, fb);
          } else {
            int bi = seg, nl = n0;
            if (p.nseg_n > 0) {
              bi = n0 / p.nseg_n;
              nl = n0 - bi * p.nseg_n;
            }
            if (!B_MN) {
              tma_load_2d(sb, &p.tb[bi], kloc, nl, fb);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) tma_load_2d(sb + 8192 * j, &p.tb[bi], nl + 64 * j, kloc, fb);
            }
          }
          ++issued;
          ++kb;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // drain the copies still in flight before the CTA may exit
        const uint32_t n_out = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
        for (uint32_t j = issued - n_out; j < issued; ++j)
          drain_wait(full_bar(j % STAGES), (j / STAGES) & 1u, p.limit_ns);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN, A_MN, B_MN, false);
      // stage-0 descriptors, computed once: the issue loop only adds constants
      const uint64_t da0 = A_MN ? sdesc_sw128(base, 8192, 1024) : sdesc_sw128(base, 16, 1024);
      const uint64_t db0 = B_MN ? sdesc_sw128(base + A_BYTES, 8192, 1024)
                                : sdesc_sw128(base + A_BYTES, 16, 1024);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, p.status, abort_flag, p.limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * BN;
        for (int i = 0; i < p.nkb; ++i) {
          if (!mbar_wait(full_bar(stage), phase, p.status, abort_flag, p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = sdesc_add(da0, stage * STAGE_BYTES);
          const uint64_t db = sdesc_add(db0, stage * STAGE_BYTES);
          const uint32_t acc0 = i != 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_f16_ss_hot(d_tmem, sdesc_add(da, A_MN ? kk * 2048 : kk * 32),
                            sdesc_add(db, B_MN ? kk * 2048 : kk * 32), idesc, kk > 0 ? 1u : acc0);
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // wait until every MMA this thread issued has completed
        umma_commit(drain_bar);
        drain_wait(drain_bar, 0, p.limit_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    int acc = 0;
    uint32_t acc_phase = 0;
    const int row = warp * 32 + lane;
    bool bad = false;   // an fp16 output out of range
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_of(p, t, mb, nb);
      const int m0 = mb * BM, n0 = nb * p.n_tile;
      const int m = m0 + row;
      if (!mbar_wait(tfull_bar(acc), acc_phase, p.status, abort_flag, p.limit_ns)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)acc * BN;
      const bool row_ok = m < p.M;
      if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t va[32], vb[32];
          tmem_ld32(tb + c * 32, va);
          tmem_ld32(tb + 128 + c * 32, vb);
          tmem_wait_ld();
          const int n = n0 + c * 32;
          if (row_ok && n < p.N) {
            float g[32], fa[32], fb[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              fa[j] = __uint_as_float(va[j]);
              fb[j] = __uint_as_float(vb[j]);
              g[j] = fa[j] * sigmoidf_(fa[j]) * fb[j];
            }
            bad |= f16_bad_n<32>(g);
            if (p.out2) bad |= f16_bad_n<32>(fa) | f16_bad_n<32>(fb);
            store16x32((ct_t*)p.out + (int64_t)m * p.ldo + n, g);
            if (p.out2) store16x32((ct_t*)p.out2 + (int64_t)m * p.ldo2 + n, fa);
            if (p.out3) store16x32((ct_t*)p.out3 + (int64_t)m * p.ldo3 + n, fb);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_wait_ld();
          const int n = n0 + c * 32;
          if (!row_ok || n >= p.N) continue;
          float f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
          if constexpr (EPI == EPI_STORE) {
            if (p.out_type == OUT_F16) bad |= f16_bad_n<32>(f);
            if (p.n_split > 0 && n >= p.n_split)
              store_any32(p.out2, (int64_t)m * p.ldo2 + (n - p.n_split), f, p.out_type);
            else
              store_any32(p.out, (int64_t)m * p.ldo + n, f, p.out_type);
          } else if constexpr (EPI == EPI_RES) {
            float r[32];
            if (p.res_f32) {
              const float4* r4 = reinterpret_cast<const float4*>((const float*)p.res +
                                                                 (int64_t)m * p.ldr + n);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 t4 = r4[q];
                r[4 * q] = t4.x; r[4 * q + 1] = t4.y; r[4 * q + 2] = t4.z; r[4 * q + 3] = t4.w;
              }
            } else {
              load16x32((const __nv_bfloat16*)p.res + (int64_t)m * p.ldr + n, r);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] += r[j];
            if (p.out_type == OUT_F16) bad |= f16_bad_n<32>(f);
            store_any32(p.out, (int64_t)m * p.ldo + n, f, p.out_type);
          } else if constexpr (EPI == EPI_F32) {
            float* dst;
            if (p.m_seg > 0) {
              const int sgi = (int)(m / p.m_seg);
              if (!TSP_INB(sgi >= 0 && sgi < 3 && p.outs[sgi] != nullptr, p.status)) continue;
              dst = (float*)p.outs[sgi] + (int64_t)(m - sgi * p.m_seg) * p.ldo + n;
            } else {
              dst = (float*)p.out + (int64_t)m * p.ldo + n;
            }
            store_f32x32(dst, f);
          } else if constexpr (EPI == EPI_SWIGLU_BWD) {
            // f = dG;  e1 = A, e2 = B (pre-activations, bf16)
            float a[32], b[32], da[32], db[32];
            load16x32((const ct_t*)p.e1 + (int64_t)m * p.lde + n, a);
            load16x32((const ct_t*)p.e2 + (int64_t)m * p.lde + n, b);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float s = sigmoidf_(a[j]);
              da[j] = f[j] * b[j] * s * (1.f + a[j] * (1.f - s));
              db[j] = f[j] * a[j] * s;
            }
            bad |= f16_bad_n<32>(da) | f16_bad_n<32>(db);
            store16x32((ct_t*)p.out + (int64_t)m * p.ldo + n, da);
            store16x32((ct_t*)p.out2 + (int64_t)m * p.ldo2 + n, db);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (bad) report_status(p.status, (int)TSP_ERR_RANGE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

template <int EPI, bool A_MN, bool B_MN, bool PAIRED>
tsp_status launch_t(const KParams& kp, int grid, cudaStream_t st, const char* name) {
  Prof prof(name, st);
  static bool attr_set[kMaxDevices] = {};   // the attribute holds for one device
  auto kern = gemm_tc_kernel<EPI, A_MN, B_MN, PAIRED>;
  const int dev = current_device();
  if (!attr_set[dev]) {
    TSP_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    attr_set[dev] = true;
  }
  kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(kp);
  TSP_CUDA_TRY(cudaGetLastError());
  return TSP_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// L2 share (bytes) that the resident operand slab of a GEMM may take: the
// rest of the 129 MB L2 holds the streamed operand's tiles in flight and the
// output lines being written back.  Measured on the 7B-shaped block forward
// (S=16384): 48 MB beats the fixed 16-M-tile order (W_1|W_3 -3.5%, W_2 and
// W_O -1.5%), while 64 MB and 96 MB slabs were 7% and 16% slower -- lines
// read by SMs of both dies seem to occupy L2 space on both, so only about
// half of the L2 is there for a resident slab.  TSP_GEMM_SLAB_MB (read once) overrides
// the default for tuning runs; 0 keeps the fixed order of 16-M-tile slabs.
size_t slab_budget() {
  static size_t v = [] {
    const char* e = getenv("TSP_GEMM_SLAB_MB");
    size_t mb = 48;
    if (e && atoll(e) >= 0 && *e) mb = (size_t)atoll(e);
    return mb << 20;
  }();
  return v;
}

// Tile order of a GEMM: which operand slab stays in L2.  A slab of g M-tiles
// (BM rows of A, all of K each) is read once and every wave of the slab
// touches all of it, so it stays resident while the B tiles stream past; B
// is then read once per slab.  DRAM reads of the operands:
//   M slabs of g tiles: A + B * ceil(tiles_m / g)
//   N slabs of g tiles: B + A * ceil(tiles_n / g)
// with g as large as the slab budget allows; the cheaper order wins.  For a
// very long K (the weight gradients, K = tokens) a slab holds few tiles and
// the reuse inside one wave dominates; those keep slabs of 16 M-tiles.
void slab_order(KParams* kp, int K) {
  const double a_tile = (double)BM * K * 2, b_tile = 256.0 * K * 2;   // fp16 operand bytes
  const double A = a_tile * kp->tiles_m, B = b_tile * kp->tiles_n;
  kp->group_n = 0;
  kp->group_m = std::min(16, kp->tiles_m);
  const double budget = (double)slab_budget();
  if (K > 16384 || budget <= 0) return;
  const int gm = (int)std::max(1.0, std::min((double)kp->tiles_m, std::floor(budget / a_tile)));
  const int gn = (int)std::max(1.0, std::min((double)kp->tiles_n, std::floor(budget / b_tile)));
  const double via_m = A + B * std::ceil((double)kp->tiles_m / gm);
  const double via_n = B + A * std::ceil((double)kp->tiles_n / gn);
  if (via_n < via_m) {
    kp->group_n = gn;
  } else {
    kp->group_m = gm;
  }
}

}  // namespace

tsp_status gemm_tc(const TcGemm& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return TSP_ERR_INVALID_ARG;
  if (g.nks < 1 || g.nks > 3) return TSP_ERR_INVALID_ARG;
  if (g.N % 32 != 0) return TSP_ERR_UNSUPPORTED;
  KParams* kp = new KParams();
  std::unique_ptr<KParams> guard(kp);
  memset(kp, 0, sizeof(KParams));
  kp->M = g.M;
  kp->N = g.N;
  kp->K = g.K;
  kp->nks = g.nks;
  int kb0 = 0;
  for (int s = 0; s < g.nks; ++s) {
    kp->kseg_kb[s] = kb0;
    const int len = g.kseg_len[s];
    if (len <= 0) return TSP_ERR_INVALID_ARG;
    if (s + 1 < g.nks && len % BK != 0) return TSP_ERR_UNSUPPORTED;
    kb0 += (len + BK - 1) / BK;
  }
  kp->kseg_kb[g.nks] = kb0;
  kp->nkb = kb0;
  kp->nseg_n = g.nseg_n;
  kp->n_tile = g.paired ? 128 : BN;
  kp->tiles_m = (g.M + BM - 1) / BM;
  kp->tiles_n = (g.N + kp->n_tile - 1) / kp->n_tile;
  slab_order(kp, g.K);
  // operand maps
  for (int s = 0; s < g.nks; ++s) {
    const int klen = g.kseg_len[s];
    if (!aligned16(g.A[s]) || (g.lda[s] * 2) % 16 != 0) return TSP_ERR_INVALID_ARG;
    bool ok = g.a_mn ? tma_map_f16(&kp->ta[s], g.A[s], g.M, klen, g.lda[s], 64)
                     : tma_map_f16(&kp->ta[s], g.A[s], klen, g.M, g.lda[s], BM);
    if (!ok) return TSP_ERR_CUDA;
  }
  const int nb_maps = g.paired ? 2 : (g.nseg_n > 0 ? (g.N + g.nseg_n - 1) / g.nseg_n : g.nks);
  if (nb_maps > 3) return TSP_ERR_UNSUPPORTED;
  if (g.nseg_n > 0 && g.nseg_n % BN != 0) return TSP_ERR_UNSUPPORTED;
  for (int s = 0; s < nb_maps; ++s) {
    if (!aligned16(g.B[s]) || (g.ldb[s] * 2) % 16 != 0) return TSP_ERR_INVALID_ARG;
    const int klen = (g.nseg_n > 0 || g.paired) ? g.K : g.kseg_len[s];
    const int nlen = g.paired ? g.N : (g.nseg_n > 0 ? g.nseg_n : g.N);
    bool ok;
    if (g.paired) ok = tma_map_f16(&kp->tb[s], g.B[s], klen, nlen, g.ldb[s], 128);
    else if (g.b_mn) ok = tma_map_f16(&kp->tb[s], g.B[s], nlen, klen, g.ldb[s], 64);
    else ok = tma_map_f16(&kp->tb[s], g.B[s], klen, nlen, g.ldb[s], BN);
    if (!ok) return TSP_ERR_CUDA;
  }
  // ring rotation over shard segments of K (k-block granularity: a block
  // that straddles a shard boundary belongs to the later shard)
  if (g.rot_D > 0) {
    if (g.rot_D > 64 || g.rot_rows <= 0 || g.rot_r0 < 0 || g.rot_r0 >= g.rot_D)
      return TSP_ERR_INVALID_ARG;
    kp->rot_D = g.rot_D;
    kp->rot_rows = g.rot_rows;
    kp->rot_r0 = g.rot_r0;
    for (int s = 0; s <= g.rot_D; ++s) {
      const int64_t e = (int64_t)s * g.K / g.rot_D;
      kp->shard_kb[s] = (s == g.rot_D) ? kp->nkb : (int)(e / BK);
    }
  }
  kp->out = g.out;
  kp->ldo = g.ldo;
  kp->out2 = g.out2;
  kp->ldo2 = g.ldo2;
  if (g.n_split < 0 || (g.n_split > 0 && (g.epi != EPI_STORE || g.n_split % BN != 0 ||
                                          g.n_split >= g.N || !g.out2)))
    return TSP_ERR_INVALID_ARG;
  kp->n_split = g.n_split;
  kp->out3 = g.out3;
  kp->ldo3 = g.ldo3;
  kp->res = g.res;
  kp->ldr = g.ldr;
  kp->res_f32 = g.res_f32 ? 1 : 0;
  kp->out_type = g.out_type;
  kp->e1 = g.e1;
  kp->e2 = g.e2;
  kp->lde = g.lde;
  kp->m_seg = g.m_seg;
  for (int i = 0; i < 3; ++i) kp->outs[i] = g.outs[i];
  kp->status = status_word();
  kp->limit_ns = wait_limit_ns();
  // tsp_debug_skip_stage: CTA 0 of this GEMM never fills its first pipeline
  // stage, which exercises the bounded-wait path (TSP_ERR_TIMEOUT in the status
  // word after TSP_WAIT_LIMIT_MS) without a fault or a hang
  kp->debug_skip = take_debug_skip() ? 1 : 0;
  const int tiles = kp->tiles_m * kp->tiles_n;
  const int grid = std::min(tiles, num_sms());
  switch (g.epi) {
    case EPI_STORE:
      if (!g.a_mn && !g.b_mn) return launch_t<EPI_STORE, false, false, false>(*kp, grid, st, g.name);
      if (!g.a_mn && g.b_mn) return launch_t<EPI_STORE, false, true, false>(*kp, grid, st, g.name);
      break;
    case EPI_RES:
      if (!g.a_mn && !g.b_mn) return launch_t<EPI_RES, false, false, false>(*kp, grid, st, g.name);
      // one rank's W_O / W_2 shard, stored transposed in the packed shard
      if (!g.a_mn && g.b_mn) return launch_t<EPI_RES, false, true, false>(*kp, grid, st, g.name);
      // weight gradients added over sequence tiles (fp32 residual = the output)
      if (g.a_mn && g.b_mn) return launch_t<EPI_RES, true, true, false>(*kp, grid, st, g.name);
      break;
    case EPI_SWIGLU:
      if (g.paired && !g.a_mn && !g.b_mn) return launch_t<EPI_SWIGLU, false, false, true>(*kp, grid, st, g.name);
      break;
    case EPI_SWIGLU_BWD:
      if (!g.a_mn && g.b_mn) return launch_t<EPI_SWIGLU_BWD, false, true, false>(*kp, grid, st, g.name);
      // one rank's W_2 shard, stored transposed in the packed ring shard
      if (!g.a_mn && !g.b_mn) return launch_t<EPI_SWIGLU_BWD, false, false, false>(*kp, grid, st, g.name);
      break;
    case EPI_F32:
      if (!g.a_mn && g.b_mn) return launch_t<EPI_F32, false, true, false>(*kp, grid, st, g.name);
      if (g.a_mn && g.b_mn) return launch_t<EPI_F32, true, true, false>(*kp, grid, st, g.name);
      if (!g.a_mn && !g.b_mn) return launch_t<EPI_F32, false, false, false>(*kp, grid, st, g.name);
      break;
    default:
      break;
  }
  return TSP_ERR_UNSUPPORTED;
}

}  // namespace tsp
