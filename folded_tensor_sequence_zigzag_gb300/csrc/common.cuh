// common.cuh -- shared device helpers of the TSP block kernels (sm_103a).
//
// Inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the
// 5th-generation tensor-core instructions (tcgen05.*), the bounded-wait
// discipline every pipeline uses, and small numeric helpers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsp.h"

namespace tsp {

// ---------------------------------------------------------------------------
// Host-side plumbing shared by the translation units
// ---------------------------------------------------------------------------

// Device address of the sticky status word (defined in api.cu).  Kernels get
// it as a parameter; they write TSP_ERR_TIMEOUT there and never trap.
int* status_word();
int num_sms();
// Ordinal of the current device (0 if it cannot be read).  Per-device state
// (function attributes, symbol addresses) is kept in arrays of kMaxDevices.
constexpr int kMaxDevices = 64;
int current_device();
// Failure-detection knob (tsp_debug_skip_stage): true for each of the next n
// tensor-core GEMM launches after tsp_debug_skip_stage(n).
bool take_debug_skip();
// Default limit of one pipeline wait, in nanoseconds of %globaltimer.
uint64_t wait_limit_ns();
// Tensor map of a row-major fp16 matrix [outer, inner] with row stride ld
// elements: box {64 inner, box_outer}, 128-byte swizzle, zero fill out of
// bounds (cuTensorMapEncodeTiled, looked up once from the driver).  False if
// the driver lacks the call or rejects the layout.
bool tma_map_f16(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld,
                 int box_outer);

// Launch accounting (api.cu): counts the kernels of one launch site and,
// while profiling is enabled (tsp_profile_enable), brackets them with CUDA
// events recorded on the launch stream.
class Prof {
 public:
  Prof(const char* name, cudaStream_t st, int kernels = 1);
  ~Prof();
  Prof(const Prof&) = delete;
  Prof& operator=(const Prof&) = delete;

 private:
  const char* name_;
  int kernels_;
  cudaStream_t st_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
  bool on_ = false;
};

#define TSP_CUDA_TRY(expr)                      \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    if (e_ != cudaSuccess) return TSP_ERR_CUDA; \
  } while (0)

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_timeout(int* status) {
  atomicCAS(status, 0, (int)TSP_ERR_TIMEOUT);
}
// Records `code` in the sticky status word unless an error is already there.
__device__ __forceinline__ void report_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

// ---- checked build -------------------------------------------------------------
// Compiled with -DTSP_CHECK, TSP_INB(cond, status) tests a computed index before
// the global access it guards: when cond fails it records TSP_ERR_BOUNDS in the
// sticky status word and the caller skips the access.  In the normal build it
// is the constant true and compiles away.
#ifdef TSP_CHECK
__device__ __forceinline__ bool tsp_inb(bool ok, int* status) {
  if (!ok) report_status(status, (int)TSP_ERR_BOUNDS);
  return ok;
}
#define TSP_INB(cond, status) ::tsp::tsp_inb((cond), (status))
#else
#define TSP_INB(cond, status) true
#endif

// Two fp32 operations in one instruction (the .f32x2 forms, sm_100 and
// later): the same rounding as two scalar ones, half the issue slots.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// fp16 range of the internal tensor-core operands: a value becomes a finite
// fp16 only if |v| < 65520 (the largest fp16, 65504, plus half its spacing);
// anything else -- NaN included -- turns into inf or NaN.  Kernels that store
// an fp16 operand OR this test over the values they store and record
// TSP_ERR_RANGE once.
__device__ __forceinline__ bool f16_bad(float v) { return !(fabsf(v) < 65520.f); }
template <int N>
__device__ __forceinline__ bool f16_bad_n(const float* f) {
  bool b = false;
#pragma unroll
  for (int j = 0; j < N; ++j) b |= f16_bad(f[j]);
  return b;
}

// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the barrier to complete, for at most limit_ns.
// On time-out it records TSP_ERR_TIMEOUT in *status, raises the CTA's abort
// flag and returns false; callers then leave their loops.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status,
                                          volatile int* abort_flag, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        report_timeout(status);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---- TMA --------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  x is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ---- tcgen05 (TMEM + UMMA) ----------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same MMA for hot issue loops: no memory clobber, so the issuing thread's
// descriptor arithmetic is scheduled freely around it.  Ordering against the
// mbarrier waits that guard the operands still holds (volatile asm statements
// keep their order), and the MMA touches no memory the compiler tracks.
// One thread issues every MMA of a CTA, so its per-instruction cost adds up:
// a K=16 step of an M=128 x N=128 MMA takes 64 tensor-core cycles, which the
// issue path (descriptor arithmetic included) must stay under.
__device__ __forceinline__ void umma_f16_ss_hot(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A (M rows = TMEM lanes,
// K = 16 fp16 values packed two per 32-bit column, lower index in the low
// half) is read from tensor memory, so only B is fetched from shared memory.
__device__ __forceinline__ void umma_f16_ts_hot(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (taddr.lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the MUFU unit (ftz); -inf gives +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 2^x of both fp16 halves of a packed pair (one MUFU operation for two)
__device__ __forceinline__ uint32_t ex2_approx_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (128-byte swizzle).
//   K-major operand: rows of 64 bf16 (128 B) along K, 8-row atoms of 1024 B;
//     sbo = 1024 (next 8 rows), lbo unused (encoded 1).
//   MN-major operand: rows of 64 bf16 along M/N, one row per K index;
//     sbo = stride between 8-K-row groups, lbo = stride between 64-wide M/N
//     blocks.
// Bits: [0,14) start>>4, [16,30) lbo>>4, [32,46) sbo>>4, bit 46 = descriptor
// version 1, [61,64) layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// A descriptor advanced by `bytes` (a multiple of 16): the start-address field
// holds address >> 4 in its low bits, and shared-memory addresses stay far
// below the field's 256 KB range, so the advance is a plain add.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) {
  return desc + (uint64_t)(bytes >> 4);
}

// Instruction descriptor, kind::f16 with 16-bit A/B (fp16: format 0, bf16:
// format 1; A and B always of the same type) and fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn_major, bool b_mn_major,
                                                     bool bf16 = false) {
  return (1u << 4)                          // D format: f32
         | ((bf16 ? 1u : 0u) << 7)          // A format
         | ((bf16 ? 1u : 0u) << 10)         // B format
         | ((a_mn_major ? 1u : 0u) << 15)   // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ---- numerics -------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// Internal tensor-core operand type of the bf16 configuration: activations
// and weights enter and leave the library as bf16, but every intermediate
// that feeds a tensor-core MMA is held in fp16 (10-bit mantissa against
// bf16's 7), with fp32 accumulation.  Same tcgen05 rate, 8x smaller rounding
// steps inside the block.
typedef __half ct_t;

// Pack/unpack two values of a 16-bit storage type T (bf16 or fp16).
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  return pack_bf16(lo, hi);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  return pack_f16(lo, hi);
}
template <typename T> __device__ __forceinline__ float lo2(uint32_t v);
template <typename T> __device__ __forceinline__ float hi2(uint32_t v);
template <> __device__ __forceinline__ float lo2<__nv_bfloat16>(uint32_t v) { return bf16_lo(v); }
template <> __device__ __forceinline__ float hi2<__nv_bfloat16>(uint32_t v) { return bf16_hi(v); }
template <> __device__ __forceinline__ float lo2<__half>(uint32_t v) { return f16_lo(v); }
template <> __device__ __forceinline__ float hi2<__half>(uint32_t v) { return f16_hi(v); }

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + __expf(-z)); }

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Zigzag map.  Buffer row of global position p (chunk j = p / c):
//   j <  D : rank j,        slot 0  ->  j * 2c + (p % c)
//   j >= D : rank 2D-1-j,   slot 1  ->  (2D-1-j) * 2c + c + (p % c)
__host__ __device__ __forceinline__ int64_t zz_row_of_pos(int64_t p, int64_t c, int D) {
  int64_t j = p / c, off = p - j * c;
  return j < D ? j * 2 * c + off : (2 * D - 1 - j) * 2 * c + c + off;
}
// The same for sequences of at most INT32_MAX positions (every row index then
// fits 32 bits): a 32-bit division, for kernels that map a row per tile in
// warps sharing schedulers with a tensor-core issuing thread.
__device__ __forceinline__ int zz_row_of_pos32(int p, int c, int D) {
  const int j = p / c, off = p - j * c;
  return j < D ? j * 2 * c + off : (2 * D - 1 - j) * 2 * c + c + off;
}
// Global position held at buffer row b.
__host__ __device__ __forceinline__ int64_t zz_pos_of_row(int64_t b, int64_t c, int D) {
  int64_t r = b / (2 * c), rem = b - r * 2 * c;
  int64_t chunk = rem < c ? r : 2 * D - 1 - r;
  return chunk * c + (rem < c ? rem : rem - c);
}

}  // namespace tsp
