// gemm_tc.h -- host interface of the tcgen05 GEMM (gemm_tc.cu).
#pragma once
#include <stdint.h>

#include "tsp.h"

namespace tsp {

enum { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 2 };
enum { EPI_STORE = 0, EPI_RES = 1, EPI_F32 = 2, EPI_SWIGLU = 3, EPI_SWIGLU_BWD = 4 };

// C[M, N] = sum over K of A(m, k) * B(n, k), fp16 operands, fp32 accumulation.
//   A K-major: stored [M, K] (row stride lda);  A MN-major: stored [K, M].
//   B K-major: stored [N, K] (nn.Linear weight); B MN-major: stored [K, N].
// K may be split into up to 3 segments, each with its own A and B pointer
// (all but the last a multiple of 64 long).  Alternatively (nseg_n > 0) the
// N range is split into segments of nseg_n columns with B pointer B[n / nseg_n]
// (and one K segment).  paired: SwiGLU tile, B[0] = W_1 and B[1] = W_3, both
// [N, K]; the output is G [M, N] = silu(A W_1^T) * (A W_3^T).
// rot_D > 0: row tile of virtual rank r = rot_r0 + m0 / rot_rows walks the K
// shards (boundaries floor(s*K/rot_D), k-block granularity) in ring order
// (r - t) mod rot_D (rot_r0: the rank of row 0, for a GEMM over a row tile).
// Epilogues (out/out2/out3 row strides ldo/ldo2/ldo3, elements):
//   EPI_STORE      out = C stored as out_type (OUT_F16 / OUT_BF16 / OUT_F32); with
//                  n_split > 0 (a multiple of 256) columns n >= n_split go to
//                  out2 at column n - n_split instead
//   EPI_RES        out = C + res, res bf16 or fp32 (res_f32), stored as out_type
//   EPI_F32        out = C (fp32); with m_seg > 0 rows go to outs[m / m_seg]
//   EPI_SWIGLU     out = f16(silu(C_1) * C_3); out2/out3 (nullable) = f16(C_1), f16(C_3)
//   EPI_SWIGLU_BWD C = dG; e1 = A, e2 = B (fp16, stride lde):
//                  out = f16(dG * B * s(A) (1 + A (1 - s(A)))), out2 = f16(dG * silu(A))
struct TcGemm {
  const char* name = "gemm_tc";  // label for launch accounting
  int M = 0, N = 0, K = 0;
  bool a_mn = false, b_mn = false;
  int nks = 1;
  const void* A[3] = {nullptr, nullptr, nullptr};
  int64_t lda[3] = {0, 0, 0};
  const void* B[3] = {nullptr, nullptr, nullptr};
  int64_t ldb[3] = {0, 0, 0};
  int kseg_len[3] = {0, 0, 0};
  int nseg_n = 0;
  bool paired = false;
  int rot_rows = 0, rot_D = 0, rot_r0 = 0;
  int epi = EPI_STORE;
  void* out = nullptr;
  int64_t ldo = 0;
  void* out2 = nullptr;
  int64_t ldo2 = 0;
  void* out3 = nullptr;
  int64_t ldo3 = 0;
  const void* res = nullptr;
  int64_t ldr = 0;
  bool res_f32 = false;
  int out_type = OUT_F16;
  const void* e1 = nullptr;
  const void* e2 = nullptr;
  int64_t lde = 0;
  int64_t m_seg = 0;
  void* outs[3] = {nullptr, nullptr, nullptr};
  int n_split = 0;
};

tsp_status gemm_tc(const TcGemm& g, cudaStream_t st);

}  // namespace tsp
