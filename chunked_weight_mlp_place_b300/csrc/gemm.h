// Description of one batched GEMM launch with a fused epilogue, shared by the
// tensor-core (bf16) and CUDA-core (fp32) back ends.
//
//   for every batch entry b = (b1, b2), b1 < nb1, b2 < nb2:
//     acc[m][n] = sum_k A_b[m][k] * B_b[k][n]          (m < M, n < N, k < K)
//     epilogue(acc) -> outputs of batch entry b
//
// An operand is a window of a row-major matrix in global memory.  Its rows are
// offset per batch entry: row = y0 + b1*ys1 + b2*ys2 + i.  For a K-major
// operand, i is the M (or N) index and the K index runs along the columns; for
// an MN-major operand, i is the K index and M (or N) runs along the columns.
#pragma once

#include <stdint.h>

namespace ipttt {

enum EpiKind : int {
  EPI_STORE = 0,  // D = acc                                  (D in the act dtype)
  EPI_GATE = 1,   // D = SiLU(acc_g) * acc_u, acc_u from B2   (D in the act dtype)
  EPI_ACCUM = 2,  // D += acc, fp32 reductions in L2          (D fp32; partial sums)
  EPI_AXPY = 3,   // D = src + alpha * acc, fp32 (CUDA cores) or split hi/lo planes (tensor cores)
};

struct Operand {
  const void* ptr = nullptr;
  int64_t rows = 0, cols = 0, ld = 0;  // matrix extent and row stride (elements)
  int mn_major = 0;                    // 1: K runs along rows
  int64_t y0 = 0, ys1 = 0, ys2 = 0;    // per-batch row offsets
};

struct OutRef {
  void* ptr = nullptr;
  int64_t ld = 0;
  int64_t y0 = 0, ys1 = 0, ys2 = 0;  // row = y0 + b1*ys1 + b2*ys2 + m, column n
  int64_t rows = 0;                  // rows of the whole matrix (needed where TMA reads or writes it)
};

struct GemmProblem {
  int64_t M = 0, N = 0, K = 0;
  int nb1 = 1, nb2 = 1;
  Operand A, B, B2;
  int epi = EPI_STORE;
  int out_bf16 = 0;  // element type of D for STORE / GATE
  OutRef D;          // primary output (AXPY on the tensor cores: the hi plane)
  OutRef src;        // AXPY: source (may equal D); fp32, or the hi plane on the tensor cores
  OutRef D_lo;       // AXPY on the tensor cores: lo planes of D and src (16-bit, same layout
  OutRef src_lo;     //   as the hi planes; see split_w in common.cuh)
  float alpha = 1.0f;
  int split_k = 0;   // tensor-core path: 1 = balance (tile, k-block) work over CTAs (needs EPI_ACCUM)
  int kind = 0;      // KernelKind label (launch counting / timing)
};

}  // namespace ipttt
