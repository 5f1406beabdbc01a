// Description of one batched GEMM launch with a fused epilogue, shared by the
// tensor-core (bf16) and CUDA-core (fp32) back ends.
//
//   for every batch entry b = (b1, b2), b1 < nb1, b2 < nb2:
//     acc[m][n] = sum_k A_b[m][k] * B_b[k][n]          (m < M, n < N, k < K)
//     epilogue(acc) -> outputs of batch entry b
//
// An operand is a window of a row-major matrix in global memory.  Its rows are
// offset per batch entry: row = y0 + b1*ys1 + b2*ys2 + i, or, where a table
// of entry starts is given (packed documents), row = y0 + ytab[b1] + b2*ys2 + i.  For a K-major
// operand, i is the M (or N) index and the K index runs along the columns; for
// an MN-major operand, i is the K index and M (or N) runs along the columns.
#pragma once

#include <stdint.h>

namespace ipttt {

// L2 eviction priority of the lines an access touches.
enum L2Hint : int { L2_NORMAL = 0, L2_EVICT_FIRST = 1, L2_EVICT_LAST = 2 };

enum EpiKind : int {
  EPI_STORE = 0,  // D = alpha * acc (+ add), block-causal mask if set   (D in the act dtype or fp32)
  EPI_GATE = 1,   // D = SiLU(acc_g) * acc_u, acc_u from B2   (D in the act dtype)
  EPI_ACCUM = 2,  // D += acc, fp32 reductions in L2          (D fp32; partial sums)
  EPI_AXPY = 3,   // D = src + alpha * acc, fp32 (CUDA cores) or split hi/lo planes (tensor cores)
};

struct Operand {
  const void* ptr = nullptr;
  int64_t rows = 0, cols = 0, ld = 0;  // matrix extent and row stride (elements)
  int mn_major = 0;                    // 1: K runs along rows
  int64_t y0 = 0, ys1 = 0, ys2 = 0;    // per-batch row offsets
  const int64_t* ytab = nullptr;       // device table replacing b1*ys1 (null: none)
};

struct OutRef {
  void* ptr = nullptr;
  int64_t ld = 0;
  int64_t y0 = 0, ys1 = 0, ys2 = 0;  // row = y0 + b1*ys1 + b2*ys2 + m, column n
  int64_t rows = 0;                  // rows of the whole matrix (needed where TMA reads or writes it)
  const int64_t* ytab = nullptr;     // device table replacing b1*ys1 (null: none)
};

// First row of batch entry (b1, b2) of an operand or output.
template <typename R>
__host__ __device__ __forceinline__ int64_t entry_row(const R& o, int b1, int b2) {
  return o.y0 + (o.ytab ? o.ytab[b1] : b1 * o.ys1) + b2 * o.ys2;
}

// The planes are stored tile-major: blocks of kPlaneRows rows x kPlaneCols
// columns, each block 4 KB contiguous (row r of a block at r * 32 bytes), the
// blocks of one row of blocks side by side, rows of blocks one after another,
// sequences (or groups) one after another; the matrix is padded with zeros to
// whole blocks.  Inside a row the two 8-column halves trade places where bit 2
// of r is set: the 32-byte swizzle of a shared-memory operand tile, so any 64
// rows of a block starting at a multiple of 8 are 2 KB that TMA copies as they
// are (rows of 512 bytes) into the MN-major 32-byte-swizzle operand layout.  A
// warp finishing 32 rows of one 16-column chunk reads and writes 1 KB contiguous.
constexpr int kPlaneRows = 128, kPlaneCols = 16, kPlaneBlock = kPlaneRows * kPlaneCols;
__host__ __device__ __forceinline__ int64_t plane_index(int64_t rb_row, int64_t cb, int64_t nblk_cols, int r, int c) {
  return (rb_row * nblk_cols + cb) * kPlaneBlock + r * kPlaneCols + (c ^ (((r >> 2) & 1) << 3));
}

// A fast weight (one d_ff x d matrix per entry) as tile-major split planes.
// Entry e = b1*es1 + b2*es2 owns row blocks e*rb .. e*rb + rb - 1.
struct Planes {
  uint16_t* hi = nullptr;
  uint16_t* lo = nullptr;
  int64_t rb = 0;   // 128-row blocks per entry
  int64_t cb = 0;   // 16-column blocks per row of blocks
  int64_t es1 = 0, es2 = 0;
  int64_t entries = 0;
};

struct GemmProblem {
  int64_t M = 0, N = 0, K = 0;
  int nb1 = 1, nb2 = 1;
  Operand A, B, B2;
  int epi = EPI_STORE;
  int out_bf16 = 0;  // element type of D for STORE / GATE
  OutRef D;          // primary output (CUDA-core AXPY: fp32 W)
  OutRef src;        // CUDA-core AXPY: fp32 source (may equal D)
  OutRef add;        // tensor-core STORE: a matrix of D's type and rows added to alpha * acc (null: none)
  // Tensor-core AXPY: the fast weight's tile-major hi/lo planes (split_w, plane_index in
  // common.cuh), read and rewritten in place.  Tensor-core ACCUM with b_planes: its B
  // operand is w.hi.
  Planes w;
  int b_planes = 0;
  float alpha = 1.0f;
  // STORE: chunk size of a block-causal mask (0: none).  Element (m, n) of a batch entry
  // is kept where n lies in an earlier chunk than m (n < (m / causal) * causal), else 0;
  // on the tensor cores, tiles with no kept element are skipped (their output stays as it was).
  int64_t causal = 0;
  int split_k = 0;   // tensor-core path: 1 = balance (tile, k-block) work over CTAs (needs EPI_ACCUM)
  int kind = 0;      // KernelKind label (launch counting / timing)
  // Tensor-core path, L2 eviction priority (L2Hint in common.cuh) of the lines the A and B
  // operand copies read, and, for the AXPY epilogue, planes_l2 = 1: the hi plane's lines
  // kept (evict last) and the lo plane's given up first -- the hi plane is read again by
  // the next apply, the lo plane only by the next update.
  int l2_a = 0, l2_b = 0, planes_l2 = 0;
  int l2_d = 0;  // STORE / GATE epilogues: L2 eviction priority of the output's bf16 stores
  // Tensor-core path, tile order (no split): 0 = groups of 16 row tiles, each swept over all
  // column tiles (B re-read once per group); band_n > 0 = bands of band_n column tiles, each
  // swept over all row tiles (A re-read once per band, the band of B held in L2).
  int band_n = 0;
  // Tensor-core path, whole tiles with a STORE (no mask) or GATE epilogue: 1 = tiles taken in
  // increasing order from a device-wide counter as CTA pairs free up, instead of a fixed
  // share per pair.  The counter is one per device: launches that use it must be ordered.
  int dyn_tiles = 0;
  // Tensor-core path, whole tiles: A triangular (M = K), its zeros skipped.  1: lower (A[m][k] = 0
  // for k > m), a tile's contraction stops after its last row; -1: upper (A[m][k] = 0 for k < m),
  // it starts at the k-block of its first row.
  int tri = 0;
  // Tensor-core path: once a CTA has issued all its operand copies it asks L2 to fetch
  // its share of pf_count ranges of pf_bytes bytes, pf_stride bytes apart, from pf_ptr
  // (the next kernel's operand; 16-byte aligned).  No result depends on it.
  const void* pf_ptr = nullptr;
  int64_t pf_bytes = 0, pf_stride = 0;
  int pf_count = 0;
};

// The MSE chunk loop of every sequence as one persistent kernel (engine_tc.cuh):
//   for k: O_k = Z_k W_k; R_k = O_k - V_k; W_{k+1} = W_k + alpha Z_k^T R_k
// split into work items per 256-column block n of W (the rule is independent across columns):
// apply items (a 256-token tile of O_k[:, n], one of `parts` slices of d_ff), whose fp32 sums
// meet in `acc` and the last of which forms O_k and R_k of that tile, and update items (256
// rows x the 256 columns of W).  Items start as soon as what they read is written.  CTA pairs
// take items in order from a device-wide counter: launches that use it must be ordered.
struct EngineMse {
  const void* Z = nullptr;       // [batch*L, d_ff] bf16, sequence s in rows s*L ..
  const void* V = nullptr;       // [batch*L, d] bf16
  void* O = nullptr;             // [batch*L, d] bf16 (out)
  float* acc = nullptr;          // [batch*B, d] fp32 scratch, zero on entry and left zero
  void* R = nullptr;             // bf16 R_k: row s*r_seq + k*r_chunk + i of sequence s, chunk k, token i
  int64_t r_seq = 0, r_chunk = 0;  // (B, 0): a [batch*B, d] scratch reused by every chunk
  const void* Zu = nullptr;      // the update's contraction operand in Z's layout (null: Z itself)
  uint32_t* counters = nullptr;  // engine_counter_words() words, zero on entry
  Planes w;                      // the fast weights (entry = sequence), read and rewritten in place
  int64_t batch = 0, L = 0, B = 0, d = 0, d_ff = 0;
  int parts = 0;                 // slices of d_ff per apply tile
  float alpha = 0.0f;            // -eta / B
  int keep_hi = 0;               // keep the hi planes in L2 (evict last)
  // Packed documents (sequence s = document s, longest first; L = the longest's chunks x B):
  // starts[s] = its first row of Z, V and O, lens[s] its tokens (its last chunk may be short: R is
  // zero past its end and scaled by B/n, O written only inside it), active[k] = the documents with
  // a chunk k (a prefix), icum[k] = the items of the chunks before k (device tables, icum[K] =
  // all); rows = the rows of Z, V and O.  Null: sequence s in rows s*L .. s*L+L-1.
  const int64_t* starts = nullptr;
  const int64_t* lens = nullptr;
  const int64_t* active = nullptr;
  const int64_t* icum = nullptr;
  int64_t icum_total = 0;  // icum[K], known on the host
  int64_t rows = 0;
};

}  // namespace ipttt
