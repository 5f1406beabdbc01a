// Host-side entry points of the kernel files, used by the C-ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.h"

namespace ipttt {

// Kernel kinds, for launch counting and the optional per-kernel event timing.
enum KernelKind : int {
  K_GATE = 0,      // gated up-projection GEMM
  K_CONV = 1,      // chunk-padded depthwise conv
  K_PROJ = 2,      // target projection GEMM
  K_APPLY = 3,     // O_k = Z_k W_k
  K_RESIDUAL = 4,  // O_k, R_k = O_k - V_k from the apply's fp32 sums
  K_UPDATE = 5,    // W_{k+1} = W_k + alpha Z_k^T R_k
  K_GROUP_SUM = 6, // additive scan: per-group Z^T V
  K_SCAN = 7,      // additive scan: exclusive prefix over groups
  K_WEIGHT = 8,    // fast-weight conversions (W_o0 -> split planes -> W_final, W_o0 -> W_final)
  K_SCORES = 9,    // additive rule, block-causal form: (eta/B) mask(Z Z^T)
  K_ENGINE = 10,   // MSE rule: the whole chunk loop in one persistent kernel
  K_WINDOW = 11,   // MSE rule in windows of chunks: Gram, inverse, transformed-Z and output GEMMs
  K_COUNT = 12
};

// Every kernel launch of the library sits inside one LaunchMark: it counts the
// launch and, while kernel timing is on, brackets it with CUDA events on `stream`.
struct LaunchMark {
  LaunchMark(int kind, cudaStream_t stream);
  ~LaunchMark();
  int kind;
  cudaStream_t stream;
  int slot;
};
// Launch `kern` so that it may start while the previous kernel of `stream` is
// still finishing (programmatic dependent launch; the kernel calls pdl_wait()
// before its first global-memory access).  cluster > 1: clusters of that many
// CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

int current_device();     // cudaGetDevice, -1 on error
void reset_launch_count(); // start counting the launches of a new C-ABI call
int device_sm_count();    // SMs of the current device (cached)

// Read the device error word of the current device (0 = no capped wait ran out) and clear it.
cudaError_t read_clear_device_error(int* code);
// Soft limit of the tensor-core kernels' pipeline waits on the current device (0: the hard limit).
cudaError_t set_wait_soft_limit(uint64_t ns);

cudaError_t launch_gemm_tc(const GemmProblem& p, cudaStream_t stream);    // bf16 operands, tcgen05
// The persistent MSE chunk engine (gemm.h EngineMse).  Shapes it takes: B, d and d_ff multiples
// of 256, parts in 1 .. d_ff / 256; cudaErrorNotSupported otherwise (nothing queued).
bool engine_mse_supported(int64_t B, int64_t d, int64_t d_ff);
int64_t engine_counter_words(int64_t batch, int64_t L, int64_t B, int64_t d, int parts);
cudaError_t launch_engine_mse(const EngineMse& a, cudaStream_t stream);
cudaError_t launch_gemm_simt(const GemmProblem& p, cudaStream_t stream);  // fp32 operands, CUDA cores

// C = chunk-padded depthwise conv of E (width 4, taps t..t+3), rows = batch*L.
// Several layers at once: rows = n_layers * e_rows, output row r is E row
// r % e_rows under the taps conv_w[r / e_rows] (conv_w: n_layers x d x 4);
// e_rows <= 0 means one layer (e_rows = rows).
cudaError_t launch_conv(const void* E, const float* conv_w, void* C, int64_t rows, int64_t L, int64_t B, int64_t d,
                        bool bf16, cudaStream_t stream, int64_t e_rows = 0);
// The same over packed documents: document i holds rows cu[i] .. cu[i+1]-1
// (cu: n_docs+1 device int64, rising from 0 to rows); chunks of B tokens are
// counted from each document's first row and the last one ends with it.
cudaError_t launch_conv_varlen(const void* E, const float* conv_w, void* C, int64_t rows, const int64_t* cu,
                               int64_t n_docs, int64_t B, int64_t d, bool bf16, cudaStream_t stream);

// Per batch entry e = b1 + nb1*b2 and chunk row i < B:
//   O[orow] = act(acc[e*B+i]);  R[e*B+i] = act(acc[e*B+i] - V[orow])  (if R);  acc[e*B+i] = 0
// with orow = o_y0 + b1*o_ys1 + b2*o_ys2 + i (otab[b1] in place of b1*o_ys1 where given).
// Packed documents (lens given): the chunk holds n = min(B, lens[b1] - o_y0)
// tokens of entry b1's document; rows i >= n lie past its end (O and V are not
// touched there, R = 0) and R is scaled by B/n, so a step of eta/B is the
// chunk's mean.  r_from_v: R = V instead of O - V (the additive rule's step).
struct ResidualArgs {
  float* acc = nullptr;
  const void* V = nullptr;
  void* O = nullptr;
  void* R = nullptr;
  int64_t B = 0, d = 0;
  int nb1 = 1, nb2 = 1;
  int64_t o_y0 = 0, o_ys1 = 0, o_ys2 = 0;
  const int64_t* otab = nullptr;
  const int64_t* lens = nullptr;
  int r_from_v = 0;
};
cudaError_t launch_residual(const ResidualArgs& a, bool bf16, cudaStream_t stream);

// The fp32 fast weight as tile-major split planes (split_w / plane_index in
// common.cuh; Planes in gemm.h), R x C per entry, C a multiple of 8:
//   split: the planes of every entry e = split(W0[e or 0]) (w0_stride elements apart, 0 = shared);
//   merge: W (entries x R x C fp32) = join(planes).
cudaError_t launch_split_planes(const float* W0, int64_t w0_stride, const Planes& w, int64_t R, int64_t C,
                                cudaStream_t stream);
cudaError_t launch_merge_planes(const Planes& w, float* W, int64_t R, int64_t C, cudaStream_t stream);
// dst[e*dst_stride + i] = act(src[e*src_stride + i]) (act = bf16 or fp32) for e < entries, i < n.
cudaError_t launch_to_act(const float* src, int64_t src_stride, void* dst, int64_t dst_stride, int64_t entries,
                          int64_t n, bool bf16, cudaStream_t stream);
// X (entries x n x n bf16, n a multiple of 8) = identity matrices.
cudaError_t launch_eye_bf16(void* X, int64_t n, int64_t entries, cudaStream_t stream);
// W[i] += alpha * S[i] for i < n (fp32).
cudaError_t launch_axpy(float* W, const float* S, float alpha, int64_t n, cudaStream_t stream);
// W[s] = W0[s or 0] (fp32 copy) for s < batch.
cudaError_t launch_copy_w(const float* W0, int64_t w0_stride, float* W, int64_t batch, int64_t n,
                          cudaStream_t stream);

// Exclusive scan over G fp32 group sums D[g], element-wise over batch*n:
//   S = W0; for g: t = D[g]; D[g] = S; S += alpha*t;  W_final = S        (fp32 mode, in place)
cudaError_t launch_group_scan(float* D, const float* W0, int64_t w0_stride, float* W_final, int64_t G,
                              int64_t batch, int64_t n, float alpha, cudaStream_t stream);
// The same scan writing each group's starting weight as the planes of entry g*batch + b.
cudaError_t launch_group_scan_planes(const float* D, const Planes& w, const float* W0, int64_t w0_stride,
                                     float* W_final, int64_t G, int64_t batch, int64_t R, int64_t C, float alpha,
                                     cudaStream_t stream);

}  // namespace ipttt
