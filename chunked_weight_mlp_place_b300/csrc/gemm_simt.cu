// fp32 back end of the batched GEMM (IPTTT_FP32 mode): CUDA-core FMA with a
// 64x64 shared-memory tile.  It exists for exact-arithmetic runs (every
// product and sum in fp32) and takes any sizes; throughput is not its job.
#include "common.cuh"
#include "gemm.h"
#include "launch.h"

namespace ipttt {
namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16, kThreads = 256;


// Load a kBK x 64 slice of operand `o` (rows i0.., K range k0..) into s[k][i].
__device__ __forceinline__ void load_tile(const Operand& o, int b1, int b2, int64_t i0, int64_t ext_i, int64_t k0,
                                          int64_t K, float (*s)[kBM + 4]) {
  const float* base = static_cast<const float*>(o.ptr);
  const int64_t r0 = entry_row(o, b1, b2);
#pragma unroll
  for (int it = 0; it < (kBK * kBM) / kThreads; ++it) {
    const int idx = threadIdx.x + it * kThreads;
    int i, k;
    if (o.mn_major) {
      i = idx % kBM;
      k = idx / kBM;
    } else {
      k = idx % kBK;
      i = idx / kBK;
    }
    const int64_t gi = i0 + i, gk = k0 + k;
    float v = 0.0f;
    if (gi < ext_i && gk < K) {
      v = o.mn_major ? base[(r0 + gk) * o.ld + gi] : base[(r0 + gi) * o.ld + gk];
    }
    s[k][i] = v;
  }
}

template <bool kGate>
__global__ void __launch_bounds__(kThreads) simt_gemm_kernel(const GemmProblem p) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  __shared__ float B2s[kGate ? kBK : 1][kBN + 4];
  const int b1 = blockIdx.z % p.nb1, b2 = blockIdx.z / p.nb1;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM, n0 = static_cast<int64_t>(blockIdx.x) * kBN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {}, acc2[4][4] = {};
  for (int64_t k0 = 0; k0 < p.K; k0 += kBK) {
    load_tile(p.A, b1, b2, m0, p.M, k0, p.K, As);
    load_tile(p.B, b1, b2, n0, p.N, k0, p.K, Bs);
    if constexpr (kGate) load_tile(p.B2, b1, b2, n0, p.N, k0, p.K, B2s);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      float a[4], b[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[k][ty * 4 + i];
        b[i] = Bs[k][tx * 4 + i];
        if constexpr (kGate) c[i] = B2s[k][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if constexpr (kGate) acc2[i][j] = fmaf(a[i], c[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
  const int64_t drow0 = entry_row(p.D, b1, b2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      float* d = static_cast<float*>(p.D.ptr) + (drow0 + m) * p.D.ld + n;
      const float v = acc[i][j];
      switch (p.epi) {
        case EPI_STORE:
          *d = (p.causal && n >= (m / p.causal) * p.causal) ? 0.0f : p.alpha * v;
          break;
        case EPI_GATE:
          *d = silu_f(v) * acc2[i][j];
          break;
        case EPI_ACCUM:
          atomicAdd(d, v);
          break;
        case EPI_AXPY: {
          const int64_t srow = entry_row(p.src, b1, b2) + m;
          const float w = static_cast<const float*>(p.src.ptr)[srow * p.src.ld + n] + p.alpha * v;
          *d = w;
          break;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmProblem& p, cudaStream_t stream) {
  if (p.M <= 0 || p.N <= 0 || p.nb1 <= 0 || p.nb2 <= 0) return cudaSuccess;
  if (p.out_bf16) return cudaErrorInvalidValue;  // fp32 mode writes fp32 activations
  if (p.add.ptr || p.dyn_tiles) return cudaErrorNotSupported;  // tensor-core features
  const int64_t gx = (p.N + kBN - 1) / kBN, gy = (p.M + kBM - 1) / kBM, gz = static_cast<int64_t>(p.nb1) * p.nb2;
  if (gy > 65535 || gz > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(gz));
  LaunchMark mark(p.kind, stream);
  if (p.epi == EPI_GATE)
    simt_gemm_kernel<true><<<grid, kThreads, 0, stream>>>(p);
  else
    simt_gemm_kernel<false><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ipttt
