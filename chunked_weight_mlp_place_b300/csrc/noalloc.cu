// ipttt_make_targets_noalloc: the target builder (chunk-padded conv, then the
// projection GEMM) with its one piece of scratch -- the conv output C -- held
// in a fixed array compiled into this library instead of the library's pool.
//
// Some callers cannot call cudaMalloc while they run this step.  A process
// whose device memory is already handed out by another allocator (a
// framework's caching allocator that reserved most of the GPU up front) can
// see a fresh cudaMalloc fail, or throw off that allocator's accounting; a
// service with a latency budget cannot afford cudaMalloc or cudaFree, which
// may synchronise the whole device.  ipttt_make_targets grows its pool with
// cudaMalloc when a call needs more than it holds; this entry point never
// allocates or frees anything.
//
// The array costs IPTTT_NOALLOC_SCRATCH_BYTES of device memory on every GPU
// that loads the library, for as long as the process lives.  All calls share
// it: two calls that overlap on the GPU (different streams, no ordering
// between them) race on it.  Nothing in it needs to start at zero: the conv
// writes every byte the projection reads before the projection runs.
#include <cuda_runtime.h>

#include "checks.h"
#include "gemm.h"
#include "ipttt.h"
#include "launch.h"

namespace ipttt {

static_assert(IPTTT_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

// The conv output of ipttt_make_targets_noalloc.  In host code this name is a
// host-side stand-in, not a device address: the address kernels use comes
// from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[IPTTT_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array in the current device's context, looked up
// on every call (cheap once the module is loaded; the first call on a device
// loads it), so that no address outlives the context it belongs to.
ipttt_status scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return IPTTT_ERR_CUDA;
  }
  *out = p;
  return IPTTT_OK;
}

}  // namespace
}  // namespace ipttt

using namespace ipttt;

extern "C" ipttt_status ipttt_make_targets_noalloc(const void* E, const float* conv_w, const void* P, void* V,
                                                   int64_t L, int64_t B, const ipttt_dims* dims,
                                                   ipttt_stream stream) {
  reset_launch_count();
  // the same checks, in the same order, as ipttt_make_targets
  ipttt_status st = check_dims(dims, true);
  if (st != IPTTT_OK) return st;
  if ((st = check_chunking(dims, L, B)) != IPTTT_OK) return st;
  const int64_t rows = dims->batch * L;
  if (rows == 0) return IPTTT_OK;
  const bool bf16 = dims->dtype == IPTTT_BF16;
  // The conv output must fit the fixed array: rows * d elements of the act type.
  const int64_t esz = bf16 ? 2 : 4;
  if (rows > static_cast<int64_t>(IPTTT_NOALLOC_SCRATCH_BYTES) / (dims->d * esz)) return IPTTT_ERR_INVALID_ARG;
  if ((st = check_ptrs({E, static_cast<const void*>(conv_w), P, static_cast<const void*>(V)})) != IPTTT_OK)
    return st;
  void* C = nullptr;
  if ((st = scratch_address(&C)) != IPTTT_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_conv(E, conv_w, C, rows, L, B, dims->d, bf16, s);
  if (e == cudaSuccess) {
    GemmProblem p;
    p.M = rows;
    p.N = dims->d;
    p.K = dims->d;
    p.A.ptr = C;
    p.A.rows = rows;
    p.A.cols = dims->d;
    p.A.ld = dims->d;
    p.B.ptr = P;
    p.B.rows = dims->d;
    p.B.cols = dims->d;
    p.B.ld = dims->d;
    p.B.mn_major = 1;
    p.epi = EPI_STORE;
    p.kind = K_PROJ;
    p.out_bf16 = bf16;
    p.D.ptr = V;
    p.D.ld = dims->d;
    e = bf16 ? launch_gemm_tc(p, s) : launch_gemm_simt(p, s);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return (e == cudaErrorInvalidValue) ? IPTTT_ERR_INVALID_ARG : IPTTT_ERR_LAUNCH;
  }
  return IPTTT_OK;
}
