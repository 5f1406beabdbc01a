// C-ABI of libipttt: argument checks, the per-device scratch pool, and the
// order of kernel launches that makes up the In-Place TTT fast-weight layer.
//
// Layer (In-Place TTT write-ups: gated MLP itsolotime §2.1, target §2.3,
// chunk-wise apply-then-update §2.2 / Fig. 1, su666666 "third axe"):
//   Z = SiLU(X W_g) * (X W_u)                          one GEMM, gate epilogue
//   V = Conv(E) P                                      conv kernel + GEMM
//   MSE rule, for k = 0 .. K-1 (sequential):
//     apply     O_acc = Z_k W_k          (bf16 hi plane of W, split over d_ff, fp32 reductions)
//     residual  O_k = O_acc; R_k = O_acc - V_k; O_acc = 0
//     update    W_{k+1} = W_k - (eta/B) Z_k^T R_k   (on the hi/lo planes of W)
//   additive rule, chunk-parallel scan over G groups of g chunks (G*g = K):
//     group sums   S_j = Z_{group j}^T V_{group j}           (all groups at once)
//     scan         W^(j) = W_0 + (eta/B) sum_{i<j} S_i; W_final = W^(G)
//     within every group at once, for its g chunks:
//       apply O_k = Z_k W; update W += (eta/B) Z_k^T V_k (not after the last)
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "ipttt.h"
#include "checks.h"
#include "gemm.h"
#include "launch.h"

namespace ipttt {

namespace {
thread_local int64_t t_launches = 0;

// Optional per-kernel timing: CUDA events recorded around every launch while
// enabled, reduced to per-kind totals when read.
struct TimingRec {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimingRec> g_timing_pending;
std::vector<cudaEvent_t> g_event_pool;
int64_t g_timing_launches[K_COUNT] = {0};
double g_timing_ms[K_COUNT] = {0};

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Fold every pending record into the totals (waits for its events).
void drain_timing_locked() {
  for (const TimingRec& r : g_timing_pending) {
    float ms = 0.0f;
    if (r.start && r.stop && cudaEventSynchronize(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      g_timing_launches[r.kind] += 1;
      g_timing_ms[r.kind] += ms;
    }
    cudaGetLastError();
    if (r.start) g_event_pool.push_back(r.start);
    if (r.stop) g_event_pool.push_back(r.stop);
  }
  g_timing_pending.clear();
}
}  // namespace

void reset_launch_count() { t_launches = 0; }

const char* kind_name(int k) {
  static const char* names[K_COUNT] = {"gate_up", "conv",  "proj",        "apply",  "residual", "update",
                                       "group_sum", "scan", "weight_copy", "scores", "engine", "window"};
  return (k >= 0 && k < K_COUNT) ? names[k] : "unknown";
}

// Every launch also sits in an NVTX range named after its kind (a no-op unless a
// profiler is attached), so traces show which step of the layer queued it.
LaunchMark::LaunchMark(int k, cudaStream_t s) : kind(k), stream(s), slot(-1) {
  ++t_launches;
  nvtxRangePushA(kind_name(k));
  std::lock_guard<std::mutex> g(g_timing_mu);
  if (!g_timing_on || k < 0 || k >= K_COUNT) return;
  TimingRec r{k, take_event(), take_event()};
  if (r.start) cudaEventRecord(r.start, s);
  g_timing_pending.push_back(r);
  slot = static_cast<int>(g_timing_pending.size()) - 1;
}

LaunchMark::~LaunchMark() {
  nvtxRangePop();
  if (slot < 0) return;
  std::lock_guard<std::mutex> g(g_timing_mu);
  if (slot < static_cast<int>(g_timing_pending.size()) && g_timing_pending[slot].stop)
    cudaEventRecord(g_timing_pending[slot].stop, stream);
  // keep memory bounded on long runs
  if (g_timing_pending.size() > 65536) drain_timing_locked();
}

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

int device_sm_count() {
  static int cache[64] = {0};
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

// ------------------------------------------------------------------- pool
struct Pool {
  void* ptr = nullptr;
  size_t size = 0;
};
std::mutex g_pool_mu;
Pool g_pools[64];

std::atomic<size_t> g_pool_limit{0};  // 0: no limit

ipttt_status pool_reserve(size_t bytes, void** out) {
  const size_t limit = g_pool_limit.load();
  if (limit && bytes > limit) return IPTTT_ERR_ALLOC;  // refused before anything is queued
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return IPTTT_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_pool_mu);
  Pool& p = g_pools[dev];
  if (bytes > p.size) {
    if (p.ptr) {
      // The old block may still be read by queued kernels of earlier calls.
      if (cudaDeviceSynchronize() != cudaSuccess) return IPTTT_ERR_CUDA;
      cudaFree(p.ptr);
      p.ptr = nullptr;
      p.size = 0;
    }
    const size_t want = (bytes + (64u << 20) - 1) & ~static_cast<size_t>((64u << 20) - 1);
    if (cudaMalloc(&p.ptr, want) != cudaSuccess) {
      cudaGetLastError();
      p.ptr = nullptr;
      return IPTTT_ERR_ALLOC;
    }
    p.size = want;
  }
  *out = p.ptr;
  return IPTTT_OK;
}

// Bump allocator over one pool block (256-byte aligned pieces).
struct Carve {
  size_t off = 0;
  template <typename T>
  size_t take(int64_t count) {
    const size_t at = off;
    off += (static_cast<size_t>(count) * sizeof(T) + 255) & ~static_cast<size_t>(255);
    return at;
  }
};

// ------------------------------------------------------------- checks
ipttt_status from_cuda(cudaError_t e) {
  switch (e) {
    case cudaSuccess:
      return IPTTT_OK;
    case cudaErrorMemoryAllocation:
      return IPTTT_ERR_ALLOC;
    case cudaErrorInvalidValue:
    case cudaErrorInvalidConfiguration:
      return IPTTT_ERR_INVALID_ARG;
    case cudaErrorNoKernelImageForDevice:
    case cudaErrorInvalidDevice:
    case cudaErrorNoDevice:
    case cudaErrorInsufficientDriver:
    case cudaErrorNotSupported:
      return IPTTT_ERR_UNSUPPORTED;
    case cudaErrorLaunchFailure:
    case cudaErrorLaunchOutOfResources:
    case cudaErrorInvalidDeviceFunction:
      return IPTTT_ERR_LAUNCH;
    default:
      return IPTTT_ERR_CUDA;
  }
}

#define IPTTT_TRY(expr)                        \
  do {                                         \
    const ipttt_status _s = (expr);            \
    if (_s != IPTTT_OK) return _s;             \
  } while (0)
#define IPTTT_CUDA(expr)                       \
  do {                                         \
    const cudaError_t _e = (expr);             \
    if (_e != cudaSuccess) {                   \
      cudaGetLastError();                      \
      return from_cuda(_e);                    \
    }                                          \
  } while (0)

}  // namespace

// ------------------------------------------------------------- checks
// (declared in checks.h: every entry point, the allocation-free one included, validates
// its arguments through these, so the same bad argument gives the same status everywhere)
namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pointer must be non-null, 16-byte aligned and reachable from the device.
ipttt_status check_ptr_host(const void* p) {
  if (!p || !aligned16(p)) return IPTTT_ERR_INVALID_ARG;
  return IPTTT_OK;
}
ipttt_status check_ptr_device(const void* p) {
  cudaPointerAttributes a;
  const cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return IPTTT_ERR_INVALID_ARG;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return IPTTT_ERR_INVALID_ARG;
  return IPTTT_OK;
}
}  // namespace

ipttt_status check_dims(const ipttt_dims* dims, bool need_batch) {
  if (!dims) return IPTTT_ERR_INVALID_ARG;
  if (dims->dtype != IPTTT_FP32 && dims->dtype != IPTTT_BF16) return IPTTT_ERR_INVALID_ARG;
  if (dims->d < 1 || dims->d_ff < 1) return IPTTT_ERR_INVALID_ARG;
  if (need_batch && dims->batch < 0) return IPTTT_ERR_INVALID_ARG;
  if (dims->w0_per_seq != 0 && dims->w0_per_seq != 1) return IPTTT_ERR_INVALID_ARG;
  if (dims->d > (1 << 20) || dims->d_ff > (1 << 20)) return IPTTT_ERR_INVALID_ARG;
  if (dims->dtype == IPTTT_BF16 && (dims->d % 8 || dims->d_ff % 8)) return IPTTT_ERR_INVALID_ARG;
  return IPTTT_OK;
}

ipttt_status check_chunking(const ipttt_dims* dims, int64_t L, int64_t B) {
  if (L < 0 || B < 1 || L % B) return IPTTT_ERR_INVALID_ARG;
  if (dims->dtype == IPTTT_BF16 && B % 16) return IPTTT_ERR_INVALID_ARG;
  // token rows and fast-weight rows are TMA coordinates (int32)
  if (dims->batch > 0 && L > (int64_t{1} << 31) / dims->batch) return IPTTT_ERR_INVALID_ARG;
  if (dims->batch > 0 && dims->d_ff * dims->batch > (int64_t{1} << 31)) return IPTTT_ERR_INVALID_ARG;
  return IPTTT_OK;
}

ipttt_status check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return IPTTT_ERR_UNSUPPORTED;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return IPTTT_ERR_UNSUPPORTED;
  }
  if (major != 10 || minor != 3) return IPTTT_ERR_UNSUPPORTED;
  return IPTTT_OK;
}

// All pointers: host-side checks first (no CUDA call), then the device checks.
ipttt_status check_ptr_list(const void* const* ps, int n) {
  for (int i = 0; i < n; ++i) IPTTT_TRY(check_ptr_host(ps[i]));
  IPTTT_TRY(check_device());
  for (int i = 0; i < n; ++i) IPTTT_TRY(check_ptr_device(ps[i]));
  return IPTTT_OK;
}

namespace {

cudaError_t gemm(const GemmProblem& p, bool bf16, cudaStream_t st) {
  return bf16 ? launch_gemm_tc(p, st) : launch_gemm_simt(p, st);
}

Operand mat(const void* ptr, int64_t rows, int64_t cols, int mn_major, int64_t y0 = 0, int64_t ys1 = 0,
            int64_t ys2 = 0) {
  Operand o;
  o.ptr = ptr;
  o.rows = rows;
  o.cols = cols;
  o.ld = cols;
  o.mn_major = mn_major;
  o.y0 = y0;
  o.ys1 = ys1;
  o.ys2 = ys2;
  return o;
}
OutRef out(void* ptr, int64_t ld, int64_t y0 = 0, int64_t ys1 = 0, int64_t ys2 = 0, int64_t rows = 0) {
  OutRef o;
  o.ptr = ptr;
  o.ld = ld;
  o.y0 = y0;
  o.ys1 = ys1;
  o.ys2 = ys2;
  o.rows = rows;
  return o;
}

size_t act_size(const ipttt_dims* d) { return d->dtype == IPTTT_BF16 ? 2 : 4; }

// ---------------------------------------------------------------- steps
// The gate's tile order: dynamic (pairs take the next tile as they free up), in bands of columns
// whose W_g | W_u tiles (4 d bytes a column of Z, 128 columns a tile) take about 34 MB, so the
// band stays in L2 while every row tile of X streams past it: X is read once per band and
// W_g | W_u about once.
void gate_tile_order(GemmProblem& p, int64_t d, bool bf16) {
  p.dyn_tiles = bf16 ? 1 : 0;
  p.band_n = bf16 ? static_cast<int>(std::max<int64_t>(1, (int64_t{33} << 20) / (4 * d * 128))) : 0;
}

ipttt_status run_gate(const void* X, const void* W_g, const void* W_u, void* Z, int64_t T, const ipttt_dims* dm,
                      cudaStream_t st) {
  const bool bf16 = dm->dtype == IPTTT_BF16;
  GemmProblem p;
  p.M = T;
  p.N = dm->d_ff;
  p.K = dm->d;
  p.A = mat(X, T, dm->d, 0);
  p.B = mat(W_g, dm->d, dm->d_ff, 1);
  p.B2 = mat(W_u, dm->d, dm->d_ff, 1);
  p.epi = EPI_GATE;
  p.kind = K_GATE;
  gate_tile_order(p, dm->d, bf16);
  p.l2_d = L2_EVICT_FIRST;  // the Z tiles (written once, read much later) leave L2 first
  p.out_bf16 = bf16;
  p.D = out(Z, dm->d_ff);
  IPTTT_CUDA(gemm(p, bf16, st));
  return IPTTT_OK;
}

ipttt_status run_targets(const void* E, const float* conv_w, const void* P, void* V, void* C, int64_t rows,
                         int64_t L, int64_t B, const ipttt_dims* dm, cudaStream_t st) {
  const bool bf16 = dm->dtype == IPTTT_BF16;
  IPTTT_CUDA(launch_conv(E, conv_w, C, rows, L, B, dm->d, bf16, st));
  GemmProblem p;
  p.M = rows;
  p.N = dm->d;
  p.K = dm->d;
  p.A = mat(C, rows, dm->d, 0);
  p.B = mat(P, dm->d, dm->d, 1);
  p.epi = EPI_STORE;
  p.kind = K_PROJ;
  p.out_bf16 = bf16;
  p.D = out(V, dm->d);
  IPTTT_CUDA(gemm(p, bf16, st));
  return IPTTT_OK;
}

bool valid_rule(ipttt_rule r) {
  return r == IPTTT_RULE_MSE || r == IPTTT_RULE_ADD || r == IPTTT_RULE_ADD_BLOCKCAUSAL;
}

// Number of groups of the additive scan: the largest divisor of K not above 8.
int64_t scan_groups(int64_t K) {
  for (int64_t G = std::min<int64_t>(8, K); G > 1; --G)
    if (K % G == 0) return G;
  return 1;
}

struct EngineLayout {
  size_t o_acc = 0, r = 0, d = 0, hi = 0, lo = 0, ac = 0, bc = 0, cnt = 0, g = 0, x = 0, zt = 0, total = 0;
};

// Slices of d_ff per apply tile in the persistent MSE engine.
int engine_parts(const ipttt_dims* dm) { return static_cast<int>(std::min<int64_t>(4, dm->d_ff / 256)); }
bool use_engine(const ipttt_dims* dm, int64_t B) {
  return dm->dtype == IPTTT_BF16 && engine_mse_supported(B, dm->d, dm->d_ff);
}
// The MSE rule in windows of m = W/B chunks (bf16, chunks below 1024 tokens): the tokens of a
// window W, the largest of 1024, 768, 512 and 256 that is a multiple of 2B and divides L, on
// which the engine runs; 0 where none fits or windows do not pay.  A window saves the fast
// weight's traffic of m - 1 chunks (8 d d_ff (m - 1) bytes) and adds about 3 W d_ff FLOP per
// token of GEMMs on short contractions; measured at 32k tokens, windows of two chunks won at
// d = 2560 (6.7 against 7.3 ms) and lost at d = 1024 (2.0 against 1.8 ms), so they are taken
// where d (m - 1) >= 2 W.
int64_t window_tokens(const ipttt_dims* dm, int64_t L, int64_t B) {
  if (dm->dtype != IPTTT_BF16) return 0;
  for (int64_t w = 1024; w >= 256; w -= 256)
    if (w % (2 * B) == 0 && L % w == 0 && engine_mse_supported(w, dm->d, dm->d_ff))
      return dm->d * (w / B - 1) >= 2 * w ? w : 0;
  return 0;
}

// Plane geometry of one d_ff x d fast weight (tile-major blocks, see common.cuh).
int64_t plane_rb(const ipttt_dims* dm) { return (dm->d_ff + kPlaneRows - 1) / kPlaneRows; }
int64_t plane_cb(const ipttt_dims* dm) { return (dm->d + kPlaneCols - 1) / kPlaneCols; }
// Whether the hi planes of all entries (2 bytes an element) take at most half of the 126 MB L2.
bool planes_fit_l2(const Planes& w) {
  return w.entries * w.rb * w.cb * kPlaneBlock * 2 <= (int64_t{63} << 20);
}
Planes planes_of(const ipttt_dims* dm, uint16_t* hi, uint16_t* lo, int64_t entries, int64_t es1, int64_t es2) {
  Planes w;
  w.hi = hi;
  w.lo = lo;
  w.rb = plane_rb(dm);
  w.cb = plane_cb(dm);
  w.es1 = es1;
  w.es2 = es2;
  w.entries = entries;
  return w;
}

// Scratch of the chunk engine.  On the tensor cores the fp32 fast weight lives
// as tile-major split hi/lo planes (bf16 hi = the apply's operand, 16-bit lo =
// the rest of the fp32 bit pattern), so one update reads and writes 8 bytes
// per element.
EngineLayout engine_layout(const ipttt_dims* dm, int64_t L, int64_t B, ipttt_rule rule, size_t base) {
  EngineLayout e;
  Carve c;
  c.off = base;
  const bool bf16 = dm->dtype == IPTTT_BF16;
  const int64_t K = L / B;
  const int64_t nw = dm->d_ff * dm->d;
  const int64_t np = plane_rb(dm) * plane_cb(dm) * kPlaneBlock;  // plane elements per entry
  if (rule == IPTTT_RULE_ADD_BLOCKCAUSAL) {
    // [Z | S] per sequence (L x (d_ff + L)), [W_0 ; V] per sequence ((d_ff + L) x d), Z^T V
    const int64_t kc = dm->d_ff + L;
    const int64_t es = static_cast<int64_t>(act_size(dm));
    e.ac = c.take<uint8_t>(dm->batch * L * kc * es);
    e.bc = c.take<uint8_t>(dm->batch * kc * dm->d * es);
    e.d = c.take<float>(dm->batch * nw);
  } else if (rule == IPTTT_RULE_MSE && window_tokens(dm, L, B)) {
    // windows: per window X = (I - A)^-1 and the masked Gram A (W x W bf16), Zt = X^T Z,
    // every chunk's R kept (the output pass reads it)
    const int64_t W = window_tokens(dm, L, B), nwin = dm->batch * (L / W);
    e.o_acc = c.take<float>(dm->batch * W * dm->d);
    e.r = c.take<uint16_t>(dm->batch * L * dm->d);
    e.hi = c.take<uint16_t>(dm->batch * np);
    e.lo = c.take<uint16_t>(dm->batch * np);
    e.cnt = c.take<uint32_t>(engine_counter_words(dm->batch, L, W, dm->d, engine_parts(dm)));
    e.g = c.take<uint16_t>(nwin * W * W);
    e.x = c.take<uint16_t>(nwin * W * W);
    e.zt = c.take<uint16_t>(dm->batch * L * dm->d_ff);
  } else if (rule == IPTTT_RULE_MSE) {
    e.o_acc = c.take<float>(dm->batch * B * dm->d);
    e.r = bf16 ? c.take<uint16_t>(dm->batch * B * dm->d) : c.take<float>(dm->batch * B * dm->d);
    if (bf16) {
      e.hi = c.take<uint16_t>(dm->batch * np);
      e.lo = c.take<uint16_t>(dm->batch * np);
    }
    if (use_engine(dm, B)) e.cnt = c.take<uint32_t>(engine_counter_words(dm->batch, L, B, dm->d, engine_parts(dm)));
  } else {
    const int64_t G = scan_groups(K);
    e.o_acc = c.take<float>(G * dm->batch * B * dm->d);
    e.d = c.take<float>(G * dm->batch * nw);
    if (bf16) {
      e.hi = c.take<uint16_t>(G * dm->batch * np);
      e.lo = c.take<uint16_t>(G * dm->batch * np);
    }
  }
  e.total = c.off;
  return e;
}

// The additive rule in its block-causal quadratic form (IPTTT_RULE_ADD_BLOCKCAUSAL):
//   O = Z W_0 + (eta/B) mask(Z Z^T) V,  W_final = W_0 + (eta/B) Z^T V,
// mask keeping, for a token of chunk q, the tokens of chunks < q.  Per sequence:
// AC = [Z | S] (L x (d_ff + L)) with S = (eta/B) mask(Z Z^T) written by one GEMM
// that skips the tiles the mask clears; BC = [W_0 ; V] ((d_ff + L) x d); then
// O = AC BC is one GEMM with K = d_ff + L, and W_final the sum GEMM plus a
// one-group scan.
ipttt_status run_quadratic(const void* Z, const void* V, const float* W0, int64_t L, int64_t B, float eta, void* O,
                           float* Wf, const ipttt_dims* dm, uint8_t* ws, const EngineLayout& lay, cudaStream_t st) {
  const bool bf16 = dm->dtype == IPTTT_BF16;
  const int64_t batch = dm->batch, d = dm->d, dff = dm->d_ff, nw = dff * d, kc = dff + L;
  const int64_t w0s = dm->w0_per_seq ? nw : 0;
  const int bint = static_cast<int>(batch);
  const size_t es = act_size(dm);
  uint8_t* AC = ws + lay.ac;
  uint8_t* BC = ws + lay.bc;
  float* D = reinterpret_cast<float*>(ws + lay.d);
  const float alpha = eta / static_cast<float>(B);
  IPTTT_CUDA(cudaMemcpy2DAsync(AC, kc * es, Z, dff * es, dff * es, batch * L, cudaMemcpyDeviceToDevice, st));
  IPTTT_CUDA(cudaMemset2DAsync(AC + dff * es, kc * es, 0, L * es, batch * L, st));
  IPTTT_CUDA(launch_to_act(W0, w0s, BC, kc * d, batch, nw, bf16, st));
  IPTTT_CUDA(cudaMemcpy2DAsync(BC + dff * d * es, kc * d * es, V, L * d * es, L * d * es, batch,
                               cudaMemcpyDeviceToDevice, st));
  {  // S = alpha * mask(Z Z^T), B operand Z read K-major (row n of Z is column n of Z^T)
    GemmProblem p;
    p.M = L;
    p.N = L;
    p.K = dff;
    p.nb1 = bint;
    p.A = mat(AC, batch * L, dff, 0, 0, L);
    p.A.ld = kc;
    p.B = p.A;
    p.epi = EPI_STORE;
    p.kind = K_SCORES;
    p.out_bf16 = bf16;
    p.alpha = alpha;
    p.causal = B;
    p.D = out(AC + dff * es, kc, 0, L, 0, batch * L);
    IPTTT_CUDA(gemm(p, bf16, st));
  }
  {  // O = [Z | S] [W_0 ; V]
    GemmProblem p;
    p.M = L;
    p.N = d;
    p.K = kc;
    p.nb1 = bint;
    p.A = mat(AC, batch * L, kc, 0, 0, L);
    p.B = mat(BC, batch * kc, d, 1, 0, kc);
    p.epi = EPI_STORE;
    p.kind = K_APPLY;
    p.out_bf16 = bf16;
    p.D = out(O, d, 0, L, 0, batch * L);
    IPTTT_CUDA(gemm(p, bf16, st));
  }
  {  // W_final = W_0 + alpha Z^T V
    GemmProblem p;
    p.M = dff;
    p.N = d;
    p.K = L;
    p.nb1 = bint;
    p.A = mat(AC, batch * L, dff, 1, 0, L);
    p.A.ld = kc;
    p.B = mat(V, batch * L, d, 1, 0, L);
    p.epi = EPI_STORE;
    p.kind = K_GROUP_SUM;
    p.out_bf16 = 0;
    p.D = out(D, d, 0, dff, 0, batch * dff);
    IPTTT_CUDA(gemm(p, bf16, st));
  }
  IPTTT_CUDA(launch_group_scan(D, W0, w0s, Wf, 1, batch, nw, alpha, st));
  return IPTTT_OK;
}

// The MSE rule over windows of m = W/B chunks (bf16).  Inside a window starting at chunk k the
// steps unroll to  O_j = Z_j W_k + alpha sum_{i<j} (Z_j Z_i^T) R_i  and  R_j = O_j - V_j
// (alpha = -eta/B), so with Y_j = Z_j W_k - V_j the window's residuals solve the block lower
// triangular system  R = Y + A R,  A = alpha mask(Z Z^T) (the blocks i < j), that is R = X Y
// with X = (I - A)^-1; and  W_{k+m} = W_k + alpha Z^T R = W_k + alpha (X^T Z)^T Y.  X depends on
// Z alone, so for every window at once:
//   A = alpha mask(Z Z^T)             one masked GEMM, bf16
//   X = I; X_j = A_{j,<j} X_{<j}      row block by row block (m - 1 GEMMs over all windows)
//   Zt = X^T Z                        one GEMM
// then the persistent engine runs on windows as its chunks (apply Z W_k, R = Y, update with Zt:
// the fast weight is read and written once per window), and last  O = X Y + V  for every window
// at once.  The same O and W_final as m chunk steps, up to rounding.
ipttt_status run_windows(const void* Z, const void* V, const float* W0, int64_t L, int64_t B, float eta, void* O,
                         float* Wf, const ipttt_dims* dm, uint8_t* ws, const EngineLayout& lay, cudaStream_t st) {
  const int64_t batch = dm->batch, d = dm->d, dff = dm->d_ff, nw = dff * d;
  const int64_t W = window_tokens(dm, L, B), m = W / B, nwin = batch * (L / W);
  const int nwi = static_cast<int>(nwin);
  const float alpha = -eta / static_cast<float>(B);
  uint16_t* G = reinterpret_cast<uint16_t*>(ws + lay.g);
  uint16_t* X = reinterpret_cast<uint16_t*>(ws + lay.x);
  uint16_t* Zt = reinterpret_cast<uint16_t*>(ws + lay.zt);
  void* R = ws + lay.r;
  IPTTT_CUDA(launch_eye_bf16(X, W, nwin, st));
  {  // A = alpha mask(Z Z^T) per window (tiles the mask clears are skipped; X_j reads none of them)
    GemmProblem p;
    p.M = W;
    p.N = W;
    p.K = dff;
    p.nb1 = nwi;
    p.A = mat(Z, batch * L, dff, 0, 0, W);
    p.B = p.A;
    p.epi = EPI_STORE;
    p.kind = K_WINDOW;
    p.out_bf16 = 1;
    p.alpha = alpha;
    p.causal = B;
    p.D = out(G, W, 0, W, 0, nwin * W);
    IPTTT_CUDA(gemm(p, true, st));
  }
  for (int64_t j = 1; j < m; ++j) {  // X[jB .. jB+B, 0 .. jB] = A[jB .. jB+B, 0 .. jB] X[0 .. jB, 0 .. jB]
    GemmProblem p;
    p.M = B;
    p.N = j * B;
    p.K = j * B;
    p.nb1 = nwi;
    p.A = mat(G, nwin * W, W, 0, j * B, W);
    p.B = mat(X, nwin * W, W, 1, 0, W);
    p.epi = EPI_STORE;
    p.kind = K_WINDOW;
    p.out_bf16 = 1;
    p.D = out(X, W, j * B, W, 0, nwin * W);
    IPTTT_CUDA(gemm(p, true, st));
  }
  {  // Zt = X^T Z per window
    GemmProblem p;
    p.M = W;
    p.N = dff;
    p.K = W;
    p.nb1 = nwi;
    p.A = mat(X, nwin * W, W, 1, 0, W);
    p.B = mat(Z, batch * L, dff, 1, 0, W);
    p.tri = -1;       // A = X^T is upper triangular
    p.dyn_tiles = 1;  // tiles of unequal contractions: pairs take them as they free up
    p.epi = EPI_STORE;
    p.kind = K_WINDOW;
    p.out_bf16 = 1;
    p.D = out(Zt, dff, 0, W, 0, batch * L);
    IPTTT_CUDA(gemm(p, true, st));
  }
  const Planes w = planes_of(dm, reinterpret_cast<uint16_t*>(ws + lay.hi), reinterpret_cast<uint16_t*>(ws + lay.lo),
                             batch, 1, 0);
  IPTTT_CUDA(launch_split_planes(W0, dm->w0_per_seq ? nw : 0, w, dff, d, st));
  float* o_acc = reinterpret_cast<float*>(ws + lay.o_acc);
  IPTTT_CUDA(cudaMemsetAsync(o_acc, 0, sizeof(float) * batch * W * d, st));
  EngineMse em;
  em.Z = Z;
  em.Zu = Zt;
  em.V = V;
  em.O = O;  // Z_w W_k here; the output pass below writes O
  em.acc = o_acc;
  em.R = R;  // Y, every window's kept
  em.r_seq = L;
  em.r_chunk = W;
  em.counters = reinterpret_cast<uint32_t*>(ws + lay.cnt);
  em.w = w;
  em.batch = batch;
  em.L = L;
  em.B = W;
  em.d = d;
  em.d_ff = dff;
  em.parts = engine_parts(dm);
  em.alpha = alpha;
  em.keep_hi = planes_fit_l2(w) ? 1 : 0;
  IPTTT_CUDA(cudaMemsetAsync(em.counters, 0, sizeof(uint32_t) * engine_counter_words(batch, L, W, d, em.parts), st));
  IPTTT_CUDA(launch_engine_mse(em, st));
  IPTTT_CUDA(launch_merge_planes(w, Wf, dff, d, st));
  {  // O = X Y + V per window
    GemmProblem p;
    p.M = W;
    p.N = d;
    p.K = W;
    p.nb1 = nwi;
    p.A = mat(X, nwin * W, W, 0, 0, W);
    p.B = mat(R, batch * L, d, 1, 0, W);
    p.tri = 1;  // X is lower triangular
    p.dyn_tiles = 1;
    p.epi = EPI_STORE;
    p.kind = K_WINDOW;
    p.out_bf16 = 1;
    p.add = out(const_cast<void*>(V), d, 0, W);
    p.D = out(O, d, 0, W, 0, batch * L);
    IPTTT_CUDA(gemm(p, true, st));
  }
  return IPTTT_OK;
}

ipttt_status run_engine(const void* Z, const void* V, const float* W0, int64_t L, int64_t B, float eta,
                        ipttt_rule rule, void* O, float* Wf, const ipttt_dims* dm, uint8_t* ws, const EngineLayout& lay,
                        cudaStream_t st) {
  const bool bf16 = dm->dtype == IPTTT_BF16;
  const int64_t batch = dm->batch, d = dm->d, dff = dm->d_ff, K = L / B, nw = dff * d;
  const int64_t w0s = dm->w0_per_seq ? nw : 0;  // element stride between sequences' W_o0
  const int64_t w0r = dm->w0_per_seq ? dff : 0;  // same, in rows
  const int bint = static_cast<int>(batch);
  float* o_acc = reinterpret_cast<float*>(ws + lay.o_acc);
  uint16_t* hi = bf16 ? reinterpret_cast<uint16_t*>(ws + lay.hi) : nullptr;
  uint16_t* lo = bf16 ? reinterpret_cast<uint16_t*>(ws + lay.lo) : nullptr;

  if (rule == IPTTT_RULE_ADD_BLOCKCAUSAL) return run_quadratic(Z, V, W0, L, B, eta, O, Wf, dm, ws, lay, st);
  if (rule == IPTTT_RULE_MSE && window_tokens(dm, L, B)) return run_windows(Z, V, W0, L, B, eta, O, Wf, dm, ws, lay, st);
  if (rule == IPTTT_RULE_MSE) {
    void* R = ws + lay.r;
    const Planes w = planes_of(dm, hi, lo, batch, 1, 0);
    if (bf16) IPTTT_CUDA(launch_split_planes(W0, w0s, w, dff, d, st));
    IPTTT_CUDA(cudaMemsetAsync(o_acc, 0, sizeof(float) * batch * B * d, st));
    const int64_t w0_rows = (dm->w0_per_seq ? batch : 1) * dff;
    // The hi planes stay in L2 from one chunk to the next when they take at most half of it.
    const bool keep_hi = bf16 && planes_fit_l2(w);
    if (use_engine(dm, B)) {
      // the whole chunk loop in one persistent kernel
      EngineMse em;
      em.Z = Z;
      em.V = V;
      em.O = O;
      em.acc = o_acc;
      em.R = R;
      em.r_seq = B;
      em.counters = reinterpret_cast<uint32_t*>(ws + lay.cnt);
      em.w = w;
      em.batch = batch;
      em.L = L;
      em.B = B;
      em.d = d;
      em.d_ff = dff;
      em.parts = engine_parts(dm);
      em.alpha = -eta / static_cast<float>(B);
      em.keep_hi = keep_hi ? 1 : 0;
      IPTTT_CUDA(cudaMemsetAsync(em.counters, 0,
                                 sizeof(uint32_t) * engine_counter_words(batch, L, B, d, em.parts), st));
      IPTTT_CUDA(launch_engine_mse(em, st));
      IPTTT_CUDA(launch_merge_planes(w, Wf, dff, d, st));
      return IPTTT_OK;
    }
    const int64_t zrow = dff * static_cast<int64_t>(act_size(dm));  // bytes of a row of Z
    for (int64_t k = 0; k < K; ++k) {
      // apply: O_acc[s] = Z_k[s] W_k[s], split over d_ff
      GemmProblem a;
      a.M = B;
      a.N = d;
      a.K = dff;
      a.nb1 = bint;
      a.A = mat(Z, batch * L, dff, 0, k * B, L);
      if (bf16) {
        a.B = mat(hi, batch * dff, d, 1, 0, dff);
        a.w = w;
        a.b_planes = 1;
        a.l2_b = keep_hi ? L2_EVICT_LAST : L2_NORMAL;
      } else
        a.B = (k == 0) ? mat(W0, w0_rows, d, 1, 0, w0r) : mat(Wf, batch * dff, d, 1, 0, dff);
      a.epi = EPI_ACCUM;
      a.kind = K_APPLY;
      a.D = out(o_acc, d, 0, B, 0, batch * B);
      a.split_k = 1;
      IPTTT_CUDA(gemm(a, bf16, st));
      // residual: O_k = O_acc, R_k = O_acc - V_k, O_acc = 0
      ResidualArgs ra;
      ra.acc = o_acc;
      ra.V = V;
      ra.O = O;
      ra.R = R;
      ra.B = B;
      ra.d = d;
      ra.nb1 = bint;
      ra.o_y0 = k * B;
      ra.o_ys1 = L;
      IPTTT_CUDA(launch_residual(ra, bf16, st));
      // update: W_{k+1} = W_k - (eta/B) Z_k^T R_k
      GemmProblem u;
      u.M = dff;
      u.N = d;
      u.K = B;
      u.nb1 = bint;
      u.A = mat(Z, batch * L, dff, 1, k * B, L);
      u.B = mat(R, batch * B, d, 1, 0, B);
      u.epi = EPI_AXPY;
      u.kind = K_UPDATE;
      if (bf16) {
        u.w = w;
        u.planes_l2 = keep_hi ? 1 : 0;
        u.l2_a = L2_EVICT_FIRST;  // the last read of Z_k
        if (k + 1 < K) {          // the next apply's Z_{k+1}, fetched into L2 as the update ends
          u.pf_ptr = static_cast<const uint8_t*>(Z) + (k + 1) * B * zrow;
          u.pf_bytes = B * zrow;
          u.pf_stride = L * zrow;
          u.pf_count = bint;
        }
      } else {
        u.D = out(Wf, d, 0, dff, 0, batch * dff);
        u.src = (k == 0) ? out(const_cast<float*>(W0), d, 0, w0r, 0, w0_rows) : out(Wf, d, 0, dff, 0, batch * dff);
      }
      u.alpha = -eta / static_cast<float>(B);
      IPTTT_CUDA(gemm(u, bf16, st));
    }
    if (bf16) IPTTT_CUDA(launch_merge_planes(w, Wf, dff, d, st));
    return IPTTT_OK;
  }

  // additive rule: chunk-parallel scan
  const int64_t G = scan_groups(K), g = K / G;
  const int gint = static_cast<int>(G);
  float* D = reinterpret_cast<float*>(ws + lay.d);
  const float alpha = eta / static_cast<float>(B);
  // group sums, all groups of all sequences at once
  GemmProblem s;
  s.M = dff;
  s.N = d;
  s.K = g * B;
  s.nb1 = bint;
  s.nb2 = gint;
  s.A = mat(Z, batch * L, dff, 1, 0, L, g * B);
  s.B = mat(V, batch * L, d, 1, 0, L, g * B);
  s.epi = EPI_STORE;
  s.kind = K_GROUP_SUM;
  s.out_bf16 = 0;
  s.D = out(D, d, 0, dff, batch * dff);
  IPTTT_CUDA(gemm(s, bf16, st));
  // exclusive scan over groups -> the fast weight at the start of each group
  const Planes w = planes_of(dm, hi, lo, G * batch, 1, batch);
  if (bf16)
    IPTTT_CUDA(launch_group_scan_planes(D, w, W0, w0s, Wf, G, batch, dff, d, alpha, st));
  else
    IPTTT_CUDA(launch_group_scan(D, W0, w0s, Wf, G, batch, nw, alpha, st));
  IPTTT_CUDA(cudaMemsetAsync(o_acc, 0, sizeof(float) * G * batch * B * d, st));
  for (int64_t i = 0; i < g; ++i) {
    GemmProblem a;
    a.M = B;
    a.N = d;
    a.K = dff;
    a.nb1 = bint;
    a.nb2 = gint;
    a.A = mat(Z, batch * L, dff, 0, i * B, L, g * B);
    a.B = bf16 ? mat(hi, G * batch * dff, d, 1, 0, dff, batch * dff) : mat(D, G * batch * dff, d, 1, 0, dff, batch * dff);
    if (bf16) {
      a.w = w;
      a.b_planes = 1;
    }
    a.epi = EPI_ACCUM;
    a.kind = K_APPLY;
    a.D = out(o_acc, d, 0, B, batch * B, G * batch * B);
    a.split_k = 1;
    IPTTT_CUDA(gemm(a, bf16, st));
    {
      ResidualArgs ra;
      ra.acc = o_acc;
      ra.O = O;
      ra.B = B;
      ra.d = d;
      ra.nb1 = bint;
      ra.nb2 = gint;
      ra.o_y0 = i * B;
      ra.o_ys1 = L;
      ra.o_ys2 = g * B;
      IPTTT_CUDA(launch_residual(ra, bf16, st));
    }
    if (i + 1 < g) {
      GemmProblem u;
      u.M = dff;
      u.N = d;
      u.K = B;
      u.nb1 = bint;
      u.nb2 = gint;
      u.A = mat(Z, batch * L, dff, 1, i * B, L, g * B);
      u.B = mat(V, batch * L, d, 1, i * B, L, g * B);
      u.epi = EPI_AXPY;
      u.kind = K_UPDATE;
      if (bf16) {
        u.w = w;
      } else {
        u.D = u.src = out(D, d, 0, dff, batch * dff, G * batch * dff);
      }
      u.alpha = alpha;
      IPTTT_CUDA(gemm(u, bf16, st));
    }
  }
  return IPTTT_OK;
}

struct LaunchScope {
  LaunchScope() { t_launches = 0; }
};

// ------------------------------------------------------- packed documents
// The layer over packed documents, the fast weight reset to W_o0 at every
// boundary (In-Place TTT, itsolotime §3.2 "boundary reset").  Documents are
// taken longest first, so the ones still running at chunk step i are a prefix
// of that order and each step is one batched apply / residual / update over
// them; a document's rows are found through a table of starts.  A document's
// last chunk may be short: the residual pass writes zeros past its end (the
// update's contraction then ignores those rows) and scales R by B/n, so the
// step is the mean over the chunk's n tokens.
struct VarlenPlan {
  int64_t T = 0, n_docs = 0, k_max = 0;
  std::vector<int64_t> order;   // sorted position -> document
  std::vector<int64_t> starts;  // sorted position -> first row
  std::vector<int64_t> lens;    // sorted position -> tokens
  std::vector<int64_t> active;  // chunk step -> documents still running
};

ipttt_status plan_varlen(const int64_t* cu, int64_t n_docs, int64_t B, VarlenPlan* pl) {
  if (!cu || n_docs < 0 || cu[0] != 0) return IPTTT_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n_docs; ++i)
    if (cu[i + 1] <= cu[i]) return IPTTT_ERR_INVALID_ARG;
  pl->n_docs = n_docs;
  pl->T = cu[n_docs];
  pl->order.resize(n_docs);
  for (int64_t i = 0; i < n_docs; ++i) pl->order[i] = i;
  std::stable_sort(pl->order.begin(), pl->order.end(),
                   [&](int64_t a, int64_t b) { return cu[a + 1] - cu[a] > cu[b + 1] - cu[b]; });
  pl->starts.resize(n_docs);
  pl->lens.resize(n_docs);
  for (int64_t s = 0; s < n_docs; ++s) {
    pl->starts[s] = cu[pl->order[s]];
    pl->lens[s] = cu[pl->order[s] + 1] - cu[pl->order[s]];
  }
  pl->k_max = n_docs ? (pl->lens[0] + B - 1) / B : 0;
  pl->active.assign(pl->k_max, 0);
  for (int64_t s = 0; s < n_docs; ++s)
    for (int64_t i = 0; i < (pl->lens[s] + B - 1) / B; ++i) ++pl->active[i];
  return IPTTT_OK;
}

ipttt_status run_varlen(const void* X, const void* E, const void* W_g, const void* W_u, const float* W0,
                        const float* conv_w, const void* P, const int64_t* cu, const VarlenPlan& pl, int64_t B,
                        float eta, ipttt_rule rule, void* O, float* Wf, const ipttt_dims* dm, cudaStream_t st) {
  const bool bf16 = dm->dtype == IPTTT_BF16;
  const int64_t n = pl.n_docs, T = pl.T, d = dm->d, dff = dm->d_ff, nw = dff * d;
  const size_t es = act_size(dm);
  const int64_t np = plane_rb(dm) * plane_cb(dm) * kPlaneBlock;
  Carve c;
  const size_t z_off = c.take<uint8_t>(T * dff * static_cast<int64_t>(es));
  const size_t v_off = c.take<uint8_t>(T * d * static_cast<int64_t>(es));
  const size_t c_off = c.take<uint8_t>(T * d * static_cast<int64_t>(es));
  const size_t acc_off = c.take<float>(n * B * d);
  const size_t r_off = c.take<uint8_t>(n * B * d * static_cast<int64_t>(es));
  const size_t hi_off = bf16 ? c.take<uint16_t>(n * np) : 0;
  const size_t lo_off = bf16 ? c.take<uint16_t>(n * np) : 0;
  const size_t cu_off = c.take<int64_t>(n + 1);
  const size_t st_off = c.take<int64_t>(n);
  const size_t ln_off = c.take<int64_t>(n);
  const size_t wt_off = c.take<int64_t>(n);
  // the persistent engine (bf16 MSE, engine shapes): documents running per chunk, items before
  // each chunk, counters
  const bool eng = bf16 && rule == IPTTT_RULE_MSE && engine_mse_supported(B, d, dff) && n > 0;
  const int parts = engine_parts(dm);
  const int64_t Lmax = pl.k_max * B;
  const size_t ac_off = eng ? c.take<int64_t>(pl.k_max) : 0;
  const size_t ic_off = eng ? c.take<int64_t>(pl.k_max + 1) : 0;
  const size_t cn_off = eng ? c.take<uint32_t>(engine_counter_words(n, Lmax, B, d, parts)) : 0;
  void* wsv = nullptr;
  IPTTT_TRY(pool_reserve(c.off, &wsv));
  uint8_t* ws = static_cast<uint8_t*>(wsv);
  int64_t* cu_d = reinterpret_cast<int64_t*>(ws + cu_off);
  int64_t* starts_d = reinterpret_cast<int64_t*>(ws + st_off);
  int64_t* lens_d = reinterpret_cast<int64_t*>(ws + ln_off);
  int64_t* wtab_d = reinterpret_cast<int64_t*>(ws + wt_off);
  std::vector<int64_t> wtab(n);
  for (int64_t s = 0; s < n; ++s) wtab[s] = pl.order[s] * dff;
  // pageable sources: each copy has read its source when the call returns
  IPTTT_CUDA(cudaMemcpyAsync(cu_d, cu, sizeof(int64_t) * (n + 1), cudaMemcpyHostToDevice, st));
  IPTTT_CUDA(cudaMemcpyAsync(starts_d, pl.starts.data(), sizeof(int64_t) * n, cudaMemcpyHostToDevice, st));
  IPTTT_CUDA(cudaMemcpyAsync(lens_d, pl.lens.data(), sizeof(int64_t) * n, cudaMemcpyHostToDevice, st));
  IPTTT_CUDA(cudaMemcpyAsync(wtab_d, wtab.data(), sizeof(int64_t) * n, cudaMemcpyHostToDevice, st));

  void* Z = ws + z_off;
  void* V = ws + v_off;
  void* R = ws + r_off;
  float* o_acc = reinterpret_cast<float*>(ws + acc_off);
  uint16_t* hi = bf16 ? reinterpret_cast<uint16_t*>(ws + hi_off) : nullptr;
  uint16_t* lo = bf16 ? reinterpret_cast<uint16_t*>(ws + lo_off) : nullptr;
  IPTTT_TRY(run_gate(X, W_g, W_u, Z, T, dm, st));
  IPTTT_CUDA(launch_conv_varlen(E, conv_w, ws + c_off, T, cu_d, n, B, d, bf16, st));
  {
    GemmProblem p;
    p.M = T;
    p.N = d;
    p.K = d;
    p.A = mat(ws + c_off, T, d, 0);
    p.B = mat(P, d, d, 1);
    p.epi = EPI_STORE;
    p.kind = K_PROJ;
    p.out_bf16 = bf16;
    p.D = out(V, d);
    IPTTT_CUDA(gemm(p, bf16, st));
  }
  // fast weights: planes in sorted order (bf16), or W_final itself in document order (fp32)
  const Planes w = planes_of(dm, hi, lo, n, 1, 0);
  if (bf16) {
    if (dm->w0_per_seq) {
      for (int64_t s = 0; s < n; ++s)
        IPTTT_CUDA(launch_split_planes(W0 + pl.order[s] * nw, 0, planes_of(dm, hi + s * np, lo + s * np, 1, 1, 0),
                                       dff, d, st));
    } else {
      IPTTT_CUDA(launch_split_planes(W0, 0, w, dff, d, st));
    }
  } else {
    IPTTT_CUDA(launch_copy_w(W0, dm->w0_per_seq ? nw : 0, Wf, n, nw, st));
  }
  IPTTT_CUDA(cudaMemsetAsync(o_acc, 0, sizeof(float) * n * B * d, st));
  const float alpha = (rule == IPTTT_RULE_MSE ? -eta : eta) / static_cast<float>(B);
  if (eng) {
    // the whole chunk loop of every document in one persistent kernel; chunk k's items cover the
    // documents still running (a prefix of the longest-first order)
    const int64_t NB = d / 256, MT = B / 256, RT = dff / 256;
    std::vector<int64_t> icum(pl.k_max + 1, 0);
    for (int64_t k = 0; k < pl.k_max; ++k) icum[k + 1] = icum[k] + NB * pl.active[k] * (MT * parts + RT);
    int64_t* act_d = reinterpret_cast<int64_t*>(ws + ac_off);
    int64_t* icum_d = reinterpret_cast<int64_t*>(ws + ic_off);
    IPTTT_CUDA(cudaMemcpyAsync(act_d, pl.active.data(), sizeof(int64_t) * pl.k_max, cudaMemcpyHostToDevice, st));
    IPTTT_CUDA(cudaMemcpyAsync(icum_d, icum.data(), sizeof(int64_t) * (pl.k_max + 1), cudaMemcpyHostToDevice, st));
    EngineMse em;
    em.Z = Z;
    em.V = V;
    em.O = O;
    em.acc = o_acc;
    em.R = R;
    em.r_seq = B;
    em.counters = reinterpret_cast<uint32_t*>(ws + cn_off);
    em.w = w;
    em.batch = n;
    em.L = Lmax;
    em.B = B;
    em.d = d;
    em.d_ff = dff;
    em.parts = parts;
    em.alpha = alpha;
    em.keep_hi = planes_fit_l2(w) ? 1 : 0;
    em.starts = starts_d;
    em.lens = lens_d;
    em.active = act_d;
    em.icum = icum_d;
    em.icum_total = icum[pl.k_max];
    em.rows = T;
    IPTTT_CUDA(cudaMemsetAsync(em.counters, 0, sizeof(uint32_t) * engine_counter_words(n, Lmax, B, d, parts), st));
    IPTTT_CUDA(launch_engine_mse(em, st));
  }
  for (int64_t i = 0; i < (eng ? 0 : pl.k_max); ++i) {
    const int na = static_cast<int>(pl.active[i]);
    GemmProblem a;
    a.M = B;
    a.N = d;
    a.K = dff;
    a.nb1 = na;
    a.A = mat(Z, T, dff, 0, i * B);
    a.A.ytab = starts_d;
    if (bf16) {
      a.B = mat(hi, n * dff, d, 1, 0, dff);
      a.w = w;
      a.b_planes = 1;
    } else {
      a.B = mat(Wf, n * dff, d, 1);
      a.B.ytab = wtab_d;
    }
    a.epi = EPI_ACCUM;
    a.kind = K_APPLY;
    a.D = out(o_acc, d, 0, B, 0, n * B);
    a.split_k = 1;
    IPTTT_CUDA(gemm(a, bf16, st));
    ResidualArgs ra;
    ra.acc = o_acc;
    ra.V = V;
    ra.O = O;
    ra.R = R;
    ra.B = B;
    ra.d = d;
    ra.nb1 = na;
    ra.o_y0 = i * B;
    ra.otab = starts_d;
    ra.lens = lens_d;
    ra.r_from_v = rule != IPTTT_RULE_MSE;
    IPTTT_CUDA(launch_residual(ra, bf16, st));
    GemmProblem u;
    u.M = dff;
    u.N = d;
    u.K = B;
    u.nb1 = na;
    u.A = mat(Z, T, dff, 1, i * B);
    u.A.ytab = starts_d;
    u.B = mat(R, n * B, d, 1, 0, B);
    u.epi = EPI_AXPY;
    u.kind = K_UPDATE;
    if (bf16) {
      u.w = w;
    } else {
      u.D = out(Wf, d, 0, 0, 0, n * dff);
      u.D.ytab = wtab_d;
      u.src = u.D;
    }
    u.alpha = alpha;
    IPTTT_CUDA(gemm(u, bf16, st));
  }
  if (bf16) {
    for (int64_t s = 0; s < n; ++s)
      IPTTT_CUDA(launch_merge_planes(planes_of(dm, hi + s * np, lo + s * np, 1, 1, 0), Wf + pl.order[s] * nw, dff, d,
                                     st));
  }
  return IPTTT_OK;
}

}  // namespace
}  // namespace ipttt

using namespace ipttt;

extern "C" {

ipttt_status ipttt_workspace_size(const ipttt_dims* dims, int64_t L, int64_t B, ipttt_rule rule,
                                  int32_t with_activations, size_t* bytes) {
  IPTTT_TRY(check_dims(dims, true));
  IPTTT_TRY(check_chunking(dims, L, B));
  if (!bytes || !valid_rule(rule)) return IPTTT_ERR_INVALID_ARG;
  size_t base = 0;
  if (with_activations) {
    Carve c;
    const int64_t T = dims->batch * L;
    const size_t es = act_size(dims);
    c.off += (static_cast<size_t>(T * dims->d_ff) * es + 255) & ~size_t(255);  // Z
    c.off += (static_cast<size_t>(T * dims->d) * es + 255) & ~size_t(255);     // V
    c.off += (static_cast<size_t>(T * dims->d) * es + 255) & ~size_t(255);     // conv output
    base = c.off;
  }
  *bytes = (L == 0 || dims->batch == 0) ? 0 : engine_layout(dims, L, B, rule, base).total;
  return IPTTT_OK;
}

ipttt_status ipttt_gate_up(const void* X, const void* W_g, const void* W_u, void* Z, int64_t n_tokens,
                           const ipttt_dims* dims, ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, false));
  if (n_tokens < 0 || n_tokens > (int64_t{1} << 31)) return IPTTT_ERR_INVALID_ARG;
  if (n_tokens == 0) return IPTTT_OK;
  IPTTT_TRY(check_ptrs({X, W_g, W_u, static_cast<const void*>(Z)}));
  return run_gate(X, W_g, W_u, Z, n_tokens, dims, static_cast<cudaStream_t>(stream));
}

ipttt_status ipttt_make_targets(const void* E, const float* conv_w, const void* P, void* V, int64_t L, int64_t B,
                                const ipttt_dims* dims, ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, true));
  IPTTT_TRY(check_chunking(dims, L, B));
  const int64_t rows = dims->batch * L;
  if (rows == 0) return IPTTT_OK;
  IPTTT_TRY(check_ptrs({E, static_cast<const void*>(conv_w), P, static_cast<const void*>(V)}));
  void* ws = nullptr;
  IPTTT_TRY(pool_reserve(static_cast<size_t>(rows * dims->d) * act_size(dims), &ws));
  return run_targets(E, conv_w, P, V, ws, rows, L, B, dims, static_cast<cudaStream_t>(stream));
}

ipttt_status ipttt_chunk_forward(const void* Z, const void* V, const float* W_o0, int64_t L, int64_t B, float eta,
                                 ipttt_rule rule, void* O, float* W_final, const ipttt_dims* dims,
                                 ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, true));
  IPTTT_TRY(check_chunking(dims, L, B));
  if (!valid_rule(rule) || !std::isfinite(eta)) return IPTTT_ERR_INVALID_ARG;
  if (dims->batch == 0) return IPTTT_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t nw = dims->d_ff * dims->d;
  if (L == 0) {
    IPTTT_TRY(check_ptrs({static_cast<const void*>(W_o0), static_cast<const void*>(W_final)}));
    IPTTT_CUDA(launch_copy_w(W_o0, dims->w0_per_seq ? nw : 0, W_final, dims->batch, nw, st));
    return IPTTT_OK;
  }
  IPTTT_TRY(check_ptrs({Z, V, static_cast<const void*>(W_o0), static_cast<const void*>(O),
                        static_cast<const void*>(W_final)}));
  const EngineLayout lay = engine_layout(dims, L, B, rule, 0);
  void* ws = nullptr;
  IPTTT_TRY(pool_reserve(lay.total, &ws));
  return run_engine(Z, V, W_o0, L, B, eta, rule, O, W_final, dims, static_cast<uint8_t*>(ws), lay, st);
}

ipttt_status ipttt_layer_forward(const void* X, const void* E, const void* W_g, const void* W_u, const float* W_o0,
                                 const float* conv_w, const void* P, int64_t L, int64_t B, float eta,
                                 ipttt_rule rule, void* O, float* W_final, const ipttt_dims* dims,
                                 ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, true));
  IPTTT_TRY(check_chunking(dims, L, B));
  if (!valid_rule(rule) || !std::isfinite(eta)) return IPTTT_ERR_INVALID_ARG;
  if (dims->batch == 0) return IPTTT_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t nw = dims->d_ff * dims->d;
  if (L == 0) {
    IPTTT_TRY(check_ptrs({static_cast<const void*>(W_o0), static_cast<const void*>(W_final)}));
    IPTTT_CUDA(launch_copy_w(W_o0, dims->w0_per_seq ? nw : 0, W_final, dims->batch, nw, st));
    return IPTTT_OK;
  }
  IPTTT_TRY(check_ptrs({X, E, W_g, W_u, static_cast<const void*>(W_o0), static_cast<const void*>(conv_w), P,
                        static_cast<const void*>(O), static_cast<const void*>(W_final)}));
  const int64_t T = dims->batch * L;
  const size_t es = act_size(dims);
  Carve c;
  const size_t z_off = c.take<uint8_t>(T * dims->d_ff * static_cast<int64_t>(es));
  const size_t v_off = c.take<uint8_t>(T * dims->d * static_cast<int64_t>(es));
  const size_t c_off = c.take<uint8_t>(T * dims->d * static_cast<int64_t>(es));
  const EngineLayout lay = engine_layout(dims, L, B, rule, c.off);
  void* wsv = nullptr;
  IPTTT_TRY(pool_reserve(lay.total, &wsv));
  uint8_t* ws = static_cast<uint8_t*>(wsv);
  IPTTT_TRY(run_gate(X, W_g, W_u, ws + z_off, T, dims, st));
  IPTTT_TRY(run_targets(E, conv_w, P, ws + v_off, ws + c_off, T, L, B, dims, st));
  return run_engine(ws + z_off, ws + v_off, W_o0, L, B, eta, rule, O, W_final, dims, ws, lay, st);
}

ipttt_status ipttt_layer_forward_varlen(const void* X, const void* E, const void* W_g, const void* W_u,
                                        const float* W_o0, const float* conv_w, const void* P,
                                        const int64_t* cu_seqlens, int64_t n_docs, int64_t B, float eta,
                                        ipttt_rule rule, void* O, float* W_final, const ipttt_dims* dims,
                                        ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, false));
  if (!valid_rule(rule) || !std::isfinite(eta)) return IPTTT_ERR_INVALID_ARG;
  if (B < 1 || n_docs < 0 || !cu_seqlens) return IPTTT_ERR_INVALID_ARG;
  if (dims->dtype == IPTTT_BF16 && B % 16) return IPTTT_ERR_INVALID_ARG;
  VarlenPlan pl;
  IPTTT_TRY(plan_varlen(cu_seqlens, n_docs, B, &pl));
  if (n_docs == 0) return IPTTT_OK;
  // token rows, fast-weight rows and chunk rows of all documents are TMA coordinates (int32)
  if (pl.T > (int64_t{1} << 31) || dims->d_ff * n_docs > (int64_t{1} << 31) || B * n_docs > (int64_t{1} << 31))
    return IPTTT_ERR_INVALID_ARG;
  IPTTT_TRY(check_ptrs({X, E, W_g, W_u, static_cast<const void*>(W_o0), static_cast<const void*>(conv_w), P,
                        static_cast<const void*>(O), static_cast<const void*>(W_final)}));
  return run_varlen(X, E, W_g, W_u, W_o0, conv_w, P, cu_seqlens, pl, B, eta, rule, O, W_final, dims,
                    static_cast<cudaStream_t>(stream));
}

ipttt_status ipttt_layers_forward(const void* X, const void* E, const void* W_g, const void* W_u, const float* W_o0,
                                  const float* conv_w, const void* P, int64_t n_layers, int64_t L, int64_t B, float eta,
                                  ipttt_rule rule, void* O, float* W_final, const ipttt_dims* dims,
                                  ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, true));
  IPTTT_TRY(check_chunking(dims, L, B));
  if (!valid_rule(rule) || !std::isfinite(eta) || n_layers < 0)
    return IPTTT_ERR_INVALID_ARG;
  if (n_layers == 0 || dims->batch == 0) return IPTTT_OK;
  const int64_t batch = dims->batch, d = dims->d, dff = dims->d_ff, nw = dff * d;
  const int64_t entries = n_layers * batch, T = batch * L, NT = n_layers * T;
  // token rows, weight rows and fast-weight rows of all layers are TMA coordinates (int32)
  if (NT > (int64_t{1} << 31) || dff * entries > (int64_t{1} << 31) || n_layers * d > (int64_t{1} << 31))
    return IPTTT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Layer l, sequence s is entry l*batch + s of the chunk engine: its rows of Z, V
  // and O sit at (l*batch + s)*L, and its fast weight at W_final[l][s].
  if (L == 0) {
    IPTTT_TRY(check_ptrs({static_cast<const void*>(W_o0), static_cast<const void*>(W_final)}));
    if (dims->w0_per_seq) {
      IPTTT_CUDA(launch_copy_w(W_o0, nw, W_final, entries, nw, st));
    } else {
      for (int64_t l = 0; l < n_layers; ++l)
        IPTTT_CUDA(launch_copy_w(W_o0 + l * nw, 0, W_final + l * batch * nw, batch, nw, st));
    }
    return IPTTT_OK;
  }
  IPTTT_TRY(check_ptrs({X, E, W_g, W_u, static_cast<const void*>(W_o0), static_cast<const void*>(conv_w), P,
                        static_cast<const void*>(O), static_cast<const void*>(W_final)}));
  const bool bf16 = dims->dtype == IPTTT_BF16;
  ipttt_dims dm = *dims;
  dm.batch = entries;
  dm.w0_per_seq = 1;
  const size_t es = act_size(dims);
  Carve c;
  const size_t z_off = c.take<uint8_t>(NT * dff * static_cast<int64_t>(es));
  const size_t v_off = c.take<uint8_t>(NT * d * static_cast<int64_t>(es));
  const size_t c_off = c.take<uint8_t>(NT * d * static_cast<int64_t>(es));
  const EngineLayout lay = engine_layout(&dm, L, B, rule, c.off);
  void* wsv = nullptr;
  IPTTT_TRY(pool_reserve(lay.total, &wsv));
  uint8_t* ws = static_cast<uint8_t*>(wsv);
  // gate of every layer: one GEMM over the layers (batch entry = layer)
  {
    GemmProblem p;
    p.M = T;
    p.N = dff;
    p.K = d;
    p.nb1 = static_cast<int>(n_layers);
    p.A = mat(X, NT, d, 0, 0, T);
    p.B = mat(W_g, n_layers * d, dff, 1, 0, d);
    p.B2 = mat(W_u, n_layers * d, dff, 1, 0, d);
    p.epi = EPI_GATE;
    p.kind = K_GATE;
    p.out_bf16 = bf16;
    gate_tile_order(p, d, bf16);
    p.l2_d = L2_EVICT_FIRST;
    p.D = out(ws + z_off, dff, 0, T, 0, NT);
    IPTTT_CUDA(gemm(p, bf16, st));
  }
  // targets of every layer from the shared embeddings: one conv launch, one projection GEMM
  IPTTT_CUDA(launch_conv(E, conv_w, ws + c_off, NT, L, B, d, bf16, st, T));
  {
    GemmProblem p;
    p.M = T;
    p.N = d;
    p.K = d;
    p.nb1 = static_cast<int>(n_layers);
    p.A = mat(ws + c_off, NT, d, 0, 0, T);
    p.B = mat(P, n_layers * d, d, 1, 0, d);
    p.epi = EPI_STORE;
    p.kind = K_PROJ;
    p.out_bf16 = bf16;
    p.D = out(ws + v_off, d, 0, T, 0, NT);
    IPTTT_CUDA(gemm(p, bf16, st));
  }
  // each entry's initial fast weight: a per-layer W_o0 shared by the sequences is copied into
  // W_final first, which the engine reads before it writes its result there
  const float* W0 = W_o0;
  if (!dims->w0_per_seq && batch > 1) {
    for (int64_t l = 0; l < n_layers; ++l)
      IPTTT_CUDA(launch_copy_w(W_o0 + l * nw, 0, W_final + l * batch * nw, batch, nw, st));
    W0 = W_final;
  }
  return run_engine(ws + z_off, ws + v_off, W0, L, B, eta, rule, O, W_final, &dm, ws, lay, st);
}

ipttt_status ipttt_additive_sums(const void* Z, const void* V, int64_t L, float* S, const ipttt_dims* dims,
                                 ipttt_stream stream) {
  LaunchScope scope;
  IPTTT_TRY(check_dims(dims, true));
  if (L < 0) return IPTTT_ERR_INVALID_ARG;
  // the contraction runs over a window of token rows: whole 16-token tensor-core steps
  if (dims->dtype == IPTTT_BF16 && L % 16) return IPTTT_ERR_INVALID_ARG;
  if (dims->batch > 0 && (L > (int64_t{1} << 31) / dims->batch || dims->d_ff * dims->batch > (int64_t{1} << 31)))
    return IPTTT_ERR_INVALID_ARG;
  if (dims->batch == 0) return IPTTT_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (L == 0) {
    IPTTT_TRY(check_ptrs({static_cast<const void*>(S)}));
    IPTTT_CUDA(cudaMemsetAsync(S, 0, sizeof(float) * dims->batch * dims->d_ff * dims->d, st));
    return IPTTT_OK;
  }
  IPTTT_TRY(check_ptrs({Z, V, static_cast<const void*>(S)}));
  const bool bf16 = dims->dtype == IPTTT_BF16;
  GemmProblem p;
  p.M = dims->d_ff;
  p.N = dims->d;
  p.K = L;
  p.nb1 = static_cast<int>(dims->batch);
  p.A = mat(Z, dims->batch * L, dims->d_ff, 1, 0, L);
  p.B = mat(V, dims->batch * L, dims->d, 1, 0, L);
  p.epi = EPI_STORE;
  p.kind = K_GROUP_SUM;
  p.out_bf16 = 0;
  p.D = out(S, dims->d, 0, dims->d_ff, 0, dims->batch * dims->d_ff);
  IPTTT_CUDA(gemm(p, bf16, st));
  return IPTTT_OK;
}

ipttt_status ipttt_weight_axpy(float* W, const float* S, float alpha, int64_t n, ipttt_stream stream) {
  LaunchScope scope;
  if (n < 0 || !std::isfinite(alpha)) return IPTTT_ERR_INVALID_ARG;
  if (n == 0) return IPTTT_OK;
  IPTTT_TRY(check_ptrs({static_cast<const void*>(W), static_cast<const void*>(S)}));
  IPTTT_CUDA(launch_axpy(W, S, alpha, n, static_cast<cudaStream_t>(stream)));
  return IPTTT_OK;
}

ipttt_status ipttt_sync_status(ipttt_stream stream) {
  const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return from_cuda(e);
  }
  int code = 0;
  if (read_clear_device_error(&code) != cudaSuccess) {
    cudaGetLastError();
    return IPTTT_ERR_CUDA;
  }
  return code ? IPTTT_ERR_TIMEOUT : IPTTT_OK;
}

ipttt_status ipttt_set_wait_limit(uint64_t ns) {
  IPTTT_TRY(check_device());
  IPTTT_CUDA(set_wait_soft_limit(ns));
  return IPTTT_OK;
}

ipttt_status ipttt_release(void) {
  std::lock_guard<std::mutex> g(g_pool_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  for (int dev = 0; dev < 64; ++dev) {
    if (!g_pools[dev].ptr) continue;
    cudaSetDevice(dev);
    cudaFree(g_pools[dev].ptr);
    g_pools[dev].ptr = nullptr;
    g_pools[dev].size = 0;
  }
  if (cur >= 0) cudaSetDevice(cur);
  cudaGetLastError();
  return IPTTT_OK;
}

int64_t ipttt_last_launch_count(void) { return t_launches; }

ipttt_status ipttt_set_pool_limit(size_t bytes) {
  g_pool_limit.store(bytes);
  return IPTTT_OK;
}

ipttt_status ipttt_kernel_timing(int32_t enable) {
  std::lock_guard<std::mutex> g(g_timing_mu);
  if (enable) {
    g_timing_pending.clear();
    for (int k = 0; k < K_COUNT; ++k) {
      g_timing_launches[k] = 0;
      g_timing_ms[k] = 0.0;
    }
  }
  g_timing_on = enable != 0;
  return IPTTT_OK;
}

ipttt_status ipttt_kernel_timing_read(int32_t kind, int64_t* launches, double* total_ms) {
  if (kind < 0 || kind >= K_COUNT || !launches || !total_ms) return IPTTT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_timing_mu);
  drain_timing_locked();
  *launches = g_timing_launches[kind];
  *total_ms = g_timing_ms[kind];
  return IPTTT_OK;
}

const char* ipttt_kernel_name(int32_t kind) { return kind_name(kind); }

const char* ipttt_status_string(ipttt_status s) {
  switch (s) {
    case IPTTT_OK:
      return "ok";
    case IPTTT_ERR_INVALID_ARG:
      return "invalid argument";
    case IPTTT_ERR_UNSUPPORTED:
      return "unsupported device (needs compute capability 10.3)";
    case IPTTT_ERR_ALLOC:
      return "scratch allocation failed";
    case IPTTT_ERR_LAUNCH:
      return "kernel launch failed";
    case IPTTT_ERR_TIMEOUT:
      return "a device-side wait ran out of time";
    case IPTTT_ERR_CUDA:
      return "CUDA runtime error";
  }
  return "unknown status";
}

int ipttt_version(void) { return IPTTT_VERSION; }

}  // extern "C"
