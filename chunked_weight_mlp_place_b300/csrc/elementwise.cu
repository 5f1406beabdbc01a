// Memory-bound kernels of the layer: the chunk-padded depthwise conv of the
// target builder, the residual / output epilogue of the apply step, the bf16
// copy of the fast weight and the group scan of the additive rule.  All are
// grid-stride loops over 16-byte vectors, sized to a multiple of the SM count.
#include "common.cuh"
#include "launch.h"

namespace ipttt {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work_items) {
  const int64_t per_wave = static_cast<int64_t>(device_sm_count()) * (2048 / kThreads);
  int64_t g = (work_items + kThreads - 1) / kThreads;
  if (g > per_wave * 4) g = per_wave * 4;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

// ---------------------------------------------------------------------- conv
// C[t, c] = sum_{j<4} w[c, j] * E[t+j, c], with E[t+j] read as zero once t+j
// leaves the chunk of B tokens holding t (In-Place TTT target, itsolotime §2.3).
// Sequences are whole chunks (L % B == 0), so chunks start at the multiples of
// B in the flattened rows.  One thread: 8 channels (16 bytes) x TT consecutive
// tokens, sliding a 4-row window; its position inside the chunk is computed
// once and stepped along the rows.  Several layers at once: output row r is
// row r % e_rows of E under layer r / e_rows's taps (e_rows a multiple of B
// and of TT, so an item stays in one layer and its taps past a layer's end
// are past a chunk end).
constexpr int kConvThreads = 128;  // three blocks per SM at up to 170 registers a thread
template <int TT>
__global__ void __launch_bounds__(kConvThreads, 3) conv_bf16x8_kernel(const __nv_bfloat16* __restrict__ E,
                                                               const float* __restrict__ w,
                                                               __nv_bfloat16* __restrict__ C, int64_t rows,
                                                               int64_t B, int64_t d, int64_t e_rows) {
  const int64_t cgroups = d / 8;
  const int64_t total = cgroups * ((rows + TT - 1) / TT);
  for (int64_t item = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; item < total;
       item += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tb = item / cgroups;
    const int64_t c0 = (item - tb * cgroups) * 8, r0 = tb * TT;
    const int64_t layer = r0 / e_rows, er0 = r0 - layer * e_rows;  // the item's layer and its first E row
    // window of rows r0 .. r0+TT+2, all loads in flight before any arithmetic
    uint4 raw[TT + 3];
#pragma unroll
    for (int i = 0; i < TT + 3; ++i)
      raw[i] = (r0 + i < rows && er0 + i < e_rows) ? *reinterpret_cast<const uint4*>(E + (er0 + i) * d + c0)
                                                   : make_uint4(0, 0, 0, 0);
    float wt[4][8];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 q = *reinterpret_cast<const float4*>(w + (layer * d + c0 + v) * 4);
      wt[0][v] = q.x;
      wt[1][v] = q.y;
      wt[2][v] = q.z;
      wt[3][v] = q.w;
    }
    int64_t pos = r0 % B;  // row r0's place in its chunk
#pragma unroll
    for (int i = 0; i < TT; ++i) {
      if (r0 + i >= rows) break;
      const int64_t room = B - pos;  // rows left in the chunk, counting this one
      float acc[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) acc[v] = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < room) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&raw[i + j])[v]);
            acc[2 * v] = fmaf(wt[j][2 * v], f.x, acc[2 * v]);
            acc[2 * v + 1] = fmaf(wt[j][2 * v + 1], f.y, acc[2 * v + 1]);
          }
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(C + (r0 + i) * d + c0) = o;
      if (++pos == B) pos = 0;
    }
  }
}

// Packed documents (launch_conv_varlen): the document holding row r, by
// binary search in cu (cu[0] = 0 <= r < cu[n_docs]).
__device__ __forceinline__ int64_t doc_of(const int64_t* cu, int64_t n_docs, int64_t r) {
  int64_t lo = 0, hi = n_docs;  // cu[lo] <= r < cu[hi]
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) / 2;
    if (cu[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

// conv_bf16x8_kernel over packed documents: chunks are counted from each
// document's first row, and a document's last row ends its last chunk.
template <int TT>
__global__ void __launch_bounds__(kConvThreads, 3) conv_bf16x8_varlen_kernel(
    const __nv_bfloat16* __restrict__ E, const float* __restrict__ w, __nv_bfloat16* __restrict__ C, int64_t rows,
    const int64_t* __restrict__ cu, int64_t n_docs, int64_t B, int64_t d) {
  const int64_t cgroups = d / 8;
  const int64_t total = cgroups * ((rows + TT - 1) / TT);
  for (int64_t item = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; item < total;
       item += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tb = item / cgroups;
    const int64_t c0 = (item - tb * cgroups) * 8, r0 = tb * TT;
    uint4 raw[TT + 3];
#pragma unroll
    for (int i = 0; i < TT + 3; ++i)
      raw[i] = (r0 + i < rows) ? *reinterpret_cast<const uint4*>(E + (r0 + i) * d + c0) : make_uint4(0, 0, 0, 0);
    float wt[4][8];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 q = *reinterpret_cast<const float4*>(w + (c0 + v) * 4);
      wt[0][v] = q.x;
      wt[1][v] = q.y;
      wt[2][v] = q.z;
      wt[3][v] = q.w;
    }
    int64_t doc = doc_of(cu, n_docs, r0);
    int64_t end = cu[doc + 1];
    int64_t pos = (r0 - cu[doc]) % B;  // row r0's place in its chunk
#pragma unroll
    for (int i = 0; i < TT; ++i) {
      const int64_t r = r0 + i;
      if (r >= rows) break;
      if (r == end) {  // the next document starts here
        ++doc;
        end = cu[doc + 1];
        pos = 0;
      }
      const int64_t room = min(B - pos, end - r);  // rows left in the chunk, counting this one
      float acc[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) acc[v] = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < room) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&raw[i + j])[v]);
            acc[2 * v] = fmaf(wt[j][2 * v], f.x, acc[2 * v]);
            acc[2 * v + 1] = fmaf(wt[j][2 * v + 1], f.y, acc[2 * v + 1]);
          }
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(C + r * d + c0) = o;
      if (++pos == B) pos = 0;
    }
  }
}

__global__ void __launch_bounds__(kThreads) conv_scalar_varlen_kernel(const float* __restrict__ E,
                                                                      const float* __restrict__ w,
                                                                      float* __restrict__ C, int64_t rows,
                                                                      const int64_t* __restrict__ cu, int64_t n_docs,
                                                                      int64_t B, int64_t d) {
  const int64_t total = rows * d;
  for (int64_t item = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; item < total;
       item += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t c = item % d, r = item / d;
    const int64_t doc = doc_of(cu, n_docs, r);
    const int64_t room = min(B - (r - cu[doc]) % B, cu[doc + 1] - r);
    float acc = 0.0f;
    for (int j = 0; j < 4 && j < room; ++j) acc = fmaf(w[c * 4 + j], E[(r + j) * d + c], acc);
    C[r * d + c] = acc;
  }
}

// Scalar-weight variant for fp32 mode with any d: one channel per thread
// (several layers as in conv_bf16x8_kernel).
__global__ void __launch_bounds__(kThreads) conv_kernel_scalar(const float* __restrict__ E,
                                                               const float* __restrict__ w, float* __restrict__ C,
                                                               int64_t rows, int64_t L, int64_t B, int64_t d,
                                                               int64_t e_rows) {
  const int64_t total = rows * d;
  for (int64_t item = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; item < total;
       item += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t c = item % d, r = item / d;
    const int64_t layer = r / e_rows, er = r - layer * e_rows;
    const int64_t t = er % L;
    const int64_t room = (t / B + 1) * B - t;
    float acc = 0.0f;
    for (int j = 0; j < 4 && j < room; ++j) acc = fmaf(w[(layer * d + c) * 4 + j], E[(er + j) * d + c], acc);
    C[r * d + c] = acc;
  }
}

// ------------------------------------------------------------------ residual
// Where row r = e*B + i of the chunk goes, and what it holds (ResidualArgs).
struct ResRow {
  int64_t orow;  // row of O and V
  float scale;   // of R
  bool valid;    // inside its document
};
__device__ __forceinline__ ResRow residual_row(const ResidualArgs& a, int64_t r) {
  const int64_t e = r / a.B, i = r % a.B;
  const int b1 = static_cast<int>(e % a.nb1), b2 = static_cast<int>(e / a.nb1);
  ResRow x;
  x.orow = a.o_y0 + (a.otab ? a.otab[b1] : b1 * a.o_ys1) + b2 * a.o_ys2 + i;
  x.valid = true;
  x.scale = 1.0f;
  if (a.lens) {
    const int64_t n = min(a.B, a.lens[b1] - a.o_y0);
    x.valid = i < n;
    x.scale = static_cast<float>(a.B) / static_cast<float>(n);
  }
  return x;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) residual_kernel(const ResidualArgs a) {
  const int64_t per_entry = a.B * a.d;
  const int64_t total = per_entry * a.nb1 * a.nb2;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx / a.d, c = idx % a.d;
    const ResRow x = residual_row(a, r);
    const float v = a.acc[idx];
    a.acc[idx] = 0.0f;
    if (x.valid) static_cast<T*>(a.O)[x.orow * a.d + c] = from_f32<T>(v);
    if (a.R) {
      float rv = 0.0f;
      if (x.valid) {
        const float t = to_f32<T>(static_cast<const T*>(a.V)[x.orow * a.d + c]);
        rv = x.scale * (a.r_from_v ? t : v - t);
      }
      static_cast<T*>(a.R)[idx] = from_f32<T>(rv);
    }
  }
}

// Vectorised bf16 variant (d % 8 == 0).  Thread (x, y): 8 columns c = 8*(128*y + x % 128)
// of kResRows consecutive rows starting at kResRows*(x / 128); all loads are
// issued before any store, so a thread keeps kResRows round trips in flight.
constexpr int kResRows = 4;
__global__ void __launch_bounds__(128) residual_kernel_bf16x8(const ResidualArgs a) {
  pdl_wait();
  pdl_trigger();
  const int64_t rows = a.B * a.nb1 * a.nb2;
  const int64_t c = (static_cast<int64_t>(blockIdx.y) * 128 + threadIdx.x) * 8;
  if (c >= a.d) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kResRows;
  float4 x[kResRows][2];
  uint4 vr[kResRows];
  ResRow rw[kResRows];
#pragma unroll
  for (int j = 0; j < kResRows; ++j) {
    const int64_t r = r0 + j;
    if (r >= rows) break;
    rw[j] = residual_row(a, r);
    uint32_t w8[8];
    ld_global_v8(a.acc + r * a.d + c, w8);  // the thread's 32 bytes of sums in one access
    x[j][0] = make_float4(__uint_as_float(w8[0]), __uint_as_float(w8[1]), __uint_as_float(w8[2]), __uint_as_float(w8[3]));
    x[j][1] = make_float4(__uint_as_float(w8[4]), __uint_as_float(w8[5]), __uint_as_float(w8[6]), __uint_as_float(w8[7]));
    if (a.R && rw[j].valid)
      vr[j] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.V) + rw[j].orow * a.d + c);
  }
#pragma unroll
  for (int j = 0; j < kResRows; ++j) {
    const int64_t r = r0 + j;
    if (r >= rows) break;
    const uint32_t zero8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    st_global_v8(a.acc + r * a.d + c, zero8);
    const float4 x0 = x[j][0], x1 = x[j][1];
    if (rw[j].valid) {
      uint4 o;
      o.x = pack_bf16x2(x0.x, x0.y);
      o.y = pack_bf16x2(x0.z, x0.w);
      o.z = pack_bf16x2(x1.x, x1.y);
      o.w = pack_bf16x2(x1.z, x1.w);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.O) + rw[j].orow * a.d + c) = o;
    }
    if (a.R) {
      float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (rw[j].valid) {
        const float acc8[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&vr[j]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 t = __bfloat1622float2(h[q]);
          y[2 * q] = rw[j].scale * (a.r_from_v ? t.x : acc8[2 * q] - t.x);
          y[2 * q + 1] = rw[j].scale * (a.r_from_v ? t.y : acc8[2 * q + 1] - t.y);
        }
      }
      uint4 rr;
      rr.x = pack_bf16x2(y[0], y[1]);
      rr.y = pack_bf16x2(y[2], y[3]);
      rr.z = pack_bf16x2(y[4], y[5]);
      rr.w = pack_bf16x2(y[6], y[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.R) + r * a.d + c) = rr;
    }
  }
}

// -------------------------------------------------------------- fast weight
// The fast weight as tile-major split planes (split_w / plane_index in
// common.cuh).  One work item: 8 consecutive columns of one row of one block
// (16 bytes of each plane); the planes' padding holds zeros.
struct PlaneItem {
  int64_t rbe;  // row block, counted over all entries
  int64_t e;    // entry
  int64_t r;    // row of the entry's matrix
  int64_t c;    // first of 8 columns
  int64_t cb;   // column block
  int row;      // row inside the block
  int half;     // 0: columns 0..7 of the block, 1: 8..15
};
__device__ __forceinline__ PlaneItem plane_item(int64_t idx, int64_t RB, int64_t CB) {
  PlaneItem it;
  it.half = static_cast<int>(idx & 1);
  it.row = static_cast<int>((idx >> 1) & (kPlaneRows - 1));
  const int64_t blk = idx >> 8;
  it.cb = blk % CB;
  it.rbe = blk / CB;
  it.e = it.rbe / RB;
  it.r = (it.rbe % RB) * kPlaneRows + it.row;
  it.c = it.cb * kPlaneCols + it.half * 8;
  return it;
}
__device__ __forceinline__ void store_split8(uint16_t* hi, uint16_t* lo, const PlaneItem& it, int64_t CB,
                                             const float (&w)[8]) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) split_w2(w[2 * q], w[2 * q + 1], h[q], l[q]);
  const int64_t at = plane_index(it.rbe, it.cb, CB, it.row, it.half * 8);
  *reinterpret_cast<uint4*>(hi + at) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo + at) = make_uint4(l[0], l[1], l[2], l[3]);
}

// W0[e or 0] (fp32, R x C row-major) -> the planes of `entries` entries.
__global__ void __launch_bounds__(kThreads) split_planes_kernel(const float* __restrict__ W0, int64_t w0_stride,
                                                                uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                                                                int64_t entries, int64_t R, int64_t C, int64_t RB,
                                                                int64_t CB) {
  const int64_t total = entries * RB * CB * kPlaneRows * 2;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const PlaneItem it = plane_item(idx, RB, CB);
    float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (it.r < R && it.c < C) {
      const float4* src = reinterpret_cast<const float4*>(W0 + it.e * w0_stride + it.r * C + it.c);
      const float4 a = src[0], b = src[1];
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
    store_split8(hi, lo, it, CB, w);
  }
}

// The planes of `entries` entries -> W (fp32, entries x R x C row-major).
__global__ void __launch_bounds__(kThreads) merge_planes_kernel(const uint16_t* __restrict__ hi,
                                                                const uint16_t* __restrict__ lo,
                                                                float* __restrict__ W, int64_t entries, int64_t R,
                                                                int64_t C, int64_t RB, int64_t CB) {
  const int64_t total = entries * RB * CB * kPlaneRows * 2;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const PlaneItem it = plane_item(idx, RB, CB);
    if (it.r >= R || it.c >= C) continue;
    const int64_t at = plane_index(it.rbe, it.cb, CB, it.row, it.half * 8);
    const uint4 h = *reinterpret_cast<const uint4*>(hi + at), l = *reinterpret_cast<const uint4*>(lo + at);
    const uint32_t hv[4] = {h.x, h.y, h.z, h.w}, lv[4] = {l.x, l.y, l.z, l.w};
    float w[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) join_w2(hv[q], lv[q], w[2 * q], w[2 * q + 1]);
    float4* dst = reinterpret_cast<float4*>(W + (it.e * R + it.r) * C + it.c);
    dst[0] = make_float4(w[0], w[1], w[2], w[3]);
    dst[1] = make_float4(w[4], w[5], w[6], w[7]);
  }
}

__global__ void __launch_bounds__(kThreads) copy_w_kernel(const float* __restrict__ W0, int64_t w0_stride,
                                                          float* __restrict__ W, int64_t batch, int64_t n) {
  const int64_t total = n * batch;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t s = idx / n, q = idx % n;
    W[idx] = W0[s * w0_stride + q];
  }
}

// Exclusive prefix over the G group sums of the additive rule (fp32 mode),
// turning each sum, in place, into the fast weight at the start of its group.
__global__ void __launch_bounds__(kThreads) group_scan_kernel(float* __restrict__ D, const float* __restrict__ W0,
                                                              int64_t w0_stride, float* __restrict__ Wf, int64_t G,
                                                              int64_t batch, int64_t n, float alpha) {
  const int64_t total = n * batch;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t s = idx / n, q = idx % n;
    float S = W0[s * w0_stride + q];
    for (int64_t g = 0; g < G; ++g) {
      const int64_t at = g * total + idx;
      const float t = D[at];
      D[at] = S;
      S = fmaf(alpha, t, S);
    }
    Wf[idx] = S;
  }
}

// The group scan of the additive rule writing the group starting weights as
// planes: S = W0; for g: state[g*batch + b] = S; S += alpha * D[g]; W_final = S.
// D is fp32 [G][batch][R][C] row-major; the planes have G*batch entries.
__global__ void __launch_bounds__(kThreads) group_scan_planes_kernel(const float* __restrict__ D,
                                                                     uint16_t* __restrict__ hi,
                                                                     uint16_t* __restrict__ lo,
                                                                     const float* __restrict__ W0, int64_t w0_stride,
                                                                     float* __restrict__ Wf, int64_t G, int64_t batch,
                                                                     int64_t R, int64_t C, int64_t RB, int64_t CB,
                                                                     float alpha) {
  const int64_t per_entry = RB * CB * kPlaneRows * 2;
  const int64_t total = batch * per_entry;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const PlaneItem it = plane_item(idx, RB, CB);  // it.e = sequence b
    const bool valid = it.r < R && it.c < C;
    float S[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) {
      const float4* w0 = reinterpret_cast<const float4*>(W0 + it.e * w0_stride + it.r * C + it.c);
      const float4 a = w0[0], b = w0[1];
      S[0] = a.x; S[1] = a.y; S[2] = a.z; S[3] = a.w;
      S[4] = b.x; S[5] = b.y; S[6] = b.z; S[7] = b.w;
    }
    for (int64_t g = 0; g < G; ++g) {
      PlaneItem ig = it;
      ig.rbe = (g * batch + it.e) * RB + it.rbe % RB;
      store_split8(hi, lo, ig, CB, S);
      if (valid) {
        const float4* t = reinterpret_cast<const float4*>(D + ((g * batch + it.e) * R + it.r) * C + it.c);
        const float4 a = t[0], b = t[1];
        S[0] = fmaf(alpha, a.x, S[0]); S[1] = fmaf(alpha, a.y, S[1]);
        S[2] = fmaf(alpha, a.z, S[2]); S[3] = fmaf(alpha, a.w, S[3]);
        S[4] = fmaf(alpha, b.x, S[4]); S[5] = fmaf(alpha, b.y, S[5]);
        S[6] = fmaf(alpha, b.z, S[6]); S[7] = fmaf(alpha, b.w, S[7]);
      }
    }
    if (valid) {
      float4* dst = reinterpret_cast<float4*>(Wf + (it.e * R + it.r) * C + it.c);
      dst[0] = make_float4(S[0], S[1], S[2], S[3]);
      dst[1] = make_float4(S[4], S[5], S[6], S[7]);
    }
  }
}

}  // namespace

cudaError_t launch_conv(const void* E, const float* conv_w, void* C, int64_t rows, int64_t L, int64_t B, int64_t d,
                        bool bf16, cudaStream_t stream, int64_t e_rows) {
  if (rows <= 0) return cudaSuccess;
  if (e_rows <= 0) e_rows = rows;
  if (rows % e_rows || e_rows % L || L % B) return cudaErrorInvalidValue;
  LaunchMark mark(K_CONV, stream);
  if (bf16) {
    if (d % 8 || e_rows % 8) return cudaErrorInvalidValue;
    constexpr int TT = 8;
    const int64_t items = (d / 8) * ((rows + TT - 1) / TT);
    const int64_t waves = static_cast<int64_t>(device_sm_count()) * 3;
    const int64_t blocks = std::min<int64_t>((items + kConvThreads - 1) / kConvThreads, waves * 4);
    conv_bf16x8_kernel<TT><<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), kConvThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(E), conv_w, static_cast<__nv_bfloat16*>(C), rows, B, d, e_rows);
  } else {
    conv_kernel_scalar<<<grid_for(rows * d), kThreads, 0, stream>>>(static_cast<const float*>(E), conv_w,
                                                                     static_cast<float*>(C), rows, L, B, d, e_rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_conv_varlen(const void* E, const float* conv_w, void* C, int64_t rows, const int64_t* cu,
                               int64_t n_docs, int64_t B, int64_t d, bool bf16, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (n_docs < 1 || B < 1 || !cu) return cudaErrorInvalidValue;
  LaunchMark mark(K_CONV, stream);
  if (bf16) {
    if (d % 8) return cudaErrorInvalidValue;
    constexpr int TT = 8;
    const int64_t items = (d / 8) * ((rows + TT - 1) / TT);
    const int64_t waves = static_cast<int64_t>(device_sm_count()) * 3;
    const int64_t blocks = std::min<int64_t>((items + kConvThreads - 1) / kConvThreads, waves * 4);
    conv_bf16x8_varlen_kernel<TT><<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), kConvThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(E), conv_w, static_cast<__nv_bfloat16*>(C), rows, cu, n_docs, B, d);
  } else {
    conv_scalar_varlen_kernel<<<grid_for(rows * d), kThreads, 0, stream>>>(
        static_cast<const float*>(E), conv_w, static_cast<float*>(C), rows, cu, n_docs, B, d);
  }
  return cudaGetLastError();
}

cudaError_t launch_residual(const ResidualArgs& a, bool bf16, cudaStream_t stream) {
  const int64_t total = a.B * a.d * a.nb1 * a.nb2;
  if (total <= 0) return cudaSuccess;
  LaunchMark mark(K_RESIDUAL, stream);
  if (bf16 && a.d % 8 == 0) {
    const int64_t rows = a.B * a.nb1 * a.nb2;
    const dim3 grid(static_cast<unsigned>((rows + kResRows - 1) / kResRows),
                    static_cast<unsigned>((a.d / 8 + 127) / 128));
    return launch_overlapped(residual_kernel_bf16x8, grid, dim3(128), 0, stream, 1, a);
  }
  else if (bf16)
    residual_kernel<__nv_bfloat16><<<grid_for(total), kThreads, 0, stream>>>(a);
  else
    residual_kernel<float><<<grid_for(total), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_split_planes(const float* W0, int64_t w0_stride, const Planes& w, int64_t R, int64_t C,
                                cudaStream_t stream) {
  if (C % 8) return cudaErrorInvalidValue;
  LaunchMark mark(K_WEIGHT, stream);
  split_planes_kernel<<<grid_for(w.entries * w.rb * w.cb * kPlaneRows * 2), kThreads, 0, stream>>>(
      W0, w0_stride, w.hi, w.lo, w.entries, R, C, w.rb, w.cb);
  return cudaGetLastError();
}

cudaError_t launch_merge_planes(const Planes& w, float* W, int64_t R, int64_t C, cudaStream_t stream) {
  if (C % 8) return cudaErrorInvalidValue;
  LaunchMark mark(K_WEIGHT, stream);
  merge_planes_kernel<<<grid_for(w.entries * w.rb * w.cb * kPlaneRows * 2), kThreads, 0, stream>>>(
      w.hi, w.lo, W, w.entries, R, C, w.rb, w.cb);
  return cudaGetLastError();
}

// dst[e*dst_stride + i] = act(src[e*src_stride + i]) for e < entries, i < n.
template <typename T>
__global__ void __launch_bounds__(kThreads) to_act_kernel(const float* __restrict__ src, int64_t src_stride,
                                                          T* __restrict__ dst, int64_t dst_stride, int64_t entries,
                                                          int64_t n) {
  const int64_t total = entries * n;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = idx / n, i = idx % n;
    dst[e * dst_stride + i] = from_f32<T>(src[e * src_stride + i]);
  }
}

cudaError_t launch_to_act(const float* src, int64_t src_stride, void* dst, int64_t dst_stride, int64_t entries,
                          int64_t n, bool bf16, cudaStream_t stream) {
  if (entries * n <= 0) return cudaSuccess;
  LaunchMark mark(K_WEIGHT, stream);
  if (bf16)
    to_act_kernel<__nv_bfloat16><<<grid_for(entries * n), kThreads, 0, stream>>>(
        src, src_stride, static_cast<__nv_bfloat16*>(dst), dst_stride, entries, n);
  else
    to_act_kernel<float><<<grid_for(entries * n), kThreads, 0, stream>>>(src, src_stride, static_cast<float*>(dst),
                                                                        dst_stride, entries, n);
  return cudaGetLastError();
}

// entries n x n bf16 identity matrices, 8 elements (16 bytes) a thread.
__global__ void __launch_bounds__(kThreads) eye_bf16_kernel(uint4* __restrict__ X, int64_t n, int64_t total8) {
  const uint32_t one = 0x3F80u;  // bf16 1.0
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e0 = (i * 8) % (n * n);  // first element of the 8 within its matrix
    const int64_t r = e0 / n, c0 = e0 % n;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (r >= c0 && r < c0 + 8) {
      const int q = static_cast<int>(r - c0);
      w[q / 2] = (q & 1) ? (one << 16) : one;
    }
    X[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_eye_bf16(void* X, int64_t n, int64_t entries, cudaStream_t stream) {
  if (n % 8) return cudaErrorInvalidValue;
  const int64_t total8 = entries * n * n / 8;
  if (total8 <= 0) return cudaSuccess;
  LaunchMark mark(K_WEIGHT, stream);
  eye_bf16_kernel<<<grid_for(total8), kThreads, 0, stream>>>(static_cast<uint4*>(X), n, total8);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(kThreads) axpy_kernel(float* __restrict__ W, const float* __restrict__ S,
                                                        float alpha, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    W[i] = fmaf(alpha, S[i], W[i]);
}

cudaError_t launch_axpy(float* W, const float* S, float alpha, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  LaunchMark mark(K_WEIGHT, stream);
  axpy_kernel<<<grid_for(n), kThreads, 0, stream>>>(W, S, alpha, n);
  return cudaGetLastError();
}

cudaError_t launch_copy_w(const float* W0, int64_t w0_stride, float* W, int64_t batch, int64_t n,
                          cudaStream_t stream) {
  LaunchMark mark(K_WEIGHT, stream);
  copy_w_kernel<<<grid_for(n * batch), kThreads, 0, stream>>>(W0, w0_stride, W, batch, n);
  return cudaGetLastError();
}

cudaError_t launch_group_scan(float* D, const float* W0, int64_t w0_stride, float* W_final, int64_t G,
                              int64_t batch, int64_t n, float alpha, cudaStream_t stream) {
  LaunchMark mark(K_SCAN, stream);
  group_scan_kernel<<<grid_for(n * batch), kThreads, 0, stream>>>(D, W0, w0_stride, W_final, G, batch, n, alpha);
  return cudaGetLastError();
}

cudaError_t launch_group_scan_planes(const float* D, const Planes& w, const float* W0, int64_t w0_stride,
                                     float* W_final, int64_t G, int64_t batch, int64_t R, int64_t C, float alpha,
                                     cudaStream_t stream) {
  if (C % 8) return cudaErrorInvalidValue;
  LaunchMark mark(K_SCAN, stream);
  group_scan_planes_kernel<<<grid_for(batch * w.rb * w.cb * kPlaneRows * 2), kThreads, 0, stream>>>(
      D, w.hi, w.lo, W0, w0_stride, W_final, G, batch, R, C, w.rb, w.cb, alpha);
  return cudaGetLastError();
}

}  // namespace ipttt
