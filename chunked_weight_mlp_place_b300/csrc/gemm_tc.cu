// Tensor-core back end of the batched GEMM (IPTTT_BF16 mode) for sm_103a.
//
// One persistent kernel template serves the four contractions of the layer:
//   gate   Z = SiLU(X W_g) * (X W_u)       A = X   (K-major)  B = [W_g | W_u] (MN-major)
//   proj   V = C P                          A = C   (K-major)  B = P           (MN-major)
//   apply  O_k = Z_k W_k  (split over K)    A = Z_k (K-major)  B = hi plane    (MN-major)
//   update W += alpha Z_k^T R_k             A = Z_k (MN-major) B = R_k         (MN-major)
// (the fast weight W is kept as split hi/lo 16-bit planes, common.cuh::split_w,
// stored tile-major in blocks of 128 rows x 16 columns, gemm.h::plane_index;
// the hi plane is the bf16 operand of the apply, read through a 3-D TMA map).
//
// Problems with more than one 128-row tile run on CTA pairs (clusters of 2,
// tcgen05 cta_group::2): one 256 x N MMA per pair, each CTA holding 128 rows
// of A and half of B's columns in its shared memory, so each SM streams half
// the B operand it would alone.
//
// Each CTA (one per SM) runs these warps:
//   warp 0      TMA producer: 128x64 A tiles and 64-wide B tiles into a ring of
//               shared-memory stages (128-byte swizzle; 32-byte for plane
//               blocks), completion on mbarriers;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128 or 256 per pair,
//               N=256, K=16) into a TMEM accumulator; tcgen05.commit frees each stage;
//   warps 2..   epilogue (4 warps; 8 for the update, two groups taking alternate
//               16-column chunks): tcgen05.ld the accumulator (one TMEM lane per
//               output row) and apply the fused epilogue.
// Two TMEM accumulators (2 x 256 columns) let the epilogue of one tile overlap
// the main loop of the next.  Work is either whole output tiles, strided over
// the CTAs or (dynamic order) taken from a device-wide counter as CTA pairs free
// up, or (split mode, for GEMMs with few tiles and a long K) an even share of
// the (tile, k-block) iteration space per CTA.
//
// The epilogues that move much data keep global accesses whole lines:
//   apply (split mode)  the epilogue stages the tile's 128 rows x 32 columns of
//                       fp32 partial sums and adds them into the fp32 sums in L2
//                       with one TMA reduce (the residual kernel then turns the
//                       sums into O and R = O - V);
//   bf16 STORE          32-column chunks staged in shared memory, one TMA store
//                       each;
//   update              no staging: a plane block's row is 32 contiguous bytes,
//                       so each thread reads and writes its row of the hi and lo
//                       planes directly and a warp moves 1 KB contiguous.
//
// Every mbarrier wait is capped (common.cuh); a CTA whose wait runs out flags
// the others, drains its in-flight TMA copies and MMAs, frees its TMEM and
// returns, leaving a code in the device error word.
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "launch.h"
#include "tmap.h"

namespace ipttt {

// Error word written by kernels whose capped waits ran out (0 = none); read
// and cleared through read_clear_device_error().  Codes: 1 = TMA-producer
// wait, 2 = MMA-issuer wait, 3 = epilogue wait, 4 = teardown drain.
__device__ int g_device_error = 0;
// Soft limit of the pipeline waits (ns): past it a CTA records a code in g_device_error and
// stops issuing MMAs and global writes, but completes its handshakes (common.cuh,
// mbar_wait_bounded).  Set from the host (ipttt_set_wait_limit); by default it equals the
// hard limit, so only a wait that hangs trips it.
__device__ unsigned long long g_wait_soft_ns = kWaitLimitNs;
// Next tile of a tensor-core GEMM launched in dynamic tile order (GemmProblem::dyn_tiles);
// zeroed on the stream before each such launch.
__device__ unsigned long long g_tile_ticket = 0;

namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;  // TMEM columns between the two accumulator buffers

template <int BN, int NB, int EPI, bool PAIR, bool OUT_BF16>
struct Cfg {
  static constexpr bool W_UPD = (EPI == EPI_AXPY);  // update epilogue on the tile-major planes
  static constexpr bool RED = (EPI == EPI_ACCUM);
  // update: two groups of four epilogue warps take alternate 16-column chunks
  static constexpr int EPI_WARPS = W_UPD ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int N_MMA = BN * NB;          // the B operands sit side by side: one MMA covers them
  static constexpr int M_MMA = PAIR ? 2 * BM : BM;
  static constexpr int B_COLS = PAIR ? N_MMA / 2 : N_MMA;  // B columns held by one CTA per stage
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_COLS * BK * 2;
  // bf16 STORE: the tile's 64-column chunks go out through TMA stores from shared memory
  static constexpr bool TMA_ST = (EPI == EPI_STORE) && OUT_BF16;
  // apply: two staging buffers of the tile's 128 rows x 32 fp32 for the TMA reductions; bf16
  // STORE: two of 128 rows x 64 bf16 for the TMA stores
  static constexpr int STG_BYTES = (RED || TMA_ST) ? BM * 32 * 4 : 0;
  static constexpr int STG_TOTAL = 2 * STG_BYTES;
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_TOTAL + BAR_BYTES;
  static_assert(N_MMA <= kAccStride && N_MMA % 16 == 0, "accumulator width");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(!PAIR || NB == 1 || BN == B_COLS, "pair: a second B operand is the peer's half");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(STAGE_BYTES % 1024 == 0 && STG_BYTES % 1024 == 0, "1024-byte aligned swizzle atoms");
  static_assert(!W_UPD || BM == kPlaneRows, "an update tile is one row of plane blocks");
};

struct Seg {
  int64_t tile;
  int kb0, kb1;
};

// Work decomposition shared by all roles (each walks it independently).
// With CTA pairs, a tile is a pair tile (2*BM rows): n_mt counts pair rows and
// the CTA of rank r in the pair owns rows 2*mt + r; the two CTAs of a cluster
// walk the same tiles and k-blocks.
struct Sched {
  int64_t n_mt, n_nt, tiles_per_batch, total_tiles;
  int kb_total;
  int group_m;
  int band_n;  // > 0: column-band order (GemmProblem::band_n)
  int tri;     // GemmProblem::tri
  int split;
  int pair;
  int64_t total_iters;
  // block-causal STORE: tiles whose every column lies in the chunk of its last row or later hold
  // no kept element and are skipped by every role
  int64_t mask_chunk, mask_m;
  int bn;

  __device__ void tile_coords(int64_t t, int& bi, int64_t& mt, int64_t& nt) const {
    bi = static_cast<int>(t / tiles_per_batch);
    const int64_t r = t % tiles_per_batch;
    if (band_n) {
      const int64_t bsz = static_cast<int64_t>(band_n) * n_mt;
      const int64_t first_n = (r / bsz) * band_n;
      const int64_t gn = min(static_cast<int64_t>(band_n), n_nt - first_n);
      const int64_t q = r % bsz;
      mt = q / gn;
      nt = first_n + q % gn;
      return;
    }
    const int64_t gsz = static_cast<int64_t>(group_m) * n_nt;
    const int64_t g = r / gsz;
    const int64_t first_m = g * group_m;
    const int64_t gm = min(static_cast<int64_t>(group_m), n_mt - first_m);
    const int64_t q = r % gsz;
    mt = first_m + q % gm;
    nt = q / gm;
  }
  // The k-blocks of tile t: all of K, or with a triangular A those that hold the tile's rows'
  // nonzeros (M = K).
  __device__ void kb_range(int64_t t, int& kb0, int& kb1) const {
    kb0 = 0;
    kb1 = kb_total;
    if (!tri) return;
    int bi;
    int64_t mt, nt;
    tile_coords(t, bi, mt, nt);
    const int64_t rows = pair ? 2 * BM : BM;
    const int64_t r0 = mt * rows, r1 = min(r0 + rows, mask_m);
    if (tri > 0)
      kb1 = static_cast<int>(min(static_cast<int64_t>(kb_total), (r1 + BK - 1) / BK));
    else
      kb0 = static_cast<int>(r0 / BK);
  }
  __device__ bool masked(int64_t t) const {
    if (!mask_chunk) return false;
    int bi;
    int64_t mt, nt;
    tile_coords(t, bi, mt, nt);
    const int64_t rows = pair ? 2 * BM : BM;
    const int64_t m_last = min(mask_m - 1, (mt + 1) * rows - 1);
    return nt * bn >= (m_last / mask_chunk) * mask_chunk;
  }
  // Split mode: worker c (a CTA, or a CTA pair) owns iterations [floor(c*T/G), floor((c+1)*T/G)).
  __device__ int64_t worker() const { return pair ? (blockIdx.x >> 1) : blockIdx.x; }
  __device__ int64_t workers() const { return pair ? (gridDim.x >> 1) : gridDim.x; }
};

struct SegIter {
  const Sched* s;
  int64_t t, it, it_end;
  __device__ void init(const Sched* sc) {
    s = sc;
    if (s->split) {
      const int64_t G = s->workers(), c = s->worker();
      it = s->total_iters * c / G;
      it_end = s->total_iters * (c + 1) / G;
    } else {
      t = s->worker();
    }
  }
  // MASK: the problem may carry a block-causal mask (STORE kernels only).
  template <bool MASK>
  __device__ bool next(Seg& g) {
    if (s->split) {
      if (it >= it_end) return false;
      g.tile = it / s->kb_total;
      g.kb0 = static_cast<int>(it % s->kb_total);
      const int64_t rem = it_end - it;
      g.kb1 = static_cast<int>(min(static_cast<int64_t>(s->kb_total), g.kb0 + rem));
      it += g.kb1 - g.kb0;
      return true;
    }
    if constexpr (MASK)
      while (t < s->total_tiles && s->masked(t)) t += s->workers();
    if (t >= s->total_tiles) return false;
    g.tile = t;
    s->kb_range(t, g.kb0, g.kb1);
    t += s->workers();
    return true;
  }
};

// Dynamic tile order (GemmProblem::dyn_tiles).  With the static order each CTA (pair) w
// takes tiles w, w + G, w + 2G, ...; over a long launch some pairs run ahead of others and
// the tiles in flight spread over more rows and columns than L2 holds.  Here one thread of
// the pair (the even CTA's producer) takes tile numbers from a global counter in increasing
// order, so the tiles in flight stay a window of consecutive ones, and publishes each number
// in a ring of kRing slots in the shared memory of both CTAs.  Every other role of both CTAs
// reads the same sequence from its own CTA's ring and releases each slot on the even CTA's
// barrier; a slot holding -1 ends the sequence.
constexpr int kRing = 8;

struct KParams {
  GemmProblem p;
  Sched s;
  unsigned long long* ticket;  // dynamic order: the tile counter (zero at launch)
};

// The tiles a role walks, in the static order (SegIter) or from the ring.
template <bool PAIR>
struct TileSrc {
  SegIter it;
  int64_t* ids;        // this CTA's ring (nullptr: static order)
  uint64_t* full;      // this CTA's ring barriers: one arrival per fill
  uint64_t* empty;     // the ring's release barriers (the even CTA's are the ones counted)
  uint32_t j;          // fills consumed

  __device__ void init(const KParams& kp, int64_t* ring_ids, uint64_t* ring_full, uint64_t* ring_empty) {
    it.init(&kp.s);
    ids = kp.p.dyn_tiles ? ring_ids : nullptr;
    full = ring_full;
    empty = ring_empty;
    j = 0;
  }
  // Consumer: the next tile.  Called by the lanes in `wmask` of one warp together (lane 0
  // among them); the warp gives up together if any lane's wait did.
  template <bool MASK>
  __device__ bool next(Seg& g, uint32_t wmask, volatile int* abort, int code, uint64_t soft_ns) {
    if (ids == nullptr) return it.template next<MASK>(g);
    const uint32_t sl = j % kRing, ph = (j / kRing) & 1;
    ++j;
    if (!__all_sync(wmask, mbar_wait_bounded<PAIR>(&full[sl], ph, abort, code, &g_device_error, soft_ns)))
      return false;
    const int64_t t = *reinterpret_cast<volatile int64_t*>(&ids[sl]);
    __syncwarp(wmask);
    if ((threadIdx.x & 31) == 0) {
      if constexpr (PAIR)
        mbar_arrive_cluster(mapa_shared(smem_u32(&empty[sl]), 0));
      else
        mbar_arrive(&empty[sl]);
    }
    if (t < 0) return false;
    g.tile = t;
    it.s->kb_range(t, g.kb0, g.kb1);
    return true;
  }
  // The even CTA's producer: its next tile.  Tile numbers are published one position ahead
  // of the producer's own walk, so the peer's producer knows its next tile while this one
  // still issues the current tile's copies.
  __device__ bool publish(uint32_t pos, unsigned long long* ticket, int64_t total, volatile int* abort,
                          uint64_t soft_ns) {
    const uint32_t sl = pos % kRing, ph = (pos / kRing) & 1;
    // every consumer of both CTAs has read the slot's previous number
    if (!mbar_wait_bounded<PAIR>(&empty[sl], ph ^ 1, abort, 1, &g_device_error, soft_ns)) return false;
    int64_t t = static_cast<int64_t>(atomicAdd(ticket, 1ull));
    if (t >= total) t = -1;
    ids[sl] = t;
    mbar_arrive(&full[sl]);
    if constexpr (PAIR) {
      st_shared_cluster_u64(mapa_shared(smem_u32(&ids[sl]), 1), static_cast<uint64_t>(t));
      mbar_arrive_cluster(mapa_shared(smem_u32(&full[sl]), 1));  // release: the store above first
    }
    return true;
  }
  __device__ bool fetch(Seg& g, unsigned long long* ticket, int64_t total, volatile int* abort, uint64_t soft_ns) {
    if (j == 0 && !publish(0, ticket, total, abort, soft_ns)) return false;
    const int64_t t = ids[j % kRing];  // published by this thread
    if (t >= 0 && !publish(j + 1, ticket, total, abort, soft_ns)) return false;
    ++j;
    if (t < 0) return false;
    g.tile = t;
    it.s->kb_range(t, g.kb0, g.kb1);
    return true;
  }
};

// Named barrier of a group of four epilogue warps (128 threads; group g uses
// barrier 1 + g); each warp re-converges first.
__device__ __forceinline__ void epi_barrier(int group) {
  __syncwarp();
  asm volatile("bar.sync %0, 128;" ::"r"(1 + group) : "memory");
}

__device__ __forceinline__ int64_t row_of(const Operand& o, int b1, int b2) { return entry_row(o, b1, b2); }
__device__ __forceinline__ int64_t row_of(const OutRef& o, int b1, int b2) { return entry_row(o, b1, b2); }

// Issue the TMA copies of one operand tile (extent EXT along M or N, BK along
// K).  With CTA pairs the completion is counted on the even CTA's barrier
// (cluster address bar_cl).
template <bool MN, int EXT, bool PAIR>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, uint32_t bar_cl,
                                             int64_t row0, int64_t i0, int64_t k0, uint64_t pol) {
  auto copy = [&](uint8_t* d, int x, int y) {
    if constexpr (PAIR)
      tma_load_2d_pair(d, map, bar_cl, x, y, pol);
    else
      tma_load_2d(d, map, bar, x, y, pol);
  };
  if constexpr (MN) {
#pragma unroll
    for (int j = 0; j < EXT / 64; ++j)
      copy(dst + j * (64 * BK * 2), static_cast<int>(i0 + 64 * j), static_cast<int>(row0 + k0));
  } else {
    copy(dst, static_cast<int>(k0), static_cast<int>(row0 + i0));
  }
}

// The B operand read from tile-major hi planes (an MN-major operand, K = rows of
// the weight).  The map views the planes as rows of 512 bytes (16 rows of a
// block), 8 to a block, blocks in storage order; one box of 4 such rows x EXT/16
// blocks lands as EXT/16 pieces of BK rows x 32 bytes, 2 KB apart, already in
// the 32-byte-swizzle layout (gemm.h::plane_index).
template <int EXT, bool PAIR>
__device__ __forceinline__ void load_plane_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                                   uint32_t bar_cl, int64_t rb0, int64_t cb, int64_t n0, int64_t k0,
                                                   uint64_t pol) {
  const int c1 = static_cast<int>((k0 % kPlaneRows) / 16);
  const int c2 = static_cast<int>((rb0 + k0 / kPlaneRows) * cb + n0 / kPlaneCols);
  if constexpr (PAIR)
    tma_load_3d_pair(dst, map, bar_cl, 0, c1, c2, pol);
  else
    tma_load_3d(dst, map, bar, 0, c1, c2, pol);
}

// Shared-memory descriptor of the k-th 16-wide K step of an operand tile.
//  K-major: rows of 128 bytes (64 K elements), 8-row groups 1024 bytes apart;
//           the K step advances the start by 32 bytes inside the swizzle atom.
//  MN-major: 64-element column blocks of 64 K rows (8 KB) side by side; 8-row
//           K groups 1024 bytes apart (SBO), column blocks 8 KB apart (LBO);
//           the K step advances the start by 16 rows = 2048 bytes.
//  plane (MN-major, 32-byte swizzle): 16-element column blocks of 64 K rows
//           (2 KB) side by side (LBO); 8-row K groups 256 bytes apart (SBO);
//           the K step advances the start by 16 rows = 512 bytes.
template <bool MN, bool PLANE = false>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kstep) {
  if constexpr (PLANE)
    return make_smem_desc(base + kstep * 512, BK * 32, 256, kLayoutSw32);
  else if constexpr (MN)
    return make_smem_desc_sw128(base + kstep * 2048, 64 * BK * 2, 1024);
  else
    return make_smem_desc_sw128(base + kstep * 32, 16, 1024);
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  return w;
}

// Output values of 32 consecutive columns n.. of row m (STORE: alpha * acc, the mask, the
// addend; GATE: SiLU(acc_g) * acc_u); columns past N are left as computed.
template <int EPI, bool OUT_BF16>
__device__ __forceinline__ void epilogue_values(const GemmProblem& p, int b1, int b2, int64_t m, int64_t n,
                                                const uint32_t (&r)[32], const uint32_t (&u)[32], float (&v)[32]) {
  const bool full = (n + 32 <= p.N);
  {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float a = __uint_as_float(r[i]);
      if constexpr (EPI == EPI_GATE)
        v[i] = silu_f(a) * __uint_as_float(u[i]);
      else
        v[i] = p.alpha * a;
    }
    if constexpr (EPI == EPI_STORE) {
      if (p.causal) {  // keep columns of earlier chunks than row m's
        const int64_t lim = (m / p.causal) * p.causal;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (n + i >= lim) v[i] = 0.0f;
      }
    }
    if constexpr (EPI == EPI_STORE) {
      if (p.add.ptr) {  // + the addend's elements (m, n .. n + 31)
        const int64_t arow = row_of(p.add, b1, b2) + m;
        if constexpr (OUT_BF16) {
          const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.add.ptr) + arow * p.add.ld + n;
          if (full) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 w = reinterpret_cast<const uint4*>(x)[q];
              const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                v[8 * q + 2 * i] += f.x;
                v[8 * q + 2 * i + 1] += f.y;
              }
            }
          } else {
            for (int i = 0; i < 32 && n + i < p.N; ++i) v[i] += __bfloat162float(x[i]);
          }
        } else {
          const float* x = static_cast<const float*>(p.add.ptr) + arow * p.add.ld + n;
          for (int i = 0; i < 32 && n + i < p.N; ++i) v[i] += x[i];
        }
      }
    }
  }
}

// Row-per-lane epilogue of 32 consecutive columns n.. of row m (gate, proj,
// group sums, and the rows of a tile that a TMA box cannot cover).
template <int EPI, bool OUT_BF16>
__device__ __forceinline__ void epilogue_chunk(const GemmProblem& p, int b1, int b2, int64_t m, int64_t n,
                                               const uint32_t (&r)[32], const uint32_t (&u)[32], uint64_t pol_d) {
  const bool full = (n + 32 <= p.N);
  if constexpr (EPI == EPI_STORE || EPI == EPI_GATE) {
    float v[32];
    epilogue_values<EPI, OUT_BF16>(p, b1, b2, m, n, r, u, v);
    const int64_t row = row_of(p.D, b1, b2) + m;
    if constexpr (OUT_BF16) {
      __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.D.ptr) + row * p.D.ld + n;
      if (full) {
#pragma unroll
        for (int q = 0; q < 4; ++q) st_global_v4_hint(reinterpret_cast<uint4*>(d) + q, pack8_bf16(v + 8 * q), pol_d);
      } else {
        for (int i = 0; i < 32 && n + i < p.N; ++i) d[i] = __float2bfloat16_rn(v[i]);
      }
    } else {
      float* d = static_cast<float*>(p.D.ptr) + row * p.D.ld + n;
      if (full) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<float4*>(d)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else {
        for (int i = 0; i < 32 && n + i < p.N; ++i) d[i] = v[i];
      }
    }
  } else if constexpr (EPI == EPI_ACCUM) {
    const int64_t row = row_of(p.D, b1, b2) + m;
    float* d = static_cast<float*>(p.D.ptr) + row * p.D.ld + n;
    if (full) {
#pragma unroll
      for (int q = 0; q < 8; ++q) red_add_v4(d + 4 * q, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    } else {
      for (int i = 0; i < 32 && n + i < p.N; ++i) red_add(d + i, __uint_as_float(r[i]));
    }
  }
}

template <int BN, int NB, bool A_MN, bool B_MN, int EPI, bool OUT_BF16, bool PAIR, bool B_PL>
__global__ void __launch_bounds__(Cfg<BN, NB, EPI, PAIR, OUT_BF16>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ KParams kp) {
  using C = Cfg<BN, NB, EPI, PAIR, OUT_BF16>;
  static_assert(!PAIR || B_MN, "pairs split an MN-major B operand by columns");
  static_assert(!B_PL || (B_MN && NB == 1), "a plane B operand is MN-major and single");
  static_assert(B_PL ? C::B_COLS % kPlaneCols == 0 : C::B_COLS % 64 == 0,
                "B columns per CTA: whole swizzle atoms (64 columns, or 16 for plane blocks)");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint8_t* stages = smem;
  uint8_t* stg = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + C::STG_TOTAL);
  uint64_t* full_bar = bars;                        // [STAGES]
  uint64_t* empty_bar = bars + C::STAGES;           // [STAGES]
  uint64_t* tfull_bar = bars + 2 * C::STAGES;       // [2]
  uint64_t* tempty_bar = bars + 2 * C::STAGES + 2;  // [2]
  uint64_t* drain_bar = bars + 2 * C::STAGES + 4;   // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* ring_full = bars + 2 * C::STAGES + 6;  // [kRing] dynamic tile order
  uint64_t* ring_empty = ring_full + kRing;        // [kRing]
  int64_t* ring_ids = reinterpret_cast<int64_t*>(ring_empty + kRing);
  static_assert((2 * C::STAGES + 6 + 3 * kRing) * 8 <= C::BAR_BYTES, "barrier area");

  const GemmProblem& p = kp.p;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // CTA pairs: rank 0 issues the pair's MMAs; both CTAs load their own A rows
  // and their half of B, and run their own epilogue on their 128 TMEM lanes.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const bool mma_cta = (rank == 0);

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < C::STAGES; ++i) {
        mbar_init(&full_bar[i], 1);
        mbar_init(&empty_bar[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&tfull_bar[i], 1);
        mbar_init(&tempty_bar[i], (PAIR ? 2 : 1) * C::EPI_WARPS);  // one arrival per epilogue warp (of both CTAs)
      }
      mbar_init(drain_bar, 1);
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&ring_full[i], 1);
        // consumers of a fill: the MMA issuer and the epilogue warps of the even CTA, and
        // with pairs the producer and epilogue warps of the odd one
        mbar_init(&ring_empty[i], PAIR ? 2 + 2 * C::EPI_WARPS : 1 + C::EPI_WARPS);
      }
      *abort_flag = 0;
      fence_mbarrier_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if constexpr (NB == 2) tma_prefetch_desc(&tmB2);
      if (C::RED || (C::TMA_ST && p.D.rows > 0)) tma_prefetch_desc(&tmD);
    }
    __syncwarp();
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // The peer signals this CTA's barriers: both CTAs' barriers exist before anyone proceeds.
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touched only this CTA's shared memory and TMEM: it overlaps
  // the previous kernel's tail.  Global memory from here on.
  pdl_wait();
  pdl_trigger();
  const uint64_t soft_ns = g_wait_soft_ns;

  SegIter iter;
  iter.init(&kp.s);
  TileSrc<PAIR> src;
  src.init(kp, ring_ids, ring_full, ring_empty);
  Seg seg;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kc = 0, pst = 0, pph = 0;  // k-blocks issued; stage and phase of the next one
      uint32_t issued_mask = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(p.l2_a), pol_b = l2_policy(p.l2_b);
      const bool fetcher = p.dyn_tiles && mma_cta;
      while (ok && (fetcher ? src.fetch(seg, kp.ticket, kp.s.total_tiles, abort_flag, soft_ns)
                            : src.template next<EPI == EPI_STORE>(seg, 1u, abort_flag, 1, soft_ns))) {
        int bi;
        int64_t mt, nt;
        kp.s.tile_coords(seg.tile, bi, mt, nt);
        if constexpr (PAIR) mt = 2 * mt + rank;
        const int b1 = bi % p.nb1, b2 = bi / p.nb1;
        const int64_t ra = row_of(p.A, b1, b2), rb = row_of(p.B, b1, b2), rb2 = row_of(p.B2, b1, b2);
        const int64_t pb0 = (b1 * p.w.es1 + b2 * p.w.es2) * p.w.rb;  // plane B operand: first row block
        for (int kb = seg.kb0; kb < seg.kb1; ++kb, ++kc) {
          const uint32_t st = pst, ph = pph;
          if (++pst == C::STAGES) {
            pst = 0;
            pph ^= 1;
          }
          if (!mbar_wait_bounded(&empty_bar[st], ph ^ 1, abort_flag, 1, &g_device_error, soft_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + st * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          // with pairs, the MMA CTA's full barrier counts both CTAs' bytes
          const uint32_t bar_cl = PAIR ? mapa_shared(smem_u32(&full_bar[st]), 0) : 0u;
          if (mma_cta) mbar_arrive_expect_tx(&full_bar[st], (PAIR ? 2 : 1) * C::STAGE_BYTES);
          issued_mask |= 1u << st;
          const int64_t k0 = static_cast<int64_t>(kb) * BK;
          load_operand<A_MN, BM, PAIR>(sa, &tmA, &full_bar[st], bar_cl, ra, mt * BM, k0, pol_a);
          if constexpr (B_PL) {
            load_plane_operand<C::B_COLS, PAIR>(sb, &tmB, &full_bar[st], bar_cl, pb0, p.w.cb,
                                                nt * BN + rank * C::B_COLS, k0, pol_b);
          } else if constexpr (PAIR && NB == 2) {
            // the even CTA holds the first B operand, its peer the second
            if (rank == 0)
              load_operand<B_MN, BN, PAIR>(sb, &tmB, &full_bar[st], bar_cl, rb, nt * BN, k0, pol_b);
            else
              load_operand<B_MN, BN, PAIR>(sb, &tmB2, &full_bar[st], bar_cl, rb2, nt * BN, k0, pol_b);
          } else if constexpr (PAIR) {
            load_operand<B_MN, C::B_COLS, PAIR>(sb, &tmB, &full_bar[st], bar_cl, rb, nt * BN + rank * C::B_COLS, k0,
                                                pol_b);
          } else {
            load_operand<B_MN, BN, PAIR>(sb, &tmB, &full_bar[st], 0u, rb, nt * BN, k0, pol_b);
            if constexpr (NB == 2)
              load_operand<B_MN, BN, PAIR>(sb + BN * BK * 2, &tmB2, &full_bar[st], 0u, rb2, nt * BN, k0, pol_b);
          }
        }
      }
      // This CTA's share of the next kernel's operand, into L2 (see GemmProblem::pf_ptr).
      if (ok && p.pf_ptr) {
        const int64_t total = p.pf_bytes * p.pf_count;
        const int64_t lo = (total * blockIdx.x / gridDim.x) & ~int64_t{255};
        const int64_t hi = (blockIdx.x + 1 == gridDim.x) ? total : ((total * (blockIdx.x + 1) / gridDim.x) & ~int64_t{255});
        for (int64_t off = lo; off < hi;) {
          const int64_t e = off / p.pf_bytes, in = off - e * p.pf_bytes;
          const int64_t n = min(min(hi - off, p.pf_bytes - in), int64_t{65536});
          prefetch_l2_bulk(static_cast<const uint8_t*>(p.pf_ptr) + e * p.pf_stride + in, static_cast<uint32_t>(n));
          off += n;
        }
      }
      // Teardown: every copy issued here must have landed before the CTA's
      // shared memory is released (matters only after an abort).  With pairs
      // the copies complete on the MMA CTA's barrier; this CTA learns that its
      // stages were consumed from its empty barriers.
      for (uint32_t st = 0; st < C::STAGES; ++st) {
        if (!(issued_mask & (1u << st))) continue;
        const uint32_t f = (kc - 1 - st) / C::STAGES;  // last fill of stage st
        if (PAIR && !mma_cta)
          mbar_wait_drain(&empty_bar[st], f & 1, 4, &g_device_error);
        else
          mbar_wait_drain(&full_bar[st], f & 1, 4, &g_device_error);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole role runs on one thread: tcgen05.mma and tcgen05.commit are
    // issued by a single thread, and a lone waiter cannot diverge from itself.
    if (lane == 0 && mma_cta) {
      constexpr uint32_t idesc = make_idesc_bf16(C::M_MMA, C::N_MMA, A_MN, B_MN);
      // Descriptors of stage 0, k step 0.  A stage or a k step moves only the start-address field
      // (bits 0-13, address >> 4; shared addresses stay below 256 KB, so the add never carries out).
      const uint32_t s0 = smem_u32(stages);
      const uint64_t a0 = operand_desc<A_MN>(s0, 0), b0 = operand_desc<B_MN, B_PL>(s0 + C::A_BYTES, 0);
      constexpr uint32_t A_KSTEP = (A_MN ? 2048u : 32u) >> 4;
      constexpr uint32_t B_KSTEP = (B_PL ? 512u : (B_MN ? 2048u : 32u)) >> 4;
      const int kb_full = static_cast<int>(p.K / BK);  // k-blocks with all BK/16 steps inside K
      uint32_t ls = 0, st = 0, ph = 0;  // tiles done; stage and phase of the next k-block
      bool ok = true;
      while (ok && src.template next<EPI == EPI_STORE>(seg, 1u, abort_flag, 2, soft_ns)) {
        const uint32_t acc = ls & 1, aph = (ls >> 1) & 1;
        if (!mbar_wait_bounded(&tempty_bar[acc], aph ^ 1, abort_flag, 2, &g_device_error, soft_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kAccStride;
        for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
          if (!mbar_wait_bounded(&full_bar[st], ph, abort_flag, 2, &g_device_error, soft_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (st * C::STAGE_BYTES) >> 4;
          const uint64_t ad = a0 + soff, bd = b0 + soff;
          const uint32_t first = (kb == seg.kb0) ? 0u : 1u;
          if (*abort_flag) {
            // aborted: no more MMAs; the commit below still frees the stage
          } else if (kb < kb_full) {
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) {
              if constexpr (PAIR)
                umma_bf16_pair(d_tmem, ad + ks * A_KSTEP, bd + ks * B_KSTEP, idesc, ks ? 1u : first);
              else
                umma_bf16(d_tmem, ad + ks * A_KSTEP, bd + ks * B_KSTEP, idesc, ks ? 1u : first);
            }
          } else {
            const int ksteps = static_cast<int>((p.K - static_cast<int64_t>(kb) * BK + 15) / 16);
            for (int ks = 0; ks < ksteps; ++ks) {
              if constexpr (PAIR)
                umma_bf16_pair(d_tmem, ad + ks * A_KSTEP, bd + ks * B_KSTEP, idesc, ks ? 1u : first);
              else
                umma_bf16(d_tmem, ad + ks * A_KSTEP, bd + ks * B_KSTEP, idesc, ks ? 1u : first);
            }
          }
          if constexpr (PAIR)
            umma_commit_pair_both(&empty_bar[st]);
          else
            umma_commit(&empty_bar[st]);
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair_both(&tfull_bar[acc]);
        else
          umma_commit(&tfull_bar[acc]);
        ++ls;
      }
      // Teardown: wait for every MMA issued here before TMEM is freed.
      if constexpr (PAIR)
        umma_commit_pair_both(drain_bar);
      else
        umma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, 4, &g_device_error);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp % 4;          // TMEM lanes 32*quarter .. +31 belong to this warp
    const int trow = quarter * 32 + lane;  // row of the tile this thread finishes
    const bool issuer = (trow == 0);       // apply: issues the tile-wide TMA reductions
    // A warp whose wait ran out (failed) skips the waits and the work from then on but
    // still walks every tile and chunk, so the apply's named barriers always fill up.
    bool failed = false;
    uint32_t ls = 0;
    if constexpr (C::W_UPD) {
      // ---- update: W = W + alpha * acc on the tile-major split planes (split_w).  A tile's
      // 128 rows are one row of plane blocks and its 16-column chunks are blocks, so thread
      // `trow` owns 32 contiguous bytes of each plane per chunk and a warp reads and writes
      // 1 KB contiguous.  Two groups of four warps take alternate chunks (group g the chunks
      // c = g, g + 2, ...).  Each group loads the planes of its next three chunks ahead,
      // across tile boundaries, and the accumulator columns of its next chunk from TMEM.
      constexpr int WC = kPlaneCols;
      constexpr int NCH = BN / WC;
      constexpr int GCH = NCH / 2;  // chunks per group and tile
      static_assert(GCH % 4 == 0, "each group's chunks come in fours");
      const int group = (warp - 2) / 4;
      struct TileW {
        uint16_t* hi;  // this thread's row of the tile's first chunk block (nullptr: no rows here)
        uint16_t* lo;
        int64_t cb0;   // the tile's first column block
      };
      auto tile_w = [&](const Seg& t) {
        TileW x{nullptr, nullptr, 0};
        int bi;
        int64_t mt, nt;
        kp.s.tile_coords(t.tile, bi, mt, nt);
        if constexpr (PAIR) mt = 2 * mt + rank;
        if (mt * BM >= p.M) return x;  // a pair's second tile past the last row block
        const int b1 = bi % p.nb1, b2 = bi / p.nb1;
        const int64_t rbk = (b1 * p.w.es1 + b2 * p.w.es2) * p.w.rb + mt;
        x.cb0 = nt * (BN / WC);
        const int64_t off = plane_index(rbk, x.cb0, p.w.cb, 0, 0) + trow * kPlaneCols;
        x.hi = p.w.hi + off;
        x.lo = p.w.lo + off;
        return x;
      };
      const int sw = (trow >> 2) & 1;  // this row's 16-byte halves trade places (plane_index)
      // planes of the chunks in flight, indexed by chunk % 4: each row's 32 bytes as stored
      // (halves swapped where sw is set), one 32-byte load per plane
      uint32_t wh[4][8], wl[4][8];
      const uint64_t pol_hi = l2_policy(p.planes_l2 ? L2_EVICT_LAST : L2_NORMAL);
      const uint64_t pol_lo = l2_policy(p.planes_l2 ? L2_EVICT_FIRST : L2_NORMAL);
      auto wload = [&](const TileW& t, int c, uint32_t (&h)[8], uint32_t (&l)[8]) {
        if (t.hi == nullptr || t.cb0 + c >= p.w.cb) return;
        ld_global_v8_hint(t.hi + static_cast<int64_t>(c) * kPlaneBlock, h, pol_hi);
        ld_global_v8_hint(t.lo + static_cast<int64_t>(c) * kPlaneBlock, l, pol_lo);
      };
      SegIter ahead = iter;
      Seg cur, nxt;
      bool have = ahead.next<EPI == EPI_STORE>(cur);
      TileW tw = have ? tile_w(cur) : TileW{nullptr, nullptr, 0};
      wload(tw, group, wh[0], wl[0]);
      wload(tw, group + 2, wh[1], wl[1]);
      wload(tw, group + 4, wh[2], wl[2]);
      while (have) {
        const bool have_next = ahead.next<EPI == EPI_STORE>(nxt);
        const TileW tn = have_next ? tile_w(nxt) : TileW{nullptr, nullptr, 0};
        const uint32_t acc = ls & 1, aph = (ls >> 1) & 1;
        if (!failed)
          failed = !__all_sync(0xffffffffu, mbar_wait_bounded(&tfull_bar[acc], aph, abort_flag, 3, &g_device_error, soft_ns));
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccStride;
        uint32_t ra[WC], rb[WC];
        tmem_ld_32x32b_x16(tbase + group * WC, ra);
#pragma unroll 1
        for (int j4 = 0; j4 < GCH; j4 += 4) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j4 + u, c = group + 2 * j;
            uint32_t(&r)[WC] = (u & 1) ? rb : ra;
            uint32_t(&rn)[WC] = (u & 1) ? ra : rb;
            tmem_wait_ld(r);
            if (j + 1 < GCH) tmem_ld_32x32b_x16(tbase + (c + 2) * WC, rn);
            // columns 2q, 2q+1 sit in stored word q ^ 4*sw
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              hw[q] = sw ? wh[u][q + 4] : wh[u][q];
              hw[q + 4] = sw ? wh[u][q] : wh[u][q + 4];
              lw[q] = sw ? wl[u][q + 4] : wl[u][q];
              lw[q + 4] = sw ? wl[u][q] : wl[u][q + 4];
            }
            // the planes of the group's chunk j + 3 go into the registers its chunk j - 1 used
            if (j + 3 < GCH)
              wload(tw, c + 6, wh[(u + 3) & 3], wl[(u + 3) & 3]);
            else
              wload(tn, c + 6 - NCH, wh[(u + 3) & 3], wl[(u + 3) & 3]);
            uint32_t ho[8], lo[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float w0, w1;
              join_w2(hw[q], lw[q], w0, w1);
              split_w2(fmaf(p.alpha, __uint_as_float(r[2 * q]), w0), fmaf(p.alpha, __uint_as_float(r[2 * q + 1]), w1),
                       ho[q], lo[q]);
            }
            if (!failed && !*abort_flag && tw.hi != nullptr && tw.cb0 + c < p.w.cb) {
              // whole 32-byte rows, halves back in stored order
              uint32_t hs[8], ls8[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                hs[q] = sw ? ho[q + 4] : ho[q];
                hs[q + 4] = sw ? ho[q] : ho[q + 4];
                ls8[q] = sw ? lo[q + 4] : lo[q];
                ls8[q + 4] = sw ? lo[q] : lo[q + 4];
              }
              st_global_v8_hint(tw.hi + static_cast<int64_t>(c) * kPlaneBlock, hs, pol_hi);
              st_global_v8_hint(tw.lo + static_cast<int64_t>(c) * kPlaneBlock, ls8, pol_lo);
            }
          }
        }
        tmem_wait_ld();
        // Hand the accumulator back to the MMA issuer (the even CTA's, with pairs).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
          else
            mbar_arrive(&tempty_bar[acc]);
        }
        ++ls;
        have = have_next;
        tw = tn;
      }
    } else {
      uint32_t sc = 0;
      const uint64_t pol_d = l2_policy(p.l2_d);  // the output's lines
      while (src.template next<EPI == EPI_STORE>(seg, 0xffffffffu, abort_flag, 3, soft_ns)) {
        const uint32_t acc = ls & 1, aph = (ls >> 1) & 1;
        // Every lane waits (each needs the acquire); the warp gives up together if any lane did.
        if (!failed)
          failed = !__all_sync(0xffffffffu, mbar_wait_bounded(&tfull_bar[acc], aph, abort_flag, 3, &g_device_error, soft_ns));
        tc_fence_after();
        int bi;
        int64_t mt, nt;
        kp.s.tile_coords(seg.tile, bi, mt, nt);
        if constexpr (PAIR) mt = 2 * mt + rank;
        const int b1 = bi % p.nb1, b2 = bi / p.nb1;
        const int64_t m = mt * BM + trow;
        // the tile goes through tile-wide TMA boxes only if all its 128 rows are rows of the problem
        const bool box_rows = (mt * BM + BM <= p.M);
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccStride;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32], u[32];
          tmem_ld_32x32b_x32(tbase + c * 32, r);
          if constexpr (EPI == EPI_GATE) tmem_ld_32x32b_x32(tbase + BN + c * 32, u);
          tmem_wait_ld();
          const int64_t n = nt * BN + c * 32;
          if (n >= p.N) continue;
          if constexpr (C::TMA_ST) {
            if (box_rows && p.D.rows > 0) {
              // 64-byte swizzle: 16-byte chunk j of row t sits at chunk j ^ ((t / 2) % 4)
              uint8_t* sbuf = stg + (sc & 1) * C::STG_BYTES;
              uint4* srow = reinterpret_cast<uint4*>(sbuf + trow * 64);
              if (!failed) {
                float v[32];
                epilogue_values<EPI, OUT_BF16>(p, b1, b2, m, n, r, u, v);
#pragma unroll
                for (int j = 0; j < 4; ++j) srow[j ^ ((trow >> 1) & 3)] = pack8_bf16(v + 8 * j);
              }
              fence_proxy_async_shared();
              if (issuer) bulk_wait_group_read<0>();  // the other buffer, written next chunk, is free
              epi_barrier(0);
              if (issuer && !failed && !*abort_flag) {
                tma_store_2d(&tmD, sbuf, static_cast<int>(n), static_cast<int>(row_of(p.D, b1, b2) + mt * BM));
                bulk_commit_group();
              }
              ++sc;
              continue;
            }
          }
          if constexpr (C::RED) {
            if (box_rows) {
              // 128-byte swizzle: 16-byte chunk j of row t sits at chunk j ^ (t % 8)
              uint8_t* sbuf = stg + (sc & 1) * C::STG_BYTES;
              float4* srow = reinterpret_cast<float4*>(sbuf + trow * 128);
              if (!failed) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  srow[j ^ (trow & 7)] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                     __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
              }
              fence_proxy_async_shared();
              if (issuer) bulk_wait_group_read<0>();  // the other buffer, written next chunk, is free
              epi_barrier(0);
              if (issuer && !failed && !*abort_flag) {
                tma_reduce_add_2d(&tmD, sbuf, static_cast<int>(n), static_cast<int>(row_of(p.D, b1, b2) + mt * BM));
                bulk_commit_group();
              }
              ++sc;
              continue;
            }
          }
          if (m < p.M && !failed && !*abort_flag) epilogue_chunk<EPI, OUT_BF16>(p, b1, b2, m, n, r, u, pol_d);
        }
        // Hand the accumulator back to the MMA issuer (the even CTA's, with pairs).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
          else
            mbar_arrive(&tempty_bar[acc]);
        }
        ++ls;
      }
      // Every bulk reduction or store has completed before the CTA exits.
      if constexpr (C::RED || C::TMA_ST) {
        if (issuer) bulk_wait_group<0>();
        __syncwarp();
      }
    }
  }

  // Roles that ran on one lane re-converge their warp first: the CTA barrier
  // below is a warp-aligned instruction, and TMEM may only be freed once every
  // warp (the epilogue's TMEM loads included) has reached it.  With pairs, the
  // barrier spans the cluster: the peer's last arrivals on this CTA's barriers
  // and the even CTA's last MMAs into the peer's TMEM are done before either frees.
  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();
  else
    __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D tensor map of a row-major matrix (rows x cols, row stride ld elements);
// the box is box_cols x box_rows and its rows are box_cols * element size
// bytes wide, swizzled with the matching pattern (32, 64 or 128 bytes).
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool fp32, int box_cols,
              int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || !ptr || rows <= 0 || cols <= 0) return false;
  const int esz = fp32 ? 4 : 2;
  const int row_bytes = box_cols * esz;
  CUtensorMapSwizzle sw;
  if (row_bytes == 128)
    sw = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (row_bytes == 64)
    sw = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (row_bytes == 32)
    sw = CU_TENSOR_MAP_SWIZZLE_32B;
  else
    return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map of tile-major hi planes read as an MN-major operand: dims (256
// elements = 512 bytes, 8 rows of 512 bytes per block, blocks of all entries);
// a box is BK/16 rows x box_cols/16 blocks, no swizzle (the planes are stored
// swizzled).
bool make_plane_map(CUtensorMap* map, const Planes& w, int box_cols) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || !w.hi || w.rb <= 0 || w.cb <= 0 || w.entries <= 0) return false;
  constexpr int kRow = 256;  // elements per 512-byte row
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(kPlaneBlock / kRow),
                        static_cast<cuuint64_t>(w.cb * w.rb * w.entries)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRow) * 2, static_cast<cuuint64_t>(kPlaneBlock) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kRow), static_cast<cuuint32_t>(BK * kPlaneCols / kRow),
                       static_cast<cuuint32_t>(box_cols / kPlaneCols)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w.hi, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int NB, bool A_MN, bool B_MN, int EPI, bool OUT_BF16, bool PAIR, bool B_PL>
static cudaError_t run(const GemmProblem& p, cudaStream_t stream) {
  using C = Cfg<BN, NB, EPI, PAIR, OUT_BF16>;
  auto kern = tc_gemm_kernel<BN, NB, A_MN, B_MN, EPI, OUT_BF16, PAIR, B_PL>;
  static std::mutex mu;
  static uint64_t attr_done = 0;  // bit per device: shared-memory size attribute set
  static int max_workers[64] = {0};  // co-resident CTAs (or CTA pairs) per device
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!(attr_done & (1ull << dev))) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      int n = device_sm_count();
      if (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (n / 2));
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        n = clusters;
      }
      if (n <= 0) return cudaErrorInvalidConfiguration;
      max_workers[dev] = n;
      attr_done |= 1ull << dev;
    }
  }

  // Operand boxes: 64 K-elements (128 bytes) wide; K-major boxes span the
  // tile's rows, MN-major boxes are 64 K-rows of 64 columns.
  CUtensorMap mA, mB, mB2, mD;
  if (!make_map(&mA, p.A.ptr, p.A.rows, p.A.cols, p.A.ld, false, 64, A_MN ? 64 : BM)) return cudaErrorInvalidValue;
  if (B_PL) {
    if (!make_plane_map(&mB, p.w, C::B_COLS)) return cudaErrorInvalidValue;
  } else if (!make_map(&mB, p.B.ptr, p.B.rows, p.B.cols, p.B.ld, false, 64, B_MN ? 64 : BN)) {
    return cudaErrorInvalidValue;
  }
  mB2 = mD = mB;
  if (NB == 2 && !make_map(&mB2, p.B2.ptr, p.B2.rows, p.B2.cols, p.B2.ld, false, 64, B_MN ? 64 : BN))
    return cudaErrorInvalidValue;
  if (C::RED && !make_map(&mD, p.D.ptr, p.D.rows, p.N, p.D.ld, true, 32, BM)) return cudaErrorInvalidValue;
  // bf16 STORE with the output's rows known: 32-column boxes (64 bytes a row) for the TMA stores
  if (C::TMA_ST && p.D.rows > 0 && !make_map(&mD, p.D.ptr, p.D.rows, p.N, p.D.ld, false, 32, BM))
    return cudaErrorInvalidValue;
  if (C::W_UPD && (!p.w.hi || !p.w.lo || p.w.rb <= 0 || p.w.cb <= 0)) return cudaErrorInvalidValue;

  KParams kp;
  kp.p = p;
  Sched& s = kp.s;
  const int64_t m_tiles = (p.M + BM - 1) / BM;
  s.pair = PAIR ? 1 : 0;
  s.n_mt = PAIR ? (m_tiles + 1) / 2 : m_tiles;
  s.n_nt = (p.N + BN - 1) / BN;
  s.tiles_per_batch = s.n_mt * s.n_nt;
  s.total_tiles = s.tiles_per_batch * p.nb1 * p.nb2;
  s.kb_total = static_cast<int>((p.K + BK - 1) / BK);
  s.group_m = static_cast<int>(s.n_mt < 16 ? s.n_mt : 16);
  s.band_n = static_cast<int>(std::min<int64_t>(std::max(p.band_n, 0), s.n_nt));
  s.tri = p.tri;
  s.split = p.split_k ? 1 : 0;
  s.total_iters = s.total_tiles * s.kb_total;
  s.mask_chunk = (EPI == EPI_STORE && !s.split) ? p.causal : 0;
  s.mask_m = p.M;
  s.bn = BN;
  const int64_t workers =
      std::min<int64_t>(max_workers[dev], s.split ? s.total_iters : s.total_tiles);
  if (workers <= 0) return cudaSuccess;
  if (p.tri && (p.M != p.K || s.split)) return cudaErrorInvalidValue;
  kp.ticket = nullptr;
  if (p.dyn_tiles) {
    // whole tiles with a plain epilogue only: the split and masked schedules and the update's
    // look-ahead walk the static order
    if (s.split || s.mask_chunk || C::RED || C::W_UPD) return cudaErrorInvalidValue;
    void* t = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&t, g_tile_ticket);
    if (e == cudaSuccess) e = cudaMemsetAsync(t, 0, sizeof(unsigned long long), stream);
    if (e != cudaSuccess) return e;
    kp.ticket = static_cast<unsigned long long*>(t);
  }
  LaunchMark mark(p.kind, stream);
  return launch_overlapped(kern, dim3(static_cast<unsigned>((PAIR ? 2 : 1) * workers)), dim3(C::THREADS),
                           C::SMEM_BYTES, stream, PAIR ? 2 : 1, mA, mB, mB2, mD, kp);
}

// Pairs of CTAs once the problem has at least two 128-row tiles.
template <int BN, int NB, bool A_MN, bool B_MN, int EPI, bool OUT_BF16, bool B_PL = false>
static cudaError_t run_any(const GemmProblem& p, cudaStream_t stream) {
  if (p.M > BM) return run<BN, NB, A_MN, B_MN, EPI, OUT_BF16, true, B_PL>(p, stream);
  return run<BN, NB, A_MN, B_MN, EPI, OUT_BF16, false, B_PL>(p, stream);
}

}  // namespace tc

cudaError_t set_wait_soft_limit(uint64_t ns) {
  const unsigned long long v = (ns == 0 || ns > kWaitLimitNs) ? kWaitLimitNs : ns;
  return cudaMemcpyToSymbol(g_wait_soft_ns, &v, sizeof(v));
}

cudaError_t read_clear_device_error(int* code) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
  return e;
}

cudaError_t launch_gemm_tc(const GemmProblem& p, cudaStream_t stream) {
  using namespace tc;
  if (p.M <= 0 || p.N <= 0 || p.K <= 0 || p.nb1 <= 0 || p.nb2 <= 0) return cudaSuccess;
  // K tails: the MMA issuer only issues the 16-wide K steps that start below K.
  // Inside the last step, elements past K must read as zero in at least one
  // operand; TMA zero-fills them when K ends at the edge of that operand's
  // matrix (gate, proj, apply).  Where K is a window of rows that continue
  // past it in both operands (update and group sums, K = a multiple of the
  // chunk), the caller guarantees K % 16 == 0.
  const bool a_mn = p.A.mn_major != 0, b_mn = p.B.mn_major != 0;
  if (p.split_k && p.epi != EPI_ACCUM) return cudaErrorInvalidValue;
  switch (p.epi) {
    case EPI_GATE:
      if (!a_mn && b_mn)
        return p.out_bf16 ? run_any<128, 2, false, true, EPI_GATE, true>(p, stream)
                          : run_any<128, 2, false, true, EPI_GATE, false>(p, stream);
      break;
    case EPI_STORE:
      // B K-major (B[k][n] read from rows n, e.g. Z^T): single CTAs (pairs split an MN-major B)
      if (!a_mn && !b_mn && p.out_bf16) return run<256, 1, false, false, EPI_STORE, true, false, false>(p, stream);
      if (!a_mn && b_mn)
        return p.out_bf16 ? run_any<256, 1, false, true, EPI_STORE, true>(p, stream)
                          : run_any<256, 1, false, true, EPI_STORE, false>(p, stream);
      if (a_mn && b_mn)
        return p.out_bf16 ? run_any<256, 1, true, true, EPI_STORE, true>(p, stream)
                          : run_any<256, 1, true, true, EPI_STORE, false>(p, stream);
      break;
    case EPI_ACCUM:
      if (!a_mn && b_mn)
        return p.b_planes ? run_any<256, 1, false, true, EPI_ACCUM, false, true>(p, stream)
                          : run_any<256, 1, false, true, EPI_ACCUM, false>(p, stream);
      break;
    case EPI_AXPY:
      if (a_mn && b_mn) return run_any<256, 1, true, true, EPI_AXPY, false>(p, stream);
      break;
  }
  return cudaErrorNotSupported;
}

}  // namespace ipttt

#include "engine_tc.cuh"
