// The MSE chunk loop of the In-Place TTT layer (itsolotime §2.2 and Fig. 1:
// apply the fast weight to a chunk, then take one gradient step on it) as one
// persistent kernel over every chunk of every sequence, for sm_103a.  A sequence
// may also be a packed document (itsolotime §3.2, the fast weight reset at every
// boundary: each document has its own), or a run of windows of chunks whose
// residuals were solved up front (the window form in api.cu).
//
// The rule is independent across the columns of W_o: column block n (256
// columns) of O_k, R_k and W_{k+1} depends only on column block n of W_k.  So
// the loop is cut into work items per column block,
//
//   apply  (k, s, n, m, p)  the 256 x 256 tile m of O_k[:, n] summed over slice p
//                           of d_ff, fp32 partial sums added into `acc` by TMA
//                           reductions; the item that completes a tile's sum
//                           (a counter) turns it into O_k and R_k = O_k - V_k and
//                           clears `acc`;
//   update (k, s, n, r)     rows 256r .. 256r+255 of W[:, n] += alpha Z_k^T R_k,
//                           on the split hi/lo planes (common.cuh split_w),
//
// and an item waits only for what it reads: an update for the residual of its
// column block, an apply of chunk k+1 for the update rows of its slice.  Items
// are numbered in an order of phases A_0, U_0, A_1, U_1, ... (the applies of a
// chunk, then its updates), each phase sequence by sequence and, within one, column
// block by column block, and CTA pairs take them in that order as they free up (a
// device-wide counter).  So the
// updates of the first column blocks start while the last applies of the chunk
// are still running, the applies of the next chunk while its last updates are,
// and no kernel boundary, wave tail or separate residual pass stands between the
// steps.  (A staggered order that mixes the phases of different blocks was
// measured slower: it spreads the working set over two chunks' activations; a
// fixed share of items per pair, w, w + P, ..., 4% slower: pairs that run ahead
// of others wait on them.)  Every dependency points to an earlier item, a pair
// finishes an item without waiting for later ones, and every item taken is held
// by a pair already running, so the order cannot deadlock.
//
// Roles as in the GEMM template (gemm_tc.cu): warp 0 the TMA producer (it also
// waits for an item's inputs), warp 1 the MMA issuer (cta_group::2, 256 x 256
// x 16 per instruction, two TMEM accumulators), warps 2..9 the epilogue as two
// groups of four.  Counters between CTAs: a writer fences its generic stores
// for the async proxy and releases; a reader acquires and fences before its
// TMA copies.  A wait past the soft limit stops the CTA's MMAs and writes but
// keeps every handshake and counter, so the grid still ends cleanly.
//
// This file is part of gemm_tc.cu's translation unit (the device error word
// and the soft wait limit are shared).

namespace ipttt {
namespace tc {

constexpr int kEngStages = 6;
constexpr int kEngEpiWarps = 8;
constexpr int kEngThreads = 64 + 32 * kEngEpiWarps;
constexpr int kEngHalf = 128 * BK * 2;                 // one CTA's A (or B) operand of a stage
constexpr int kEngStageBytes = 2 * kEngHalf;
constexpr int kEngStgBytes = 128 * 32 * 4;             // a group's staging tile: 128 rows x 32 fp32
constexpr int kEngSmem = 1024 + kEngStages * kEngStageBytes + 2 * kEngStgBytes + 512;
static_assert(kEngSmem <= 227 * 1024, "shared memory");

struct EngParams {
  EngineMse a;
  int64_t K, NB, MT, RT;    // chunks; column blocks, token tiles and d_ff tiles of 256
  int64_t NAb, NUb;         // items of one column block's apply phase and update phase
  // counter regions (words): apply slices done per (sequence, chunk, block, token tile, half);
  // residual halves done per (sequence, chunk, block, token tile); update tiles done per
  // (sequence, chunk, block, d_ff slice)
  int64_t off_apply, off_resid, off_upd;
  int64_t total;                  // items
  unsigned long long* ticket;     // the item counter (zero at launch)
};

struct EItem {
  int upd;  // 0: apply, 1: update
  int s, n, m, p, r;
  int64_t k;
  int kb0, kb1;  // k-blocks of its contraction
};

// First d_ff tile (of 256 rows) of slice p.
__device__ __forceinline__ int eng_part_begin(int p, int P, int64_t RT) {
  return static_cast<int>(static_cast<int64_t>(p) * RT / P);
}
__device__ __forceinline__ int eng_part_of(int r, int P, int64_t RT) {
  int p = 0;
  while (p + 1 < P && eng_part_begin(p + 1, P, RT) <= r) ++p;
  return p;
}


// First row of sequence (document) s in Z, V and O.
__device__ __forceinline__ int64_t eng_row0(const EngineMse& a, int s) {
  return a.starts ? a.starts[s] : static_cast<int64_t>(s) * a.L;
}

// Position in the order: item j of phase slot tau (slot 2k: the applies of chunk k, every
// column block's in turn; slot 2k + 1: its updates).
struct ECursor {
  int64_t tau, j;
  // Item g of the whole order.
  __device__ void at(const EngParams& e, int64_t g) {
    int64_t k, base, act;
    if (e.a.icum) {  // packed documents: chunk k holds items icum[k] .. icum[k+1] - 1
      int64_t lo = 0, hi = e.K - 1;
      while (lo < hi) {
        const int64_t mid = (lo + hi + 1) / 2;
        if (e.a.icum[mid] <= g)
          lo = mid;
        else
          hi = mid - 1;
      }
      k = lo;
      base = e.a.icum[k];
      act = e.a.active[k];
    } else {
      act = e.a.batch;
      k = g / (e.NB * (e.NAb + e.NUb));
      base = k * e.NB * (e.NAb + e.NUb);
    }
    const int64_t sa = e.NB * act * e.MT * e.a.parts, rem = g - base;
    tau = 2 * k + (rem >= sa ? 1 : 0);
    j = rem >= sa ? rem - sa : rem;
  }
};

// The items a role of a pair walks.  The even CTA's producer takes item numbers from the
// counter in increasing order, one ahead of its own walk, and publishes each in a ring of
// kRing slots in both CTAs' shared memory (as gemm_tc.cu's TileSrc does for tiles); the other
// roles of both CTAs read the same sequence and release each slot on the even CTA's barrier;
// -1 ends it.
struct EngSrc {
  int64_t* ids;     // this CTA's ring
  uint64_t* full;   // this CTA's ring barriers
  uint64_t* empty;  // release barriers (the even CTA's are the ones counted)
  uint32_t j;       // ring positions walked

  __device__ void init(int64_t* ring_ids, uint64_t* ring_full, uint64_t* ring_empty) {
    ids = ring_ids;
    full = ring_full;
    empty = ring_empty;
    j = 0;
  }
  // Consumer: the next item.  Called by the lanes of `wmask` of one warp together (lane 0
  // among them), which give up together.
  __device__ bool next(const EngParams& e, ECursor& c, uint32_t wmask, volatile int* abort, int code,
                       uint64_t soft_ns) {
    const uint32_t sl = j % kRing, ph = (j / kRing) & 1;
    ++j;
    if (!__all_sync(wmask, mbar_wait_bounded<true>(&full[sl], ph, abort, code, &g_device_error, soft_ns)))
      return false;
    const int64_t g = *reinterpret_cast<volatile int64_t*>(&ids[sl]);
    __syncwarp(wmask);
    if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&empty[sl]), 0));
    if (g < 0) return false;
    c.at(e, g);
    return true;
  }
  // The item after the one `next` returned last, if already published.  Consumes nothing.
  __device__ bool peek(const EngParams& e, ECursor& c) const {
    const uint32_t sl = j % kRing, ph = (j / kRing) & 1;
    if (!mbar_try_wait<true>(&full[sl], ph)) return false;
    const int64_t g = *reinterpret_cast<volatile int64_t*>(&ids[sl]);
    if (g < 0) return false;
    c.at(e, g);
    return true;
  }
  __device__ bool publish(const EngParams& e, uint32_t pos, volatile int* abort, uint64_t soft_ns) {
    const uint32_t sl = pos % kRing, ph = (pos / kRing) & 1;
    if (!mbar_wait_bounded<true>(&empty[sl], ph ^ 1, abort, 1, &g_device_error, soft_ns)) return false;
    int64_t g = static_cast<int64_t>(atomicAdd(e.ticket, 1ull));
    if (g >= e.total) g = -1;
    ids[sl] = g;
    mbar_arrive(&full[sl]);
    st_shared_cluster_u64(mapa_shared(smem_u32(&ids[sl]), 1), static_cast<uint64_t>(g));
    mbar_arrive_cluster(mapa_shared(smem_u32(&full[sl]), 1));  // release: the store above first
    return true;
  }
  // The even CTA's producer: its next item (the item after it is published first).
  __device__ bool fetch(const EngParams& e, ECursor& c, volatile int* abort, uint64_t soft_ns) {
    if (j == 0 && !publish(e, 0, abort, soft_ns)) return false;
    const int64_t g = ids[j % kRing];
    if (g >= 0 && !publish(e, j + 1, abort, soft_ns)) return false;
    ++j;
    if (g < 0) return false;
    c.at(e, g);
    return true;
  }
};

// Within a phase the items run sequence by sequence, each sequence's column block by column
// block: one sequence's Z_k rows serve all its column blocks while they are in L2 (with many
// sequences or documents, a chunk's rows of all of them exceed it).
__device__ __forceinline__ EItem eng_decode(const EngParams& e, const ECursor& cur) {
  EItem it;
  const int64_t ph = cur.tau;
  const int P = e.a.parts;
  const int64_t per = (ph & 1) ? e.RT : e.MT * P;  // items of one column block of one sequence
  it.s = static_cast<int>(cur.j / (e.NB * per));
  int64_t rem = cur.j - it.s * (e.NB * per);
  it.n = static_cast<int>(rem / per);
  rem -= it.n * per;
  it.k = ph / 2;
  if (!(ph & 1)) {
    it.upd = 0;
    it.p = static_cast<int>(rem % P);
    it.m = static_cast<int>(rem / P);
    it.r = 0;
    it.kb0 = eng_part_begin(it.p, P, e.RT) * 4;
    it.kb1 = eng_part_begin(it.p + 1, P, e.RT) * 4;
  } else {
    it.upd = 1;
    it.r = static_cast<int>(rem);
    it.m = it.p = 0;
    it.kb0 = 0;
    it.kb1 = static_cast<int>(e.a.B / BK);
  }
  return it;
}

__device__ __forceinline__ uint32_t* eng_cnt_apply(const EngParams& e, const EItem& it, uint32_t rank) {
  return e.a.counters + e.off_apply + (((it.s * e.K + it.k) * e.NB + it.n) * e.MT + it.m) * 2 + rank;
}
__device__ __forceinline__ uint32_t* eng_cnt_resid(const EngParams& e, int s, int64_t k, int n, int m) {
  return e.a.counters + e.off_resid + ((s * e.K + k) * e.NB + n) * e.MT + m;
}
__device__ __forceinline__ uint32_t* eng_cnt_upd(const EngParams& e, int s, int64_t k, int n, int p) {
  return e.a.counters + e.off_upd + ((s * e.K + k) * e.NB + n) * e.a.parts + p;
}

// A wait for another CTA's counter gives up after half the hard limit of the pipeline waits: the
// MMA issuer and the epilogue of this pair, waiting behind it on their mbarriers, then see their
// data arrive before their own limit, so the pair never takes the hard exit with copies in flight.
constexpr uint64_t kEngDepLimitNs = kWaitLimitNs / 2;

// Wait until *c >= target (acquire).  Past the soft limit the CTA aborts softly (error code 5);
// past kEngDepLimitNs the wait gives up and the item goes ahead on whatever is there, the CTA
// still only softly aborted (no more MMAs or writes, every handshake kept), so that no role of it
// stops waiting for copies or MMAs already in flight.
__device__ __forceinline__ void eng_wait_count(const uint32_t* c, uint32_t target, volatile int* abort,
                                               uint64_t soft_ns) {
  if (ld_acquire_u32(c) >= target) return;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u32(c) < target) {
    if (*abort == kAbortHard) return;
    const uint64_t el = globaltimer_ns() - t0;
    if (el > soft_ns && *abort == 0) {
      atomicMax(const_cast<int*>(abort), kAbortSoft);
      atomicCAS(&g_device_error, 0, 5);
    }
    if (el > kEngDepLimitNs) {
      atomicMax(const_cast<int*>(abort), kAbortSoft);
      atomicCAS(&g_device_error, 0, 5);
      return;
    }
    __nanosleep(64);
  }
}

// The 256 epilogue threads (both groups).
__device__ __forceinline__ void eng_epi_all_barrier() {
  __syncwarp();
  asm volatile("bar.sync 3, 256;" ::: "memory");
}

// O_k and R_k of this CTA's 128 rows x 256 columns of an apply tile, from the finished fp32
// sums, which are cleared for the next chunk.  A packed document's last chunk may hold n < B
// tokens: past them O is not written and R is zero, and R is scaled by B/n, so the step is the
// mean over the chunk's n tokens.  Warp ew takes rows ew, ew + 8, ...; lane l columns
// 8l .. 8l+7, so every row is one coalesced pass.
__device__ __forceinline__ void eng_residual(const EngParams& e, const EItem& it, uint32_t rank, int ew, int lane) {
  const EngineMse& a = e.a;
  const int64_t row0 = it.m * 256 + rank * 128;           // in the chunk
  const int64_t arow0 = it.s * a.B + row0;                  // acc rows
  const int64_t rrow0 = it.s * a.r_seq + it.k * a.r_chunk + row0;  // R rows
  const int64_t trow0 = eng_row0(a, it.s) + it.k * a.B + row0;  // O and V rows
  const int64_t ntok = a.lens ? min(a.B, a.lens[it.s] - it.k * a.B) : a.B;
  const float scale = static_cast<float>(a.B) / static_cast<float>(ntok);
  const int64_t c0 = static_cast<int64_t>(it.n) * 256 + lane * 8;
  const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(a.V);
  __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.O);
  __nv_bfloat16* R = static_cast<__nv_bfloat16*>(a.R);
#pragma unroll 1
  for (int i = ew; i < 128; i += 2 * kEngEpiWarps) {
    uint32_t x[2][8];
    uint4 v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t ii = i + h * kEngEpiWarps;
      ld_global_v8(a.acc + (arow0 + ii) * a.d + c0, x[h]);
      v[h] = (row0 + ii < ntok) ? *reinterpret_cast<const uint4*>(V + (trow0 + ii) * a.d + c0) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t ii = i + h * kEngEpiWarps;
      const uint32_t zero8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      st_global_v8(a.acc + (arow0 + ii) * a.d + c0, zero8);
      const __nv_bfloat162* vh = reinterpret_cast<const __nv_bfloat162*>(&v[h]);
      const bool valid = (row0 + ii < ntok);
      uint32_t o4[4], r4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float s0 = __uint_as_float(x[h][2 * q]), s1 = __uint_as_float(x[h][2 * q + 1]);
        const float2 t = __bfloat1622float2(vh[q]);
        o4[q] = pack_bf16x2(s0, s1);
        r4[q] = valid ? pack_bf16x2(scale * (s0 - t.x), scale * (s1 - t.y)) : 0u;
      }
      if (valid) *reinterpret_cast<uint4*>(O + (trow0 + ii) * a.d + c0) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      *reinterpret_cast<uint4*>(R + (rrow0 + ii) * a.d + c0) = make_uint4(r4[0], r4[1], r4[2], r4[3]);
    }
  }
}

__global__ void __launch_bounds__(kEngThreads, 1)
    engine_mse_kernel(const __grid_constant__ CUtensorMap tmZk, const __grid_constant__ CUtensorMap tmZm,
                      const __grid_constant__ CUtensorMap tmHi, const __grid_constant__ CUtensorMap tmR,
                      const __grid_constant__ CUtensorMap tmAcc, const __grid_constant__ EngParams e) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint8_t* stages = smem;
  uint8_t* stg = smem + kEngStages * kEngStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + 2 * kEngStgBytes);
  uint64_t* full_bar = bars;                          // [kEngStages]
  uint64_t* empty_bar = bars + kEngStages;            // [kEngStages]
  uint64_t* tfull_bar = bars + 2 * kEngStages;        // [2]
  uint64_t* tempty_bar = bars + 2 * kEngStages + 2;   // [2]
  uint64_t* drain_bar = bars + 2 * kEngStages + 4;    // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kEngStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* last_flag = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  uint64_t* ring_full = bars + 2 * kEngStages + 7;  // [kRing] item numbers
  uint64_t* ring_empty = ring_full + kRing;          // [kRing]
  int64_t* ring_ids = reinterpret_cast<int64_t*>(ring_empty + kRing);
  static_assert((2 * kEngStages + 7 + 3 * kRing) * 8 <= 512, "barrier area");

  const EngineMse& a = e.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool mma_cta = (rank == 0);

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < kEngStages; ++i) {
        mbar_init(&full_bar[i], 1);
        mbar_init(&empty_bar[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&tfull_bar[i], 1);
        mbar_init(&tempty_bar[i], 2 * kEngEpiWarps);  // every epilogue warp of both CTAs
      }
      mbar_init(drain_bar, 1);
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&ring_full[i], 1);
        // the even CTA's MMA issuer and epilogue warps, the odd CTA's producer and epilogue warps
        mbar_init(&ring_empty[i], 2 + 2 * kEngEpiWarps);
      }
      *abort_flag = 0;
      *last_flag = 0;
      fence_mbarrier_init();
      tma_prefetch_desc(&tmZk);
      tma_prefetch_desc(&tmZm);
      tma_prefetch_desc(&tmHi);
      tma_prefetch_desc(&tmR);
      tma_prefetch_desc(&tmAcc);
    }
    __syncwarp();
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t soft_ns = g_wait_soft_ns;
  EngSrc src;
  src.init(ring_ids, ring_full, ring_empty);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kc = 0, pst = 0, pph = 0, issued_mask = 0;
      bool ok = true;
      const uint64_t pol_hi = l2_policy(a.keep_hi ? L2_EVICT_LAST : L2_NORMAL);
      const uint64_t pol_n = l2_policy(L2_NORMAL);
      ECursor cur;
      while (ok && (mma_cta ? src.fetch(e, cur, abort_flag, soft_ns) : src.next(e, cur, 1u, abort_flag, 1, soft_ns))) {
        const EItem it = eng_decode(e, cur);
        // what the item reads must be written: the residual of its column block (update), or
        // the previous chunk's update of its d_ff slice (apply)
        if (it.upd) {
          // (token tile by token tile, in the k loop below)
        } else if (it.k > 0) {
          const int nt = eng_part_begin(it.p + 1, a.parts, e.RT) - eng_part_begin(it.p, a.parts, e.RT);
          eng_wait_count(eng_cnt_upd(e, it.s, it.k - 1, it.n, it.p), static_cast<uint32_t>(2 * nt), abort_flag,
                         soft_ns);
        }
        fence_proxy_async_global();
        const int64_t col = static_cast<int64_t>(it.n) * 256 + rank * 128;  // this CTA's B columns
        for (int kb = it.kb0; kb < it.kb1; ++kb, ++kc) {
          if (it.upd && kb % 4 == 0) {
            // an update contracts over the chunk's tokens: those of token tile kb / 4 are ready
            // once both halves of that tile's residual are written
            eng_wait_count(eng_cnt_resid(e, it.s, it.k, it.n, kb / 4), 2u, abort_flag, soft_ns);
            fence_proxy_async_global();
          }
          const uint32_t st = pst, ph = pph;
          if (++pst == kEngStages) {
            pst = 0;
            pph ^= 1;
          }
          if (!mbar_wait_bounded(&empty_bar[st], ph ^ 1, abort_flag, 1, &g_device_error, soft_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + st * kEngStageBytes;
          uint8_t* sb = sa + kEngHalf;
          const uint32_t bar_cl = mapa_shared(smem_u32(&full_bar[st]), 0);
          if (mma_cta) mbar_arrive_expect_tx(&full_bar[st], 2 * kEngStageBytes);
          issued_mask |= 1u << st;
          const int64_t k0 = static_cast<int64_t>(kb) * BK;
          if (!it.upd) {
            // A: rows of Z_k (this CTA's 128 of the 256-token tile), d_ff columns k0 ..
            const int64_t zrow = eng_row0(a, it.s) + it.k * a.B + it.m * 256 + rank * 128;
            tma_load_2d_pair(sa, &tmZk, bar_cl, static_cast<int>(k0), static_cast<int>(zrow), pol_n);
            // B: the hi plane, d_ff rows k0 .., this CTA's 128 columns of block n
            const int c1 = static_cast<int>((k0 % kPlaneRows) / 16);
            const int c2 = static_cast<int>((it.s * a.w.rb + k0 / kPlaneRows) * a.w.cb + col / kPlaneCols);
            tma_load_3d_pair(sb, &tmHi, bar_cl, 0, c1, c2, pol_hi);
          } else {
            // A: Z_k^T (or the Zu operand's rows of the chunk), tokens k0 .., this CTA's 128 d_ff
            // rows of tile r
            const int64_t trow = eng_row0(a, it.s) + it.k * a.B + k0;
            const int64_t frow = static_cast<int64_t>(it.r) * 256 + rank * 128;
            // B: R_k, the same tokens, this CTA's 128 columns of block n
            const int64_t rrow = it.s * a.r_seq + it.k * a.r_chunk + k0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              tma_load_2d_pair(sa + j * (64 * BK * 2), &tmZm, bar_cl, static_cast<int>(frow + 64 * j),
                               static_cast<int>(trow), pol_n);
              tma_load_2d_pair(sb + j * (64 * BK * 2), &tmR, bar_cl, static_cast<int>(col + 64 * j),
                               static_cast<int>(rrow), pol_n);
            }
          }
        }
        // An update item of chunk k brings its share of Z_{k+1} (the next applies' A operand)
        // into L2: the chunk's update items split those rows of every sequence evenly.
        if (ok && it.upd && it.k + 1 < e.K && rank == 0 && !a.starts) {
          const int64_t seg = a.B * a.d_ff * 2;  // bytes of one sequence's chunk of Z
          const int64_t total = a.batch * seg, nu = e.NB * e.NUb;
          const int64_t u = (static_cast<int64_t>(it.n) * a.batch + it.s) * e.RT + it.r;
          int64_t off = (total * u / nu) & ~int64_t{255};
          const int64_t end = (u + 1 == nu) ? total : ((total * (u + 1) / nu) & ~int64_t{255});
          while (off < end) {
            const int64_t sq = off / seg, in = off - sq * seg;
            const int64_t n = min(min(end - off, seg - in), int64_t{65536});
            prefetch_l2_bulk(static_cast<const uint8_t*>(a.Z) + ((sq * a.L + (it.k + 1) * a.B) * a.d_ff) * 2 + in,
                             static_cast<uint32_t>(n));
            off += n;
          }
        }
      }
      // Teardown: every copy issued here has landed before shared memory is released.  The
      // copies complete on the MMA CTA's barriers; its peer learns of them from its empty
      // barriers (the MMAs that read them have finished).
      for (uint32_t st = 0; st < kEngStages; ++st) {
        if (!(issued_mask & (1u << st))) continue;
        const uint32_t f = (kc - 1 - st) / kEngStages;  // last fill of stage st
        if (!mma_cta)
          mbar_wait_drain(&empty_bar[st], f & 1, 4, &g_device_error);
        else
          mbar_wait_drain(&full_bar[st], f & 1, 4, &g_device_error);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && mma_cta) {
      constexpr uint32_t idesc_apply = make_idesc_bf16(2 * BM, 256, false, true);
      constexpr uint32_t idesc_upd = make_idesc_bf16(2 * BM, 256, true, true);
      const uint32_t s0 = smem_u32(stages);
      const uint64_t a_apply = operand_desc<false>(s0, 0), b_apply = operand_desc<true, true>(s0 + kEngHalf, 0);
      const uint64_t a_upd = operand_desc<true>(s0, 0), b_upd = operand_desc<true>(s0 + kEngHalf, 0);
      uint32_t ls = 0, st = 0, ph = 0;
      bool ok = true;
      ECursor cur;
      while (ok && src.next(e, cur, 1u, abort_flag, 2, soft_ns)) {
        const EItem it = eng_decode(e, cur);
        const uint32_t acc = ls & 1, aph = (ls >> 1) & 1;
        if (!mbar_wait_bounded(&tempty_bar[acc], aph ^ 1, abort_flag, 2, &g_device_error, soft_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kAccStride;
        const uint64_t a0 = it.upd ? a_upd : a_apply, b0 = it.upd ? b_upd : b_apply;
        const uint32_t idesc = it.upd ? idesc_upd : idesc_apply;
        const uint32_t ak = it.upd ? (2048u >> 4) : (32u >> 4);   // a k step: 16 rows MN-major, 32 bytes K-major
        const uint32_t bk = it.upd ? (2048u >> 4) : (512u >> 4);  // 16 rows MN-major, 512 bytes of plane rows
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait_bounded(&full_bar[st], ph, abort_flag, 2, &g_device_error, soft_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!*abort_flag) {
            const uint32_t soff = (st * kEngStageBytes) >> 4;
            const uint32_t first = (kb == it.kb0) ? 0u : 1u;
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              umma_bf16_pair(d_tmem, a0 + soff + ks * ak, b0 + soff + ks * bk, idesc, ks ? 1u : first);
          }
          umma_commit_pair_both(&empty_bar[st]);
          if (++st == kEngStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair_both(&tfull_bar[acc]);
        ++ls;
      }
      umma_commit_pair_both(drain_bar);
      mbar_wait_drain(drain_bar, 0, 4, &g_device_error);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                // 0 .. 7
    const int grp = ew / 4;                 // two groups of four warps
    const int quarter = warp % 4;           // TMEM lanes 32*quarter .. +31
    const int trow = quarter * 32 + lane;   // row of this CTA's 128 that this thread finishes
    const bool issuer = (quarter == 0 && lane == 0);  // one per group: the TMA reductions
    uint8_t* buf = stg + grp * kEngStgBytes;
    const uint64_t pol_hi = l2_policy(a.keep_hi ? L2_EVICT_LAST : L2_NORMAL);
    const uint64_t pol_lo = l2_policy(a.keep_hi ? L2_EVICT_FIRST : L2_NORMAL);
    const int sw = (trow >> 2) & 1;  // this row's 16-byte halves trade places in a plane block
    // This thread's row of an update item's plane blocks (the CTA's 128 rows of the tile).
    auto plane_row = [&](const EItem& x, uint16_t* base) {
      const int64_t rbk = x.s * a.w.rb + static_cast<int64_t>(x.r) * 2 + rank;
      return base + plane_index(rbk, static_cast<int64_t>(x.n) * (256 / kPlaneCols), a.w.cb, 0, 0) + trow * kPlaneCols;
    };
    uint32_t wh[4][8], wl[4][8];  // plane rows of the chunks in flight, by chunk % 4
    bool pre = false;             // the first three chunks of this update item are already loaded
    bool failed = false;
    uint32_t ls = 0;
    ECursor cur;
    while (src.next(e, cur, 0xffffffffu, abort_flag, 3, soft_ns)) {
      const EItem it = eng_decode(e, cur);
      // The next item's planes may be loaded during this one only once what writes them has
      // finished: a complete residual of the first token tile of its column block means every
      // apply of that tile is done, and those waited for the previous chunk's updates of all
      // the block's rows.  (Only if the next item is already published.)
      ECursor nx;
      bool nx_upd = false;
      if (it.upd && src.peek(e, nx)) {
        const EItem nit = eng_decode(e, nx);
        nx_upd = nit.upd && ld_acquire_u32(eng_cnt_resid(e, nit.s, nit.k, nit.n, 0)) >= 2u;
      }
      nx_upd = __all_sync(0xffffffffu, nx_upd);
      const uint32_t acc = ls & 1, aph = (ls >> 1) & 1;
      if (!failed)
        failed = !__all_sync(0xffffffffu,
                             mbar_wait_bounded(&tfull_bar[acc], aph, abort_flag, 3, &g_device_error, soft_ns));
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccStride;
      if (!it.upd) {
        // ---- apply: this slice's partial sums of the tile, added into acc by TMA reductions
        const int64_t orow = it.s * a.B + it.m * 256 + rank * 128;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          const int c = grp + 2 * j;  // 32-column chunk of the tile
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + c * 32, r);
          tmem_wait_ld();
          if (issuer) bulk_wait_group_read<0>();  // the buffer's last reduction has read it
          epi_barrier(grp);
          if (!failed) {
            // 128-byte swizzle: 16-byte chunk q of row t sits at chunk q ^ (t % 8)
            float4* srow = reinterpret_cast<float4*>(buf + trow * 128);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              srow[q ^ (trow & 7)] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
          }
          fence_proxy_async_shared();
          epi_barrier(grp);
          if (issuer && !failed && !*abort_flag) {
            if (j == 0) fence_proxy_async_global();  // after the clearing of acc by the last residual
            tma_reduce_add_2d(&tmAcc, buf, static_cast<int>(static_cast<int64_t>(it.n) * 256 + c * 32),
                              static_cast<int>(orow));
            bulk_commit_group();
          }
        }
        // the accumulator has been read: hand it back to the MMA issuer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
        // this slice's sums are in memory before it is counted
        if (issuer) {
          bulk_wait_group<0>();
          fence_proxy_async_global();
        }
        eng_epi_all_barrier();
        if (ew == 0 && lane == 0) {
          fence_acq_rel_gpu();
          const uint32_t old = atom_add_acq_rel_u32(eng_cnt_apply(e, it, rank), 1u);
          *last_flag = (old + 1 == static_cast<uint32_t>(a.parts)) ? 1u : 0u;
        }
        eng_epi_all_barrier();
        if (*last_flag) {
          // the last slice of this half tile: every slice's sums are in acc
          fence_acq_rel_gpu();
          if (!failed && !*abort_flag) eng_residual(e, it, rank, ew, lane);
          fence_proxy_async_global();  // R is read next by TMA copies
          eng_epi_all_barrier();
          if (ew == 0 && lane == 0) {
            fence_acq_rel_gpu();
            red_add_release_u32(eng_cnt_resid(e, it.s, it.k, it.n, it.m), 1u);
          }
        }
      } else {
        // ---- update: W = W + alpha * acc on this CTA's 128 plane rows of the tile.  The rows
        // are one row of plane blocks; group g takes the 16-column chunks g, g + 2, ...; each
        // thread reads and writes its row's 32 bytes of each plane, three chunks ahead.
        constexpr int WC = kPlaneCols;
        constexpr int GCH = 256 / WC / 2;  // chunks per group
        static_assert(GCH % 4 == 0, "a group's chunks come in fours");
        uint16_t* const hi = plane_row(it, a.w.hi);
        uint16_t* const lo = plane_row(it, a.w.lo);
        auto wload = [&](uint16_t* h0, uint16_t* l0, int c, uint32_t (&h)[8], uint32_t (&l)[8]) {
          ld_global_v8_hint(h0 + static_cast<int64_t>(c) * kPlaneBlock, h, pol_hi);
          ld_global_v8_hint(l0 + static_cast<int64_t>(c) * kPlaneBlock, l, pol_lo);
        };
        if (!pre) {
          wload(hi, lo, grp, wh[0], wl[0]);
          wload(hi, lo, grp + 2, wh[1], wl[1]);
          wload(hi, lo, grp + 4, wh[2], wl[2]);
        }
        // the next update item's rows (its first three chunks are loaded during this one's last)
        uint16_t* nhi = hi;
        uint16_t* nlo = lo;
        if (nx_upd) {
          const EItem nit = eng_decode(e, nx);
          nhi = plane_row(nit, a.w.hi);
          nlo = plane_row(nit, a.w.lo);
        }
        uint32_t ra[WC], rb[WC];
        tmem_ld_32x32b_x16(tbase + grp * WC, ra);
#pragma unroll 1
        for (int j4 = 0; j4 < GCH; j4 += 4) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int jj = j4 + u, c = grp + 2 * jj;
            uint32_t(&rr)[WC] = (u & 1) ? rb : ra;
            uint32_t(&rn)[WC] = (u & 1) ? ra : rb;
            tmem_wait_ld(rr);
            if (jj + 1 < GCH) tmem_ld_32x32b_x16(tbase + (c + 2) * WC, rn);
            // columns 2q, 2q+1 sit in stored word q ^ 4*sw
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              hw[q] = sw ? wh[u][q + 4] : wh[u][q];
              hw[q + 4] = sw ? wh[u][q] : wh[u][q + 4];
              lw[q] = sw ? wl[u][q + 4] : wl[u][q];
              lw[q + 4] = sw ? wl[u][q] : wl[u][q + 4];
            }
            if (jj + 3 < GCH)
              wload(hi, lo, c + 6, wh[(u + 3) & 3], wl[(u + 3) & 3]);
            else if (nx_upd)
              wload(nhi, nlo, grp + 2 * (jj + 3 - GCH), wh[(u + 3) & 3], wl[(u + 3) & 3]);
            uint32_t ho[8], lo8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float w0, w1;
              join_w2(hw[q], lw[q], w0, w1);
              split_w2(fmaf(a.alpha, __uint_as_float(rr[2 * q]), w0), fmaf(a.alpha, __uint_as_float(rr[2 * q + 1]), w1),
                       ho[q], lo8[q]);
            }
            if (!failed && !*abort_flag) {
              uint32_t hs[8], ls8[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                hs[q] = sw ? ho[q + 4] : ho[q];
                hs[q + 4] = sw ? ho[q] : ho[q + 4];
                ls8[q] = sw ? lo8[q + 4] : lo8[q];
                ls8[q + 4] = sw ? lo8[q] : lo8[q + 4];
              }
              st_global_v8_hint(hi + static_cast<int64_t>(c) * kPlaneBlock, hs, pol_hi);
              st_global_v8_hint(lo + static_cast<int64_t>(c) * kPlaneBlock, ls8, pol_lo);
            }
          }
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
        // the new rows are read next by TMA copies (the next chunk's applies)
        fence_proxy_async_global();
        eng_epi_all_barrier();
        if (ew == 0 && lane == 0) {
          fence_acq_rel_gpu();
          red_add_release_u32(eng_cnt_upd(e, it.s, it.k, it.n, eng_part_of(it.r, a.parts, e.RT)), 1u);
        }
      }
      pre = it.upd && nx_upd;
      ++ls;
    }
    if (issuer) bulk_wait_group<0>();
    __syncwarp();
  }

  // Teardown: the roles that ran on one lane re-converge; with the pair, the cluster barrier
  // keeps both CTAs until the last MMAs into either TMEM and the last arrivals on either
  // CTA's barriers are done; then TMEM is freed.
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace tc

bool engine_mse_supported(int64_t B, int64_t d, int64_t d_ff) {
  return B > 0 && d > 0 && d_ff > 0 && B % 256 == 0 && d % 256 == 0 && d_ff % 256 == 0;
}

int64_t engine_counter_words(int64_t batch, int64_t L, int64_t B, int64_t d, int parts) {
  const int64_t K = L / B, NB = d / 256, MT = B / 256;
  return batch * K * NB * (3 * MT + parts);
}

cudaError_t launch_engine_mse(const EngineMse& a, cudaStream_t stream) {
  using namespace tc;
  if (!engine_mse_supported(a.B, a.d, a.d_ff) || a.batch < 1 || a.L < a.B || a.L % a.B || a.parts < 1 ||
      a.parts > a.d_ff / 256 || !a.counters || !a.w.hi || !a.w.lo)
    return cudaErrorNotSupported;
  static std::mutex mu;
  static uint64_t attr_done = 0;
  static int max_pairs[64] = {0};
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!(attr_done & (1ull << dev))) {
      cudaError_t err = cudaFuncSetAttribute(engine_mse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kEngSmem);
      if (err != cudaSuccess) return err;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (device_sm_count() / 2));
      cfg.blockDim = dim3(kEngThreads);
      cfg.dynamicSmemBytes = kEngSmem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      err = cudaOccupancyMaxActiveClusters(&clusters, engine_mse_kernel, &cfg);
      if (err != cudaSuccess) return err;
      if (clusters <= 0) return cudaErrorInvalidConfiguration;
      max_pairs[dev] = clusters;
      attr_done |= 1ull << dev;
    }
  }
  CUtensorMap mZk, mZm, mHi, mR, mAcc;
  const int64_t T = a.rows > 0 ? a.rows : a.batch * a.L, BR = a.batch * a.B;
  if ((a.starts || a.lens || a.active || a.icum) && !(a.starts && a.lens && a.active && a.icum && a.icum_total > 0))
    return cudaErrorInvalidValue;
  if (!make_map(&mZk, a.Z, T, a.d_ff, a.d_ff, false, 64, BM)) return cudaErrorInvalidValue;
  if (!make_map(&mZm, a.Zu ? a.Zu : a.Z, T, a.d_ff, a.d_ff, false, 64, 64)) return cudaErrorInvalidValue;
  if (!make_plane_map(&mHi, a.w, 128)) return cudaErrorInvalidValue;
  if (a.r_seq < a.B || a.r_chunk < 0) return cudaErrorInvalidValue;
  const int64_t RR = (a.batch - 1) * a.r_seq + (a.L / a.B - 1) * a.r_chunk + a.B;  // rows of R
  if (!make_map(&mR, a.R, RR, a.d, a.d, false, 64, 64)) return cudaErrorInvalidValue;
  if (!make_map(&mAcc, a.acc, BR, a.d, a.d, true, 32, BM)) return cudaErrorInvalidValue;

  EngParams e;
  e.a = a;
  e.K = a.L / a.B;
  e.NB = a.d / 256;
  e.MT = a.B / 256;
  e.RT = a.d_ff / 256;
  e.NAb = a.batch * e.MT * a.parts;
  e.NUb = a.batch * e.RT;
  const int64_t total = a.icum ? a.icum_total : e.K * e.NB * (e.NAb + e.NUb);
  e.off_apply = 0;
  e.off_resid = a.batch * e.K * e.NB * e.MT * 2;
  e.off_upd = e.off_resid + a.batch * e.K * e.NB * e.MT;
  const int64_t pairs = std::min<int64_t>(max_pairs[dev], total);
  e.total = total;
  {
    void* t = nullptr;
    cudaError_t err = cudaGetSymbolAddress(&t, g_tile_ticket);
    if (err == cudaSuccess) err = cudaMemsetAsync(t, 0, sizeof(unsigned long long), stream);
    if (err != cudaSuccess) return err;
    e.ticket = static_cast<unsigned long long*>(t);
  }

  LaunchMark mark(K_ENGINE, stream);
  // The grid is the number of clusters that fit on the device together; should other work
  // hold SMs, the late pairs start as it leaves and take whatever items are left.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(kEngThreads);
  cfg.dynamicSmemBytes = kEngSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, engine_mse_kernel, mZk, mZm, mHi, mR, mAcc, e);
  return err;
}

}  // namespace ipttt
