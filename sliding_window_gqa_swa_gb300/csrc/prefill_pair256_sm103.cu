// Prefill attention at head size 256 for an even GQA group: the two query
// heads 2g and 2g + 1 of one KV head share every tensor-core product
// (tcgen05 cta_group::2, M = 256), on 128-key tiles.
//
// A cluster of two CTAs serves 128-row query tiles for the two heads; CTA r
// holds head 2g + r's Q rows (64 KB) and its own rows of every accumulator.
// The kernel is persistent: one cluster per SM pair walks a list of work items
// (query tile, head pair, sequence), longest first, so no partial wave is left
// and the next item's Q and key tiles load, and its first score products run,
// while the softmax warps write the previous item's output.  Each CTA loads half of every key tile: keys [64 r, 64 r + 64)
// of K (the B operand of S = Q K^T is split by its N dimension) and
// head-dimension columns [128 r, 128 r + 128) of V (the B operand of
// O += P V is split by its N dimension), so each SM streams 64 KB per 128-key
// tile instead of 128 KB; a single SM's TMA stream is what bounds the
// one-CTA kernel at this head size.
//
// Per key tile j: S_j = Q K_j^T (M = 256, N = 128, sixteen K = 16 steps) into
// one of two 128-column S buffers in tensor memory; the softmax warps of each
// CTA turn their rows of S_j into bf16 probabilities P_j, written over the
// first 64 columns of the same buffer; O += P_j V_j (M = 256, N = 256, eight
// K = 16 steps, A = P_j from tensor memory, V read MN-major), then S_{j+2}
// into the buffer S_j came from (the tensor pipe runs one thread's MMAs in
// order, so S_{j+2} overwrites P_j only after PV_j read it).  The softmax of
// tile j + 1 overlaps PV_j and S_{j+2}.  Tensor memory per CTA: O (256
// columns) + two S buffers = 512 columns.  Shared memory per CTA: Q (64 KB),
// a ring of four 32 KB slots (a K or V half-tile each), a 32 KB output
// staging area (the output leaves through TMA stores: stores from registers
// would write 32 rows per warp instruction), the row-maximum exchange,
// barriers: 226 KB.
//
// Warp roles (both CTAs): warp 0 TMA producer; warp 1 lane 0 issues the MMAs
// (even CTA) or forwards "P_j written" to the even CTA (odd CTA); warps 2-9
// softmax in two warpgroups, one query row per thread (its TMEM lane), group g
// owning key columns [64 g, 64 g + 64) of every tile and output columns
// [128 g, 128 g + 128).  The two threads of a row agree on each tile's maximum
// through shared memory; O is rescaled lazily (only when the maximum grows by
// more than 2^32).  PV uses the bf16-rounded probabilities and O is
// normalised by the sum of the same rounded values; lse uses the unrounded
// sum.
// Every wait is bounded; a timeout sets the device error word, makes all
// roles stop, lets in-flight copies and MMAs finish, and frees TMEM.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary and Compilation behavior (causal square-prefill plan,
// generic plan for future same-image pairs); "Add SDPA attention
// implementation", Summary (K/V shared by the query heads of a group).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace swa {
namespace {

using namespace ptx;

constexpr int BM = kPlanBM;      // 128 query rows per CTA
constexpr int BN = 128;          // keys per tile
constexpr int HD = 256;          // head dimension
constexpr int QBOX = 128 * 128;  // one {64 columns, 128 rows} bf16 box: 16 KB
constexpr int KBOX = 64 * 128;   // one {64 columns, 64 keys} bf16 box: 8 KB
constexpr int SLOT = 32768;      // K half-tile (64 keys x 256) or V half-tile (128 keys x 128)
constexpr int NST = 4;           // ring slots
constexpr int THREADS = 512;
// Per-thread registers after the split (launch: 65536 / 512 = 128 each); the
// four warpgroups' shares add up to the launch's 65536 registers
constexpr int REGS_CTRL = 56, REGS_SOFTMAX = 168, REGS_EPI = 120;
static_assert(REGS_CTRL + 2 * REGS_SOFTMAX + REGS_EPI <= 4 * (65536 / THREADS), "register split");
constexpr int OFF_Q = 0;
constexpr int OFF_RING = OFF_Q + 4 * QBOX;
constexpr int OFF_STAGE = OFF_RING + NST * SLOT;  // output staging: two {64 columns, 128 rows} boxes
constexpr int OFF_PMAX = OFF_STAGE + 2 * QBOX;    // [128 rows] fp32: the two groups' exchange
constexpr int OFF_ROWS = OFF_PMAX + BM * 4;       // [128 rows] x {1 / l, lse}: softmax -> epilogue
constexpr int OFF_BAR = OFF_ROWS + BM * 8;
constexpr int N_BARS = 2 * NST + 11;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024 B
static_assert(SMEM <= 232448, "shared memory budget");

constexpr uint32_t TM_O = 0, TM_S = 256, TM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(2 * BM, BN, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(2 * BM, HD, true);
// O and the row sums are rescaled only when the row maximum grows by more than
// 2^32: probabilities then stay below 2^32 (bf16 and fp32 hold them exactly
// as well as below 1), so the fp32 accumulators keep ample headroom, and the
// rescale (a read-modify-write of O in tensor memory) practically never runs
constexpr float kRescaleLog2 = 32.f;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (NST + s); }
  __device__ uint32_t q() const { return base + 8 * (2 * NST); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (2 * NST + 1 + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (2 * NST + 3 + b); }
  __device__ uint32_t pv_done(int b) const { return base + 8 * (2 * NST + 5 + b); }
  __device__ uint32_t teardown() const { return base + 8 * (2 * NST + 7); }
  __device__ uint32_t q_free() const { return base + 8 * (2 * NST + 8); }  // the item's score MMAs are done
  __device__ uint32_t o_free() const { return base + 8 * (2 * NST + 9); }  // the epilogue has read O
  __device__ uint32_t rows_ready() const { return base + 8 * (2 * NST + 10); }  // 1 / l and lse of every row
};

// Bounded wait on one phase of an mbarrier (cluster-scope acquire when the
// phase is completed by the peer CTA or by the pair's MMAs).  Gives up when
// another role has aborted or after kTimeoutNs, recording the timeout.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  auto poll = [&] { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (poll()) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        if (err) atomicCAS(err, 0, kErrTimeout);
        return false;
      }
    }
  }
}

// Bounded wait of a single thread on the critical path (the MMA issuer and
// the forwarder): polled with test_wait, because a thread suspended in
// try_wait was measured to resume up to ~1500 SM clocks after the phase
// completed.  kCluster: acquire at cluster scope (the peer's arrivals).
template <bool kCluster>
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  auto poll = [&] {
    if (!kCluster) return mbar_test_wait(bar, parity);
    if (!mbar_test_wait_relaxed_cluster(bar, parity)) return false;
    fence_acquire_cluster();
    return true;
  };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (poll()) return true;
    if ((it & 255) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        if (err) atomicCAS(err, 0, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x on the special-function unit (subnormal results flush to 0; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// One work item: query tile qt (128 rows) of sequence b for the head pair
// `pair` (query heads 2 pair, 2 pair + 1).  Items are numbered longest first
// (late query tiles of a causal sequence have the most key tiles).
struct Item {
  int qt, pair, b;
};
__device__ __forceinline__ Item item_of(int it, int npairs, int batch, int nqt) {
  const int per_tile = npairs * batch;
  Item x;
  x.qt = nqt - 1 - it / per_tile;
  const int rest = it % per_tile;
  x.pair = rest % npairs;
  x.b = rest / npairs;
  return x;
}

// Key tiles [kt_lo, kt_lo + n) that some row of query tile (b, qt) needs.
__device__ __forceinline__ void tile_range(const PrefillArgs& a, int b, int qt, int& kt_lo, int& n) {
  int k_lo = 0, k_hi = 0;
  if (a.generic) {
    const PlanLayout L = plan_layout(a.batch, a.chunk_len);
    const int nqt = (a.chunk_len + BM - 1) / BM;
    const char* plan = static_cast<const char*>(a.plan);
    k_lo = reinterpret_cast<const int32_t*>(plan + L.off_tlo)[b * nqt + qt];
    k_hi = reinterpret_cast<const int32_t*>(plan + L.off_thi)[b * nqt + qt];
  } else {
    const int vs = a.valid_start ? a.valid_start[b] : 0;
    const int q0 = a.chunk_start + qt * BM;
    const int qlast = min(q0 + BM - 1, a.chunk_start + a.chunk_len - 1);
    if (qlast >= vs) {
      int lo, hi;
      causal_interval(max(q0, vs), vs, a.window, lo, hi);
      k_lo = lo;
      k_hi = qlast + 1;
    }
  }
  k_hi = min(k_hi, a.key_rows);
  kt_lo = k_lo / BN;
  n = (k_hi > k_lo) ? ((k_hi - 1) / BN - kt_lo + 1) : 0;
}

// Persistent: cluster c (CTAs 2c, 2c + 1) serves items c, c + C, c + 2C, ...
// (C clusters).  The ring, the S buffers and every barrier keep running
// across items, so the next item's Q and first key tiles load, and its first
// two score products run, while the softmax warps finish the previous item.
__global__ void __launch_bounds__(THREADS, 1)
prefill_pair256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_ki, const __grid_constant__ CUtensorMap tm_vi,
                       const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + OFF_Q, sRing = base + OFF_RING;
  const Bars bars{base + OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_MISC + 4);
  int32_t* err = a.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = int(cluster_ctarank());  // 0: issues the pair's MMAs
  const bool issuer = crank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int group = a.q_heads / a.kv_heads;
  const int npairs = a.q_heads / 2;
  const int nqt = (a.chunk_len + BM - 1) / BM;
  const int nitems = nqt * npairs * a.batch;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    mbar_init(bars.q(), 1);
    mbar_init(bars.q_free(), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full(i), 1);
      // the issuing CTA also counts the one arrival its peer forwards
      mbar_init(bars.p_full(i), issuer ? 257 : 256);
      mbar_init(bars.pv_done(i), 1);
    }
    mbar_init(bars.o_free(), issuer ? 129 : 128);
    mbar_init(bars.rows_ready(), 128);
    mbar_init(bars.teardown(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
    if (a.k_in) {
      prefetch_tmap(&tm_ki);
      prefetch_tmap(&tm_vi);
    }
  }
  tc_fence_before();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive or copy
  tc_fence_after();
  // programmatic dependent launch: the K/V write launched behind this kernel
  // may start now (it reads only the chunk's inputs); this kernel's own inputs
  // are read after the wait for the kernel launched before it
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;

  // each role's code follows its warpgroup's register split in the same branch
  if (warp < 4) {
  regs_dec<REGS_CTRL>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per item: Q (once the previous item's score products are done), then the
    // ring in the order the MMAs consume it: K_0, K_1, and per tile j: V_j,
    // K_{j+2}.  Both CTAs' halves complete on the even CTA's barriers.
    bool ok = true;
    int idx = 0, qn = 0;
    auto load = [&](int kt, bool is_v, int hk, int b) {
      const int s = idx % NST;
      // polled by one lane: a suspended wait resumes late and eats the ring's lookahead
      bool got = true;
      if (lane == 0) got = wait_spin<false>(bars.empty(s), ((idx / NST) & 1) ^ 1, abort_flag, err);
      ok = __shfl_sync(0xffffffffu, got, 0);
      if (ok && lane == 0) {
        int k0 = kt * BN;
        const uint32_t dst = sRing + s * SLOT;
        const uint32_t bar = map_shared(bars.full(s), 0);
        if (issuer) mbar_arrive_expect_tx(bars.full(s), 2 * SLOT);
        // keys of the chunk itself come from its inputs when the kernel reads them
        const bool from_in = a.k_in != nullptr && k0 >= a.chunk_start;
        if (from_in) k0 -= a.chunk_start;
        if (is_v) {
          // head-dimension columns [128 crank, 128 crank + 128) of all 128 keys
          for (int c = 0; c < 2; ++c)
            tma_load_4d_pair(dst + c * QBOX, from_in ? &tm_vi : &tm_v, bar, 128 * crank + 64 * c, k0, hk, b);
        } else {
          // keys [k0 + 64 crank, k0 + 64 crank + 64), all 256 columns
          for (int c = 0; c < 4; ++c)
            tma_load_4d_pair(dst + c * KBOX, from_in ? &tm_ki : &tm_k, bar, 64 * c, k0 + 64 * crank, hk, b);
        }
      }
      __syncwarp();
      ++idx;
    };
    for (int it = cid; it < nitems && ok; it += ncl) {
      const Item x = item_of(it, npairs, a.batch, nqt);
      const int hq = 2 * x.pair + crank, hk = hq / group;
      int kt_lo, n;
      tile_range(a, x.b, x.qt, kt_lo, n);
      if (n == 0) continue;
      if (qn > 0) ok = __all_sync(0xffffffffu, wait_bar<true>(bars.q_free(), (qn - 1) & 1, abort_flag, err));
      if (!ok) break;
      if (lane == 0) {
        if (issuer) mbar_arrive_expect_tx(bars.q(), 2 * 4 * QBOX);
        for (int c = 0; c < 4; ++c)
          tma_load_4d_pair(sQ + c * QBOX, &tm_q, map_shared(bars.q(), 0), 64 * c, x.qt * BM, hq, x.b);
      }
      __syncwarp();
      ++qn;
      for (int t = 0; t < 2 && t < n && ok; ++t) load(kt_lo + t, false, hk, x.b);
      for (int j = 0; j < n && ok; ++j) {
        load(kt_lo + j, true, hk, x.b);
        if (j + 2 < n && ok) load(kt_lo + j + 2, false, hk, x.b);
      }
    }
  } else if (warp == 1) {
    if (issuer && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      bool ok = true;
      auto commit = [&](uint32_t bar) { mma_pair_commit(bar, 0x3); };
      // S_t = Q K_t^T into S buffer sb from the K half-tiles in ring slot s
      auto qk = [&](int sb, int s) {
        const uint32_t kslot = sRing + s * SLOT;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const int c = kk >> 2;  // 64-column box of the contraction
          const uint64_t ad = sdesc_sw128(sQ + c * QBOX + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kslot + c * KBOX + (kk & 3) * 32, 16, 1024);
          mma_pair_bf16_ss(tmem + TM_S + sb * BN, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      int idx = 0, T = 0, qn = 0, on = 0;
      for (int it = cid; it < nitems && ok; it += ncl) {
        const Item x = item_of(it, npairs, a.batch, nqt);
        int kt_lo, n;
        tile_range(a, x.b, x.qt, kt_lo, n);
        if (n == 0) continue;
        ok = wait_spin<false>(bars.q(), qn & 1, abort_flag, err);
        ++qn;
        for (int t = 0; t < 2 && t < n && ok; ++t) {
          ok = wait_spin<false>(bars.full(idx % NST), (idx / NST) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          qk((T + t) & 1, idx % NST);
          commit(bars.s_full((T + t) & 1));
          commit(bars.empty(idx % NST));
          if (t == n - 1) commit(bars.q_free());
          ++idx;
        }
        // V_j and K_{j+2} of tile j landed: tile 0 here, tile j + 1 right after
        // tile j's MMAs are issued (the wait overlaps their execution)
        auto wait_data = [&](int j) {
          return wait_spin<false>(bars.full(idx % NST), (idx / NST) & 1, abort_flag, err) &&
                 (j + 2 >= n || wait_spin<false>(bars.full((idx + 1) % NST), ((idx + 1) / NST) & 1, abort_flag, err));
        };
        if (ok) ok = wait_data(0);
        // the previous item's epilogue has read O (both CTAs) before PV_0 overwrites it
        if (ok && on > 0) ok = wait_spin<true>(bars.o_free(), (on - 1) & 1, abort_flag, err);
        ++on;
        for (int j = 0; j < n && ok; ++j) {
          const int tj = T + j, sb = tj & 1;
          const bool next = j + 2 < n;  // S_{j+2} goes to the buffer S_j came from
          const int sv = idx % NST, sk = (idx + 1) % NST;
          // P_j written in both CTAs (its data landed already)
          ok = wait_spin<true>(bars.p_full(sb), (tj >> 1) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vslot = sRing + sv * SLOT;
          const uint32_t pbase = tmem + TM_S + sb * BN;
#pragma unroll
          for (int p = 0; p < BN / 16; ++p) {
            // V is [keys][head dim]: MN-major B; 64-column boxes QBOX apart, 8-key
            // row groups 1024 B apart; P_j: 16 keys per step = 8 columns of bf16 pairs
            const uint64_t bd = sdesc_sw128(vslot + p * 2048, QBOX, 1024);
            mma_pair_bf16_ts(tmem + TM_O, pbase + 8 * p, bd, IDESC_PV, (j > 0 || p > 0) ? 1u : 0u);
          }
          commit(bars.pv_done(sb));
          commit(bars.empty(sv));
          if (next) {
            qk(sb, sk);
            commit(bars.s_full(sb));
            commit(bars.empty(sk));
            if (j + 2 == n - 1) commit(bars.q_free());
          }
          idx += next ? 2 : 1;
          if (j + 1 < n) ok = wait_data(j + 1);
        }
        T += n;
      }
    } else if (!issuer && lane == 0) {
      // ---------------------------------------------------------- forwarder
      // each P_j and each finished epilogue of this CTA is announced to the
      // issuing CTA with one cluster-scope arrival
      bool ok = true;
      int T = 0, on = 0;
      for (int it = cid; it < nitems && ok; it += ncl) {
        const Item x = item_of(it, npairs, a.batch, nqt);
        int kt_lo, n;
        tile_range(a, x.b, x.qt, kt_lo, n);
        if (n == 0) continue;
        for (int j = 0; j < n && ok; ++j) {
          const int tj = T + j;
          ok = wait_spin<false>(bars.p_full(tj & 1), (tj >> 1) & 1, abort_flag, err);
          // the softmax threads' tcgen05.wait::st preceded their local arrivals
          if (ok) mbar_arrive_remote_relaxed(map_shared(bars.p_full(tj & 1), 0));
        }
        if (ok) ok = wait_spin<false>(bars.o_free(), on & 1, abort_flag, err);
        if (ok) mbar_arrive_remote_relaxed(map_shared(bars.o_free(), 0));
        ++on;
        T += n;
      }
    }
  }
  } else if (warp < 12) {
    regs_inc<REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax
    const int grp = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    constexpr int HC = BN / 2;  // key columns per group
    const int cb = grp * HC;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    // the two groups of a row exchange through one value per row: group 0
    // writes, both meet, group 1 combines and writes, both meet, group 0 reads
    float* xch = reinterpret_cast<float*>(gbase + OFF_PMAX) + r;
    float2* rows = reinterpret_cast<float2*>(gbase + OFF_ROWS) + r;
    const int bar_id = 1 + q4;  // named barrier of this quadrant's two warps
    const float c2 = a.scale_log2;
    auto combine = [&](float v, bool is_max) {
      if (grp == 0) *xch = v;
      named_sync(bar_id);
      if (grp == 1) *xch = v = is_max ? fmaxf(v, *xch) : v + *xch;
      named_sync(bar_id);
      if (grp == 0) v = *xch;
      return v;
    };
    // The two warps of a row meet at a named barrier for every tile and at the
    // end of every item; a warp that gives up (timeout or abort) keeps meeting
    // its partner there and skips the rest, so the arrivals stay paired.
    bool ok = true;
    int T = 0;
    for (int it = cid; it < nitems; it += ncl) {
      const Item x = item_of(it, npairs, a.batch, nqt);
      const int b = x.b;
      int kt_lo, n;
      tile_range(a, b, x.qt, kt_lo, n);
      if (n == 0) continue;  // the epilogue warps write the zero rows
      const int i = x.qt * BM + r;
      int lo = 0, hi = -1;
      if (i < a.chunk_len) {
        if (a.generic) {
          const PlanLayout L = plan_layout(a.batch, a.chunk_len);
          const char* plan = static_cast<const char*>(a.plan);
          lo = reinterpret_cast<const int32_t*>(plan + L.off_lo)[(long long)b * a.chunk_len + i];
          hi = reinterpret_cast<const int32_t*>(plan + L.off_hi)[(long long)b * a.chunk_len + i];
        } else {
          causal_interval(a.chunk_start + i, a.valid_start ? a.valid_start[b] : 0, a.window, lo, hi);
        }
        hi = min(hi, a.key_rows - 1);
      }
      // m_run: the reference maximum (exp2 domain); l_run sums the bf16-rounded
      // probabilities (normalises O, which the tensor core accumulates from the
      // same rounded values, so O stays a convex combination of V rows);
      // l_exact sums the unrounded ones (gives lse)
      float m_run = -CUDART_INF_F, l_run = 0.f, l_exact = 0.f;
      for (int t = 0; t < n; ++t) {
        const int tt = T + t, sb = tt & 1;
        // polled: a suspended wait resumes late, and S is on the critical path
        if (ok) ok = __all_sync(0xffffffffu, wait_spin<true>(bars.s_full(sb), (tt >> 1) & 1, abort_flag, err));
        if (ok) tc_fence_after();
        const uint32_t tS = tmem + lane_off + TM_S + sb * BN;
        // this group's keys [k0, k0 + 64): columns outside the row's interval are masked
        const int k0 = (kt_lo + t) * BN + cb;
        const bool need_lo = !__all_sync(0xffffffffu, k0 >= lo);
        const bool need_hi = !__all_sync(0xffffffffu, k0 + HC - 1 <= hi);
        uint32_t sr[HC];
        float mraw = -CUDART_INF_F;
        if (ok) {
          tmem_ld32(tS + cb, sr);
          tmem_ld32(tS + cb + 32, sr + 32);
          tmem_ld_wait();
          const int clo = lo - k0, chi = hi - k0;  // admitted columns [clo, chi]
          if (need_lo && need_hi) {
#pragma unroll
            for (int c = 0; c < HC; ++c)
              sr[c] = (c >= clo && c <= chi) ? sr[c] : __float_as_uint(-CUDART_INF_F);
          } else if (need_hi) {  // the diagonal tile: a prefix of the columns
#pragma unroll
            for (int c = 0; c < HC; ++c) sr[c] = c <= chi ? sr[c] : __float_as_uint(-CUDART_INF_F);
          } else if (need_lo) {  // the tile at the window's start: a suffix
#pragma unroll
            for (int c = 0; c < HC; ++c) sr[c] = c >= clo ? sr[c] : __float_as_uint(-CUDART_INF_F);
          }
          float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
          for (int c = 0; c < HC; c += 8) {
            m4[0] = max3(m4[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            m4[1] = max3(m4[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            m4[2] = max3(m4[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
            m4[3] = max3(m4[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
          }
          mraw = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        // the two groups of this row agree on the tile maximum; after this
        // exchange both have read their S columns, so P may overwrite them
        mraw = combine(mraw, true);
        if (!ok) continue;
        const float mt = mraw * c2;
        // lazy rescale: move the reference only when the maximum grows by > 2^32
        const bool move = (m_run == -CUDART_INF_F) ? (mt > -CUDART_INF_F) : (mt > m_run + kRescaleLog2);
        const bool rescale = move && m_run != -CUDART_INF_F;  // O holds data relative to m_run
        if (__any_sync(0xffffffffu, rescale)) {
          // PV of the previous tile, the only MMA that may still write O, must be done
          ok = __all_sync(0xffffffffu, wait_bar<true>(bars.pv_done((tt - 1) & 1), ((tt - 1) >> 1) & 1, abort_flag, err));
          if (!ok) continue;
          tc_fence_after();
          const float alpha = rescale ? exp2f(m_run - mt) : 1.f;
#pragma unroll 1
          for (int c0 = grp * (HD / 2); c0 < (grp + 1) * (HD / 2); c0 += 16) {
            uint32_t o[16];
            tmem_ld16(tmem + lane_off + TM_O + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(tmem + lane_off + TM_O + c0, o);
          }
          tmem_st_wait();
          if (rescale) {
            l_run *= alpha;
            l_exact *= alpha;
          }
        }
        if (move) m_run = mt;
        // probabilities exp2(s * scale_log2 - m_run), packed to bf16 pairs
        const float nm = (m_run == -CUDART_INF_F) ? 0.f : -m_run;
        // the packed pair of scores c, c + 1 replaces score c / 2 (already read)
        uint64_t lr[2] = {0ull, 0ull}, le[2] = {0ull, 0ull};  // packed fp32 pairs
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          float x0 = __uint_as_float(sr[c]), x1 = __uint_as_float(sr[c + 1]);
          fma2(x0, x1, c2, nm);
          const float p0 = ex2(x0), p1 = ex2(x1);  // -inf -> 0
          const uint32_t w = pack_bf16(p0, p1);
          add2(le[(c >> 1) & 1], p0, p1);
          add2(lr[(c >> 1) & 1], __uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
          sr[c / 2] = w;
        }
        l_run += pair_sum(lr[0]) + pair_sum(lr[1]);
        l_exact += pair_sum(le[0]) + pair_sum(le[1]);
        // P: keys [64 grp, 64 grp + 64) go to columns [32 grp, 32 grp + 32) of
        // the S buffer (the A operand layout of PV: 16 keys per 8 columns)
        tmem_st32(tS + 32 * grp, sr);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bars.p_full(sb));
      }
      // the row's normaliser and lse go to the epilogue warps (group 0 holds both
      // groups' sums after the exchanges); their previous values were read
      // before the epilogue released O for this item's first PV
      const float l_tot = combine(l_run, false);
      const float e_tot = combine(l_exact, false);
      if (grp == 0) {
        *rows = make_float2(l_tot > 0.f ? 1.f / l_tot : 0.f,
                            e_tot > 0.f ? (m_run + log2f(e_tot)) * 0.69314718055994530942f : -CUDART_INF_F);
        mbar_arrive(bars.rows_ready());
      }
      T += n;
    }
  } else {
    regs_dec<REGS_EPI>();
    // ------------------------------------------------------------ epilogue
    // Per item: O (this thread's row, 256 columns) / l -> bf16 -> the staging
    // boxes -> TMA stores, in two rounds of 128 columns; O is released for the
    // next item's first PV as soon as the second round's columns are read
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const float2* rows = reinterpret_cast<const float2*>(gbase + OFF_ROWS) + r;
    const bool elected = warp == 12 && lane == 0;
    uint8_t* stage_row = gbase + OFF_STAGE + r * 128;
    auto epi_sync = [] { asm volatile("bar.sync 5, 128;" ::: "memory"); };
    // bf16 pair u (0..7) of 16-byte unit `unit` of this row in staging box g
    auto put = [&](int g, int unit, uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3) {
      *reinterpret_cast<uint4*>(stage_row + g * QBOX + ((unit ^ (r & 7)) << 4)) = make_uint4(x0, x1, x2, x3);
    };
    // the staging boxes hold head-dimension columns [128 h, 128 h + 128): store them
    auto flush = [&](int h, int qt, int hq, int b) {
      fence_proxy_async_smem();
      epi_sync();
      if (elected) {
        for (int g = 0; g < 2; ++g) tma_store_4d(&tm_o, base + OFF_STAGE + g * QBOX, 128 * h + 64 * g, qt * BM, hq, b);
        bulk_commit_group();
      }
    };
    auto staging_free = [&] {
      if (elected) bulk_wait_read_all();  // the previous round's stores have read the staging
      epi_sync();
    };
    bool ok = true;
    int T = 0, on = 0;
    for (int it = cid; it < nitems; it += ncl) {
      const Item x = item_of(it, npairs, a.batch, nqt);
      const int hq = 2 * x.pair + crank, b = x.b;
      int kt_lo, n;
      tile_range(a, b, x.qt, kt_lo, n);
      const int i = x.qt * BM + r;
      float inv = 0.f, lse = -CUDART_INF_F;
      bool have_o = false;
      if (n > 0) {
        if (ok) ok = __all_sync(0xffffffffu, wait_bar<false>(bars.rows_ready(), on & 1, abort_flag, err));
        if (ok)
          ok = __all_sync(0xffffffffu, wait_bar<true>(bars.pv_done((T + n - 1) & 1), ((T + n - 1) >> 1) & 1,
                                                      abort_flag, err));
        tc_fence_after();
        have_o = ok;
        if (ok) {
          const float2 v = *rows;
          inv = v.x;
          lse = v.y;
        }
      }
      auto cvt = [&](const uint32_t* o, int e) {
        return have_o ? pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv) : 0u;
      };
      // round 0: columns [0, 128) straight into the staging boxes
      staging_free();
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        uint32_t o[32];
        if (have_o) {
          tmem_ld32(tmem + lane_off + TM_O + 32 * h4, o);
          tmem_ld_wait();
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          put(h4 >> 1, (h4 & 1) * 4 + u, cvt(o, 4 * u), cvt(o, 4 * u + 1), cvt(o, 4 * u + 2), cvt(o, 4 * u + 3));
      }
      flush(0, x.qt, hq, b);
      // round 1: columns [128, 256) into registers; then O is free
      uint32_t w[64];
#pragma unroll
      for (int h8 = 0; h8 < 8; ++h8) {
        uint32_t o[16];
        if (have_o) {
          tmem_ld16(tmem + lane_off + TM_O + 128 + 16 * h8, o);
          tmem_ld_wait();
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) w[8 * h8 + e] = cvt(o, e);
      }
      if (n > 0) {  // O read: the next item's first PV may overwrite it
        tc_fence_before();
        mbar_arrive(bars.o_free());
        ++on;
      }
      staging_free();
#pragma unroll
      for (int u = 0; u < 16; ++u) put(u >> 3, u & 7, w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
      flush(1, x.qt, hq, b);
      if (a.lse && i < a.chunk_len) a.lse[((long long)b * a.chunk_len + i) * a.q_heads + hq] = lse;
      T += n;
    }
  }

  // ------------------------------------------------------------ teardown
  if (warp == 12 && lane == 0) bulk_wait_all();  // the output stores have completed
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let the MMAs and TMA copies this CTA issued finish before TMEM and
    // shared memory are released
    if (warp == 1 && lane == 0 && issuer) {
      mma_pair_commit(bars.teardown(), 0x1);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bars.teardown(), 0) && globaltimer_ns() - t0 < kTimeoutNs) {
      }
    }
    if (warp == 0 && lane == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
    __syncthreads();
  }
  cluster_sync();  // the peer no longer reads or writes this CTA's shared memory or TMEM
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, TM_COLS);
}

}  // namespace

// Clusters of two prefill CTAs the current device runs at once (cached per device).
int max_clusters() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_pair256_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      int sms = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      n = sms > 1 ? sms / 2 : 1;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t launch_prefill_pair256(const PrefillArgs& a, cudaStream_t s) {
  if (a.head_dim != HD || (a.q_heads / a.kv_heads) % 2 != 0) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_pair256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint64_t D = HD;
  CUtensorMap mq, mk, mv;
  // K / V: dims {D, key rows, Hkv, B} with the caller's strides; K in boxes of
  // 64 keys (one CTA's half of a tile), V in boxes of 128 keys
  const uint64_t kd[4] = {D, uint64_t(a.key_dim_rows), uint64_t(a.kv_heads), uint64_t(a.batch)};
  const uint64_t ks[3] = {uint64_t(a.key_row_stride) * 2, uint64_t(a.key_head_stride) * 2,
                          uint64_t(a.key_seq_stride > 0 ? a.key_seq_stride : a.key_dim_rows * a.key_row_stride) * 2};
  // Q [B, C, Hq, D]: dims {D, C, Hq, B}
  const uint64_t qd[4] = {D, uint64_t(a.chunk_len), uint64_t(a.q_heads), uint64_t(a.batch)};
  const uint64_t qs[3] = {uint64_t(a.q_heads) * D * 2, D * 2, uint64_t(a.chunk_len) * a.q_heads * D * 2};
  CUtensorMap mo;  // the output has Q's layout
  if (!make_tmap_bf16(&mk, a.k, kd, ks, BN / 2) || !make_tmap_bf16(&mv, a.v, kd, ks, BN) ||
      !make_tmap_bf16(&mq, a.q, qd, qs, BM) || !make_tmap_bf16(&mo, a.out, qd, qs, BM))
    return cudaErrorInvalidValue;
  // the chunk's own K/V [B, C, Hkv, D]: dims {D, C, Hkv, B}
  CUtensorMap mki = mk, mvi = mv;
  if (a.k_in) {
    const uint64_t id[4] = {D, uint64_t(a.chunk_len), uint64_t(a.kv_heads), uint64_t(a.batch)};
    const uint64_t is[3] = {uint64_t(a.kv_heads) * D * 2, D * 2, uint64_t(a.chunk_len) * a.kv_heads * D * 2};
    if (!make_tmap_bf16(&mki, a.k_in, id, is, BN / 2) || !make_tmap_bf16(&mvi, a.v_in, id, is, BN))
      return cudaErrorInvalidValue;
  }
  const int nqt = (a.chunk_len + BM - 1) / BM;
  const long long nitems = (long long)nqt * (a.q_heads / 2) * a.batch;
  const int ncl = int(std::min<long long>(nitems, max_clusters()));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ncl, 1, 1);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // programmatic dependent launch: set-up overlaps the previous kernel's tail
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, prefill_pair256_kernel, mq, mk, mv, mo, mki, mvi, a);
}

bool prefill_reads_chunk_inputs(const PrefillArgs& a) {
  return a.head_dim == HD && (a.q_heads / a.kv_heads) % 2 == 0 && a.k_in != nullptr && a.v_in != nullptr &&
         a.chunk_start % BN == 0;
}

}  // namespace swa
