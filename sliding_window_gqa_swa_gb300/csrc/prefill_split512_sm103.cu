// Prefill attention at head size 512 for an even GQA group, with every
// product computed once.  The output row of 512 fp32 columns fills a whole
// tensor memory, so no CTA can hold O beside its scores; the work of one
// (head pair, 128-row query tile) item is split over a cluster of four CTAs:
//
//   ranks 0, 1 (score pair): query heads 2g and 2g + 1 of one KV head, the
//     same 128 query rows.  Q is staged once through shared memory into
//     tensor memory (A operand of every score MMA).  S = Q K^T over the whole
//     512-column contraction with pair MMAs (cta_group::2, M = 256: rank 0
//     holds head 2g's rows, rank 1 head 2g + 1's) on 128-key tiles: N = 128
//     runs the tensor pipe at its full rate (N = 64 would cost ~45 SM clocks
//     per 32 clocks of work).  Q and two S buffers fill the tensor memory, so
//     S_{t+1} is computed while the softmax works on S_t.
//     Each warp writes its 32 rows of P (bf16) into local staging and sends
//     them with one bulk copy into the shared memory of the output CTA of
//     the same head (rank + 2), the rows' rescale factors with remote
//     stores; both count their bytes on that CTA's barrier;
//   ranks 2, 3 (output pair): O (128 rows x 512 columns, fp32, all of tensor
//     memory) += P V with pair MMAs, two N = 256 halves per 16-key step, P
//     from the received buffer and V from a ring of TMA tiles.  A rescale
//     factor other than 1 (the row maximum grew by more than 2^8) is applied
//     to O before the tile's product; at the end O / l goes out through
//     shared-memory staging and TMA stores.
// Both pairs do the same tensor work per key tile (Q K^T: 256 x 128 x 512;
// P V: 256 x 512 x 128), so in steady state neither waits for the other, and
// the head-512 forward does the algorithmic FLOP only.
//
// Warp roles (320 threads in every CTA):
//   warp 0      TMA producer: Q once (into K ring slots 2-3 and the P
//               staging, which it leaves before either is used) and K
//               tiles (score pair: two slots per tile, the contraction
//               halves), V tiles (output pair: two slots per tile, 64 keys
//               each), into rings of 32 KB slots (128-byte swizzle);
//   warp 1      lane 0 of the even CTA of each pair issues that pair's MMAs;
//               in rank 1 it forwards "S read" to rank 0;
//   warps 2-9   score pair: Q into TMEM, then the softmax, two warpgroups
//               of one query row per thread (TMEM lane), group g owning keys
//               [64g, 64g + 64) of a tile; output pair: warps 4-7 apply the
//               rescale factors, and all eight write the output.
// Every wait is bounded; a timeout sets the device error word, makes the
// CTA's roles stop, lets its in-flight copies and MMAs finish, and frees TMEM.
//
// Sources: "Add SDPA attention implementation", Summary (packed documents,
// head size 512, K/V shared by query-head groups); "Enable compact
// sliding-window attention for Gemma 3 and Gemma 4 variants", Compilation
// behavior (the generic plan's per-row key intervals).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace swa {
namespace {

using namespace ptx;

constexpr int BM = kPlanBM;  // 128 query rows per item
constexpr int BN = 128;      // keys per tile
constexpr int HD = 512;      // head size
constexpr int THREADS = 320;
constexpr int Q_BOX = BM * 128;        // one 64-column box of Q: 16 KB
constexpr int Q_BYTES = Q_BOX * (HD / 64);
constexpr int K_BOX = (BN / 2) * 128;  // this CTA's 64 keys of one 64-column box of K: 8 KB
constexpr int K_SLOT = K_BOX * 4;      // one contraction half (256 columns) of them
constexpr int V_BOX = 64 * 128;        // 64 keys of one 64-column box of V: 8 KB
constexpr int V_SLOT = V_BOX * 4;      // 64 keys x this CTA's 256 columns of V
constexpr int P_BYTES = BM * BN * 2;   // one tile of P: 32 KB (two 64-key halves)
constexpr int NSTK = 4;                // K ring slots, two per tile
constexpr int NSTV = 4;                // V ring slots, two per tile
constexpr int NB = 2;                  // P buffers in each output CTA
constexpr int NS = 2;                  // S buffers in the score pair's TMEM
constexpr int KSTEPS = HD / 16;        // K = 16 steps of one score tile

// Shared memory (bytes from the 1024-aligned base).  The score and output
// CTAs use the main region differently; the barriers sit at the same offset
// in every CTA, so a multicast commit reaches the same barrier in each.
constexpr int OFF_K = 0;                              // score: K ring
constexpr int OFF_PSTAGE = OFF_K + NSTK * K_SLOT;     // score: P staging [NB]
constexpr int OFF_QSTAGE = OFF_K + 2 * K_SLOT;        // score: Q [8 boxes] until it is in TMEM
constexpr int OFF_V = 0;                              // output: V ring (the output staging at the end)
constexpr int OFF_RECV = OFF_V + NSTV * V_SLOT;       // output: P buffers
constexpr int OFF_ALPHA = OFF_RECV + NB * P_BYTES;    // output: rescale factors [NB][128]
constexpr int OFF_FIN = OFF_ALPHA + NB * BM * 4;      // output: 1 / l [128]
constexpr int MAIN_SCORE = OFF_PSTAGE + NB * P_BYTES, MAIN_OUT = OFF_FIN + BM * 4;
constexpr int MAIN = MAIN_SCORE > MAIN_OUT ? MAIN_SCORE : MAIN_OUT;
static_assert(OFF_QSTAGE + Q_BYTES <= MAIN_SCORE, "Q staging");
static_assert(8 * Q_BOX <= NSTV * V_SLOT, "output staging reuses the V ring");
constexpr int OFF_PMAX = MAIN;                        // score: [2 tiles][2 groups][128 rows] fp32
constexpr int OFF_BAR = OFF_PMAX + 4 * BM * 4;
constexpr int N_BARS = 2 * NSTK + 1 + 2 * NS + NB + 2 * NSTV + 2 * NB + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024 B
static_assert(SMEM <= 232448, "shared memory budget");

// score CTAs: S buffer b in columns [128 b, 128 b + 128), Q in [256, 512)
// (column c holds the bf16 pair of contraction columns 2c, 2c + 1); output
// CTAs: O
constexpr uint32_t TM_Q = NS * BN;
constexpr uint32_t TM_COLS = 512;
static_assert(TM_Q + HD / 2 <= TM_COLS, "score TMEM budget");
constexpr uint32_t IDESC_QK2 = idesc_bf16_f32(2 * BM, BN, false);
static_assert(BN <= 256 && TM_Q + HD / 2 <= 512, "tensor memory");
constexpr uint32_t IDESC_PV2 = idesc_bf16_f32(2 * BM, 256, true);
constexpr float kRescaleLog2 = 8.f;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Bars {
  uint32_t base;
  __device__ uint32_t at(int i) const { return base + 8 * i; }
  __device__ uint32_t k_full(int s) const { return at(s); }
  __device__ uint32_t k_empty(int s) const { return at(NSTK + s); }
  __device__ uint32_t q() const { return at(2 * NSTK); }
  __device__ uint32_t s_full(int b) const { return at(2 * NSTK + 1 + b); }
  __device__ uint32_t s_free(int b) const { return at(2 * NSTK + 1 + NS + b); }
  // score CTAs: the output pair's MMAs finished reading P buffer b
  __device__ uint32_t recv_free(int b) const { return at(2 * NSTK + 1 + 2 * NS + b); }
  __device__ uint32_t v_full(int s) const { return at(2 * NSTK + 1 + 2 * NS + NB + s); }
  __device__ uint32_t v_empty(int s) const { return at(2 * NSTK + 1 + 2 * NS + NB + NSTV + s); }
  // output CTAs: P buffer b and its factors arrived (transaction bytes)
  __device__ uint32_t p_recv(int b) const { return at(2 * NSTK + 1 + 2 * NS + NB + 2 * NSTV + b); }
  // output leader: both output CTAs rescaled O for the tile in buffer b
  __device__ uint32_t ready(int b) const { return at(2 * NSTK + 1 + 2 * NS + 2 * NB + 2 * NSTV + b); }
  __device__ uint32_t pv_done(int b) const { return at(2 * NSTK + 1 + 2 * NS + 3 * NB + 2 * NSTV + b); }
  __device__ uint32_t fin() const { return at(2 * NSTK + 1 + 2 * NS + 3 * NB + 2 * NSTV + 2); }
  __device__ uint32_t teardown() const { return at(2 * NSTK + 1 + 2 * NS + 3 * NB + 2 * NSTV + 3); }
  // score CTAs: Q is in TMEM (the leader also counts its peer's forwarded arrival)
  __device__ uint32_t q_tmem() const { return at(2 * NSTK + 1 + 2 * NS + 3 * NB + 2 * NSTV + 4); }
};

// Bounded wait on one phase of an mbarrier (the whole warp polls).  Gives up
// when another role has aborted or after kTimeoutNs, recording the timeout.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  auto poll = [&] { return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
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

// Bounded wait of the single thread on the critical path (an MMA issuer, the
// forwarder): polled with test_wait, because a thread suspended in try_wait
// can resume well over a thousand SM clocks after the phase completed.
// kCluster: the phase completes by a peer's relaxed arrival, so a successful
// test is followed by an acquire fence at cluster scope.
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

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Key tiles of one item: [kt_lo, kt_lo + n) of BN keys.
__device__ __forceinline__ void tile_range(const PrefillArgs& a, int b, int qt, int& kt_lo, int& n) {
  const int q0 = a.chunk_start + qt * BM;
  int k_lo = 0, k_hi = 0;
  if (a.generic) {
    const PlanLayout L = plan_layout(a.batch, a.chunk_len);
    const int nqt = (a.chunk_len + BM - 1) / BM;
    const char* plan = static_cast<const char*>(a.plan);
    k_lo = reinterpret_cast<const int32_t*>(plan + L.off_tlo)[b * nqt + qt];
    k_hi = reinterpret_cast<const int32_t*>(plan + L.off_thi)[b * nqt + qt];
  } else {
    const int vs = a.valid_start ? a.valid_start[b] : 0;
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

__global__ void __launch_bounds__(THREADS, 1)
prefill_split512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const Bars bars{base + OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_MISC + 4);
  int32_t* err = a.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = int(cluster_ctarank());
  const bool score = crank < 2;           // score pair (ranks 0, 1) or output pair (2, 3)
  const bool leader = (crank & 1) == 0;   // issues its pair's MMAs
  const int lead_rank = crank & 2;        // the leader of this CTA's pair
  const int hq = 2 * int(blockIdx.x >> 2) + (crank & 1);
  const int hk = hq / (a.q_heads / a.kv_heads);
  // query tiles late in a causal sequence or document have the most key
  // tiles: they are scheduled first, so the short ones fill the tail
  const int qt = int(gridDim.y - 1 - blockIdx.y), b = blockIdx.z;
  const int i0 = qt * BM;
  int kt_lo, n;
  tile_range(a, b, qt, kt_lo, n);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTK; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
    }
    mbar_init(bars.q(), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(bars.s_full(i), 1);
      // the score leader also counts the one arrival its peer forwards
      mbar_init(bars.s_free(i), crank == 0 ? 257 : 256);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(bars.recv_free(i), 1);
      mbar_init(bars.p_recv(i), 1);
      mbar_init(bars.ready(i), 8);  // the four rescaling warps of both output CTAs
    }
    for (int s = 0; s < NSTV; ++s) {
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(bars.pv_done(i), 1);
    mbar_init(bars.fin(), 1);
    mbar_init(bars.teardown(), 1);
    mbar_init(bars.q_tmem(), crank == 0 ? 257 : 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    if (score) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
    } else {
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_o);
    }
  }
  tc_fence_before();
  cluster_sync();  // every CTA's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (one lane; its waits are polled: a suspended wait resumes late and eats
    // the ring's lookahead)
    if (n > 0 && lane == 0) {
      bool ok = true;
      if (score) {
        // this CTA's Q rows into the staging slots (this CTA's softmax
        // threads move them to TMEM)
        mbar_arrive_expect_tx(bars.q(), Q_BYTES);
        for (int c = 0; c < HD / 64; ++c) tma_load_4d(base + OFF_QSTAGE + c * Q_BOX, &tm_q, bars.q(), 64 * c, i0, hq, b);
        // K tile t: this CTA's 64 of its 128 keys; slot 2t % NSTK holds
        // contraction columns [0, 256), the next slot [256, 512).  Tile 1
        // goes to slots 2-3 once Q has left them (P_0 is written after S_0,
        // which needs Q in TMEM)
        for (int t = 0; t < n && ok; ++t) {
          if (t == 1) ok = wait_bar<true>(bars.q_tmem(), 0, abort_flag, err);
          const int k0 = (kt_lo + t) * BN + (crank & 1) * (BN / 2);
          for (int h = 0; h < 2 && ok; ++h) {
            const int u = 2 * t + h, s = u % NSTK;
            ok = wait_spin<true>(bars.k_empty(s), ((u / NSTK) & 1) ^ 1, abort_flag, err);
            if (!ok) break;
            if (leader) mbar_arrive_expect_tx(bars.k_full(s), 2 * K_SLOT);
            for (int c = 0; c < 4; ++c)
              tma_load_4d_pair(base + OFF_K + s * K_SLOT + c * K_BOX, &tm_k, map_shared(bars.k_full(s), lead_rank),
                               256 * h + 64 * c, k0, hk, b);
          }
        }
      } else {
        // V tile t, keys [64 h, 64 h + 64) in slot (2t + h) % NSTV: head-dimension
        // columns 256 m + 128 (rank & 1) + [0, 128) for the two N = 256 halves m
        for (int t = 0; t < n && ok; ++t) {
          for (int h = 0; h < 2 && ok; ++h) {
            const int u = 2 * t + h, s = u % NSTV;
            ok = wait_spin<true>(bars.v_empty(s), ((u / NSTV) & 1) ^ 1, abort_flag, err);
            if (!ok) break;
            if (leader) mbar_arrive_expect_tx(bars.v_full(s), 2 * V_SLOT);
            const int k0 = (kt_lo + t) * BN + 64 * h;
            for (int c = 0; c < 4; ++c)
              tma_load_4d_pair(base + OFF_V + s * V_SLOT + c * V_BOX, &tm_v, map_shared(bars.v_full(s), lead_rank),
                               256 * (c >> 1) + 128 * (crank & 1) + 64 * (c & 1), k0, hk, b);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (n > 0 && lane == 0) {
      bool ok = true;
      if (score && leader) {
        // ---------------------------------------------------------- score MMAs
        // S_t = Q K_t^T into S buffer t % 2: 32 steps of K = 16, the first
        // 16 from the slot of contraction columns [0, 256), the rest from the
        // next.  The descriptors of a slot differ by constants (the start
        // address is bits 0-13 in 16-byte units), so each step is one add.
        ok = wait_spin<true>(bars.q_tmem(), 0, abort_flag, err);
        const uint64_t kdesc0 = sdesc_sw128(base + OFF_K, 16, 1024);
        for (int t = 0; t < n && ok; ++t) {
          const int sb = t % NS, s0 = (2 * t) % NSTK, s1 = (2 * t + 1) % NSTK;
          // the softmax read S_{t-2} (both CTAs); K_t is in both halves' slots
          if (t >= NS) ok = wait_spin<true>(bars.s_free(sb), ((t / NS) - 1) & 1, abort_flag, err);
          if (ok) ok = wait_spin<false>(bars.k_full(s0), ((2 * t) / NSTK) & 1, abort_flag, err);
          if (ok) ok = wait_spin<false>(bars.k_full(s1), ((2 * t + 1) / NSTK) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bd[2] = {kdesc0 + uint64_t((s0 * K_SLOT) >> 4), kdesc0 + uint64_t((s1 * K_SLOT) >> 4)};
          const uint32_t d = tmem + sb * BN;
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const int h = kk >> 4, kl = kk & 15;
            mma_pair_bf16_ts(d, tmem + TM_Q + kk * 8, bd[h] + uint64_t(((kl >> 2) * K_BOX + (kl & 3) * 32) >> 4),
                             IDESC_QK2, kk ? 1u : 0u);
          }
          mma_pair_commit(bars.k_empty(s0), 0x3);
          mma_pair_commit(bars.k_empty(s1), 0x3);
          mma_pair_commit(bars.s_full(sb), 0x3);
        }
      } else if (score) {
        // ---------------------------------------------------------- forwarder
        // rank 1 tells the leader that its Q is in TMEM and that its softmax
        // read S_t, with relaxed cluster-scope arrivals: the tensor-memory
        // accesses finished (tcgen05.wait) before the local arrivals, and the
        // leader acquires at cluster scope
        ok = wait_spin<false>(bars.q_tmem(), 0, abort_flag, err);
        if (ok) mbar_arrive_remote_relaxed(map_shared(bars.q_tmem(), 0));
        for (int t = 0; t < n && ok; ++t) {
          ok = wait_spin<false>(bars.s_free(t % NS), (t / NS) & 1, abort_flag, err);
          if (ok) mbar_arrive_remote_relaxed(map_shared(bars.s_free(t % NS), 0));
        }
      } else if (leader) {
        // ---------------------------------------------------------- output MMAs
        // O[:, 256 m + (0..255)] += P_t V_t[:, 256 m + (0..255)], 16 keys per step
        for (int t = 0; t < n && ok; ++t) {
          const int pb = t % NB, s0 = (2 * t) % NSTV, s1 = (2 * t + 1) % NSTV;
          ok = wait_spin<true>(bars.ready(pb), (t / NB) & 1, abort_flag, err) &&
               wait_spin<false>(bars.v_full(s0), ((2 * t) / NSTV) & 1, abort_flag, err) &&
               wait_spin<false>(bars.v_full(s1), ((2 * t + 1) / NSTV) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pbuf = base + OFF_RECV + pb * P_BYTES;
#pragma unroll
          for (int p = 0; p < BN / 16; ++p) {
            // P (K-major, two 64-key halves of 128-byte rows): 16 keys = 32
            // bytes per step.  V is [keys][head dim]: MN-major B, 64-column
            // boxes V_BOX apart, 8-key row groups 1024 B apart
            const uint64_t ad = sdesc_sw128(pbuf + (p >> 2) * (P_BYTES / 2) + (p & 3) * 32, 16, 1024);
            const uint32_t vs = base + OFF_V + ((p >> 2) ? s1 : s0) * V_SLOT + (p & 3) * 2048;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const uint64_t bd = sdesc_sw128(vs + m * 2 * V_BOX, V_BOX, 1024);
              mma_pair_bf16_ss(tmem + 256 * m, ad, bd, IDESC_PV2, (t > 0 || p > 0) ? 1u : 0u);
            }
          }
          mma_pair_commit(bars.v_empty(s0), 0xC);
          mma_pair_commit(bars.v_empty(s1), 0xC);
          mma_pair_commit(bars.recv_free(pb), 0x3);  // the score CTAs may refill buffer pb
          mma_pair_commit(bars.pv_done(t & 1), 0xC);
        }
      }
    }
    __syncwarp();
  } else if (score) {
    // ------------------------------------------------------------ softmax
    // Warp w serves TMEM lane quadrant (w % 4), one query row per thread; the
    // two threads of a row (one per group) take identical rescaling decisions
    // because both see the same row maximum.
    const int grp = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int i = i0 + r;
    const bool row_ok = i < a.chunk_len;
    int lo = 0, hi = -1;
    if (row_ok) {
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
    constexpr int HC = BN / 2;  // keys per group
    const int cb = grp * HC;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    float* pmax = reinterpret_cast<float*>(gbase + OFF_PMAX);  // [group][row]
    const int bar_id = 1 + q4;  // named barrier of this quadrant's two warps
    const int out_rank = crank + 2;
    // this warp's 32 rows of this group's 64-key half of P (4 KB, the same
    // layout in the staging and in the output CTA's buffers), and the row's
    // factor in the output CTA
    const uint32_t p_off = grp * (P_BYTES / 2) + q4 * 32 * 128;
    uint8_t* stage_row = gbase + OFF_PSTAGE + p_off + lane * 128;
    const uint32_t recv_warp = map_shared(base + OFF_RECV, out_rank) + p_off;
    const uint32_t alpha_row = map_shared(base + OFF_ALPHA, out_rank) + r * 4;
    const float c2 = a.scale_log2;

    bool ok = true;
    if (n > 0) {
      // Q row r, contraction columns [256 grp, 256 grp + 256): staging boxes
      // 4 grp .. 4 grp + 3 -> TMEM columns TM_Q + 128 grp + [0, 128)
      ok = __all_sync(0xffffffffu, wait_bar(bars.q(), 0, abort_flag, err));
      if (ok) {
        const uint8_t* qrow = gbase + OFF_QSTAGE + r * 128;
#pragma unroll 1
        for (int c = 4 * grp; c < 4 * grp + 4; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + c * Q_BOX + ((u ^ (r & 7)) << 4));
            w[4 * u] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
          }
          tmem_st32(tmem + lane_off + TM_Q + 32 * c, w);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bars.q_tmem());
      }
    }

    // m_run is the reference maximum in the exp2 domain; l_run sums the
    // bf16-rounded probabilities (normalises O, which the tensor core
    // accumulates from the same rounded values); l_exact sums the unrounded
    // ones (gives the lse)
    float m_run = -CUDART_INF_F, l_run = 0.f, l_exact = 0.f;
    // The two warps of a row meet at a named barrier for every tile; a warp
    // that gives up keeps meeting its partner there and skips the rest.
    for (int t = 0; t < n; ++t) {
      const int pb = t % NB;
      // polled: a suspended wait resumes late, and S is on the critical path
      if (ok) ok = __all_sync(0xffffffffu, wait_spin<true>(bars.s_full(t % NS), (t / NS) & 1, abort_flag, err));
      if (ok) tc_fence_after();
      const uint32_t tS = tmem + lane_off + (t % NS) * BN + cb;
      const int k0 = (kt_lo + t) * BN;
      const bool masked = !__all_sync(0xffffffffu, (k0 >= lo) && (k0 + BN - 1 <= hi));
      uint32_t sr[HC];
      float mraw = -CUDART_INF_F;
      if (ok) {
        // this group's 64 scores; the S buffer is released for S_{t+2} as
        // soon as it is read
        tmem_ld32(tS, sr);
        tmem_ld32(tS + 32, sr + 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bars.s_free(t % NS));
        // keys outside the row's interval [lo, hi] -> -inf
        if (masked) {
          const int clo = lo - (k0 + cb), chi = hi - (k0 + cb);
#pragma unroll
          for (int c = 0; c < HC; ++c)
            if (c < clo || c > chi) sr[c] = __float_as_uint(-CUDART_INF_F);
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
      // the two groups of this row agree on the tile maximum (pmax is double
      // buffered by tile parity, so one barrier per tile suffices)
      float* pm = pmax + (t & 1) * 2 * BM;
      pm[grp * BM + r] = mraw;
      named_sync(bar_id, 64);
      mraw = fmaxf(mraw, pm[(grp ^ 1) * BM + r]);
      if (!ok) continue;
      const float mt = mraw * c2;
      // lazy rescale: move the reference only when the maximum grows by > 2^8
      const bool move = (m_run == -CUDART_INF_F) ? (mt > -CUDART_INF_F) : (mt > m_run + kRescaleLog2);
      const bool rescale = move && m_run != -CUDART_INF_F;  // O holds data relative to m_run
      const float alpha = rescale ? exp2f(m_run - mt) : 1.f;
      if (rescale) {
        l_run *= alpha;
        l_exact *= alpha;
      }
      if (move) m_run = mt;
      // probabilities exp2(s * scale_log2 - m_run), packed to bf16 pairs
      const float nm = (m_run == -CUDART_INF_F) ? 0.f : -m_run;
      uint64_t lr[2] = {0ull, 0ull}, le[2] = {0ull, 0ull};  // packed fp32 pairs
#pragma unroll
      for (int c = 0; c < HC; c += 2) {
        float x0 = __uint_as_float(sr[c]), x1 = __uint_as_float(sr[c + 1]);
        fma2(x0, x1, c2, nm);
        const float p0 = ex2(x0), p1 = ex2(x1);  // -inf -> 0
        const uint32_t w = pack_bf16(p0, p1);
        add2(le[(c >> 1) & 1], p0, p1);
        add2(lr[(c >> 1) & 1], __uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
        sr[c / 2] = w;  // score c / 2 was read already
      }
      l_run += pair_sum(lr[0]) + pair_sum(lr[1]);
      l_exact += pair_sum(le[0]) + pair_sum(le[1]);
      // staging pb (and the output CTA's buffer pb) is free once the output
      // pair's PV of tile t - NB completed
      if (t >= NB) ok = __all_sync(0xffffffffu, wait_bar<true>(bars.recv_free(pb), ((t / NB) - 1) & 1, abort_flag, err));
      if (!ok) continue;
      // P_t -> staging (K-major, 128-byte swizzle: 16-byte unit u of row r at
      // u ^ (r % 8)), then this warp's 4 KB -> the output CTA in one bulk
      // copy; it and the factors count their bytes on the output CTA's p_recv(pb)
      const uint32_t pbar = map_shared(bars.p_recv(pb), out_rank);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(stage_row + pb * P_BYTES + ((u ^ (r & 7)) << 4)) =
            make_uint4(sr[4 * u], sr[4 * u + 1], sr[4 * u + 2], sr[4 * u + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) bulk_copy_to_peer(recv_warp + pb * P_BYTES, base + OFF_PSTAGE + pb * P_BYTES + p_off, 4096, pbar);
      if (grp == 0) st_async_u32(alpha_row + pb * (BM * 4), __float_as_uint(alpha), pbar);
    }
    // row sums of both groups
    named_sync(bar_id, 64);
    pmax[grp * BM + r] = l_run;
    named_sync(bar_id, 64);
    const float l_tot = l_run + pmax[(grp ^ 1) * BM + r];
    named_sync(bar_id, 64);
    pmax[grp * BM + r] = l_exact;
    named_sync(bar_id, 64);
    const float e_tot = l_exact + pmax[(grp ^ 1) * BM + r];
    if (grp == 0) {
      // 1 / l -> the output CTA (counted on its fin barrier); the lse here
      if (n > 0)
        st_async_u32(map_shared(base + OFF_FIN + r * 4, out_rank),
                     __float_as_uint(ok && l_tot > 0.f ? 1.f / l_tot : 0.f), map_shared(bars.fin(), out_rank));
      if (row_ok && a.lse)
        a.lse[((long long)b * a.chunk_len + i) * a.q_heads + hq] =
            n > 0 && ok && e_tot > 0.f ? (m_run + log2f(e_tot)) * 0.69314718055994530942f : -CUDART_INF_F;
    }
    // the output pair's last commits to recv_free have landed before this CTA
    // leaves (nothing arrives in its shared memory after the teardown)
    if (warp == 2 && lane == 0 && ok)
      for (int t = max(0, n - NB); t < n; ++t)
        if (!wait_bar<true>(bars.recv_free(t % NB), (t / NB) & 1, abort_flag, err)) break;
  } else {
    // ------------------------------------------------------------ output rows
    // One row per thread (TMEM lane quadrant warp % 4).  Warps 4-7 apply each
    // tile's rescale factor to O before its product; then all eight warps
    // write O / l, warpgroup e (warps 4-7: e = 0; 8, 9, 2, 3: e = 1) the
    // output columns [256 e, 256 e + 256).
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int eg = (warp >= 4 && warp < 8) ? 0 : 1;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const bool elected = warp == 4 && lane == 0;
    bool ok = true;
    if (eg == 0) {
      if (n > 0 && elected) mbar_arrive_expect_tx(bars.fin(), BM * 4);
      for (int t = 0; t < n && ok; ++t) {
        const int pb = t % NB;
        if (elected) mbar_arrive_expect_tx(bars.p_recv(pb), P_BYTES + BM * 4);
        ok = __all_sync(0xffffffffu, wait_spin<true>(bars.p_recv(pb), (t / NB) & 1, abort_flag, err));
        if (!ok) break;
        // the received P is read next by the tensor core (async proxy)
        fence_proxy_async_smem();
        const float alpha = reinterpret_cast<const float*>(gbase + OFF_ALPHA + pb * (BM * 4))[r];
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // O of tile t - 1 must be complete (t >= 1: the first tile never rescales)
          ok = __all_sync(0xffffffffu,
                          wait_bar<true>(bars.pv_done((t - 1) & 1), ((t - 1) >> 1) & 1, abort_flag, err));
          if (!ok) break;
          tc_fence_after();
          for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_off + c0, o);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(bars.ready(pb));
          else
            mbar_arrive_remote_relaxed(map_shared(bars.ready(pb), lead_rank));
        }
      }
    }
    // epilogue: O / l -> bf16 -> staging boxes (the drained V ring) -> TMA stores
    float inv = 0.f;
    bool have_o = false;
    if (n > 0) {
      if (ok) ok = __all_sync(0xffffffffu, wait_bar<true>(bars.fin(), 0, abort_flag, err));
      if (ok)
        ok = __all_sync(0xffffffffu,
                        wait_bar<true>(bars.pv_done((n - 1) & 1), ((n - 1) >> 1) & 1, abort_flag, err));
      tc_fence_after();
      have_o = ok;
      if (ok) inv = reinterpret_cast<const float*>(gbase + OFF_FIN)[r];
    }
    uint8_t* stage_row = gbase + OFF_V + r * 128;
#pragma unroll 1
    for (int g = 4 * eg; g < 4 * eg + 4; ++g) {
      uint32_t o[64];
      if (have_o) {
        tmem_ld32(tmem + lane_off + 64 * g, o);
        tmem_ld32(tmem + lane_off + 64 * g + 32, o + 32);
        tmem_ld_wait();
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 8 * u + 2 * e;
          w[e] = have_o ? pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv) : 0u;
        }
        *reinterpret_cast<uint4*>(stage_row + g * Q_BOX + ((u ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    named_sync(5, 256);
    if (elected) {
      for (int g = 0; g < HD / 64; ++g) tma_store_4d(&tm_o, base + OFF_V + g * Q_BOX, 64 * g, i0, hq, b);
      bulk_commit_group();
      bulk_wait_read_all();  // shared memory is released at the teardown
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let the MMAs and TMA copies this CTA issued finish before TMEM and
    // shared memory are released
    if (warp == 1 && lane == 0 && leader) {
      mma_pair_commit(bars.teardown(), uint16_t(1u << crank));
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
  cluster_sync();  // no CTA reads or writes another's shared memory any more
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, TM_COLS);
}

}  // namespace

bool prefill_split512_eligible(const PrefillArgs& a) {
  return a.head_dim == HD && a.kv_heads > 0 && (a.q_heads / a.kv_heads) % 2 == 0;
}

cudaError_t launch_prefill_split512(const PrefillArgs& a, cudaStream_t s) {
  if (!prefill_split512_eligible(a)) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_split512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint64_t D = HD;
  CUtensorMap mq, mk, mv, mo;
  // K / V: dims {D, key rows, Hkv, B} with the caller's strides; boxes of
  // 64 keys (a score CTA loads half of a K tile, an output CTA a V tile in
  // two halves)
  const uint64_t kd[4] = {D, uint64_t(a.key_dim_rows), uint64_t(a.kv_heads), uint64_t(a.batch)};
  const uint64_t ks[3] = {uint64_t(a.key_row_stride) * 2, uint64_t(a.key_head_stride) * 2,
                          uint64_t(a.key_seq_stride > 0 ? a.key_seq_stride : a.key_dim_rows * a.key_row_stride) * 2};
  // Q and O [B, C, Hq, D]: dims {D, C, Hq, B}, boxes of 128 rows
  const uint64_t qd[4] = {D, uint64_t(a.chunk_len), uint64_t(a.q_heads), uint64_t(a.batch)};
  const uint64_t qs[3] = {uint64_t(a.q_heads) * D * 2, D * 2, uint64_t(a.chunk_len) * a.q_heads * D * 2};
  if (!make_tmap_bf16(&mk, a.k, kd, ks, BN / 2) || !make_tmap_bf16(&mv, a.v, kd, ks, 64) ||
      !make_tmap_bf16(&mq, a.q, qd, qs, BM) || !make_tmap_bf16(&mo, a.out, qd, qs, BM))
    return cudaErrorInvalidValue;
  const int nqt = (a.chunk_len + BM - 1) / BM;
  cudaLaunchConfig_t cfg = {};
  // four CTAs per (head pair, query tile)
  cfg.gridDim = dim3(2 * a.q_heads, nqt, a.batch);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 4;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_split512_kernel, mq, mk, mv, mo, a);
}

}  // namespace swa
