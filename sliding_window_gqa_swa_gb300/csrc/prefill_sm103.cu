// Prefill attention on the 5th-generation tensor cores (tcgen05) on 64-key
// tiles, for head size 512 and an odd GQA group (an even group runs
// prefill_split512_kernel; head size 256 runs prefill_pair256_kernel or
// prefill128_kernel).
//
// A cluster of two CTAs computes 128 query rows of one query head against the
// key tiles (64 keys each) its rows need; the tile range comes from the causal
// arithmetic or from the plan built on the device (generic plan: image
// blocks, documents).  The two CTAs hold the two 256-column halves of the
// head (a column pair): each computes a partial S over its half of the
// contraction and sends it into one of the peer's two exchange buffers with
// asynchronous remote stores; both add the two partials (fp32 addition
// commutes: the same S bit for bit), run the identical softmax, and
// accumulate their own half of O -- no MMA is done twice.
// Warp roles:
//   warp 0     TMA producer: K and V slices into a ring of slots (128-byte
//              swizzled, 64-column boxes), in the order the MMA thread
//              consumes them: K_0 .. K_{NS-1}, then V_j, K_{j+NS} for each j;
//   warp 1     one thread issues the MMAs: S_0 .. S_{NS-1}, then for each
//              tile j one group that interleaves O += P_j V_j (4 MMAs, V read
//              MN-major) with S_{j+NS} = Q K_{j+NS}^T (16 MMAs of N = 64) into
//              the S buffer S_j came from;
//   warps 2-9  softmax: two warpgroups, one query row per thread (its TMEM
//              lane); group g owns score columns [32g, 32g + 32) of each tile
//              and output columns [128g, 128g + 128).  Per tile: apply the
//              row's key interval [lo, hi], take the row maximum, online
//              softmax in the exp2 domain with lazy rescaling of O (only when
//              the maximum grows by more than 2^8), write P (bf16); finally
//              normalise O and store it;
//   warp 10    forwards "exchange buffer read" to the peer.
// Every wait is bounded; a timeout sets the device error word, makes all
// roles stop, lets in-flight copies and MMAs finish, and frees TMEM.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary and Compilation behavior (causal square-prefill plan,
// generic plan for future same-image pairs); "Add SDPA attention
// implementation", Summary (packed documents, head size 512, K/V shared by
// query-head groups).

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

constexpr int BM = kPlanBM;    // 128 query rows per CTA
constexpr int BN = 64;         // keys per tile
constexpr int HS = 256;        // head-dimension slice per CTA
// TMA warp, MMA warp, two softmax warpgroups and a warp that forwards the
// partial-score exchange's "buffer consumed" signal to the peer
constexpr int THREADS = 352;
constexpr int KV_CHUNK = BN * 128;  // one 64-column box of K or V: 8 KB
constexpr int KV_BYTES = KV_CHUNK * (HS / 64);
constexpr int P_BYTES = BM * BN * 2;
constexpr int XS_BYTES = BM * BN * 4;  // one partial-S exchange buffer (head size 512; two of them)

// Shared memory: the K/V ring, two P buffers, two exchange buffers, the
// row-maximum exchange, barriers.  Q lives in tensor memory.
struct Layout {
  static constexpr int SLOT = KV_BYTES;                          // one ring slot
  static constexpr int NST = 4;                                  // ring slots
  static constexpr int NS = 2;                                   // S buffers in TMEM
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_P = OFF_KV + NST * SLOT;
  static constexpr int OFF_XS = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_PMAX = OFF_XS + 2 * XS_BYTES;  // [2 groups][128 rows] fp32
  static constexpr int OFF_BAR = OFF_PMAX + 2 * BM * 4;
  static constexpr int N_BARS = 2 * NST + 15;
  static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024 B
  static_assert(SMEM <= 232448, "shared memory budget");
};

// TMEM columns: O, then the S buffers (TM_S + b * BN), then the Q slice
constexpr uint32_t TM_O = 0, TM_S = HS, TM_Q = HS + 2 * BN, TM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, HS, true);
constexpr float kRescaleLog2 = 8.f;
constexpr uint64_t kTimeoutNs = 2000000000ull;
static_assert(TM_Q + HS / 2 <= TM_COLS && TM_S + 2 * (2 * BN) <= TM_COLS, "TMEM budget");

template <int NST>
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (NST + s); }
  __device__ uint32_t q() const { return base + 8 * (2 * NST); }  // Q slice ready for the MMAs
  __device__ uint32_t s_full(int b) const { return base + 8 * (2 * NST + 1 + b); }  // b < 2
  __device__ uint32_t p_full(int b) const { return base + 8 * (2 * NST + 4 + b); }
  __device__ uint32_t pv_done(int b) const { return base + 8 * (2 * NST + 6 + b); }
  __device__ uint32_t teardown() const { return base + 8 * (2 * NST + 8); }
  // head size 512, exchange buffer b: the peer's partial arrived (transaction
  // bytes of its stores), this CTA consumed it, the peer consumed this CTA's
  __device__ uint32_t xs_full(int b) const { return base + 8 * (2 * NST + 9 + b); }
  __device__ uint32_t xs_cons(int b) const { return base + 8 * (2 * NST + 11 + b); }
  __device__ uint32_t xs_free(int b) const { return base + 8 * (2 * NST + 13 + b); }
};

// Bounded wait on one phase of an mbarrier.  Gives up when another role has
// aborted or after kTimeoutNs, recording the timeout.
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

// Maximum of the scores sr[0, NC), whose key indices are kbase + c.  When
// `masked`, scores outside the row's interval [lo, hi] are first set to -inf
// (raw domain: the scale is positive).  Four partial maxima keep the
// dependency chains short.
template <int NC>
__device__ __forceinline__ float mask_max(uint32_t* sr, int kbase, int lo, int hi, bool masked) {
  if (masked) {
    const int clo = lo - kbase, chi = hi - kbase;
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (c < clo || c > chi) sr[c] = __float_as_uint(-CUDART_INF_F);
  }
  float m[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
  for (int c = 0; c < NC; ++c) m[c & 3] = fmaxf(m[c & 3], __uint_as_float(sr[c]));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

__device__ __forceinline__ void named_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

__global__ void __launch_bounds__(THREADS, 1)
prefill_colpair_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const PrefillArgs a) {
  using LY = Layout;
  constexpr int NST = LY::NST;
  constexpr int NS = LY::NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sKV = base + LY::OFF_KV, sP = base + LY::OFF_P;
  const Bars<NST> bars{base + LY::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + LY::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + LY::OFF_MISC + 4);
  int32_t* err = a.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the cluster's two CTAs hold the two 256-column halves of query head hq
  const int half = int(cluster_ctarank());  // column half of O
  const int peer = half ^ 1;
  const int col0 = half * HS;
  const int hq = int(blockIdx.x >> 1);
  // query tiles late in a causal sequence or document have the most key tiles:
  // they are scheduled first, so the short ones fill the tail of the grid
  const int qt = int(gridDim.y - 1 - blockIdx.y), b = blockIdx.z;
  const int hk = hq / (a.q_heads / a.kv_heads);
  const int i0 = qt * BM;
  const int q0 = a.chunk_start + i0;

  // key range [k_lo, k_hi) any row of this tile needs
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
  const int kt_lo = k_lo / BN;
  const int n = (k_hi > k_lo) ? ((k_hi - 1) / BN - kt_lo + 1) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    // the softmax threads copy Q into TMEM
    mbar_init(bars.q(), 256);
    for (int i = 0; i < 2; ++i) mbar_init(bars.s_full(i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.p_full(i), 256);
      mbar_init(bars.pv_done(i), 1);
    }
    mbar_init(bars.teardown(), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.xs_full(i), 1);
      mbar_init(bars.xs_cons(i), 256);
      mbar_init(bars.xs_free(i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // ring order: K_0 .. K_{NS-1}, then V_j, K_{j+NS} for j = 0 .. n-1; this
    // CTA's 256 columns of each
    if (n > 0) {
      bool ok = true;
      int idx = 0;
      auto load = [&](int tile, bool is_v) {
        const int s = idx % NST;
        ok = __all_sync(0xffffffffu, wait_bar(bars.empty(s), ((idx / NST) & 1) ^ 1, abort_flag, err));
        if (ok && lane == 0) {
          const int k0 = (kt_lo + tile) * BN;
          const uint32_t dst = sKV + s * LY::SLOT;
          mbar_arrive_expect_tx(bars.full(s), KV_BYTES);
          const CUtensorMap* m = is_v ? &tm_v : &tm_k;
          for (int c = 0; c < HS / 64; ++c) tma_load_4d(dst + c * KV_CHUNK, m, bars.full(s), col0 + 64 * c, k0, hk, b);
        }
        __syncwarp();
        ++idx;
      };
      for (int t = 0; t < NS && t < n && ok; ++t) load(t, false);
      for (int j = 0; j < n && ok; ++j) {
        load(j, true);
        if (j + NS < n && ok) load(j + NS, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // one thread issues every MMA; the other lanes of the warp stay idle
    if (n > 0 && lane == 0) {
      bool ok = wait_bar(bars.q(), 0, abort_flag, err);
      auto commit = [&](uint32_t bar) { mma_commit(bar); };
      // one K=16 step of S_b = Q K^T into S buffer b; K (K-major) from ring slot
      // kslot; Q from TMEM
      auto qk_step = [&](int sbuf, uint32_t kslot, int kk) {
        const int c = kk >> 2, sub = kk & 3;
        const uint64_t bd = sdesc_sw128(kslot + c * KV_CHUNK + sub * 32, 16, 1024);
        mma_bf16_ts(tmem + TM_S + sbuf * BN, tmem + TM_Q + kk * 8, bd, IDESC_QK, kk > 0 ? 1u : 0u);
      };
      int idx = 0;
      for (int t = 0; t < NS && t < n && ok; ++t) {
        const int s = idx % NST;
        ok = wait_bar(bars.full(s), (idx / NST) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HS / 16; ++kk) qk_step(t, sKV + s * LY::SLOT, kk);
        commit(bars.s_full(t));
        commit(bars.empty(s));
        ++idx;
      }
      for (int j = 0; j < n && ok; ++j) {
        const int pb = j & 1;
        const bool next = j + NS < n;  // S_{j+NS} goes to the buffer S_j came from
        const int sbuf = j % NS;
        const int sv = idx % NST, sk = (idx + 1) % NST;
        // P_j written (so S_j read), V_j and K_{j+NS} loaded: one round of polls,
        // then bounded waits for whatever is still pending
        const bool pf = mbar_try_wait(bars.p_full(pb), (j >> 1) & 1);
        const bool vf = mbar_try_wait(bars.full(sv), (idx / NST) & 1);
        const bool kf = !next || mbar_try_wait(bars.full(sk), ((idx + 1) / NST) & 1);
        if (!(pf & vf & kf)) {
          ok = wait_bar(bars.p_full(pb), (j >> 1) & 1, abort_flag, err) &&
               wait_bar(bars.full(sv), (idx / NST) & 1, abort_flag, err) &&
               (!next || wait_bar(bars.full(sk), ((idx + 1) / NST) & 1, abort_flag, err));
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t vslot = sKV + sv * LY::SLOT, kslot = sKV + sk * LY::SLOT;
#pragma unroll
        for (int p = 0; p < BN / 16; ++p) {
          // V is [keys][head dim]: MN-major B; 64-column boxes are KV_CHUNK apart,
          // 8-key row groups 1024 B apart
          const uint64_t bd = sdesc_sw128(vslot + p * 2048, KV_CHUNK, 1024);
          mma_bf16_ss(tmem + TM_O, sdesc_sw128(sP + pb * P_BYTES + p * 32, 16, 1024), bd, IDESC_PV,
                      (j > 0 || p > 0) ? 1u : 0u);
          if (next) {
#pragma unroll
            for (int kk = 4 * p; kk < 4 * p + 4; ++kk) qk_step(sbuf, kslot, kk);
          }
        }
        if (next) commit(bars.s_full(sbuf));
        commit(bars.pv_done(pb));
        commit(bars.empty(sv));
        if (next) commit(bars.empty(sk));
        idx += next ? 2 : 1;
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ exchange forwarder (head size 512)
    // this CTA consumed the peer's partial in buffer t & 1: the peer may refill it
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      ok = __all_sync(0xffffffffu, wait_bar(bars.xs_cons(t & 1), (t >> 1) & 1, abort_flag, err));
      if (ok && lane == 0) mbar_arrive_remote(map_shared(bars.xs_free(t & 1), peer));
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w serves TMEM lane quadrant (w % 4), i.e. one query row per
    // thread; the two threads of a row (one per group) take identical
    // rescaling decisions because both see the same row maximum.
    const int grp = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int i = i0 + r;
    const bool row_ok = i < a.chunk_len;
    const int q = a.chunk_start + i;
    int lo = 0, hi = -1;
    if (row_ok) {
      if (a.generic) {
        const PlanLayout L = plan_layout(a.batch, a.chunk_len);
        const char* plan = static_cast<const char*>(a.plan);
        lo = reinterpret_cast<const int32_t*>(plan + L.off_lo)[(long long)b * a.chunk_len + i];
        hi = reinterpret_cast<const int32_t*>(plan + L.off_hi)[(long long)b * a.chunk_len + i];
      } else {
        causal_interval(q, a.valid_start ? a.valid_start[b] : 0, a.window, lo, hi);
      }
      hi = min(hi, a.key_rows - 1);
    }
    constexpr int HC = BN / 2;  // score columns per group
    constexpr int OC = HS / 2;  // output columns per group
    const int cb = grp * HC;    // first score column of this group
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    float* pmax = reinterpret_cast<float*>(gbase + LY::OFF_PMAX);  // [group][row]
    const int bar_id = 1 + q4;  // named barrier of this quadrant's two warps
    // my row slice of the exchange buffer, and the same slice in the peer's buffer
    const uint32_t xs_row = base + LY::OFF_XS + (r * BN + cb) * 4;
    const uint32_t xs_row_peer = map_shared(xs_row, peer);

    const float c2 = a.scale_log2;

    // this group's half of the row's Q slice -> TMEM (A operand of the score MMAs);
    // 32-bit column c holds the bf16 pair (2c, 2c + 1), the lower index in the low half
    if (n > 0) {
      const uint4* qrow = reinterpret_cast<const uint4*>(
          a.q + (((long long)b * a.chunk_len + i) * a.q_heads + hq) * a.head_dim + col0 + grp * (HS / 2));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = row_ok ? __ldg(qrow + h * 8 + e) : make_uint4(0, 0, 0, 0);
          w[4 * e] = v.x;
          w[4 * e + 1] = v.y;
          w[4 * e + 2] = v.z;
          w[4 * e + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + TM_Q + grp * (HS / 4) + h * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bars.q());
    }

    // m_run is the reference maximum in the exp2 domain; l_run sums the
    // bf16-rounded probabilities of this group's columns (normalises O, which
    // the tensor core accumulates from the same rounded values); l_exact sums
    // the unrounded ones (gives the lse)
    float m_run = -CUDART_INF_F, l_run = 0.f, l_exact = 0.f;
    // The two warps of a row (one per group) meet at a named barrier for every
    // tile; a warp that gives up (timeout or abort) keeps meeting its partner
    // there and skips the rest of each tile, so the barrier's arrivals stay
    // paired and every role reaches the teardown.
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int sb = t % NS, pb = t & 1;
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(bars.s_full(sb), (t / NS) & 1, abort_flag, err));
      if (ok) tc_fence_after();
      const uint32_t tS = tmem + lane_off + TM_S + sb * BN;
      const int k0 = (kt_lo + t) * BN;
      // the masking pass runs only when some row of the warp needs it
      const bool masked = !__all_sync(0xffffffffu, (k0 >= lo) && (k0 + BN - 1 <= hi));
      // sr[0, HC): this group's columns
      uint32_t sr[HC];
      float mraw = -CUDART_INF_F;
      {
        if (ok) {
          tmem_ld32(tS + cb, sr);
          {
            tmem_ld_wait();
            // send my partial slice into the peer's exchange buffer xb (once the
            // peer has consumed what this CTA sent there two tiles ago); the
            // stores count their bytes on the peer's xs_full(xb)
            const int xb = t & 1;
            if (t >= 2)
              ok = __all_sync(0xffffffffu, wait_bar<true>(bars.xs_free(xb), ((t >> 1) - 1) & 1, abort_flag, err));
            if (ok) {
              const uint32_t fbar = map_shared(bars.xs_full(xb), peer);
#pragma unroll
              for (int c = 0; c < HC; c += 4)
                st_async_u32x4(xs_row_peer + xb * XS_BYTES + c * 4, sr[c], sr[c + 1], sr[c + 2], sr[c + 3], fbar);
              // this CTA receives one whole partial tile per tile
              if (threadIdx.x == 64) mbar_arrive_expect_tx(bars.xs_full(xb), XS_BYTES);
              ok = __all_sync(0xffffffffu, wait_bar(bars.xs_full(xb), (t >> 1) & 1, abort_flag, err));
            }
            if (ok) {
              const float* xr = reinterpret_cast<const float*>(gbase + LY::OFF_XS + xb * XS_BYTES) + r * BN + cb;
#pragma unroll
              for (int c = 0; c < HC; c += 4) {
                const float4 v = *reinterpret_cast<const float4*>(xr + c);
                sr[c] = __float_as_uint(__uint_as_float(sr[c]) + v.x);
                sr[c + 1] = __float_as_uint(__uint_as_float(sr[c + 1]) + v.y);
                sr[c + 2] = __float_as_uint(__uint_as_float(sr[c + 2]) + v.z);
                sr[c + 3] = __float_as_uint(__uint_as_float(sr[c + 3]) + v.w);
              }
              mbar_arrive(bars.xs_cons(xb));  // the forwarding warp tells the peer
            }
          }
          if (ok) mraw = mask_max<HC>(sr, k0 + cb, lo, hi, masked);
        }
        // the two groups of this row agree on the tile maximum
        pmax[grp * BM + r] = mraw;
        named_sync(bar_id);
        mraw = fmaxf(mraw, pmax[(grp ^ 1) * BM + r]);
        named_sync(bar_id);
        if (!ok) continue;
      }
      const float mt = mraw * c2;
      // lazy rescale: move the reference only when the maximum grows by > 2^8
      const bool move = (m_run == -CUDART_INF_F) ? (mt > -CUDART_INF_F) : (mt > m_run + kRescaleLog2);
      const bool rescale = move && m_run != -CUDART_INF_F;  // O holds data relative to m_run
      if (__any_sync(0xffffffffu, rescale)) {
        ok = __all_sync(0xffffffffu, wait_bar(bars.pv_done((t - 1) & 1), ((t - 1) >> 1) & 1, abort_flag, err));
        if (!ok) continue;
        tc_fence_after();
        const float alpha = rescale ? exp2f(m_run - mt) : 1.f;
        for (int c0 = grp * OC; c0 < grp * OC + OC; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + TM_O + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tmem + lane_off + TM_O + c0, o);
        }
        tmem_st_wait();
        if (rescale) {
          l_run *= alpha;
          l_exact *= alpha;
        }
      }
      if (move) m_run = mt;
      // probabilities exp2(s * scale_log2 - m_run), packed to bf16
      const float nm = (m_run == -CUDART_INF_F) ? 0.f : -m_run;
      uint32_t pk[HC / 2];
      float ls[2] = {0.f, 0.f}, es[2] = {0.f, 0.f};
#pragma unroll
      for (int c = 0; c < HC; c += 2) {
        const float x0 = __uint_as_float(sr[c]), x1 = __uint_as_float(sr[c + 1]);
        const float p0 = ex2(fmaf(x0, c2, nm));  // -inf -> 0
        const float p1 = ex2(fmaf(x1, c2, nm));
        const uint32_t w = pack_bf16(p0, p1);
        ls[(c >> 1) & 1] += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
        es[(c >> 1) & 1] += p0 + p1;
        pk[c / 2] = w;
      }
      l_run += ls[0] + ls[1];
      l_exact += es[0] + es[1];
      {
        if (t >= 2) {  // P buffer pb is free once PV_{t-2} completed
          ok = __all_sync(0xffffffffu, wait_bar(bars.pv_done(pb), ((t - 2) >> 1) & 1, abort_flag, err));
          if (!ok) continue;
        }
        uint8_t* prow = gbase + LY::OFF_P + pb * P_BYTES + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(prow + (((grp * 4 + j) ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(bars.p_full(pb));
    }
    // row sums of both groups
    pmax[grp * BM + r] = l_run;
    named_sync(bar_id);
    const float l_tot = l_run + pmax[(grp ^ 1) * BM + r];
    named_sync(bar_id);
    pmax[grp * BM + r] = l_exact;
    named_sync(bar_id);
    const float e_tot = l_exact + pmax[(grp ^ 1) * BM + r];
    // epilogue: O / l -> bf16, this group's columns of the CTA's slice
    bool have_o = n > 0 && ok;
    if (have_o)
      have_o = __all_sync(0xffffffffu, wait_bar(bars.pv_done((n - 1) & 1), ((n - 1) >> 1) & 1, abort_flag, err));
    tc_fence_after();
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    uint16_t* orow = a.out + (((long long)b * a.chunk_len + i) * a.q_heads + hq) * a.head_dim + col0;
    for (int c0 = grp * OC; c0 < grp * OC + OC; c0 += 32) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(tmem + lane_off + TM_O + c0, o);
        tmem_ld_wait();
      }
      if (row_ok) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = have_o ? pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv) : 0u;
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    }
    if (row_ok && a.lse && half == 0 && grp == 0)
      a.lse[((long long)b * a.chunk_len + i) * a.q_heads + hq] =
          e_tot > 0.f ? (m_run + log2f(e_tot)) * 0.69314718055994530942f : -CUDART_INF_F;
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let the MMAs and TMA copies this CTA issued finish before TMEM and
    // shared memory are released
    if (warp == 1 && lane == 0) {
      mma_commit(bars.teardown());
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
  cluster_sync();  // the peer no longer reads or writes this CTA's shared memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

cudaError_t launch_colpair(const CUtensorMap& mk, const CUtensorMap& mv, const PrefillArgs& a, cudaStream_t s) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_colpair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int nqt = (a.chunk_len + BM - 1) / BM;
  cudaLaunchConfig_t cfg = {};
  // two CTAs per query head (the two column halves of O)
  cfg.gridDim = dim3(a.q_heads * 2, nqt, a.batch);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Layout::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_colpair_kernel, mk, mv, a);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_bf16(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t box[4] = {64, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides_bytes, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  if (a.head_dim != 256 && a.head_dim != 512) return cudaErrorInvalidValue;
  if (a.head_dim == 256)
    return (a.q_heads / a.kv_heads) % 2 == 0 ? launch_prefill_pair256(a, s) : launch_prefill_t128(a, s);
  // head size 512: four-CTA clusters for an even GQA group, column pairs otherwise
  if (prefill_split512_eligible(a)) return launch_prefill_split512(a, s);
  const uint64_t D = uint64_t(a.head_dim);
  CUtensorMap mk, mv;
  // K / V: dims {D, key rows, Hkv, B} with the caller's strides (Q is read
  // with 16-byte row loads into TMEM)
  const uint64_t kd[4] = {D, uint64_t(a.key_dim_rows), uint64_t(a.kv_heads), uint64_t(a.batch)};
  const uint64_t ks[3] = {uint64_t(a.key_row_stride) * 2, uint64_t(a.key_head_stride) * 2,
                          uint64_t(a.key_seq_stride > 0 ? a.key_seq_stride : a.key_dim_rows * a.key_row_stride) * 2};
  if (!make_tmap_bf16(&mk, a.k, kd, ks, BN) || !make_tmap_bf16(&mv, a.v, kd, ks, BN)) return cudaErrorInvalidValue;
  return launch_colpair(mk, mv, a, s);
}

}  // namespace swa
