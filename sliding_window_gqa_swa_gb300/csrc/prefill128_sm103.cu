// Prefill attention at head size 256 on 128-key tiles (tcgen05, one CTA per
// 128 query rows of one query head).
//
// Per key tile j (128 keys): S_j = Q K_j^T (M = N = 128, one chain of sixteen
// K = 16 steps over the head dimension) into one of two 128-column S buffers
// in tensor memory; the softmax warps turn S_j into bf16 probabilities P_j,
// written over the first 64 columns of the same buffer; then O += P_j V_j as
// two independent chains of N = 128 (the two 128-column halves of O, eight
// K = 16 steps each, A = P_j from tensor memory, V read MN-major).  The MMA
// thread issues PV_j followed by S_{j+2} (which overwrites P_j: the tensor
// pipe runs one thread's MMAs in order), so the softmax of tile j + 1 overlaps
// both.  Tensor memory: O (256 columns) + two S buffers = 512 columns.
// Shared memory: Q (64 KB, loaded once), a ring of five 32 KB slots each
// holding 128 keys x 128 head-dimension columns of K or V (a K or V tile
// takes two slots), the row-maximum exchange, barriers: 226 KB.
//
// Warp roles: warp 0 TMA producer; warp 1 one thread issues the MMAs; warps
// 2-9 softmax in two warpgroups, one query row per thread (its TMEM lane);
// group g owns key columns [64 g, 64 g + 64) of every tile and output
// columns [128 g, 128 g + 128).  The two threads of a row agree on each
// tile's maximum through shared memory, so they rescale identically; O is
// rescaled lazily (only when the maximum grows by more than 2^8).  The
// probabilities are rounded to bf16 for PV and the normaliser is the sum of
// the same rounded values; lse uses the unrounded sum.
// Every wait is bounded; a timeout sets the device error word, makes all
// roles stop, lets in-flight copies and MMAs finish, and frees TMEM.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary and Compilation behavior (causal square-prefill plan,
// generic plan for future same-image pairs); "Add SDPA attention
// implementation", Summary (packed documents, K/V shared by query-head
// groups).

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

constexpr int BM = kPlanBM;      // 128 query rows per CTA
constexpr int BN = 128;          // keys per tile
constexpr int HD = 256;          // head dimension
constexpr int BOX = 128 * 128;   // one {64 columns, 128 rows} bf16 box: 16 KB
constexpr int SLOT = 2 * BOX;    // 128 keys x 128 columns of K or V: 32 KB
constexpr int NST = 5;           // ring slots
constexpr int THREADS = 320;
constexpr int OFF_Q = 0;
constexpr int OFF_RING = OFF_Q + 4 * BOX;
constexpr int OFF_PMAX = OFF_RING + NST * SLOT;  // [2 groups][128 rows] fp32
constexpr int OFF_BAR = OFF_PMAX + 2 * BM * 4;
constexpr int N_BARS = 2 * NST + 8;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024 B
static_assert(SMEM <= 232448, "shared memory budget");

constexpr uint32_t TM_O = 0, TM_S = 256, TM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, 128, true);
constexpr float kRescaleLog2 = 8.f;
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
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
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

__device__ __forceinline__ void named_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

__global__ void __launch_bounds__(THREADS, 1)
prefill128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
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
  const int hq = blockIdx.x;
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
    mbar_init(bars.q(), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full(i), 1);
      mbar_init(bars.p_full(i), 256);
      mbar_init(bars.pv_done(i), 1);
    }
    mbar_init(bars.teardown(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Q once; then the ring in the order the MMAs consume it: K_0, K_1, and per
    // tile j: V_j, K_{j+2} (a tile takes two slots: head-dimension columns
    // [0, 128) and [128, 256))
    if (n > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bars.q(), 4 * BOX);
        for (int c = 0; c < 4; ++c) tma_load_4d(sQ + c * BOX, &tm_q, bars.q(), 64 * c, i0, hq, b);
      }
      __syncwarp();
      bool ok = true;
      int idx = 0;
      auto load = [&](const CUtensorMap* m, int tile, int part) {
        const int s = idx % NST;
        ok = __all_sync(0xffffffffu, wait_bar(bars.empty(s), ((idx / NST) & 1) ^ 1, abort_flag, err));
        if (ok && lane == 0) {
          const int k0 = (kt_lo + tile) * BN;
          const uint32_t dst = sRing + s * SLOT;
          mbar_arrive_expect_tx(bars.full(s), SLOT);
          for (int c = 0; c < 2; ++c) tma_load_4d(dst + c * BOX, m, bars.full(s), 128 * part + 64 * c, k0, hk, b);
        }
        __syncwarp();
        ++idx;
      };
      for (int t = 0; t < 2 && t < n && ok; ++t)
        for (int part = 0; part < 2 && ok; ++part) load(&tm_k, t, part);
      for (int j = 0; j < n && ok; ++j) {
        for (int part = 0; part < 2 && ok; ++part) load(&tm_v, j, part);
        if (j + 2 < n)
          for (int part = 0; part < 2 && ok; ++part) load(&tm_k, j + 2, part);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0 && lane == 0) {
      bool ok = wait_bar(bars.q(), 0, abort_flag, err);
      // S_t = Q K_t^T into S buffer sb from ring slots (idx, idx + 1)
      auto qk = [&](int sb, int idx) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const int c = kk >> 2;  // 64-column box of the contraction
          const uint32_t slot = sRing + ((idx + (c >> 1)) % NST) * SLOT;
          const uint64_t ad = sdesc_sw128(sQ + c * BOX + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(slot + (c & 1) * BOX + (kk & 3) * 32, 16, 1024);
          mma_bf16_ss(tmem + TM_S + sb * BN, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      int idx = 0;
      for (int t = 0; t < 2 && t < n && ok; ++t) {
        ok = wait_bar(bars.full(idx % NST), (idx / NST) & 1, abort_flag, err) &&
             wait_bar(bars.full((idx + 1) % NST), ((idx + 1) / NST) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        qk(t, idx);
        mma_commit(bars.s_full(t));
        mma_commit(bars.empty(idx % NST));
        mma_commit(bars.empty((idx + 1) % NST));
        idx += 2;
      }
      for (int j = 0; j < n && ok; ++j) {
        const int sb = j & 1;
        const bool next = j + 2 < n;  // S_{j+2} goes to the buffer S_j came from
        // P_j written, V_j loaded (slots idx, idx + 1), K_{j+2} loaded (idx + 2, idx + 3)
        ok = wait_bar(bars.p_full(sb), (j >> 1) & 1, abort_flag, err);
        for (int u = 0; u < (next ? 4 : 2) && ok; ++u)
          ok = wait_bar(bars.full((idx + u) % NST), ((idx + u) / NST) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t pbase = tmem + TM_S + sb * BN;
        const uint32_t v0 = sRing + (idx % NST) * SLOT, v1 = sRing + ((idx + 1) % NST) * SLOT;
#pragma unroll
        for (int p = 0; p < BN / 16; ++p) {
          // V is [keys][head dim]: MN-major B, 64-column boxes BOX apart, 8-key
          // row groups 1024 B apart; P_j: 16 keys per step = 8 columns of bf16 pairs
          const uint32_t acc = (j > 0 || p > 0) ? 1u : 0u;
          mma_bf16_ts(tmem + TM_O, pbase + 8 * p, sdesc_sw128(v0 + p * 2048, BOX, 1024), IDESC_PV, acc);
          mma_bf16_ts(tmem + TM_O + 128, pbase + 8 * p, sdesc_sw128(v1 + p * 2048, BOX, 1024), IDESC_PV, acc);
        }
        mma_commit(bars.pv_done(sb));
        mma_commit(bars.empty(idx % NST));
        mma_commit(bars.empty((idx + 1) % NST));
        if (next) {
          qk(sb, idx + 2);
          mma_commit(bars.s_full(sb));
          mma_commit(bars.empty((idx + 2) % NST));
          mma_commit(bars.empty((idx + 3) % NST));
        }
        idx += next ? 4 : 2;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
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
    constexpr int HC = BN / 2;  // key columns per group
    constexpr int OC = HD / 2;  // output columns per group
    const int cb = grp * HC;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    float* pmax = reinterpret_cast<float*>(gbase + OFF_PMAX);  // [group][row]
    const int bar_id = 1 + q4;  // named barrier of this quadrant's two warps
    const float c2 = a.scale_log2;

    float m_run = -CUDART_INF_F, l_run = 0.f, l_exact = 0.f;
    // The two warps of a row meet at a named barrier for every tile; a warp
    // that gives up (timeout or abort) keeps meeting its partner there and
    // skips the rest of each tile, so the arrivals stay paired.
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int sb = t & 1;
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(bars.s_full(sb), (t >> 1) & 1, abort_flag, err));
      if (ok) tc_fence_after();
      const uint32_t tS = tmem + lane_off + TM_S + sb * BN;
      const int k0 = (kt_lo + t) * BN;
      const bool masked = !__all_sync(0xffffffffu, (k0 >= lo) && (k0 + BN - 1 <= hi));
      uint32_t sr[HC];
      float mraw = -CUDART_INF_F;
      if (ok) {
        tmem_ld32(tS + cb, sr);
        tmem_ld32(tS + cb + 32, sr + 32);
        tmem_ld_wait();
        if (masked) {
          const int clo = lo - (k0 + cb), chi = hi - (k0 + cb);
#pragma unroll
          for (int c = 0; c < HC; ++c)
            if (c < clo || c > chi) sr[c] = __float_as_uint(-CUDART_INF_F);
        }
        float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int c = 0; c < HC; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sr[c]));
        mraw = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      // the two groups of this row agree on the tile maximum; after this
      // barrier both have read their S columns, so P may overwrite them
      pmax[grp * BM + r] = mraw;
      named_sync(bar_id);
      mraw = fmaxf(mraw, pmax[(grp ^ 1) * BM + r]);
      named_sync(bar_id);
      if (!ok) continue;
      const float mt = mraw * c2;
      // lazy rescale: move the reference only when the maximum grows by > 2^8
      const bool move = (m_run == -CUDART_INF_F) ? (mt > -CUDART_INF_F) : (mt > m_run + kRescaleLog2);
      const bool rescale = move && m_run != -CUDART_INF_F;  // O holds data relative to m_run
      if (__any_sync(0xffffffffu, rescale)) {
        // PV_{t-1}, the only MMA that may still write O, must be done
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
      // probabilities exp2(s * scale_log2 - m_run), packed to bf16 pairs
      const float nm = (m_run == -CUDART_INF_F) ? 0.f : -m_run;
      uint32_t pk[HC / 2];
      float ls[2] = {0.f, 0.f}, es[2] = {0.f, 0.f};
#pragma unroll
      for (int c = 0; c < HC; c += 2) {
        const float p0 = ex2(fmaf(__uint_as_float(sr[c]), c2, nm));  // -inf -> 0
        const float p1 = ex2(fmaf(__uint_as_float(sr[c + 1]), c2, nm));
        const uint32_t w = pack_bf16(p0, p1);
        ls[(c >> 1) & 1] += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
        es[(c >> 1) & 1] += p0 + p1;
        pk[c / 2] = w;
      }
      l_run += ls[0] + ls[1];
      l_exact += es[0] + es[1];
      // P_t: keys [64 grp, 64 grp + 64) go to columns [32 grp, 32 grp + 32) of
      // the S buffer (the A operand layout of PV: 16 keys per 8 columns)
      tmem_st32(tS + 32 * grp, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bars.p_full(sb));
    }
    // row sums of both groups
    pmax[grp * BM + r] = l_run;
    named_sync(bar_id);
    const float l_tot = l_run + pmax[(grp ^ 1) * BM + r];
    named_sync(bar_id);
    pmax[grp * BM + r] = l_exact;
    named_sync(bar_id);
    const float e_tot = l_exact + pmax[(grp ^ 1) * BM + r];
    // epilogue: O / l -> bf16, this group's output columns
    bool have_o = n > 0 && ok;
    if (have_o)
      have_o = __all_sync(0xffffffffu, wait_bar(bars.pv_done((n - 1) & 1), ((n - 1) >> 1) & 1, abort_flag, err));
    tc_fence_after();
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    uint16_t* orow = a.out + (((long long)b * a.chunk_len + i) * a.q_heads + hq) * a.head_dim;
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
    if (row_ok && a.lse && grp == 0)
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
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

cudaError_t launch_prefill_t128(const PrefillArgs& a, cudaStream_t s) {
  if (a.head_dim != HD) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint64_t D = HD;
  CUtensorMap mq, mk, mv;
  // K / V: dims {D, key rows, Hkv, B} with the caller's strides
  const uint64_t kd[4] = {D, uint64_t(a.key_dim_rows), uint64_t(a.kv_heads), uint64_t(a.batch)};
  const uint64_t ks[3] = {uint64_t(a.key_row_stride) * 2, uint64_t(a.key_head_stride) * 2,
                          uint64_t(a.key_seq_stride > 0 ? a.key_seq_stride : a.key_dim_rows * a.key_row_stride) * 2};
  // Q [B, C, Hq, D]: dims {D, C, Hq, B}
  const uint64_t qd[4] = {D, uint64_t(a.chunk_len), uint64_t(a.q_heads), uint64_t(a.batch)};
  const uint64_t qs[3] = {uint64_t(a.q_heads) * D * 2, D * 2, uint64_t(a.chunk_len) * a.q_heads * D * 2};
  if (!make_tmap_bf16(&mk, a.k, kd, ks, BN) || !make_tmap_bf16(&mv, a.v, kd, ks, BN) ||
      !make_tmap_bf16(&mq, a.q, qd, qs, BM))
    return cudaErrorInvalidValue;
  const int nqt = (a.chunk_len + BM - 1) / BM;
  prefill128_kernel<<<dim3(a.q_heads, nqt, a.batch), THREADS, SMEM, s>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace swa
