// Backward pass of sliding-window attention on the 5th-generation tensor
// cores (tcgen05), for training over whole sequences or packed documents.
//
// For a query row i of head h with key interval [lo_i, hi_i] (the prefill
// plan), upstream gradient dO_i, forward output O_i and lse_i:
//   P_ij  = exp(scale * q_i.k_j - lse_i)            j in [lo_i, hi_i], else 0
//   dP_ij = dO_i . v_j
//   dS_ij = scale * P_ij * (dP_ij - delta_i),       delta_i = dO_i . O_i
//   dQ_i  = sum_j dS_ij k_j,   dK_j = sum_i dS_ij q_i,   dV_j = sum_i P_ij dO_i
// (dK and dV also sum over the query heads of a GQA group).
//
// At head size 512 the accumulators of one 128-key tile's dK and dV alone
// need 1024 of the 512 tensor-memory columns an SM has, so the three
// products cannot share one pass over the scores.  The pass is split into
// kernels that each fit:
//   1. delta_kernel:  delta = rowsum(dO * O), one warp per (row, head);
//   2. scores_kernel: one CTA per (sequence, head, 128-row query tile) walks
//      the tile's 128-key tiles; per tile two MMA chains over the head
//      dimension, S = Q K^T and dP = dO V^T (M = N = 128, double-buffered in
//      tensor memory: 4 x 128 columns), then the epilogue warps write P^T, dS
//      and dS^T as bf16 tiles to global memory, already in the 128-byte
//      swizzled layout the next kernel's MMAs read;
//   3. grads_kernel:  one CTA per 128 x 256 block of dQ, dK or dV sums the
//      products of the stored tiles with Q, K or dO tiles (MN-major B
//      operand, M = 128, N = 256, one 256-column accumulator in tensor
//      memory).  dK and dV run over every (query head of the group, query
//      tile) whose band holds the key tile, dQ over the query tile's band.
// The score tiles cost 3 x 32 KB of HBM traffic per (query tile, key tile,
// head) in each direction; every product runs on the tensor cores once.
//
// Warp roles (scores / grads): warp 0 TMA and bulk-copy producer, warp 1 one
// thread issues the MMAs, then 8 / 4 epilogue warps (one row per thread, the
// TMEM lane of its warp's quadrant).  Every wait is bounded; a timeout sets
// the device error word, makes all roles stop, lets in-flight copies and
// MMAs finish, and frees tensor memory.
//
// Sources: "Add SDPA attention implementation", Summary (head size 512
// models must train; packed documents given by cu_seqlens; K/V shared by the
// query heads of a group) and its fwd+bwd benchmark table; "Enable compact
// sliding-window attention for Gemma 3 and Gemma 4 variants", Summary (the
// sliding-window / image-block / padding mask the plan encodes).

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

constexpr int BT = kBwdTile;                     // queries / keys per score tile
static_assert(BT == kPlanBM, "the plan's query tiles are the score tiles");
constexpr int BOX = BT * 128;                    // one {64 columns, 128 rows} bf16 box: 16 KB
constexpr uint32_t TILE = uint32_t(kBwdTileBytes);  // one score tile: two boxes, 32 KB
constexpr int GN = 256;                          // gradient columns per grads job
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// scores kernel: ring stages of {Q, dO, K, V} 64-column chunks
constexpr int SC_NST = 3;
constexpr int SC_STAGE = 4 * BOX;                // 64 KB
constexpr int SC_THREADS = 320;                  // TMA, MMA, 8 epilogue warps
constexpr int SC_OFF_BAR = SC_NST * SC_STAGE;
constexpr int SC_NBARS = 2 * SC_NST + 5;
constexpr int SC_OFF_MISC = SC_OFF_BAR + 8 * SC_NBARS;
constexpr int SC_SMEM = SC_OFF_MISC + 16 + 1024;
static_assert(SC_SMEM <= 232448, "shared memory budget");
constexpr uint32_t IDESC_S = idesc_bf16_f32(BT, BT, false);

// grads kernel: ring stages of {A score tile, B 128 x 256 operand}
constexpr int GR_NST = 2;
constexpr int GR_A = int(TILE);
constexpr int GR_STAGE = GR_A + 4 * BOX;         // 96 KB
constexpr int GR_THREADS = 192;                  // TMA, MMA, 4 epilogue warps
constexpr int GR_OFF_BAR = GR_NST * GR_STAGE;
constexpr int GR_NBARS = 2 * GR_NST + 2;
constexpr int GR_OFF_MISC = GR_OFF_BAR + 8 * GR_NBARS;
constexpr int GR_SMEM = GR_OFF_MISC + 16 + 1024;
static_assert(GR_SMEM <= 232448, "shared memory budget");
constexpr uint32_t IDESC_G = idesc_bf16_f32(BT, GN, true);

// Bounded wait on one phase of an mbarrier (gives up when another role has
// aborted or after kTimeoutNs, recording the timeout).
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

// 2^x on the special-function unit (-inf -> 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of element (row, col) in a 128 x 128 bf16 tile stored as two
// 128-byte-swizzled {64 columns, 128 rows} boxes: the image TMA would leave in
// shared memory, so one bulk copy makes it an MMA operand.
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
  return uint32_t((col >> 6) * BOX + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2);
}

// Key-tile range [kt_lo, kt_lo + n) of query tile qt of sequence b (from the
// plan's per-tile key range); n = 0 when the tile has no admitted key, and
// when the range exceeds the workspace band (recorded as kErrBand).
__device__ __forceinline__ void tile_band(const char* plan, const PlanLayout& L, int nqt, int b, int qt, int band,
                                          int32_t* err, bool report, int& kt_lo, int& n) {
  const int klo = reinterpret_cast<const int32_t*>(plan + L.off_tlo)[b * nqt + qt];
  const int khi = reinterpret_cast<const int32_t*>(plan + L.off_thi)[b * nqt + qt];
  kt_lo = klo / BT;
  n = khi > klo ? (khi - 1) / BT - kt_lo + 1 : 0;
  if (n > band) {
    if (report && err) atomicCAS(err, 0, kErrBand);
    n = 0;
  }
}

__device__ __forceinline__ size_t tile_slot(int b, int h, int qt, int j, int q_heads, int nqt, int band) {
  return ((size_t(b) * q_heads + h) * nqt + qt) * band + j;
}

// Release tensor memory and shared memory safely after an abort: let the
// MMAs and copies this CTA issued finish first.
__device__ __forceinline__ void drain_after_abort(int warp, int lane, uint32_t teardown_bar) {
  if (warp == 1 && lane == 0) {
    mma_commit(teardown_bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(teardown_bar, 0) && globaltimer_ns() - t0 < kTimeoutNs) {
    }
  }
  if (warp == 0 && lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
}

// ---------------------------------------------------------------- delta
__global__ void __launch_bounds__(256) delta_kernel(const uint16_t* __restrict__ out,
                                                    const uint16_t* __restrict__ dout, float* __restrict__ delta,
                                                    long long rows, int head_dim) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* o = reinterpret_cast<const uint4*>(out + row * head_dim);
  const uint4* g = reinterpret_cast<const uint4*>(dout + row * head_dim);
  float acc = 0.f;
  for (int c = lane; c < head_dim / 8; c += 32) {
    const uint4 a = __ldg(o + c), b = __ldg(g + c);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
      acc = fmaf(__uint_as_float(aw[e] & 0xffff0000u), __uint_as_float(bw[e] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
  if (lane == 0) delta[row] = acc;
}

// ---------------------------------------------------------------- scores
// grid (Hq, n_tiles, B)
__global__ void __launch_bounds__(SC_THREADS, 1)
scores_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const BackwardArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + SC_OFF_BAR;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (SC_NST + s); };
  auto s_full = [&](int b) { return bar0 + 8 * (2 * SC_NST + b); };
  auto t_free = [&](int b) { return bar0 + 8 * (2 * SC_NST + 2 + b); };
  const uint32_t teardown = bar0 + 8 * (2 * SC_NST + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + SC_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + SC_OFF_MISC + 4);
  int32_t* err = a.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the last query tiles of a causal sequence have the most key tiles: they are
  // scheduled first, so the short ones fill the tail of the grid
  const int h = blockIdx.x, qt = int(gridDim.y - 1 - blockIdx.y), b = blockIdx.z;
  const int hk = h / (a.q_heads / a.kv_heads);
  const int nqt = (a.seq_len + BT - 1) / BT;
  const PlanLayout L = plan_layout(a.batch, a.seq_len);
  const char* plan = static_cast<const char*>(a.plan);
  int kt_lo, n;
  tile_band(plan, L, nqt, b, qt, a.band, err, threadIdx.x == 0 && h == 0, kt_lo, n);
  const int NC = a.head_dim / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SC_NST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(t_free(i), 256);
    }
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int idx = 0;
    for (int j = 0; j < n && ok; ++j) {
      const int k0 = (kt_lo + j) * BT;
      for (int c = 0; c < NC && ok; ++c, ++idx) {
        const int s = idx % SC_NST;
        ok = __all_sync(0xffffffffu, wait_bar(empty(s), ((idx / SC_NST) & 1) ^ 1, abort_flag, err));
        if (ok && lane == 0) {
          const uint32_t dst = base + s * SC_STAGE;
          mbar_arrive_expect_tx(full(s), SC_STAGE);
          tma_load_4d(dst, &tm_q, full(s), 64 * c, qt * BT, h, b);
          tma_load_4d(dst + BOX, &tm_do, full(s), 64 * c, qt * BT, h, b);
          tma_load_4d(dst + 2 * BOX, &tm_k, full(s), 64 * c, k0, hk, b);
          tma_load_4d(dst + 3 * BOX, &tm_v, full(s), 64 * c, k0, hk, b);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // S_j = Q K_j^T into columns [256 (j & 1), +128), dP_j = dO V_j^T into the
    // next 128; the two chains alternate step by step
    if (lane == 0) {
      bool ok = true;
      int idx = 0;
      for (int j = 0; j < n && ok; ++j) {
        const int tb = j & 1;
        if (j >= 2) ok = wait_bar(t_free(tb), ((j >> 1) - 1) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_s = tmem + tb * 256, d_p = d_s + 128;
        for (int c = 0; c < NC && ok; ++c, ++idx) {
          const int s = idx % SC_NST;
          ok = wait_bar(full(s), (idx / SC_NST) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = base + s * SC_STAGE;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (c | kk) ? 1u : 0u;
            mma_bf16_ss(d_s, sdesc_sw128(st + kk * 32, 16, 1024), sdesc_sw128(st + 2 * BOX + kk * 32, 16, 1024),
                        IDESC_S, acc);
            mma_bf16_ss(d_p, sdesc_sw128(st + BOX + kk * 32, 16, 1024),
                        sdesc_sw128(st + 3 * BOX + kk * 32, 16, 1024), IDESC_S, acc);
          }
          mma_commit(empty(s));
        }
        if (ok) mma_commit(s_full(tb));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp w serves TMEM lane quadrant w % 4 (query row r); group g takes the
    // key columns [64 g, 64 g + 64) of every tile
    const int grp = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int i = qt * BT + r;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    int lo = 1, hi = 0;  // empty unless the row exists and admits a key
    float l2 = 0.f, dl = 0.f;
    if (i < a.seq_len) {
      const long long row = (long long)b * a.seq_len + i;
      lo = reinterpret_cast<const int32_t*>(plan + L.off_lo)[row];
      hi = reinterpret_cast<const int32_t*>(plan + L.off_hi)[row];
      if (hi >= lo) {
        l2 = a.lse[row * a.q_heads + h] * kLog2e;
        dl = a.delta[row * a.q_heads + h];
      }
    }
    const float c2 = a.scale * kLog2e;
    const float sc = a.scale;
    const int band = a.band;
    char* t_ds = a.t_ds;
    char* t_pt = a.t_pt;
    char* t_dst = a.t_dst;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int tb = j & 1;
      ok = __all_sync(0xffffffffu, wait_bar(s_full(tb), (j >> 1) & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const size_t slot = tile_slot(b, h, qt, j, a.q_heads, nqt, band) * TILE;
      char* ds_tile = t_ds + slot;
      char* pt_tile = t_pt + slot;
      char* dst_tile = t_dst + slot;
      const int kbase = (kt_lo + j) * BT;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int col = grp * 64 + cc * 32;  // first key column of this chunk
        uint32_t sr[32], pr[32];
        tmem_ld32(tmem + lane_off + tb * 256 + col, sr);
        tmem_ld32(tmem + lane_off + tb * 256 + 128 + col, pr);
        tmem_ld_wait();
        if (cc == 1) {  // every TMEM read of this tile is done: the MMAs may reuse it
          tc_fence_before();
          mbar_arrive(t_free(tb));
        }
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p[2], d[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int key = kbase + col + e + u;
            const bool in = key >= lo && key <= hi;
            // selects, not products with p = 0: masked entries are exactly 0
            // whatever the caller's dout holds in rows without keys
            p[u] = in ? ex2(fmaf(__uint_as_float(sr[e + u]), c2, -l2)) : 0.f;
            d[u] = in ? p[u] * (__uint_as_float(pr[e + u]) - dl) * sc : 0.f;
          }
          pw[e / 2] = pack_bf16(p[0], p[1]);
          dw[e / 2] = pack_bf16(d[0], d[1]);
        }
        // dS: row r, key columns [col, col + 32): four 16-byte units
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(ds_tile + tile_off(r, col + 8 * u)) =
              make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
        // P^T and dS^T: row = key, column r.  Lanes r and r + 1 (r even) hold
        // the two halves of one 4-byte word of each row: per pair of keys
        // (c, c + 1) the even lane stores row c and the odd lane row c + 1,
        // after one exchange of the half each needs
        const bool odd = lane & 1;
        const int r0 = r & ~1;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint32_t pwv = pw[e >> 1], dwv = dw[e >> 1];  // lo: key col + e, hi: key col + e + 1
          const uint32_t px = __shfl_xor_sync(0xffffffffu, odd ? (pwv & 0xffffu) : (pwv >> 16), 1);
          const uint32_t dx = __shfl_xor_sync(0xffffffffu, odd ? (dwv & 0xffffu) : (dwv >> 16), 1);
          const uint32_t off = tile_off(col + e + (odd ? 1 : 0), r0);
          *reinterpret_cast<uint32_t*>(pt_tile + off) = odd ? (px | (pwv & 0xffff0000u)) : ((pwv & 0xffffu) | (px << 16));
          *reinterpret_cast<uint32_t*>(dst_tile + off) = odd ? (dx | (dwv & 0xffff0000u)) : ((dwv & 0xffffu) | (dx << 16));
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    drain_after_abort(warp, lane, teardown);
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- grads
// One job: a 128 x 256 block of dV, dK (key tile `tile` of KV head `head`) or
// dQ (query tile `tile` of query head `head`).  Linear grid: the dV / dK jobs
// (longer: they sum over every head of the group) first, then dQ.
struct GradJob {
  int kind;  // 0: dV, 1: dK, 2: dQ
  int b, head, tile, half;
};

__device__ __forceinline__ GradJob grad_job(const BackwardArgs& a, int nqt) {
  const int halves = a.head_dim / GN;
  long long x = blockIdx.x;
  const long long nkv = (long long)a.batch * a.kv_heads * nqt * halves;
  GradJob j;
  if (x < 2 * nkv) {
    j.kind = int(x & 1);
    x >>= 1;
  } else {
    j.kind = 2;
    x -= 2 * nkv;
  }
  j.half = int(x % halves);
  x /= halves;
  j.tile = int(x % nqt);
  // dQ: the last query tiles have the widest bands, so they go first (dV / dK:
  // the first key tiles are admitted by the most query tiles and already lead)
  if (j.kind == 2) j.tile = nqt - 1 - j.tile;
  x /= nqt;
  const int heads = j.kind == 2 ? a.q_heads : a.kv_heads;
  j.head = int(x % heads);
  j.b = int(x / heads);
  return j;
}

// Visit the job's items in order: f(slot, b_row_tile, b_head) per item, where
// slot indexes the stored score tile (A operand) and (b_row_tile, b_head)
// locate the B operand.  dQ: the key tiles of the query tile's band (B = K).
// dV / dK: every (query head of the group, query tile) whose band holds the
// key tile (B = dO or Q), found 32 query tiles at a time with a warp ballot.
// Called by all 32 lanes of a warp; f runs warp-uniformly and returns false
// to stop.  Returns the number of items visited.
template <typename F>
__device__ __forceinline__ int for_each_item(const BackwardArgs& a, const GradJob& j, int nqt, int lane, F&& f) {
  const char* plan = static_cast<const char*>(a.plan);
  const PlanLayout L = plan_layout(a.batch, a.seq_len);
  int count = 0;
  if (j.kind == 2) {
    int kt_lo, n;
    tile_band(plan, L, nqt, j.b, j.tile, a.band, a.err, false, kt_lo, n);
    const int hk = j.head / (a.q_heads / a.kv_heads);
    for (int t = 0; t < n; ++t) {
      if (!f(tile_slot(j.b, j.head, j.tile, t, a.q_heads, nqt, a.band), kt_lo + t, hk)) return count;
      ++count;
    }
    return count;
  }
  const int G = a.q_heads / a.kv_heads;
  for (int q0 = 0; q0 < nqt; q0 += 32) {
    const int qt = q0 + lane;
    int kt_lo = 0, n = 0;
    if (qt < nqt) tile_band(plan, L, nqt, j.b, qt, a.band, a.err, false, kt_lo, n);
    const uint32_t hits = __ballot_sync(0xffffffffu, j.tile >= kt_lo && j.tile < kt_lo + n);
    for (int hh = 0; hh < G; ++hh) {
      const int h = j.head * G + hh;
      for (uint32_t m = hits; m; m &= m - 1) {
        const int src = __ffs(m) - 1;
        const int klo = __shfl_sync(0xffffffffu, kt_lo, src);
        if (!f(tile_slot(j.b, h, q0 + src, j.tile - klo, a.q_heads, nqt, a.band), q0 + src, h)) return count;
        ++count;
      }
    }
  }
  return count;
}

__global__ void __launch_bounds__(GR_THREADS, 1)
grads_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
             const __grid_constant__ CUtensorMap tm_k, const BackwardArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + GR_OFF_BAR;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (GR_NST + s); };
  const uint32_t acc_full = bar0 + 8 * (2 * GR_NST);
  const uint32_t teardown = bar0 + 8 * (2 * GR_NST + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + GR_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + GR_OFF_MISC + 4);
  int32_t* err = a.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = (a.seq_len + BT - 1) / BT;
  const GradJob job = grad_job(a, nqt);
  // item count (every role walks the same list)
  const int n = for_each_item(a, job, nqt, lane, [](size_t, int, int) { return true; });

  if (threadIdx.x == 0) {
    for (int s = 0; s < GR_NST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), GN);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(job.kind == 0 ? &tm_do : job.kind == 1 ? &tm_q : &tm_k);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const char* tiles = job.kind == 0 ? a.t_pt : job.kind == 1 ? a.t_dst : a.t_ds;
    const CUtensorMap* mb = job.kind == 0 ? &tm_do : job.kind == 1 ? &tm_q : &tm_k;
    const int col0 = job.half * GN;
    int idx = 0;
    for_each_item(a, job, nqt, lane, [&](size_t slot, int brow, int bhead) {
      const int s = idx % GR_NST;
      const bool ok = __all_sync(0xffffffffu, wait_bar(empty(s), ((idx / GR_NST) & 1) ^ 1, abort_flag, err));
      if (ok && lane == 0) {
        const uint32_t dst = base + s * GR_STAGE;
        const char* src = tiles + slot * TILE;
        mbar_arrive_expect_tx(full(s), GR_STAGE);
        bulk_load(dst, src, TILE / 2, full(s));
        bulk_load(dst + TILE / 2, src + TILE / 2, TILE / 2, full(s));
        for (int c = 0; c < GN / 64; ++c)
          tma_load_4d(dst + GR_A + c * BOX, mb, full(s), col0 + 64 * c, brow * BT, bhead, job.b);
      }
      __syncwarp();
      ++idx;
      return ok;
    });
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % GR_NST;
        ok = wait_bar(full(s), (t / GR_NST) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = base + s * GR_STAGE;
#pragma unroll
        for (int p = 0; p < BT / 16; ++p) {
          // A: the score tile, K-major (two 64-column boxes); B: 128 rows x 256
          // columns, MN-major (four 64-column boxes of 128 rows)
          const uint64_t ad = sdesc_sw128(st + (p >> 2) * BOX + (p & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(st + GR_A + p * 2048, BOX, 1024);
          mma_bf16_ss(tmem, ad, bd, IDESC_G, (t | p) ? 1u : 0u);
        }
        mma_commit(empty(s));
      }
      if (ok && n > 0) mma_commit(acc_full);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int row = job.tile * BT + r;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    bool have = n > 0;
    if (have) have = __all_sync(0xffffffffu, wait_bar(acc_full, 0, abort_flag, err));
    tc_fence_after();
    uint16_t* dst = nullptr;
    if (row < a.seq_len) {
      const long long srow = (long long)job.b * a.seq_len + row;
      if (job.kind == 2)
        dst = a.dq + (srow * a.q_heads + job.head) * a.head_dim;
      else
        dst = (job.kind == 0 ? a.dv : a.dk) + (srow * a.kv_heads + job.head) * a.head_dim;
      dst += job.half * GN;
    }
    // an aborted job leaves its block unwritten (the error word reports it)
    if (n == 0 || have) {
      for (int c0 = 0; c0 < GN; c0 += 32) {
        uint32_t o[32];
        if (have) {
          tmem_ld32(tmem + lane_off + c0, o);
          tmem_ld_wait();
        }
        if (dst) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = have ? pack_bf16(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])) : 0u;
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    drain_after_abort(warp, lane, teardown);
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, GN);
}

}  // namespace

BackwardLayout backward_layout(int batch, int seq_len, int q_heads, int window, bool images) {
  BackwardLayout l;
  l.n_tiles = (seq_len + BT - 1) / BT;
  const int span = 1 + (window - 1 + BT - 1) / BT;
  l.band = images ? l.n_tiles : (span < l.n_tiles ? span : l.n_tiles);
  const size_t tiles = size_t(batch) * q_heads * l.n_tiles * l.band * kBwdTileBytes;
  l.off_delta = 0;
  l.off_ds = align256(size_t(batch) * seq_len * q_heads * sizeof(float));
  l.off_pt = l.off_ds + tiles;
  l.off_dst = l.off_pt + tiles;
  l.total = l.off_dst + tiles;
  return l;
}

cudaError_t launch_prefill_backward(const BackwardArgs& a, cudaStream_t s) {
  if (a.head_dim != 256 && a.head_dim != 512) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(grads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GR_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint64_t D = uint64_t(a.head_dim), S = uint64_t(a.seq_len);
  // [B, S, H, D] tensors: dims {D, S, H, B}
  const uint64_t qd[4] = {D, S, uint64_t(a.q_heads), uint64_t(a.batch)};
  const uint64_t qs[3] = {uint64_t(a.q_heads) * D * 2, D * 2, S * a.q_heads * D * 2};
  const uint64_t kd[4] = {D, S, uint64_t(a.kv_heads), uint64_t(a.batch)};
  const uint64_t ks[3] = {uint64_t(a.kv_heads) * D * 2, D * 2, S * a.kv_heads * D * 2};
  CUtensorMap mq, mdo, mk, mv;
  if (!make_tmap_bf16(&mq, a.q, qd, qs, BT) || !make_tmap_bf16(&mdo, a.dout, qd, qs, BT) ||
      !make_tmap_bf16(&mk, a.k, kd, ks, BT) || !make_tmap_bf16(&mv, a.v, kd, ks, BT))
    return cudaErrorInvalidValue;

  const long long rows = (long long)a.batch * a.seq_len * a.q_heads;
  delta_kernel<<<unsigned((rows + 7) / 8), 256, 0, s>>>(a.out, a.dout, a.delta, rows, a.head_dim);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int nqt = (a.seq_len + BT - 1) / BT;
  scores_kernel<<<dim3(a.q_heads, nqt, a.batch), SC_THREADS, SC_SMEM, s>>>(mq, mdo, mk, mv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const long long halves = a.head_dim / GN;
  const long long jobs = 2LL * a.batch * a.kv_heads * nqt * halves + (long long)a.batch * a.q_heads * nqt * halves;
  grads_kernel<<<unsigned(jobs), GR_THREADS, GR_SMEM, s>>>(mq, mdo, mk, a);
  return cudaGetLastError();
}

}  // namespace swa
