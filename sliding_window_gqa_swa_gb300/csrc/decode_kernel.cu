// Single-token decode over the compact cache: append, split-K attention and
// the merge of the splits, in one launch.
//
// Grid (nsplit, Hkv, B).  Each CTA owns a contiguous range of rows of one
// (sequence, kv head) slab.  A producer warp issues bulk asynchronous copies
// of the range, in chunks of contiguous rows (32 KB of K + V per chunk), into
// a 3-stage shared-memory ring: the first chunks at once, later chunks only
// when the runtime mask admits one of their rows.  It also stages the step's
// new K/V row (used in place of the cache row it replaces) and appends it to
// the cache.  Four compute warps each take a quarter of the rows of every
// chunk and keep their own online-softmax state for all G query heads of the
// group (each loaded K/V row serves the whole group); a row is split across
// LPR lanes so a lane group reads a contiguous 128-byte span of it.  The
// warps are merged in a fixed order.  Then:
//   * one split: the CTA writes the output;
//   * a cluster of splits (at most 8): the CTAs of a slab form a thread-block
//     cluster and rank 0 merges their partials through distributed shared
//     memory;
//   * more splits: partials go to the workspace and the last CTA of the slab
//     (atomic ticket, no waiting) merges them and resets the ticket.
// The merge order is fixed everywhere, so results are deterministic.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary (the step's new row goes into the compact cache at its
// row index; one runtime mask per step) and Compilation behavior (decode
// reads only the 1088 rows of the compact buffer); "Add SDPA attention implementation", Summary
// (K/V shared by query-head groups).

#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

// Scratch of swa_decode_noalloc (tickets, split statistics, split partials)
// for callers that cannot allocate device memory.  Every GPU that loads the
// library holds it until the process exits.  In host code this name is only a
// host-side stand-in: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[SWA_DECODE_STATIC_SCRATCH_BYTES];

namespace swa {
namespace {

using namespace ptx;

constexpr int kStages = 3;
constexpr int kStageBytes = 32768;                  // K chunk + V chunk
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D, int G, int NW>
struct Shape {
  static constexpr int CH = kStageBytes / (2 * D * 2);  // rows per chunk
  static constexpr int RPC = CH / NW;                   // rows per warp per chunk
  static constexpr int kWant = D * G / 32;              // lanes per row keeping q + acc in registers
  static constexpr int kMin = 32 / RPC;                 // a warp pass must not exceed its rows
  static constexpr int kLpr = kWant > kMin ? kWant : kMin;
  static constexpr int kMax = D / 8 < 32 ? D / 8 : 32;  // a lane holds at least one 16-byte vector
  static constexpr int LPR = kLpr < 8 ? 8 : (kLpr > kMax ? kMax : kLpr);  // lanes per row
  static constexpr int E = D / LPR;                     // elements per lane
  static constexpr int V16 = E / 8;                     // 16-byte vectors per lane per row
  static constexpr int RPW = 32 / LPR;                  // rows per warp pass
  static constexpr int PASSES = RPC / RPW;
  static_assert(PASSES >= 1 && RPC % RPW == 0, "chunk shape");
};

// Shared-memory slots the warp merge uses: as many as fit in the ring next
// to the CTA accumulator and the combine's statistics (a power of two that
// divides the warp count).
__host__ __device__ constexpr int merge_slots(int nw, int g, int d) {
  return (nw + 2) * g * d * 4 + 3 * g * 64 * 4 <= kStages * kStageBytes       ? nw
         : (nw / 2 + 2) * g * d * 4 + 3 * g * 64 * 4 <= kStages * kStageBytes ? nw / 2
         : (nw / 4 + 2) * g * d * 4 + 3 * g * 64 * 4 <= kStages * kStageBytes ? nw / 4
         : (nw / 8 + 2) * g * d * 4 + 3 * g * 64 * 4 <= kStages * kStageBytes ? nw / 8
                                                                               : 1;
}

// Packed fp32 pairs: (lo, hi) in one 64-bit register and d += a * b on both.
__device__ __forceinline__ uint64_t pair_f32(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ void ffma2(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ float pair_lo(uint64_t x) { return __uint_as_float(uint32_t(x)); }
__device__ __forceinline__ float pair_hi(uint64_t x) { return __uint_as_float(uint32_t(x >> 32)); }
// bf16 pair (element 0 in the low half) widened to an fp32 pair
__device__ __forceinline__ uint64_t bf16x2_to_pair(uint32_t w) { return pair_f32(w << 16, w & 0xffff0000u); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicCAS(err, 0, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Shared memory (dynamic): ring [kStages][K chunk | V chunk] (reused after the
// chunk loop for the per-warp accumulators [warps][G][D], the CTA accumulator
// [G][D] and the combine's split statistics) | new K row | new V row | mask
// bytes of the range | chunk flags | barriers.
template <int D, int G, int NW>
__global__ void __launch_bounds__(32 * (NW + 1), 16 / NW)
decode_kernel(const DecodeArgs a) {
  constexpr int kComputeWarps = NW;
  constexpr int kThreads = 32 * (NW + 1);  // + one producer warp
  using S = Shape<D, G, NW>;
  constexpr int LPR = S::LPR, E = S::E, V16 = S::V16, RPW = S::RPW, CH = S::CH, RPC = S::RPC,
                PASSES = S::PASSES;
  constexpr int CHUNK_BYTES = CH * D * 2;

  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int R = a.rows;
  const int r0 = split * a.rows_per_split;
  const int r1 = min(R, r0 + a.rows_per_split);
  const int nrows = max(0, r1 - r0);
  const int nchunks = (nrows + CH - 1) / CH;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  uint8_t* kn_s = smem + kStages * kStageBytes;
  uint8_t* vn_s = kn_s + D * 2;
  uint8_t* mask_s = vn_s + D * 2;
  const int mask_bytes = (a.rows_per_split + 15) & ~15;
  uint8_t* chunk_on = mask_s + mask_bytes;
  const int flag_bytes = ((a.rows_per_split + CH - 1) / CH + 15) & ~15;
  uint64_t* bars = reinterpret_cast<uint64_t*>(chunk_on + flag_bytes);  // full[kStages], empty[kStages]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  __shared__ float s_m[kComputeWarps][G], s_l[kComputeWarps][G];
  __shared__ float s_M[G], s_L[G];
  __shared__ int s_last;
  // cluster merge by pushes: every CTA sends each CTA of the cluster (M, L) and
  // that CTA's slice of its accumulator with asynchronous remote stores; each
  // CTA waits for its slice from all and finishes it (no cluster barrier after
  // the compute).  Used when the slices are equal and fit these buffers.
  constexpr int kNf = G * D / 4;  // float4s of one CTA's accumulator
  constexpr bool kPushable = G <= 2 && kNf <= 256;
  __shared__ __align__(16) float4 s_recv[kPushable ? 16 + kNf : 1];
  __shared__ __align__(8) uint64_t s_merge_bar;
  const bool push = kPushable && a.cluster && a.nsplit > 1 && a.nsplit <= 16 && kNf % a.nsplit == 0;
  const int slice = push ? kNf / a.nsplit : 0;
  const uint32_t sring = smem_u32(smem);
  const uint32_t bar_full0 = smem_u32(bars), bar_empty0 = smem_u32(bars + kStages);

  // the next kernel of the stream may start its own cache prefetch now
  if (tid == 0) pdl_launch_dependents();
  swa_device_state* st = a.state;
  const long long slab = (((long long)a.layer * a.batch + b) * a.kv_heads + h) * (long long)R * D;
  uint16_t* Kc = a.k_cache + slab;
  uint16_t* Vc = a.v_cache + slab;
  // KV-sharing layer (no k_new / v_new): attend over rows the owning layer's
  // decode already wrote this step, without appending; the owner may be the
  // kernel launched just before, so even the cache is read after the wait
  const bool append = a.k_new != nullptr;
  if (!append) pdl_wait();
  const uint16_t* kn = append ? a.k_new + ((long long)b * a.kv_heads + h) * D : nullptr;
  const uint16_t* vn = append ? a.v_new + ((long long)b * a.kv_heads + h) * D : nullptr;
  // Chunks loaded before the mask is read: the first ones that can hold an
  // admitted row.  In an anchored cache the admitted rows of a sequence are
  // one interval, [max(0, valid_start - origin, cur_row - W + 1), cur_row],
  // computed here from the state the step's mask kernel left (every kernel
  // that writes the state completes before a decode of the step starts); in
  // a ring cache the first chunks are taken.  Chunks before c_first are never
  // fetched; later ones only when the mask admits one of their rows.
  int c_first = 0, c_end = nchunks;
  if (!a.ring && append && nchunks > kStages) {
    const int cr = st->cur_row, org = st->origin, vs = a.valid_start[b];
    const int lo = max(max(0, vs - org), max(-org, cr - a.window + 1)) - r0;
    const int hi = min(min(cr, R - 1) - r0, nrows - 1);  // within this split's rows
    if (cr < 0 || cr >= R || hi < 0 || lo >= nrows || lo > hi) {
      c_first = c_end = 0;  // nothing of this split is admitted (or the state is off: the mask decides)
    } else {
      c_first = max(0, lo) / CH;
      c_end = hi / CH + 1;
    }
  }
  // chunks [c_first, c_first + nspec) are fetched early; c_end <= nchunks
  const int nspec = max(0, min(kStages, c_end - c_first));
  // a range that fits in the ring is loaded at once by every thread with
  // 16-byte asynchronous copies (lowest latency); longer ranges stream
  // through the ring with bulk copies
  const bool oneshot = nchunks <= kStages;
  if (oneshot) {
    constexpr int U = D / 8;  // 16-byte units per row
    const int units = nrows * U;
    for (int x = tid; x < 2 * units; x += kThreads) {
      const int kv = x >= units, y = kv ? x - units : x;
      const int row = y / U, col = y % U;
      const int c = row / CH, rr = row % CH;
      const uint32_t dst = sring + c * kStageBytes + kv * CHUNK_BYTES + (rr * U + col) * 16;
      cp_async_16(dst, (kv ? Vc : Kc) + (long long)(r0 + row) * D + col * 8);
    }
  }

  if (warp == kComputeWarps) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(bar_full0 + 8 * s, 1);
        mbar_init(bar_empty0 + 8 * s, kComputeWarps);
      }
      *abort_flag = 0;
      if (push) {  // phase 0 completes when every CTA's slice (header + accumulator) landed
        mbar_init(smem_u32(&s_merge_bar), 1);
        mbar_arrive_expect_tx(smem_u32(&s_merge_bar), uint32_t(a.nsplit * (1 + slice) * 16));
      }
      fence_mbar_init();
      for (int i = 0; i < (oneshot ? 0 : nspec); ++i) {
        const int c = c_first + i;
        const uint32_t bytes = uint32_t(min(CH, nrows - c * CH)) * D * 2;
        mbar_arrive_expect_tx(bar_full0 + 8 * i, 2 * bytes);
        const long long row = r0 + c * CH;
        bulk_load(sring + i * kStageBytes, Kc + row * D, bytes, bar_full0 + 8 * i);
        bulk_load(sring + i * kStageBytes + CHUNK_BYTES, Vc + row * D, bytes, bar_full0 + 8 * i);
      }
    }
    // everything above read only this layer's cache rows, which no earlier
    // kernel of the stream writes; the inputs below may come from the kernel
    // launched just before this one
    pdl_wait();
    // the new row, the mask bytes of the range
    for (int i = lane; append && i < D / 8; i += 32) {
      reinterpret_cast<uint4*>(kn_s)[i] = reinterpret_cast<const uint4*>(kn)[i];
      reinterpret_cast<uint4*>(vn_s)[i] = reinterpret_cast<const uint4*>(vn)[i];
    }
    const uint8_t* mrow = a.mask + (long long)b * R + r0;
    for (int i = lane; i < nrows; i += 32) mask_s[i] = mrow[i];
  }
  // the compute warps fetch their query slices before the first barrier so the
  // load overlaps the state, mask and K/V round trip
  uint4 qraw[G][V16];
  if (warp < kComputeWarps) {
    pdl_wait();
    const int li = lane % LPR;
    const uint16_t* qp = a.q + ((long long)b * a.q_heads + (long long)h * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < V16; ++j) qraw[g][j] = *reinterpret_cast<const uint4*>(qp + g * D + (j * LPR + li) * 8);
  }
  const int cur = st->cur_row;
  const bool state_ok = cur >= 0 && cur < R;
  if (oneshot) cp_async_wait_all();
  __syncthreads();
  // the merge barrier is initialised: peers may push once they pass the matching wait
  if (push) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  if (warp == kComputeWarps) {
    for (int c = lane; c < nchunks; c += 32) {
      uint8_t any = 0;
      for (int i = c * CH; i < min(nrows, (c + 1) * CH); ++i) any |= mask_s[i];
      chunk_on[c] = oneshot || (c >= c_first && c < c_first + nspec) || (c >= c_first + nspec && state_ok && any);
    }
  }
  if (!state_ok) {
    if (split == 0 && tid == 0) atomicCAS(&st->error, 0, kErrRowRange);
    for (int i = tid; i < nrows; i += kThreads) mask_s[i] = 0;
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int idx = nspec;
      for (int c = c_first + nspec; c < nchunks; ++c) {
        if (!chunk_on[c]) continue;
        const int s = idx % kStages;
        if (!wait_bar(bar_empty0 + 8 * s, ((idx / kStages) & 1) ^ 1, abort_flag, &st->error)) break;
        const uint32_t bytes = uint32_t(min(CH, nrows - c * CH)) * D * 2;
        mbar_arrive_expect_tx(bar_full0 + 8 * s, 2 * bytes);
        const long long row = r0 + c * CH;
        bulk_load(sring + s * kStageBytes, Kc + row * D, bytes, bar_full0 + 8 * s);
        bulk_load(sring + s * kStageBytes + CHUNK_BYTES, Vc + row * D, bytes, bar_full0 + 8 * s);
        ++idx;
      }
    }
    // append the step's row to the cache (the compute warps read it from kn_s / vn_s)
    if (append && state_ok && cur >= r0 && cur < r1) {
      for (int i = lane; i < D / 8; i += 32) {
        reinterpret_cast<uint4*>(Kc + (long long)cur * D)[i] = reinterpret_cast<const uint4*>(kn_s)[i];
        reinterpret_cast<uint4*>(Vc + (long long)cur * D)[i] = reinterpret_cast<const uint4*>(vn_s)[i];
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int li = lane % LPR, rg = lane / LPR;
    // query slice as fp32 pairs, pre-scaled into the exp2 domain
    uint64_t qr[G][E / 2];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < V16; ++j) {
        float f[8];
        bf16x8_to_f32(qraw[g][j], f);
#pragma unroll
        for (int e = 0; e < 8; e += 2)
          qr[g][(j * 8 + e) / 2] = pair_f32(__float_as_uint(f[e] * a.scale_log2), __float_as_uint(f[e + 1] * a.scale_log2));
      }
    float m_run[G], l_run[G];
    uint64_t acc[G][E / 2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -CUDART_INF_F;
      l_run[g] = 0.f;
#pragma unroll
      for (int e = 0; e < E / 2; ++e) acc[g][e] = 0ull;
    }
    // the step's row within the range (may be outside); without an append it
    // is read from the cache like any other row
    const int cur_i = append ? cur - r0 : -1;
    int idx = 0;
    for (int c = 0; c < nchunks; ++c) {
      if (!chunk_on[c]) continue;
      const int s = oneshot ? c : idx % kStages;
      if (!oneshot) {
        const bool ok = __all_sync(0xffffffffu, wait_bar(bar_full0 + 8 * s, (idx / kStages) & 1, abort_flag,
                                                           &st->error));
        if (!ok) break;
      }
      const uint8_t* Ks = smem + s * kStageBytes;
      const uint8_t* Vs = Ks + CHUNK_BYTES;
      float sc[PASSES][G];
      bool valid[PASSES];
      float cmax[G];
#pragma unroll
      for (int g = 0; g < G; ++g) cmax[g] = -CUDART_INF_F;
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const int rr = warp * RPC + p * RPW + rg;  // row within the chunk
        const int ri = c * CH + rr;                // row within the range
        valid[p] = ri < nrows && mask_s[ri] != 0;
        const uint8_t* krow = (ri == cur_i) ? kn_s : Ks + rr * D * 2;
        uint64_t acc2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc2[g] = 0ull;
#pragma unroll
        for (int j = 0; j < V16; ++j) {
          const uint4 kv = *reinterpret_cast<const uint4*>(krow + (j * LPR + li) * 16);
          const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint64_t k2 = bf16x2_to_pair(w[e]);
#pragma unroll
            for (int g = 0; g < G; ++g) ffma2(acc2[g], qr[g][j * 4 + e], k2);
          }
        }
        float acc_s[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          acc_s[g] = pair_lo(acc2[g]) + pair_hi(acc2[g]);
#pragma unroll
          for (int o = LPR / 2; o > 0; o >>= 1) acc_s[g] += __shfl_xor_sync(0xffffffffu, acc_s[g], o);
          sc[p][g] = valid[p] ? acc_s[g] : -CUDART_INF_F;
          cmax[g] = fmaxf(cmax[g], sc[p][g]);
        }
      }
      // chunk maximum over the warp's rows, then rescale the running state
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) cmax[g] = fmaxf(cmax[g], __shfl_xor_sync(0xffffffffu, cmax[g], o));
        const float mn = fmaxf(m_run[g], cmax[g]);
        if (mn > m_run[g]) {
          const float alpha = (m_run[g] == -CUDART_INF_F) ? 0.f : exp2f(m_run[g] - mn);
          l_run[g] *= alpha;
          const uint64_t a2 = pair_f32(__float_as_uint(alpha), __float_as_uint(alpha));
#pragma unroll
          for (int e = 0; e < E / 2; ++e) {
            uint64_t z = 0ull;
            ffma2(z, acc[g][e], a2);
            acc[g][e] = z;
          }
          m_run[g] = mn;
        }
      }
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        if (!valid[p]) continue;
        const int rr = warp * RPC + p * RPW + rg;
        const uint8_t* vrow = (c * CH + rr == cur_i) ? vn_s : Vs + rr * D * 2;
        uint64_t w2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float w = exp2f(sc[p][g] - m_run[g]);
          l_run[g] += w;
          w2[g] = pair_f32(__float_as_uint(w), __float_as_uint(w));
        }
#pragma unroll
        for (int j = 0; j < V16; ++j) {
          const uint4 vv = *reinterpret_cast<const uint4*>(vrow + (j * LPR + li) * 16);
          const uint32_t wv[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint64_t v2 = bf16x2_to_pair(wv[e]);
#pragma unroll
            for (int g = 0; g < G; ++g) ffma2(acc[g][j * 4 + e], w2[g], v2);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && !oneshot) mbar_arrive(bar_empty0 + 8 * s);
      ++idx;
    }
    // reduce the warp's row groups (every lane of a group holds the same weights)
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) l_run[g] += __shfl_xor_sync(0xffffffffu, l_run[g], o);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        float lo = pair_lo(acc[g][e]), hi = pair_hi(acc[g][e]);
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) {
          lo += __shfl_xor_sync(0xffffffffu, lo, o);
          hi += __shfl_xor_sync(0xffffffffu, hi, o);
        }
        acc[g][e] = pair_f32(__float_as_uint(lo), __float_as_uint(hi));
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s_m[warp][g] = m_run[g];
        s_l[warp][g] = l_run[g];
      }
    }
    // every warp rescales to the CTA maximum and the warps are summed into
    // kSlots shared-memory slots in a fixed order (round r adds warps
    // [r * kSlots, (r + 1) * kSlots)); the ring is free once all compute warps
    // are past their chunk loops
    constexpr int kSlots = merge_slots(NW, G, D);
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");
    float* red = reinterpret_cast<float*>(smem);  // [kSlots][G][D]
    float scale_w[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, s_m[w][g]);
      scale_w[g] = (m_run[g] == -CUDART_INF_F) ? 0.f : exp2f(m_run[g] - M);
    }
    const int slot = warp % kSlots;
#pragma unroll 1
    for (int r = 0; r < kComputeWarps / kSlots; ++r) {
      if (warp / kSlots == r && rg == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int j = 0; j < V16; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float* d = &red[(slot * G + g) * D + (j * LPR + li) * 8 + e];
              const uint64_t pr = acc[g][(j * 8 + e) / 2];
              const float v = scale_w[g] * ((e & 1) ? pair_hi(pr) : pair_lo(pr));
              *d = (r == 0) ? v : *d + v;
            }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");
    }
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  if (aborted && tid == kComputeWarps * 32) {
    // let bulk copies in flight land before shared memory is reused or released
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }

  // ---- this CTA's (M, L) and accumulator (slots summed in a fixed order)
  constexpr int kSlots = merge_slots(NW, G, D);
  if (tid < G) {
    float M = -CUDART_INF_F;
    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, s_m[w][tid]);
    float L = 0.f;
    for (int w = 0; w < kComputeWarps; ++w)
      if (s_m[w][tid] != -CUDART_INF_F) L += exp2f(s_m[w][tid] - M) * s_l[w][tid];
    s_M[tid] = M;
    s_L[tid] = L;
  }
  float* red = reinterpret_cast<float*>(smem);
  float* cta_acc = red + kSlots * G * D;  // [G][D]
  for (int i = tid; i < G * D; i += kThreads) {
    float o = red[i];
#pragma unroll
    for (int k = 1; k < kSlots; ++k) o += red[k * G * D + i];
    cta_acc[i] = o;
  }
  __syncthreads();
  const long long head0 = (long long)b * a.q_heads + (long long)h * G;
  const int nsplit = a.nsplit;

  if (nsplit == 1) {
    if (!aborted) {
      for (int i = tid; i < G * D / 2; i += kThreads) {
        const int g = (2 * i) / D;
        const float L = s_L[g];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<uint32_t*>(a.out + head0 * D)[i] = pack_bf16(cta_acc[2 * i] * inv, cta_acc[2 * i + 1] * inv);
      }
      if (tid < G && a.lse)
        a.lse[head0 + tid] = s_L[tid] > 0.f ? (s_M[tid] + log2f(s_L[tid])) * 0.69314718055994530942f : -CUDART_INF_F;
    }
    return;
  }

  if (push) {
    // ---- cluster merge by pushes (see s_recv)
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    const int rank = int(cluster_ctarank());
    const float4* acc4 = reinterpret_cast<const float4*>(cta_acc);
    for (int x = tid; x < nsplit * (1 + slice); x += kThreads) {
      const int k = x / (1 + slice), j = x % (1 + slice);
      // item 0 of each destination: this CTA's (M, L) per query head
      const float4 val = (j == 0) ? make_float4(s_M[0], s_L[0], s_M[G - 1], s_L[G - 1]) : acc4[k * slice + j - 1];
      st_async_u32x4(map_shared(smem_u32(&s_recv[rank * (1 + slice) + j]), uint32_t(k)), __float_as_uint(val.x),
                     __float_as_uint(val.y), __float_as_uint(val.z), __float_as_uint(val.w),
                     map_shared(smem_u32(&s_merge_bar), uint32_t(k)));
    }
    // this CTA's slice from every CTA of the cluster (bounded wait)
    bool got = true;
    if (tid < slice) {
      const uint64_t t0 = globaltimer_ns();
      while (!(got = mbar_try_wait(smem_u32(&s_merge_bar), 0)) && globaltimer_ns() - t0 < 2000000000ull) {
      }
      if (!got) atomicCAS(&st->error, 0, kErrTimeout);
    }
    if (tid < slice && got && !aborted) {
      const int f = rank * slice + tid;
      const int g = (4 * f) / D;
      float M = -CUDART_INF_F;
      for (int r = 0; r < nsplit; ++r) {
        const float4 hdr = s_recv[r * (1 + slice)];
        M = fmaxf(M, g ? hdr.z : hdr.x);
      }
      float L = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < nsplit; ++r) {  // fixed order: CTA rank
        const float4 hdr = s_recv[r * (1 + slice)];
        const float ms = g ? hdr.z : hdr.x, ls = g ? hdr.w : hdr.y;
        const float w = (ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
        const float4 v = s_recv[r * (1 + slice) + 1 + tid];
        L += w * ls;
        o.x = fmaf(w, v.x, o.x);
        o.y = fmaf(w, v.y, o.y);
        o.z = fmaf(w, v.z, o.z);
        o.w = fmaf(w, v.w, o.w);
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      reinterpret_cast<uint2*>(a.out + head0 * D)[f] =
          make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
      if (a.lse && 4 * f == g * D)
        a.lse[head0 + g] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -CUDART_INF_F;
    }
    return;
  }

  if (a.cluster) {
    // ---- cluster merge: rank 0 reads every CTA's (M, L, accumulator) through
    // distributed shared memory; every CTA reaches both cluster barriers
    cluster_sync();
    if (!aborted) {
      // every CTA merges its own slice of the output columns from all CTAs of
      // the cluster (remote loads issued together; fixed summation order)
      float* wts = cta_acc + G * D;  // [G][nsplit]
      float* sms = wts + G * nsplit;
      float* sls = sms + G * nsplit;
      __shared__ float s_gM[G], s_gL[G];
      for (int x = tid; x < G * nsplit; x += kThreads) {
        const int g = x / nsplit, r = x % nsplit;
        sms[x] = ld_dsmem_f32(map_shared(smem_u32(&s_M[g]), r));
        sls[x] = ld_dsmem_f32(map_shared(smem_u32(&s_L[g]), r));
      }
      __syncthreads();
      if (tid < G) {
        const int g = tid;
        float M = -CUDART_INF_F;
        for (int r = 0; r < nsplit; ++r) M = fmaxf(M, sms[g * nsplit + r]);
        float L = 0.f;
        for (int r = 0; r < nsplit; ++r) {
          const float ms = sms[g * nsplit + r];
          const float w = (ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
          wts[g * nsplit + r] = w;
          L += w * sls[g * nsplit + r];
        }
        s_gM[g] = M;
        s_gL[g] = L;
      }
      __syncthreads();
      const int nf = G * D / 4;
      const int rank = int(cluster_ctarank());
      const int f0 = rank * nf / nsplit, f1 = (rank + 1) * nf / nsplit;
      for (int f = f0 + tid; f < f1; f += kThreads) {
        const int g = (4 * f) / D;
        const uint32_t local = smem_u32(cta_acc + 4 * f);
        float4 v[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < nsplit) v[r] = ld_dsmem_f32x4(map_shared(local, r));
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < nsplit) {
            const float w = wts[g * nsplit + r];
            o.x = fmaf(w, v[r].x, o.x);
            o.y = fmaf(w, v[r].y, o.y);
            o.z = fmaf(w, v[r].z, o.z);
            o.w = fmaf(w, v[r].w, o.w);
          }
        const float L = s_gL[g];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<uint2*>(a.out + head0 * D)[f] =
            make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
      }
      if (rank == 0 && tid < G && a.lse)
        a.lse[head0 + tid] = s_gL[tid] > 0.f ? (s_gM[tid] + log2f(s_gL[tid])) * 0.69314718055994530942f : -CUDART_INF_F;
    }
    cluster_sync();
    return;
  }

  // ---- workspace merge.  Every CTA takes a ticket, an aborted one with a
  // mark in the upper bits, so the last CTA of the slab always resets the
  // counter (the workspace is ready for the next call) and writes the output
  // only when no CTA of the slab gave up.
  if (!aborted) {
    for (int i = tid; i < G * D; i += kThreads) {
      const int g = i / D, d = i % D;
      a.ws_acc[((head0 + g) * nsplit + split) * D + d] = cta_acc[i];
    }
    if (tid < G) {
      a.ws_ml[((head0 + tid) * nsplit + split) * 2 + 0] = s_M[tid];
      a.ws_ml[((head0 + tid) * nsplit + split) * 2 + 1] = s_L[tid];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    constexpr int kAbortMark = 1 << 16;
    const int ticket = atomicAdd(&a.counters[b * a.kv_heads + h], aborted ? 1 + kAbortMark : 1);
    const bool last = (ticket & (kAbortMark - 1)) == nsplit - 1;
    const bool any_abort = aborted || ticket >= kAbortMark;
    if (last && any_abort) a.counters[b * a.kv_heads + h] = 0;
    s_last = last && !any_abort;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA of the slab: statistics staged with independent loads, then the
  // accumulators 16 splits at a time as float4 (fixed summation order)
  float* wts = cta_acc + G * D;  // [G][nsplit]
  float* sms = wts + G * nsplit;
  float* sls = sms + G * nsplit;
  for (int x = tid; x < G * nsplit; x += kThreads) {
    const int g = x / nsplit, s = x % nsplit;
    sms[x] = __ldcg(&a.ws_ml[((head0 + g) * nsplit + s) * 2]);
    sls[x] = __ldcg(&a.ws_ml[((head0 + g) * nsplit + s) * 2 + 1]);
  }
  __syncthreads();
  if (tid < G) {
    const int g = tid;
    float M = -CUDART_INF_F;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, sms[g * nsplit + s]);
    float Lsum = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = sms[g * nsplit + s];
      const float w = (ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
      wts[g * nsplit + s] = w;
      Lsum += w * sls[g * nsplit + s];
    }
    s_M[g] = M;
    s_L[g] = Lsum;
  }
  __syncthreads();
  for (int f = tid; f < G * D / 4; f += kThreads) {
    const int g = (4 * f) / D, d = (4 * f) % D;
    const float4* src = reinterpret_cast<const float4*>(a.ws_acc + (head0 + g) * nsplit * (long long)D + d);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += 16) {
      float4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (s0 + u < nsplit) v[u] = __ldcg(src + (long long)(s0 + u) * (D / 4));
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (s0 + u < nsplit) {
          const float w = wts[g * nsplit + s0 + u];
          o.x = fmaf(w, v[u].x, o.x);
          o.y = fmaf(w, v[u].y, o.y);
          o.z = fmaf(w, v[u].z, o.z);
          o.w = fmaf(w, v[u].w, o.w);
        }
    }
    const float L = s_L[g];
    const float inv = L > 0.f ? 1.f / L : 0.f;
    reinterpret_cast<uint2*>(a.out + head0 * D)[f] =
        make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
  }
  if (tid < G && a.lse)
    a.lse[head0 + tid] = s_L[tid] > 0.f ? (s_M[tid] + log2f(s_L[tid])) * 0.69314718055994530942f : -CUDART_INF_F;
  if (tid == 0) a.counters[b * a.kv_heads + h] = 0;
}

size_t smem_bytes(int rows_per_split, int ch, int d) {
  const size_t ring = size_t(kStages) * kStageBytes;
  const size_t mask = (size_t(rows_per_split) + 15) & ~size_t(15);
  const size_t flags = ((size_t(rows_per_split) + ch - 1) / ch + 15) & ~size_t(15);
  return ring + 4 * size_t(d) + mask + flags + 2 * kStages * 8 + 16;
}

template <int D, int G, int NW>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
  // the merge areas reuse the ring
  if (size_t(merge_slots(NW, G, D) + 1) * G * D * 4 + size_t(3) * G * a.nsplit * 4 > size_t(kStages) * kStageBytes)
    return cudaErrorInvalidValue;
  const size_t smem = smem_bytes(a.rows_per_split, Shape<D, G, NW>::CH, D);
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(decode_kernel<D, G, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, 110 * 1024);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(decode_kernel<D, G, NW>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr != cudaSuccess) return attr;
  if (smem > 110 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.kv_heads, a.batch);
  cfg.blockDim = dim3(32 * (NW + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  // programmatic dependent launch: the kernel prefetches its cache rows while
  // the previous kernel of the stream finishes (it waits before reading inputs)
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (a.cluster) {
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = a.nsplit;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, G, NW>, a);
}

template <int D, int G>
cudaError_t launch_w(const DecodeArgs& a, cudaStream_t s) {
  return a.warps == 16 ? launch_t<D, G, 16>(a, s) : launch_t<D, G, 8>(a, s);
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
  switch (a.q_heads / a.kv_heads) {
    case 1: return launch_w<D, 1>(a, s);
    case 2: return launch_w<D, 2>(a, s);
    case 4: return launch_w<D, 4>(a, s);
    case 8: return launch_w<D, 8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

DecodeSplit decode_split(int batch, int q_heads, int kv_heads, int head_dim, int rows, int sm_count,
                         int max_cluster) {
  DecodeSplit d;
  const int ch = kStageBytes / (2 * head_dim * 2);
  const long long pairs = (long long)batch * kv_heads;
  const int sms = sm_count > 0 ? sm_count : 152;
  const int min_rows = 2 * ch > 64 ? 2 * ch : 64;
  long long max_ns = (rows + min_rows - 1) / min_rows;
  if (max_ns > 64) max_ns = 64;
  long long ns;
  if (pairs >= sms) {
    // throughput regime: 8 compute warps, two CTAs per SM, a few splits per
    // slab for load balance, merged through the workspace
    d.warps = 8;
    ns = (8LL * sms + pairs - 1) / pairs;
    if (ns > 4) ns = 4;
  } else {
    // latency regime: 16 compute warps, as many CTAs as the cluster allows
    d.warps = 16;
    ns = (2LL * sms + pairs - 1) / pairs;
    if (ns > max_cluster && (rows + max_cluster - 1) / max_cluster <= 8 * ch) ns = max_cluster;
  }
  if (ns > max_ns) ns = max_ns;
  if (ns < 1) ns = 1;
  d.rows_per_split = int((rows + ns - 1) / ns);
  d.nsplit = (rows + d.rows_per_split - 1) / d.rows_per_split;
  d.cluster = (d.warps == 16 && d.nsplit > 1 && d.nsplit <= max_cluster) ? 1 : 0;
  const size_t counters = size_t(pairs) * sizeof(int32_t);
  const size_t ml = size_t(batch) * q_heads * d.nsplit * 2 * sizeof(float);
  const size_t acc = size_t(batch) * q_heads * d.nsplit * head_dim * sizeof(float);
  d.off_ml = align256(counters);
  d.off_acc = d.off_ml + align256(ml);
  d.total = d.off_acc + align256(acc);
  return d;
}

int decode_max_cluster() {
  // the largest cluster of decode CTAs the current device can co-schedule
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int best = 8;
    if (cudaFuncSetAttribute(decode_kernel<256, 2, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess &&
        cudaFuncSetAttribute(decode_kernel<256, 2, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 110 * 1024) ==
            cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1, 1);
      cfg.blockDim = dim3(32 * 17);
      cfg.dynamicSmemBytes = smem_bytes(128, Shape<256, 2, 16>::CH, 256);
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 16;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<256, 2, 16>, &cfg) == cudaSuccess && n >= 2) best = 16;
      cudaGetLastError();
    }
    cached[dev] = best;
  }
  return cached[dev];
}

cudaError_t decode_static_scratch(void** ptr) {
  static std::mutex mu;
  static void* cached[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // with this device current
    if (e != cudaSuccess) return e;
    // the ticket area starts at zero (the array is zero at load; cleared once
    // more here, synchronously); every decode leaves its tickets at zero
    e = cudaMemset(p, 0, align256(size_t(SWA_DECODE_STATIC_MAX_SLABS) * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    cached[dev] = p;
  }
  *ptr = cached[dev];
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  // the latency regime (16 compute warps: few slabs) goes to the tensor-core kernel
  if (a.warps == 16 && decode_small_eligible(a)) return launch_decode_small(a, s);
  switch (a.head_dim) {
    case 64: return launch_d<64>(a, s);
    case 128: return launch_d<128>(a, s);
    case 256: return launch_d<256>(a, s);
    case 512: return launch_d<512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swa
