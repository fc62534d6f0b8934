// Single-token decode for few (sequence, KV head) slabs: the latency regime
// (the single-stream workload: B = 1, Hkv = 2, 1088 rows per slab).
//
// Launch: one thread-block cluster of `nsplit` CTAs (at most 16) per slab;
// CTA k owns rows [k R / nsplit, ...) of the slab (at most 128, 96 at head size 512).  The work is
// tiny (68 rows x 2 heads x 256 columns per CTA) and on the critical path of a
// dependent chain of launches, so the kernel is built for latency:
//   * before griddepcontrol.wait (i.e. while the previous kernel of the stream
//     still runs) every thread copies the CTA's K and V rows into shared
//     memory with 16-byte asynchronous copies, 128-byte-swizzled so the
//     warp-level tensor-core loads below are free of bank conflicts;
//   * after the wait: the runtime mask, the query, the cache state and the
//     step's new row arrive in one round trip;
//   * scores S = K q^T with warp-level tensor-core products (mma.sync
//     m16n8k16, bf16 in, fp32 out): a warp takes 16 rows, the G query heads
//     of the group are the N dimension (one loaded K row serves the whole
//     group), two accumulator chains over the head dimension;
//   * one warp per query head takes the maximum and the exponentials over the
//     CTA's rows (bf16 probabilities, the normaliser is the sum of the same
//     rounded values, lse uses the unrounded sum);
//   * O = P V with the same products, each warp owning a slice of the head
//     dimension for all rows, so no merge between warps is needed;
//   * the CTAs of the cluster merge (M, L, O) by pushes into each other's
//     shared memory (each CTA finishes 1 / nsplit of the output columns).
// The current step's row comes from k_new / v_new (and is appended to the
// cache by the CTA that owns it); a KV-sharing call (no k_new) reads the
// cache after the wait.  The tensor-core products here are 16 x 8 tiles on
// the warp-level path: with 68 rows per CTA the latency of one dependent
// chain matters, not throughput.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary (the step's new row goes into the compact cache at its
// row index; one runtime mask per step) and Compilation behavior (decode
// reads only the rows of the compact buffer); "Add SDPA attention
// implementation", Summary (K/V shared by query-head groups).

#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace swa {
namespace {

using namespace ptx;

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
// rows per CTA: at most 128, and K + V of them within 192 KB of shared memory
__host__ __device__ constexpr int max_rows(int d) { return (192 * 1024) / (4 * d) < 128 ? ((192 * 1024) / (4 * d)) & ~15 : 128; }
constexpr uint64_t kTimeoutNs = 2000000000ull;

// Offset of 16-byte unit `u` of row `r` in a row-major tile of `units`
// units per row, with the unit index XOR-swizzled by the row (8 rows cover
// all 32 banks for any 16-byte column).
__device__ __forceinline__ uint32_t swz(int r, int u, int units) { return uint32_t((r * units + (u ^ (r & 7))) * 16); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// d += a * b, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x on the special-function unit (subnormal results flush to 0; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Shared memory (dynamic): K [RP][D] | V [RP][D] (swizzled bf16, RP = rows
// rounded up to 16) | per-block statistics [3][G][8] fp32 (maximum, rounded
// and unrounded sums of each 16-row block) | P [G][RP] bf16 | O [G][D] fp32 |
// the step's new K and V rows [2][D] bf16 | mask bytes [RP].  The merge area
// is static.
template <int D>
struct SmallLayout {
  static constexpr int U = D / 8;  // 16-byte units per row
  __host__ __device__ static size_t kv(int rp) { return size_t(rp) * D * 2; }
  __host__ __device__ static size_t off_v(int rp) { return kv(rp); }
  __host__ __device__ static size_t off_s(int rp) { return 2 * kv(rp); }
  __host__ __device__ static size_t off_p(int rp, int g) { return off_s(rp) + size_t(3 * 8) * g * 4; }
  __host__ __device__ static size_t off_o(int rp, int g) { return (off_p(rp, g) + size_t(g) * rp * 2 + 15) & ~size_t(15); }
  __host__ __device__ static size_t off_n(int rp, int g) { return off_o(rp, g) + size_t(g) * D * 4; }
  __host__ __device__ static size_t off_m(int rp, int g) { return off_n(rp, g) + size_t(2) * D * 2; }
  __host__ __device__ static size_t total(int rp, int g) { return off_m(rp, g) + size_t(rp); }
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) decode_small_kernel(const DecodeArgs a) {
  using LY = SmallLayout<D>;
  constexpr int U = LY::U;
  constexpr int KSTEPS = D / 16;
  constexpr int NB = D / 8 / kWarps;  // 8-column output blocks per warp
  static_assert(NB >= 1 && G <= 2, "shape");
  constexpr int kNf = G * D / 4;  // float4s of one CTA's accumulator
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int R = a.rows;
  const int r0 = split * a.rows_per_split;
  const int r1 = min(R, r0 + a.rows_per_split);
  const int nrows = max(0, r1 - r0);
  const int RP = (a.rows_per_split + 15) & ~15;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nsplit = a.nsplit;
  const int slice = kNf / nsplit;

  uint8_t* sK = smem;
  uint8_t* sV = smem + LY::off_v(RP);
  float* sB = reinterpret_cast<float*>(smem + LY::off_s(RP));          // [3][G][8] block statistics
  uint16_t* sP = reinterpret_cast<uint16_t*>(smem + LY::off_p(RP, G));  // [G][RP]
  float* sO = reinterpret_cast<float*>(smem + LY::off_o(RP, G));        // [G][D]
  uint8_t* sN = smem + LY::off_n(RP, G);                                // new K row | new V row
  uint8_t* mask_s = smem + LY::off_m(RP, G);
  __shared__ __align__(16) float4 s_recv[32 + kNf];  // 16 CTAs x 2 header items + accumulator slices
  __shared__ __align__(8) uint64_t s_merge_bar;
  __shared__ float s_M[G], s_L[G], s_E[G];
  const uint32_t kbase = smem_u32(sK), vbase = smem_u32(sV);

  if (tid == 0) pdl_launch_dependents();
  swa_device_state* st = a.state;
  const long long slab = (((long long)a.layer * a.batch + b) * a.kv_heads + h) * (long long)R * D;
  uint16_t* Kc = a.k_cache + slab;
  uint16_t* Vc = a.v_cache + slab;
  const bool append = a.k_new != nullptr;
  // KV-sharing layer: the owning layer's decode, possibly the kernel launched
  // just before, writes this step's row: even the cache is read after the wait
  if (!append) pdl_wait();
  // rows [nrows, RP) of the last 16-row block are zero: they meet zero weights
  for (int x = tid; x < (RP - nrows) * U; x += kThreads) {
    const int r = nrows + x / U, u = x % U;
    *reinterpret_cast<uint4*>(sK + swz(r, u, U)) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(sV + swz(r, u, U)) = make_uint4(0, 0, 0, 0);
  }
  for (int x = tid; x < 2 * nrows * U; x += kThreads) {
    const int kv = x >= nrows * U, y = kv ? x - nrows * U : x;
    const int r = y / U, u = y % U;
    cp_async_16((kv ? vbase : kbase) + swz(r, u, U), (kv ? Vc : Kc) + (long long)(r0 + r) * D + u * 8);
  }
  if (tid == 0 && nsplit > 1) {
    // phase 0 completes when every CTA's slice (header + accumulator) landed
    mbar_init(smem_u32(&s_merge_bar), 1);
    mbar_arrive_expect_tx(smem_u32(&s_merge_bar), uint32_t(nsplit * (2 + slice) * 16));
    fence_mbar_init();
  }
  // everything above read only this layer's cache rows, which no earlier
  // kernel of the stream writes; the inputs below may come from the kernel
  // launched just before this one, unless the caller said they were ready
  // before it (then they are read first and the wait overlaps their round trip)
  int cur;
  const int gq = lane >> 2;
  uint32_t bq[KSTEPS][2];
  auto read_inputs = [&] {
    cur = st->cur_row;
    for (int i = tid; i < nrows; i += kThreads) mask_s[i] = a.mask[(long long)b * R + r0 + i];
    // score operand: the group's queries, lane l holding heads g = l / 4 (zero
    // beyond G) at columns 16 kk + 2 (l % 4) + {0, 1} and + 8
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q + ((long long)b * a.q_heads + (long long)h * G + gq) * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      bq[kk][0] = gq < G ? qp[kk * 8 + (lane & 3)] : 0u;
      bq[kk][1] = gq < G ? qp[kk * 8 + 4 + (lane & 3)] : 0u;
    }
    // the step's new row, in the same round trip (only the owning CTA uses it)
    if (append && tid < 2 * U) {
      const int kv = tid >= U, u = kv ? tid - U : tid;
      cp_async_16(smem_u32(sN) + tid * 16, (kv ? a.v_new : a.k_new) + ((long long)b * a.kv_heads + h) * D + u * 8);
    }
  };
  const bool early = a.inputs_ready && append;
  if (early) read_inputs();
  pdl_wait();
  if (!early) read_inputs();
  const bool state_ok = cur >= 0 && cur < R;
  const int cur_i = (append && state_ok) ? cur - r0 : -1;
  cp_async_wait_all();
  __syncthreads();  // (cp.async data, mask bytes)
  // the merge barrier is initialised: peers may push once they pass the matching wait
  if (nsplit > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  if (cur_i >= 0 && cur_i < nrows) {
    // this CTA owns the step's row: it replaces the prefetched row and is appended
    for (int u = tid; u < 2 * U; u += kThreads) {
      const int kv = u >= U, uu = kv ? u - U : u;
      const uint4 x = reinterpret_cast<const uint4*>(sN)[u];
      *reinterpret_cast<uint4*>((kv ? sV : sK) + swz(cur_i, uu, U)) = x;
      reinterpret_cast<uint4*>((kv ? Vc : Kc) + (long long)cur * D)[uu] = x;
    }
  }
  if (!state_ok && split == 0 && tid == 0) atomicCAS(&st->error, 0, kErrRowRange);
  __syncthreads();

  // ---- scores: warp w takes 16-row blocks w, w + 8, ...  A lane holds rows
  // rb * 16 + l / 4 (+ 8) of heads 2 (l % 4) (+ 1): for G <= 2 the lanes
  // with l % 4 == 0.  Each block's maximum goes to shared memory; after one
  // barrier every warp turns its own block into probabilities.
  const float c2 = a.scale_log2;
  float sc[2][4];  // scores of this warp's blocks (exp2 domain; -inf when masked)
  const int nblk = RP / 16;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rb = warp + t * kWarps;
    if (rb >= nblk) break;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int ar = rb * 16 + (lane & 15);  // row this lane addresses for ldmatrix
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      uint32_t af[4];
      ldsm_x4(kbase + swz(ar, 2 * kk + (lane >> 4), U), af[0], af[1], af[2], af[3]);
      mma16816(acc[kk & 1], af, bq[kk][0], bq[kk][1]);
    }
    float bm[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int rr = rb * 16 + (lane >> 2) + ((e & 2) ? 8 : 0);
      const bool in = (lane & 3) == 0 && rr < nrows && state_ok && mask_s[rr] != 0;
      sc[t][e] = in ? (acc[0][e] + acc[1][e]) * c2 : -CUDART_INF_F;
      bm[e & 1] = fmaxf(bm[e & 1], sc[t][e]);
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      bm[0] = fmaxf(bm[0], __shfl_xor_sync(0xffffffffu, bm[0], o));
      bm[1] = fmaxf(bm[1], __shfl_xor_sync(0xffffffffu, bm[1], o));
    }
    if (lane == 0) {  // the lanes with l % 4 == 0 were reduced into lane 0
#pragma unroll
      for (int g = 0; g < G; ++g) sB[g * 8 + rb] = bm[g];
    }
  }
  __syncthreads();

  // ---- probabilities of the warp's blocks against the CTA maximum M: P in
  // bf16; the block's rounded and unrounded sums
  float M[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = -CUDART_INF_F;
    for (int k = 0; k < nblk; ++k) M[g] = fmaxf(M[g], sB[g * 8 + k]);
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rb = warp + t * kWarps;
    if (rb >= nblk) break;
    float lr[2] = {0.f, 0.f}, le[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int g = e & 1;
      if (g < G && (lane & 3) == 0) {
        const int rr = rb * 16 + (lane >> 2) + ((e & 2) ? 8 : 0);
        const float p = ex2(sc[t][e] - (M[g] == -CUDART_INF_F ? 0.f : M[g]));  // -inf -> 0
        const __nv_bfloat16 pb = __float2bfloat16_rn(p);
        sP[g * RP + rr] = *reinterpret_cast<const uint16_t*>(&pb);
        lr[g] += __bfloat162float(pb);
        le[g] += p;
      }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        lr[g] += __shfl_xor_sync(0xffffffffu, lr[g], o);
        le[g] += __shfl_xor_sync(0xffffffffu, le[g], o);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        sB[(G + g) * 8 + rb] = lr[g];
        sB[(2 * G + g) * 8 + rb] = le[g];
      }
    }
  }
  __syncthreads();
  if (tid < G) {  // the CTA's statistics: maximum, rounded and unrounded sums
    float L = 0.f, E = 0.f;
    for (int k = 0; k < nblk; ++k) {
      L += sB[(G + tid) * 8 + k];
      E += sB[(2 * G + tid) * 8 + k];
    }
    s_M[tid] = tid == 0 ? M[0] : M[G - 1];
    s_L[tid] = L;
    s_E[tid] = E;
  }

  // ---- O = P V: warp w takes head-dimension columns [w D / 8, (w + 1) D / 8)
  {
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    const int n0u = warp * NB;  // first 16-byte unit (8 columns) of this warp
    for (int kb = 0; kb < RP / 16; ++kb) {
      // A: probabilities of head l / 4 (zero beyond G), keys kb * 16 + 2 (l % 4) + {0, 1} and + 8
      uint32_t af[4] = {0u, 0u, 0u, 0u};
      if (gq < G) {
        const uint32_t* pp = reinterpret_cast<const uint32_t*>(sP + gq * RP + kb * 16);
        af[0] = pp[lane & 3];
        af[2] = pp[4 + (lane & 3)];
      }
      // B: V rows kb * 16 + (l % 16), two 8-column blocks per ldmatrix
#pragma unroll
      for (int nb = 0; nb < NB; nb += 2) {
        uint32_t b0, b1, b2, b3;
        const int vr = kb * 16 + (lane & 15);
        const int vu = n0u + nb + (lane >> 4);
        ldsm_x4_t(vbase + swz(vr, vu, U), b0, b1, b2, b3);
        mma16816(acc[nb], af, b0, b1);
        if (nb + 1 < NB) mma16816(acc[nb + 1], af, b2, b3);
      }
    }
    // lane l holds head l / 4 at columns 8 (n0u + nb) + 2 (l % 4) + {0, 1}
    if (gq < G) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        *reinterpret_cast<float2*>(sO + gq * D + (n0u + nb) * 8 + 2 * (lane & 3)) = make_float2(acc[nb][0], acc[nb][1]);
    }
  }
  __syncthreads();

  const long long head0 = (long long)b * a.q_heads + (long long)h * G;
  if (nsplit == 1) {
    for (int i = tid; i < G * D / 2; i += kThreads) {
      const int g = (2 * i) / D;
      const float L = s_L[g];
      const float inv = L > 0.f ? 1.f / L : 0.f;
      reinterpret_cast<uint32_t*>(a.out + head0 * D)[i] = pack_bf16(sO[2 * i] * inv, sO[2 * i + 1] * inv);
    }
    if (tid < G && a.lse)
      a.lse[head0 + tid] = s_E[tid] > 0.f ? (s_M[tid] + log2f(s_E[tid])) * 0.69314718055994530942f : -CUDART_INF_F;
    return;
  }

  // ---- cluster merge by pushes: every CTA sends each CTA of the cluster two
  // header items, (M, L, E) of each query head (maximum, rounded and
  // unrounded sums), and that CTA's slice of its accumulator, with
  // asynchronous remote stores; each CTA waits for its slice from all and
  // finishes it (fixed summation order: CTA rank)
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  const int rank = int(cluster_ctarank());
  constexpr int HDR = 2;
  const int item = HDR + slice;
  const float4* acc4 = reinterpret_cast<const float4*>(sO);
  for (int x = tid; x < nsplit * item; x += kThreads) {
    const int k = x / item, j = x % item;
    const int gh = (j == 1) ? G - 1 : 0;
    const float4 val = (j < HDR) ? make_float4(s_M[gh], s_L[gh], s_E[gh], 0.f) : acc4[k * slice + j - HDR];
    st_async_u32x4(map_shared(smem_u32(&s_recv[rank * item + j]), uint32_t(k)), __float_as_uint(val.x),
                   __float_as_uint(val.y), __float_as_uint(val.z), __float_as_uint(val.w),
                   map_shared(smem_u32(&s_merge_bar), uint32_t(k)));
  }
  bool got = true;
  if (tid < slice) {
    const uint64_t t0 = globaltimer_ns();
    while (!(got = mbar_test_wait(smem_u32(&s_merge_bar), 0)) && globaltimer_ns() - t0 < kTimeoutNs) {
    }
    if (!got) atomicCAS(&st->error, 0, kErrTimeout);
  }
  if (tid < slice && got) {
    const int f = rank * slice + tid;
    const int g = (4 * f) / D;
    float M = -CUDART_INF_F;
    for (int r = 0; r < nsplit; ++r) M = fmaxf(M, s_recv[r * item + (g ? 1 : 0)].x);
    float L = 0.f, E = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < nsplit; ++r) {
      const float4 hdr = s_recv[r * item + (g ? 1 : 0)];
      const float w = (hdr.x == -CUDART_INF_F) ? 0.f : exp2f(hdr.x - M);
      const float4 v = s_recv[r * item + HDR + tid];
      L += w * hdr.y;
      E += w * hdr.z;
      o.x = fmaf(w, v.x, o.x);
      o.y = fmaf(w, v.y, o.y);
      o.z = fmaf(w, v.z, o.z);
      o.w = fmaf(w, v.w, o.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    reinterpret_cast<uint2*>(a.out + head0 * D)[f] =
        make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
    if (a.lse && 4 * f == g * D)
      a.lse[head0 + g] = E > 0.f ? (M + log2f(E)) * 0.69314718055994530942f : -CUDART_INF_F;
  }
}

template <int D, int G>
cudaError_t launch_small(const DecodeArgs& a, cudaStream_t s) {
  const int rp = (a.rows_per_split + 15) & ~15;
  const size_t smem = SmallLayout<D>::total(rp, G);
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(decode_small_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(SmallLayout<D>::total(max_rows(D), G)));
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(decode_small_kernel<D, G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.kv_heads, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (a.nsplit > 1) {
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = a.nsplit;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, decode_small_kernel<D, G>, a);
}

template <int D>
cudaError_t launch_small_d(const DecodeArgs& a, cudaStream_t s) {
  return (a.q_heads / a.kv_heads) == 1 ? launch_small<D, 1>(a, s) : launch_small<D, 2>(a, s);
}

}  // namespace

bool decode_small_eligible(const DecodeArgs& a) {
  const int g = a.q_heads / a.kv_heads;
  if (g < 1 || g > 2) return false;
  if (a.head_dim != 128 && a.head_dim != 256 && a.head_dim != 512) return false;
  if (a.rows_per_split > max_rows(a.head_dim) || a.nsplit < 1 || a.nsplit > 16) return false;
  if (a.nsplit > 1 && !a.cluster) return false;
  const int nf = g * a.head_dim / 4;  // float4s of one CTA's accumulator
  return nf <= 256 && nf % a.nsplit == 0;
}

cudaError_t launch_decode_small(const DecodeArgs& a, cudaStream_t s) {
  switch (a.head_dim) {
    case 128: return launch_small_d<128>(a, s);
    case 256: return launch_small_d<256>(a, s);
    case 512: return launch_small_d<512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swa
