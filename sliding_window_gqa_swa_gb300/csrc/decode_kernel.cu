// Single-token decode over the compact cache: append, split-K partial
// attention and the combine, in one launch.
//
// Grid (nsplit, Hkv, B); each CTA owns a contiguous range of cache rows of
// one (sequence, kv head) slab and serves all G = Hq / Hkv query heads of the
// group from every K/V row it loads (grouped-query reuse).  A row is split
// across LPR lanes so each 16-byte load instruction of a lane group covers a
// contiguous 128-byte span of the row; rows the runtime mask rejects are
// never loaded.  Partial (max, sum, accumulator) go to the workspace; the
// last CTA of each (sequence, kv head) -- found with an atomic ticket, no
// waiting -- merges them, writes the bf16 output and resets the ticket.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary (decode writes through the compact cache index; one
// runtime mask per step) and Compilation behavior (decode scans only the
// compact 1088-row allocation); "Add SDPA attention implementation", Summary
// (K/V shared by query-head groups).

#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"

// Scratch of swa_decode_noalloc (tickets, split statistics, split partials)
// for callers that cannot allocate device memory.  Every GPU that loads the
// library holds it until the process exits.  In host code this name is only a
// host-side stand-in: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[SWA_DECODE_STATIC_SCRATCH_BYTES];

namespace swa {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kDecodeWarps = kDecodeThreads / 32;

template <int D, int G>
struct DecodeShape {
  static constexpr int kWant = D * G / 64;
  static constexpr int LPR = kWant < 8 ? 8 : (kWant > 32 ? 32 : kWant);  // lanes per row
  static constexpr int E = D / LPR;        // elements per lane
  static constexpr int V16 = E / 8;        // 16-byte vectors per lane per row
  static constexpr int RPW = 32 / LPR;     // rows per warp pass
  static constexpr int U = (V16 * 2 <= 8) ? 4 : 2;  // passes in flight
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(const DecodeArgs a) {
  using S = DecodeShape<D, G>;
  constexpr int LPR = S::LPR, E = S::E, V16 = S::V16, RPW = S::RPW, U = S::U;
  constexpr int ROWS_PER_PASS = kDecodeWarps * RPW;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int R = a.rows;
  const int r0 = split * a.rows_per_split;
  const int r1 = min(R, r0 + a.rows_per_split);
  const int nrows = max(0, r1 - r0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int li = lane % LPR, rg = lane / LPR;

  extern __shared__ float smem[];
  const int sc_len = max(a.rows_per_split, a.nsplit);
  float* sc = smem;                  // [G][sc_len]: scores, then weights, then merge weights
  float* red = smem + G * sc_len;    // [warps][G][D] per-warp partial sums (fixed-order reduction)
  __shared__ float s_m[G], s_l[G];
  __shared__ int s_last;

  const int cur = a.state->cur_row;
  const bool state_ok = cur >= 0 && cur < R;
  if (!state_ok && split == 0 && tid == 0) atomicCAS(&a.state->error, 0, kErrRowRange);

  const long long slab = (((long long)a.layer * a.batch + b) * a.kv_heads + h) * (long long)R * D;
  uint16_t* Kc = a.k_cache + slab;
  uint16_t* Vc = a.v_cache + slab;
  const uint16_t* kn = a.k_new + ((long long)b * a.kv_heads + h) * D;
  const uint16_t* vn = a.v_new + ((long long)b * a.kv_heads + h) * D;
  const uint8_t* mrow = a.mask + (long long)b * R;

  // append the new row (only the CTA whose range holds it)
  if (state_ok && cur >= r0 && cur < r1) {
    for (int i = tid; i < D / 8; i += kDecodeThreads) {
      reinterpret_cast<uint4*>(Kc + (long long)cur * D)[i] = reinterpret_cast<const uint4*>(kn)[i];
      reinterpret_cast<uint4*>(Vc + (long long)cur * D)[i] = reinterpret_cast<const uint4*>(vn)[i];
    }
  }

  // this lane's slice of the G query vectors, pre-scaled into the exp2 domain
  float qr[G][E];
  {
    const uint16_t* qp = a.q + ((long long)b * a.q_heads + (long long)h * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < V16; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(qp + g * D + (j * LPR + li) * 8);
        float f[8];
        bf16x8_to_f32(v, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qr[g][j * 8 + e] = f[e] * a.scale_log2;
      }
  }

  // ---- pass 1: scores of every row of the range
  for (int p0 = 0; p0 < nrows; p0 += ROWS_PER_PASS * U) {
    uint4 kv[U][V16];
    bool act[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + p0 + u * ROWS_PER_PASS + warp * RPW + rg;
      act[u] = state_ok && r < r1 && mrow[r] != 0;
      if (act[u]) {
        const uint16_t* src = (r == cur) ? kn : Kc + (long long)r * D;
#pragma unroll
        for (int j = 0; j < V16; ++j) kv[u][j] = ld_stream(src + (j * LPR + li) * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float s[G];
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = 0.f;
      if (act[u]) {
#pragma unroll
        for (int j = 0; j < V16; ++j) {
          float f[8];
          bf16x8_to_f32(kv[u][j], f);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[g] = fmaf(qr[g][j * 8 + e], f[e], s[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) s[g] += __shfl_xor_sync(0xffffffffu, s[g], o);
      const int r = r0 + p0 + u * ROWS_PER_PASS + warp * RPW + rg;
      if (li == 0 && r < r1) {
#pragma unroll
        for (int g = 0; g < G; ++g) sc[g * sc_len + (r - r0)] = act[u] ? s[g] : -CUDART_INF_F;
      }
    }
  }
  __syncthreads();

  // ---- softmax statistics of the range (per query head)
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float m = -CUDART_INF_F;
    for (int i = tid; i < nrows; i += kDecodeThreads) m = fmaxf(m, sc[g * sc_len + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (tid == 0) {
      float mm = red[0];
      for (int w = 1; w < kDecodeWarps; ++w) mm = fmaxf(mm, red[w]);
      s_m[g] = mm;
    }
    __syncthreads();
    const float mg = s_m[g];
    float l = 0.f;
    for (int i = tid; i < nrows; i += kDecodeThreads) {
      const float x = sc[g * sc_len + i];
      const float p = (x == -CUDART_INF_F) ? 0.f : exp2f(x - mg);
      sc[g * sc_len + i] = p;
      l += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    __syncthreads();
    if (lane == 0) red[warp] = l;
    __syncthreads();
    if (tid == 0) {
      float ll = 0.f;
      for (int w = 0; w < kDecodeWarps; ++w) ll += red[w];
      s_l[g] = ll;
    }
    __syncthreads();
  }

  // ---- pass 2: weighted sum of the value rows
  float acc[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
  for (int p0 = 0; p0 < nrows; p0 += ROWS_PER_PASS * U) {
    uint4 vv[U][V16];
    bool act[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + p0 + u * ROWS_PER_PASS + warp * RPW + rg;
      act[u] = state_ok && r < r1 && mrow[r] != 0;
      if (act[u]) {
        const uint16_t* src = (r == cur) ? vn : Vc + (long long)r * D;
#pragma unroll
        for (int j = 0; j < V16; ++j) vv[u][j] = ld_stream(src + (j * LPR + li) * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!act[u]) continue;
      const int r = r0 + p0 + u * ROWS_PER_PASS + warp * RPW + rg;
      float p[G];
#pragma unroll
      for (int g = 0; g < G; ++g) p[g] = sc[g * sc_len + (r - r0)];
#pragma unroll
      for (int j = 0; j < V16; ++j) {
        float f[8];
        bf16x8_to_f32(vv[u][j], f);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[g][j * 8 + e] = fmaf(p[g], f[e], acc[g][j * 8 + e]);
      }
    }
  }
  // reduce across the row groups of the warp, then across warps
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
  if (rg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < V16; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) red[(warp * G + g) * D + (j * LPR + li) * 8 + e] = acc[g][j * 8 + e];
  }
  __syncthreads();

  // ---- partial result of this split (warps summed in a fixed order: deterministic)
  const int nsplit = a.nsplit;
  const long long head0 = (long long)b * a.q_heads + (long long)h * G;
  for (int i = tid; i < G * D; i += kDecodeThreads) {
    const int g = i / D, d = i % D;
    float sum = red[i];
#pragma unroll
    for (int w = 1; w < kDecodeWarps; ++w) sum += red[w * G * D + i];
    a.ws_acc[((head0 + g) * nsplit + split) * D + d] = sum;
  }
  if (tid < G) {
    a.ws_ml[((head0 + tid) * nsplit + split) * 2 + 0] = s_m[tid];
    a.ws_ml[((head0 + tid) * nsplit + split) * 2 + 1] = s_l[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(&a.counters[b * a.kv_heads + h], 1);
    s_last = (ticket == nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- combine (last CTA of this sequence and kv head)
  // split statistics are staged in shared memory with independent loads; the
  // accumulator loads are issued eight at a time; the summation order over
  // splits stays fixed (deterministic)
  float* wts = red;                     // [G][nsplit] merge weights
  float* sms = red + G * nsplit;        // [G][nsplit] split maxima
  float* sls = red + 2 * G * nsplit;    // [G][nsplit] split sums
  __shared__ float s_M[G], s_L[G];
  for (int x = tid; x < G * nsplit; x += kDecodeThreads) {
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
  for (int i = tid; i < G * D; i += kDecodeThreads) {
    const int g = i / D, d = i % D;
    const float* src = a.ws_acc + (head0 + g) * nsplit * (long long)D + d;
    const float* w = wts + g * nsplit;
    float o = 0.f;
    int s = 0;
    for (; s + 8 <= nsplit; s += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (long long)(s + u) * D);
#pragma unroll
      for (int u = 0; u < 8; ++u) o = fmaf(w[s + u], v[u], o);
    }
    for (; s < nsplit; ++s) o = fmaf(w[s], __ldcg(src + (long long)s * D), o);
    const float L = s_L[g];
    o = L > 0.f ? o / L : 0.f;
    a.out[(head0 + g) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
  }
  if (tid < G && a.lse) {
    const float L = s_L[tid];
    a.lse[head0 + tid] = L > 0.f ? (s_M[tid] + log2f(L)) * 0.69314718055994530942f : -CUDART_INF_F;
  }
  if (tid == 0) a.counters[b * a.kv_heads + h] = 0;
}

template <int D, int G>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
  const int sc_len = a.rows_per_split > a.nsplit ? a.rows_per_split : a.nsplit;
  const size_t smem = sizeof(float) * (size_t(G) * sc_len + size_t(kDecodeWarps) * G * D);
  auto k = decode_kernel<D, G>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(a.nsplit, a.kv_heads, a.batch);
  k<<<grid, kDecodeThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
  switch (a.q_heads / a.kv_heads) {
    case 1: return launch_t<D, 1>(a, s);
    case 2: return launch_t<D, 2>(a, s);
    case 4: return launch_t<D, 4>(a, s);
    case 8: return launch_t<D, 8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

DecodeSplit decode_split(int batch, int q_heads, int kv_heads, int head_dim, int rows, int sm_count) {
  DecodeSplit d;
  const long long pairs = (long long)batch * kv_heads;
  const long long target = 4LL * (sm_count > 0 ? sm_count : 152);
  long long ns = (target + pairs - 1) / pairs;
  const int min_rows = 32;
  long long max_ns = (rows + min_rows - 1) / min_rows;
  if (max_ns > 64) max_ns = 64;
  if (ns > max_ns) ns = max_ns;
  if (ns < 1) ns = 1;
  d.nsplit = int(ns);
  d.rows_per_split = (rows + d.nsplit - 1) / d.nsplit;
  d.nsplit = (rows + d.rows_per_split - 1) / d.rows_per_split;
  const size_t counters = size_t(pairs) * sizeof(int32_t);
  const size_t ml = size_t(batch) * q_heads * d.nsplit * 2 * sizeof(float);
  const size_t acc = size_t(batch) * q_heads * d.nsplit * head_dim * sizeof(float);
  d.off_ml = align256(counters);
  d.off_acc = d.off_ml + align256(ml);
  d.total = d.off_acc + align256(acc);
  return d;
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
    cached[dev] = p;
  }
  *ptr = cached[dev];
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  switch (a.head_dim) {
    case 64: return launch_d<64>(a, s);
    case 128: return launch_d<128>(a, s);
    case 256: return launch_d<256>(a, s);
    case 512: return launch_d<512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swa
