// Prefill attention on CUDA cores for head size 512: one warp per (sequence,
// query row, query head), online softmax over the row's key interval.  The
// head-size-256 path runs on the tensor cores (prefill_sm103.cu).
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary and Compilation behavior (narrow causal plan and generic
// plan); "Add SDPA attention implementation", Summary (packed documents).

#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"

namespace swa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) prefill_simt_kernel(const PrefillArgs a) {
  constexpr int E = D / 32;  // elements per lane
  const long long gw = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long total = (long long)a.batch * a.chunk_len * a.q_heads;
  if (gw >= total) return;
  const int hq = int(gw % a.q_heads);
  const int i = int((gw / a.q_heads) % a.chunk_len);
  const int b = int(gw / ((long long)a.q_heads * a.chunk_len));
  const int q = a.chunk_start + i;
  const int hk = hq / (a.q_heads / a.kv_heads);

  int lo, hi;
  if (a.generic) {
    const char* plan = static_cast<const char*>(a.plan);
    const PlanLayout L = plan_layout(a.batch, a.chunk_len);
    lo = reinterpret_cast<const int32_t*>(plan + L.off_lo)[(long long)b * a.chunk_len + i];
    hi = reinterpret_cast<const int32_t*>(plan + L.off_hi)[(long long)b * a.chunk_len + i];
  } else {
    causal_interval(q, a.valid_start ? a.valid_start[b] : 0, a.window, lo, hi);
  }
  if (hi > a.key_rows - 1) hi = a.key_rows - 1;
  if (lo < 0) lo = 0;

  const long long qoff = (((long long)b * a.chunk_len + i) * a.q_heads + hq) * D;
  float qv[E];
#pragma unroll
  for (int e = 0; e < E; ++e)
    qv[e] = __bfloat162float(__ushort_as_bfloat16(a.q[qoff + lane * E + e])) * a.scale_log2;

  const uint16_t* kb = a.k + b * a.key_seq_stride + hk * a.key_head_stride;
  const uint16_t* vb = a.v + b * a.key_seq_stride + hk * a.key_head_stride;
  float m = -CUDART_INF_F, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int k = lo; k <= hi; ++k) {
    const uint16_t* kr = kb + k * a.key_row_stride + lane * E;
    const uint16_t* vr = vb + k * a.key_row_stride + lane * E;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) s = fmaf(qv[e], __bfloat162float(__ushort_as_bfloat16(kr[e])), s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmaxf(m, s);
    const float corr = exp2f(m - mn);  // m = -inf on the first key -> 0
    const float p = exp2f(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < E; ++e)
      acc[e] = fmaf(p, __bfloat162float(__ushort_as_bfloat16(vr[e])), acc[e] * corr);
    m = mn;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float o = l > 0.f ? acc[e] / l : 0.f;
    a.out[qoff + lane * E + e] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
  }
  if (a.lse && lane == 0) {
    a.lse[((long long)b * a.chunk_len + i) * a.q_heads + hq] =
        l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
  }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t s) {
  const long long warps = (long long)a.batch * a.chunk_len * a.q_heads;
  const long long blocks = (warps * 32 + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  switch (a.head_dim) {
    case 256: prefill_simt_kernel<256><<<unsigned(blocks), 256, 0, s>>>(a); break;
    case 512: prefill_simt_kernel<512><<<unsigned(blocks), 256, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace swa
