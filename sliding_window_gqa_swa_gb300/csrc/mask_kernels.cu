// Runtime-mask builders: the per-step decode mask, the prefill plan (one key
// interval per query row plus per-tile key ranges) and a dense expansion of
// the plan for tests.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary (one fixed-shape runtime mask shared by all sliding
// layers; a key counts when it lies in the window and is causal or in the
// query's image block) and Compilation behavior (positions, rows not yet
// written, where the window sits, padding and image regions are device data,
// not constants of the compiled program); "Add SDPA attention implementation", Summary
// (document boundaries from cu_seqlens).

#include "internal.h"

namespace swa {
namespace {

constexpr int kMaskThreads = 512;

// Position held by row r: anchored (origin + r), or in a ring of `rows` rows
// the latest position congruent to r that is <= p ("Gemma3 Local Attention
// Cache", Steps 2-3: positions assigned with % and wrapping around).
__device__ __forceinline__ int row_position(int r, int origin, int p, int rows, bool ring) {
  return ring ? p - (((p - r) % rows) + rows) % rows : origin + r;
}

// Decode mask of the step about to run (one block).  Every thread reads the
// state first; thread 0 advances it after a barrier.
__global__ void __launch_bounds__(kMaskThreads)
decode_mask_kernel(swa_device_state* st, const int32_t* __restrict__ vs, int batch, int rows, int ring,
                   uint8_t* __restrict__ mask) {
  const int origin = st->origin;
  const int cur = st->next_row;
  const int p = st->prompt_len + st->step;
  const int window = st->window;
  // a ring writes position p to row p % rows; an anchored cache never past its end
  const bool ok = cur >= 0 && cur < rows && (!ring || cur == p % rows);
  const long long n = (long long)batch * rows;
  if ((rows & 15) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15) == 0) {
    // 16 rows per thread-iteration, written as one 16-byte store
    const long long nv = n / 16;
    for (long long i = threadIdx.x; i < nv; i += blockDim.x) {
      const int b = int((i * 16) / rows);
      const int r0 = int((i * 16) % rows);
      const int v = vs[b];
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t x = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = r0 + j * 4 + e;
          const int pos = row_position(r, origin, p, rows, ring);
          const bool m = ok && (ring || r <= cur) && pos > p - window && pos >= v && pos >= 0;
          x |= uint32_t(m) << (8 * e);
        }
        w[j] = x;
      }
      reinterpret_cast<uint4*>(mask)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (long long i = threadIdx.x; i < n; i += blockDim.x) {
      const int b = int(i / rows);
      const int r = int(i % rows);
      const int pos = row_position(r, origin, p, rows, ring);
      mask[i] = uint8_t(ok && (ring || r <= cur) && pos > p - window && pos >= vs[b] && pos >= 0);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (ok) {
      st->cur_row = cur;
      st->next_row = (ring && cur + 1 == rows) ? 0 : cur + 1;
      st->step = st->step + 1;
    } else {
      atomicCAS(&st->error, 0, ring ? kErrRowRange : kErrRollDue);
    }
  }
}

constexpr int kPlanThreads = 1024;
constexpr int kInf = 0x7fffffff;

__device__ __forceinline__ int warp_min(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = min(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ int warp_max(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// One block per sequence.  Query rows are walked from the chunk end towards
// its start in tiles of 1024 (aligned to 128-row query tiles) so that the end
// of every image run is found with a block-wide suffix minimum over "run
// start" positions.
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(swa_prefill_meta meta, char* plan) {
  const int b = blockIdx.x;
  const int C = meta.chunk_len;
  const int c0 = meta.chunk_start;
  const int W = meta.window;
  const PlanLayout L = plan_layout(meta.batch, C);
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(plan);
  int32_t* row_lo = reinterpret_cast<int32_t*>(plan + L.off_lo) + (long long)b * C;
  int32_t* row_hi = reinterpret_cast<int32_t*>(plan + L.off_hi) + (long long)b * C;
  const int nqt = (C + kPlanBM - 1) / kPlanBM;
  int32_t* tlo = reinterpret_cast<int32_t*>(plan + L.off_tlo) + (long long)b * nqt;
  int32_t* thi = reinterpret_cast<int32_t*>(plan + L.off_thi) + (long long)b * nqt;
  const int32_t* img = meta.img_id ? meta.img_id + (long long)b * meta.seq_len : nullptr;
  const int vs = meta.valid_start ? meta.valid_start[b] : 0;

  __shared__ int s_suffix[kPlanThreads];
  __shared__ int s_wmin[32], s_wmax[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // The host zero-fills the header (error word included) before the launch.
  if (b == 0 && tid == 0) {
    hdr->magic = kPlanMagic;
    hdr->batch = meta.batch;
    hdr->chunk_start = c0;
    hdr->chunk_len = C;
    hdr->seq_len = meta.seq_len;
    hdr->window = W;
    hdr->n_qtiles = nqt;
  }
  if (img && tid == 0) {
    const int e = c0 + C;
    if (e < meta.seq_len && img[e - 1] >= 0 && img[e] == img[e - 1])
      atomicCAS(&hdr->error, 0, kErrImageCrossesChunk);
  }

  int carry = c0 + C;  // smallest run start seen above the current tile
  const int last_tile = ((C - 1) / kPlanThreads) * kPlanThreads;
  for (int base = last_tile; base >= 0; base -= kPlanThreads) {
    const int i = base + tid;
    const int q = c0 + i;
    int lo = 0, hi = -1;
    if (img) {
      // run start marker: position q (> c0) where the id changes
      int mark = kInf;
      if (i > 0 && i < C && img[q] != img[q - 1]) mark = q;
      // inclusive suffix minimum within the warp
      int x = mark;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x = min(x, y);
      }
      if (lane == 0) s_wmin[warp] = x;
      __syncthreads();
      if (warp == 0) {
        int z = s_wmin[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, z, o);
          if (lane + o < 32) z = min(z, y);
        }
        s_wmin[lane] = z;  // suffix minimum over warps >= lane
      }
      __syncthreads();
      const int after = warp + 1 < 32 ? s_wmin[warp + 1] : kInf;
      s_suffix[tid] = min(x, after);
      __syncthreads();
      const int next = min(tid + 1 < kPlanThreads ? s_suffix[tid + 1] : kInf, carry);
      if (i < C) {
        causal_interval(q, vs, W, lo, hi);
        if (hi >= lo && img[q] >= 0) hi = max(q, next - 1);
      }
      const int tile_min = s_suffix[0];
      __syncthreads();
      carry = min(carry, tile_min);
    } else if (i < C) {
      if (meta.cu_seqlens) {
        // document of q: the last d with cu[d] <= q
        int a = 0, z = meta.num_docs;  // cu[a] <= q < cu[z]
        if (q < meta.cu_seqlens[0] || q >= meta.cu_seqlens[z]) {
          atomicCAS(&hdr->error, 0, kErrBadDocs);
        } else {
          while (z - a > 1) {
            const int m = (a + z) >> 1;
            if (meta.cu_seqlens[m] <= q) a = m; else z = m;
          }
          causal_interval(q, meta.cu_seqlens[a], W, lo, hi);
        }
      } else {
        causal_interval(q, vs, W, lo, hi);
      }
    }
    if (i < C) {
      row_lo[i] = lo;
      row_hi[i] = hi;
    }
    // per 128-row query tile: [min lo, max hi + 1) over non-empty rows
    const bool nonempty = i < C && hi >= lo;
    const int wlo = warp_min(nonempty ? lo : kInf);
    const int whi = warp_max(nonempty ? hi + 1 : -1);
    if (lane == 0) {
      s_wmin[warp] = wlo;
      s_wmax[warp] = whi;
    }
    __syncthreads();
    if (tid < kPlanThreads / kPlanBM) {
      const int t = (base / kPlanBM) + tid;
      if (t < nqt) {
        int mn = kInf, mx = -1;
        for (int w = 0; w < kPlanBM / 32; ++w) {
          mn = min(mn, s_wmin[tid * (kPlanBM / 32) + w]);
          mx = max(mx, s_wmax[tid * (kPlanBM / 32) + w]);
        }
        tlo[t] = mx < 0 ? 0 : mn;
        thi[t] = mx < 0 ? 0 : mx;
      }
    }
    __syncthreads();
  }
}

// Dense [B, C, seq_len] expansion of the key intervals the prefill kernel uses.
__global__ void dense_debug_kernel(swa_prefill_meta meta, uint8_t* __restrict__ out) {
  const long long n = (long long)meta.batch * meta.chunk_len * meta.seq_len;
  const PlanLayout L = plan_layout(meta.batch, meta.chunk_len);
  const char* plan = static_cast<const char*>(meta.plan);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int k = int(i % meta.seq_len);
    const long long rowi = i / meta.seq_len;  // b * C + row
    const int b = int(rowi / meta.chunk_len);
    const int q = meta.chunk_start + int(rowi % meta.chunk_len);
    int lo, hi;
    if (plan) {
      lo = reinterpret_cast<const int32_t*>(plan + L.off_lo)[rowi];
      hi = reinterpret_cast<const int32_t*>(plan + L.off_hi)[rowi];
    } else {
      causal_interval(q, meta.valid_start ? meta.valid_start[b] : 0, meta.window, lo, hi);
    }
    out[i] = uint8_t(k >= lo && k <= hi);
  }
}

}  // namespace

cudaError_t launch_decode_mask(swa_device_state* st, const int32_t* vs, int batch, int rows, bool ring,
                               uint8_t* mask, cudaStream_t s) {
  decode_mask_kernel<<<1, kMaskThreads, 0, s>>>(st, vs, batch, rows, ring ? 1 : 0, mask);
  return cudaGetLastError();
}

cudaError_t launch_prefill_plan(const swa_prefill_meta& meta, void* plan, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(plan, 0, sizeof(PlanHeader), s);
  if (e != cudaSuccess) return e;
  plan_kernel<<<meta.batch, kPlanThreads, 0, s>>>(meta, static_cast<char*>(plan));
  return cudaGetLastError();
}

cudaError_t launch_dense_debug(const swa_prefill_meta& meta, uint8_t* out, cudaStream_t s) {
  const long long n = (long long)meta.batch * meta.chunk_len * meta.seq_len;
  long long g = (n + 255) / 256;
  if (g > 32LL * device_sm_count()) g = 32LL * device_sm_count();
  if (g < 1) g = 1;
  dense_debug_kernel<<<int(g), 256, 0, s>>>(meta, out);
  return cudaGetLastError();
}

}  // namespace swa
