// Cache movement kernels: state initialisation, the prefill K/V write, the
// compaction at first decode and the 64-row roll.  All are plain 16-byte
// copies (HBM-bound), bit-exact.
//
// Sources: "Enable compact sliding-window attention for Gemma 3 and Gemma 4
// variants", Summary (prompt-sized caches compacted at first decode into
// window + 64 anchored buffers; every 64 decode tokens the rows shift down by
// a fixed offset with device-to-device copies).

#include <mutex>

#include "internal.h"

namespace swa {

int device_sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

__global__ void init_state_kernel(swa_device_state* st, int32_t* vs_dst, const int32_t* vs_src,
                                  int batch, swa_device_state init) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t == 0) *st = init;
  for (int i = t; i < batch; i += blockDim.x * gridDim.x) vs_dst[i] = vs_src ? vs_src[i] : 0;
}

// Chunk K/V [B, C, Hkv, D] -> cache rows [c0, c0 + C) of one layer.
// kAfterReader: a programmatic dependent launch behind a prefill kernel that
// reads the chunk's keys from k / v (not from these cache rows): the copy
// starts at once and waits for that kernel only before exiting.
template <bool kAfterReader>
__global__ void write_rows_kernel(uint4* __restrict__ ck, uint4* __restrict__ cv,
                                  const uint4* __restrict__ k, const uint4* __restrict__ v,
                                  int batch, int chunk_len, int kv_heads, int d8, int rows,
                                  int layer, int c0) {
  if (kAfterReader && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long n = (long long)batch * chunk_len * kv_heads * d8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int dv = int(i % d8);
    long long r = i / d8;
    const int h = int(r % kv_heads);
    r /= kv_heads;
    const int t = int(r % chunk_len);
    const int b = int(r / chunk_len);
    const long long dst =
        ((((long long)layer * batch + b) * kv_heads + h) * rows + c0 + t) * d8 + dv;
    ck[dst] = k[i];
    cv[dst] = v[i];
  }
  if (kAfterReader) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Compact rows [0, W) <- prefill rows [S - W, S) (zero for negative positions).
__global__ void compact_kernel(uint4* __restrict__ dk, uint4* __restrict__ dv,
                               const uint4* __restrict__ sk, const uint4* __restrict__ sv,
                               long long slabs, int src_rows, int dst_rows, int window,
                               int prompt_len, int d8, int ring) {
  const long long n = slabs * window * d8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = int(i % d8);
    const long long rr = i / d8;
    const int r = int(rr % window);
    const long long slab = rr / window;
    const int pos = prompt_len - window + r;
    uint4 a = make_uint4(0, 0, 0, 0), b = a;
    if (pos >= 0) {
      const long long src = (slab * src_rows + pos) * d8 + c;
      a = sk[src];
      b = sv[src];
    }
    const int dr = ring ? ((pos % window) + window) % window : r;  // ring: row pos % W
    const long long dst = (slab * dst_rows + dr) * d8 + c;
    dk[dst] = a;
    dv[dst] = b;
  }
}

// In-place shift of rows [64, R) to rows [0, W) of one slab column strip.
// A block owns a strip of up to 8 16-byte columns of every row of one slab
// (K or V) and walks the rows upwards in passes of 64 rows: each pass loads
// its source rows into registers, synchronises, then stores.  A pass writes
// rows that an earlier pass read (before an earlier barrier) and reads rows
// that only a later pass writes, so the overlapping copy is race-free.
constexpr int kRollThreads = 256;
constexpr int kRollStrip = 8;                                 // 16-byte columns per strip
constexpr int kRollRowsPerLoad = kRollThreads / kRollStrip;   // 32
constexpr int kRollLoads = SWA_ROLL_ROWS / kRollRowsPerLoad;  // 2 -> 64 rows per pass

__global__ void __launch_bounds__(kRollThreads)
roll_kernel(uint4* __restrict__ k, uint4* __restrict__ v, long long slabs, int rows, int window,
            int d8, swa_device_state* st) {
  const long long sid = blockIdx.x;  // [0, 2 * slabs): K slabs then V slabs
  const int strip = blockIdx.y;
  uint4* base = sid < slabs ? k + sid * rows * (long long)d8 : v + (sid - slabs) * rows * (long long)d8;
  const int col = strip * kRollStrip + (threadIdx.x % kRollStrip);
  const int rsub = threadIdx.x / kRollStrip;
  const bool col_ok = col < d8;
  for (int p0 = 0; p0 < window; p0 += SWA_ROLL_ROWS) {
    uint4 buf[kRollLoads];
#pragma unroll
    for (int j = 0; j < kRollLoads; ++j) {
      const int dst = p0 + j * kRollRowsPerLoad + rsub;
      if (col_ok && dst < window) buf[j] = base[(long long)(dst + SWA_ROLL_ROWS) * d8 + col];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRollLoads; ++j) {
      const int dst = p0 + j * kRollRowsPerLoad + rsub;
      if (col_ok && dst < window) base[(long long)dst * d8 + col] = buf[j];
    }
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    st->origin += SWA_ROLL_ROWS;
    st->next_row = window;
  }
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  const long long cap = 64LL * device_sm_count();  // grid-stride loops: 64 CTAs per SM at most
  if (g > cap) g = cap;
  return g < 1 ? 1 : int(g);
}

}  // namespace

cudaError_t launch_init_state(swa_device_state* st, int32_t* vs_dst, const int32_t* vs_src,
                              int batch, swa_device_state init, cudaStream_t s) {
  const int threads = 256;
  init_state_kernel<<<(batch + threads - 1) / threads + 1, threads, 0, s>>>(st, vs_dst, vs_src, batch, init);
  return cudaGetLastError();
}

cudaError_t launch_write_rows(uint16_t* cache_k, uint16_t* cache_v, const uint16_t* k,
                              const uint16_t* v, int batch, int chunk_len, int kv_heads,
                              int head_dim, int rows, int layer, int chunk_start, bool after_reader,
                              cudaStream_t s) {
  const int d8 = head_dim / 8;
  const long long n = (long long)batch * chunk_len * kv_heads * d8;
  if (n == 0) return cudaSuccess;
  uint4* ck = reinterpret_cast<uint4*>(cache_k);
  uint4* cv = reinterpret_cast<uint4*>(cache_v);
  const uint4* k4 = reinterpret_cast<const uint4*>(k);
  const uint4* v4 = reinterpret_cast<const uint4*>(v);
  if (!after_reader) {
    write_rows_kernel<false><<<grid_for(n, 256), 256, 0, s>>>(ck, cv, k4, v4, batch, chunk_len, kv_heads, d8, rows,
                                                              layer, chunk_start);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(n, 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, write_rows_kernel<true>, ck, cv, k4, v4, batch, chunk_len, kv_heads, d8, rows,
                            layer, chunk_start);
}

cudaError_t launch_compact(uint16_t* dk, uint16_t* dv, const uint16_t* sk, const uint16_t* sv,
                           long long slabs, int src_rows, int dst_rows, int window,
                           int prompt_len, int head_dim, bool ring, cudaStream_t s) {
  const int d8 = head_dim / 8;
  const long long n = slabs * window * d8;
  if (n == 0) return cudaSuccess;
  compact_kernel<<<grid_for(n, 256), 256, 0, s>>>(
      reinterpret_cast<uint4*>(dk), reinterpret_cast<uint4*>(dv),
      reinterpret_cast<const uint4*>(sk), reinterpret_cast<const uint4*>(sv), slabs, src_rows,
      dst_rows, window, prompt_len, d8, ring ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_roll(uint16_t* k, uint16_t* v, long long slabs, int rows, int window,
                        int head_dim, swa_device_state* st, cudaStream_t s) {
  const int d8 = head_dim / 8;
  dim3 grid((unsigned)(2 * slabs), (d8 + kRollStrip - 1) / kRollStrip);
  roll_kernel<<<grid, kRollThreads, 0, s>>>(reinterpret_cast<uint4*>(k), reinterpret_cast<uint4*>(v),
                                            slabs, rows, window, d8, st);
  return cudaGetLastError();
}

}  // namespace swa
