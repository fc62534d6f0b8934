// Internal declarations shared by the CUDA translation units of libswa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "swa.h"

namespace swa {

// Device-side error codes recorded in swa_device_state::error / the plan header.
enum DevError : int32_t {
  kErrNone = 0,
  kErrRowRange = 1,          // decode saw cur_row outside [0, rows)
  kErrRollDue = 2,           // decode mask built while next_row == rows
  kErrImageCrossesChunk = 3, // an image block runs past the chunk end
  kErrBadDocs = 4,           // cu_seqlens does not cover the query rows
  kErrTimeout = 5,           // a bounded wait inside a kernel gave up
  kErrBand = 6,              // a query tile's key tiles exceed the backward workspace band
};

// Query rows per prefill tile; the plan's per-tile key ranges use it.
constexpr int kPlanBM = 128;
constexpr int32_t kPlanMagic = 0x53574150;

struct PlanHeader {
  int32_t magic;
  int32_t batch;
  int32_t chunk_start;
  int32_t chunk_len;
  int32_t seq_len;
  int32_t window;
  int32_t n_qtiles;
  int32_t error;
};

// Plan buffer: header (256 B) | row_lo [B*C] | row_hi [B*C] | tile_klo [B*T] | tile_khi [B*T]
// (T = ceil(C / kPlanBM)); each array starts on a 256-byte boundary.
struct PlanLayout {
  size_t off_lo, off_hi, off_tlo, off_thi, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline PlanLayout plan_layout(int batch, int chunk_len) {
  PlanLayout p;
  size_t rows = size_t(batch) * size_t(chunk_len) * sizeof(int32_t);
  size_t tiles = size_t(batch) * size_t((chunk_len + kPlanBM - 1) / kPlanBM) * sizeof(int32_t);
  p.off_lo = 256;
  p.off_hi = p.off_lo + align256(rows);
  p.off_tlo = p.off_hi + align256(rows);
  p.off_thi = p.off_tlo + align256(tiles);
  p.total = p.off_thi + align256(tiles);
  return p;
}

// Keys a query at position q attends in the narrow causal plan: the interval
// [lo, hi] (empty when hi < lo).  Pad queries attend nothing.
__host__ __device__ inline void causal_interval(int q, int vs, int window, int& lo, int& hi) {
  if (q < vs) {
    lo = 0;
    hi = -1;
    return;
  }
  int a = q - window + 1;
  lo = a > vs ? a : vs;
  if (lo < 0) lo = 0;
  hi = q;
}

// ---------------------------------------------------------------- launches
// Each returns the launch's cudaError_t (cudaGetLastError after the launch).

cudaError_t launch_init_state(swa_device_state* st, int32_t* vs_dst, const int32_t* vs_src,
                              int batch, swa_device_state init, cudaStream_t s);

// after_reader: launched right after a prefill kernel that reads the chunk's
// keys from its inputs, as a programmatic dependent launch: the copy may run
// on SMs that kernel leaves idle, and the kernel does not complete before the
// prefill kernel has (so later work on the stream stays ordered after both).
cudaError_t launch_write_rows(uint16_t* cache_k, uint16_t* cache_v, const uint16_t* k,
                              const uint16_t* v, int batch, int chunk_len, int kv_heads,
                              int head_dim, int rows, int layer, int chunk_start, bool after_reader,
                              cudaStream_t s);

// ring: position pos goes to row pos % window instead of row pos - (S - W)
cudaError_t launch_compact(uint16_t* dk, uint16_t* dv, const uint16_t* sk, const uint16_t* sv,
                           long long slabs, int src_rows, int dst_rows, int window,
                           int prompt_len, int head_dim, bool ring, cudaStream_t s);

cudaError_t launch_roll(uint16_t* k, uint16_t* v, long long slabs, int rows, int window,
                        int head_dim, swa_device_state* st, cudaStream_t s);

cudaError_t launch_decode_mask(swa_device_state* st, const int32_t* vs, int batch, int rows, bool ring,
                               uint8_t* mask, cudaStream_t s);

cudaError_t launch_prefill_plan(const swa_prefill_meta& meta, void* plan, cudaStream_t s);

cudaError_t launch_dense_debug(const swa_prefill_meta& meta, uint8_t* out, cudaStream_t s);

struct DecodeArgs {
  const uint16_t* q;      // [B, Hq, D]
  const uint16_t* k_new;  // [B, Hkv, D]
  const uint16_t* v_new;
  const uint8_t* mask;    // [B, R]
  uint16_t* k_cache;      // layer 0 base, [L, B, Hkv, R, D]
  uint16_t* v_cache;
  swa_device_state* state;
  uint16_t* out;          // [B, Hq, D]
  float* lse;             // [B, Hq] or null
  int32_t* counters;      // [B * Hkv]
  float* ws_ml;           // [B, Hq, nsplit, 2]
  float* ws_acc;          // [B, Hq, nsplit, D]
  int batch, q_heads, kv_heads, head_dim, rows, layer;
  int nsplit, rows_per_split;
  int cluster;            // 1: the splits of a slab form one cluster and merge in shared memory
  int warps;              // compute warps per CTA: 8 (throughput) or 16 (latency)
  float scale_log2;       // scale * log2(e)
  const int32_t* valid_start;  // [B] left-pad counts (the cache's copy)
  int window;
  int ring;               // 1: modular ring cache (rows hold positions p - ((p - r) mod W))
  int inputs_ready;       // 1: q, k_new, v_new, the mask and the state may be read before the launch wait
};

// SMs of the current device (cached per device; 152 if the query fails).
int device_sm_count();

// Split choice and workspace size shared by the host API and the launcher.
struct DecodeSplit {
  int nsplit, rows_per_split, cluster, warps;
  size_t off_ml, off_acc, total;
};
DecodeSplit decode_split(int batch, int q_heads, int kv_heads, int head_dim, int rows, int sm_count,
                         int max_cluster);
// Largest decode cluster the current device co-schedules (16 or 8).
int decode_max_cluster();

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// Latency-regime decode (few slabs, one cluster per slab, at most 128 rows per
// CTA, Hq / Hkv <= 2, head size 128-512): warp-level tensor-core products and
// no merge between warps.  launch_decode uses it whenever eligible.
bool decode_small_eligible(const DecodeArgs& a);
cudaError_t launch_decode_small(const DecodeArgs& a, cudaStream_t s);

// Device address, on the current device, of the static scratch array that
// swa_decode_noalloc uses (SWA_DECODE_STATIC_SCRATCH_BYTES); looked up once
// per device.
cudaError_t decode_static_scratch(void** ptr);

struct PrefillArgs {
  const uint16_t* q;        // [B, C, Hq, D] (packed: [T, Hq, D], B = 1)
  const uint16_t* k;        // key base: cache layer base or packed keys
  const uint16_t* v;
  uint16_t* out;
  float* lse;
  const int32_t* valid_start;  // causal mode
  const void* plan;            // generic mode
  int batch, chunk_start, chunk_len, q_heads, kv_heads, head_dim, window;
  long long key_seq_stride;    // elements between sequences' key bases
  long long key_head_stride;   // elements between kv heads
  long long key_row_stride;    // elements between key rows
  int key_rows;                // keys a row may attend lie below this bound
  int key_dim_rows;            // rows of the key tensor per (sequence, head): Rp or T
  int generic;
  float scale_log2;
  int32_t* err;                // device error word (cache state or plan header)
  // The chunk's own K/V [B, C, Hkv, D] when the kernel reads keys
  // [chunk_start, chunk_start + C) from them instead of the cache (which the
  // K/V write then fills concurrently); null: every key comes from k / v.
  const uint16_t* k_in;
  const uint16_t* v_in;
};

// Tensor-core (tcgen05) prefill.  Head size 256: the two query heads of a
// KV head share a CTA pair on 128-key tiles when the group size is even
// (launch_prefill_pair256), else one CTA per head on 128-key tiles
// (launch_prefill_t128).  Head size 512: four-CTA clusters on 128-key tiles
// for an even group (launch_prefill_split512), else column pairs on 64-key
// tiles.
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_prefill_t128(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_prefill_pair256(const PrefillArgs& a, cudaStream_t s);
// True when launch_prefill_tc runs the pair kernel for these arguments and it
// can read the chunk's keys from k_in / v_in (the chunk starts on a key tile).
bool prefill_reads_chunk_inputs(const PrefillArgs& a);

// Head size 512, even GQA group: a four-CTA cluster per (head pair, query
// tile), one CTA pair computing S and the softmax, the other accumulating O.
cudaError_t launch_prefill_split512(const PrefillArgs& a, cudaStream_t s);
bool prefill_split512_eligible(const PrefillArgs& a);

// 4-D bf16 tensor map with a {64, box_rows, 1, 1} box and 128-byte swizzle
// (dims innermost first, strides in bytes of dims 1..3); false on failure.
bool make_tmap_bf16(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                    uint32_t box_rows);

// ---------------------------------------------------------------- backward
// Score tiles of the backward pass are 128 queries x 128 keys (the plan's
// query tile); each is stored as the 128-byte-swizzled image of two
// {64 columns, 128 rows} boxes (32 KB).
constexpr int kBwdTile = 128;
constexpr size_t kBwdTileBytes = size_t(kBwdTile) * kBwdTile * 2;

struct BackwardLayout {
  int n_tiles;       // query (= key) tiles per sequence: ceil(S / 128)
  int band;          // key tiles reserved per query tile
  size_t off_delta;  // [B, S, Hq] fp32: rowsum(dout * out)
  size_t off_ds;     // dS tiles   [B, Hq, n_tiles, band] (rows: queries, columns: keys)
  size_t off_pt;     // P^T tiles  (rows: keys, columns: queries)
  size_t off_dst;    // dS^T tiles
  size_t total;
};
// band = n_tiles when image blocks are present (future keys up to the block
// end), else the most 128-key tiles a 128-row query tile can span under a
// window of `window` keys: 1 + ceil((window - 1) / 128), capped at n_tiles.
BackwardLayout backward_layout(int batch, int seq_len, int q_heads, int window, bool images);

struct BackwardArgs {
  const uint16_t* q;     // [B, S, Hq, D]
  const uint16_t* k;     // [B, S, Hkv, D]
  const uint16_t* v;
  const uint16_t* out;   // forward output [B, S, Hq, D]
  const uint16_t* dout;  // upstream gradient of out
  const float* lse;      // forward lse [B, S, Hq]
  uint16_t* dq;          // [B, S, Hq, D]
  uint16_t* dk;          // [B, S, Hkv, D]
  uint16_t* dv;
  const void* plan;      // prefill plan of the whole sequences
  float* delta;          // workspace parts (BackwardLayout)
  char* t_ds;
  char* t_pt;
  char* t_dst;
  int batch, seq_len, q_heads, kv_heads, head_dim, band;
  float scale;
  int32_t* err;          // plan header error word
};

// Three launches on `s`: delta, scores (P and dS tiles), gradients (dQ, dK, dV).
cudaError_t launch_prefill_backward(const BackwardArgs& a, cudaStream_t s);

}  // namespace swa
