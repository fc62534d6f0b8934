// The C ABI of libswa: argument validation, the host mirror of the cache
// index map, and kernel launches.  Every argument is checked before the first
// CUDA call of an entry point, so a rejected call touches no device memory.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "internal.h"
#include "swa.h"

struct swa_cache {
  swa_cache_desc desc;  // rows resolved
  char* base;
  swa_device_state* state;
  int32_t* valid_start;
  uint16_t* k;
  uint16_t* v;
  size_t kv_bytes;
  // host mirror of the device index map
  int32_t origin, next_row, cur_row, step;
};

namespace {

thread_local std::string g_error;

swa_status fail(swa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return st;
}

swa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SWA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct Layout {
  size_t off_vs, off_k, off_v, kv_bytes, total;
};

// Validate a desc and resolve rows; returns false with g_error set.
// Caches that decode: the anchored compact buffer and the modular ring.
bool decodes(int32_t kind) { return kind == SWA_CACHE_COMPACT || kind == SWA_CACHE_RING; }

bool resolve_desc(const swa_cache_desc* in, swa_cache_desc* out) {
  if (!in) {
    fail(SWA_EINVAL, "desc is NULL");
    return false;
  }
  swa_cache_desc d = *in;
  if (d.kind != SWA_CACHE_PREFILL && d.kind != SWA_CACHE_COMPACT && d.kind != SWA_CACHE_RING) {
    fail(SWA_EINVAL, "desc.kind must be SWA_CACHE_PREFILL, SWA_CACHE_COMPACT or SWA_CACHE_RING");
    return false;
  }
  if (d.layers < 1 || d.batch < 1 || d.kv_heads < 1) {
    fail(SWA_EINVAL, "layers, batch and kv_heads must be >= 1");
    return false;
  }
  if (d.head_dim < 64 || d.head_dim > 512 || (d.head_dim & 63)) {
    fail(SWA_EINVAL, "head_dim must be a multiple of 64 in [64, 512]");
    return false;
  }
  if (d.window < 1 || d.prompt_len < 0) {
    fail(SWA_EINVAL, "window must be >= 1 and prompt_len >= 0");
    return false;
  }
  if (d.kind == SWA_CACHE_COMPACT) {
    if (d.window < SWA_ROLL_ROWS) {
      fail(SWA_EINVAL, "a compact cache needs window >= %d", SWA_ROLL_ROWS);
      return false;
    }
    const int32_t want = d.window + SWA_ROLL_ROWS;
    if (d.rows != 0 && d.rows != want) {
      fail(SWA_EINVAL, "a compact cache has exactly window + %d rows", SWA_ROLL_ROWS);
      return false;
    }
    d.rows = want;
  } else if (d.kind == SWA_CACHE_RING) {
    if (d.rows != 0 && d.rows != d.window) {
      fail(SWA_EINVAL, "a ring cache has exactly window rows");
      return false;
    }
    d.rows = d.window;
  } else {
    const int64_t minr = std::max<int64_t>(d.prompt_len, int64_t(d.window) + SWA_ROLL_ROWS);
    if (d.rows == 0) d.rows = int32_t(std::min<int64_t>(minr, INT32_MAX));
    if (d.rows < d.prompt_len) {
      fail(SWA_EINVAL, "prefill cache rows (%d) < prompt_len (%d)", d.rows, d.prompt_len);
      return false;
    }
  }
  *out = d;
  return true;
}

Layout layout_of(const swa_cache_desc& d) {
  Layout l;
  l.off_vs = 64;
  l.kv_bytes = size_t(d.layers) * d.batch * d.kv_heads * size_t(d.rows) * d.head_dim * 2;
  l.off_k = swa::align256(l.off_vs + size_t(d.batch) * 4);
  l.off_v = l.off_k + swa::align256(l.kv_bytes);
  l.total = l.off_v + swa::align256(l.kv_bytes);
  return l;
}

bool check_meta(const swa_prefill_meta* m) {
  if (!m) {
    fail(SWA_EINVAL, "meta is NULL");
    return false;
  }
  if (m->batch < 1 || m->seq_len < 1 || m->window < 1) {
    fail(SWA_EINVAL, "meta: batch, seq_len and window must be >= 1");
    return false;
  }
  if (m->chunk_len < 1 || m->chunk_start < 0 || int64_t(m->chunk_start) + m->chunk_len > m->seq_len) {
    fail(SWA_EINVAL, "meta: chunk [%d, %d) outside [0, %d)", m->chunk_start,
         m->chunk_start + m->chunk_len, m->seq_len);
    return false;
  }
  if (m->cu_seqlens) {
    if (m->valid_start || m->img_id) {
      fail(SWA_EUNSUPPORTED, "meta: packed documents take neither valid_start nor img_id");
      return false;
    }
    if (m->batch != 1 || m->num_docs < 1 || m->chunk_start != 0 || m->chunk_len != m->seq_len) {
      fail(SWA_EINVAL, "meta: packed documents need batch 1, num_docs >= 1 and the whole range");
      return false;
    }
  }
  if ((m->valid_start && !aligned16(m->valid_start)) || (m->img_id && !aligned16(m->img_id)) ||
      (m->cu_seqlens && !aligned16(m->cu_seqlens)) || (m->plan && !aligned16(m->plan))) {
    fail(SWA_EINVAL, "meta: device pointers must be 16-byte aligned");
    return false;
  }
  return true;
}

// Meta accepted by the backward pass: whole sequences and a plan.  Returns
// SWA_OK or the failing status (g_error set).
swa_status check_backward_meta(const swa_prefill_meta* meta) {
  if (!check_meta(meta)) return SWA_EINVAL;
  if (meta->chunk_start != 0 || meta->chunk_len != meta->seq_len)
    return fail(SWA_EUNSUPPORTED, "backward covers whole sequences (chunk_start 0, chunk_len = seq_len)");
  if (!meta->plan) return fail(SWA_EINVAL, "backward needs meta->plan (swa_build_mask(SWA_MASK_PREFILL))");
  return SWA_OK;
}

}  // namespace

extern "C" {

int32_t swa_version(void) { return 100; }

const char* swa_last_error(void) { return g_error.c_str(); }

const char* swa_status_string(swa_status s) {
  switch (s) {
    case SWA_OK: return "SWA_OK";
    case SWA_EINVAL: return "SWA_EINVAL";
    case SWA_ESTATE: return "SWA_ESTATE";
    case SWA_EUNSUPPORTED: return "SWA_EUNSUPPORTED";
    case SWA_ECUDA: return "SWA_ECUDA";
    case SWA_ETIMEOUT: return "SWA_ETIMEOUT";
    case SWA_EDEVICE: return "SWA_EDEVICE";
  }
  return "SWA_UNKNOWN";
}

size_t swa_cache_bytes(const swa_cache_desc* desc) {
  swa_cache_desc d;
  if (!resolve_desc(desc, &d)) return 0;
  return layout_of(d).total;
}

swa_status swa_cache_alloc(const swa_cache_desc* desc, void* dev_mem, size_t bytes,
                           const int32_t* dev_valid_start, swa_stream_t stream, swa_cache** out) {
  if (!out) return fail(SWA_EINVAL, "out is NULL");
  *out = nullptr;
  swa_cache_desc d;
  if (!resolve_desc(desc, &d)) return SWA_EINVAL;
  if (!dev_mem) return fail(SWA_EINVAL, "dev_mem is NULL");
  if (reinterpret_cast<uintptr_t>(dev_mem) & 255) return fail(SWA_EINVAL, "dev_mem must be 256-byte aligned");
  const Layout l = layout_of(d);
  if (bytes < l.total) return fail(SWA_EINVAL, "bytes (%zu) < swa_cache_bytes (%zu)", bytes, l.total);
  if (dev_valid_start && (reinterpret_cast<uintptr_t>(dev_valid_start) & 3))
    return fail(SWA_EINVAL, "dev_valid_start must be 4-byte aligned");

  swa_cache* c = new (std::nothrow) swa_cache;
  if (!c) return fail(SWA_EINVAL, "out of host memory");
  c->desc = d;
  c->base = static_cast<char*>(dev_mem);
  c->state = reinterpret_cast<swa_device_state*>(c->base);
  c->valid_start = reinterpret_cast<int32_t*>(c->base + l.off_vs);
  c->k = reinterpret_cast<uint16_t*>(c->base + l.off_k);
  c->v = reinterpret_cast<uint16_t*>(c->base + l.off_v);
  c->kv_bytes = l.kv_bytes;
  swa_device_state init;
  if (d.kind == SWA_CACHE_COMPACT) {
    init.origin = d.prompt_len - d.window;
    init.next_row = d.window;
  } else if (d.kind == SWA_CACHE_RING) {
    init.origin = 0;
    init.next_row = d.prompt_len % d.window;
  } else {
    init.origin = 0;
    init.next_row = d.prompt_len;
  }
  init.cur_row = -1;
  init.step = 0;
  init.prompt_len = d.prompt_len;
  init.window = d.window;
  init.rows = d.rows;
  init.error = 0;
  c->origin = init.origin;
  c->next_row = init.next_row;
  c->cur_row = -1;
  c->step = 0;

  cudaError_t e = cudaMemsetAsync(dev_mem, 0, l.total, stream);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cudaMemsetAsync");
  }
  e = swa::launch_init_state(c->state, c->valid_start, dev_valid_start, d.batch, init, stream);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "init_state launch");
  }
  *out = c;
  return SWA_OK;
}

void swa_cache_free(swa_cache* cache) { delete cache; }

swa_status swa_cache_info(const swa_cache* c, swa_cache_desc* desc_out, void** k_out, void** v_out,
                          void** state_out) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  if (desc_out) *desc_out = c->desc;
  if (k_out) *k_out = c->k;
  if (v_out) *v_out = c->v;
  if (state_out) *state_out = c->state;
  return SWA_OK;
}

swa_status swa_cache_position(const swa_cache* c, int32_t* origin, int32_t* next_row, int32_t* step) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  if (origin) *origin = c->origin;
  if (next_row) *next_row = c->next_row;
  if (step) *step = c->step;
  return SWA_OK;
}

swa_status swa_cache_advance(swa_cache* c, int32_t steps) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  if (!decodes(c->desc.kind)) return fail(SWA_ESTATE, "only a compact or ring cache decodes");
  if (steps < 0) return fail(SWA_EINVAL, "steps must be >= 0");
  if (steps == 0) return SWA_OK;
  if (c->desc.kind == SWA_CACHE_RING) {  // never rolls
    const int32_t R = c->desc.rows;
    c->cur_row = int32_t((int64_t(c->next_row) + steps - 1) % R);
    c->next_row = int32_t((int64_t(c->next_row) + steps) % R);
    c->step += steps;
    return SWA_OK;
  }
  if (int64_t(c->next_row) + steps > c->desc.rows)
    return fail(SWA_ESTATE, "advancing %d steps runs past a due roll (next_row = %d, rows = %d)", steps,
                c->next_row, c->desc.rows);
  c->cur_row = c->next_row + steps - 1;
  c->next_row += steps;
  c->step += steps;
  return SWA_OK;
}

swa_status swa_cache_check(swa_cache* c, swa_stream_t stream) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t err = 0;
  e = cudaMemcpy(&err, &c->state->error, sizeof err, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  if (err != 0) {
    const int32_t zero = 0;
    cudaMemcpy(&c->state->error, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (err == swa::kErrTimeout) return fail(SWA_ETIMEOUT, "a bounded wait inside a kernel gave up");
    return fail(SWA_EDEVICE, "device error %d recorded in the cache state (%s)", err,
                err == swa::kErrRowRange  ? "decode row out of range"
                : err == swa::kErrRollDue ? "decode mask built while a roll was due"
                                          : "unknown");
  }
  return SWA_OK;
}

size_t swa_prefill_plan_bytes(const swa_prefill_meta* meta) {
  if (!check_meta(meta)) return 0;
  return swa::plan_layout(meta->batch, meta->chunk_len).total;
}

swa_status swa_plan_check(const void* plan, swa_stream_t stream) {
  if (!plan || !aligned16(plan)) return fail(SWA_EINVAL, "plan is NULL or misaligned");
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  swa::PlanHeader h;
  e = cudaMemcpy(&h, plan, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  if (h.magic != swa::kPlanMagic) return fail(SWA_ESTATE, "buffer does not hold a built plan");
  if (h.error == swa::kErrImageCrossesChunk)
    return fail(SWA_EDEVICE, "an image block crosses the chunk end (its future keys are not written yet)");
  if (h.error == swa::kErrBadDocs) return fail(SWA_EDEVICE, "cu_seqlens does not cover every token");
  if (h.error == swa::kErrTimeout) return fail(SWA_ETIMEOUT, "a bounded wait inside a kernel gave up");
  if (h.error != 0) return fail(SWA_EDEVICE, "device error %d recorded in the plan", h.error);
  return SWA_OK;
}

swa_status swa_build_mask(swa_cache* c, int32_t kind, const swa_prefill_meta* meta, void* dev_out,
                          swa_stream_t stream) {
  if (!dev_out) return fail(SWA_EINVAL, "dev_out is NULL");
  if (kind == SWA_MASK_DECODE) {
    if (!c) return fail(SWA_EINVAL, "a decode mask needs a cache");
    if (!decodes(c->desc.kind)) return fail(SWA_ESTATE, "a decode mask needs a compact or ring cache");
    if (meta) return fail(SWA_EINVAL, "a decode mask takes no prefill meta");
    const bool ring = c->desc.kind == SWA_CACHE_RING;
    if (!ring && c->next_row >= c->desc.rows)
      return fail(SWA_ESTATE, "a roll is due before the next decode step (next_row == rows)");
    cudaError_t e = swa::launch_decode_mask(c->state, c->valid_start, c->desc.batch, c->desc.rows, ring,
                                            static_cast<uint8_t*>(dev_out), stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode mask launch");
    c->cur_row = c->next_row;
    c->next_row = (ring && c->next_row + 1 == c->desc.rows) ? 0 : c->next_row + 1;
    c->step += 1;
    return SWA_OK;
  }
  if (kind == SWA_MASK_PREFILL || kind == SWA_MASK_DENSE_DEBUG) {
    if (!check_meta(meta)) return SWA_EINVAL;
    if (!aligned16(dev_out)) return fail(SWA_EINVAL, "dev_out must be 16-byte aligned");
    if (c && (c->desc.kind != SWA_CACHE_PREFILL || c->desc.batch != meta->batch ||
              c->desc.rows < meta->seq_len))
      return fail(SWA_EINVAL, "meta does not match the prefill cache");
    cudaError_t e;
    if (kind == SWA_MASK_PREFILL) {
      e = swa::launch_prefill_plan(*meta, dev_out, stream);
    } else {
      e = swa::launch_dense_debug(*meta, static_cast<uint8_t*>(dev_out), stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "mask launch");
    return SWA_OK;
  }
  return fail(SWA_EINVAL, "unknown mask kind %d", kind);
}

swa_status swa_prefill(swa_cache* c, int32_t layer, int32_t mode, int32_t q_heads, int32_t kv_heads,
                       int32_t head_dim, const swa_prefill_meta* meta, const swa_bf16* q,
                       const swa_bf16* k, const swa_bf16* v, float scale, swa_bf16* out, float* lse,
                       swa_stream_t stream) {
  if (!check_meta(meta)) return SWA_EINVAL;
  if (mode != SWA_MODE_CAUSAL && mode != SWA_MODE_GENERIC) return fail(SWA_EINVAL, "unknown mode %d", mode);
  if (q_heads < 1 || kv_heads < 1 || q_heads % kv_heads)
    return fail(SWA_EINVAL, "q_heads must be a positive multiple of kv_heads");
  if (head_dim != 256 && head_dim != 512) return fail(SWA_EUNSUPPORTED, "prefill supports head_dim 256 and 512");
  if (!q || !out) return fail(SWA_EINVAL, "q and out are required");
  if (!aligned16(q) || !aligned16(out) || (k && !aligned16(k)) || (v && !aligned16(v)) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3)))
    return fail(SWA_EINVAL, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(SWA_EINVAL, "scale must be finite");
  if (mode == SWA_MODE_CAUSAL && meta->img_id) return fail(SWA_EINVAL, "the causal plan takes no img_id (use SWA_MODE_GENERIC)");
  if (mode == SWA_MODE_GENERIC && !meta->plan) return fail(SWA_EINVAL, "the generic plan needs meta->plan");
  swa::PrefillArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.out = out;
  a.lse = lse;
  a.valid_start = meta->valid_start;
  a.plan = meta->plan;
  a.batch = meta->batch;
  a.chunk_start = meta->chunk_start;
  a.chunk_len = meta->chunk_len;
  a.q_heads = q_heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.window = meta->window;
  a.generic = mode == SWA_MODE_GENERIC;
  a.scale_log2 = scale * 1.4426950408889634f;
  if (c) {
    const swa_cache_desc& d = c->desc;
    if (d.kind != SWA_CACHE_PREFILL) return fail(SWA_ESTATE, "prefill needs a prefill cache");
    if (layer < 0 || layer >= d.layers) return fail(SWA_EINVAL, "layer %d out of range", layer);
    if (d.kv_heads != kv_heads || d.head_dim != head_dim || d.batch != meta->batch)
      return fail(SWA_EINVAL, "shape does not match the cache");
    if (meta->seq_len > d.rows || meta->window != d.window)
      return fail(SWA_EINVAL, "meta (seq_len, window) does not match the cache");
    if (meta->cu_seqlens) return fail(SWA_EINVAL, "packed documents take no cache");
    if ((k == nullptr) != (v == nullptr)) return fail(SWA_EINVAL, "k and v must both be given or both NULL");
    const long long slab = (long long)d.rows * d.head_dim;
    a.k = c->k + (long long)layer * d.batch * d.kv_heads * slab;
    a.v = c->v + (long long)layer * d.batch * d.kv_heads * slab;
    a.key_seq_stride = (long long)d.kv_heads * slab;
    a.key_head_stride = slab;
    a.key_row_stride = d.head_dim;
    a.key_rows = meta->chunk_start + meta->chunk_len;
    a.key_dim_rows = d.rows;
    a.err = &c->state->error;
    if (k) {
      // the chunk's K/V go into the cache rows [chunk_start, chunk_start + C):
      // either before the attention kernel (which then reads every key from
      // the cache), or concurrently with it when it reads the chunk's keys
      // from k / v
      a.k_in = reinterpret_cast<const uint16_t*>(k);
      a.v_in = reinterpret_cast<const uint16_t*>(v);
      const bool concurrent = swa::prefill_reads_chunk_inputs(a);
      if (!concurrent) {
        a.k_in = a.v_in = nullptr;
        cudaError_t e = swa::launch_write_rows(c->k, c->v, k, v, d.batch, meta->chunk_len, d.kv_heads, d.head_dim,
                                               d.rows, layer, meta->chunk_start, false, stream);
        if (e != cudaSuccess) return cuda_fail(e, "write_rows launch");
      }
      cudaError_t e = swa::launch_prefill_tc(a, stream);
      if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
      if (concurrent) {
        e = swa::launch_write_rows(c->k, c->v, k, v, d.batch, meta->chunk_len, d.kv_heads, d.head_dim, d.rows,
                                   layer, meta->chunk_start, true, stream);
        if (e != cudaSuccess) return cuda_fail(e, "write_rows launch");
      }
      return SWA_OK;
    }
  } else {
    if (!meta->cu_seqlens) return fail(SWA_EINVAL, "without a cache, prefill needs packed documents (cu_seqlens)");
    if (mode != SWA_MODE_GENERIC) return fail(SWA_EINVAL, "packed documents use SWA_MODE_GENERIC");
    if (!k || !v) return fail(SWA_EINVAL, "packed documents need k and v");
    a.k = k;
    a.v = v;
    a.key_seq_stride = 0;
    a.key_head_stride = head_dim;
    a.key_row_stride = (long long)kv_heads * head_dim;
    a.key_rows = meta->seq_len;
    a.key_dim_rows = meta->seq_len;
    a.err = reinterpret_cast<int32_t*>(const_cast<void*>(meta->plan)) + offsetof(swa::PlanHeader, error) / 4;
  }
  cudaError_t e = swa::launch_prefill_tc(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return SWA_OK;
}

size_t swa_prefill_backward_workspace_bytes(int32_t q_heads, const swa_prefill_meta* meta) {
  if (check_backward_meta(meta) != SWA_OK) return 0;
  if (q_heads < 1) {
    fail(SWA_EINVAL, "q_heads must be >= 1");
    return 0;
  }
  return swa::backward_layout(meta->batch, meta->seq_len, q_heads, meta->window, meta->img_id != nullptr).total;
}

swa_status swa_prefill_backward(int32_t q_heads, int32_t kv_heads, int32_t head_dim, const swa_prefill_meta* meta,
                                const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const swa_bf16* out,
                                const swa_bf16* dout, const float* lse, float scale, swa_bf16* dq, swa_bf16* dk,
                                swa_bf16* dv, void* workspace, size_t ws_bytes, swa_stream_t stream) {
  const swa_status ms = check_backward_meta(meta);
  if (ms != SWA_OK) return ms;
  if (q_heads < 1 || kv_heads < 1 || q_heads % kv_heads)
    return fail(SWA_EINVAL, "q_heads must be a positive multiple of kv_heads");
  if (head_dim != 256 && head_dim != 512) return fail(SWA_EUNSUPPORTED, "backward supports head_dim 256 and 512");
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !workspace)
    return fail(SWA_EINVAL, "q, k, v, out, dout, lse, dq, dk, dv and workspace are required");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return fail(SWA_EINVAL, "tensor pointers must be 16-byte aligned (lse 4-byte)");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(SWA_EINVAL, "workspace must be 256-byte aligned");
  if (!std::isfinite(scale)) return fail(SWA_EINVAL, "scale must be finite");
  const swa::BackwardLayout L =
      swa::backward_layout(meta->batch, meta->seq_len, q_heads, meta->window, meta->img_id != nullptr);
  if (ws_bytes < L.total)
    return fail(SWA_EINVAL, "workspace too small: %zu bytes, need %zu", ws_bytes, L.total);
  char* ws = static_cast<char*>(workspace);
  swa::BackwardArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.plan = meta->plan;
  a.delta = reinterpret_cast<float*>(ws + L.off_delta);
  a.t_ds = ws + L.off_ds;
  a.t_pt = ws + L.off_pt;
  a.t_dst = ws + L.off_dst;
  a.batch = meta->batch;
  a.seq_len = meta->seq_len;
  a.q_heads = q_heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.band = L.band;
  a.scale = scale;
  a.err = reinterpret_cast<int32_t*>(const_cast<void*>(meta->plan)) + offsetof(swa::PlanHeader, error) / 4;
  cudaError_t e = swa::launch_prefill_backward(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return SWA_OK;
}

swa_status swa_compact(const swa_cache* p, swa_cache* c, swa_stream_t stream) {
  if (!p || !c) return fail(SWA_EINVAL, "cache is NULL");
  if (p->desc.kind != SWA_CACHE_PREFILL || !decodes(c->desc.kind))
    return fail(SWA_ESTATE, "compaction goes from a prefill cache to a compact or ring cache");
  const swa_cache_desc &a = p->desc, &b = c->desc;
  if (a.layers != b.layers || a.batch != b.batch || a.kv_heads != b.kv_heads || a.head_dim != b.head_dim ||
      a.window != b.window || a.prompt_len != b.prompt_len)
    return fail(SWA_EINVAL, "prefill and compact caches differ in shape, window or prompt length");
  if (c->step != 0) return fail(SWA_ESTATE, "the compact cache has already been decoded into");
  const long long slabs = (long long)a.layers * a.batch * a.kv_heads;
  cudaError_t e = swa::launch_compact(c->k, c->v, p->k, p->v, slabs, a.rows, b.rows, b.window,
                                      b.prompt_len, b.head_dim, b.kind == SWA_CACHE_RING, stream);
  if (e != cudaSuccess) return cuda_fail(e, "compact launch");
  return SWA_OK;
}

size_t swa_decode_workspace_bytes(const swa_cache* c, int32_t q_heads) {
  if (!c) {
    fail(SWA_EINVAL, "cache is NULL");
    return 0;
  }
  if (q_heads < 1 || q_heads % c->desc.kv_heads) {
    fail(SWA_EINVAL, "q_heads must be a positive multiple of kv_heads");
    return 0;
  }
  const swa_cache_desc& d = c->desc;
  return swa::decode_split(d.batch, q_heads, d.kv_heads, d.head_dim, d.rows, swa::device_sm_count(),
                        swa::decode_max_cluster()).total;
}

swa_status swa_decode(swa_cache* c, int32_t layer, int32_t q_heads, const swa_bf16* q,
                      const swa_bf16* k_new, const swa_bf16* v_new, const uint8_t* mask, float scale,
                      swa_bf16* out, float* lse, void* workspace, size_t ws_bytes, swa_stream_t stream) {
  return swa_decode_ex(c, layer, q_heads, q, k_new, v_new, mask, scale, out, lse, workspace, ws_bytes, 0u, stream);
}

swa_status swa_decode_ex(swa_cache* c, int32_t layer, int32_t q_heads, const swa_bf16* q,
                         const swa_bf16* k_new, const swa_bf16* v_new, const uint8_t* mask, float scale,
                         swa_bf16* out, float* lse, void* workspace, size_t ws_bytes, uint32_t flags,
                         swa_stream_t stream) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  if (flags & ~uint32_t(SWA_DECODE_INPUTS_READY)) return fail(SWA_EINVAL, "unknown decode flags 0x%x", flags);
  const swa_cache_desc& d = c->desc;
  if (!decodes(d.kind)) return fail(SWA_ESTATE, "decode needs a compact or ring cache");
  if (layer < 0 || layer >= d.layers) return fail(SWA_EINVAL, "layer %d out of range", layer);
  if (q_heads < 1 || q_heads % d.kv_heads) return fail(SWA_EINVAL, "q_heads must be a positive multiple of kv_heads");
  const int g = q_heads / d.kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return fail(SWA_EUNSUPPORTED, "decode supports Hq/Hkv in {1, 2, 4, 8}");
  if (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256 && d.head_dim != 512)
    return fail(SWA_EUNSUPPORTED, "decode supports head_dim 64, 128, 256 and 512");
  if (!q || !mask || !out || !workspace) return fail(SWA_EINVAL, "q, mask, out and workspace are required");
  if (!k_new != !v_new) return fail(SWA_EINVAL, "k_new and v_new are both given or both NULL (KV-sharing layer)");
  if (!aligned16(q) || (k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new)) || !aligned16(out) ||
      !aligned16(workspace) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3)))
    return fail(SWA_EINVAL, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(SWA_EINVAL, "scale must be finite");
  if (c->cur_row < 0) return fail(SWA_ESTATE, "build the step's decode mask before decoding");
  const swa::DecodeSplit sp =
      swa::decode_split(d.batch, q_heads, d.kv_heads, d.head_dim, d.rows, swa::device_sm_count(),
                        swa::decode_max_cluster());
  if (ws_bytes < sp.total) return fail(SWA_EINVAL, "workspace too small (%zu < %zu)", ws_bytes, sp.total);
  swa::DecodeArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.mask = mask;
  a.k_cache = c->k;
  a.v_cache = c->v;
  a.state = c->state;
  a.out = out;
  a.lse = lse;
  char* ws = static_cast<char*>(workspace);
  a.counters = reinterpret_cast<int32_t*>(ws);
  a.ws_ml = reinterpret_cast<float*>(ws + sp.off_ml);
  a.ws_acc = reinterpret_cast<float*>(ws + sp.off_acc);
  a.batch = d.batch;
  a.q_heads = q_heads;
  a.kv_heads = d.kv_heads;
  a.head_dim = d.head_dim;
  a.rows = d.rows;
  a.layer = layer;
  a.nsplit = sp.nsplit;
  a.rows_per_split = sp.rows_per_split;
  a.cluster = sp.cluster;
  a.warps = sp.warps;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.valid_start = c->valid_start;
  a.window = d.window;
  a.ring = d.kind == SWA_CACHE_RING;
  a.inputs_ready = (flags & SWA_DECODE_INPUTS_READY) && k_new ? 1 : 0;
  cudaError_t e = swa::launch_decode(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return SWA_OK;
}

swa_status swa_decode_noalloc(swa_cache* c, int32_t layer, int32_t q_heads, const swa_bf16* q,
                              const swa_bf16* k_new, const swa_bf16* v_new, const uint8_t* mask, float scale,
                              swa_bf16* out, float* lse, swa_stream_t stream) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  const swa_cache_desc& d = c->desc;
  if (!decodes(d.kind)) return fail(SWA_ESTATE, "decode needs a compact or ring cache");
  if (layer < 0 || layer >= d.layers) return fail(SWA_EINVAL, "layer %d out of range", layer);
  if (q_heads < 1 || q_heads % d.kv_heads) return fail(SWA_EINVAL, "q_heads must be a positive multiple of kv_heads");
  const int g = q_heads / d.kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return fail(SWA_EUNSUPPORTED, "decode supports Hq/Hkv in {1, 2, 4, 8}");
  if (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256 && d.head_dim != 512)
    return fail(SWA_EUNSUPPORTED, "decode supports head_dim 64, 128, 256 and 512");
  if (!q || !mask || !out) return fail(SWA_EINVAL, "q, mask and out are required");
  if (!k_new != !v_new) return fail(SWA_EINVAL, "k_new and v_new are both given or both NULL (KV-sharing layer)");
  if (!aligned16(q) || (k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new)) || !aligned16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3)))
    return fail(SWA_EINVAL, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(SWA_EINVAL, "scale must be finite");
  if (c->cur_row < 0) return fail(SWA_ESTATE, "build the step's decode mask before decoding");
  const swa::DecodeSplit sp =
      swa::decode_split(d.batch, q_heads, d.kv_heads, d.head_dim, d.rows, swa::device_sm_count(),
                        swa::decode_max_cluster());
  // The static array: a fixed ticket area for up to SWA_DECODE_STATIC_MAX_SLABS
  // (sequence, KV head) slabs, then the split statistics and partials.  Only
  // the workspace merge (several splits that are not one cluster) uses it.
  const size_t pairs = size_t(d.batch) * d.kv_heads;
  const size_t tickets = swa::align256(size_t(SWA_DECODE_STATIC_MAX_SLABS) * sizeof(int32_t));
  const size_t partials = sp.total - sp.off_ml;
  const bool uses_scratch = sp.nsplit > 1 && !sp.cluster;
  if (uses_scratch && (pairs > size_t(SWA_DECODE_STATIC_MAX_SLABS) ||
                       tickets + partials > size_t(SWA_DECODE_STATIC_SCRATCH_BYTES)))
    return fail(SWA_EUNSUPPORTED,
                "this shape needs %zu bytes of decode scratch for %zu slabs; the static array holds %zu bytes "
                "(tickets for %d slabs)",
                tickets + partials, pairs, size_t(SWA_DECODE_STATIC_SCRATCH_BYTES), SWA_DECODE_STATIC_MAX_SLABS);
  void* scratch = nullptr;
  cudaError_t e = swa::decode_static_scratch(&scratch);  // first call on a device: address and cleared tickets
  if (e != cudaSuccess) return cuda_fail(e, "decode static scratch set-up");
  swa::DecodeArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.mask = mask;
  a.k_cache = c->k;
  a.v_cache = c->v;
  a.state = c->state;
  a.out = out;
  a.lse = lse;
  char* ws = static_cast<char*>(scratch);
  a.counters = reinterpret_cast<int32_t*>(ws);
  a.ws_ml = reinterpret_cast<float*>(ws + tickets);
  a.ws_acc = reinterpret_cast<float*>(ws + tickets + (sp.off_acc - sp.off_ml));
  a.batch = d.batch;
  a.q_heads = q_heads;
  a.kv_heads = d.kv_heads;
  a.head_dim = d.head_dim;
  a.rows = d.rows;
  a.layer = layer;
  a.nsplit = sp.nsplit;
  a.rows_per_split = sp.rows_per_split;
  a.cluster = sp.cluster;
  a.warps = sp.warps;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.valid_start = c->valid_start;
  a.window = d.window;
  a.ring = d.kind == SWA_CACHE_RING;
  a.inputs_ready = 0;
  e = swa::launch_decode(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return SWA_OK;
}

swa_status swa_roll(swa_cache* c, swa_stream_t stream) {
  if (!c) return fail(SWA_EINVAL, "cache is NULL");
  const swa_cache_desc& d = c->desc;
  if (d.kind == SWA_CACHE_RING) return fail(SWA_ESTATE, "a ring cache never rolls");
  if (d.kind != SWA_CACHE_COMPACT) return fail(SWA_ESTATE, "only a compact cache rolls");
  if (c->next_row != d.rows)
    return fail(SWA_ESTATE, "a roll is due only when next_row == rows (next_row = %d)", c->next_row);
  const long long slabs = (long long)d.layers * d.batch * d.kv_heads;
  cudaError_t e = swa::launch_roll(c->k, c->v, slabs, d.rows, d.window, d.head_dim, c->state, stream);
  if (e != cudaSuccess) return cuda_fail(e, "roll launch");
  c->origin += SWA_ROLL_ROWS;
  c->next_row = d.window;
  return SWA_OK;
}

}  // extern "C"
