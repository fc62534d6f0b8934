"""Thin ctypes binding of libswa (include/swa.h): argument marshalling only.

Every step of the attention path runs in the CUDA kernels of libswa.so; this
module turns torch tensors into device pointers and raises ``SwaError`` when a
call returns a status other than SWA_OK.  Importing it fails loudly when the
library has not been built (there is no fallback).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libswa.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                      "or python -m sliding_window_gqa_swa_gb300.build")

_lib = ctypes.CDLL(LIB_PATH)

# status codes and enums (include/swa.h)
OK, EINVAL, ESTATE, EUNSUPPORTED, ECUDA, ETIMEOUT, EDEVICE = range(7)
CACHE_PREFILL, CACHE_COMPACT, CACHE_RING = 0, 1, 2
MODE_CAUSAL, MODE_GENERIC = 0, 1
MASK_DECODE, MASK_PREFILL, MASK_DENSE_DEBUG = 0, 1, 2
ROLL_ROWS = 64


class SwaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kind", "layers", "batch", "kv_heads", "head_dim", "window", "prompt_len", "rows")]


class PrefillMeta(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seq_len", ctypes.c_int32), ("chunk_start", ctypes.c_int32),
                ("chunk_len", ctypes.c_int32), ("window", ctypes.c_int32), ("num_docs", ctypes.c_int32),
                ("valid_start", ctypes.c_void_p), ("img_id", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("plan", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGS = {
    "swa_cache_bytes": (_SZ, [ctypes.POINTER(CacheDesc)]),
    "swa_cache_alloc": (_I, [ctypes.POINTER(CacheDesc), _P, _SZ, _P, _P, ctypes.POINTER(_P)]),
    "swa_cache_free": (None, [_P]),
    "swa_cache_info": (_I, [_P, ctypes.POINTER(CacheDesc), ctypes.POINTER(_P), ctypes.POINTER(_P),
                            ctypes.POINTER(_P)]),
    "swa_cache_position": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "swa_cache_advance": (_I, [_P, _I]),
    "swa_cache_check": (_I, [_P, _P]),
    "swa_prefill_plan_bytes": (_SZ, [ctypes.POINTER(PrefillMeta)]),
    "swa_build_mask": (_I, [_P, _I, ctypes.POINTER(PrefillMeta), _P, _P]),
    "swa_plan_check": (_I, [_P, _P]),
    "swa_prefill": (_I, [_P, _I, _I, _I, _I, _I, ctypes.POINTER(PrefillMeta), _P, _P, _P, _F, _P, _P, _P]),
    "swa_prefill_backward_workspace_bytes": (_SZ, [_I, ctypes.POINTER(PrefillMeta)]),
    "swa_prefill_backward": (_I, [_I, _I, _I, ctypes.POINTER(PrefillMeta), _P, _P, _P, _P, _P, _P, _F, _P, _P, _P,
                                  _P, _SZ, _P]),
    "swa_compact": (_I, [_P, _P, _P]),
    "swa_decode_workspace_bytes": (_SZ, [_P, _I]),
    "swa_decode": (_I, [_P, _I, _I, _P, _P, _P, _P, _F, _P, _P, _P, _SZ, _P]),
    "swa_decode_ex": (_I, [_P, _I, _I, _P, _P, _P, _P, _F, _P, _P, _P, _SZ, ctypes.c_uint32, _P]),
    "swa_decode_noalloc": (_I, [_P, _I, _I, _P, _P, _P, _P, _F, _P, _P, _P]),
    "swa_roll": (_I, [_P, _P]),
    "swa_last_error": (ctypes.c_char_p, []),
    "swa_status_string": (ctypes.c_char_p, [_I]),
    "swa_version": (_I, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def lib():
    return _lib


def last_error() -> str:
    return _lib.swa_last_error().decode()


def check(status: int, what: str) -> None:
    if status != OK:
        raise SwaError(status, f"{what}: {_lib.swa_status_string(status).decode()}: {last_error()}")


def ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _bf16(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")


# ------------------------------------------------------------------ cache
def cache_bytes(kind, layers, batch, kv_heads, head_dim, window, prompt_len, rows=0) -> int:
    d = CacheDesc(kind, layers, batch, kv_heads, head_dim, window, prompt_len, rows)
    return int(_lib.swa_cache_bytes(ctypes.byref(d)))


class Cache:
    """A sliding cache in torch-owned device memory (one buffer: state, K, V)."""

    def __init__(self, kind: int, layers: int, batch: int, kv_heads: int, head_dim: int, window: int,
                 prompt_len: int, valid_start: Optional[torch.Tensor] = None, rows: int = 0,
                 device=None, stream=None, mem: Optional[torch.Tensor] = None):
        """``mem``: optional caller-owned uint8 device buffer (>= the cache's bytes,
        256-byte aligned) to bind instead of a fresh allocation."""
        desc = CacheDesc(kind, layers, batch, kv_heads, head_dim, window, prompt_len, rows)
        nbytes = int(_lib.swa_cache_bytes(ctypes.byref(desc)))
        if nbytes == 0:
            raise SwaError(EINVAL, f"swa_cache_bytes: {last_error()}")
        device = torch.device("cuda") if device is None else torch.device(device)
        if mem is not None:
            if mem.dtype != torch.uint8 or not mem.is_cuda or mem.numel() < nbytes:
                raise SwaError(EINVAL, f"mem must be a CUDA uint8 tensor of at least {nbytes} bytes")
            self.mem = mem[:nbytes]
        else:
            self.mem = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.valid_start = None
        if valid_start is not None:
            self.valid_start = valid_start.to(device=device, dtype=torch.int32).contiguous()
        self.handle = None
        self._desc_in = desc
        self.bind(stream)
        d = CacheDesc()
        kp, vp, sp = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        check(_lib.swa_cache_info(self.handle, ctypes.byref(d), ctypes.byref(kp), ctypes.byref(vp),
                                  ctypes.byref(sp)), "swa_cache_info")
        self.desc = d
        base = self.mem.data_ptr()
        shape = (d.layers, d.batch, d.kv_heads, d.rows, d.head_dim)
        n = d.layers * d.batch * d.kv_heads * d.rows * d.head_dim
        self.k = self.mem[kp.value - base: kp.value - base + 2 * n].view(torch.bfloat16).view(shape)
        self.v = self.mem[vp.value - base: vp.value - base + 2 * n].view(torch.bfloat16).view(shape)
        self._state = self.mem[sp.value - base: sp.value - base + 32].view(torch.int32)

    def bind(self, stream=None) -> None:
        """(Re)bind a fresh handle to the same memory: zero-fill + initial state."""
        self.close()
        h = ctypes.c_void_p()
        check(_lib.swa_cache_alloc(ctypes.byref(self._desc_in), ptr(self.mem), self.mem.numel(), ptr(self.valid_start),
                                   stream_handle(stream), ctypes.byref(h)), "swa_cache_alloc")
        self.handle = h

    @property
    def rows(self) -> int:
        return self.desc.rows

    def state(self) -> dict:
        """Device state (synchronises via the copy)."""
        vals = self._state.cpu().tolist()
        return dict(zip(("origin", "next_row", "cur_row", "step", "prompt_len", "window", "rows", "error"), vals))

    def position(self):
        o, n, s = _I(), _I(), _I()
        check(_lib.swa_cache_position(self.handle, ctypes.byref(o), ctypes.byref(n), ctypes.byref(s)),
              "swa_cache_position")
        return o.value, n.value, s.value

    def needs_roll(self) -> bool:
        # a ring cache never rolls
        return self.desc.kind == CACHE_COMPACT and self.position()[1] == self.rows

    def advance(self, steps: int = 1) -> None:
        """Advance the host mirror for steps replayed from a captured graph."""
        check(_lib.swa_cache_advance(self.handle, steps), "swa_cache_advance")

    def check(self, stream=None) -> None:
        check(_lib.swa_cache_check(self.handle, stream_handle(stream)), "swa_cache_check")

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            _lib.swa_cache_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ masks
class Meta:
    """Owns a PrefillMeta and keeps the tensors it points to alive."""

    def __init__(self, batch, seq_len, chunk_start, chunk_len, window, valid_start=None, img_id=None,
                 cu_seqlens=None, plan=None):
        self._keep = [t for t in (valid_start, img_id, cu_seqlens, plan) if t is not None]
        num_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
        self.c = PrefillMeta(batch, seq_len, chunk_start, chunk_len, window, num_docs,
                             ptr(valid_start), ptr(img_id), ptr(cu_seqlens), ptr(plan))
        self.plan = plan

    def with_plan(self, plan: torch.Tensor) -> "Meta":
        self.plan = plan
        self._keep.append(plan)
        self.c.plan = ptr(plan)
        return self

    def plan_bytes(self) -> int:
        n = int(_lib.swa_prefill_plan_bytes(ctypes.byref(self.c)))
        if n == 0:
            raise SwaError(EINVAL, f"swa_prefill_plan_bytes: {last_error()}")
        return n


def build_decode_mask(cache: Cache, mask_out: torch.Tensor, stream=None) -> None:
    check(_lib.swa_build_mask(cache.handle, MASK_DECODE, None, ptr(mask_out), stream_handle(stream)),
          "swa_build_mask(decode)")


def build_prefill_plan(meta: Meta, cache: Optional[Cache] = None, stream=None, device=None,
                       out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Build the prefill plan (into ``out`` when given, else a new buffer);
    attaches it to ``meta``."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    plan = torch.empty(meta.plan_bytes(), dtype=torch.uint8, device=dev) if out is None else out
    check(_lib.swa_build_mask(cache.handle if cache else None, MASK_PREFILL, ctypes.byref(meta.c),
                              ptr(plan), stream_handle(stream)), "swa_build_mask(prefill)")
    meta.with_plan(plan)
    return plan


def dense_debug_mask(meta: Meta, stream=None, device=None) -> torch.Tensor:
    dev = torch.device("cuda") if device is None else torch.device(device)
    out = torch.empty((meta.c.batch, meta.c.chunk_len, meta.c.seq_len), dtype=torch.uint8, device=dev)
    check(_lib.swa_build_mask(None, MASK_DENSE_DEBUG, ctypes.byref(meta.c), ptr(out), stream_handle(stream)),
          "swa_build_mask(dense_debug)")
    return out


def plan_check(plan: torch.Tensor, stream=None) -> None:
    check(_lib.swa_plan_check(ptr(plan), stream_handle(stream)), "swa_plan_check")


# ------------------------------------------------------------------ compute
def prefill(cache: Optional[Cache], layer: int, mode: int, q: torch.Tensor, k: Optional[torch.Tensor],
            v: Optional[torch.Tensor], meta: Meta, scale: float, out: torch.Tensor,
            lse: Optional[torch.Tensor] = None, kv_heads: Optional[int] = None, stream=None) -> None:
    _bf16(q, "q")
    _bf16(out, "out")
    hq, d = q.shape[-2], q.shape[-1]
    if kv_heads is None:
        kv_heads = cache.desc.kv_heads if cache is not None else k.shape[-2]
    check(_lib.swa_prefill(cache.handle if cache else None, layer, mode, hq, kv_heads, d, ctypes.byref(meta.c),
                           ptr(q), ptr(k), ptr(v), float(scale), ptr(out), ptr(lse), stream_handle(stream)),
          "swa_prefill")


def backward_workspace_bytes(q_heads: int, meta: Meta) -> int:
    n = int(_lib.swa_prefill_backward_workspace_bytes(q_heads, ctypes.byref(meta.c)))
    if n == 0:
        raise SwaError(EINVAL, f"swa_prefill_backward_workspace_bytes: {last_error()}")
    return n


def backward_workspace(q_heads: int, meta: Meta, device=None) -> torch.Tensor:
    """A workspace for swa_prefill_backward (no initialisation needed)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return torch.empty(backward_workspace_bytes(q_heads, meta), dtype=torch.uint8, device=dev)


def prefill_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, dout: torch.Tensor,
                     lse: torch.Tensor, meta: Meta, scale: float, dq: torch.Tensor, dk: torch.Tensor,
                     dv: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _bf16(t, n)
    hq, hkv, d = q.shape[-2], k.shape[-2], q.shape[-1]
    check(_lib.swa_prefill_backward(hq, hkv, d, ctypes.byref(meta.c), ptr(q), ptr(k), ptr(v), ptr(out), ptr(dout),
                                    ptr(lse), float(scale), ptr(dq), ptr(dk), ptr(dv), ptr(workspace),
                                    workspace.numel(), stream_handle(stream)), "swa_prefill_backward")


def compact(prefill_cache: Cache, compact_cache: Cache, stream=None) -> None:
    check(_lib.swa_compact(prefill_cache.handle, compact_cache.handle, stream_handle(stream)), "swa_compact")


def decode_workspace_bytes(cache: Cache, q_heads: int) -> int:
    n = int(_lib.swa_decode_workspace_bytes(cache.handle, q_heads))
    if n == 0:
        raise SwaError(EINVAL, f"swa_decode_workspace_bytes: {last_error()}")
    return n


def decode_workspace(cache: Cache, q_heads: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for swa_decode."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return torch.zeros(decode_workspace_bytes(cache, q_heads), dtype=torch.uint8, device=dev)


DECODE_INPUTS_READY = 1


def decode(cache: Cache, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
           mask: torch.Tensor, scale: float, out: torch.Tensor, workspace: torch.Tensor,
           lse: Optional[torch.Tensor] = None, stream=None, inputs_ready: bool = False) -> None:
    """swa_decode; ``inputs_ready`` calls swa_decode_ex with SWA_DECODE_INPUTS_READY
    (the inputs were written before the previously enqueued kernel, which does
    not write them: see include/swa.h)."""
    _bf16(q, "q")
    if inputs_ready:
        check(_lib.swa_decode_ex(cache.handle, layer, q.shape[-2], ptr(q), ptr(k_new), ptr(v_new), ptr(mask),
                                 float(scale), ptr(out), ptr(lse), ptr(workspace), workspace.numel(),
                                 DECODE_INPUTS_READY, stream_handle(stream)), "swa_decode_ex")
        return
    check(_lib.swa_decode(cache.handle, layer, q.shape[-2], ptr(q), ptr(k_new), ptr(v_new), ptr(mask),
                          float(scale), ptr(out), ptr(lse), ptr(workspace), workspace.numel(),
                          stream_handle(stream)), "swa_decode")


def roll(cache: Cache, stream=None) -> None:
    check(_lib.swa_roll(cache.handle, stream_handle(stream)), "swa_roll")
