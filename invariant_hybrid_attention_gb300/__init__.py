"""Python binding of the g4attn C ABI (include/g4attn.h): argument marshalling only.

Every step of the attention path runs in the CUDA kernels of libg4attn.so, loaded with
ctypes from this directory. There is no Python, PyTorch or CPU implementation to fall back
on: if the library is missing or a call fails, an exception says so.

The functions take torch tensors (device memory and streams come from PyTorch) and pass
their raw pointers; names follow the C entry points.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libg4attn.so")

G4_OK, G4_ERR_INVALID, G4_ERR_UNSUPPORTED, G4_ERR_CUDA, G4_ERR_TIMEOUT, G4_ERR_DEVICE, G4_ERR_SCRATCH = range(7)
G4_SLIDING, G4_GLOBAL = 0, 1
PAGE_SIZE = 16
DECODE_STATIC_SCRATCH_BYTES = 32 << 20   # the static scratch of g4attn_decode_static, per device

EXPORTS = ("g4attn_rope_apply", "g4attn_prefill", "g4attn_prefill_stage", "g4attn_prefill_attend",
           "g4attn_prefill_normed", "g4attn_prefill_vision", "g4attn_kv_append_normed", "g4attn_decode_normed",
           "g4attn_decode_exact", "g4attn_decode_exact_workspace_bytes",
           "g4attn_kv_append", "g4attn_decode_workspace_bytes",
           "g4attn_decode", "g4attn_decode_static", "g4attn_provenance", "g4attn_status_sync", "g4attn_status_string",
           "g4attn_set_wait_limit_ns", "g4attn_wait_limit_ns", "g4attn_prefill_partial", "g4attn_merge_partials")
DEFAULT_WAIT_LIMIT_NS = 2_000_000_000   # the kernels' bounded waits give up after 2 s by default


class g4attn_layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rope_partial", ctypes.c_float), ("softmax_scale", ctypes.c_float), ("kv_shared", ctypes.c_int32)]


class g4attn_norms(ctypes.Structure):
    _fields_ = [("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p), ("v_norm", ctypes.c_int32),
                ("eps", ctypes.c_float)]


class g4attn_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_rot", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32)]


class G4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: Optional[str] = None):
    """Loads libg4attn.so (built by __graft_entry__.build() or build.build()). Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libg4attn.so not found at {p}: build it first (the library has no fallback path)")
    lib = ctypes.CDLL(p)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    L, C = ctypes.POINTER(g4attn_layer), ctypes.POINTER(g4attn_cache)
    N = ctypes.POINTER(g4attn_norms)
    sigs = {
        "g4attn_rope_apply": (I32, [L, P, P, I32, I32, P, P]),
        "g4attn_prefill": (I32, [L, P, P, P, I32, P, P, P, I32, C, P, I32, P, P]),
        "g4attn_prefill_stage": (I32, [L, P, P, P, I32, P, P, P, I32, C, P, I32, P, P]),
        "g4attn_prefill_attend": (I32, [L, P, I32, P, P, P, I32, C, P, I32, P, P]),
        "g4attn_prefill_normed": (I32, [L, N, P, P, P, I32, P, P, P, I32, C, P, I32, P, P]),
        "g4attn_prefill_vision": (I32, [L, N, P, P, P, I32, P, P, P, I32, P, C, P, I32, P, P]),
        "g4attn_kv_append_normed": (I32, [L, N, P, P, I32, P, P, P, I32, C, P, I32, P]),
        "g4attn_decode_normed": (I32, [L, N, P, P, P, P, I32, C, P, I32, P, P, SZ, P]),
        "g4attn_decode_exact": (I32, [L, N, P, P, P, P, I32, C, P, I32, P, P, SZ, P]),
        "g4attn_decode_exact_workspace_bytes": (SZ, [I32]),
        "g4attn_kv_append": (I32, [L, P, P, I32, P, P, P, I32, C, P, I32, P]),
        "g4attn_decode_workspace_bytes": (SZ, [L, I32, I32]),
        "g4attn_decode": (I32, [L, P, P, P, P, I32, C, P, I32, P, P, SZ, P]),
        "g4attn_decode_static": (I32, [L, P, P, P, P, I32, C, P, I32, P, P]),
        "g4attn_provenance": (I32, [L, ctypes.c_char_p, SZ]),
        "g4attn_status_sync": (I32, [P]),
        "g4attn_status_string": (ctypes.c_char_p, [I32]),
        "g4attn_set_wait_limit_ns": (I32, [ctypes.c_uint64]),
        "g4attn_wait_limit_ns": (ctypes.c_uint64, []),
        "g4attn_prefill_partial": (I32, [L, P, I32, P, P, P, I32, P, P, C, P, I32, P, P, P]),
        "g4attn_merge_partials": (I32, [L, I32, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                                        I32, P, P, I32, P, P]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().g4attn_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - used while formatting errors
        return "unknown"


def sliding_layer(window: int = 1024, softmax_scale: Optional[float] = None, tp: int = 1) -> g4attn_layer:
    """The sliding layer, or (tp > 1) one tensor-parallel rank's slice of it: 32/tp query heads,
    16/tp KV heads."""
    return g4attn_layer(G4_SLIDING, 32 // tp, 16 // tp, 256, int(window), 1.0e4, 1.0,
                        1.0 / math.sqrt(256) if softmax_scale is None else float(softmax_scale), 0)


def global_layer(softmax_scale: Optional[float] = None, tp: int = 1) -> g4attn_layer:
    """The global K==V layer, or (tp > 1) one rank's slice: 32/tp query heads and max(1, 4/tp) KV
    heads (at tp = 8 two ranks hold the same KV head)."""
    return g4attn_layer(G4_GLOBAL, 32 // tp, max(1, 4 // tp), 512, 0, 1.0e6, 0.25,
                        1.0 / math.sqrt(512) if softmax_scale is None else float(softmax_scale), 1)


def make_cache(k, v, num_pages: int, k_rot=None) -> g4attn_cache:
    return g4attn_cache(_ptr(k), _ptr(v), _ptr(k_rot), int(num_pages), PAGE_SIZE)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(status: int, what: str):
    if status != G4_OK:
        raise G4Error(status, what)


def g4attn_rope_apply(layer: g4attn_layer, x, pos, out=None, stream=None):
    """out[r][h] = RoPE(x[r][h], pos[r]); x [T, H, D] bf16, pos int32 [T] (device)."""
    out = x if out is None else out
    T, H = int(x.shape[0]), int(x.shape[1])
    _check(load().g4attn_rope_apply(ctypes.byref(layer), _ptr(x), _ptr(pos), T, H, _ptr(out), _stream(stream)),
           "g4attn_rope_apply")
    return out


def g4attn_kv_append(layer, k, v, q_start, q_len, ctx_start, cache: g4attn_cache, page_table, stream=None):
    T, B = int(k.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_kv_append(ctypes.byref(layer), _ptr(k), _ptr(v), T, _ptr(q_start), _ptr(q_len),
                                   _ptr(ctx_start), B, ctypes.byref(cache), _ptr(page_table),
                                   int(page_table.shape[1]), _stream(stream)), "g4attn_kv_append")


def g4attn_prefill(layer, q, k, v, q_start, q_len, ctx_start, cache: g4attn_cache, page_table, out, stream=None):
    T, B = int(q.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_prefill(ctypes.byref(layer), _ptr(q), _ptr(k), _ptr(v), T, _ptr(q_start), _ptr(q_len),
                                 _ptr(ctx_start), B, ctypes.byref(cache), _ptr(page_table), int(page_table.shape[1]),
                                 _ptr(out), _stream(stream)), "g4attn_prefill")
    return out


def g4attn_prefill_stage(layer, q, k, v, q_start, q_len, ctx_start, cache: g4attn_cache, page_table, out,
                         stream=None):
    T, B = int(q.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_prefill_stage(ctypes.byref(layer), _ptr(q), _ptr(k), _ptr(v), T, _ptr(q_start),
                                       _ptr(q_len), _ptr(ctx_start), B, ctypes.byref(cache), _ptr(page_table),
                                       int(page_table.shape[1]), _ptr(out), _stream(stream)), "g4attn_prefill_stage")
    return out


def g4attn_prefill_attend(layer, q, q_start, q_len, ctx_start, cache: g4attn_cache, page_table, out, stream=None):
    """The attention step of a prefill: q the raw query rows (rotated in the kernel), or None when
    g4attn_prefill_stage staged the roped queries in out."""
    T, B = int(out.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_prefill_attend(ctypes.byref(layer), _ptr(q), T, _ptr(q_start), _ptr(q_len), _ptr(ctx_start),
                                        B, ctypes.byref(cache), _ptr(page_table), int(page_table.shape[1]),
                                        _ptr(out), _stream(stream)), "g4attn_prefill_attend")
    return out


def g4attn_decode_workspace_bytes(layer, B: int, max_pages: int) -> int:
    return int(load().g4attn_decode_workspace_bytes(ctypes.byref(layer), int(B), int(max_pages)))


def g4attn_decode(layer, q, k_new, v_new, seq_len, cache: g4attn_cache, page_table, out, workspace, stream=None):
    B = int(q.shape[0])
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().g4attn_decode(ctypes.byref(layer), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(seq_len), B,
                                ctypes.byref(cache), _ptr(page_table), int(page_table.shape[1]), _ptr(out),
                                _ptr(workspace), nbytes, _stream(stream)), "g4attn_decode")
    return out


def g4attn_decode_static(layer, q, k_new, v_new, seq_len, cache: g4attn_cache, page_table, out, stream=None):
    """g4attn_decode with the library's static scratch instead of a workspace: for callers that
    cannot allocate device memory at decode time. Allocates nothing (this wrapper included).
    Raises G4Error(G4_ERR_SCRATCH) when the step needs more than DECODE_STATIC_SCRATCH_BYTES.
    Calls that may overlap on the GPU (unordered streams) share the scratch and race."""
    B = int(q.shape[0])
    _check(load().g4attn_decode_static(ctypes.byref(layer), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(seq_len), B,
                                       ctypes.byref(cache), _ptr(page_table), int(page_table.shape[1]), _ptr(out),
                                       _stream(stream)), "g4attn_decode_static")
    return out


def g4attn_provenance(layer) -> str:
    buf = ctypes.create_string_buffer(2048)
    n = load().g4attn_provenance(ctypes.byref(layer), buf, len(buf))
    if n < 0:
        raise G4Error(G4_ERR_UNSUPPORTED, "g4attn_provenance")
    return buf.value.decode()


def g4attn_status_sync(stream=None) -> int:
    return int(load().g4attn_status_sync(_stream(stream)))


def make_norms(q_weight=None, k_weight=None, v_norm: bool = False, eps: float = 1e-6) -> g4attn_norms:
    """Per-head norm arguments: q_weight / k_weight are bf16 [head_dim] device tensors or None."""
    return g4attn_norms(_ptr(q_weight), _ptr(k_weight), 1 if v_norm else 0, float(eps))


def g4attn_prefill_normed(layer, norms: g4attn_norms, q, k, v, q_start, q_len, ctx_start, cache: g4attn_cache,
                          page_table, out, stream=None):
    T, B = int(q.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_prefill_normed(ctypes.byref(layer), ctypes.byref(norms), _ptr(q), _ptr(k), _ptr(v), T,
                                        _ptr(q_start), _ptr(q_len), _ptr(ctx_start), B, ctypes.byref(cache),
                                        _ptr(page_table), int(page_table.shape[1]), _ptr(out), _stream(stream)),
           "g4attn_prefill_normed")
    return out


def g4attn_prefill_vision(layer, norms, q, k, v, q_start, q_len, ctx_start, span, cache: g4attn_cache,
                          page_table, out, stream=None):
    """g4attn_prefill_normed with image spans: span is an int32 [T, 2] device tensor (or None),
    row t's image [s0, s1) of absolute positions, s1 <= s0 for a text row. norms may be None."""
    T, B = int(q.shape[0]), int(q_start.shape[0])
    nrm = None if norms is None else ctypes.byref(norms)
    _check(load().g4attn_prefill_vision(ctypes.byref(layer), nrm, _ptr(q), _ptr(k), _ptr(v), T,
                                        _ptr(q_start), _ptr(q_len), _ptr(ctx_start), B, _ptr(span),
                                        ctypes.byref(cache), _ptr(page_table), int(page_table.shape[1]), _ptr(out),
                                        _stream(stream)),
           "g4attn_prefill_vision")
    return out


def g4attn_kv_append_normed(layer, norms: g4attn_norms, k, v, q_start, q_len, ctx_start, cache: g4attn_cache,
                            page_table, stream=None):
    T, B = int(k.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_kv_append_normed(ctypes.byref(layer), ctypes.byref(norms), _ptr(k), _ptr(v), T,
                                          _ptr(q_start), _ptr(q_len), _ptr(ctx_start), B, ctypes.byref(cache),
                                          _ptr(page_table), int(page_table.shape[1]), _stream(stream)),
           "g4attn_kv_append_normed")


def g4attn_decode_normed(layer, norms: g4attn_norms, q, k_new, v_new, seq_len, cache: g4attn_cache, page_table,
                         out, workspace, stream=None):
    B = int(q.shape[0])
    _check(load().g4attn_decode_normed(ctypes.byref(layer), ctypes.byref(norms), _ptr(q), _ptr(k_new), _ptr(v_new),
                                       _ptr(seq_len), B, ctypes.byref(cache), _ptr(page_table),
                                       int(page_table.shape[1]), _ptr(out), _ptr(workspace),
                                       int(workspace.numel() * workspace.element_size()), _stream(stream)),
           "g4attn_decode_normed")
    return out


def g4attn_decode_exact_workspace_bytes(B: int) -> int:
    return int(load().g4attn_decode_exact_workspace_bytes(int(B)))


def g4attn_decode_exact(layer, norms, q, k_new, v_new, seq_len, cache: g4attn_cache, page_table, out, workspace,
                        stream=None):
    """One decode step through the prefill kernels: the rows' bits equal a prefill's. norms may be
    None; workspace holds at least g4attn_decode_exact_workspace_bytes(B) bytes."""
    B = int(q.shape[0])
    nrm = None if norms is None else ctypes.byref(norms)
    _check(load().g4attn_decode_exact(ctypes.byref(layer), nrm, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(seq_len), B,
                                      ctypes.byref(cache), _ptr(page_table), int(page_table.shape[1]), _ptr(out),
                                      _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                      _stream(stream)),
           "g4attn_decode_exact")
    return out


def g4attn_set_wait_limit_ns(ns: int) -> None:
    """Bound of every protocol wait in kernels launched from now on (0 .. 2e9 ns; default 2 s)."""
    _check(load().g4attn_set_wait_limit_ns(int(ns)), "g4attn_set_wait_limit_ns")


def g4attn_wait_limit_ns() -> int:
    return int(load().g4attn_wait_limit_ns())


def g4attn_prefill_partial(layer, q, q_start, q_len, ctx_start, key_begin, key_end, cache: g4attn_cache, page_table,
                           o_part, ml_part, stream=None):
    """A global layer's attention restricted to each sequence's keys key_begin .. key_end-1 (int32 [B]
    device tensors): writes the un-normalised fp32 output o_part [T, Hq, 512] and the softmax state
    ml_part [T, Hq, 2] (max in log2 units, sum) of every sequence row."""
    T, B = int(q.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_prefill_partial(ctypes.byref(layer), _ptr(q), T, _ptr(q_start), _ptr(q_len), _ptr(ctx_start),
                                         B, _ptr(key_begin), _ptr(key_end), ctypes.byref(cache), _ptr(page_table),
                                         int(page_table.shape[1]), _ptr(o_part), _ptr(ml_part), _stream(stream)),
           "g4attn_prefill_partial")


def g4attn_merge_partials(layer, o_parts, ml_parts, q_start, q_len, out, stream=None):
    """Merges the partials (lists of device tensors, in rank order) into out [T, Hq, 512] bf16."""
    n = len(o_parts)
    arr_o = (ctypes.c_void_p * n)(*[_ptr(t) for t in o_parts])
    arr_m = (ctypes.c_void_p * n)(*[_ptr(t) for t in ml_parts])
    T, B = int(out.shape[0]), int(q_start.shape[0])
    _check(load().g4attn_merge_partials(ctypes.byref(layer), n, arr_o, arr_m, T, _ptr(q_start), _ptr(q_len), B,
                                        _ptr(out), _stream(stream)), "g4attn_merge_partials")
    return out
