"""Thin ctypes binding of ``libmla.so`` (declared in ``include/mla.h``).

Argument marshalling only: torch provides device memory and the current CUDA
stream, every computation runs in the library's kernels.  There is no fallback:
if the library is missing or a call fails, an exception says so.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

_lib = None


class MLAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("s_q", ctypes.c_int), ("d_c", ctypes.c_int),
                ("d_rope", ctypes.c_int), ("d_nope", ctypes.c_int), ("d_v", ctypes.c_int),
                ("scale", ctypes.c_float)]


class Cache(ctypes.Structure):
    _fields_ = [("kv", ctypes.c_void_p), ("seq_stride", ctypes.c_longlong), ("capacity", ctypes.c_int),
                ("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int), ("page_size", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("seq_lens", ctypes.c_void_p), ("max_seq_len", ctypes.c_int),
                ("kv_dtype", ctypes.c_int), ("kv_scale", ctypes.c_float)]


KV_BF16, KV_E4M3 = 0, 1
ABI_VERSION = 2
SPLITS_BALANCED = -1  # num_splits asking for the balanced plan (MLA_SPLITS_BALANCED)


EXPORTS = ("mla_status_string", "mla_abi_version", "mla_absorb_q", "mla_decode_workspace_size",
           "mla_decode_num_splits", "mla_decode_attn", "mla_out_proj", "mla_naive_workspace_size",
           "mla_naive_decode", "mla_read_status", "mla_decode_attn_noalloc", "mla_cache_append_workspace_size",
           "mla_cache_append", "mla_decode_sparse_workspace_size", "mla_decode_attn_sparse", "mla_prefill_crossover",
           "mla_prefill_expand_workspace_size", "mla_prefill_expand", "mla_prefill_workspace_size", "mla_prefill",
           "mla_decode_step", "mla_set_wait_limit_ns")
PATH_ABSORB, PATH_EXPAND = 0, 1


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Open libmla.so (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"MLA CUDA library not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    pd, pc = ctypes.POINTER(Dims), ctypes.POINTER(Cache)
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [I]
    lib.mla_abi_version.restype = I
    lib.mla_absorb_q.argtypes = [pd, P, P, P, P, P]
    lib.mla_absorb_q.restype = I
    lib.mla_decode_workspace_size.argtypes = [pd, pc, I]
    lib.mla_decode_workspace_size.restype = SZ
    lib.mla_decode_num_splits.argtypes = [pd, pc]
    lib.mla_decode_num_splits.restype = I
    lib.mla_decode_attn.argtypes = [pd, P, pc, P, P, P, SZ, I, P]
    lib.mla_decode_attn.restype = I
    lib.mla_out_proj.argtypes = [pd, P, P, P, P]
    lib.mla_out_proj.restype = I
    lib.mla_naive_workspace_size.argtypes = [pd, pc]
    lib.mla_naive_workspace_size.restype = SZ
    lib.mla_naive_decode.argtypes = [pd, P, P, pc, P, P, P, P, P, SZ, P]
    lib.mla_naive_decode.restype = I
    lib.mla_decode_sparse_workspace_size.argtypes = [pd, pc, I, I]
    lib.mla_decode_sparse_workspace_size.restype = SZ
    lib.mla_decode_attn_sparse.argtypes = [pd, P, pc, P, I, P, P, P, SZ, I, P]
    lib.mla_decode_attn_sparse.restype = I
    lib.mla_cache_append_workspace_size.argtypes = [pd, I]
    lib.mla_cache_append_workspace_size.restype = SZ
    lib.mla_cache_append.argtypes = [pd, I, P, P, P, pc, P, SZ, P]
    lib.mla_cache_append.restype = I
    lib.mla_read_status.argtypes = [P, ctypes.POINTER(I), P]
    lib.mla_read_status.restype = I
    lib.mla_decode_step.argtypes = [pd, P, P, pc, P, P, P, P, P, P, P, SZ, I, P]
    lib.mla_decode_step.restype = I
    lib.mla_prefill_crossover.argtypes = [pd, ctypes.c_longlong]
    lib.mla_prefill_crossover.restype = ctypes.c_double
    lib.mla_prefill_expand_workspace_size.argtypes = [pd, pc]
    lib.mla_prefill_expand_workspace_size.restype = SZ
    lib.mla_prefill_expand.argtypes = [pd, P, P, pc, P, P, P, P, P, SZ, P]
    lib.mla_prefill_expand.restype = I
    lib.mla_prefill_workspace_size.argtypes = [pd, pc]
    lib.mla_prefill_workspace_size.restype = SZ
    lib.mla_prefill.argtypes = [pd, P, P, pc, P, P, P, P, P, SZ, ctypes.POINTER(I), P]
    lib.mla_prefill.restype = I
    lib.mla_decode_attn_noalloc.argtypes = [pd, P, pc, P, P, I, P, P]
    lib.mla_decode_attn_noalloc.restype = I
    lib.mla_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.mla_set_wait_limit_ns.restype = I
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().mla_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != 0:
        raise MLAError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Problem:
    """Sizes of one decode step (mirrors ``mla_dims``)."""
    B: int
    H: int
    s_q: int
    d_c: int
    d_rope: int
    d_nope: int
    d_v: int
    scale: float

    def dims(self) -> Dims:
        return Dims(self.B, self.H, self.s_q, self.d_c, self.d_rope, self.d_nope, self.d_v, float(self.scale))

    @classmethod
    def of(cls, cfg) -> "Problem":
        return cls(cfg.B, cfg.H, cfg.s_q, cfg.d_c, cfg.d_rope, cfg.d_nope, cfg.d_v, cfg.scale)


def make_cache(prob: Problem, kv: torch.Tensor, seq_lens: torch.Tensor, block_table=None,
               page_size: int = 64, max_seq_len: int = 0, kv_scale: float | None = None) -> Cache:
    """Cache descriptor for a contiguous [B, T_max, W] (any sequence stride) or paged
    [P, page, W] latent cache already on the device: bf16 values, or FP8 E4M3 codes
    (uint8 or float8_e4m3fn) with their ``kv_scale`` (value = kv_scale * code)."""
    W = prob.d_c + prob.d_rope
    fp8 = kv.dtype in (torch.uint8, torch.float8_e4m3fn)
    if (kv.dtype != torch.bfloat16 and not fp8) or kv.shape[-1] != W or kv.stride(-1) != 1:
        raise ValueError("kv must be bf16 or FP8 codes with rows of d_c + d_rope contiguous values")
    if fp8 and kv_scale is None:
        raise ValueError("an FP8 cache needs its kv_scale")
    dt, sc = (KV_E4M3, float(kv_scale)) if fp8 else (KV_BF16, 1.0)
    if block_table is None:
        if kv.dim() != 3 or kv.stride(1) != W:
            raise ValueError("contiguous kv must be [B, T_max, W] with dense token rows")
        return Cache(kv.data_ptr(), kv.stride(0), kv.shape[1], None, 0, page_size, 0,
                     seq_lens.data_ptr(), int(max_seq_len), dt, sc)
    if not kv.is_contiguous() or kv.dim() != 3:
        raise ValueError("paged kv must be a dense [P, page, W] pool")
    if block_table.dtype != torch.int32 or not block_table.is_contiguous():
        raise ValueError("block_table must be a dense int32 [B, max_pages] tensor")
    return Cache(kv.data_ptr(), 0, 0, block_table.data_ptr(), block_table.shape[1], kv.shape[1],
                 kv.shape[0], seq_lens.data_ptr(), int(max_seq_len), dt, sc)


# ---------------------------------------------------------------------------- entry points
def absorb_q(prob: Problem, q_nope, q_rope, w_uk, q_cat=None, stream=None):
    lib = load()
    if q_cat is None:
        q_cat = torch.empty(prob.B, prob.s_q, prob.H, prob.d_c + prob.d_rope, dtype=torch.bfloat16,
                            device=q_nope.device)
    d = prob.dims()
    _check(lib.mla_absorb_q(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(q_cat),
                            _stream(stream)), "mla_absorb_q")
    return q_cat


def decode_workspace_size(prob: Problem, cache: Cache, num_splits: int = 0) -> int:
    d = prob.dims()
    n = load().mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(cache), int(num_splits))
    if n == 0:
        raise ValueError("mla_decode_workspace_size rejected the arguments")
    return int(n)


def decode_num_splits(prob: Problem, cache: Cache) -> int:
    d = prob.dims()
    return int(load().mla_decode_num_splits(ctypes.byref(d), ctypes.byref(cache)))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def decode_attn(prob: Problem, q_cat, cache: Cache, o_lat=None, lse=None, workspace=None, num_splits: int = 0,
                stream=None):
    lib = load()
    dev = q_cat.device
    if o_lat is None:
        o_lat = torch.empty(prob.B, prob.s_q, prob.H, prob.d_c, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(prob.B, prob.s_q, prob.H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(decode_workspace_size(prob, cache, num_splits), dev)
    d = prob.dims()
    _check(lib.mla_decode_attn(ctypes.byref(d), _ptr(q_cat), ctypes.byref(cache), _ptr(o_lat), _ptr(lse),
                               _ptr(workspace), workspace.numel(), int(num_splits), _stream(stream)),
           "mla_decode_attn")
    return o_lat, lse, workspace


def out_proj(prob: Problem, o_lat, w_uv, out=None, stream=None):
    lib = load()
    if out is None:
        out = torch.empty(prob.B, prob.s_q, prob.H, prob.d_v, dtype=torch.bfloat16, device=o_lat.device)
    d = prob.dims()
    _check(lib.mla_out_proj(ctypes.byref(d), _ptr(o_lat), _ptr(w_uv), _ptr(out), _stream(stream)),
           "mla_out_proj")
    return out


def decode_sparse_workspace_size(prob: Problem, cache: Cache, topk: int, num_splits: int = 0) -> int:
    d = prob.dims()
    n = load().mla_decode_sparse_workspace_size(ctypes.byref(d), ctypes.byref(cache), int(topk), int(num_splits))
    if n == 0:
        raise ValueError("mla_decode_sparse_workspace_size rejected the arguments")
    return int(n)


def decode_attn_sparse(prob: Problem, q_cat, cache: Cache, indices, num_splits: int = 0, o_lat=None, lse=None,
                       workspace=None, stream=None):
    """mla_decode_attn_sparse: attention over the listed tokens (indices int32 [B, s_q, topk])."""
    lib = load()
    dev = q_cat.device
    topk = int(indices.shape[-1])
    if o_lat is None:
        o_lat = torch.empty(prob.B, prob.s_q, prob.H, prob.d_c, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(prob.B, prob.s_q, prob.H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(decode_sparse_workspace_size(prob, cache, topk, num_splits), dev)
    d = prob.dims()
    _check(lib.mla_decode_attn_sparse(ctypes.byref(d), _ptr(q_cat), ctypes.byref(cache), _ptr(indices), topk,
                                      _ptr(o_lat), _ptr(lse), _ptr(workspace), workspace.numel(), int(num_splits),
                                      _stream(stream)), "mla_decode_attn_sparse")
    return o_lat, lse, workspace


def cache_append_workspace_size(prob: Problem, d_model: int) -> int:
    d = prob.dims()
    n = load().mla_cache_append_workspace_size(ctypes.byref(d), int(d_model))
    if n == 0:
        raise ValueError("mla_cache_append_workspace_size rejected the arguments")
    return int(n)


def cache_append(prob: Problem, x, w_dkv, k_rope, cache: Cache, workspace=None, stream=None):
    """mla_cache_append: c = x . W_DKV of the new tokens, written with k_rope into
    rows seq_lens[b] - s_q + i of the cache (whose kv buffer is modified)."""
    lib = load()
    if workspace is None:
        workspace = alloc_workspace(cache_append_workspace_size(prob, int(x.shape[-1])), x.device)
    d = prob.dims()
    _check(lib.mla_cache_append(ctypes.byref(d), int(x.shape[-1]), _ptr(x), _ptr(w_dkv), _ptr(k_rope),
                                ctypes.byref(cache), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mla_cache_append")
    return workspace


def naive_workspace_size(prob: Problem, cache: Cache) -> int:
    d = prob.dims()
    n = load().mla_naive_workspace_size(ctypes.byref(d), ctypes.byref(cache))
    if n == 0:
        raise ValueError("mla_naive_workspace_size rejected the arguments")
    return int(n)


def naive_decode(prob: Problem, q_nope, q_rope, cache: Cache, w_uk, w_uv, out=None, lse=None, workspace=None,
                 stream=None):
    lib = load()
    dev = q_nope.device
    if out is None:
        out = torch.empty(prob.B, prob.s_q, prob.H, prob.d_v, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(prob.B, prob.s_q, prob.H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(naive_workspace_size(prob, cache), dev)
    d = prob.dims()
    _check(lib.mla_naive_decode(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), ctypes.byref(cache), _ptr(w_uk),
                                _ptr(w_uv), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                _stream(stream)), "mla_naive_decode")
    return out, lse, workspace


def prefill_crossover(prob: Problem, L: int) -> float:
    """mla_prefill_crossover: the query count S* where both bracketings tie (host only)."""
    d = prob.dims()
    return float(load().mla_prefill_crossover(ctypes.byref(d), int(L)))


def _prefill_outputs(prob, dev, out, lse):
    if out is None:
        out = torch.empty(prob.B, prob.s_q, prob.H, prob.d_v, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(prob.B, prob.s_q, prob.H, dtype=torch.float32, device=dev)
    return out, lse


def prefill_expand(prob: Problem, q_nope, q_rope, cache: Cache, w_uk, w_uv, out=None, lse=None, workspace=None,
                   stream=None):
    """mla_prefill_expand: K, V re-expanded per head, then per-head attention."""
    lib = load()
    out, lse = _prefill_outputs(prob, q_nope.device, out, lse)
    d = prob.dims()
    if workspace is None:
        n = lib.mla_prefill_expand_workspace_size(ctypes.byref(d), ctypes.byref(cache))
        if n == 0:
            raise ValueError("mla_prefill_expand_workspace_size rejected the arguments")
        workspace = alloc_workspace(n, q_nope.device)
    _check(lib.mla_prefill_expand(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), ctypes.byref(cache), _ptr(w_uk),
                                  _ptr(w_uv), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "mla_prefill_expand")
    return out, lse, workspace


def prefill(prob: Problem, q_nope, q_rope, cache: Cache, w_uk, w_uv, out=None, lse=None, workspace=None,
            stream=None):
    """mla_prefill: absorbed below the crossover S*, expanded at or above it.
    Returns (out, lse, workspace, path)."""
    lib = load()
    out, lse = _prefill_outputs(prob, q_nope.device, out, lse)
    d = prob.dims()
    if workspace is None:
        n = lib.mla_prefill_workspace_size(ctypes.byref(d), ctypes.byref(cache))
        if n == 0:
            raise ValueError("mla_prefill_workspace_size rejected the arguments")
        workspace = alloc_workspace(n, q_nope.device)
    path = ctypes.c_int(-1)
    _check(lib.mla_prefill(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), ctypes.byref(cache), _ptr(w_uk), _ptr(w_uv),
                           _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), ctypes.byref(path),
                           _stream(stream)), "mla_prefill")
    return out, lse, workspace, int(path.value)


def decode_attn_noalloc(prob: Problem, q_cat, cache: Cache, o_lat, lse, num_splits: int = 0,
                        device_status=None, stream=None):
    """mla_decode_attn_noalloc: the same attention with the library's built-in
    scratch array instead of a workspace (for callers that cannot allocate)."""
    d = prob.dims()
    _check(load().mla_decode_attn_noalloc(ctypes.byref(d), _ptr(q_cat), ctypes.byref(cache), _ptr(o_lat),
                                          _ptr(lse), int(num_splits), _ptr(device_status), _stream(stream)),
           "mla_decode_attn_noalloc")
    return o_lat, lse


def set_wait_limit_ns(ns: int) -> None:
    """mla_set_wait_limit_ns: the bound of the attention kernels' waits for work
    (0: the default 2 s).  For tests of the timeout path."""
    _check(load().mla_set_wait_limit_ns(int(ns)), "mla_set_wait_limit_ns")


def read_status(workspace, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(load().mla_read_status(_ptr(workspace), ctypes.byref(v), _stream(stream)), "mla_read_status")
    return int(v.value)


class Decoder:
    """One layer's absorbed decode step with its buffers allocated once:
    absorb_q -> decode_attn -> out_proj on the current stream."""

    def __init__(self, prob: Problem, kv, seq_lens, w_uk, w_uv, block_table=None, page_size=64,
                 max_seq_len=0, num_splits=0, kv_scale=None):
        self.prob = prob
        self.kv, self.seq_lens, self.block_table = kv, seq_lens, block_table
        self.w_uk, self.w_uv = w_uk, w_uv
        self.cache = make_cache(prob, kv, seq_lens, block_table, page_size, max_seq_len, kv_scale)
        self.num_splits = num_splits
        dev = kv.device
        B, s_q, H = prob.B, prob.s_q, prob.H
        self.q_cat = torch.empty(B, s_q, H, prob.d_c + prob.d_rope, dtype=torch.bfloat16, device=dev)
        self.o_lat = torch.empty(B, s_q, H, prob.d_c, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B, s_q, H, dtype=torch.float32, device=dev)
        self.out = torch.empty(B, s_q, H, prob.d_v, dtype=torch.bfloat16, device=dev)
        self.workspace = alloc_workspace(decode_workspace_size(prob, self.cache, num_splits), dev)

    def absorb(self, q_nope, q_rope, stream=None):
        return absorb_q(self.prob, q_nope, q_rope, self.w_uk, self.q_cat, stream)

    def attend(self, stream=None):
        return decode_attn(self.prob, self.q_cat, self.cache, self.o_lat, self.lse, self.workspace,
                           self.num_splits, stream)

    def project(self, stream=None):
        return out_proj(self.prob, self.o_lat, self.w_uv, self.out, stream)

    def step(self, q_nope, q_rope, stream=None):
        """mla_decode_step: the three launches as one call, overlapping."""
        d = self.prob.dims()
        _check(load().mla_decode_step(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), ctypes.byref(self.cache),
                                      _ptr(self.w_uk), _ptr(self.w_uv), _ptr(self.q_cat), _ptr(self.o_lat),
                                      _ptr(self.out), _ptr(self.lse), _ptr(self.workspace), self.workspace.numel(),
                                      int(self.num_splits), _stream(stream)), "mla_decode_step")
        return self.out

    def __call__(self, q_nope, q_rope, stream=None):
        self.absorb(q_nope, q_rope, stream)
        self.attend(stream)
        self.project(stream)
        return self.out
