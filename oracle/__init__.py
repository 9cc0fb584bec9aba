"""fp64 CPU oracle for weight-absorbed MLA decode -- TEST INFRASTRUCTURE.

This package is what the CUDA path is checked against, not the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  It shares no code with the CUDA library and never
imports it; the two meet only through the seeded input generators, which hold
none of the method's arithmetic.

The numerics live in ``mla_oracle.c`` (plain fp64 loops, OpenMP over output
rows), compiled on first use with the host C compiler; ``counts.py`` holds the
closed-form FLOP / byte counters the pages print.  Inputs are the exact bf16
tensors handed to the GPU (bit patterns, widened to fp64 inside the C code) or,
for an FP8 latent cache, its E4M3 codes (uint8) and the cache's one scale;
activations returned here are float64 CPU tensors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``liboracle.so`` (skipped when up to date)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        # No OpenMP runtime on this host: the pragmas are ignored, results are identical.
        subprocess.run(base, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("s_q", ctypes.c_int),
                ("d_c", ctypes.c_int), ("d_rope", ctypes.c_int), ("d_nope", ctypes.c_int),
                ("d_v", ctypes.c_int), ("scale", ctypes.c_double)]


class _Cache(ctypes.Structure):
    _fields_ = [("kv", ctypes.c_void_p), ("seq_stride", ctypes.c_longlong),
                ("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int),
                ("page_size", ctypes.c_int), ("capacity", ctypes.c_longlong),
                ("seq_lens", ctypes.c_void_p), ("elem", ctypes.c_int), ("kv_scale", ctypes.c_double)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, LL = ctypes.c_void_p, ctypes.c_longlong
            lib.orc_threads.restype = ctypes.c_int
            lib.orc_e4m3_to_f64.restype = ctypes.c_double
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_f64_to_e4m3.restype = ctypes.c_uint8
            lib.orc_f64_to_e4m3.argtypes = [ctypes.c_double]
            lib.orc_encode_e4m3.argtypes = [LL, P, P]
            lib.orc_absorb_q.argtypes = [ctypes.POINTER(_Dims), P, P, P, P]
            lib.orc_attend.argtypes = [ctypes.POINTER(_Dims), P, ctypes.POINTER(_Cache), P, LL, P, P]
            lib.orc_attend_partial.argtypes = [ctypes.POINTER(_Dims), P, ctypes.POINTER(_Cache),
                                               LL, LL, LL, P, P, P]
            lib.orc_combine.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P]
            lib.orc_out_proj.argtypes = [ctypes.POINTER(_Dims), P, P, P]
            lib.orc_naive.argtypes = [ctypes.POINTER(_Dims), P, P, ctypes.POINTER(_Cache), P, P,
                                      P, LL, P, P]
            lib.orc_down_proj.argtypes = [LL, ctypes.c_int, ctypes.c_int, P, P, P]
            lib.orc_attend_sparse.argtypes = [ctypes.POINTER(_Dims), P, ctypes.POINTER(_Cache), P, ctypes.c_int,
                                              P, LL, P, P]
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses (the host's affinity unless OMP_NUM_THREADS says otherwise)."""
    return int(_load().orc_threads())


# ----------------------------------------------------------------------------- marshalling
def _bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> contiguous int16 view of its bit patterns (CPU)."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"oracle expects bf16 inputs, got {t.dtype}")
    return t.detach().to("cpu").contiguous().view(torch.int16)


def _f64(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu", torch.float64).contiguous()


def _i32(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu", torch.int32).contiguous()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dims(d) -> _Dims:
    return _Dims(int(d.B), int(d.H), int(d.s_q), int(d.d_c), int(d.d_rope), int(d.d_nope),
                 int(d.d_v), float(d.scale))


class _CacheArgs:
    """Keeps the marshalled cache tensors alive while the C call runs.

    Contiguous cache: ``kv`` is [B, T_max, d_c + d_rope] (any strides; copied
    contiguous here).  Paged cache: ``kv`` is the pool [P, page_size, d_c + d_rope]
    and ``block_table`` is [B, max_pages].  ``kv`` is bf16, or uint8 /
    float8_e4m3fn E4M3 codes together with ``kv_scale`` (value = kv_scale * code)."""

    def __init__(self, d, kv, seq_lens, block_table=None, page_size=64, kv_scale=None):
        if kv.dtype in (torch.uint8, torch.float8_e4m3fn):
            if kv_scale is None:
                raise ValueError("an FP8 cache needs its kv_scale")
            self.kv = kv.detach().to("cpu").contiguous().view(torch.uint8)
            elem, scale = 1, float(kv_scale)
        else:
            self.kv = _bits(kv)
            elem, scale = 0, 1.0
        self.seq_lens = _i32(seq_lens)
        self.block_table = _i32(block_table) if block_table is not None else None
        W = d.d_c + d.d_rope
        if int(kv.shape[-1]) != W:
            raise ValueError("cache rows must be d_c + d_rope wide")
        if self.block_table is None:
            t_max = int(kv.shape[1])
            self.c = _Cache(_ptr(self.kv).value, t_max * W, None, 0, int(page_size), t_max,
                            _ptr(self.seq_lens).value, elem, scale)
        else:
            max_pages = int(self.block_table.shape[1])
            self.c = _Cache(_ptr(self.kv).value, 0, _ptr(self.block_table).value, max_pages,
                            int(page_size), max_pages * int(page_size), _ptr(self.seq_lens).value, elem, scale)


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64)).contiguous()
    return r, int(r.numel())


# ----------------------------------------------------------------------------- public API
def absorb_q(d, q_nope, q_rope, w_uk) -> torch.Tensor:
    """q_cat [B, s_q, H, d_c + d_rope] float64 (see orc_absorb_q)."""
    lib = _load()
    qn, qr, wk = _bits(q_nope), _bits(q_rope), _bits(w_uk)
    out = torch.empty(d.B, d.s_q, d.H, d.d_c + d.d_rope, dtype=torch.float64)
    lib.orc_absorb_q(ctypes.byref(_dims(d)), _ptr(qn), _ptr(qr), _ptr(wk), _ptr(out))
    return out


def e4m3_to_f64(code: int) -> float:
    """Value of one OCP FP8 E4M3 code (see orc_e4m3_to_f64)."""
    return float(_load().orc_e4m3_to_f64(int(code) & 0xFF))


def e4m3_encode(values) -> torch.Tensor:
    """E4M3 codes (uint8) of float64 values: nearest, ties to even, saturating at
    +-448 (see orc_f64_to_e4m3)."""
    v = _f64(torch.as_tensor(values))
    out = torch.empty(v.shape, dtype=torch.uint8)
    _load().orc_encode_e4m3(int(v.numel()), _ptr(v), _ptr(out))
    return out


def attend(d, q_cat, kv, seq_lens, block_table=None, page_size=64, rows=None, kv_scale=None):
    """(o_lat [B, s_q, H, d_c], lse [B, s_q, H]) float64 from a float64-widened q_cat.

    ``rows`` optionally lists flat row indices (b*s_q + i)*H + h to compute; other
    rows are returned as NaN.  An FP8 cache (uint8 codes) needs ``kv_scale``."""
    lib = _load()
    q = _f64(q_cat)
    ca = _CacheArgs(d, kv, seq_lens, block_table, page_size, kv_scale)
    o = torch.full((d.B, d.s_q, d.H, d.d_c), float("nan"), dtype=torch.float64)
    lse = torch.full((d.B, d.s_q, d.H), float("nan"), dtype=torch.float64)
    r, n = _rows_arg(rows)
    lib.orc_attend(ctypes.byref(_dims(d)), _ptr(q), ctypes.byref(ca.c), _ptr(r), n, _ptr(o), _ptr(lse))
    return o, lse


def attend_sparse(d, q_cat, kv, seq_lens, indices, block_table=None, page_size=64, rows=None, kv_scale=None):
    """Sparse top-k attention: (o_lat, lse) float64 over the listed tokens only.

    ``indices`` [B, s_q, topk] int32: token positions per query token, shared by
    the heads; entries that do not name a visible token (e.g. -1) take no part."""
    lib = _load()
    q = _f64(q_cat)
    ca = _CacheArgs(d, kv, seq_lens, block_table, page_size, kv_scale)
    idx = _i32(indices)
    topk = int(idx.shape[-1])
    o = torch.full((d.B, d.s_q, d.H, d.d_c), float("nan"), dtype=torch.float64)
    lse = torch.full((d.B, d.s_q, d.H), float("nan"), dtype=torch.float64)
    r, n = _rows_arg(rows)
    lib.orc_attend_sparse(ctypes.byref(_dims(d)), _ptr(q), ctypes.byref(ca.c), _ptr(idx), topk, _ptr(r), n,
                          _ptr(o), _ptr(lse))
    return o, lse


def attend_partial(d, q_cat, kv, seq_lens, row, j0, j1, block_table=None, page_size=64, kv_scale=None):
    """Unnormalised partial (m, l, acc[d_c]) of one flat row over tokens [j0, j1)."""
    lib = _load()
    q = _f64(q_cat)
    ca = _CacheArgs(d, kv, seq_lens, block_table, page_size, kv_scale)
    m = torch.zeros(1, dtype=torch.float64)
    l = torch.zeros(1, dtype=torch.float64)
    acc = torch.zeros(d.d_c, dtype=torch.float64)
    lib.orc_attend_partial(ctypes.byref(_dims(d)), _ptr(q), ctypes.byref(ca.c), int(row), int(j0),
                           int(j1), _ptr(m), _ptr(l), _ptr(acc))
    return float(m.item()), float(l.item()), acc


def combine(m, l, acc):
    """Merge partials: m, l [n] and acc [n, width] -> (o [width], lse)."""
    lib = _load()
    m = _f64(torch.as_tensor(m, dtype=torch.float64))
    l = _f64(torch.as_tensor(l, dtype=torch.float64))
    acc = _f64(torch.as_tensor(acc, dtype=torch.float64))
    n, width = int(acc.shape[0]), int(acc.shape[1])
    o = torch.zeros(width, dtype=torch.float64)
    lse = torch.zeros(1, dtype=torch.float64)
    lib.orc_combine(n, width, _ptr(m), _ptr(l), _ptr(acc), _ptr(o), _ptr(lse))
    return o, float(lse.item())


def out_proj(d, o_lat, w_uv) -> torch.Tensor:
    """out [B, s_q, H, d_v] float64 from a float64-widened o_lat."""
    lib = _load()
    o = _f64(o_lat)
    wv = _bits(w_uv)
    out = torch.empty(d.B, d.s_q, d.H, d.d_v, dtype=torch.float64)
    lib.orc_out_proj(ctypes.byref(_dims(d)), _ptr(o), _ptr(wv), _ptr(out))
    return out


def down_proj(x, w_dkv) -> torch.Tensor:
    """c = x . W_DKV in fp64: x [..., d_model] bf16, w_dkv [d_model, d_c] bf16 -> [..., d_c]."""
    lib = _load()
    xb, wb = _bits(x), _bits(w_dkv)
    d_model, d_c = int(w_dkv.shape[0]), int(w_dkv.shape[1])
    M = xb.numel() // d_model
    c = torch.empty(M, d_c, dtype=torch.float64)
    lib.orc_down_proj(M, d_model, d_c, _ptr(xb), _ptr(wb), _ptr(c))
    return c.view(*x.shape[:-1], d_c)


def cache_append(d, x, w_dkv, k_rope, kv, seq_lens, block_table=None, page_size=64, kv_scale=None):
    """The cache after appending the new tokens, in fp64, and a bool mask of the
    rows written ("MLA, dim by dim", "MLA Decode": c = x . W_DKV is appended).

    Token i of sequence b (x [B, s_q, d_model], k_rope [B, s_q, d_rope]) lands at
    position L_b - s_q + i (seq_lens already count the new tokens): row
    [c | k_rope] of the contiguous cache [B, T_max, W], or of page
    block_table[b][pos // page_size] of the pool [P, page_size, W].  Invalid
    lengths or page ids write nothing.  For an FP8 cache (uint8 codes with
    ``kv_scale``) the returned cache holds the exact values divided by kv_scale
    for the written rows (the codes a quantiser must round) and the old codes'
    values elsewhere; e4m3_encode turns it into codes."""
    c = down_proj(x, w_dkv)
    fp8 = kv.dtype in (torch.uint8, torch.float8_e4m3fn)
    if fp8:
        if kv_scale is None:
            raise ValueError("an FP8 cache needs its kv_scale")
        out = kv.detach().to("cpu").contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        c = c / float(kv_scale)
    else:
        out = kv.detach().to("cpu", torch.float64).clone()
    written = torch.zeros(out.shape[:-1], dtype=torch.bool)
    kr = k_rope.detach().to("cpu", torch.float64)
    if fp8:
        kr = kr / float(kv_scale)
    lens = [int(v) for v in seq_lens.detach().to("cpu")]
    bt = block_table.detach().to("cpu") if block_table is not None else None
    cap = int(bt.shape[1]) * page_size if bt is not None else int(kv.shape[1])
    for b in range(d.B):
        L = lens[b]
        if L < d.s_q or L > cap:
            continue
        for i in range(d.s_q):
            pos = L - d.s_q + i
            if bt is None:
                idx = (b, pos)
            else:
                page = int(bt[b, pos // page_size])
                if page < 0 or page >= int(kv.shape[0]):
                    continue
                idx = (page, pos % page_size)
            out[idx][: d.d_c] = c[b, i]
            out[idx][d.d_c:] = kr[b, i]
            written[idx] = True
    return out, written


def naive(d, q_nope, q_rope, kv, seq_lens, w_uk, w_uv, block_table=None, page_size=64, rows=None):
    """Naive decompress-then-attend: (out [B, s_q, H, d_v], lse [B, s_q, H]) float64."""
    lib = _load()
    qn, qr, wk, wv = _bits(q_nope), _bits(q_rope), _bits(w_uk), _bits(w_uv)
    ca = _CacheArgs(d, kv, seq_lens, block_table, page_size)
    out = torch.full((d.B, d.s_q, d.H, d.d_v), float("nan"), dtype=torch.float64)
    lse = torch.full((d.B, d.s_q, d.H), float("nan"), dtype=torch.float64)
    r, n = _rows_arg(rows)
    lib.orc_naive(ctypes.byref(_dims(d)), _ptr(qn), _ptr(qr), ctypes.byref(ca.c), _ptr(wk), _ptr(wv),
                  _ptr(r), n, _ptr(out), _ptr(lse))
    return out, lse


def decode(d, q_nope, q_rope, kv, seq_lens, w_uk, w_uv, block_table=None, page_size=64, rows=None,
           kv_scale=None):
    """Absorbed decode end to end in fp64: dict(q_cat, o_lat, lse, out).

    With ``rows`` the attention runs on those rows only; out is then valid on
    those rows only."""
    q_cat = absorb_q(d, q_nope, q_rope, w_uk)
    o_lat, lse = attend(d, q_cat, kv, seq_lens, block_table, page_size, rows, kv_scale)
    out = out_proj(d, torch.nan_to_num(o_lat, nan=0.0) if rows is not None else o_lat, w_uv)
    if rows is not None:
        keep = torch.zeros(d.B * d.s_q * d.H, dtype=torch.bool)
        keep[torch.as_tensor(np.asarray(rows, dtype=np.int64))] = True
        out.view(-1, d.d_v)[~keep] = float("nan")
    return {"q_cat": q_cat, "o_lat": o_lat, "lse": lse, "out": out}
