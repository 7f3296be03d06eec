"""fp64 CPU oracle for absorbed-MLA DCP decode attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

The arithmetic lives in ``mla_oracle.c`` (plain C, double precision); this
module only compiles it with gcc, loads it with ctypes and marshals numpy
arrays.  Work is split over query tokens across threads (ctypes releases the
GIL), which changes no arithmetic: every (token, head) row is computed by the
same sequential C loop.

Inputs follow the library's layouts: bf16 tensors are passed as ``uint16``
numpy arrays holding the bf16 bit patterns, indices as ``int32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "libmla_oracle.so")

KV_LORA_RANK = 512
ROPE_DIM = 64

_lock = threading.Lock()
_lib = None


def build(force: bool = False, extra_flags: tuple[str, ...] = (), out: str | None = None) -> str:
    """Compile ``mla_oracle.c`` into a shared object with gcc; returns its path.

    ``extra_flags``/``out`` let the mutation tests build deliberately broken
    copies of the oracle next to the real one.
    """
    target = out or _LIB
    if not force and os.path.exists(target) and os.path.getmtime(target) >= os.path.getmtime(_SRC):
        return target
    tmp = target + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *extra_flags, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    return target


def _bind(lib):
    i64, f64, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.mla_oracle_local_len.argtypes = [i64, i64, i64]
    lib.mla_oracle_local_len.restype = i64
    lib.mla_oracle_key_visible.argtypes = [i64, i64, i64, i64]
    lib.mla_oracle_key_visible.restype = ctypes.c_int
    lib.mla_oracle_visible_count.argtypes = [i64, i64, i64, i64]
    lib.mla_oracle_visible_count.restype = i64
    lib.mla_oracle_causal_dense.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f64, i64, i64, vp, vp, vp, vp]
    lib.mla_oracle_causal_dense.restype = None
    lib.mla_oracle_dcp_decode.argtypes = [vp, vp, vp, i64, vp, i64, vp, vp, i64, i64, i64, i64, f64, i64, i64,
                                          vp, vp, vp, vp, vp]
    lib.mla_oracle_dcp_decode.restype = None
    lib.mla_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.mla_oracle_e4m3_to_double.restype = f64
    lib.mla_oracle_dcp_decode_kv8.argtypes = [vp, vp, vp, f64, i64, vp, i64, vp, vp, i64, i64, i64, i64, f64, i64,
                                              i64, vp, vp, vp, vp, vp]
    lib.mla_oracle_dcp_decode_kv8.restype = None
    lib.mla_oracle_sparse_dcp_decode.argtypes = [vp, vp, vp, i64, vp, i64, vp, vp, i64, i64, vp, i64, vp, i64, i64,
                                                 f64, i64, i64, vp, vp, vp, vp, vp]
    lib.mla_oracle_sparse_dcp_decode.restype = None
    lib.mla_oracle_lse_merge.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp]
    lib.mla_oracle_lse_merge.restype = None
    lib.mla_oracle_wuv_project.argtypes = [vp, vp, i64, i64, i64, vp]
    lib.mla_oracle_wuv_project.restype = None
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _token_ranges(T, t_lo, t_hi, threads):
    lo, hi = t_lo, (T if t_hi is None else t_hi)
    n = max(1, min(threads, hi - lo))
    cuts = np.linspace(lo, hi, n + 1).astype(np.int64)
    return [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def local_len(L: int, D: int, r: int, lib=None) -> int:
    return int((lib or load()).mla_oracle_local_len(L, D, r))


def key_visible(P: int, D: int, r: int, j: int, lib=None) -> bool:
    return bool((lib or load()).mla_oracle_key_visible(P, D, r, j))


def visible_count(P: int, L: int, D: int, r: int, lib=None) -> int:
    return int((lib or load()).mla_oracle_visible_count(P, L, D, r))


def causal_dense(q_nope, q_pe, kv, kv_start, seq_lens, qsl, scale, t_lo=0, t_hi=None,
                 threads=None, lib=None):
    """Unsharded causal MLA over logical per-request KV rows.

    kv: uint16 [sum L, 576]; kv_start int64 [B] row offsets.  Returns
    (out float64 [n, H, 512], lse float64 [n, H]) for the n = t_hi - t_lo
    tokens [t_lo, t_hi).
    """
    lib = lib or load()
    q_nope, q_pe, kv = _c(q_nope, np.uint16), _c(q_pe, np.uint16), _c(kv, np.uint16)
    kv_start, seq_lens, qsl = _c(kv_start, np.int64), _c(seq_lens, np.int32), _c(qsl, np.int32)
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    t_hi = T if t_hi is None else t_hi
    out = np.full((t_hi - t_lo, H, KV_LORA_RANK), np.nan)
    lse = np.full((t_hi - t_lo, H), np.nan)
    maxL = int(seq_lens.max()) if B else 0

    def run(rng):
        keys = (ctypes.c_void_p * max(1, maxL))()
        s = np.empty(max(1, maxL))
        lib.mla_oracle_causal_dense(_p(q_nope), _p(q_pe), _p(kv), _p(kv_start), _p(seq_lens), _p(qsl), B, H,
                                    float(scale), rng[0], rng[1], _p(out[rng[0] - t_lo:]), _p(lse[rng[0] - t_lo:]),
                                    ctypes.cast(keys, ctypes.c_void_p), _p(s))

    _parallel(run, _token_ranges(T, t_lo, t_hi, threads or default_threads()))
    return out, lse


def dcp_decode(q_nope, q_pe, kv_cache, block_table, seq_lens, qsl, D, r, scale, t_lo=0, t_hi=None,
               threads=None, lib=None):
    """Dense attention of DCP shard r of D, read through its paged cache.

    kv_cache uint16 [num_blocks, page_size, 576]; block_table int32 [B, W]
    (shard-local pages); seq_lens are global lengths.  Returns (out [n,H,512],
    lse [n,H], row_counts int32 [n]) for the n = t_hi - t_lo tokens [t_lo, t_hi).
    """
    lib = lib or load()
    q_nope, q_pe, kv_cache = _c(q_nope, np.uint16), _c(q_pe, np.uint16), _c(kv_cache, np.uint16)
    block_table, seq_lens, qsl = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(qsl, np.int32)
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    ps = kv_cache.shape[1]
    t_hi = T if t_hi is None else t_hi
    out = np.full((t_hi - t_lo, H, KV_LORA_RANK), np.nan)
    lse = np.full((t_hi - t_lo, H), np.nan)
    counts = np.full((t_hi - t_lo,), -1, dtype=np.int32)
    maxL = int(seq_lens.max()) if B else 0

    def run(rng):
        keys = (ctypes.c_void_p * max(1, maxL))()
        s = np.empty(max(1, maxL))
        o = rng[0] - t_lo
        lib.mla_oracle_dcp_decode(_p(q_nope), _p(q_pe), _p(kv_cache), ps, _p(block_table), block_table.shape[1],
                                  _p(seq_lens), _p(qsl), B, H, D, r, float(scale), rng[0], rng[1], _p(out[o:]),
                                  _p(lse[o:]), _p(counts[o:]), ctypes.cast(keys, ctypes.c_void_p), _p(s))

    _parallel(run, _token_ranges(T, t_lo, t_hi, threads or default_threads()))
    return out, lse, counts


def e4m3_to_double(code: int, lib=None) -> float:
    """Exact value of one FP8 E4M3 code (NaN for S.1111.111)."""
    return float((lib or load()).mla_oracle_e4m3_to_double(int(code) & 0xFF))


def dcp_decode_kv8(q_nope, q_pe, kv_cache, kv_scale, block_table, seq_lens, qsl, D, r, scale, t_lo=0, t_hi=None,
                   threads=None, lib=None):
    """dcp_decode over an FP8 E4M3 cache: kv_cache uint8 codes [num_blocks,
    page_size, 576], each value kv_scale * decode(code).  Returns (out [n,H,512],
    lse [n,H], row_counts int32 [n]) for tokens [t_lo, t_hi)."""
    lib = lib or load()
    q_nope, q_pe, kv_cache = _c(q_nope, np.uint16), _c(q_pe, np.uint16), _c(kv_cache, np.uint8)
    block_table, seq_lens, qsl = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(qsl, np.int32)
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    ps = kv_cache.shape[1]
    t_hi = T if t_hi is None else t_hi
    out = np.full((t_hi - t_lo, H, KV_LORA_RANK), np.nan)
    lse = np.full((t_hi - t_lo, H), np.nan)
    counts = np.full((t_hi - t_lo,), -1, dtype=np.int32)
    maxL = int(seq_lens.max()) if B else 0

    def run(rng):
        keys = (ctypes.c_void_p * max(1, maxL))()
        s = np.empty(max(1, maxL))
        o = rng[0] - t_lo
        lib.mla_oracle_dcp_decode_kv8(_p(q_nope), _p(q_pe), _p(kv_cache), float(kv_scale), ps, _p(block_table),
                                      block_table.shape[1], _p(seq_lens), _p(qsl), B, H, D, r, float(scale), rng[0],
                                      rng[1], _p(out[o:]), _p(lse[o:]), _p(counts[o:]),
                                      ctypes.cast(keys, ctypes.c_void_p), _p(s))

    _parallel(run, _token_ranges(T, t_lo, t_hi, threads or default_threads()))
    return out, lse, counts


def sparse_dcp_decode(q_nope, q_pe, kv_cache, block_table, seq_lens, qsl, topk, valid, D, r, scale, t_lo=0,
                      t_hi=None, threads=None, lib=None):
    """Sparse (top-k index list) attention of DCP shard r of D.

    topk int32 [T, K] global positions (-1 padded); valid int32 [T].  Returns
    (out [n,H,512], lse [n,H], local_counts int32 [n]) for tokens [t_lo, t_hi).
    """
    lib = lib or load()
    q_nope, q_pe, kv_cache = _c(q_nope, np.uint16), _c(q_pe, np.uint16), _c(kv_cache, np.uint16)
    block_table, seq_lens, qsl = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(qsl, np.int32)
    topk, valid = _c(topk, np.int32), _c(valid, np.int32)
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    K = topk.shape[1]
    ps = kv_cache.shape[1]
    t_hi = T if t_hi is None else t_hi
    out = np.full((t_hi - t_lo, H, KV_LORA_RANK), np.nan)
    lse = np.full((t_hi - t_lo, H), np.nan)
    counts = np.full((t_hi - t_lo,), -1, dtype=np.int32)

    def run(rng):
        keys = (ctypes.c_void_p * max(1, K))()
        s = np.empty(max(1, K))
        o = rng[0] - t_lo
        lib.mla_oracle_sparse_dcp_decode(_p(q_nope), _p(q_pe), _p(kv_cache), ps, _p(block_table),
                                         block_table.shape[1], _p(seq_lens), _p(qsl), B, H, _p(topk), K, _p(valid), D,
                                         r, float(scale), rng[0], rng[1], _p(out[o:]), _p(lse[o:]), _p(counts[o:]),
                                         ctypes.cast(keys, ctypes.c_void_p), _p(s))

    _parallel(run, _token_ranges(T, t_lo, t_hi, threads or default_threads()))
    return out, lse, counts


def lse_merge(partials, lses, valid_counts=None, lib=None):
    """LSE-weighted merge.  partials [D, T, H, W] (any float; widened to
    float64), lses [D, T, H], valid_counts int32 [D, T] or None.
    Returns (out float64 [T, H, W], lse float64 [T, H])."""
    lib = lib or load()
    partials = _c(partials, np.float64)
    lses = _c(lses, np.float64)
    D, T, H, W = partials.shape
    vc = None if valid_counts is None else _c(valid_counts, np.int32)
    out = np.empty((T, H, W))
    lse = np.empty((T, H))
    lib.mla_oracle_lse_merge(_p(partials), _p(lses), _p(vc), D, T, H, W, _p(out), _p(lse))
    return out, lse


def wuv_project(o, w_uv, lib=None):
    """y[t,h,:] = o[t,h,:] @ W_UV[h]; o float [T,H,512], w_uv uint16 (bf16 bits)
    [H, 512, V].  Returns float64 [T, H, V]."""
    lib = lib or load()
    o = _c(o, np.float64)
    w_uv = _c(w_uv, np.uint16)
    T, H, _ = o.shape
    V = w_uv.shape[2]
    y = np.empty((T, H, V))
    lib.mla_oracle_wuv_project(_p(o), _p(w_uv), T, H, V, _p(y))
    return y


def _parallel(fn, ranges):
    if len(ranges) <= 1:
        for r in ranges:
            fn(r)
        return
    with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
        list(ex.map(fn, ranges))
