"""Helpers shared by the GPU parity tests: run the fp64 oracle on a workload
and compare element by element.

Tolerances (written here once, used by every parity test):
  * outputs: |gpu - oracle| <= 1e-2 + 2e-2 * |oracle| element-wise (the
    allclose reading of "max-abs 1e-2 and max-rel 2e-2"), max-abs and
    max-rel reported on failure;
  * LSE: |gpu - oracle| <= 1e-3, and -inf exactly where the oracle is -inf;
  * counts: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mla_decode_attention_04_gb300 import workloads as wl

OUT_ATOL, OUT_RTOL, LSE_ATOL = 1e-2, 2e-2, 1e-3


class HostInputs:
    """Host copies (bf16 bit patterns / int32) of a workload's tensors."""

    def __init__(self, w):
        self.q_nope = wl.bf16_bits(w.q_nope)
        self.q_pe = wl.bf16_bits(w.q_pe)
        self.seq_lens = w.seq_lens.cpu().numpy()
        self.qsl = w.query_start_loc.cpu().numpy()
        self.caches = [wl.bf16_bits(s.cache) for s in w.shards]
        self.tables = [s.block_table.cpu().numpy() for s in w.shards]
        self.w_uv = None if w.w_uv is None else wl.bf16_bits(w.w_uv)
        self.topk = None if w.topk is None else w.topk.cpu().numpy()
        self.valid = None if w.topk_valid is None else w.topk_valid.cpu().numpy()
        self.D, self.scale = w.dcp_world, w.scale


def oracle_shard(h: HostInputs, r: int, t_lo=0, t_hi=None, sparse=False, threads=None):
    if sparse:
        return oracle.sparse_dcp_decode(h.q_nope, h.q_pe, h.caches[r], h.tables[r], h.seq_lens, h.qsl, h.topk, h.valid,
                                        h.D, r, h.scale, t_lo=t_lo, t_hi=t_hi, threads=threads)
    return oracle.dcp_decode(h.q_nope, h.q_pe, h.caches[r], h.tables[r], h.seq_lens, h.qsl, h.D, r, h.scale,
                             t_lo=t_lo, t_hi=t_hi, threads=threads)


def oracle_step(h: HostInputs, tokens=None, sparse=False, threads=None):
    """Per-shard results and the merged (and W_UV-projected) output for the
    given token indices (all tokens if None).  Returns dict of float64 arrays
    restricted to ``tokens``."""
    T = h.q_nope.shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    parts, lses, counts = [], [], []
    for r in range(h.D):
        ps, ls, cs = [], [], []
        for t in tokens:
            o, l, c = oracle_shard(h, r, int(t), int(t) + 1, sparse=sparse, threads=1)
            ps.append(o[0]), ls.append(l[0]), cs.append(c[0])
        parts.append(np.stack(ps)), lses.append(np.stack(ls)), counts.append(np.array(cs, np.int32))
    parts, lses, counts = np.stack(parts), np.stack(lses), np.stack(counts)
    merged, mlse = oracle.lse_merge(parts, lses, counts)
    out = oracle.wuv_project(merged, h.w_uv) if h.w_uv is not None else merged
    return dict(parts=parts, lses=lses, counts=counts, merged=merged, lse=mlse, out=out, tokens=tokens)


def oracle_step_threaded(h: HostInputs, tokens, sparse=False, threads=None):
    """Same as oracle_step but parallel over tokens (ctypes releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    tokens = list(tokens)
    n = threads or oracle.default_threads()
    chunks = [tokens[i::n] for i in range(n) if tokens[i::n]]
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        res = list(ex.map(lambda c: oracle_step(h, c, sparse=sparse), chunks))
    order = np.concatenate([r["tokens"] for r in res])
    inv = np.argsort(order)
    out = {}
    for k in ("parts", "lses", "counts"):
        out[k] = np.concatenate([r[k] for r in res], axis=1)[:, inv]
    for k in ("merged", "lse", "out"):
        out[k] = np.concatenate([r[k] for r in res], axis=0)[inv]
    out["tokens"] = order[inv]
    return out


_WORKLOAD_REFS = {}


def oracle_workload(name, w):
    """The oracle on every token of a named benchmark workload: each shard's
    (partial, lse, count) and the merged (and W_UV-projected) result.  The
    workloads are seeded, so the result is kept per name for the tests of
    both routes in one process."""
    if name not in _WORKLOAD_REFS:
        ref = oracle_step_threaded(HostInputs(w), range(w.num_tokens), sparse=w.topk is not None)
        _WORKLOAD_REFS[name] = ref
    return _WORKLOAD_REFS[name]


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ref)
    if bad.any():
        rel = err / np.maximum(np.abs(ref), 1e-30)
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; max abs {err.max():.3e}, "
                             f"max rel {rel.max():.3e}; first bad {idx}")


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern differs"
    fin = ~ninf
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        assert err.max() <= LSE_ATOL, f"{what}: max lse error {err.max():.3e}"


def to_np(t):
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def oracle_step_kv8(h: HostInputs, caches8, kv_scale, tokens=None):
    """oracle_step over FP8 shard caches (uint8 E4M3 codes, value = kv_scale *
    decode(code)), parallel over tokens."""
    from concurrent.futures import ThreadPoolExecutor
    T = h.q_nope.shape[0]
    tokens = list(range(T)) if tokens is None else list(tokens)
    n = oracle.default_threads()
    chunks = [tokens[i::n] for i in range(n) if tokens[i::n]]

    def run(chunk):
        parts, lses, counts = [], [], []
        for r in range(h.D):
            ps, ls, cs = [], [], []
            for t in chunk:
                o, l, c = oracle.dcp_decode_kv8(h.q_nope, h.q_pe, caches8[r], kv_scale, h.tables[r], h.seq_lens, h.qsl,
                                                h.D, r, h.scale, t_lo=t, t_hi=t + 1, threads=1)
                ps.append(o[0]), ls.append(l[0]), cs.append(c[0])
            parts.append(np.stack(ps)), lses.append(np.stack(ls)), counts.append(np.array(cs, np.int32))
        return np.stack(parts), np.stack(lses), np.stack(counts)

    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        res = list(ex.map(run, chunks))
    order = np.concatenate([np.asarray(c) for c in chunks])
    inv = np.argsort(order)
    parts = np.concatenate([r[0] for r in res], axis=1)[:, inv]
    lses = np.concatenate([r[1] for r in res], axis=1)[:, inv]
    counts = np.concatenate([r[2] for r in res], axis=1)[:, inv]
    merged, mlse = oracle.lse_merge(parts, lses, counts)
    out = oracle.wuv_project(merged, h.w_uv) if h.w_uv is not None else merged
    return dict(parts=parts, lses=lses, counts=counts, merged=merged, lse=mlse, out=out)
