"""Checks that pin the fp64 oracle to facts outside itself.

Each ``check_*`` takes a loaded oracle library (``oracle.load()`` or a
deliberately broken build) and raises AssertionError when the oracle
disagrees with:
  * the mask tables and the seqlen_k example printed on the page
    "[Attention] add DCP support for FLASH_ATTN_MLA backend" (review thread),
    stored under tests/golden/;
  * closed forms (floor formula for visible counts, two-key sigmoid,
    zero-query mean, identical keys);
  * library routines (torch scaled_dot_product_attention and logsumexp in
    float64, numpy einsum);
  * invariants the pages state: the LSE-weighted merge over the D shards
    reproduces unsharded attention, and W_UV commutes with the merge
    ("[Attention] DCP sparse MLA output-merge optimizations", summary);
  * brute force on tiny inputs.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from mla_decode_attention_04_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits(t):
    return wl.bf16_bits(t)


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


# ------------------------------------------------------------------ golden


def read_mask_tables():
    tables, cur = [], None
    with open(os.path.join(GOLDEN, "dcp_mask_seq6_q4_d2.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("table"):
                _, name, _, D, _, r = line.split()
                cur = dict(name=name, D=int(D), r=int(r), rows={})
                tables.append(cur)
            elif line.startswith("keys"):
                cur["keys"] = [int(x) for x in line.split()[1:]]
            else:
                q, vals = line.split(":")
                cur["rows"][int(q)] = [int(x) for x in vals.split()]
    return tables


def read_seqlen_example():
    out = {}
    with open(os.path.join(GOLDEN, "dcp_seqlen_k_q2_d2.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("seq_len"):
                p = line.split()
                out["L"], out["q"], out["D"] = int(p[1]), int(p[3]), int(p[5])
            else:
                r, vals = line.split(":")
                out.setdefault("ranks", {})[int(r.split()[1])] = [int(x) for x in vals.split()]
    return out


def check_mask_tables(lib):
    L, q_len = 6, 4
    for tab in read_mask_tables():
        D, r = tab["D"], tab["r"]
        # the listed columns are the shard's tokens, in local order
        assert oracle.local_len(L, D, r, lib=lib) == len(tab["keys"]), tab["name"]
        for i, row in tab["rows"].items():
            P = L - q_len + i
            got = [int(oracle.key_visible(P, D, r, j, lib=lib)) for j in range(len(tab["keys"]))]
            assert got == row, (tab["name"], i, got, row)
            assert oracle.visible_count(P, L, D, r, lib=lib) == sum(row), (tab["name"], i)


def check_seqlen_example(lib):
    ex = read_seqlen_example()
    for r, want in ex["ranks"].items():
        got = [oracle.visible_count(ex["L"] - ex["q"] + i, ex["L"], ex["D"], r, lib=lib) for i in range(ex["q"])]
        assert got == want, (r, got, want)


def check_count_closed_form(lib):
    # floor formula and partition of the prefix over the shards
    for D in range(1, 9):
        for L in range(0, 40):
            for r in range(D):
                want = (L - r - 1) // D + 1 if L > r else 0
                assert oracle.local_len(L, D, r, lib=lib) == want, (L, D, r)
            for P in range(max(0, L - 8), L):
                tot = 0
                for r in range(D):
                    n = oracle.visible_count(P, L, D, r, lib=lib)
                    assert n == ((P - r) // D + 1 if P >= r else 0), (P, L, D, r, n)
                    tot += n
                assert tot == P + 1


# --------------------------------------------------------------- attention


def _dense_inputs(seq_lens, q_lens, H=2, D=1, seed=0, q_std=0.3, ps=4, topk=None):
    return wl.custom(seq_lens, q_lens, H, D, page_size=ps, seed=seed, q_std=q_std, topk=topk)


def _run_shard(w, r, lib):
    sh = w.shards[r]
    return oracle.dcp_decode(_bits(w.q_nope), _bits(w.q_pe), _bits(sh.cache), sh.block_table.numpy(),
                             w.seq_lens.numpy(), w.query_start_loc.numpy(), w.dcp_world, r, w.scale, lib=lib,
                             threads=1)


def _run_dense(w, lib):
    return oracle.causal_dense(_bits(w.q_nope), _bits(w.q_pe), _bits(w.kv_logical), w.kv_start.numpy(),
                               w.seq_lens.numpy(), w.query_start_loc.numpy(), w.scale, lib=lib, threads=1)


def check_sdpa_d1(lib):
    """D=1 reduces to textbook bottom-right causal attention over q=[q_nope|q_pe],
    k=[kv_c|k_pe], v=kv_c: compare with torch SDPA in float64."""
    w = _dense_inputs([5, 9, 3], [2, 3, 3], H=3, D=1, seed=3)
    out, lse, counts = _run_shard(w, 0, lib)
    qsl = w.query_start_loc.numpy()
    for b, L in enumerate(w.seq_lens.tolist()):
        t0, t1 = qsl[b], qsl[b + 1]
        ql = t1 - t0
        q = torch.cat([w.q_nope[t0:t1], w.q_pe[t0:t1]], dim=-1).to(torch.float64).transpose(0, 1)  # [H, q, 576]
        kv = w.kv_logical[int(w.kv_start[b]):int(w.kv_start[b]) + L].to(torch.float64)
        k = kv.unsqueeze(0).expand(q.shape[0], L, 576)
        v = kv[:, :512].unsqueeze(0).expand(q.shape[0], L, 512)
        pos = torch.arange(L - ql, L).unsqueeze(1)
        mask = torch.arange(L).unsqueeze(0) <= pos  # [q, L]
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=w.scale)
        logits = (q @ k.transpose(-1, -2)) * w.scale
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)  # [H, q]
        np.testing.assert_allclose(out[t0:t1], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t0:t1], ref_lse.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        assert counts[t0:t1].tolist() == (pos.squeeze(1) + 1).tolist()


def check_two_key_closed_form(lib):
    """Two visible keys: weight of key 1 is the logistic of s1 - s0."""
    w = _dense_inputs([2], [1], H=2, D=1, seed=5, q_std=1.0)
    out, lse, _ = _run_shard(w, 0, lib)
    kv = _f64(w.kv_logical)
    q = np.concatenate([_f64(w.q_nope), _f64(w.q_pe)], -1)[0]  # [H, 576]
    for h in range(2):
        s0 = w.scale * float(np.dot(q[h], kv[0]))
        s1 = w.scale * float(np.dot(q[h], kv[1]))
        p1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(out[0, h], (1 - p1) * kv[0, :512] + p1 * kv[1, :512], rtol=0, atol=1e-12)
        assert abs(lse[0, h] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-12


def check_zero_query_mean(lib):
    """q = 0: every score is 0, so LSE = ln(n visible) and the output is the mean
    of the visible kv_c rows -- per shard, which pins the mask through values."""
    w = _dense_inputs([6, 11], [4, 3], H=2, D=3, seed=7, ps=2)
    w.q_nope.zero_()
    w.q_pe.zero_()
    kv = _f64(w.kv_logical)
    qsl = w.query_start_loc.numpy()
    for r in range(3):
        out, lse, counts = _run_shard(w, r, lib)
        for b, L in enumerate(w.seq_lens.tolist()):
            for i in range(qsl[b + 1] - qsl[b]):
                t = qsl[b] + i
                P = L - (qsl[b + 1] - qsl[b]) + i
                vis = [p for p in range(r, L, 3) if p <= P]  # brute force
                assert counts[t] == len(vis)
                if not vis:
                    assert np.all(lse[t] == -np.inf) and np.all(out[t] == 0.0)
                    continue
                mean = kv[int(w.kv_start[b]) + np.array(vis), :512].mean(0)
                np.testing.assert_allclose(out[t], np.broadcast_to(mean, out[t].shape), rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[t], math.log(len(vis)), rtol=0, atol=1e-12)


def check_identical_keys(lib):
    """All keys equal: the output is that key's kv_c for any query."""
    w = _dense_inputs([7], [3], H=2, D=1, seed=9, q_std=1.0)
    w.kv_logical[:] = w.kv_logical[0]
    sh = w.shards[0]
    sh.cache[:] = w.kv_logical[0]
    out, lse, _ = _run_shard(w, 0, lib)
    c = _f64(w.kv_logical[0, :512])
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-12)


def check_paged_equals_logical(lib):
    """D=1 through the paged cache equals the logical-sequence route."""
    w = _dense_inputs([13, 4, 9], [1, 4, 2], H=2, D=1, seed=11, ps=4)
    out, lse, _ = _run_shard(w, 0, lib)
    ref, ref_lse = _run_dense(w, lib)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-13)


def check_shard_merge_equals_unsharded(lib):
    """LSE-merge of the D shard results equals unsharded causal attention."""
    for D in (1, 2, 4, 8):
        w = _dense_inputs([3, 17, 26, 9], [3, 1, 4, 2], H=2, D=D, seed=20 + D, ps=2, q_std=1.0)
        parts, lses, counts = zip(*[_run_shard(w, r, lib) for r in range(D)])
        merged, mlse = oracle.lse_merge(np.stack(parts), np.stack(lses), np.stack(counts), lib=lib)
        ref, ref_lse = _run_dense(w, lib)
        np.testing.assert_allclose(merged, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(mlse, ref_lse, rtol=0, atol=1e-12)
        merged2, _ = oracle.lse_merge(np.stack(parts), np.stack(lses), None, lib=lib)
        np.testing.assert_allclose(merged2, ref, rtol=0, atol=1e-12)


def check_merge_lse_logsumexp(lib):
    """Merged LSE equals a library logsumexp over the shards that take part."""
    rng = np.random.default_rng(1)
    D, T, H, W = 5, 4, 3, 8
    parts = rng.standard_normal((D, T, H, W))
    lses = rng.standard_normal((D, T, H)) * 3
    counts = rng.integers(0, 3, size=(D, T)).astype(np.int32)
    counts[:, 0] = 0  # token 0: no shard takes part
    out, lse = oracle.lse_merge(parts, lses, counts, lib=lib)
    for t in range(T):
        use = counts[:, t] > 0
        if not use.any():
            assert np.all(lse[t] == -np.inf) and np.all(out[t] == 0)
            continue
        ref = torch.logsumexp(torch.from_numpy(lses[use, t]), dim=0).numpy()
        np.testing.assert_allclose(lse[t], ref, rtol=0, atol=1e-12)
        wts = np.exp(lses[use, t] - ref)  # [n, H]
        np.testing.assert_allclose(out[t], np.einsum("nh,nhw->hw", wts, parts[use, t]), rtol=0, atol=1e-12)


def check_merge_ignores_empty_shards(lib):
    """Shard rows with valid count 0 are not read: NaN partials behind them
    change nothing; a row with every shard empty is 0 with LSE -inf."""
    w = _dense_inputs([2, 9], [2, 3], H=2, D=2, seed=31, ps=2)
    parts, lses, counts = [np.stack(x) for x in zip(*[_run_shard(w, r, lib) for r in range(2)])]
    assert (counts == 0).any()  # seq_len 2, q_len 2, D=2: q_A has no key on rank 1
    clean, clean_lse = oracle.lse_merge(parts, lses, counts, lib=lib)
    poisoned = parts.copy()
    plse = lses.copy()
    for r in range(2):
        for t in range(parts.shape[1]):
            if counts[r, t] == 0:
                poisoned[r, t] = np.nan
                plse[r, t] = np.nan
    out, lse = oracle.lse_merge(poisoned, plse, counts, lib=lib)
    np.testing.assert_array_equal(out, clean)
    np.testing.assert_array_equal(lse, clean_lse)
    none = np.zeros_like(counts)
    out0, lse0 = oracle.lse_merge(poisoned, plse, none, lib=lib)
    assert np.all(out0 == 0) and np.all(lse0 == -np.inf)


def check_empty_row(lib):
    """A query with no visible key on a shard gives LSE -inf and output 0."""
    w = _dense_inputs([2], [2], H=2, D=2, seed=2, ps=1)
    out, lse, counts = _run_shard(w, 1, lib)
    assert counts.tolist() == [0, 1]
    assert np.all(lse[0] == -np.inf) and np.all(out[0] == 0.0)
    assert np.all(np.isfinite(lse[1])) and np.all(np.isfinite(out[1]))


def check_wuv_library(lib):
    rng = np.random.default_rng(3)
    T, H, V = 3, 2, 16
    o = rng.standard_normal((T, H, 512))
    w = torch.randn(H, 512, V, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    y = oracle.wuv_project(o, _bits(w), lib=lib)
    np.testing.assert_allclose(y, np.einsum("thd,hdv->thv", o, _f64(w)), rtol=1e-13, atol=1e-12)


def check_wuv_commutes(lib):
    """Projecting each shard's partial through W_UV and then merging equals
    merging and then projecting."""
    w = _dense_inputs([5, 12, 30], [2, 1, 3], H=2, D=4, seed=41, ps=4)
    wuv = torch.randn(2, 512, 128, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    parts, lses, counts = [np.stack(x) for x in zip(*[_run_shard(w, r, lib) for r in range(4)])]
    merged, _ = oracle.lse_merge(parts, lses, counts, lib=lib)
    after = oracle.wuv_project(merged, _bits(wuv), lib=lib)
    proj = np.stack([oracle.wuv_project(parts[r], _bits(wuv), lib=lib) for r in range(4)])
    before, _ = oracle.lse_merge(proj, lses, counts, lib=lib)
    np.testing.assert_allclose(before, after, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ sparse


def _run_sparse(w, r, lib, topk=None, valid=None):
    sh = w.shards[r]
    topk = w.topk.numpy() if topk is None else topk
    valid = w.topk_valid.numpy() if valid is None else valid
    return oracle.sparse_dcp_decode(_bits(w.q_nope), _bits(w.q_pe), _bits(sh.cache), sh.block_table.numpy(),
                                    w.seq_lens.numpy(), w.query_start_loc.numpy(), topk, valid, w.dcp_world, r,
                                    w.scale, lib=lib, threads=1)


def check_sparse_full_prefix_is_dense(lib):
    """Index lists holding the whole visible prefix reproduce dense causal
    attention after the merge, and each shard count equals the dense count."""
    D = 3
    w = _dense_inputs([7, 12], [3, 2], H=2, D=D, seed=51, ps=2, q_std=1.0)
    T = w.num_tokens
    K = 12
    topk = np.full((T, K), -1, np.int32)
    valid = np.zeros(T, np.int32)
    qsl = w.query_start_loc.numpy()
    rng = np.random.default_rng(0)
    for b, L in enumerate(w.seq_lens.tolist()):
        ql = qsl[b + 1] - qsl[b]
        for i in range(ql):
            P = L - ql + i
            topk[qsl[b] + i, :P + 1] = rng.permutation(P + 1)
            valid[qsl[b] + i] = P + 1
    res = [_run_sparse(w, r, lib, topk, valid) for r in range(D)]
    dense = [_run_shard(w, r, lib) for r in range(D)]
    for r in range(D):
        assert res[r][2].tolist() == dense[r][2].tolist()
    parts, lses, counts = [np.stack(x) for x in zip(*res)]
    merged, mlse = oracle.lse_merge(parts, lses, counts, lib=lib)
    ref, ref_lse = _run_dense(w, lib)
    np.testing.assert_allclose(merged, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(mlse, ref_lse, rtol=0, atol=1e-12)


def check_sparse_subset(lib):
    """A sparse list equals dense attention over a sequence made of exactly the
    listed keys (a one-query request that sees all of them); counts by brute
    force; padding, entries past the valid count and past the query position
    are ignored."""
    D = 2
    w = _dense_inputs([20, 9], [2, 1], H=2, D=D, seed=61, ps=4, q_std=1.0)
    T, K = w.num_tokens, 8
    rng = np.random.default_rng(5)
    topk = np.full((T, K), -1, np.int32)
    valid = np.array([6, 8, 5], np.int32)
    qsl = w.query_start_loc.numpy()
    for b, L in enumerate(w.seq_lens.tolist()):
        ql = qsl[b + 1] - qsl[b]
        for i in range(ql):
            t = qsl[b] + i
            P = L - ql + i
            n = min(K, P + 1)
            topk[t, :n] = rng.choice(P + 1, n, replace=False)
    topk[0, 2] = -1            # padding inside the valid range
    topk[0, 5] = 19            # token 0 sits at position 18: key 19 is in its future, ignored
    topk[1, 6] = 25            # beyond the sequence: ignored
    kv = w.kv_logical
    for r in range(D):
        out, lse, counts = _run_sparse(w, r, lib, topk, valid)
        for b, L in enumerate(w.seq_lens.tolist()):
            ql = qsl[b + 1] - qsl[b]
            for i in range(ql):
                t = qsl[b] + i
                P = L - ql + i
                keep = [int(p) for p in topk[t, :valid[t]] if 0 <= p <= P and p % D == r]
                assert counts[t] == len(keep), (r, t)
                if not keep:
                    assert np.all(lse[t] == -np.inf) and np.all(out[t] == 0)
                    continue
                sub = kv[int(w.kv_start[b]) + torch.tensor(keep)]
                ref, ref_lse = oracle.causal_dense(_bits(w.q_nope[t:t + 1]), _bits(w.q_pe[t:t + 1]), _bits(sub),
                                                   np.array([0]), np.array([len(keep)], np.int32),
                                                   np.array([0, 1], np.int32), w.scale, lib=lib, threads=1)
                np.testing.assert_allclose(out[t], ref[0], rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[t], ref_lse[0], rtol=0, atol=1e-12)


def two_stage_lists(w):
    """Index lists of the two-stage decomposition: per query token, the
    request's context [0, L - q_len) (every query row sees all of it) and its
    q_len new positions [L - q_len, L) (a row keeps those <= its own
    position, i.e. the causal part).  Returns (ctx, ctx_valid, new, new_valid)."""
    L = w.seq_lens.numpy()
    qsl = w.query_start_loc.numpy()
    T = w.num_tokens
    K = int(max(1, L.max()))
    ctx = np.full((T, K), -1, np.int32)
    new = np.full((T, K), -1, np.int32)
    ctx_valid = np.zeros(T, np.int32)
    new_valid = np.zeros(T, np.int32)
    for b in range(len(L)):
        ql = int(qsl[b + 1] - qsl[b])
        c = int(L[b]) - ql
        for t in range(qsl[b], qsl[b + 1]):
            ctx[t, :c] = np.arange(c)
            ctx_valid[t] = c
            new[t, :ql] = np.arange(c, c + ql)
            new_valid[t] = ql
    return ctx, ctx_valid, new, new_valid


def check_two_stage_decomposition(lib):
    """A non-causal pass over the context keys plus a causal pass over the
    q_len new keys, merged by LSE over both passes and every shard, is the
    one-pass causal attention: the two-stage alternative to a custom mask
    offered in the review thread of "[Attention] add DCP support for
    FLASH_ATTN_MLA backend" (context keys with causal off, the query's own
    keys with causal on)."""
    for D in (1, 2, 3):
        w = _dense_inputs([9, 14, 5, 3], [3, 4, 1, 3], H=2, D=D, seed=71 + D, ps=2, q_std=1.0)
        ctx, ctx_valid, new, new_valid = two_stage_lists(w)
        res = []
        for r in range(D):
            res.append(_run_sparse(w, r, lib, ctx, ctx_valid))
            res.append(_run_sparse(w, r, lib, new, new_valid))
        parts, lses, counts = [np.stack(x) for x in zip(*res)]
        merged, mlse = oracle.lse_merge(parts, lses, counts, lib=lib)
        ref, ref_lse = _run_dense(w, lib)
        np.testing.assert_allclose(merged, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(mlse, ref_lse, rtol=0, atol=1e-12)
        # the passes split every row's visible keys: counts add up to P + 1
        assert (counts.sum(axis=0) == [P + 1 for P in _positions(w)]).all()


def _positions(w):
    L = w.seq_lens.numpy()
    qsl = w.query_start_loc.numpy()
    out = []
    for b in range(len(L)):
        ql = int(qsl[b + 1] - qsl[b])
        out += [int(L[b]) - ql + i for i in range(ql)]
    return out


# ----------------------------------------------------------- FP8 cache


def check_e4m3_decode_library(lib):
    """Every FP8 E4M3 code decodes to torch's float8_e4m3fn value (NaN for
    S.1111.111, signed zero, the subnormals at exponent 0, 448 at the top)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c, lib=lib) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def _fp8_case(kv_scale, seed):
    w = _dense_inputs([9, 70, 33], [2, 1, 3], H=3, D=2, seed=seed, ps=8)
    codes, views = wl.fp8_cache(w, kv_scale)
    # the bf16 cache holding exactly kv_scale * decode(code) (an E4M3 value
    # has at most 4 significant bits, times 1 or 0.75 at most 6: exact in bf16)
    twin = (wl.e4m3_values(codes) * kv_scale).to(torch.bfloat16)
    return w, views, twin


def check_kv8_reduces_to_bf16(lib):
    """The FP8 shard decode equals the (pinned) bf16 shard decode on a bf16
    cache holding the dequantised values, for kv_scale 1 and 0.75."""
    for kv_scale, seed in ((1.0, 11), (0.75, 12)):
        w, views, twin = _fp8_case(kv_scale, seed)
        for r, sh in enumerate(w.shards):
            tw = twin[sh.page_base:sh.page_base + sh.cache.shape[0]]
            args = (w.seq_lens.numpy(), w.query_start_loc.numpy(), w.dcp_world, r, w.scale)
            o8, l8, c8 = oracle.dcp_decode_kv8(_bits(w.q_nope), _bits(w.q_pe), views[r].numpy(), kv_scale,
                                              sh.block_table.numpy(), *args, lib=lib, threads=1)
            ob, lb, cb = oracle.dcp_decode(_bits(w.q_nope), _bits(w.q_pe), _bits(tw), sh.block_table.numpy(), *args,
                                           lib=lib, threads=1)
            assert np.array_equal(c8, cb)
            assert np.array_equal(np.isneginf(l8), np.isneginf(lb))
            np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-12)
            fin = np.isfinite(lb)
            np.testing.assert_allclose(l8[fin], lb[fin], rtol=0, atol=1e-12)


def check_kv8_zero_query(lib):
    """q = 0 over an FP8 cache: LSE = ln(n visible), output = kv_scale times
    the mean of the decoded visible kv_c rows (decoded here by torch)."""
    kv_scale = 0.5
    w, views, _ = _fp8_case(kv_scale, 13)
    w.q_nope.zero_()
    w.q_pe.zero_()
    codes, _ = wl.fp8_cache(w, kv_scale)
    vals = wl.e4m3_values(codes).double().numpy()
    qsl = w.query_start_loc.numpy()
    for r, sh in enumerate(w.shards):
        out, lse, counts = oracle.dcp_decode_kv8(_bits(w.q_nope), _bits(w.q_pe), views[r].numpy(), kv_scale,
                                                 sh.block_table.numpy(), w.seq_lens.numpy(), qsl, 2, r, w.scale,
                                                 lib=lib, threads=1)
        bt = sh.block_table.numpy()
        for b, L in enumerate(w.seq_lens.tolist()):
            for i in range(qsl[b + 1] - qsl[b]):
                t = qsl[b] + i
                P = L - (qsl[b + 1] - qsl[b]) + i
                vis = [p // 2 for p in range(r, L, 2) if p <= P]  # local slots, brute force
                assert counts[t] == len(vis)
                if not vis:
                    assert np.all(np.isneginf(lse[t])) and np.all(out[t] == 0.0)
                    continue
                rows = np.stack([vals[sh.page_base + bt[b, j // 8], j % 8, :512] for j in vis])
                np.testing.assert_allclose(out[t], np.broadcast_to(kv_scale * rows.mean(0), out[t].shape), rtol=0,
                                           atol=1e-12)
                np.testing.assert_allclose(lse[t], math.log(len(vis)), rtol=0, atol=1e-12)


ALL_CHECKS = [
    check_mask_tables, check_seqlen_example, check_count_closed_form, check_sdpa_d1, check_two_key_closed_form,
    check_zero_query_mean, check_identical_keys, check_paged_equals_logical, check_shard_merge_equals_unsharded,
    check_merge_lse_logsumexp, check_merge_ignores_empty_shards, check_empty_row, check_wuv_library,
    check_wuv_commutes, check_sparse_full_prefix_is_dense, check_sparse_subset, check_two_stage_decomposition,
    check_e4m3_decode_library, check_kv8_reduces_to_bf16, check_kv8_zero_query,
]
