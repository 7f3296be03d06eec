"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Counts bit-exact; outputs within 1e-2 + 2e-2*|ref| element-wise; LSE within
1e-3 (see parity_utils).  Every case compares every element, the benchmark
workloads at full size included (in the launch configuration the benchmark
times).
"""
import math

import numpy as np
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build
from mla_decode_attention_04_gb300 import pipeline
from mla_decode_attention_04_gb300 import workloads as wl
from parity_utils import (HostInputs, assert_lse_close, assert_out_close, oracle_shard, oracle_step,
                          oracle_workload, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mla_build.build()
    mla.load_library()


def _shard_calls(w, out_dtype=torch.bfloat16, num_splits=0):
    res = []
    for r, s in enumerate(w.shards):
        out, lse, cnt = mla.mla_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc,
                                           w.max_query_len, w.max_seq_len, w.dcp_world, r, w.scale,
                                           out_dtype=out_dtype, num_splits=num_splits)
        res.append((out, lse, cnt))
    torch.cuda.synchronize()
    return res


def _check_shards(w, res, h=None, sparse=False):
    h = h or HostInputs(w)
    for r, (out, lse, cnt) in enumerate(res):
        ro, rl, rc = oracle_shard(h, r, sparse=sparse)
        assert cnt.cpu().numpy().tolist() == rc.tolist(), f"shard {r} counts"
        assert_out_close(to_np(out), ro, f"shard {r} out")
        assert_lse_close(to_np(lse), rl, f"shard {r} lse")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_tiny_shards(out_dtype, num_splits):
    w = wl.tiny().to("cuda")
    _check_shards(w, _shard_calls(w, out_dtype, num_splits))


def test_tiny_step_with_wuv():
    w = wl.tiny().to("cuda")
    step = pipeline.step_for_workload(w)
    out, lse = step.run()
    torch.cuda.synchronize()
    ref = oracle_step(HostInputs(w))
    assert step.counts.cpu().numpy().tolist() == ref["counts"].tolist()
    assert_out_close(to_np(out), ref["out"], "merged W_UV output")
    assert_lse_close(to_np(lse), ref["lse"], "merged lse")


def test_tiny_step_without_wuv_bf16_partials():
    w = wl.tiny().to("cuda")
    w.w_uv = None
    step = pipeline.step_for_workload(w, partial_dtype=torch.bfloat16)
    out, lse = step.run()
    torch.cuda.synchronize()
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["out"], "merged output")
    assert_lse_close(to_np(lse), ref["lse"], "merged lse")


EDGE = {
    "shard_without_tokens": dict(seq_lens=[1, 3, 2], q_lens=[1, 2, 2], num_heads=16, dcp_world=4, page_size=16),
    "prefill_from_empty": dict(seq_lens=[5, 70], q_lens=[5, 70], num_heads=4, dcp_world=2, page_size=8),
    "empty_request": dict(seq_lens=[10, 7, 12, 1], q_lens=[2, 0, 1, 1], num_heads=16, dcp_world=2, page_size=16),
    "page_32": dict(seq_lens=[100, 257], q_lens=[3, 1], num_heads=16, dcp_world=3, page_size=32),
    "page_128": dict(seq_lens=[1000, 129], q_lens=[1, 4], num_heads=8, dcp_world=2, page_size=128),
    "heads_1": dict(seq_lens=[300, 50], q_lens=[1, 1], num_heads=1, dcp_world=1, page_size=64),
    "heads_17_ragged_groups": dict(seq_lens=[77, 130], q_lens=[3, 2], num_heads=17, dcp_world=2, page_size=16),
    "heads_128": dict(seq_lens=[200, 65], q_lens=[2, 1], num_heads=128, dcp_world=8, page_size=64),
    "many_splits": dict(seq_lens=[9000], q_lens=[3], num_heads=16, dcp_world=2, page_size=64),
    "d8_ragged_shards": dict(seq_lens=[1001, 64, 7], q_lens=[2, 1, 7], num_heads=16, dcp_world=8, page_size=16),
    # 64-row units in gangs of 3 CTAs, requests with 1, 2 or 3 row groups
    "gangs_mixed_groups": dict(seq_lens=[900, 40, 2000, 7, 1500], q_lens=[3, 1, 2, 3, 3], num_heads=64, dcp_world=2,
                               page_size=32),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_shapes(name):
    w = wl.custom(seed=sorted(EDGE).index(name), **EDGE[name]).to("cuda")
    _check_shards(w, _shard_calls(w, torch.float32))


def test_fused_query_strides():
    """q_nope / q_pe as views of one [T, H, 576] query (row stride 576)."""
    w = wl.tiny().to("cuda")
    q = torch.cat([w.q_nope, w.q_pe], dim=-1).contiguous()
    w.q_nope, w.q_pe = q[..., :512], q[..., 512:]
    _check_shards(w, _shard_calls(w))


def test_unused_block_table_entries_are_not_read():
    """Entries past a request's pages do not change anything."""
    w = wl.custom([40, 300], [2, 1], 16, 2, page_size=16, seed=5).to("cuda")
    base = _shard_calls(w, torch.float32)
    for r, s in enumerate(w.shards):
        for b, L in enumerate(w.seq_lens.tolist()):
            pages = -(-len(range(r, L, w.dcp_world)) // w.page_size)
            s.block_table[b, pages:] = 10 ** 6  # out of range: would be flagged (and change results) if read
    res = _shard_calls(w, torch.float32)
    for (o0, l0, c0), (o1, l1, c1) in zip(base, res):
        assert torch.equal(o0, o1) and torch.equal(l0, l1) and torch.equal(c0, c1)


def test_device_check_flags_bad_page_without_faulting():
    """A page id past the cache is reported in the status word; the access is skipped."""
    w = wl.custom([200], [1], 16, 1, page_size=16, seed=3).to("cuda")
    s = w.shards[0]
    s.block_table[0, 2] = s.cache.shape[0] + 7
    ws = torch.empty(mla.decode_workspace_size(1, 1, 16, 1, 200, 1), dtype=torch.uint8, device="cuda")
    mla.mla_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc, 1, 200, 1, 0, w.scale,
                       workspace=ws)
    rc, detail = mla.workspace_status(ws)
    assert rc == mla.MLA_ERR_DEVICE_CHECK and detail == 1
    # a clean call resets the word
    s.block_table[0, 2] = 0
    mla.mla_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc, 1, 200, 1, 0, w.scale,
                       workspace=ws)
    assert mla.workspace_status(ws) == (mla.MLA_OK, 0)


# ------------------------------------------------------------------- merge


@pytest.mark.parametrize("wuv", [False, True])
@pytest.mark.parametrize("partial_dtype", [torch.float32, torch.bfloat16])
def test_merge_against_oracle_with_poisoned_empty_rows(wuv, partial_dtype):
    import oracle
    g = torch.Generator().manual_seed(7)
    D, T, H = 4, 37, 16
    parts = torch.randn(D, T, H, 512, generator=g).to(partial_dtype)
    lses = torch.randn(D, T, H, generator=g) * 2
    counts = torch.randint(0, 3, (D, T), generator=g, dtype=torch.int32)
    counts[:, 5] = 0
    poisoned = parts.clone()
    plse = lses.clone()
    for r in range(D):
        for t in range(T):
            if counts[r, t] == 0:
                poisoned[r, t] = float("nan")
                plse[r, t] = float("nan")
    w_uv = torch.randn(H, 512, 128, generator=g).to(torch.bfloat16) if wuv else None
    out, lse = mla.dcp_lse_merge(poisoned.cuda(), plse.cuda(), counts.cuda(), None if w_uv is None else w_uv.cuda())
    torch.cuda.synchronize()
    ref, ref_lse = oracle.lse_merge(parts.double().numpy(), lses.double().numpy(), counts.numpy())
    if wuv:
        ref = oracle.wuv_project(ref, wl.bf16_bits(w_uv))
    assert_out_close(to_np(out), ref, "merge")
    assert_lse_close(to_np(lse), ref_lse, "merge lse")
    assert torch.all(out[5] == 0) and torch.all(torch.isneginf(lse[5]))


def test_merge_without_counts_uses_neg_inf_lse():
    import oracle
    g = torch.Generator().manual_seed(8)
    D, T, H = 3, 9, 4
    parts = torch.randn(D, T, H, 512, generator=g)
    lses = torch.randn(D, T, H, generator=g)
    lses[1, :4] = -math.inf
    lses[:, 7] = -math.inf
    out, lse = mla.dcp_lse_merge(parts.cuda(), lses.cuda(), None, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.lse_merge(parts.double().numpy(), lses.double().numpy(), None)
    assert_out_close(to_np(out), ref, "merge")
    assert_lse_close(to_np(lse), ref_lse, "merge lse")


# ------------------------------------------------------------------ sparse


def _sparse_calls(w):
    res = []
    for r, s in enumerate(w.shards):
        res.append(mla.mla_sparse_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc,
                                             w.topk, w.topk_valid, w.dcp_world, r, w.scale, out_dtype=torch.float32))
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("H,D,K", [(16, 2, 64), (24, 3, 100), (64, 4, 256), (1, 1, 7)])
def test_sparse_small(H, D, K):
    w = wl.custom([300, 90, 700, 45], [2, 1, 4, 3], H, D, page_size=16, seed=H + D + K, topk=K,
                  short_valid_frac=0.3, force_zero_valid=1).to("cuda")
    _check_shards(w, _sparse_calls(w), sparse=True)


def test_sparse_step_with_wuv():
    w = wl.custom([300, 90, 700, 45], [2, 1, 4, 3], 64, 4, page_size=64, seed=11, topk=128, short_valid_frac=0.3,
                  force_zero_valid=1).to("cuda")
    step = pipeline.step_for_workload(w)
    out, lse = step.run()
    torch.cuda.synchronize()
    ref = oracle_step(HostInputs(w), sparse=True)
    assert step.counts.cpu().numpy().tolist() == ref["counts"].tolist()
    assert_out_close(to_np(out), ref["out"], "sparse merged W_UV output")
    assert_lse_close(to_np(lse), ref["lse"], "sparse merged lse")


# ------------------------------------------------------------- CUDA graphs


def test_graph_replay_matches_eager():
    w = wl.custom([500, 1300, 80], [2, 1, 2], 16, 4, page_size=64, seed=21).to("cuda")
    step = pipeline.step_for_workload(w, num_splits=4)
    out, lse = step.run()
    torch.cuda.synchronize()
    eager_out, eager_lse = out.clone(), lse.clone()
    out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.run(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager_out) and torch.equal(lse, eager_lse)


# ------------------------------------------------- benchmark workloads, full size


@pytest.mark.parametrize("name", ["plain_decode_d1", "plain_decode_d2", "mtp", "long_context", "sparse_mixed"])
def test_benchmark_workload_every_token(name):
    """The D shard calls + merge of a benchmark workload at full size, in the
    launch configuration the benchmark times, against the oracle on every
    token: each shard's partials, LSEs and counts (bit-exact), and the merged
    (W_UV-projected) result."""
    w = wl.NAMED[name](device="cuda")
    step = pipeline.step_for_workload(w)
    out, lse = step.run()
    torch.cuda.synchronize()
    rc, detail = mla.workspace_status(step.workspace)
    assert rc == mla.MLA_OK, detail
    ref = oracle_workload(name, w)
    assert step.counts.cpu().numpy().tolist() == ref["counts"].tolist(), f"{name} counts"
    for r in range(w.dcp_world):
        assert_out_close(to_np(step.partials[r]), ref["parts"][r], f"{name} shard {r}")
        assert_lse_close(to_np(step.lses[r]), ref["lses"][r], f"{name} shard {r} lse")
    assert_out_close(to_np(out), ref["out"], f"{name} merged")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} merged lse")


# ------------------------------------------------ two-stage decomposition


def test_two_stage_decomposition_on_the_gpu():
    """A second GPU path: per shard, the sparse decode over each token's
    context keys (every row sees them all) and over its request's q_len new
    keys (the kernel keeps those up to the row's position), the 2 D results
    merged by LSE, against the oracle and against the dense decode."""
    from oracle_pins import two_stage_lists
    w = wl.custom([700, 1300, 90, 4], [3, 4, 2, 4], 16, 2, page_size=64, seed=31).to("cuda")
    ctx, ctx_valid, new, new_valid = [torch.from_numpy(x).to("cuda") for x in two_stage_lists(w.to("cpu"))]
    parts, lses, counts = [], [], []
    for r, s in enumerate(w.shards):
        for idx, valid in ((ctx, ctx_valid), (new, new_valid)):
            o, l, c = mla.mla_sparse_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens,
                                                w.query_start_loc, idx, valid, w.dcp_world, r, w.scale,
                                                out_dtype=torch.float32)
            parts.append(o), lses.append(l), counts.append(c)
    out, lse = mla.dcp_lse_merge(torch.stack(parts), torch.stack(lses), torch.stack(counts), None,
                                 out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["merged"], "two-stage merged output")
    assert_lse_close(to_np(lse), ref["lse"], "two-stage merged lse")
    dense_out, dense_lse = mla.mla_dcp_decode_fused(w.q_nope, w.q_pe, [s.cache for s in w.shards],
                                                    [s.block_table for s in w.shards], w.seq_lens,
                                                    w.query_start_loc, w.max_query_len, w.max_seq_len, w.scale,
                                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_out_close(to_np(out), to_np(dense_out).astype(np.float64), "two-stage vs one-pass on the GPU")
