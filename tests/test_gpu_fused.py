"""GPU parity of the shard-fused dense decode (mla_dcp_decode_fused): one
launch over all D shards whose online softmax runs over every shard's
visible keys, checked against the oracle's D shard attentions merged by LSE
(and, with W_UV, projected), element by element."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build
from mla_decode_attention_04_gb300 import pipeline, workloads as wl
from parity_utils import HostInputs, assert_lse_close, assert_out_close, oracle_step, oracle_workload, to_np
from test_gpu_parity import EDGE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mla_build.build()
    mla.load_library()


def _fused(w, out_dtype=torch.float32, num_splits=0):
    out, lse = mla.mla_dcp_decode_fused(w.q_nope, w.q_pe, [s.cache for s in w.shards],
                                        [s.block_table for s in w.shards], w.seq_lens, w.query_start_loc,
                                        w.max_query_len, w.max_seq_len, w.scale, out_dtype=out_dtype,
                                        num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_tiny_fused(out_dtype, num_splits):
    w = wl.tiny().to("cuda")
    out, lse = _fused(w, out_dtype, num_splits)
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["merged"], "fused merged output")
    assert_lse_close(to_np(lse), ref["lse"], "fused merged lse")


@pytest.mark.parametrize("name", sorted(EDGE))
def test_fused_edge_shapes(name):
    w = wl.custom(seed=sorted(EDGE).index(name), **EDGE[name]).to("cuda")
    out, lse = _fused(w)
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["merged"], f"{name} fused output")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} fused lse")


def test_tiny_fused_step_with_wuv():
    w = wl.tiny().to("cuda")
    step = pipeline.fused_step_for_workload(w)
    out, lse = step.run()
    torch.cuda.synchronize()
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["out"], "fused step W_UV output")
    assert_lse_close(to_np(lse), ref["lse"], "fused step lse")


def test_fused_needs_one_cache_and_table_per_shard():
    w = wl.tiny().to("cuda")
    with pytest.raises(ValueError):
        mla.mla_dcp_decode_fused(w.q_nope, w.q_pe, [w.shards[0].cache], [], w.seq_lens, w.query_start_loc,
                                 w.max_query_len, w.max_seq_len, w.scale)


@pytest.mark.parametrize("name", ["plain_decode_d1", "plain_decode_d2", "mtp", "long_context"])
def test_fused_benchmark_workload_every_token(name):
    """The benchmarked shard-fused step at full size against the oracle's
    merged (W_UV-projected) result on every token."""
    w = wl.NAMED[name](device="cuda")
    step = pipeline.fused_step_for_workload(w)
    out, lse = step.run()
    torch.cuda.synchronize()
    rc, detail = mla.workspace_status(step.workspace)
    assert rc == mla.MLA_OK, detail
    ref = oracle_workload(name, w)
    assert_out_close(to_np(out), ref["out"], f"{name} fused step")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} fused lse")


def test_fused_matches_shard_calls_on_every_token():
    # the two routes on the GPU agree everywhere (the oracle checks samples)
    w = wl.NAMED["plain_decode_d2"](device="cuda")
    fused_out, fused_lse = pipeline.fused_step_for_workload(w).run()
    step = pipeline.step_for_workload(w, partial_dtype=torch.float32)
    out, lse = step.run()
    torch.cuda.synchronize()
    assert_out_close(to_np(fused_out), to_np(out).astype(np.float64), "fused vs shard calls")
    assert_lse_close(to_np(fused_lse), to_np(lse).astype(np.float64), "fused vs shard calls lse")


# ------------------------------------------------------------------ sparse


def _sparse_fused(w, out_dtype=torch.float32):
    kept = torch.empty((w.num_tokens,), dtype=torch.int32, device="cuda")
    out, lse, kept = mla.mla_sparse_dcp_decode_fused(w.q_nope, w.q_pe, [s.cache for s in w.shards],
                                                     [s.block_table for s in w.shards], w.seq_lens,
                                                     w.query_start_loc, w.topk, w.topk_valid, w.scale,
                                                     out_dtype=out_dtype, kept_counts=kept)
    torch.cuda.synchronize()
    return out, lse, kept


@pytest.mark.parametrize("H,D,K", [(16, 2, 64), (24, 3, 100), (64, 4, 256), (1, 1, 7), (32, 8, 300)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_sparse_fused_small(H, D, K, out_dtype):
    # short valid counts and a row with none: the merged result over every
    # shard's kept entries, and the kept count = the shard counts' sum
    w = wl.custom([300, 90, 700, 45], [2, 1, 4, 3], H, D, page_size=16, seed=H + D + K, topk=K,
                  short_valid_frac=0.3, force_zero_valid=1).to("cuda")
    out, lse, kept = _sparse_fused(w, out_dtype)
    ref = oracle_step(HostInputs(w), sparse=True)
    assert kept.cpu().numpy().tolist() == ref["counts"].sum(axis=0).tolist()
    assert_out_close(to_np(out), ref["merged"], "sparse fused output")
    assert_lse_close(to_np(lse), ref["lse"], "sparse fused lse")


def test_sparse_fused_matches_shard_calls_merged():
    # the fused call against the D shard calls + merge on the GPU, every token
    w = wl.custom([1200, 333, 2050, 64, 900], [1, 4, 2, 1, 3], 64, 4, page_size=64, seed=5, topk=512,
                  short_valid_frac=0.2, force_zero_valid=1).to("cuda")
    fused_out, fused_lse, _ = _sparse_fused(w)
    parts = [mla.mla_sparse_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc,
                                       w.topk, w.topk_valid, w.dcp_world, r, w.scale, out_dtype=torch.float32)
             for r, s in enumerate(w.shards)]
    out, lse = mla.dcp_lse_merge(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]),
                                 torch.stack([p[2] for p in parts]), None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_out_close(to_np(fused_out), to_np(out).astype(np.float64), "sparse fused vs shard calls")
    assert_lse_close(to_np(fused_lse), to_np(lse).astype(np.float64), "sparse fused vs shard calls lse")


def test_sparse_fused_step_with_wuv():
    w = wl.custom([300, 90, 700, 45], [2, 1, 4, 3], 64, 4, page_size=64, seed=11, topk=128, short_valid_frac=0.3,
                  force_zero_valid=1).to("cuda")
    step = pipeline.fused_step_for_workload(w)
    out, lse = step.run()
    torch.cuda.synchronize()
    ref = oracle_step(HostInputs(w), sparse=True)
    assert_out_close(to_np(out), ref["out"], "sparse fused W_UV output")
    assert_lse_close(to_np(lse), ref["lse"], "sparse fused lse")


def test_sparse_fused_benchmark_workload_every_token():
    """The benchmarked sparse shard-fused step at full size against the
    oracle on every token, kept counts (the shard counts' sum) bit-exact."""
    w = wl.NAMED["sparse_mixed"](device="cuda")
    step = pipeline.fused_step_for_workload(w)
    kept = torch.empty((w.num_tokens,), dtype=torch.int32, device="cuda")
    step.kept_counts = kept
    out, lse = step.run()
    torch.cuda.synchronize()
    rc, detail = mla.workspace_status(step.workspace)
    assert rc == mla.MLA_OK, detail
    ref = oracle_workload("sparse_mixed", w)
    assert kept.cpu().numpy().tolist() == ref["counts"].sum(axis=0).tolist()
    assert_out_close(to_np(out), ref["out"], "sparse_mixed fused step")
    assert_lse_close(to_np(lse), ref["lse"], "sparse_mixed fused lse")


# ---------------------------------------------- graph replay with new lengths


@pytest.mark.parametrize("sparse", [False, True])
def test_graph_replays_new_lengths(sparse):
    """The split plan is derived on the device from the lengths in memory, so
    one captured step serves a later step whose lengths, query lengths and
    lists differ (same buffers, same bounds): the replay equals an eager call
    on the new inputs."""
    kw = dict(topk=256, short_valid_frac=0.2, force_zero_valid=1) if sparse else {}
    w = wl.custom([700, 1300, 90, 500], [3, 4, 2, 4], 32, 2, page_size=64, seed=41, with_w_uv=False, **kw).to("cuda")
    step = pipeline.fused_step_for_workload(w)
    step.run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.run(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    # the next step: shorter sequences, other query lengths (same token
    # count), other queries; the block tables and caches stay valid
    w.seq_lens.copy_(torch.tensor([400, 1300, 60, 9], dtype=torch.int32))
    w.query_start_loc.copy_(torch.tensor([0, 4, 7, 10, 13], dtype=torch.int32))
    w.q_nope.copy_(torch.randn_like(w.q_nope, dtype=torch.float32).to(torch.bfloat16) * 0.1)
    if sparse:
        w.topk_valid.copy_(torch.clamp(w.topk_valid, max=100))
    g.replay()
    torch.cuda.synchronize()
    out_g, lse_g = step.out.clone(), step.lse.clone()
    step.out.zero_()
    step.run()
    torch.cuda.synchronize()
    rc, detail = mla.workspace_status(step.workspace)
    assert rc == mla.MLA_OK, detail
    assert torch.equal(out_g, step.out) and torch.equal(lse_g, step.lse)


@pytest.mark.parametrize("fused", [False, True])
def test_sparse_long_lists(fused):
    # lists longer than one 2048-entry pass of the key-list kernel, page 32,
    # a request whose prefix is shorter than the list, short and empty rows
    w = wl.custom([6100, 700, 2600], [2, 1, 3], 24, 3, page_size=32, seed=13, topk=5000, short_valid_frac=0.3,
                  force_zero_valid=1).to("cuda")
    ref = oracle_step(HostInputs(w), sparse=True)
    if fused:
        out, lse, kept = _sparse_fused(w)
        assert kept.cpu().numpy().tolist() == ref["counts"].sum(axis=0).tolist()
    else:
        parts = [mla.mla_sparse_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc,
                                           w.topk, w.topk_valid, w.dcp_world, r, w.scale, out_dtype=torch.float32)
                 for r, s in enumerate(w.shards)]
        counts = torch.stack([p[2] for p in parts])
        assert counts.cpu().numpy().tolist() == ref["counts"].tolist()
        out, lse = mla.dcp_lse_merge(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]), counts,
                                     None, out_dtype=torch.float32)
        torch.cuda.synchronize()
    assert_out_close(to_np(out), ref["merged"], "long-list sparse output")
    assert_lse_close(to_np(lse), ref["lse"], "long-list sparse lse")
