"""GPU parity of the two-stage decomposition (mla_dcp_decode_two_stage).

"[Attention] add DCP support for FLASH_ATTN_MLA backend", review thread:
context keys with the causal mask off plus the query's own keys with it
on, merged, in place of a custom DCP mask.  The call runs stage 1 (dense,
non-causal, over each request's context), stage 2 (sparse, over each
token's new positions up to its own) and their LSE merge, all on the device.
Checked element by element against the oracle's causal DCP attention (its D
shard attentions merged by LSE) and against the one-pass fused call."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build
from mla_decode_attention_04_gb300 import workloads as wl
from parity_utils import HostInputs, assert_lse_close, assert_out_close, oracle_step, oracle_workload, to_np
from test_gpu_parity import EDGE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mla_build.build()
    mla.load_library()


def _two_stage(w, out_dtype=torch.float32, workspace=None):
    out, lse = mla.mla_dcp_decode_two_stage(w.q_nope, w.q_pe, [s.cache for s in w.shards],
                                            [s.block_table for s in w.shards], w.seq_lens, w.query_start_loc,
                                            w.max_query_len, w.max_seq_len, w.scale, out_dtype=out_dtype,
                                            workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def _fused(w):
    out, lse = mla.mla_dcp_decode_fused(w.q_nope, w.q_pe, [s.cache for s in w.shards],
                                        [s.block_table for s in w.shards], w.seq_lens, w.query_start_loc,
                                        w.max_query_len, w.max_seq_len, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    return out, lse


def _workspace(w):
    B = w.seq_lens.shape[0]
    need = mla.two_stage_workspace_size(B, w.num_tokens, w.num_heads, w.max_query_len, w.max_seq_len)
    return torch.empty((need,), dtype=torch.uint8, device="cuda")


CASES = ["tiny"] + sorted(EDGE)


def _case(name):
    if name == "tiny":
        return wl.tiny().to("cuda")
    return wl.custom(seed=100 + sorted(EDGE).index(name), **EDGE[name]).to("cuda")


@pytest.mark.parametrize("name", CASES)
def test_two_stage_matches_oracle_and_one_pass(name):
    w = _case(name)
    ws = _workspace(w)
    out, lse = _two_stage(w, workspace=ws)
    assert mla.workspace_status(ws) == (mla.MLA_OK, 0)
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["merged"], f"{name} out")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} lse")
    # the one-pass causal call: the same attention, another summation order
    out1, lse1 = _fused(w)
    np.testing.assert_allclose(to_np(out), to_np(out1), atol=1e-3, rtol=1e-3)
    a, b = to_np(lse), to_np(lse1)
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = ~np.isneginf(b)
    assert np.abs(a[fin] - b[fin]).max(initial=0.0) <= 1e-4


def test_two_stage_bf16_output():
    w = wl.tiny().to("cuda")
    out, lse = _two_stage(w, out_dtype=torch.bfloat16)
    ref = oracle_step(HostInputs(w))
    assert_out_close(to_np(out), ref["merged"], "tiny bf16 out")
    assert_lse_close(to_np(lse), ref["lse"], "tiny bf16 lse")


@pytest.mark.parametrize("name", ["mtp", "plain_decode_d2"])
def test_two_stage_benchmark_workload_every_token(name):
    """Every token of a full-size workload (MTP: q_len 2, D=4, 128 requests;
    plain decode: q_len 1, D=2) against the oracle."""
    w = wl.NAMED[name](device="cuda")
    out, lse = _two_stage(w)
    ref = oracle_workload(name, w)
    assert_out_close(to_np(out), ref["merged"], f"{name} out")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} lse")


def test_two_stage_status_reports_the_second_stage():
    """A page id past the cache that only stage 2 reads (the page holding a
    request's new keys, after a context of exactly 3 full pages) is reported
    in the call's status word; a clean call resets it."""
    w = wl.custom([50], [2], 16, 1, page_size=16, seed=9).to("cuda")
    s = w.shards[0]
    good = int(s.block_table[0, 3])
    s.block_table[0, 3] = s.cache.shape[0] + 5
    ws = _workspace(w)
    _two_stage(w, workspace=ws)
    rc, detail = mla.workspace_status(ws)
    assert rc == mla.MLA_ERR_DEVICE_CHECK and detail == 1
    s.block_table[0, 3] = good
    _two_stage(w, workspace=ws)
    assert mla.workspace_status(ws) == (mla.MLA_OK, 0)


def test_two_stage_replays_in_a_cuda_graph():
    """The call allocates nothing and reads its lengths on the device: one
    captured call replays bit for bit like the eager call, also after the
    lengths change within the captured bounds."""
    w = wl.custom([300, 41, 1000, 7], [2, 1, 4, 3], 16, 2, page_size=16, seed=21).to("cuda")
    ws = _workspace(w)
    out = torch.empty((w.num_tokens, w.num_heads, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.num_tokens, w.num_heads), dtype=torch.float32, device="cuda")

    def call():
        mla.mla_dcp_decode_two_stage(w.q_nope, w.q_pe, [s.cache for s in w.shards], [s.block_table for s in w.shards],
                                     w.seq_lens, w.query_start_loc, w.max_query_len, w.max_seq_len, w.scale,
                                     out=out, lse=lse, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for lens in ([300, 41, 1000, 7], [290, 12, 999, 3]):
        w.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        o_graph, l_graph = out.clone(), lse.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_graph, out) and torch.equal(l_graph, lse)
        assert mla.workspace_status(ws) == (mla.MLA_OK, 0)
