"""A decode whose pipeline waits give up ends cleanly (GPU).

Every pipeline wait inside the decode kernels is bounded.  When one gives
up, its CTA stops issuing work, waits (with a bound of its own) for the
copies and MMAs it already issued, frees its tensor memory and exits; the
call completes, mla_workspace_status reports check 3, the workspace names
the first site that gave up, and the context stays usable.  Here the test
hook shortens the budget to 1 ns so that waits give up on purpose (no fault
is involved: a wait that runs out is an ordinary outcome of the kernel).
"""
import numpy as np
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build
from mla_decode_attention_04_gb300 import pipeline, workloads as wl
from parity_utils import HostInputs, assert_lse_close, assert_out_close, oracle_step, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mla_build.build()
    lib = mla.load_library()
    yield lib
    lib.mla_debug_set_wait_budget_ns(0)


@pytest.mark.parametrize("route", ["shards", "fused", "fused_fp8", "sparse_fused"])
def test_waits_give_up_cleanly_then_the_next_call_is_right(lib, route):
    if route == "sparse_fused":
        w = wl.custom([300, 90, 700, 45], [2, 1, 4, 3], 64, 4, page_size=16, seed=7, topk=128, short_valid_frac=0.3,
                      force_zero_valid=1).to("cuda")
    else:
        w = wl.tiny().to("cuda")
    ws = torch.empty(max(mla.decode_workspace_size(w.num_requests, w.num_tokens, w.num_heads, w.max_query_len,
                                                   w.max_seq_len, w.dcp_world),
                         mla.fused_workspace_size(w.num_requests, w.num_tokens, w.num_heads, w.max_query_len,
                                                  w.max_seq_len),
                         mla.sparse_workspace_size(w.num_tokens, w.num_heads, 128, w.dcp_world)),
                     dtype=torch.uint8, device="cuda")
    tables = [s.block_table for s in w.shards]
    views = wl.fp8_cache(w, 0.25)[1] if route == "fused_fp8" else None

    def run():
        if route == "shards":
            s = w.shards[1]
            return mla.mla_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc,
                                      w.max_query_len, w.max_seq_len, w.dcp_world, 1, w.scale,
                                      out_dtype=torch.float32, workspace=ws)[:2]
        if route == "fused":
            return mla.mla_dcp_decode_fused(w.q_nope, w.q_pe, [s.cache for s in w.shards], tables, w.seq_lens,
                                            w.query_start_loc, w.max_query_len, w.max_seq_len, w.scale,
                                            out_dtype=torch.float32, workspace=ws)
        if route == "fused_fp8":
            return mla.mla_dcp_decode_fused_fp8(w.q_nope, w.q_pe, views, 0.25, tables, w.seq_lens,
                                                w.query_start_loc, w.max_query_len, w.max_seq_len, w.scale,
                                                out_dtype=torch.float32, workspace=ws)
        out, lse, _ = mla.mla_sparse_dcp_decode_fused(w.q_nope, w.q_pe, [s.cache for s in w.shards], tables,
                                                      w.seq_lens, w.query_start_loc, w.topk, w.topk_valid, w.scale,
                                                      out_dtype=torch.float32, workspace=ws)
        return out, lse

    lib.mla_debug_set_wait_budget_ns(1)
    try:
        run()
        rc, detail = mla.workspace_status(ws)
    finally:
        lib.mla_debug_set_wait_budget_ns(0)
    assert rc == mla.MLA_ERR_DEVICE_CHECK and detail == 3, (rc, detail)
    assert mla.workspace_wait_site(ws) > 0
    # the context is usable: the same call with the default budget is right
    out, lse = run()
    assert mla.workspace_status(ws) == (mla.MLA_OK, 0)
    assert mla.workspace_wait_site(ws) == 0
    torch.cuda.synchronize()
    if route == "shards":
        ref = oracle_step(HostInputs(w))
        assert_out_close(to_np(out), ref["parts"][1], "after give-up")
        assert_lse_close(to_np(lse), ref["lses"][1], "after give-up lse")
    elif route in ("fused", "sparse_fused"):
        ref = oracle_step(HostInputs(w), sparse=route == "sparse_fused")
        assert_out_close(to_np(out), ref["merged"], "after give-up")
        assert_lse_close(to_np(lse), ref["lse"], "after give-up lse")
    else:
        assert torch.isfinite(out).all()
