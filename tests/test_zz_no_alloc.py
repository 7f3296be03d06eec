"""The decode entry point for callers that cannot allocate device memory.

mla_dcp_decode_static_scratch takes no workspace: its scratch is a fixed
device array inside the library.  This file is collected last so that a run
stopping at the first failure has already run every other test.  It checks,
through the C ABI, two calls in a row against mla_dcp_decode with a caller
workspace (same tolerance as the other parity tests), two calls on
different problems issued back to back on one stream with no synchronise in
between, and that a problem whose scratch would not fit the array is
refused before anything runs.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build
from mla_decode_attention_04_gb300 import workloads as wl
from parity_utils import assert_lse_close, assert_out_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mla_build.build()
    return mla.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_static(lib, w, r, out, lse, counts):
    s = w.shards[r]
    return lib.mla_dcp_decode_static_scratch(
        _p(w.q_nope), w.q_nope.stride(1), _p(w.q_pe), w.q_pe.stride(1), _p(s.cache), s.cache.shape[0], w.page_size,
        mla.MLA_DTYPE_BF16, _p(s.block_table), s.block_table.shape[1], _p(w.seq_lens), _p(w.query_start_loc),
        w.num_requests, w.num_tokens, w.num_heads, w.max_query_len, w.max_seq_len, w.dcp_world, r,
        ctypes.c_float(w.scale), _p(out), mla.MLA_DTYPE_F32, _p(lse), _p(counts), 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["tiny", "mtp_small"])
def test_static_scratch_matches_workspace_entry_point(lib, name):
    if name == "tiny":
        w = wl.tiny().to("cuda")
    else:
        w = wl.mtp(device="cuda", batch=16)
    assert lib.mla_dcp_decode_workspace_size(w.num_requests, w.num_tokens, w.num_heads, w.max_query_len,
                                             w.max_seq_len, w.dcp_world, 0) <= mla.MLA_STATIC_SCRATCH_BYTES
    for r, s in enumerate(w.shards):
        ref_out, ref_lse, ref_cnt = mla.mla_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens,
                                                       w.query_start_loc, w.max_query_len, w.max_seq_len,
                                                       w.dcp_world, r, w.scale, out_dtype=torch.float32)
        for _ in range(2):  # two calls in a row share the array
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            cnt = torch.full_like(ref_cnt, -1)
            rc = _call_static(lib, w, r, out, lse, cnt)
            assert rc == mla.MLA_OK, lib.mla_last_error().decode()
            torch.cuda.synchronize()
            assert torch.equal(cnt, ref_cnt)
            assert_out_close(to_np(out), to_np(ref_out).astype(np.float64), f"{name} shard {r}")
            assert_lse_close(to_np(lse), to_np(ref_lse).astype(np.float64), f"{name} shard {r} lse")


def test_static_scratch_back_to_back_on_one_stream(lib):
    """Calls on one stream are ordered, so consecutive calls may share the
    array: two different problems, launched back to back without a
    synchronise, each match the workspace entry point."""
    cases = [wl.tiny().to("cuda"), wl.mtp(device="cuda", batch=16)]
    refs, outs = [], []
    for w in cases:
        s = w.shards[1]
        refs.append(mla.mla_dcp_decode(w.q_nope, w.q_pe, s.cache, s.block_table, w.seq_lens, w.query_start_loc,
                                       w.max_query_len, w.max_seq_len, w.dcp_world, 1, w.scale,
                                       out_dtype=torch.float32))
    torch.cuda.synchronize()
    for w, (ro, rl, rc) in zip(cases, refs):
        o = torch.full_like(ro, float("nan"))
        l = torch.full_like(rl, float("nan"))
        c = torch.full_like(rc, -1)
        assert _call_static(lib, w, 1, o, l, c) == mla.MLA_OK, lib.mla_last_error().decode()
        outs.append((o, l, c))
    torch.cuda.synchronize()
    for (ro, rl, rc), (o, l, c) in zip(refs, outs):
        assert torch.equal(c, rc)
        assert_out_close(to_np(o), to_np(ro).astype(np.float64), "back-to-back static call")
        assert_lse_close(to_np(l), to_np(rl).astype(np.float64), "back-to-back static call lse")


def test_static_scratch_refuses_oversized_problems(lib):
    # The dense workspace is bounded by the SM count (2 partial slots of up
    # to 64 rows per SM): a problem with 64-row units (here 2 query tokens x
    # 128 heads per request) needs about 40 MB on a 152-SM GPU, more than the
    # array, so it is refused before anything runs.
    B, T, H, L = 32, 64, 128, 32768
    need = lib.mla_dcp_decode_workspace_size(B, T, H, 2, L, 8, 0)
    if need <= mla.MLA_STATIC_SCRATCH_BYTES:
        pytest.skip(f"every dense problem fits the static array on this GPU (largest workspace {need} bytes)")
    dummy = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    a = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.mla_dcp_decode_static_scratch(a, 512, a, 64, a, 100, 64, mla.MLA_DTYPE_BF16, a, 8, a, a, B, T, H, 2, L, 8,
                                           0, ctypes.c_float(0.07), a, mla.MLA_DTYPE_F32, a, None, 0, None)
    assert rc == mla.MLA_ERR_WORKSPACE
    assert "static" in lib.mla_last_error().decode()
