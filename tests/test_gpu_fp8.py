"""GPU parity of the FP8 latent cache calls (mla_dcp_decode_fp8 and
mla_dcp_decode_fused_fp8) against the fp64 oracle's FP8 decode: each cache
value is kv_scale times the exact value of its E4M3 code.  Same tolerances
as the bf16 calls (parity_utils)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build
from mla_decode_attention_04_gb300 import workloads as wl
from parity_utils import HostInputs, assert_lse_close, assert_out_close, oracle_step_kv8, to_np
from test_gpu_parity import EDGE

pytestmark = pytest.mark.gpu
KV_SCALE = 0.25


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mla_build.build()
    mla.load_library()


def _fp8(w, kv_scale=KV_SCALE):
    codes, views = wl.fp8_cache(w, kv_scale)
    return codes, views, [v.cpu().numpy() for v in views]


def _shard_calls(w, views, kv_scale=KV_SCALE, out_dtype=torch.float32, num_splits=0):
    res = []
    for r, s in enumerate(w.shards):
        res.append(mla.mla_dcp_decode_fp8(w.q_nope, w.q_pe, views[r], kv_scale, s.block_table, w.seq_lens,
                                          w.query_start_loc, w.max_query_len, w.max_seq_len, w.dcp_world, r, w.scale,
                                          out_dtype=out_dtype, num_splits=num_splits))
    torch.cuda.synchronize()
    return res


def _fused(w, views, kv_scale=KV_SCALE, out_dtype=torch.float32):
    out, lse = mla.mla_dcp_decode_fused_fp8(w.q_nope, w.q_pe, views, kv_scale, [s.block_table for s in w.shards],
                                            w.seq_lens, w.query_start_loc, w.max_query_len, w.max_seq_len, w.scale,
                                            out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, lse


def test_e4m3_widening_is_exact():
    """Zero queries and one visible key per token: the output is the key's
    kv_c times kv_scale, so every finite E4M3 code (subnormals, signed zero,
    +-448) must come back exactly."""
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    B = 6
    w = wl.custom([1] * B, [1] * B, 4, 1, page_size=8, seed=3).to("cuda")
    w.q_nope.zero_()
    w.q_pe.zero_()
    rng = np.random.default_rng(0)
    codes = torch.zeros(w.cache_all.shape, dtype=torch.uint8)
    for p in range(codes.shape[0]):
        for slot in range(codes.shape[1]):
            codes[p, slot] = torch.from_numpy(rng.permutation(np.resize(finite, 576)).astype(np.uint8))
    codes = codes.cuda()
    sh = w.shards[0]
    view = codes[sh.page_base:sh.page_base + sh.cache.shape[0]]
    out, lse, cnt = mla.mla_dcp_decode_fp8(w.q_nope, w.q_pe, view, 0.5, sh.block_table, w.seq_lens,
                                           w.query_start_loc, 1, 1, 1, 0, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert cnt.cpu().tolist() == [1] * B
    bt = sh.block_table.cpu().numpy()
    vals = wl.e4m3_values(view.cpu()).numpy()
    for b in range(B):
        want = 0.5 * vals[bt[b, 0], 0, :512]
        got = out[b].cpu().numpy()
        for h in range(w.num_heads):
            assert np.array_equal(got[h], want.astype(np.float32)), f"request {b} head {h}"
    assert torch.all(lse == 0)


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tiny_fp8_shards_and_fused(num_splits, out_dtype):
    w = wl.tiny().to("cuda")
    _, views, host8 = _fp8(w)
    ref = oracle_step_kv8(HostInputs(w), host8, KV_SCALE)
    for r, (out, lse, cnt) in enumerate(_shard_calls(w, views, out_dtype=out_dtype, num_splits=num_splits)):
        assert cnt.cpu().numpy().tolist() == ref["counts"][r].tolist()
        assert_out_close(to_np(out), ref["parts"][r], f"fp8 shard {r}")
        assert_lse_close(to_np(lse), ref["lses"][r], f"fp8 shard {r} lse")
    out, lse = _fused(w, views, out_dtype=out_dtype)
    assert_out_close(to_np(out), ref["merged"], "fp8 fused")
    assert_lse_close(to_np(lse), ref["lse"], "fp8 fused lse")


@pytest.mark.parametrize("name", sorted(EDGE))
def test_fp8_edge_shapes(name):
    w = wl.custom(seed=sorted(EDGE).index(name), **EDGE[name]).to("cuda")
    _, views, host8 = _fp8(w, 0.125)
    ref = oracle_step_kv8(HostInputs(w), host8, 0.125)
    for r, (out, lse, cnt) in enumerate(_shard_calls(w, views, 0.125)):
        assert cnt.cpu().numpy().tolist() == ref["counts"][r].tolist()
        assert_out_close(to_np(out), ref["parts"][r], f"{name} fp8 shard {r}")
        assert_lse_close(to_np(lse), ref["lses"][r], f"{name} fp8 shard {r} lse")
    out, lse = _fused(w, views, 0.125)
    assert_out_close(to_np(out), ref["merged"], f"{name} fp8 fused")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} fp8 fused lse")


@pytest.mark.parametrize("name", ["plain_decode_d2", "mtp"])
def test_fp8_benchmark_workload_every_token(name):
    """The benchmark workloads with an FP8 cache, at full size, every token:
    the fused call's merged result and each shard call against the oracle."""
    w = wl.NAMED[name](device="cuda")
    _, views, host8 = _fp8(w)
    ref = oracle_step_kv8(HostInputs(w), host8, KV_SCALE)
    out, lse = _fused(w, views)
    assert_out_close(to_np(out), ref["merged"], f"{name} fp8 fused")
    assert_lse_close(to_np(lse), ref["lse"], f"{name} fp8 fused lse")
    for r, (o, l, c) in enumerate(_shard_calls(w, views)):
        assert c.cpu().numpy().tolist() == ref["counts"][r].tolist()
        assert_out_close(to_np(o), ref["parts"][r], f"{name} fp8 shard {r}")
        assert_lse_close(to_np(l), ref["lses"][r], f"{name} fp8 shard {r} lse")
