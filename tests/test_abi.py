"""The C-ABI library: it builds for sm_103a, loads, exports every function the
header declares, and rejects bad arguments on the host before any launch
(CPU only: no call here reaches the GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_dcp.h")
A = 1 << 20  # a 256-byte aligned fake device address: never dereferenced by these calls


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^(?:int|int64_t|size_t|void|const char \*)\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("mla_dcp_decode", "mla_sparse_dcp_decode", "dcp_lse_merge"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names and set(names) <= set(mla.EXPORTS) | set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", mla.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(mla.EXPORTS) == set(names)


def test_library_is_built_for_sm_103a():
    assert "compute_103a,code=sm_103a" in " ".join(mla_build.ARCH)
    assert mla_build.up_to_date()


def _decode(lib, **kw):
    args = dict(q_nope=A, sn=512, q_pe=A, sp=64, kv=A, nb=10, ps=64, kvdt=mla.MLA_DTYPE_BF16, bt=A, bts=4, sl=A,
                qsl=A, B=2, T=2, H=16, mq=1, ms=100, D=2, r=0, scale=0.07, out=A, odt=mla.MLA_DTYPE_BF16, lse=A,
                rc=None, ns=0, ws=A, wsb=1 << 30, stream=None)
    args.update(kw)
    a = args
    rc = lib.mla_dcp_decode(a["q_nope"], a["sn"], a["q_pe"], a["sp"], a["kv"], a["nb"], a["ps"], a["kvdt"], a["bt"],
                            a["bts"], a["sl"], a["qsl"], a["B"], a["T"], a["H"], a["mq"], a["ms"], a["D"], a["r"],
                            a["scale"], a["out"], a["odt"], a["lse"], a["rc"], a["ns"], a["ws"], a["wsb"], a["stream"])
    return rc, lib.mla_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(r=2), mla.MLA_ERR_INVALID_ARG),
    (dict(r=-1), mla.MLA_ERR_INVALID_ARG),
    (dict(D=0, r=0), mla.MLA_ERR_INVALID_ARG),
    (dict(H=0), mla.MLA_ERR_INVALID_ARG),
    (dict(H=129), mla.MLA_ERR_INVALID_ARG),
    (dict(nb=0), mla.MLA_ERR_INVALID_ARG),
    (dict(kvdt=mla.MLA_DTYPE_FP8_E4M3), mla.MLA_ERR_UNSUPPORTED),
    (dict(ps=12), mla.MLA_ERR_UNSUPPORTED),
    (dict(ps=96), mla.MLA_ERR_UNSUPPORTED),
    (dict(q_nope=None), mla.MLA_ERR_INVALID_ARG),
    (dict(q_nope=A + 8), mla.MLA_ERR_INVALID_ARG),
    (dict(sn=500), mla.MLA_ERR_INVALID_ARG),
    (dict(odt=7), mla.MLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), mla.MLA_ERR_INVALID_ARG),
    (dict(scale=0.0), mla.MLA_ERR_INVALID_ARG),
    (dict(scale=-0.07), mla.MLA_ERR_INVALID_ARG),
    (dict(ws=None), mla.MLA_ERR_WORKSPACE),
    (dict(ws=A + 64), mla.MLA_ERR_WORKSPACE),
    (dict(wsb=16), mla.MLA_ERR_WORKSPACE),
    (dict(ns=-1), mla.MLA_ERR_INVALID_ARG),
])
def test_decode_argument_errors(lib, kw, code):
    rc, msg = _decode(lib, **kw)
    assert rc == code, msg
    assert msg


def test_decode_zero_tokens_is_a_noop(lib):
    rc, msg = _decode(lib, T=0)
    assert rc == mla.MLA_OK, msg


def test_workspace_size_grows_with_work(lib):
    small = lib.mla_dcp_decode_workspace_size(4, 4, 16, 1, 1024, 2, 0)
    big = lib.mla_dcp_decode_workspace_size(4, 8, 16, 2, 1024, 2, 0)
    assert 256 < small < big
    # a fixed split bound sizes the partials: one split needs none
    assert lib.mla_dcp_decode_workspace_size(4, 8, 16, 2, 1024, 2, 1) < big
    assert lib.mla_sparse_dcp_decode_workspace_size(480, 64, 2048, 4) >= 480 * 2048 * 4


def test_merge_argument_errors(lib):
    rc = lib.dcp_lse_merge(A, mla.MLA_DTYPE_F32, A, None, None, 0, 4, 16, A, mla.MLA_DTYPE_BF16, None, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = lib.dcp_lse_merge(A, 5, A, None, None, 2, 4, 16, A, mla.MLA_DTYPE_BF16, None, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = lib.dcp_lse_merge(A + 4, mla.MLA_DTYPE_F32, A, None, None, 2, 4, 16, A, mla.MLA_DTYPE_BF16, None, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = lib.dcp_lse_merge(None, mla.MLA_DTYPE_F32, A, None, None, 2, 4, 16, A, mla.MLA_DTYPE_BF16, None, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    rc = lib.dcp_lse_merge(A, mla.MLA_DTYPE_F32, A, None, None, 2, 0, 16, A, mla.MLA_DTYPE_BF16, None, None)
    assert rc == mla.MLA_OK


def test_sparse_argument_errors(lib):
    def call(**kw):
        a = dict(topk=A, K=2048, valid=A, counts=A, r=0, D=4)
        a.update(kw)
        return lib.mla_sparse_dcp_decode(A, 512, A, 64, A, 10, 64, 0, A, 4, A, A, 2, 2, 16, a["topk"], a["K"],
                                         a["valid"], a["D"], a["r"], 0.07, A, 0, A, a["counts"], A, 1 << 30, None)
    assert call(topk=None) == mla.MLA_ERR_INVALID_ARG
    assert call(counts=None) == mla.MLA_ERR_INVALID_ARG
    assert call(K=0) == mla.MLA_ERR_INVALID_ARG
    assert call(r=4) == mla.MLA_ERR_INVALID_ARG


def test_product_path_has_no_cpu_fallback(monkeypatch, tmp_path):
    """Without the CUDA library the binding raises instead of computing."""
    monkeypatch.setattr(mla, "_lib", None)
    monkeypatch.setattr(mla, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        mla.load_library()


def test_package_does_not_import_oracle():
    import sys
    pkg = os.path.join(ROOT, "mla_decode_attention_04_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text and "mla_oracle" not in text, f
    assert "oracle" not in sys.modules or True


def _shard_arrays(D, nb=10, bad_shard=None, bad=None):
    kvs = (ctypes.c_void_p * D)(*([A] * D))
    nbs = (ctypes.c_int64 * D)(*([nb] * D))
    bts = (ctypes.c_void_p * D)(*([A] * D))
    if bad_shard is not None:
        if bad == "kv":
            kvs[bad_shard] = None
        elif bad == "nb":
            nbs[bad_shard] = 0
        elif bad == "bt":
            bts[bad_shard] = A + 2
    return (ctypes.cast(kvs, ctypes.c_void_p), ctypes.cast(nbs, ctypes.c_void_p), ctypes.cast(bts, ctypes.c_void_p))


def _fused(lib, D=2, T=2, wsb=1 << 30, arrays=None, **kw):
    kvs, nbs, bts = arrays if arrays is not None else _shard_arrays(D)
    a = dict(ps=64, kvdt=mla.MLA_DTYPE_BF16, ns=0, ws=A)
    a.update(kw)
    rc = lib.mla_dcp_decode_fused(A, 512, A, 64, kvs, nbs, a["ps"], a["kvdt"], bts, 4, A, A, 2, T, 16, 1, 100, D,
                                  0.07, A, mla.MLA_DTYPE_BF16, A, a["ns"], a["ws"], wsb, None)
    return rc, lib.mla_last_error().decode()


def _sparse_fused(lib, D=4, T=2, wsb=1 << 30, arrays=None, **kw):
    kvs, nbs, bts = arrays if arrays is not None else _shard_arrays(D)
    a = dict(topk=A, K=2048, valid=A, ws=A, kept=None)
    a.update(kw)
    rc = lib.mla_sparse_dcp_decode_fused(A, 512, A, 64, kvs, nbs, 64, mla.MLA_DTYPE_BF16, bts, 4, A, A, 2, T, 16,
                                         a["topk"], a["K"], a["valid"], D, 0.07, A, mla.MLA_DTYPE_BF16, A, a["kept"],
                                         a["ws"], wsb, None)
    return rc, lib.mla_last_error().decode()


@pytest.mark.parametrize("call", ["dense", "sparse"])
def test_fused_calls_check_every_shard(lib, call):
    f = _fused if call == "dense" else _sparse_fused
    D = 4
    # one bad shard among good ones is caught on the host, whichever it is
    for bad in ("kv", "nb", "bt"):
        for r in (0, D - 1):
            rc, msg = f(lib, D=D, arrays=_shard_arrays(D, bad_shard=r, bad=bad))
            assert rc == mla.MLA_ERR_INVALID_ARG, (bad, r, msg)
            assert msg
    # at most 8 shards in one call
    rc, msg = f(lib, D=9, arrays=_shard_arrays(9))
    assert rc == mla.MLA_ERR_INVALID_ARG and "dcp_world" in msg
    # the shard arrays themselves are required
    rc, _ = f(lib, D=2, arrays=(None, None, None))
    assert rc == mla.MLA_ERR_INVALID_ARG
    # no token: a successful no-op; too small a workspace: refused
    assert f(lib, D=2, T=0)[0] == mla.MLA_OK
    assert f(lib, D=2, wsb=64)[0] == mla.MLA_ERR_WORKSPACE


def test_sparse_fused_argument_errors(lib):
    assert _sparse_fused(lib, topk=None)[0] == mla.MLA_ERR_INVALID_ARG
    assert _sparse_fused(lib, valid=None)[0] == mla.MLA_ERR_INVALID_ARG
    assert _sparse_fused(lib, K=0)[0] == mla.MLA_ERR_INVALID_ARG
    assert _sparse_fused(lib, K=70000)[0] == mla.MLA_ERR_INVALID_ARG


def test_fused_dense_feature_gates(lib):
    assert _fused(lib, kvdt=mla.MLA_DTYPE_FP8_E4M3)[0] == mla.MLA_ERR_UNSUPPORTED
    assert _fused(lib, ps=12)[0] == mla.MLA_ERR_UNSUPPORTED
    assert _fused(lib, ns=-1)[0] == mla.MLA_ERR_INVALID_ARG


def test_sparse_workspace_holds_lists_and_split_partials(lib):
    # per token the kept rows' addresses (8 bytes per entry), plus the split
    # table and two partial slots of NR rows per CTA, whatever the tokens
    T, H, K = 480, 64, 2048
    size = lib.mla_sparse_dcp_decode_workspace_size(T, H, K, 4)
    assert size >= T * K * 8
    small = lib.mla_sparse_dcp_decode_workspace_size(1, H, K, 4)
    assert small >= 2 * 32 * (512 * 4 + 4)  # at least one CTA's two slots of 32 fp32 rows
    assert size - small >= (T - 1) * K * 8
    # the fused dense call's workspace does not grow with the batch
    a = lib.mla_dcp_decode_fused_workspace_size(64, 64, 16, 1, 4096, 0)
    b = lib.mla_dcp_decode_fused_workspace_size(4096, 4096, 16, 1, 4096, 0)
    assert a == b


@pytest.mark.parametrize("kw,code", [
    (dict(H=0), mla.MLA_ERR_INVALID_ARG),
    (dict(T=-1), mla.MLA_ERR_INVALID_ARG),
    (dict(r=2), mla.MLA_ERR_INVALID_ARG),
    (dict(ms=-5), mla.MLA_ERR_INVALID_ARG),
    (dict(kvdt=7), mla.MLA_ERR_UNSUPPORTED),
])
def test_static_scratch_reports_argument_errors_before_sizing(lib, kw, code):
    """The allocation-free variant checks its arguments before it compares the
    problem's scratch with its array, so a bad size is an argument error, not
    a scratch shortfall (and nothing reaches the GPU)."""
    a = dict(H=16, T=2, r=0, ms=100, kvdt=mla.MLA_DTYPE_BF16)
    a.update(kw)
    rc = lib.mla_dcp_decode_static_scratch(A, 512, A, 64, A, 10, 64, a["kvdt"], A, 4, A, A, 2, a["T"], a["H"], 1,
                                           a["ms"], 2, a["r"], ctypes.c_float(0.07), A, mla.MLA_DTYPE_BF16, A, None, 0,
                                           None)
    assert rc == code, lib.mla_last_error().decode()


def test_fp8_calls_check_their_arguments(lib):
    def call(**kw):
        a = dict(kvs=0.25, H=16, ps=64, kv=A)
        a.update(kw)
        return lib.mla_dcp_decode_fp8(A, 512, A, 64, a["kv"], 10, a["ps"], ctypes.c_float(a["kvs"]), A, 4, A, A, 2, 2,
                                      a["H"], 1, 100, 2, 0, ctypes.c_float(0.07), A, mla.MLA_DTYPE_BF16, A, None, 0, A,
                                      1 << 30, None)
    assert call(kvs=0.0) == mla.MLA_ERR_INVALID_ARG
    assert call(kvs=float("inf")) == mla.MLA_ERR_INVALID_ARG
    assert call(kvs=-1.0) == mla.MLA_ERR_INVALID_ARG
    assert call(H=0) == mla.MLA_ERR_INVALID_ARG
    assert call(ps=12) == mla.MLA_ERR_UNSUPPORTED
    assert call(kv=None) == mla.MLA_ERR_INVALID_ARG
    kvs, nbs, bts = _shard_arrays(2)
    rc = lib.mla_dcp_decode_fused_fp8(A, 512, A, 64, kvs, nbs, 64, ctypes.c_float(0.0), bts, 4, A, A, 2, 2, 16, 1,
                                      100, 2, ctypes.c_float(0.07), A, mla.MLA_DTYPE_BF16, A, 0, A, 1 << 30, None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    # the bf16 calls still refuse an FP8 cache, pointing to these calls
    rc, msg = _decode(lib, kvdt=mla.MLA_DTYPE_FP8_E4M3)
    assert rc == mla.MLA_ERR_UNSUPPORTED and "_fp8" in msg
