"""GB300 (sm_103a) absorbed-MLA paged decode attention under decode context
parallelism (DCP).

The compute lives in the CUDA library ``libmla_dcp.so`` behind the C ABI of
``include/mla_dcp.h``.  This module is a thin ctypes binding with the same
names: it checks tensor shapes/dtypes, allocates outputs and workspace with
torch when the caller does not pass them, and forwards raw device pointers,
sizes and the current CUDA stream.  Every step of the computation runs in the
library's kernels; there is no other implementation to fall back to, and a
missing or unloadable library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import workloads  # noqa: F401  (seeded inputs; no kernel arithmetic)

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_dcp.so")

KV_LORA_RANK = 512
ROPE_DIM = 64
V_HEAD_DIM = 128

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_WORKSPACE, MLA_ERR_DEVICE_CHECK = range(6)
MLA_DTYPE_BF16, MLA_DTYPE_F32, MLA_DTYPE_FP8_E4M3 = 0, 1, 2

EXPORTS = [
    "mla_last_error", "mla_dcp_decode_workspace_size", "mla_dcp_decode", "mla_sparse_dcp_decode_workspace_size",
    "mla_sparse_dcp_decode", "dcp_lse_merge", "mla_workspace_status", "mla_kernel_launch_count",
    "mla_dcp_decode_static_scratch", "mla_dcp_decode_fused_workspace_size", "mla_dcp_decode_fused",
    "mla_sparse_dcp_decode_fused", "mla_dcp_decode_fp8", "mla_dcp_decode_fused_fp8", "mla_debug_set_wait_budget_ns",
    "mla_dcp_decode_two_stage_workspace_size", "mla_dcp_decode_two_stage",
]

# Size of the library's fixed device scratch array used by
# mla_dcp_decode_static_scratch (the entry point for callers that cannot
# allocate device memory); see include/mla_dcp.h.
MLA_STATIC_SCRATCH_BYTES = 24 * 1024 * 1024


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None


def _bind(lib):
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.mla_last_error.restype = ctypes.c_char_p
    lib.mla_last_error.argtypes = []
    lib.mla_dcp_decode_workspace_size.restype = sz
    lib.mla_dcp_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.mla_dcp_decode.restype = ctypes.c_int
    lib.mla_dcp_decode.argtypes = [vp, i64, vp, i64, vp, i64, i32, i32, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                   i32, f32, vp, i32, vp, vp, i32, vp, sz, vp]
    lib.mla_sparse_dcp_decode_workspace_size.restype = sz
    lib.mla_sparse_dcp_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.mla_sparse_dcp_decode.restype = ctypes.c_int
    lib.mla_sparse_dcp_decode.argtypes = [vp, i64, vp, i64, vp, i64, i32, i32, vp, i32, vp, vp, i32, i32, i32, vp,
                                          i32, vp, i32, i32, f32, vp, i32, vp, vp, vp, sz, vp]
    lib.dcp_lse_merge.restype = ctypes.c_int
    lib.dcp_lse_merge.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, vp, i32, vp, vp]
    lib.mla_workspace_status.restype = ctypes.c_int
    lib.mla_workspace_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.mla_kernel_launch_count.restype = i64
    lib.mla_kernel_launch_count.argtypes = []
    lib.mla_dcp_decode_fused_workspace_size.restype = sz
    lib.mla_dcp_decode_fused_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.mla_dcp_decode_fused.restype = ctypes.c_int
    lib.mla_dcp_decode_fused.argtypes = [vp, i64, vp, i64, vp, vp, i32, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                         i32, i32, ctypes.c_float, vp, i32, vp, i32, vp, sz, vp]
    lib.mla_sparse_dcp_decode_fused.restype = ctypes.c_int
    lib.mla_sparse_dcp_decode_fused.argtypes = [vp, i64, vp, i64, vp, vp, i32, i32, vp, i32, vp, vp, i32, i32, i32,
                                                vp, i32, vp, i32, f32, vp, i32, vp, vp, vp, sz, vp]
    lib.mla_dcp_decode_fp8.restype = ctypes.c_int
    lib.mla_dcp_decode_fp8.argtypes = [vp, i64, vp, i64, vp, i64, i32, f32, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                       i32, i32, f32, vp, i32, vp, vp, i32, vp, sz, vp]
    lib.mla_dcp_decode_fused_fp8.restype = ctypes.c_int
    lib.mla_dcp_decode_fused_fp8.argtypes = [vp, i64, vp, i64, vp, vp, i32, f32, vp, i32, vp, vp, i32, i32, i32, i32,
                                             i32, i32, f32, vp, i32, vp, i32, vp, sz, vp]
    lib.mla_dcp_decode_two_stage_workspace_size.restype = sz
    lib.mla_dcp_decode_two_stage_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.mla_dcp_decode_two_stage.restype = ctypes.c_int
    lib.mla_dcp_decode_two_stage.argtypes = [vp, i64, vp, i64, vp, vp, i32, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                             i32, i32, f32, vp, i32, vp, vp, sz, vp]
    lib.mla_debug_set_wait_budget_ns.restype = None
    lib.mla_debug_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
    lib.mla_dcp_decode_static_scratch.restype = ctypes.c_int
    lib.mla_dcp_decode_static_scratch.argtypes = [vp, i64, vp, i64, vp, i64, i32, i32, vp, i32, vp, vp, i32, i32, i32,
                                                  i32, i32, i32, i32, f32, vp, i32, vp, vp, i32, vp]
    return lib


def load_library(path: str | None = None):
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with mla_decode_attention_04_gb300.build.build()")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def _check(rc: int):
    if rc != MLA_OK:
        raise MlaError(rc, load_library().mla_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


_DT = {torch.bfloat16: MLA_DTYPE_BF16, torch.float32: MLA_DTYPE_F32}


def _row_stride(q, width, name):
    if q.dim() != 3 or q.shape[2] != width or q.stride(2) != 1 or q.stride(0) != q.shape[1] * q.stride(1):
        raise ValueError(f"{name} must be [T, H, {width}] with unit last stride and rows of equal stride")
    return q.stride(1)


def _i32(t, name):
    if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def workspace_wait_site(workspace) -> int:
    """The workspace header's diagnostic word: the site of the first pipeline
    wait that gave up (0 if none); read after mla_workspace_status."""
    return int(workspace[8:12].view(torch.int32).item())


def decode_workspace_size(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, dcp_world,
                          num_splits=0) -> int:
    return int(load_library().mla_dcp_decode_workspace_size(num_requests, num_tokens, num_heads, max_query_len,
                                                             max_seq_len, dcp_world, num_splits))


def sparse_workspace_size(num_tokens, num_heads, topk, dcp_world) -> int:
    return int(load_library().mla_sparse_dcp_decode_workspace_size(num_tokens, num_heads, topk, dcp_world))


def _kv_args(kv_cache):
    if kv_cache.dim() != 3 or kv_cache.shape[2] != KV_LORA_RANK + ROPE_DIM or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be a contiguous [num_blocks, page_size, 576] tensor")
    dt = {torch.bfloat16: MLA_DTYPE_BF16}.get(kv_cache.dtype, MLA_DTYPE_FP8_E4M3)
    return kv_cache.shape[0], kv_cache.shape[1], dt


def mla_dcp_decode(q_nope, q_pe, kv_cache, block_table, seq_lens, query_start_loc, max_query_len, max_seq_len,
                   dcp_world, dcp_rank, scale, out=None, lse=None, row_counts=None, out_dtype=torch.bfloat16,
                   num_splits=0, workspace=None, stream=None, return_counts=True):
    """Dense DCP shard decode.  Returns (out [T,H,512], lse [T,H], row_counts [T])."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    nb, ps, kv_dt = _kv_args(kv_cache)
    _i32(block_table, "block_table"), _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if row_counts is None and return_counts:
        row_counts = torch.empty((T,), dtype=torch.int32, device=dev)
    if workspace is None:  # (the library checks a given workspace's size itself)
        need = decode_workspace_size(B, T, H, max_query_len, max_seq_len, dcp_world, num_splits)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    _check(lib.mla_dcp_decode(_ptr(q_nope), sn, _ptr(q_pe), sp, _ptr(kv_cache), nb, ps, kv_dt, _ptr(block_table),
                              block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), B, T, H,
                              int(max_query_len), int(max_seq_len), int(dcp_world), int(dcp_rank), float(scale),
                              _ptr(out), _DT[out.dtype], _ptr(lse), _ptr(row_counts), int(num_splits),
                              _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse, row_counts


def _kv8(kv_cache):
    if (kv_cache.dtype != torch.uint8 or kv_cache.dim() != 3 or kv_cache.shape[2] != KV_LORA_RANK + ROPE_DIM
            or not kv_cache.is_contiguous()):
        raise ValueError("an FP8 kv_cache must be a contiguous uint8 [num_blocks, page_size, 576] tensor of E4M3 codes")
    return kv_cache.shape[0], kv_cache.shape[1]


def mla_dcp_decode_fp8(q_nope, q_pe, kv_cache, kv_scale, block_table, seq_lens, query_start_loc, max_query_len,
                       max_seq_len, dcp_world, dcp_rank, scale, out=None, lse=None, row_counts=None,
                       out_dtype=torch.bfloat16, num_splits=0, workspace=None, stream=None):
    """mla_dcp_decode over an FP8 E4M3 cache (uint8 codes, value = kv_scale *
    decode(code)).  Returns (out [T,H,512], lse [T,H], row_counts [T])."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    nb, ps = _kv8(kv_cache)
    _i32(block_table, "block_table"), _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if row_counts is None:
        row_counts = torch.empty((T,), dtype=torch.int32, device=dev)
    if workspace is None:  # (the size query covers the bf16 and FP8 calls)
        need = decode_workspace_size(B, T, H, max_query_len, max_seq_len, dcp_world, num_splits)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    _check(lib.mla_dcp_decode_fp8(_ptr(q_nope), sn, _ptr(q_pe), sp, _ptr(kv_cache), nb, ps, float(kv_scale),
                                  _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), B, T,
                                  H, int(max_query_len), int(max_seq_len), int(dcp_world), int(dcp_rank),
                                  float(scale), _ptr(out), _DT[out.dtype], _ptr(lse), _ptr(row_counts),
                                  int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))
    return out, lse, row_counts


def mla_dcp_decode_fused_fp8(q_nope, q_pe, kv_caches, kv_scale, block_tables, seq_lens, query_start_loc,
                             max_query_len, max_seq_len, scale, out=None, lse=None, out_dtype=torch.bfloat16,
                             num_splits=0, workspace=None, stream=None):
    """mla_dcp_decode_fused over FP8 E4M3 shard caches (uint8 codes, value =
    kv_scale * decode(code)).  Returns the merged (out [T,H,512], lse [T,H])."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    D = len(kv_caches)
    if len(block_tables) != D or D < 1:
        raise ValueError("kv_caches and block_tables need one entry per shard")
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    kv_args = [_kv8(c) for c in kv_caches]
    ps = kv_args[0][1]
    if any(a[1] != ps for a in kv_args):
        raise ValueError("all shard caches need the same page size")
    bt_stride = block_tables[0].shape[1]
    for bt in block_tables:
        _i32(bt, "block_table")
        if bt.shape[1] != bt_stride:
            raise ValueError("all block tables need the same row stride")
    _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if workspace is None:
        need = fused_workspace_size(B, T, H, max_query_len, max_seq_len, num_splits)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    kv_ptrs = (ctypes.c_void_p * D)(*[c.data_ptr() for c in kv_caches])
    nbs = (ctypes.c_int64 * D)(*[a[0] for a in kv_args])
    bt_ptrs = (ctypes.c_void_p * D)(*[bt.data_ptr() for bt in block_tables])
    _check(lib.mla_dcp_decode_fused_fp8(_ptr(q_nope), sn, _ptr(q_pe), sp, ctypes.cast(kv_ptrs, ctypes.c_void_p),
                                        ctypes.cast(nbs, ctypes.c_void_p), ps, float(kv_scale),
                                        ctypes.cast(bt_ptrs, ctypes.c_void_p), bt_stride, _ptr(seq_lens),
                                        _ptr(query_start_loc), B, T, H, int(max_query_len), int(max_seq_len), D,
                                        float(scale), _ptr(out), _DT[out.dtype], _ptr(lse), int(num_splits),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))
    return out, lse


def fused_workspace_size(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, num_splits=0) -> int:
    return int(load_library().mla_dcp_decode_fused_workspace_size(num_requests, num_tokens, num_heads, max_query_len,
                                                                   max_seq_len, num_splits))


def two_stage_workspace_size(num_requests, num_tokens, num_heads, max_query_len, max_seq_len) -> int:
    return int(load_library().mla_dcp_decode_two_stage_workspace_size(num_requests, num_tokens, num_heads,
                                                                       max_query_len, max_seq_len))


def mla_dcp_decode_two_stage(q_nope, q_pe, kv_caches, block_tables, seq_lens, query_start_loc, max_query_len,
                             max_seq_len, scale, out=None, lse=None, out_dtype=torch.bfloat16, workspace=None,
                             stream=None):
    """The two-stage decomposition of the step over all D shards: each
    query row over its request's context without a mask, then over the new
    keys up to its own position, the two merged by LSE.  Returns the merged
    (out [T,H,512], lse [T,H]); equals ``mla_dcp_decode_fused`` up to
    rounding."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    D = len(kv_caches)
    if len(block_tables) != D or D < 1:
        raise ValueError("kv_caches and block_tables need one entry per shard")
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    kv_args = [_kv_args(c) for c in kv_caches]
    ps, kv_dt = kv_args[0][1], kv_args[0][2]
    if any(a[1] != ps or a[2] != kv_dt for a in kv_args):
        raise ValueError("all shard caches need the same page size and dtype")
    bt_stride = block_tables[0].shape[1]
    for bt in block_tables:
        _i32(bt, "block_table")
        if bt.shape[1] != bt_stride:
            raise ValueError("all block tables need the same row stride")
    _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if workspace is None:  # (the library checks a given workspace's size itself)
        need = two_stage_workspace_size(B, T, H, max_query_len, max_seq_len)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    kv_ptrs = (ctypes.c_void_p * D)(*[c.data_ptr() for c in kv_caches])
    nbs = (ctypes.c_int64 * D)(*[a[0] for a in kv_args])
    bt_ptrs = (ctypes.c_void_p * D)(*[bt.data_ptr() for bt in block_tables])
    _check(lib.mla_dcp_decode_two_stage(_ptr(q_nope), sn, _ptr(q_pe), sp, ctypes.cast(kv_ptrs, ctypes.c_void_p),
                                        ctypes.cast(nbs, ctypes.c_void_p), ps, kv_dt,
                                        ctypes.cast(bt_ptrs, ctypes.c_void_p), bt_stride, _ptr(seq_lens),
                                        _ptr(query_start_loc), B, T, H, int(max_query_len), int(max_seq_len), D,
                                        float(scale), _ptr(out), _DT[out.dtype], _ptr(lse), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def mla_dcp_decode_fused(q_nope, q_pe, kv_caches, block_tables, seq_lens, query_start_loc, max_query_len,
                         max_seq_len, scale, out=None, lse=None, out_dtype=torch.bfloat16, num_splits=0,
                         workspace=None, stream=None):
    """All D DCP shards of a decode step in one launch: the shard caches and
    block tables (lists of D tensors) are read in turn by one online softmax,
    which is the LSE merge over the shards.  Returns the merged (out
    [T,H,512], lse [T,H])."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    D = len(kv_caches)
    if len(block_tables) != D or D < 1:
        raise ValueError("kv_caches and block_tables need one entry per shard")
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    kv_args = [_kv_args(c) for c in kv_caches]
    ps, kv_dt = kv_args[0][1], kv_args[0][2]
    if any(a[1] != ps or a[2] != kv_dt for a in kv_args):
        raise ValueError("all shard caches need the same page size and dtype")
    bt_stride = block_tables[0].shape[1]
    for bt in block_tables:
        _i32(bt, "block_table")
        if bt.shape[1] != bt_stride:
            raise ValueError("all block tables need the same row stride")
    _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if workspace is None:  # (the library checks a given workspace's size itself)
        need = fused_workspace_size(B, T, H, max_query_len, max_seq_len, num_splits)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    kv_ptrs = (ctypes.c_void_p * D)(*[c.data_ptr() for c in kv_caches])
    nbs = (ctypes.c_int64 * D)(*[a[0] for a in kv_args])
    bt_ptrs = (ctypes.c_void_p * D)(*[bt.data_ptr() for bt in block_tables])
    _check(lib.mla_dcp_decode_fused(_ptr(q_nope), sn, _ptr(q_pe), sp, ctypes.cast(kv_ptrs, ctypes.c_void_p),
                                    ctypes.cast(nbs, ctypes.c_void_p), ps, kv_dt,
                                    ctypes.cast(bt_ptrs, ctypes.c_void_p), bt_stride, _ptr(seq_lens),
                                    _ptr(query_start_loc), B, T, H, int(max_query_len), int(max_seq_len), D,
                                    float(scale), _ptr(out), _DT[out.dtype], _ptr(lse), int(num_splits),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def mla_sparse_dcp_decode_fused(q_nope, q_pe, kv_caches, block_tables, seq_lens, query_start_loc, topk_indices,
                                topk_valid, scale, out=None, lse=None, kept_counts=None, out_dtype=torch.bfloat16,
                                workspace=None, stream=None):
    """Sparse decode of all D DCP shards in one call (the shard caches and
    block tables are lists of D tensors): each token attends over every used
    entry of its list, which is the merge of the D shard results.  Returns
    the merged (out [T,H,512], lse [T,H], kept_counts [T] or None)."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    D = len(kv_caches)
    if len(block_tables) != D or D < 1:
        raise ValueError("kv_caches and block_tables need one entry per shard")
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    kv_args = [_kv_args(c) for c in kv_caches]
    ps, kv_dt = kv_args[0][1], kv_args[0][2]
    if any(a[1] != ps or a[2] != kv_dt for a in kv_args):
        raise ValueError("all shard caches need the same page size and dtype")
    bt_stride = block_tables[0].shape[1]
    for bt in block_tables:
        _i32(bt, "block_table")
        if bt.shape[1] != bt_stride:
            raise ValueError("all block tables need the same row stride")
    _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    _i32(topk_indices, "topk_indices"), _i32(topk_valid, "topk_valid")
    K = topk_indices.shape[1]
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if workspace is None:  # (the library checks a given workspace's size itself)
        need = sparse_workspace_size(T, H, K, D)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    kv_ptrs = (ctypes.c_void_p * D)(*[c.data_ptr() for c in kv_caches])
    nbs = (ctypes.c_int64 * D)(*[a[0] for a in kv_args])
    bt_ptrs = (ctypes.c_void_p * D)(*[bt.data_ptr() for bt in block_tables])
    _check(lib.mla_sparse_dcp_decode_fused(_ptr(q_nope), sn, _ptr(q_pe), sp, ctypes.cast(kv_ptrs, ctypes.c_void_p),
                                           ctypes.cast(nbs, ctypes.c_void_p), ps, kv_dt,
                                           ctypes.cast(bt_ptrs, ctypes.c_void_p), bt_stride, _ptr(seq_lens),
                                           _ptr(query_start_loc), B, T, H, _ptr(topk_indices), K, _ptr(topk_valid), D,
                                           float(scale), _ptr(out), _DT[out.dtype], _ptr(lse), _ptr(kept_counts),
                                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))
    return out, lse, kept_counts


def mla_sparse_dcp_decode(q_nope, q_pe, kv_cache, block_table, seq_lens, query_start_loc, topk_indices, topk_valid,
                          dcp_world, dcp_rank, scale, out=None, lse=None, local_counts=None, out_dtype=torch.bfloat16,
                          workspace=None, stream=None):
    """Sparse (top-k list) DCP shard decode.  Returns (out, lse, local_counts)."""
    lib = load_library()
    T, H = q_nope.shape[0], q_nope.shape[1]
    B = seq_lens.shape[0]
    sn, sp = _row_stride(q_nope, KV_LORA_RANK, "q_nope"), _row_stride(q_pe, ROPE_DIM, "q_pe")
    nb, ps, kv_dt = _kv_args(kv_cache)
    _i32(block_table, "block_table"), _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc")
    _i32(topk_indices, "topk_indices"), _i32(topk_valid, "topk_valid")
    K = topk_indices.shape[1]
    dev = q_nope.device
    if out is None:
        out = torch.empty((T, H, KV_LORA_RANK), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if local_counts is None:
        local_counts = torch.empty((T,), dtype=torch.int32, device=dev)
    if workspace is None:  # (the library checks a given workspace's size itself)
        need = sparse_workspace_size(T, H, K, dcp_world)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    _check(lib.mla_sparse_dcp_decode(_ptr(q_nope), sn, _ptr(q_pe), sp, _ptr(kv_cache), nb, ps, kv_dt,
                                     _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
                                     B, T, H, _ptr(topk_indices), K, _ptr(topk_valid), int(dcp_world), int(dcp_rank),
                                     float(scale), _ptr(out), _DT[out.dtype], _ptr(lse), _ptr(local_counts),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse, local_counts


def dcp_lse_merge(partials, lses, valid_counts=None, w_uv=None, out=None, lse_out=None, out_dtype=torch.bfloat16,
                  stream=None, return_lse=True):
    """LSE merge of [D, T, H, 512] partials (+ optional W_UV [H, 512, 128]).
    Returns (out [T, H, 512 or 128], lse [T, H] or None)."""
    lib = load_library()
    D, T, H, W = partials.shape
    if W != KV_LORA_RANK or not partials.is_contiguous():
        raise ValueError("partials must be a contiguous [D, T, H, 512] tensor")
    if lses.shape != (D, T, H) or lses.dtype != torch.float32 or not lses.is_contiguous():
        raise ValueError("lses must be a contiguous float32 [D, T, H] tensor")
    if valid_counts is not None and (valid_counts.shape != (D, T) or valid_counts.dtype != torch.int32):
        raise ValueError("valid_counts must be int32 [D, T]")
    if w_uv is not None and (w_uv.shape != (H, KV_LORA_RANK, V_HEAD_DIM) or w_uv.dtype != torch.bfloat16
                             or not w_uv.is_contiguous()):
        raise ValueError("w_uv must be a contiguous bf16 [H, 512, 128] tensor")
    width = V_HEAD_DIM if w_uv is not None else KV_LORA_RANK
    if out is None:
        out = torch.empty((T, H, width), dtype=out_dtype, device=partials.device)
    if lse_out is None and return_lse:
        lse_out = torch.empty((T, H), dtype=torch.float32, device=partials.device)
    _check(lib.dcp_lse_merge(_ptr(partials), _DT[partials.dtype], _ptr(lses), _ptr(valid_counts), _ptr(w_uv), D, T, H,
                             _ptr(out), _DT[out.dtype], _ptr(lse_out), _stream(stream)))
    return out, lse_out


def kernel_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().mla_kernel_launch_count())


def workspace_status(workspace, stream=None):
    """Synchronise and read the kernels' status word: (status, detail)."""
    lib = load_library()
    detail = ctypes.c_int32(0)
    rc = lib.mla_workspace_status(_ptr(workspace), _stream(stream), ctypes.byref(detail))
    return rc, detail.value
