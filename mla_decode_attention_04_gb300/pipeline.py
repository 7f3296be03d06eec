"""One DCP decode step on one GPU: the D shard decodes, then the merge.

On one device the D DCP shards are D disjoint slices of the cache in the same
HBM, so the step is D calls of the shard decode (dense or sparse) writing into
one [D, T, H, 512] partial buffer, and one call of the LSE merge (optionally
fused with W_UV).  Everything here is argument marshalling around the C ABI;
all buffers are allocated once by ``DcpStep`` so that a step allocates
nothing and can be captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import (KV_LORA_RANK, V_HEAD_DIM, decode_workspace_size, dcp_lse_merge, fused_workspace_size, mla_dcp_decode,
               mla_dcp_decode_fused, mla_dcp_decode_fused_fp8, mla_sparse_dcp_decode, mla_sparse_dcp_decode_fused,
               sparse_workspace_size)


class DcpStep:
    """Preallocated buffers + the launch sequence of one decode step.

    ``shards``: list of (kv_cache slice, block_table) per DCP rank.
    ``partial_dtype``: dtype of the per-shard outputs handed to the merge.
    ``None`` picks float32 when the merge projects through W_UV (whose
    unit-scale weights amplify input rounding by about sqrt(512)) and bfloat16
    otherwise (the 512-wide merge keeps bf16 partials well inside tolerance).
    """

    def __init__(self, q_nope, q_pe, shards, seq_lens, query_start_loc, max_query_len, max_seq_len, scale, w_uv=None,
                 topk=None, topk_valid=None, partial_dtype=None, out_dtype=torch.bfloat16, num_splits=0,
                 use_counts=True):
        self.q_nope, self.q_pe, self.shards = q_nope, q_pe, shards
        self.seq_lens, self.qsl = seq_lens, query_start_loc
        self.max_query_len, self.max_seq_len, self.scale = int(max_query_len), int(max_seq_len), float(scale)
        self.w_uv, self.topk, self.topk_valid = w_uv, topk, topk_valid
        self.num_splits = num_splits
        self.use_counts = use_counts
        D = len(shards)
        T, H = q_nope.shape[0], q_nope.shape[1]
        dev = q_nope.device
        self.D, self.T, self.H = D, T, H
        if partial_dtype is None:
            partial_dtype = torch.float32 if w_uv is not None else torch.bfloat16
        self.partials = torch.empty((D, T, H, KV_LORA_RANK), dtype=partial_dtype, device=dev)
        self.lses = torch.empty((D, T, H), dtype=torch.float32, device=dev)
        self.counts = torch.empty((D, T), dtype=torch.int32, device=dev)
        width = V_HEAD_DIM if w_uv is not None else KV_LORA_RANK
        self.out = torch.empty((T, H, width), dtype=out_dtype, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        B = seq_lens.shape[0]
        if topk is not None:
            need = sparse_workspace_size(T, H, topk.shape[1], D)
        else:
            need = decode_workspace_size(B, T, H, max_query_len, max_seq_len, D, num_splits)
        self.workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)

    def run(self, stream=None):
        for r, (cache, bt) in enumerate(self.shards):
            if self.topk is not None:
                mla_sparse_dcp_decode(self.q_nope, self.q_pe, cache, bt, self.seq_lens, self.qsl, self.topk,
                                      self.topk_valid, self.D, r, self.scale, out=self.partials[r], lse=self.lses[r],
                                      local_counts=self.counts[r], workspace=self.workspace, stream=stream)
            else:
                mla_dcp_decode(self.q_nope, self.q_pe, cache, bt, self.seq_lens, self.qsl, self.max_query_len,
                               self.max_seq_len, self.D, r, self.scale, out=self.partials[r], lse=self.lses[r],
                               row_counts=self.counts[r], num_splits=self.num_splits, workspace=self.workspace,
                               stream=stream)
        dcp_lse_merge(self.partials, self.lses, self.counts if self.use_counts else None, self.w_uv, out=self.out,
                      lse_out=self.lse, stream=stream)
        return self.out, self.lse


class FusedDcpStep:
    """The step in one decode call over all D shards, followed, with W_UV,
    by the projection (``dcp_lse_merge`` of the one merged result).  Dense:
    ``mla_dcp_decode_fused`` (the online softmax runs over shard 0's keys,
    then shard 1's, ..., which is the LSE merge); sparse (``topk`` given):
    ``mla_sparse_dcp_decode_fused`` (each token over every used entry of its
    list).  Same outputs as ``DcpStep`` (``out``, ``lse``); no per-shard
    partials or counts.  ``kv_scale`` given: the shard caches hold FP8 E4M3
    codes (uint8) with that dequantisation scale (``mla_dcp_decode_fused_fp8``)."""

    def __init__(self, q_nope, q_pe, shards, seq_lens, query_start_loc, max_query_len, max_seq_len, scale, w_uv=None,
                 out_dtype=torch.bfloat16, num_splits=0, topk=None, topk_valid=None, kv_scale=None):
        self.q_nope, self.q_pe = q_nope, q_pe
        self.caches = [c for c, _ in shards]
        self.tables = [bt for _, bt in shards]
        self.seq_lens, self.qsl = seq_lens, query_start_loc
        self.max_query_len, self.max_seq_len, self.scale = int(max_query_len), int(max_seq_len), float(scale)
        self.w_uv, self.num_splits = w_uv, num_splits
        self.kv_scale = None if kv_scale is None else float(kv_scale)
        if self.kv_scale is not None and topk is not None:
            raise ValueError("FP8 caches are served by the dense decode only")
        T, H = q_nope.shape[0], q_nope.shape[1]
        dev = q_nope.device
        self.D, self.T, self.H = len(shards), T, H
        width = V_HEAD_DIM if w_uv is not None else KV_LORA_RANK
        self.out = torch.empty((T, H, width), dtype=out_dtype, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        # with W_UV the merged 512-wide output stays fp32 until the projection
        self.merged = (torch.empty((1, T, H, KV_LORA_RANK), dtype=torch.float32, device=dev)
                       if w_uv is not None else None)
        self.merged_lse = torch.empty((1, T, H), dtype=torch.float32, device=dev) if w_uv is not None else None
        self.topk, self.topk_valid = topk, topk_valid
        # sparse: an int32 [T] tensor here receives each token's used-entry count
        self.kept_counts = None
        if topk is not None:
            need = sparse_workspace_size(T, H, topk.shape[1], self.D)
        else:
            need = fused_workspace_size(seq_lens.shape[0], T, H, max_query_len, max_seq_len, num_splits)
        self.workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)

    def decode(self, out, lse, stream=None):
        """The fused decode call alone, into ``out`` / ``lse``."""
        if self.topk is not None:
            mla_sparse_dcp_decode_fused(self.q_nope, self.q_pe, self.caches, self.tables, self.seq_lens, self.qsl,
                                        self.topk, self.topk_valid, self.scale, out=out, lse=lse,
                                        kept_counts=self.kept_counts, workspace=self.workspace, stream=stream)
        elif self.kv_scale is not None:
            mla_dcp_decode_fused_fp8(self.q_nope, self.q_pe, self.caches, self.kv_scale, self.tables, self.seq_lens,
                                     self.qsl, self.max_query_len, self.max_seq_len, self.scale, out=out, lse=lse,
                                     num_splits=self.num_splits, workspace=self.workspace, stream=stream)
        else:
            mla_dcp_decode_fused(self.q_nope, self.q_pe, self.caches, self.tables, self.seq_lens, self.qsl,
                                 self.max_query_len, self.max_seq_len, self.scale, out=out, lse=lse,
                                 num_splits=self.num_splits, workspace=self.workspace, stream=stream)

    def run(self, stream=None):
        if self.w_uv is None:
            self.decode(self.out, self.lse, stream)
        else:
            self.decode(self.merged[0], self.merged_lse[0], stream)
            dcp_lse_merge(self.merged, self.merged_lse, None, self.w_uv, out=self.out, lse_out=self.lse,
                          stream=stream)
        return self.out, self.lse


def fused_step_for_workload(w, num_splits=0, sparse=None, fp8_caches=None, kv_scale=None):
    """FusedDcpStep for a ``workloads.Workload`` already on the GPU
    (``fp8_caches`` + ``kv_scale``: per-shard FP8 code caches in the
    workload's page layout, in place of its bf16 caches)."""
    sparse = (w.topk is not None) if sparse is None else sparse
    caches = fp8_caches if fp8_caches is not None else [s.cache for s in w.shards]
    shards = [(c, s.block_table) for c, s in zip(caches, w.shards)]
    return FusedDcpStep(w.q_nope, w.q_pe, shards, w.seq_lens, w.query_start_loc, w.max_query_len, w.max_seq_len,
                        w.scale, w_uv=w.w_uv, num_splits=num_splits, topk=w.topk if sparse else None,
                        topk_valid=w.topk_valid if sparse else None,
                        kv_scale=kv_scale if fp8_caches is not None else None)


def step_for_workload(w, partial_dtype=None, num_splits=0, sparse=None):
    """DcpStep for a ``workloads.Workload`` already on the GPU."""
    sparse = (w.topk is not None) if sparse is None else sparse
    shards = [(s.cache, s.block_table) for s in w.shards]
    return DcpStep(w.q_nope, w.q_pe, shards, w.seq_lens, w.query_start_loc, w.max_query_len, w.max_seq_len, w.scale,
                   w_uv=w.w_uv, topk=w.topk if sparse else None, topk_valid=w.topk_valid if sparse else None,
                   partial_dtype=partial_dtype, num_splits=num_splits)
