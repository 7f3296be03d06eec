"""Seeded synthetic inputs for MLA decode attention under DCP.

This module draws inputs and lays them out; it computes none of the
attention, masking or merge arithmetic.  The same tensors (same bf16 bits)
feed the CUDA library and the CPU oracle.

Layout produced (the library's input contract):
  * ``q_nope`` bf16 [T, H, 512], ``q_pe`` bf16 [T, H, 64]: the absorbed query
    split as in the flashattn_mla backend's ``_forward_decode``.
  * one latent KV row per token: kv_c (512) followed by k_pe (64), bf16.
  * DCP interleaving (pages "[Attention] add DCP support for FLASH_ATTN_MLA
    backend", review-thread tables): token p of a request is stored on shard
    p % D in that shard's local slot p // D.  Each shard's rows are paged
    (``page_size`` rows per page) through its own block table; the pages of
    all shards live in one tensor, shard r owning the contiguous slice
    ``cache[page_base[r] : page_base[r] + num_pages[r]]`` whose block-table
    entries are local to the slice.  Page order inside a slice is a seeded
    random permutation.  Unused block-table entries hold 0 (a valid page).
  * ``seq_lens`` are global lengths, new tokens included; query token i of a
    request with q_len new tokens sits at global position seq_len - q_len + i.
  * sparse lists (``topk``): per query token, distinct global positions drawn
    without replacement from that token's visible prefix [0, position], -1
    padded past ``topk_valid``.

Five named workloads mirror the benchmark configurations (tiny, plain
decode, MTP, long context, sparse + mixed); ``custom`` builds any other.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

KV_LORA_RANK = 512
ROPE_DIM = 64
ROW = KV_LORA_RANK + ROPE_DIM
V_HEAD_DIM = 128
SOFTMAX_SCALE = 1.0 / math.sqrt(128 + 64)  # (qk_nope_head_dim + qk_rope_head_dim) ** -0.5


@dataclass
class Shard:
    cache: torch.Tensor        # bf16 [num_pages, page_size, 576] (a view into Workload.cache_all)
    block_table: torch.Tensor  # int32 [B, W]
    page_base: int             # first page of this shard in Workload.cache_all


@dataclass
class Workload:
    name: str
    seed: int
    seq_lens: torch.Tensor          # int32 [B]
    query_start_loc: torch.Tensor   # int32 [B+1]
    q_nope: torch.Tensor            # bf16 [T, H, 512]
    q_pe: torch.Tensor              # bf16 [T, H, 64]
    cache_all: torch.Tensor         # bf16 [total_pages, ps, 576]
    shards: list                    # [Shard] * D
    dcp_world: int
    page_size: int
    scale: float
    w_uv: torch.Tensor | None = None        # bf16 [H, 512, 128]
    topk: torch.Tensor | None = None        # int32 [T, K]
    topk_valid: torch.Tensor | None = None  # int32 [T]
    kv_logical: torch.Tensor | None = None  # bf16 [sum L, 576] (kept only when asked)
    kv_start: torch.Tensor | None = None    # int64 [B]
    meta: dict = field(default_factory=dict)

    @property
    def num_requests(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_nope.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q_nope.shape[1])

    @property
    def max_query_len(self) -> int:
        return int(self.meta["max_query_len"])

    @property
    def max_seq_len(self) -> int:
        return int(self.meta["max_seq_len"])

    def to(self, device) -> "Workload":
        def mv(x):
            return None if x is None else x.to(device)
        cache_all = self.cache_all.to(device)
        shards = []
        for s in self.shards:
            n = s.cache.shape[0]
            shards.append(Shard(cache_all[s.page_base:s.page_base + n], s.block_table.to(device), s.page_base))
        return Workload(self.name, self.seed, mv(self.seq_lens), mv(self.query_start_loc), mv(self.q_nope),
                        mv(self.q_pe), cache_all, shards, self.dcp_world, self.page_size, self.scale, mv(self.w_uv),
                        mv(self.topk), mv(self.topk_valid), mv(self.kv_logical), mv(self.kv_start), dict(self.meta))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _randn(gen, shape, device, scale=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def custom(seq_lens, q_lens, num_heads, dcp_world, page_size=64, seed=0, q_std=1.0, with_w_uv=True, topk=None,
           short_valid_frac=0.0, force_zero_valid=0, device="cpu", keep_logical=True, name="custom",
           spare_pages=0):
    """Build a workload from explicit per-request lengths.

    seq_lens[b] (global) >= q_lens[b] >= 0.  ``topk`` (int) adds sparse lists
    of that length; ``short_valid_frac`` of the tokens get a valid count drawn
    uniformly below topk, of which ``force_zero_valid`` are forced to 0.
    """
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(seq_lens) == len(q_lens)
    for L, q in zip(seq_lens, q_lens):
        assert 0 <= q <= L, (L, q)
    B, H, D, ps = len(seq_lens), int(num_heads), int(dcp_world), int(page_size)
    T = sum(q_lens)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    cpu_rng = np.random.default_rng(seed)

    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    q_nope = _randn(gen, (T, H, KV_LORA_RANK), device, q_std)
    q_pe = _randn(gen, (T, H, ROPE_DIM), device, q_std)

    kv_start = np.zeros(B, dtype=np.int64)
    kv_start[1:] = np.cumsum(seq_lens)[:-1]
    total_L = int(sum(seq_lens))
    kv_logical = _randn(gen, (max(total_L, 1), ROW), device)

    # DCP interleaving: token p -> shard p % D, local slot p // D; pages per shard.
    shard_tokens = []  # per shard: list per request of the logical token ids in local order
    for r in range(D):
        shard_tokens.append([np.arange(r, L, D, dtype=np.int64) for L in seq_lens])
    pages_per_req = [[-(-len(tok) // ps) for tok in shard_tokens[r]] for r in range(D)]
    # every shard owns at least one page (a cache allocation is never empty)
    num_pages = [max(1, sum(p) + spare_pages) for p in pages_per_req]
    page_base = np.zeros(D, dtype=np.int64)
    page_base[1:] = np.cumsum(num_pages)[:-1]
    total_pages = max(1, int(sum(num_pages)))
    cache_all = torch.zeros((total_pages, ps, ROW), dtype=torch.bfloat16, device=device)
    flat = cache_all.view(-1, ROW)
    shards = []
    for r in range(D):
        # one row width for every shard's table (the fused calls take one stride)
        W = max(1, max(max(p) for p in pages_per_req) if B else 1)
        bt = np.zeros((B, W), dtype=np.int32)
        perm = cpu_rng.permutation(num_pages[r]).astype(np.int64)
        off = 0
        dst_rows, src_rows = [], []
        for b in range(B):
            npg = pages_per_req[r][b]
            pages = perm[off:off + npg]
            off += npg
            bt[b, :npg] = pages
            tok = shard_tokens[r][b]
            if len(tok):
                j = np.arange(len(tok), dtype=np.int64)
                dst_rows.append((page_base[r] + pages[j // ps]) * ps + j % ps)
                src_rows.append(kv_start[b] + tok)
        if dst_rows:
            dst = torch.from_numpy(np.concatenate(dst_rows)).to(device)
            src = torch.from_numpy(np.concatenate(src_rows)).to(device)
            flat.index_copy_(0, dst, kv_logical.index_select(0, src))
        cache_r = cache_all[int(page_base[r]):int(page_base[r]) + num_pages[r]]
        shards.append(Shard(cache_r, torch.from_numpy(bt).to(device), int(page_base[r])))

    w_uv = _randn(gen, (H, KV_LORA_RANK, V_HEAD_DIM), device) if with_w_uv else None

    topk_t = valid_t = None
    if topk:
        K = int(topk)
        idx = np.full((T, K), -1, dtype=np.int32)
        valid = np.zeros(T, dtype=np.int32)
        t = 0
        for b in range(B):
            for i in range(q_lens[b]):
                pos = seq_lens[b] - q_lens[b] + i
                n = min(K, pos + 1)
                idx[t, :n] = cpu_rng.choice(pos + 1, size=n, replace=False)
                valid[t] = n
                t += 1
        if T and short_valid_frac > 0:
            nshort = max(1, int(round(short_valid_frac * T)))
            rows = cpu_rng.choice(T, size=nshort, replace=False)
            for k, row in enumerate(rows):
                v = 0 if k < force_zero_valid else int(cpu_rng.integers(0, K))
                valid[row] = min(valid[row], v)
        for row in range(T):
            idx[row, valid[row]:] = -1
        topk_t = torch.from_numpy(idx).to(device)
        valid_t = torch.from_numpy(valid).to(device)

    meta = dict(q_lens=q_lens, max_query_len=max(q_lens) if B else 0, max_seq_len=max(seq_lens) if B else 0,
                num_pages=num_pages, total_L=total_L)
    return Workload(name, seed, torch.tensor(seq_lens, dtype=torch.int32, device=device),
                    torch.from_numpy(qsl).to(device), q_nope, q_pe, cache_all, shards, D, ps, SOFTMAX_SCALE, w_uv,
                    topk_t, valid_t, kv_logical if keep_logical else None,
                    torch.from_numpy(kv_start).to(device) if keep_logical else None, meta)


# --------------------------------------------------------------- named configs


def fp8_cache(w: "Workload", kv_scale: float = 0.25):
    """An FP8 E4M3 latent cache for workload w: the bf16 cache values divided
    by ``kv_scale`` and rounded to E4M3 codes (torch's float8_e4m3fn cast),
    stored as uint8 [total_pages, page_size, 576] in the same page layout (a
    shard's slice at the same page range).  Returns (codes, per-shard views).
    Input drawing only: the cache holds kv_scale * decode(code), a value
    near the bf16 draw."""
    x = w.cache_all.float() / float(kv_scale)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
    views = [codes[s.page_base:s.page_base + s.cache.shape[0]] for s in w.shards]
    return codes, views


def e4m3_values(codes: torch.Tensor) -> torch.Tensor:
    """float32 values of uint8 E4M3 codes (torch's float8_e4m3fn widening)."""
    return codes.view(torch.float8_e4m3fn).float()


def tiny(device="cpu", **kw):
    """4 requests, lengths {6,37,130,300}, q_len {4,1,2,2} (request 0 is the
    6-key / 4-query case of the mask tables), D=2, H=16, page 16, q scaled by
    1/sqrt(576), seed 0."""
    args = dict(seq_lens=[6, 37, 130, 300], q_lens=[4, 1, 2, 2], num_heads=16, dcp_world=2, page_size=16, seed=0,
                q_std=1.0 / math.sqrt(576.0), with_w_uv=True, device=device, name="tiny")
    args.update(kw)
    return custom(**args)


def plain_decode(dcp_world=2, device="cpu", batch=64, context=4096, **kw):
    """batch 64, q_len 1, H=16, context 4096 each, D in {1, 2}, page 64."""
    args = dict(seq_lens=[context] * batch, q_lens=[1] * batch, num_heads=16, dcp_world=dcp_world, page_size=64,
                seed=1, with_w_uv=False, device=device, keep_logical=False, name=f"plain_decode_d{dcp_world}")
    args.update(kw)
    return custom(**args)


def mtp(device="cpu", batch=128, lo=1024, hi=8192, **kw):
    """batch 128, q_len 2, H=16, context ~ U[1024, 8192], D=4, page 64, W_UV."""
    rng = np.random.default_rng(2)
    L = rng.integers(lo, hi + 1, size=batch).tolist()
    args = dict(seq_lens=L, q_lens=[2] * batch, num_heads=16, dcp_world=4, page_size=64, seed=2, with_w_uv=True,
                device=device, keep_logical=False, name="mtp")
    args.update(kw)
    return custom(**args)


def long_context(device="cpu", batch=32, lo=16384, hi=32768, **kw):
    """batch 32, q_len 2, H=128, context ~ U[16384, 32768], D=8, page 64, W_UV."""
    rng = np.random.default_rng(3)
    L = rng.integers(lo, hi + 1, size=batch).tolist()
    args = dict(seq_lens=L, q_lens=[2] * batch, num_heads=128, dcp_world=8, page_size=64, seed=3, with_w_uv=True,
                device=device, keep_logical=False, name="long_context")
    args.update(kw)
    return custom(**args)


def sparse_mixed(device="cpu", n_decode=96, n_prefill=4, prefill_len=64, lo=4096, hi=65536, topk=2048, **kw):
    """96 requests with q_len in {1, 2, 4} plus 4 chunked-prefill requests of
    64 query tokens, H=64, context ~ U[4096, 65536], top-k 2048 per query
    token, 10% of tokens with fewer valid entries (at least one with 0), D=4,
    page 64, W_UV."""
    rng = np.random.default_rng(4)
    q = rng.choice([1, 2, 4], size=n_decode).tolist() + [prefill_len] * n_prefill
    L = rng.integers(lo, hi + 1, size=n_decode + n_prefill).tolist()
    args = dict(seq_lens=L, q_lens=q, num_heads=64, dcp_world=4, page_size=64, seed=4, with_w_uv=True, topk=topk,
                short_valid_frac=0.10, force_zero_valid=max(1, (sum(q) + 99) // 100), device=device,
                keep_logical=False, name="sparse_mixed")
    args.update(kw)
    return custom(**args)


def sparse_mixed_profile(device="cpu", **kw):
    """The sparse + mixed recipe at a size an ncu capture replays quickly:
    24 decode requests plus 1 chunked prefill, context ~ U[4096, 16384]
    (cache ~0.3 GB, still larger than L2)."""
    args = dict(n_decode=24, n_prefill=1, lo=4096, hi=16384, name="sparse_mixed_profile")
    args.update(kw)
    return sparse_mixed(device=device, **args)


NAMED = {
    "tiny": tiny,
    "plain_decode_d1": lambda **kw: plain_decode(dcp_world=1, **kw),
    "plain_decode_d2": lambda **kw: plain_decode(dcp_world=2, **kw),
    "mtp": mtp,
    "long_context": long_context,
    "sparse_mixed": sparse_mixed,
    "sparse_mixed_profile": sparse_mixed_profile,
}
