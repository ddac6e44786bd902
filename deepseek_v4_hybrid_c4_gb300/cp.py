"""Context-parallel split of one request's C4 decode step over R ranks ("SGLang 如何为
DeepSeek V4 打造「Day-0」推理加速", sec. "3.1 长上下文预填充：Context Parallelism (CP)").

Rank r holds the contiguous candidate range [lo_r, hi_r) of the request -- its index-key rows
and compressed rows -- and the last rank also the raw rows of the sliding window.  A step:

  1. local:    csa_index_score over the range, csa_topk with keys (sorted, local indices);
  2. exchange: all-gather of the R (key, index) lists, rank order;
  3. local:    csa_topk_merge -> the exact global top k and the rows of it this rank holds;
  4. local:    csa_sparse_attn_partial over those rows (+ the window on the last rank);
  5. exchange: all-gather of the R partials (fp32 rows, lse), then csa_attn_merge.

Every computation runs in libcsa's kernels; this module holds the per-rank buffers, passes
pointers and moves the exchanged tensors.  An exchange object provides `world` and
`all_gather(t)` -> the ranks' tensors concatenated along dim 0 in rank order:
TorchDistExchange uses torch.distributed (NCCL between GPUs, gloo between CPU processes);
`run_local` runs R shards on one device, the exchanges being concatenations.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import (CSA_BF16, csa_attn_merge, csa_index_score, csa_paged, csa_sparse_attn_partial,
               csa_sparse_attn_workspace_size, csa_topk, csa_topk_merge, csa_topk_merge_workspace_size,
               csa_topk_workspace_size)


@dataclass
class CPShard:
    """Rank `rank`'s share of one request (device tensors through csa_paged descriptors)."""
    rank: int
    world: int
    rank_lo: torch.Tensor        # device int64 [world + 1]: the ranks' candidate ranges
    lo: int                      # this rank's range [lo, hi) (host copies of rank_lo[rank], [rank + 1])
    hi: int
    kidx: csa_paged              # index-key rows of [lo, hi) (bf16 or fp8), local row ids 0 .. hi - lo - 1
    kv_c: csa_paged              # compressed rows of [lo, hi), same local row ids
    kv_raw: csa_paged | None     # raw rows (the last rank: the window's source), else None
    n_tokens: int                # raw tokens of the request (the window is the last min(swa, N))
    H: int
    Hi: int
    k: int
    swa: int
    scale: float
    kdtype: int = CSA_BF16
    bufs: dict = field(default_factory=dict)

    def buffers(self, device):
        """Per-rank device buffers, made once and reused by every step."""
        if not self.bufs:
            G = self.hi - self.lo
            b = self.bufs
            b["scores"] = torch.empty(max(G, 1), dtype=torch.float32, device=device)
            b["idx"] = torch.empty(self.k, dtype=torch.int32, device=device)
            b["keys"] = torch.empty(self.k, dtype=torch.int32, device=device)
            b["topk_ws"] = torch.empty(max(csa_topk_workspace_size(1, max(G, 1), self.k), 16), dtype=torch.uint8,
                                       device=device)
            b["merge_ws"] = torch.empty(max(csa_topk_merge_workspace_size(self.world, self.k), 16),
                                        dtype=torch.uint8, device=device)
            b["sel_local"] = torch.empty(self.k, dtype=torch.int32, device=device)
            b["sel_global"] = torch.empty(self.k, dtype=torch.int32, device=device)
            swa = self.swa if self.kv_raw is not None else 0
            b["attn_ws"] = torch.empty(max(csa_sparse_attn_workspace_size(self.H, self.k, swa), 16),
                                       dtype=torch.uint8, device=device)
            b["o"] = torch.empty((self.H, 512), dtype=torch.float32, device=device)
            b["lse"] = torch.empty(self.H, dtype=torch.float32, device=device)
        return self.bufs


class LibcsaBackend:
    """The steps of one rank, each a libcsa call on the rank's device."""

    def local_topk(self, sh: CPShard, q_idx, w_h, stream=None):
        b = sh.buffers(q_idx.device)
        G = sh.hi - sh.lo
        if G > 0:
            csa_index_score(q_idx, w_h, sh.Hi, sh.kidx, sh.kdtype, G, b["scores"], stream)
        # G == 0: every entry is padding (index -1, key 0)
        csa_topk(b["scores"], G, sh.k, b["idx"], b["keys"], b["topk_ws"], b["topk_ws"].numel(), stream)
        return b["keys"], b["idx"]

    def global_select(self, sh: CPShard, keys_all, idx_all, stream=None):
        b = sh.buffers(keys_all.device)
        csa_topk_merge(keys_all, idx_all, sh.rank_lo, sh.world, sh.k, sh.rank, b["sel_local"], b["sel_global"], None,
                       b["merge_ws"], b["merge_ws"].numel(), stream)
        return b["sel_local"], b["sel_global"]

    def attn_partial(self, sh: CPShard, q, stream=None):
        b = sh.buffers(q.device)
        raw = sh.kv_raw if sh.kv_raw is not None else sh.kv_c
        swa = sh.swa if sh.kv_raw is not None else 0
        csa_sparse_attn_partial(q, sh.H, sh.scale, sh.kv_c, b["sel_local"], sh.k, raw, sh.n_tokens, swa, b["o"],
                                b["lse"], b["attn_ws"], b["attn_ws"].numel(), stream)
        return b["o"], b["lse"]

    def merge(self, o_all, lse_all, R: int, H: int, out, lse, stream=None):
        csa_attn_merge(o_all, lse_all, R, H, out, lse, stream)


class TorchDistExchange:
    """All-gather over a torch.distributed process group (rank order)."""

    def __init__(self, dist, group=None):
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        parts = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(parts, t.contiguous(), group=self.group)
        return torch.cat(parts, dim=0)


def cp_decode_step(sh: CPShard, q, q_idx, w_h, backend, exchange, out, lse, stream=None):
    """One rank's part of the step; every rank ends with the same out [H, 512] bf16 and lse [H].
    Returns the global selection (device int32 [k], by (score desc, index asc))."""
    keys, idx = backend.local_topk(sh, q_idx, w_h, stream)
    keys_all = exchange.all_gather(keys)
    idx_all = exchange.all_gather(idx)
    _, sel_global = backend.global_select(sh, keys_all, idx_all, stream)
    o, l = backend.attn_partial(sh, q, stream)
    backend.merge(exchange.all_gather(o), exchange.all_gather(l), sh.world, sh.H, out, lse, stream)
    return sel_global


def run_local(shards, q, q_idx, w_h, backend, out, lse, stream=None):
    """The R shards of one request on one device, stage by stage; the exchanges are
    concatenations in rank order, as an all-gather would deliver them."""
    lists = [backend.local_topk(sh, q_idx, w_h, stream) for sh in shards]
    keys_all = torch.cat([k for k, _ in lists])
    idx_all = torch.cat([i for _, i in lists])
    sels = [backend.global_select(sh, keys_all, idx_all, stream)[1] for sh in shards]
    parts = [backend.attn_partial(sh, q, stream) for sh in shards]
    o_all = torch.cat([o for o, _ in parts])
    lse_all = torch.cat([l for _, l in parts])
    backend.merge(o_all, lse_all, len(shards), shards[0].H, out, lse, stream)
    return sels[0]


def contiguous_ranges(G: int, world: int, multiple: int = 16) -> list[int]:
    """Range starts of `world` contiguous shards of G candidates, each a multiple of
    `multiple` long except the last (whole pages per shard)."""
    per = -(-G // world)
    per = -(-per // multiple) * multiple
    return [min(G, r * per) for r in range(world)] + [G]
