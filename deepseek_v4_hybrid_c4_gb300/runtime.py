"""Device-resident decode batch: holds the pools, page tables, per-request
queries and the workspace on the GPU and fills one csa_decode_params.

PyTorch is used here only to own device memory; every stage runs in libcsa.
"""
from __future__ import annotations

import torch

from . import (CSA_BF16, CSA_FP8_E4M3, csa_decode, csa_decode_params, csa_decode_timed,
               csa_decode_workspace_size)


def _dev(x, dtype, device):
    t = x if isinstance(x, torch.Tensor) else torch.as_tensor(x)
    return t.to(device=device, dtype=dtype).contiguous()


def _bits(x, dev):
    """Move bf16/fp8 data (typed tensor or numpy bit patterns) to the device without conversion."""
    if isinstance(x, torch.Tensor):
        t = x
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        return t.to(dev).contiguous()
    import numpy as np
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def _np_bits(x):
    """numpy bit patterns as a C-contiguous int16 array (bf16 rows)."""
    import numpy as np
    a = np.ascontiguousarray(x)
    return a.view(np.int16) if a.dtype == np.uint16 else a


def _pack(dev, parts):
    """One device buffer holding every tensor of `parts`, each at a 256-byte boundary, and a
    view of the buffer for each (the data copied in), so that the group moves in one copy."""
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.zeros(max(total, 256), dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(parts, offs):
        v = buf[o: o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class DecodeBatch:
    """One fused decode step over B requests.

    Pools (bf16 / fp8 data given as raw bit patterns or typed tensors):
      raw_pool   [n_pages * rows_per_page, 512] bf16      raw latent KV, 64-token pages
      c_pool     [n_pages * c_rpp, 512] bf16              compressed entries (shadow pages unless
                                                          c_page_table is given)
      kidx_pool  [n_pages * c_rpp, 128] bf16 / fp8        index keys (C4 only)
    page_table [B, P] int32, n_tokens / n_groups_done [B] int64, q [B, H, 512] bf16,
    q_idx [B, Hi, 128] bf16, w_h [B, Hi] fp32, w_gate [512] fp32, b_pos [ratio] fp32.
    Speculative verify: n_q query positions per request; q, q_idx, w_h and the outputs then have
    B * n_q leading entries in (request, query) order.
    HiSparse (hs_slots > 0, C4 with an explicit c_page_table): the compressed pool becomes a
    mirror in pinned host memory, with a GPU working set of hs_slots pages; `hs_update()` after a
    step brings the pages it missed in, and `hs_step` stamps the next step.
    Optional compression-state rings: ring_pool [n_rings * ring_size, 512] bf16 and ring_page [B]
    int32 (request b's token t in row ring_page[b] * ring_size + t % ring_size); the pending
    groups are then compressed from the ring.
    The per-step inputs q, q_idx and w_h are views of one device buffer (`step_in`), and the
    outputs out and lse of another (`step_out`), so each group moves in a single copy.
    """

    def __init__(self, *, ratio, H, Hi, k, swa, scale, kdtype, rows_per_page, raw_pool, c_pool, kidx_pool,
                 page_table, n_tokens, n_groups_done, q, q_idx, w_h, w_gate, b_pos, n_pages, max_tokens=None,
                 c_page_table=None, c_rows_per_page=0, c_n_pages=0, ring_pool=None, ring_page=None, ring_size=0,
                 n_q=1, hs_slots=0, device="cuda"):
        dev = torch.device(device)
        i32, i64, f32 = torch.int32, torch.int64, torch.float32
        self.ratio, self.H, self.Hi, self.k, self.swa = ratio, H, Hi, k, swa
        self.raw_pool = _bits(raw_pool, dev)
        self.hs_slots = int(hs_slots)
        if self.hs_slots:  # the full compressed pool as a pinned host mirror the kernels read directly
            src = c_pool.cpu() if isinstance(c_pool, torch.Tensor) else torch.from_numpy(_np_bits(c_pool))
            self.c_pool = torch.empty(src.shape, dtype=torch.int16, pin_memory=True)
            self.c_pool.copy_(src.view(torch.int16))
        else:
            self.c_pool = _bits(c_pool, dev)
        self.kidx_pool = None if kidx_pool is None else _bits(kidx_pool, dev)
        self.page_table = _dev(page_table, i32, dev)
        self.c_page_table = None if c_page_table is None else _dev(c_page_table, i32, dev)
        self.n_tokens = _dev(n_tokens, i64, dev)
        self.n_groups_done = _dev(n_groups_done, i64, dev)
        self.B = int(self.n_tokens.shape[0])
        self.n_q = max(1, int(n_q))
        Bq = self.B * self.n_q  # (request, query position) entries of q, q_idx, w_h and the outputs
        for name, x in (("q", q), ("q_idx", q_idx), ("w_h", w_h)):
            if x is not None and int(x.shape[0]) != Bq:
                raise ValueError(f"{name} has {int(x.shape[0])} entries; B * n_q = {Bq}")
        self.step_in, (self.q, self.q_idx, self.w_h) = _pack(dev, [
            _bits(q, dev),
            _bits(q_idx, dev) if Hi else torch.zeros(8, dtype=torch.int16, device=dev),
            _dev(w_h, f32, dev) if Hi else torch.zeros(4, dtype=f32, device=dev)])
        self.w_gate = _dev(w_gate, f32, dev)
        self.b_pos = _dev(b_pos, f32, dev)
        self.step_out, (self.out, self.lse) = _pack(dev, [
            torch.zeros((Bq, H, 512), dtype=torch.bfloat16, device=dev),
            torch.zeros((Bq, H), dtype=f32, device=dev)])
        self.sel = torch.zeros((Bq, max(k, 1)), dtype=i32, device=dev) if ratio == 4 else None
        if max_tokens is None:
            max_tokens = int(torch.as_tensor(n_tokens).max())
        c_rpp = c_rows_per_page if c_page_table is not None else rows_per_page // ratio
        p = csa_decode_params()
        p.B, p.ratio, p.H, p.Hi, p.k, p.swa = self.B, ratio, H, Hi, k, swa
        p.scale = float(scale)
        p.k_dtype = CSA_BF16 if kdtype == "bf16" else CSA_FP8_E4M3
        p.max_tokens = int(max_tokens)
        p.n_tokens = self.n_tokens.data_ptr()
        p.n_groups_done = self.n_groups_done.data_ptr()
        p.kv_raw = self.raw_pool.data_ptr()
        p.raw_rows_per_page = rows_per_page
        p.raw_page_stride = rows_per_page * 1024
        p.kv_c = self.c_pool.data_ptr()
        p.c_page_stride = c_rpp * 1024
        if self.kidx_pool is not None:
            p.k_idx = self.kidx_pool.data_ptr()
            p.kidx_page_stride = c_rpp * (256 if kdtype == "bf16" else 128)
        p.n_pages = int(n_pages)
        p.page_table = self.page_table.data_ptr()
        p.page_table_stride = int(self.page_table.shape[1])
        if self.c_page_table is not None:
            p.c_page_table = self.c_page_table.data_ptr()
            p.c_page_table_stride = int(self.c_page_table.shape[1])
            p.c_rows_per_page = c_rows_per_page
            p.c_n_pages = int(c_n_pages)
        p.w_gate = self.w_gate.data_ptr()
        p.b_pos = self.b_pos.data_ptr()
        p.q = self.q.data_ptr()
        p.q_idx = self.q_idx.data_ptr()
        p.w_h = self.w_h.data_ptr()
        p.out = self.out.data_ptr()
        p.lse = self.lse.data_ptr()
        p.sel = self.sel.data_ptr() if self.sel is not None else None
        p.n_q = self.n_q
        self.ring_pool = None if ring_pool is None else _bits(ring_pool, dev)
        self.ring_page = None if ring_page is None else _dev(ring_page, i32, dev)
        if self.ring_pool is not None:
            p.ring_pool = self.ring_pool.data_ptr()
            p.ring_page = self.ring_page.data_ptr()
            p.ring_size = int(ring_size)
            p.ring_n_pages = int(self.ring_pool.shape[0]) // int(ring_size)
        self.hs = None
        if self.hs_slots:
            stride = int(self.c_page_table.shape[1])
            self.hs_pool = torch.zeros((self.hs_slots * c_rpp, 512), dtype=torch.int16, device=dev)
            self.hs_table = torch.full((self.B, stride), -1, dtype=i32, device=dev)
            self.hs_touch = torch.zeros((self.B, stride), dtype=i32, device=dev)
            p.hs_ws_pool = self.hs_pool.data_ptr()
            p.hs_ws_table = self.hs_table.data_ptr()
            p.hs_n_slots = self.hs_slots
            p.hs_touch = self.hs_touch.data_ptr()
            p.hs_step = 1
            from . import csa_hisparse_create
            self.hs = csa_hisparse_create(self.B, stride, self.hs_slots)
        self.params = p
        self.ws_bytes = csa_decode_workspace_size(p)  # 0 also when the parameters are rejected: run() reports why
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self._shape = dict(ratio=ratio, H=H, Hi=Hi, k=k, swa=swa, scale=scale, kdtype=kdtype,
                           rows_per_page=rows_per_page, n_pages=n_pages, max_tokens=max_tokens,
                           c_rows_per_page=c_rows_per_page, c_n_pages=c_n_pages, ring_size=ring_size, n_q=n_q,
                           hs_slots=hs_slots, device=device)

    def clone(self) -> "DecodeBatch":
        """The same step over copies of every device buffer (same values, other addresses):
        e.g. the next layer of a model whose layers hold identical synthetic caches."""
        c = lambda t: None if t is None else t.clone()
        return DecodeBatch(raw_pool=c(self.raw_pool), c_pool=c(self.c_pool), kidx_pool=c(self.kidx_pool),
                           page_table=c(self.page_table), n_tokens=c(self.n_tokens),
                           n_groups_done=c(self.n_groups_done), q=c(self.q), q_idx=c(self.q_idx) if self.Hi else None,
                           w_h=c(self.w_h) if self.Hi else None, w_gate=c(self.w_gate), b_pos=c(self.b_pos),
                           c_page_table=c(self.c_page_table), ring_pool=c(self.ring_pool),
                           ring_page=c(self.ring_page), **self._shape)

    @property
    def hs_step(self) -> int:
        return int(self.params.hs_step)

    @hs_step.setter
    def hs_step(self, v: int) -> None:
        self.params.hs_step = int(v)

    def hs_update(self, stream=None):
        """After a step: bring the pages it read from the mirror into the working set ->
        (pages brought in, pages evicted)."""
        from . import csa_hisparse_update
        return csa_hisparse_update(self.hs, self.params, stream)

    def hs_collect(self, stream=None):
        """After a step: enqueue the readback of its stamps (no wait)."""
        from . import csa_hisparse_collect
        csa_hisparse_collect(self.hs, self.params, stream)

    def hs_apply(self, n_tokens_host, stream=None, side_stream=None):
        """Bring in the pages the collected step missed, beside the next steps -> (n_in, n_evicted)."""
        from . import csa_hisparse_apply
        return csa_hisparse_apply(self.hs, self.params, n_tokens_host, stream, side_stream)

    def __del__(self):
        if getattr(self, "hs", None):
            from . import csa_hisparse_destroy
            csa_hisparse_destroy(self.hs)
            self.hs = None

    def run(self, stream=None, events=None) -> None:
        if events is None:
            csa_decode(self.params, self.ws, self.ws_bytes, stream)
        else:
            csa_decode_timed(self.params, self.ws, self.ws_bytes, stream, events)
