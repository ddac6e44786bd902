"""Seeded synthetic inputs for the C4 sparse-attention decode step.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds no arithmetic of the method (no gate, score,
selection or attention): only random draws (Philox4x32-10 + Box-Muller, in
``synth.c``), their encoding into bf16 / fp8-e4m3 / fp32 storage, page-table
permutations and the scatter of logical rows into paged pools.

Every tensor of a workload has its own stream id, so each tensor (and each row
range of it) is reproducible on its own from (seed, stream).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None

D_LATENT = 512
D_INDEX = 128

# stream ids: (tensor kind << 32) | request index
S_RAW, S_CPOOL, S_KIDX, S_QIDX, S_WH, S_Q, S_WGATE, S_BPOS, S_PAGES, S_LENS, S_CODEBOOK, S_CODEIDX, S_SCORES = range(1, 14)


def build(force: bool = False) -> str:
    """Compile libsynth.so beside its source (gcc; portable C, no ISA flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, u64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        for name in ("synth_normal_bf16", "synth_normal_f32", "synth_normal_e4m3", "synth_uniform_f32"):
            getattr(lib, name).argtypes = [vp, i64, i64, u64, u64, dbl, dbl, i32]
        lib.synth_u32.argtypes = [vp, i64, i64, u64, u64]
        lib.synth_permutation.argtypes = [vp, i64, u64, u64]
        lib.synth_uniform_int.argtypes = [vp, i64, i64, i64, u64, u64]
        lib.synth_scatter_pages.argtypes = [vp, i64, i64, ctypes.c_int32, vp, i64, vp]
        lib.synth_gather_pages.argtypes = [vp, i64, i64, ctypes.c_int32, vp, i64, vp]
        lib.synth_philox4x32_10_raw.argtypes = [vp, vp, vp]
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def stream_id(kind: int, request: int = 0) -> int:
    return (kind << 32) | request


def philox_block(counter, key) -> list[int]:
    c = np.asarray(counter, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    _L().synth_philox4x32_10_raw(_ptr(c), _ptr(k), _ptr(o))
    return [int(x) for x in o]


def normal_bf16(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0, begin: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, std^2) draws, round-to-nearest-even."""
    out = np.empty(shape, dtype=np.uint16)
    _L().synth_normal_bf16(_ptr(out), begin, out.size, seed, stream, mean, std, _threads())
    return out


def normal_f32(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0, begin: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().synth_normal_f32(_ptr(out), begin, out.size, seed, stream, mean, std, _threads())
    return out


def normal_e4m3(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0, begin: int = 0) -> np.ndarray:
    """fp8-e4m3 (OCP E4M3FN) bit patterns of N(mean, std^2) draws, RNE, saturating to +-448."""
    out = np.empty(shape, dtype=np.uint8)
    _L().synth_normal_e4m3(_ptr(out), begin, out.size, seed, stream, mean, std, _threads())
    return out


def uniform_f32(shape, seed: int, stream: int, lo: float = 0.0, hi: float = 1.0, begin: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().synth_uniform_f32(_ptr(out), begin, out.size, seed, stream, lo, hi, _threads())
    return out


def u32(n: int, seed: int, stream: int, begin: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    _L().synth_u32(_ptr(out), begin, n, seed, stream)
    return out


def permutation(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _L().synth_permutation(_ptr(out), n, seed, stream)
    return out


def uniform_int(n: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    _L().synth_uniform_int(_ptr(out), n, lo, hi, seed, stream)
    return out


def scatter_pages(logical: np.ndarray, rows_per_page: int, page_table: np.ndarray, pool: np.ndarray,
                  page_stride_bytes: int) -> None:
    """pool[page_table[r // rpp]] slot r % rpp <- logical row r (pure data movement)."""
    logical = np.ascontiguousarray(logical)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    row_bytes = logical.nbytes // max(1, logical.shape[0])
    _L().synth_scatter_pages(_ptr(logical), logical.shape[0], row_bytes, rows_per_page, _ptr(pt),
                             page_stride_bytes, _ptr(pool))


def gather_pages(pool: np.ndarray, n_rows: int, row_shape, dtype, rows_per_page: int, page_table: np.ndarray,
                 page_stride_bytes: int) -> np.ndarray:
    out = np.empty((n_rows,) + tuple(row_shape), dtype=dtype)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    row_bytes = out.nbytes // max(1, n_rows)
    _L().synth_gather_pages(_ptr(pool), n_rows, row_bytes, rows_per_page, _ptr(pt), page_stride_bytes, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Workload recipes
# --------------------------------------------------------------------------

@dataclass
class Request:
    n_tokens: int
    n_groups_done: int
    raw: np.ndarray        # bf16 bits [N, 512]
    cpool: np.ndarray      # bf16 bits [G, 512]; rows >= n_groups_done are zero (the step computes them)
    kidx: np.ndarray       # bf16 bits [G, 128] (uint16) or e4m3 bits [G, 128] (uint8); None for dense C128
    q: np.ndarray          # bf16 bits [H, 512]
    q_idx: np.ndarray      # bf16 bits [Hi, 128]
    w_h: np.ndarray        # fp32 [Hi]
    pages: np.ndarray      # int32 physical page ids of this request's logical pages


@dataclass
class DecodeCase:
    name: str
    seed: int
    ratio: int
    H: int
    Hi: int
    k: int
    swa: int
    kdtype: str            # "bf16" | "fp8"
    rows_per_page: int     # raw tokens per page (compressed pools use rows_per_page // ratio: shadow pages)
    scale: float
    w_gate: np.ndarray     # fp32 [512]
    b_pos: np.ndarray      # fp32 [ratio]
    requests: list = field(default_factory=list)
    n_pages: int = 0       # physical pages in each pool

    @property
    def B(self) -> int:
        return len(self.requests)

    def page_table(self) -> np.ndarray:
        """int32 [B, max_pages]; unused entries -1."""
        mp = max(len(r.pages) for r in self.requests)
        pt = np.full((self.B, mp), -1, dtype=np.int32)
        for b, r in enumerate(self.requests):
            pt[b, : len(r.pages)] = r.pages
        return pt

    # physical pools (host), built from the logical tensors through the page table
    def raw_pool(self) -> np.ndarray:
        pool = np.zeros((self.n_pages * self.rows_per_page, D_LATENT), dtype=np.uint16)
        for r in self.requests:
            scatter_pages(r.raw, self.rows_per_page, r.pages, pool, self.rows_per_page * D_LATENT * 2)
        return pool

    def c_rows_per_page(self) -> int:
        return max(1, self.rows_per_page // self.ratio)

    def c_pool(self) -> np.ndarray:
        rpp = self.c_rows_per_page()
        pool = np.zeros((self.n_pages * rpp, D_LATENT), dtype=np.uint16)
        for r in self.requests:
            scatter_pages(r.cpool, rpp, self.c_pages(r), pool, rpp * D_LATENT * 2)
        return pool

    def c_pages(self, r: Request) -> np.ndarray:
        """Pages of the compressed pools.  With rows_per_page % ratio == 0 they are the shadow of the raw
        pages (same physical ids); otherwise (C128 with small raw pages) the request's compressed rows use
        the first ceil(G / c_rpp) of its page ids."""
        G = r.n_tokens // self.ratio
        rpp = self.c_rows_per_page()
        return r.pages[: (G + rpp - 1) // rpp]

    def kidx_pool(self) -> np.ndarray:
        rpp = self.c_rows_per_page()
        dt = np.uint16 if self.kdtype == "bf16" else np.uint8
        pool = np.zeros((self.n_pages * rpp, D_INDEX), dtype=dt)
        rb = D_INDEX * (2 if self.kdtype == "bf16" else 1)
        for r in self.requests:
            scatter_pages(r.kidx, rpp, self.c_pages(r), pool, rpp * rb)
        return pool


def make_decode_case(name: str, seed: int, lengths, H: int, Hi: int, *, ratio: int = 4, k: int = 512,
                     swa: int = 128, kdtype: str = "bf16", rows_per_page: int = 64, paged: bool = True,
                     n_pending: int = 1, tie_codebook: bool = False, spare_pages: int = 0) -> DecodeCase:
    """Draw one decode workload.

    Recipe (per request b; all streams keyed by (seed, kind, b)):
      raw latent KV   [N_b, 512]  bf16 ~ N(0, 1)
      compressed pool [G_b, 512]  bf16 ~ N(0, 1) for groups < G_b - n_pending (already-compressed entries
                                  are an input of the decode step); pending rows are left 0
      index keys      [G_b, 128]  bf16 ~ N(0, 1), or fp8-e4m3 ~ N(0, 1); with tie_codebook each row is a
                                  copy of one of ceil(G_b / 16) codebook rows (many exact score ties)
      q [H, 512] bf16 ~ N(0,1); q_idx [Hi, 128] bf16 ~ N(0,1); w_h [Hi] fp32 ~ U(0,1)
    Layer weights: w_gate [512] fp32 ~ N(0, 1/512); b_pos [ratio] fp32 ~ N(0, 0.1) (second argument of N is
    the variance).  scale = 1/sqrt(512).  Pages: `rows_per_page` raw tokens per page; the physical page ids
    of all requests are one seeded permutation of the pool's pages (identity order when paged=False).
    """
    lengths = [int(n) for n in lengths]
    for n in lengths:
        assert n % ratio == 0 and n > 0
    w_gate = normal_f32((D_LATENT,), seed, stream_id(S_WGATE), 0.0, 1.0 / np.sqrt(512.0))
    b_pos = normal_f32((ratio,), seed, stream_id(S_BPOS), 0.0, float(np.sqrt(0.1)))
    case = DecodeCase(name=name, seed=seed, ratio=ratio, H=H, Hi=Hi, k=k, swa=swa, kdtype=kdtype,
                      rows_per_page=rows_per_page, scale=float(np.float32(1.0 / np.sqrt(512.0))),
                      w_gate=w_gate, b_pos=b_pos)
    pages_per_req = [(n + rows_per_page - 1) // rows_per_page for n in lengths]
    total_pages = sum(pages_per_req) + spare_pages
    perm = permutation(total_pages, seed, stream_id(S_PAGES)) if paged else np.arange(total_pages, dtype=np.int32)
    case.n_pages = total_pages
    off = 0
    for b, n in enumerate(lengths):
        G = n // ratio
        done = max(0, G - n_pending)
        raw = normal_bf16((n, D_LATENT), seed, stream_id(S_RAW, b))
        cpool = np.zeros((G, D_LATENT), dtype=np.uint16)
        if done:
            cpool[:done] = normal_bf16((done, D_LATENT), seed, stream_id(S_CPOOL, b))
        kidx = None
        if ratio == 4 or Hi > 0:
            if tie_codebook:
                C = (G + 15) // 16
                book = (normal_e4m3 if kdtype == "fp8" else normal_bf16)((C, D_INDEX), seed, stream_id(S_CODEBOOK, b))
                which = uniform_int(G, 0, C - 1, seed, stream_id(S_CODEIDX, b))
                kidx = np.ascontiguousarray(book[which])
            else:
                kidx = (normal_e4m3 if kdtype == "fp8" else normal_bf16)((G, D_INDEX), seed, stream_id(S_KIDX, b))
        req = Request(n_tokens=n, n_groups_done=done, raw=raw, cpool=cpool, kidx=kidx,
                      q=normal_bf16((H, D_LATENT), seed, stream_id(S_Q, b)),
                      q_idx=normal_bf16((max(Hi, 1), D_INDEX), seed, stream_id(S_QIDX, b))[:Hi],
                      w_h=uniform_f32((max(Hi, 1),), seed, stream_id(S_WH, b))[:Hi],
                      pages=np.ascontiguousarray(perm[off: off + pages_per_req[b]]))
        off += pages_per_req[b]
        case.requests.append(req)
    return case


def ragged_lengths(B: int, lo: int, hi: int, multiple: int, seed: int) -> list[int]:
    """B context lengths ~ U[lo, hi] restricted to multiples of `multiple`."""
    u = uniform_int(B, lo // multiple, hi // multiple, seed, stream_id(S_LENS))
    return [int(x) * multiple for x in u]


# The five workloads: tiny, 128K, 1M paged, ragged fp8 batch, C128 dense.
def config(i: int, *, scale_down: int = 1) -> DecodeCase:
    """Workload i (seed i).  `scale_down` > 1 shrinks context lengths (parity at oracle-friendly sizes)."""
    if i == 0:
        return make_decode_case("tiny-4K", 0, [4096], H=16, Hi=4, paged=False)
    if i == 1:
        return make_decode_case("c4-128K", 1, [131072 // scale_down], H=64, Hi=8, paged=False)
    if i == 2:
        return make_decode_case("c4-1M-paged", 2, [1048576 // scale_down], H=128, Hi=8, paged=True)
    if i == 3:
        lens = ragged_lengths(32, 4096 // scale_down, 131072 // scale_down, 4, 3)
        return make_decode_case("ragged32-fp8", 3, lens, H=64, Hi=8, kdtype="fp8", paged=True, tie_codebook=True)
    if i == 4:
        return make_decode_case("c128-dense-bs8", 4, [524288 // scale_down] * 8, H=64, Hi=0, ratio=128,
                                paged=True)
    raise ValueError(i)
