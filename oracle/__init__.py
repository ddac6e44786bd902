"""CPU oracle of the C4 hybrid-sparse-attention decode step (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never calls it and has no CPU fallback.

Thin numpy/ctypes marshalling over ``oracle.c`` (plain single-threaded C,
fp64 compression and attention, fp32 fixed-order index score, total-order sort
for the top-k).  The C file documents each stage, the passage of the pages it
follows and the independent checks that pin it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
D_LATENT = 512
D_INDEX = 128


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc: no contraction of a*b+c, no fast-math."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f32.restype = f32
        lib.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_f32.restype = f32
        lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.orc_f64_to_bf16.restype = ctypes.c_uint16
        lib.orc_score_key.argtypes = [f32]
        lib.orc_score_key.restype = ctypes.c_uint32
        lib.orc_compress.argtypes = [vp, i64, i32, vp, vp, i64, i64, vp, vp, vp]
        lib.orc_compress.restype = i32
        lib.orc_index_score.argtypes = [vp, vp, i32, vp, i32, i64, vp]
        lib.orc_index_score.restype = None
        lib.orc_topk.argtypes = [vp, i64, i32, vp, vp]
        lib.orc_topk.restype = i32
        lib.orc_topk_select.argtypes = [vp, i64, i32, vp, vp]
        lib.orc_topk_select.restype = i32
        lib.orc_attention.argtypes = [vp, i32, f32, vp, i64, vp, vp, vp]
        lib.orc_attention.restype = None
        lib.orc_sparse_attn.argtypes = [vp, i32, f32, vp, i64, vp, i32, vp, i64, i32, vp, vp, vp]
        lib.orc_sparse_attn.restype = i32
        lib.orc_decode_request.argtypes = [vp, i64, vp, i64, i32, i32, vp, vp, vp, vp, i32, vp, i32, i32, vp, i32,
                                           f32, i32, vp, vp, vp, vp, vp]
        lib.orc_decode_request.restype = i32
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous numpy"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ decoders
def bf16_to_f32(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def e4m3_to_f32(bits) -> np.ndarray:
    lib = _L()
    table = np.array([lib.orc_e4m3_to_f32(i) for i in range(256)], dtype=np.float32)
    return table[_c(bits, np.uint8)]


def f64_to_bf16(x) -> np.ndarray:
    lib = _L()
    x = np.asarray(x, dtype=np.float64)
    return np.array([lib.orc_f64_to_bf16(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def score_key(s: float) -> int:
    return int(_L().orc_score_key(float(s)))


# ------------------------------------------------------------------ stages
def compress(x_bf16, ratio: int, w_gate, b_pos, first_group: int = 0, n_groups: int | None = None,
             want_f64: bool = False, want_gates: bool = False):
    """Stage 1 over groups [first_group, first_group+n_groups) of x [n_tokens, 512] (bf16 bits)."""
    x = _c(x_bf16, np.uint16)
    n_tokens = x.shape[0]
    if n_groups is None:
        n_groups = n_tokens // ratio - first_group
    out = np.zeros((n_groups, D_LATENT), dtype=np.uint16)
    f64 = np.zeros((n_groups, D_LATENT), dtype=np.float64) if want_f64 else None
    gates = np.zeros((n_groups, ratio), dtype=np.float64) if want_gates else None
    rc = _L().orc_compress(_p(x), n_tokens, ratio, _p(_c(w_gate, np.float32)), _p(_c(b_pos, np.float32)),
                           first_group, n_groups, _p(out), _p(f64), _p(gates))
    if rc:
        raise ValueError(f"orc_compress rc={rc}")
    res = [out]
    if want_f64:
        res.append(f64)
    if want_gates:
        res.append(gates)
    return res[0] if len(res) == 1 else tuple(res)


def index_score(q_idx_bf16, w_h, k_idx, k_fp8: bool) -> np.ndarray:
    q = _c(q_idx_bf16, np.uint16)
    Hi = q.shape[0]
    k = _c(k_idx, np.uint8 if k_fp8 else np.uint16)
    G = k.shape[0]
    out = np.zeros(G, dtype=np.float32)
    _L().orc_index_score(_p(q), _p(_c(w_h, np.float32)), Hi, _p(k), int(bool(k_fp8)), G, _p(out))
    return out


def topk(scores, k: int, want_keys: bool = False):
    s = _c(scores, np.float32)
    idx = np.zeros(k, dtype=np.int32)
    keys = np.zeros(k, dtype=np.uint32) if want_keys else None
    rc = _L().orc_topk(_p(s), s.shape[0], k, _p(idx), _p(keys))
    if rc:
        raise ValueError(f"orc_topk rc={rc}")
    return (idx, keys) if want_keys else idx


def topk_select(scores, k: int, want_keys: bool = False):
    """topk by selection (partition to rank k, then sort only the k): the same result."""
    s = _c(scores, np.float32)
    idx = np.zeros(k, dtype=np.int32)
    keys = np.zeros(k, dtype=np.uint32) if want_keys else None
    rc = _L().orc_topk_select(_p(s), s.shape[0], k, _p(idx), _p(keys))
    if rc:
        raise ValueError(f"orc_topk_select rc={rc}")
    return (idx, keys) if want_keys else idx


def attention(q_bf16, scale: float, rows_bf16):
    """Stage 4 over explicit rows [n, 512]. Returns (out bf16 bits [H,512], out f64, lse f64 [H])."""
    q = _c(q_bf16, np.uint16)
    rows = _c(rows_bf16, np.uint16).reshape(-1, D_LATENT)
    H = q.shape[0]
    out = np.zeros((H, D_LATENT), dtype=np.uint16)
    f64 = np.zeros((H, D_LATENT), dtype=np.float64)
    lse = np.zeros(H, dtype=np.float64)
    _L().orc_attention(_p(q), H, scale, _p(rows), rows.shape[0], _p(out), _p(f64), _p(lse))
    return out, f64, lse


def sparse_attn(q_bf16, scale: float, cpool_bf16, sel, raw_bf16, swa: int):
    q = _c(q_bf16, np.uint16)
    cpool = _c(cpool_bf16, np.uint16)
    raw = _c(raw_bf16, np.uint16)
    sel = _c(sel, np.int32)
    H = q.shape[0]
    out = np.zeros((H, D_LATENT), dtype=np.uint16)
    f64 = np.zeros((H, D_LATENT), dtype=np.float64)
    lse = np.zeros(H, dtype=np.float64)
    rc = _L().orc_sparse_attn(_p(q), H, scale, _p(cpool), cpool.shape[0], _p(sel), sel.shape[0], _p(raw),
                              raw.shape[0], swa, _p(out), _p(f64), _p(lse))
    if rc:
        raise ValueError(f"orc_sparse_attn rc={rc}")
    return out, f64, lse


def decode_request(req, *, ratio: int, w_gate, b_pos, k: int, swa: int, scale: float, kdtype: str = "bf16",
                   dense: bool | None = None):
    """The decode step of one request (attributes as in synth.Request).

    Returns dict(out bf16 [H,512], out_f64, lse [H], sel [k] (C4 only), scores [G] (C4 only),
    cpool [G,512] with the pending groups filled in)."""
    if dense is None:
        dense = ratio != 4
    raw = _c(req.raw, np.uint16)
    N = raw.shape[0]
    G = N // ratio
    cpool = np.array(req.cpool, dtype=np.uint16, copy=True, order="C")
    q = _c(req.q, np.uint16)
    H = q.shape[0]
    out = np.zeros((H, D_LATENT), dtype=np.uint16)
    f64 = np.zeros((H, D_LATENT), dtype=np.float64)
    lse = np.zeros(H, dtype=np.float64)
    sel = np.zeros(max(k, 1), dtype=np.int32)
    scores = np.zeros(max(G, 1), dtype=np.float32)
    fp8 = kdtype == "fp8"
    if dense:
        qi = np.zeros((1, D_INDEX), dtype=np.uint16)
        wh = np.zeros(1, dtype=np.float32)
        kk = np.zeros((1, D_INDEX), dtype=np.uint16)
        Hi = 0
    else:
        qi = _c(req.q_idx, np.uint16)
        wh = _c(req.w_h, np.float32)
        kk = _c(req.kidx, np.uint8 if fp8 else np.uint16)
        Hi = qi.shape[0]
    rc = _L().orc_decode_request(_p(raw), N, _p(cpool), int(req.n_groups_done), ratio, int(bool(dense)),
                                 _p(_c(w_gate, np.float32)), _p(_c(b_pos, np.float32)), _p(qi), _p(wh), Hi, _p(kk),
                                 int(fp8), k, _p(q), H, scale, swa, _p(out), _p(f64), _p(lse), _p(sel),
                                 _p(scores))
    if rc:
        raise ValueError(f"orc_decode_request rc={rc}")
    res = dict(out=out, out_f64=f64, lse=lse, cpool=cpool)
    if not dense:
        res["sel"] = sel[:k]
        res["scores"] = scores[:G]
    return res


def decode_queries(req, queries, *, ratio: int, w_gate, b_pos, k: int, swa: int, scale: float,
                   kdtype: str = "bf16"):
    """Speculative verify of one request: `queries` = [(q, q_idx, w_h)] for its last n_q token
    positions.  Query j sits at token N - n_q + j, so it is the decode step of the same request
    cut to its first N - n_q + j + 1 tokens (the groups completed within them, its own top k and
    SWA window).  Returns one decode_request result per query."""
    from types import SimpleNamespace
    N, nq = int(req.n_tokens), len(queries)
    res = []
    for j, (q, q_idx, w_h) in enumerate(queries):
        Nj = N - nq + j + 1
        sub = SimpleNamespace(raw=req.raw[:Nj], cpool=req.cpool, q=q, q_idx=q_idx, w_h=w_h, kidx=req.kidx,
                              n_groups_done=min(int(req.n_groups_done), Nj // ratio))
        res.append(decode_request(sub, ratio=ratio, w_gate=w_gate, b_pos=b_pos, k=k, swa=swa, scale=scale,
                                  kdtype=kdtype))
    return res


def decode_case(case):
    """The decode step for every request of a synth.DecodeCase (requests are independent)."""
    return [decode_request(r, ratio=case.ratio, w_gate=case.w_gate, b_pos=case.b_pos, k=case.k, swa=case.swa,
                           scale=case.scale, kdtype=case.kdtype) for r in case.requests]
