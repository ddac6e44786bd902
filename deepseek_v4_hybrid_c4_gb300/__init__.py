"""Python binding of libcsa (the C4 hybrid-sparse-attention decode step on GB300).

Argument marshalling only: every stage runs in libcsa's CUDA kernels.  The
functions keep the names of the C entry points (include/csa.h) and take torch
CUDA tensors (or raw device addresses) plus an optional torch stream.  There is
no CPU path: if libcsa.so is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")
_lib = None

CSA_OK, CSA_ERR_INVALID_ARG, CSA_ERR_UNSUPPORTED, CSA_ERR_CUDA, CSA_ERR_TIMEOUT, CSA_ERR_DEVICE_BOUNDS, \
    CSA_ERR_WORKSPACE = range(7)
CSA_BF16, CSA_FP8_E4M3, CSA_FP32 = range(3)


class CsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (csa_status {code})")


class csa_paged(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("rows_per_page", ctypes.c_int32),
                ("page_stride_bytes", ctypes.c_int64), ("n_pages", ctypes.c_int64)]


CSA_COPY_MAX = 16


class csa_copy(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("bytes", ctypes.c_uint64)]


class csa_decode_params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("ratio", ctypes.c_int32), ("H", ctypes.c_int32), ("Hi", ctypes.c_int32),
        ("k", ctypes.c_int32), ("swa", ctypes.c_int32), ("scale", ctypes.c_float), ("k_dtype", ctypes.c_int32),
        ("max_tokens", ctypes.c_int64), ("n_tokens", ctypes.c_void_p), ("n_groups_done", ctypes.c_void_p),
        ("kv_raw", ctypes.c_void_p), ("raw_rows_per_page", ctypes.c_int32), ("raw_page_stride", ctypes.c_int64),
        ("kv_c", ctypes.c_void_p), ("c_page_stride", ctypes.c_int64),
        ("k_idx", ctypes.c_void_p), ("kidx_page_stride", ctypes.c_int64), ("n_pages", ctypes.c_int64),
        ("page_table", ctypes.c_void_p), ("page_table_stride", ctypes.c_int64),
        ("c_page_table", ctypes.c_void_p), ("c_page_table_stride", ctypes.c_int64),
        ("c_rows_per_page", ctypes.c_int32), ("c_n_pages", ctypes.c_int64),
        ("w_gate", ctypes.c_void_p), ("b_pos", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("w_h", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("sel", ctypes.c_void_p),
        ("ring_pool", ctypes.c_void_p), ("ring_page", ctypes.c_void_p), ("ring_size", ctypes.c_int32),
        ("ring_n_pages", ctypes.c_int64), ("n_q", ctypes.c_int32),
        ("hs_ws_pool", ctypes.c_void_p), ("hs_ws_table", ctypes.c_void_p), ("hs_n_slots", ctypes.c_int64),
        ("hs_touch", ctypes.c_void_p), ("hs_step", ctypes.c_uint32),
    ]


def lib() -> ctypes.CDLL:
    """The loaded libcsa.so (built by __graft_entry__.build() / deepseek_v4_hybrid_c4_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcsa.so is not built ({LIB_PATH}); run `python -c 'import __graft_entry__ as g; "
                               f"g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        L.csa_compress.argtypes = [csa_paged, i64, i32, vp, vp, i64, i64, csa_paged, vp]
        L.csa_index_score.argtypes = [vp, vp, i32, csa_paged, i32, i64, vp, vp]
        L.csa_index_score_bounds.argtypes = [vp, vp, i32, csa_paged, i32, i64, vp, vp, vp]
        L.csa_topk.argtypes = [vp, i64, i32, vp, vp, vp, sz, vp]
        L.csa_topk_batched.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp, sz, vp]
        L.csa_topk_cluster.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp]
        L.csa_topk_workspace_size.argtypes = [i32, i64, i32]
        L.csa_topk_workspace_size.restype = sz
        L.csa_sparse_attn.argtypes = [vp, i32, f32, csa_paged, vp, i32, csa_paged, i64, i32, vp, vp, vp, sz, vp]
        L.csa_sparse_attn_workspace_size.argtypes = [i32, i32, i32]
        L.csa_sparse_attn_workspace_size.restype = sz
        L.csa_topk_merge_workspace_size.argtypes = [i32, i32]
        L.csa_topk_merge_workspace_size.restype = sz
        L.csa_topk_merge.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.csa_sparse_attn_partial.argtypes = [vp, i32, f32, csa_paged, vp, i32, csa_paged, i64, i32, vp, vp, vp, sz,
                                              vp]
        L.csa_attn_merge.argtypes = [vp, vp, i32, i32, vp, vp, vp]
        L.csa_decode.argtypes = [ctypes.POINTER(csa_decode_params), vp, sz, vp]
        L.csa_decode_timed.argtypes = [ctypes.POINTER(csa_decode_params), vp, sz, vp, ctypes.POINTER(vp)]
        L.csa_decode_noalloc.argtypes = [ctypes.POINTER(csa_decode_params), vp]
        L.csa_decode_workspace_size.argtypes = [ctypes.POINTER(csa_decode_params)]
        L.csa_decode_workspace_size.restype = sz
        L.csa_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.csa_status_string.argtypes = [i32]
        L.csa_status_string.restype = ctypes.c_char_p
        L.csa_version.restype = i32
        L.csa_selftest_bounded_wait.argtypes = [vp]
        L.csa_copy_batch.argtypes = [i32, ctypes.POINTER(csa_copy), vp]
        L.csa_hisparse_create.argtypes = [i32, i64, i64, ctypes.POINTER(vp)]
        L.csa_hisparse_destroy.argtypes = [vp]
        L.csa_hisparse_destroy.restype = None
        L.csa_hisparse_plan.argtypes = [vp, vp, ctypes.c_uint32, vp, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.csa_hisparse_table.argtypes = [vp]
        L.csa_hisparse_table.restype = ctypes.POINTER(ctypes.c_int32)
        L.csa_hisparse_collect.argtypes = [vp, ctypes.POINTER(csa_decode_params), vp]
        L.csa_hisparse_apply.argtypes = [vp, ctypes.POINTER(csa_decode_params), vp, vp, vp, ctypes.POINTER(i64),
                                         ctypes.POINTER(i64)]
        L.csa_hisparse_update.argtypes = [vp, ctypes.POINTER(csa_decode_params), vp, ctypes.POINTER(i64),
                                          ctypes.POINTER(i64)]
        for name in ("csa_compress", "csa_index_score", "csa_index_score_bounds", "csa_topk", "csa_topk_batched",
                     "csa_topk_cluster", "csa_topk_merge", "csa_sparse_attn_partial", "csa_attn_merge", "csa_sparse_attn",
                     "csa_decode", "csa_decode_timed", "csa_decode_noalloc", "csa_read_device_status",
                     "csa_hisparse_create", "csa_hisparse_plan", "csa_hisparse_update", "csa_hisparse_collect",
                     "csa_hisparse_apply", "csa_selftest_bounded_wait", "csa_copy_batch"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(code: int) -> str:
    try:
        return lib().csa_status_string(int(code)).decode()
    except Exception:  # library not loadable: still describe the code
        return str(code)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("libcsa takes device tensors")
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != CSA_OK:
        raise CsaError(rc, where)


def paged(base, rows_per_page: int, row_bytes: int, page_table=None, page_stride_bytes: int | None = None,
          n_pages: int | None = None) -> csa_paged:
    """Describe a (paged or contiguous) row buffer; see csa_paged in csa.h.  The returned
    struct keeps references to the tensors it points into, so they stay allocated."""
    stride = page_stride_bytes if page_stride_bytes is not None else rows_per_page * row_bytes
    if n_pages is None:
        n_pages = max(1, base.numel() * base.element_size() // stride) if not isinstance(base, int) else 1
    p = csa_paged(_ptr(base), _ptr(page_table), rows_per_page, stride, n_pages)
    p._keep = (base, page_table)
    return p


# ---------------------------------------------------------------- entry points
def csa_compress(kv_raw: csa_paged, n_tokens: int, ratio: int, w_gate, b_pos, first_group: int, n_groups: int,
                 kv_c_out: csa_paged, stream=None) -> None:
    _check(lib().csa_compress(kv_raw, n_tokens, ratio, _ptr(w_gate), _ptr(b_pos), first_group, n_groups, kv_c_out,
                              _stream(stream)), "csa_compress")


def csa_index_score(q_idx, w_h, Hi: int, k_idx: csa_paged, k_dtype: int, G: int, scores, stream=None) -> None:
    _check(lib().csa_index_score(_ptr(q_idx), _ptr(w_h), Hi, k_idx, k_dtype, G, _ptr(scores), _stream(stream)),
           "csa_index_score")


def csa_index_score_bounds(q_idx, w_h, Hi: int, k_idx: csa_paged, k_dtype: int, G: int, lower, upper,
                           stream=None) -> None:
    _check(lib().csa_index_score_bounds(_ptr(q_idx), _ptr(w_h), Hi, k_idx, k_dtype, G,
                                        _ptr(lower) if lower is not None else None, _ptr(upper), _stream(stream)),
           "csa_index_score_bounds")


def csa_topk_workspace_size(B: int, max_G: int, k: int) -> int:
    return int(lib().csa_topk_workspace_size(B, max_G, k))


def _scratch(nbytes: int, like):
    import torch
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=like.device if hasattr(like, "device") else "cuda")


def csa_topk(scores, G: int, k: int, idx_out, keys_out=None, workspace=None, ws_bytes: int = 0,
             stream=None) -> None:
    """workspace None: a scratch tensor of csa_topk_workspace_size(1, G, k) bytes is allocated."""
    if workspace is None:
        ws_bytes = csa_topk_workspace_size(1, G, k)
        workspace = _scratch(ws_bytes, scores)
    _check(lib().csa_topk(_ptr(scores), G, k, _ptr(idx_out), _ptr(keys_out), _ptr(workspace), ws_bytes,
                          _stream(stream)), "csa_topk")


def csa_topk_batched(scores, offsets, B: int, max_G: int, k: int, idx_out, keys_out=None, workspace=None,
                     ws_bytes: int = 0, stream=None) -> None:
    if workspace is None:
        ws_bytes = csa_topk_workspace_size(B, max_G, k)
        workspace = _scratch(ws_bytes, scores)
    _check(lib().csa_topk_batched(_ptr(scores), _ptr(offsets), B, max_G, k, _ptr(idx_out), _ptr(keys_out),
                                  _ptr(workspace), ws_bytes, _stream(stream)), "csa_topk_batched")


def csa_topk_cluster(scores, offsets, B: int, max_G: int, k: int, idx_out, keys_out=None, stream=None) -> None:
    _check(lib().csa_topk_cluster(_ptr(scores), _ptr(offsets), B, max_G, k, _ptr(idx_out), _ptr(keys_out),
                                  _stream(stream)), "csa_topk_cluster")


def csa_sparse_attn_workspace_size(H: int, n_sel: int, swa: int) -> int:
    return int(lib().csa_sparse_attn_workspace_size(H, n_sel, swa))


def csa_sparse_attn(q, H: int, scale: float, kv_c: csa_paged, sel, n_sel: int, kv_raw: csa_paged, n_tokens: int,
                    swa: int, out, lse=None, workspace=None, ws_bytes: int = 0, stream=None) -> None:
    _check(lib().csa_sparse_attn(_ptr(q), H, scale, kv_c, _ptr(sel), n_sel, kv_raw, n_tokens, swa, _ptr(out),
                                 _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)), "csa_sparse_attn")


def csa_topk_merge_workspace_size(R: int, k: int) -> int:
    return int(lib().csa_topk_merge_workspace_size(R, k))


def csa_topk_merge(keys, idx, rank_lo, R: int, k: int, rank: int = -1, sel_local=None, idx_out=None, keys_out=None,
                   workspace=None, ws_bytes: int = 0, stream=None) -> None:
    if workspace is None:
        ws_bytes = csa_topk_merge_workspace_size(R, k)
        workspace = _scratch(ws_bytes, keys)
    _check(lib().csa_topk_merge(_ptr(keys), _ptr(idx), _ptr(rank_lo), R, k, rank, _ptr(sel_local), _ptr(idx_out),
                                _ptr(keys_out), _ptr(workspace), ws_bytes, _stream(stream)), "csa_topk_merge")


def csa_sparse_attn_partial(q, H: int, scale: float, kv_c: csa_paged, sel, n_sel: int, kv_raw: csa_paged,
                            n_tokens: int, swa: int, o_part, lse_part, workspace=None, ws_bytes: int = 0,
                            stream=None) -> None:
    if workspace is None:
        ws_bytes = csa_sparse_attn_workspace_size(H, n_sel, swa)
        workspace = _scratch(ws_bytes, q)
    _check(lib().csa_sparse_attn_partial(_ptr(q), H, scale, kv_c, _ptr(sel), n_sel, kv_raw, n_tokens, swa,
                                         _ptr(o_part), _ptr(lse_part), _ptr(workspace), ws_bytes, _stream(stream)),
           "csa_sparse_attn_partial")


def csa_attn_merge(o_parts, lse_parts, R: int, H: int, out, lse=None, stream=None) -> None:
    _check(lib().csa_attn_merge(_ptr(o_parts), _ptr(lse_parts), R, H, _ptr(out), _ptr(lse), _stream(stream)),
           "csa_attn_merge")


def csa_decode_workspace_size(p: csa_decode_params) -> int:
    return int(lib().csa_decode_workspace_size(ctypes.byref(p)))


def copy_batch_args(pairs) -> "ctypes.Array":
    """The csa_copy array for csa_copy_batch from (src, dst[, bytes]) pairs of tensors or raw
    pointers; bytes defaults to the source tensor's size."""
    def addr(x):  # a device tensor, a pinned host tensor, or a raw pointer
        if isinstance(x, int):
            return x
        if not x.is_cuda and not x.is_pinned():
            raise ValueError("csa_copy_batch takes device or pinned host tensors")
        return x.data_ptr()
    arr = (csa_copy * len(pairs))()
    for i, pr in enumerate(pairs):
        src, dst = pr[0], pr[1]
        nbytes = pr[2] if len(pr) > 2 else src.numel() * src.element_size()
        arr[i] = csa_copy(addr(src), addr(dst), nbytes)
    return arr


def csa_copy_batch(copies, stream=None) -> None:
    """Enqueue up to CSA_COPY_MAX copies as one kernel (device or pinned host memory on either
    side; 16-byte aligned, sizes multiples of 16).  `copies`: a csa_copy array (copy_batch_args)."""
    _check(lib().csa_copy_batch(len(copies), copies, _stream(stream)), "csa_copy_batch")


def csa_selftest_bounded_wait(stream=None) -> None:
    """Enqueue the bounded-wait self-test: its wait runs out and sets CSA_ERR_TIMEOUT in the
    device status word (read it with csa_read_device_status)."""
    _check(lib().csa_selftest_bounded_wait(_stream(stream)), "csa_selftest_bounded_wait")


def csa_hisparse_create(B: int, table_stride: int, n_slots: int) -> int:
    """A HiSparse coordinator (an opaque handle); release it with csa_hisparse_destroy."""
    h = ctypes.c_void_p()
    _check(lib().csa_hisparse_create(B, table_stride, n_slots, ctypes.byref(h)), "csa_hisparse_create")
    return h.value


def csa_hisparse_destroy(h: int) -> None:
    lib().csa_hisparse_destroy(h)


def csa_hisparse_plan(h: int, touch, step: int, max_plan: int):
    """The host-side LRU decision for `touch` (numpy uint32 [B, table_stride]) -> (plan [n, 3]
    int32 rows (request, logical page, slot), number evicted)."""
    import numpy as np
    t = np.ascontiguousarray(touch, dtype=np.uint32)
    plan = np.zeros((max(int(max_plan), 1), 3), dtype=np.int32)
    n_in, n_ev = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().csa_hisparse_plan(h, t.ctypes.data, step, plan.ctypes.data, int(max_plan), ctypes.byref(n_in),
                                   ctypes.byref(n_ev)), "csa_hisparse_plan")
    return plan[: n_in.value].copy(), n_ev.value


def csa_hisparse_table(h: int, B: int, table_stride: int):
    """A copy of the coordinator's residency table (numpy int32 [B, table_stride])."""
    import numpy as np
    ptr = lib().csa_hisparse_table(h)
    return np.ctypeslib.as_array(ptr, shape=(B * table_stride,)).reshape(B, table_stride).copy()


def csa_hisparse_update(h: int, p: csa_decode_params, stream=None):
    """After a decode step: bring the pages it missed into the working set -> (n_in, n_evicted)."""
    n_in, n_ev = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().csa_hisparse_update(h, ctypes.byref(p), _stream(stream), ctypes.byref(n_in), ctypes.byref(n_ev)),
           "csa_hisparse_update")
    return n_in.value, n_ev.value


def csa_hisparse_collect(h: int, p: csa_decode_params, stream=None) -> None:
    """After a decode step: enqueue the readback of its page stamps (no wait)."""
    _check(lib().csa_hisparse_collect(h, ctypes.byref(p), _stream(stream)), "csa_hisparse_collect")


def csa_hisparse_apply(h: int, p: csa_decode_params, n_tokens_host, stream=None, side_stream=None):
    """Plan from the collected stamps; evictions on `stream`, the swap on `side_stream`
    (n_tokens_host: numpy int64 [B], the token counts of the last enqueued step) -> (n_in, n_evicted)."""
    import numpy as np
    nt = np.ascontiguousarray(n_tokens_host, dtype=np.int64)
    n_in, n_ev = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().csa_hisparse_apply(h, ctypes.byref(p), nt.ctypes.data, _stream(stream), _stream(side_stream),
                                    ctypes.byref(n_in), ctypes.byref(n_ev)), "csa_hisparse_apply")
    return n_in.value, n_ev.value


def csa_decode(p: csa_decode_params, workspace, ws_bytes: int, stream=None) -> None:
    _check(lib().csa_decode(ctypes.byref(p), _ptr(workspace), ws_bytes, _stream(stream)), "csa_decode")


def csa_decode_timed(p: csa_decode_params, workspace, ws_bytes: int, stream=None, events=None) -> None:
    """events: 5 torch.cuda.Event(enable_timing=True) recorded around the four stages (or None)."""
    arr = None
    if events is not None:
        arr = (ctypes.c_void_p * 5)(*[e.cuda_event for e in events])
    _check(lib().csa_decode_timed(ctypes.byref(p), _ptr(workspace), ws_bytes, _stream(stream), arr),
           "csa_decode_timed")


def csa_decode_noalloc(p: csa_decode_params, stream=None) -> None:
    """csa_decode with the library's own fixed 32 MiB scratch (for callers that cannot allocate)."""
    _check(lib().csa_decode_noalloc(ctypes.byref(p), _stream(stream)), "csa_decode_noalloc")


def csa_read_device_status(stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib().csa_read_device_status(_stream(stream), ctypes.byref(v)), "csa_read_device_status")
    return int(v.value)


def csa_version() -> int:
    return int(lib().csa_version())


from .runtime import DecodeBatch  # noqa: E402  (device-resident batch + params builder)
