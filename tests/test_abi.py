"""The C ABI: the shared library loads and exports every entry point declared in include/csa.h
(no compute: this runs without a GPU)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    from deepseek_v4_hybrid_c4_gb300 import build
    return build.build()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["csa_compress", "csa_index_score", "csa_topk", "csa_sparse_attn", "csa_decode"]:
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (csa_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_library_loads_and_answers_host_queries(libpath):
    import ctypes
    import deepseek_v4_hybrid_c4_gb300 as csa
    L = csa.lib()
    assert csa.csa_version() >= 100
    assert csa.status_string(csa.CSA_ERR_WORKSPACE) == "workspace missing or too small"
    for n in declared_functions():
        assert hasattr(L, n)
    # argument validation is synchronous and touches no device memory
    assert L.csa_topk(None, 10, 4, None, None, None, 0, None) == csa.CSA_ERR_INVALID_ARG
    assert L.csa_topk(None, 10, 0, None, None, None, 0, None) == csa.CSA_ERR_UNSUPPORTED
    assert csa.csa_topk_workspace_size(1, 1000, 512) > 0 and csa.csa_topk_workspace_size(0, 1000, 512) == 0
    assert csa.csa_topk_workspace_size(1, 1000, 0) == 0 and csa.csa_topk_workspace_size(1, 1000, 2049) == 0
    assert csa.csa_topk_workspace_size(32, 1000, 512) > csa.csa_topk_workspace_size(1, 1000, 512)
    assert csa.csa_topk_workspace_size(1, -1, 512) == 0
    p = csa.csa_decode_params()
    assert L.csa_decode(ctypes.byref(p), None, 0, None) == csa.CSA_ERR_UNSUPPORTED
    assert csa.csa_decode_workspace_size(p) == 0


def test_index_score_bounds_validates_its_arguments(libpath):
    """csa_index_score_bounds rejects synchronously, with nothing enqueued: fp8 keys and head
    counts outside 1..16 (unsupported), missing or misaligned pointers, a negative or oversized G,
    a page table whose pages are not whole 16-row boxes."""
    import ctypes
    import deepseek_v4_hybrid_c4_gb300 as csa
    L = csa.lib()
    a16 = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    a4 = ctypes.c_void_p(0x10004)
    contiguous = csa.csa_paged(0x20000, None, 16, 16 * 256, 4)
    f = L.csa_index_score_bounds
    assert f(a16, a16, 8, contiguous, csa.CSA_FP8_E4M3, 64, None, a16, None) == csa.CSA_ERR_UNSUPPORTED
    assert f(a16, a16, 0, contiguous, csa.CSA_BF16, 64, None, a16, None) == csa.CSA_ERR_UNSUPPORTED
    assert f(a16, a16, 17, contiguous, csa.CSA_BF16, 64, None, a16, None) == csa.CSA_ERR_UNSUPPORTED
    assert f(None, a16, 8, contiguous, csa.CSA_BF16, 64, None, a16, None) == csa.CSA_ERR_INVALID_ARG
    assert f(a4, a16, 8, contiguous, csa.CSA_BF16, 64, None, a16, None) == csa.CSA_ERR_INVALID_ARG
    assert f(a16, a16, 8, contiguous, csa.CSA_BF16, 64, None, None, None) == csa.CSA_ERR_INVALID_ARG
    assert f(a16, a16, 8, contiguous, csa.CSA_BF16, 64, ctypes.c_void_p(0x10002), a16, None) == csa.CSA_ERR_INVALID_ARG
    assert f(a16, a16, 8, contiguous, csa.CSA_BF16, -1, None, a16, None) == csa.CSA_ERR_INVALID_ARG
    assert f(a16, a16, 8, contiguous, csa.CSA_BF16, 1 << 31, None, a16, None) == csa.CSA_ERR_INVALID_ARG
    paged8 = csa.csa_paged(0x20000, 0x30000, 8, 8 * 256, 4)
    assert f(a16, a16, 8, paged8, csa.CSA_BF16, 64, None, a16, None) == csa.CSA_ERR_UNSUPPORTED
    assert f(a16, a16, 8, contiguous, csa.CSA_BF16, 0, None, a16, None) == csa.CSA_OK  # nothing to do


def test_binding_has_the_c_names():
    import deepseek_v4_hybrid_c4_gb300 as csa
    for n in declared_functions():
        if n not in ("csa_status_string",):
            assert callable(getattr(csa, n)), n


def test_product_path_does_not_reach_the_oracle():
    """The package never imports the oracle or the generators."""
    pkg = os.path.join(ROOT, "deepseek_v4_hybrid_c4_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+(oracle|synth)\b", src, re.M), f
                assert "liboracle" not in src and "orc_" not in src, f


def test_every_workload_fits_the_noalloc_scratch(libpath):
    """csa_decode_noalloc serves each of the five synthetic workloads at full size: the
    workspace each needs (a host-side computation, no device) fits its fixed 32 MiB array."""
    import synth
    import deepseek_v4_hybrid_c4_gb300 as csa
    for i in range(5):
        c = synth.config(i)
        p = csa.csa_decode_params()
        p.B, p.ratio, p.H, p.Hi, p.k, p.swa = len(c.requests), c.ratio, c.H, c.Hi, c.k, c.swa
        p.scale = 0.04
        p.k_dtype = csa.CSA_BF16 if c.kdtype == "bf16" else csa.CSA_FP8_E4M3
        p.max_tokens = max(r.n_tokens for r in c.requests)
        for f in ("n_tokens", "n_groups_done", "kv_raw", "kv_c", "k_idx", "w_gate", "b_pos", "q", "q_idx", "w_h",
                  "out", "lse", "sel", "page_table", "c_page_table"):
            setattr(p, f, 4096)  # never dereferenced by the size query
        p.raw_rows_per_page, p.raw_page_stride, p.n_pages = c.rows_per_page, c.rows_per_page * 1024, 1 << 20
        p.c_rows_per_page, p.c_page_stride, p.c_n_pages = 16, 16 * 1024, 1 << 20
        p.kidx_page_stride = 16 * 256
        need = csa.csa_decode_workspace_size(p)
        assert 0 < need <= 32 << 20, (i, need)


def test_ring_parameters_are_validated(libpath):
    """The compression-state ring is checked on the host: a ring size that is not a multiple
    of the ratio, a misaligned pool or no ring pages reject the call (workspace size 0)."""
    import synth
    import deepseek_v4_hybrid_c4_gb300 as csa
    c = synth.config(0)
    p = csa.csa_decode_params()
    p.B, p.ratio, p.H, p.Hi, p.k, p.swa = len(c.requests), c.ratio, c.H, c.Hi, c.k, c.swa
    p.scale, p.k_dtype, p.max_tokens = 0.04, csa.CSA_BF16, max(r.n_tokens for r in c.requests)
    for f in ("n_tokens", "n_groups_done", "kv_raw", "kv_c", "k_idx", "w_gate", "b_pos", "q", "q_idx", "w_h",
              "out", "lse", "sel", "page_table"):
        setattr(p, f, 4096)  # never dereferenced by the size query
    p.raw_rows_per_page, p.raw_page_stride, p.n_pages = c.rows_per_page, c.rows_per_page * 1024, 1 << 20
    p.c_page_stride, p.kidx_page_stride = (c.rows_per_page // 4) * 1024, (c.rows_per_page // 4) * 256
    base = csa.csa_decode_workspace_size(p)
    assert base > 0
    p.ring_pool, p.ring_page, p.ring_size, p.ring_n_pages = 8192, 4096, 8, 4
    assert csa.csa_decode_workspace_size(p) == base
    for field, bad in (("ring_size", 6), ("ring_size", 2), ("ring_pool", 8200), ("ring_n_pages", 0), ("ring_page", None)):
        good = getattr(p, field)
        setattr(p, field, bad)
        assert csa.csa_decode_workspace_size(p) == 0, (field, bad)
        setattr(p, field, good)


def _ref_lru(state, touch, step):
    """The documented coordinator policy, restated: refresh this step's resident pages; then each
    missed page of this step, in (request, page) order, takes a free slot (lowest first) or
    evicts the resident page with the oldest stamp other than this step's (lowest slot on ties)."""
    import numpy as np
    table, owner, stamp = state
    flat = table.reshape(-1)
    t = touch.reshape(-1)
    for e in np.nonzero(t == step)[0]:
        if flat[e] >= 0:
            stamp[flat[e]] = step
    cand = [s for s in range(len(owner)) if owner[s] < 0]
    cand += sorted([s for s in range(len(owner)) if owner[s] >= 0 and stamp[s] != step], key=lambda s: (stamp[s], s))
    plan, ev = [], 0
    for e in np.nonzero(t == step)[0]:
        if flat[e] >= 0:
            continue
        if not cand:
            break
        s = cand.pop(0)
        if owner[s] >= 0:
            flat[owner[s]] = -1
            ev += 1
        owner[s], stamp[s], flat[e] = e, step, s
        plan.append((e // table.shape[1], e % table.shape[1], s))
    return plan, ev


def test_hisparse_plan_is_lru(libpath):
    """The coordinator's host-side decisions over random access traces equal the restated
    policy, keep slots and table consistent, and never evict a page read in the same step."""
    import numpy as np
    import deepseek_v4_hybrid_c4_gb300 as csa
    rng = np.random.default_rng(5)
    B, stride, slots = 3, 40, 24
    h = csa.csa_hisparse_create(B, stride, slots)
    try:
        state = (np.full((B, stride), -1, np.int64), np.full(slots, -1, np.int64), np.zeros(slots, np.int64))
        for step in range(1, 30):
            touch = np.zeros((B, stride), np.uint32)
            hot = rng.integers(0, 8)  # a drifting hot set plus random pages
            for b in range(B):
                touch[b, (hot + np.arange(5)) % stride] = step
                touch[b, rng.integers(0, stride, size=rng.integers(0, 9))] = step
            touch[touch == 0] = rng.integers(0, step, size=int((touch == 0).sum()))  # older stamps
            plan, ev = csa.csa_hisparse_plan(h, touch, step, slots)
            rplan, rev = _ref_lru(state, touch, step)
            assert [tuple(x) for x in plan.tolist()] == rplan and ev == rev, step
            table = csa.csa_hisparse_table(h, B, stride)
            assert np.array_equal(table, state[0])
            held = table[table >= 0]
            assert len(np.unique(held)) == len(held)  # no slot twice
            n_touched = int((touch == step).sum())
            assert int(((table >= 0) & (touch == step)).sum()) == min(n_touched, slots)
    finally:
        csa.csa_hisparse_destroy(h)


def test_ctypes_structs_match_the_header(tmp_path):
    """Every field offset and the size of csa_paged, csa_decode_params and csa_copy, as a C
    compiler lays them out from include/csa.h, equal the ctypes binding's."""
    import ctypes
    import shutil
    import subprocess
    import deepseek_v4_hybrid_c4_gb300 as csa
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "csa.h"', "int main(void) {"]
    for st in (csa.csa_paged, csa.csa_decode_params, csa.csa_copy):
        cname = st.__name__
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in st._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        name, field, value = line.split()
        got[(name, field)] = int(value)
    for st in (csa.csa_paged, csa.csa_decode_params, csa.csa_copy):
        assert got[(st.__name__, "size")] == ctypes.sizeof(st), st.__name__
        for f, _ in st._fields_:
            assert got[(st.__name__, f)] == getattr(st, f).offset, (st.__name__, f)


def _valid_params(csa, synth):
    """Decode parameters of workload 0 that the host accepts (pointers never dereferenced)."""
    c = synth.config(0)
    p = csa.csa_decode_params()
    p.B, p.ratio, p.H, p.Hi, p.k, p.swa = len(c.requests), c.ratio, c.H, c.Hi, c.k, c.swa
    p.scale, p.k_dtype, p.max_tokens = 0.04, csa.CSA_BF16, max(r.n_tokens for r in c.requests)
    for f in ("n_tokens", "n_groups_done", "kv_raw", "kv_c", "k_idx", "w_gate", "b_pos", "q", "q_idx", "w_h",
              "out", "lse", "sel", "page_table"):
        setattr(p, f, 4096)
    p.raw_rows_per_page, p.raw_page_stride, p.n_pages = c.rows_per_page, c.rows_per_page * 1024, 1 << 20
    p.c_page_stride, p.kidx_page_stride = (c.rows_per_page // 4) * 1024, (c.rows_per_page // 4) * 256
    return p


def test_query_positions_are_validated(libpath):
    """n_q: 0 and 1 are one position; up to 16 positions; B * n_q within the grid limit.  The
    workspace grows with the positions (scores, histograms, lists, partials per position)."""
    import synth
    import deepseek_v4_hybrid_c4_gb300 as csa
    p = _valid_params(csa, synth)
    one = csa.csa_decode_workspace_size(p)
    p.n_q = 1
    assert csa.csa_decode_workspace_size(p) == one
    p.n_q = 4
    four = csa.csa_decode_workspace_size(p)
    assert four > one
    for bad in (17, -1):
        p.n_q = bad
        assert csa.csa_decode_workspace_size(p) == 0, bad
    p.n_q, p.B = 16, 5000  # 80,000 batch entries > 65,535
    assert csa.csa_decode_workspace_size(p) == 0


def test_hisparse_parameters_are_validated(libpath):
    """HiSparse needs ratio 4, an explicit compressed page table, a residency table, at least one
    slot and a 16-byte aligned working set; otherwise the call is refused on the host."""
    import synth
    import deepseek_v4_hybrid_c4_gb300 as csa
    p = _valid_params(csa, synth)
    p.c_page_table, p.c_page_table_stride, p.c_rows_per_page, p.c_n_pages = 4096, 64, 16, 1 << 20
    base = csa.csa_decode_workspace_size(p)
    assert base > 0
    p.hs_ws_pool, p.hs_ws_table, p.hs_n_slots, p.hs_touch, p.hs_step = 8192, 4096, 32, 4096, 1
    assert csa.csa_decode_workspace_size(p) == base  # the working set needs no workspace
    for field, bad in (("hs_ws_table", None), ("hs_n_slots", 0), ("hs_ws_pool", 8200), ("c_page_table", None)):
        good = getattr(p, field)
        setattr(p, field, bad)
        assert csa.csa_decode_workspace_size(p) == 0, (field, bad)
        setattr(p, field, good)
    p.ratio = 128  # C128 is dense: every step reads every entry, so no mirror
    assert csa.csa_decode_workspace_size(p) == 0


def test_hisparse_coordinator_rejects_bad_arguments(libpath):
    import deepseek_v4_hybrid_c4_gb300 as csa
    for args in ((0, 10, 4), (2, 0, 4), (2, 10, 0)):
        with pytest.raises(csa.CsaError):
            csa.csa_hisparse_create(*args)
    h = csa.csa_hisparse_create(1, 8, 2)
    try:
        import numpy as np
        plan, ev = csa.csa_hisparse_plan(h, np.zeros((1, 8), np.uint32), 1, 2)
        assert len(plan) == 0 and ev == 0  # nothing read in step 1: nothing to bring in
        assert (csa.csa_hisparse_table(h, 1, 8) == -1).all()
    finally:
        csa.csa_hisparse_destroy(h)


def test_copy_batch_validates_its_arguments(libpath):
    """csa_copy_batch rejects, before enqueueing anything: no copies or more than CSA_COPY_MAX, a
    null array or pointer, a source or destination not 16-byte aligned, a size not a multiple of
    16; an all-empty batch is accepted with nothing to do (no GPU touched: the pointers below are
    never dereferenced)."""
    import deepseek_v4_hybrid_c4_gb300 as csa
    f = csa.lib().csa_copy_batch
    one = (csa.csa_copy * 1)()
    assert f(0, one, None) == csa.CSA_ERR_INVALID_ARG
    assert f(csa.CSA_COPY_MAX + 1, (csa.csa_copy * (csa.CSA_COPY_MAX + 1))(), None) == csa.CSA_ERR_INVALID_ARG
    assert f(1, None, None) == csa.CSA_ERR_INVALID_ARG
    for src, dst, n in [(0, 32, 16), (16, 0, 16), (8, 32, 16), (16, 40, 16), (16, 32, 24)]:
        one[0] = csa.csa_copy(src, dst, n)
        assert f(1, one, None) == csa.CSA_ERR_INVALID_ARG, (src, dst, n)
    one[0] = csa.csa_copy(16, 32, 0)
    assert f(1, one, None) == csa.CSA_OK
