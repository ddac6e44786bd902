"""The fused decode step (csa_decode through the C ABI) against the oracle on the five
workloads: tiny; 128K; 1M paged; ragged batch of 32 with fp8 keys and planted ties; C128 dense.
Reduced-size variants run first; the full sizes follow (the oracle is plain C, so it finishes
them in seconds).  Selections are compared exactly, outputs within the bf16 tolerance."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, bf16_bits_to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def entry():
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v4_hybrid_c4_gb300 as m
    m.csa_read_device_status()
    return __graft_entry__


def run_and_check(entry, case):
    import deepseek_v4_hybrid_c4_gb300 as m
    batch = entry.case_to_batch(case)
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    return _check_against_oracle(case, batch)


def _check_against_oracle(case, batch):
    refs = oracle.decode_case(case)
    out = batch.out.float().cpu().numpy().astype(np.float64)
    lse = batch.lse.cpu().numpy()
    c_rpp = case.c_rows_per_page()
    for b, (r, ref) in enumerate(zip(case.requests, refs)):
        if case.ratio == 4:
            # the step's selection is the top-k set (csa_topk's order is tested in the stage tests)
            got_sel = batch.sel[b].cpu().numpy()
            n = int((ref["sel"] >= 0).sum())
            assert (got_sel[n:] == -1).all(), f"request {b}: padding"
            assert np.array_equal(np.sort(got_sel[:n]), np.sort(ref["sel"][:n])), f"request {b}: top-k set differs"
        assert_close(out[b], ref["out_f64"], f"{case.name} request {b} output")
        assert np.abs(lse[b] - ref["lse"]).max() <= 1e-3 * max(1.0, np.abs(ref["lse"]).max())
        # the pending groups were compressed into the pool
        G = r.n_tokens // case.ratio
        if r.n_groups_done < G:
            pages = case.c_pages(r)
            rows = [int(pages[g // c_rpp]) * c_rpp + g % c_rpp for g in range(r.n_groups_done, G)]
            got_rows = batch.c_pool[torch.tensor(rows, device=batch.c_pool.device)].cpu().numpy().view(np.uint16)
            ref_rows = oracle.compress(r.raw, case.ratio, case.w_gate, case.b_pos, r.n_groups_done,
                                       G - r.n_groups_done, want_f64=True)[1]
            assert_close(bf16_bits_to_f64(got_rows), ref_rows, f"{case.name} request {b} compressed rows")
    return batch


@pytest.mark.parametrize("cfg,scale_down", [(0, 1), (1, 8), (2, 16), (3, 16), (4, 64)])
def test_decode_reduced(entry, cfg, scale_down):
    run_and_check(entry, synth.config(cfg, scale_down=scale_down))


def test_decode_paged_equals_contiguous(entry):
    a = synth.make_decode_case("pg", 11, [20000], H=64, Hi=8, paged=True, spare_pages=40)
    b = synth.make_decode_case("ct", 11, [20000], H=64, Hi=8, paged=False)
    ba = run_and_check(entry, a)
    bb = run_and_check(entry, b)
    assert torch.equal(ba.sel, bb.sel)
    assert torch.equal(ba.out, bb.out)


def test_decode_ragged_with_short_requests(entry):
    """Ragged batch including a request with a single candidate (G < k) and two pending groups."""
    case = synth.make_decode_case("rg", 12, [4096, 516, 12000, 4, 2048], H=16, Hi=4, k=128, n_pending=2)
    run_and_check(entry, case)


@pytest.mark.parametrize("G", [6000, 10240])
def test_decode_select_all_scores_equal(entry, G):
    """Every index key equal, so every score ties: the select refines down to the index digits
    (its general path; above 8,192 candidates it rereads them from L2 each round).  Ties go to
    the lower index, so the set is candidates 0 .. k-1 -- checked in closed form besides the
    oracle."""
    case = synth.make_decode_case("eq", 13, [4 * G], H=16, Hi=4, k=512)
    for r in case.requests:
        r.kidx[:] = r.kidx[0]
    batch = run_and_check(entry, case)
    assert np.array_equal(np.sort(batch.sel[0].cpu().numpy()), np.arange(512))


def _rings(case, ring_size, spare=3):
    """Per-request compression-state rings holding each request's last ring_size tokens (token t
    in row ring_page[b] * ring_size + t % ring_size); ring pages are a seeded permutation."""
    B = len(case.requests)
    page = synth.permutation(B + spare, case.seed, 31)[:B].copy()
    pool = np.zeros(((B + spare) * ring_size, 512), np.uint16)
    for b, r in enumerate(case.requests):
        for t in range(max(0, r.n_tokens - ring_size), r.n_tokens):
            pool[page[b] * ring_size + t % ring_size] = r.raw[t]
    return dict(ring_pool=pool, ring_page=page, ring_size=ring_size)


@pytest.mark.parametrize("ratio,ring_size,n_pending", [(4, 8, 1), (4, 8, 2), (4, 16, 3), (128, 128, 1),
                                                       (128, 256, 2)])
def test_decode_ring_matches_oracle(entry, ratio, ring_size, n_pending):
    """Pending groups compressed from the compression-state rings: the whole step matches."""
    case = synth.make_decode_case(f"ring{ratio}", 40 + ring_size, [4096 + 4 * ratio, 8192, 1024 + ratio * n_pending],
                                  H=64, Hi=8, ratio=ratio, n_pending=n_pending)
    case.name = f"ring r{ratio} size {ring_size}"
    import deepseek_v4_hybrid_c4_gb300 as m
    batch = entry.case_to_batch(case, **_rings(case, ring_size))
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    _check_against_oracle(case, batch)


def test_decode_ring_is_the_source(entry):
    """With rings set, the raw pool's pending rows are never read by the compressor: zero them
    and the compressed rows still match the oracle on the true tokens."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case("ringsrc", 45, [4096, 2048 + 8], H=16, Hi=4, n_pending=2)
    batch = entry.case_to_batch(case, **_rings(case, 8))
    rpp = case.rows_per_page
    for r in case.requests:
        G = r.n_tokens // case.ratio
        for t in range(r.n_groups_done * case.ratio, G * case.ratio):
            batch.raw_pool[int(r.pages[t // rpp]) * rpp + t % rpp] = 0
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    c_rpp = case.c_rows_per_page()
    for b, r in enumerate(case.requests):
        G = r.n_tokens // case.ratio
        pages = case.c_pages(r)
        rows = [int(pages[g // c_rpp]) * c_rpp + g % c_rpp for g in range(r.n_groups_done, G)]
        got = batch.c_pool[torch.tensor(rows, device="cuda")].cpu().numpy().view(np.uint16)
        ref = oracle.compress(r.raw, case.ratio, case.w_gate, case.b_pos, r.n_groups_done, G - r.n_groups_done,
                              want_f64=True)[1]
        assert_close(bf16_bits_to_f64(got), ref, f"ring-sourced compressed rows, request {b}")


def test_decode_ring_too_small_sets_status(entry):
    """A ring that no longer holds every pending token: the device status reports a bounds
    error (no fault, no trap)."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case("ringsmall", 46, [4096], H=16, Hi=4, n_pending=2)
    batch = entry.case_to_batch(case, **_rings(case, 4))
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 1 << (m.CSA_ERR_DEVICE_BOUNDS - 1)
    assert m.csa_read_device_status() == 0  # read-and-clear


def _spec_queries(case, n_q, seed_stream=300):
    """n_q query positions per request: q, q_idx, w_h drawn like the case's own (own streams)."""
    qs = []
    for b, r in enumerate(case.requests):
        q = synth.normal_bf16((n_q, case.H, 512), case.seed, seed_stream + 3 * b)
        qi = synth.normal_bf16((n_q, max(case.Hi, 1), 128), case.seed, seed_stream + 3 * b + 1)
        wh = synth.uniform_f32((n_q, max(case.Hi, 1)), case.seed, seed_stream + 3 * b + 2)
        qs.append([(q[j], qi[j], wh[j]) for j in range(n_q)])
    return qs


@pytest.mark.parametrize("ratio,n_q,n_pending", [(4, 2, 1), (4, 4, 2), (4, 3, 1), (128, 4, 1), (128, 2, 2)])
def test_decode_speculative_verify(entry, ratio, n_q, n_pending):
    """n_q query positions per request, each with its own candidates (groups completed before
    it), top k and SWA window, against the oracle run once per position."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case(f"spec{ratio}", 50 + n_q, [8192, 4096 + 4 * ratio, 20000 // ratio * ratio],
                                  H=64 if ratio == 128 else 16, Hi=8, ratio=ratio, n_pending=n_pending)
    qs = _spec_queries(case, n_q)
    flat = [x for per in qs for x in per]  # (request, query) order
    batch = entry.case_to_batch(case, n_q=n_q, q=np.stack([x[0] for x in flat]),
                                q_idx=np.stack([x[1] for x in flat]), w_h=np.stack([x[2] for x in flat]))
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    out = batch.out.float().cpu().numpy().astype(np.float64)
    lse = batch.lse.cpu().numpy()
    for b, r in enumerate(case.requests):
        refs = oracle.decode_queries(r, qs[b], ratio=ratio, w_gate=case.w_gate, b_pos=case.b_pos, k=case.k,
                                     swa=case.swa, scale=case.scale, kdtype=case.kdtype)
        for j, ref in enumerate(refs):
            e = b * n_q + j
            if ratio == 4:
                got = batch.sel[e].cpu().numpy()
                n = int((ref["sel"] >= 0).sum())
                assert (got[n:] == -1).all() and np.array_equal(np.sort(got[:n]), np.sort(ref["sel"][:n])), (b, j)
            assert_close(out[e], ref["out_f64"], f"spec verify request {b} query {j}")
            assert np.abs(lse[e] - ref["lse"]).max() <= 1e-3 * max(1.0, np.abs(ref["lse"]).max())


def test_decode_one_query_position_is_the_plain_step(entry):
    """n_q = 1 is the ordinary decode step, bit for bit."""
    case = synth.config(0)
    a = entry.case_to_batch(case)
    b = entry.case_to_batch(case, n_q=1)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.sel, b.sel) and torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)


def _hisparse_batch(entry, case, slots):
    """The case with its C4 pool as a pinned host mirror (the shadow paging made explicit) and a
    GPU working set of `slots` pages, empty at first."""
    c_rpp = case.rows_per_page // case.ratio
    return entry.case_to_batch(case, c_page_table=case.page_table(), c_rows_per_page=c_rpp, c_n_pages=case.n_pages,
                               hs_slots=slots), c_rpp


def test_hisparse_mirror_and_working_set(entry):
    """Step 1 reads every selected row from the host mirror and stamps their pages; the
    coordinator then brings those pages in; step 2 reads them from the working set.  Both steps
    match the oracle, the stamps are exactly the selected pages, and the slots hold the mirror's
    bytes."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case("hs", 60, [65536, 20000], H=16, Hi=8, n_pending=1)
    batch, c_rpp = _hisparse_batch(entry, case, slots=2048)
    batch.hs_step = 1
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    _check_against_oracle(case, batch)
    touch = batch.hs_touch.cpu().numpy()
    want = np.zeros_like(touch)
    for b in range(len(case.requests)):
        s = batch.sel[b].cpu().numpy()
        want[b, np.unique(s[s >= 0] // c_rpp)] = 1
    assert np.array_equal(touch, want)
    n_in, n_ev = batch.hs_update()
    assert n_in == int(want.sum()) and n_ev == 0
    table = batch.hs_table.cpu().numpy()
    assert ((table >= 0) == (want == 1)).all()
    pt = case.page_table()
    pool = batch.c_pool.numpy()
    slots = batch.hs_pool.cpu().numpy()
    for b, lp in zip(*np.nonzero(table >= 0)):
        sl = table[b, lp]
        assert np.array_equal(slots[sl * c_rpp:(sl + 1) * c_rpp], pool[pt[b, lp] * c_rpp:(pt[b, lp] + 1) * c_rpp])
    batch.out.zero_()
    batch.hs_step = 2
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    _check_against_oracle(case, batch)
    assert np.array_equal(batch.hs_touch.cpu().numpy(), want * 2)


def test_hisparse_many_requests_pages_on_both_sides(entry):
    """Twenty-four requests, so each attention split takes two key tiles (the lookups of a tile
    are issued a tile ahead of its gather), with a working set that holds only part of the
    selected pages: rows come from slots and from the mirror in the same tiles.  Both steps
    match the oracle."""
    import deepseek_v4_hybrid_c4_gb300 as m
    lengths = [6000 + 100 * i for i in range(24)]
    case = synth.make_decode_case("hs5", 64, lengths, H=16, Hi=4, n_pending=1)
    batch, c_rpp = _hisparse_batch(entry, case, slots=700)
    for step in (1, 2):
        batch.out.zero_()
        batch.hs_step = step
        batch.run()
        torch.cuda.synchronize()
        assert m.csa_read_device_status() == 0
        _check_against_oracle(case, batch)
        n_in, _ = batch.hs_update()
        if step == 1:
            assert n_in == 700
    table = batch.hs_table.cpu().numpy()
    touch = batch.hs_touch.cpu().numpy()
    assert (table >= 0).sum() == 700 and (touch == 2).sum() > 700  # some selected pages stayed in the mirror


def test_hisparse_small_working_set_evicts(entry):
    """A working set smaller than one step's pages: the coordinator fills it, the rest stay in
    the mirror, and the step still matches the oracle with pages on both sides."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case("hs2", 61, [40000], H=16, Hi=4, n_pending=1)
    batch, c_rpp = _hisparse_batch(entry, case, slots=64)
    for step in (1, 2, 3):
        batch.hs_step = step
        batch.run()
        torch.cuda.synchronize()
        assert m.csa_read_device_status() == 0
        _check_against_oracle(case, batch)
        n_in, n_ev = batch.hs_update()
        resident = int((batch.hs_table.cpu().numpy() >= 0).sum())
        assert resident == 64 and n_in == (64 if step == 1 else 0)


def test_hisparse_new_rows_reach_mirror_and_slot(entry):
    """The pending group's compressed row goes to the mirror and, its page being resident, to
    the slot as well."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case("hs3", 62, [8192 + 64], H=16, Hi=4, n_pending=1)
    batch, c_rpp = _hisparse_batch(entry, case, slots=8)
    r = case.requests[0]
    G = r.n_tokens // 4
    lp = (G - 1) // c_rpp
    batch.hs_table[0, lp] = 5
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    ref = oracle.compress(r.raw, 4, case.w_gate, case.b_pos, G - 1, 1, want_f64=True)[1]
    page = int(case.page_table()[0, lp])
    in_mirror = batch.c_pool.numpy().view(np.uint16)[page * c_rpp + (G - 1) % c_rpp]
    in_slot = batch.hs_pool.cpu().numpy().view(np.uint16)[5 * c_rpp + (G - 1) % c_rpp]
    assert_close(bf16_bits_to_f64(in_mirror[None]), ref, "new row in the mirror")
    assert np.array_equal(in_slot, in_mirror)


def test_hisparse_async_swaps_beside_the_steps(entry):
    """The asynchronous coordinator: each step's stamps are collected, and the swap they call for
    is applied after the next step is enqueued -- evictions on the decode stream, the copies and
    installs on a side stream beside the following steps.  The queries change every step, so
    pages come and go; every step still matches the oracle, and the final slots hold the
    mirror's bytes."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.make_decode_case("hs4", 63, [65536, 30000], H=16, Hi=8, n_pending=1)
    batch, c_rpp = _hisparse_batch(entry, case, slots=96)
    s, side = torch.cuda.Stream(), torch.cuda.Stream()
    n_tok = np.array([r.n_tokens for r in case.requests], np.int64)
    steps, outs, moved = 6, [], []
    qs = []
    for t in range(1, steps + 1):
        q = [synth.normal_bf16((case.H, 512), 63, 900 + 10 * t + b) for b in range(len(case.requests))]
        qi = [synth.normal_bf16((case.Hi, 128), 63, 950 + 10 * t + b) for b in range(len(case.requests))]
        qs.append((q, qi))
        with torch.cuda.stream(s):
            batch.q.copy_(torch.from_numpy(np.stack(q).view(np.int16)))
            batch.q_idx.copy_(torch.from_numpy(np.stack(qi).view(np.int16)))
            batch.hs_step = t
            batch.run(s)
            outs.append((batch.out.clone(), batch.lse.clone(), batch.sel.clone()))
            if t > 1:
                moved.append(batch.hs_apply(n_tok, s, side))  # the previous step's stamps
            batch.hs_collect(s)
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    assert sum(n for n, _ in moved) > 0 and sum(e for _, e in moved) > 0  # pages came in and went out
    for t, ((q, qi), (out, lse, sel)) in enumerate(zip(qs, outs)):
        for b, r in enumerate(case.requests):
            r.q, r.q_idx = q[b], qi[b]
        batch.out.copy_(out)
        batch.lse.copy_(lse)
        batch.sel.copy_(sel)
        _check_against_oracle(case, batch)
    table = batch.hs_table.cpu().numpy()
    assert np.array_equal(table, m.csa_hisparse_table(batch.hs, batch.B, table.shape[1]))
    pt = case.page_table()
    pool = batch.c_pool.numpy()
    slots = batch.hs_pool.cpu().numpy()
    assert (table >= 0).sum() > 0
    for b, lp in zip(*np.nonzero(table >= 0)):
        sl = table[b, lp]
        assert np.array_equal(slots[sl * c_rpp:(sl + 1) * c_rpp], pool[pt[b, lp] * c_rpp:(pt[b, lp] + 1) * c_rpp])
        G = case.requests[b].n_tokens // 4
        assert lp < (G - 1) // c_rpp  # the page still receiving rows was never brought in


def test_decode_graph_capture_replay(entry):
    """The step enqueues only device work: it can be captured once and replayed."""
    case = synth.config(0)
    batch = entry.case_to_batch(case)
    s = torch.cuda.Stream()
    batch.run(s)  # warm (sets kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        batch.run(s)
    batch.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.decode_case(case)[0]
    assert np.array_equal(np.sort(batch.sel[0].cpu().numpy()), np.sort(ref["sel"]))
    assert_close(batch.out[0].float().cpu().numpy(), ref["out_f64"], "graph replay")


@pytest.mark.parametrize("cfg,sd", [(0, 1), (3, 16), (4, 16)])
def test_decode_outputs_into_pinned_host_memory(entry, cfg, sd):
    """out and lse given as page-locked host memory: the merge kernel writes them over the host
    link, and the host receives the same bits the device-side outputs hold (one request, 32
    ragged requests, 8 dense C128 requests), from a captured graph."""
    import deepseek_v4_hybrid_c4_gb300 as m
    case = synth.config(cfg, scale_down=sd)
    batch = entry.case_to_batch(case)
    batch.run()
    torch.cuda.synchronize()
    out_d, lse_d = batch.out.cpu(), batch.lse.cpu()
    h_out = torch.full(out_d.shape, -1, dtype=out_d.dtype).pin_memory()
    h_lse = torch.full(lse_d.shape, float("nan"), dtype=lse_d.dtype).pin_memory()
    p = type(batch.params).from_buffer_copy(batch.params)
    p.out, p.lse = h_out.data_ptr(), h_lse.data_ptr()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.csa_decode(p, batch.ws, batch.ws_bytes, s)
    g.replay()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    assert torch.equal(h_out.view(torch.int16), out_d.view(torch.int16))
    assert torch.equal(h_lse.view(torch.int32), lse_d.view(torch.int32))


def test_decode_is_deterministic(entry):
    """Two runs of the same step give the same selection order and the same output bits."""
    case = synth.config(3, scale_down=16)
    batch = entry.case_to_batch(case)
    batch.run()
    torch.cuda.synchronize()
    sel, out, lse = batch.sel.clone(), batch.out.clone(), batch.lse.clone()
    for _ in range(2):
        batch.sel.fill_(-7)
        batch.out.zero_()
        batch.run()
        torch.cuda.synchronize()
        assert torch.equal(batch.sel, sel)
        assert torch.equal(batch.out, out)
        assert torch.equal(batch.lse, lse)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_decode_full_size(entry, cfg):
    run_and_check(entry, synth.config(cfg))
