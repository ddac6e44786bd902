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
            got_rows = batch.c_pool[torch.tensor(rows, device="cuda")].cpu().numpy().view(np.uint16)
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
