"""Stage 2 as tensor-core brackets (csa_index_score_bounds) and the decode step's select built
on them.  Every bracket must hold the oracle's fixed-order score (lower <= s <= upper, as
floats); its half-width must be the stated 2^-13 * max_j |k_gj| * sum_h |w_h| ||q_h||_1 (+1e-30);
non-finite cases must give (-inf, +inf).  The decode step (bf16 keys) then selects exactly the
oracle's top k, including inputs built to put many exact ties and near-ties at the threshold."""
import numpy as np
import pytest

import oracle
import synth
from helpers import dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def csa():
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v4_hybrid_c4_gb300 as m
    m.csa_read_device_status()
    return m


def _bf16(x):
    """fp32 -> bf16 bits (round to nearest even), as uint16."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _bounds(csa, q, w, k, paged=False, seed=0):
    G = k.shape[0]
    Hi = q.shape[0]
    if paged:
        rpp = 16
        n_pages = (G + rpp - 1) // rpp + 2
        pt = synth.permutation(n_pages, seed, 4)[: (G + rpp - 1) // rpp].copy()
        pool = np.zeros((n_pages * rpp, 128), np.uint16)
        synth.scatter_pages(k, rpp, pt, pool, rpp * 256)
        kp = csa.paged(dev(pool, torch), rpp, 256, page_table=dev(pt, torch), n_pages=n_pages)
    else:
        kp = csa.paged(dev(k, torch), 16, 256, n_pages=(G + 15) // 16)
    lo = torch.full((G,), float("nan"), device="cuda")
    up = torch.full((G,), float("nan"), device="cuda")
    csa.csa_index_score_bounds(dev(q, torch), dev(w, torch), Hi, kp, csa.CSA_BF16, G, lo, up)
    torch.cuda.synchronize()
    return lo.cpu().numpy(), up.cpu().numpy()


def _half_width(q, w, k):
    """The stated half-width in fp64 (before the kernel's upward rounding)."""
    qf = _f32(q).astype(np.float64)
    kf = np.abs(_f32(k).astype(np.float64)).max(axis=1)
    c = (np.abs(w.astype(np.float64)) * np.abs(qf).sum(axis=1)).sum()
    return 2.0 ** -13 * kf * c + 1e-30


def _check_bracket(lo, up, s, what):
    bad = ~((lo <= s) & (s <= up))
    assert not bad.any(), f"{what}: {int(bad.sum())} brackets miss the score, first at {int(np.argmax(bad))}"


@pytest.mark.parametrize("Hi", [1, 4, 8, 13, 16])
@pytest.mark.parametrize("G,paged", [(1, False), (127, False), (1000, True), (40000, True), (40001, False)])
def test_bounds_hold_the_fixed_order_score(csa, Hi, G, paged):
    seed = 700 + Hi + G
    k = synth.normal_bf16((G, 128), seed, 1)
    q = synth.normal_bf16((Hi, 128), seed, 2)
    w = synth.uniform_f32((Hi,), seed, 3)
    lo, up = _bounds(csa, q, w, k, paged, seed)
    s = oracle.index_score(q, w, k, False)
    _check_bracket(lo, up, s, f"Hi={Hi} G={G}")
    e = _half_width(q, w, k)
    hw = (up.astype(np.float64) - lo.astype(np.float64)) / 2
    # the stated half-width, rounded up once or twice in fp32 (and the 0.1% the kernel adds)
    assert np.all(hw >= e * (1 - 1e-6)), "bracket narrower than stated"
    assert np.all(hw <= e * 1.002 + np.abs(s) * 2.0 ** -22 + 1e-37), "bracket wider than stated"
    assert csa.csa_read_device_status() == 0


def test_bounds_cancellation_signs_and_zeros(csa):
    """Dots that cancel to zero from large terms, negative weights, a zero query head, keys
    spanning many binades: the bracket still holds the fixed-order score."""
    G, Hi = 4096, 8
    rng = np.random.default_rng(5)
    k = rng.standard_normal((G, 128)).astype(np.float32)
    k[:1024, 1::2] = -k[:1024, 0::2]                     # pairs that cancel against q = 1
    k[1024:2048] *= np.float32(2.0) ** rng.integers(-60, 60, (1024, 1)).astype(np.float32)
    k[2048:2100] = 0.0
    q = rng.standard_normal((Hi, 128)).astype(np.float32)
    q[0] = 1.0
    q[3] = 0.0
    w = rng.uniform(-1.0, 1.0, Hi).astype(np.float32)
    kb, qb = _bf16(k), _bf16(q)
    lo, up = _bounds(csa, qb, w, kb)
    s = oracle.index_score(qb, w, kb, False)
    _check_bracket(lo, up, s, "cancellation")
    assert np.all(np.isfinite(lo)) and np.all(np.isfinite(up))
    assert csa.csa_read_device_status() == 0


def test_bounds_non_finite_give_the_whole_line(csa):
    """A NaN or infinite key, or products that overflow fp32, give (-inf, +inf); the other rows
    keep finite brackets."""
    G, Hi = 256, 4
    k = synth.normal_bf16((G, 128), 9, 1)
    q = synth.normal_bf16((Hi, 128), 9, 2)
    w = synth.uniform_f32((Hi,), 9, 3)
    k[3, 7] = 0x7FC0       # NaN
    k[40, 0] = 0x7F80      # +inf
    k[41, 5] = 0xFF80      # -inf
    k[100, :] = 0x7F00     # 1.7e38 in every dim: the dots overflow
    lo, up = _bounds(csa, q, w, k)
    odd = [3, 40, 41, 100]
    assert np.all(np.isneginf(lo[odd])) and np.all(np.isposinf(up[odd]))
    rest = np.setdiff1d(np.arange(G), odd)
    s = oracle.index_score(q, w, k, False)
    _check_bracket(lo[rest], up[rest], s[rest], "finite rows")
    assert csa.csa_read_device_status() == 0


def test_bounds_reject_fp8(csa):
    k = torch.zeros((16, 128), dtype=torch.uint8, device="cuda")
    q = torch.zeros((4, 128), dtype=torch.int16, device="cuda")
    w = torch.zeros(4, device="cuda")
    up = torch.zeros(16, device="cuda")
    with pytest.raises(RuntimeError):
        csa.csa_index_score_bounds(q, w, 4, csa.paged(k, 16, 128, n_pages=1), csa.CSA_FP8_E4M3, 16, None, up)


# ------------------------------------------------------------------ the decode step on the bounds
def _decode_check(entry, case, n_q=1):
    """One step of the case, every selection compared as a set with the oracle's, outputs within
    the bf16 tolerance.  n_q > 1: every request verifies n_q draft positions with its own query
    (the same keys, fewer candidates for the earlier positions) -- the tensor-core bounds path."""
    import deepseek_v4_hybrid_c4_gb300 as m
    from test_gpu_2_decode import _check_against_oracle
    from helpers import assert_close
    if n_q == 1:
        batch = entry.case_to_batch(case)
        batch.run()
        torch.cuda.synchronize()
        assert m.csa_read_device_status() == 0
        _check_against_oracle(case, batch)
        return batch
    per = [[(r.q, r.q_idx, r.w_h)] * n_q for r in case.requests]
    flat = [x for p in per for x in p]
    batch = entry.case_to_batch(case, n_q=n_q, q=np.stack([x[0] for x in flat]),
                                q_idx=np.stack([x[1] for x in flat]), w_h=np.stack([x[2] for x in flat]))
    batch.run()
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    out = batch.out.float().cpu().numpy().astype(np.float64)
    for b, r in enumerate(case.requests):
        refs = oracle.decode_queries(r, per[b], ratio=case.ratio, w_gate=case.w_gate, b_pos=case.b_pos, k=case.k,
                                     swa=case.swa, scale=case.scale, kdtype=case.kdtype)
        for j, ref in enumerate(refs):
            e = b * n_q + j
            got = batch.sel[e].cpu().numpy()
            n = int((ref["sel"] >= 0).sum())
            assert (got[n:] == -1).all() and np.array_equal(np.sort(got[:n]), np.sort(ref["sel"][:n])), (b, j)
            assert_close(out[e], ref["out_f64"], f"{case.name} request {b} query {j}")
    return batch


@pytest.fixture(scope="module")
def entry(csa):
    import __graft_entry__
    return __graft_entry__


@pytest.mark.parametrize("n_q", [1, 2, 4])
@pytest.mark.parametrize("G,rows_per_book", [(30000, 16), (65536, 64), (5000, 2)])
def test_decode_bf16_ties_at_the_threshold(entry, G, rows_per_book, n_q):
    """bf16 keys drawn from a small codebook: groups of candidates with identical exact scores,
    so whole tie groups straddle the k-th place and the lower indices must win."""
    case = synth.make_decode_case("bf16-ties", 40 + rows_per_book, [4 * G], H=16, Hi=8, paged=True)
    r = case.requests[0]
    rng = np.random.default_rng(G)
    book = r.kidx[rng.integers(0, G, max(1, G // rows_per_book))]
    r.kidx[:] = book[rng.integers(0, book.shape[0], G)]
    _decode_check(entry, case, n_q)


@pytest.mark.parametrize("n_q", [1, 2, 3])
def test_decode_near_ties_inside_the_bounds(entry, n_q):
    """Candidates whose exact scores differ by a few ulps (keys that differ in one low bit):
    inside any bracket's width, so only the exact rescoring can order them."""
    G = 20000
    case = synth.make_decode_case("near", 77, [4 * G], H=16, Hi=4, paged=False)
    r = case.requests[0]
    base = r.kidx[int(np.argmax(oracle.index_score(r.q_idx, r.w_h, r.kidx, False)))].copy()  # a top row
    rng = np.random.default_rng(1)
    for i in rng.choice(G, 3000, replace=False):
        row = base.copy()
        j = rng.integers(0, 128, 3)
        row[j] ^= np.uint16(1)  # one-ulp changes in three dims
        r.kidx[i] = row
    _decode_check(entry, case, n_q)


@pytest.mark.parametrize("n_q", [1, 2, 4])
def test_decode_negative_weights_and_batch(entry, n_q):
    """Index weights of both signs (scores below zero) in a ragged bf16 batch."""
    case = synth.make_decode_case("negw", 91, [4096, 40000, 516, 131072 // 8], H=64, Hi=8, paged=True, n_pending=2)
    rng = np.random.default_rng(3)
    for r in case.requests:
        r.w_h[:] = rng.uniform(-1.0, 1.0, r.w_h.shape).astype(np.float32)
    _decode_check(entry, case, n_q)


def test_decode_all_scores_equal_on_the_bounds(entry):
    """Every key equal, four positions: every bracket is the same, every candidate is rescored
    (more than the exact select ranks in shared memory: its radix path over the lists), and the
    set is candidates 0 .. k-1 at every position."""
    case = synth.make_decode_case("eq4", 13, [4 * 10240], H=16, Hi=4, k=512)
    for r in case.requests:
        r.kidx[:] = r.kidx[0]
    batch = _decode_check(entry, case, 4)
    for e in range(4):
        assert np.array_equal(np.sort(batch.sel[e].cpu().numpy()), np.arange(512))
