"""Pins of the CPU oracle against facts that do not come from the oracle itself:
closed forms, brute force, library routines (numpy, torch casts, Python's sorted),
exact rational arithmetic and hand-derived golden cases (tests/golden/).

Each test names the stage it pins; a plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a different summation order) fails
at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f2bf(x) -> np.ndarray:
    """float -> bf16 bits through torch's cast (a library routine, RNE)."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf2f(b) -> np.ndarray:
    return torch.tensor(np.asarray(b, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


# ----------------------------------------------------------------- storage types
def test_bf16_decode_matches_torch_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(codes)
    ref = bf2f(codes)
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).float().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert ((ours == ref) | both_nan).all()
    # OCP table values
    assert ours[0x7E] == 448.0 and ours[0x38] == 1.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def _nearest_bf16_bruteforce(x: float) -> int:
    """Nearest bf16 by exact rational comparison of the two neighbours (ties to even mantissa)."""
    f = np.float32(x)
    cands = set()
    for v in (f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))):
        b = int(np.array(v, dtype=np.float32).view(np.uint32))
        cands.add(b >> 16)
        cands.add(((b >> 16) + 1) & 0xFFFF)
        cands.add(((b >> 16) - 1) & 0xFFFF)
    best = None
    X = Fraction(x)
    for c in cands:
        v = float(bf2f(np.array([c], dtype=np.uint16))[0])
        if not math.isfinite(v):
            continue
        d = abs(Fraction(v) - X)
        key = (d, c & 1)  # equal distance: the even code wins
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_f64_to_bf16_single_rounding_bruteforce():
    rng = np.random.default_rng(123)
    xs = list(rng.standard_normal(400) * 10.0 ** rng.integers(-30, 30, 400))
    # exact midpoints between bf16 neighbours (ties) and values just off them
    for m in range(128, 256, 7):
        mid = (m + 0.5) / 128.0
        xs += [mid, -mid, math.nextafter(mid, 0), math.nextafter(mid, 2)]
    xs += [1e-40, -3e-39, 2.0 ** -133, 1.5 * 2.0 ** -133]  # subnormals
    for x in xs:
        assert int(oracle.f64_to_bf16([x])[0]) == _nearest_bf16_bruteforce(float(x)), x


# ----------------------------------------------------------------- stage 1: compressor
def _gate_inputs(seed=7, ratio=4, n_groups=3):
    x = synth.normal_bf16((n_groups * ratio, 512), seed, 11)
    w = synth.normal_f32((512,), seed, 12, 0.0, 1 / math.sqrt(512))
    b = synth.normal_f32((ratio,), seed, 13, 0.0, math.sqrt(0.1))
    return x, w, b


@pytest.mark.parametrize("ratio", [4, 128])
def test_compress_identical_tokens_give_that_token(ratio):
    x, w, b = _gate_inputs(ratio=ratio)
    for g in range(3):
        x[g * ratio:(g + 1) * ratio] = x[g * ratio]
    out = oracle.compress(x, ratio, w, b)
    for g in range(3):
        assert np.array_equal(out[g], x[g * ratio])


@pytest.mark.parametrize("ratio", [4, 128])
def test_compress_gates_sum_to_one_and_follow_definition(ratio):
    x, w, b = _gate_inputs(ratio=ratio)
    _, gates = oracle.compress(x, ratio, w, b, want_gates=True)
    assert np.allclose(gates.sum(axis=1), 1.0, atol=1e-12, rtol=0)
    # gate logits from numpy (library dot products) -> softmax
    xf = bf2f(x).astype(np.float64).reshape(3, ratio, 512)
    s = xf @ w.astype(np.float64) + b.astype(np.float64)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    assert np.allclose(gates, e / e.sum(axis=1, keepdims=True), atol=1e-12, rtol=0)


def test_compress_zero_gate_is_arithmetic_mean():
    x, _, _ = _gate_inputs()
    out, f64 = oracle.compress(x, 4, np.zeros(512, np.float32), np.zeros(4, np.float32), want_f64=True)
    mean = bf2f(x).astype(np.float64).reshape(3, 4, 512).mean(axis=1)
    assert np.allclose(f64, mean, atol=1e-15, rtol=0)
    # the bf16 output is the fp64 mean rounded once, to nearest with ties to even: 8 significant
    # bits from frexp's mantissa in [0.5, 1), rounded by rint (half to even); all values normal
    m, e = np.frexp(mean)
    expect = np.ldexp(np.rint(m * 256.0), e - 8)
    assert np.array_equal(out, f2bf(expect.astype(np.float32)))  # expect is on the bf16 grid: exact


def test_compress_one_hot_bias_selects_token():
    x, w, _ = _gate_inputs()
    for i in range(4):
        b = np.zeros(4, np.float32)
        b[i] = 1e4
        out = oracle.compress(x, 4, w, b)
        for g in range(3):
            assert np.array_equal(out[g], x[g * 4 + i])


def test_compress_permutation_of_tokens_with_bias():
    x, w, b = _gate_inputs()
    _, ref = oracle.compress(x, 4, w, b, want_f64=True)
    perm = np.array([2, 0, 3, 1])
    xp = x.reshape(3, 4, 512)[:, perm].reshape(12, 512).copy()
    _, got = oracle.compress(xp, 4, w, b[perm].copy(), want_f64=True)
    assert np.allclose(got, ref, atol=1e-12, rtol=0)


def test_compress_group_range_and_later_groups_only():
    x, w, b = _gate_inputs()
    full = oracle.compress(x, 4, w, b)
    part = oracle.compress(x, 4, w, b, first_group=1, n_groups=2)
    assert np.array_equal(part, full[1:])


def test_compress_golden_closed_form():
    rows = {}
    for line in open(os.path.join(GOLDEN, "compress_c4_closed_form.txt")):
        if line.startswith("dim "):
            d, vals = line[4:].split(":")
            rows[int(d)] = [float(v) for v in vals.split()]
    x = np.zeros((4, 512), np.float32)
    for d, vals in rows.items():
        x[:, d] = vals
    xb = f2bf(x)
    assert np.array_equal(bf2f(xb), x)  # fixture values are bf16-exact
    w = np.zeros(512, np.float32)
    w[0] = 1.0
    out, f64 = oracle.compress(xb, 4, w, np.zeros(4, np.float32), want_f64=True)
    z = sum(math.exp(i) for i in range(4))
    a = [math.exp(i) / z for i in range(4)]
    for d in range(512):
        exp_val = sum(a[i] * float(x[i, d]) for i in range(4))
        assert abs(f64[0, d] - exp_val) <= 1e-13 * max(1.0, abs(exp_val)), d
        assert int(out[0, d]) == _nearest_bf16_bruteforce(exp_val), d


# ----------------------------------------------------------------- stage 2: index score
def _parse_score_cases():
    cases, cur = [], None
    for raw in open(os.path.join(GOLDEN, "score_chunk_order.txt")):
        line = raw.split("#")[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = dict(name=tok[1], heads=[], kdtype="bf16")
            cases.append(cur)
        elif tok[0] == "kdtype":
            cur["kdtype"] = tok[1]
        elif tok[0] == "w":
            cur["w"] = [float(v) for v in tok[1:]]
        elif tok[0].startswith("h"):
            cur["heads"].append([t.split(":") for t in tok[1:]])
        elif tok[0] == "expect":
            cur["expect"] = eval(" ".join(tok[1:]), {"__builtins__": {}})
    return cases


@pytest.mark.parametrize("case", _parse_score_cases(), ids=lambda c: c["name"])
def test_score_golden_chunk_order(case):
    Hi = len(case["heads"])
    q = np.zeros((Hi, 128), np.float32)
    fp8 = case["kdtype"] == "fp8"
    k = np.zeros(128, np.uint8) if fp8 else np.zeros(128, np.float32)
    for h, triples in enumerate(case["heads"]):
        for d, qv, kv in triples:
            q[h, int(d)] = float(qv)
            if fp8:
                k[int(d)] = int(kv, 16)
            else:
                k[int(d)] = float(kv)
    qb = f2bf(q)
    assert np.array_equal(bf2f(qb), q)
    kk = k[None, :] if fp8 else f2bf(k)[None, :]
    s = oracle.index_score(qb, np.array(case["w"], np.float32), kk, fp8)
    assert float(s[0]) == float(np.float32(case["expect"])), (s[0], case["expect"])


def test_score_small_integers_exact():
    """Small-integer inputs: every fp32 operation is exact, so the score equals the exact integer formula."""
    rng = np.random.default_rng(5)
    Hi, G = 6, 200
    q = rng.integers(-3, 4, (Hi, 128)).astype(np.float32)
    k = rng.integers(-3, 4, (G, 128)).astype(np.float32)
    w = np.array([1, 0.5, 2, 0.25, 4, 1], np.float32)
    s = oracle.index_score(f2bf(q), w, f2bf(k), False)
    dots = k.astype(np.int64) @ q.astype(np.int64).T  # exact integers
    ref = (np.maximum(dots, 0) * w.astype(np.float64)).sum(axis=1)
    assert np.array_equal(s.astype(np.float64), ref)


def test_score_single_head_error_bound_vs_exact():
    """Hi = 1, w = 1: score = max(q.k, 0) within the fp32 bound of 11 roundings of the stated tree."""
    q = synth.normal_bf16((1, 128), 9, 1)
    k = synth.normal_bf16((64, 128), 9, 2)
    s = oracle.index_score(q, np.ones(1, np.float32), k, False)
    qf, kf = bf2f(q)[0], bf2f(k)
    u = 2.0 ** -24
    for g in range(64):
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qf, kf[g]))
        bound = 11 * u * sum(abs(float(a) * float(b)) for a, b in zip(qf, kf[g])) * (1 + 1e-6)
        ref = max(exact, Fraction(0))
        assert abs(Fraction(float(s[g])) - ref) <= Fraction(bound), g


def test_score_relu_and_weight_scaling():
    q = synth.normal_bf16((8, 128), 10, 1)
    k = synth.normal_bf16((300, 128), 10, 2)
    w = synth.uniform_f32((8,), 10, 3)
    s1 = oracle.index_score(q, w, k, False)
    s2 = oracle.index_score(q, 2 * w, k, False)
    assert np.array_equal(s2, 2 * s1)  # doubling every weight doubles the score exactly
    neg = oracle.index_score(q, w, (k.astype(np.uint32) ^ 0x8000).astype(np.uint16), False)  # k -> -k
    # each head keeps exactly one of ReLU(d), ReLU(-d): the two scores sum to sum_h w_h |d_h| (no score < 0)
    assert (s1 >= 0).all() and (neg >= 0).all()


def test_score_fp8_matches_bf16_of_same_values():
    """fp8 keys decode exactly into bf16, so an fp8 row and its bf16 copy score identically."""
    q = synth.normal_bf16((8, 128), 11, 1)
    k8 = synth.normal_e4m3((500, 128), 11, 2)
    kb = f2bf(oracle.e4m3_to_f32(k8))
    w = synth.uniform_f32((8,), 11, 3)
    assert np.array_equal(oracle.index_score(q, w, k8, True), oracle.index_score(q, w, kb, False))


# ----------------------------------------------------------------- stage 3: top-k
def _brute_topk(scores, k):
    order = sorted(range(len(scores)), key=lambda g: (-float(scores[g]), g))
    res = order[:k]
    return res + [-1] * (k - len(res))


@pytest.mark.parametrize("G,k", [(1, 4), (7, 16), (64, 8), (64, 64), (200, 17), (1000, 512)])
def test_topk_equals_brute_force_with_ties(G, k):
    rng = np.random.default_rng(G * 1000 + k)
    vals = np.array([0.0, -0.0, 1.5, -2.0, np.inf, -np.inf, 3.25, 1e-30, -1e-30], np.float32)
    s = np.where(rng.random(G) < 0.5, vals[rng.integers(0, len(vals), G)], rng.standard_normal(G).astype(np.float32))
    assert oracle.topk(s, k).tolist() == _brute_topk(s, k)


@pytest.mark.parametrize("G,k", [(1, 4), (7, 16), (64, 8), (64, 64), (200, 17), (1000, 512), (20000, 512)])
def test_topk_by_selection_equals_brute_force(G, k):
    """The selection form (partition to rank k, sort the k) against the brute-force order."""
    rng = np.random.default_rng(G * 7 + k)
    vals = np.array([0.0, -0.0, 1.5, -2.0, np.inf, -np.inf, 3.25], np.float32)
    s = np.where(rng.random(G) < 0.5, vals[rng.integers(0, len(vals), G)], rng.standard_normal(G).astype(np.float32))
    idx, keys = oracle.topk_select(s, k, want_keys=True)
    assert idx.tolist() == _brute_topk(s, k)
    assert np.array_equal(keys[: min(k, G)], np.array([oracle.score_key(s[g]) for g in idx[: min(k, G)]], np.uint32))
    assert (keys[min(k, G):] == 0).all()


def test_topk_all_equal_and_k_ge_G():
    s = np.full(50, 2.0, np.float32)
    assert oracle.topk(s, 10).tolist() == list(range(10))
    assert oracle.topk(s, 64).tolist() == list(range(50)) + [-1] * 14
    s[17] = -0.0
    s[3] = 0.0
    s[:] = 0.0
    s[9] = -0.0
    assert oracle.topk(s, 50).tolist() == list(range(50))  # -0 ties +0


def test_topk_key_is_order_preserving():
    rng = np.random.default_rng(3)
    x = np.sort(np.concatenate([rng.standard_normal(500) * 1e3, [-np.inf, np.inf, 0.0, 1e-40, -1e-40]]).astype(np.float32))
    keys = [oracle.score_key(v) for v in x]
    for a, b, ka, kb in zip(x[:-1], x[1:], keys[:-1], keys[1:]):
        assert (ka < kb) == (a < b) and (ka == kb) == (a == b)


# ----------------------------------------------------------------- stage 4: attention
def test_attention_single_key_returns_its_row():
    q = synth.normal_bf16((16, 512), 20, 1)
    row = synth.normal_bf16((1, 512), 20, 2)
    sc = float(np.float32(0.044))
    out, _, lse = oracle.attention(q, sc, row)
    assert np.array_equal(out, np.repeat(row, 16, axis=0))
    ref = sc * (bf2f(q).astype(np.float64) @ bf2f(row)[0].astype(np.float64))
    assert np.allclose(lse, ref, atol=1e-12, rtol=0)


def test_attention_equal_logits_give_mean_and_log_n():
    rows = synth.normal_bf16((37, 512), 21, 1)
    q = np.zeros((4, 512), np.uint16)  # q = 0 -> all logits 0
    _, f64, lse = oracle.attention(q, 0.1, rows)
    assert np.allclose(f64, bf2f(rows).astype(np.float64).mean(axis=0), atol=1e-14, rtol=0)
    assert np.allclose(lse, math.log(37), atol=1e-14, rtol=0)


def test_attention_matches_numpy_textbook():
    q = synth.normal_bf16((8, 512), 22, 1)
    rows = synth.normal_bf16((300, 512), 22, 2)
    scale = float(np.float32(1 / math.sqrt(512)))
    _, f64, lse = oracle.attention(q, scale, rows)
    Q, K = bf2f(q).astype(np.float64), bf2f(rows).astype(np.float64)
    L = scale * Q @ K.T
    m = L.max(axis=1, keepdims=True)
    P = np.exp(L - m)
    ref = (P / P.sum(axis=1, keepdims=True)) @ K
    assert np.allclose(f64, ref, atol=1e-12, rtol=0)
    assert np.allclose(lse, (m[:, 0] + np.log(P.sum(axis=1))), atol=1e-12, rtol=0)


def test_sparse_attn_key_set_is_selection_plus_swa():
    rng = np.random.default_rng(4)
    G, N, swa = 300, 1200, 128
    cpool = synth.normal_bf16((G, 512), 23, 1)
    raw = synth.normal_bf16((N, 512), 23, 2)
    q = synth.normal_bf16((4, 512), 23, 3)
    sel = rng.permutation(G)[:50].astype(np.int32)
    sel_padded = np.concatenate([sel, -np.ones(14, np.int32)])
    _, f64, lse = oracle.sparse_attn(q, 0.05, cpool, sel_padded, raw, swa)
    rows = np.concatenate([cpool[sel], raw[N - swa:]])
    _, f64r, lser = oracle.attention(q, 0.05, rows[::-1].copy())  # any order of the key set
    assert np.allclose(f64, f64r, atol=1e-12, rtol=0) and np.allclose(lse, lser, atol=1e-12, rtol=0)
    # short context: W = min(swa, N)
    _, f64s, _ = oracle.sparse_attn(q, 0.05, cpool, sel, raw[:40], swa)
    _, f64t, _ = oracle.attention(q, 0.05, np.concatenate([cpool[sel], raw[:40]]))
    assert np.allclose(f64s, f64t, atol=1e-12, rtol=0)


def test_selecting_every_candidate_is_dense_attention():
    G, N = 64, 256
    cpool = synth.normal_bf16((G, 512), 24, 1)
    raw = synth.normal_bf16((N, 512), 24, 2)
    q = synth.normal_bf16((2, 512), 24, 3)
    sc = float(np.float32(0.05))  # the oracle takes the scale as fp32
    _, f64, _ = oracle.sparse_attn(q, sc, cpool, np.arange(G, dtype=np.int32), raw, 128)
    Q = bf2f(q).astype(np.float64)
    K = np.concatenate([bf2f(cpool), bf2f(raw[N - 128:])]).astype(np.float64)
    L = sc * Q @ K.T
    P = np.exp(L - L.max(axis=1, keepdims=True))
    assert np.allclose(f64, (P / P.sum(axis=1, keepdims=True)) @ K, atol=1e-12, rtol=0)


# ----------------------------------------------------------------- the decode step
def test_decode_composes_the_stages():
    case = synth.make_decode_case("t", 5, [2048], H=16, Hi=4, k=64, n_pending=2)
    r = case.requests[0]
    res = oracle.decode_request(r, ratio=4, w_gate=case.w_gate, b_pos=case.b_pos, k=64, swa=128, scale=case.scale)
    G = 512
    comp = oracle.compress(r.raw, 4, case.w_gate, case.b_pos, first_group=G - 2, n_groups=2)
    assert np.array_equal(res["cpool"][G - 2:], comp)
    assert np.array_equal(res["cpool"][:G - 2], r.cpool[:G - 2])
    s = oracle.index_score(r.q_idx, r.w_h, r.kidx, False)
    assert np.array_equal(res["scores"], s)
    assert res["sel"].tolist() == _brute_topk(s, 64)
    out, f64, lse = oracle.sparse_attn(r.q, case.scale, res["cpool"], res["sel"], r.raw, 128)
    assert np.array_equal(res["out"], out) and np.allclose(res["lse"], lse, atol=0, rtol=0)


def test_decode_dense_c128():
    case = synth.make_decode_case("t", 6, [1024, 2048], H=8, Hi=0, ratio=128, k=0)
    res = oracle.decode_case(case)
    for r, o in zip(case.requests, res):
        G = r.n_tokens // 128
        assert np.array_equal(o["cpool"][G - 1], oracle.compress(r.raw, 128, case.w_gate, case.b_pos, G - 1, 1)[0])
        ref = oracle.sparse_attn(r.q, case.scale, o["cpool"], np.arange(G, dtype=np.int32), r.raw, 128)
        assert np.array_equal(o["out"], ref[0])


def test_decode_queries_positions_and_candidates():
    """Speculative verify in the oracle: query j of n_q sees the first N - n_q + j + 1 tokens.
    The last query is the plain decode step; a query whose prefix holds no completed group
    attends only its SWA window (textbook attention over those raw rows); and a query's
    candidates are exactly the groups completed within its prefix (floor), scored as before."""
    case = synth.make_decode_case("t", 7, [1024 + 8], H=16, Hi=4, k=64, n_pending=2)
    r = case.requests[0]
    kw = dict(ratio=4, w_gate=case.w_gate, b_pos=case.b_pos, k=64, swa=128, scale=case.scale)
    qs = [(synth.normal_bf16((16, 512), 7, 90 + j), r.q_idx, r.w_h) for j in range(3)] + [(r.q, r.q_idx, r.w_h)]
    res = oracle.decode_queries(r, qs, **kw)
    plain = oracle.decode_request(r, **kw)
    assert np.array_equal(res[3]["out"], plain["out"]) and np.array_equal(res[3]["sel"], plain["sel"])
    N = r.n_tokens
    for j in range(3):
        Nj = N - 4 + j + 1
        s = oracle.index_score(r.q_idx, r.w_h, r.kidx[: Nj // 4], False)
        assert np.array_equal(res[j]["scores"], s)              # floor(Nj / 4) candidates
        assert res[j]["sel"].tolist() == _brute_topk(s, 64)
    # a prefix of 3 tokens: no completed group, only the window
    tiny = synth.make_decode_case("t", 8, [8], H=4, Hi=4, k=4, n_pending=2)
    t = tiny.requests[0]
    q0 = synth.normal_bf16((4, 512), 8, 95)
    one = oracle.decode_queries(t, [(q0, t.q_idx, t.w_h)] + [(t.q, t.q_idx, t.w_h)] * 5,
                                ratio=4, w_gate=tiny.w_gate, b_pos=tiny.b_pos, k=4, swa=128, scale=tiny.scale)
    _, f64, lse = oracle.attention(q0, tiny.scale, t.raw[:3])
    assert np.allclose(one[0]["out_f64"], f64, atol=0, rtol=0) and (one[0]["sel"] == -1).all()


def test_fp8_tie_codebook_creates_straddling_ties():
    """Workload 3's recipe: codebook index keys make exact score ties around rank k."""
    case = synth.make_decode_case("t", 3, [8192], H=4, Hi=8, kdtype="fp8", tie_codebook=True, k=512)
    r = case.requests[0]
    s = oracle.index_score(r.q_idx, r.w_h, r.kidx, True)
    idx = oracle.topk(s, 513)
    assert s[idx[511]] == s[idx[512]]  # the k-th and (k+1)-th candidates tie: the lower index must win
