"""Per-stage parity of the CUDA path (through the C ABI) against the CPU oracle.

Index scores and top-k are compared bit for bit; compressed rows and attention
outputs within max-abs 2e-2 and relative-L2 5e-3 of the oracle's fp64 result.
Sizes span several tiles/units and ragged tails, plus the degenerate cases.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, bf16_bits_to_f64, dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def csa():
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v4_hybrid_c4_gb300 as m
    m.csa_read_device_status()  # start from a clear status word
    return m


def _status_clean(csa):
    torch.cuda.synchronize()
    assert csa.csa_read_device_status() == 0


# ------------------------------------------------------------------ stage 2: index score
@pytest.mark.parametrize("kdtype", ["bf16", "fp8"])
@pytest.mark.parametrize("Hi", [1, 4, 8, 16])
@pytest.mark.parametrize("G,paged", [(1, False), (17, False), (1000, True), (40000, True), (40001, False)])
def test_index_score_bitexact(csa, kdtype, Hi, G, paged):
    seed = 100 + Hi + G
    fp8 = kdtype == "fp8"
    k = (synth.normal_e4m3 if fp8 else synth.normal_bf16)((G, 128), seed, 1)
    q = synth.normal_bf16((Hi, 128), seed, 2)
    w = synth.uniform_f32((Hi,), seed, 3)
    rb = 128 if fp8 else 256
    if paged:
        rpp = 16
        n_pages = (G + rpp - 1) // rpp + 3
        pt = synth.permutation(n_pages, seed, 4)[: (G + rpp - 1) // rpp].copy()
        pool = np.zeros((n_pages * rpp, 128), k.dtype)
        synth.scatter_pages(k, rpp, pt, pool, rpp * rb)
        kp = csa.paged(dev(pool, torch), rpp, rb, page_table=dev(pt, torch), n_pages=n_pages)
    else:
        kp = csa.paged(dev(k, torch), 16, rb, n_pages=(G + 15) // 16)
    out = torch.full((G,), float("nan"), device="cuda")
    csa.csa_index_score(dev(q, torch), dev(w, torch), Hi, kp, csa.CSA_FP8_E4M3 if fp8 else csa.CSA_BF16, G, out)
    ref = oracle.index_score(q, w, k, fp8)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
        f"{int((got.view(np.uint32) != ref.view(np.uint32)).sum())} of {G} scores differ"
    _status_clean(csa)


def test_index_score_golden_cases(csa):
    """The hand-derived chunk-order cases (tests/golden/score_chunk_order.txt) on the GPU."""
    from test_oracle_pins import _parse_score_cases, f2bf
    for case in _parse_score_cases():
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
        kk = k[None, :] if fp8 else f2bf(k)[None, :]
        out = torch.zeros(1, device="cuda")
        csa.csa_index_score(dev(f2bf(q), torch), dev(np.array(case["w"], np.float32), torch), Hi,
                            csa.paged(dev(kk, torch), 16, 128 if fp8 else 256, n_pages=1),
                            csa.CSA_FP8_E4M3 if fp8 else csa.CSA_BF16, 1, out)
        assert float(out.item()) == float(np.float32(case["expect"])), case["name"]


# ------------------------------------------------------------------ stage 3: top-k
def _scores_with_ties(G, seed):
    rng = np.random.default_rng(seed)
    base = rng.standard_normal(G).astype(np.float32) * 10
    pool = np.array([0.0, -0.0, 3.5, 7.25, -1.0, np.inf, 12.0], np.float32)
    pick = rng.random(G) < 0.3
    base[pick] = pool[rng.integers(0, len(pool), pick.sum())]
    return base


def _topk_gpu(csa, s, k):
    sd = torch.from_numpy(s).cuda()
    idx = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    keys = torch.zeros((k,), dtype=torch.int32, device="cuda")
    csa.csa_topk(sd, s.shape[0], k, idx, keys)
    return idx.cpu().numpy(), keys.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("G", [1, 5, 511, 512, 513, 4096, 40000, 262144])
@pytest.mark.parametrize("k", [1, 7, 512, 2048])
def test_topk_bitexact(csa, G, k):
    s = _scores_with_ties(G, G * 7 + k)
    idx, keys = _topk_gpu(csa, s, k)
    ref, rkeys = oracle.topk(s, k, want_keys=True)
    assert np.array_equal(idx, ref)
    assert np.array_equal(keys, rkeys)
    _status_clean(csa)


def test_topk_all_equal_and_straddling_ties(csa):
    s = np.full(100000, 2.5, np.float32)
    idx, _ = _topk_gpu(csa, s, 512)
    assert np.array_equal(idx, np.arange(512))
    # a tie group straddling rank k spread over every CTA of the cluster
    s = np.zeros(262144, np.float32)
    s[::97] = 1.0   # 2703 equal scores at the top, k=512 takes the lowest indices
    idx, _ = _topk_gpu(csa, s, 512)
    assert np.array_equal(idx, oracle.topk(s, 512))
    _status_clean(csa)


def test_topk_candidate_overflow_path(csa):
    """More than the shared-memory candidate capacity share the threshold's bins."""
    rng = np.random.default_rng(9)
    s = np.ones(300000, np.float32)
    s[rng.integers(0, 300000, 100)] = 2.0
    s[rng.integers(0, 300000, 50000)] = np.float32(1.0000001)
    idx, _ = _topk_gpu(csa, s, 2048)
    assert np.array_equal(idx, oracle.topk(s, 2048))
    _status_clean(csa)


def test_topk_batched_ragged(csa):
    lens = [1, 300, 512, 513, 70000, 4097, 0, 33000]
    segs = [_scores_with_ties(n, 50 + i) for i, n in enumerate(lens)]
    flat = np.concatenate(segs).astype(np.float32)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    k = 512
    idx = torch.full((len(lens), k), -7, dtype=torch.int32, device="cuda")
    csa.csa_topk_batched(torch.from_numpy(flat).cuda(), torch.from_numpy(offs).cuda(), len(lens), max(lens), k, idx)
    got = idx.cpu().numpy()
    for b, sgm in enumerate(segs):
        assert np.array_equal(got[b], oracle.topk(sgm, k)), b
    _status_clean(csa)


def _straddling(G, k, seed):
    """Ragged random scores whose k-th largest value is shared by a group of about 3k entries
    spread over the whole range, so the tie group straddles rank k."""
    s = _scores_with_ties(G, seed)
    t = np.float32(np.partition(s, G - k)[G - k])
    rng = np.random.default_rng(seed + 1)
    s[rng.integers(0, G, min(G, 3 * k))] = t
    return s


@pytest.mark.parametrize("G", [1, 511, 513, 20000, 262144, 300001])
@pytest.mark.parametrize("k", [1, 512, 2048])
def test_topk_cluster_bitexact(csa, G, k):
    """The single-cluster form (distributed-shared-memory histograms) at any size."""
    s = _straddling(G, k, G + 3 * k) if G > k else _scores_with_ties(G, G + 3 * k)
    sd = torch.from_numpy(s).cuda()
    idx = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    keys = torch.zeros((k,), dtype=torch.int32, device="cuda")
    csa.csa_topk_cluster(sd, None, 1, G, k, idx, keys)
    ref, rkeys = oracle.topk(s, k, want_keys=True)
    assert np.array_equal(idx.cpu().numpy(), ref)
    assert np.array_equal(keys.cpu().numpy().view(np.uint32), rkeys)
    _status_clean(csa)


def test_topk_cluster_batched_ragged(csa):
    lens = [1, 300, 512, 513, 70000, 0, 33000, 262144]
    segs = [_scores_with_ties(n, 90 + i) for i, n in enumerate(lens)]
    flat = np.concatenate(segs).astype(np.float32)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    k = 512
    idx = torch.full((len(lens), k), -7, dtype=torch.int32, device="cuda")
    csa.csa_topk_cluster(torch.from_numpy(flat).cuda(), torch.from_numpy(offs).cuda(), len(lens), max(lens), k, idx)
    got = idx.cpu().numpy()
    for b, sgm in enumerate(segs):
        assert np.array_equal(got[b], oracle.topk(sgm, k)), b
    _status_clean(csa)


@pytest.mark.parametrize("G", [4194305, 6000000])
@pytest.mark.parametrize("k", [512, 2048])
def test_topk_above_the_wide_select(csa, G, k):
    """csa_topk and csa_topk_batched above 4,194,304 scores per request (the cluster form, its
    candidates overflowing shared memory and re-read from L2 each round), a tie group
    straddling rank k."""
    s = _straddling(G, k, G + k)
    idx, keys = _topk_gpu(csa, s, k)
    ref, rkeys = oracle.topk(s, k, want_keys=True)
    assert np.array_equal(idx, ref)
    assert np.array_equal(keys, rkeys)
    small = _scores_with_ties(1000, 5)
    flat = np.concatenate([small, s]).astype(np.float32)
    offs = np.array([0, 1000, 1000 + G], np.int64)
    got = torch.full((2, k), -7, dtype=torch.int32, device="cuda")
    csa.csa_topk_batched(torch.from_numpy(flat).cuda(), torch.from_numpy(offs).cuda(), 2, G, k, got)
    got = got.cpu().numpy()
    assert np.array_equal(got[0], oracle.topk(small, k))
    assert np.array_equal(got[1], ref)
    _status_clean(csa)


# ------------------------------------------------------------------ stage 1: compressor
@pytest.mark.parametrize("ratio,n_tokens,paged", [(4, 4096, False), (4, 8192 + 64, True), (128, 4096, True),
                                                  (128, 128 * 37, False),
                                                  # chunks that fill every SM take the streaming kernel:
                                                  # ragged last stage, stages across page boundaries
                                                  (4, 4 * 1300, False), (4, 4 * 1300, True),
                                                  (128, 128 * 160, True), (128, 128 * 170, False)])
def test_compress_matches_oracle(csa, ratio, n_tokens, paged):
    seed = ratio + n_tokens
    x = synth.normal_bf16((n_tokens, 512), seed, 1)
    wg = synth.normal_f32((512,), seed, 2, 0.0, 1 / math.sqrt(512))
    bp = synth.normal_f32((ratio,), seed, 3, 0.0, math.sqrt(0.1))
    G = n_tokens // ratio
    first = 3 if G > 10 else 0
    ng = G - first
    rpp = 64
    n_pages = (n_tokens + rpp - 1) // rpp
    if paged:
        pt = synth.permutation(n_pages + 5, seed, 4)[:n_pages].copy()
        pool = np.zeros(((n_pages + 5) * rpp, 512), np.uint16)
        synth.scatter_pages(x, rpp, pt, pool, rpp * 1024)
        raw = csa.paged(dev(pool, torch), rpp, 1024, page_table=dev(pt, torch), n_pages=n_pages + 5)
    else:
        raw = csa.paged(dev(x, torch), rpp, 1024, n_pages=n_pages)
    out = torch.zeros((G, 512), dtype=torch.int16, device="cuda")
    csa.csa_compress(raw, n_tokens, ratio, dev(wg, torch), dev(bp, torch), first, ng,
                     csa.paged(out, 1, 1024, n_pages=G))
    _, ref = oracle.compress(x, ratio, wg, bp, first_group=first, n_groups=ng, want_f64=True)
    got = bf16_bits_to_f64(out.cpu().numpy()[first:])
    assert_close(got, ref, f"compress r{ratio}")
    assert not out.cpu().numpy()[:first].any()  # groups before first_group untouched
    _status_clean(csa)


def test_compress_identical_tokens_exact(csa):
    x = synth.normal_bf16((64, 512), 5, 1)
    x = np.repeat(x[::4], 4, axis=0)  # every group of 4 is one token repeated
    wg = synth.normal_f32((512,), 5, 2, 0.0, 1 / math.sqrt(512))
    bp = synth.normal_f32((4,), 5, 3, 0.0, math.sqrt(0.1))
    out = torch.zeros((16, 512), dtype=torch.int16, device="cuda")
    csa.csa_compress(csa.paged(dev(x, torch), 64, 1024, n_pages=1), 64, 4, dev(wg, torch), dev(bp, torch), 0, 16,
                     csa.paged(out, 16, 1024, n_pages=1))
    got = out.cpu().numpy().view(np.uint16)
    diff = np.abs(bf16_bits_to_f64(got) - bf16_bits_to_f64(x[::4]))
    # gates sum to 1 in fp32: the result may move by at most one bf16 ulp
    assert (diff <= np.abs(bf16_bits_to_f64(x[::4])) * 2 ** -7).all()


# ------------------------------------------------------------------ stage 4: attention
def _attn_case(seed, H, G, n_sel, N, n_invalid=0):
    cpool = synth.normal_bf16((G, 512), seed, 1)
    raw = synth.normal_bf16((N, 512), seed, 2)
    q = synth.normal_bf16((H, 512), seed, 3)
    rng = np.random.default_rng(seed)
    sel = rng.permutation(G)[:n_sel].astype(np.int32)
    if n_invalid:
        sel[rng.permutation(n_sel)[:n_invalid]] = -1
    return cpool, raw, q, sel


def _attn_gpu(csa, cpool, raw, q, sel, swa, scale, paged_raw=None, dense_n=None):
    H = q.shape[0]
    G = cpool.shape[0]
    N = raw.shape[0]
    kc = csa.paged(dev(cpool, torch), 1, 1024, n_pages=G)
    if paged_raw is not None:
        pool, pt, n_pages = paged_raw
        kr = csa.paged(dev(pool, torch), 64, 1024, page_table=dev(pt, torch), n_pages=n_pages)
    else:
        kr = csa.paged(dev(raw, torch), 1, 1024, n_pages=max(N, 1))
    n_sel = dense_n if sel is None else len(sel)
    ws_n = csa.csa_sparse_attn_workspace_size(H, n_sel, swa)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = torch.zeros((H, 512), dtype=torch.int16, device="cuda")
    lse = torch.zeros(H, dtype=torch.float32, device="cuda")
    seld = None if sel is None else dev(sel, torch)
    csa.csa_sparse_attn(dev(q, torch), H, scale, kc, seld, n_sel, kr, N, swa, out, lse, ws, ws_n)
    return out.cpu().numpy().view(np.uint16), lse.cpu().numpy()


@pytest.mark.parametrize("H", [16, 64, 128])
@pytest.mark.parametrize("n_sel,N,n_invalid", [(512, 4096, 0), (512, 4096, 37), (100, 50, 0), (2048, 9000, 5),
                                               (1, 3, 0), (0, 200, 0)])
def test_sparse_attn_matches_oracle(csa, H, n_sel, N, n_invalid):
    scale = float(np.float32(1 / math.sqrt(512)))
    cpool, raw, q, sel = _attn_case(H * 1000 + n_sel, H, 4096, n_sel, N, n_invalid)
    out, lse = _attn_gpu(csa, cpool, raw, q, sel, 128, scale)
    _, f64, rlse = oracle.sparse_attn(q, scale, cpool, sel, raw, 128)
    assert_close(bf16_bits_to_f64(out), f64, f"attn H={H} n_sel={n_sel}")
    assert np.abs(lse - rlse).max() <= 1e-3 * max(1.0, np.abs(rlse).max())
    _status_clean(csa)


def test_dense_attn_c128_and_paged_raw(csa):
    scale = float(np.float32(1 / math.sqrt(512)))
    cpool, raw, q, _ = _attn_case(77, 64, 4096, 0, 8192)
    rpp = 64
    n_pages = 8192 // rpp
    pt = synth.permutation(n_pages + 3, 77, 9)[:n_pages].copy()
    pool = np.zeros(((n_pages + 3) * rpp, 512), np.uint16)
    synth.scatter_pages(raw, rpp, pt, pool, rpp * 1024)
    out, lse = _attn_gpu(csa, cpool, raw, q, None, 128, scale, paged_raw=(pool, pt, n_pages + 3), dense_n=4096)
    _, f64, rlse = oracle.sparse_attn(q, scale, cpool, np.arange(4096, dtype=np.int32), raw, 128)
    assert_close(bf16_bits_to_f64(out), f64, "dense C128 attention")
    _status_clean(csa)


@pytest.mark.parametrize("H", [16, 64])
def test_attn_padded_page_stride(csa, H):
    """Raw pages padded by half a row: the page stride is not a whole number of rows, so a
    row's address is page * stride + slot * 1 KiB, never page * rows_per_page + slot."""
    scale = float(np.float32(1 / math.sqrt(512)))
    cpool, raw, q, sel = _attn_case(91 + H, H, 4096, 700, 3000, 11)
    rpp, stride = 64, 64 * 1024 + 512
    n_pages = (3000 + rpp - 1) // rpp
    pt = synth.permutation(n_pages + 2, 91, 9)[:n_pages].copy()
    pool = np.zeros(((n_pages + 2) * stride) // 2, np.uint16)
    synth.scatter_pages(raw, rpp, pt, pool, stride)
    kc = csa.paged(dev(cpool, torch), 1, 1024, n_pages=4096)
    kr = csa.paged(dev(pool, torch), rpp, 1024, page_table=dev(pt, torch), page_stride_bytes=stride,
                   n_pages=n_pages + 2)
    ws_n = csa.csa_sparse_attn_workspace_size(H, 700, 128)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = torch.zeros((H, 512), dtype=torch.int16, device="cuda")
    lse = torch.zeros(H, dtype=torch.float32, device="cuda")
    csa.csa_sparse_attn(dev(q, torch), H, scale, kc, dev(sel, torch), 700, kr, 3000, 128, out, lse, ws, ws_n)
    _, f64, rlse = oracle.sparse_attn(q, scale, cpool, sel, raw, 128)
    assert_close(bf16_bits_to_f64(out.cpu().numpy().view(np.uint16)), f64, f"attn padded pages H={H}")
    assert np.abs(lse.cpu().numpy() - rlse).max() <= 1e-3 * max(1.0, np.abs(rlse).max())
    _status_clean(csa)


def test_attn_single_key_returns_its_row(csa):
    cpool, raw, q, _ = _attn_case(5, 16, 16, 0, 4)
    out, lse = _attn_gpu(csa, cpool, raw, q, np.array([7], np.int32), 0, 0.044)
    assert np.array_equal(out, np.repeat(cpool[7:8], 16, axis=0))


def test_attn_rescale_path_increasing_logits(csa):
    """Logits that rise by ~10 (log2 units) per 64-key tile: with 8192 keys each CTA owns several tiles,
    so the running max moves past the threshold inside a CTA and O is rescaled in TMEM.  Head 0's query
    is scaled up so the key rows (and the outputs) stay well inside O(1)."""
    H, G = 64, 8192
    q = synth.normal_bf16((H, 512), 8, 1)
    qf = bf16_bits_to_f64(q)
    qf[0] *= 256.0
    q[0] = np.asarray(np.asarray(qf[0], np.float32).view(np.uint32) >> 16, np.uint16)
    qf = bf16_bits_to_f64(q)
    cpool = synth.normal_bf16((G, 512), 8, 2)
    noise = bf16_bits_to_f64(cpool)
    unit = qf[0] / np.linalg.norm(qf[0])
    scale = float(np.float32(1 / math.sqrt(512)))
    # logit_j(head 0) ~ scale * |q0| * c * j with 64 * c * scale * |q0| * log2(e) = 10 per tile
    c = 10.0 / (64 * scale * np.linalg.norm(qf[0]) * 1.4426950408889634)
    for j in range(G):
        v = unit * (c * j) + noise[j] * 0.1
        cpool[j] = np.asarray(np.asarray(v, np.float32).view(np.uint32) >> 16, np.uint16)
    raw = synth.normal_bf16((128, 512), 8, 3)
    sel = np.arange(G, dtype=np.int32)
    out, lse = _attn_gpu(csa, cpool, raw, q, sel, 128, scale)
    _, f64, rlse = oracle.sparse_attn(q, scale, cpool, sel, raw, 128)
    assert np.abs(bf16_bits_to_f64(cpool)).max() < 1
    assert_close(bf16_bits_to_f64(out), f64, "attention with rising maxima")
    assert np.abs(lse - rlse).max() <= 1e-3 * max(1.0, np.abs(rlse).max())


# ------------------------------------------------------------------ device status (no fault)
def test_bad_page_id_sets_device_status_without_fault(csa):
    G = 64
    k = synth.normal_bf16((G, 128), 1, 1)
    pool = np.zeros((4 * 16, 128), np.uint16)
    pt = np.array([0, 1, 99, 2], np.int32)  # logical page 2 -> physical 99: outside the 4-page pool
    synth.scatter_pages(k[:32], 16, pt[:2], pool, 16 * 256)
    out = torch.zeros(G, device="cuda")
    csa.csa_index_score(dev(synth.normal_bf16((4, 128), 1, 2), torch), dev(np.ones(4, np.float32), torch), 4,
                        csa.paged(dev(pool, torch), 16, 256, page_table=dev(pt, torch), n_pages=4), csa.CSA_BF16, G,
                        out)
    torch.cuda.synchronize()
    st = csa.csa_read_device_status()
    assert st & (1 << (csa.CSA_ERR_DEVICE_BOUNDS - 1))
    assert csa.csa_read_device_status() == 0  # read clears it


def test_bounded_wait_runs_out_without_fault(csa):
    """A wait that nothing satisfies (an mbarrier no one arrives on) runs out after its bounded
    spin, sets CSA_ERR_TIMEOUT in the device status word and returns; the context stays usable
    (a score call afterwards is correct and leaves the status clean)."""
    csa.csa_read_device_status()
    csa.csa_selftest_bounded_wait()
    torch.cuda.synchronize()
    st = csa.csa_read_device_status()
    assert st & (1 << (csa.CSA_ERR_TIMEOUT - 1))
    assert csa.csa_read_device_status() == 0
    k = synth.normal_bf16((64, 128), 3, 1)
    q = synth.normal_bf16((4, 128), 3, 2)
    w = np.ones(4, np.float32)
    out = torch.zeros(64, device="cuda")
    csa.csa_index_score(dev(q, torch), dev(w, torch), 4, csa.paged(dev(k, torch), 64, 256, n_pages=1), csa.CSA_BF16,
                        64, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32),
                          oracle.index_score(q, w, k, False).view(np.uint32))
    _status_clean(csa)


def test_copy_batch_moves_every_byte(csa):
    """csa_copy_batch: pinned host -> device, device -> pinned host and device -> device copies of
    several sizes (one 16-byte chunk up to a few MB, an empty one), up to CSA_COPY_MAX in one
    launch, each destination byte-equal to its source and the bytes around it untouched."""
    import deepseek_v4_hybrid_c4_gb300 as m
    g = torch.Generator().manual_seed(11)
    sizes = [16, 4096, 137728, 131584, 0, (1 << 21) + 48, 1040, 16 * 1000]
    pairs, checks = [], []
    for i, n in enumerate(sizes):
        src_host = (i % 2) == 0
        words = max(n // 4, 1) + 8
        data = torch.randint(-2**31, 2**31 - 1, (words,), generator=g, dtype=torch.int32)
        src = data.pin_memory() if src_host else data.cuda()
        dst_host = i % 3 == 1
        fill = torch.full((words,), 0x5A5A5A5A, dtype=torch.int32)
        dst = fill.pin_memory() if dst_host else fill.cuda()
        pairs.append((src, dst, n))
        checks.append((data, dst, n, words))
    while len(pairs) < m.CSA_COPY_MAX:  # device -> device to fill the batch
        n = 16 * (len(pairs) + 1)
        data = torch.randint(-2**31, 2**31 - 1, (n // 4 + 8,), generator=g, dtype=torch.int32)
        dst = torch.full((n // 4 + 8,), 0x5A5A5A5A, dtype=torch.int32).cuda()
        pairs.append((data.cuda(), dst, n))
        checks.append((data, dst, n, n // 4 + 8))
    m.csa_copy_batch(m.copy_batch_args(pairs))
    torch.cuda.synchronize()
    assert m.csa_read_device_status() == 0
    for data, dst, n, words in checks:
        got = dst.cpu()
        assert torch.equal(got[: n // 4], data[: n // 4]), n
        assert (got[n // 4:] == 0x5A5A5A5A).all(), n
