"""The context-parallel split of one request on one GPU: R contiguous shards of the
candidates run every stage through the C ABI (csa_index_score, csa_topk with keys,
csa_topk_merge, csa_sparse_attn_partial, csa_attn_merge), the exchanges being
concatenations in rank order.  The global selection must equal the single-request oracle's
top k bit for bit and in order; the output is held to the oracle's fp64 result within the
bf16 tolerance."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def csa():
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v4_hybrid_c4_gb300 as m
    m.csa_read_device_status()
    return m


def _shards(csa, cp, case, r, R, kidx, cpool, raw):
    G = r.n_tokens // case.ratio
    ranges = cp.contiguous_ranges(G, R)
    rank_lo = torch.tensor(ranges, dtype=torch.int64, device="cuda")
    rb = 256 if case.kdtype == "bf16" else 128
    shards = []
    for rank in range(R):
        lo, hi = ranges[rank], ranges[rank + 1]
        n = max(1, (hi - lo + 15) // 16)
        kp = csa.paged(kidx[lo:hi] if hi > lo else kidx, 16, rb, n_pages=n)
        cp_ = csa.paged(cpool[lo:hi] if hi > lo else cpool, 16, 1024, n_pages=n)
        rawp = csa.paged(raw, 64, 1024, n_pages=(r.n_tokens + 63) // 64) if rank == R - 1 else None
        shards.append(cp.CPShard(rank=rank, world=R, rank_lo=rank_lo, lo=lo, hi=hi, kidx=kp, kv_c=cp_, kv_raw=rawp,
                                 n_tokens=r.n_tokens, H=case.H, Hi=case.Hi, k=case.k, swa=case.swa,
                                 scale=case.scale,
                                 kdtype=csa.CSA_BF16 if case.kdtype == "bf16" else csa.CSA_FP8_E4M3))
    return shards


@pytest.mark.parametrize("n_tokens,R", [(65536, 2), (65536, 4), (16384, 3), (1048576, 4)])
def test_context_parallel_split_matches_single_request(csa, n_tokens, R):
    from deepseek_v4_hybrid_c4_gb300 import cp
    case = synth.make_decode_case("cp", 2, [n_tokens], H=128, Hi=8, paged=False, n_pending=0)
    r = case.requests[0]
    ref = oracle.decode_request(r, ratio=4, w_gate=case.w_gate, b_pos=case.b_pos, k=case.k, swa=case.swa,
                                scale=case.scale)
    kidx, cpool, raw = dev(r.kidx, torch), dev(r.cpool, torch), dev(r.raw, torch)
    shards = _shards(csa, cp, case, r, R, kidx, cpool, raw)
    out = torch.empty((case.H, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty(case.H, dtype=torch.float32, device="cuda")
    sel = cp.run_local(shards, dev(r.q, torch), dev(r.q_idx, torch), dev(r.w_h, torch), cp.LibcsaBackend(), out, lse)
    torch.cuda.synchronize()
    assert csa.csa_read_device_status() == 0
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])  # the global top k, by (score desc, index asc)
    got = out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    assert_close(got.view(np.float32).astype(np.float64), ref["out_f64"], f"CP R={R} output")
    assert np.abs(lse.cpu().numpy() - ref["lse"]).max() <= 1e-3 * max(1.0, np.abs(ref["lse"]).max())


def test_topk_merge_ties_across_ranks_and_padding(csa):
    """Local top-k lists with equal keys in different ranks and ranks shorter than k."""
    from test_gpu_1_stages import _scores_with_ties
    rng = np.random.default_rng(3)
    s = _scores_with_ties(9000, 77)
    s[rng.integers(0, 9000, 800)] = np.float32(4.0)  # a tie group spread over every rank
    ranges = [0, 100, 4096, 4200, 9000]              # ranks of 100 and 104 candidates hold fewer than k
    R, k = 4, 512
    keys = torch.empty((R, k), dtype=torch.int32, device="cuda")
    idx = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sd = torch.from_numpy(s).cuda()
    for q in range(R):
        lo, hi = ranges[q], ranges[q + 1]
        csa.csa_topk(sd[lo:hi], hi - lo, k, idx[q], keys[q])
    rank_lo = torch.tensor(ranges, dtype=torch.int64, device="cuda")
    glob = torch.empty(k, dtype=torch.int32, device="cuda")
    gk = torch.empty(k, dtype=torch.int32, device="cuda")
    loc = torch.empty(k, dtype=torch.int32, device="cuda")
    csa.csa_topk_merge(keys, idx, rank_lo, R, k, 2, loc, glob, gk)
    ref, rkeys = oracle.topk(s, k, want_keys=True)
    g = glob.cpu().numpy()
    assert np.array_equal(g, ref)
    assert np.array_equal(gk.cpu().numpy().view(np.uint32), rkeys)
    mine = np.where((g >= 4096) & (g < 4200), g - 4096, -1)
    assert np.array_equal(loc.cpu().numpy(), mine)
    assert csa.csa_read_device_status() == 0


def test_attn_partial_empty_share_and_merge(csa):
    """A share with no selected rows and no window contributes nothing to the merge."""
    H = 64
    case = synth.make_decode_case("cp-empty", 5, [8192], H=H, Hi=8, paged=False, n_pending=0)
    r = case.requests[0]
    q = dev(r.q, torch)
    cpool = dev(r.cpool, torch)
    cpd = csa.paged(cpool, 16, 1024, n_pages=cpool.shape[0] // 16)
    raw = csa.paged(dev(r.raw, torch), 64, 1024, n_pages=r.n_tokens // 64)
    o = torch.full((2, H, 512), 7.0, dtype=torch.float32, device="cuda")
    l = torch.zeros((2, H), dtype=torch.float32, device="cuda")
    empty = torch.full((64,), -1, dtype=torch.int32, device="cuda")
    csa.csa_sparse_attn_partial(q, H, case.scale, cpd, empty, 64, raw, r.n_tokens, 0, o[0], l[0])
    sel = torch.arange(0, 2048, 7, dtype=torch.int32, device="cuda")[:64]
    csa.csa_sparse_attn_partial(q, H, case.scale, cpd, sel, 64, raw, r.n_tokens, 128, o[1], l[1])
    torch.cuda.synchronize()
    assert torch.all(o[0] == 0) and torch.all(torch.isinf(l[0])) and torch.all(l[0] < 0)
    out = torch.empty((H, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty(H, dtype=torch.float32, device="cuda")
    csa.csa_attn_merge(o, l, 2, H, out, lse)
    rows = np.concatenate([r.cpool[sel.cpu().numpy()], r.raw[r.n_tokens - 128:]])
    _, f64, rl = oracle.attention(r.q, case.scale, rows)
    got = out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    assert_close(got.view(np.float32).astype(np.float64), f64, "merge of an empty and a full share")
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max())
    assert np.abs(l[1].cpu().numpy() - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max())
    assert csa.csa_read_device_status() == 0
