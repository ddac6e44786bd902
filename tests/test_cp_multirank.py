"""The context-parallel split of one request (deepseek_v4_hybrid_c4_gb300.cp) across processes:
world size 2 over gloo at 127.0.0.1, on the CPU.

Each rank holds a contiguous half of the request's candidates; cp_decode_step runs the step
with the real exchange (torch.distributed all-gathers) and a CPU stand-in for the per-rank
stages built on the oracle (index score, sorted top k with keys, attention over the rank's
rows).  The stand-in restates on the host what the CUDA stages compute, so the test checks
the split's logic and exchange: both ranks must end with the single-request oracle's selection
(bit-exact, in order) and output (within 1e-5: both sides are the oracle's fp64 attention, the
partials passing through fp32 once)."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _key_to_score(keys_u32: np.ndarray) -> np.ndarray:
    k = keys_u32.astype(np.uint32)
    bits = np.where(k & 0x80000000, k ^ 0x80000000, ~k).astype(np.uint32)
    return bits.view(np.float32)


class OracleBackend:
    """Host restatement of the per-rank stages (tests only)."""

    def local_topk(self, sh, q_idx, w_h, stream=None):
        import torch
        import oracle
        G = sh.hi - sh.lo
        scores = oracle.index_score(q_idx, w_h, sh.kidx, False) if G else np.zeros(0, np.float32)
        idx, keys = oracle.topk(scores, sh.k, want_keys=True)
        return torch.from_numpy(keys.view(np.int32).copy()), torch.from_numpy(idx.copy())

    def global_select(self, sh, keys_all, idx_all, stream=None):
        import torch
        import oracle
        keys = keys_all.numpy().view(np.uint32)
        idx = idx_all.numpy()
        pos = oracle.topk(_key_to_score(keys), sh.k)
        ranges = sh.rank_lo.numpy()
        glob = np.full(sh.k, -1, np.int32)
        for i, p in enumerate(pos):
            if p >= 0 and idx[p] >= 0:
                glob[i] = ranges[p // sh.k] + idx[p]
        local = np.where((glob >= sh.lo) & (glob < sh.hi), glob - sh.lo, -1).astype(np.int32)
        self.local = local
        return torch.from_numpy(local), torch.from_numpy(glob)

    def attn_partial(self, sh, q, stream=None):
        import torch
        import oracle
        rows = [sh.kv_c[i] for i in self.local if i >= 0]
        if sh.kv_raw is not None:
            W = min(sh.swa, sh.n_tokens)
            rows += list(sh.kv_raw[sh.n_tokens - W: sh.n_tokens])
        if not rows:
            return torch.zeros((sh.H, 512), dtype=torch.float32), torch.full((sh.H,), -np.inf, dtype=torch.float32)
        _, f64, lse = oracle.attention(q, sh.scale, np.stack(rows))
        return torch.from_numpy(f64.astype(np.float32)), torch.from_numpy(lse.astype(np.float32))

    def merge(self, o_all, lse_all, R, H, out, lse, stream=None):
        o = o_all.numpy().astype(np.float64).reshape(R, H, 512)
        l = lse_all.numpy().astype(np.float64).reshape(R, H)
        M = l.max(axis=0)
        w = np.exp(l - M)
        L = w.sum(axis=0)
        out.copy_(__import__("torch").from_numpy((w[:, :, None] * o).sum(axis=0) / L[:, None]))
        lse.copy_(__import__("torch").from_numpy(M + np.log(L)))


def _worker(rank, world, port, q_out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist
    import synth
    from deepseek_v4_hybrid_c4_gb300 import cp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = synth.make_decode_case("cp-cpu", 11, [4096], H=16, Hi=4, k=64, paged=False, n_pending=0)
        r = case.requests[0]
        G = r.n_tokens // case.ratio
        ranges = cp.contiguous_ranges(G, world)
        lo, hi = ranges[rank], ranges[rank + 1]
        sh = cp.CPShard(rank=rank, world=world, rank_lo=torch.tensor(ranges, dtype=torch.int64), lo=lo, hi=hi,
                        kidx=r.kidx[lo:hi], kv_c=r.cpool[lo:hi], kv_raw=r.raw if rank == world - 1 else None,
                        n_tokens=r.n_tokens, H=case.H, Hi=case.Hi, k=case.k, swa=case.swa, scale=case.scale)
        out = torch.empty((case.H, 512), dtype=torch.float64)
        lse = torch.empty(case.H, dtype=torch.float64)
        sel = cp.cp_decode_step(sh, r.q, r.q_idx, r.w_h, OracleBackend(), cp.TorchDistExchange(dist), out, lse)
        q_out.put((rank, sel.numpy().copy(), out.numpy().copy(), lse.numpy().copy()))
    finally:
        dist.destroy_process_group()


def test_context_parallel_step_over_two_processes():
    import torch.multiprocessing as mp
    import oracle
    import synth
    from helpers import assert_close
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    case = synth.make_decode_case("cp-cpu", 11, [4096], H=16, Hi=4, k=64, paged=False, n_pending=0)
    r = case.requests[0]
    ref = oracle.decode_request(r, ratio=4, w_gate=case.w_gate, b_pos=case.b_pos, k=case.k, swa=case.swa,
                                scale=case.scale)
    for rank, sel, out, lse in got:
        assert np.array_equal(sel, ref["sel"]), rank      # the global top k, in order, on every rank
        assert_close(out, ref["out_f64"], f"rank {rank} output", max_abs=1e-5, rel_l2=1e-6)
        assert np.abs(lse - ref["lse"]).max() <= 1e-5 * max(1.0, np.abs(ref["lse"]).max())


def test_contiguous_ranges_cover_the_request():
    from deepseek_v4_hybrid_c4_gb300 import cp
    for G, world in [(1024, 2), (1000, 3), (262144, 4), (17, 4), (5, 8)]:
        rg = cp.contiguous_ranges(G, world)
        assert rg[0] == 0 and rg[-1] == G and len(rg) == world + 1
        assert all(a <= b for a, b in zip(rg, rg[1:]))
        assert all(x % 16 == 0 or x == G for x in rg)  # every shard starts on a 16-row page
