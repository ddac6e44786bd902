"""Benchmark of the C4 sparse-attention decode step (libcsa on GB300).

One step = the fused decode of one C4 layer at 1M context, bs = 1 (N = 1,048,576 raw
tokens -> 262,144 candidates -> top-512, plus SWA 128; 128 query heads, 8 index heads,
64-token pages under a random page-table permutation; one pending group compressed).
Prints one JSON line.  Inputs are synthetic (seeded generators) and resident in HBM
before timing.  The timed region is exactly K steps back to back between two CUDA events,
running the layers of a 6-layer stack in turn, each layer with its own copy of every buffer:
a step's ~68 MB of inputs were last touched five steps earlier and 340 MB of other layers'
traffic (> 129 MB L2) has evicted them -- data cold, code warm.  As a model captures its
decode loop, one CUDA graph holds the six layers' steps (K // 6 replays, then K mod 6
one-layer graphs), so a graph launch (about 4 us on the GPU) is paid once per six steps.
Two more timings go alongside: each one-layer graph alone between its own events
("value_step_alone"), and the same after an explicit L2 flush (a 256 MiB write, then a
256 MiB read of a second buffer; "value_l2_flushed").  An eager pass records CUDA events
between the stages for the per-stage breakdown and the roofline of the dominant kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the CPU oracle (the only reference this method has: the pages
ship no code) on the same workload.
Multi-GPU: one process per GPU (torchrun); requests are independent, so ranks run
replicas with no collective on the data path ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS = 6  # layers cycled by the timed steps
METRIC = "C4 sparse-attn decode µs/layer-step @1M ctx bs=1; HBM GB/s as % of GB300 peak"
WORKLOAD = "c4-decode-1M-bs1-paged (N=1048576, G=262144, k=512, SWA=128, H=128, Hi=8, 64-token pages)"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(case):
    """Bytes the step must move through HBM, summed over the batch's requests (scores, lists and
    partials stay in L2 and are not counted)."""
    kidx = pages = gather = q = out = comp = 0
    for r in case.requests:
        G = r.n_tokens // case.ratio
        if case.ratio == 4:  # index keys streamed, then k selected rows gathered
            kidx += G * 128 * (2 if case.kdtype == "bf16" else 1)
            gather += min(case.k, G) * 1024
        else:                # dense: every compressed row
            gather += G * 1024
        gather += min(case.swa, r.n_tokens) * 1024
        pages += (r.n_tokens + case.rows_per_page - 1) // case.rows_per_page * 4  # page table (int32)
        q += case.H * 512 * 2 + case.Hi * 128 * 2 + case.Hi * 4
        out += case.H * 512 * 2 + case.H * 4
        comp += (G - r.n_groups_done) * (case.ratio * 1024 + 1024)
    return dict(total=kidx + pages + gather + q + out + comp, score_kernel=kidx)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    def __init__(self, out_csv):
        self.out_csv = out_csv
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.out_csv, "w")
            dev = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
            sel = [f"--id={dev}"] if dev.isdigit() else []
            self.proc = subprocess.Popen(["nvidia-smi"] + sel + [f"--query-gpu={q}", "--format=csv,noheader",
                                                                 "-lms", "20"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [l.strip().split(",") for l in open(self.out_csv) if l.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1].split()[0]))
                mx = float(r[2].split()[0])
                for n, v in zip(names, r[5:9]):
                    if "Active" in v and "Not" not in v:
                        reasons.add(n)
            except Exception:
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_step_times(case, n_min, budget_s):
    """The oracle's decode step (single-threaded, as it stands), repeated."""
    import oracle
    oracle.build()
    r = case.requests[0]
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < n_min or (time.perf_counter() < t_end and len(times) < 50):
        t0 = time.perf_counter()
        oracle.decode_request(r, ratio=case.ratio, w_gate=case.w_gate, b_pos=case.b_pos, k=case.k, swa=case.swa,
                              scale=case.scale, kdtype=case.kdtype)
        times.append(time.perf_counter() - t0)
    return times


def oracle_stage_times(case, reps=3):
    """The oracle's stages on the workload's request, each timed alone (median of `reps`):
    compress the pending groups, score every candidate, select by full sort and by selection
    (partition to rank k, then sort the k), attend the selected rows plus the window."""
    import numpy as np
    import oracle
    oracle.build()
    r = case.requests[0]
    G = r.n_tokens // case.ratio
    fp8 = case.kdtype == "fp8"

    def med(fn):
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            v = fn()
            ts.append(time.perf_counter() - t0)
        return statistics.median(ts) * 1e6, v

    t_comp, _ = med(lambda: oracle.compress(r.raw, case.ratio, case.w_gate, case.b_pos, r.n_groups_done,
                                            G - r.n_groups_done))
    t_score, scores = med(lambda: oracle.index_score(r.q_idx, r.w_h, r.kidx, fp8))
    t_sort, sel = med(lambda: oracle.topk(scores, case.k))
    t_nth, sel2 = med(lambda: oracle.topk_select(scores, case.k))
    assert np.array_equal(sel, sel2)
    rows = np.concatenate([r.cpool[sel[sel >= 0]], r.raw[r.n_tokens - min(case.swa, r.n_tokens):]])
    t_attn, _ = med(lambda: oracle.attention(r.q, case.scale, rows))
    return {"compress": round(t_comp, 1), "score": round(t_score, 1), "select_full_sort": round(t_sort, 1),
            "select_partition_then_sort": round(t_nth, 1), "attention": round(t_attn, 1)}


def run_reference(args, rank):
    """--impl reference: the CPU oracle on the host cores, rank 0 only."""
    if rank != 0:
        return
    import synth
    case = synth.config(2)
    times = oracle_step_times(case, args.warmup + args.steps, 0.0)[args.warmup:]
    us = statistics.mean(times) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "µs/layer-step",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 index score)",
            "data": "synthetic (seeded Philox4x32-10 generators)",
            "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": round(us, 1), "unit": "µs/layer-step", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} full decode steps of the 1M workload after {args.warmup} "
                                       f"untimed; host nproc={os.cpu_count()}"},
            "e2e": {"value": round(us, 1), "unit": "µs/layer-step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def other_workloads(torch, csa, entry, synth, stream, flush_l2, peak):
    """The other measured rows: the top-512 select alone over the 1M workload's 262,144 scores;
    the ragged fp8 batch and the C128 dense batch as decode steps; the prefill compressors
    (C128 over 8 x 524,288 tokens, C4 over 1,048,576) as bandwidth.  Each step or call is timed
    alone between CUDA events after an L2 flush (write then read).  The event timer advances in
    steps of about 2 us on these GPUs, so a median of single-call samples sits on that grid; the
    reported time is the mean of the middle 80% of the samples, which resolves below a step."""
    import numpy as np
    res = {}

    def timed(fn, n, flush=True):
        ts = []
        for _ in range(n):
            with torch.cuda.stream(stream):
                if flush:
                    flush_l2()
                else:  # keep the GPU busy (~50 us) while the host enqueues the events and the call
                    torch.cuda._sleep(100000)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        ts.sort()
        cut = len(ts) // 10
        mid = ts[cut:len(ts) - cut] or ts
        return statistics.fmean(mid), ts[int(0.9 * (len(ts) - 1))]

    def back_to_back(batch, n_layers=6, reps=20):
        """Per-step time of `batch`'s step with n_layers copies of its buffers stepped in turn in one
        CUDA graph, replayed back to back (the protocol of the headline value); the copies are
        freed again."""
        layers_ = [batch] + [batch.clone() for _ in range(n_layers - 1)]
        with torch.cuda.stream(stream):
            for lb in layers_:
                lb.run(stream)
        torch.cuda.synchronize()
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            for lb in layers_:
                lb.run(stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g_.replay()
            e1.record(stream)
        e1.synchronize()
        assert csa.csa_read_device_status(stream) == 0
        del g_, layers_
        torch.cuda.empty_cache()
        return e0.elapsed_time(e1) * 1e3 / (reps * n_layers)

    # ---- the select alone: csa_topk (sorted output) on the 1M workload's scores
    case2 = synth.config(2)
    b2 = entry.case_to_batch(case2)
    r2 = case2.requests[0]
    G2 = r2.n_tokens // case2.ratio
    c_rpp = case2.c_rows_per_page()
    kp = csa.paged(b2.kidx_pool, c_rpp, 256, page_table=b2.page_table[0], n_pages=case2.n_pages)
    scores = torch.empty(G2, dtype=torch.float32, device="cuda")
    idx = torch.empty(case2.k, dtype=torch.int32, device="cuda")
    ws_bytes = csa.csa_topk_workspace_size(1, G2, case2.k)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        csa.csa_index_score(b2.q_idx, b2.w_h, case2.Hi, kp, csa.CSA_BF16, G2, scores, stream.cuda_stream)
    torch.cuda.synchronize()
    topk = lambda: csa.csa_topk(scores, G2, case2.k, idx, None, ws, ws_bytes, stream.cuda_stream)
    # "alone": one call between two events, as one graph launch -- timed eagerly, the host's enqueue
    # of the call's kernels after the first event would be measured too (and hidden by the flush
    # when there is one, which made the flushed call look faster)
    topk()
    torch.cuda.synchronize()
    g_topk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_topk, stream=stream):
        topk()
    warm, warm90 = timed(g_topk.replay, 50, flush=False)
    cold, cold90 = timed(g_topk.replay, 50, flush=True)
    with torch.cuda.stream(stream):  # 200 calls back to back: per-call launch latency pipelined
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(200):
            topk()
        e1.record(stream)
    e1.synchronize()
    res["topk_262144_to_512"] = {"us_per_call_back_to_back": round(e0.elapsed_time(e1) * 1e3 / 200, 2),
                                 "us_alone_scores_in_l2": round(warm, 2), "us_p90_alone_scores_in_l2": round(warm90, 2),
                                 "us_alone_l2_flushed": round(cold, 2), "us_p90_alone_l2_flushed": round(cold90, 2),
                                 "output": "sorted by (score desc, index asc); four kernels per call (clear the "
                                           "histograms, first digit, scan, finish); alone = one graph launch "
                                           "between two events"}
    # the same select in its single-cluster form (csa_topk_cluster: every digit's histogram summed
    # across the cluster through distributed shared memory), same scores, same box
    idx_c = torch.empty(case2.k, dtype=torch.int32, device="cuda")
    topk_c = lambda: csa.csa_topk_cluster(scores, None, 1, G2, case2.k, idx_c, None, stream.cuda_stream)
    topk_c()
    torch.cuda.synchronize()
    g_topk_c = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_topk_c, stream=stream):
        topk_c()
    warm_c, warm90_c = timed(g_topk_c.replay, 50, flush=False)
    cold_c, cold90_c = timed(g_topk_c.replay, 50, flush=True)
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(200):
            topk_c()
        e1.record(stream)
    e1.synchronize()
    assert torch.equal(idx_c, idx)
    res["topk_262144_to_512_cluster_form"] = {
        "us_per_call_back_to_back": round(e0.elapsed_time(e1) * 1e3 / 200, 2),
        "us_alone_scores_in_l2": round(warm_c, 2), "us_p90_alone_scores_in_l2": round(warm90_c, 2),
        "us_alone_l2_flushed": round(cold_c, 2), "us_p90_alone_l2_flushed": round(cold90_c, 2),
        "output": "identical indices; one cluster of 16 CTAs, one kernel per call"}
    # ---- C4 prefill compressor over the 1M workload's raw pool
    rp = csa.paged(b2.raw_pool, case2.rows_per_page, 1024, page_table=b2.page_table[0], n_pages=case2.n_pages)
    cout = torch.empty((G2, 512), dtype=torch.int16, device="cuda")
    cp = csa.paged(cout, G2, 1024)
    comp4 = lambda: csa.csa_compress(rp, r2.n_tokens, 4, b2.w_gate, b2.b_pos, 0, G2, cp, stream.cuda_stream)
    t, t90 = timed(comp4, 10)
    by = r2.n_tokens * 1024 + G2 * 1024
    res["c4_prefill_compress_1M"] = {"us": round(t, 1), "GB_s": round(by / t / 1e3, 1),
                                     "frac_of_peak": round(by / t / 1e3 / peak, 4), "bytes": by}
    del b2, cout, scores
    torch.cuda.empty_cache()
    # ---- decode steps of the ragged fp8 batch and of the C128 dense batch
    for cfg, name in [(0, "tiny_4K_decode"), (1, "c4_128K_decode"), (3, "ragged32_fp8_decode"),
                      (4, "c128_dense_bs8_decode")]:
        case = synth.config(cfg)
        b = entry.case_to_batch(case)
        with torch.cuda.stream(stream):
            for _ in range(3):
                b.run(stream)
        torch.cuda.synchronize()
        assert csa.csa_read_device_status(stream) == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            b.run(stream)
        t, t90 = timed(g.replay, 30)
        t_b2b = back_to_back(b)
        by = algorithmic_bytes(case)["total"]
        res[name] = {"us_per_step": round(t, 2), "us_p90": round(t90, 2),
                     "us_per_step_back_to_back": round(t_b2b, 2), "algorithmic_bytes": by,
                     "GB_s": round(by / t / 1e3, 1), "frac_of_peak": round(by / t / 1e3 / peak, 4),
                     "requests": len(case.requests)}
        if cfg == 4:  # ---- C128 prefill compressor over the same 8 x 524,288 tokens
            outs = [torch.empty((r.n_tokens // 128, 512), dtype=torch.int16, device="cuda") for r in case.requests]
            descs = [(csa.paged(b.raw_pool, case.rows_per_page, 1024, page_table=b.page_table[i], n_pages=case.n_pages),
                      csa.paged(o, o.shape[0], 1024), r.n_tokens) for i, (r, o) in enumerate(zip(case.requests, outs))]

            def comp128():
                for rp_, op_, n_ in descs:
                    csa.csa_compress(rp_, n_, 128, b.w_gate, b.b_pos, 0, n_ // 128, op_, stream.cuda_stream)
            t, t90 = timed(comp128, 10)
            by = sum(r.n_tokens * 1024 + (r.n_tokens // 128) * 1024 for r in case.requests)
            res["c128_prefill_compress_8x512K"] = {"us": round(t, 1), "GB_s": round(by / t / 1e3, 1),
                                                   "frac_of_peak": round(by / t / 1e3 / peak, 4), "bytes": by}
            del outs, descs
        del g, b
        torch.cuda.empty_cache()
    # ---- speculative verify at 1M context, bs = 1: n_q query positions (draft tokens) per step,
    #      each with its own candidates, top k and SWA window.  Two to four positions take one pass
    #      over the keys on the tensor cores (brackets, then the candidates they leave open
    #      rescored in the fixed order).
    case = synth.config(2)
    G = case.requests[0].n_tokens // case.ratio
    for nq in (2, 3, 4):
        b = entry.case_to_batch(case, n_q=nq, q=synth.normal_bf16((nq, case.H, 512), case.seed, 400),
                                q_idx=synth.normal_bf16((nq, case.Hi, 128), case.seed, 401),
                                w_h=synth.uniform_f32((nq, case.Hi), case.seed, 402))
        with torch.cuda.stream(stream):
            for _ in range(3):
                b.run(stream)
        torch.cuda.synchronize()
        assert csa.csa_read_device_status(stream) == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            b.run(stream)
        t, t90 = timed(g.replay, 30)
        t_b2b = back_to_back(b)
        one_pass = nq >= 2
        res[f"spec_verify_1M_{nq}_positions"] = {
            "us_per_step": round(t, 2), "us_p90": round(t90, 2), "us_per_step_back_to_back": round(t_b2b, 2),
            "us_per_query_position": round(t / nq, 2),
            "query_positions": nq, "index_key_bytes_per_step": (1 if one_pass else nq) * G * 256,
            "score": "one pass over the keys for every position: tcgen05 brackets, then exact rescoring of the "
                     "candidates they leave open" if one_pass else "the fixed-order kernel once per position"}
        del g, b
        torch.cuda.empty_cache()
    # ---- context-parallel split of the 1M request into 4 contiguous shards, on this one GPU: the
    #      stages of the rank holding the last shard (which also attends the window), with the
    #      exchanged lists and partials already in place, and the full 4-shard step run in turn
    from deepseek_v4_hybrid_c4_gb300 import cp as cpm
    case = synth.config(2)
    r = case.requests[0]
    G = r.n_tokens // case.ratio
    R = 4
    ranges = cpm.contiguous_ranges(G, R)
    rank_lo = torch.tensor(ranges, dtype=torch.int64, device="cuda")
    kidx_d = torch.from_numpy(np.ascontiguousarray(r.kidx).view(np.int16)).cuda()
    cpool_d = torch.from_numpy(np.ascontiguousarray(r.cpool).view(np.int16)).cuda()
    raw_d = torch.from_numpy(np.ascontiguousarray(r.raw).view(np.int16)).cuda()
    shards = []
    for q_ in range(R):
        lo, hi = ranges[q_], ranges[q_ + 1]
        shards.append(cpm.CPShard(
            rank=q_, world=R, rank_lo=rank_lo, lo=lo, hi=hi,
            kidx=csa.paged(kidx_d[lo:hi], 16, 256, n_pages=(hi - lo + 15) // 16),
            kv_c=csa.paged(cpool_d[lo:hi], 16, 1024, n_pages=(hi - lo + 15) // 16),
            kv_raw=csa.paged(raw_d, 64, 1024, n_pages=r.n_tokens // 64) if q_ == R - 1 else None,
            n_tokens=r.n_tokens, H=case.H, Hi=case.Hi, k=case.k, swa=case.swa, scale=case.scale))
    qd = torch.from_numpy(np.ascontiguousarray(r.q).view(np.int16)).cuda()
    qid = torch.from_numpy(np.ascontiguousarray(r.q_idx).view(np.int16)).cuda()
    whd = torch.from_numpy(r.w_h.astype(np.float32)).cuda()
    be = cpm.LibcsaBackend()
    out_d = torch.empty((case.H, 512), dtype=torch.int16, device="cuda")
    lse_d = torch.empty(case.H, dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        cpm.run_local(shards, qd, qid, whd, be, out_d, lse_d, stream.cuda_stream)
        lists = [be.local_topk(sh, qid, whd, stream.cuda_stream) for sh in shards]
        keys_all = torch.cat([k_ for k_, _ in lists])
        idx_all = torch.cat([i_ for _, i_ in lists])
        parts = [be.attn_partial(sh, qd, stream.cuda_stream) for sh in shards]
        o_all = torch.cat([o_ for o_, _ in parts])
        l_all = torch.cat([l_ for _, l_ in parts])
    torch.cuda.synchronize()
    last = shards[-1]

    def one_rank():  # the last rank's stages, the exchanged tensors in place
        be.local_topk(last, qid, whd, stream.cuda_stream)
        be.global_select(last, keys_all, idx_all, stream.cuda_stream)
        be.attn_partial(last, qd, stream.cuda_stream)
        be.merge(o_all, l_all, R, case.H, out_d, lse_d, stream.cuda_stream)

    g_rank, g_all = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()  # no host launch cost in the timing
    with torch.cuda.graph(g_rank, stream=stream):
        one_rank()
    with torch.cuda.graph(g_all, stream=stream):
        cpm.run_local(shards, qd, qid, whd, be, out_d, lse_d, stream.cuda_stream)
    t_rank, t_rank90 = timed(g_rank.replay, 30)
    t_all, _ = timed(g_all.replay, 10)
    assert csa.csa_read_device_status(stream) == 0
    res["cp_split_1M_4_shards_one_gpu"] = {
        "us_one_rank_stages": round(t_rank, 2), "us_p90_one_rank_stages": round(t_rank90, 2),
        "us_all_4_shards_in_turn": round(t_all, 2), "shards": R, "candidates_per_shard": ranges[1] - ranges[0],
        "note": "one GPU, CUDA graphs: a rank's own work (score and top-k of its shard, global merge, partial "
                "attention with the window, final merge) with the exchanged lists and partials in place, and the "
                "4 shards' stages in turn; the all-gathers between GPUs are not measured (one GPU per box)"}
    del g_rank, g_all, shards, kidx_d, cpool_d, raw_d, o_all, l_all, keys_all, idx_all, parts, lists
    torch.cuda.empty_cache()
    # ---- HiSparse at 1M context: the C4 pool (256 MiB) as a pinned host mirror with a GPU working
    #      set of a quarter of its pages.  Cold: every selected row comes from the mirror; warm:
    #      after the coordinator brought the step's pages in.
    case = synth.config(2)
    c_rpp = case.rows_per_page // case.ratio
    slots = case.n_pages // 4
    b = entry.case_to_batch(case, c_page_table=case.page_table(), c_rows_per_page=c_rpp, c_n_pages=case.n_pages,
                            hs_slots=slots)
    b.hs_step = 1
    with torch.cuda.stream(stream):
        for _ in range(3):
            b.run(stream)
    torch.cuda.synchronize()
    assert csa.csa_read_device_status(stream) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        b.run(stream)
    t_cold, _ = timed(g.replay, 30)
    t0 = time.perf_counter()
    n_in, n_ev = b.hs_update(stream)
    torch.cuda.synchronize()
    t_upd = (time.perf_counter() - t0) * 1e6
    t_warm, _ = timed(g.replay, 30)  # the graph reads the residency table, so it now hits
    assert csa.csa_read_device_status(stream) == 0
    # the asynchronous coordinator in a decode loop: after each step its stamps are collected and
    # the swap of the previous step's misses is applied (evictions on the decode stream, copies on a
    # side stream).  Two query sets alternate, so every step selects pages the previous one did not.
    # Each loop is host-driven (eager steps); the coordinator's cost is the loop's time per step
    # against the same loop without it.
    side = torch.cuda.Stream()
    n_tok = np.array([rq.n_tokens for rq in case.requests], np.int64)
    q_alt = [b.q.clone(), torch.from_numpy(synth.normal_bf16((1, case.H, 512), case.seed, 410).view(np.int16)).cuda()]
    qi_alt = [b.q_idx.clone(),
              torch.from_numpy(synth.normal_bf16((1, case.Hi, 128), case.seed, 411).view(np.int16)).cuda()]
    step_no = [10]

    def loop(T, coord):
        moved = 0
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for t in range(T):
                b.q.copy_(q_alt[t % 2])
                b.q_idx.copy_(qi_alt[t % 2])
                step_no[0] += 1
                b.hs_step = step_no[0]
                b.run(stream)
                if coord:
                    if t > 0:
                        moved += b.hs_apply(n_tok, stream, side)[0]
                    b.hs_collect(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / T, moved

    loop(6, True)
    t_plain, _ = loop(60, False)
    t_coord, moved = loop(60, True)
    assert csa.csa_read_device_status(stream) == 0
    res["hisparse_1M_quarter_working_set"] = {
        "us_per_step_cold": round(t_cold, 2), "us_per_step_warm": round(t_warm, 2),
        "us_update_host_wall": round(t_upd, 1), "pages_brought_in": int(n_in), "pages_evicted": int(n_ev),
        "working_set_pages": int(slots), "mirror_pages": int(case.n_pages), "page_bytes": c_rpp * 1024,
        "async_loop_us_per_step_with_coordinator": round(t_coord, 2),
        "async_loop_us_per_step_without": round(t_plain, 2),
        "async_coordinator_us_per_step": round(t_coord - t_plain, 2),
        "async_pages_moved_per_step": round(moved / 59, 1),
        "note": "cold: the 512 selected rows are read from pinned host memory over NVLink-C2C; async loop: "
                "eager (host-driven) steps alternating two query sets, collect after each step, apply after "
                "the next is enqueued"}
    del g, b
    torch.cuda.empty_cache()
    assert csa.csa_read_device_status(stream) == 0
    return res


def _attn_splits(case):
    """Key splits of the attention launch (a merge kernel follows when there are several)."""
    T = (case.k + case.swa + 63) // 64
    return max(1, min(T, 16, 76 // max(1, case.B)))


def _score_source_sha():
    p = os.path.join(ROOT, "deepseek_v4_hybrid_c4_gb300", "csrc", "score.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def rank_barrier(dist, sync=None):
    """Every rank's queued device work done (sync), then every rank here."""
    if sync:
        sync()
    if dist:
        dist.barrier()


def rank_max(dist, x: float, device="cuda") -> float:
    """The largest x over the ranks (a time: the job takes as long as its slowest rank)."""
    if not dist:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_step(ms_per_step_max: float, world: int) -> float:
    """Replicas: `world` ranks each run the timed steps, so the job does world x K layer-steps in
    the slowest rank's time; the line reports µs per layer-step of the whole job."""
    return ms_per_step_max * 1e3 / world


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the other measured rows (select alone, ragged and C128 batches, prefill compressors)")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layers cycled by the timed steps (1: a small run for profiler captures)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        return run_reference(args, rank)

    import torch
    import synth
    import __graft_entry__
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    __graft_entry__.build()
    import deepseek_v4_hybrid_c4_gb300 as csa

    case = synth.config(2)
    batch = __graft_entry__.case_to_batch(case, f"cuda:{local}")
    # LAYERS layers of the same shape, each with its own copy of every buffer; consecutive steps
    # run consecutive layers, so a step's inputs were last touched LAYERS - 1 steps earlier and
    # the LAYERS * ~68 MB read per round (> 129 MB L2) has evicted them by then
    n_layers = max(1, args.layers)
    layers = [batch] + [batch.clone() for _ in range(n_layers - 1)]
    stream = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")
    flush_sum = torch.empty((), dtype=torch.int64, device="cuda")

    def flush_l2():  # on the current stream, outside the timed region
        flush.zero_()
        torch.sum(flush_rd, dim=0, dtype=torch.int64, out=flush_sum)

    def barrier():
        rank_barrier(dist, torch.cuda.synchronize)

    def max_over_ranks(x):
        return rank_max(dist, x, "cuda")

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for lb in layers:
                lb.run(stream)
    barrier()
    assert csa.csa_read_device_status(stream) == 0

    # ---- the step as one CUDA graph per layer
    graphs = []
    for lb in layers:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            lb.run(stream)
        graphs.append(g)
    # and one graph over the whole stack, as a model captures its decode loop
    stack = torch.cuda.CUDAGraph()
    with torch.cuda.graph(stack, stream=stream):
        for lb in layers:
            lb.run(stream)

    def run_steps(K):  # exactly K layer-steps: K // n_layers stack replays, then single layers
        full, rem = divmod(K, n_layers)
        for _ in range(full):
            stack.replay()
        for i in range(rem):
            graphs[i].replay()

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup) * n_layers):
            graphs[i % n_layers].replay()
        for _ in range(max(3, args.warmup)):
            stack.replay()
    barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clk_path = os.path.join(tempfile.gettempdir(), f"bench_clocks_{os.getpid()}.csv")
    clocks = ClockSampler(clk_path)
    barrier()
    with clocks:
        # the timed region: exactly K steps back to back, as a model's layer loop runs them
        with torch.cuda.stream(stream):
            e_start.record(stream)
            run_steps(args.steps)
            e_end.record(stream)
        barrier()
        ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps)
        assert csa.csa_read_device_status(stream) == 0
        # each step alone between two events (its own launch latency inside)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                ev[i][0].record(stream)
                graphs[i % n_layers].replay()
                ev[i][1].record(stream)
        barrier()
        ms_alone = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev))
        # each step alone after an explicit flush of L2 (256 MiB write, then 256 MiB read of a
        # second buffer): data and code both cold
        evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_l2()
                evf[i][0].record(stream)
                graphs[i % n_layers].replay()
                evf[i][1].record(stream)
        barrier()
        ms_flushed = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evf))

    # ---- eager pass with events between the stages (breakdown + dominant-kernel roofline)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for row in sev:  # libcsa re-records these inside the step; torch only needs to know they exist
        for e in row:
            e.record(stream)
    barrier()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            layers[i % n_layers].run(stream, sev[i])
    barrier()
    stage_ms = [[sev[i][j].elapsed_time(sev[i][j + 1]) for i in range(args.steps)] for j in range(4)]
    eager_ms = statistics.mean(sev[i][0].elapsed_time(sev[i][4]) for i in range(args.steps))

    # ---- end to end through host buffers: the new token's state goes up, the output comes back.
    #      Per layer one CUDA graph holds the step with its copies: the packed per-step inputs
    #      (q | q_idx | w_h), the completed group's raw rows and its index row up from pinned
    #      host memory in one csa_copy_batch launch; the step writes its outputs (out, lse)
    #      straight into pinned host memory (the same bytes the device-side outputs hold).
    h_in = batch.step_in.cpu().pin_memory()
    h_out = torch.empty(batch.step_out.shape, dtype=batch.step_out.dtype).pin_memory()
    r0 = case.requests[0]
    G = r0.n_tokens // case.ratio
    t0 = r0.n_groups_done * case.ratio
    row0 = int(r0.pages[t0 // case.rows_per_page]) * case.rows_per_page + t0 % case.rows_per_page
    n_new = (G - r0.n_groups_done) * case.ratio  # the completed group's raw tokens (inside one page)
    hraw = batch.raw_pool[row0: row0 + n_new].cpu().pin_memory()
    c_rpp = case.c_rows_per_page()
    krow = int(r0.pages[(G - 1) // c_rpp]) * c_rpp + (G - 1) % c_rpp
    hkidx = batch.kidx_pool[krow: krow + 1].cpu().pin_memory()
    h2d = h_in.numel() + hraw.numel() * 2 + hkidx.numel() * hkidx.element_size()
    d2h = h_out.numel()
    e2e_graphs = []
    for lb in layers:
        g = torch.cuda.CUDAGraph()
        up = csa.copy_batch_args([(h_in, lb.step_in), (hraw, lb.raw_pool[row0: row0 + n_new]),
                                  (hkidx, lb.kidx_pool[krow: krow + 1])])
        ph = type(lb.params).from_buffer_copy(lb.params)  # the layer's step with host outputs
        ph.out = h_out.data_ptr() + (lb.out.data_ptr() - lb.step_out.data_ptr())
        ph.lse = h_out.data_ptr() + (lb.lse.data_ptr() - lb.step_out.data_ptr())
        with torch.cuda.graph(g, stream=stream):
            csa.csa_copy_batch(up, stream)
            csa.csa_decode(ph, lb.ws, lb.ws_bytes, stream)
        e2e_graphs.append((g, ph))
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup) * n_layers):
            e2e_graphs[i % n_layers][0].replay()
    barrier()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_graphs[i % n_layers][0].replay()
            e1.record(stream)
            e1.synchronize()  # the host holds the step's output before the next step goes up
            e2e_ms.append(e0.elapsed_time(e1))
    barrier()
    assert csa.csa_read_device_status(stream) == 0
    # the host copy is the step's output: the last layer's device-side output, recomputed
    # eagerly from the same inputs, holds the same bits
    lb = layers[(args.steps - 1) % n_layers]
    with torch.cuda.stream(stream):
        lb.run(stream)
    torch.cuda.synchronize()
    hb, db = h_out.view(torch.uint8), lb.step_out.cpu().view(torch.uint8)
    for t in (lb.out, lb.lse):
        o = t.data_ptr() - lb.step_out.data_ptr()
        n = t.numel() * t.element_size()
        assert torch.equal(hb[o: o + n], db[o: o + n]), "the step's host outputs differ from its device outputs"

    e2e = max_over_ranks(statistics.mean(e2e_ms))

    if rank != 0:
        dist.destroy_process_group()
        return
    peak, peak_kind = peaks()
    ab = algorithmic_bytes(case)
    score_ms = statistics.mean(stage_ms[1])
    achieved = ab["score_kernel"] / (score_ms * 1e-3) / 1e9
    step_gbs = ab["total"] / (ms * 1e-3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "score_kernel_traffic.json")
    if os.path.exists(tp):
        try:
            d = json.load(open(tp))
            if d.get("kernel_source_sha") == _score_source_sha():
                traffic = d.get("traffic_bytes_per_launch")
        except Exception:
            traffic = None
    line = {
        "metric": METRIC, "value": round(job_us_per_step(ms, world), 3), "unit": "µs/layer-step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate; fp32 fixed-order index score)",
        "data": "synthetic (seeded Philox4x32-10 generators; shapes of the 1M-context workload)",
        "config": {"workload": WORKLOAD, "l2": f"inputs larger than L2: {n_layers} layers with their own buffers, stepped in turn "
                               f"({n_layers} x {ab['total'] / 1e6:.0f} MB per round vs 129 MB L2; no flush)",
                   "launch": f"one CUDA graph over the {n_layers} layers' steps, replayed K // {n_layers} "
                             f"times, then K mod {n_layers} one-layer graphs; K steps back to back between "
                             "two events (value_step_alone: each one-layer graph between its own events; "
                             "value_l2_flushed: the same after an explicit L2 flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "value_step_alone": round(ms_alone * 1e3 / world, 3),
        "value_l2_flushed": round(ms_flushed * 1e3 / world, 3),
        "stages_us_eager": {n: round(statistics.mean(v) * 1e3, 3) for n, v in
                            zip(["compress", "score", "topk", "attn"], stage_ms)},
        "eager_step_us": round(eager_ms * 1e3, 3),
        "step_roofline": {"bound": "hbm", "algorithmic_bytes": ab["total"], "achieved": round(step_gbs, 1),
                          "peak": peak, "unit": "GB/s", "frac": round(step_gbs / peak, 4),
                          "peak_source": f"{peak_kind} (copy)"},
        "roofline": {"kernel": "score_kernel (stage 2, index score)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": ab["score_kernel"],
                     "peak_source": f"{peak_kind} (burst copy)"},
        "e2e": {"value": round(e2e * 1e3 / world, 3), "unit": "µs/layer-step", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": args.steps * (5 + (1 if _attn_splits(case) > 1 else 0)),  # compress, score, select scan + finish, attention (+ merge)
        "clocks": clocks.summary(),
    }
    if not args.no_other_workloads:
        del graphs, stack, e2e_graphs
        layers = layers[:1]
        torch.cuda.empty_cache()
        line["other_workloads"] = other_workloads(torch, csa, __graft_entry__, synth, stream, flush_l2, peak)
    if not args.no_cpu_baseline:
        times = oracle_step_times(case, 3, 15.0)
        line["cpu_baseline"] = {"value": round(statistics.median(times) * 1e6, 1), "unit": "µs/layer-step",
                                "cores": 1, "kind": "oracle",
                                "sample": f"{len(times)} full decode steps of the same 1M workload (median); "
                                          f"host nproc={os.cpu_count()}",
                                "stages_us": oracle_stage_times(case)}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
