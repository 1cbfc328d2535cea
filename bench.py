#!/usr/bin/env python
"""Benchmark of the speculative-decoding sampling round on one GB300.

One step = spec_round: the draft-side softmax + multinomial over every
draft row, keeping each row's normaliser (the pass of spec_draft_sample_lse),
then the softmax of every target row, accept test, first rejection and
residual or bonus draw with those normalisers (the pass of spec_verify_lse),
in one call, on the ragged adaptive-k batch (B = 512 sequences, k_b uniform
in 1..10, V = 128256, bf16 logits, T = 1).  Inputs are resident in HBM and
larger than L2 (no flush needed).  The same round as two calls (each pass
timed by itself) and the standalone spec_verify (which streams the draft
rows again) are timed on the same batch beside it.

metric: verified logit rows/s (R_t + R_d rows per step) and achieved HBM
GB/s of algorithmic bytes (every logit row once, plus one row-equivalent
per sampled sequence for the resample).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the batch (the
path shards by sequence with no collective: weak scaling); timing is the
max over ranks.  --impl reference times the fp64 CPU oracle on the host
cores (rank 0 only) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified logit rows/sec and achieved HBM GB/s (fraction of 8 TB/s), 1xGB300"
UNIT = "rows/s"
MAIN_CONFIG = 5
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=MAIN_CONFIG)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--extra-configs", default="3,4",
                    help="other workloads measured kernel-only (comma list, '' for none)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--tree", type=int, default=1, help="also time the tree verify workload (0: skip)")
    ap.add_argument("--vocab-shard", default="2,4,8",
                    help="rank counts of the vocab-sharded verify to time ('' to skip)")
    ap.add_argument("--k-sweep", default="1,2,3,4,5,6,7,8,9,10",
                    help="draft lengths k of the spec_round sweep (B=512, V=128256, bf16, T=1; '' to skip)")
    return ap.parse_args()


def line_config(w, world: int) -> dict:
    """The workload as both arms describe it on their JSON lines."""
    return {"workload": w.name, "B": w.B, "V": w.V, "k": "uniform 1..10 per sequence",
            "temperature": 1.0, "logits": w.dtype, "rows_target": w.rows_target, "rows_draft": w.rows_draft,
            "step": "one sampling round: the draft-side softmax + multinomial of every draft row, then the "
                    "verify-and-resample of every sequence (spec_round)",
            "l2": "inputs > L2 (no flush)", "parallelism": f"replicas x{world}"}


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "spec_round_traffic_B512_ragged_k1to10_V128256_bf16.txt")


# the sources of the kernels a verify call launches
VERIFY_SOURCES = ("spec_verify.cu", "device_utils.cuh", "verify_common.cuh", "host_common.h")


def strip_comments(src: str) -> str:
    """C++ source without its // and /* */ comments and without blank lines
    (string and character literals kept as they are), so that an edit of a
    comment leaves the code's hash alone."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = ("".join(out)).split("\n")
    return "\n".join(ln.rstrip() for ln in lines if ln.strip())


def kernel_source_hash() -> str:
    """sha256 over the code of spec_verify's kernels (file names and their
    sources without comments)."""
    import hashlib
    d = os.path.join(ROOT, "speculative_decoding_verification_61_gb300", "csrc")
    h = hashlib.sha256()
    for name in VERIFY_SOURCES:
        h.update(name.encode())
        with open(os.path.join(d, name), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per spec_round call from the committed ncu summary, if
    it was taken on this workload with the current kernel sources; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("workload") != workload or kv.get("csrc_sha256") != kernel_source_hash():
        return None
    return int(kv["traffic_bytes_per_call"])


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.enabled = enabled
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        if not self.enabled:
            return self
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.enabled or self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def to_device(w, torch, dev):
    import numpy as np

    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            x = x.view(torch.bfloat16)
        return x.to(dev)
    return dict(tl=t(w.target_logits), dl=t(w.draft_logits), ua=t(w.u_accept), ur=t(w.u_resample),
                ud=t(w.u_draft), T=t(w.temperature), ko=t(w.k_offsets))


def measure(w, steps, warmup, torch, sv, dev, sampler=None, barrier=None, mode="fused", keep_outputs=False):
    """Device-resident timing of one sampling round with CUDA events on the
    launching stream.  mode "round": spec_round (both passes in one call);
    "fused": spec_draft_sample_lse + spec_verify_lse (each row read once);
    "separate": spec_draft_sample + spec_verify.  Returns per-step and
    per-call times (ms; in round mode the draft slot is empty) and, with
    keep_outputs, the last step's draft tokens, tokens and counts (host)."""
    fused = mode == "fused"
    d = to_device(w, torch, dev)
    toks = torch.empty(w.rows_draft, dtype=torch.int32, device=dev)
    lse2 = torch.empty(max(w.rows_draft, 1), dtype=torch.float64, device=dev)
    out_t = torch.empty(w.rows_target, dtype=torch.int32, device=dev)
    out_n = torch.empty(w.B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def draft():
        if mode == "round":
            return
        if fused:
            sv.spec_draft_sample_lse(d["dl"], d["T"], d["ud"], d["ko"], out_draft_tokens=toks, out_draft_lse2=lse2)
        else:
            sv.spec_draft_sample(d["dl"], d["T"], d["ud"], d["ko"], out_draft_tokens=toks)

    def verify():
        if mode == "round":
            sv.spec_round(d["tl"], d["dl"], d["ud"], d["ua"], d["ur"], d["T"], d["ko"], out_draft_tokens=toks,
                          out_tokens=out_t, out_num_accepted=out_n)
        elif fused:
            sv.spec_verify_lse(d["tl"], d["dl"], lse2, toks, d["ua"], d["ur"], d["T"], d["ko"], out_tokens=out_t,
                               out_num_accepted=out_n)
        else:
            sv.spec_verify(d["tl"], d["dl"], toks, d["ua"], d["ur"], d["T"], d["ko"], out_tokens=out_t,
                           out_num_accepted=out_n)

    for _ in range(max(3, warmup)):
        draft()
        verify()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        t0.record(stream)
        if mode == "round":
            # one call per step: only the bracketing events
            for _ in range(steps):
                verify()
        else:
            for i in range(steps):
                e = ev[i]
                e[0].record(stream)
                draft()
                e[1].record(stream)
                verify()
                e[2].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    if barrier:
        barrier()
    total = t0.elapsed_time(t1)
    if mode == "round":
        draft, ver = [0.0], [total / steps]
    else:
        draft = [e[0].elapsed_time(e[1]) for e in ev]
        ver = [e[1].elapsed_time(e[2]) for e in ev]
    n_acc = out_n.float().mean().item()
    outs = (toks.cpu().numpy(), out_t.cpu().numpy(), out_n.cpu().numpy()) if keep_outputs else None
    del d
    return dict(step_ms=total / steps, draft_ms=statistics.mean(draft), verify_ms=statistics.mean(ver),
                verify_ms_median=statistics.median(ver), mean_accepted=n_acc, outputs=outs)


def back_to_back(w, reps, warmup, torch, sv, dev):
    """spec_verify, spec_verify_lse, spec_round and spec_draft_sample on one
    workload, each called reps times back to back on the stream (the draft
    tokens and normalisers from one draft pass), bracketed by one pair of
    CUDA events: calls chain by programmatic dependent launch as in a
    serving loop.  Inputs exceed L2 for the measured workloads.  ms per call."""
    d = to_device(w, torch, dev)
    toks = torch.empty(max(w.rows_draft, 1), dtype=torch.int32, device=dev)
    lse2 = torch.empty(max(w.rows_draft, 1), dtype=torch.float64, device=dev)
    out_t = torch.empty(w.rows_target, dtype=torch.int32, device=dev)
    out_n = torch.empty(w.B, dtype=torch.int32, device=dev)
    sv.spec_draft_sample_lse(d["dl"], d["T"], d["ud"], d["ko"], out_draft_tokens=toks, out_draft_lse2=lse2)
    toks2 = torch.empty_like(toks)
    calls = {
        "verify": lambda: sv.spec_verify(d["tl"], d["dl"], toks, d["ua"], d["ur"], d["T"], d["ko"],
                                         out_tokens=out_t, out_num_accepted=out_n),
        "verify_lse": lambda: sv.spec_verify_lse(d["tl"], d["dl"], lse2, toks, d["ua"], d["ur"], d["T"], d["ko"],
                                                 out_tokens=out_t, out_num_accepted=out_n),
        "round": lambda: sv.spec_round(d["tl"], d["dl"], d["ud"], d["ua"], d["ur"], d["T"], d["ko"],
                                       out_draft_tokens=toks2, out_tokens=out_t, out_num_accepted=out_n),
        "draft_sample": lambda: sv.spec_draft_sample(d["dl"], d["T"], d["ud"], d["ko"], out_draft_tokens=toks2),
    }
    stream = torch.cuda.current_stream()
    out = {}
    for name, fn in calls.items():
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / reps
    del d
    return out


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def measure_tree(torch, sv, dev, reps, warmup):
    """Tree verify on the tree workload (64 sequences, full 3/2/1 trees of 16
    nodes, V = 128256, bf16): tokens drawn once by spec_tree_draft_sample,
    then spec_tree_verify timed with CUDA events on the launching stream."""
    import numpy as np
    import workloads
    w = workloads.make_tree_config()

    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(torch.bfloat16) if a.dtype == np.uint16 else x).to(dev)
    d = {k: t(getattr(w, k)) for k in ("target_logits", "draft_logits", "node_offsets", "parent", "u_accept",
                                       "u_resample", "u_draft", "temperature")}
    args_draft = (d["draft_logits"], d["node_offsets"], d["parent"], d["temperature"], d["u_draft"])
    toks = sv.spec_tree_draft_sample(*args_draft)
    toks = torch.where(toks < 0, torch.zeros_like(toks), toks)
    out = (torch.empty(w.nodes, dtype=torch.int32, device=dev), torch.empty(w.B, dtype=torch.int32, device=dev),
           torch.empty(w.B, dtype=torch.int32, device=dev))
    draft_out = torch.empty(w.nodes, dtype=torch.int32, device=dev)

    def verify():
        sv.spec_tree_verify(d["target_logits"], d["draft_logits"], d["node_offsets"], d["parent"], toks,
                            d["u_accept"], d["u_resample"], d["temperature"], out_tokens=out[0],
                            out_num_accepted=out[1], out_last_node=out[2])

    def draft():
        sv.spec_tree_draft_sample(*args_draft, out_tokens=draft_out)
    stream = torch.cuda.current_stream()
    res = {}
    for name, fn in (("verify", verify), ("draft", draft)):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
    nbytes = workloads.tree_algorithmic_bytes(w)
    internal = int(w.internal().sum())
    draft_bytes = w.elem_bytes * w.V * internal
    gbs = nbytes / (res["verify"] * 1e-3) / 1e9
    return {"workload": w.name, "B": w.B, "nodes": w.nodes, "verify_ms": round(res["verify"], 5),
            "verify_gbs": gbs, "verify_frac_of_8tbs": gbs / 8000.0, "verify_bytes": nbytes,
            "nodes_per_s": w.nodes / (res["verify"] * 1e-3),
            "mean_accepted": out[1].float().mean().item(),
            "draft_sample_ms": round(res["draft"], 5),
            "draft_sample_gbs": draft_bytes / (res["draft"] * 1e-3) / 1e9,
            "calls": "spec_tree_verify (setup + stats_kernel tree mode + tree_walk_kernel); "
                     "spec_tree_draft_sample (setup + stats_kernel tree-draft mode + tree_draft_select_kernel)"}


def measure_vocab_shard(torch, sv, dev, reps, warmup, Gs):
    """One rank's share of the vocab-sharded verify on the 512-sequence ragged
    workload (V = 128256, bf16, T = 1) with the vocabulary split over G
    ranks.  The G ranks are emulated on this GPU: every rank's columns are
    cut out once, the gathered records and masses (the inputs of decide and
    draw) come from one untimed pass over all ranks, then each rank's three
    calls (spec_shard_stats, spec_shard_decide, spec_shard_draw) are timed
    with CUDA events, the ranks interleaved so that a rank's columns leave
    L2 before its next run.  On G GPUs the ranks run in parallel: the
    slowest rank's time is the step's, plus two all-gathers and one
    all-reduce that are not measured here."""
    import workloads
    from speculative_decoding_verification_61_gb300.vocab_shard import VocabShardVerifier, even_bounds
    w = workloads.make_config(5)
    d = to_device(w, torch, dev)
    toks = sv.spec_draft_sample(d["dl"], d["T"], d["ud"], d["ko"])
    ab = workloads.algorithmic_bytes(w)
    stream = torch.cuda.current_stream()
    out = {}
    for G in Gs:
        bounds = even_bounds(w.V, G)
        vs = [VocabShardVerifier(bounds, r, w.B, sv.BF16, dev) for r in range(G)]
        cols = [(d["tl"][:, a:b].contiguous(), d["dl"][:, a:b].contiguous()) for a, b in zip(bounds, bounds[1:])]
        recs = torch.stack([v.stats(t, q, toks, d["T"], d["ko"]) for v, (t, q) in zip(vs, cols)])
        outs = [v.decide(recs, d["ua"]) for v in vs]
        mass = torch.stack([o[2] for o in outs])
        tok_out = [o[0] for o in outs]

        def rank_call(r):
            v, (t, q) = vs[r], cols[r]
            v.stats(t, q, toks, d["T"], d["ko"])
            v.decide(recs, d["ua"])
            v.draw(mass, d["ur"], tok_out[r])
        for _ in range(max(3, warmup)):
            for r in range(G):
                rank_call(r)
        torch.cuda.synchronize()
        # each rank's calls as one CUDA graph (what a serving loop replays),
        # and issued one by one from Python (host-bound at small widths)
        graphs = []
        for r in range(G):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                rank_call(r)
            graphs.append(g)
        torch.cuda.synchronize()

        def timed(run):
            ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(G)]
                  for _ in range(reps)]
            for i in range(reps):
                for r in range(G):
                    ev[i][r][0].record(stream)
                    run(r)
                    ev[i][r][1].record(stream)
            torch.cuda.synchronize()
            return [statistics.mean(ev[i][r][0].elapsed_time(ev[i][r][1]) for i in range(reps)) for r in range(G)]
        per_rank_eager = timed(rank_call)
        for _ in range(3):
            for r in range(G):
                graphs[r].replay()
        per_rank = timed(lambda r: graphs[r].replay())
        worst = max(per_rank)
        Vs_max = max(b - a for a, b in zip(bounds, bounds[1:]))
        rows_rec = w.rows_target + w.rows_draft
        # the rank's columns of every needed row once, one row-equivalent of
        # them per sampled sequence for the draw, its records out and all
        # ranks' records in
        rank_bytes = (w.elem_bytes * Vs_max * (ab["rows_needed"] + ab["sampled_sequences"]) +
                      16 * rows_rec * (1 + G) + 16 * w.B * (1 + G))
        gbs = rank_bytes / (worst * 1e-3) / 1e9
        out[str(G)] = {"ranks": G, "columns_per_rank": Vs_max, "rank_ms_max": round(worst, 5),
                       "rank_ms_mean": round(statistics.mean(per_rank), 5),
                       "rank_ms_max_eager": round(max(per_rank_eager), 5), "rank_bytes": int(rank_bytes),
                       "rank_gbs": gbs, "rank_frac_of_8tbs": gbs / 8000.0,
                       "rows_per_s_without_exchanges": rows_rec / (worst * 1e-3)}
        del vs, cols, recs, outs, mass, tok_out, graphs
    del d
    return {"workload": w.name, "by_ranks": out,
            "calls": "per rank, replayed as one CUDA graph (rank_ms_*; issued from Python: rank_ms_max_eager): "
                     "spec_shard_stats (stats_kernel shard mode + shard_row_kernel), "
                     "spec_shard_decide (shard_decide_kernel), spec_shard_draw (shard_draw_kernel); exchanges not timed"}


def k_sweep(torch, sv, dev, ks, reps, warmup, peak):
    """spec_round on B = 512 sequences that all draft k tokens, V = 128256,
    bf16, T = 1, for each k in ks ("【大模型】- 推测解码", optimize_parameters:
    the draft length tried over 1..10).  One seeded batch with k = max(ks)
    is generated; the batch for a smaller k keeps each sequence's first k
    drafted positions and its target row at position k (the bonus row after
    k acceptances), with their uniforms, cut out on the device.  Per k: the
    round's time, rows/s, algorithmic GB/s and its fraction of the measured
    copy peak, the mean accepted count and the emitted tokens per second
    (B * (n + 1) per round); best_k maximises the latter for this step."""
    import numpy as np
    import workloads
    kmax, B, V = max(ks), 512, 128256
    w = workloads.make_case(B=B, k=kmax, V=V, dtype=workloads.BF16, temperature=1.0, a=1.1, sigma_t=1.0,
                            sigma_d=0.5, seed=1105, name=f"B{B}_k{kmax}_V{V}_bf16_T1")
    d = to_device(w, torch, dev)
    stream = torch.cuda.current_stream()
    out = {}
    for k in ks:
        bb = torch.arange(B, device=dev)
        t_idx = (bb[:, None] * (kmax + 1) + torch.arange(k + 1, device=dev)[None, :]).reshape(-1)
        d_idx = (bb[:, None] * kmax + torch.arange(k, device=dev)[None, :]).reshape(-1)
        tl, dl = d["tl"].index_select(0, t_idx), d["dl"].index_select(0, d_idx)
        ua, ud, ur = d["ua"][d_idx], d["ud"][d_idx], d["ur"][t_idx]
        ko = (torch.arange(B + 1, device=dev, dtype=torch.int32) * k).contiguous()
        toks = torch.empty(B * k, dtype=torch.int32, device=dev)
        out_t = torch.empty(B * (k + 1), dtype=torch.int32, device=dev)
        out_n = torch.empty(B, dtype=torch.int32, device=dev)

        def call():
            sv.spec_round(tl, dl, ud, ua, ur, d["T"], ko, out_draft_tokens=toks, out_tokens=out_t,
                          out_num_accepted=out_n)
        for _ in range(max(3, warmup)):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        sub = workloads.Workload(name=f"k{k}", B=B, V=V, dtype=w.dtype, k_offsets=np.arange(B + 1, dtype=np.int32) * k,
                                 temperature=w.temperature, target_logits=None, draft_logits=None,
                                 u_accept=None, u_resample=None, u_draft=None)
        ab = workloads.algorithmic_bytes(sub)
        nbytes = ab["verify_lse"] + ab["draft_sample"]
        gbs = nbytes / (ms * 1e-3) / 1e9
        n_acc = out_n.float().mean().item()
        out[str(k)] = {"k": k, "round_ms": round(ms, 5), "rows_per_s": (B * (2 * k + 1)) / (ms * 1e-3),
                       "gbs": gbs, "frac_of_peak": gbs / peak, "bytes": nbytes, "mean_accepted": n_acc,
                       "acceptance_per_draft": n_acc / k, "emitted_tokens_per_s": B * (n_acc + 1) / (ms * 1e-3)}
        del tl, dl, ua, ud, ur, toks, out_t, out_n
    del d
    best = max(out.values(), key=lambda r: r["emitted_tokens_per_s"])["k"]
    return {"workload": f"B{B}, every sequence k drafted tokens, V={V}, bf16, T=1 (sigma_t 1, sigma_d 0.5, "
                        f"seed 1105; batches cut from one k={kmax} batch)",
            "step": "spec_round", "reps_per_k": reps, "by_k": out, "best_k_by_emitted_tokens_per_s": best}


def adaptive_k_timing(torch, sv, dev, B=4096, reps=1000):
    """Device time of one adaptive-k update (spec_adapt_update) for B
    sequences, the round-to-round step of a serving loop."""
    import numpy as np
    ctl = sv.AdaptiveK(B, 1, 10, device=dev)
    rng = np.random.default_rng(7)
    counts = [torch.from_numpy(rng.integers(0, 6, size=B).astype(np.int32)).to(dev) for _ in range(8)]
    for i in range(20):
        ctl.update(counts[i % 8])
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        ctl.update(counts[i % 8])
    e1.record(stream)
    torch.cuda.synchronize()
    return {"B": B, "update_us": 1000.0 * e0.elapsed_time(e1) / reps, "launches_per_update": 1,
            "kernel": "update_kernel (one block; history update, exact mean test, k_offsets scan)"}


def e2e(w, steps, torch, sv):
    """Through the public host-buffer entry point: H2D of the step's inputs
    from pinned memory, draft sample + verify, D2H of the results."""
    import numpy as np

    def h(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(torch.bfloat16) if a.dtype == np.uint16 else x).pin_memory()
    hs = dict(tl=h(w.target_logits), dl=h(w.draft_logits), ud=h(w.u_draft), ua=h(w.u_accept),
              ur=h(w.u_resample), T=h(w.temperature), ko=h(w.k_offsets))
    outs = (torch.empty(w.rows_draft, dtype=torch.int32).pin_memory(),
            torch.empty(w.rows_target, dtype=torch.int32).pin_memory(),
            torch.empty(w.B, dtype=torch.int32).pin_memory())

    def call():
        sv.spec_round_host(hs["tl"], hs["dl"], hs["ud"], hs["ua"], hs["ur"], hs["T"], hs["ko"],
                           out_draft_tokens=outs[0], out_tokens=outs[1], out_num_accepted=outs[2])
    call()
    call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(v.numel() * v.element_size() for v in hs.values())
    d2h = sum(v.numel() * v.element_size() for v in outs)
    return ms, h2d, d2h


class OracleSample:
    """The oracle as it stands, on host cores, on the first n sequences of
    the workload: draft sample + verify of that sub-batch is one step."""

    def __init__(self, w, nthreads, n):
        import workloads
        self.w, self.nthreads = w, nthreads
        self.n = n = int(min(w.B, max(1, n)))
        ko = w.k_offsets[:n + 1].copy()
        R_d, R_t = int(ko[-1]), int(ko[-1]) + n
        self.s = workloads.Workload(name=w.name, B=n, V=w.V, dtype=w.dtype, k_offsets=ko,
                                    temperature=w.temperature[:n].copy(),
                                    target_logits=w.target_logits[:R_t], draft_logits=w.draft_logits[:R_d],
                                    u_accept=w.u_accept[:R_d], u_resample=w.u_resample[:R_t],
                                    u_draft=w.u_draft[:R_d])
        self.rows = self.s.rows_target + self.s.rows_draft

    def step(self):
        import oracle
        s = self.s
        t = time.perf_counter()
        ds = oracle.draft_sample(s.draft_logits, s.temperature, s.u_draft, s.k_offsets, nthreads=self.nthreads)
        oracle.verify(s.target_logits, s.draft_logits, ds.tokens, s.u_accept, s.u_resample, s.temperature,
                      s.k_offsets, nthreads=self.nthreads)
        return time.perf_counter() - t

    @classmethod
    def sized(cls, w, nthreads, seconds):
        """A sample whose step takes about `seconds` (at least one sequence
        per thread)."""
        probe = cls(w, nthreads, max(nthreads, 4))
        t = probe.step()
        return cls(w, nthreads, max(probe.n, probe.n * seconds / max(t, 1e-3)))

    def describe(self, reps, t):
        how = "OpenMP over sequences" if self.nthreads > 1 else "one thread"
        return (f"first {self.n} of {self.w.B} sequences of {self.w.name} x{reps} ({self.rows * reps} rows), "
                f"draft sample + verify, fp64 C oracle, {how}, {t:.1f} s")


def _timed_sample(w, nthreads, seconds):
    smp = OracleSample.sized(w, nthreads, seconds)
    reps, t = 1, smp.step()
    while t * (reps + 1) / reps < seconds and reps < 64:
        t += smp.step()
        reps += 1
    return dict(value=smp.rows * reps / t, unit=UNIT, cores=nthreads, kind="oracle",
                sequences_per_s=smp.n * reps / t, sample=smp.describe(reps, t))


def cpu_baseline(w, seconds, nthreads):
    """The oracle on bounded samples of the workload: about `seconds` of CPU
    time with OpenMP over sequences on every host core, and a third of that
    on one thread."""
    line = _timed_sample(w, nthreads, seconds)
    line["single_thread"] = _timed_sample(w, 1, seconds / 3)
    return line


FLAG_MARGIN = 1e-5


def oracle_parity(w, gpu_outputs, nthreads):
    """The timed round's outputs for every sequence of the workload against
    the oracle (part of the CPU-baseline leg, outside every timed region):
    the draft tokens against the oracle's draft sampling, then the verify
    outputs against the oracle's verify on the same draft tokens.  Decisions
    whose oracle margin is <= 1e-5 are flagged: counted, and not required to
    match.  Returns the counts."""
    import numpy as np
    import oracle
    g_draft, g_tok, g_num = gpu_outputs
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets, nthreads=nthreads)
    dflag = ds.margin <= FLAG_MARGIN
    dsame = g_draft == ds.tokens
    ov = oracle.verify(w.target_logits, w.draft_logits, g_draft, w.u_accept, w.u_resample, w.temperature,
                       w.k_offsets, nthreads=nthreads)
    flagged = flagged_match = mismatches = 0
    for b in range(w.B):
        o, k = int(w.k_offsets[b]) + b, int(w.k_offsets[b + 1] - w.k_offsets[b])
        same = bool(g_num[b] == ov.num_accepted[b] and np.array_equal(g_tok[o:o + k + 1], ov.tokens[o:o + k + 1]))
        if ov.num_accepted[b] >= 0 and ov.margin[b] <= FLAG_MARGIN:
            flagged += 1
            flagged_match += int(same)
        elif not same:
            mismatches += 1
    return {"oracle": "fp64 C oracle (oracle/)", "flag_margin": FLAG_MARGIN, "sequences": int(w.B),
            "flagged_sequences": flagged, "flagged_match": flagged_match,
            "mismatched_sequences_outside_flags": mismatches,
            "draft_rows": int(w.rows_draft), "draft_flagged_rows": int(dflag.sum()),
            "draft_flagged_match": int((dflag & dsame).sum()),
            "draft_mismatched_rows_outside_flags": int((~dflag & ~dsame).sum())}


# ------------------------------------------------------------------ main
def run_reference(args):
    """The reference arm: the fp64 oracle timed on the host cores, rank 0
    only.  One step = draft sample + verify of a fixed sample of the
    workload, sized once so that the W + K steps take about two minutes in
    all (at least one sequence per thread)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import workloads
    w = workloads.make_config(args.config)
    nthreads = oracle.cores()
    per_step = min(args.cpu_seconds if args.cpu_seconds > 0 else 15.0, 120.0 / max(1, args.steps + args.warmup))
    smp = OracleSample.sized(w, nthreads, per_step)
    for _ in range(args.warmup):
        smp.step()
    times = [smp.step() for _ in range(args.steps)]
    v = smp.rows / statistics.median(times)
    rows_step = w.rows_target + w.rows_draft
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * rows_step / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Zipf-like logits)",
            "config": line_config(w, world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                             "sample": smp.describe(args.steps, sum(times)) + " (median step)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import workloads
    import speculative_decoding_verification_61_gb300 as sv

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))
        barrier = dist.barrier
    sv.lib()
    peak, peak_kind = peaks()

    w = workloads.make_config(args.config)
    ab = workloads.algorithmic_bytes(w)
    sampler = ClockSampler(local, enabled=(rank == 0 and not args.no_clocks))
    m = measure(w, args.steps, args.warmup, torch, sv, dev, sampler=sampler, barrier=barrier, mode="round",
                keep_outputs=(rank == 0))
    step_ms = m["step_ms"]
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([step_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    rows = w.rows_target + w.rows_draft
    value = world * rows / (step_ms * 1e-3)
    step_bytes = ab["verify_lse"] + ab["draft_sample"]
    gbs = lambda nbytes, ms: nbytes / (ms * 1e-3) / 1e9  # noqa: E731
    step_gbs = gbs(step_bytes, step_ms)

    # the same round as two calls (each pass timed by itself), and the
    # separate calls (spec_verify streams the draft rows again)
    reps = max(50, args.steps // 4)
    two = measure(w, reps, args.warmup, torch, sv, dev, mode="fused") if rank == 0 else None
    sep = measure(w, reps, args.warmup, torch, sv, dev, mode="separate") if rank == 0 else None

    extra = {}
    for c in [int(x) for x in args.extra_configs.split(",") if x.strip()] if rank == 0 else []:
        wc = workloads.make_config(c)
        abc = workloads.algorithmic_bytes(wc)
        reps = max(50, args.steps // 4)
        bb = back_to_back(wc, reps, args.warmup, torch, sv, dev)
        mc = measure(wc, reps, args.warmup, torch, sv, dev, mode="separate")
        extra[wc.name] = {
            "timing": "each call back to back (events around the loop); *_in_loop: events around every "
                      "call of a draft-then-verify loop, which stops the calls from chaining",
            "verify_ms": round(bb["verify"], 5), "draft_sample_ms": round(bb["draft_sample"], 5),
            "verify_rows_per_s": (wc.rows_target + wc.rows_draft) / (bb["verify"] * 1e-3),
            "verify_gbs": gbs(abc["verify"], bb["verify"]),
            "verify_frac_of_8tbs": gbs(abc["verify"], bb["verify"]) / 8000.0,
            "verify_bytes": abc["verify"], "mean_accepted": mc["mean_accepted"],
            "verify_ms_in_loop": round(mc["verify_ms"], 5),
            "verify_frac_of_8tbs_in_loop": gbs(abc["verify"], mc["verify_ms"]) / 8000.0,
            # (the mean above takes any host stall between two calls; the
            # median of the per-call times does not)
            "verify_ms_in_loop_median": round(mc["verify_ms_median"], 5),
            "verify_lse_ms": round(bb["verify_lse"], 5),
            "verify_lse_gbs": gbs(abc["verify_lse"], bb["verify_lse"]),
            "verify_lse_frac_of_8tbs": gbs(abc["verify_lse"], bb["verify_lse"]) / 8000.0,
            "round_ms": round(bb["round"], 5),
            "round_rows_per_s": (wc.rows_target + wc.rows_draft) / (bb["round"] * 1e-3),
            "round_gbs": gbs(abc["verify_lse"] + abc["draft_sample"], bb["round"]),
            "round_frac_of_8tbs": gbs(abc["verify_lse"] + abc["draft_sample"], bb["round"]) / 8000.0}
        del wc

    adapt = adaptive_k_timing(torch, sv, dev) if rank == 0 else None
    sweep_ks = [int(x) for x in args.k_sweep.split(",") if x.strip()]
    sweep = (k_sweep(torch, sv, dev, sweep_ks, max(50, args.steps // 10), args.warmup, peak)
             if rank == 0 and sweep_ks else None)
    tree = measure_tree(torch, sv, dev, max(50, args.steps // 4), args.warmup) if rank == 0 and args.tree else None
    shard_gs = [int(x) for x in args.vocab_shard.split(",") if x.strip()]
    vshard = (measure_vocab_shard(torch, sv, dev, max(20, args.steps // 20), args.warmup, shard_gs)
              if rank == 0 and shard_gs else None)

    e2e_line = None
    if rank == 0 and args.e2e_steps > 0:
        ms, h2d, d2h = e2e(w, args.e2e_steps, torch, sv)
        e2e_line = {"value": rows / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": args.e2e_steps,
                    "api": "spec_round_host (pinned host buffers)"}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    import oracle
    cpu = cpu_baseline(w, args.cpu_seconds, oracle.cores()) if args.cpu_seconds > 0 else None
    # the CPU-baseline leg also checks the timed round's outputs against the oracle
    parity = oracle_parity(w, m["outputs"], oracle.cores()) if args.cpu_seconds > 0 else None
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Zipf-like logits + Gaussian noise)",
        "config": line_config(w, world),
        "hbm_gbs": step_bytes / (step_ms * 1e-3) / 1e9,
        "frac_of_8tbs": step_bytes / (step_ms * 1e-3) / 8e12,
        "bytes_per_step": step_bytes,
        "kernels": {"mean_accepted": m["mean_accepted"],
                    "two_calls": None if two is None else {
                        "step": "spec_draft_sample_lse + spec_verify_lse",
                        "step_ms": two["step_ms"], "rows_per_s": rows / (two["step_ms"] * 1e-3),
                        "spec_verify_lse_ms": two["verify_ms"],
                        "spec_verify_lse_gbs": gbs(ab["verify_lse"], two["verify_ms"]),
                        "spec_verify_lse_frac_of_peak": gbs(ab["verify_lse"], two["verify_ms"]) / peak,
                        "spec_draft_sample_lse_ms": two["draft_ms"],
                        "spec_draft_sample_lse_gbs": gbs(ab["draft_sample"], two["draft_ms"])},
                    "separate_calls": None if sep is None else {
                        "step_ms": sep["step_ms"],
                        "rows_per_s": rows / (sep["step_ms"] * 1e-3),
                        "spec_verify_ms": sep["verify_ms"],
                        "spec_verify_gbs": gbs(ab["verify"], sep["verify_ms"]),
                        "spec_verify_frac_of_8tbs": gbs(ab["verify"], sep["verify_ms"]) / 8000.0,
                        "spec_draft_sample_ms": sep["draft_ms"]}},
        "roofline": {"bound": "hbm",
                     "kernel": "spec_round, all five launches (stats_kernel over the draft rows, draft_select_kernel, "
                               "stats_kernel over the target rows, decide_stream_kernel, resid_draw_kernel), "
                               "timed as the step",
                     "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                     "frac": step_gbs / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": measured_traffic(w.name), "algorithmic_bytes_per_launch": step_bytes,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum over the round's five "
                                       "kernels, one capture per kernel (profiles/, null unless taken with the "
                                       "current kernel sources)"},
        # per step (spec_round on B=512): stats_kernel + draft_select_kernel, stats_kernel +
        # decide_stream_kernel + resid_draw_kernel
        "gpu_launches": 5 * args.steps,
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": e2e_line,
        "clocks": clocks,
        "other_workloads": extra,
        "adaptive_k": adapt,
        "tree_verify": tree,
        "vocab_sharded_verify": vshard,
        "k_sweep": sweep,
    }
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
