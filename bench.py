#!/usr/bin/env python
"""Draft-tree build + verify throughput on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
stage-1 log-softmax/Top-K over the vocabulary, tree selection, tree mask and
position ids, and the acceptance walk -- dt_build_tree, dt_tree_mask,
dt_verify through the C ABI.  Default workload: a single request at the Qwen3
vocabulary (batch 1, L=16, V=151936, bf16 logits with a +8 spike on one token
per position with probability 0.7), DDTree with K=B=256, greedy verification
against target rows whose spike matches the drafter's with probability 0.8.

Timing: every step reads a different copy of the inputs (rotating copies
whose drafter logits alone exceed twice the L2 size, so no step reads logits
another step left in L2); one CUDA graph holds the steps of a pass over all
copies and is replayed; CUDA events on the launching stream bracket exactly K
steps, with a barrier and a device synchronise on both sides; max over ranks.

Prints one JSON line.  --impl reference times the CPU oracle (the plain
restatement the tests check the kernels against) on the host cores instead.
"""
import argparse
import concurrent.futures
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft trees built+verified/sec and logit-read HBM GB/s (% of GB300 peak) at V=151936"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal

# ncu dram__bytes_read.sum + dram__bytes_write.sum per launch of the stage-1
# kernel, keyed by (kernel, workload, sha1 of the kernel's sources -- code only,
# comments and whitespace dropped -- when the capture was taken); a changed
# kernel reports null until it is captured again.
KN1_TRAFFIC = {
    ('kn1_kernel', 'ddtree_b1_L16_V151936_K128_B128', 'cbcf81db6862727ca848226199f3ec3a09787490'): 4932437,
    ('kn1_kernel', 'ddtree_b1_L16_V151936_K256_B256', 'cbcf81db6862727ca848226199f3ec3a09787490'): 4932523,
    ('kn1_kernel', 'ddtree_b1_L16_V151936_K64_B64', 'cbcf81db6862727ca848226199f3ec3a09787490'): 4932608,
    ('kn1_kernel', 'ddtree_t1_b1_L16_V151936_K256_B256', 'cbcf81db6862727ca848226199f3ec3a09787490'): 4932267,
    ('kn1b_kernel', 'dartree_b8_L16_V151936_W32_K16_B512_beta0', 'f17fce87448e4d8e01b396ff5ed69d6396ca1699'): 38964139,
    ('kn1b_kernel', 'ddtree_t1_b16_L16_V151936_K256_B256', 'f17fce87448e4d8e01b396ff5ed69d6396ca1699'): 78302464,
    ('kn1b_kernel', 'ddtree_t1_b4_L16_V151936_K256_B256', 'f17fce87448e4d8e01b396ff5ed69d6396ca1699'): 19515136,
    ('kn1b_kernel', 'talon_b64_L16_V151936_k10_mu0.03_N1024', 'f17fce87448e4d8e01b396ff5ed69d6396ca1699'): 325276075,
    ('kn1b_kernel', 'talon_b64_L16_V151936_k10_mu0.03_N60', 'f17fce87448e4d8e01b396ff5ed69d6396ca1699'): 315164501,
}
STAGE1_SOURCES = {
    "kn1_kernel": ("kn1_candidates.cu", "kn1_common.cuh", "dt_device.cuh"),
    "kn1b_kernel": ("kn1b_rows.cu", "kn1_common.cuh", "dt_device.cuh"),
}


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed: what the compiler sees,
    so that a comment edit does not void counters taken on unchanged code."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def stage1_source_hash(kernel):
    h = hashlib.sha1()
    for f in STAGE1_SOURCES[kernel]:
        with open(os.path.join(ROOT, "speculative_decoding_draft_bf16_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def workloads():
    from speculative_decoding_draft_bf16_gb300 import workloads as wk
    return {
        "single_request_B256": wk.single_request(256),
        "single_request_B128": wk.single_request(128),
        "single_request_B64": wk.single_request(64),
        "stochastic_b1": wk.stochastic_batch(1),
        "stochastic_b4": wk.stochastic_batch(4),
        "stochastic_b16": wk.stochastic_batch(16),
        "stochastic_iter_residual_b16": wk.stochastic_rule(16, "iter_residual"),
        "stochastic_target_match_b16": wk.stochastic_rule(16, "target_match"),
        "dartree_beta0": wk.dartree_supertree(0.0),
        "dartree_beta-0.5": wk.dartree_supertree(-0.5),
        "dartree_norm_beta0": wk.dartree_normalised(0.0),
        "dartree_norm_t1": wk.dartree_normalised_t1(0.0),
        "dartree_fixed": wk.dartree_fixed(),
        "ddtree_saba_b16": wk.ddtree_saba(16),
        "heap_markov": wk.heap_markov(False),
        "heap_markov_norm": wk.heap_markov(True),
        "heap_tdes": wk.heap_tdes(256),
        "talon_N60": wk.talon_gated(60),
        "talon_N1024": wk.talon_gated(1024),
    }


def max_over_ranks(value, world, device="cpu"):
    """Largest value over all ranks (replicas are timed independently; the job
    takes as long as its slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(steps, batch_per_rank, world, max_ms):
    """Whole-job trees/s: every rank's trees over the slowest rank's time."""
    return steps * batch_per_rank * world / (max_ms / 1000.0)


def headline(steps, batch_per_rank, world, max_ms):
    """The line's throughput keys for `steps` steps of `batch_per_rank` trees on
    each of `world` replicas, the slowest taking max_ms."""
    return {"value": job_throughput(steps, batch_per_rank, world, max_ms), "unit": "trees/s", "n_gpus": world,
            "steps": steps, "ms_per_step": max_ms / steps, "scaling": "weak"}


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--copies", type=int, default=0, help="rotating input copies (0: enough to exceed 2x L2)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="single_request_B256")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def normaliser_roofline(wl, stage_us, peaks):
    """The tensor-core normaliser's roofline (the dominant kernel of the
    normalised DARTree workload): 2 * rows * V * R flops of the contraction per
    launch over its measured stage time, against the sustained bf16 peak (it
    runs inside a long step)."""
    rows = wl.batch * wl.L * wl.K
    flops = 2.0 * rows * wl.V * wl.R
    tflops = flops / (stage_us["normalise"] * 1e-6) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
    source = ("measured (MEASURED_PEAKS.json bf16_tflops_sustained)" if "bf16_tflops_sustained" in peaks
              else "fallback (1.7 PFLOP/s, an earlier sustained GB300 bf16 measurement)")
    return {"roofline_normaliser": {
        "bound": "tensor", "kernel": "kn3n_kernel (tcgen05 [rows x 64] x [64 x V] + log-sum-exp)",
        "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
        "peak_source": source, "traffic": None,
        "algorithmic_flops_per_launch": flops,
        "note": "one exp per (row, token) in the epilogue: %.0f M per launch" % (rows * wl.V / 1e6)}}


def ceiling_fields(stage_us, draft_bytes, achieved, peak):
    """The read floor of the same launch (cluster stage 1 only): the same bytes
    read by a kernel with stage 1's grid, chunks, shared memory and launch mode
    that does nothing but take each chunk's maximum."""
    if "stage1_ceiling" not in stage_us:
        return {"ceiling": None}
    us = stage_us["stage1_ceiling"]
    gbs = draft_bytes / (us * 1e-6) / 1e9
    return {"ceiling": {"kernel": "kn0_kernel (stage 1's cluster launch; bulk copy + chunk max only)",
                        "us": us, "gbs": gbs, "frac_of_peak": gbs / peak},
            "frac_of_ceiling": achieved / gbs}


def params_for(wl, U=None, Vt=None, tdes=None, budgets=None):
    from speculative_decoding_draft_bf16_gb300 import dtree
    td = None
    if tdes is not None:
        Ap, Ac, Dd, w, b0, s = tdes
        td = dtree.Tdes(Ap, Ac, Dd, w, b0=b0, s=s)
    return dtree.Params(mode=wl.mode, batch=wl.batch, L=wl.L, V=wl.V, dtype=wl.dtype, K=wl.K, B=wl.B, W=wl.W,
                        beta=wl.beta, R=wl.R, U=U, Vt=Vt, talon_k=wl.talon_k, mu=wl.mu, N=wl.N,
                        markov_norm=wl.markov_norm, tdes=td, budget_policy=wl.budget_policy, budgets=budgets)


def max_nodes_of(wl):
    if wl.mode == "dartree":
        return min(wl.B, wl.W * wl.L) + 1
    return wl.max_nodes


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return None
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, wl, rank, world, local):
    import torch
    import torch.distributed as dist
    from speculative_decoding_draft_bf16_gb300 import dtree
    from speculative_decoding_draft_bf16_gb300 import workloads as wk

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dtree.lib()
    U = Vt = tdes = None
    if wl.R > 0 and wl.mode in ("dartree", "heap"):
        U, Vt = wk.markov_tables(wl.V, wl.R, device=dev)
    if wl.H > 0:
        tdes = wk.tdes_weights(wl.V, wl.L, wl.H, device=dev)
    saba = None
    if wl.saba_cv > 0:  # one history for the batch rows; the budgets feed the selection
        saba = dict(st=dtree.SabaState(wl.batch, 8, device=dev),
                    budget=torch.full((wl.batch,), wl.B, dtype=torch.int32, device=dev),
                    state=torch.zeros((wl.batch, 4), device=dev))
    p = params_for(wl, U, Vt, tdes, saba["budget"] if saba else None)
    plan_kind, plan_cluster = dtree.stage1_plan(p)
    Mmax = max_nodes_of(wl)
    esize = 2 if wl.dtype == "bf16" else 4
    draft_bytes = wl.batch * wl.L * wl.V * esize
    target_bytes = wl.batch * Mmax * wl.V * esize
    R = max(2, math.ceil(2 * L2_BYTES / draft_bytes))
    R = min(R, max(2, int(40e9 // max(target_bytes, 1))))
    if args.copies > 0:
        R = args.copies
    temperature = wl.temperature

    # rotating copies: distinct requests per copy and per rank
    copies = []
    for r in range(R):
        first = (rank * R + r) * wl.batch
        x, spikes = wk.draft_logits(wl, device=dev, first_req=first)
        tree = dtree.TreeBuffers(wl.batch, wl.L, p.Kc, Mmax, device=dev)
        ws = dtree.make_workspace(p, device=dev)
        dtree.build_tree(p, x, tree, workspace=ws)
        torch.cuda.synchronize()
        tgt = wk.target_logits(wl, tree.depth, tree.n_nodes, spikes, device=dev, first_req=first, rows=Mmax)
        uni = wk.uniforms(wl, device=dev, first_req=first) if temperature == 1.0 else None
        mask, pos = dtree.alloc_mask(tree, device=dev)
        out = dtree.alloc_verify_out(tree, device=dev)
        cmax = (torch.empty((wl.batch * wl.L, plan_cluster), device=dev) if plan_kind == "cluster" else None)
        copies.append(dict(x=x, tree=tree, ws=ws, tgt=tgt, uni=uni, mask=mask, pos=pos, out=out, cmax=cmax))

    markov_t1 = wl.mode == "dartree" and wl.markov_norm and temperature == 1.0

    def step(c, stages=("buildmask", "verify")):
        if saba is not None and ("buildmask" in stages or "saba" in stages):
            # SABA from this copy's previous round: its stage-1 tables and accepted lengths
            dtree.saba_budget(c["tree"], saba["st"], wl.saba_cv, wl.saba_cf, 1, wl.B, saba["budget"],
                              saba["state"], prev_acc_len=c["out"][1])
        if "buildmask" in stages:  # stage 1, selection, and the mask written by the selection kernel
            dtree.build_tree_mask(p, c["x"], c["tree"], c["mask"], c["pos"], workspace=c["ws"])
        if "build" in stages:
            dtree.build_tree(p, c["x"], c["tree"], workspace=c["ws"])
        if "cand" in stages:
            dtree.candidates(p, c["x"], c["tree"])
        if "ceil" in stages:  # the read floor of the cluster stage-1 launch
            dtree.stage1_ceiling(p, c["x"], c["cmax"])
        if "norm" in stages:
            dtree.markov_norm(p, c["x"], c["tree"], c["ws"])
        if "select" in stages:
            dtree.select(p, c["tree"], workspace=c["ws"])
        if "selmask" in stages:
            dtree.select_mask(p, c["tree"], c["mask"], c["pos"], workspace=c["ws"])
        if "mask" in stages:
            dtree.tree_mask(c["tree"], c["mask"], c["pos"])
        if "verify" in stages and markov_t1:  # T=1 against the normalised proposal q~
            dtree.verify_markov(p, c["tree"], c["tgt"], c["x"], dtree.znorm_view(p, c["ws"]), c["uni"],
                                out=c["out"])
        elif "verify" in stages:
            dtree.verify(c["tree"], c["tgt"], temperature=temperature,
                         draft=c["x"] if temperature and wl.verify_rule != "target_match" else None,
                         uniforms=c["uni"], out=c["out"], rule=wl.verify_rule or None)

    stream = torch.cuda.Stream(device=dev)

    def capture(stages, n_copies):
        """One CUDA graph running `stages` on copies 0..n_copies-1 in order."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in copies[:n_copies]:
                step(c, stages)
        return g

    def barrier():
        if world > 1:
            dist.barrier()

    def run_steps(stages, n, graphs):
        """Enqueue exactly n steps: full passes over the copies, then a prefix."""
        full, rem = divmod(n, R)
        for _ in range(full):
            graphs[R].replay()
        if rem:
            if rem not in graphs:
                graphs[rem] = capture(stages, rem)
            graphs[rem].replay()

    def timed(stages, n, warm):
        for c in copies:
            step(c, stages)  # eager call first (kernel attributes are set outside capture)
        torch.cuda.synchronize()
        graphs = {R: capture(stages, R)}
        for k in {n % R, warm % R} - {0}:
            graphs[k] = capture(stages, k)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            run_steps(stages, warm, graphs)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            run_steps(stages, n, graphs)
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        del graphs
        return ms

    clocks = ClockSampler(local)
    full_stages = ("buildmask", "verify")
    # the clock sampler runs over the timed region only
    for c in copies:
        step(c, full_stages)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    ms = timed(full_stages, args.steps, args.warmup)
    clk = clocks.stop()

    # per-stage device time (same rotating inputs, graphs of one stage)
    stage_us = {}
    stage_list = [("candidates", ("cand",)), ("select+mask", ("selmask",)), ("select", ("select",)),
                  ("mask", ("mask",)), ("verify", ("verify",))]
    if wl.markov_norm:
        stage_list.insert(1, ("normalise", ("norm",)))
    if saba is not None:
        stage_list.insert(1, ("saba", ("saba",)))
    if plan_kind == "cluster":
        stage_list.insert(1, ("stage1_ceiling", ("ceil",)))
    for name, stages in stage_list:
        n = max(R, (args.steps // R) * R)
        stage_us[name] = timed(stages, n, R) * 1000.0 / n

    # end to end: pinned host inputs copied in, results copied out, every step
    e2e = None
    if args.e2e_steps > 0:
        hx = [copies[i]["x"].cpu().pin_memory() for i in range(2)]
        ht = [copies[i]["tgt"].cpu().pin_memory() for i in range(2)]
        hu = [copies[i]["uni"].cpu().pin_memory() if copies[i]["uni"] is not None else None for i in range(2)]
        c = copies[0]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in c["out"]]
        htok = torch.empty(c["tree"].node_tok.shape, dtype=torch.int32, pin_memory=True)
        h2d = hx[0].numel() * hx[0].element_size() + ht[0].numel() * ht[0].element_size()
        if hu[0] is not None:
            h2d += hu[0].numel() * 4
        d2h = sum(t.numel() * 4 for t in hout) + htok.numel() * 4

        def e2e_step(i):
            j = i % 2
            c["x"].copy_(hx[j], non_blocking=True)
            c["tgt"].copy_(ht[j], non_blocking=True)
            if hu[j] is not None:
                c["uni"].copy_(hu[j], non_blocking=True)
            step(c)
            for h, d in zip(hout, c["out"]):
                h.copy_(d, non_blocking=True)
            htok.copy_(c["tree"].node_tok, non_blocking=True)

        with torch.cuda.stream(stream):
            for i in range(3):
                e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.e2e_steps):
                e2e_step(i)
            e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": job_throughput(args.e2e_steps, wl.batch, world, ems), "unit": "trees/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    status = sum(int(c["tree"].status.abs().sum()) for c in copies)
    # stage 1, selection (writing the mask), walk; the heap's separate mask kernel; the Markov or TDES
    # edge table; the normalised correction's table conversion, normaliser and merge
    edge_table = wl.mode in ("dartree", "heap") and (wl.R > 0 or wl.H > 0)
    launches_per_step = (3 + (1 if wl.mode == "heap" else 0) + (1 if edge_table else 0) +
                         (3 if wl.markov_norm else 0) + (1 if saba is not None else 0))
    kn1_s = stage_us["candidates"] / 1e6
    achieved = draft_bytes / kn1_s / 1e9
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_source = ("measured (MEASURED_PEAKS.json hbm_gbs)" if "hbm_gbs" in peaks
                   else "fallback (6.8 TB/s, an earlier GB300 copy measurement; no MEASURED_PEAKS.json value)")
    kn1_name = "kn1_kernel" if plan_kind == "cluster" else "kn1b_kernel"
    kn1_desc = ("%s (log-softmax + Top-K, a cluster of %d CTAs per row)" % (kn1_name, plan_cluster)
                if plan_kind == "cluster" else "%s (log-softmax + Top-K, one CTA per row)" % kn1_name)
    traffic = KN1_TRAFFIC.get((kn1_name, wl.name, stage1_source_hash(kn1_name)))
    result = {
        "metric": METRIC,
        **headline(args.steps, wl.batch, world, ms),
        "warmup": args.warmup,
        "higher_is_better": True,
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded Gaussian logits with confident-token spikes; Qwen3 vocabulary)",
        "config": {"workload": wl.name, "mode": wl.mode, "batch_per_gpu": wl.batch, "L": wl.L, "V": wl.V,
                   "K": wl.K, "B": wl.B, "W": wl.W, "beta": wl.beta, "N": wl.N, "R": wl.R, "H": wl.H,
                   "markov_norm": wl.markov_norm, "budget_policy": wl.budget_policy,
                   "saba": {"c_verify": wl.saba_cv, "c_fixed": wl.saba_cf} if saba is not None else None,
                   "temperature": temperature,
                   "verify_rule": wl.verify_rule or ("ratio" if temperature else "greedy"),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "rotating %d input copies (drafter logits %.0f MB > 2x L2)" % (R, R * draft_bytes / 1e6)},
        "roofline": {"bound": "hbm", "kernel": kn1_desc, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_source,
                     "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic, "algorithmic_bytes_per_launch": draft_bytes,
                     **ceiling_fields(stage_us, draft_bytes, achieved, peak)},
        "stages_us": stage_us,
        **(normaliser_roofline(wl, stage_us, peaks) if wl.markov_norm else {}),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "device_status_nonzero": status,
    }
    return result, copies


# ---------------------------------------------------------------------------
# CPU oracle: baseline leg and reference arm
# ---------------------------------------------------------------------------
def oracle_round(wl, x, tgt, uni, M):
    """One tree through the oracle: stage 1, selection, mask, walk.  M: the
    edge-term weights (U, Vt: Markov; tdes: TDES) as host arrays.  Returns a
    dict: tree, lps (the stage-1 table), check (selection_check arguments for
    this mode), walk ((acc_nodes, acc_len, next_tok), or None without targets)."""
    import numpy as np
    import oracle
    _, l32, ids, lps = oracle.candidates(x, wl.Kc)
    Mmax = max_nodes_of(wl)
    U, Vt = M["U"], M["Vt"]
    check = {"mode": wl.mode}
    z = None
    if wl.mode == "ddtree":
        B = wl.B
        if wl.saba_cv > 0:  # SABA budget from this tree's state (no history yet)
            B, _ = oracle.saba(lps[:, 0], None, oracle.SabaState(8), -1, wl.saba_cv, wl.saba_cf, 1, wl.B)
        t = oracle.ddtree(lps, ids, B, Mmax=Mmax)
    elif wl.mode == "dartree":
        z = oracle.markov_norm(x, ids, U, Vt, -1) if wl.markov_norm else None
        widths = oracle.uniform_widths(wl.B, wl.L) if wl.budget_policy == "uniform" else None
        W = int(widths.max()) if widths is not None else wl.W
        t, _, _ = oracle.dartree(lps, ids, U, Vt, -1, W, wl.beta, wl.B, Mmax=Mmax, znorm=z, widths=widths)
        if U is not None:
            check.update(E=oracle.markov_table(ids, U, Vt, -1), znorm=z, beta=wl.beta)
    elif wl.mode == "heap":
        E = None
        if M["tdes"] is not None:
            Ap, Ac, Dd, w, b0, s = M["tdes"]
            E = oracle.tdes_table(ids, Ap, Ac, Dd, w, b0, s, -1)
        elif U is not None:
            E = oracle.markov_table(ids, U, Vt, -1)
            z = oracle.markov_norm(x, ids, U, Vt, -1) if wl.markov_norm else None
        t = oracle.heap_select(lps, ids, wl.B, E=E, znorm=z, Mmax=Mmax)
        check.update(E=E, znorm=z)
    else:
        t = oracle.talon(lps, ids, wl.talon_k, wl.log_mu, wl.N, Mmax=Mmax)
        check.update(log_mu=wl.log_mu)
    oracle.tree_mask(t, Mmax, wl.L)
    walk = None
    if tgt is not None:
        if wl.temperature == 1.0 and wl.mode == "dartree" and wl.markov_norm:
            walk = oracle.verify_t1_markov(t, tgt, x, l32, U, Vt, -1, z, uni, wl.L, Mmax)[:3]
        elif wl.temperature == 1.0:
            walk = oracle.verify_t1(t, tgt, x, l32, uni, wl.L, Mmax, rule=wl.verify_rule or "ratio")[:3]
        else:
            walk = oracle.verify_greedy(t, tgt, wl.L)
    return {"tree": t, "lps": lps, "check": check, "walk": walk}


def oracle_inputs(wl, n_trees, seed_base=10_000):
    """Host inputs for n_trees requests; targets follow the oracle's own trees."""
    import numpy as np
    import torch
    from speculative_decoding_draft_bf16_gb300 import workloads as wk
    M = {"U": None, "Vt": None, "tdes": None}
    if wl.R > 0 and wl.mode in ("dartree", "heap"):
        M["U"], M["Vt"] = (t.numpy() for t in wk.markov_tables(wl.V, wl.R))
    if wl.H > 0:
        M["tdes"] = tuple(v.numpy() if hasattr(v, "numpy") else v for v in wk.tdes_weights(wl.V, wl.L, wl.H))
    one = wl.with_(batch=1)
    items = []
    for i in range(n_trees):
        x, spikes = wk.draft_logits(one, first_req=seed_base + i)
        xf = x[0].float().numpy()
        t = oracle_round(wl, xf, None, None, M)["tree"]
        Mmax = max_nodes_of(wl)
        depth = np.zeros((1, Mmax), np.int32)
        depth[0, :t.n] = t.depth[:t.n]
        tgt = wk.target_logits(one, depth, [t.n], spikes, first_req=seed_base + i, rows=Mmax)[0].float().numpy()
        uni = wk.uniforms(one, first_req=seed_base + i)[0].numpy() if wl.temperature == 1.0 else None
        items.append((xf, tgt, uni))
    return items, M


def time_oracle(wl, items, M, threads):
    """Seconds for the oracle rounds of `items` on `threads` host threads, and their results."""
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(lambda it: oracle_round(wl, it[0], it[1], it[2], M), items))
    return time.perf_counter() - t0, res


# Tolerance of the normaliser table of the normalised DARTree correction,
# added to the per-log-prob 1e-5 for the edge terms that subtract it.
ZNORM_TOL = 1e-5


def parity_sample(wl, items, results, n_max=16):
    """The GPU's trees and walks against the oracle's on the first n_max
    requests of the CPU sample (untimed): every selection difference must be a
    near-tie (oracle.selection_check, the per-log-prob tolerance 1e-5 summed
    along each path); the count is reported.  Walks are compared on requests
    whose trees agree node for node.  SABA budgets depend on each request's
    history, which the sample does not carry: not compared."""
    import numpy as np
    import torch
    import oracle
    from speculative_decoding_draft_bf16_gb300 import dtree
    from speculative_decoding_draft_bf16_gb300 import workloads as wk
    if wl.saba_cv > 0:
        return {"compared": 0, "reason": "SABA budgets depend on per-request history"}
    dev = torch.device("cuda", torch.cuda.current_device())
    one = wl.with_(batch=1)
    # the oracle's tables are drawn on the host (a device generator draws other values): the same here
    U = Vt = tdes = None
    if wl.R > 0 and wl.mode in ("dartree", "heap"):
        U, Vt = (t.to(dev) for t in wk.markov_tables(wl.V, wl.R))
    if wl.H > 0:
        tdes = tuple(v.to(dev) if torch.is_tensor(v) else v for v in wk.tdes_weights(wl.V, wl.L, wl.H))
    p = params_for(one, U, Vt, tdes)
    tot = {"requests": 0, "near_ties": 0, "consequences": 0, "order_swaps": 0, "mismatches": 0,
           "order_mismatches": 0, "score_err_viol": 0, "score_err_max": 0.0, "tolerance_max": 0.0,
           "walks_compared": 0, "walk_mismatches": 0}
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    Mmax = max_nodes_of(wl)
    for (xf, tgt, uni), res in list(zip(items, results))[:n_max]:
        x = torch.from_numpy(xf).to(dt).reshape(1, wl.L, wl.V).to(dev)
        tree = dtree.TreeBuffers(1, wl.L, p.Kc, Mmax, device=dev)
        ws = dtree.make_workspace(p, device=dev)
        dtree.build_tree(p, x, tree, workspace=ws)
        t_dev = torch.from_numpy(tgt).to(dt).reshape(1, Mmax, wl.V).to(dev)
        u_dev = torch.from_numpy(uni).reshape(1, 2, Mmax).to(dev) if uni is not None else None
        if wl.temperature == 1.0 and wl.mode == "dartree" and wl.markov_norm:
            out = dtree.verify_markov(p, tree, t_dev, x, dtree.znorm_view(p, ws), u_dev)
        else:
            out = dtree.verify(tree, t_dev, temperature=wl.temperature,
                               draft=x if wl.temperature and wl.verify_rule != "target_match" else None,
                               uniforms=u_dev, rule=wl.verify_rule or None)
        torch.cuda.synchronize()
        n = int(tree.n_nodes[0])
        g = oracle.Tree(*(getattr(tree, f)[0].cpu().numpy()[:n].copy() for f in
                          ("node_tok", "parent", "depth", "rank", "score")), n)
        kw = dict(res["check"])
        mode = kw.pop("mode")
        eps_z = ZNORM_TOL if kw.get("znorm") is not None else 0.0
        rep = oracle.selection_check(g, res["tree"].trimmed(), res["lps"], mode, eps_z=eps_z, got_scores=g.score,
                                     **kw)
        tot["requests"] += 1
        for k in ("near_ties", "consequences", "order_swaps", "order_mismatches", "score_err_viol"):
            tot[k] += rep[k]
        tot["mismatches"] += len(rep["mismatches"])
        tot["score_err_max"] = max(tot["score_err_max"], rep["score_err_max"])
        tot["tolerance_max"] = max(tot["tolerance_max"], rep["tau_max"])
        o = res["tree"]
        if g.n == o.n and np.array_equal(g.tok, o.tok[:n]) and np.array_equal(g.parent, o.parent[:n]):
            acc, alen, nxt = res["walk"]
            tot["walks_compared"] += 1
            same = (out[0][0].cpu().tolist() == list(acc) and int(out[1][0]) == alen and int(out[2][0]) == nxt)
            tot["walk_mismatches"] += 0 if same else 1
    return tot


def cpu_baseline(wl, cpu_seconds=20.0):
    """The oracle on the host cores, one tree per thread, on a sample sized to
    about `cpu_seconds` of CPU work (one tree is timed first to size it); then
    the GPU's trees on the first requests of the same sample against the
    oracle's (untimed)."""
    from oracle import build as ob
    ob.build()
    cores = os.cpu_count() or 1
    probe, M = oracle_inputs(wl, 1, seed_base=20_000)
    t1, _ = time_oracle(wl, probe, M, 1)
    trees = int(max(cores, min(4 * cores, cpu_seconds / max(t1, 1e-3))))
    items, M = oracle_inputs(wl, trees)
    sec, results = time_oracle(wl, items, M, cores)
    base = {"value": trees / sec, "unit": "trees/s", "cores": cores, "kind": "oracle",
            "sample": "%d single-request trees of the %s workload (stage 1, selection, mask, walk; "
                      "%.2f s per tree on one core), one thread per tree over %d host cores"
                      % (trees, wl.name, t1, cores)}
    return base, parity_sample(wl, items, results)


def run_reference(args, wl, rank, world, budget_s=150.0, warm_budget_s=30.0):
    """The oracle as the reference arm: each step is one tree per host core.
    The requested warm-up steps run untimed (at least min(3, requested); more
    only while they fit in about `warm_budget_s` seconds); timed steps beyond
    what fits in about `budget_s` seconds are not run.  The line reports the
    steps actually run beside the requested ones."""
    if rank != 0:
        return None
    from oracle import build as ob
    ob.build()
    cores = os.cpu_count() or 1
    per_step = cores
    items, M = oracle_inputs(wl, per_step)
    warm, _ = time_oracle(wl, items, M, cores)  # the first untimed warm-up step, which also sizes the rest
    warmup = max(1, min(args.warmup, max(3, int(warm_budget_s / max(warm, 1e-3)))))
    for _ in range(warmup - 1):
        time_oracle(wl, items, M, cores)
    steps = max(1, min(args.steps, int(budget_s / max(warm, 1e-3))))
    total = 0.0
    for _ in range(steps):
        total += time_oracle(wl, items, M, cores)[0]
    value = steps * per_step / total
    sample = "%d single-request trees per step (one per host core), %d of %d requested steps timed after %d " \
             "of %d requested warm-up steps" % (per_step, steps, args.steps, warmup, args.warmup)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "trees/s", "n_gpus": world,
        "steps": steps, "steps_requested": args.steps, "warmup": warmup, "warmup_requested": args.warmup,
        "ms_per_step": 1000.0 * total / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded Gaussian logits with confident-token spikes; Qwen3 vocabulary)",
        "config": {"workload": wl.name, "mode": wl.mode, "batch_per_step": per_step, "L": wl.L, "V": wl.V,
                   "K": wl.K, "B": wl.B, "temperature": wl.temperature},
        "cpu_baseline": {"value": value, "unit": "trees/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "trees/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def launch_plan(gpus, env, argv, port=None):
    """How `bench.py --gpus N` runs.  Under a launcher that set WORLD_SIZE (the
    driver's torchrun) each process is one rank and WORLD_SIZE must equal N:
    ("ranks", None), or ("single", None) for N = 1.  Without one, N = 1 runs
    here and N > 1 re-launches this script as N local ranks, one per GPU,
    through torch.distributed.run on 127.0.0.1: ("spawn", command).  Requests
    are independent, so the ranks are replicas that share only the final
    max-over-ranks time reduction."""
    world = env.get("WORLD_SIZE")
    if world is not None:
        if int(world) != gpus:
            raise SystemExit("bench.py: --gpus %d does not match WORLD_SIZE=%s" % (gpus, world))
        return ("ranks", None) if gpus > 1 else ("single", None)
    if gpus <= 1:
        return ("single", None)
    if port is None:
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
    return ("spawn", [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(gpus),
                      "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv])


def main():
    args = parse()
    mode, cmd = launch_plan(args.gpus, os.environ, sys.argv[1:])
    if mode == "spawn":
        sys.exit(subprocess.call(cmd))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workloads()[args.workload]
    if args.impl == "reference":
        out = run_reference(args, wl, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    result, copies = run_ours(args, wl, rank, world, local)
    del copies
    if rank == 0:
        if not args.no_cpu_baseline:
            result["cpu_baseline"], par = cpu_baseline(wl)
            result["parity_sample"] = par
            result["near_ties"] = par.get("near_ties")
            result["mismatches"] = (par["mismatches"] + par["order_mismatches"] + par["score_err_viol"] +
                                    par["walk_mismatches"]) if par.get("requests") else None
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
