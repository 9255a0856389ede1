#!/usr/bin/env python3
"""Benchmark of ancestor-masked tree attention over a shared page-prefix KV
cache on one or more GPUs (one process per GPU, weak scaling).

A step runs both regimes of the hot path on the serving-scale workload:
  * branch decode: 512 pages, prefix U[4000, 6144] tokens, 8-60 branches per
    page (zero-copy forks of the page prefix), own suffix U[0, 1024], one
    query token per live branch (about 17.6 k branches); kernels: the cascade
    prefix pass and the own-suffix pass with the log-sum-exp merge;
  * tree-varlen forward and its backward (dQ, dK, dV): 8 packed sequences of
    16384 tokens built from the same page-length distributions.
`value` is branch-decode attention tokens per second (query tokens of all
ranks divided by the slowest rank's decode time); the forward's and the
backward's TFLOP/s and the roofline fractions ride along in the same JSON
line.  The same timed loop also runs two smaller decode steps on pages of
their own and reports them under kernels.branch_decode and kernels.verify:
  * branch decode over 16 pages (prefix 4809, 8-40 branches, own suffix
    U[0, 512], one query per branch);
  * speculative verify over 64 pages (the same shapes, a draft tree of up
    to 16 nodes per branch), followed by the accept step over every draft
    node's 151,936 logits.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "branch-decode attn tokens/s & % HBM roofline; tree-varlen fwd TFLOP/s & % peak"
WORKLOADS = {
    "serving": "serving-scale: branch decode over 512 pages (prefix U[4000,6144], 8-60 branches/page, own suffix "
               "U[0,1024], 1 query/branch)",
    "branch": "branch decode over 16 pages (prefix 4809, 8-40 branches/page, own suffix U[0,512], 1 query/branch)",
    "verify": "speculative verify over 64 pages (prefix 4809, 8-40 branches/page, own suffix U[0,512], draft tree "
              "of up to 16 nodes per branch)",
}


def workload_name(kind: str, fwd_seqs: int) -> str:
    return (WORKLOADS[kind] + f" + tree-varlen forward and backward over {fwd_seqs} x 16384 packed tokens; "
            "bf16, Hq=16, Hkv=8, d=128")


WORKLOAD = workload_name("serving", 8)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "of measured"
    return FALLBACK_PEAKS, "of fallback"


# ---------------------------------------------------------------- CPU oracle legs


def _oracle_decode_pages(args):
    """Child process: the oracle's branch decode over sampled pages, timed."""
    seed, page_ids = args
    sys.path.insert(0, ROOT)
    from oracle import tree_attention as ta
    from tree_structured_shared_gb300 import workloads as wl
    full = wl.serving_decode(seed)
    sub = wl.DecodeWorkload("sample", [full.pages[i] for i in page_ids], full.Hq, full.Hkv, full.d,
                            full.value_scale)
    vals = wl.decode_values(sub, seed + 17)
    t0 = time.perf_counter()
    ta.branch_decode(sub, vals, tree=False)
    return time.perf_counter() - t0, sub.n_queries


def _oracle_forward_rows(args):
    """Child process: the oracle's forward on sampled rows of one packed page."""
    seed, n_rows = args
    sys.path.insert(0, ROOT)
    import numpy as np
    from oracle import tree_attention as ta
    from tree_structured_shared_gb300 import workloads as wl
    full = wl.packed_sequences(seed)
    page = wl.TreeWorkload("p", [full.pages[0]], full.Hq, full.Hkv, full.d, "bf16", 0.5, [0])
    q, k, v = wl.tree_qkv(page, seed)
    rng = np.random.default_rng(seed)
    rows = sorted(rng.choice(page.n_tokens, n_rows, replace=False).tolist())
    anc = ta.ancestor_positions(page.pages)
    pairs = sum(len(anc[r]) for r in rows)
    t0 = time.perf_counter()
    ta.tree_forward(q, k, v, page.pages, positions=rows)
    return time.perf_counter() - t0, 4.0 * page.d * page.Hq * pairs


def cpu_oracle_baseline(seed: int, n_pages: int, fwd_rows: int):
    """The oracle as it stands, on the host cores, over a bounded sample."""
    cores = len(os.sched_getaffinity(0))
    used = min(cores, n_pages)
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(processes=used) as pool:
        res = pool.map(_oracle_decode_pages, [(seed, [i]) for i in range(n_pages)])
        nf = min(used, 4)
        fwd = pool.map(_oracle_forward_rows, [(seed + i, fwd_rows) for i in range(nf)])
    wall = time.perf_counter() - t0
    dec_tokens = sum(r[1] for r in res)
    dec_cpu = sum(r[0] for r in res)
    fwd_cpu = sum(r[0] for r in fwd)
    return {
        "value": dec_tokens / (dec_cpu / used),
        "unit": "tokens/s",
        "cores": used,
        "kind": "oracle",
        "sample": (f"{n_pages} of the 512 decode pages ({dec_tokens} branch queries), one page per process, "
                   f"float64 NumPy; rate = queries / (summed oracle seconds / processes); forward: {fwd_rows} "
                   f"sampled query rows of one packed page in each of {nf} processes"),
        "cpu_seconds": round(dec_cpu + fwd_cpu, 2),
        "wall_seconds": round(wall, 2),
        "forward_tflops": sum(r[1] for r in fwd) / (fwd_cpu / nf) / 1e12,
    }


def run_reference(args, rank: int) -> int:
    """Reference arm: the float64 oracle on host cores, same metric."""
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0))
    per_step = max(1, min(cores, 4))
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=per_step) as pool:
        for w in range(args.warmup):
            pool.map(_oracle_decode_pages, [(args.seed, [w % 512])])
        toks = 0
        t0 = time.perf_counter()
        for s in range(args.steps):
            ids = [(s * per_step + i) % 512 for i in range(per_step)]
            res = pool.map(_oracle_decode_pages, [(args.seed, [i]) for i in ids])
            toks += sum(r[1] for r in res)
        total = time.perf_counter() - t0
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "reference": "float64 CPU oracle (the pages publish no implementation)",
                   "per_step": f"{per_step} decode pages, one per process"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": per_step, "kind": "oracle",
                         "sample": f"{per_step} pages of the 512-page decode workload per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="padoc_clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx = float(p[2])
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm


def traffic_for(kernel: str, units: float):
    """DRAM bytes per launch from the committed ncu summary, scaled by units,
    or None when the kernel's source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "tree_structured_shared_gb300", "csrc", d["source"])
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha"]:
        return None
    return d["dram_bytes"] / d["units"] * units


def bwd_traffic(units: float):
    """DRAM bytes of the dQ and dK/dV passes (the row-sum pass is not
    captured), or None when either kernel changed since the capture."""
    a, b = traffic_for("bwd_dq", units), traffic_for("bwd_dkv", units)
    return None if a is None or b is None else a + b


def decode_report(dec, dw, t_pre: float, t_own: float, hbm: float, tf_sus: float) -> dict:
    """Per-pass and whole-step figures of one decode / verify step: times,
    algorithmic bytes (unique KV once per page, own tokens once, the query
    block, O and LSE) and flops (4 d Hq per query-ancestor pair), the
    fractions of HBM and sustained tensor peak, and the roofline bound time
    max(bytes / BW, flops / peak)."""
    own_b, pre_b, all_b = dec.own_bytes(), dec.prefix_bytes(), dec.unique_kv_bytes()
    dec_fl = dec.flops()
    pre_fl = 4.0 * dw.d * dw.Hq * sum(pg.q_len[j] * pg.branch_prefix_len[j] for pg in dw.pages
                                      for j in range(len(pg.q_len)))
    own_fl = dec_fl - pre_fl
    t_dec = t_pre + t_own

    def part(ms, b, fl):
        gbs, tfs = b / (ms * 1e-3) / 1e9, fl / (ms * 1e-3) / 1e12
        bound = max(b / (hbm * 1e9), fl / (tf_sus * 1e12)) * 1e3
        return {"ms": ms, "algorithmic_bytes": b, "algorithmic_flops": fl, "achieved_gbs": gbs,
                "frac_hbm": gbs / hbm, "achieved_tflops": tfs, "frac_tensor": tfs / tf_sus,
                "bound_time_ms": bound, "frac_of_bound": bound / ms}

    step = dict(part(t_dec, all_b, dec_fl), tokens_per_s=dec.nq / (t_dec * 1e-3),
                frac_spec_8tbs=all_b / (t_dec * 1e-3) / 1e9 / 8000.0)
    if dec._plan.fused():
        # one kernel: the prefix pass call launches nothing
        return {"fused_pass": dict(part(t_dec, all_b, dec_fl), kernel="attn_tc_kernel<MODE_VERIFY>"),
                "step": step, "pages": len(dw.pages), "branches": dw.n_branches, "query_tokens": dec.nq}
    return {"prefix_pass": part(t_pre, pre_b, pre_fl), "own_pass": part(t_own, own_b, own_fl),
            "step": step, "pages": len(dw.pages), "branches": dw.n_branches, "query_tokens": dec.nq}


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-pages", type=int, default=32, help="decode pages in the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default="serving", choices=sorted(WORKLOADS),
                    help="serving (the default bench line); branch and verify are smaller cases for profiling")
    ap.add_argument("--fwd-seqs", type=int, default=8, help="packed 16384-token sequences in the forward")
    ap.add_argument("--vocab", type=int, default=151936, help="vocabulary of the verify workload's accept step")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the 16-page branch decode and 64-page verify steps timed beside the serving step")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")

    # the CPU baseline's process pool runs before any CUDA work (spawn)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "serving":
        cpu = cpu_oracle_baseline(args.seed, args.cpu_pages, 64)

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    from tree_structured_shared_gb300 import build, harness, padoc
    from tree_structured_shared_gb300 import workloads as wl
    if not os.path.exists(padoc.LIB_PATH):
        build.build()
    seed = args.seed + 1000 * rank  # independent pages per rank

    dw = {"serving": wl.serving_decode, "branch": wl.branch_decode, "verify": wl.spec_verify}[args.workload](seed)
    fw = wl.packed_sequences(seed, n_seq=args.fwd_seqs)
    dec = harness.Decode(dw, seed=seed, tree=args.workload == "verify")
    fwd = harness.Forward(fw, seed=seed)
    bwd = harness.Backward(fwd, seed=seed)
    dec.plan()
    stream = torch.cuda.current_stream()
    acc = None
    if args.workload == "verify":
        # the accept step over next-token logits of every draft node
        trees = [t for pg in dw.pages for t in pg.parents]
        acc = harness.Accept(trees, args.vocab, seed)

    def accept_step():
        if acc is not None:
            acc.run()

    # Beside the serving step, the same loop times the 16-page branch decode
    # and the 64-page speculative verify step (attention + accept), each on
    # its own seeded pages.
    side = {}
    if args.workload == "serving" and not args.no_side:
        bw = wl.branch_decode(seed)
        side["branch_decode"] = {"w": bw, "dec": harness.Decode(bw, seed=seed + 1, tree=False)}
        vw = wl.spec_verify(seed)
        side["verify"] = {"w": vw, "dec": harness.Decode(vw, seed=seed + 2, tree=True),
                          "acc": harness.Accept([t for pg in vw.pages for t in pg.parents], args.vocab, seed + 3)}
        for sd in side.values():
            sd["dec"].plan()

    def side_step(evs):
        i = 0
        for name in ("branch_decode", "verify"):
            if name not in side:
                continue
            sd = side[name]
            evs[i].record(stream)
            sd["dec"].prefix_pass()
            evs[i + 1].record(stream)
            sd["dec"].own_pass()
            evs[i + 2].record(stream)
            if "acc" in sd:
                sd["acc"].run()
            evs[i + 3].record(stream)
            i += 4

    n_side_ev = 4 * len(side)
    for _ in range(args.warmup):
        dec.prefix_pass()
        dec.own_pass()
        accept_step()
        fwd.run()
        bwd.run()
        side_step([torch.cuda.Event() for _ in range(n_side_ev)])
    torch.cuda.synchronize()
    padoc.device_status()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_side_ev)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for s in range(K):
        ev[s][0].record(stream)
        dec.prefix_pass()
        ev[s][1].record(stream)
        dec.own_pass()
        ev[s][2].record(stream)
        accept_step()
        ev[s][3].record(stream)
        fwd.run()
        ev[s][4].record(stream)
        bwd.run()
        ev[s][5].record(stream)
        side_step(sev[s])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    padoc.device_status()
    t_pre = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    t_own = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    t_acc = sum(e[2].elapsed_time(e[3]) for e in ev) / K
    t_fwd = sum(e[3].elapsed_time(e[4]) for e in ev) / K
    t_bwd = sum(e[4].elapsed_time(e[5]) for e in ev) / K
    t_dec = t_pre + t_own
    t_side = [sum(e[i].elapsed_time(e[i + 1]) for e in sev) / K for i in range(n_side_ev) if i % 4 != 3]
    times = torch.tensor([t_dec, t_fwd, t_pre, t_own, t_acc, t_bwd] + t_side, dtype=torch.float64, device="cuda")
    if world > 1:
        dist.all_reduce(times, op=dist.ReduceOp.MAX)
    t_dec, t_fwd, t_pre, t_own, t_acc, t_bwd = [float(x) for x in times.tolist()[:6]]
    t_side = [float(x) for x in times.tolist()[6:]]

    # end to end through the all-in-one C-ABI call, inputs from pinned host memory
    e2e = None
    nq = dec.nq
    if not args.no_e2e:
        h_q = torch.empty(dec.q.shape, dtype=dec.q.dtype, pin_memory=True)
        h_k = torch.empty(dec.k_new.shape, dtype=dec.k_new.dtype, pin_memory=True)
        h_v = torch.empty(dec.v_new.shape, dtype=dec.v_new.dtype, pin_memory=True)
        h_q.copy_(dec.q)
        h_k.copy_(dec.k_new)
        h_v.copy_(dec.v_new)
        # Two sets of device inputs and outputs, and a copy stream for each
        # direction: the copies of one step run beside the kernels of the
        # other, while every step still copies its own inputs in and its own
        # result out inside the timed region.
        n_sets = 2
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        d_in = [(torch.empty_like(dec.q), torch.empty_like(dec.k_new), torch.empty_like(dec.v_new))
                for _ in range(n_sets)]
        d_out = [(torch.empty_like(dec.o), torch.empty_like(dec.lse)) for _ in range(n_sets)]
        h_out = [(torch.empty(dec.o.shape, dtype=dec.o.dtype, pin_memory=True),
                  torch.empty(dec.lse.shape, dtype=dec.lse.dtype, pin_memory=True)) for _ in range(n_sets)]
        ev_in = [torch.cuda.Event() for _ in range(n_sets)]    # inputs of set b copied in
        ev_done = [torch.cuda.Event() for _ in range(n_sets)]  # the step that read set b has run
        ev_out = [torch.cuda.Event() for _ in range(n_sets)]   # the result in set b copied out
        for b in range(n_sets):
            ev_done[b].record(comp)
            ev_out[b].record(comp)
        step_no = [0]

        def e2e_step():
            b = step_no[0] % n_sets
            step_no[0] += 1
            dq, dk, dv = d_in[b]
            o, l = d_out[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[b])
                dq.copy_(h_q, non_blocking=True)
                dk.copy_(h_k, non_blocking=True)
                dv.copy_(h_v, non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])
            padoc.branch_decode(dec.pool, dec.batch, dw.Hq, dq, dk, dv, dec.tree_bits, o, l, dec.ws, dec.ws_bytes,
                                stream=comp)
            ev_done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                h_out[b][0].copy_(o, non_blocking=True)
                h_out[b][1].copy_(l, non_blocking=True)
                ev_out[b].record(s_out)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        torch.cuda.synchronize()
        te = torch.tensor([(time.perf_counter() - t0) / K], dtype=torch.float64, device="cuda")
        if world > 1:
            dist.all_reduce(te, op=dist.ReduceOp.MAX)
        te = float(te.item())
        e2e = {"value": nq * world / te, "unit": "tokens/s",
               "h2d_bytes_per_step": (h_q.numel() + h_k.numel() + h_v.numel()) * 2,
               "d2h_bytes_per_step": h_out[0][0].numel() * 2 + h_out[0][1].numel() * 4, "ms_per_step": te * 1000,
               "includes": ("host plan build, block-table and plan upload, both passes, input and output copies; "
                            "two buffer sets, so one step's copies overlap the other's kernels")}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tf_sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    own_b, pre_b, all_b = dec.own_bytes(), dec.prefix_bytes(), dec.unique_kv_bytes()
    # algorithmic flops (4 d Hq per query-ancestor pair): the whole step, and
    # the prefix pass's share (each query row against its page prefix)
    dec_fl = dec.flops()
    pre_fl = 4.0 * dw.d * dw.Hq * sum(pg.q_len[j] * pg.branch_prefix_len[j] for pg in dw.pages
                                      for j in range(len(pg.q_len)))
    fl = fwd.flops
    fwd_ex = fwd.executed_flops  # tensor-core work incl. masked / padded tile elements
    own_gbs = own_b / (t_own * 1e-3) / 1e9
    pre_gbs = pre_b / (t_pre * 1e-3) / 1e9
    dec_gbs = all_b / (t_dec * 1e-3) / 1e9
    fwd_tf = fl / (t_fwd * 1e-3) / 1e12
    own_units = sum(sum(p.own_len) for p in dw.pages)
    line = {
        "metric": METRIC,
        "value": nq * world / (t_dec * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": t_dec,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(args.workload, args.fwd_seqs), "pages": len(dw.pages), "branches": dw.n_branches, "query_tokens": nq,
                   "forward_tokens": fw.n_tokens,
                   "l2": "inputs larger than L2 (decode KV about 48 GB, forward Q/K/V 1.3 GB)",
                   "step": ("value and ms_per_step cover the decode step (prefix pass + own pass); the forward "
                            "and its backward run in the same timed loop and are reported under 'forward' and "
                            "'backward'"),
                   "parallelism": f"dp{world} (independent pages per GPU)"},
        "roofline": {"bound": "hbm", "kernel": "own_pass_kernel", "achieved": own_gbs, "peak": hbm,
                     "unit": "GB/s", "frac": own_gbs / hbm, "peak_source": peak_src,
                     "traffic": traffic_for("own_pass", own_units), "algorithmic_bytes": own_b, "ms": t_own},
        "kernels": {
            "prefix_pass": {"ms": t_pre, "achieved_gbs": pre_gbs, "frac_hbm": pre_gbs / hbm,
                            "algorithmic_bytes": pre_b, "algorithmic_flops": pre_fl,
                            "achieved_tflops": pre_fl / (t_pre * 1e-3) / 1e12,
                            "frac_tensor": pre_fl / (t_pre * 1e-3) / 1e12 / tf_sus,
                            "bound_time_ms": max(pre_b / (hbm * 1e9), pre_fl / (tf_sus * 1e12)) * 1e3,
                            "traffic": traffic_for("prefix_pass", sum(max(p.branch_prefix_len or [0]) for p in dw.pages))},
            "own_pass": {"ms": t_own, "achieved_gbs": own_gbs, "frac_hbm": own_gbs / hbm,
                         "algorithmic_bytes": own_b},
            "decode_step": {"ms": t_dec, "achieved_gbs": dec_gbs, "frac_hbm": dec_gbs / hbm,
                            "frac_spec_8tbs": dec_gbs / 8000.0, "algorithmic_bytes": all_b,
                            "algorithmic_flops": dec_fl, "frac_tensor": dec_fl / (t_dec * 1e-3) / 1e12 / tf_sus,
                            "bound_time_ms": max(all_b / (hbm * 1e9), dec_fl / (tf_sus * 1e12)) * 1e3},
        },
        "forward": {"ms": t_fwd, "tflops": fwd_tf * world, "tflops_per_gpu": fwd_tf, "bound": "tensor",
                    "peak": tf_sus, "peak_kind": "bf16 sustained " + peak_src, "frac": fwd_tf / tf_sus,
                    "frac_spec_2250": fwd_tf / 2250.0, "algorithmic_flops": fl,
                    "executed_flops": fwd_ex, "executed_frac": fwd_ex / (t_fwd * 1e-3) / 1e12 / tf_sus,
                    "traffic": traffic_for("forward", fw.n_tokens)},
        "backward": {"ms": t_bwd, "tflops": bwd.flops / (t_bwd * 1e-3) / 1e12 * world,
                     "tflops_per_gpu": bwd.flops / (t_bwd * 1e-3) / 1e12, "bound": "tensor", "peak": tf_sus,
                     "peak_kind": "bf16 sustained " + peak_src,
                     "frac": bwd.flops / (t_bwd * 1e-3) / 1e12 / tf_sus, "algorithmic_flops": bwd.flops,
                     "what": "dQ, dK, dV of the same forward (launches: row sums, dQ pass, dK/dV pass)",
                     "traffic": bwd_traffic(fw.n_tokens)},
        "gpu_launches": ((1 if dec._plan.fused() else 2) + (2 if acc is not None else 0) + 1 + 3) * K,
        "clocks": clk,
    }
    if dec._plan.fused():
        # the step is one kernel (the prefix pass call launches nothing)
        fused_gbs = all_b / (t_dec * 1e-3) / 1e9
        pre_units = sum(max(p.branch_prefix_len or [0]) for p in dw.pages)
        line["roofline"] = {"bound": "hbm", "kernel": "attn_tc_kernel<MODE_VERIFY>", "achieved": fused_gbs, "peak": hbm,
                            "unit": "GB/s", "frac": fused_gbs / hbm, "peak_source": peak_src,
                            "traffic": traffic_for("verify_fused", own_units + pre_units), "algorithmic_bytes": all_b,
                            "ms": t_dec}
        del line["kernels"]["prefix_pass"], line["kernels"]["own_pass"]
        line["kernels"]["fused_pass"] = {"ms": t_dec, "achieved_gbs": fused_gbs, "frac_hbm": fused_gbs / hbm,
                                         "algorithmic_bytes": all_b, "algorithmic_flops": dec_fl,
                                         "achieved_tflops": dec_fl / (t_dec * 1e-3) / 1e12}
        line["config"]["step"] = ("value and ms_per_step cover the decode step (one fused verify pass); the forward "
                                  "and its backward run in the same timed loop and are reported under 'forward' and "
                                  "'backward'")
    if acc is not None:
        acc_gbs = acc.bytes / (t_acc * 1e-3) / 1e9
        line["kernels"]["accept"] = {
            "ms": t_acc, "achieved_gbs": acc_gbs, "frac_hbm": acc_gbs / hbm, "algorithmic_bytes": acc.bytes,
            "traffic": traffic_for("accept", acc.nq * args.vocab),
            "vocab": args.vocab, "draft_nodes": acc.nq, "mean_accepted": acc.mean_accepted(),
            "what": "row argmax over every draft node's logits + greedy tree walk (tau 0.75)"}
        line["kernels"]["verify_step"] = {"ms": t_dec + t_acc, "tokens_per_s": nq * world / ((t_dec + t_acc) * 1e-3)}
    for i, name in enumerate(n for n in ("branch_decode", "verify") if n in side):
        sd = side[name]
        t_p, t_o, t_a = t_side[3 * i], t_side[3 * i + 1], t_side[3 * i + 2]
        rep = decode_report(sd["dec"], sd["w"], t_p, t_o, hbm, tf_sus)
        rep["workload"] = WORKLOADS["branch" if name == "branch_decode" else name]
        sw = sd["w"]
        own_units = sum(sum(pg.own_len) for pg in sw.pages)
        pre_units = sum(max(pg.branch_prefix_len or [0]) for pg in sw.pages)
        if "fused_pass" in rep:
            rep["fused_pass"]["traffic"] = traffic_for("verify_fused", own_units + pre_units)
        elif name == "verify":
            rep["own_pass"]["kernel"] = "own_kmajor_kernel"
            rep["own_pass"]["traffic"] = traffic_for("own_kmajor_verify", own_units)
            rep["prefix_pass"]["traffic"] = traffic_for("prefix_pass_verify", pre_units)
        else:
            rep["own_pass"]["kernel"] = "own_pass_kernel"
            rep["own_pass"]["traffic"] = traffic_for("own_pass", own_units)
            rep["prefix_pass"]["traffic"] = traffic_for("prefix_pass", pre_units)
        if "acc" in sd:
            a = sd["acc"]
            a_gbs = a.bytes / (t_a * 1e-3) / 1e9
            rep["accept"] = {"ms": t_a, "algorithmic_bytes": a.bytes, "achieved_gbs": a_gbs, "frac_hbm": a_gbs / hbm,
                             "vocab": args.vocab, "draft_nodes": a.nq, "mean_accepted": a.mean_accepted(),
                             "traffic": traffic_for("accept", a.nq * args.vocab)}
            t_v = rep["step"]["ms"] + t_a
            rep["verify_step"] = {"ms": t_v, "tokens_per_s": sd["dec"].nq * world / (t_v * 1e-3),
                                  "what": ("fused verify pass" if "fused_pass" in rep else "prefix pass + own pass") +
                                          " + accept (row argmax, tree walk at tau 0.75)"}
        line["kernels"][name] = rep
    if side:
        # branch decode: prefix + own pass; verify: the fused pass (or prefix + own pass) + row argmax + tree walk
        n_side = 2 * ("branch_decode" in side)
        if "verify" in side:
            n_side += (1 if side["verify"]["dec"]._plan.fused() else 2) + 2
        line["gpu_launches"] += n_side * K
    if e2e:
        line["e2e"] = e2e
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
