#!/usr/bin/env python
"""Decode-step benchmark of the persistent MoE decode megakernel.

Prints ONE JSON line on rank 0.  Default workload: the pages-scale synthetic MoE
(48 parallel attention+MoE layers, d 2048, 32/4 heads x 128, 128 experts top-8,
ffn 768, vocab 151936) at batch 1 with 8192 cached tokens, one decode step per
megakernel launch, inputs resident in HBM.  The per-step working set (~6.9 GB of
weights + KV) is far larger than the 129 MB L2, so no L2 flush is needed between
steps.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

N > 1 runs under torchrun as independent replicas (the step has no data-parallel
split; each rank decodes its own batch): value = all ranks' tokens / max-over-ranks
time.  `--impl reference` times the CPU oracle on the host cores: whole decode steps
of the same workload, over the benchmark's own inputs.
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

METRIC = "decode tok/s at bs1 & bs8; achieved HBM GB/s as % of weight+KV SoL"
UNIT = "tok/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--workload", default="pages_b1_8k")
    ap.add_argument("--mode", default="mega", choices=["mega", "perop", "graph"])
    ap.add_argument("--deterministic", action="store_true",
                    help="deterministic steps (fixed-point layer accumulators) for the main measurement")
    ap.add_argument("--lm-umma", action="store_true",
                    help="the LM head on the tcgen05 tensor cores (every handle of the run)")
    ap.add_argument("--ffn-umma", action="store_true",
                    help="with --lm-umma: the bf16 expert and dense-FFN items on the tensor cores too")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-baselines", action="store_true", help="skip per-op / graph arms")
    ap.add_argument("--no-bs8", action="store_true", help="skip the batch-8 ragged measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ablate-orders", default="",
                    help="comma-separated wave orders (letters r q a m o x: router, QKV, "
                         "attention, MoE items, O-proj, ADD_RMSNORM) to time one after another "
                         "on the same buffers, e.g. rqamox,qramox,rqaomx")
    ap.add_argument("--multistep", type=int, default=16,
                    help="also time greedy decode with this many steps per launch (tokens fed "
                         "back on the device); 0 skips it")
    ap.add_argument("--no-long", action="store_true", help="skip the batch-1 128K-context measurement")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-expert batch-8 measurement")
    ap.add_argument("--oracle-probe", default="", help=argparse.SUPPRESS)
    ap.add_argument("--trace", default="",
                    help="after timing, record one step's task timeline and write a per-opcode "
                         "summary (JSON) to this path")
    return ap.parse_args()


# ----------------------------------------------------------------------------- dist
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int, device="cuda") -> float:
    """Max of a per-rank value over all ranks (the slowest replica sets the time)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(",") for ln in self.f.read().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, spec sheet


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "persistent_moe_decode_cta_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except Exception:
        return None
    e = t.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def build_state(workload, seed, device, deterministic=False):
    import torch

    import synth
    from persistent_moe_decode_cta_gb300 import binding as B
    cfg = synth.model_config(workload)
    seq = synth.seq_lens_for(workload, seed)
    W = synth.make_weights(cfg, seed=seed, device=device)
    # a handle sized for the workload's batch where the packing depends on it (FP8 expert
    # items are 32 rows of d_ff below batch 4, 64 from 4 up)
    mk = B.Megakernel(cfg, W, max_batch=len(seq) if cfg.get("expert_dtype") == "fp8" else 8)
    if deterministic:
        mk.set_deterministic(True)
    st = plan_workload(mk, cfg, workload, seq, seed, device)
    return cfg, mk, st, W


def plan_workload(mk, cfg, workload, seq, seed, device):
    import torch

    import synth
    pt, npages = synth.make_page_table(seq, steps=1, seed=seed)
    k, v = synth.make_kv(cfg, npages, seed=seed, device=device)
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=seed, device=device)
    pt_dev = torch.as_tensor(pt, device=device)
    mk.plan(seq, pt_dev, npages)
    mk.set_fixed(True)
    logits = torch.empty(len(seq), cfg["vocab"], device=device)
    return dict(seq=seq, pt=pt_dev, npages=npages, k=k, v=v, tokens=tokens, logits=logits,
                workload=workload)


def time_device(run_step, K, W, ws, stream):
    """W untimed steps; then K steps bracketed by barrier + synchronize, with CUDA
    events on the launching stream around every launch.  Returns (total_s,
    per-launch seconds)."""
    import torch
    for _ in range(W):
        run_step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # (an NVTX range around the timed steps: a profiler's launch list can be restricted
    # to it with `ncu --nvtx --nvtx-include "timed/"`)
    torch.cuda.nvtx.range_push("timed")
    t0.record(stream)
    for i in range(K):
        evs[i][0].record(stream)
        run_step()
        evs[i][1].record(stream)
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(ws)
    total = t0.elapsed_time(t1) / 1e3
    per = [a.elapsed_time(b) / 1e3 for a, b in evs]
    return total, per


OPNAMES = {1: "EMBED", 2: "QKV_PROJ", 3: "ROUTER", 4: "ATTN_DRAIN", 5: "MOE_DRAIN", 7: "O_PROJ",
           8: "LM_HEAD", 9: "ADD_RMSNORM"}


def task_trace_summary(mk, st, path):
    """One traced megakernel step: per opcode, the mean time a task spends waiting for
    its dependency, for its operands / first chunk, in its MMA loop and after it (us)."""
    import numpy as np
    import torch
    mk.trace_on(1 << 18)
    mk.step(st["tokens"], st["k"], st["v"], st["logits"])
    torch.cuda.synchronize()
    r = mk.trace_records().astype(np.int64)
    mk.trace_off()
    op = (r[:, 0] >> 8) & 0xFF
    t0 = r[:, 2].min()
    out = {"span_us": float((r[:, 7].max() - t0) / 1e3), "tasks": int(len(r)), "per_opcode": {}}
    for o in sorted(set(op.tolist())):
        m = op == o
        def mean(a, b):
            x = r[m, b] - r[m, a]
            x = x[(r[m, a] > 0) & (r[m, b] > 0)]
            return float(x.mean() / 1e3) if len(x) else None
        out["per_opcode"][OPNAMES.get(o, str(o))] = dict(
            n=int(m.sum()), dep_wait=mean(2, 3), operand_wait=mean(3, 4), loop=mean(4, 5),
            after_loop=mean(5, 7), total=mean(2, 7))
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    np.save(os.path.splitext(path)[0] + ".npy", r)
    return {"path": path, "span_us": out["span_us"]}


def union_sizes(mk, L):
    return [len(a) for a in mk.active()][:L]


# ----------------------------------------------------------------------------- CPU oracle
class OracleSteps:
    """Whole CPU-oracle decode steps of a workload (every layer, the full LM head) on
    the host cores, over the same inputs as the GPU arm: the benchmark's seeded weights
    and K/V (device tensors, copied to the host once, during an untimed first step) and
    its page table and tokens.  Without a GPU the weights and pages are drawn on the
    host from the same per-tensor seeds (other values, same shapes and distribution)."""

    def __init__(self, workload, seed, W=None, kv=None):
        import numpy as np  # noqa: F401

        import oracle
        import synth
        self.O = oracle
        self.workload = workload
        self.cfg = synth.model_config(workload)
        self.seq = synth.seq_lens_for(workload, seed)
        self.B = len(self.seq)
        self.pt, _ = synth.make_page_table(self.seq, steps=1, seed=seed)
        self.tokens = synth.make_tokens(self.B, self.cfg["vocab"], seed=seed).numpy()
        if W is not None:
            self.W = synth.HostWeights(W, cache_experts=True)
            self.kv = synth.HostKV(*kv, cache=True)
            self.source = "the benchmark's device weights and K/V, copied to the host once"
        else:
            self.W = synth.LazyHostWeights(self.cfg, seed)
            self.kv = synth.LazyHostKV(self.cfg, seed)
            self.source = "weights and K/V drawn on the host"
        self.step()            # untimed: brings every tensor the step reads to the host

    def step(self, n_layers=None):
        """Seconds of one decode step.  With n_layers, a bounded sample of it: the
        embedding, the first n_layers layers and the full LM head, each timed, the
        layers' time scaled to all of them (every layer has the same shapes)."""
        O, cfg = self.O, self.cfg
        L = cfg["n_layers"]
        if n_layers is None or n_layers >= L:
            t0 = time.perf_counter()
            O.decode_step(cfg, self.W, self.kv, self.tokens, self.seq, self.pt)
            return time.perf_counter() - t0
        t0 = time.perf_counter()
        x = O.embed(self.W, self.tokens)
        t1 = time.perf_counter()
        for l in range(n_layers):
            x, _ = O.layer_step(cfg, self.W, self.kv, l, x, self.seq, self.pt)
        t2 = time.perf_counter()
        O.lm_head(cfg, self.W, x)
        t3 = time.perf_counter()
        return (t1 - t0) + (t2 - t1) * L / n_layers + (t3 - t2)

    def describe(self, n, n_layers=None):
        L = self.cfg["n_layers"]
        if n_layers is None or n_layers >= L:
            return (f"{self.workload}: {n} whole float64 numpy oracle step(s) ({L} layers "
                    f"+ the full LM head, batch {self.B}) over {self.source}")
        return (f"{self.workload}: {n} sampled float64 numpy oracle step(s), each the embedding, the "
                f"first {n_layers} of {L} layers (time scaled by {L}/{n_layers}) and the full LM head, "
                f"batch {self.B}, over {self.source}")


def cpu_cores():
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(threads) if threads else os.cpu_count()


def oracle_probe(workload, steps):
    """Median seconds of `steps` whole oracle steps of a small workload (host-drawn
    inputs); run in a child process for the single-core measurement."""
    o = OracleSteps(workload, 0)
    return statistics.median(o.step() for _ in range(steps))


def small_configs_cpu(steps=3):
    """The tiny and small parity models, whole oracle steps, median of `steps`, with all
    cores and with one core (a child interpreter with one BLAS thread)."""
    out = {}
    for wl in ("tiny_b1_64", "small_b1_2k"):
        allc = oracle_probe(wl, steps)
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-probe", wl,
                            "--steps", str(steps)], env=env, capture_output=True, text=True, timeout=600)
        one = float(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
        out[wl] = {"tok_s_all_cores": 1.0 / allc, "tok_s_one_core": (1.0 / one) if one else None,
                   "cores": cpu_cores(), "steps": steps}
    return out


def run_reference(args, rank, ws):
    """The reference arm: the CPU oracle, as it stands, timed on the host cores with
    whole decode steps -- args.warmup untimed, then args.steps timed -- of the
    workload's batch, over the benchmark's own inputs."""
    if rank != 0:
        return 0
    W = kv = None
    try:
        import torch
        if torch.cuda.is_available():
            import synth
            cfg = synth.model_config(args.workload)
            seq = synth.seq_lens_for(args.workload, args.seed)
            W = synth.make_weights(cfg, seed=args.seed, device="cuda")
            _, npages = synth.make_page_table(seq, steps=1, seed=args.seed)
            kv = synth.make_kv(cfg, npages, seed=args.seed, device="cuda")
    except Exception:
        W = kv = None
    o = OracleSteps(args.workload, args.seed, W, kv)
    # whole steps while warm-up + timed steps fit the time budget; else each step is a
    # bounded sample of the layers (the first warm-up step, or one extra untimed step,
    # measures a whole step)
    budget_s = 150.0
    t_whole = o.step()
    n_steps = max(1, args.warmup + args.steps)
    n_layers = None
    if t_whole * n_steps > budget_s:
        n_layers = max(1, int(o.cfg["n_layers"] * budget_s / (n_steps * t_whole)))
    for _ in range(max(0, args.warmup - 1)):
        o.step(n_layers)
    per = [o.step(n_layers) for _ in range(args.steps)]
    step_s = statistics.mean(per)
    value = o.B / step_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "batch": o.B, "seq_lens": o.seq, "mode": "oracle"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": o.describe(args.steps, n_layers)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main
def main():
    args = parse_args()
    if args.oracle_probe:
        print(oracle_probe(args.oracle_probe, args.steps))
        return 0
    rank, ws, local = dist_init()
    if args.impl == "reference":
        return run_reference(args, rank, ws)

    import torch

    from persistent_moe_decode_cta_gb300 import binding as Bd
    from persistent_moe_decode_cta_gb300 import sol
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    stream = torch.cuda.current_stream()
    args.lm_umma = args.lm_umma or args.ffn_umma
    if args.lm_umma:
        os.environ["MK_LM_UMMA"] = "1"  # read by mk_create
    if args.ffn_umma:
        os.environ["MK_MOE_UMMA"] = "1"
    cfg, mk, st, W = build_state(args.workload, args.seed, device, deterministic=args.deterministic)
    B = len(st["seq"])
    full = args.workload == "pages_b1_8k"
    if not full:
        # the unpacked weights are only needed again to build the batch-8 handles and
        # for the CPU oracle's copy of the workload
        W = None
        torch.cuda.empty_cache()

    def step_mega():
        mk.step(st["tokens"], st["k"], st["v"], st["logits"])

    def step_perop():
        mk.step_perop(st["tokens"], st["k"], st["v"], st["logits"], use_graph=False)

    def step_graph():
        mk.step_perop(st["tokens"], st["k"], st["v"], st["logits"], use_graph=True)

    run = {"mega": step_mega, "perop": step_perop, "graph": step_graph}[args.mode]
    launches_per_step = 1 if args.mode == "mega" else mk.query(Bd.MK_Q_PEROP_LAUNCHES)
    clocks = ClockSampler(local)
    # warm-up outside the sampler, then the timed region with the sampler running
    run()
    torch.cuda.synchronize()
    status = mk.status()
    if status["code"] != 0:
        raise RuntimeError(f"device error: {status}")
    clocks.start()
    total_s, per = time_device(run, args.steps, args.warmup, ws, stream)
    ck = clocks.stop()
    status = mk.status()
    if status["code"] != 0:
        raise RuntimeError(f"device error: {status}")
    total_s = max_over_ranks(total_s, ws, device)
    ms_per_step = total_s / args.steps * 1e3
    value = ws * B * args.steps / total_s

    # algorithmic bytes of one step (union of routed experts read back from the GPU)
    us = union_sizes(mk, cfg["n_layers"])
    sb = sol.step_bytes(cfg, st["seq"], us)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    launch_s = statistics.mean(per) / launches_per_step if args.mode != "mega" else statistics.mean(per)
    achieved = sb["total"] / statistics.mean(per) / 1e9
    # (the committed DRAM counters were taken on the default kernel build)
    traffic = profiled_traffic(args.workload) if args.mode == "mega" and not (args.deterministic or args.lm_umma) else None
    sol_tok = sol.sol_tok_s(sb["total"], hbm * 1e9, B)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3" if cfg.get("expert_dtype") == "fp8" else "bf16",
            "data": "synthetic (seeded random bf16 weights ~N(0,0.02), K/V ~N(0,1))",
            "config": {"workload": args.workload, "batch": B, "seq_lens": st["seq"]
                       if B <= 8 else None, "mode": args.mode,
                       "l2": "per-step working set %.2f GB >> 129 MB L2; no flush" % (sb["total"] / 1e9),
                       "parallelism": f"replicas x{ws}",
                       **({"accumulators": "64-bit fixed point (deterministic)"} if args.deterministic else {}),
                       **({"lm_head": "tcgen05"} if args.lm_umma else {}),
                       **({"ffn": "tcgen05"} if args.ffn_umma else {})},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": traffic,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": sb["total"],
                         "launch_ms": launch_s * 1e3},
            "sol": {"bytes_per_step": sb["total"], "weights": sb["weights"], "kv": sb["kv"],
                    "writes": sb["writes"], "sol_tok_s": sol_tok,
                    "frac_of_sol": value / ws / sol_tok,
                    # against the spec-sheet HBM3e bandwidth instead of the measured copy
                    "nominal_hbm_gbs": NOMINAL_HBM_GBS,
                    "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
                    "union_experts_mean": statistics.mean(us)},
            "clocks": ck}

    # ---- end to end through the C ABI with host buffers (copies inside the timed region)
    if not args.no_e2e and args.mode == "mega":
        tok_h = st["tokens"].cpu().pin_memory()
        log_h = torch.empty(B, cfg["vocab"], dtype=torch.float32).pin_memory()
        for _ in range(args.warmup):
            mk.step_host(tok_h, st["k"], st["v"], log_h)
        barrier(ws)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            mk.step_host(tok_h, st["k"], st["v"], log_h)
        el = max_over_ranks(time.perf_counter() - t0, ws, device)
        barrier(ws)
        line["e2e"] = {"value": ws * B * args.steps / el, "unit": UNIT,
                       "h2d_bytes_per_step": B * 4, "d2h_bytes_per_step": B * cfg["vocab"] * 4}

    # ---- greedy multi-step decode: n steps per launch, each step's token fed to the next
    # on the device (fixed positions, as above, so every step moves the same bytes)
    if args.multistep > 0 and args.mode == "mega":
        n = args.multistep
        tok_out = torch.empty(n, B, dtype=torch.int32, device=device)

        def step_multi():
            mk.steps(st["tokens"], n, st["k"], st["v"], st["logits"], tok_out)

        k2 = max(3, args.steps // n)
        t, _ = time_device(step_multi, k2, 2, ws, stream)
        t = max_over_ranks(t, ws, device)
        if mk.status()["code"] != 0:
            raise RuntimeError("device error in the multi-step arm")
        ms = {"steps_per_launch": n, "launches": k2, "value": ws * B * n * k2 / t, "unit": UNIT,
              "ms_per_step": t / (n * k2) * 1e3}
        if not args.no_e2e:
            # end to end: host tokens in and the n greedy tokens back, once per launch
            tok_h = st["tokens"].cpu().pin_memory()
            out_h = torch.empty(n, B, dtype=torch.int32).pin_memory()
            tok_d = torch.empty_like(st["tokens"])
            barrier(ws)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(k2):
                tok_d.copy_(tok_h, non_blocking=True)
                mk.steps(tok_d, n, st["k"], st["v"], st["logits"], tok_out)
                out_h.copy_(tok_out, non_blocking=True)
                torch.cuda.synchronize()
            el = max_over_ranks(time.perf_counter() - t0, ws, device)
            barrier(ws)
            ms["e2e"] = {"value": ws * B * n * k2 / el, "unit": UNIT, "h2d_bytes_per_launch": B * 4,
                         "d2h_bytes_per_launch": n * B * 4}
        line["multistep"] = ms

    # ---- wave-order ablation: the same step re-planned with each order (the order is a
    # plan-time property of the per-SM lists; outputs do not depend on it)
    if args.ablate_orders and args.mode == "mega":
        abl = {}
        k2 = max(5, args.steps // 4)
        for order in [o for o in args.ablate_orders.split(",") if o]:
            os.environ["MK_WAVE_ORDER"] = order
            mk.plan(st["seq"], st["pt"], st["npages"])
            mk.set_fixed(True)
            t, _ = time_device(step_mega, k2, 2, ws, stream)
            t = max_over_ranks(t, ws, device)
            if mk.status()["code"] != 0:
                raise RuntimeError(f"device error with wave order {order}")
            abl[order] = {"value": ws * B * k2 / t, "ms_per_step": t / k2 * 1e3}
        os.environ.pop("MK_WAVE_ORDER", None)
        mk.plan(st["seq"], st["pt"], st["npages"])
        mk.set_fixed(True)
        line["wave_order_ablation"] = abl

    if args.trace:
        line["trace"] = task_trace_summary(mk, st, args.trace)

    # ---- the same opcodes as separate launches, and as one CUDA graph
    if not args.no_baselines and args.mode == "mega":
        bl = {}
        for name, fn in (("perop", step_perop), ("graph", step_graph)):
            k2 = max(5, args.steps // 4)
            t, _ = time_device(fn, k2, 2, ws, stream)
            t = max_over_ranks(t, ws, device)
            bl[name] = {"value": ws * B * k2 / t, "ms_per_step": t / k2 * 1e3,
                        "launches_per_step": mk.query(Bd.MK_Q_PEROP_LAUNCHES)}
        if mk.status()["code"] != 0:
            raise RuntimeError("device error in per-op arms")
        line["baselines"] = bl

    # ---- CPU oracle baseline (rank 0, N = 1): whole oracle steps over this workload's
    # inputs, and the two small parity models with all cores and with one
    if not args.no_cpu and rank == 0 and ws == 1:
        o = OracleSteps(args.workload, args.seed, W, (st["k"], st["v"]))
        per = [o.step() for _ in range(2)]
        line["cpu_baseline"] = {"value": o.B / statistics.mean(per), "unit": UNIT, "cores": cpu_cores(),
                                "kind": "oracle", "sample": o.describe(len(per)),
                                "small_configs": small_configs_cpu()}
        del o

    # ---- batch 1 at the 128K context (131072 cached tokens): the same handle, re-planned
    if not args.no_long and full and args.mode == "mega":
        import synth
        wl5 = "pages_b1_128k"
        cfg5 = synth.model_config(wl5)
        seq5 = synth.seq_lens_for(wl5, args.seed)
        del st
        torch.cuda.empty_cache()
        st5 = plan_workload(mk, cfg5, wl5, seq5, args.seed, device)

        def step5():
            mk.step(st5["tokens"], st5["k"], st5["v"], st5["logits"])
        step5()
        k5 = max(10, args.steps // 2)
        t5, per5 = time_device(step5, k5, args.warmup, ws, stream)
        if mk.status()["code"] != 0:
            raise RuntimeError("device error in the 128K arm")
        t5 = max_over_ranks(t5, ws, device)
        sb5 = sol.step_bytes(cfg5, seq5, union_sizes(mk, cfg5["n_layers"]))
        ach5 = sb5["total"] / statistics.mean(per5) / 1e9
        line["long128k"] = {"workload": wl5, "value": ws * k5 / t5, "unit": UNIT, "ms_per_step": t5 / k5 * 1e3,
                            "bytes_per_step": sb5["total"], "achieved_gbs": ach5, "frac": ach5 / hbm,
                            "sol_tok_s": sol.sol_tok_s(sb5["total"], hbm * 1e9, 1)}
        del st5
        torch.cuda.empty_cache()

    # ---- batch 8, ragged lengths, sliding window on odd layers (same weights), in bf16
    # and with the routed experts stored as FP8
    if not args.no_bs8 and full:
        import synth
        wl8 = "pages_b8_ragged_swa"
        cfg8 = synth.model_config(wl8)
        seq8 = synth.seq_lens_for(wl8, args.seed)
        arms = [("bs8", cfg8)]
        if not args.no_fp8:
            arms.append(("fp8_b8", dict(cfg8, expert_dtype="fp8")))
        for key, c8 in arms:
            # the sliding window is a plan-time property of the layers: a handle of its own
            mk.close()
            torch.cuda.empty_cache()
            mk = Bd.Megakernel(c8, W, max_batch=8)
            st8 = plan_workload(mk, c8, wl8, seq8, args.seed, device)

            def step8():
                mk.step(st8["tokens"], st8["k"], st8["v"], st8["logits"])
            step8()
            k8 = max(10, args.steps // 2)
            t8, per8 = time_device(step8, k8, args.warmup, ws, stream)
            if mk.status()["code"] != 0:
                raise RuntimeError(f"device error in the {key} arm")
            t8 = max_over_ranks(t8, ws, device)
            us8 = union_sizes(mk, c8["n_layers"])
            sb8 = sol.step_bytes(c8, seq8, us8)
            ach8 = sb8["total"] / statistics.mean(per8) / 1e9
            line[key] = {"workload": wl8 + ("" if key == "bs8" else " (FP8 experts)"), "value": ws * 8 * k8 / t8,
                         "unit": UNIT, "ms_per_step": t8 / k8 * 1e3, "bytes_per_step": sb8["total"],
                         "achieved_gbs": ach8, "frac": ach8 / hbm,
                         "sol_tok_s": sol.sol_tok_s(sb8["total"], hbm * 1e9, 8),
                         "union_experts_mean": statistics.mean(us8), "seq_lens": seq8}
            del st8

    mk.close()
    del W
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
