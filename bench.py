"""Benchmark: draft positions verified per second on one GB300, with the
achieved HBM bandwidth of the verification kernel against the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the verification hot path over one batch:
  dflash   (default) block-draft chain verify, B=256 K=8 V=151936 fp32,
           T=1, top-k 50 -- the chain-verification workload large enough
           to be bound by HBM bandwidth
  eagle3   chain verify B=64 K=3 V=128256 bf16, T=0.8
  eagle3_greedy  greedy verify on the same shape
  chain_small    chain verify B=4 K=4 V=1000
  ddtree   DDTree build (B=32, L=16, budget 64, V=151936) + tree walk
  dspark   DSpark verify length + ragged chain verify (B=512, Kmax=8, V=128256 bf16)

Inputs are seeded synthetic tensors (see workloads/), resident in HBM before
the timed region.  Successive steps rotate over 3 independently seeded input
copies, so no step re-reads rows the previous one left in L2 (each copy's
rows read per step exceed the 126 MB L2 for dflash/dspark).

Multi-GPU (torchrun): every rank verifies its own batch (weak scaling, no
collective on the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

METRIC = "draft positions verified/sec; achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0


def kernel_source_hash():
    """Hash of the library's kernel and header sources (ties a profile to the code it measured)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "speculative_decoding_draft_sampling_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(pkg, "*.cu")) + glob.glob(os.path.join(pkg, "*.cuh"))
                   + glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, algorithmic_bytes):
    """DRAM bytes per launch from the committed ncu summary of the same kernel
    sources (scaled from its captured case by the bytes read), else None."""
    path = os.path.join(ROOT, "profiles", f"chain_kernel_{workload}_b64_full.md")
    if not os.path.exists(path):
        return None
    sha = ratio = None
    with open(path) as f:
        for line in f:
            t = line.strip()
            if t.startswith("source_sha256:"):
                sha = t.split(":", 1)[1].strip()
            elif t.startswith("traffic_ratio:"):
                ratio = float(t.split(":", 1)[1])
    if sha != kernel_source_hash() or ratio is None:
        return None
    return ratio * algorithmic_bytes


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"spec_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads: (setup) -> step callable, positions, algorithmic bytes
# ---------------------------------------------------------------------------
def chain_bytes(w, res):
    """Bytes a chain verify must move: logits rows 0..n_b of every request,
    a 32-byte sector per q(y) point read, the q values of the top-k set (or
    the whole q row without top-k) at a rejection, and the small arrays."""
    n = res.num_accepted.cpu().numpy().astype(np.int64)
    st = res.status.cpu().numpy()
    K, V, B = w.K, w.V, w.B
    es = w.logits.element_size()
    rows = n + 1
    rej = (n < K) & ((st & 1) == 0)
    q_pts = np.minimum(n + rej, K)
    topk = 0 < w.top_k < V
    per_rej = (w.top_k * 32) if topk else V * 4
    small = B * (K * 4 + (K + 1) * 4 + (K + 1) * 4 + 8)
    return int(rows.sum() * V * es + q_pts.sum() * 32 + rej.sum() * per_rej + small)


def make_chain_case(name, dev, copies, greedy=False, over=None):
    import workloads
    import speculative_decoding_draft_sampling_gb300 as sv
    ws = [workloads.make_chain(name, device=dev, seed=workloads.seed_of(name) + 100 * i, **(over or {}))
          for i in range(copies)]
    outs = []
    for w in ws:
        if greedy:
            outs.append(sv.verify_greedy(w.logits, w.draft_greedy))
        else:
            outs.append(sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k))
    torch.cuda.synchronize()
    if greedy:
        nbytes = []
        for w, r in zip(ws, outs):
            n = r.num_accepted.cpu().numpy().astype(np.int64)
            nbytes.append(int((n + 1).sum() * w.V * w.logits.element_size() + w.B * (w.K * 4 + (w.K + 1) * 4 + 8)))
    else:
        nbytes = [chain_bytes(w, r) for w, r in zip(ws, outs)]

    def step(i):
        w, r = ws[i % copies], outs[i % copies]
        if greedy:
            sv.verify_greedy(w.logits, w.draft_greedy, out=r)
        else:
            sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, out=r)

    w0 = ws[0]
    cfg = dict(workload=name + ("_greedy" if greedy else ""), B=w0.B, K=w0.K, V=w0.V,
               logits_dtype=str(w0.logits.dtype).replace("torch.", ""), temperature=w0.temperature,
               top_k=w0.top_k, mode="greedy" if greedy else "stochastic")
    return dict(step=step, positions=w0.B * w0.K, bytes=nbytes, cfg=cfg, inputs=ws, outs=outs,
                dtype="f32" if w0.logits.dtype == torch.float32 else "bf16")


def make_tree_case(dev, copies):
    import workloads
    import speculative_decoding_draft_sampling_gb300 as sv
    ts = [workloads.make_tree("ddtree", device=dev, seed=workloads.seed_of("ddtree") + 100 * i) for i in range(copies)]
    trees = [sv.tree_build(t.q, t.budget) for t in ts]
    tls = [workloads.tree_target_logits(t, tr.depth) for t, tr in zip(ts, trees)]
    walks = [sv.verify_tree(tl, tr.token, tr.parent, tr.num_nodes, t.q.shape[1]) for t, tl, tr in zip(ts, tls, trees)]
    torch.cuda.synchronize()
    nbytes = []
    for t, tr, wk, tl in zip(ts, trees, walks, tls):
        B, L, V = t.q.shape
        dep = tr.depth.cpu().numpy()
        rows = 0
        for b in range(B):
            dmax = dep[b].max()
            first = int(np.argmax(dep[b] == dmax))
            need = dmax if (first == t.budget - 1 or dmax == L) else dmax + 1
            rows += need
        walk_rows = int((wk.num_accepted.cpu().numpy() + 1).sum())
        nbytes.append(int(rows * V * 4 + walk_rows * V * tl.element_size()))

    def step(i):
        t, tr, tl, wk = ts[i % copies], trees[i % copies], tls[i % copies], walks[i % copies]
        sv.tree_build(t.q, t.budget, out=tr)
        sv.verify_tree(tl, tr.token, tr.parent, tr.num_nodes, t.q.shape[1], out=wk)

    B, L, V = ts[0].q.shape
    cfg = dict(workload="ddtree", B=B, L=L, V=V, budget=ts[0].budget, q_dtype="float32", target_dtype="bfloat16")
    return dict(step=step, positions=B * (ts[0].budget - 1), bytes=nbytes, cfg=cfg, inputs=ts, outs=walks,
                dtype="f32+bf16")


def make_dspark_case(dev, copies):
    import workloads
    import speculative_decoding_draft_sampling_gb300 as sv
    ws = [workloads.make_chain("dspark", device=dev, seed=workloads.seed_of("dspark") + 100 * i) for i in range(copies)]
    lens = [sv.adaptive_len(w.conf, 1.0, 0.15) for w in ws]
    packs = [workloads.pack_ragged(w.logits, w.q, a.k, a.l_row_off, a.q_row_off) for w, a in zip(ws, lens)]
    outs = [sv.verify_chain(pl, pq, w.draft, w.uniforms, w.temperature, w.top_k, k_per_req=a.k,
                            l_row_off=a.l_row_off, q_row_off=a.q_row_off)
            for w, a, (pl, pq) in zip(ws, lens, packs)]
    torch.cuda.synchronize()
    nbytes, pos = [], []
    for w, a, r in zip(ws, lens, outs):
        k = a.k.cpu().numpy().astype(np.int64)
        n = r.num_accepted.cpu().numpy().astype(np.int64)
        rej = n < k
        es = w.logits.element_size()
        nbytes.append(int((n + 1).sum() * w.V * es + (np.minimum(n + rej, k)).sum() * 32 + rej.sum() * w.top_k * 32
                          + w.B * (w.K * 4 * 2 + 8 * 3 + w.K * 8)))
        pos.append(int(k.sum()))

    def step(i):
        w, a, (pl, pq), r = ws[i % copies], lens[i % copies], packs[i % copies], outs[i % copies]
        sv.adaptive_len(w.conf, 1.0, 0.15, out=a)
        sv.verify_chain(pl, pq, w.draft, w.uniforms, w.temperature, w.top_k, k_per_req=a.k,
                        l_row_off=a.l_row_off, q_row_off=a.q_row_off, out=r)

    w0 = ws[0]
    cfg = dict(workload="dspark", B=w0.B, Kmax=w0.K, V=w0.V, logits_dtype="bfloat16", temperature=1.0,
               top_k=w0.top_k, a=1.0, b=0.15, mode="adaptive ragged (compact)")
    return dict(step=step, positions=pos, bytes=nbytes, cfg=cfg, inputs=ws, outs=outs, dtype="bf16")


def make_case(name, dev, copies, over=None):
    """`over` shrinks or reshapes a chain workload (e.g. {"B": 64}) for sweeps;
    the default bench line always uses the workload's own sizes."""
    if name == "ddtree":
        return make_tree_case(dev, copies)
    if name == "dspark":
        return make_dspark_case(dev, copies)
    if name == "eagle3_greedy":
        return make_chain_case("eagle3", dev, copies, greedy=True, over=over)
    return make_chain_case(name, dev, copies, over=over)


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def host_view(t: torch.Tensor) -> np.ndarray:
    """Host copy in the oracle's input format (bf16 as raw uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def oracle_sample(case, budget_s=12.0):
    import oracle
    name = case["cfg"]["workload"]
    t0 = time.perf_counter()
    done_pos = 0
    n_req = 0
    if name == "ddtree":
        t = case["inputs"][0]
        B = t.q.shape[0]
        b = 0
        while time.perf_counter() - t0 < budget_s and b < B:
            tr = oracle.tree_build(host_view(t.q[b:b + 1]), t.budget)
            tl = __import__("workloads").tree_target_logits(t, torch.from_numpy(tr["depth"]).to(t.q.device))
            oracle.verify_tree(host_view(tl[b:b + 1]), tr["token"], tr["parent"], tr["num_nodes"], t.q.shape[1])
            done_pos += t.budget - 1
            b += 1
            n_req += 1
    else:
        w = case["inputs"][0]
        B = w.B
        b = 0
        while time.perf_counter() - t0 < budget_s and b < B:
            sl = slice(b, b + 1)
            if name == "eagle3_greedy":
                oracle.verify_greedy(host_view(w.logits[sl]), host_view(w.draft_greedy[sl]))
            else:
                oracle.verify_chain(host_view(w.logits[sl]), host_view(w.q[sl]), host_view(w.draft[sl]),
                                    host_view(w.uniforms[sl]), w.temperature, w.top_k)
            done_pos += w.K
            b += 1
            n_req += 1
    el = time.perf_counter() - t0
    return done_pos / el, n_req, el


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, rank, world):
    """--impl reference: the float64 oracle on the host cores, bounded sample per step."""
    if rank != 0:
        return 0
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    case = make_case_cpu_or_gpu(args.workload, dev)
    vals = []
    for i in range(args.warmup + args.steps):
        v, n_req, el = oracle_sample(case, budget_s=max(1.0, min(6.0, 60.0 / max(1, args.steps))))
        if i >= args.warmup:
            vals.append(v)
    val = statistics.mean(vals)
    line = dict(impl="reference", metric=METRIC, value=val, unit=UNIT, n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=case["cfg"],
                cpu_baseline=dict(value=val, unit=UNIT, cores=1, kind="oracle",
                                  sample=f"whole requests of the same workload, ~{n_req} per step, single-threaded C"),
                e2e=dict(value=val, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def make_case_cpu_or_gpu(name, dev):
    if dev.type == "cuda":
        import speculative_decoding_draft_sampling_gb300 as sv
        sv.build()
        return make_case(name, dev, 1)
    raise SystemExit("the reference arm generates its inputs on the GPU; no GPU found")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dflash",
                    choices=["dflash", "eagle3", "eagle3_greedy", "chain_small", "ddtree", "dspark"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--B", type=int, default=0, help="override the batch size of a chain workload (sweeps)")
    ap.add_argument("--slices", type=int, default=0, help="slices per row (0 = automatic)")
    ap.add_argument("--ctas-per-sm", type=int, default=0, help="resident CTAs per SM (0 = occupancy limit)")
    args = ap.parse_args()
    rank, world, local = dist_setup()
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import speculative_decoding_draft_sampling_gb300 as sv
    if rank == 0 or world == 1:
        sv.build()
    barrier(world)
    sv.build()
    dev = torch.device("cuda", local)
    sv.set_tuning(args.slices, args.ctas_per_sm)
    case = make_case(args.workload, dev, args.copies, over={"B": args.B} if args.B > 0 else None)
    step = case["step"]
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # timed region: per-step events on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clk = ClockSampler(local)
    clk.start()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    clocks = clk.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_total = max_over_ranks(sum(step_ms), world)
    ms_per_step = ms_total / args.steps

    pos = case["positions"]
    pos_step = statistics.mean(pos[i % args.copies] for i in range(args.steps)) if isinstance(pos, list) else pos
    bytes_step = statistics.mean(case["bytes"][i % args.copies] for i in range(args.steps))
    value = pos_step * world / (ms_per_step / 1e3)
    peak, peak_kind = peaks()
    achieved = bytes_step / (statistics.mean(step_ms) / 1e3) / 1e9

    # end to end through the public API from pinned host buffers
    e2e = None
    if args.e2e_steps > 0 and args.workload not in ("ddtree", "dspark"):
        e2e = run_e2e(case, args.e2e_steps, args.workload == "eagle3_greedy")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n_req, el = oracle_sample(case, budget_s=15.0)
        cpu = dict(value=v, unit=UNIT, cores=1, kind="oracle",
                   sample=f"{n_req} whole requests of copy 0 run one by one by the single-threaded float64 C oracle "
                          f"({el:.1f} s)")

    if rank == 0:
        cfg = dict(case["cfg"])
        cfg.update(parallelism=f"dp{world}", l2=f"steps rotate over {args.copies} seeded input copies",
                   bytes_per_step=int(bytes_step))
        line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
                    ms_per_step=ms_per_step, higher_is_better=True, scaling="weak", vs_baseline=None,
                    dtype=case["dtype"], data="synthetic (seeded)", config=cfg,
                    roofline=dict(bound="hbm", achieved=achieved, peak=peak, unit="GB/s", frac=achieved / peak,
                                  traffic=profiled_traffic(args.workload, bytes_step), peak_kind=peak_kind),
                    cpu_baseline=cpu, e2e=e2e, gpu_launches=args.steps * (2 if args.workload in ("ddtree", "dspark") else 1),
                    clocks=clocks, wall_s=wall)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(case, steps, greedy):
    import speculative_decoding_draft_sampling_gb300 as sv
    w = case["inputs"][0]
    pin = lambda t: t.cpu().pin_memory()
    h_logits, h_draft, h_u = pin(w.logits), pin(w.draft_greedy if greedy else w.draft), pin(w.uniforms)
    h_q = None if greedy else pin(w.q)
    d_logits, d_draft, d_u = torch.empty_like(w.logits), torch.empty_like(w.draft), torch.empty_like(w.uniforms)
    d_q = None if greedy else torch.empty_like(w.q)
    B, K = w.B, w.K
    o_tok = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    o_n = torch.empty(B, dtype=torch.int32).pin_memory()
    o_st = torch.empty(B, dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream()

    def one():
        d_logits.copy_(h_logits, non_blocking=True)
        d_draft.copy_(h_draft, non_blocking=True)
        d_u.copy_(h_u, non_blocking=True)
        if greedy:
            r = sv.verify_greedy(d_logits, d_draft)
        else:
            d_q.copy_(h_q, non_blocking=True)
            r = sv.verify_chain(d_logits, d_q, d_draft, d_u, w.temperature, w.top_k)
        o_tok.copy_(r.tokens, non_blocking=True)
        o_n.copy_(r.num_accepted, non_blocking=True)
        o_st.copy_(r.status, non_blocking=True)

    one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(t.numel() * t.element_size() for t in (h_logits, h_draft, h_u) + (() if h_q is None else (h_q,)))
    d2h = sum(t.numel() * t.element_size() for t in (o_tok, o_n, o_st))
    return dict(value=B * K / (ms / 1e3), unit=UNIT, h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                ms_per_step=ms)


if __name__ == "__main__":
    sys.exit(main())
