"""Benchmark: draft positions verified per second on one GB300, with the
achieved HBM bandwidth of the verification kernel against the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the verification hot path over one batch:
  dflash   (default) block-draft chain verify, B=256 K=8 V=151936 fp32,
           T=1, top-k 50 -- the chain-verification workload large enough
           to be bound by HBM bandwidth
  dflash_vs  the same shape, every row with its own logit scale and offset
  eagle3   chain verify B=64 K=3 V=128256 bf16, T=0.8
  eagle3_greedy  greedy verify on the same shape
  chain_small    chain verify B=4 K=4 V=1000
  ddtree   DDTree build (B=32, L=16, budget 64, V=151936) + tree walk
  dspark   DSpark verify length + ragged chain verify (B=512, Kmax=8, V=128256 bf16)
  eagle2   EAGLE-2 dynamic tree: six expansion steps + rerank (B=32, V=151936 fp32)

Inputs are seeded synthetic tensors (see workloads/), resident in HBM before
the timed region.  Successive steps rotate over 3 independently seeded input
copies, so no step re-reads rows the previous one left in L2 (each copy's
rows read per step exceed the 126 MB L2 for dflash/dspark).

The line also carries: `parity` -- every request of input copy 0 re-run on
the float64 oracle (threads over requests on the host cores) and compared
with the GPU's outputs; `cpu_baseline` -- that oracle timed on one thread and
on every host core; `e2e` -- the same step through the public API on
inputs in pinned host memory, which the kernels read in place over the
CPU-GPU link (only the rows the step needs cross it), with the results read
back to the host inside the timed region; `e2e_copy_all` -- the same with
every input copied to the device first.

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
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal


def kernel_source_hash():
    """Hash of the chain kernel's sources -- its translation unit and the
    headers it includes (ties a profile to the code it measured)."""
    import hashlib
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "speculative_decoding_draft_sampling_gb300", "csrc")
    files = [os.path.join(pkg, f) for f in ("spec_chain.cu", "spec_chain.cuh", "spec_engine.cuh", "spec_common.cuh",
                                             "spec_select.cuh")]
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
def chain_bytes(K, V, es, top_k, n, st, k=None):
    """Bytes a chain verify must move: logits rows 0..n_b of every request,
    a 32-byte sector per q(y) point read, the q values of the top-k set (or
    the whole q row without top-k) at a rejection, and the small per-request
    arrays (drafts, uniforms, outputs)."""
    n = np.asarray(n, np.int64)
    st = np.asarray(st)
    kk = np.full_like(n, K) if k is None else np.asarray(k, np.int64)
    B = n.shape[0]
    rej = (n < kk) & ((st & 1) == 0)
    q_pts = np.minimum(n + rej, kk)
    topk = 0 < top_k < V
    per_rej = (top_k * 32) if topk else V * 4
    small = B * (K * 4 + (K + 1) * 4 + (K + 1) * 4 + 8) + (B * 12 if k is not None else 0)
    return int((n + 1).sum() * V * es + q_pts.sum() * 32 + rej.sum() * per_rej + small)


def pinned(t):
    return t.cpu().pin_memory()


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
    nbytes = []
    for w, r in zip(ws, outs):
        n = r.num_accepted.cpu().numpy().astype(np.int64)
        if greedy:
            nbytes.append(int((n + 1).sum() * w.V * w.logits.element_size() + w.B * (w.K * 4 + (w.K + 1) * 4 + 8)))
        else:
            nbytes.append(chain_bytes(w.K, w.V, w.logits.element_size(), w.top_k, n, r.status.cpu().numpy()))

    def step(i):
        w, r = ws[i % copies], outs[i % copies]
        if greedy:
            sv.verify_greedy(w.logits, w.draft_greedy, out=r)
        else:
            sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, out=r)

    def e2e():
        w = ws[0]
        h_in = [pinned(t) for t in ([w.logits, w.draft_greedy] if greedy else [w.logits, w.draft, w.uniforms, w.q])]

        def call(x):
            if greedy:
                r = sv.verify_greedy(x[0], x[1])
            else:
                r = sv.verify_chain(x[0], x[3], x[1], x[2], w.temperature, w.top_k)
            return [r.tokens, r.num_accepted, r.status]
        return h_in, call

    w0 = ws[0]
    cfg = dict(workload=name + ("_greedy" if greedy else ""), B=w0.B, K=w0.K, V=w0.V,
               logits_dtype=str(w0.logits.dtype).replace("torch.", ""), temperature=w0.temperature,
               top_k=w0.top_k, mode="greedy" if greedy else "stochastic")
    return dict(step=step, positions=w0.B * w0.K, bytes=nbytes, cfg=cfg, inputs=ws, outs=outs,
                launches_per_step=1, e2e=e2e, dtype="f32" if w0.logits.dtype == torch.float32 else "bf16")


def tree_bytes(q_shape, budget, depth, walk_n, target_es):
    """DDTree step bytes: the q rows the best-first order consults (per
    request, up to the deepest kept depth, plus the next one unless the budget
    filled at that depth's first node or the depth limit), and the target rows
    on the walked path."""
    B, L, V = q_shape
    rows = 0
    for b in range(B):
        dmax = depth[b].max()
        first = int(np.argmax(depth[b] == dmax))
        rows += dmax if (first == budget - 1 or dmax == L) else dmax + 1
    return int(rows * V * 4 + (np.asarray(walk_n) + 1).sum() * V * target_es)


def make_tree_case(dev, copies):
    import workloads
    import speculative_decoding_draft_sampling_gb300 as sv
    ts = [workloads.make_tree("ddtree", device=dev, seed=workloads.seed_of("ddtree") + 100 * i) for i in range(copies)]
    trees = [sv.tree_build(t.q, t.budget) for t in ts]
    tls = [workloads.tree_target_logits(t, tr.depth) for t, tr in zip(ts, trees)]
    walks = [sv.verify_tree(tl, tr.token, tr.parent, tr.num_nodes, t.q.shape[1]) for t, tl, tr in zip(ts, tls, trees)]
    torch.cuda.synchronize()
    nbytes = [tree_bytes(t.q.shape, t.budget, tr.depth.cpu().numpy(), wk.num_accepted.cpu().numpy(),
                         tl.element_size()) for t, tr, wk, tl in zip(ts, trees, walks, tls)]
    L = ts[0].q.shape[1]

    def step(i):
        t, tr, tl, wk = ts[i % copies], trees[i % copies], tls[i % copies], walks[i % copies]
        sv.tree_build(t.q, t.budget, out=tr)
        sv.verify_tree(tl, tr.token, tr.parent, tr.num_nodes, L, out=wk)

    def e2e():
        t, tl = ts[0], tls[0]
        h_in = [pinned(t.q), pinned(tl)]

        def call(x):
            tr = sv.tree_build(x[0], t.budget)
            wk = sv.verify_tree(x[1], tr.token, tr.parent, tr.num_nodes, L)
            return [wk.tokens, wk.num_accepted, wk.path_nodes, wk.status]
        return h_in, call

    B, L, V = ts[0].q.shape
    cfg = dict(workload="ddtree", B=B, L=L, V=V, budget=ts[0].budget, q_dtype="float32", target_dtype="bfloat16")
    return dict(step=step, positions=B * (ts[0].budget - 1), bytes=nbytes, cfg=cfg, inputs=ts, outs=walks,
                trees=trees, target=tls, launches_per_step=2, e2e=e2e, dtype="f32+bf16")


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
        nbytes.append(chain_bytes(w.K, w.V, w.logits.element_size(), w.top_k, r.num_accepted.cpu().numpy(),
                                  r.status.cpu().numpy(), k=k) + w.B * w.K * (4 + 8))
        pos.append(int(k.sum()))

    def step(i):
        w, a, (pl, pq), r = ws[i % copies], lens[i % copies], packs[i % copies], outs[i % copies]
        sv.adaptive_len(w.conf, 1.0, 0.15, out=a)
        sv.verify_chain(pl, pq, w.draft, w.uniforms, w.temperature, w.top_k, k_per_req=a.k,
                        l_row_off=a.l_row_off, q_row_off=a.q_row_off, out=r)

    def e2e():
        # the target's rows arrive packed for the verify lengths the
        # confidences give (the same on the host and the device)
        w, (pl, pq) = ws[0], packs[0]
        h_in = [pinned(t) for t in (w.conf, pl, pq, w.draft, w.uniforms)]

        def call(x):
            a = sv.adaptive_len(x[0], 1.0, 0.15)
            r = sv.verify_chain(x[1], x[2], x[3], x[4], w.temperature, w.top_k, k_per_req=a.k,
                                l_row_off=a.l_row_off, q_row_off=a.q_row_off)
            return [r.tokens, r.num_accepted, r.status, a.k]
        return h_in, call

    w0 = ws[0]
    cfg = dict(workload="dspark", B=w0.B, Kmax=w0.K, V=w0.V, logits_dtype="bfloat16", temperature=1.0,
               top_k=w0.top_k, a=1.0, b=0.15, mode="adaptive ragged (compact)")
    return dict(step=step, positions=pos, bytes=nbytes, cfg=cfg, inputs=ws, outs=outs, lens=lens, packs=packs,
                launches_per_step=2, e2e=e2e, dtype="bf16")


def eagle_node_paths(token, parent, num_gen, b):
    """token path of every generated node of request b (host arrays)"""
    out = {0: ()}
    for i in range(1, int(num_gen[b])):
        out[i] = out[int(parent[b, i])] + (int(token[b, i]),)
    return out


class EagleInputs:
    """The conditional draft rows of every expansion step of an EAGLE-2
    tree: step s's rows q[s] [B, F_s, V] belong to the frontier that step
    s - 1 selected (found once by a first run, the same every run)."""

    def __init__(self, cfg, q, fronts):
        self.cfg = cfg
        self.q = q              # list of [B, F_s, V] tensors
        self.fronts = fronts    # list of (front [B, F_s] int32, num_front [B] int32) tensors
        self.B, self.V = cfg["B"], cfg["V"]
        self.K2, self.Fn, self.steps, self.N = cfg["K2"], cfg["Fn"], cfg["steps"], cfg["N"]
        self.G = 1 + self.K2 + (self.steps - 1) * self.Fn * self.K2


def eagle_rows_for(state_host, front, nfront, V, seed, dev):
    import workloads
    tok, par, ng = state_host
    paths = []
    for b in range(front.shape[0]):
        pb = eagle_node_paths(tok, par, ng, b)
        paths.append([pb[int(front[b, f])] if f < nfront[b] else None for f in range(front.shape[1])])
    return workloads.eagle2_rows(paths, V, seed, device=dev)


def make_eagle_case(dev, copies):
    import workloads
    import speculative_decoding_draft_sampling_gb300 as sv
    cfg = dict(workloads.DEFAULTS["eagle2"])
    B, V, K2, Fn, steps, N = cfg["B"], cfg["V"], cfg["K2"], cfg["Fn"], cfg["steps"], cfg["N"]
    G = 1 + K2 + (steps - 1) * Fn * K2
    seed = workloads.seed_of("eagle2")
    st = sv.eagle_state(B, G, dev)
    front = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    nf = torch.ones(B, dtype=torch.int32, device=dev)
    qs, fronts = [], []
    for _ in range(steps):
        q = eagle_rows_for((st.token.cpu().numpy(), st.parent.cpu().numpy(), st.num_gen.cpu().numpy()),
                           front.cpu().numpy(), nf.cpu().numpy(), V, seed, dev)
        qs.append(q)
        fronts.append((front, nf))
        front, nf, _ = sv.eagle_expand(q, st, front, nf, K2, Fn)
    inp = EagleInputs(cfg, qs, fronts)
    # preallocated outputs and workspaces: each step's calls are fixed
    outs_f = [(torch.empty((B, Fn), dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(steps)]
    ws = [sv.workspace(sv.lib().spec_eagle_expand_workspace_size(B, q.shape[1], K2), dev) for q in qs]
    tree = sv.eagle_rerank(st, N)
    torch.cuda.synchronize()
    rows = sum(int(fr[1].cpu().numpy().clip(0, q.shape[1]).sum()) for q, fr in zip(qs, fronts))
    nbytes = rows * V * 4 + B * G * (4 * 3 + 8) + B * N * (4 * 3 + 8 + 8)

    def step(i):
        st.num_gen.fill_(1)
        fr, n = fronts[0]
        for s in range(steps):
            fo, no, so = outs_f[s]
            sv.eagle_expand(qs[s], st, fr, n, K2, Fn, front_out=fo, num_front_out=no, status=so, ws=ws[s])
            fr, n = fo, no
        sv.eagle_rerank(st, N, out=tree)

    def e2e():
        h_in = [pinned(q) for q in qs]

        def call(x):
            s2 = sv.eagle_state(B, G, dev)
            fr, n = fronts[0]
            for s in range(steps):
                fr, n, _ = sv.eagle_expand(x[s], s2, fr, n, K2, Fn)
            t = sv.eagle_rerank(s2, N)
            return [t.token, t.parent, t.depth, t.num_nodes]
        return h_in, call

    ccfg = dict(workload="eagle2", B=B, V=V, steps=steps, children_per_node=K2, frontier=Fn, budget=N,
                q_dtype="float32", node_capacity=G)
    return dict(step=step, positions=B * (N - 1), bytes=[nbytes] * copies, cfg=ccfg, inputs=[inp], outs=[tree],
                state=st, launches_per_step=2 * steps + 1, e2e=e2e, dtype="f32")


WORKLOAD_CHOICES = ["dflash", "dflash_vs", "eagle3", "eagle3_greedy", "chain_small", "ddtree", "dspark", "eagle2"]


def make_case(name, dev, copies, over=None):
    """`over` shrinks or reshapes a chain workload (e.g. {"B": 64}) for sweeps;
    the default bench line always uses the workload's own sizes."""
    if name == "ddtree":
        return make_tree_case(dev, copies)
    if name == "dspark":
        return make_dspark_case(dev, copies)
    if name == "eagle2":
        return make_eagle_case(dev, copies)
    if name == "eagle3_greedy":
        return make_chain_case("eagle3", dev, copies, greedy=True, over=over)
    return make_chain_case(name, dev, copies, over=over)


# ---------------------------------------------------------------------------
# the float64 oracle: whole requests of input copy 0, on the host cores
# ---------------------------------------------------------------------------
def host_view(t: torch.Tensor) -> np.ndarray:
    """Host copy in the oracle's input format (bf16 as raw uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


class OracleJob:
    """Host copies of one input copy and the oracle for requests [lo, hi).

    `target` (DDTree) is the tree's target logits; `tree_depth` the depth
    array they were generated from.  Nothing here calls the CUDA library."""

    def __init__(self, name, w, target=None):
        self.name = name
        self.w = w
        if name == "eagle2":
            self.q = [host_view(q) for q in w.q]
            self.B, self.V = w.B, w.V
            self.per_req = w.N - 1
            return
        if name == "ddtree":
            self.q = host_view(w.q)
            self.tl = host_view(target)
            self.B, self.L, self.V = w.q.shape
            self.per_req = w.budget - 1
        else:
            self.lg, self.qq = host_view(w.logits), host_view(w.q)
            self.d = host_view(w.draft_greedy if name == "eagle3_greedy" else w.draft)
            self.u = host_view(w.uniforms)
            self.conf = host_view(w.conf) if w.conf is not None else None
            self.B, self.K, self.V = w.B, w.K, w.V
            self.per_req = None if name == "dspark" else w.K

    def run(self, lo, hi):
        import oracle
        w = self.w
        if self.name == "eagle2":
            st = oracle.eagle_init(hi - lo, w.G)
            fr = np.zeros((hi - lo, 1), np.int32)
            nf = np.ones(hi - lo, np.int32)
            for s in range(w.steps):
                fr, nf, _ = oracle.eagle_expand(self.q[s][lo:hi], st, fr, nf, w.K2, w.Fn)
            out = {f"tree_{k}": v for k, v in oracle.eagle_rerank(st, w.N).items()}
            out["positions"] = np.full(hi - lo, self.per_req, np.int64)
            return out
        if self.name == "ddtree":
            tr = oracle.tree_build(self.q[lo:hi], w.budget)
            wk = oracle.verify_tree(self.tl[lo:hi], tr["token"], tr["parent"], tr["num_nodes"], self.L)
            out = {f"tree_{k}": v for k, v in tr.items()}
            out.update(wk)
            out["positions"] = np.full(hi - lo, self.per_req, np.int64)
            return out
        if self.name == "eagle3_greedy":
            out = oracle.verify_greedy(self.lg[lo:hi], self.d[lo:hi])
            out["positions"] = np.full(hi - lo, self.K, np.int64)
            return out
        if self.name == "dspark":
            a = oracle.adaptive_len(self.conf[lo:hi], 1.0, 0.15)
            k = a["k"]
            lo_off = np.concatenate([[0], np.cumsum(k + 1)]).astype(np.int32)
            qo_off = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
            pl = np.concatenate([self.lg[j, :k[j - lo] + 1] for j in range(lo, hi)])
            pq = np.concatenate([self.qq[j, :k[j - lo]] for j in range(lo, hi)] + [np.zeros((1, self.V), np.float32)])
            out = oracle.verify_chain(pl, pq, self.d[lo:hi], self.u[lo:hi], w.temperature, w.top_k, K=self.K,
                                      V=self.V, k_per_req=k, l_row_off=lo_off, q_row_off=qo_off)
            out["k"] = k
            out["positions"] = k.astype(np.int64)
            return out
        out = oracle.verify_chain(self.lg[lo:hi], self.qq[lo:hi], self.d[lo:hi], self.u[lo:hi], w.temperature,
                                  w.top_k)
        out["positions"] = np.full(hi - lo, self.K, np.int64)
        return out


def run_threads(job, reqs, threads):
    """The oracle over the listed requests, one request per task on
    `threads` host threads (the oracle's C calls release the GIL).
    Returns (results in request order, positions, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda b: job.run(b, b + 1), reqs))
    el = time.perf_counter() - t0
    res = {k: np.concatenate([p[k] for p in parts]) for k in parts[0]} if parts else {}
    return res, int(res["positions"].sum()) if parts else 0, el


def cpu_baseline(job, budget_s=12.0):
    """The oracle as it stands on one thread (requests one by one for about
    budget_s/2 seconds) and on every host core (a pool over the next
    requests, about as long)."""
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    b, pos1 = 0, 0
    while b < job.B and time.perf_counter() - t0 < budget_s / 2:
        pos1 += int(job.run(b, b + 1)["positions"].sum())
        b += 1
    el1 = time.perf_counter() - t0
    n1 = b
    # all cores: as many requests as one thread did in its half, times the
    # cores (cycling over the batch)
    reqs = [(n1 + i) % job.B for i in range(max(cores, min(job.B * 4, n1 * cores)))]
    _, posn, eln = run_threads(job, reqs, cores)
    return dict(value=posn / eln, unit=UNIT, cores=cores, kind="oracle", cpu_model=cpu_model(),
                sample=f"{len(reqs)} whole requests of input copy 0 on {cores} host threads ({eln:.1f} s); "
                       f"float64 C oracle, one request per task",
                single_thread=dict(value=pos1 / el1, cores=1,
                                   sample=f"{n1} whole requests one by one ({el1:.1f} s)"))


def parity_report(case, job):
    """Every request of input copy 0 on the oracle (all host cores), compared
    with the GPU's outputs for the same inputs: decisions and tokens must be
    equal except at the near-ties the oracle flags."""
    name = case["cfg"]["workload"]
    ref, _, el = run_threads(job, list(range(job.B)), os.cpu_count() or 1)
    out = case["outs"][0]
    mism, near, flagged = 0, 0, 0
    if name == "eagle2":
        for k in ("token", "parent", "depth", "score", "num_nodes", "status"):
            g = getattr(out, k).cpu().numpy()
            mism += int((g != ref["tree_" + k]).reshape(g.shape[0], -1).any(1).sum())
    elif name == "ddtree":
        tr = case["trees"][0]
        for k in ("token", "parent", "depth", "score", "num_nodes", "status"):
            g = getattr(tr, k).cpu().numpy()
            mism += int((g != ref["tree_" + k]).reshape(g.shape[0], -1).any(1).sum())
        for k in ("tokens", "num_accepted", "path_nodes", "status"):
            g = getattr(out, k).cpu().numpy()
            mism += int((g != ref[k]).reshape(g.shape[0], -1).any(1).sum())
    else:
        tok = out.tokens.cpu().numpy()
        n = out.num_accepted.cpu().numpy()
        st = out.status.cpu().numpy()
        nt = ref.get("near_tie", np.zeros(job.B, np.uint32))
        flagged = int((nt != 0).sum())
        for b in range(job.B):
            same = n[b] == ref["num_accepted"][b] and (tok[b] == ref["tokens"][b]).all() and st[b] == ref["status"][b]
            if not same:
                if nt[b] != 0:
                    near += 1
                else:
                    mism += 1
        if name == "dspark":
            mism += int((case["lens"][0].k.cpu().numpy() != ref["k"]).sum())
    return dict(requests=job.B, mismatches=mism, near_tie_mismatches=near, near_tie_flagged=flagged,
                oracle_s=round(el, 2))


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


def reference_job(name):
    """Inputs for the reference arm, built by the seeded generator and, where
    the method's own earlier step decides the layout (the DDTree target rows
    depend on the tree), by the oracle: the CUDA library is not used."""
    import workloads
    import oracle
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    if name == "eagle2":
        # the frontier of every step from the oracle itself
        cfg = dict(workloads.DEFAULTS["eagle2"])
        B, V, K2, Fn, steps, N = cfg["B"], cfg["V"], cfg["K2"], cfg["Fn"], cfg["steps"], cfg["N"]
        G = 1 + K2 + (steps - 1) * Fn * K2
        st = oracle.eagle_init(B, G)
        fr, nf = np.zeros((B, 1), np.int32), np.ones(B, np.int32)
        qs, fronts = [], []
        for _ in range(steps):
            q = eagle_rows_for((st["token"], st["parent"], st["num_gen"]), fr, nf, V, workloads.seed_of("eagle2"), dev)
            qs.append(q)
            fronts.append((fr, nf))
            fr, nf, _ = oracle.eagle_expand(host_view(q), st, fr, nf, K2, Fn)
        ccfg = dict(workload="eagle2", B=B, V=V, steps=steps, children_per_node=K2, frontier=Fn, budget=N,
                    q_dtype="float32", node_capacity=G)
        return OracleJob(name, EagleInputs(cfg, qs, fronts)), ccfg
    if name == "ddtree":
        t = workloads.make_tree("ddtree", device=dev)
        depth = oracle.tree_build(host_view(t.q), t.budget)["depth"]
        tl = workloads.tree_target_logits(t, torch.from_numpy(depth).to(dev))
        cfg = dict(workload="ddtree", B=t.q.shape[0], L=t.q.shape[1], V=t.q.shape[2], budget=t.budget,
                   q_dtype="float32", target_dtype="bfloat16")
        return OracleJob(name, t, tl), cfg
    base = "eagle3" if name == "eagle3_greedy" else name
    w = workloads.make_chain(base, device=dev)
    if name == "dspark":
        cfg = dict(workload="dspark", B=w.B, Kmax=w.K, V=w.V, logits_dtype="bfloat16", temperature=1.0,
                   top_k=w.top_k, a=1.0, b=0.15, mode="adaptive ragged (compact)")
    else:
        cfg = dict(workload=name, B=w.B, K=w.K, V=w.V, logits_dtype=str(w.logits.dtype).replace("torch.", ""),
                   temperature=w.temperature, top_k=w.top_k,
                   mode="greedy" if name == "eagle3_greedy" else "stochastic")
    return OracleJob(name, w), cfg


def run_reference(args, rank, world):
    """--impl reference: the float64 oracle on every host core, a bounded
    sample of whole requests of the same workload per step."""
    if rank != 0:
        return 0
    job, cfg = reference_job(args.workload)
    cores = os.cpu_count() or 1
    budget = max(1.0, min(6.0, 60.0 / max(1, args.steps)))
    # requests per step: about `budget` seconds on every core (from a probe)
    t0 = time.perf_counter()
    job.run(0, 1)
    per_req = max(1e-3, time.perf_counter() - t0)
    n = max(cores, int(budget / per_req * cores))
    vals, nreq = [], 0
    start = 1
    for i in range(args.warmup + args.steps):
        reqs = [(start + j) % job.B for j in range(n)]
        start = (start + n) % job.B
        _, pos, el = run_threads(job, reqs, cores)
        if i >= args.warmup:
            vals.append(pos / el)
            nreq = n
    val = statistics.mean(vals)
    line = dict(impl="reference", metric=METRIC, value=val, unit=UNIT, n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic (seeded)", config=cfg,
                cpu_baseline=dict(value=val, unit=UNIT, cores=cores, kind="oracle", cpu_model=cpu_model(),
                                  sample=f"{nreq} whole requests of the same workload per step, one per task "
                                         f"on {cores} host threads, float64 C oracle"),
                e2e=dict(value=val, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(case, steps, world=1):
    """The same step through the public API on inputs in pinned host memory,
    timed with its results read back to the host every step, two ways:

    - zero-copy (the reported `e2e`): the host tensors go to the call as they
      are and the kernels read them in place over the CPU-GPU link, so only
      the rows the step needs cross it (rows past a rejection stay on the
      host); `h2d_bytes_per_step` is the step's algorithmic bytes, the bytes
      the kernels read;
    - copy-all (`e2e_copy_all`): every input is first copied to device
      memory, then the call runs there; its bytes are the whole inputs.
    """
    h_in, call = case["e2e"]()
    d_in = [torch.empty_like(t, device=torch.device("cuda", torch.cuda.current_device())) for t in h_in]
    outs = call(d_in)
    h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    stream = torch.cuda.current_stream()

    def zero_copy():
        res = call(h_in)
        for h, o in zip(h_out, res):
            h.copy_(o, non_blocking=True)

    def copy_all():
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        res = call(d_in)
        for h, o in zip(h_out, res):
            h.copy_(o, non_blocking=True)

    def timed(one):
        one()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            one()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    pos = case["positions"]
    pos0 = pos[0] if isinstance(pos, list) else pos
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    ms_zc = max_over_ranks(timed(zero_copy), world)
    ms_cp = max_over_ranks(timed(copy_all), world)
    whole = sum(t.numel() * t.element_size() for t in h_in)
    zc = dict(value=pos0 * world / (ms_zc / 1e3), unit=UNIT, h2d_bytes_per_step=int(case["bytes"][0]),
              d2h_bytes_per_step=int(d2h), ms_per_step=ms_zc,
              mode="zero-copy: the kernels read the pinned host inputs in place over NVLink-C2C; "
                   "h2d bytes = the rows and values they read")
    cp = dict(value=pos0 * world / (ms_cp / 1e3), unit=UNIT, h2d_bytes_per_step=int(whole), d2h_bytes_per_step=int(d2h),
              ms_per_step=ms_cp, mode="copy-all: every input copied host -> device, then the call")
    return zc, cp


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dflash", choices=WORKLOAD_CHOICES)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls instead of CUDA-graph replays")
    ap.add_argument("--B", type=int, default=0, help="override the batch size of a chain workload (sweeps)")
    ap.add_argument("--slices", type=int, default=0, help="CTAs per cluster, one row slice each (0 = automatic)")
    ap.add_argument("--slots-per-cta", type=int, default=0, help="requests in flight per CTA (0 = automatic)")
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
    sv.set_tuning(args.slices, args.slots_per_cta)
    case = make_case(args.workload, dev, args.copies, over={"B": args.B} if args.B > 0 else None)
    step = case["step"]
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if not args.no_graph:
        # the steps as a serving loop issues them: each input copy's calls
        # captured once into a CUDA graph and replayed (the library's calls
        # are one memset and one kernel launch each, on the caller's stream)
        graphs = []
        cap_stream = torch.cuda.Stream()
        with torch.cuda.stream(cap_stream):
            for c in range(args.copies):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="thread_local"):
                    step(c)
                graphs.append(g)
        torch.cuda.synchronize()
        eager = step
        step = lambda i: graphs[i % args.copies].replay()
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

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

    e2e, e2e_copy = run_e2e(case, args.e2e_steps, world) if args.e2e_steps > 0 else (None, None)

    cpu = parity = None
    if rank == 0 and not (args.no_cpu_baseline and args.no_parity):
        job = OracleJob(args.workload, case["inputs"][0],
                        case["target"][0] if args.workload == "ddtree" else None)
        if not args.no_parity:
            parity = parity_report(case, job)
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(job)

    if rank == 0:
        cfg = dict(case["cfg"])
        cfg.update(parallelism=f"dp{world}", l2=f"steps rotate over {args.copies} seeded input copies",
                   bytes_per_step=int(bytes_step),
                   launch="eager calls" if args.no_graph else "CUDA-graph replay of the library calls")
        line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
                    ms_per_step=ms_per_step, higher_is_better=True, scaling="weak", vs_baseline=None,
                    dtype=case["dtype"], data="synthetic (seeded)", config=cfg,
                    roofline=dict(bound="hbm", achieved=achieved, peak=peak, unit="GB/s", frac=achieved / peak,
                                  traffic=profiled_traffic(args.workload, bytes_step), peak_kind=peak_kind,
                                  nominal_peak=NOMINAL_HBM_GBS, frac_of_nominal=achieved / NOMINAL_HBM_GBS),
                    parity=parity, cpu_baseline=cpu, e2e=e2e, e2e_copy_all=e2e_copy,
                    gpu_launches=args.steps * case["launches_per_step"],
                    clocks=clocks, wall_s=wall)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
