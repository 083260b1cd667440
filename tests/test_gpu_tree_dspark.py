"""GPU parity: DDTree build and tree walk, DSpark verify length and the
ragged (compact) chain verify it feeds, against the float64 oracle through
the C ABI.

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §5 (DDTree, DSpark) and §9 (compact ragged verify).
Tree outputs and verify lengths are compared bit for bit: the GPU forms
Q(u) and the DSpark ratios with the same fp64 operations in the same order.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_sampling_gb300 as sv
import workloads
from gpu_util import assert_chain_parity, compare_exact, host, run_chunks

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TREE_KEYS = ("token", "parent", "depth", "score", "anc_mask", "num_nodes", "status")


@pytest.fixture(autouse=True, scope="module")
def _built():
    sv.build()
    sv.set_tuning(0, 0)
    yield
    sv.set_tuning(0, 0)


def _tree_np(t):
    out = {k: getattr(t, k).cpu().numpy() for k in TREE_KEYS}
    out["anc_mask"] = out["anc_mask"].view(np.uint64)
    return out


def _assert_tree_equal(gpu, ref, rows=None):
    for k in TREE_KEYS:
        a, b = gpu[k], ref[k]
        if rows is not None:
            a = a[rows]
        assert np.array_equal(a, b), k


# ---------------------------------------------------------------------------
# DDTree build
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,L,V,N", [(4, 6, 3000, 24), (8, 16, 20011, 64), (3, 4, 777, 2), (5, 3, 500, 1),
                                     (4, 16, 10007, 200), (2, 5, 64, 40)])
@pytest.mark.parametrize("slices", [0, 2])
def test_tree_build_parity(B, L, V, N, slices):
    sv.set_tuning(slices, 0)
    t = workloads.make_tree("ddtree", device=DEV, B=B, L=L, V=V, N=N, seed=B * 1000 + V)
    g = sv.tree_build(t.q, t.budget)
    ref = oracle.tree_build(host(t.q), t.budget)
    _assert_tree_equal(_tree_np(g), ref)
    assert sv.workspace_error(g.ws) == 0
    sv.set_tuning(0, 0)


def test_tree_build_ties_and_uniform_rows():
    B, L, V, N = 4, 5, 300, 30
    q = torch.randint(1, 4, (B, L, V), device=DEV).float()
    q[0] = 1.0
    q = (q / q.sum(-1, keepdim=True)).contiguous()
    g = sv.tree_build(q, N)
    ref = oracle.tree_build(host(q), N)
    _assert_tree_equal(_tree_np(g), ref)


def test_tree_build_stale_depth_hints():
    """The per-depth filter hints persist in the workspace across calls.  A
    call whose rows are much flatter at some depths and much sharper at
    others than the previous call's makes those hints wrong (too high: the
    row is read again unhinted; too low: many more candidates); the trees
    must still equal the oracle's."""
    B, L, V, N = 8, 6, 20011, 48
    t1 = workloads.make_tree("ddtree", device=DEV, B=B, L=L, V=V, N=N, seed=7)
    g1 = sv.tree_build(t1.q, N)
    _assert_tree_equal(_tree_np(g1), oracle.tree_build(host(t1.q), N))
    scale = torch.tensor([0.25, 2.5, 0.5, 2.0, 0.3, 3.0], device=DEV).view(1, L, 1)
    q2 = torch.softmax(t1.q_logits * scale, dim=-1).float().contiguous()
    for q in (q2, t1.q):                      # stale hints both ways, on the same workspace
        g = sv.tree_build(q, N, ws=g1.ws)
        _assert_tree_equal(_tree_np(g), oracle.tree_build(host(q), N))
        assert sv.workspace_error(g.ws) == 0


def test_tree_build_never_reads_past_needed_rows():
    t = workloads.make_tree("ddtree", device=DEV, B=8, L=16, V=20000, N=64)
    ref = oracle.tree_build(host(t.q), 64)
    q = t.q.clone()
    for b in range(8):
        q[b, ref["rows_needed"][b]:] = float("nan")
    g = sv.tree_build(q, 64)
    _assert_tree_equal(_tree_np(g), ref)


def _oracle_tree_all(qh, budget):
    out = run_chunks(lambda a, b: {k: v for k, v in oracle.tree_build(qh[a:b], budget).items()}, qh.shape[0], chunk=1)
    return out


def test_tree_build_full_size_every_request():
    t = workloads.make_tree("ddtree", device=DEV)
    g = _tree_np(sv.tree_build(t.q, t.budget))
    ref = _oracle_tree_all(host(t.q), t.budget)
    _assert_tree_equal(g, ref)
    assert (g["num_nodes"] == t.budget).all()


# ---------------------------------------------------------------------------
# tree walk
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,L,V,N", [(6, 6, 3000, 24), (8, 16, 20011, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tree_walk_parity(B, L, V, N, dtype):
    t = workloads.make_tree("ddtree", device=DEV, B=B, L=L, V=V, N=N)
    g = sv.tree_build(t.q, t.budget)
    ref_t = oracle.tree_build(host(t.q), t.budget)
    tl = workloads.tree_target_logits(t, g.depth, dtype=dtype)
    w = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, L)
    ref = oracle.verify_tree(host(tl), ref_t["token"], ref_t["parent"], ref_t["num_nodes"], L)
    for k in ("path_nodes", "tokens", "num_accepted", "status"):
        assert np.array_equal(getattr(w, k).cpu().numpy(), ref[k]), k
    assert sv.workspace_error(w.ws) == 0


def test_tree_walk_full_size_every_request():
    t = workloads.make_tree("ddtree", device=DEV)
    g = sv.tree_build(t.q, t.budget)
    tl = workloads.tree_target_logits(t, g.depth)
    w = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, 16)
    ref_t = _oracle_tree_all(host(t.q), t.budget)
    tlh = host(tl)
    ref = run_chunks(lambda a, b: oracle.verify_tree(tlh[a:b], ref_t["token"][a:b], ref_t["parent"][a:b],
                                                     ref_t["num_nodes"][a:b], 16), t.q.shape[0])
    for k in ("path_nodes", "tokens", "num_accepted", "status"):
        assert np.array_equal(getattr(w, k).cpu().numpy(), ref[k]), k
    assert (w.num_accepted.cpu().numpy() >= 1).mean() > 0.5     # the walk gets somewhere


def test_tree_walk_rows_off_path_never_read():
    t = workloads.make_tree("ddtree", device=DEV, B=6, L=6, V=3000, N=24)
    g = sv.tree_build(t.q, t.budget)
    tl = workloads.tree_target_logits(t, g.depth)
    w = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, 6)
    keep = torch.zeros(tl.shape[:2], dtype=torch.bool, device=DEV)
    pn = w.path_nodes.cpu().numpy()
    for b in range(6):
        for n in pn[b]:
            if n >= 0:
                keep[b, n] = True
    tl2 = tl.clone()
    tl2[~keep] = float("nan")
    w2 = sv.verify_tree(tl2, g.token, g.parent, g.num_nodes, 6)
    assert torch.equal(w.tokens, w2.tokens) and torch.equal(w.status, w2.status)


# ---------------------------------------------------------------------------
# stochastic tree walk
# ---------------------------------------------------------------------------
def _compare_walk(w, ref, B):
    """Every request equal to the oracle unless a draw sat within 1e-6 of a
    CDF boundary (counted, bounded)."""
    near = 0
    got = {k: getattr(w, k).cpu().numpy() for k in ("path_nodes", "tokens", "num_accepted", "status")}
    for b in range(B):
        same = all(np.array_equal(got[k][b], ref[k][b]) for k in got)
        if not same:
            assert ref["near_tie"][b] != 0, (b, {k: (got[k][b], ref[k][b]) for k in got})
            near += 1
    assert near <= max(2, B // 100), near
    return near


@pytest.mark.parametrize("B,L,V,N,dtype,T,top_k", [(8, 6, 3000, 24, torch.bfloat16, 1.0, 50),
                                                   (8, 6, 3000, 24, torch.float32, 0.9, 0),
                                                   (12, 16, 20011, 64, torch.bfloat16, 0.7, 20),
                                                   (32, 16, 151936, 64, torch.bfloat16, 1.0, 50)])
def test_tree_sample_parity(B, L, V, N, dtype, T, top_k):
    t = workloads.make_tree("ddtree", device=DEV, B=B, L=L, V=V, N=N)
    g = sv.tree_build(t.q, t.budget)
    tl = workloads.tree_target_logits(t, g.depth, dtype=dtype)
    u = workloads.tree_uniforms(t, L)
    w = sv.verify_tree_sample(tl, g.token, g.parent, g.num_nodes, u, L, T, top_k)
    torch.cuda.synchronize()
    assert sv.workspace_error(w.ws) == 0
    ref_t = oracle.tree_build(host(t.q), t.budget)
    tlh, uh = host(tl), host(u)
    ref = run_chunks(lambda a, b: oracle.verify_tree_sample(tlh[a:b], ref_t["token"][a:b], ref_t["parent"][a:b],
                                                            ref_t["num_nodes"][a:b], uh[a:b], L, T, top_k), B)
    near = _compare_walk(w, ref, B)
    print(f"tree sample B={B} V={V} top_k={top_k}: {near} near-tie(s) excused")


def test_tree_sample_top1_equals_greedy_walk_on_gpu():
    t = workloads.make_tree("ddtree", device=DEV, B=16, L=8, V=20011, N=48)
    g = sv.tree_build(t.q, t.budget)
    tl = workloads.tree_target_logits(t, g.depth, dtype=torch.float32)
    u = workloads.tree_uniforms(t, 8)
    s1 = sv.verify_tree_sample(tl, g.token, g.parent, g.num_nodes, u, 8, 1.0, 1)
    gw = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, 8)
    for k in ("path_nodes", "tokens", "num_accepted", "status"):
        assert torch.equal(getattr(s1, k), getattr(gw, k)), k


# ---------------------------------------------------------------------------
# accepted-path KV compaction
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,R,M", [(torch.bfloat16, 1024, 40), (torch.uint8, 37, 23), (torch.float32, 5, 17)])
def test_kv_compact_matches_oracle(dtype, R, M):
    """The KV rows of a real tree walk's accepted path, gathered into a
    cache at per-request positions; byte for byte against the oracle (a
    16-byte-aligned layout, and layouts that take 4-byte or byte copies)."""
    t = workloads.make_tree("ddtree", device=DEV, B=8, L=6, V=3000, N=24)
    g = sv.tree_build(t.q, t.budget)
    tl = workloads.tree_target_logits(t, g.depth)
    w = sv.verify_tree(tl, g.token, g.parent, g.num_nodes, 6)
    P, B, N = 5, 8, 24
    gen = torch.Generator(device=DEV)
    gen.manual_seed(R)
    src = torch.randint(0, 250, (P, B, N, R), generator=gen, device=DEV).to(dtype)
    dst = torch.randint(0, 250, (P, B, M, R), generator=gen, device=DEV).to(dtype)
    pos = torch.randint(0, M - 7 + 1, (B,), generator=gen, device=DEV, dtype=torch.int32)
    want = oracle.kv_compact(host(src), host(dst), host(w.path_nodes), host(w.num_accepted), dst_pos=host(pos))
    sv.kv_compact(src, dst, w.path_nodes, w.num_accepted, dst_pos=pos)
    torch.cuda.synchronize()
    assert np.array_equal(host(dst), want)


# ---------------------------------------------------------------------------
# DSpark verify length + ragged chain verify
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,Kmax", [(512, 8), (3, 1), (1000, 16), (7, 0)])
def test_adaptive_len_bit_exact(B, Kmax):
    g = torch.Generator(device="cpu")
    g.manual_seed(B + Kmax)
    c = torch.distributions.Beta(8.0, 2.0).sample((B, Kmax)).float()
    if B > 3:
        c[0] = 1.0
        c[1] = 0.0
    cg = c.to(DEV)
    a = sv.adaptive_len(cg, 1.0, 0.15)
    ref = oracle.adaptive_len(c.numpy(), 1.0, 0.15)
    assert np.array_equal(a.k.cpu().numpy(), ref["k"])
    assert np.array_equal(a.surv.cpu().numpy(), ref["surv"])
    assert np.array_equal(a.exp_adv.cpu().numpy(), ref["exp_adv"])
    assert np.array_equal(a.l_row_off.cpu().numpy(), ref["l_row_off"])
    assert np.array_equal(a.q_row_off.cpu().numpy(), ref["q_row_off"])


def _ragged(w, a):
    pl, pq = workloads.pack_ragged(w.logits, w.q, a.k, a.l_row_off, a.q_row_off)
    return pl, pq


@pytest.mark.parametrize("over", [dict(B=48, V=30011), dict()])
def test_ragged_verify_parity(over):
    """The DSpark workload (over={} is the full B=512, Kmax=8, V=128256
    configuration the benchmark times): verify lengths from the library, then
    the ragged chain verify; every request compared with the oracle, which
    packs its own rows from its own verify lengths."""
    w = workloads.make_chain("dspark", device=DEV, **over)
    a = sv.adaptive_len(w.conf, 1.0, 0.15)
    pl, pq = _ragged(w, a)
    r = sv.verify_chain(pl, pq, w.draft, w.uniforms, w.temperature, w.top_k,
                        k_per_req=a.k, l_row_off=a.l_row_off, q_row_off=a.q_row_off, diag=True)
    torch.cuda.synchronize()
    assert sv.workspace_error(r.ws) == 0
    aref = oracle.adaptive_len(host(w.conf), 1.0, 0.15)
    k = aref["k"]
    assert np.array_equal(a.k.cpu().numpy(), k)
    lh, qh, dh, uh = host(w.logits), host(w.q), host(w.draft), host(w.uniforms)

    def part(lo_b, hi_b):
        sel_k = k[lo_b:hi_b]
        lo = np.concatenate([[0], np.cumsum(sel_k + 1)]).astype(np.int32)
        qo = np.concatenate([[0], np.cumsum(sel_k)]).astype(np.int32)
        pl_h = np.concatenate([lh[j, :sel_k[j - lo_b] + 1] for j in range(lo_b, hi_b)])
        pq_h = np.concatenate([qh[j, :sel_k[j - lo_b]] for j in range(lo_b, hi_b)] + [np.zeros((1, w.V), np.float32)])
        return oracle.verify_chain(pl_h, pq_h, dh[lo_b:hi_b], uh[lo_b:hi_b], w.temperature, w.top_k,
                                   K=w.K, V=w.V, k_per_req=sel_k, l_row_off=lo, q_row_off=qo)

    ref = run_chunks(part, w.B)
    near = assert_chain_parity(r, ref, w.K, draft=w.draft)
    print(f"dspark {over}: {w.B} requests compared, {near} near-tie(s) excused")


@pytest.mark.parametrize("over", [dict(B=64, V=30011), dict()])
def test_cap_accept_parity(over):
    """Page §9's "cap-accept" mode: the dense rows of the full window, each
    request verifying and committing only its first k_b positions (k_b from
    the verify-length step); every request against the oracle."""
    w = workloads.make_chain("dspark", device=DEV, **over)
    a = sv.adaptive_len(w.conf, 1.0, 0.15)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, k_per_req=a.k, diag=True)
    torch.cuda.synchronize()
    assert sv.workspace_error(r.ws) == 0
    k = a.k.cpu().numpy()
    lh, qh, dh, uh = host(w.logits), host(w.q), host(w.draft), host(w.uniforms)
    ref = run_chunks(lambda lo, hi: oracle.verify_chain(lh[lo:hi], qh[lo:hi], dh[lo:hi], uh[lo:hi], w.temperature,
                                                        w.top_k, k_per_req=k[lo:hi]), w.B)
    assert_chain_parity(r, ref, w.K, draft=w.draft)
    g = sv.verify_greedy(w.logits, w.draft, k_per_req=a.k)
    gref = run_chunks(lambda lo, hi: oracle.verify_greedy(lh[lo:hi], dh[lo:hi], k_per_req=k[lo:hi]), w.B)
    compare_exact(g.tokens, g.num_accepted, gref)


@pytest.mark.parametrize("B,Kmax", [(512, 8), (1000, 16), (5, 0)])
def test_adaptive_len_table_bit_exact(B, Kmax):
    g = torch.Generator(device="cpu")
    g.manual_seed(7 * B + Kmax)
    c = torch.distributions.Beta(8.0, 2.0).sample((B, Kmax)).float()
    table = (torch.cumsum(torch.rand(Kmax + 1, generator=g, dtype=torch.float64) * 0.4 + 0.05, 0) + 0.5)
    a = sv.adaptive_len(c.to(DEV), 1.0, 0.15, cost=table.to(DEV))
    ref = oracle.adaptive_len(c.numpy(), 1.0, 0.15, cost=table.numpy())
    for key in ("k", "surv", "exp_adv", "l_row_off", "q_row_off"):
        assert np.array_equal(getattr(a, key).cpu().numpy(), ref[key]), key


def test_ragged_greedy_and_bad_lengths():
    w = workloads.make_chain("dspark", device=DEV, B=20, V=4099)
    k = torch.randint(0, w.K + 1, (w.B,), dtype=torch.int32)
    k[3] = w.K + 1                        # out of range
    k[4] = -2
    kk = k.clamp(0, w.K)
    lo = torch.zeros(w.B + 1, dtype=torch.int32)
    qo = torch.zeros(w.B + 1, dtype=torch.int32)
    lo[1:] = torch.cumsum(kk + 1, 0)
    qo[1:] = torch.cumsum(kk, 0)
    pl, pq = workloads.pack_ragged(w.logits, w.q, kk, lo, qo)
    kg, log, qog = k.to(DEV), lo.to(DEV), qo.to(DEV)
    r = sv.verify_chain(pl, pq, w.draft, w.uniforms, w.temperature, w.top_k, k_per_req=kg, l_row_off=log,
                        q_row_off=qog)
    ref = oracle.verify_chain(host(pl), host(pq), host(w.draft), host(w.uniforms), w.temperature, w.top_k,
                              K=w.K, V=w.V, k_per_req=k.numpy(), l_row_off=lo.numpy(), q_row_off=qo.numpy())
    assert_chain_parity(r, ref, w.K, check_diag=False)
    assert r.status[3].item() == 16 and r.status[4].item() == 16
    g = sv.verify_greedy(pl, w.draft, k_per_req=kg, l_row_off=log)
    gref = oracle.verify_greedy(host(pl), host(w.draft), K=w.K, V=w.V, k_per_req=k.numpy(), l_row_off=lo.numpy())
    compare_exact(g.tokens, g.num_accepted, gref)
