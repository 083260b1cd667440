"""GPU parity: chain speculative sampling and greedy verification against
the float64 oracle, through the C ABI (libspecverify.so).

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §1.  Decisions must match the oracle except at
near-ties the oracle flags; diag probabilities within 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_sampling_gb300 as sv
import workloads
from conftest import load_golden
from gpu_util import (assert_chain_parity, compare_chain, compare_exact, host, max_near, oracle_chain,
                      oracle_chain_all, run_chunks)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(autouse=True, scope="module")
def _built():
    sv.build()
    sv.set_tuning(0, 0)
    yield
    sv.set_tuning(0, 0)


def _ws_ok(r):
    assert sv.workspace_error(r.ws) == 0


# ---------------------------------------------------------------------------
# the page's worked example: A B C D -> A B R, NaN rows never read
# ---------------------------------------------------------------------------
def test_worked_example_on_gpu():
    g = load_golden("worked_example_abcd.json")
    K, V = g["K"], g["V"]
    lg = torch.tensor(g["logits"]).view(1, K + 1, V).to(DEV)
    q = torch.tensor(g["q"]).view(1, K, V).to(DEV)
    d = torch.tensor([g["draft"]], dtype=torch.int32, device=DEV)
    for us in g["uniform_sets"]:
        u = torch.tensor([us], dtype=torch.float32, device=DEV)
        r = sv.verify_chain(lg, q, d, u, 1.0, 0, diag=True)
        assert r.tokens[0].tolist() == g["expected_tokens"]
        assert int(r.num_accepted[0]) == g["expected_num_accepted"]
        assert int(r.status[0]) == g["expected_status"]
        _ws_ok(r)


# ---------------------------------------------------------------------------
# parity on each workload family, shrunk so the oracle finishes in seconds
# while rows still span several slices and end in a ragged tail
# ---------------------------------------------------------------------------
CASES = [
    ("chain_small", {}, 0),
    ("chain_small", dict(B=64, V=1000), 1),
    ("eagle3", dict(B=24, V=50021), 0),
    ("eagle3", dict(B=16, K=5, V=12345), 1),
    ("dflash", dict(B=24, V=40001), 0),
    ("dflash", dict(B=12, K=8, V=151936), 1),
    ("dspark", dict(B=24, V=30011), 0),
]


@pytest.mark.parametrize("name,over,seed_off", CASES)
@pytest.mark.parametrize("slices", [0, 1, 2, 3])
def test_chain_parity(name, over, seed_off, slices):
    sv.set_tuning(slices, 0)
    w = workloads.make_chain(name, device=DEV, seed=workloads.seed_of(name) + 17 * seed_off, **over)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, diag=True)
    torch.cuda.synchronize()
    ref = oracle_chain(w)
    assert_chain_parity(r, ref, w.K, draft=w.draft)
    _ws_ok(r)
    sv.set_tuning(0, 0)


@pytest.mark.parametrize("name,over", [("chain_small", {}), ("eagle3", dict(B=24, V=50021)),
                                       ("dflash", dict(B=16, V=40001))])
def test_greedy_parity(name, over):
    w = workloads.make_chain(name, device=DEV, **over)
    draft = w.draft_greedy if w.draft_greedy is not None else w.draft
    # make some drafts match the target argmax so the walk goes deeper
    am = torch.argmax(w.logits[:, :w.K].float(), dim=-1).to(torch.int32)
    mix = torch.where(torch.rand(draft.shape, device=DEV) < 0.7, am, draft).contiguous()
    r = sv.verify_greedy(w.logits, mix)
    ref = oracle.verify_greedy(host(w.logits), host(mix))
    compare_exact(r.tokens, r.num_accepted, ref)
    assert np.array_equal(r.status.cpu().numpy(), ref["status"])
    _ws_ok(r)


def test_greedy_bf16_ties_lowest_index():
    B, K, V = 32, 3, 4099
    base = torch.randint(0, 5, (B, K + 1, V), device=DEV).float()   # massive exact ties
    lg = base.to(torch.bfloat16)
    am = torch.argmax(base[:, :K], dim=-1).to(torch.int32)          # torch: first maximal index
    r = sv.verify_greedy(lg, am.contiguous())
    ref = oracle.verify_greedy(host(lg), host(am))
    compare_exact(r.tokens, r.num_accepted, ref)
    assert (r.num_accepted.cpu().numpy() == K).all()


# ---------------------------------------------------------------------------
# full-size workloads, exactly the inputs the benchmark times (copy 0): every
# request compared with the oracle, near-ties counted and bounded
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["eagle3", "dflash"])
def test_chain_full_size_every_request(name):
    w = workloads.make_chain(name, device=DEV)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, diag=True)
    torch.cuda.synchronize()
    _ws_ok(r)
    ref = oracle_chain_all(w)
    near = assert_chain_parity(r, ref, w.K, draft=w.draft)
    print(f"{name}: {w.B} requests compared, {near} near-tie(s) excused")


def test_varying_scale_rows_after_a_dflash_call():
    """Rows whose logit scale and offset change from row to row (and from
    call to call): any threshold carried over from the previous row or the
    previous call on the same workspace is wrong.  Two calls in a row after a
    DFlash-like call, every request compared."""
    d = workloads.make_chain("dflash", device=DEV)          # same (B, K, V, top_k): same workspace size
    r0 = sv.verify_chain(d.logits, d.q, d.draft, d.uniforms, d.temperature, d.top_k)
    del d
    for seed_off in (0, 1):
        w = workloads.make_chain("dflash_vs", device=DEV, seed=workloads.seed_of("dflash_vs") + seed_off)
        r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k, diag=True, ws=r0.ws)
        torch.cuda.synchronize()
        _ws_ok(r)
        ref = oracle_chain_all(w)
        near = assert_chain_parity(r, ref, w.K, draft=w.draft)
        print(f"dflash_vs call {seed_off}: {w.B} requests compared, {near} near-tie(s) excused")
        del w, r, ref


def test_greedy_full_size_every_request():
    w = workloads.make_chain("eagle3", device=DEV)
    r = sv.verify_greedy(w.logits, w.draft_greedy)
    lg, dg = host(w.logits), host(w.draft_greedy)
    ref = run_chunks(lambda a, b: oracle.verify_greedy(lg[a:b], dg[a:b]), w.B)
    compare_exact(r.tokens, r.num_accepted, ref)
    assert np.array_equal(r.status.cpu().numpy(), ref["status"])


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
def test_empty_batch_is_a_no_op():
    lg = torch.zeros((0, 3, 10), device=DEV)
    q = torch.zeros((0, 2, 10), device=DEV)
    d = torch.zeros((0, 2), dtype=torch.int32, device=DEV)
    u = torch.zeros((0, 3), device=DEV)
    r = sv.verify_chain(lg, q, d, u, 1.0, 0)
    assert r.tokens.shape == (0, 3)


@pytest.mark.parametrize("V", [1, 2, 3, 17, 64, 65])
@pytest.mark.parametrize("top_k", [0, 1, 2])
def test_tiny_vocabularies(V, top_k):
    g = torch.Generator(device=DEV)
    g.manual_seed(V * 7 + top_k)
    B, K = 40, 3
    lg = torch.randn((B, K + 1, V), generator=g, device=DEV) * 2
    q = torch.softmax(torch.randn((B, K, V), generator=g, device=DEV), -1)
    d = torch.multinomial(q.view(-1, V), 1, generator=g).view(B, K).to(torch.int32)
    u = torch.rand((B, K + 1), generator=g, device=DEV)
    r = sv.verify_chain(lg, q, d, u, 0.9, top_k, diag=True)
    ref = oracle.verify_chain(host(lg), host(q), host(d), host(u), 0.9, top_k)
    assert_chain_parity(r, ref, K, draft=d)


def test_k_zero_is_plain_sampling():
    w = workloads.make_chain("chain_small", device=DEV, K=0, B=32)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, 1.0, 0)
    ref = oracle_chain(w)
    assert_chain_parity(r, ref, 0, check_diag=False)
    assert (r.num_accepted == 0).all()


def test_strided_and_unaligned_rows_take_the_plain_path():
    w = workloads.make_chain("dflash", device=DEV, B=8, V=9001)
    # a row stride of V+3 elements breaks 16-byte alignment of every row
    big = torch.zeros((w.B, w.K + 1, w.V + 3), device=DEV)
    big[:, :, :w.V] = w.logits
    lg = big[:, :, :w.V]
    qb = torch.zeros((w.B, w.K, w.V + 1), device=DEV)
    qb[:, :, :w.V] = w.q
    q = qb[:, :, :w.V]
    r = sv.verify_chain(lg, q, w.draft, w.uniforms, w.temperature, w.top_k, diag=True)
    ref = oracle.verify_chain(host(w.logits), host(w.q), host(w.draft), host(w.uniforms), w.temperature, w.top_k)
    assert_chain_parity(r, ref, w.K, draft=w.draft)


def test_status_paths_match_oracle():
    w = workloads.make_chain("eagle3", device=DEV, B=12, V=5000)
    lg = w.logits.clone()
    q = w.q.clone()
    d = w.draft.clone()
    d[0, 0] = w.V + 5                       # out-of-range token
    d[1, 0] = -1
    q[2, 0, d[2, 0]] = 0.0                  # q(y) = 0
    lg[3, 0, 17] = float("nan")             # NaN in the first row
    lg[4, 1, :] = float("-inf")             # a row with no finite value
    lg[5, 2, 3] = float("inf")
    r = sv.verify_chain(lg, q, d, w.uniforms, w.temperature, 0, diag=True)
    ref = oracle.verify_chain(host(lg), host(q), host(d), host(w.uniforms), w.temperature, 0)
    bad, near = compare_chain(r, ref, w.K, check_diag=False)
    assert not bad, bad
    assert near <= max_near(w.B)
    st = r.status.cpu().numpy()
    assert st[0] & 8 and st[1] & 8 and st[3] & 1


def test_massive_ties_use_the_exact_path():
    B, K, V = 6, 2, 20000
    lg = torch.zeros((B, K + 1, V), device=DEV)             # every logit tied: S = whole vocabulary
    lg[1] = torch.randint(0, 3, (K + 1, V), device=DEV).float()
    q = torch.softmax(torch.randn((B, K, V), device=DEV), -1)
    d = torch.multinomial(q.view(-1, V), 1).view(B, K).to(torch.int32)
    u = torch.rand((B, K + 1), device=DEV)
    r = sv.verify_chain(lg, q, d, u, 1.0, 50, diag=True)
    ref = oracle.verify_chain(host(lg), host(q), host(d), host(u), 1.0, 50)
    assert_chain_parity(r, ref, K, draft=d)


def test_top1_equals_greedy_on_gpu():
    w = workloads.make_chain("dflash", device=DEV, B=32, V=30000)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, 1.0, 1)
    g = sv.verify_greedy(w.logits, w.draft)
    assert torch.equal(r.tokens, g.tokens) and torch.equal(r.num_accepted, g.num_accepted)


def test_rows_past_rejection_are_never_read():
    w = workloads.make_chain("dflash", device=DEV, B=16, V=40001)
    r = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)
    n = r.num_accepted.cpu().numpy()
    lg = w.logits.clone()
    q = w.q.clone()
    for b in range(w.B):
        if n[b] < w.K:                       # rejected at row n: rows n+1.. are dead
            lg[b, n[b] + 1:] = float("nan")
            q[b, n[b] + 1:] = float("nan")
    r2 = sv.verify_chain(lg, q, w.draft, w.uniforms, w.temperature, w.top_k)
    assert torch.equal(r.tokens, r2.tokens) and torch.equal(r.status, r2.status)


def test_broadcast_batch_stride_zero():
    V, K, B = 8, 2, 5000
    lg1 = torch.randn((1, K + 1, V), device=DEV)
    q1 = torch.softmax(torch.randn((1, K, V), device=DEV), -1)
    lg = lg1.expand(B, K + 1, V)
    q = q1.expand(B, K, V)
    d = torch.multinomial(q1[0], B, replacement=True).t().contiguous().to(torch.int32)
    u = torch.rand((B, K + 1), device=DEV)
    r = sv.verify_chain(lg, q, d, u, 1.0, 0)
    ref = oracle.verify_chain(host(lg1), host(q1), host(d), host(u), 1.0, 0, K=K, V=V,
                              l_strides=(0, V), q_strides=(0, V))
    assert_chain_parity(r, ref, K, check_diag=False, draft=d)


def test_repeated_calls_reuse_the_workspace():
    w = workloads.make_chain("dflash", device=DEV, B=16, V=20000)
    r1 = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)
    t1 = r1.tokens.clone()
    for _ in range(3):
        r2 = sv.verify_chain(w.logits, w.q, w.draft, w.uniforms, w.temperature, w.top_k)
        assert torch.equal(t1, r2.tokens)
