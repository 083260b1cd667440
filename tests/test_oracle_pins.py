"""Pins for the float64 oracle, against what the source page and mathematics
fix -- never against the oracle's own formulas.

Source page: "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
(chzhyang.github.io), §1 (acceptance rule, residual, bonus token, greedy
consistency, temperature/top-k folded into p), §5 (DDTree Q(u), best-first
heap, tree walk; DSpark s_j and expected advance).

Each pin is chosen so that a plausible slip in the oracle fails it: a ratio
written q/p, a dropped min, a residual taken as |p-q| or q-p, the wrong
uniform index, top-k ties dropped, temperature applied after truncation in a
way that changes S, a missing factor in Q(u), an off-by-one in depth or rank,
a wrong tie order in the heap, an inverted cost in DSpark.

Statistical tests use fixed seeds; their thresholds (p-value >= 1e-3 and
5-sigma binomial bands) are fixed here, not tuned after the fact.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

import oracle

from conftest import load_golden

# ---------------------------------------------------------------------------
# helpers: inputs whose target distribution is known by construction
# ---------------------------------------------------------------------------


def logits_for(p, T=1.0, excluded_gap=None):
    """Logits l with softmax(l/T) == p on supp(p).  Entries with p == 0 get
    -inf, or -- when ``excluded_gap`` is given -- a finite value that far below
    every kept entry, so that only the top-k truncation removes them."""
    p = np.asarray(p, np.float64)
    l = np.empty_like(p)
    kept = p > 0
    l[kept] = T * np.log(p[kept])
    l[~kept] = -np.inf if excluded_gap is None else l[kept].min() - excluded_gap
    return l.astype(np.float32)


def draw(rng, probs, n):
    """n iid draws from a discrete distribution (inverse CDF on numpy's own
    uniforms; independent of the oracle)."""
    c = np.cumsum(probs)
    c /= c[-1]
    return np.searchsorted(c, rng.random(n), side="right").astype(np.int32)


def chi2_pvalue(counts, probs):
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    sup = probs > 0
    assert counts[~sup].sum() == 0, "a token with zero target probability was committed"
    exp = probs[sup] / probs[sup].sum() * counts.sum()
    return stats.chisquare(counts[sup], exp).pvalue


# ---------------------------------------------------------------------------
# §1 worked example: drafts A B C D, commit A B R
# ---------------------------------------------------------------------------


def test_worked_example_abcd():
    g = load_golden("worked_example_abcd.json")
    K, V = g["K"], g["V"]
    logits = g["logits"].reshape(1, K + 1, V)
    q = g["q"].reshape(1, K, V)
    draft = np.array([g["draft"]], np.int32)
    for us in g["uniform_sets"]:
        out = oracle.verify_chain(logits, q, draft, np.array([us], np.float32),
                                  g["temperature"], g["top_k"])
        assert out["tokens"][0].tolist() == g["expected_tokens"], us
        assert out["num_accepted"][0] == g["expected_num_accepted"]
        assert out["status"][0] == g["expected_status"]     # NaN rows never read
        assert out["rows_read"][0] == 3


def test_worked_example_ragged_layout():
    g = load_golden("worked_example_abcd.json")
    K, V = g["K"], g["V"]
    out = oracle.verify_chain(g["logits"], g["q"], np.array([g["draft"]], np.int32),
                              np.array([g["uniform_sets"][3]], np.float32), 1.0, 0,
                              K=K, V=V, k_per_req=[K], l_row_off=[0, K + 1], q_row_off=[0, K])
    assert out["tokens"][0].tolist() == g["expected_tokens"]


# ---------------------------------------------------------------------------
# §1 acceptance rule: P(accept) = sum_x q(x) min(1, p(x)/q(x)) = sum min(p, q)
# ---------------------------------------------------------------------------


def test_acceptance_rate_is_one_minus_tv():
    rng = np.random.default_rng(7)
    p = np.array([0.30, 0.25, 0.15, 0.10, 0.08, 0.06, 0.04, 0.02])
    q = np.array([0.05, 0.10, 0.30, 0.20, 0.05, 0.10, 0.15, 0.05])
    n = 1_000_000
    logits = np.stack([logits_for(p), logits_for(p)])[None]          # [1, 2, 8]
    qa = q.astype(np.float32)[None, None]                            # [1, 1, 8]
    y = draw(rng, q, n)[:, None]
    u = rng.random((n, 2), dtype=np.float32)
    out = oracle.verify_chain(logits, qa, y, u, 1.0, 0, K=1, V=8,
                              l_strides=(0, 8), q_strides=(0, 8))
    acc = (out["num_accepted"] == 1).mean()
    expect = np.minimum(p, q).sum()                                  # 1 - TV(p, q)
    swapped = (q * np.minimum(1, q / p)).sum()                      # a q/p slip
    sig = math.sqrt(expect * (1 - expect) / n)
    assert abs(acc - expect) < 5 * sig, (acc, expect)
    assert abs(swapped - expect) > 20 * sig


# ---------------------------------------------------------------------------
# §1 distribution preservation, with temperature and top-k folded into p
# ---------------------------------------------------------------------------

P_ROWS = np.array([
    [0.40, 0.30, 0.20, 0.10, 0.00, 0.00],
    [0.00, 0.50, 0.25, 0.00, 0.15, 0.10],
    [0.25, 0.25, 0.00, 0.30, 0.20, 0.00],
    [0.10, 0.00, 0.45, 0.00, 0.25, 0.20],
])
Q_ROWS = np.array([
    [0.10, 0.10, 0.30, 0.30, 0.10, 0.10],
    [0.30, 0.20, 0.20, 0.10, 0.10, 0.10],
    [0.20, 0.40, 0.10, 0.10, 0.10, 0.10],
])


def _run_chain_trials(n, T, top_k, seed):
    rng = np.random.default_rng(seed)
    K, V = 3, 6
    # with top-k the zero-mass entries are finite and only truncation removes them
    gap = 1.0 if top_k else None
    logits = np.stack([logits_for(r, T=T, excluded_gap=gap) for r in P_ROWS])[None]   # [1, 4, 6]
    qa = Q_ROWS.astype(np.float32)[None]
    y = np.stack([draw(rng, Q_ROWS[i], n) for i in range(K)], 1)
    u = rng.random((n, K + 1), dtype=np.float32)
    return oracle.verify_chain(logits, qa, y, u, T, top_k, K=K, V=V,
                               l_strides=(0, V), q_strides=(0, V))


@pytest.mark.parametrize("T,top_k", [(1.0, 0), (0.7, 4)])
def test_committed_tokens_follow_target(T, top_k):
    n = 1_000_000
    out = _run_chain_trials(n, T, top_k, seed=11 if top_k else 12)
    tok, na = out["tokens"], out["num_accepted"]
    for pos in range(4):
        sel = na >= pos                      # the token at `pos` was committed
        c = np.bincount(tok[sel, pos], minlength=6)
        assert chi2_pvalue(c, P_ROWS[pos]) > 1e-3, (pos, c)


def test_residual_law_after_rejection():
    n = 1_000_000
    out = _run_chain_trials(n, 1.0, 0, seed=13)
    rej = out["num_accepted"] == 0
    r = np.maximum(P_ROWS[0] - Q_ROWS[0], 0.0)
    c = np.bincount(out["tokens"][rej, 0], minlength=6)
    assert chi2_pvalue(c, r) > 1e-3
    # the residual mass of the rejection row is the total variation distance
    R = out["diag"][rej, 0, 3]
    np.testing.assert_allclose(R, r.sum(), rtol=1e-6)


def test_markov_target_joint_over_rounds():
    """Repeated draft/verify rounds on a first-order Markov target reproduce
    the target's joint law of the first three tokens."""
    rng = np.random.default_rng(21)
    V, K, L, n = 4, 2, 3, 300_000
    P = np.array([[0.50, 0.20, 0.20, 0.10],
                  [0.10, 0.60, 0.10, 0.20],
                  [0.25, 0.25, 0.25, 0.25],
                  [0.05, 0.15, 0.30, 0.50],
                  [0.30, 0.30, 0.20, 0.20]])       # row 4 = start state
    Qd = np.array([[0.25, 0.25, 0.25, 0.25],
                   [0.40, 0.20, 0.20, 0.20],
                   [0.10, 0.10, 0.40, 0.40],
                   [0.30, 0.30, 0.30, 0.10],
                   [0.10, 0.60, 0.20, 0.10]])
    logP = np.log(P).astype(np.float32)
    seqs = [[] for _ in range(n)]
    active = np.arange(n)
    while active.size:
        prev = np.array([seqs[i][-1] if seqs[i] else 4 for i in active])
        y = np.empty((active.size, K), np.int32)
        ctx = prev.copy()
        for j in range(K):
            cs = np.cumsum(Qd[ctx], 1)
            y[:, j] = (rng.random(active.size)[:, None] >= cs).sum(1)
            ctx = y[:, j]
        rows_ctx = np.stack([prev, y[:, 0], y[:, 1]], 1)             # target context per row
        logits = logP[rows_ctx]                                      # [A, 3, 4]
        qa = Qd[np.stack([prev, y[:, 0]], 1)].astype(np.float32)     # [A, 2, 4]
        u = rng.random((active.size, K + 1), dtype=np.float32)
        out = oracle.verify_chain(logits, qa, y, u, 1.0, 0)
        keep = []
        for j, i in enumerate(active):
            m = out["num_accepted"][j] + 1
            seqs[i].extend(out["tokens"][j, :m].tolist())
            if len(seqs[i]) < L:
                keep.append(i)
        active = np.array(keep, dtype=np.int64)
    idx = np.array([s[0] * 16 + s[1] * 4 + s[2] for s in seqs])
    counts = np.bincount(idx, minlength=64)
    joint = np.array([P[4, a] * P[a, b] * P[b, c]
                      for a in range(4) for b in range(4) for c in range(4)])
    assert chi2_pvalue(counts, joint) > 1e-3


# ---------------------------------------------------------------------------
# §1 special cases that reduce to closed forms or to greedy decoding
# ---------------------------------------------------------------------------


def test_p_equals_q_always_accepts():
    rng = np.random.default_rng(3)
    n, K, V = 200_000, 3, 6
    logits = np.stack([logits_for(r) for r in P_ROWS])[None]
    qa = P_ROWS[:K].astype(np.float32)[None]
    y = np.stack([draw(rng, P_ROWS[i], n) for i in range(K)], 1)
    u = rng.random((n, K + 1), dtype=np.float32)
    out = oracle.verify_chain(logits, qa, y, u, 1.0, 0, K=K, V=V, l_strides=(0, V), q_strides=(0, V))
    # p/q == 1 up to float32 rounding of q: reject only if u lands in that sliver
    assert (out["num_accepted"] == K).mean() > 0.9999
    c = np.bincount(out["tokens"][out["num_accepted"] == K, K], minlength=6)
    assert chi2_pvalue(c, P_ROWS[3]) > 1e-3


def test_top1_stochastic_equals_greedy():
    rng = np.random.default_rng(5)
    B, K, V = 400, 4, 50
    logits = rng.permutation(np.arange(B * (K + 1) * V)).reshape(B, K + 1, V).astype(np.float32) / 100
    q = rng.dirichlet(np.ones(V), size=(B, K)).astype(np.float32)
    am = logits[:, :K].argmax(-1).astype(np.int32)
    draft = np.where(rng.random((B, K)) < 0.6, am, rng.integers(0, V, (B, K))).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    s = oracle.verify_chain(logits, q, draft, u, 1.0, 1)
    g = oracle.verify_greedy(logits, draft)
    np.testing.assert_array_equal(s["tokens"], g["tokens"])
    np.testing.assert_array_equal(s["num_accepted"], g["num_accepted"])


def test_tiny_temperature_equals_greedy():
    rng = np.random.default_rng(6)
    B, K, V = 200, 3, 40
    logits = (rng.permutation(B * (K + 1) * V).reshape(B, K + 1, V) * 0.1).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(B, K)).astype(np.float32)
    am = logits[:, :K].argmax(-1).astype(np.int32)
    draft = np.where(rng.random((B, K)) < 0.5, am, rng.integers(0, V, (B, K))).astype(np.int32)
    u = np.clip(rng.random((B, K + 1), dtype=np.float32), 1e-3, None)
    s = oracle.verify_chain(logits, q, draft, u, 1e-3, 0)
    g = oracle.verify_greedy(logits, draft)
    np.testing.assert_array_equal(s["tokens"], g["tokens"])


def test_one_hot_draft_with_zero_target_mass_always_rejects():
    V = 5
    logits = np.array([[logits_for([0.5, 0.5, 0, 0, 0], excluded_gap=30.0)] * 2], np.float32)
    q = np.zeros((1, 1, V), np.float32)
    q[0, 0, 3] = 1.0
    for u0 in (0.0, 0.3, 0.999):
        out = oracle.verify_chain(logits, q, np.array([[3]], np.int32),
                                  np.array([[u0, 0.25]], np.float32), 1.0, 2)
        assert out["num_accepted"][0] == 0
        assert out["tokens"][0, 0] == 0            # residual = p; u=0.25 -> token 0
        assert out["diag"][0, 0, 0] == 0.0         # p(y) = 0 outside the top-2 set


def test_normaliser_closed_forms_and_ties_kept():
    # weights 4,2,1,1 -> Z = (4+2+1+1)/4 = 2
    l = np.log(np.array([4, 2, 1, 1], np.float64)).astype(np.float32)
    logits = np.stack([l, l])[None]
    q = np.full((1, 1, 4), 0.25, np.float32)
    out = oracle.verify_chain(logits, q, np.array([[0]], np.int32),
                              np.array([[0.5, 0.5]], np.float32), 1.0, 0)
    np.testing.assert_allclose(out["diag"][0, 0, 2], 2.0, rtol=1e-7)
    # ties at the top-k threshold are kept: [3,2,2,2,1], k=2 -> S = {0,1,2,3}
    l = np.array([3, 2, 2, 2, 1], np.float32)
    logits = np.stack([l, l])[None]
    q = np.full((1, 1, 5), 0.2, np.float32)
    out = oracle.verify_chain(logits, q, np.array([[3]], np.int32),
                              np.array([[0.0, 0.5]], np.float32), 1.0, 2)
    np.testing.assert_allclose(out["diag"][0, 0, 2], 1 + 3 * math.exp(-1), rtol=1e-12)
    assert out["diag"][0, 0, 0] > 0                # token 3 is tied at tau: kept
    # temperature divides the logit gap: T = 2 -> Z = 1 + 3 e^{-1/2}
    out = oracle.verify_chain(logits, q, np.array([[3]], np.int32),
                              np.array([[0.0, 0.5]], np.float32), 2.0, 2)
    np.testing.assert_allclose(out["diag"][0, 0, 2], 1 + 3 * math.exp(-0.5), rtol=1e-12)


def test_residual_mass_closed_form():
    p = [0.5, 0.5, 0.0, 0.0]
    logits = np.stack([logits_for(p, excluded_gap=40.0)] * 2)[None]
    q = np.full((1, 1, 4), 0.25, np.float32)
    # draft token 2: p = 0 (with top-2), reject; R = sum [p-q]+ = 0.5
    out = oracle.verify_chain(logits, q, np.array([[2]], np.int32),
                              np.array([[0.1, 0.75]], np.float32), 1.0, 2)
    np.testing.assert_allclose(out["diag"][0, 0, 3], 0.5, rtol=1e-12)
    # residual is 0.25 on tokens 0 and 1; u*R = 0.375 -> token 1
    assert out["tokens"][0].tolist() == [1, -1]


def test_near_tie_flags_at_the_accept_boundary():
    """p = (1/2, 1/2) and q = (5/8, 3/8): drafting token 0 gives p/q = 4/5
    exactly.  |u - 4/5| = 5e-7 sets the position's near-tie bit; 5e-6 does not
    (the window is 1e-6); the decision itself follows u < p/q."""
    logits = np.zeros((1, 2, 2), np.float32)
    q = np.array([[[0.625, 0.375]]], np.float32)
    d = np.array([[0]], np.int32)
    for du, flagged in ((-5e-7, True), (5e-7, True), (-5e-6, False), (5e-6, False)):
        u0 = np.float32(0.8 + du)
        out = oracle.verify_chain(logits, q, d, np.array([[u0, 0.3]], np.float32), 1.0, 0)
        assert bool(out["near_tie"][0] & 1) == flagged, du
        assert out["num_accepted"][0] == (1 if du < 0 else 0), du
        assert not (out["near_tie"][0] >> 31), du     # the sample is far from its CDF edges


def test_near_tie_flags_at_a_cdf_boundary():
    """Position 0 always accepts (p = q); the bonus row has p = (1/4, 3/4),
    so its CDF boundary is 1/4.  u within 5e-7 of it sets bit 31, 5e-6 away
    does not; the token is 0 below the boundary and 1 above it."""
    logits = np.zeros((1, 2, 2), np.float32)
    logits[0, 1] = [0.0, np.log(3.0)]
    q = np.full((1, 1, 2), 0.5, np.float32)
    d = np.array([[1]], np.int32)
    for du, flagged in ((-5e-7, True), (5e-7, True), (-5e-6, False), (5e-6, False)):
        us = np.float32(0.25 + du)
        out = oracle.verify_chain(logits, q, d, np.array([[0.3, us]], np.float32), 1.0, 0)
        assert out["num_accepted"][0] == 1
        assert bool(out["near_tie"][0] >> 31) == flagged, du
        assert out["tokens"][0, 1] == (0 if du < 0 else 1), du
        assert not (out["near_tie"][0] & 1)
    # the residual's boundaries: a rejection whose residual is one token
    # (p = (1/2, 1/2), q = (5/8, 3/8): [p - q]_+ = (0, 1/8)) has its CDF edges
    # at 0 and R, i.e. at u = 0 and u = 1
    logits = np.zeros((1, 2, 2), np.float32)
    q = np.array([[[0.625, 0.375]]], np.float32)
    d = np.array([[0]], np.int32)
    for us, flagged in ((5e-7, True), (5e-6, False), (0.5, False)):
        out = oracle.verify_chain(logits, q, d, np.array([[0.9, us]], np.float32), 1.0, 0)
        assert out["num_accepted"][0] == 0 and out["tokens"][0, 0] == 1
        assert bool(out["near_tie"][0] >> 31) == flagged, us


def test_uniform_indexing_accept_vs_sample():
    """u[b, i] decides position i; u[b, k] drives the single sample."""
    p = [0.5, 0.5, 0.0, 0.0]
    logits = np.stack([logits_for(p, excluded_gap=40.0)] * 3)[None]
    q = np.array([[[0.25, 0.25, 0.25, 0.25], [0.25, 0.25, 0.25, 0.25]]], np.float32)
    d = np.array([[0, 1]], np.int32)
    # ratio = 2 at both positions: accepted; the bonus then uses u[2]
    out = oracle.verify_chain(logits, q, d, np.array([[0.99, 0.99, 0.2]], np.float32), 1.0, 2)
    assert out["tokens"][0].tolist() == [0, 1, 0]
    out = oracle.verify_chain(logits, q, d, np.array([[0.99, 0.99, 0.7]], np.float32), 1.0, 2)
    assert out["tokens"][0].tolist() == [0, 1, 1]


def test_status_bits():
    V = 4
    base = logits_for([0.4, 0.3, 0.2, 0.1])
    logits = np.stack([base, base, base])[None].copy()
    q = np.full((1, 2, V), 0.25, np.float32)
    u = np.array([[0.5, 0.5, 0.5]], np.float32)
    # drafted id out of range: flagged, rejected, correction sampled
    out = oracle.verify_chain(logits, q, np.array([[7, 0]], np.int32), u, 1.0, 0)
    assert out["status"][0] & oracle.ST_BAD_TOKEN and out["num_accepted"][0] == 0
    assert out["tokens"][0, 0] >= 0
    # q(y) = 0 with p(y) > 0: infinite ratio, accepted, flagged
    q0 = q.copy(); q0[0, 0] = [0.0, 1 / 3, 1 / 3, 1 / 3]
    out = oracle.verify_chain(logits, q0, np.array([[0, 0]], np.int32), u, 1.0, 0)
    assert out["status"][0] & oracle.ST_Q_ZERO and out["tokens"][0, 0] == 0
    # NaN in a read row: the walk stops with no correction token
    bad = logits.copy(); bad[0, 1, 2] = np.nan
    out = oracle.verify_chain(bad, q, np.array([[0, 0]], np.int32),
                              np.array([[0.0, 0.5, 0.5]], np.float32), 1.0, 0)
    assert out["status"][0] & oracle.ST_BAD_ROW
    assert out["tokens"][0].tolist() == [0, -1, -1] and out["num_accepted"][0] == 1
    # ragged length out of range
    out = oracle.verify_chain(logits.reshape(3, V), q.reshape(2, V), np.array([[0, 0]], np.int32),
                              u, 1.0, 0, K=2, V=V, k_per_req=[3], l_row_off=[0, 3], q_row_off=[0, 2])
    assert out["status"][0] == oracle.ST_BAD_K and out["tokens"][0].tolist() == [-1, -1, -1]


def test_ragged_equals_dense_per_request():
    rng = np.random.default_rng(9)
    B, K, V = 12, 5, 30
    logits = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, K)).astype(np.float32)
    draft = np.stack([[draw(rng, q[b, i], 1)[0] for i in range(K)] for b in range(B)]).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    k = rng.integers(0, K + 1, B).astype(np.int32)
    lo = np.concatenate([[0], np.cumsum(k + 1)]).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    pl = np.concatenate([logits[b, :k[b] + 1] for b in range(B)])
    pq = np.concatenate([q[b, :k[b]] for b in range(B)] + [np.zeros((1, V), np.float32)])
    rg = oracle.verify_chain(pl, pq, draft, u, 0.9, 7, K=K, V=V, k_per_req=k, l_row_off=lo, q_row_off=qo)
    for b in range(B):
        kb = int(k[b])
        uu = np.concatenate([u[b, :kb], [u[b, kb]]])[None].astype(np.float32)
        d1 = oracle.verify_chain(logits[b:b + 1, :kb + 1], q[b:b + 1, :max(kb, 1)] if kb else
                                 np.zeros((1, 1, V), np.float32),
                                 draft[b:b + 1, :kb] if kb else np.zeros((1, 0), np.int32), uu, 0.9, 7,
                                 K=kb, V=V)
        assert rg["tokens"][b, :kb + 1].tolist() == d1["tokens"][0].tolist()
        assert rg["num_accepted"][b] == d1["num_accepted"][0]


def test_cap_accept_equals_compact_and_dense_prefix():
    """Page §9's ragged modes: "cap-accept" keeps the full dense window and
    caps the commit at k_b; "compact" packs only the k_b + 1 rows; both equal
    a dense verify of the first k_b + 1 rows of each request."""
    rng = np.random.default_rng(19)
    B, K, V = 30, 6, 40
    logits = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, K)).astype(np.float32)
    draft = np.stack([[draw(rng, q[b, i], 1)[0] for i in range(K)] for b in range(B)]).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    k = rng.integers(0, K + 1, B).astype(np.int32)
    for top_k in (0, 5):
        cap = oracle.verify_chain(logits, q, draft, u, 0.8, top_k, k_per_req=k)
        lo = np.concatenate([[0], np.cumsum(k + 1)]).astype(np.int32)
        qo = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
        pl = np.concatenate([logits[b, :k[b] + 1] for b in range(B)])
        pq = np.concatenate([q[b, :k[b]] for b in range(B)] + [np.zeros((1, V), np.float32)])
        comp = oracle.verify_chain(pl, pq, draft, u, 0.8, top_k, K=K, V=V, k_per_req=k, l_row_off=lo, q_row_off=qo)
        for key in ("tokens", "num_accepted", "status", "rows_read"):
            np.testing.assert_array_equal(cap[key], comp[key], err_msg=key)
        for b in range(B):
            kb = int(k[b])
            uu = np.concatenate([u[b, :kb], [u[b, kb]]])[None].astype(np.float32)
            d1 = oracle.verify_chain(logits[b:b + 1, :kb + 1],
                                     q[b:b + 1, :kb] if kb else np.zeros((1, 1, V), np.float32),
                                     draft[b:b + 1, :kb] if kb else np.zeros((1, 0), np.int32), uu, 0.8, top_k,
                                     K=kb, V=V)
            assert cap["tokens"][b, :kb + 1].tolist() == d1["tokens"][0].tolist()
            assert (cap["tokens"][b, kb + 1:] == -1).all()
            assert cap["num_accepted"][b] == d1["num_accepted"][0] <= kb
    # every k_b = K: the cap never binds, the result is the static (dense) one
    full = oracle.verify_chain(logits, q, draft, u, 0.8, 5, k_per_req=np.full(B, K, np.int32))
    dense = oracle.verify_chain(logits, q, draft, u, 0.8, 5)
    np.testing.assert_array_equal(full["tokens"], dense["tokens"])
    np.testing.assert_array_equal(full["num_accepted"], dense["num_accepted"])


# ---------------------------------------------------------------------------
# greedy: argmax with the lowest index on ties
# ---------------------------------------------------------------------------


def test_greedy_against_library_argmax_with_ties():
    rng = np.random.default_rng(17)
    B, K, V = 300, 4, 64
    logits = np.round(rng.standard_normal((B, K + 1, V)) * 3) / 4     # many exact ties
    logits = logits.astype(np.float32)
    am = logits.argmax(-1)                                            # numpy: first maximal index
    draft = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    out = oracle.verify_greedy(logits, draft)
    for b in range(B):
        n = 0
        while n < K and draft[b, n] == am[b, n]:
            n += 1
        assert out["num_accepted"][b] == n
        assert out["tokens"][b, :n + 1].tolist() == list(draft[b, :n]) + [am[b, n]]
        assert out["rows_read"][b] == n + 1


def test_greedy_bf16_bits_roundtrip():
    rng = np.random.default_rng(2)
    f = (rng.standard_normal((3, 3, 16)) * 3).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)               # truncation is a valid bf16
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    d = back[:, :2].argmax(-1).astype(np.int32)
    a = oracle.verify_greedy(bits, d)
    b = oracle.verify_greedy(back, d)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])


# ---------------------------------------------------------------------------
# §5 DDTree: Q(u) = prod q_i(u_i), best-first heap under the node budget
# ---------------------------------------------------------------------------


def _rand_q(rng, B, L, V, ties=False):
    if ties:
        q = rng.integers(1, 4, size=(B, L, V)).astype(np.float64)
    else:
        q = rng.random((B, L, V)) + 0.05
    return (q / q.sum(-1, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("V,L", [(2, 4), (3, 3), (4, 4), (3, 1), (6, 3), (5, 4)])
@pytest.mark.parametrize("budget", [1, 2, 3, 4, 5, 17, 64])
@pytest.mark.parametrize("ties", [False, True])
def test_tree_heap_equals_bruteforce(V, L, budget, ties):
    """The brute force enumerates every prefix over all V tokens of every
    depth (ranks counted pairwise), so cases with budget - 1 < V also pin
    the heap's per-depth cut to the budget - 1 most probable tokens."""
    rng = np.random.default_rng(100 + V * 10 + L + budget + (7 if ties else 0))
    q = _rand_q(rng, 6, L, V, ties)
    if ties:
        q[0] = 1.0 / V                                               # one fully uniform block
    h = oracle.tree_build(q, budget)
    bf = oracle.tree_build_bruteforce(q, budget)
    for key in ("token", "parent", "depth", "score", "anc_mask", "num_nodes"):
        np.testing.assert_array_equal(h[key], bf[key], err_msg=key)


def test_tree_invariants_and_product_score():
    rng = np.random.default_rng(31)
    B, L, V, N = 8, 6, 40, 64
    q = _rand_q(rng, B, L, V)
    q[:, :, :3] *= 20                                                # a few dominant tokens
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    t = oracle.tree_build(q, N)
    for b in range(B):
        nn = t["num_nodes"][b]
        assert nn == N
        assert t["depth"][b, 0] == 0 and t["parent"][b, 0] == -1 and t["score"][b, 0] == 1.0
        for n in range(1, nn):
            par = t["parent"][b, n]
            assert 0 <= par < n                                      # parents come first
            assert t["depth"][b, n] == t["depth"][b, par] + 1
            assert t["score"][b, n] <= t["score"][b, par]
            # Q(u) as the product of q along the path, root to node
            path = []
            m = n
            while m > 0:
                path.append(m)
                m = t["parent"][b, m]
            s = 1.0
            for m in reversed(path):
                s = s * float(q[b, t["depth"][b, m] - 1, t["token"][b, m]])
            assert s == t["score"][b, n]
            # visibility: the node itself and exactly its ancestors
            anc = set(path) | {0}
            mask = int(t["anc_mask"][b, n, 0])
            assert {i for i in range(64) if mask >> i & 1} == anc
            assert bin(mask).count("1") - 1 == t["depth"][b, n]
        # siblings carry distinct tokens
        pairs = {(t["parent"][b, n], t["token"][b, n]) for n in range(1, nn)}
        assert len(pairs) == nn - 1
        # the pop order is non-increasing in Q
        assert np.all(np.diff(t["score"][b, :nn]) <= 0)


def test_tree_rows_beyond_needed_are_never_consulted():
    rng = np.random.default_rng(41)
    B, L, V, N = 10, 8, 300, 64
    q = np.exp(rng.standard_normal((B, L, V)) * 3)
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    full = oracle.tree_build(q, N)
    assert (full["rows_needed"] < L).any()
    poisoned = q.copy()
    for b in range(B):
        poisoned[b, full["rows_needed"][b]:] = np.nan
    cut = oracle.tree_build(poisoned, N)
    assert (cut["status"] == 0).all()
    for key in ("token", "parent", "depth", "score", "anc_mask", "num_nodes"):
        np.testing.assert_array_equal(full[key], cut[key], err_msg=key)
    # the deepest kept node is at rows_needed - 1 or rows_needed
    for b in range(B):
        dmax = full["depth"][b].max()
        assert full["rows_needed"][b] in (dmax, dmax + 1)


# ---------------------------------------------------------------------------
# §5 DDTree verification walk
# ---------------------------------------------------------------------------


def test_tree_walk_follows_constructed_target():
    rng = np.random.default_rng(51)
    B, L, V, N = 6, 5, 30, 20
    q = _rand_q(rng, B, L, V)
    t = oracle.tree_build(q, N)
    logits = rng.standard_normal((B, N, V)).astype(np.float32)
    expect = []
    for b in range(B):
        # intended path: from the root, take a random child while one exists,
        # stopping early for some requests
        cur, path, toks = 0, [0], []
        stop_at = rng.integers(0, L + 1)
        while True:
            kids = [c for c in range(t["num_nodes"][b]) if t["parent"][b, c] == cur]
            if not kids or len(toks) >= stop_at:
                used = {t["token"][b, c] for c in kids}
                bonus = next(x for x in range(V) if x not in used)
                logits[b, cur, bonus] = 100.0
                toks.append(bonus)
                break
            c = kids[rng.integers(len(kids))]
            logits[b, cur, t["token"][b, c]] = 100.0
            toks.append(int(t["token"][b, c]))
            path.append(c)
            cur = c
        expect.append((path, toks))
    out = oracle.verify_tree(logits, t["token"], t["parent"], t["num_nodes"], L)
    for b, (path, toks) in enumerate(expect):
        assert out["num_accepted"][b] == len(path) - 1
        assert out["path_nodes"][b, :len(path)].tolist() == path
        assert out["tokens"][b, :len(toks)].tolist() == toks
        assert (out["tokens"][b, len(toks):] == -1).all()


# ---------------------------------------------------------------------------
# §1 + §5 stochastic tree walk: every committed token is a target draw
# ---------------------------------------------------------------------------


def _walk_case(seed, B=40, L=5, V=60, N=24):
    rng = np.random.default_rng(seed)
    t = oracle.tree_build(_rand_q(rng, B, L, V), N)
    # distinct logits (no tied maximum), with the tree's tokens pushed up so
    # that walks go deep
    logits = (rng.permutation(B * N * V).reshape(B, N, V) * 1e-3).astype(np.float32)
    for b in range(B):
        for c in range(1, N):
            par = t["parent"][b, c]
            if par >= 0 and rng.random() < 0.6:
                logits[b, par, t["token"][b, c]] += 500.0 + rng.random()
    return rng, t, logits, L


def test_tree_sample_top1_equals_greedy_walk():
    rng, t, logits, L = _walk_case(71)
    u = rng.random((logits.shape[0], L + 1), dtype=np.float32)
    s = oracle.verify_tree_sample(logits, t["token"], t["parent"], t["num_nodes"], u, L, 1.0, 1)
    g = oracle.verify_tree(logits, t["token"], t["parent"], t["num_nodes"], L)
    for k in ("path_nodes", "tokens", "num_accepted", "status"):
        np.testing.assert_array_equal(s[k], g[k], err_msg=k)
    assert (g["num_accepted"] >= 1).mean() > 0.3


def test_tree_sample_tiny_temperature_equals_greedy_walk():
    rng, t, logits, L = _walk_case(72)
    u = np.clip(rng.random((logits.shape[0], L + 1), dtype=np.float32), 1e-3, 1 - 1e-3)
    s = oracle.verify_tree_sample(logits, t["token"], t["parent"], t["num_nodes"], u, L, 1e-4, 0)
    g = oracle.verify_tree(logits, t["token"], t["parent"], t["num_nodes"], L)
    for k in ("path_nodes", "tokens", "num_accepted"):
        np.testing.assert_array_equal(s[k], g[k], err_msg=k)


def test_tree_sample_tokens_follow_target():
    """A hand tree over V = 6: root -> tokens 0 (node 1) and 2 (node 2);
    node 1 -> tokens 1 (node 3) and 3 (node 4); node 2 -> token 5 (node 5).
    Over 10^6 walks the first committed token follows p_root, and the second
    follows the p of the node the first one reached (the joint law of the
    first two tokens is p_root(a) p_node(a)(b) whenever a has a node)."""
    rng = np.random.default_rng(73)
    V, L, n = 6, 2, 1_000_000
    P = np.array([[0.30, 0.10, 0.25, 0.05, 0.20, 0.10],    # root
                  [0.05, 0.40, 0.10, 0.25, 0.10, 0.10],    # node 1 (after token 0)
                  [0.20, 0.10, 0.10, 0.10, 0.10, 0.40],    # node 2 (after token 2)
                  [0.50, 0.10, 0.10, 0.10, 0.10, 0.10],
                  [0.10, 0.50, 0.10, 0.10, 0.10, 0.10],
                  [0.10, 0.10, 0.50, 0.10, 0.10, 0.10]])
    token = np.array([-1, 0, 2, 1, 3, 5], np.int32)
    parent = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    N = 6
    logits = np.log(P).astype(np.float32)[None]                      # [1, N, V], broadcast
    u = rng.random((n, L + 1), dtype=np.float32)
    out = oracle.verify_tree_sample(logits, np.broadcast_to(token, (n, N)), np.broadcast_to(parent, (n, N)),
                                    np.full(n, N, np.int32), u, L, 1.0, 0, l_strides=(0, V))
    tok = out["tokens"]
    assert chi2_pvalue(np.bincount(tok[:, 0], minlength=V), P[0]) > 1e-3
    node_of = {0: 1, 2: 2}
    for a, node in node_of.items():
        sel = tok[:, 0] == a
        assert (out["num_accepted"][sel] >= 1).all()
        assert chi2_pvalue(np.bincount(tok[sel, 1], minlength=V), P[node]) > 1e-3
    # tokens without a node end the walk: nothing after them
    ends = ~np.isin(tok[:, 0], [0, 2])
    assert (out["num_accepted"][ends] == 0).all() and (tok[ends, 1] == -1).all()
    # the joint of the first two tokens over the walks that reached depth 1
    pairs = tok[:, 0] * V + np.where(tok[:, 1] >= 0, tok[:, 1], 0)
    deep = np.isin(tok[:, 0], [0, 2])
    joint = np.zeros(V * V)
    for a, node in node_of.items():
        joint[a * V:(a + 1) * V] = P[0, a] * P[node]
    assert chi2_pvalue(np.bincount(pairs[deep], minlength=V * V), joint) > 1e-3


# ---------------------------------------------------------------------------
# §5 DDTree: the KV cache keeps only the accepted path
# ---------------------------------------------------------------------------


def test_kv_compact_keeps_the_walked_path_in_depth_order():
    """Rows tagged with their own (plane, request, node) coordinates: after a
    constructed walk the destination holds exactly the root and the accepted
    nodes' rows, in depth order, at each request's cache position; every
    other destination row keeps its contents."""
    rng, t, logits, L = _walk_case(81, B=12, L=5, V=60, N=24)
    walk = oracle.verify_tree(logits, t["token"], t["parent"], t["num_nodes"], L)
    P, B, N, R = 3, 12, 24, 4
    src = np.zeros((P, B, N, R), np.int32)
    for p in range(P):
        for b in range(B):
            for n in range(N):
                src[p, b, n] = [p, b, n, 7]
    M = 40
    pos = rng.integers(0, M - (L + 1), B).astype(np.int32)
    dst = np.full((P, B, M, R), -9, np.int32)
    out = oracle.kv_compact(src, dst, walk["path_nodes"], walk["num_accepted"], dst_pos=pos)
    for p in range(P):
        for b in range(B):
            n = walk["num_accepted"][b]
            path = walk["path_nodes"][b, :n + 1]
            assert path[0] == 0                                        # the root first
            for j, node in enumerate(path):
                assert out[p, b, pos[b] + j].tolist() == [p, b, node, 7]
            # depth order: each kept node's parent is the row before it
            for j in range(1, n + 1):
                assert t["parent"][b, path[j]] == path[j - 1]
            mask = np.ones(M, bool)
            mask[pos[b]:pos[b] + n + 1] = False
            assert (out[p, b, mask] == -9).all()


# ---------------------------------------------------------------------------
# §5 DSpark: s_j = prod c_i, advance 1 + sum s_j, k maximising advance/cost
# ---------------------------------------------------------------------------


def test_adaptive_closed_forms():
    Kmax = 8
    one = oracle.adaptive_len(np.ones((3, Kmax), np.float32), 1.0, 0.15)
    assert (one["k"] == Kmax).all()                                  # (1+k)/(1+0.15k) increases
    np.testing.assert_array_equal(one["exp_adv"], Kmax + 1.0)
    zero = oracle.adaptive_len(np.zeros((3, Kmax), np.float32), 1.0, 0.15)
    assert (zero["k"] == 0).all() and (zero["exp_adv"] == 1.0).all()
    np.testing.assert_array_equal(zero["l_row_off"], [0, 1, 2, 3])
    np.testing.assert_array_equal(zero["q_row_off"], [0, 0, 0, 0])


def test_adaptive_exact_ties_go_to_the_smaller_k():
    """c = 1 and cost a + b k with a = b = 1: E(k)/cost(k) = (1+k)/(1+k) = 1
    exactly for every k, so the smaller-k tie rule picks k = 0; the same with
    the cost table 1 + k, and a two-way tie at k = 2, 5 from a table."""
    Kmax = 6
    c = np.ones((2, Kmax), np.float32)
    assert (oracle.adaptive_len(c, 1.0, 1.0)["k"] == 0).all()
    assert (oracle.adaptive_len(c, 1.0, 0.0, cost=np.arange(1, Kmax + 2, dtype=np.float64))["k"] == 0).all()
    # E = 1..7; cost chosen so that E/cost = 1.5 exactly at k = 2 and k = 5, 1 elsewhere
    cost = np.array([1, 2, 2, 4, 5, 4, 7], np.float64)
    o = oracle.adaptive_len(c, 1.0, 0.0, cost=cost)
    assert (o["k"] == 2).all()


def test_adaptive_hand_example():
    # c = 0.9, 0.8, 0.5, 0.5: s = .9, .72, .36, .18; E = 1.9, 2.62, 2.98, 3.16
    # E/(1+0.15k): 1.6522, 1.9407, 2.0552, 1.9750  -> k = 3
    c = np.array([[0.9, 0.8, 0.5, 0.5]], np.float32)
    o = oracle.adaptive_len(c, 1.0, 0.15)
    assert o["k"][0] == 3
    np.testing.assert_allclose(o["surv"][0], [0.9, 0.72, 0.36, 0.18], rtol=1e-6)
    np.testing.assert_allclose(o["exp_adv"][0], 2.98, rtol=1e-6)
    np.testing.assert_array_equal(o["l_row_off"], [0, 4])
    np.testing.assert_array_equal(o["q_row_off"], [0, 3])


def test_adaptive_exact_rational_bruteforce():
    rng = np.random.default_rng(61)
    B, Kmax = 2000, 8
    c = rng.beta(8, 2, size=(B, Kmax)).astype(np.float32)
    a, b = 1.0, 0.15
    o = oracle.adaptive_len(c, a, b)
    A, Bq = Fraction(float(np.float32(a))), Fraction(float(np.float32(b)))
    lo = [0]
    for r in range(B):
        s, E = Fraction(1), Fraction(1)
        ratios = [E / (A + Bq * 0)]
        for j in range(Kmax):
            s *= Fraction(float(c[r, j]))
            E += s
            ratios.append(E / (A + Bq * (j + 1)))
        best = max(range(Kmax + 1), key=lambda k: (ratios[k], -k))
        if not o["near_tie"][r]:
            assert o["k"][r] == best, r
        lo.append(lo[-1] + int(o["k"][r]) + 1)
        np.testing.assert_allclose(o["surv"][r], np.cumprod(c[r].astype(np.float64)), rtol=1e-14)
    np.testing.assert_array_equal(o["l_row_off"], lo)
    np.testing.assert_array_equal(np.diff(o["q_row_off"]), o["k"])


def test_adaptive_cost_table_of_a_linear_cost_is_the_linear_rule():
    rng = np.random.default_rng(62)
    B, Kmax = 3000, 8
    c = rng.beta(8, 2, size=(B, Kmax)).astype(np.float32)
    a, b = 1.0, 0.15
    table = np.float64(np.float32(a)) + np.float64(np.float32(b)) * np.arange(Kmax + 1, dtype=np.float64)
    lin = oracle.adaptive_len(c, a, b)
    tab = oracle.adaptive_len(c, 7.0, 3.0, cost=table)        # a, b ignored with a table
    for key in ("k", "surv", "exp_adv", "l_row_off", "q_row_off"):
        np.testing.assert_array_equal(lin[key], tab[key], err_msg=key)


def test_adaptive_cost_table_hand_example():
    # E = 1, 1.9, 2.62, 2.98, 3.16 (as in the linear hand example, where k = 3);
    # a table where two positions cost as much as none and the third doubles
    # the price: E/cost = 1, 1.9, 2.62, 1.192, 1.264 -> k = 2
    c = np.array([[0.9, 0.8, 0.5, 0.5]], np.float32)
    o = oracle.adaptive_len(c, 1.0, 0.15, cost=np.array([1.0, 1.0, 1.0, 2.5, 2.5]))
    assert o["k"][0] == 2
    np.testing.assert_allclose(o["exp_adv"][0], 2.62, rtol=1e-6)
    np.testing.assert_array_equal(o["l_row_off"], [0, 3])


def test_adaptive_cost_table_exact_rational_bruteforce():
    rng = np.random.default_rng(63)
    B, Kmax = 1500, 8
    c = rng.beta(8, 2, size=(B, Kmax)).astype(np.float32)
    table = np.cumsum(rng.random(Kmax + 1) * 0.4 + 0.05) + 0.5
    o = oracle.adaptive_len(c, 1.0, 0.15, cost=table)
    Ct = [Fraction(float(x)) for x in table]
    for r in range(B):
        s, E = Fraction(1), Fraction(1)
        ratios = [E / Ct[0]]
        for j in range(Kmax):
            s *= Fraction(float(c[r, j]))
            E += s
            ratios.append(E / Ct[j + 1])
        best = max(range(Kmax + 1), key=lambda k: (ratios[k], -k))
        if not o["near_tie"][r]:
            assert o["k"][r] == best, r
