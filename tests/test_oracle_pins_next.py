"""Pins of the oracle's rows that follow the core path (CPU only): appending to
the paged cache, exact speculative sampling and top-p page selection.

As in the core pins, each test ties the oracle to something outside itself: an
independent construction of the same cache, values worked by hand, the
distribution theorem of speculative sampling, or brute-force enumeration."""
import itertools
import os

import numpy as np
import pytest

from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.helpers import custom

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- f1 append

def _pair(lens, T, H_q=4, H_kv=2, D=16, ps=16, seed=30):
    """The same cache built twice by the test helper's scatter: once whole, once
    with the last T tokens of each sequence replaced by garbage."""
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((n, H_kv, D)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((n, H_kv, D)).astype(np.float32) for n in lens]
    Kg = [k.copy() for k in K]
    Vg = [v.copy() for v in V]
    for k, v in zip(Kg, Vg):
        k[len(k) - T:] = 1000.0
        v[len(v) - T:] = -1000.0
    full = custom(lens, H_q, H_kv, D, ps, rng=np.random.default_rng(seed + 1), K=K, V=V)
    hole = custom(lens, H_q, H_kv, D, ps, rng=np.random.default_rng(seed + 1), K=Kg, V=Vg)
    k_new = np.stack([wl.f32_to_bf16_bits(k[len(k) - T:]) for k in K])
    v_new = np.stack([wl.f32_to_bf16_bits(v[len(v) - T:]) for v in V])
    return full, hole, k_new, v_new


@pytest.mark.parametrize("lens,T", [([33, 16, 17, 64], 1), ([40, 23, 30], 7), ([80, 50], 40)])
def test_append_rebuilds_the_whole_cache(oracle_mod, lens, T):
    """Writing the last T tokens into the holed cache gives the whole cache bit for bit
    (other slots, other sequences and the unused tails are untouched)."""
    full, hole, k_new, v_new = _pair(lens, T)
    assert np.array_equal(full.page_table, hole.page_table)
    K, V = oracle_mod.append(hole, T, k_new, v_new)
    assert np.array_equal(K, full.K) and np.array_equal(V, full.V)


def test_append_all_at_once_equals_one_token_at_a_time(oracle_mod):
    lens, T = [45, 20, 33], 6
    full, hole, k_new, v_new = _pair(lens, T, seed=31)
    K, V = oracle_mod.append(hole, T, k_new, v_new)
    w = hole
    for t in range(T):
        step = wl.Workload(**{**w.__dict__})
        step.seq_lens = (np.asarray(lens) - T + t + 1).astype(np.int32)
        step.K, step.V = w.K, w.V
        step.K, step.V = oracle_mod.append(step, 1, k_new[:, t:t + 1], v_new[:, t:t + 1])
        w = step
    assert np.array_equal(w.K, K) and np.array_equal(w.V, V)


def test_summaries_after_append_match_the_whole_cache(oracle_mod):
    lens, T = [47, 16, 65], 3
    full, hole, k_new, v_new = _pair(lens, T, seed=32)
    after = wl.Workload(**{**hole.__dict__})
    after.K, after.V = oracle_mod.append(hole, T, k_new, v_new)
    s_full = oracle_mod.summarize(full)
    s_after = oracle_mod.summarize(after)
    used = np.unique(full.page_table[full.page_table >= 0])
    assert np.array_equal(s_full[used], s_after[used])
    # a fresh page holding one appended token has that key as both min and max
    b, pos = 1, 15                      # len 16: the last token is slot 15 of page 0
    ph = full.page_table[b, pos // 16]
    k = wl.bf16_bits_to_f32(k_new[b, -1]).astype(np.float64)
    assert np.all(s_after[ph, :, 0] <= k) and np.all(k <= s_after[ph, :, 1])


# ---------------------------------------------------------------- f2 speculative sampling

def _golden_spec(fname="spec_accept_cases.txt"):
    out = []
    for line in open(os.path.join(HERE, "golden", fname)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kn, p, q, draft, uacc, ures, nacc, toks = [x.strip() for x in line.split("|")]
        k, n = map(int, kn.split())
        rows = lambda s: np.array([[float(v) for v in r.split()] for r in s.split(";")], np.float32)
        out.append((k, n, rows(p), rows(q), [int(x) for x in draft.split()],
                    [float(x) for x in uacc.split()], float(ures), int(nacc),
                    [int(x) for x in toks.split()]))
    return out


@pytest.mark.parametrize("case", _golden_spec(), ids=lambda c: f"k{c[0]}n{c[1]}")
def test_spec_accept_hand_worked_cases(oracle_mod, case):
    k, n, p, q, draft, uacc, ures, nacc, toks = case
    assert p.shape == (k, n) and q.shape == (k + 1, n)
    na, tk = oracle_mod.spec_accept(p[None], q[None], np.array([draft]), np.array([uacc], np.float32),
                                    np.array([ures], np.float32))
    assert na[0] == nacc and tk[0].tolist() == toks


def test_spec_accept_output_follows_the_target_distribution(oracle_mod):
    """The first emitted token is distributed as q_0 whatever the drafter p_0 (the
    theorem that makes speculative sampling exact), and the first draft is accepted
    with probability sum_x min(p_0(x), q_0(x))."""
    rng = np.random.default_rng(40)
    n, k, N = 6, 2, 40000
    p = rng.dirichlet(np.ones(n), size=k).astype(np.float32)
    q = rng.dirichlet(np.ones(n), size=k + 1).astype(np.float32)
    P = np.broadcast_to(p, (N, k, n))
    Q = np.broadcast_to(q, (N, k + 1, n))
    draft = np.stack([rng.choice(n, size=N, p=p[i] / p[i].sum()) for i in range(k)], axis=1)
    u_acc = rng.random((N, k), dtype=np.float32)
    u_res = rng.random(N, dtype=np.float32)
    nacc, toks = oracle_mod.spec_accept(P, Q, draft, u_acc, u_res)
    q0 = q[0].astype(np.float64) / q[0].sum()
    freq = np.bincount(toks[:, 0], minlength=n) / N
    sigma = np.sqrt(q0 * (1 - q0) / N)
    assert np.all(np.abs(freq - q0) <= 5 * sigma + 1e-9), (freq, q0)
    p0 = p[0].astype(np.float64) / p[0].sum()
    alpha = np.minimum(p0, q0).sum()
    got = np.mean(nacc >= 1)
    assert abs(got - alpha) <= 5 * np.sqrt(alpha * (1 - alpha) / N)


def test_spec_accept_rejection_draws_from_the_residual(oracle_mod):
    """At a rejection the emitted token follows max(0, q - p) normalised (drafts are
    forced to be rejected with u = 1 - 2^-24 on a draft whose p exceeds q), so tokens
    with q <= p are never emitted and the others with frequencies within 5 sigma."""
    rng = np.random.default_rng(42)
    n, N = 8, 40000
    p = rng.dirichlet(np.ones(n)).astype(np.float32)
    q = rng.dirichlet(np.ones(n)).astype(np.float32)
    x = int(np.argmax(p.astype(np.float64) - q))       # a draft the target likes less
    P = np.broadcast_to(p, (N, 1, n))
    Q = np.broadcast_to(np.stack([q, q]), (N, 2, n))
    u_acc = np.full((N, 1), np.float32(1 - 2.0 ** -24))  # u * p(x) >= q(x): rejected
    nacc, toks = oracle_mod.spec_accept(P, Q, np.full((N, 1), x), u_acc, rng.random(N, dtype=np.float32))
    assert np.all(nacc == 0)
    r = np.maximum(0.0, q.astype(np.float64) - p)
    r /= r.sum()
    freq = np.bincount(toks[:, 0], minlength=n) / N
    assert np.all(freq[r == 0] == 0)
    sigma = np.sqrt(r * (1 - r) / N)
    assert np.all(np.abs(freq - r) <= 5 * sigma + 1e-9), (freq, r)


def test_spec_accept_identical_distributions_accept_everything(oracle_mod):
    rng = np.random.default_rng(41)
    n, k, B = 50, 6, 64
    p = rng.dirichlet(np.ones(n), size=(B, k)).astype(np.float32)
    bonus = rng.integers(0, n, size=B)
    q = np.concatenate([p, np.eye(n, dtype=np.float32)[bonus][:, None]], axis=1)
    draft = rng.integers(0, n, size=(B, k))
    nacc, toks = oracle_mod.spec_accept(p, q, draft, rng.random((B, k), dtype=np.float32) * 0.999,
                                        rng.random(B, dtype=np.float32))
    assert np.all(nacc == k)
    assert np.array_equal(toks[:, :k], draft) and np.array_equal(toks[:, k], bonus)


# ---------------------------------------------------------------- f3 top-p selection

def _scores_workload(P, ps=16, H_kv=1):
    return custom([P * ps], H_kv, H_kv, 8, ps, rng=np.random.default_rng(50))


@pytest.mark.parametrize("P,sink,local,top_p,k_max", [
    (9, 1, 1, 0.5, 9), (9, 1, 2, 0.8, 9), (10, 0, 0, 0.9, 10), (10, 1, 1, 0.95, 5),
    (8, 1, 1, 0.3, 8), (7, 0, 1, 0.99, 7)])
def test_top_p_is_the_smallest_sufficient_set(oracle_mod, P, sink, local, top_p, k_max):
    """Brute force over all subsets that hold the mandatory pages: the oracle's set has
    the least size reaching the weight share top_p (or k_max pages if none does), and
    the largest weight among sets of that size."""
    rng = np.random.default_rng(51 + P + local)
    w = _scores_workload(P)
    scale = 0.7
    for trial in range(4):
        sc = rng.standard_normal((1, 1, P)) * 3.0
        pol = wl.BudgetPolicy("fixed", fixed_pages=P, sink_pages=sink, local_pages=local)
        sel, nsel = oracle_mod.select_top_p(w, sc, top_p, score_scale=scale, k_max=k_max, policy=pol)
        got = set(sel[0, 0, : nsel[0, 0]].tolist())
        weight = np.exp(scale * (sc[0, 0] - sc[0, 0].max()))
        need = top_p * weight.sum()
        mand = {p for p in range(P) if p < sink or p >= P - local}
        rest = [p for p in range(P) if p not in mand]
        best = None
        for r in range(len(rest) + 1):
            if len(mand) + r > k_max:
                break
            cands = [mand | set(c) for c in itertools.combinations(rest, r)]
            ok = [c for c in cands if weight[list(c)].sum() >= need] if cands else []
            if ok:
                best = max(ok, key=lambda c: weight[list(c)].sum())
                break
        if best is None:   # nothing reaches top_p within k_max: the k_max best pages
            r = k_max - len(mand)
            best = max((mand | set(c) for c in itertools.combinations(rest, r)),
                       key=lambda c: weight[list(c)].sum())
        assert got == best, (trial, sorted(got), sorted(best))
        assert sel[0, 0, : nsel[0, 0]].tolist() == sorted(got)


def test_top_p_edge_cases(oracle_mod):
    w = _scores_workload(6)
    pol0 = wl.BudgetPolicy("fixed", fixed_pages=6, sink_pages=0, local_pages=0)
    pol = wl.BudgetPolicy("fixed", fixed_pages=6, sink_pages=1, local_pages=1)
    sc = np.array([[[0.0, 1.0, 50.0, 2.0, 3.0, 0.5]]])
    # top_p = 0: the empty set suffices, so only mandatory pages are held
    sel, nsel = oracle_mod.select_top_p(w, sc, 0.0, score_scale=1.0, policy=pol0)
    assert nsel[0, 0] == 0
    sel, nsel = oracle_mod.select_top_p(w, sc, 0.0, score_scale=1.0, policy=pol)
    assert sel[0, 0, : nsel[0, 0]].tolist() == [0, 5]
    # one dominant page carries almost all the weight
    sel, nsel = oracle_mod.select_top_p(w, sc, 0.9, score_scale=1.0, policy=pol)
    assert sel[0, 0, : nsel[0, 0]].tolist() == [0, 2, 5]
    # top_p = 1 with distinct finite scores needs every page with positive weight
    sc2 = np.array([[[0.0, 0.1, 0.2, 0.3, 0.4, 0.5]]])
    sel, nsel = oracle_mod.select_top_p(w, sc2, 1.0, score_scale=1.0, policy=pol0)
    assert nsel[0, 0] >= 5
    # k_max caps the count
    sel, nsel = oracle_mod.select_top_p(w, sc2, 1.0, score_scale=1.0, k_max=3, policy=pol)
    assert sel[0, 0, : nsel[0, 0]].tolist() == [0, 4, 5]
