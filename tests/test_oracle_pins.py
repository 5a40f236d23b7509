"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test ties one oracle step to a closed form, an invariant the mathematics
fixes, a brute-force enumeration on a tiny input, or a value worked by hand from
the workload definitions -- never to a retyped copy of the oracle's own formula.
"""
import itertools
import os

import numpy as np
import pytest

from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.helpers import custom, f, token_kv

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- a1 summaries

def test_summary_is_attained_bound_over_valid_tokens(oracle_mod):
    """min/max bound every valid key, are attained by one, and ignore the slots past len."""
    rng = np.random.default_rng(1)
    w = custom([37, 16, 5, 64], 4, 2, 16, 16, rng=rng)
    summ = oracle_mod.summarize(w)
    for b in range(w.B):
        for h in range(w.H_kv):
            Kt, _ = token_kv(w, b, h)
            for p in range(w.pages(b)):
                toks = Kt[p * 16: min(len(Kt), (p + 1) * 16)]
                s = summ[w.page_table[b, p], h]
                assert np.all(s[0] <= toks) and np.all(toks <= s[1])
                assert np.all(np.any(toks == s[0], axis=0)) and np.all(np.any(toks == s[1], axis=0))
                # the poison (+64) in the unused slots of a partial page never shows up
                assert np.all(s[1] < wl.POISON_K)


def test_summary_of_single_token_page_is_the_key(oracle_mod):
    w = custom([17], 2, 1, 8, 16, rng=np.random.default_rng(2))
    summ = oracle_mod.summarize(w)
    k = f(w.K[w.page_table[0, 1], 0, 0])
    s = summ[w.page_table[0, 1], 0]
    assert np.array_equal(s[0], k) and np.array_equal(s[1], k)


# ---------------------------------------------------------------- a2 scores

def test_upper_bound_dominates_every_true_logit(oracle_mod):
    rng = np.random.default_rng(3)
    w = custom([70, 33], 6, 2, 32, 16, rng=rng)
    summ = oracle_mod.summarize(w)
    sc = oracle_mod.scores(w, summ)
    qf = f(w.q)
    for b in range(w.B):
        for h in range(w.H_kv):
            Kt, _ = token_kv(w, b, h)
            for p in range(w.pages(b)):
                toks = Kt[p * 16: min(len(Kt), (p + 1) * 16)]
                true_max = max(float(np.max(toks @ qf[b, h * w.G + g])) for g in range(w.G))
                assert sc[b, h, p] >= true_max - 1e-12


def test_upper_bound_is_exact_for_one_token_page(oracle_mod):
    """A page holding one key: the bound equals the largest q.k over the group (closed form)."""
    rng = np.random.default_rng(4)
    w = custom([33], 4, 1, 16, 16, rng=rng)
    sc = oracle_mod.scores(w, oracle_mod.summarize(w))
    k = f(w.K[w.page_table[0, 2], 0, 0])
    qf = f(w.q[0])
    exact = max(float(np.dot(qf[g], k)) for g in range(4))
    assert abs(sc[0, 0, 2] - exact) <= 1e-12 * (1 + abs(exact))


def test_upper_bound_sign_cases(oracle_mod):
    """q >= 0 picks the channel maxima, q <= 0 the minima (closed forms)."""
    rng = np.random.default_rng(5)
    D = 8
    q = np.abs(rng.standard_normal((1, 2, D))).astype(np.float32)
    q[0, 1] = -q[0, 1]
    w = custom([16], 2, 2, D, 16, q=q, rng=rng)
    summ = oracle_mod.summarize(w)
    sc = oracle_mod.scores(w, summ)
    qf = f(w.q[0])
    s0 = summ[w.page_table[0, 0], 0]
    s1 = summ[w.page_table[0, 0], 1]
    assert sc[0, 0, 0] == pytest.approx(float(qf[0] @ s0[1]), rel=1e-14)
    assert sc[0, 1, 0] == pytest.approx(float(qf[1] @ s1[0]), rel=1e-14)


def test_group_score_is_max_over_heads(oracle_mod):
    """One head of the group has q = 0 (bound 0): the group score is max(0, other head's bound)."""
    rng = np.random.default_rng(6)
    D = 8
    q = rng.standard_normal((1, 2, D)).astype(np.float32)
    q[0, 0] = 0.0
    w = custom([48], 2, 1, D, 16, q=q, rng=np.random.default_rng(60))
    summ = oracle_mod.summarize(w)
    sc = oracle_mod.scores(w, summ)
    # same seed and shapes: the one-head workload draws the same keys
    w1 = custom([48], 1, 1, D, 16, q=q[:, 1:2], rng=np.random.default_rng(60))
    sc1 = oracle_mod.scores(w1, oracle_mod.summarize(w1))
    assert np.allclose(sc[0, 0, :3], np.maximum(0.0, sc1[0, 0, :3]), rtol=0, atol=0)


# ---------------------------------------------------------------- a3 budget

def _golden_budgets():
    rows = []
    with open(os.path.join(HERE, "golden", "budget_schedule.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if line:
                mode, n, ps, exp = line.split()
                rows.append((mode, int(n), int(ps), int(exp)))
    return rows


@pytest.mark.parametrize("mode,length,ps,expected", _golden_budgets())
def test_budget_matches_hand_worked_values(oracle_mod, mode, length, ps, expected):
    if mode == "linear":
        pol = wl.spec("sweep", ps).policy
    elif mode == "fraction":
        pol = wl.spec("longtail").policy
    else:
        pol = wl.spec("q8b").policy if expected == 64 else wl.spec("q17b").policy
    assert oracle_mod.budget_pages(pol, length, ps) == expected


def test_k_eff_edge_cases(oracle_mod):
    pol = wl.BudgetPolicy("fixed", fixed_pages=3, sink_pages=1, local_pages=4)
    assert oracle_mod.k_eff(pol, 16 * 10, 16, 64) == 5      # budget below |mandatory| = 5
    assert oracle_mod.k_eff(pol, 16 * 2, 16, 64) == 2       # fewer pages than mandatory
    pol = wl.BudgetPolicy("fixed", fixed_pages=100, sink_pages=1, local_pages=4)
    assert oracle_mod.k_eff(pol, 16 * 10, 16, 64) == 10     # budget above the page count
    assert oracle_mod.k_eff(pol, 16 * 90, 16, 64) == 64     # capped by the buffer size k_max
    assert oracle_mod.k_eff(pol, 0, 16, 64) == 0            # empty sequence
    assert oracle_mod.k_eff(pol, 1, 16, 64) == 1


# ---------------------------------------------------------------- a4 selection

def _sel_workload(P, ps=16):
    return custom([P * ps], 1, 1, 4, ps, rng=np.random.default_rng(7))


def test_selection_equals_brute_force_best_subset(oracle_mod):
    """All subsets of the non-mandatory pages: the max-sum one of the right size is chosen."""
    rng = np.random.default_rng(8)
    for trial in range(30):
        P = int(rng.integers(3, 11))
        sink, local = int(rng.integers(0, 2)), int(rng.integers(0, 3))
        budget = int(rng.integers(0, P + 2))
        w = _sel_workload(P)
        pol = wl.BudgetPolicy("fixed", fixed_pages=budget, sink_pages=sink, local_pages=local)
        sc = np.full((1, 1, w.max_pages_per_seq), -np.inf)
        sc[0, 0, :P] = rng.standard_normal(P)
        sel, nsel = oracle_mod.select(w, sc, policy=pol, k_max=P)
        got = set(sel[0, 0, : nsel[0, 0]].tolist())
        mand = {p for p in range(P) if p < sink or p >= P - local}
        k = min(P, max(budget, len(mand)))
        rest = [p for p in range(P) if p not in mand]
        best, best_sum = None, -np.inf
        for sub in itertools.combinations(rest, k - len(mand)):
            s = sum(sc[0, 0, p] for p in sub)
            if s > best_sum:
                best, best_sum = set(sub), s
        assert got == mand | best, (trial, P, sink, local, budget)


def test_selection_ties_prefer_lower_page_ids(oracle_mod):
    P = 12
    w = _sel_workload(P)
    pol = wl.BudgetPolicy("fixed", fixed_pages=5, sink_pages=1, local_pages=1)
    sc = np.zeros((1, 1, P))
    sel, nsel = oracle_mod.select(w, sc, policy=pol, k_max=P)
    assert sel[0, 0, : nsel[0, 0]].tolist() == [0, 1, 2, 3, 11]


def test_selection_invariants_on_generated_workload(oracle_mod):
    w = wl.named("q17b", B=6, len_lo=300, len_hi=4000, policy_over=dict(fixed_pages=20))
    res = oracle_mod.decode_step(w, threads=4)
    for b in range(w.B):
        P = w.pages(b)
        k = oracle_mod.k_eff(w.policy, int(w.seq_lens[b]), w.page_size, w.k_max)
        for h in range(w.H_kv):
            s = res["sel"][b, h, : res["nsel"][b, h]].tolist()
            assert len(s) == k
            assert s == sorted(set(s))
            assert 0 in s and all(p in s for p in range(max(0, P - 4), P))
            assert all(0 <= p < P for p in s)


def test_selection_with_budget_over_all_pages_keeps_everything(oracle_mod):
    w = wl.named("tiny", policy_over=dict(fixed_pages=1000), k_max=64)
    res = oracle_mod.decode_step(w, threads=2)
    for b in range(w.B):
        for h in range(w.H_kv):
            assert res["sel"][b, h, : res["nsel"][b, h]].tolist() == list(range(64))


# ---------------------------------------------------------------- a5 sparse attention

def _attn_all(oracle_mod, w):
    P = w.max_pages_per_seq
    sel = np.tile(np.arange(P, dtype=np.int32), (w.B, w.H_kv, 1))
    nsel = np.array([[w.pages(b)] * w.H_kv for b in range(w.B)], dtype=np.int32)
    return oracle_mod.sparse_attn(w, sel, nsel)


def test_single_token_returns_its_value_exactly(oracle_mod):
    w = custom([1], 2, 1, 8, 16, rng=np.random.default_rng(9))
    o, lse = _attn_all(oracle_mod, w)
    v = f(w.V[w.page_table[0, 0], 0, 0])
    k = f(w.K[w.page_table[0, 0], 0, 0])
    for g in range(2):
        assert np.array_equal(o[0, g], v)
        assert lse[0, g] == pytest.approx(float(f(w.q[0, g]) @ k) / np.sqrt(8), rel=1e-14)


def test_two_tokens_closed_form(oracle_mod):
    """Two keys: the weights are a logistic of the scaled logit gap (catches a lost scale or sign)."""
    D = 4
    K = [np.array([[[1, 0, 0, 0]], [[0, 2, 0, 0]]], dtype=np.float32)]
    V = [np.array([[[1, 0, 0, 0]], [[0, 1, 0, 0]]], dtype=np.float32)]
    q = np.array([[[3, 1, 0, 0]]], dtype=np.float32)
    w = custom([2], 1, 1, D, 16, K=K, V=V, q=q)
    o, lse = _attn_all(oracle_mod, w)
    z1, z2 = 3 / 2, 2 / 2          # scale 1/sqrt(4)
    w1 = 1 / (1 + np.exp(z2 - z1))
    assert o[0, 0, 0] == pytest.approx(w1, rel=1e-14)
    assert o[0, 0, 1] == pytest.approx(1 - w1, rel=1e-13)
    assert lse[0, 0] == pytest.approx(np.log(np.exp(z1) + np.exp(z2)), rel=1e-14)


def test_equal_keys_give_the_mean_and_log_count(oracle_mod):
    rng = np.random.default_rng(10)
    n, D = 45, 16
    k = rng.standard_normal(D).astype(np.float32)
    K = [np.tile(k, (n, 1, 1))]
    w = custom([n], 2, 1, D, 16, K=K, rng=rng)
    o, lse = _attn_all(oracle_mod, w)
    _, Vt = token_kv(w, 0, 0)
    kf = f(w.K[w.page_table[0, 0], 0, 0])
    for g in range(2):
        assert np.allclose(o[0, g], Vt.mean(axis=0), rtol=0, atol=1e-14)
        z = float(f(w.q[0, g]) @ kf) / 4.0
        assert lse[0, g] == pytest.approx(z + np.log(n), rel=1e-13, abs=1e-13)


def test_weights_are_a_distribution(oracle_mod):
    """V = one-hot per token exposes the weights: non-negative, sum 1, ratios e^{z_i - z_j}."""
    rng = np.random.default_rng(11)
    n = D = 24
    V = [np.eye(n, dtype=np.float32).reshape(n, 1, D)]
    w = custom([n], 1, 1, D, 16, V=V, rng=rng)
    o, _ = _attn_all(oracle_mod, w)
    wts = o[0, 0]
    assert np.all(wts > 0) and wts.sum() == pytest.approx(1.0, abs=1e-14)
    Kt, _ = token_kv(w, 0, 0)
    z = (Kt @ f(w.q[0, 0])) / np.sqrt(D)
    assert wts[3] / wts[7] == pytest.approx(np.exp(z[3] - z[7]), rel=1e-12)


def test_value_shift_and_constant_values(oracle_mod):
    """Weights sum to one: V + c gives o + c; constant V gives that constant."""
    rng = np.random.default_rng(12)
    V = [(rng.integers(-32, 32, size=(50, 1, 8)) / 8).astype(np.float32)]   # exact in bf16, also + 0.5
    K = [rng.standard_normal((50, 1, 8)).astype(np.float32)]
    q = rng.standard_normal((1, 2, 8)).astype(np.float32)
    o, _ = _attn_all(oracle_mod, custom([50], 2, 1, 8, 16, K=K, V=V, q=q))
    o2, _ = _attn_all(oracle_mod, custom([50], 2, 1, 8, 16, K=K, V=[V[0] + 0.5], q=q))
    assert np.allclose(o2, o + 0.5, rtol=0, atol=1e-13)
    o3, _ = _attn_all(oracle_mod, custom([50], 2, 1, 8, 16, K=K, q=q,
                                         V=[np.full((50, 1, 8), 1.25, dtype=np.float32)]))
    assert np.allclose(o3, 1.25, rtol=0, atol=1e-15)


def test_masked_slots_and_physical_layout_do_not_matter(oracle_mod):
    """Changing the bytes past len, or the physical page order, leaves every result unchanged."""
    rng = np.random.default_rng(13)
    K = [rng.standard_normal((n, 2, 16)).astype(np.float32) for n in (41, 70)]
    V = [rng.standard_normal((n, 2, 16)).astype(np.float32) for n in (41, 70)]
    q = rng.standard_normal((2, 4, 16)).astype(np.float32)
    pol = wl.BudgetPolicy("fixed", fixed_pages=3, sink_pages=1, local_pages=1)
    wa = custom([41, 70], 4, 2, 16, 16, K=K, V=V, q=q, permute=False, poison=True, policy=pol)
    wb = custom([41, 70], 4, 2, 16, 16, K=K, V=V, q=q, permute=True, poison=False,
                rng=np.random.default_rng(99), policy=pol)
    ra = oracle_mod.decode_step(wa, threads=1)
    rb = oracle_mod.decode_step(wb, threads=1)
    for key in ("scores", "sel", "nsel", "o", "lse"):
        assert np.array_equal(ra[key], rb[key]), key


def test_sparse_over_all_pages_equals_dense_decode(oracle_mod):
    w = wl.named("tiny", policy_over=dict(fixed_pages=64))
    o, lse = _attn_all(oracle_mod, w)
    od, lsed = oracle_mod.verify(w, 1, q=w.q.reshape(w.B, 1, w.H_q, w.D))
    assert np.allclose(o, od[:, 0], rtol=0, atol=1e-14)
    assert np.allclose(lse, lsed[:, 0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- a6 merge

def test_merge_of_any_page_partition_equals_unsplit(oracle_mod):
    rng = np.random.default_rng(14)
    w = custom([100, 61], 4, 2, 16, 16, rng=rng)
    o, lse = _attn_all(oracle_mod, w)
    P = w.max_pages_per_seq
    for S in (1, 2, 3, 7):
        cut = np.sort(rng.choice(np.arange(1, P), size=min(S - 1, P - 1), replace=False))
        parts = np.split(np.arange(P), cut)
        parts += [np.array([], dtype=int)] * (S - len(parts))   # empty splits: lse = -inf
        po, pl = [], []
        for part in parts:
            sel = np.full((w.B, w.H_kv, P), -1, dtype=np.int32)
            nsel = np.zeros((w.B, w.H_kv), dtype=np.int32)
            for b in range(w.B):
                mine = [p for p in part if p < w.pages(b)]
                sel[b, :, : len(mine)] = mine
                nsel[b, :] = len(mine)
            a, l = oracle_mod.sparse_attn(w, sel, nsel)
            po.append(a.reshape(-1, w.D))
            pl.append(l.reshape(-1))
        mo, ml = oracle_mod.merge(np.stack(po), np.stack(pl))
        assert np.allclose(mo, o.reshape(-1, w.D), rtol=0, atol=1e-13)
        assert np.allclose(ml, lse.reshape(-1), rtol=0, atol=1e-12)


def test_merge_of_empty_partials(oracle_mod):
    po = np.zeros((3, 2, 4))
    pl = np.full((3, 2), -np.inf)
    pl[1, 0] = 0.7
    po[1, 0] = [1, 2, 3, 4]
    o, lse = oracle_mod.merge(po, pl)
    assert np.array_equal(o[0], [1, 2, 3, 4]) and lse[0] == 0.7
    assert np.array_equal(o[1], np.zeros(4)) and lse[1] == -np.inf


# ---------------------------------------------------------------- a7 verify

def test_verify_is_causal_and_rows_match_shorter_dense_decodes(oracle_mod):
    rng = np.random.default_rng(15)
    T = 3
    w = custom([40, 19], 4, 2, 16, 16, T=T, rng=rng)
    o, lse = oracle_mod.verify(w, T)
    for t in range(T):
        wt = custom([40, 19], 4, 2, 16, 16, T=T, rng=np.random.default_rng(15))
        wt.seq_lens = (w.seq_lens - T + t + 1).astype(np.int32)
        ot, lt = oracle_mod.verify(wt, 1, q=np.ascontiguousarray(w.q_verify[:, t: t + 1]))
        assert np.array_equal(o[:, t], ot[:, 0]) and np.array_equal(lse[:, t], lt[:, 0])
    # future tokens: changing the last token's K/V leaves rows 0..T-2 unchanged
    w2 = custom([40, 19], 4, 2, 16, 16, T=T, rng=np.random.default_rng(15))
    for b in range(2):
        j = int(w2.seq_lens[b]) - 1
        w2.K[w2.page_table[b, j // 16], :, j % 16] = wl.f32_to_bf16_bits(np.full(16, 9.0, np.float32))
    o2, _ = oracle_mod.verify(w2, T)
    assert np.array_equal(o2[:, : T - 1], o[:, : T - 1])
    assert not np.array_equal(o2[:, T - 1], o[:, T - 1])


def test_verify_row_sees_exactly_len_minus_T_plus_t_plus_1_tokens(oracle_mod):
    """Identical keys: lse = z + log(visible count) pins the causal offset."""
    T, n, D = 4, 35, 8
    k = np.ones(D, dtype=np.float32)
    w = custom([n], 1, 1, D, 16, K=[np.tile(k, (n, 1, 1))], T=T, rng=np.random.default_rng(16))
    o, lse = oracle_mod.verify(w, T)
    for t in range(T):
        z = float(f(w.q_verify[0, t, 0]) @ k) / np.sqrt(D)
        assert lse[0, t, 0] == pytest.approx(z + np.log(n - T + t + 1), rel=1e-13, abs=1e-13)
