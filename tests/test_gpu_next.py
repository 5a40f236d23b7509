"""GPU parity of the rows that follow the core path, through the C ABI against the
fp64 oracle: the fused cache append + summary refresh (bit-exact)."""
import numpy as np
import pytest

import oracle
from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.gpu_helpers import Gpu, assert_close_outputs, compare_selection, np_bf16, summ_bits
from tests.helpers import custom

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _new_tokens(w, T, seed):
    rng = np.random.default_rng(seed)
    shape = (w.B, T, w.H_kv, w.D)
    return (wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32)),
            wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32)))


def _check_append(w, T, seed=0):
    g = Gpu(w)
    summ = g.summarize()                       # summaries of the cache before the append
    before = summ_bits(summ).copy()
    k_new, v_new = _new_tokens(w, T, seed)
    g.append(T, k_new, v_new, summ)
    assert g.sync_status() == 0
    K_ref, V_ref = oracle.append(w, T, k_new, v_new, threads=8)
    assert np.array_equal(_bits(g.d["K"]), K_ref), "K cache differs"
    assert np.array_equal(_bits(g.d["V"]), V_ref), "V cache differs"
    after = wl.Workload(**{**w.__dict__})
    after.K, after.V = K_ref, V_ref
    s_ref = oracle.summarize(after, threads=8)
    got = summ_bits(summ)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        touched = set(range(max(0, L - T) // w.page_size, (L - 1) // w.page_size + 1))
        for p in range(w.max_pages_per_seq):
            if p in touched:
                exp = wl.f32_to_bf16_bits(s_ref[w.page_table[b, p]].astype(np.float32))
                assert np.array_equal(got[b, :, p], exp), (b, p)
            else:
                assert np.array_equal(got[b, :, p], before[b, :, p]), (b, p, "untouched page changed")


@pytest.mark.parametrize("ps", [16, 32, 64])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("T", [1, 7, 40])
def test_append_refresh_bit_exact(ps, D, T):
    # lengths put the new tokens at a page start, mid-page, at a page end and across pages
    lens = [T, ps + 1, 2 * ps, 3 * ps + 5, 5 * ps - 1, 90]
    lens = [max(L, T) for L in lens]
    w = custom(lens, 4, 2, D, ps, rng=np.random.default_rng(ps + D + T))
    _check_append(w, T, seed=T)


@pytest.mark.parametrize("name,kw", [("q8b", dict(B=6, len_lo=700, len_hi=2200)),
                                     ("sweep", dict(page_size=32, B=3, len_lo=2000, len_hi=5000))])
def test_append_refresh_on_workloads(name, kw):
    w = wl.named(name, threads=4, **kw)
    _check_append(w, 1, seed=5)
    _check_append(w, 7, seed=6)


def test_append_rejects_short_sequences_without_touching_them():
    w = custom([3, 40], 4, 2, 64, 16, rng=np.random.default_rng(9))
    g = Gpu(w)
    summ = g.summarize()
    K0 = _bits(g.d["K"]).copy()
    k_new, v_new = _new_tokens(w, 5, 1)
    g.append(5, k_new, v_new, summ)
    assert g.sync_status() == 0x8
    K1 = _bits(g.d["K"])
    # sequence 0 (len 3 < T = 5) is untouched; sequence 1 got its tokens
    K_ref, _ = oracle.append(w, 5, k_new, v_new, seqs=[1])
    assert np.array_equal(K1, K_ref)
    assert np.array_equal(K1[w.page_table[0, 0]], K0[w.page_table[0, 0]])


def test_append_then_decode_matches_oracle_pipeline():
    """A decode step on the appended cache: refresh, score, select and attend equal the
    oracle run on the cache with the token written."""
    from tests.gpu_helpers import assert_close_outputs, compare_selection, np_bf16
    w = wl.named("q8b", threads=4, B=4, len_lo=900, len_hi=1500)
    g = Gpu(w)
    summ = g.summarize()
    k_new, v_new = _new_tokens(w, 1, 11)
    g.append(1, k_new, v_new, summ)
    sel, nsel, sc, _ = g.score_select(summ)
    o, lse, _ = g.sparse_attn(sel, nsel)
    assert g.sync_status() == 0
    after = wl.Workload(**{**w.__dict__})
    after.K, after.V = oracle.append(w, 1, k_new, v_new)
    ref = oracle.decode_step(after, threads=8)
    same = compare_selection(after, sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy(),
                             ref["sel"], ref["nsel"], ref["scores"])
    rows = [b for b in range(w.B) if all((b, h) in same for h in range(w.H_kv))]
    assert rows
    assert_close_outputs(np_bf16(o)[rows], ref["o"][rows], lse.cpu().numpy()[rows], ref["lse"][rows])


# ---------------------------------------------------------------- f2 speculative sampling

def _spec_gpu(p, q, draft, u_acc, u_res):
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    dev = "cuda"
    P = torch.from_numpy(np.ascontiguousarray(p, np.float32)).to(dev)
    Q = torch.from_numpy(np.ascontiguousarray(q, np.float32)).to(dev)
    Dr = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).to(dev)
    Ua = torch.from_numpy(np.ascontiguousarray(u_acc, np.float32)).to(dev)
    Ur = torch.from_numpy(np.ascontiguousarray(u_res, np.float32)).to(dev)
    B, k, n = p.shape
    nacc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    toks = torch.full((B, k + 1), -7, dtype=torch.int32, device=dev)
    spd.spec_accept(P, Q, Dr, Ua, Ur, nacc, toks)
    torch.cuda.synchronize()
    return nacc.cpu().numpy(), toks.cpu().numpy(), spd.spd_device_status(clear=True)


def _emitted_agrees(p, q, nacc, u_res, tok_gpu, tok_ref):
    """The kernel's emitted token against the oracle's.  The oracle draws on real
    numbers; the kernel weighs each token on a 2^-40 grid (each weight within one
    grid step of 2^40 times the real one, so running sums within n steps and the
    threshold within n + 1).  The tokens must be equal unless the oracle's threshold
    lies within (2n + 2) grid steps (plus the fp64 rounding of the sums) of a
    boundary of both tokens' intervals -- or the residual's real total is itself
    within the grid of zero, where the kernel may fall back to the target row."""
    if tok_gpu == tok_ref:
        return True
    k, n = p.shape[0], q.shape[-1]
    pos = lambda v: np.where(v > 0, v, 0.0)
    qr = q[nacc].astype(np.float64)
    w = pos(qr - p[nacc].astype(np.float64)) if nacc < k else pos(qr)
    if nacc < k and w.sum() <= (n + 1) * 2.0 ** -40:
        if w.sum() == 0:
            w = pos(qr)
        elif tok_gpu >= 0 and qr[tok_gpu] > 0:
            return True  # the kernel's grid saw no residual and drew from the target row
    C = np.cumsum(w)
    T = float(u_res) * C[-1]
    band = (2 * n + 2) * 2.0 ** -40 + 4 * n * 2.0 ** -53 * C[-1]

    def near(x):
        if x < 0:
            return False
        lo = C[x - 1] if x > 0 else 0.0
        return abs(T - lo) <= band or abs(C[x] - T) <= band
    return near(tok_ref) and near(tok_gpu)


def _compare_spec(d):
    """Accept counts and accepted drafts equal to the oracle's (the same exact fp64
    test), the emitted token equal unless the draw lies within the grid band."""
    import oracle as orc
    na_r, tk_r = orc.spec_accept(d["p"], d["q"], d["draft"], d["u_acc"], d["u_res"])
    na_g, tk_g, st = _spec_gpu(d["p"], d["q"], d["draft"], d["u_acc"], d["u_res"])
    assert st == 0, st
    assert np.array_equal(na_g, na_r)
    for b in range(len(na_r)):
        a = int(na_r[b])
        assert tk_g[b, :a].tolist() == tk_r[b, :a].tolist() and np.all(tk_g[b, a + 1:] == -1), b
        assert _emitted_agrees(d["p"][b], d["q"][b], a, d["u_res"][b], int(tk_g[b, a]), int(tk_r[b, a])), \
            (b, tk_g[b, a], tk_r[b, a])
    return na_r


def test_spec_accept_hand_worked_cases_on_gpu():
    """The hand-worked cases of the rule (equal, or within the grid band), and the
    kernel's own grid cases exactly."""
    from tests.test_oracle_pins_next import _golden_spec
    for k, n, p, q, draft, uacc, ures, nacc, toks in _golden_spec():
        na, tk, st = _spec_gpu(p[None], q[None], np.array([draft]), np.array([uacc], np.float32),
                               np.array([ures], np.float32))
        assert st == 0 and na[0] == nacc and tk[0, :nacc].tolist() == toks[:nacc], (k, n, na, tk)
        assert _emitted_agrees(p, q, nacc, np.float32(ures), int(tk[0, nacc]), toks[nacc]), (k, n, tk, toks)
    for k, n, p, q, draft, uacc, ures, nacc, toks in _golden_spec("spec_accept_grid_cases.txt"):
        na, tk, st = _spec_gpu(p[None], q[None], np.array([draft]), np.array([uacc], np.float32),
                               np.array([ures], np.float32))
        assert st == 0 and na[0] == nacc and tk[0].tolist() == toks, (k, n, na, tk)


@pytest.mark.parametrize("n", [1000, 4099, 151936])
def test_spec_accept_matches_oracle(n):
    d = wl.spec_inputs(B=24, k=6, n=n, seed=77 + n)
    nacc = _compare_spec(d)
    assert nacc.min() < 6 and nacc.max() > 0     # both rejections and acceptances occur


def test_spec_accept_all_accepted_zero_residual_and_empty_rows():
    rng = np.random.default_rng(5)
    n, k, B = 4096, 6, 6
    p = rng.random((B, k, n)).astype(np.float32)
    q = np.concatenate([p, rng.random((B, 1, n)).astype(np.float32)], axis=1)
    draft = rng.integers(0, n, size=(B, k)).astype(np.int32)
    u_acc = (rng.random((B, k)) * 0.999).astype(np.float32)
    # row 1: target = drafter / 2 at position 2, rejected there with a zero residual
    q[1, 2] = p[1, 2] * 0.5
    u_acc[1, 2] = 0.75
    # row 2: the bonus row is all zero -> no token
    q[2, k] = 0.0
    # row 3: rejected at 0 with residual and target both zero -> no token
    q[3, 0] = 0.0
    d = dict(p=p, q=q, draft=draft, u_acc=u_acc, u_res=rng.random(B, dtype=np.float32))
    nacc = _compare_spec(d)
    assert nacc.tolist() == [6, 2, 6, 0, 6, 6]
    na_g, tk_g, _ = _spec_gpu(p, q, draft, u_acc, d["u_res"])
    assert tk_g[2, k] == -1 and tk_g[3, 0] == -1


def _grid_row_mixed(n, rng):
    """A residual row (p, q) whose grid weights W = max(0, floor(2^40 q) - floor(2^40 p))
    are known exactly: most tiles hold only values below 2^-10 (the kernel's 32-bit
    form), a few also hold values of 2^-10 and above, negative residuals and
    subnormals (its 64-bit form).  The total stays below 2^23, so a float32 u can
    place the draw's threshold on any integer."""
    g = 2.0 ** -40
    p = np.zeros(n, np.float64)
    q = np.zeros(n, np.float64)
    tiles = n // 128
    wide = set(rng.choice(tiles, size=max(3, tiles // 6), replace=False).tolist())
    for t in range(tiles):
        base = t * 128
        xs = rng.choice(128, size=40, replace=False) + base
        for x in xs[:24]:                                   # tiny: W = m
            q[x] = int(rng.integers(1, 3000)) * g
        for x in xs[24:30]:                                 # just below 2^-10: W = 64 j
            v = 2.0 ** -10 - int(rng.integers(1, 50)) * 2.0 ** -34
            q[x], p[x] = v, v - int(rng.integers(1, 40)) * 2.0 ** -34
        q[xs[30]] = 2.0 ** -140                             # subnormal: W = 0
        if t in wide:
            q[xs[31]], p[xs[31]] = 2.0 ** -10 + 2.0 ** -33, 2.0 ** -10           # W = 128
            q[xs[32]], p[xs[32]] = 2.0 ** -9, 2.0 ** -9 - 3 * 2.0 ** -33         # W = 384
            q[xs[33]], p[xs[33]] = 0.25 + int(rng.integers(1, 4)) * 2.0 ** -24, 0.25   # W = 2^16 j
            q[xs[34]], p[xs[34]] = 0.5, 0.5 + 2.0 ** -24                       # residual < 0: W = 0
            q[xs[35]], p[xs[35]] = 2.0 ** -10, 2.0 ** -10                     # W = 0 at the bound
    p32, q32 = p.astype(np.float32), q.astype(np.float32)
    assert np.array_equal(p32.astype(np.float64), p) and np.array_equal(q32.astype(np.float64), q)
    F = lambda v: int(np.floor(np.ldexp(float(v), 40))) if v > 0 else 0
    W = [max(0, F(qq) - F(pp)) for qq, pp in zip(q32.tolist(), p32.tolist())]
    return p32, q32, W


def test_spec_accept_grid_sums_exact_in_32_and_64_bit_tiles():
    """The draw's running sums are exact on the 2^-40 grid in both of the kernel's
    forms of a tile: thresholds on either side of running-sum boundaries spread
    over every tile, where one grid step of error anywhere before the boundary
    moves the token.  (The kernel's documented arithmetic, as in the grid cases.)"""
    from fractions import Fraction
    rng = np.random.default_rng(2024)
    n, k = 4096, 2
    p0, q0, W = _grid_row_mixed(n, rng)
    C = np.cumsum(np.array(W, dtype=np.int64))
    total = int(C[-1])
    assert 0 < total < 2 ** 23
    nz = [x for x in range(n) if W[x] > 0]
    picks = [nz[i] for i in np.linspace(1, len(nz) - 1, 24).astype(int)]
    thresholds, expect = [], []
    for x in picks:
        for T in (int(C[x - 1]), int(C[x]) - 1):   # both draw x
            thresholds.append(T)
            expect.append(x)
    B = len(thresholds)
    u = []
    for T in thresholds:
        f = np.float32(float(Fraction(2 * T + 1, 2 * total)))
        while int(Fraction(float(f)) * total) > T:
            f = np.nextafter(f, np.float32(0))
        while int(Fraction(float(f)) * total) < T:
            f = np.nextafter(f, np.float32(1))
        assert int(Fraction(float(f)) * total) == T
        u.append(f)
    zero = [x for x in range(n) if p0[x] == 0 and q0[x] == 0][0]   # rejected: u_acc * 0 < 0 fails
    p = np.broadcast_to(p0, (B, k, n)).copy()
    q = np.broadcast_to(q0, (B, k + 1, n)).copy()
    draft = np.full((B, k), zero, np.int32)
    na, tk, st = _spec_gpu(p, q, draft, np.full((B, k), 0.5, np.float32), np.array(u, np.float32))
    assert st == 0 and np.all(na == 0)
    assert tk[:, 0].tolist() == expect
    assert np.all(tk[:, 1:] == -1)


def test_spec_accept_bad_draft_token_sets_status():
    d = wl.spec_inputs(B=3, k=2, n=512, seed=3)
    d["draft"][1, 1] = 512
    na, tk, st = _spec_gpu(d["p"], d["q"], d["draft"], d["u_acc"], d["u_res"])
    assert st == 0x10 and na[1] == 0 and np.all(tk[1] == -1)


# ---------------------------------------------------------------- f3 top-p selection

TOP_P_TOL = 1e-3   # relative weight tolerance at the top_p boundary (fp32 scores, 2^-31 grid)


def _check_top_p(w, top_p, scale, k_max=None):
    import dataclasses
    from tests.gpu_helpers import TIE_BAND
    k_max = k_max or w.max_pages_per_seq
    pol = dataclasses.replace(w.policy, mode="top_p", top_p=top_p, score_scale=scale)
    g = Gpu(w)
    summ = g.summarize()
    sel, nsel, sc, _ = g.score_select(summ, policy=pol, k_max=k_max)
    assert g.sync_status() == 0
    sel_g, nsel_g, sc_g = sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy().astype(np.float64)
    sc_o = oracle.scores(w, oracle.summarize(w, threads=8), threads=8)
    sel_o, nsel_o = oracle.select_top_p(w, sc_o, top_p, scale, k_max=k_max, policy=pol)
    exact = 0
    for b in range(w.B):
        P = w.pages(b)
        sink, local = min(pol.sink_pages, P), min(pol.local_pages, P)
        mand = {p for p in range(P) if p < sink or p >= P - local}
        for h in range(w.H_kv):
            g_set = sel_g[b, h, : nsel_g[b, h]].tolist()
            o_set = sel_o[b, h, : nsel_o[b, h]].tolist()
            assert g_set == sorted(set(g_set)) and mand <= set(g_set)
            if g_set == o_set:
                exact += 1
                continue
            s = sc_o[b, h, :P]
            wgt = np.exp(scale * (s - s.max()))
            need = top_p * wgt.sum()
            order = sorted((p for p in range(P) if p not in mand), key=lambda p: (-s[p], p))
            n = len(g_set) - len(mand)
            held = lambda m: wgt[list(mand)].sum() + wgt[order[:m]].sum()
            # the count is right up to the weight tolerance
            assert n == k_max - len(mand) or held(n) >= need * (1 - TOP_P_TOL), (b, h, n)
            assert n == 0 or held(n - 1) < need * (1 + TOP_P_TOL), (b, h, n)
            # the pages are the best n by score, up to the tie band
            kth = s[order[n - 1]] if n else np.inf
            band = {p for p in order if abs(s[p] - kth) <= TIE_BAND * abs(kth)}
            assert set(g_set) - band == (set(order[:n]) | mand) - band, (b, h)
    return exact


@pytest.mark.parametrize("top_p", [0.0, 0.5, 0.9, 0.99, 1.0])
def test_top_p_selection_matches_oracle(top_p):
    w = wl.named("q8b", threads=4, B=5, len_lo=700, len_hi=2200)
    exact = _check_top_p(w, top_p, 1.0 / np.sqrt(w.D))
    assert exact >= w.B * w.H_kv // 2


@pytest.mark.parametrize("name,kw,scale", [
    ("sweep", dict(page_size=32, B=3, len_lo=2000, len_hi=6000), 0.05),
    ("longtail", dict(B=2, len_lo=4000, len_hi=9000, T=1), 0.2),
    ("tiny", dict(), 0.125)])
def test_top_p_selection_other_workloads(name, kw, scale):
    w = wl.named(name, threads=4, **kw)
    _check_top_p(w, 0.8, scale)
    _check_top_p(w, 0.8, scale, k_max=max(8, w.policy.sink_pages + w.policy.local_pages))


def test_top_p_then_sparse_attention():
    """The top-p selection feeds the sparse attention like a top-k one."""
    import dataclasses
    from tests.gpu_helpers import assert_close_outputs, np_bf16
    w = wl.named("q8b", threads=4, B=3, len_lo=800, len_hi=1500)
    pol = dataclasses.replace(w.policy, mode="top_p", top_p=0.7, score_scale=1.0 / np.sqrt(w.D))
    g = Gpu(w)
    sel, nsel, _, _ = g.score_select(g.summarize(), policy=pol, k_max=w.max_pages_per_seq)
    o, lse, _ = g.sparse_attn(sel, nsel)
    assert g.sync_status() == 0
    o_ref, lse_ref = oracle.sparse_attn(w, sel.cpu().numpy(), nsel.cpu().numpy(), threads=8)
    assert_close_outputs(np_bf16(o), o_ref, lse.cpu().numpy(), lse_ref)


# ---------------------------------------------------------------- f1 fused into scoring

@pytest.mark.parametrize("name,kw", [("q8b", dict(B=6, len_lo=700, len_hi=2200)),
                                     ("sweep", dict(page_size=32, B=3, len_lo=2000, len_hi=5000)),
                                     ("sweep", dict(page_size=64, B=3, len_lo=2000, len_hi=5000)),
                                     ("tiny", dict())])
def test_fused_append_score_select_equals_the_two_calls(name, kw):
    """pages_append_score_select gives the same bits as kv_append_refresh(T=1) then
    pages_score_select: cache, summaries, scores and selection."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = wl.named(name, threads=4, **kw)
    k_new, v_new = _new_tokens(w, 1, 21)
    outs = []
    for one_call in (False, True):
        g = Gpu(w)
        summ = g.summarize()
        kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda()
        vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda()
        sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
        nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((w.B, w.H_kv, w.max_pages_per_seq), float("nan"), device="cuda")
        ws = g.ws(spd.spd_score_select_workspace_size(g.dims))
        d = g.d
        if one_call:
            spd.pages_append_score_select(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn,
                                          d["q"], summ, w.policy, sel, nsel, w.k_max, ws, scores=sc)
        else:
            spd.kv_append_refresh(g.dims, 1, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, summ)
            spd.pages_score_select(g.dims, d["q"], summ, d["seq_lens"], w.policy, sel, nsel, w.k_max, ws,
                                   scores=sc)
        assert g.sync_status() == 0
        outs.append([_bits(d["K"]), _bits(d["V"]), summ_bits(summ), sel.cpu().numpy(), nsel.cpu().numpy(),
                     sc.view(torch.int32).cpu().numpy()])
    for x, y, what in zip(outs[0], outs[1], ["K", "V", "summ", "sel", "nsel", "scores"]):
        assert np.array_equal(x, y), what


def test_fused_append_flags_empty_sequences_and_bad_pages():
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = custom([0, 40, 50], 4, 2, 64, 16, rng=np.random.default_rng(3))
    w.page_table[2, 3] = w.num_phys_pages + 9      # the last page of sequence 2
    g = Gpu(w)
    summ = torch.zeros((w.B, w.H_kv, w.max_pages_per_seq, 2, w.D), dtype=torch.bfloat16, device="cuda")
    k_new, v_new = _new_tokens(w, 1, 4)
    kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda()
    vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda()
    sel = torch.zeros((w.B, w.H_kv, w.k_max), dtype=torch.int32, device="cuda")
    nsel = torch.zeros((w.B, w.H_kv), dtype=torch.int32, device="cuda")
    ws = g.ws(spd.spd_score_select_workspace_size(g.dims))
    d = g.d
    spd.pages_append_score_select(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, d["q"],
                                  summ, w.policy, sel, nsel, w.k_max, ws)
    assert g.sync_status() == 0x8 | 0x1


# ---------------------------------------------------------------- the decode step in one call

def _top_p(w):
    """The workload with a top-p budget (0.9 of the page weight) and room for every page."""
    import dataclasses
    import math
    w.policy = dataclasses.replace(w.policy, mode="top_p", top_p=0.9, score_scale=1.0 / math.sqrt(w.D))
    w.k_max = w.max_pages_per_seq
    return w


def _wide_table(w, max_pages=1040):
    """The workload with a page table (and summary array) of max_pages slots per sequence."""
    extra = max_pages - w.max_pages_per_seq
    w.page_table = np.pad(w.page_table, ((0, 0), (0, extra)), constant_values=-1)
    w.max_pages_per_seq = max_pages
    return w


# name, overrides, append, variant.  The step chains its kernels row by row in every
# case; the row count (B x 8 KV heads, tiny: x 2) sets the chained selection's CTA width
# on a 152-SM part: 128 threads above two rows per SM, 256 up to two, 512 up to one
# (few rows: split attention units and the fused merge)
STEP_CASES = [
    ("q8b", dict(), True, None),                                            # full size, 512 rows
    ("q8b", dict(B=5, len_lo=700, len_hi=2200), True, None),                # 40 rows, split units
    ("q17b", dict(B=48, len_lo=2000, len_hi=6000), False, None),            # 384 rows
    ("q8b", dict(B=30, len_lo=2000, len_hi=5000), True, None),              # 240 rows
    ("longtail", dict(B=2, len_lo=4000, len_hi=9000, T=1), True, None),     # 16 rows, split units
    ("q8b", dict(B=40, len_lo=2000, len_hi=5000, page_size=32), True, None),
    ("q8b", dict(B=40, len_lo=2000, len_hi=5000, page_size=64), False, None),
    ("tiny", dict(B=200), True, None),                                      # D = 64, 400 rows
    ("tiny", dict(B=1000), True, None),                                     # 2,000 rows: ~7 claimed per CTA
    ("q8b", dict(B=40, len_lo=2000, len_hi=5000), True, "top_p"),
    ("q8b", dict(B=40, len_lo=2000, len_hi=5000), True, "wide_table"),
]


@pytest.mark.parametrize("name,kw,append,variant", STEP_CASES)
def test_decode_step_equals_the_separate_calls(name, kw, append, variant):
    """sparse_decode_step gives the bits of append + score_select + sparse attention, for
    two steps in a row with different queries through one workspace (so the chain's
    counters must have been reset by the first), chained row by row or as calls in turn,
    at page sizes 16 / 32 / 64, head dims 64 / 128, top-p budgets and page tables
    wider than the sequences."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = wl.named(name, threads=8, **kw)
    if variant == "top_p":
        w = _top_p(w)
    elif variant == "wide_table":
        w = _wide_table(w)
    k_new, v_new = _new_tokens(w, 1, 31)
    rng = np.random.default_rng(32)
    q2 = torch.from_numpy(wl.f32_to_bf16_bits(rng.standard_normal(w.q.shape).astype(np.float32))).view(
        torch.bfloat16).cuda()
    outs = []
    for one_call in (False, True):
        g = Gpu(w)
        summ = g.summarize()
        d = g.d
        kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda() if append else None
        vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda() if append else None
        sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
        nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
        o = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.B, w.H_q), float("nan"), device="cuda")
        ws = g.ws(spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max))
        wss = g.ws(spd.spd_score_select_workspace_size(g.dims))
        wsa = g.ws(spd.spd_sparse_decode_workspace_size(g.dims, w.k_max, 0))
        res = []
        for q in (d["q"], q2):
            if one_call:
                spd.sparse_decode_step(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, q,
                                       summ, w.policy, sel, nsel, w.k_max, o, ws, lse=lse)
            else:
                if append:
                    spd.kv_append_refresh(g.dims, 1, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn,
                                          summ)
                spd.pages_score_select(g.dims, q, summ, d["seq_lens"], w.policy, sel, nsel, w.k_max, wss)
                spd.sparse_decode_attn(g.dims, q, d["K"], d["V"], d["page_table"], d["seq_lens"], sel, nsel,
                                       w.k_max, o, wsa, lse=lse)
            assert g.sync_status() == 0
            res += [_bits(d["K"]), summ_bits(summ), sel.cpu().numpy(), nsel.cpu().numpy(), _bits(o),
                    lse.view(torch.int32).cpu().numpy()]
        outs.append(res)
    names = ["K", "summ", "sel", "nsel", "o", "lse"] * 2
    for x, y, what in zip(outs[0], outs[1], names):
        assert np.array_equal(x, y), what


def _edge_lens(n_seq, ps):
    """Lengths cycling through the edge cases: empty, one token, a page minus one, a
    page, a page plus one, and longer ragged rows."""
    pattern = [0, 1, ps - 1, ps, ps + 1, 2 * ps + 1, 100, 20 * ps + 3]
    return [pattern[i % len(pattern)] for i in range(n_seq)]


@pytest.mark.parametrize("case", ["q17b_short", "tiny_d64", "edges_d128", "edges_d64_ps32", "rows192",
                                  "rows64_long"])
def test_decode_step_against_the_oracle(case):
    """The chained decode step (no append) against the fp64 oracle: selections equal
    outside the tie band, outputs within tolerance on the rows selected alike, empty
    rows give o = 0 and lse = -inf.  The row counts cover each width of the chained
    selection on a 152-SM part: 320 / 400 rows (128 threads), 192 rows (256) and 64 rows
    of 750-1,250 pages (512 threads, several radix levels, split attention units)."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    if case == "q17b_short":
        w = wl.named("q17b", threads=8, B=40, len_lo=300, len_hi=1500,
                     policy=wl.BudgetPolicy("fixed", fixed_pages=24, sink_pages=1, local_pages=4))
    elif case == "tiny_d64":
        w = wl.named("tiny", threads=8, B=200)
    elif case == "rows192":
        w = wl.named("tiny", threads=8, B=96, len_lo=3000, len_hi=8000,
                     policy=wl.BudgetPolicy("fixed", fixed_pages=24, sink_pages=1, local_pages=4))
    elif case == "rows64_long":
        w = wl.named("tiny", threads=8, B=32, len_lo=12000, len_hi=20000,
                     policy=wl.BudgetPolicy("fraction", frac_num=1, frac_den=16, sink_pages=1, local_pages=4))
    else:
        D, ps = (128, 16) if case == "edges_d128" else (64, 32)
        pol = wl.BudgetPolicy("fixed", fixed_pages=3, sink_pages=1, local_pages=1)
        w = custom(_edge_lens(200, ps), 4, 2, D, ps, rng=np.random.default_rng(D + ps), policy=pol, k_max=8)
    ref = oracle.decode_step(w, threads=8)
    g = Gpu(w)
    summ = g.summarize()
    d = g.d
    sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
    nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
    o = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H_q), float("nan"), device="cuda")
    ws = g.ws(spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max))
    spd.sparse_decode_step(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], None, None, d["q"], summ,
                           w.policy, sel, nsel, w.k_max, o, ws, lse=lse)
    assert g.sync_status() == 0
    _, _, sc, _ = g.score_select(summ)   # the GPU's own scores, for the validity check
    same = compare_selection(w, sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy(), ref["sel"], ref["nsel"],
                             ref["scores"])
    seqs_same = sorted({b for b, h in same if all((b, hh) in same for hh in range(w.H_kv))})
    assert len(seqs_same) >= w.B // 2
    assert_close_outputs(np_bf16(o)[seqs_same], ref["o"][seqs_same], lse.cpu().numpy()[seqs_same],
                         ref["lse"][seqs_same], what=f"decode step {case}")
    empty = [b for b in range(w.B) if int(w.seq_lens[b]) == 0]
    if empty:
        assert not np_bf16(o)[empty].any()
        assert np.all(np.isneginf(lse.cpu().numpy()[empty]))
        assert not nsel.cpu().numpy()[empty].any()


def test_decode_step_wait_runs_out_and_the_next_call_is_clean():
    """A bounded wait that runs out, on purpose and safely: a step workspace whose two
    tile counters start past the end, so each scoring warp scores its fixed first
    chunk and no more.  The rows beyond those chunks never get all their scores, so
    their selections (waiting for the scores) and attention units (waiting for the
    selections) give up after a 1 ms limit.  The call returns, SPD_DEV_TIMEOUT is set,
    and the same step on a fresh zeroed workspace then gives the bits of a clean run
    on a fresh cache (the append writes the same token again)."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = wl.named("q8b", threads=8, len_lo=3000, len_hi=6000)
    k_new, v_new = _new_tokens(w, 1, 41)
    kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda()
    vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda()

    def setup():
        g = Gpu(w)
        summ = g.summarize()
        out = dict(sel=torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda"),
                   nsel=torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda"),
                   o=torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda"),
                   lse=torch.full((w.B, w.H_q), float("nan"), device="cuda"))
        return g, summ, out

    def step(g, summ, out, ws):
        d = g.d
        spd.sparse_decode_step(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, d["q"], summ,
                               w.policy, out["sel"], out["nsel"], w.k_max, out["o"], ws, lse=out["lse"])
        torch.cuda.synchronize()

    def bits(g, summ, out):
        return [_bits(g.d["K"]), summ_bits(summ), out["sel"].cpu().numpy(), out["nsel"].cpu().numpy(),
                _bits(out["o"]), out["lse"].view(torch.int32).cpu().numpy()]

    g, summ, out = setup()
    ws_bytes = spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max)
    ws = g.ws(ws_bytes)
    chain = -(-spd.spd_score_select_workspace_size(g.dims) // 256) * 256  # the chain part of the workspace
    ws[chain:chain + 16].view(torch.int64).fill_(1 << 40)                 # both tile counters past the end
    spd.spd_set_wait_limit_ns(1_000_000)
    try:
        step(g, summ, out, ws)
    finally:
        spd.spd_set_wait_limit_ns(2_000_000_000)
    st = spd.spd_device_status(clear=True)
    assert st & spd.DEV_TIMEOUT, st
    step(g, summ, out, g.ws(ws_bytes))               # a fresh zeroed workspace
    assert spd.spd_device_status(clear=True) == 0
    g2, summ2, out2 = setup()
    step(g2, summ2, out2, g2.ws(ws_bytes))            # a clean run
    assert spd.spd_device_status(clear=True) == 0
    for x, y, what in zip(bits(g, summ, out), bits(g2, summ2, out2), ["K", "summ", "sel", "nsel", "o", "lse"]):
        assert np.array_equal(x, y), what


def test_decode_step_bad_page_id_sets_status_and_does_not_fault():
    """A page-table entry outside the cache in the chained step (where the selection
    hands the attention each selected page's physical page): the sink page of one
    sequence, always selected, points past the last physical page.  The step sets
    SPD_DEV_BAD_PAGE, skips that page, faults nowhere, and the other sequences get the
    bits of a run on the good table; the next call on the good table is clean."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = wl.named("q17b", threads=8, B=16, len_lo=300, len_hi=1500,
                 policy=wl.BudgetPolicy("fixed", fixed_pages=24, sink_pages=1, local_pages=4))

    def run(page_table):
        g = Gpu(w)
        summ = g.summarize()
        d = g.d
        sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
        nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
        o = torch.zeros((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros((w.B, w.H_q), device="cuda")
        ws = g.ws(spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max))
        spd.sparse_decode_step(g.dims, d["K"], d["V"], page_table(d), d["seq_lens"], None, None, d["q"], summ,
                               w.policy, sel, nsel, w.k_max, o, ws, lse=lse)
        torch.cuda.synchronize()
        return spd.spd_device_status(clear=True), _bits(o), lse.view(torch.int32).cpu().numpy()

    def bad_table(d):
        t = d["page_table"].clone()
        t[3, 0] = w.num_phys_pages + 5
        return t

    st_bad, o_bad, lse_bad = run(bad_table)
    assert st_bad == spd.DEV_BAD_PAGE, st_bad
    st_good, o_good, lse_good = run(lambda d: d["page_table"])
    assert st_good == 0, st_good
    others = [b for b in range(w.B) if b != 3]
    assert np.array_equal(o_bad[others], o_good[others])
    assert np.array_equal(lse_bad[others], lse_good[others])


def test_decode_step_ties_go_to_lower_pages():
    """Pages with identical keys score alike: the chained step takes the mandatory pages
    and then the lowest page ids, at 41 and at 100 pages per row."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    ps, D, H_kv = 16, 64, 2
    lens = [16 * 40 + 5 if i % 2 == 0 else 16 * 99 + 1 for i in range(200)]
    rng = np.random.default_rng(77)
    K = []
    for n in lens:
        tok = rng.standard_normal((1, H_kv, D)).astype(np.float32)
        K.append(np.repeat(tok, n, axis=0))
    pol = wl.BudgetPolicy("fixed", fixed_pages=8, sink_pages=1, local_pages=1)
    w = custom(lens, 4, H_kv, D, ps, rng=rng, K=K, policy=pol, k_max=8)
    g = Gpu(w)
    summ = g.summarize()
    d = g.d
    sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
    nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
    o = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    ws = g.ws(spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max))
    spd.sparse_decode_step(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], None, None, d["q"], summ,
                           w.policy, sel, nsel, w.k_max, o, ws)
    assert g.sync_status() == 0
    sel_h, nsel_h = sel.cpu().numpy(), nsel.cpu().numpy()
    ref = oracle.decode_step(w, threads=8)
    for b in range(w.B):
        P = w.pages(b)
        expect = [0, 1, 2, 3, 4, 5, 6, P - 1]
        for h in range(H_kv):
            assert nsel_h[b, h] == 8
            assert sel_h[b, h].tolist() == expect, (b, h, sel_h[b, h].tolist())
            assert ref["sel"][b, h, :8].tolist() == expect


def test_rollouts_sharing_prompt_pages():
    """A group of rollouts of one prompt (as in a GRPO group) shares the prompt's
    physical pages: every sequence's page table points at the same 21 prefix pages,
    followed by pages of its own.  The summaries are stored per sequence, so each
    sharer gets its own copy of a shared page's summary: the copies are identical
    and equal the oracle's; the one-call decode step (each sequence appending to a
    page of its own) then matches the oracle on every sequence."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    ps, H_q, H_kv, D, shared = 16, 8, 2, 128, 21
    lens = [shared * ps + 3, shared * ps + 40, shared * ps + 200, shared * ps + 517]
    pol = wl.BudgetPolicy("fixed", fixed_pages=12, sink_pages=1, local_pages=2)
    w = custom(lens, H_q, H_kv, D, ps, rng=np.random.default_rng(71), policy=pol, k_max=12)
    for b in range(1, w.B):        # sequences 1.. reuse sequence 0's prompt pages
        w.page_table[b, :shared] = w.page_table[0, :shared]
    k_new, v_new = _new_tokens(w, 1, 72)
    K2, V2 = oracle.append(w, 1, k_new, v_new)   # appends land in pages of each sequence's own
    import dataclasses
    w2 = dataclasses.replace(w, K=K2, V=V2)
    ref = oracle.decode_step(w2, threads=4)
    g = Gpu(w)
    summ = g.summarize()
    d = g.d
    got = summ_bits(summ)
    for b in range(1, w.B):
        assert np.array_equal(got[b, :, :shared], got[0, :, :shared]), b
    kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda()
    vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda()
    sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
    nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
    o = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H_q), float("nan"), device="cuda")
    ws = g.ws(spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max))
    spd.sparse_decode_step(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, d["q"], summ,
                           w.policy, sel, nsel, w.k_max, o, ws, lse=lse)
    assert g.sync_status() == 0
    got = summ_bits(summ)
    for b in range(w.B):
        for p in range(w.pages(b)):
            exp = wl.f32_to_bf16_bits(ref["summ"][w.page_table[b, p]].astype(np.float32))
            assert np.array_equal(got[b, :, p], exp), (b, p)
    _, _, sc, _ = g.score_select(summ)
    same = compare_selection(w2, sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy(), ref["sel"],
                             ref["nsel"], ref["scores"])
    rows = [b for b in range(w.B) if all((b, h) in same for h in range(w.H_kv))]
    assert len(rows) >= 3
    assert_close_outputs(np_bf16(o)[rows], ref["o"][rows], lse.cpu().numpy()[rows], ref["lse"][rows],
                         what="shared prompt pages")
