"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on small
seeded cases of every workload (several tiles, ragged tails) and on edge cases."""
import numpy as np
import pytest

import oracle
from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.gpu_helpers import (Gpu, assert_close_outputs, compare_selection, np_bf16, summ_bits)
from tests.helpers import custom

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": dict(name="tiny"),
    "q17b": dict(name="q17b", B=6, len_lo=300, len_hi=3000, policy_over=dict(fixed_pages=24)),
    "q8b": dict(name="q8b", B=5, len_lo=700, len_hi=2200),
    "sweep16": dict(name="sweep", page_size=16, B=4, len_lo=2000, len_hi=9000),
    "sweep32": dict(name="sweep", page_size=32, B=4, len_lo=2000, len_hi=9000),
    "sweep64": dict(name="sweep", page_size=64, B=4, len_lo=2000, len_hi=9000),
    "longtail": dict(name="longtail", B=3, len_lo=4000, len_hi=9000, T=1),
}


def small(key):
    kw = dict(SMALL[key])
    name = kw.pop("name")
    return wl.named(name, threads=4, **kw)


@pytest.fixture(scope="module", params=sorted(SMALL))
def case(request):
    w = small(request.param)
    ref = oracle.decode_step(w, threads=8)
    g = Gpu(w)
    return request.param, w, ref, g


def test_summaries_bit_exact(case):
    _, w, ref, g = case
    summ = g.summarize()
    assert g.sync_status() == 0
    got = summ_bits(summ)
    for b in range(w.B):
        for p in range(w.pages(b)):
            exp = wl.f32_to_bf16_bits(ref["summ"][w.page_table[b, p]].astype(np.float32))
            assert np.array_equal(got[b, :, p], exp), (b, p)


def test_scores_and_selection(case):
    _, w, ref, g = case
    summ = g.summarize()
    sel, nsel, sc, _ = g.score_select(summ)
    assert g.sync_status() == 0
    sc_g = sc.cpu().numpy().astype(np.float64)
    for b in range(w.B):
        P = w.pages(b)
        d = np.abs(sc_g[b, :, :P] - ref["scores"][b, :, :P])
        assert np.all(d <= 2e-5 * (1 + np.abs(ref["scores"][b, :, :P]))), (b, d.max())
    compare_selection(w, sel.cpu().numpy(), nsel.cpu().numpy(), sc_g, ref["sel"], ref["nsel"],
                      ref["scores"])


def test_sparse_attention_on_the_oracle_selection(case):
    key, w, ref, g = case
    for splits in (0, 1, 2, 3):
        o, lse, _ = g.sparse_attn(ref["sel"], ref["nsel"], num_splits=splits)
        assert g.sync_status() == 0
        assert_close_outputs(np_bf16(o), ref["o"], lse.cpu().numpy(), ref["lse"],
                             what=f"{key} sparse splits={splits}")


def test_full_pipeline(case):
    key, w, ref, g = case
    summ = g.summarize()
    sel, nsel, sc, _ = g.score_select(summ)
    o, lse, _ = g.sparse_attn(sel, nsel)
    assert g.sync_status() == 0
    same = compare_selection(w, sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy(),
                             ref["sel"], ref["nsel"], ref["scores"])
    seqs_same = sorted({b for b, h in same if all((b, hh) in same for hh in range(w.H_kv))})
    assert len(seqs_same) >= 1
    assert_close_outputs(np_bf16(o)[seqs_same], ref["o"][seqs_same],
                         lse.cpu().numpy()[seqs_same], ref["lse"][seqs_same], what=f"{key} pipeline")


def test_dense_verify(case):
    key, w, ref, g = case
    T = w.T or 1
    q = w.q_verify if w.T else w.q.reshape(w.B, 1, w.H_q, w.D)
    o_ref, lse_ref = oracle.verify(w, T, q=np.ascontiguousarray(q), threads=8)
    qd = g.torch.from_numpy(np.ascontiguousarray(q)).view(g.torch.bfloat16).cuda()
    for splits in (0, 1, 3):
        o, lse, _ = g.verify(T, q=qd, num_splits=splits)
        assert g.sync_status() == 0
        assert_close_outputs(np_bf16(o), o_ref, lse.cpu().numpy(), lse_ref,
                             what=f"{key} verify T={T} splits={splits}")


# ------------------------------------------------------------------ edge cases

def _edge_workload(ps=16, D=64, T=0, permute=True, H_q=4, H_kv=2, poison=True, lens=None):
    lens = lens or [0, 1, 15, 16, 17, 33, 100, 16 * 20 + 3]
    pol = wl.BudgetPolicy("fixed", fixed_pages=3, sink_pages=1, local_pages=1)
    return custom(lens, H_q, H_kv, D, ps, rng=np.random.default_rng(ps + D + T), T=T,
                  policy=pol, k_max=8, permute=permute, poison=poison)


@pytest.mark.parametrize("ps", [16, 32, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_edge_lengths_all_stages(ps, D):
    w = _edge_workload(ps, D, T=3)
    ref = oracle.decode_step(w, threads=4)
    g = Gpu(w)
    summ = g.summarize()
    sel, nsel, sc, _ = g.score_select(summ)
    compare_selection(w, sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy(), ref["sel"],
                      ref["nsel"], ref["scores"])
    for splits in (0, 1, 2, 5):
        o, lse, _ = g.sparse_attn(ref["sel"], ref["nsel"], num_splits=splits)
        assert_close_outputs(np_bf16(o), ref["o"], lse.cpu().numpy(), ref["lse"], what="edge sparse")
    # the empty sequence: o = 0 and lse = -inf
    assert np.all(np_bf16(o)[0] == 0) and np.all(np.isneginf(lse.cpu().numpy()[0]))
    o_ref, lse_ref = oracle.verify(w, 3)
    for splits in (0, 1, 4):
        o, lse, _ = g.verify(3, num_splits=splits)
        assert_close_outputs(np_bf16(o), o_ref, lse.cpu().numpy(), lse_ref, what="edge verify")
    assert g.sync_status() == 0


def test_nan_in_unused_cache_slots_is_ignored():
    w = _edge_workload(16, 128, T=2, lens=[17, 40, 100, 33])
    nan = np.uint16(0x7FC0)
    for b in range(w.B):
        n = int(w.seq_lens[b])
        if n % 16:
            ph = w.page_table[b, n // 16]
            w.K[ph, :, n % 16:, :] = nan
            w.V[ph, :, n % 16:, :] = nan
    ref = oracle.decode_step(w, threads=4)
    g = Gpu(w)
    summ = g.summarize()
    sel, nsel, sc, _ = g.score_select(summ)
    compare_selection(w, sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy(), ref["sel"],
                      ref["nsel"], ref["scores"])
    o, lse, _ = g.sparse_attn(ref["sel"], ref["nsel"])
    assert_close_outputs(np_bf16(o), ref["o"], lse.cpu().numpy(), ref["lse"], what="nan slots")
    o_ref, lse_ref = oracle.verify(w, 2)
    o, lse, _ = g.verify(2)
    assert_close_outputs(np_bf16(o), o_ref, lse.cpu().numpy(), lse_ref, what="nan slots verify")
    assert g.sync_status() == 0


def test_identical_pages_tie_to_lower_ids():
    n, D = 16 * 12, 64
    k = np.random.default_rng(3).standard_normal(D).astype(np.float32)
    K = [np.tile(k, (n, 2, 1))]
    pol = wl.BudgetPolicy("fixed", fixed_pages=5, sink_pages=1, local_pages=1)
    w = custom([n], 4, 2, D, 16, K=K, policy=pol, k_max=8, rng=np.random.default_rng(4))
    g = Gpu(w)
    sel, nsel, _, _ = g.score_select(g.summarize())
    assert g.sync_status() == 0
    for h in range(2):
        assert sel.cpu().numpy()[0, h, : nsel[0, h]].tolist() == [0, 1, 2, 3, 11]


def test_more_tied_pages_than_are_ranked_take_the_lowest_ids():
    """300 identical pages (more tied candidates than the selection ranks pairwise):
    the exact-key path takes the lowest page ids after the mandatory ones."""
    n, D = 16 * 300, 64
    k = np.random.default_rng(5).standard_normal(D).astype(np.float32)
    K = [np.tile(k, (n, 2, 1))]
    pol = wl.BudgetPolicy("fixed", fixed_pages=20, sink_pages=1, local_pages=2)
    w = custom([n], 4, 2, D, 16, K=K, policy=pol, k_max=24, rng=np.random.default_rng(6))
    g = Gpu(w)
    sel, nsel, _, _ = g.score_select(g.summarize())
    assert g.sync_status() == 0
    for h in range(2):
        assert sel.cpu().numpy()[0, h, : nsel[0, h]].tolist() == list(range(18)) + [298, 299]


@pytest.mark.parametrize("top_p", [None, 0.8])
def test_scores_of_both_signs_select_as_the_oracle(top_p):
    """Pages whose scores straddle zero (keys +-(1 + p/97) times one vector, so every
    candidate's score is distinct and the order-preserving keys differ in the sign
    bit): the radix select and the top-p descent agree with the oracle."""
    import dataclasses
    ps, D, P = 16, 64, 150
    rng = np.random.default_rng(8)
    base = rng.standard_normal(D).astype(np.float32)
    K = []
    for _ in range(2):
        rows = []
        for p in range(P):
            sgn = 1.0 if (p * 7) % 3 else -1.0
            rows.append(np.tile(sgn * (1.0 + p / 97.0) * base, (ps, 2, 1)))
        K.append(np.concatenate(rows).astype(np.float32))
    pol = wl.BudgetPolicy("fixed", fixed_pages=23, sink_pages=1, local_pages=3)
    if top_p is not None:
        pol = dataclasses.replace(pol, mode="top_p", top_p=top_p, score_scale=0.125)
    w = custom([P * ps, P * ps - 5], 4, 2, D, ps, K=K, policy=pol, k_max=P, rng=rng)
    ref = oracle.decode_step(w, threads=4)
    g = Gpu(w)
    sel, nsel, sc, _ = g.score_select(g.summarize())
    assert g.sync_status() == 0
    sc_g = sc.cpu().numpy()
    assert (sc_g[:, :, :P] < 0).any() and (sc_g[:, :, :P] > 0).any()
    compare_selection(w, sel.cpu().numpy(), nsel.cpu().numpy(), sc_g.astype(np.float64), ref["sel"],
                      ref["nsel"], ref["scores"])


def test_bad_page_id_sets_status_and_does_not_fault():
    w = _edge_workload(16, 64, lens=[40, 50])
    w.page_table[1, 1] = w.num_phys_pages + 5
    g = Gpu(w)
    summ = g.summarize()
    sel, nsel, _, _ = g.score_select(summ)
    g.sparse_attn(sel, nsel)
    g.verify(1, q=g.d["q"].view(w.B, 1, w.H_q, w.D))
    st = g.sync_status()
    assert st == 0x1, st
    assert g.sync_status() == 0  # cleared


@pytest.mark.parametrize("bad", ["long", "negative"])
def test_length_beyond_the_page_table_sets_status_and_empties_the_row(bad):
    """A seq_lens entry the page table cannot hold (longer than max_pages * page_size,
    or negative) sets SPD_DEV_BAD_LEN in scoring, attention and verification; that
    row gets nothing selected and o = 0 / lse = -inf, and every other row is
    bit-identical to a run without the bad entry."""
    import torch
    w = _edge_workload(16, 64, lens=[40, 50, 70, 33])
    g = Gpu(w)
    summ = g.summarize()
    assert g.sync_status() == 0
    ref_sel, ref_nsel, _, _ = g.score_select(summ)
    ref_o, ref_lse, _ = g.sparse_attn(ref_sel, ref_nsel)
    ref_ov, ref_lv, _ = g.verify(1, q=g.d["q"].view(w.B, 1, w.H_q, w.D))
    assert g.sync_status() == 0
    g.d["seq_lens"][2] = w.max_pages_per_seq * w.page_size + 9 if bad == "long" else -5
    sel, nsel, _, _ = g.score_select(summ)
    o, lse, _ = g.sparse_attn(sel, nsel)
    ov, lv, _ = g.verify(1, q=g.d["q"].view(w.B, 1, w.H_q, w.D))
    assert g.sync_status() == 0x8
    ns = nsel.cpu().numpy()
    assert not ns[2].any()
    assert not np_bf16(o)[2].any() and np.all(np.isneginf(lse.cpu().numpy()[2]))
    assert not np_bf16(ov)[2].any() and np.all(np.isneginf(lv.cpu().numpy()[2]))
    keep = [0, 1, 3]
    assert np.array_equal(ns[keep], ref_nsel.cpu().numpy()[keep])
    for b in keep:
        for h in range(w.H_kv):
            n = ns[b, h]
            assert np.array_equal(sel.cpu().numpy()[b, h, :n], ref_sel.cpu().numpy()[b, h, :n])
    for x, y in ((o, ref_o), (lse, ref_lse), (ov, ref_ov), (lv, ref_lv)):
        xb = x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32).cpu().numpy()[keep]
        yb = y.view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32).cpu().numpy()[keep]
        assert np.array_equal(xb, yb)


def test_bad_selection_entry_sets_status_and_does_not_fault():
    w = _edge_workload(16, 64, lens=[40, 50])
    g = Gpu(w)
    sel = np.zeros((w.B, w.H_kv, 4), dtype=np.int32)
    sel[:, :, 1], sel[:, :, 2], sel[:, :, 3] = 1, 2, 7       # page 7 is past both sequences
    nsel = np.full((w.B, w.H_kv), 4, dtype=np.int32)
    g.sparse_attn(sel, nsel)
    st = g.sync_status()
    assert st == 0x2, st
    nsel[0, 0] = 9                                           # more entries than k_max
    g.sparse_attn(sel, nsel)
    assert g.sync_status() & 0x2


def test_incremental_summary_matches_full():
    w = _edge_workload(16, 128, lens=[40, 100, 333])
    g = Gpu(w)
    full = summ_bits(g.summarize())
    last = [b * w.max_pages_per_seq + (int(w.seq_lens[b]) - 1) // 16 for b in range(w.B)]
    sentinel = g.torch.full((w.B, w.H_kv, w.max_pages_per_seq, 2, w.D), 3.0, dtype=g.torch.bfloat16,
                            device="cuda")
    inc = summ_bits(g.summarize(only_pages=last, summ=sentinel))
    assert g.sync_status() == 0
    s3 = wl.f32_to_bf16_bits(np.float32(3.0))
    for b in range(w.B):
        for p in range(w.max_pages_per_seq):
            if b * w.max_pages_per_seq + p in last:
                assert np.array_equal(inc[b, :, p], full[b, :, p])
            else:
                assert np.all(inc[b, :, p] == s3)


def test_workspace_reuse_gives_identical_results():
    w = small("longtail")
    ref = oracle.decode_step(w, threads=8)
    g = Gpu(w)
    ws = g.ws(g.spd.spd_sparse_decode_workspace_size(g.dims, w.k_max, 0))
    t = g.torch
    sel = t.as_tensor(ref["sel"], device="cuda")
    nsel = t.as_tensor(ref["nsel"], device="cuda")
    outs = []
    for _ in range(3):
        o = t.empty((w.B, w.H_q, w.D), dtype=t.bfloat16, device="cuda")
        g.spd.sparse_decode_attn(g.dims, g.d["q"], g.d["K"], g.d["V"], g.d["page_table"],
                                 g.d["seq_lens"], sel, nsel, w.k_max, o, ws)
        outs.append(o.view(t.int16).cpu().numpy())
    assert g.sync_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert int(ws[:256].sum()) == 0  # counters back to zero


@pytest.mark.parametrize("T,G", [(1, 8), (7, 4), (16, 4), (8, 8), (20, 2)])
def test_verify_row_tiles(T, G):
    H_kv = 2
    w = custom([T + 5, 3 * 16 + T, 200], G * H_kv, H_kv, 128, 16, T=T,
               rng=np.random.default_rng(T * 10 + G))
    o_ref, lse_ref = oracle.verify(w, T)
    g = Gpu(w)
    o, lse, _ = g.verify(T)
    assert g.sync_status() == 0
    assert_close_outputs(np_bf16(o), o_ref, lse.cpu().numpy(), lse_ref, what=f"verify T={T} G={G}")


def test_lse_merge_against_oracle():
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    rng = np.random.default_rng(5)
    for S, rows, D in ((1, 7, 64), (3, 33, 128), (40, 5, 128)):
        po = rng.standard_normal((S, rows, D)).astype(np.float32)
        pl = (rng.standard_normal((S, rows)) * 3).astype(np.float32)
        pl[rng.random((S, rows)) < 0.3] = -np.inf
        pl[:, 0] = -np.inf
        o_ref, lse_ref = oracle.merge(po.astype(np.float64), pl.astype(np.float64))
        o = torch.empty((rows, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(rows, device="cuda")
        spd.lse_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), o, lse)
        torch.cuda.synchronize()
        assert_close_outputs(np_bf16(o), o_ref, lse.cpu().numpy(), lse_ref, what=f"merge S={S}")


@pytest.mark.parametrize("key", ["tiny", "q8b"])
def test_dense_all_pages_equals_sparse_all_pages(key):
    """Budget = every page: sparse attention is dense decode attention.  Both kernels
    sum in fp32 in different orders and round o to bf16, so an element may differ by
    one bf16 rounding step of its magnitude; otherwise they agree within 1e-3, on
    average within 1e-4, and the (unrounded) lse within 1e-5."""
    w = small(key)
    g = Gpu(w)
    P = w.max_pages_per_seq
    sel = np.tile(np.arange(P, dtype=np.int32), (w.B, w.H_kv, 1))
    nsel = np.array([[w.pages(b)] * w.H_kv for b in range(w.B)], dtype=np.int32)
    o_s, lse_s, _ = g.sparse_attn(sel, nsel)
    o_d, lse_d, _ = g.verify(1, q=g.d["q"].view(w.B, 1, w.H_q, w.D))
    assert g.sync_status() == 0
    a, b = np_bf16(o_s), np_bf16(o_d)[:, 0]
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(a), np.abs(b)) + 1e-30)) - 7)  # one bf16 ulp
    diff = np.abs(a - b)
    assert np.all(diff <= np.maximum(1e-3, step)), diff.max()
    assert diff.mean() <= 1e-4
    assert np.abs(lse_s.cpu().numpy() - lse_d.cpu().numpy()[:, 0]).max() <= 1e-5


@pytest.mark.parametrize("key", ["q8b", "tiny"])
def test_one_workspace_serves_the_calls_in_turn(key):
    """One zeroed buffer of the largest workspace size serves scoring + selection,
    sparse attention and verification one after the other, twice (each call leaves
    the counters the others need at zero): results bit-identical to separate
    workspaces."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = small(key)
    g = Gpu(w)
    summ = g.summarize()
    sel0, nsel0, _, _ = g.score_select(summ)
    o0, lse0, _ = g.sparse_attn(sel0, nsel0)
    qv = g.d["q"].view(w.B, 1, w.H_q, w.D)
    ov0, lv0, _ = g.verify(1, q=qv)
    ws = g.ws(max(spd.spd_score_select_workspace_size(g.dims),
                  spd.spd_sparse_decode_workspace_size(g.dims, w.k_max, 0),
                  spd.spd_dense_verify_workspace_size(g.dims, 1, 0)))
    d = g.d
    for _ in range(2):
        sel = torch.full_like(sel0, -1)
        nsel = torch.full_like(nsel0, -7)
        o = torch.full_like(o0, float("nan"))
        lse = torch.full_like(lse0, float("nan"))
        ov = torch.full_like(ov0, float("nan"))
        lv = torch.full_like(lv0, float("nan"))
        spd.pages_score_select(g.dims, d["q"], summ, d["seq_lens"], w.policy, sel, nsel, w.k_max, ws)
        spd.sparse_decode_attn(g.dims, d["q"], d["K"], d["V"], d["page_table"], d["seq_lens"], sel, nsel,
                               w.k_max, o, ws, lse=lse)
        spd.dense_verify_attn(g.dims, 1, qv, d["K"], d["V"], d["page_table"], d["seq_lens"], ov, ws, lse=lv)
        assert g.sync_status() == 0
        assert torch.equal(nsel, nsel0)
        for b in range(w.B):
            for h in range(w.H_kv):
                n = int(nsel0[b, h])
                assert torch.equal(sel[b, h, :n], sel0[b, h, :n])
        for x, y in ((o, o0), (lse, lse0), (ov, ov0), (lv, lv0)):
            assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                               y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))


def test_workspace_sizes_do_not_change_after_first_launch():
    """Auto split counts (and so workspace sizes) are the same before and after launches."""
    w = small("q8b")
    g = Gpu(w)
    before = (g.spd.spd_sparse_decode_workspace_size(g.dims, w.k_max, 0),
              g.spd.spd_dense_verify_workspace_size(g.dims, 7, 0))
    summ = g.summarize()
    sel, nsel, _, _ = g.score_select(summ)
    g.sparse_attn(sel, nsel)
    g.verify(7)
    after = (g.spd.spd_sparse_decode_workspace_size(g.dims, w.k_max, 0),
             g.spd.spd_dense_verify_workspace_size(g.dims, 7, 0))
    assert before == after
    assert g.sync_status() == 0
