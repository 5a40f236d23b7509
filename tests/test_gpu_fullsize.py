"""GPU parity at the full workload sizes, in the launch configuration the benchmark
uses (automatic split counts), checked against the fp64 oracle on sampled
sequences (the oracle computes those sequences one by one)."""
import numpy as np
import pytest

import oracle
from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.gpu_helpers import Gpu, assert_close_outputs, compare_selection, np_bf16, summ_bits

pytestmark = pytest.mark.gpu

FULL = [("q17b", None), ("q8b", None), ("sweep", 16), ("sweep", 32), ("sweep", 64), ("longtail", None)]


@pytest.mark.parametrize("name,ps", FULL, ids=[f"{n}{p or ''}" for n, p in FULL])
def test_full_size_sampled(name, ps):
    w = wl.named(name, ps)
    rng = np.random.default_rng(7)
    sample = sorted(set([0, w.B - 1] + rng.choice(w.B, size=min(3, w.B), replace=False).tolist()))
    g = Gpu(w)
    summ = g.summarize()
    sel, nsel, sc, _ = g.score_select(summ)
    o, lse, _ = g.sparse_attn(sel, nsel)
    assert g.sync_status() == 0
    sel_g, nsel_g, sc_g = sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy()

    s_ref = oracle.summarize(w, seqs=sample, threads=16)
    got = summ_bits(summ)
    for b in sample:
        for p in range(w.pages(b)):
            ph = w.page_table[b, p]
            assert np.array_equal(got[b, :, p], wl.f32_to_bf16_bits(s_ref[ph].astype(np.float32))), (b, p)
    sc_ref = oracle.scores(w, s_ref, seqs=sample, threads=16)
    sel_ref, nsel_ref = oracle.select(w, sc_ref, seqs=sample, threads=16)
    for b in sample:
        P = w.pages(b)
        d = np.abs(sc_g[b, :, :P] - sc_ref[b, :, :P])
        assert np.all(d <= 2e-5 * (1 + np.abs(sc_ref[b, :, :P]))), (b, d.max())
    same = compare_selection(w, sel_g, nsel_g, sc_g, sel_ref, nsel_ref, sc_ref, seqs=sample)

    # attention on the oracle's selection for the sampled sequences
    mix_sel, mix_n = sel_g.copy(), nsel_g.copy()
    for b in sample:
        mix_sel[b], mix_n[b] = sel_ref[b], nsel_ref[b]
    o_m, lse_m, _ = g.sparse_attn(mix_sel, mix_n)
    o_ref, lse_ref = oracle.sparse_attn(w, sel_ref, nsel_ref, seqs=sample, threads=16)
    assert_close_outputs(np_bf16(o_m)[sample], o_ref[sample], lse_m.cpu().numpy()[sample],
                         lse_ref[sample], what=f"{name} sparse")
    # the GPU pipeline itself, on sampled sequences whose selections match exactly
    rows = [b for b in sample if all((b, h) in same for h in range(w.H_kv))]
    if rows:
        assert_close_outputs(np_bf16(o)[rows], o_ref[rows], lse.cpu().numpy()[rows], lse_ref[rows],
                             what=f"{name} pipeline")

    # dense verification (the q8b workload's T = 7) or dense decode (T = 1)
    if w.T or name == "longtail":
        T = w.T or 1
        q = w.q_verify if w.T else np.ascontiguousarray(w.q.reshape(w.B, 1, w.H_q, w.D))
        qd = g.torch.from_numpy(q).view(g.torch.bfloat16).cuda()
        ov, lv, _ = g.verify(T, q=qd)
        assert g.sync_status() == 0
        ov_ref, lv_ref = oracle.verify(w, T, q=q, seqs=sample, threads=16)
        assert_close_outputs(np_bf16(ov)[sample], ov_ref[sample], lv.cpu().numpy()[sample],
                             lv_ref[sample], what=f"{name} verify T={T}")


def _sample(w, seed=11):
    rng = np.random.default_rng(seed)
    return sorted(set([0, w.B - 1] + rng.choice(w.B, size=min(3, w.B), replace=False).tolist()))


def _new_token(w, seed):
    rng = np.random.default_rng(seed)
    shape = (w.B, 1, w.H_kv, w.D)
    return (wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32)),
            wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32)))


def _check_append_and_selection(w, g, k_new, v_new, summ, sel_g, nsel_g, sc_g, sample):
    """The cache and summaries after the step's append against the oracle's append
    (K / V bits of every sequence, summaries of the sampled ones), the GPU's scores
    and selection against the oracle's on the sampled sequences.  Returns the oracle's
    appended workload, its selection and the (b, h) rows selected alike."""
    import dataclasses
    import torch
    K2, V2 = oracle.append(w, 1, k_new, v_new, threads=16)
    w2 = dataclasses.replace(w, K=K2, V=V2)
    Kg = g.d["K"].view(torch.int16).cpu().numpy().view(np.uint16)
    Vg = g.d["V"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(Kg, K2) and np.array_equal(Vg, V2)  # the whole cache, every sequence
    for b in range(w.B):
        L = int(w.seq_lens[b])
        ph, slot = w.page_table[b, (L - 1) // w.page_size], (L - 1) % w.page_size
        assert np.array_equal(K2[ph, :, slot], k_new[b, 0]) and not np.array_equal(w.K[ph, :, slot], k_new[b, 0])
    s_ref = oracle.summarize(w2, seqs=sample, threads=16)
    got = summ_bits(summ)
    for b in sample:
        for p in range(w.pages(b)):
            ph = w.page_table[b, p]
            assert np.array_equal(got[b, :, p], wl.f32_to_bf16_bits(s_ref[ph].astype(np.float32))), (b, p)
    sc_ref = oracle.scores(w2, s_ref, seqs=sample, threads=16)
    sel_ref, nsel_ref = oracle.select(w2, sc_ref, seqs=sample, threads=16)
    for b in sample:
        P = w.pages(b)
        d = np.abs(sc_g[b, :, :P] - sc_ref[b, :, :P])
        assert np.all(d <= 2e-5 * (1 + np.abs(sc_ref[b, :, :P]))), (b, d.max())
    same = compare_selection(w2, sel_g, nsel_g, sc_g, sel_ref, nsel_ref, sc_ref, seqs=sample)
    return w2, sel_ref, nsel_ref, same


def test_decode_step_full_size_with_append_against_oracle():
    """The benchmark's exact call -- sparse_decode_step with the step's token appended,
    at the full Qwen3-8B shape (B = 64, 512 rows of 512..1022 pages), twice through one
    workspace -- against the fp64 oracle on sampled sequences: the appended cache and
    summaries bit-exact, the selection equal outside the tie band, o and lse within
    tolerance."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = wl.named("q8b")
    sample = _sample(w)
    k_new, v_new = _new_token(w, 5)
    g = Gpu(w)
    summ = g.summarize()
    d = g.d
    kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda()
    vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda()
    sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
    nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
    o = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H_q), float("nan"), device="cuda")
    ws = g.ws(spd.spd_sparse_decode_step_workspace_size(g.dims, w.k_max))
    outs = []
    for _ in range(2):  # the second call rewrites the same token: the same bits, counters reset by the first
        spd.sparse_decode_step(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, d["q"], summ,
                               w.policy, sel, nsel, w.k_max, o, ws, lse=lse)
        assert g.sync_status() == 0
        outs.append([sel.cpu().numpy(), nsel.cpu().numpy(), o.view(torch.int16).cpu().numpy(),
                     lse.view(torch.int32).cpu().numpy(), summ_bits(summ)])
    for x, y in zip(*outs):
        assert np.array_equal(x, y)
    _, _, sc, _ = g.score_select(summ)   # the GPU's own scores of the updated summaries
    sel_g, nsel_g, sc_g = sel.cpu().numpy(), nsel.cpu().numpy(), sc.cpu().numpy()
    w2, sel_ref, nsel_ref, same = _check_append_and_selection(w, g, k_new, v_new, summ, sel_g, nsel_g, sc_g,
                                                              sample)
    o_ref, lse_ref = oracle.sparse_attn(w2, sel_ref, nsel_ref, seqs=sample, threads=16)
    rows = [b for b in sample if all((b, h) in same for h in range(w.H_kv))]
    assert rows, "no sampled sequence selected alike"
    assert_close_outputs(np_bf16(o)[rows], o_ref[rows], lse.cpu().numpy()[rows], lse_ref[rows],
                         what="q8b decode step with append")


def test_append_score_select_full_size_against_oracle():
    """pages_append_score_select (the step's first pass, with its scores written out)
    at the full Qwen3-8B shape against the fp64 oracle on sampled sequences."""
    import torch
    import sparse_attention_decode_pages_gb300 as spd
    w = wl.named("q8b")
    sample = _sample(w, seed=12)
    k_new, v_new = _new_token(w, 6)
    g = Gpu(w)
    summ = g.summarize()
    d = g.d
    kn = torch.from_numpy(k_new).view(torch.bfloat16).cuda()
    vn = torch.from_numpy(v_new).view(torch.bfloat16).cuda()
    sel = torch.full((w.B, w.H_kv, w.k_max), -1, dtype=torch.int32, device="cuda")
    nsel = torch.full((w.B, w.H_kv), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((w.B, w.H_kv, w.max_pages_per_seq), float("nan"), device="cuda")
    ws = g.ws(spd.spd_score_select_workspace_size(g.dims))
    spd.pages_append_score_select(g.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], kn, vn, d["q"], summ,
                                  w.policy, sel, nsel, w.k_max, ws, scores=sc)
    assert g.sync_status() == 0
    _check_append_and_selection(w, g, k_new, v_new, summ, sel.cpu().numpy(), nsel.cpu().numpy(),
                                sc.cpu().numpy(), sample)
