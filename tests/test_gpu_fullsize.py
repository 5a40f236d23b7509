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
