"""GPU parity of the rows that follow the core path, through the C ABI against the
fp64 oracle: the fused cache append + summary refresh (bit-exact)."""
import numpy as np
import pytest

import oracle
from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.gpu_helpers import Gpu, summ_bits
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
