"""sparse_decode_attn_noalloc: the variant for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: an engine that owns all GPU
memory through a fixed arena, or a decode loop that must not call cudaMalloc
(it can synchronise the device).  For them the library keeps the scratch of the
sparse attention (unit queue, split tickets, split partials) in a fixed array of
its own.  This test calls that entry point through the C ABI twice in a row and
checks it against the workspace entry point, within the tolerances the other
parity tests use.  It lives in a file of its own, collected last.
"""
import numpy as np
import pytest

from sparse_attention_decode_pages_gb300 import workloads as wl
from tests.gpu_helpers import O_MAX_ABS, O_MEAN_ABS, LSE_ABS

pytestmark = pytest.mark.gpu


def _compare(o_a, lse_a, o_b, lse_b):
    """Within the tolerances the other parity tests use, and -- the same kernel with
    the same split count -- bit for bit."""
    d = np.abs(o_a - o_b)
    assert np.all(np.isfinite(o_a)) and d.max() <= O_MAX_ABS and d.mean() <= O_MEAN_ABS
    both = np.isneginf(lse_a) & np.isneginf(lse_b)
    assert np.all(np.where(both, 0.0, np.abs(lse_a - lse_b)) <= LSE_ABS)
    assert np.array_equal(o_a, o_b) and np.array_equal(lse_a.view(np.int32), lse_b.view(np.int32))


@pytest.mark.parametrize("splits", [0, 3])
def test_noalloc_matches_workspace_entry_point_twice(splits):
    import torch
    import sparse_attention_decode_pages_gb300 as spd

    w = wl.named("q8b", B=6, len_lo=600, len_hi=2500, threads=4)
    d = wl.to_device(w)
    dims = spd.dims_of(w.B, w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, w.num_phys_pages)
    summ = torch.empty((w.B, w.H_kv, w.max_pages_per_seq, 2, w.D), dtype=torch.bfloat16, device="cuda")
    spd.pages_summarize(dims, d["K"], d["page_table"], d["seq_lens"], summ)
    sel = torch.empty((w.B, w.H_kv, w.k_max), dtype=torch.int32, device="cuda")
    nsel = torch.empty((w.B, w.H_kv), dtype=torch.int32, device="cuda")
    spd.pages_score_select(dims, d["q"], summ, d["seq_lens"], w.policy, sel, nsel,
                           w.k_max, spd.workspace(spd.spd_score_select_workspace_size(dims)))

    def run(fn, **kw):
        o = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.B, w.H_q), float("nan"), device="cuda")
        fn(dims, d["q"], d["K"], d["V"], d["page_table"], d["seq_lens"], sel, nsel, w.k_max, o,
           lse=lse, num_splits=splits, **kw)
        torch.cuda.synchronize()
        return o.float().cpu().numpy(), lse.cpu().numpy()

    ws = spd.workspace(spd.spd_sparse_decode_workspace_size(dims, w.k_max, splits))
    ref_o, ref_lse = run(lambda *a, **k: spd.sparse_decode_attn(*a[:10], ws, **k))
    for _ in range(2):  # the fixed array keeps the last call's contents
        o, lse = run(spd.sparse_decode_attn_noalloc)
        _compare(o, lse, ref_o, ref_lse)
    assert spd.spd_device_status(clear=True) == 0


def test_noalloc_one_unit_per_row_needs_no_partials():
    """With one attention unit per row (B = 512 at the Qwen3-8B heads: 4,096 rows) a
    call writes no split partials, so it needs only the unit queue and the split
    tickets of the fixed array -- although one split's partials alone (4,096 rows x
    4 heads x 128 channels x 4 bytes = 8 MiB) would fill it.  Bit-identical to the
    workspace entry point, twice in a row.  (The automatic split count gives every
    row at least one unit per attention worker only when rows are few, so its
    partials stay near 4 MB on this GPU and never need lowering to fit.)"""
    import torch
    import sparse_attention_decode_pages_gb300 as spd

    w = wl.named("q8b", B=512, len_lo=100, len_hi=400, threads=8)
    d = wl.to_device(w)
    dims = spd.dims_of(w.B, w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, w.num_phys_pages)
    summ = torch.empty((w.B, w.H_kv, w.max_pages_per_seq, 2, w.D), dtype=torch.bfloat16, device="cuda")
    spd.pages_summarize(dims, d["K"], d["page_table"], d["seq_lens"], summ)
    k_max = 16
    sel = torch.empty((w.B, w.H_kv, k_max), dtype=torch.int32, device="cuda")
    nsel = torch.empty((w.B, w.H_kv), dtype=torch.int32, device="cuda")
    pol = wl.BudgetPolicy("fixed", fixed_pages=k_max, sink_pages=1, local_pages=4)
    spd.pages_score_select(dims, d["q"], summ, d["seq_lens"], pol, sel, nsel, k_max,
                           spd.workspace(spd.spd_score_select_workspace_size(dims)))

    def run(fn, **kw):
        o = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.B, w.H_q), float("nan"), device="cuda")
        fn(dims, d["q"], d["K"], d["V"], d["page_table"], d["seq_lens"], sel, nsel, k_max, o, lse=lse, **kw)
        torch.cuda.synchronize()
        return o.float().cpu().numpy(), lse.cpu().numpy()

    ws = spd.workspace(spd.spd_sparse_decode_workspace_size(dims, k_max, 0))
    ref_o, ref_lse = run(lambda *a, **k: spd.sparse_decode_attn(*a[:10], ws, **k))
    for _ in range(2):
        o, lse = run(spd.sparse_decode_attn_noalloc)
        _compare(o, lse, ref_o, ref_lse)
    assert spd.spd_device_status(clear=True) == 0


def test_noalloc_rejects_scratch_beyond_its_fixed_size():
    import torch
    import sparse_attention_decode_pages_gb300 as spd

    # 512 (sequence, KV head) rows x 4 heads x 128 channels: 1 MiB of partials per split
    w = wl.named("q8b", len_lo=100, len_hi=300, threads=4)
    d = wl.to_device(w)
    dims = spd.dims_of(w.B, w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, w.num_phys_pages)
    sel = torch.zeros((w.B, w.H_kv, 16), dtype=torch.int32, device="cuda")
    nsel = torch.ones((w.B, w.H_kv), dtype=torch.int32, device="cuda")
    o = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(spd.SpdError) as e:
        spd.sparse_decode_attn_noalloc(dims, d["q"], d["K"], d["V"], d["page_table"], d["seq_lens"],
                                       sel, nsel, 16, o, num_splits=16)
    assert e.value.status == 2 and "fixed array" in str(e.value)
