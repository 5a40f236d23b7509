"""Runs the CUDA path on a workload through the Python binding and returns numpy results."""
from __future__ import annotations

import numpy as np

from sparse_attention_decode_pages_gb300 import workloads as wl

# Tolerances: selected sets bit-exact outside the band of pages whose score is
# within TIE_BAND (relative) of the k-th score; outputs vs the fp64 oracle.
TIE_BAND = 1e-3
O_MAX_ABS, O_MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


class Gpu:
    """Device copies of a workload plus the library calls on them."""

    def __init__(self, w: wl.Workload):
        import torch
        import sparse_attention_decode_pages_gb300 as spd
        self.torch, self.spd, self.w = torch, spd, w
        self.d = wl.to_device(w)
        self.dims = spd.dims_of(w.B, w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq,
                                w.num_phys_pages)

    def ws(self, nbytes):
        return self.spd.workspace(nbytes)

    def summarize(self, only_pages=None, summ=None):
        t, w = self.torch, self.w
        if summ is None:
            summ = t.zeros((w.B, w.H_kv, w.max_pages_per_seq, 2, w.D), dtype=t.bfloat16, device="cuda")
        op = None if only_pages is None else t.as_tensor(np.asarray(only_pages, np.int32), device="cuda")
        self.spd.pages_summarize(self.dims, self.d["K"], self.d["page_table"], self.d["seq_lens"],
                                 summ, only_pages=op)
        return summ

    def score_select(self, summ, policy=None, k_max=None, q=None):
        t, w = self.torch, self.w
        k_max = w.k_max if k_max is None else k_max
        sel = t.full((w.B, w.H_kv, k_max), -1, dtype=t.int32, device="cuda")
        nsel = t.full((w.B, w.H_kv), -7, dtype=t.int32, device="cuda")
        scores = t.full((w.B, w.H_kv, w.max_pages_per_seq), float("nan"), device="cuda")
        ws = self.ws(self.spd.spd_score_select_workspace_size(self.dims))
        self.spd.pages_score_select(self.dims, self.d["q"] if q is None else q, summ,
                                    self.d["seq_lens"],
                                    policy or w.policy, sel, nsel, k_max, ws, scores=scores)
        return sel, nsel, scores, ws

    def sparse_attn(self, sel, nsel, num_splits=0, k_max=None):
        t, w = self.torch, self.w
        if isinstance(sel, np.ndarray):
            sel = t.as_tensor(np.ascontiguousarray(sel, np.int32), device="cuda")
            nsel = t.as_tensor(np.ascontiguousarray(nsel, np.int32), device="cuda")
        k_max = sel.shape[-1] if k_max is None else k_max
        o = t.full((w.B, w.H_q, w.D), float("nan"), dtype=t.bfloat16, device="cuda")
        lse = t.full((w.B, w.H_q), float("nan"), device="cuda")
        ws = self.ws(self.spd.spd_sparse_decode_workspace_size(self.dims, k_max, num_splits))
        self.spd.sparse_decode_attn(self.dims, self.d["q"], self.d["K"], self.d["V"],
                                    self.d["page_table"], self.d["seq_lens"], sel, nsel, k_max, o,
                                    ws, lse=lse, num_splits=num_splits)
        return o, lse, ws

    def verify(self, T, q=None, num_splits=0):
        t, w = self.torch, self.w
        q = self.d["q_verify"] if q is None else q
        o = t.full((w.B, T, w.H_q, w.D), float("nan"), dtype=t.bfloat16, device="cuda")
        lse = t.full((w.B, T, w.H_q), float("nan"), device="cuda")
        ws = self.ws(self.spd.spd_dense_verify_workspace_size(self.dims, T, num_splits))
        self.spd.dense_verify_attn(self.dims, T, q, self.d["K"], self.d["V"], self.d["page_table"],
                                   self.d["seq_lens"], o, ws, lse=lse, num_splits=num_splits)
        return o, lse, ws

    def append(self, T, k_new, v_new, summ):
        """kv_append_refresh on the device copies of K / V (k_new, v_new: numpy bf16 bits)."""
        t = self.torch
        kn = t.from_numpy(np.ascontiguousarray(k_new)).view(t.bfloat16).cuda()
        vn = t.from_numpy(np.ascontiguousarray(v_new)).view(t.bfloat16).cuda()
        self.spd.kv_append_refresh(self.dims, T, self.d["K"], self.d["V"], self.d["page_table"],
                                   self.d["seq_lens"], kn, vn, summ)
        return summ

    def sync_status(self):
        self.torch.cuda.synchronize()
        return self.spd.spd_device_status(clear=True)


def np_bf16(t):
    """A device bf16 tensor -> float64 numpy."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def summ_bits(t):
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close_outputs(o_gpu, o_ref, lse_gpu=None, lse_ref=None, rows=None, what=""):
    """Max-abs / mean-abs on o and abs on lse against the fp64 oracle (over the given rows)."""
    og, orf = np.asarray(o_gpu, np.float64), np.asarray(o_ref, np.float64)
    if rows is not None:
        og, orf = og[rows], orf[rows]
    assert np.all(np.isfinite(og)), f"{what}: non-finite outputs"
    err = np.abs(og - orf)
    assert err.max() <= O_MAX_ABS, f"{what}: max abs error {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean abs error {err.mean():.3e}"
    if lse_gpu is not None:
        lg, lr = np.asarray(lse_gpu, np.float64), np.asarray(lse_ref, np.float64)
        if rows is not None:
            lg, lr = lg[rows], lr[rows]
        both_inf = np.isneginf(lg) & np.isneginf(lr)
        d = np.where(both_inf, 0.0, np.abs(lg - lr))
        assert np.nanmax(d) <= LSE_ABS and not np.any(np.isnan(d)), f"{what}: lse error {np.nanmax(d):.3e}"
    return err.max(), err.mean()


def compare_selection(w, sel_g, nsel_g, sc_g, sel_o, nsel_o, sc_o, seqs=None):
    """Selected sets equal outside the tie band; GPU's choice valid under its own scores.

    Returns the list of (b, h) rows whose sets are identical."""
    same_rows = []
    seqs = range(w.B) if seqs is None else seqs
    for b in seqs:
        P = w.pages(b)
        sink, local = min(w.policy.sink_pages, P), min(w.policy.local_pages, P)
        mand = {p for p in range(P) if p < sink or p >= P - local}
        for h in range(w.H_kv):
            assert nsel_g[b, h] == nsel_o[b, h], (b, h, nsel_g[b, h], nsel_o[b, h])
            g = sel_g[b, h, : nsel_g[b, h]].tolist()
            o = sel_o[b, h, : nsel_o[b, h]].tolist()
            assert g == sorted(set(g)), (b, h, "not ascending/unique")
            assert mand <= set(g), (b, h, "mandatory page missing")
            if g == o:
                same_rows.append((b, h))
                continue
            picked = [p for p in o if p not in mand]
            if not picked:
                raise AssertionError((b, h, "sets differ with nothing to pick"))
            kth = min(sc_o[b, h, p] for p in picked)
            band = {p for p in range(P)
                    if p not in mand and abs(sc_o[b, h, p] - kth) <= TIE_BAND * abs(kth)}
            assert set(g) - band == set(o) - band, (b, h, sorted(set(g) ^ set(o)), sorted(band))
            # validity under the GPU's own scores: no unselected page beats a selected one
            sg = sc_g[b, h]
            chosen = [p for p in g if p not in mand]
            rest = [p for p in range(P) if p not in mand and p not in g]
            if chosen and rest:
                lo = min(chosen, key=lambda p: (sg[p], -p))
                hi = max(rest, key=lambda p: (sg[p], -p))
                assert (sg[lo], -lo) > (sg[hi], -hi), (b, h, "GPU selection not a top-k of its scores")
    return same_rows
