"""fp64 CPU oracle for sparse paged decode attention (ctypes over ``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg, never by the library.  It shares no
code with the CUDA path; both read the same seeded inputs from
``sparse_attention_decode_pages_gb300.workloads``.

Each wrapper runs the C oracle one sequence at a time; sequences are spread
over a thread pool (ctypes releases the GIL during the foreign call), so the
number of threads used is what ``threads`` says.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

MODES = {"fixed": 0, "linear": 1, "fraction": 2}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (plain gcc, IEEE double)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
        L.oracle_summarize_seq.argtypes = [i, i, i, i, P, P, P, i, P]
        L.oracle_score_seq.argtypes = [i, i, i, i, i, P, P, P, P, i, P]
        L.oracle_budget_pages.argtypes = [i, l, l, l, l, i, i]
        L.oracle_budget_pages.restype = l
        L.oracle_k_eff.argtypes = [i, l, i, i, i]
        L.oracle_k_eff.restype = i
        L.oracle_select_seq.argtypes = [i, i, i, P, i, i, l, l, l, l, i, i, i, P, P]
        L.oracle_sparse_attn_seq.argtypes = [i, i, i, i, i, P, P, P, P, P, i, P, P, i, d, P, P]
        L.oracle_merge_row.argtypes = [i, i, P, P, P, P]
        L.oracle_verify_seq.argtypes = [i, i, i, i, i, i, P, P, P, P, P, i, d, P, P]
        L.oracle_append_seq.argtypes = [i, i, i, i, i, P, P, P, P, i, P, P]
        L.oracle_spec_accept_seq.argtypes = [i, i, P, P, P, P, ctypes.c_float, P]
        L.oracle_spec_accept_seq.restype = i
        L.oracle_select_top_p_seq.argtypes = [i, i, i, P, i, d, d, i, i, i, P, P]
        for f in ("oracle_summarize_seq", "oracle_score_seq", "oracle_select_seq",
                  "oracle_sparse_attn_seq", "oracle_merge_row", "oracle_verify_seq",
                  "oracle_append_seq", "oracle_select_top_p_seq"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _run(fn, items, threads):
    threads = threads or min(16, os.cpu_count() or 1)
    if threads <= 1:
        for x in items:
            fn(x)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fn, items))


def _policy_args(pol):
    m = MODES[pol.mode]
    if m == 0:
        return m, pol.fixed_pages, 0, 1, 0
    if m == 1:
        return m, pol.min_tokens, pol.slope_num, pol.slope_den, pol.intercept
    return m, pol.frac_num, pol.frac_den, 0, 0


def _seqs(w, seqs):
    return range(w.B) if seqs is None else list(seqs)


def summarize(w, seqs=None, threads=None) -> np.ndarray:
    """Step a1: float64 [num_phys_pages][H_kv][2][D]; pages not used by ``seqs`` stay NaN."""
    L = lib()
    out = np.full((w.num_phys_pages, w.H_kv, 2, w.D), np.nan)
    _run(lambda b: L.oracle_summarize_seq(w.H_kv, w.D, w.page_size, w.max_pages_per_seq,
                                          _p(w.K), _p(w.page_table), _p(w.seq_lens), b, _p(out)),
         _seqs(w, seqs), threads)
    return out


def scores(w, summ, q=None, seqs=None, threads=None) -> np.ndarray:
    """Step a2: float64 [B][H_kv][max_pages]; slots past a sequence's last page are -inf."""
    L = lib()
    q = w.q if q is None else q
    out = np.full((w.B, w.H_kv, w.max_pages_per_seq), -np.inf)

    def one(b):
        L.oracle_score_seq(w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, _p(q), _p(summ),
                           _p(w.page_table), _p(w.seq_lens), b, out[b].ctypes.data)
    _run(one, _seqs(w, seqs), threads)
    return out


def budget_pages(pol, length: int, page_size: int) -> int:
    m, a, b, c, d = _policy_args(pol)
    return lib().oracle_budget_pages(m, a, b, c, d, length, page_size)


def k_eff(pol, length: int, page_size: int, k_max: int) -> int:
    P = -(-length // page_size)
    return lib().oracle_k_eff(P, budget_pages(pol, length, page_size), k_max, pol.sink_pages,
                              pol.local_pages)


def select(w, sc, policy=None, k_max=None, seqs=None, threads=None):
    """Step a4: (sel int32 [B][H_kv][k_max], nsel int32 [B][H_kv]); unused slots are -1."""
    pol = w.policy if policy is None else policy
    if pol.mode == "top_p":
        return select_top_p(w, sc, pol.top_p, pol.score_scale, k_max=k_max, policy=pol, seqs=seqs,
                            threads=threads)
    L = lib()
    k_max = w.k_max if k_max is None else k_max
    m, a, b_, c, d = _policy_args(pol)
    sel = np.full((w.B, w.H_kv, k_max), -1, dtype=np.int32)
    nsel = np.zeros((w.B, w.H_kv), dtype=np.int32)
    sc = np.ascontiguousarray(sc, dtype=np.float64)

    def one(b):
        L.oracle_select_seq(w.H_kv, w.page_size, w.max_pages_per_seq, sc[b].ctypes.data,
                            int(w.seq_lens[b]), m, a, b_, c, d, pol.sink_pages, pol.local_pages,
                            k_max, sel[b].ctypes.data, nsel[b].ctypes.data)
    _run(one, _seqs(w, seqs), threads)
    return sel, nsel


def sparse_attn(w, sel, nsel, q=None, seqs=None, threads=None, scale=None):
    """Step a5: (o float64 [B][H_q][D], lse float64 [B][H_q]) over the given selection."""
    L = lib()
    q = w.q if q is None else q
    k_max = sel.shape[-1]
    scale = w.scale if scale is None else scale
    o = np.full((w.B, w.H_q, w.D), np.nan)
    lse = np.full((w.B, w.H_q), np.nan)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    nsel = np.ascontiguousarray(nsel, dtype=np.int32)

    def one(b):
        L.oracle_sparse_attn_seq(w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, _p(q),
                                 _p(w.K), _p(w.V), _p(w.page_table), _p(w.seq_lens), b,
                                 sel[b].ctypes.data, nsel[b].ctypes.data, k_max, scale,
                                 o[b].ctypes.data, lse[b].ctypes.data)
    _run(one, _seqs(w, seqs), threads)
    return o, lse


def verify(w, T, q=None, seqs=None, threads=None, scale=None):
    """Step a7: (o float64 [B][T][H_q][D], lse float64 [B][T][H_q]); q is [B][T][H_q][D]."""
    L = lib()
    q = w.q_verify if q is None else q
    scale = w.scale if scale is None else scale
    o = np.full((w.B, T, w.H_q, w.D), np.nan)
    lse = np.full((w.B, T, w.H_q), np.nan)

    def one(b):
        L.oracle_verify_seq(T, w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, _p(q),
                            _p(w.K), _p(w.V), _p(w.page_table), _p(w.seq_lens), b, scale,
                            o[b].ctypes.data, lse[b].ctypes.data)
    _run(one, _seqs(w, seqs), threads)
    return o, lse


def merge(part_o: np.ndarray, part_lse: np.ndarray):
    """Step a6: part_o [S][rows][D], part_lse [S][rows] -> (o [rows][D], lse [rows])."""
    L = lib()
    S, rows, D = part_o.shape
    po = np.ascontiguousarray(np.transpose(part_o, (1, 0, 2)), dtype=np.float64)
    pl = np.ascontiguousarray(np.transpose(part_lse, (1, 0)), dtype=np.float64)
    o = np.empty((rows, D))
    lse = np.empty(rows)
    for r in range(rows):
        L.oracle_merge_row(S, D, po[r].ctypes.data, pl[r].ctypes.data, o[r].ctypes.data,
                           lse[r:r + 1].ctypes.data)
    return o, lse


def decode_step(w, threads=None):
    """Steps a1-a5 for the decode query: summaries, scores, selection, sparse attention."""
    summ = summarize(w, threads=threads)
    sc = scores(w, summ, threads=threads)
    sel, nsel = select(w, sc, threads=threads)
    o, lse = sparse_attn(w, sel, nsel, threads=threads)
    return dict(summ=summ, scores=sc, sel=sel, nsel=nsel, o=o, lse=lse)


def append(w, T, k_new, v_new, seqs=None, threads=None):
    """Row f1: (K, V) copies of the cache with the T newest tokens of each sequence
    written from k_new / v_new (bf16 bits [B][T][H_kv][D]); the inputs are untouched."""
    L = lib()
    K, V = w.K.copy(), w.V.copy()
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    assert k_new.shape == (w.B, T, w.H_kv, w.D) and v_new.shape == k_new.shape
    _run(lambda b: L.oracle_append_seq(T, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, _p(K),
                                       _p(V), _p(w.page_table), _p(w.seq_lens), b, _p(k_new),
                                       _p(v_new)),
         _seqs(w, seqs), threads)
    return K, V


def spec_accept(p, q, draft, u_acc, u_res):
    """Row f2: exact speculative sampling per sequence.

    p float32 [B][k][n], q float32 [B][k+1][n], draft int32 [B][k], u_acc float32
    [B][k], u_res float32 [B] -> (n_accepted int32 [B], tokens int32 [B][k+1])."""
    L = lib()
    p = np.ascontiguousarray(p, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    u_acc = np.ascontiguousarray(u_acc, dtype=np.float32)
    u_res = np.ascontiguousarray(u_res, dtype=np.float32)
    B, k, n = p.shape
    assert q.shape == (B, k + 1, n) and draft.shape == (B, k) and u_acc.shape == (B, k)
    tokens = np.full((B, k + 1), -1, dtype=np.int32)
    nacc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        nacc[b] = L.oracle_spec_accept_seq(k, n, p[b].ctypes.data, q[b].ctypes.data,
                                           draft[b].ctypes.data, u_acc[b].ctypes.data,
                                           float(u_res[b]), tokens[b].ctypes.data)
    return nacc, tokens


def select_top_p(w, sc, top_p, score_scale=None, k_max=None, policy=None, seqs=None, threads=None):
    """Row f3: top-p page selection -> (sel int32 [B][H_kv][k_max], nsel int32 [B][H_kv])."""
    L = lib()
    pol = w.policy if policy is None else policy
    k_max = w.k_max if k_max is None else k_max
    score_scale = w.scale if score_scale is None else score_scale
    sel = np.full((w.B, w.H_kv, k_max), -1, dtype=np.int32)
    nsel = np.zeros((w.B, w.H_kv), dtype=np.int32)
    sc = np.ascontiguousarray(sc, dtype=np.float64)

    def one(b):
        L.oracle_select_top_p_seq(w.H_kv, w.page_size, w.max_pages_per_seq, sc[b].ctypes.data,
                                  int(w.seq_lens[b]), float(top_p), float(score_scale),
                                  pol.sink_pages, pol.local_pages, k_max, sel[b].ctypes.data,
                                  nsel[b].ctypes.data)
    _run(one, _seqs(w, seqs), threads)
    return sel, nsel
