"""Test helpers: hand-built workloads with explicit values (no method arithmetic)."""
from __future__ import annotations

import numpy as np

from sparse_attention_decode_pages_gb300 import workloads as wl


def custom(lens, H_q, H_kv, D, ps, *, rng=None, K=None, V=None, q=None, q_verify=None, T=0,
           policy=None, k_max=None, permute=True, poison=True):
    """A Workload from explicit float32 token arrays.

    K, V: per sequence, float32 [len_b][H_kv][D] (token-major); they are scattered
    into pages of ``ps`` tokens over a (optionally permuted) physical page order.
    Missing arrays are drawn N(0, 1) from ``rng``.  Values are rounded to bf16.
    """
    rng = rng or np.random.default_rng(0)
    lens = np.asarray(lens, dtype=np.int32)
    B = len(lens)
    pages = (lens.astype(np.int64) + ps - 1) // ps
    max_pages = max(1, int(pages.max()))
    P_phys = max(1, int(pages.sum()))
    order = rng.permutation(P_phys) if permute else np.arange(P_phys)
    pt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        pt[b, : pages[b]] = order[off: off + pages[b]]
        off += int(pages[b])
    Kp = np.zeros((P_phys, H_kv, ps, D), dtype=np.float32)
    Vp = np.zeros_like(Kp)
    if poison:
        Kp[:] = wl.POISON_K
        Vp[:] = wl.POISON_V
    for b in range(B):
        n = int(lens[b])
        kb = K[b] if K is not None else rng.standard_normal((n, H_kv, D)).astype(np.float32)
        vb = V[b] if V is not None else rng.standard_normal((n, H_kv, D)).astype(np.float32)
        for j in range(n):
            Kp[pt[b, j // ps], :, j % ps, :] = kb[j]
            Vp[pt[b, j // ps], :, j % ps, :] = vb[j]
    qq = q if q is not None else rng.standard_normal((B, H_q, D)).astype(np.float32)
    qv = None
    if T:
        qv = q_verify if q_verify is not None else rng.standard_normal((B, T, H_q, D)).astype(np.float32)
        qv = wl.f32_to_bf16_bits(np.asarray(qv, dtype=np.float32))
    policy = policy or wl.BudgetPolicy("fixed", fixed_pages=max_pages, sink_pages=1, local_pages=1)
    return wl.Workload("custom", B, H_q, H_kv, D, ps, max_pages, P_phys, lens, pt,
                       wl.f32_to_bf16_bits(np.asarray(qq, dtype=np.float32)),
                       wl.f32_to_bf16_bits(Kp), wl.f32_to_bf16_bits(Vp), policy,
                       k_max if k_max is not None else max_pages, T, qv)


def f(h):
    """bf16 bits -> float64."""
    return wl.bf16_bits_to_f32(h).astype(np.float64)


def token_kv(w, b, h):
    """float64 keys and values of sequence b, KV head h, in token order: ([len][D], [len][D])."""
    n = int(w.seq_lens[b])
    ps = w.page_size
    idx = [(w.page_table[b, j // ps], j % ps) for j in range(n)]
    Kt = np.array([f(w.K[p, h, t]) for p, t in idx]).reshape(n, w.D)
    Vt = np.array([f(w.V[p, h, t]) for p, t in idx]).reshape(n, w.D)
    return Kt, Vt
