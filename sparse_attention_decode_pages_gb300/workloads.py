"""Seeded synthetic inputs for sparse paged decode attention.

This module holds only input generation: shapes, seeds, random draws and the
float32 -> bfloat16 storage conversion.  It contains none of the method's
arithmetic (no summaries, scores, selection or softmax), so both the CUDA path
and the fp64 oracle can be fed from it without sharing any computation.

The five workloads follow the shapes of the Qwen3 rollout studies on the
Sparrow project page ("Control Study 2", page-size study) and the S3R appendix
(Table 4 settings, Table 7 draft/verify with k=6), at synthetic values:

=========  ===  ========  ===  ==========================  ====  =========================================
name        B   Hq / Hkv   D   context length (tokens)       ps   budget (pages)
=========  ===  ========  ===  ==========================  ====  =========================================
tiny        2    4 / 2     64   1024 each                    16   8 fixed, sink page 0 + last page
q17b       64   16 / 8    128   U[4096, 16384]               16   128 fixed (2048 tokens), sink + 4 local
q8b        64   32 / 8    128   8192 + U[0, 8192]            16   64 fixed (1024 tokens), sink + 4 local;
                                                                   dense verify of k+1 = 7 positions
sweep      32   32 / 8    128   U[16384, 32768]              16/32/64  ceil(max(512, len/50 + 256) / ps)
longtail    8   32 / 8    128   U[65536, 131072]             32   ceil(len / 16 / ps), split-K
=========  ===  ========  ===  ==========================  ====  =========================================

Recipe (all draws from numpy PCG64, seed ``1000 + index`` with index 1..5 in
the order above; the sweep adds the page size to the seed):

* lengths: uniform integers in the stated inclusive range.
* physical pages: the sequences' logical pages are laid out over a random
  permutation of ``sum_b ceil(len_b / ps)`` physical pages; page-table slots
  past a sequence's last page hold -1 and are never read.
* q, K, V: N(0, 1) rounded to bf16, except the sweep's keys, which are
  Student-t with 3 degrees of freedom (unscaled).
* planted retrieval tokens (q17b, sweep: 8 per sequence): positions drawn
  uniformly outside the sink page and the local window; at each, every KV
  head g gets the key ``4 * qbar_g / rms(qbar_g)``, where ``qbar_g`` is the
  mean of that head's group of decode queries.
* sink-biased first page (longtail): token 0 gets the same aligned key.
* cache slots past ``len_b`` inside a sequence's last page are filled with
  +64 (K) and -64 (V): a kernel that fails to mask them produces a visibly
  wrong answer.

Large arrays are generated in fixed chunks, each with its own child seed, so
the bytes do not depend on how many threads generate them.

Speculative-sampling inputs (``spec_inputs``; S3R Table 7: k = 6 drafts per
round, Qwen3's 151,936-token vocabulary): each drafter row p_i is a Dirichlet
draw with concentration 0.05 per token (peaked, like a sampled LM
distribution); each target row is (1 - eps) * p_i + eps * (an independent
Dirichlet draw), eps = 0.3, and the row after the last draft is a fresh
Dirichlet draw.  Drafted tokens are drawn from p_i; the uniform numbers are
float32 draws in [0, 1).  Seed 1006.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

POISON_K = 64.0
POISON_V = -64.0
_CHUNK = 1 << 24  # elements per independently seeded chunk


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class BudgetPolicy:
    """Per-sequence page budget.

    mode "fixed": ``fixed_pages`` pages.
    mode "linear": ``ceil(max(min_tokens, slope_num * len / slope_den + intercept) / ps)`` pages,
        evaluated in exact integer arithmetic.
    mode "fraction": ``ceil(len * frac_num / (frac_den * ps))`` pages.
    mode "top_p": the smallest set holding ``top_p`` of the page weight
        ``exp(score_scale * (score - max score))``, at most k_max pages.
    ``sink_pages`` leading pages and ``local_pages`` trailing pages are always kept.
    """

    mode: str = "fixed"
    fixed_pages: int = 0
    min_tokens: int = 0
    slope_num: int = 0
    slope_den: int = 1
    intercept: int = 0
    frac_num: int = 1
    frac_den: int = 1
    sink_pages: int = 1
    local_pages: int = 1
    top_p: float = 0.0
    score_scale: float = 0.0


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    page_size: int
    max_pages_per_seq: int
    num_phys_pages: int
    seq_lens: np.ndarray  # int32 [B]
    page_table: np.ndarray  # int32 [B][max_pages_per_seq]
    q: np.ndarray  # uint16 (bf16 bits) [B][H_q][D]
    K: np.ndarray  # uint16 [num_phys_pages][H_kv][page_size][D]
    V: np.ndarray  # uint16 [num_phys_pages][H_kv][page_size][D]
    policy: BudgetPolicy
    k_max: int
    T: int = 0  # draft positions verified (0 = no verify query)
    q_verify: np.ndarray | None = None  # uint16 [B][T][H_q][D]
    planted: list = dataclasses.field(default_factory=list)  # per sequence: token positions

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def pages(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.page_size)


@dataclasses.dataclass
class Spec:
    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    page_size: int
    len_lo: int
    len_hi: int
    policy: BudgetPolicy
    seed: int
    T: int = 0
    planted_per_seq: int = 0
    sink_biased: bool = False
    keys: str = "normal"  # or "student_t3"
    k_max: int | None = None


def _k_max_for(spec: Spec) -> int:
    """Largest selection any sequence of this spec can need (sizes the selection buffer)."""
    if spec.k_max is not None:
        return spec.k_max
    ps = spec.page_size
    pmax = -(-spec.len_hi // ps)
    p = spec.policy
    if p.mode == "fixed":
        need = p.fixed_pages
    elif p.mode == "linear":
        tok = max(p.min_tokens, -(-(p.slope_num * spec.len_hi) // p.slope_den) + p.intercept)
        need = -(-tok // ps)
    else:
        need = -(-(spec.len_hi * p.frac_num) // (p.frac_den * ps))
    need = max(need, p.sink_pages + p.local_pages)
    return int(min(pmax, need))


def spec(name: str, page_size: int | None = None, **over) -> Spec:
    """The named workload's specification; keyword arguments override fields (for small cases)."""
    if name == "tiny":
        s = Spec("tiny", 2, 4, 2, 64, 16, 1024, 1024,
                 BudgetPolicy("fixed", fixed_pages=8, sink_pages=1, local_pages=1), seed=1001)
    elif name == "q17b":
        s = Spec("q17b", 64, 16, 8, 128, 16, 4096, 16384,
                 BudgetPolicy("fixed", fixed_pages=128, sink_pages=1, local_pages=4), seed=1002,
                 planted_per_seq=8)
    elif name == "q8b":
        s = Spec("q8b", 64, 32, 8, 128, 16, 8192, 16384,
                 BudgetPolicy("fixed", fixed_pages=64, sink_pages=1, local_pages=4), seed=1003, T=7)
    elif name == "sweep":
        ps = page_size or 16
        s = Spec("sweep", 32, 32, 8, 128, ps, 16384, 32768,
                 BudgetPolicy("linear", min_tokens=512, slope_num=1, slope_den=50, intercept=256,
                              sink_pages=1, local_pages=4), seed=1004 + ps, planted_per_seq=8,
                 keys="student_t3")
    elif name == "longtail":
        s = Spec("longtail", 8, 32, 8, 128, 32, 65536, 131072,
                 BudgetPolicy("fraction", frac_num=1, frac_den=16, sink_pages=1, local_pages=4),
                 seed=1005, sink_biased=True)
    else:
        raise ValueError(f"unknown workload {name!r}")
    if page_size is not None and name != "sweep":
        s.page_size = page_size
    for k, v in over.items():
        if k == "policy_over":
            s.policy = dataclasses.replace(s.policy, **v)
        else:
            setattr(s, k, v)
    return s


def _fill(out: np.ndarray, ss: np.random.SeedSequence, kind: str, threads: int) -> None:
    """Fill a flat uint16 array with bf16-rounded draws, chunk i seeded by ss.spawn order."""
    n = out.size
    nchunks = -(-n // _CHUNK)
    children = ss.spawn(nchunks)

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        rng = np.random.Generator(np.random.PCG64(children[i]))
        if kind == "normal":
            x = rng.standard_normal(hi - lo, dtype=np.float32)
        elif kind == "student_t3":
            x = rng.standard_t(3, hi - lo).astype(np.float32)
        else:
            raise ValueError(kind)
        out[lo:hi] = f32_to_bf16_bits(x)

    if threads <= 1 or nchunks == 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))


def _aligned_keys(qb: np.ndarray, H_kv: int) -> np.ndarray:
    """Per KV head g: 4 * qbar_g / rms(qbar_g), qbar_g = mean of the group's queries (float32)."""
    H_q, D = qb.shape
    G = H_q // H_kv
    qf = bf16_bits_to_f32(qb).reshape(H_kv, G, D).astype(np.float64)
    qbar = qf.mean(axis=1)
    rms = np.sqrt((qbar * qbar).mean(axis=1, keepdims=True))
    rms[rms == 0] = 1.0
    return (4.0 * qbar / rms).astype(np.float32)


def make(s: Spec, threads: int | None = None) -> Workload:
    """Generate the workload described by ``s``.  Deterministic in ``s``."""
    threads = threads or min(16, os.cpu_count() or 1)
    root = np.random.SeedSequence(s.seed)
    ss_len, ss_perm, ss_q, ss_k, ss_v, ss_plant, ss_qv = root.spawn(7)
    ps = s.page_size
    rng_len = np.random.Generator(np.random.PCG64(ss_len))
    lens = rng_len.integers(s.len_lo, s.len_hi + 1, size=s.B).astype(np.int32)
    pages = (lens.astype(np.int64) + ps - 1) // ps
    max_pages = int(-(-s.len_hi // ps))
    P_phys = int(pages.sum())
    perm = np.random.Generator(np.random.PCG64(ss_perm)).permutation(P_phys).astype(np.int32)
    page_table = np.full((s.B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(s.B):
        page_table[b, : pages[b]] = perm[off: off + pages[b]]
        off += int(pages[b])

    q = np.empty((s.B, s.H_q, s.D), dtype=np.uint16)
    _fill(q.reshape(-1), ss_q, "normal", 1)
    K = np.empty((P_phys, s.H_kv, ps, s.D), dtype=np.uint16)
    V = np.empty_like(K)
    _fill(K.reshape(-1), ss_k, s.keys, threads)
    _fill(V.reshape(-1), ss_v, "normal", threads)

    pk = f32_to_bf16_bits(np.float32(POISON_K))
    pv = f32_to_bf16_bits(np.float32(POISON_V))
    for b in range(s.B):
        tail = int(lens[b]) % ps
        if tail:
            last = page_table[b, pages[b] - 1]
            K[last, :, tail:, :] = pk
            V[last, :, tail:, :] = pv

    rng_plant = np.random.Generator(np.random.PCG64(ss_plant))
    planted = []
    W = s.policy.local_pages
    S0 = s.policy.sink_pages
    for b in range(s.B):
        pos_list = []
        keys = None
        if s.planted_per_seq:
            lo, hi = S0 * ps, (int(pages[b]) - W) * ps
            if hi - lo >= s.planted_per_seq:
                pos_list = sorted(rng_plant.choice(np.arange(lo, hi), s.planted_per_seq,
                                                   replace=False).tolist())
        if s.sink_biased:
            pos_list = [0] + pos_list
        if pos_list:
            keys = f32_to_bf16_bits(_aligned_keys(q[b], s.H_kv))  # [H_kv][D]
            for pos in pos_list:
                K[page_table[b, pos // ps], :, pos % ps, :] = keys
        planted.append(pos_list)

    q_verify = None
    if s.T:
        q_verify = np.empty((s.B, s.T, s.H_q, s.D), dtype=np.uint16)
        _fill(q_verify.reshape(-1), ss_qv, "normal", 1)

    return Workload(s.name, s.B, s.H_q, s.H_kv, s.D, ps, max_pages, P_phys, lens, page_table,
                    q, K, V, s.policy, _k_max_for(s), s.T, q_verify, planted)


def named(name: str, page_size: int | None = None, threads: int | None = None, **over) -> Workload:
    return make(spec(name, page_size, **over), threads)


def to_device(w: Workload, device="cuda") -> dict:
    """Copy a workload's arrays to the GPU as torch tensors (bf16 data keeps its bit patterns)."""
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)

    out = dict(
        q=bf(w.q), K=bf(w.K), V=bf(w.V),
        page_table=torch.from_numpy(w.page_table).to(device),
        seq_lens=torch.from_numpy(w.seq_lens).to(device),
    )
    if w.q_verify is not None:
        out["q_verify"] = bf(w.q_verify)
    return out


VOCAB_QWEN3 = 151936


def _dirichlet_rows(rng, rows: int, n: int, alpha: float) -> np.ndarray:
    g = rng.standard_gamma(alpha, size=(rows, n))
    g /= g.sum(axis=1, keepdims=True)
    return g


def spec_inputs(B: int = 64, k: int = 6, n: int = VOCAB_QWEN3, seed: int = 1006,
                alpha: float = 0.05, eps: float = 0.3) -> dict:
    """Seeded drafter / target probability rows and the random numbers of one round.

    Returns p float32 [B][k][n], q float32 [B][k+1][n], draft int32 [B][k], u_acc
    float32 [B][k], u_res float32 [B]."""
    rng = np.random.default_rng(seed)
    p = np.empty((B, k, n), np.float32)
    q = np.empty((B, k + 1, n), np.float32)
    draft = np.empty((B, k), np.int32)
    for b in range(B):
        pb = _dirichlet_rows(rng, k, n, alpha)
        mix = _dirichlet_rows(rng, k + 1, n, alpha)
        p[b] = pb
        q[b, :k] = (1.0 - eps) * pb + eps * mix[:k]
        q[b, k] = mix[k]
        c = np.cumsum(pb, axis=1)
        u = rng.random(k)
        draft[b] = np.minimum([np.searchsorted(c[i], u[i] * c[i, -1], side="right") for i in range(k)], n - 1)
    u_acc = rng.random((B, k), dtype=np.float32)
    u_res = rng.random(B, dtype=np.float32)
    return dict(p=p, q=q, draft=draft, u_acc=u_acc, u_res=u_res)


def round_inputs(w: Workload, k: int = 6, seed: int = 1007, n_vocab: int = 0) -> dict:
    """Seeded inputs of one S3R round on workload ``w`` (k sparse draft steps, then
    verification of k + 1 positions), with w.seq_lens as the verification lengths.

    Draft step s appends position L0 + s with L0 = seq_lens - (k + 1), so its lengths
    are L0 + s + 1.  Returns seq_lens int32 [k+1][B]; q_draft [k][B][H_q][D],
    k_draft / v_draft [k][B][H_kv][D], q_verify [B][k+1][H_q][D], k_verify / v_verify
    [B][k+1][H_kv][D] (bf16 bits, N(0, 1)); with n_vocab > 0 also the sampling inputs
    of ``spec_inputs`` (p, q, draft, u_acc, u_res)."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D = w.B, w.H_q, w.H_kv, w.D
    L0 = w.seq_lens.astype(np.int64) - (k + 1)
    if L0.min() < 0:
        raise ValueError("every sequence needs at least k + 1 tokens")
    lens = np.stack([L0 + s + 1 for s in range(k)] + [w.seq_lens.astype(np.int64)]).astype(np.int32)
    bf = lambda shape: f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    out = dict(seq_lens=lens, q_draft=bf((k, B, Hq, D)), k_draft=bf((k, B, Hkv, D)),
               v_draft=bf((k, B, Hkv, D)), q_verify=bf((B, k + 1, Hq, D)),
               k_verify=bf((B, k + 1, Hkv, D)), v_verify=bf((B, k + 1, Hkv, D)))
    if n_vocab:
        out.update(spec_inputs(B=B, k=k, n=n_vocab, seed=seed + 1))
    return out
