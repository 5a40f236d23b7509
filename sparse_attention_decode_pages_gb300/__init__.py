"""Sparse paged decode attention for GB300: a thin Python binding over ``libspd.so``.

The functions here carry the names of the C ABI (``include/spd.h``) and only
marshal arguments: every step runs in the library's CUDA kernels.  PyTorch
supplies device memory and the current stream.  There is no fallback: if the
library is missing or a call fails, a ``SpdError`` is raised.

Tensors: bf16 data may be ``torch.bfloat16`` or ``torch.uint16`` (same bits);
index data is ``torch.int32``; everything contiguous and on the current device.
Workspaces are zero-initialised byte tensors (see ``workspace``); each call
leaves its counters at zero, so a workspace can be reused on one stream.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "SpdError", "Dims", "Policy", "RoundDesc", "Round", "lib", "dims_of", "policy_of", "workspace",
    "pages_summarize", "kv_append_refresh", "pages_score_select", "pages_append_score_select",
    "sparse_decode_attn", "sparse_decode_attn_noalloc", "sparse_decode_step", "dense_verify_attn",
    "lse_merge", "spec_accept", "spd_device_status", "spd_score_select_workspace_size",
    "spd_sparse_decode_workspace_size", "spd_dense_verify_workspace_size",
    "spd_sparse_decode_step_workspace_size", "spd_set_wait_limit_ns", "spd_wait_limit_ns",
    "DEV_BAD_PAGE", "DEV_BAD_SEL", "DEV_TIMEOUT", "DEV_BAD_LEN", "DEV_BAD_TOKEN",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspd.so")

# device status bits (SPD_DEV_* in include/spd.h)
DEV_BAD_PAGE, DEV_BAD_SEL, DEV_TIMEOUT, DEV_BAD_LEN, DEV_BAD_TOKEN = 0x1, 0x2, 0x4, 0x8, 0x10
_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "WORKSPACE"}
_MODES = {"fixed": 0, "linear": 1, "fraction": 2, "top_p": 3}


class SpdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"spd {_STATUS.get(status, status)}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_phys_pages", ctypes.c_int64)]


class Policy(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("fixed_pages", ctypes.c_int32),
                ("min_tokens", ctypes.c_int64), ("slope_num", ctypes.c_int64),
                ("slope_den", ctypes.c_int64), ("intercept", ctypes.c_int64),
                ("frac_num", ctypes.c_int64), ("frac_den", ctypes.c_int64),
                ("sink_pages", ctypes.c_int32), ("local_pages", ctypes.c_int32),
                ("top_p", ctypes.c_float), ("score_scale", ctypes.c_float)]


class RoundDesc(ctypes.Structure):
    _fields_ = [("dims", Dims), ("k", ctypes.c_int32),
                ("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("summ", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("q_draft", ctypes.c_void_p), ("k_draft", ctypes.c_void_p), ("v_draft", ctypes.c_void_p),
                ("q_verify", ctypes.c_void_p), ("k_verify", ctypes.c_void_p), ("v_verify", ctypes.c_void_p),
                ("policy", Policy), ("k_max", ctypes.c_int32),
                ("sel", ctypes.c_void_p), ("nsel", ctypes.c_void_p),
                ("o_draft", ctypes.c_void_p), ("lse_draft", ctypes.c_void_p),
                ("o_verify", ctypes.c_void_p), ("lse_verify", ctypes.c_void_p),
                ("n_vocab", ctypes.c_int32),
                ("p_draft", ctypes.c_void_p), ("q_target", ctypes.c_void_p),
                ("draft_tokens", ctypes.c_void_p), ("u_acc", ctypes.c_void_p), ("u_res", ctypes.c_void_p),
                ("n_accepted", ctypes.c_void_p), ("tokens", ctypes.c_void_p),
                ("ws_select", ctypes.c_void_p), ("ws_select_bytes", ctypes.c_size_t),
                ("ws_sparse", ctypes.c_void_p), ("ws_sparse_bytes", ctypes.c_size_t),
                ("ws_verify", ctypes.c_void_p), ("ws_verify_bytes", ctypes.c_size_t),
                ("sparse_splits", ctypes.c_int32), ("verify_splits", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


_lib = None


def lib():
    """Load libspd.so (fails loudly when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise SpdError(3, f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        DP, PP = ctypes.POINTER(Dims), ctypes.POINTER(Policy)
        L.spd_version.restype = i32
        L.spd_last_error.restype = ctypes.c_char_p
        L.spd_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        L.spd_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.spd_wait_limit_ns.restype = ctypes.c_uint64
        L.spd_score_select_workspace_size.argtypes = [DP]
        L.spd_score_select_workspace_size.restype = sz
        L.spd_sparse_decode_workspace_size.argtypes = [DP, i32, i32]
        L.spd_sparse_decode_workspace_size.restype = sz
        L.spd_dense_verify_workspace_size.argtypes = [DP, i32, i32]
        L.spd_dense_verify_workspace_size.restype = sz
        L.pages_summarize.argtypes = [DP, P, P, P, P, i32, P, P]
        L.pages_score_select.argtypes = [DP, P, P, P, PP, P, P, i32, P, P, sz, P]
        L.sparse_decode_attn.argtypes = [DP, P, P, P, P, P, P, P, i32, i32, ctypes.c_float,
                                         P, P, P, sz, P]
        L.dense_verify_attn.argtypes = [DP, i32, P, P, P, P, P, i32, ctypes.c_float, P, P, P, sz, P]
        L.sparse_decode_attn_noalloc.argtypes = [DP, P, P, P, P, P, P, P, i32, i32, ctypes.c_float,
                                                 P, P, P]
        L.lse_merge.argtypes = [i32, i32, i32, P, P, P, P, P]
        L.kv_append_refresh.argtypes = [DP, i32, P, P, P, P, P, P, P, P]
        L.spec_accept.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P]
        L.pages_append_score_select.argtypes = [DP, P, P, P, P, P, P, P, P, PP, P, P, i32, P, P, sz, P]
        L.spd_sparse_decode_step_workspace_size.argtypes = [DP, i32]
        L.spd_sparse_decode_step_workspace_size.restype = sz
        L.sparse_decode_step.argtypes = [DP, P, P, P, P, P, P, P, P, PP, P, P, i32, ctypes.c_float, P, P,
                                         P, sz, P]
        L.spd_round_create.argtypes = [ctypes.POINTER(RoundDesc), ctypes.POINTER(ctypes.c_void_p)]
        L.spd_round_launch.argtypes = [P, i32, P]
        L.spd_round_destroy.argtypes = [P]
        L.spd_round_destroy.restype = None
        for f in ("spd_device_status", "spd_set_wait_limit_ns", "pages_summarize", "pages_score_select",
                  "sparse_decode_attn", "dense_verify_attn", "lse_merge",
                  "sparse_decode_attn_noalloc", "kv_append_refresh", "spec_accept",
                  "pages_append_score_select", "sparse_decode_step",
                  "spd_round_create", "spd_round_launch"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise SpdError(status, lib().spd_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise SpdError(1, "tensor is not on a CUDA device")
    if not t.is_contiguous():
        raise SpdError(1, "tensor is not contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def dims_of(B, H_q, H_kv, D, page_size, max_pages_per_seq, num_phys_pages) -> Dims:
    return Dims(B, H_q, H_kv, D, page_size, max_pages_per_seq, num_phys_pages)


def policy_of(p) -> Policy:
    """A ``Policy`` from any object with the fields of ``workloads.BudgetPolicy``."""
    return Policy(_MODES[p.mode] if isinstance(p.mode, str) else int(p.mode), p.fixed_pages,
                  p.min_tokens, p.slope_num, p.slope_den, p.intercept, p.frac_num, p.frac_den,
                  p.sink_pages, p.local_pages, float(getattr(p, "top_p", 0.0)),
                  float(getattr(p, "score_scale", 0.0)))


def _size(v: int, what: str) -> int:
    if v == 0:
        raise SpdError(1, f"{what}: " + lib().spd_last_error().decode(errors="replace"))
    return v


def spd_score_select_workspace_size(dims: Dims) -> int:
    """Bytes of workspace pages_score_select needs for these dims."""
    return _size(lib().spd_score_select_workspace_size(ctypes.byref(dims)), "score_select workspace")


def spd_sparse_decode_workspace_size(dims: Dims, k_max: int, num_splits: int = 0) -> int:
    """Bytes of workspace sparse_decode_attn needs (num_splits 0: the automatic split count)."""
    return _size(lib().spd_sparse_decode_workspace_size(ctypes.byref(dims), k_max, num_splits),
                 "sparse_decode workspace")


def spd_dense_verify_workspace_size(dims: Dims, T: int, num_splits: int = 0) -> int:
    """Bytes of workspace dense_verify_attn needs for T positions."""
    return _size(lib().spd_dense_verify_workspace_size(ctypes.byref(dims), T, num_splits),
                 "dense_verify workspace")


def workspace(nbytes: int, device=None):
    """A zeroed byte tensor usable as a workspace (allocated by PyTorch, not the library)."""
    import torch
    return torch.zeros(max(1, int(nbytes)), dtype=torch.uint8, device=device or "cuda")


def spd_device_status(clear: bool = False) -> int:
    """The device status word (DEV_* bits raised by kernels since the last clear); waits for the device."""
    v = ctypes.c_uint32(0)
    _check(lib().spd_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


def spd_set_wait_limit_ns(ns: int):
    """Limit (ns) of every bounded wait in kernels launched from now on (2 s by default)."""
    _check(lib().spd_set_wait_limit_ns(int(ns)))


def spd_wait_limit_ns() -> int:
    """The current limit of the kernels' bounded waits, in nanoseconds."""
    return int(lib().spd_wait_limit_ns())


def pages_summarize(dims: Dims, K, page_table, seq_lens, summ, only_pages=None, stream=None):
    """Per-page key min / max summaries into summ (all pages, or the listed b * max_pages + p slots)."""
    n_only = 0 if only_pages is None else only_pages.numel()
    _check(lib().pages_summarize(ctypes.byref(dims), _ptr(K), _ptr(page_table), _ptr(seq_lens),
                                 _ptr(only_pages), n_only, _ptr(summ), _stream(stream)))


def kv_append_refresh(dims: Dims, T: int, K, V, page_table, seq_lens, k_new, v_new, summ,
                      stream=None):
    """Write the T newest tokens into the paged cache and rebuild the summaries of their pages."""
    _check(lib().kv_append_refresh(ctypes.byref(dims), T, _ptr(K), _ptr(V), _ptr(page_table),
                                   _ptr(seq_lens), _ptr(k_new), _ptr(v_new), _ptr(summ),
                                   _stream(stream)))


def spec_accept(p_draft, q_target, draft, u_acc, u_res, n_accepted, tokens, stream=None):
    """p_draft [B][k][n], q_target [B][k+1][n] (fp32), draft int32 [B][k], u_acc [B][k], u_res [B]."""
    B, k, n = p_draft.shape
    _check(lib().spec_accept(B, k, n, _ptr(p_draft), _ptr(q_target), _ptr(draft), _ptr(u_acc),
                             _ptr(u_res), _ptr(n_accepted), _ptr(tokens), _stream(stream)))


def pages_append_score_select(dims: Dims, K, V, page_table, seq_lens, k_new, v_new, q, summ, policy,
                              sel, nsel, k_max: int, ws, scores=None, stream=None):
    """kv_append_refresh (T = 1) fused into pages_score_select's pass over the summaries."""
    pol = policy if isinstance(policy, Policy) else policy_of(policy)
    _check(lib().pages_append_score_select(ctypes.byref(dims), _ptr(K), _ptr(V), _ptr(page_table),
                                           _ptr(seq_lens), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(summ),
                                           ctypes.byref(pol), _ptr(sel), _ptr(nsel), k_max, _ptr(scores),
                                           _ptr(ws), ws.numel(), _stream(stream)))


def spd_sparse_decode_step_workspace_size(dims: Dims, k_max: int) -> int:
    """Bytes of workspace sparse_decode_step needs."""
    return _size(lib().spd_sparse_decode_step_workspace_size(ctypes.byref(dims), k_max), "decode step workspace")


def sparse_decode_step(dims: Dims, K, V, page_table, seq_lens, k_new, v_new, q, summ, policy, sel, nsel,
                       k_max: int, o, ws, lse=None, softmax_scale: float | None = None, stream=None):
    """Append (k_new / v_new may be None) + score + select + sparse attention in one call."""
    pol = policy if isinstance(policy, Policy) else policy_of(policy)
    scale = 1.0 / math.sqrt(dims.D) if softmax_scale is None else softmax_scale
    _check(lib().sparse_decode_step(ctypes.byref(dims), _ptr(K), _ptr(V), _ptr(page_table), _ptr(seq_lens),
                                    _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(summ), ctypes.byref(pol), _ptr(sel),
                                    _ptr(nsel), k_max, scale, _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(stream)))


def pages_score_select(dims: Dims, q, summ, seq_lens, policy, sel, nsel, k_max: int, ws,
                       scores=None, stream=None):
    """Page upper-bound scores and the budgeted selection (ascending page ids) per (sequence, KV head)."""
    pol = policy if isinstance(policy, Policy) else policy_of(policy)
    _check(lib().pages_score_select(ctypes.byref(dims), _ptr(q), _ptr(summ), _ptr(seq_lens),
                                    ctypes.byref(pol), _ptr(sel), _ptr(nsel), k_max,
                                    _ptr(scores), _ptr(ws), ws.numel(), _stream(stream)))


def sparse_decode_attn(dims: Dims, q, K, V, page_table, seq_lens, sel, nsel, k_max: int, o, ws,
                       lse=None, num_splits: int = 0, softmax_scale: float | None = None,
                       stream=None):
    """Attention of the decode query over the selected pages (split-K, merged)."""
    scale = 1.0 / math.sqrt(dims.D) if softmax_scale is None else softmax_scale
    _check(lib().sparse_decode_attn(ctypes.byref(dims), _ptr(q), _ptr(K), _ptr(V), _ptr(page_table),
                                    _ptr(seq_lens), _ptr(sel), _ptr(nsel), k_max, num_splits,
                                    scale, _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(stream)))


def sparse_decode_attn_noalloc(dims: Dims, q, K, V, page_table, seq_lens, sel, nsel, k_max: int, o,
                               lse=None, num_splits: int = 0, softmax_scale: float | None = None,
                               stream=None):
    """sparse_decode_attn without a workspace: its scratch is a fixed array inside the library."""
    scale = 1.0 / math.sqrt(dims.D) if softmax_scale is None else softmax_scale
    _check(lib().sparse_decode_attn_noalloc(ctypes.byref(dims), _ptr(q), _ptr(K), _ptr(V),
                                            _ptr(page_table), _ptr(seq_lens), _ptr(sel), _ptr(nsel),
                                            k_max, num_splits, scale, _ptr(o), _ptr(lse),
                                            _stream(stream)))


def dense_verify_attn(dims: Dims, T: int, q, K, V, page_table, seq_lens, o, ws, lse=None,
                      num_splits: int = 0, softmax_scale: float | None = None, stream=None):
    """Causal attention of the T newest positions over the whole cache."""
    scale = 1.0 / math.sqrt(dims.D) if softmax_scale is None else softmax_scale
    _check(lib().dense_verify_attn(ctypes.byref(dims), T, _ptr(q), _ptr(K), _ptr(V),
                                   _ptr(page_table), _ptr(seq_lens), num_splits, scale, _ptr(o),
                                   _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def lse_merge(part_o, part_lse, o, lse=None, stream=None):
    """Merge split partials (part_o [S][rows][D], part_lse [S][rows]) by the log-sum-exp rule."""
    S, rows, D = part_o.shape
    _check(lib().lse_merge(S, rows, D, _ptr(part_o), _ptr(part_lse), _ptr(o), _ptr(lse),
                           _stream(stream)))


class Round:
    """spd_round: one S3R round (k sparse draft steps, verification, sampling) as two
    CUDA graphs built by the library.  Takes device tensors laid out as include/spd.h
    states; keeps them referenced while the round lives.  ``sampling`` is None or a dict
    with p_draft, q_target, draft_tokens, u_acc, u_res, n_accepted, tokens."""

    def __init__(self, dims: Dims, k: int, K, V, summ, page_table, seq_lens, q_draft, k_draft,
                 v_draft, q_verify, k_verify, v_verify, policy, k_max: int, sel, nsel, o_draft,
                 o_verify, ws_select, ws_sparse, ws_verify, lse_draft=None, lse_verify=None,
                 sampling=None, sparse_splits: int = 0, verify_splits: int = 0,
                 softmax_scale: float | None = None):
        pol = policy if isinstance(policy, Policy) else policy_of(policy)
        scale = 1.0 / math.sqrt(dims.D) if softmax_scale is None else softmax_scale
        smp = sampling or {}
        self._keep = [K, V, summ, page_table, seq_lens, q_draft, k_draft, v_draft, q_verify,
                      k_verify, v_verify, sel, nsel, o_draft, o_verify, ws_select, ws_sparse,
                      ws_verify, lse_draft, lse_verify, *smp.values()]
        n_vocab = int(smp["q_target"].shape[-1]) if smp else 0
        g = lambda name: _ptr(smp.get(name))
        d = RoundDesc(dims, k, _ptr(K), _ptr(V), _ptr(summ), _ptr(page_table), _ptr(seq_lens),
                      _ptr(q_draft), _ptr(k_draft), _ptr(v_draft), _ptr(q_verify), _ptr(k_verify),
                      _ptr(v_verify), pol, k_max, _ptr(sel), _ptr(nsel), _ptr(o_draft),
                      _ptr(lse_draft), _ptr(o_verify), _ptr(lse_verify), n_vocab,
                      g("p_draft"), g("q_target"), g("draft_tokens"), g("u_acc"), g("u_res"),
                      g("n_accepted"), g("tokens"),
                      _ptr(ws_select), ws_select.numel(), _ptr(ws_sparse), ws_sparse.numel(),
                      _ptr(ws_verify), ws_verify.numel(), sparse_splits, verify_splits, scale)
        h = ctypes.c_void_p()
        _check(lib().spd_round_create(ctypes.byref(d), ctypes.byref(h)))
        self._h = h

    def launch(self, part: int = 2, stream=None):
        """Replay part 0 (draft steps), 1 (verification + sampling) or 2 (both)."""
        _check(lib().spd_round_launch(self._h, part, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            lib().spd_round_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
