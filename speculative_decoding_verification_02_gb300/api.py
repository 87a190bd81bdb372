"""ctypes binding over libspecverify.so.

The functions carry the C entry points' names and do argument marshalling
only: shapes and dtypes are read off torch tensors, pointers and strides are
passed through, outputs are allocated on the inputs' device, and the call is
enqueued on the current torch stream.  Every step of verification runs in the
library's CUDA kernels; there is no fallback.  Loading fails loudly when the
library has not been built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK, SPEC_EINVAL, SPEC_EDTYPE, SPEC_EWORKSPACE, SPEC_ECUDA = 0, -1, -2, -3, -4
STATUS_OK, STATUS_TOKEN_RANGE, STATUS_BAD_TREE, STATUS_BAD_LENGTH = 0, 1, 2, 3
DTYPE_F32, DTYPE_BF16 = 0, 1
OP_NGRAM, OP_GREEDY, OP_SAMPLE, OP_TREE, OP_DRAW, OP_FILTER = 0, 1, 2, 3, 4, 5
CHAIN_AUTO, CHAIN_TWO_PASS, CHAIN_FUSED, CHAIN_CHUNKED = 0, 1, 2, 3
TREE_SIBLINGS_WITHOUT_REPLACEMENT = 1

_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class SpecError(RuntimeError):
    """A libspecverify call returned a non-zero status."""


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, F, Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_size_t)
        L.spec_ngram_draft.argtypes = [P, P, I, I, I, I, P, P, P, P]
        L.spec_verify_greedy.argtypes = [P, I64, I64, I, I, I, I, P, P, P, P, P, P, P, P, Z, P]
        L.spec_verify_sample.argtypes = [P, I64, P, I64, I64, I, I, I, I, F, P, P, P, P, P, P, P,
                                         P, P, P, P, P, Z, P]
        L.spec_verify_tree.argtypes = [P, I64, P, I64, I64, I, I, I, I, F, P, P, P, I, P, P, P, P,
                                       P, P, Z, P]
        L.spec_verify_tree_ex.argtypes = [P, I64, P, I64, I64, I, I, I, I, F, P, P, P, I, I, P, P, P, P,
                                          P, P, Z, P]
        L.spec_workspace_size.argtypes = [I, I, I, I, I]
        L.spec_workspace_size.restype = Z
        L.spec_status_string.argtypes = [I]
        L.spec_status_string.restype = ctypes.c_char_p
        L.spec_last_error.argtypes = []
        L.spec_last_error.restype = ctypes.c_char_p
        L.spec_trace_enable.argtypes = [I]
        L.spec_trace_repeat.argtypes = [I]
        L.spec_trace_collect.argtypes = [P, P, P, I]
        L.spec_launch_count.argtypes = []
        L.spec_launch_count.restype = ctypes.c_int64
        L.spec_set_chain_path.argtypes = [I]
        L.spec_tree_rerank.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, P, P, P]
        L.spec_sample.argtypes = [P, I64, I, I, I, F, P, P, P, P, P, Z, P]
        L.spec_verify_sample_topkp.argtypes = [P, I64, P, I64, I64, I, I, I, I, F, I, F, P, P, P, P, P, P, P, P,
                                               P, P, P, P, Z, P]
        L.spec_sample_topkp.argtypes = [P, I64, I, I, I, F, I, F, P, P, P, P, P, Z, P]
        L.spec_filter_rows.argtypes = [P, I64, I, I, I, F, I, F, P, P, P, Z, P]
        D = ctypes.c_double
        L.spec_expected_tokens.argtypes = [D, I, P]
        L.spec_speedup.argtypes = [D, I, D, P]
        L.spec_best_k.argtypes = [D, D, I, P, P]
        L.spec_alpha_estimate.argtypes = [P, P, I, I, P, P]
        _lib = L
        return L


# ------------------------------------------------------------------ helpers

def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != SPEC_OK:
        L = lib()
        msg = L.spec_status_string(rc).decode()
        err = L.spec_last_error().decode()
        detail = err and rc in (SPEC_ECUDA, SPEC_EWORKSPACE)
        raise SpecError(f"{what}: {msg}" + (f" [{err}]" if detail else ""))


def _call(dev, fn, *args):
    """fn(*args) with the tensors' device current: the library sizes its
    launches for the current device, and the no-allocation entry point looks
    up its scratch array there."""
    with torch.cuda.device(dev):
        return fn(*args)


def _i32(t, shape, name, device):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or t.device != device:
        raise TypeError(f"{name} must be an int32 tensor on {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.contiguous()


def _f32(t, shape, name, device):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.device != device:
        raise TypeError(f"{name} must be a float32 tensor on {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.contiguous()


def _logits3(t, name):
    if t.dim() != 3 or (t.stride(2) != 1 and t.numel() > 0 and t.shape[2] > 1):
        raise ValueError(f"{name} must be [B, rows, V] with contiguous rows")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    return t


def spec_workspace_size(op: int, B: int, rows_per_req: int, V: int, dtype: int) -> int:
    return int(lib().spec_workspace_size(op, B, rows_per_req, V, dtype))


def workspace(nbytes: int, device, stream=None) -> torch.Tensor:
    """A 256-byte aligned workspace of at least nbytes.

    One buffer is cached per (device, stream): calls on one stream are
    ordered, so they may share it, while calls on different streams could
    overlap and must not."""
    device = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < max(nbytes, 1):
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)  # needs no initialisation
        if ws.data_ptr() % 256:
            raise RuntimeError("workspace allocation is not 256-byte aligned")
        _workspaces[key] = ws
    return ws


def set_chain_path(path: int):
    """Chain verification path for later calls, process-wide: CHAIN_AUTO,
    CHAIN_TWO_PASS, CHAIN_FUSED or CHAIN_CHUNKED (same results, different
    speed)."""
    _check(lib().spec_set_chain_path(int(path)), "spec_set_chain_path")


def trace_enable(on: bool = True):
    lib().spec_trace_enable(1 if on else 0)


def trace_repeat(reps: int = 1):
    """While tracing, launch each kernel reps times inside its event pair."""
    _check(lib().spec_trace_repeat(int(reps)), "spec_trace_repeat")


def trace_collect(cap: int = 16) -> dict:
    """{kernel name: (total ms, launches)} since the last collect."""
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_double * cap)()
    cnt = (ctypes.c_int64 * cap)()
    n = lib().spec_trace_collect(ctypes.cast(names, ctypes.c_void_p), ctypes.cast(ms, ctypes.c_void_p),
                                 ctypes.cast(cnt, ctypes.c_void_p), cap)
    if n < 0:
        _check(n, "spec_trace_collect")
    return {names[i].decode(): (ms[i], cnt[i]) for i in range(min(n, cap))}


def launch_count() -> int:
    return int(lib().spec_launch_count())


# --------------------------------------------------------------- entry points

def spec_ngram_draft(history: torch.Tensor, hist_len: torch.Tensor, window: int, k: int, *,
                     out=None, stream=None) -> dict:
    """history int32 [B, H], hist_len int32 [B] -> draft [B, k], draft_len [B], status [B]."""
    dev = history.device
    B, H = history.shape
    history = _i32(history, (B, H), "history", dev)
    hist_len = _i32(hist_len, (B,), "hist_len", dev)
    o = out or dict(draft=torch.empty((B, k), dtype=torch.int32, device=dev),
                    draft_len=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    rc = _call(dev, lib().spec_ngram_draft, _p(history), _p(hist_len), B, H, int(window), int(k), _p(o["draft"]),
                                _p(o["draft_len"]), _p(o["status"]), _stream(stream, dev))
    _check(rc, "spec_ngram_draft")
    return o


def spec_verify_greedy(target: torch.Tensor, draft: torch.Tensor, draft_len=None, max_emit=None, *,
                       out=None, ws=None, stream=None) -> dict:
    """target [B, k+1, V] fp32/bf16, draft int32 [B, k] -> accepted, out_tokens, n_emit, status."""
    target = _logits3(target, "target")
    dev = target.device
    B, R, V = target.shape
    k = R - 1
    draft = _i32(draft, (B, k), "draft", dev)
    draft_len = _i32(draft_len, (B,), "draft_len", dev)
    max_emit = _i32(max_emit, (B,), "max_emit", dev)
    dt = _dtype_code(target)
    need = spec_workspace_size(OP_GREEDY, B, k, V, dt)
    ws = ws if ws is not None else workspace(need, dev, stream)
    o = out or dict(accepted=torch.empty(B, dtype=torch.int32, device=dev),
                    out_tokens=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
                    n_emit=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    rc = _call(dev, lib().spec_verify_greedy, _p(target), target.stride(0), target.stride(1), dt, B, k, V,
                                  _p(draft), _p(draft_len), _p(max_emit), _p(o["accepted"]),
                                  _p(o["out_tokens"]), _p(o["n_emit"]), _p(o["status"]), _p(ws),
                                  ws.numel(), _stream(stream, dev))
    _check(rc, "spec_verify_greedy")
    return o


def spec_verify_sample(target: torch.Tensor, draft_logits: torch.Tensor, draft: torch.Tensor,
                       uniforms: torch.Tensor, temperature: float = 1.0, draft_len=None,
                       max_emit=None, *, probs: bool = True, top_k: int = 0, top_p: float = 1.0, out=None,
                       ws=None, stream=None) -> dict:
    """target [B, k+1, V], draft_logits [B, k, V] (same dtype), draft int32 [B, k],
    uniforms fp32 [B, k+1] -> accepted, out_tokens, n_emit, p_tok, q_tok, resid_mass, status.
    top_k / top_p (0 / 1.0: off) filter p and q alike (spec_verify_sample_topkp)."""
    target = _logits3(target, "target")
    draft_logits = _logits3(draft_logits, "draft_logits")
    dev = target.device
    B, R, V = target.shape
    k = R - 1
    if tuple(draft_logits.shape) != (B, k, V) or draft_logits.dtype != target.dtype:
        raise ValueError("draft_logits must be [B, k, V] with the target's dtype")
    if k > 1 and draft_logits.stride(1) != target.stride(1):
        raise ValueError("target and draft rows must share a row stride")
    draft = _i32(draft, (B, k), "draft", dev)
    uniforms = _f32(uniforms, (B, k + 1), "uniforms", dev)
    draft_len = _i32(draft_len, (B,), "draft_len", dev)
    max_emit = _i32(max_emit, (B,), "max_emit", dev)
    dt = _dtype_code(target)
    need = spec_workspace_size(OP_SAMPLE, B, k, V, dt)
    ws = ws if ws is not None else workspace(need, dev, stream)
    o = out
    if o is None:
        o = dict(accepted=torch.empty(B, dtype=torch.int32, device=dev),
                 out_tokens=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
                 n_emit=torch.empty(B, dtype=torch.int32, device=dev),
                 status=torch.empty(B, dtype=torch.int32, device=dev))
        if probs:
            o.update(p_tok=torch.empty((B, k), dtype=torch.float32, device=dev),
                     q_tok=torch.empty((B, k), dtype=torch.float32, device=dev),
                     resid_mass=torch.empty(B, dtype=torch.float32, device=dev))
    head = (_p(target), target.stride(0), _p(draft_logits), draft_logits.stride(0), target.stride(1), dt, B, k, V,
            float(temperature))
    tail = (_p(draft), _p(draft_len), _p(max_emit), _p(uniforms), _p(o["accepted"]), _p(o["out_tokens"]),
            _p(o["n_emit"]), _p(o.get("p_tok")), _p(o.get("q_tok")), _p(o.get("resid_mass")), _p(o["status"]),
            _p(ws), ws.numel(), _stream(stream, dev))
    if top_k or top_p != 1.0:
        _check(_call(dev, lib().spec_verify_sample_topkp, *head, int(top_k), float(top_p), *tail), "spec_verify_sample_topkp")
    else:
        _check(_call(dev, lib().spec_verify_sample, *head, *tail), "spec_verify_sample")
    return o


def spec_verify_tree(target: torch.Tensor, draft_logits, parents: torch.Tensor, node_tok: torch.Tensor,
                     uniforms: torch.Tensor, temperature: float, max_depth: int, *, flags: int = 0, out=None,
                     stream=None) -> dict:
    """target/draft_logits [B, N, V], parents/node_tok int32 [B, N], uniforms fp32 [B, N+1]
    -> accepted_len, path_nodes, out_tokens, n_emit, status.  temperature <= 0: greedy.
    flags != 0 (TREE_SIBLINGS_WITHOUT_REPLACEMENT) goes through spec_verify_tree_ex."""
    target = _logits3(target, "target")
    dev = target.device
    B, N, V = target.shape
    greedy = not temperature > 0
    if draft_logits is not None:
        draft_logits = _logits3(draft_logits, "draft_logits")
        if tuple(draft_logits.shape) != (B, N, V) or draft_logits.dtype != target.dtype:
            raise ValueError("draft_logits must be [B, N, V] with the target's dtype")
        if N > 1 and draft_logits.stride(1) != target.stride(1):
            raise ValueError("target and draft rows must share a row stride")
    elif not greedy:
        raise ValueError("sampling tree verification needs draft_logits")
    parents = _i32(parents, (B, N), "parents", dev)
    node_tok = _i32(node_tok, (B, N), "node_tok", dev)
    uniforms = _f32(uniforms, (B, N + 1), "uniforms", dev)
    W = max_depth + 1
    o = out or dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                    path_nodes=torch.empty((B, W), dtype=torch.int32, device=dev),
                    out_tokens=torch.empty((B, W), dtype=torch.int32, device=dev),
                    n_emit=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    d_req = draft_logits.stride(0) if draft_logits is not None else 0
    head = (_p(target), target.stride(0), _p(draft_logits), d_req, target.stride(1), _dtype_code(target), B, N,
            V, float(temperature), _p(parents), _p(node_tok), _p(uniforms), int(max_depth))
    tail = (_p(o["accepted_len"]), _p(o["path_nodes"]), _p(o["out_tokens"]), _p(o["n_emit"]), _p(o["status"]),
            None, 0, _stream(stream, dev))
    if flags:
        rc = _call(dev, lib().spec_verify_tree_ex, *head, int(flags), *tail)
        _check(rc, "spec_verify_tree_ex")
    else:
        rc = _call(dev, lib().spec_verify_tree, *head, *tail)
        _check(rc, "spec_verify_tree")
    return o


def spec_sample(logits: torch.Tensor, uniforms: torch.Tensor, temperature: float = 1.0, *, probs: bool = True,
                top_k: int = 0, top_p: float = 1.0, out=None, ws=None, stream=None) -> dict:
    """logits [B, V] (fp32 or bf16, each row contiguous), uniforms fp32 [B]
    -> tokens int32 [B] drawn from softmax(logits / T), probs fp32 [B] (the
    drawn tokens' probabilities), status.  top_k / top_p (0 / 1.0: off):
    draw from the filtered rows (spec_sample_topkp)."""
    if not isinstance(logits, torch.Tensor) or logits.dim() != 2:
        raise ValueError("logits must be a [B, V] tensor")
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    if logits.stride(1) != 1:
        logits = logits.contiguous()
    dev = logits.device
    B, V = logits.shape
    uniforms = _f32(uniforms, (B,), "uniforms", dev)
    dt = _dtype_code(logits)
    need = spec_workspace_size(OP_DRAW, B, 0, V, dt)
    ws = ws if ws is not None else workspace(need, dev, stream)
    o = out or dict(tokens=torch.empty(B, dtype=torch.int32, device=dev),
                    probs=torch.empty(B, dtype=torch.float32, device=dev) if probs else None,
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    tail = (_p(uniforms), _p(o["tokens"]), _p(o.get("probs")), _p(o["status"]), _p(ws), ws.numel(),
            _stream(stream, dev))
    if top_k or top_p != 1.0:
        rc = _call(dev, lib().spec_sample_topkp, _p(logits), logits.stride(0), dt, B, V, float(temperature), int(top_k),
                                     float(top_p), *tail)
        _check(rc, "spec_sample_topkp")
    else:
        _check(_call(dev, lib().spec_sample, _p(logits), logits.stride(0), dt, B, V, float(temperature), *tail), "spec_sample")
    return o


def spec_filter_rows(logits: torch.Tensor, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0, *,
                     out=None, stream=None) -> dict:
    """logits [R, V] (fp32 or bf16, each row contiguous) -> theta fp32 [R]
    (the smallest logit the top-k / top-p filter keeps) and kept int32 [R]."""
    if not isinstance(logits, torch.Tensor) or logits.dim() != 2:
        raise ValueError("logits must be a [R, V] tensor")
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    if logits.stride(1) != 1:
        logits = logits.contiguous()
    dev = logits.device
    R, V = logits.shape
    dt = _dtype_code(logits)
    ws = workspace(spec_workspace_size(OP_FILTER, R, 0, V, dt), dev, stream)
    o = out or dict(theta=torch.empty(R, dtype=torch.float32, device=dev),
                    kept=torch.empty(R, dtype=torch.int32, device=dev))
    _check(_call(dev, lib().spec_filter_rows, _p(logits), logits.stride(0), dt, R, V, float(temperature), int(top_k),
                                  float(top_p), _p(o["theta"]), _p(o.get("kept")), _p(ws), ws.numel(),
                                  _stream(stream, dev)), "spec_filter_rows")
    return o


def spec_tree_rerank(parents: torch.Tensor, conf: torch.Tensor, m: int, max_depth: int = 64, node_tok=None, *,
                     mask: bool = True, out=None, stream=None) -> dict:
    """parents int32 [B, N], conf fp32 [B, N] (node_tok int32 [B, N] or None)
    -> sel_nodes, sel_parents, sel_depth, sel_value, sel_tok (with node_tok),
    mask uint8 [B, m, m] (unless mask=False), n_sel, status."""
    dev = parents.device
    if parents.dim() != 2:
        raise ValueError("parents must be [B, N]")
    B, N = parents.shape
    parents = _i32(parents, (B, N), "parents", dev)
    conf = _f32(conf, (B, N), "conf", dev)
    node_tok = _i32(node_tok, (B, N), "node_tok", dev) if node_tok is not None else None
    i32 = dict(dtype=torch.int32, device=dev)
    o = out or dict(sel_nodes=torch.empty((B, m), **i32), sel_parents=torch.empty((B, m), **i32),
                    sel_depth=torch.empty((B, m), **i32),
                    sel_value=torch.empty((B, m), dtype=torch.float32, device=dev),
                    sel_tok=torch.empty((B, m), **i32) if node_tok is not None else None,
                    mask=torch.empty((B, m, m), dtype=torch.uint8, device=dev) if mask else None,
                    n_sel=torch.empty(B, **i32), status=torch.empty(B, **i32))
    rc = _call(dev, lib().spec_tree_rerank, _p(parents), _p(conf), _p(node_tok), B, N, int(m), int(max_depth),
                                _p(o["sel_nodes"]), _p(o["sel_parents"]), _p(o["sel_depth"]),
                                _p(o.get("sel_value")), _p(o.get("sel_tok")), _p(o.get("mask")),
                                _p(o["n_sel"]), _p(o.get("status")), _stream(stream, dev))
    _check(rc, "spec_tree_rerank")
    return o


def spec_verify_sample_noalloc(target: torch.Tensor, draft_logits: torch.Tensor, draft: torch.Tensor,
                               uniforms: torch.Tensor, temperature: float = 1.0, draft_len=None,
                               max_emit=None, *, out=None, stream=None) -> dict:
    """spec_verify_sample without a workspace, for callers that cannot allocate
    device memory while they run: the library's fixed scratch array is used
    instead (SPEC_NOALLOC_SCRATCH_BYTES; larger problems raise SpecError).
    Outputs are allocated here unless `out` is given."""
    L = lib()
    fn = L.spec_verify_sample_noalloc
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [P, I64, P, I64, I64, I, I, I, I, F, P, P, P, P, P, P, P, P, P, P, P, P]
    target = _logits3(target, "target")
    draft_logits = _logits3(draft_logits, "draft_logits")
    dev = target.device
    B, R, V = target.shape
    k = R - 1
    if tuple(draft_logits.shape) != (B, k, V) or draft_logits.dtype != target.dtype:
        raise ValueError("draft_logits must be [B, k, V] with the target's dtype")
    if k > 1 and draft_logits.stride(1) != target.stride(1):
        raise ValueError("target and draft rows must share a row stride")
    draft = _i32(draft, (B, k), "draft", dev)
    uniforms = _f32(uniforms, (B, k + 1), "uniforms", dev)
    draft_len = _i32(draft_len, (B,), "draft_len", dev)
    max_emit = _i32(max_emit, (B,), "max_emit", dev)
    o = out or dict(accepted=torch.empty(B, dtype=torch.int32, device=dev),
                    out_tokens=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
                    n_emit=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev),
                    p_tok=torch.empty((B, k), dtype=torch.float32, device=dev),
                    q_tok=torch.empty((B, k), dtype=torch.float32, device=dev),
                    resid_mass=torch.empty(B, dtype=torch.float32, device=dev))
    rc = _call(dev, fn, _p(target), target.stride(0), _p(draft_logits), draft_logits.stride(0), target.stride(1),
            _dtype_code(target), B, k, V, float(temperature), _p(draft), _p(draft_len), _p(max_emit),
            _p(uniforms), _p(o["accepted"]), _p(o["out_tokens"]), _p(o["n_emit"]), _p(o.get("p_tok")),
            _p(o.get("q_tok")), _p(o.get("resid_mass")), _p(o["status"]), _stream(stream, dev))
    _check(rc, "spec_verify_sample_noalloc")
    return o


# ------------------------------------------------------- host analysis helpers
# Host-side (no GPU): the choice of the draft length from measured acceptance.

def expected_tokens(alpha: float, k: int) -> float:
    """Expected tokens per round, 1 + alpha + ... + alpha^k."""
    out = ctypes.c_double()
    _check(lib().spec_expected_tokens(float(alpha), int(k), ctypes.byref(out)), "spec_expected_tokens")
    return out.value


def speedup(alpha: float, k: int, draft_cost: float) -> float:
    """Expected tokens per round over the round's cost k c + 1 (in target forwards)."""
    out = ctypes.c_double()
    _check(lib().spec_speedup(float(alpha), int(k), float(draft_cost), ctypes.byref(out)), "spec_speedup")
    return out.value


def best_k(alpha: float, draft_cost: float, k_max: int) -> tuple:
    """(k in [0, k_max] with the largest speedup, that speedup)."""
    k = ctypes.c_int()
    s = ctypes.c_double()
    _check(lib().spec_best_k(float(alpha), float(draft_cost), int(k_max), ctypes.byref(k), ctypes.byref(s)),
           "spec_best_k")
    return k.value, s.value


def alpha_estimate(accepted, draft_len=None, k: int = 0) -> tuple:
    """(alpha, positions tested) from rounds' accepted counts (host arrays or
    tensors, copied to the host) and draft lengths (None: all k)."""
    import numpy as np
    acc = np.ascontiguousarray(torch.as_tensor(accepted).cpu().numpy(), dtype=np.int32).reshape(-1)
    dl = None if draft_len is None else np.ascontiguousarray(torch.as_tensor(draft_len).cpu().numpy(),
                                                             dtype=np.int32).reshape(-1)
    if dl is not None and dl.size != acc.size:
        raise ValueError("draft_len must match accepted")
    a = ctypes.c_double()
    t = ctypes.c_int64()
    _check(lib().spec_alpha_estimate(acc.ctypes.data, None if dl is None else dl.ctypes.data, acc.size, int(k),
                                     ctypes.byref(a), ctypes.byref(t)), "spec_alpha_estimate")
    return a.value, t.value
