"""fp64 CPU oracle for speculative-decoding verification -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never loads it, and it
never loads the product library: the two share nothing but the seeded inputs
from ``speculative_decoding_verification_02_gb300.workloads``.

The arithmetic lives in ``spec_oracle.c`` (plain C, fp64, built here with
gcc); the helpers in ``analysis.py`` are plain Python.  Parity of every
function is pinned by ``tests/test_oracle_*.py`` against values the pages
print, closed forms and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ST_OK, ST_TOKEN_RANGE, ST_BAD_TREE, ST_BAD_LENGTH = 0, 1, 2, 3
VARIANT_LOSSLESS, VARIANT_RESAMPLE_FROM_P, VARIANT_NAIVE_EQUAL = 0, 1, 2
TREE_VARIANT_NO_RESIDUAL_UPDATE = 1   # planted mistake
TREE_VARIANT_WITHOUT_REPLACEMENT = 2  # siblings drawn from q without replacement


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_softmax.argtypes = [P, I, I, D, P]
        lib.orc_argmax.argtypes = [P, I, I]
        lib.orc_inverse_cdf.argtypes = [P, I, D]
        lib.orc_residual.argtypes = [P, P, I, P]
        lib.orc_residual.restype = D
        lib.orc_ngram_draft.argtypes = [P, P, I, I, I, I, P, P, P]
        lib.orc_verify_greedy.argtypes = [P, I, I, I, I, I64, I64, P, P, P, P, P, P, P]
        lib.orc_verify_sample.argtypes = [P, I64, P, I64, I64, I, I, I, I, D, I, D, P, P, P, P,
                                          P, P, P, P, P, P, P, I, I, P, P]
        lib.orc_filter_row.argtypes = [P, I, I, D, I, D, P, P, P]
        lib.orc_verify_tree.argtypes = [P, I64, P, I64, I64, I, I, I, I, D, P, P, P, I,
                                        P, P, P, P, P, I, I, P]
        lib.orc_tree_rerank.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, P, P]
        lib.orc_max_threads.argtypes = []
        _lib = lib
        return lib


# ----------------------------------------------------------------- helpers

def _ptr(a):
    return None if a is None else a.ctypes.data


def _logits(x):
    """(array, dtype code, element strides).  fp32 -> 0, bf16 bits (uint16) -> 1."""
    x = np.asarray(x)
    if x.dtype == np.float32:
        code = 0
    elif x.dtype == np.uint16:
        code = 1
    else:
        raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {x.dtype}")
    if x.strides[-1] != x.itemsize and x.size > 0 and x.shape[-1] > 1:
        raise ValueError("logit rows must be contiguous along V")
    return x, code


def _strides(x):
    """Element strides of a [B, R, V] logits view (0 allowed for broadcasts)."""
    return x.strides[0] // x.itemsize, x.strides[1] // x.itemsize


def _i32(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.int32)
    if shape is not None and a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def max_threads() -> int:
    return int(_load().orc_max_threads())


# ------------------------------------------------------------ distributions

def softmax(row, T: float = 1.0) -> np.ndarray:
    """p = softmax(row / T) in fp64, from fp32 or bf16-bit logits."""
    row, code = _logits(np.ascontiguousarray(row))
    p = np.empty(row.shape[-1], dtype=np.float64)
    _check(_load().orc_softmax(_ptr(row), code, row.shape[-1], float(T), _ptr(p)), "softmax")
    return p


def argmax(row) -> int:
    """Index of the largest logit, ties to the lowest index."""
    row, code = _logits(np.ascontiguousarray(row))
    r = _load().orc_argmax(_ptr(row), code, row.shape[-1])
    if r < 0:
        raise ValueError("argmax failed")
    return int(r)


def inverse_cdf(d, u: float) -> int:
    """Smallest v with d[0] + ... + d[v] > u (d normalised, fp64)."""
    d = np.ascontiguousarray(d, dtype=np.float64)
    return int(_load().orc_inverse_cdf(_ptr(d), d.size, float(u)))


def residual(p, q):
    """(norm(max(0, p - q)), sum max(0, p - q)) in fp64."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    r = np.empty_like(p)
    R = _load().orc_residual(_ptr(p), _ptr(q), p.size, _ptr(r))
    return r, float(R)


# ------------------------------------------------------------------ drafter

def ngram_draft(history, hist_len, window: int, k: int):
    """Returns (draft [B,k] int32 padded -1, draft_len [B], status [B])."""
    history = np.ascontiguousarray(history, dtype=np.int32)
    B, H = history.shape
    hist_len = _i32(hist_len, (B,))
    draft = np.empty((B, k), dtype=np.int32)
    dlen = np.empty(B, dtype=np.int32)
    status = np.empty(B, dtype=np.int32)
    _check(_load().orc_ngram_draft(_ptr(history), _ptr(hist_len), B, H, int(window), int(k),
                                   _ptr(draft), _ptr(dlen), _ptr(status)), "ngram_draft")
    return draft, dlen, status


# ---------------------------------------------------------------- verifiers

def verify_greedy(target, draft, draft_len=None, max_emit=None):
    """Greedy chain verification.  target: [B, k+1, V] logits (fp32 or bf16 bits)."""
    target, code = _logits(target)
    B, R, V = target.shape
    k = R - 1
    draft = _i32(draft, (B, k))
    t_req, row = _strides(target)
    out = dict(accepted=np.empty(B, np.int32), out_tokens=np.empty((B, k + 1), np.int32),
               n_emit=np.empty(B, np.int32), status=np.empty(B, np.int32))
    _check(_load().orc_verify_greedy(_ptr(target), code, B, k, V, t_req, row, _ptr(draft),
                                     _ptr(_i32(draft_len, (B,))), _ptr(_i32(max_emit, (B,))),
                                     _ptr(out["accepted"]), _ptr(out["out_tokens"]),
                                     _ptr(out["n_emit"]), _ptr(out["status"])), "verify_greedy")
    return out


def verify_sample(target, draft_logits, draft, uniforms, T: float = 1.0, draft_len=None,
                  max_emit=None, variant: int = VARIANT_LOSSLESS, threads: int = 1, top_k: int = 0,
                  top_p: float = 1.0, top_p_rows=None):
    """Sampling chain verification.

    target: [B, k+1, V], draft_logits: [B, k, V] (fp32 or bf16 bits; request
    strides may be 0 to broadcast one problem), draft: [B, k] int32,
    uniforms: [B, k+1] float32.  top_k / top_p filter p and q alike before
    verification (0 / 1.0: off; see filter_row).  top_p_rows: optional
    [B, 2k+1] float64, one top_p per row (target rows 0..k, then draft rows
    0..k-1) in place of top_p.
    """
    target, code = _logits(target)
    draft_logits, code_d = _logits(draft_logits)
    if code_d != code:
        raise TypeError("target and draft logits must share a dtype")
    B, R, V = target.shape
    k = R - 1
    if draft_logits.shape != (B, k, V):
        raise ValueError(f"draft logits must be {(B, k, V)}, got {draft_logits.shape}")
    t_req, row = _strides(target)
    d_req, d_row = _strides(draft_logits)
    if k > 1 and d_row != row:
        raise ValueError("target and draft rows must share a row stride")
    if k <= 1:
        d_row = row
    draft = _i32(draft, (B, k))
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    if uniforms.shape != (B, k + 1):
        raise ValueError(f"uniforms must be {(B, k + 1)}")
    out = dict(accepted=np.empty(B, np.int32), out_tokens=np.empty((B, k + 1), np.int32),
               n_emit=np.empty(B, np.int32), p_tok=np.empty((B, k)), q_tok=np.empty((B, k)),
               resid_mass=np.empty(B), status=np.empty(B, np.int32))
    degen = np.zeros(1, dtype=np.int64)
    if top_p_rows is not None:
        top_p_rows = np.ascontiguousarray(top_p_rows, dtype=np.float64)
        if top_p_rows.shape != (B, 2 * k + 1) or not np.all((top_p_rows > 0) & (top_p_rows <= 1)):
            raise ValueError(f"top_p_rows must be {(B, 2 * k + 1)} values in (0, 1]")
    _check(_load().orc_verify_sample(
        _ptr(target), t_req, _ptr(draft_logits), d_req, row, code, B, k, V, float(T), int(top_k), float(top_p),
        _ptr(draft), _ptr(_i32(draft_len, (B,))), _ptr(_i32(max_emit, (B,))), _ptr(uniforms),
        _ptr(out["accepted"]), _ptr(out["out_tokens"]), _ptr(out["n_emit"]),
        _ptr(out["p_tok"]), _ptr(out["q_tok"]), _ptr(out["resid_mass"]), _ptr(out["status"]),
        int(variant), int(threads), _ptr(degen), _ptr(top_p_rows)), "verify_sample")
    out["degenerate"] = int(degen[0])
    return out


def filter_row(row, T: float = 1.0, top_k: int = 0, top_p: float = 1.0):
    """Top-k then top-p filtering of one logit row (fp32 or bf16 bits), in
    fp64: (p' [V] float64, theta = the smallest kept logit, kept count).
    top_k keeps every logit >= the top_k-th largest; top_p then keeps, over
    those renormalised, the smallest descending prefix whose mass reaches
    top_p, ties at its last logit included."""
    row, code = _logits(row)
    row = np.ascontiguousarray(row).reshape(-1)
    V = row.size
    p = np.empty(V)
    theta = ctypes.c_double()
    kept = ctypes.c_int32()
    _check(_load().orc_filter_row(_ptr(row), code, V, float(T), int(top_k), float(top_p), _ptr(p),
                                  ctypes.byref(theta), ctypes.byref(kept)), "filter_row")
    return p, theta.value, kept.value


def verify_tree(target, draft_logits, parents, node_tok, uniforms, T: float, max_depth: int,
                variant: int = VARIANT_LOSSLESS, threads: int = 1):
    """Tree verification.  target/draft_logits: [B, N, V]; parents, node_tok: [B, N];
    uniforms: [B, N+1].  T <= 0 walks the tree greedily (draft_logits may be None)."""
    target, code = _logits(target)
    B, N, V = target.shape
    t_req, row = _strides(target)
    if draft_logits is not None:
        draft_logits, code_d = _logits(draft_logits)
        if code_d != code or draft_logits.shape != (B, N, V):
            raise ValueError("draft logits must match the target's dtype and shape")
        d_req, d_row = _strides(draft_logits)
        if N > 1 and d_row != row:
            raise ValueError("target and draft rows must share a row stride")
    else:
        d_req = 0
    parents = _i32(parents, (B, N))
    node_tok = _i32(node_tok, (B, N))
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    if uniforms.shape != (B, N + 1):
        raise ValueError(f"uniforms must be {(B, N + 1)}")
    W = max_depth + 1
    out = dict(accepted_len=np.empty(B, np.int32), path_nodes=np.empty((B, W), np.int32),
               out_tokens=np.empty((B, W), np.int32), n_emit=np.empty(B, np.int32),
               status=np.empty(B, np.int32))
    degen = np.zeros(1, dtype=np.int64)
    _check(_load().orc_verify_tree(
        _ptr(target), t_req, _ptr(draft_logits), d_req, row, code, B, N, V, float(T),
        _ptr(parents), _ptr(node_tok), _ptr(uniforms), int(max_depth),
        _ptr(out["accepted_len"]), _ptr(out["path_nodes"]), _ptr(out["out_tokens"]),
        _ptr(out["n_emit"]), _ptr(out["status"]), int(variant), int(threads), _ptr(degen)),
        "verify_tree")
    out["degenerate"] = int(degen[0])
    return out


def tree_rerank(parents, conf, m: int, max_depth: int = 64, node_tok=None, mask: bool = True):
    """EAGLE-2 post-processing of candidate trees.  parents: [B, N] int32
    (parents[0] = -1, parents[i] < i); conf: [B, N] fp32 draft confidences in
    [0, 1] (conf[:, 0] unused); node_tok: [B, N] or None.  Returns the kept
    nodes in flattened order with their flattened parents, depths, values,
    tokens, the [B, m, m] attention mask, n_sel and status."""
    parents = _i32(parents, None)
    B, N = parents.shape
    conf = np.ascontiguousarray(conf, dtype=np.float32)
    if conf.shape != (B, N):
        raise ValueError(f"conf must be {(B, N)}")
    if node_tok is not None:
        node_tok = _i32(node_tok, (B, N))
    out = dict(sel_nodes=np.empty((B, m), np.int32), sel_parents=np.empty((B, m), np.int32),
               sel_depth=np.empty((B, m), np.int32), sel_value=np.empty((B, m), np.float32),
               sel_tok=np.empty((B, m), np.int32) if node_tok is not None else None,
               mask=np.empty((B, m, m), np.uint8) if mask else None,
               n_sel=np.empty(B, np.int32), status=np.empty(B, np.int32))
    _check(_load().orc_tree_rerank(
        _ptr(parents), _ptr(conf), _ptr(node_tok), B, N, int(m), int(max_depth), _ptr(out["sel_nodes"]),
        _ptr(out["sel_parents"]), _ptr(out["sel_depth"]), _ptr(out["sel_value"]), _ptr(out["sel_tok"]),
        _ptr(out["mask"]), _ptr(out["n_sel"]), _ptr(out["status"])), "tree_rerank")
    return out
