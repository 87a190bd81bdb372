"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before launching."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verification_02_gb300 import api, build
    build.build()
    return api.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = _declared()
    for n in ("spec_ngram_draft", "spec_verify_greedy", "spec_verify_sample", "spec_verify_tree"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_header_constants_match_binding():
    from speculative_decoding_verification_02_gb300 import api
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define (SPEC_\w+) \(?(-?\d+)\)?", text))
    assert int(consts["SPEC_OK"]) == api.SPEC_OK and int(consts["SPEC_EINVAL"]) == api.SPEC_EINVAL
    assert int(consts["SPEC_EDTYPE"]) == api.SPEC_EDTYPE
    assert int(consts["SPEC_EWORKSPACE"]) == api.SPEC_EWORKSPACE
    assert int(consts["SPEC_ECUDA"]) == api.SPEC_ECUDA
    assert int(consts["SPEC_DTYPE_BF16"]) == api.DTYPE_BF16
    assert int(consts["SPEC_STATUS_BAD_TREE"]) == api.STATUS_BAD_TREE
    assert int(consts["SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT"]) == api.TREE_SIBLINGS_WITHOUT_REPLACEMENT
    assert (int(consts["SPEC_CHAIN_AUTO"]), int(consts["SPEC_CHAIN_TWO_PASS"]), int(consts["SPEC_CHAIN_FUSED"]),
            int(consts["SPEC_CHAIN_CHUNKED"])) == (api.CHAIN_AUTO, api.CHAIN_TWO_PASS, api.CHAIN_FUSED,
                                                   api.CHAIN_CHUNKED)


def test_chain_path_switch(L):
    L.spec_set_chain_path.argtypes = [ctypes.c_int]
    for bad in (-1, 4, 5, 1 << 20):
        assert L.spec_set_chain_path(bad) == -1          # SPEC_EINVAL
    for good in (3, 2, 1, 0):
        assert L.spec_set_chain_path(good) == 0


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails validation


def _sample(L, **kw):
    a = dict(target=FAKE, t_req=5 * 1024, draft=FAKE, d_req=4 * 1024, row=1024, dtype=1, B=2, k=4,
             V=1024, T=1.0, x=FAKE, dlen=None, maxe=None, u=FAKE, acc=FAKE, out=FAKE, ne=FAKE,
             pt=None, qt=None, rm=None, st=FAKE, ws=ctypes.c_void_p(0x100000), wsb=1 << 30, stream=None)
    a.update(kw)
    return L.spec_verify_sample(*a.values())


def test_sample_argument_checks(L):
    from speculative_decoding_verification_02_gb300 import api
    n0 = L.spec_launch_count()
    assert _sample(L, dtype=7) == api.SPEC_EDTYPE
    assert _sample(L, B=-1) == api.SPEC_EINVAL
    assert _sample(L, k=65) == api.SPEC_EINVAL
    assert _sample(L, V=0) == api.SPEC_EINVAL
    assert _sample(L, T=0.0) == api.SPEC_EINVAL
    assert _sample(L, T=float("inf")) == api.SPEC_EINVAL
    assert _sample(L, T=float("nan")) == api.SPEC_EINVAL
    assert _sample(L, target=None) == api.SPEC_EINVAL
    assert _sample(L, u=None) == api.SPEC_EINVAL
    assert _sample(L, row=-1) == api.SPEC_EINVAL
    assert _sample(L, ws=None) == api.SPEC_EWORKSPACE
    assert _sample(L, ws=ctypes.c_void_p(0x100010)) == api.SPEC_EWORKSPACE       # misaligned
    assert _sample(L, wsb=16) == api.SPEC_EWORKSPACE                             # too small
    assert _sample(L, B=0) == api.SPEC_OK                                        # nothing to do
    assert L.spec_launch_count() == n0                                           # nothing launched


def test_greedy_tree_ngram_argument_checks(L):
    from speculative_decoding_verification_02_gb300 import api
    n0 = L.spec_launch_count()
    ws = ctypes.c_void_p(0x100000)
    assert L.spec_verify_greedy(FAKE, 0, 0, 0, 1, 2, 0, FAKE, None, None, FAKE, FAKE, FAKE, None, ws,
                                1 << 20, None) == api.SPEC_EINVAL
    assert L.spec_verify_greedy(FAKE, 0, 0, 3, 1, 2, 10, FAKE, None, None, FAKE, FAKE, FAKE, None, ws,
                                1 << 20, None) == api.SPEC_EDTYPE
    assert L.spec_verify_greedy(None, 0, 0, 0, 1, 2, 10, FAKE, None, None, FAKE, FAKE, FAKE, None, ws,
                                1 << 20, None) == api.SPEC_EINVAL
    tree = lambda **kw: L.spec_verify_tree(*dict(dict(t=FAKE, tr=0, d=FAKE, dr=0, r=64, dt=0, B=1, N=4, V=64,
                                                      T=1.0, par=FAKE, tok=FAKE, u=FAKE, md=3, al=FAKE,
                                                      pn=FAKE, ot=FAKE, ne=FAKE, st=FAKE, ws=None, wb=0,
                                                      s=None), **kw).values())
    assert tree(N=0) == api.SPEC_EINVAL
    assert tree(N=4097) == api.SPEC_EINVAL
    assert tree(md=65) == api.SPEC_EINVAL
    assert tree(md=-1) == api.SPEC_EINVAL
    assert tree(T=float("nan")) == api.SPEC_EINVAL
    assert tree(d=None) == api.SPEC_EINVAL            # sampling needs draft logits
    assert tree(par=None) == api.SPEC_EINVAL
    assert tree(dt=9) == api.SPEC_EDTYPE
    assert tree(B=0) == api.SPEC_OK
    tree_ex = lambda **kw: L.spec_verify_tree_ex(*dict(dict(t=FAKE, tr=0, d=FAKE, dr=0, r=64, dt=0, B=1, N=4, V=64,
                                                            T=1.0, par=FAKE, tok=FAKE, u=FAKE, md=3, fl=1, al=FAKE,
                                                            pn=FAKE, ot=FAKE, ne=FAKE, st=FAKE, ws=None, wb=0,
                                                            s=None), **kw).values())
    assert tree_ex(fl=2) == api.SPEC_EINVAL            # unknown flag bit
    assert tree_ex(fl=-1) == api.SPEC_EINVAL
    assert tree_ex(N=0) == api.SPEC_EINVAL
    assert tree_ex(d=None) == api.SPEC_EINVAL
    assert tree_ex(B=0) == api.SPEC_OK
    assert tree_ex(B=0, fl=0) == api.SPEC_OK
    ng = lambda **kw: L.spec_ngram_draft(*dict(dict(h=FAKE, hl=FAKE, B=2, hs=16, w=3, k=4, d=FAKE, dl=FAKE,
                                                    st=None, s=None), **kw).values())
    assert ng(w=0) == api.SPEC_EINVAL
    assert ng(w=65) == api.SPEC_EINVAL
    assert ng(k=65) == api.SPEC_EINVAL
    assert ng(hl=None) == api.SPEC_EINVAL
    assert ng(B=0) == api.SPEC_OK
    assert L.spec_launch_count() == n0


def test_workspace_sizes(L):
    from speculative_decoding_verification_02_gb300 import api
    s1 = L.spec_workspace_size(api.OP_SAMPLE, 1, 4, 248320, 1)
    s64 = L.spec_workspace_size(api.OP_SAMPLE, 64, 8, 128256, 1)
    assert 0 < s1 < s64 and s1 % 256 == 0 and s64 % 256 == 0
    assert L.spec_workspace_size(api.OP_GREEDY, 64, 4, 32000, 0) > 0
    assert L.spec_workspace_size(api.OP_TREE, 16, 60, 128256, 1) == 0
    assert L.spec_workspace_size(api.OP_SAMPLE, -1, 4, 10, 1) == 0
    assert L.spec_workspace_size(api.OP_SAMPLE, 1, 4, 10, 5) == 0
    # the streaming pass keeps 16 bytes per (row, 16 KB chunk): small next to the logits
    assert s64 < 0.01 * 64 * 17 * 128256 * 2
    # a 16-byte partial per (row, streaming chunk) at least
    assert s1 >= 9 * 16 and L.spec_workspace_size(api.OP_GREEDY, 4, 4, 2048, 0) >= 4 * 5 * 16


def test_status_strings(L):
    assert L.spec_status_string(0) == b"ok"
    assert b"workspace" in L.spec_status_string(-3)
    assert b"tree" in L.spec_status_string(102)
    assert L.spec_status_string(104) == b"unknown code"
    assert L.spec_last_error() is not None


def test_tree_rerank_argument_checks(L):
    P_ = ctypes.c_void_p
    L.spec_tree_rerank.argtypes = [P_, P_, P_, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int] + [P_] * 9
    def call(parents=FAKE, conf=FAKE, tok=None, B=2, N=8, m=4, depth=8, nodes=FAKE, par=FAKE, dep=FAKE,
             val=None, stok=None, mask=None, nsel=FAKE, st=None):
        return L.spec_tree_rerank(parents, conf, tok, B, N, m, depth, nodes, par, dep, val, stok, mask, nsel, st,
                                  None)
    assert call(N=0) == -1 and call(N=4097) == -1
    assert call(m=0) == -1 and call(m=4097) == -1
    assert call(depth=-1) == -1 and call(depth=65) == -1
    assert call(B=-1) == -1
    assert call(B=0) == 0                       # nothing to do, nothing launched
    for kw in ("parents", "conf", "nodes", "par", "dep", "nsel"):
        assert call(**{kw: None}) == -1, kw
    assert call(stok=FAKE) == -1                # tokens out without tokens in


def test_sample_draw_argument_checks(L):
    P_ = ctypes.c_void_p
    L.spec_sample.argtypes = [P_, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                              P_, P_, P_, P_, P_, ctypes.c_size_t, P_]
    L.spec_workspace_size.restype = ctypes.c_size_t
    need = L.spec_workspace_size(4, 8, 0, 1000, 1)
    assert need > 0 and need >= L.spec_workspace_size(2, 8, 0, 1000, 1)
    ws = ctypes.c_void_p(0x100000)
    def call(logits=FAKE, stride=1000, dtype=1, B=8, V=1000, T=1.0, u=FAKE, tok=FAKE, w=ws, wsb=need):
        return L.spec_sample(logits, stride, dtype, B, V, T, u, tok, None, None, w, wsb, None)
    assert call(dtype=7) == -2
    assert call(B=-1) == -1 and call(V=0) == -1 and call(stride=-1) == -1
    assert call(T=0.0) == -1 and call(T=float("inf")) == -1 and call(T=float("nan")) == -1
    assert call(logits=None) == -1 and call(u=None) == -1 and call(tok=None) == -1
    assert call(wsb=need - 1) == -3 and call(w=None) == -3 and call(w=ctypes.c_void_p(0x100010)) == -3
    assert call(B=0) == 0


def test_topkp_argument_checks(L):
    """spec_verify_sample_topkp, spec_sample_topkp and spec_filter_rows reject
    bad filters and arguments on the host, launching nothing."""
    P_, I, I64, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.spec_verify_sample_topkp.argtypes = [P_, I64, P_, I64, I64, I, I, I, I, F, I, F] + [P_] * 12 + [Z, P_]
    L.spec_sample_topkp.argtypes = [P_, I64, I, I, I, F, I, F, P_, P_, P_, P_, P_, Z, P_]
    L.spec_filter_rows.argtypes = [P_, I64, I, I, I, F, I, F, P_, P_, P_, Z, P_]
    L.spec_workspace_size.restype = ctypes.c_size_t
    ws = ctypes.c_void_p(0x100000)
    n0 = L.spec_launch_count()

    def verify(top_k=50, top_p=0.9, dtype=1, B=2, k=4, V=1024, T=1.0):
        return L.spec_verify_sample_topkp(FAKE, 5 * 1024, FAKE, 4 * 1024, 1024, dtype, B, k, V, T, top_k, top_p,
                                          FAKE, None, None, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, ws,
                                          1 << 30, None)
    for bad in (dict(top_k=-1), dict(top_p=0.0), dict(top_p=-0.5), dict(top_p=1.5), dict(top_p=float("nan")),
                dict(T=0.0), dict(k=65), dict(V=0)):
        assert verify(**bad) == -1, bad
    assert verify(dtype=7) == -2
    assert verify(B=0) == 0

    def draw(top_k=50, top_p=0.9, B=8, V=1000, T=1.0, w=ws, wsb=None):
        wsb = L.spec_workspace_size(4, B, 0, V, 1) if wsb is None else wsb
        return L.spec_sample_topkp(FAKE, V, 1, B, V, T, top_k, top_p, FAKE, FAKE, None, None, w, wsb, None)
    assert draw(top_k=-3) == -1 and draw(top_p=2.0) == -1 and draw(T=float("inf")) == -1
    assert draw(wsb=16) == -3 and draw(w=None) == -3 and draw(w=ctypes.c_void_p(0x100010)) == -3
    assert draw(B=0) == 0

    def rows(top_k=50, top_p=0.9, R=4, V=1000, T=1.0, theta=FAKE, w=ws, wsb=None, dtype=1):
        wsb = L.spec_workspace_size(5, R, 0, V, dtype) if wsb is None else wsb
        return L.spec_filter_rows(FAKE, V, dtype, R, V, T, top_k, top_p, theta, None, w, wsb, None)
    assert rows(top_k=-1) == -1 and rows(top_p=0.0) == -1 and rows(R=-1) == -1 and rows(V=0) == -1
    assert rows(theta=None) == -1 and rows(dtype=3) == -2
    assert rows(wsb=8) == -3 and rows(w=None) == -3
    assert rows(V=786_433) == -1                       # more than 16 slices of 96 KB of bf16
    assert rows(V=393_217, dtype=0) == -1              # the same for fp32
    assert rows(R=0) == 0
    assert L.spec_launch_count() == n0
