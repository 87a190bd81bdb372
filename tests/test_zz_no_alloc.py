"""spec_verify_sample_noalloc: the entry point for callers that cannot
allocate device memory (a serving loop with a fixed memory budget, code that
must not stall on cudaMalloc) must give the same results as
spec_verify_sample with a caller-supplied workspace.

The library's fixed scratch array is shared by every call and keeps the
previous call's contents, so two different calls run back to back through
the C ABI and each is compared with the workspace entry point.  A problem
too large for the array must be refused with a clear message.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import TOL, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    lib = api.lib()
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.spec_verify_sample_noalloc.argtypes = [P, I64, P, I64, I64, I, I, I, I, F, P, P, P, P, P, P, P, P, P,
                                               P, P, P]
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc_call(L, prob):
    """Outputs of one spec_verify_sample_noalloc call made through ctypes."""
    T, D = to_dev(prob["target"]), to_dev(prob["draft_logits"])
    X, U = to_dev(prob["draft"]), to_dev(prob["uniforms"])
    B, R, V = T.shape
    k = R - 1
    out = dict(accepted=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               out_tokens=torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda"),
               n_emit=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               status=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               p_tok=torch.full((B, k), -7.0, device="cuda"), q_tok=torch.full((B, k), -7.0, device="cuda"),
               resid_mass=torch.full((B,), -7.0, device="cuda"))
    dt = api.DTYPE_BF16 if T.dtype == torch.bfloat16 else api.DTYPE_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.spec_verify_sample_noalloc(_ptr(T), T.stride(0), _ptr(D), D.stride(0), T.stride(1), dt, B, k, V,
                                      float(prob["T"]), _ptr(X), None, None, _ptr(U), _ptr(out["accepted"]),
                                      _ptr(out["out_tokens"]), _ptr(out["n_emit"]), _ptr(out["p_tok"]),
                                      _ptr(out["q_tok"]), _ptr(out["resid_mass"]), _ptr(out["status"]), stream)
    assert rc == api.SPEC_OK, L.spec_last_error()
    torch.cuda.synchronize()
    return host(out)


def _workspace_call(prob):
    o = api.spec_verify_sample(to_dev(prob["target"]), to_dev(prob["draft_logits"]), to_dev(prob["draft"]),
                               to_dev(prob["uniforms"]), prob["T"])
    torch.cuda.synchronize()
    return host(o)


def _same(a, b):
    for key in ("accepted", "out_tokens", "n_emit", "status"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    for key in ("p_tok", "q_tok", "resid_mass"):
        assert np.max(np.abs(a[key] - b[key])) <= TOL, key


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(L):
    first = workloads.chain_problem(301, 16, 4, 30000, "bf16", 1.0, target_std=2.0, noise_std=1.0)
    second = workloads.chain_problem(302, 6, 7, 5001, "fp32", 0.8, target_std=1.5, noise_std=0.5)
    for prob in (first, second):                 # two calls in a row on the shared array
        got = _noalloc_call(L, prob)
        _same(got, _workspace_call(prob))
        assert np.all(got["status"] == 0) and np.all(got["n_emit"] >= 1)


def test_noalloc_refuses_problems_beyond_its_scratch(L):
    # B=4096, k=64, V=2048 fp32 needs several MiB of per-chunk statistics
    need = L.spec_workspace_size(api.OP_SAMPLE, 4096, 64, 2048, api.DTYPE_F32)
    assert need > 4 << 20
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the call is refused first
    rc = L.spec_verify_sample_noalloc(fake, 65 * 2048, fake, 64 * 2048, 2048, api.DTYPE_F32, 4096, 64, 2048,
                                      1.0, fake, None, None, fake, fake, fake, fake, None, None, None, None, None)
    assert rc == api.SPEC_EWORKSPACE
    assert b"needs" in L.spec_last_error() and b"scratch" in L.spec_last_error()


def test_noalloc_python_binding_matches_workspace_binding(L):
    """The Python wrapper api.spec_verify_sample_noalloc (argument checks,
    strides, draft_len / max_emit, current device) against api.spec_verify_sample,
    and its refusal of an oversized problem with the library's message."""
    prob = workloads.chain_problem(303, 12, 5, 20000, "bf16", 0.9, target_std=2.0, noise_std=0.7)
    rng = np.random.default_rng(303)
    dl = to_dev(rng.integers(0, 6, 12).astype(np.int32))
    me = to_dev(rng.integers(1, 7, 12).astype(np.int32))
    args = (to_dev(prob["target"]), to_dev(prob["draft_logits"]), to_dev(prob["draft"]), to_dev(prob["uniforms"]),
            prob["T"], dl, me)
    for _ in range(2):
        got = host(api.spec_verify_sample_noalloc(*args))
        torch.cuda.synchronize()
        _same(got, host(api.spec_verify_sample(*args)))
    # B=4096, k=64: 4096 x 129 row partials of 16 bytes, more than the 4 MiB array
    big = torch.zeros((4096, 65, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(api.SpecError, match="needs .* bytes of scratch"):
        api.spec_verify_sample_noalloc(big, big[:, :64], torch.zeros((4096, 64), dtype=torch.int32, device="cuda"),
                                       torch.zeros((4096, 65), dtype=torch.float32, device="cuda"), 1.0)
