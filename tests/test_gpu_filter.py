"""GPU parity of top-k / top-p filtering and filtered verification against
the oracle.

- spec_filter_rows: the threshold and the kept count are the oracle's,
  exactly for top-k; for top-p the cut may sit one value group off only where
  the oracle's cumulative mass at that cut is within 1e-6 of top_p (counted).
- spec_verify_sample_topkp: every request's outputs under the chain decision
  rule of tests/parity.py against the oracle's filtered verification.  Where
  the GPU's filter cut of a row differs from the oracle's (only allowed where
  the cut's fp64 mass is within 1e-6 of top_p; counted), the oracle filters
  that row with the top_p that gives the GPU's cut, so no request is left out.
  On the headline shape, on both accept kernels (cluster, chunked, each
  forced in turn),
  bf16 ties at the top-k cut, masked logits, drafts outside the filtered q,
  lengths, caps and bad tokens; both filters off reproduce spec_verify_sample
  bit for bit.
- spec_sample_topkp: tokens and q'(x) against the oracle, and 200,000 draws
  from one row follow the filtered distribution.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import TOL, _near_draw, check_chain_sample, host, poison_like, to_dev

pytestmark = pytest.mark.gpu
NEAR = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _cut_ok(row, T, top_k, top_p, theta_g):
    """True when the GPU's kept set {x >= theta_g} is the oracle's, or a top-p
    cut the oracle's fp64 masses put within NEAR of top_p."""
    x = workloads.logits_as_f64(row).reshape(-1)
    _, theta_o, _ = oracle.filter_row(row, T, top_k, top_p)
    if theta_g == theta_o:
        return True, False
    if top_p >= 1.0:
        return False, False
    z = x / T
    p = np.exp(z - z.max())
    vals = np.unique(x)[::-1]
    if 0 < top_k < x.size:
        tk = np.sort(x)[::-1][top_k - 1]
        vals = vals[vals >= tk]
        keep = x >= tk
    else:
        keep = np.ones(x.size, bool)
    SK = p[keep].sum()
    cum = np.array([p[x >= v].sum() for v in vals]) / SK
    i_o = int(np.flatnonzero(vals == theta_o)[0])
    i_g = np.flatnonzero(vals == theta_g)
    if i_g.size == 0:
        return False, False
    i_g = int(i_g[0])
    lo = min(i_o, i_g)
    return abs(i_o - i_g) == 1 and abs(cum[lo] - top_p) < NEAR, True


@pytest.mark.parametrize("seed,R,V,dtype,T,top_k,top_p", [
    (1, 9, 248_320, "bf16", 1.0, 50, 1.0), (2, 9, 248_320, "bf16", 1.0, 0, 0.9),
    (3, 9, 248_320, "bf16", 0.7, 40, 0.8), (4, 16, 32_000, "fp32", 1.0, 100, 0.95),
    (5, 32, 3001, "fp32", 1.3, 7, 1.0), (6, 32, 3001, "bf16", 1.0, 0, 0.5),
    (7, 8, 128_256, "bf16", 1.0, 1, 1.0), (8, 12, 9, "fp32", 1.0, 3, 0.6),
    (9, 4, 5000, "fp32", 1.0, 0, 1.0), (10, 6, 393_216, "fp32", 1.0, 20, 0.9)])
def test_filter_rows_match_oracle(seed, R, V, dtype, T, top_k, top_p):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((R, V)) * 3).astype(np.float32)
    for r in range(R):
        x[r, rng.choice(V, min(5, V), replace=False)] += 8.0
    rows = workloads.bf16_bits(x) if dtype == "bf16" else x
    g = host(api.spec_filter_rows(to_dev(rows), T, top_k, top_p))
    near = 0
    for r in range(R):
        pf, theta_o, kept_o = oracle.filter_row(rows[r], T, top_k, top_p)
        ok, was_near = _cut_ok(rows[r], T, top_k, top_p, float(g["theta"][r]))
        assert ok, (r, g["theta"][r], theta_o, g["kept"][r], kept_o)
        if was_near:
            near += 1
        else:
            assert g["kept"][r] == kept_o, (r, g["kept"][r], kept_o)
    assert near <= R // 4
    print("near-cut rows", near)


def test_filter_rows_ties_and_masks():
    """bf16 rows with the maximum and the cut value repeated, -inf logits,
    an all-equal row, and -0 next to +0."""
    rng = np.random.default_rng(21)
    V = 70_000
    x = rng.integers(-4, 4, (6, V)).astype(np.float32)
    x[1, rng.random(V) < 0.5] = -np.inf
    x[2] = 1.5
    x[3, :10] = 0.0
    x[3, 10:20] = -0.0
    x[3, 20:] = -5.0
    rows = workloads.bf16_bits(x)
    for top_k, top_p in [(1, 1.0), (100, 1.0), (25_000, 1.0), (15, 1.0), (0, 0.3), (0, 0.99), (5000, 0.7)]:
        g = host(api.spec_filter_rows(to_dev(rows), 1.0, top_k, top_p))
        for r in range(6):
            _, theta_o, kept_o = oracle.filter_row(rows[r], 1.0, top_k, top_p)
            ok, was_near = _cut_ok(rows[r], 1.0, top_k, top_p, float(g["theta"][r]))
            assert ok and (was_near or g["kept"][r] == kept_o), (top_k, top_p, r, g["theta"][r], theta_o,
                                                                   g["kept"][r], kept_o)


def _filtered_chain(seed, B, k, V, dtype, T, top_k, top_p, draft_from_filtered=True):
    prob = workloads.chain_problem(seed, B, k, V, dtype, T, target_std=1.5,
                                   noise_std=np.linspace(0.3, 1.5, B).astype(np.float32))
    rng = np.random.default_rng(seed + 1)
    if draft_from_filtered and k:
        for b in range(B):
            for i in range(k):
                qf = oracle.filter_row(prob["draft_logits"][b, i], T, top_k, top_p)[0]
                prob["draft"][b, i] = rng.choice(V, p=qf / qf.sum())
    return prob


def _gpu_cut_top_p(row, T, top_k, top_p, theta_g):
    """A top_p for which the oracle's filter of `row` keeps exactly the GPU's
    set {x >= theta_g}: top_p itself when the two cuts agree; otherwise (a
    cut one value group off, allowed only where the fp64 mass at the cut is
    within NEAR of top_p) the middle of theta_g's value group in the oracle's
    own fp64 masses, so that the oracle's descending walk reaches it inside
    that group."""
    ok, near = _cut_ok(row, T, top_k, top_p, theta_g)
    assert ok, (theta_g, oracle.filter_row(row, T, top_k, top_p)[1])
    if not near:
        return top_p, False
    x = workloads.logits_as_f64(row).reshape(-1)
    z = x / T
    p = np.exp(z - z.max())
    keep = x >= np.sort(x)[::-1][top_k - 1] if 0 < top_k < x.size else np.ones(x.size, bool)
    SK = p[keep].sum()
    before = p[keep & (x > theta_g)].sum() / SK
    group = p[keep & (x == theta_g)].sum() / SK
    return before + group / 2, True


def _top_p_rows(prob, top_k, top_p):
    """Each verified row's top_p for the oracle, [B, 2k+1] (target rows 0..k,
    then draft rows 0..k-1): top_p, except on rows where the GPU's filter cut
    sits one value group off the oracle's (a top-p cut whose fp64 mass is
    within NEAR of top_p) -- there the value that gives the oracle the GPU's
    cut, so that every request is still compared in full.  (spec_filter_rows
    runs the same filter kernel, with the same slices and arithmetic, as the
    filtered verification.)"""
    B, R, V = prob["target"].shape
    k = R - 1
    rows = np.concatenate([prob["target"].reshape(B * R, V), prob["draft_logits"].reshape(B * k, V)])
    g = host(api.spec_filter_rows(to_dev(rows), prob["T"], top_k, top_p))
    tp = np.full((B, 2 * k + 1), float(top_p))
    near = 0
    for j in range(rows.shape[0]):
        _, theta_o, _ = oracle.filter_row(rows[j], prob["T"], top_k, top_p)
        if float(g["theta"][j]) != theta_o:
            b, col = (j // R, j % R) if j < B * R else ((j - B * R) // k, k + 1 + (j - B * R) % k)
            tp[b, col], was_near = _gpu_cut_top_p(rows[j], prob["T"], top_k, top_p, float(g["theta"][j]))
            near += was_near
    assert near <= max(1, rows.shape[0] // 8), near
    return tp, near


def _run(prob, top_k, top_p, draft_len=None, max_emit=None):
    args = dict(draft_len=None if draft_len is None else to_dev(draft_len),
                max_emit=None if max_emit is None else to_dev(max_emit), top_k=top_k, top_p=top_p)
    T, D = to_dev(prob["target"]), to_dev(prob["draft_logits"])
    x, u = to_dev(prob["draft"]), to_dev(prob["uniforms"])
    o = api.spec_verify_sample(T, D, x, u, prob["T"], **args)
    poison_like(o)
    o = api.spec_verify_sample(T, D, x, u, prob["T"], out=o, **args)
    torch.cuda.synchronize()
    return host(o)


def _check(prob, g, top_k, top_p, draft_len=None, max_emit=None):
    """Every request of a filtered verification against the oracle's, the
    oracle run with each row's top_p from _top_p_rows."""
    tp, near = _top_p_rows(prob, top_k, top_p)
    if near:
        print("rows with a near top-p cut", near)
    r = oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"], prob["T"],
                             draft_len=draft_len, max_emit=max_emit, top_k=top_k, top_p=top_p,
                             top_p_rows=tp, threads=oracle.max_threads())
    return check_chain_sample_filtered(prob, g, r, top_k, tp, draft_len)


def check_chain_sample_filtered(prob, g, r, top_k, tp, draft_len=None):
    """check_chain_sample with the near-threshold replays on filtered p and q
    (tp: each row's top_p, [B, 2k+1])."""
    B, R, V = prob["target"].shape
    k = R - 1
    np.testing.assert_array_equal(g["status"], r["status"])
    near = 0
    for b in range(B):
        L = k if draft_len is None else int(draft_len[b])
        if r["status"][b] != 0:
            assert g["n_emit"][b] == 0
            continue
        pt, qt = r["p_tok"][b], r["q_tok"][b]
        assert np.all(np.abs(g["p_tok"][b, :L] - pt[:L]) <= TOL) and np.all(np.abs(g["q_tok"][b, :L] - qt[:L]) <= TOL)
        mg, mo = int(g["accepted"][b]), int(r["accepted"][b])
        if mg != mo:
            i = min(mg, mo)
            thr = min(1.0, pt[i] / qt[i]) if qt[i] > 0 else float(pt[i] > 0)
            assert abs(float(prob["uniforms"][b, i]) - thr) < TOL, (b, mg, mo)
            near += 1
            continue
        np.testing.assert_array_equal(g["out_tokens"][b, :mo], r["out_tokens"][b, :mo])
        assert g["n_emit"][b] == r["n_emit"][b]
        assert abs(g["resid_mass"][b] - r["resid_mass"][b]) <= TOL
        ne = int(r["n_emit"][b])
        if mo < ne and g["out_tokens"][b, mo] != r["out_tokens"][b, mo]:
            pf = oracle.filter_row(prob["target"][b, mo], prob["T"], top_k, tp[b, mo])[0]
            if mo < L:
                qf = oracle.filter_row(prob["draft_logits"][b, mo], prob["T"], top_k, tp[b, k + 1 + mo])[0]
                dist, Rm = oracle.residual(pf, qf)
                if Rm <= 0:
                    dist = pf
            else:
                dist = pf
            assert _near_draw(dist, float(prob["uniforms"][b, k]), int(g["out_tokens"][b, mo]),
                              int(r["out_tokens"][b, mo])), (b, "final token")
            near += 1
    return near


@pytest.fixture(params=["cluster", "chunked"])
def accept_kernel(request):
    """The accept kernel after the filter: the cluster one where the plan
    fits (AUTO), or the chunked one on every call."""
    api.set_chain_path(api.CHAIN_AUTO if request.param == "cluster" else api.CHAIN_CHUNKED)
    yield request.param
    api.set_chain_path(api.CHAIN_AUTO)


@pytest.mark.parametrize("seed,B,k,V,dtype,T,top_k,top_p", [
    (1, 1, 4, 248_320, "bf16", 1.0, 50, 1.0), (2, 2, 4, 248_320, "bf16", 1.0, 0, 0.6),
    (3, 16, 4, 3000, "fp32", 1.0, 20, 0.9), (4, 64, 3, 2048, "bf16", 0.8, 0, 0.95),
    (5, 400, 2, 4000, "bf16", 1.0, 40, 0.9), (6, 8, 6, 40_003, "bf16", 1.2, 100, 1.0),
    (7, 4, 0, 50_000, "fp32", 1.0, 10, 0.8)])
def test_filtered_verification_parity(seed, B, k, V, dtype, T, top_k, top_p, accept_kernel):
    """B=400 takes the chunked accept kernel on either setting."""
    prob = _filtered_chain(seed, B, k, V, dtype, T, top_k, top_p)
    g = _run(prob, top_k, top_p)
    print("near", _check(prob, g, top_k, top_p))


def test_filtered_drafts_outside_the_filter_lengths_caps(accept_kernel):
    """Drafts drawn from the unfiltered q (some fall outside q'), variable
    lengths, caps and a bad token, masked logits."""
    B, k, V, top_k, top_p = 24, 5, 6000, 30, 0.9
    prob = _filtered_chain(31, B, k, V, "bf16", 1.0, top_k, top_p, draft_from_filtered=False)
    rng = np.random.default_rng(5)
    t = workloads.bf16_to_f32(prob["target"]).copy()
    t[rng.random(t.shape) < 0.2] = -np.inf
    prob["target"] = workloads.bf16_bits(t)
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    draft_len[0] = -1
    prob["draft"][1, 0] = V
    draft_len[1] = 2
    max_emit = rng.integers(0, k + 2, B).astype(np.int32)
    g = _run(prob, top_k, top_p, draft_len, max_emit)
    _check(prob, g, top_k, top_p, draft_len, max_emit)
    assert list(g["status"][:2]) == [3, 1]
    assert (g["q_tok"][g["status"] == 0] == 0).any()      # some drafts lie outside q'


def test_filters_off_is_the_unfiltered_path():
    prob = workloads.chain_problem(41, 16, 4, 30_000, "bf16", 1.0, target_std=1.5, noise_std=0.8)
    a = _run(prob, 0, 1.0)
    b = _run(prob, 30_000, 1.0)   # top_k = V: off
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_filtered_draws_and_their_distribution():
    rng = np.random.default_rng(9)
    B, V, T, top_k, top_p = 6, 50_000, 0.9, 200, 0.85
    x = workloads.bf16_bits((rng.standard_normal((B, V)) * 2).astype(np.float32))
    u = rng.random(B, dtype=np.float32)
    g = host(api.spec_sample(to_dev(x), to_dev(u), T, top_k=top_k, top_p=top_p))
    for b in range(B):
        pf = oracle.filter_row(x[b], T, top_k, top_p)[0]
        r = oracle.verify_sample(np.ascontiguousarray(x[b:b + 1, None]), np.zeros((1, 0, V), x.dtype),
                                 np.zeros((1, 0), np.int32), u[b:b + 1, None], T, top_k=top_k, top_p=top_p)
        rt, gt = int(r["out_tokens"][0, 0]), int(g["tokens"][b])
        assert rt == gt or _near_draw(pf, float(u[b]), rt, gt)
        assert abs(g["probs"][b] - pf[gt]) <= TOL
    # 200,000 draws from one filtered row (a V=2048 row, broadcast)
    row = workloads.chain_small()["draft_logits"][0, 0]
    n = 200_000
    pf = oracle.filter_row(row, 1.0, 64, 0.9)[0]
    uu = np.random.default_rng(10).random(n, dtype=np.float32)
    g = host(api.spec_sample(to_dev(row)[None].expand(n, row.size), to_dev(uu), 1.0, top_k=64, top_p=0.9))
    counts = np.bincount(g["tokens"], minlength=row.size)
    kept = pf > 0
    assert counts[~kept].sum() == 0
    # Pearson chi-square over the kept tokens: dof = kept - 1 for a correct
    # sampler, its standard deviation sqrt(2 dof); a bound of 6 standard deviations
    chi2 = np.sum((counts[kept] - n * pf[kept]) ** 2 / (n * pf[kept]))
    dof = kept.sum() - 1
    assert chi2 < dof + 6 * np.sqrt(2 * dof), (chi2, dof)
    print("kept", kept.sum(), "chi2", chi2, "dof", dof)


def _path_rows(kind, V, rng):
    """Rows that steer the filter kernel down each of its paths (with top_k =
    50): the max's top-byte bin holding >= 50 logits ("bin0"); fewer, with the
    bin below completing them ("bin1"); a top bin too full for the per-CTA
    list ("dense"); a negative max ("negative"); a max in the two lowest
    bins, the window reaching bin 1 ("tiny"); a max of +0, where the window
    is not tried ("zero")."""
    x = (rng.standard_normal(V) * 0.3).astype(np.float32)
    if kind == "bin0":
        x = (rng.standard_normal(V) * 2.5).astype(np.float32)
    elif kind == "bin1":
        x[rng.choice(V, 300, replace=False)] = rng.uniform(2.5, 7.5, 300)
        x[rng.choice(V, 3, replace=False)] = 20.0
    elif kind == "dense":
        x = rng.uniform(8.5, 30.0, V).astype(np.float32)
    elif kind == "negative":
        x = rng.uniform(-30.0, -1.5, V).astype(np.float32)
    elif kind == "tiny":
        x[:] = -np.inf
        x[rng.choice(V, 60, replace=False)] = -1e38
        x[rng.choice(V, 3, replace=False)] = -2e37
    elif kind == "zero":
        x = -np.abs(x)
        x[rng.choice(V, 70, replace=False)] = 0.0
    return x


@pytest.mark.parametrize("dtype,top_p,reps", [("bf16", 1.0, 1), ("fp32", 1.0, 1), ("bf16", 0.7, 1), ("fp32", 0.7, 1),
                                               ("bf16", 1.0, 52), ("bf16", 0.7, 52), ("fp32", 0.7, 52)])
def test_filter_paths(dtype, top_p, reps):
    """Every path of the filter kernel: the thresholds and kept counts of
    spec_filter_rows, and filtered verification (p_tok, q_tok and the
    residual mass test the kept mass) on requests made of the same rows.
    reps = 52 gives 312 rows and 66 requests of 5 verified rows, enough rows
    for the kernel's row mode (one CTA per row, no staged slices)."""
    rng = np.random.default_rng(77)
    V, top_k, T = 128_256, 50, 1.0
    kinds = ["bin0", "bin1", "dense", "negative", "tiny", "zero"] * reps
    x = np.stack([_path_rows(kd, V, rng) for kd in kinds])
    rows = workloads.bf16_bits(x) if dtype == "bf16" else x
    api.trace_enable(True)
    api.trace_collect()
    try:
        g = host(api.spec_filter_rows(to_dev(rows), T, top_k, top_p))
        launched = api.trace_collect()
    finally:
        api.trace_enable(False)
    assert ("chain_filter_rows" if reps > 1 else "chain_filter") in launched, launched
    for r in range(len(kinds)):
        ok, was_near = _cut_ok(rows[r], T, top_k, top_p, float(g["theta"][r]))
        _, theta_o, kept_o = oracle.filter_row(rows[r], T, top_k, top_p)
        assert ok, (r, kinds[r], g["theta"][r], theta_o)
        assert was_near or g["kept"][r] == kept_o, (r, kinds[r], g["kept"][r], kept_o)
    # requests: target rows 0..k from one kind, draft rows = target + noise
    # (66 requests x 5 rows in the row-mode case)
    if reps > 1:
        x = x[:66]
    B, k = x.shape[0], 2
    tgt = np.repeat(x[:, None, :], k + 1, axis=1).copy()
    tgt[:, 1:] += (rng.standard_normal((B, k, V)) * 0.05).astype(np.float32)
    dl = tgt[:, :k] + (rng.standard_normal((B, k, V)) * 0.2).astype(np.float32)
    cast = workloads.bf16_bits if dtype == "bf16" else (lambda a: np.ascontiguousarray(a, np.float32))
    prob = dict(target=cast(tgt), draft_logits=cast(dl), T=T, B=B, k=k, V=V, dtype=dtype,
                draft=np.zeros((B, k), np.int32), uniforms=workloads.uniforms(rng, (B, k + 1)))
    for b in range(B):
        for i in range(k):
            qf = oracle.filter_row(prob["draft_logits"][b, i], T, top_k, top_p)[0]
            prob["draft"][b, i] = rng.choice(V, p=qf / qf.sum())
    gv = _run(prob, top_k, top_p)
    _check(prob, gv, top_k, top_p)
