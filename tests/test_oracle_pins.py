"""Pins for the CPU FP64 oracle: every check compares it with something other
than itself (hand-worked values, an explicit S-matrix form, the chunked WY
form with a library inverse, O(T^2) closed forms, exact retrieval, structural
identities).  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import pin_forms as pf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def rand_case(rng, B=1, T=37, H=2, K=6, V=5, delta=True, h0=True, lengths=None,
              g_mu=1.0):
    """Small FP64 inputs with unit-norm keys and queries."""
    if lengths is not None:
        B, T = 1, int(sum(lengths))
    q = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, H)))) if delta else None
    g = -np.log1p(np.exp(-(rng.standard_normal((B, T, H)) + g_mu)))
    cu = None
    N = B
    if lengths is not None:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
        N = len(lengths)
    hz = 0.1 * rng.standard_normal((N, H, K, V)) if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu=cu, h0=hz)


def slice_tokens(c, a, b):
    """Dense case restricted to tokens [a, b) (h0 kept)."""
    out = dict(c)
    for key in ("q", "k", "v", "g", "beta"):
        if c[key] is not None:
            out[key] = c[key][:, a:b]
    return out


def run_oracle(c, **kw):
    o, ht, _ = oracle.forward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                              cu_seqlens=c["cu"], h0=c["h0"], **kw)
    return o, ht


# --------------------------------------------------------------------------
# hand-worked values
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked(case):
    K, V = case["K"], case["V"]
    T = len(case["alpha"])
    q = np.array(case["q"], dtype=np.float64).reshape(1, T, 1, K)
    k = np.array(case["k"], dtype=np.float64).reshape(1, T, 1, K)
    v = np.array(case["v"], dtype=np.float64).reshape(1, T, 1, V)
    g = np.log(np.array(case["alpha"])).reshape(1, T, 1)
    beta = None if case["beta"] is None else np.array(case["beta"]).reshape(1, T, 1)
    h0 = None if case["h0"] is None else np.array(case["h0"]).reshape(1, 1, K, V)
    o, ht, _ = oracle.forward(q, k, v, g, beta, h0=h0)
    np.testing.assert_allclose(o.reshape(T, V), np.array(case["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(ht.reshape(K, V), np.array(case["ht"]), rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# brute force: explicit S-matrix product and the chunked WY formulation
# --------------------------------------------------------------------------
@pytest.mark.parametrize("delta", [True, False])
@pytest.mark.parametrize("T", [1, 15, 64, 65, 130])
def test_matrix_form(delta, T):
    rng = np.random.default_rng(T + 100 * delta)
    c = rand_case(rng, B=2, T=T, H=2, K=8, V=7, delta=delta)
    o, ht = run_oracle(c)
    mo, mht = pf.matrix_form(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                             1 / math.sqrt(8))
    assert pf.rel(o, mo) < 1e-12
    assert pf.rel(ht, mht) < 1e-12


@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("T", [63, 64, 65, 127, 130, 257])
@pytest.mark.parametrize("delta", [True, False])
def test_chunked_wy_form(chunk, T, delta):
    rng = np.random.default_rng(1000 + T + chunk + delta)
    c = rand_case(rng, B=1, T=T, H=2, K=8, V=6, delta=delta)
    o, ht = run_oracle(c)
    co, cht = pf.chunked_form(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                              1 / math.sqrt(8), chunk)
    assert pf.rel(o, co) < 1e-12
    assert pf.rel(ht, cht) < 1e-12


def test_chunked_wy_form_varlen():
    rng = np.random.default_rng(7)
    lengths = [1, 63, 64, 65, 130, 7]
    c = rand_case(rng, H=2, K=8, V=8, lengths=lengths)
    o, ht = run_oracle(c)
    co, cht = pf.chunked_form(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                              1 / math.sqrt(8), 64, cu=c["cu"])
    assert pf.rel(o, co) < 1e-12
    assert pf.rel(ht, cht) < 1e-12


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 50, 129])
def test_beta_free_closed_form(T):
    rng = np.random.default_rng(T)
    c = rand_case(rng, B=2, T=T, H=3, K=8, V=5, delta=False)
    o, ht = run_oracle(c)
    co, cht = pf.gla_closed_form(c["q"], c["k"], c["v"], c["g"], c["h0"], 1 / math.sqrt(8))
    assert pf.rel(o, co) < 1e-12
    assert pf.rel(ht, cht) < 1e-12


def test_literal_beta_zero():
    """beta = 0 freezes every write: o_t = e^{G_t} h0^T q_t / sqrt(K) and
    ht = e^{G_T} h0 (G: sequence-global cumsum)."""
    rng = np.random.default_rng(3)
    c = rand_case(rng, B=1, T=90, H=2, K=8, V=4)
    c["beta"] = np.zeros_like(c["g"])
    o, ht = run_oracle(c)
    G = np.cumsum(c["g"][0], axis=0)  # [T, H]
    exp_o = np.einsum("th,hkv,thk->thv", np.exp(G), c["h0"][0], c["q"][0]) / math.sqrt(8)
    np.testing.assert_allclose(o[0], exp_o, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(ht[0], np.exp(G[-1])[:, None, None] * c["h0"][0],
                               rtol=1e-12, atol=1e-15)


def test_exact_retrieval_orthonormal_keys():
    """alpha = 1, beta = 1, orthonormal keys, h0 = 0: the state maps each
    written key to its value, a query on key j returns v_j / sqrt(K), an
    unwritten orthonormal key reads 0, and re-writing a key overwrites."""
    rng = np.random.default_rng(11)
    K, V = 16, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm.T  # rows orthonormal
    T = K + 4
    k = np.zeros((1, T, 1, K))
    k[0, :K, 0] = keys
    k[0, K:, 0] = keys[:4]  # rewrite keys 0..3
    v = rng.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    q = np.zeros((1, T, 1, K))
    q[0, :, 0] = keys[0]  # always query key 0
    o, ht, _ = oracle.forward(q, k, v, g, beta)
    s = 1 / math.sqrt(K)
    for t in range(T):
        want = v[0, K, 0] if t >= K else v[0, 0, 0]
        np.testing.assert_allclose(o[0, t, 0], want * s, atol=1e-12)
    # the final state maps every key to its latest value
    S = ht[0, 0].T  # V x K
    for j in range(K):
        latest = K + j if j < 4 else j
        np.testing.assert_allclose(S @ keys[j], v[0, latest, 0], atol=1e-12)
    # a key not yet written reads zero
    q2 = np.zeros_like(q)
    q2[0, :, 0] = keys[K - 1]
    o2, _, _ = oracle.forward(q2, k, v, g, beta)
    np.testing.assert_allclose(o2[0, :K - 1, 0], 0.0, atol=1e-12)


# --------------------------------------------------------------------------
# structural identities
# --------------------------------------------------------------------------
def test_varlen_equals_independent_runs():
    rng = np.random.default_rng(5)
    lengths = [3, 64, 100, 1, 65]
    c = rand_case(rng, H=2, K=8, V=8, lengths=lengths)
    o, ht = run_oracle(c)
    cu = c["cu"]
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        sl = (slice(0, 1), slice(a, b))
        on, htn, _ = oracle.forward(c["q"][sl], c["k"][sl], c["v"][sl], c["g"][sl],
                                    c["beta"][sl], h0=c["h0"][n:n + 1])
        assert np.array_equal(on, o[sl])
        assert np.array_equal(htn, ht[n:n + 1])


@pytest.mark.parametrize("t1", [1, 63, 64, 77])
def test_state_carry(t1):
    rng = np.random.default_rng(t1)
    c = rand_case(rng, B=1, T=150, H=2, K=8, V=6)
    o, ht = run_oracle(c)
    oa, hta = run_oracle(slice_tokens(c, 0, t1))
    b = slice_tokens(c, t1, 150)
    b["h0"] = hta
    ob, htb = run_oracle(b)
    assert pf.rel(np.concatenate([oa, ob], axis=1), o) < 1e-12
    assert pf.rel(htb, ht) < 1e-12


def test_linearity_in_v_and_h0():
    rng = np.random.default_rng(9)
    c1 = rand_case(rng, B=1, T=70, H=2, K=8, V=6)
    c2 = dict(c1)
    c2["v"] = rng.standard_normal(c1["v"].shape)
    c2["h0"] = rng.standard_normal(c1["h0"].shape)
    lam = -1.7
    c3 = dict(c1)
    c3["v"] = c1["v"] + lam * c2["v"]
    c3["h0"] = c1["h0"] + lam * c2["h0"]
    o1, h1 = run_oracle(c1)
    o2, h2 = run_oracle(c2)
    o3, h3 = run_oracle(c3)
    assert pf.rel(o3, o1 + lam * o2) < 1e-12
    assert pf.rel(h3, h1 + lam * h2) < 1e-12


def test_stability_invariant():
    """Unit keys and beta in [0, 1] make (I - beta k k^T) non-expanding, so
    ||h_t|| <= e^{g_t} ||h_{t-1}|| + beta_t ||k_t|| ||v_t|| (Frobenius)."""
    rng = np.random.default_rng(13)
    c = rand_case(rng, B=1, T=60, H=1, K=8, V=6, g_mu=4.0)
    h = c["h0"]
    for t in range(60):
        step = slice_tokens(c, t, t + 1)
        step["h0"] = h
        _, hn = run_oracle(step)
        bound = (math.exp(c["g"][0, t, 0]) * np.linalg.norm(h)
                 + c["beta"][0, t, 0] * np.linalg.norm(c["v"][0, t, 0]))
        assert np.linalg.norm(hn) <= bound * (1 + 1e-12)
        h = hn


@pytest.mark.parametrize("S", [2, 4, 8, 16])
@pytest.mark.parametrize("delta", [True, False])
def test_segment_split_composition(S, delta):
    rng = np.random.default_rng(S)
    lengths = [200, 64 * 5 + 3, 40]
    c = rand_case(rng, H=2, K=6, V=5, lengths=lengths, delta=delta)
    o, ht = run_oracle(c)
    so, sht = oracle.forward_segmented(c["q"], c["k"], c["v"], c["g"], c["beta"],
                                       cu_seqlens=c["cu"], h0=c["h0"], n_segments=S)
    assert pf.rel(so, o) < 1e-10
    assert pf.rel(sht, ht) < 1e-10


@pytest.mark.parametrize("S", [2, 4, 16])
@pytest.mark.parametrize("delta", [True, False])
def test_segment_split_common_length(S, delta):
    """One run length for the whole batch (ceil(longest / S) chunks): the
    short sequences stay one run, the long one is cut; the composition still
    rebuilds the serial result."""
    rng = np.random.default_rng(100 + S)
    lengths = [64 * 9 + 5, 64, 0, 70, 130]
    c = rand_case(rng, H=2, K=6, V=5, lengths=lengths, delta=delta)
    o, ht = run_oracle(c)
    so, sht = oracle.forward_segmented(c["q"], c["k"], c["v"], c["g"], c["beta"],
                                       cu_seqlens=c["cu"], h0=c["h0"], n_segments=S,
                                       common=True)
    assert pf.rel(so, o) < 1e-10
    assert pf.rel(sht, ht) < 1e-10


def test_affine_map_matches_recurrence():
    """M h_in + c equals the recurrence run from h_in, for random h_in."""
    rng = np.random.default_rng(21)
    c = rand_case(rng, B=1, T=45, H=1, K=7, V=4)
    M, cc = oracle.affine(c["k"][0, :, 0], c["v"][0, :, 0], c["g"][0, :, 0],
                          c["beta"][0, :, 0])
    for _ in range(3):
        hin = rng.standard_normal((1, 1, 7, 4))
        _, ht, _ = oracle.forward(c["q"], c["k"], c["v"], c["g"], c["beta"], h0=hin)
        assert pf.rel(M @ hin[0, 0] + cc, ht[0, 0]) < 1e-12


def test_segment_bounds():
    assert oracle.segment_bounds(0, 4) == []
    assert oracle.segment_bounds(65, 4) == [(0, 64), (64, 65)]
    assert oracle.segment_bounds(64 * 16, 16) == [(64 * i, 64 * (i + 1)) for i in range(16)]
    assert oracle.segment_bounds(64 * 10, 4) == [(0, 192), (192, 384), (384, 576), (576, 640)]
    # a common run length: 3 chunks a run whatever the sequence's own length
    assert oracle.segment_bounds(64 * 2 + 1, 4, per=3) == [(0, 129)]
    assert oracle.segment_bounds(64 * 7, 4, per=3) == [(0, 192), (192, 384), (384, 448)]


def test_pair_mask_limits_work():
    rng = np.random.default_rng(2)
    c = rand_case(rng, B=2, T=20, H=3, K=4, V=4)
    o, ht = run_oracle(c)
    mask = np.zeros(6, dtype=bool)
    mask[4] = True  # sequence 1, head 1
    om, htm = run_oracle(c, pair_mask=mask)
    assert np.array_equal(om[1, :, 1], o[1, :, 1])
    assert np.array_equal(htm[1, 1], ht[1, 1])
    assert np.isnan(om[0]).all() and np.isnan(htm[0]).all()


def test_rejects_bad_cu_seqlens():
    rng = np.random.default_rng(2)
    c = rand_case(rng, lengths=[5, 5], K=4, V=4)
    c["cu"] = np.array([0, 6, 5], dtype=np.int64)
    with pytest.raises(ValueError):
        run_oracle(c)
