"""Pins for the oracle's backward pass (``oracle.backward``): the gradient of
L = <do, o> + <dht, ht> with respect to q, k, v, g, beta and h0.

The pins stand on the forward oracle (itself pinned in
``test_oracle_pins.py``) and on the mathematics, not on the backward code:

* central finite differences of L along random directions, for every input,
  on dense and varlen batches whose sequences span several 64-token replay
  blocks, ragged tails and empty sequences, delta rule and beta-free;
* exact identities of a function that is linear in some of its inputs: for
  fixed q, k, g, beta the pair (o, ht) is linear in (v, h0), so
  <do, o> + <dht, ht> = <dv, v> + <dh0, h0>; o is linear in q and ht does not
  depend on it, so <do, o> = <dq, q>;
* an empty sequence passes the final-state gradient straight through
  (dh0 = dht); varlen equals independent per-sequence runs;
* the closed form of the scalar case (K = V = 1, two tokens), derived by
  the chain rule on the explicit composition of the two steps.

Planted mistakes in copies of the C source (a dropped term, a wrong sign, a
state read one token off, a missing decay factor) must each fail one pin.
"""
import numpy as np
import pytest

import oracle
from test_oracle_mutants import SRC, _case, _compile

NAMES = ("q", "k", "v", "g", "beta", "h0")


def _loss(lib, args, cu, do, dht):
    q, k, v, g, beta, h0 = args
    o, ht, _ = oracle.forward(q, k, v, g, beta, cu_seqlens=cu, h0=h0, lib=lib)
    out = float(np.sum(o * do))
    if dht is not None:
        out += float(np.sum(ht * dht))
    return out


def fd_errors(lib, args, cu, do, dht, rng, eps=1e-6):
    """Relative gap between <grad, d> and the central difference of L along a
    random direction d, per input."""
    grads = oracle.backward(*args[:5], cu_seqlens=cu, h0=args[5], do=do, dht=dht, lib=lib)
    errs = {}
    for i, name in enumerate(NAMES):
        if args[i] is None:
            continue
        d = rng.standard_normal(args[i].shape)
        plus, minus = list(args), list(args)
        plus[i] = args[i] + eps * d
        minus[i] = args[i] - eps * d
        fd = (_loss(lib, plus, cu, do, dht) - _loss(lib, minus, cu, do, dht)) / (2 * eps)
        an = float(np.sum(grads[i] * d))
        errs[name] = abs(fd - an) / max(abs(an), 1e-300)
    return errs


def _cases(rng):
    """(args, cu, do, dht) for the pinned configurations."""
    out = []
    for delta in (True, False):
        q, k, v, g, beta, cu, h0 = _case(rng, B=2, T=150, H=2, K=5, V=3, delta=delta)
        do = rng.standard_normal(v.shape)
        dht = rng.standard_normal(h0.shape)
        out.append(((q, k, v, g, beta, h0), None, do, dht))
    q, k, v, g, beta, cu, h0 = _case(rng, H=2, K=5, V=3, lengths=[0, 1, 70, 64, 3])
    do = rng.standard_normal(v.shape)
    out.append(((q, k, v, g, beta, h0), cu, do, rng.standard_normal(h0.shape)))
    out.append(((q, k, v, g, beta, h0), cu, do, None))  # no final-state term
    return out


def scalar_two_token_grads(q, k, v, g, b, s0, do, dht, scale, delta=True):
    """Gradients of L = do1 o1 + do2 o2 + dht h2 for K = V = 1 and two
    tokens, by the chain rule on the explicit composition
        h1 = a1 s0 (1 - b1 k1^2) + b1 k1 v1,  h2 = a2 h1 (1 - b2 k2^2) + b2 k2 v2
    (beta-free: h_t = a_t h_{t-1} + k_t v_t), o_t = scale q_t h_t.
    Returns dq, dk, dv, dg, dbeta (arrays of 2) and ds0."""
    a = np.exp(g)
    if not delta:
        b = np.zeros(2)
    p = 1 - b * k * k if delta else np.ones(2)       # the transition factor
    w = b * k * v if delta else k * v                # the write
    h1 = a[0] * s0 * p[0] + w[0]
    h2 = a[1] * h1 * p[1] + w[1]
    D2 = scale * q[1] * do[1] + dht                  # dL/dh2
    D1 = scale * q[0] * do[0] + D2 * a[1] * p[1]     # dL/dh1
    hp = np.array([s0, h1])                          # state before each token
    D = np.array([D1, D2])
    dq = scale * np.array([h1, h2]) * do
    dg = D * a * hp * p
    if delta:
        dk = D * (a * hp * (-2 * b * k) + b * v)
        dv = D * b * k
        db = D * (-a * hp * k * k + k * v)
    else:
        dk = D * v
        dv = D * k
        db = None
    ds0 = D1 * a[0] * p[0]
    return dq, dk, dv, dg, db, ds0


def scalar_closed_form_errors(lib, rng):
    """Largest relative gap between the oracle and the scalar closed form
    over a few random cases, delta rule and beta-free."""
    worst = 0.0
    for delta in (True, False):
        for _ in range(4):
            q, k, v = rng.standard_normal(2), rng.standard_normal(2), rng.standard_normal(2)
            g = -np.abs(rng.standard_normal(2))
            b = 1 / (1 + np.exp(-rng.standard_normal(2)))
            s0, dht = rng.standard_normal(), rng.standard_normal()
            do = rng.standard_normal(2)
            scale = 0.7
            ref = scalar_two_token_grads(q, k, v, g, b, s0, do, dht, scale, delta)
            out = oracle.backward(q.reshape(1, 2, 1, 1), k.reshape(1, 2, 1, 1),
                                  v.reshape(1, 2, 1, 1), g.reshape(1, 2, 1),
                                  b.reshape(1, 2, 1) if delta else None,
                                  h0=np.array(s0).reshape(1, 1, 1, 1), do=do.reshape(1, 2, 1, 1),
                                  dht=np.array(dht).reshape(1, 1, 1, 1), scale=scale, lib=lib)
            for got, want in zip(out, ref):
                if want is None:
                    continue
                got = np.asarray(got).reshape(-1)
                want = np.asarray(want).reshape(-1)
                worst = max(worst, float(np.max(np.abs(got - want) / (np.abs(want) + 1e-12))))
    return worst


def bwd_battery(lib) -> list:
    """Runs the backward pins against ``lib``; returns the names that failed."""
    failed = []
    rng = np.random.default_rng(1)
    if not scalar_closed_form_errors(lib, rng) < 1e-12:
        failed.append("scalar_two_token_closed_form")
    for ci, (args, cu, do, dht) in enumerate(_cases(rng)):
        for name, err in fd_errors(lib, args, cu, do, dht, rng).items():
            if not err < 1e-6:
                failed.append(f"finite_difference:{ci}:{name}")
        q, k, v, g, beta, h0 = args
        o, ht, _ = oracle.forward(q, k, v, g, beta, cu_seqlens=cu, h0=h0, lib=lib)
        dq, dk, dv, dg, dbeta, dh0 = oracle.backward(q, k, v, g, beta, cu_seqlens=cu, h0=h0,
                                                     do=do, dht=dht, lib=lib)
        lhs = np.sum(o * do) + (np.sum(ht * dht) if dht is not None else 0.0)
        rhs = np.sum(dv * v) + np.sum(dh0 * h0)
        if not abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs)):
            failed.append(f"linear_in_v_h0:{ci}")
        if not abs(np.sum(o * do) - np.sum(dq * q)) <= 1e-12 * max(1.0, abs(lhs)):
            failed.append(f"linear_in_q:{ci}")
    # empty sequence: dh0 = dht; other sequences unaffected by their neighbours
    q, k, v, g, beta, cu, h0 = _case(rng, H=1, K=4, V=3, lengths=[0, 9, 66])
    do = rng.standard_normal(v.shape)
    dht = rng.standard_normal(h0.shape)
    full = oracle.backward(q, k, v, g, beta, cu_seqlens=cu, h0=h0, do=do, dht=dht, lib=lib)
    if not np.array_equal(full[5][0], dht[0]):
        failed.append("empty_sequence_passes_dht")
    for n in (1, 2):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = (slice(0, 1), slice(a, b))
        one = oracle.backward(q[sl], k[sl], v[sl], g[sl], beta[sl], h0=h0[n:n + 1],
                              do=do[sl], dht=dht[n:n + 1], lib=lib)
        for i in range(5):
            if not np.array_equal(one[i], full[i][sl]):
                failed.append(f"varlen_independent:{n}:{i}")
        if not np.array_equal(one[5], full[5][n:n + 1]):
            failed.append(f"varlen_independent:{n}:dh0")
    return failed


def test_backward_pins_hold():
    assert bwd_battery(None) == []


def test_scalar_two_token_closed_form():
    """K = V = 1, two tokens: the oracle's gradients equal the hand-derived
    chain rule of the explicit composition, delta rule and beta-free."""
    assert scalar_closed_form_errors(None, np.random.default_rng(11)) < 1e-12


def test_finite_differences_are_tight():
    """The directional derivatives agree with central differences to about
    1e-9 (the differences' own truncation and rounding error)."""
    rng = np.random.default_rng(5)
    args, cu, do, dht = _cases(rng)[0]
    errs = fd_errors(None, args, cu, do, dht, rng)
    assert max(errs.values()) < 1e-7, errs


BWD_MUTANTS = {
    "dq_uses_previous_state": ("acc += hcur[i * V + j] * dot[j];",
                               "acc += hprev[i * V + j] * dot[j];"),
    "readout_grad_drops_scale": ("dh[i * V + j] += J->scale * qt[i] * dot[j];",
                                 "dh[i * V + j] += qt[i] * dot[j];"),
    "state_grad_drops_prediction_term": ("dh[i * V + j] += kt[i] * dy;",
                                         "dh[i * V + j] += 0.0 * kt[i] * dy;"),
    "dk_drops_prediction_term": ("dkt[i] += acc;", "dkt[i] += 0.0 * acc;"),
    "dbeta_sign": ("db += du[j] * (vt[j] - y[j]);", "db += du[j] * (vt[j] + y[j]);"),
    "dv_drops_beta": ("dvt[j] = bb * du[j];", "dvt[j] = du[j];"),
    "dg_drops_gate_factor": ("J->dg[tok] = a * da;", "J->dg[tok] = da;"),
    "state_grad_not_decayed": ("dh[i] *= a;", "dh[i] *= 1.0;"),
    "replay_skips_block_start": ("memcpy(st, ck + b * KV, sizeof(double) * (size_t)KV);",
                                 "memcpy(st, ck + (b > 0 ? b - 1 : 0) * KV, sizeof(double) * (size_t)KV);"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_mutant_is_caught(name, tmp_path):
    source = open(SRC).read()
    old, new = BWD_MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    lib = _compile(source.replace(old, new), str(tmp_path / f"{name}.so"))
    assert bwd_battery(lib), f"pins did not catch mutant {name}"
