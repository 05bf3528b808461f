"""Plants plausible mistakes in copies of the oracle's C source (a dropped
term, a wrong sign, a wrong operand or index) and checks that the pins reject
every copy.  The mistakes live only in temporary copies compiled here, on the
CPU; the committed oracle is untouched."""
import json
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
import pin_forms as pf

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")

MUTANTS = {
    "delta_sign": ("u[j] = b * (vt[j] - u[j]);", "u[j] = b * (vt[j] + u[j]);"),
    "dropped_beta": ("u[j] = b * (vt[j] - u[j]);", "u[j] = (vt[j] - u[j]);"),
    "dropped_decay": ("S[i] *= a;", "S[i] *= 1.0;"),
    "readout_uses_k": ("ot[j] += Si[j] * qi;", "ot[j] += Si[j] * kt[i];"),
    "dropped_scale": ("ot[j] *= J->scale;", "ot[j] *= 1.0;"),
    "prediction_uses_q": ("u[j] += Si[j] * ki;", "u[j] += Si[j] * qt[i];"),
    "no_delta_correction": ("Si[j] += ki * u[j];", "Si[j] += ki * vt[j] * (J->beta ? J->beta[tok] : 1.0);"),
    "gate_sign": ("const double a = exp(J->g[tok]);", "const double a = exp(-J->g[tok]);"),
    "dropped_head_index": ("const int64_t tok = (row * J->T + t) * H + hh;",
                           "const int64_t tok = (row * J->T + t) * H;"),
    "h0_transposed": ("memcpy(S, J->h0 + sidx, sizeof(double) * (size_t)(K * V));",
                      "for (int64_t i = 0; i < K * V; ++i) S[i] = J->h0[sidx + (i % K) * V + i / K];"),
    "varlen_drops_last_token": ("t1 = J->cu[n + 1];", "t1 = J->cu[n + 1] - 1;"),
    "affine_transition_sign": ("M[i * K + j] = a * (M[i * K + j] - b * kt[i] * r[j]);",
                               "M[i * K + j] = a * (M[i * K + j] + b * kt[i] * r[j]);"),
    "affine_dropped_beta_write": ("b * kt[i] * vt[j];", "kt[i] * vt[j];"),
    "affine_beta_free_no_decay": ("c[i * V + j] = a * c[i * V + j] + kt[i] * vt[j];",
                                  "c[i * V + j] = c[i * V + j] + kt[i] * vt[j];"),
}


def _compile(src_text, out):
    c_path = out + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    c_path, "-o", out, "-lm"], check=True)
    return oracle.load_library(out)


def _case(rng, B=1, T=70, H=2, K=6, V=5, delta=True, lengths=None):
    if lengths is not None:
        B, T = 1, int(sum(lengths))
    q = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, H)))) if delta else None
    g = -np.log1p(np.exp(-(rng.standard_normal((B, T, H)) + 1.0)))
    N = len(lengths) if lengths is not None else B
    cu = None if lengths is None else np.concatenate([[0], np.cumsum(lengths)])
    h0 = 0.1 * rng.standard_normal((N, H, K, V))
    return q, k, v, g, beta, cu, h0


def battery(lib) -> list:
    """Runs the pin checks against ``lib``; returns the names that failed."""
    failed = []
    for case in json.load(open(GOLDEN))["cases"]:
        K, V, T = case["K"], case["V"], len(case["alpha"])
        args = (np.array(case["q"], float).reshape(1, T, 1, K),
                np.array(case["k"], float).reshape(1, T, 1, K),
                np.array(case["v"], float).reshape(1, T, 1, V),
                np.log(np.array(case["alpha"])).reshape(1, T, 1),
                None if case["beta"] is None else np.array(case["beta"]).reshape(1, T, 1))
        h0 = None if case["h0"] is None else np.array(case["h0"]).reshape(1, 1, K, V)
        o, ht, _ = oracle.forward(*args, h0=h0, lib=lib)
        if not (np.allclose(o.reshape(T, V), case["o"], atol=1e-12)
                and np.allclose(ht.reshape(K, V), case["ht"], atol=1e-12)):
            failed.append("golden:" + case["name"])
    rng = np.random.default_rng(0)
    for delta in (True, False):
        q, k, v, g, beta, cu, h0 = _case(rng, B=2, H=2, K=6, V=5, delta=delta)
        o, ht, _ = oracle.forward(q, k, v, g, beta, h0=h0, lib=lib)
        mo, mht = pf.matrix_form(q, k, v, g, beta, h0, 1 / math.sqrt(6))
        if not (pf.rel(o, mo) < 1e-12 and pf.rel(ht, mht) < 1e-12):
            failed.append(f"matrix_form:delta={delta}")
        lengths = [5, 64, 70]
        q, k, v, g, beta, cu, h0 = _case(rng, H=2, K=6, V=5, delta=delta, lengths=lengths)
        o, ht, _ = oracle.forward(q, k, v, g, beta, cu_seqlens=cu, h0=h0, lib=lib)
        co, cht = pf.chunked_form(q, k, v, g, beta, h0, 1 / math.sqrt(6), 64, cu=cu)
        if not (pf.rel(o, co) < 1e-12 and pf.rel(ht, cht) < 1e-12):
            failed.append(f"chunked_form_varlen:delta={delta}")
        try:
            so, sht = oracle.forward_segmented(q, k, v, g, beta, cu_seqlens=cu, h0=h0,
                                               n_segments=2, lib=lib)
            if not (pf.rel(sht, cht) < 1e-10 and pf.rel(so, co) < 1e-10):
                failed.append(f"segment_split:delta={delta}")
        except ValueError:
            failed.append(f"segment_split:delta={delta}")
    return failed


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


def test_unmutated_source_passes(source, tmp_path):
    lib = _compile(source, str(tmp_path / "clean.so"))
    assert battery(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    lib = _compile(source.replace(old, new), str(tmp_path / f"{name}.so"))
    assert battery(lib), f"pins did not catch mutant {name}"
