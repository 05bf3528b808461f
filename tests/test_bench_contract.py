"""bench.py's contract on the CPU: the reference arm's JSON line carries every
key the launch contract asks for, and the roofline numerators (algorithmic
bytes and flops) are defined for every kernel the library reports."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "cpu_baseline", "e2e", "gpu_launches"}


def _bench():
    spec = importlib.util.spec_from_file_location("bench_contract", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_reference_arm_line(which):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--pass", which, "--steps", "1",
           "--warmup", "0", "--workload", "tiny_dense_f32"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert REQUIRED <= set(line), REQUIRED - set(line)
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"]
    assert ("gdr_chunk_bwd" in line["metric"]) == (which == "bwd")
    cb = line["cpu_baseline"]
    assert {"value", "unit", "cores", "kind", "sample"} <= set(cb) and cb["kind"] == "oracle"
    assert cb["value"] == line["value"] and cb["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny_dense_f32"


def test_roofline_numerators_cover_every_kernel():
    import chunked_gated_delta_rule_gb300 as pkg
    from chunked_gated_delta_rule_gb300 import synthetic
    b = _bench()
    names = set()
    for kid in range(64):
        n = pkg.gdr_kernel_name(kid)
        if n != "?":
            names.add(n)
    fwd = {"tc_prep", "tc_chain_serial", "tc_chain_prescan", "tc_prescan_dual",
           "tc_chain_segment_out", "tc_gla_serial", "tc_gla_prescan", "tc_gla_segment_out",
           "compose_delta", "compose_scalar", "simt_prep", "simt_scan_serial",
           "simt_scan_segment_out", "simt_output"}
    bwd = {"bwd_gram", "bwd_dscan", "bwd_lk", "bwd_local", "simt_prep", "simt_scan_serial"}
    assert fwd <= names and bwd <= names
    for wname in ("wide_varlen_bf16", "gla_k256_v512_bf16", "tiny_dense_f32"):
        x = synthetic.make_inputs(synthetic.small(synthetic.WORKLOADS[wname], T=256)
                                  if wname != "wide_varlen_bf16" else
                                  synthetic.WORKLOADS[wname], lengths=None)
        c = b.counts(x, 4)
        for k in fwd:
            v = b.algorithmic_bytes(k, x, c)
            assert v is not None and v > 0, (wname, k)
        for k in bwd:
            by, fl = b.bwd_algorithmic(k, x, c)
            assert by > 0 and fl >= 0, (wname, k)
        assert b.algorithmic_bytes("call", x, c) > 0


def test_traffic_records_follow_each_kernels_includes():
    """A kernel's source hash covers its .cu file and the headers it
    includes, so the host-only header does not enter a tensor-core kernel's
    hash, and every record in the committed summary names a known kernel."""
    b = _bench()
    assert b.kernel_sources("tc_prep")[0] == "tc_prep.cu"
    assert "gdr_internal.cuh" in b.kernel_sources("tc_prep")
    assert "gdr_launch.cuh" not in b.kernel_sources("tc_prep")
    assert "simt_tile.cuh" in b.kernel_sources("bwd_local")
    h1 = b.source_hash("tc_prep")
    assert len(h1) == 16 and h1 == b.source_hash("tc_prep")
    assert b.source_hash("tc_prep") != b.source_hash("tc_chain_serial")
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    kernels = set()
    for line in open(path):
        if line.startswith("kernel="):
            f = dict(kv.split("=", 1) for kv in line.split())
            kernels.add(f["kernel"])
            assert float(f["dram_bytes_per_launch"]) >= 0
    assert {"tc_prep", "tc_chain_serial", "tc_bwd_grad", "tc_bwd_scan"} <= kernels


def test_measured_traffic_stays_near_the_algorithmic_bytes():
    """Every committed DRAM record is within 1.25x of the kernel's
    algorithmic bytes for its workload (no kernel re-reads its operands
    wholesale); values below 1 are writes still in L2 when the launch ends."""
    import chunked_gated_delta_rule_gb300 as pkg
    from chunked_gated_delta_rule_gb300 import synthetic
    b = _bench()
    cache = {}
    checked = 0
    for line in open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")):
        if not line.startswith("kernel="):
            continue
        f = dict(kv.split("=", 1) for kv in line.split())
        k, w, t = f["kernel"], f["workload"], float(f["dram_bytes_per_launch"])
        backward = w.startswith("bwd_")  # a backward-pass kernel, on workload w[4:]
        if w not in cache:
            x = synthetic.make_inputs(synthetic.WORKLOADS[w[4:] if backward else w])
            cu = x["cu_seqlens"]
            plan = pkg.gdr_plan_query(x["B"], x["T"], x["H"], x["K"], x["V"],
                                      N=x["N"] if cu is not None else 0,
                                      dtype={"f32": 0, "bf16": 1, "f16": 2}[x["dtype"]],
                                      beta_free=x["beta"] is None,
                                      max_len=int((cu[1:] - cu[:-1]).max()) if cu is not None
                                      else 0)
            cache[w] = (x, b.counts(x, plan["n_segments"], b.common_segments(x, plan)))
        x, c = cache[w]
        if backward:
            a = b.bwd_algorithmic(k, x, c)[0]
        elif k.startswith("bwd_"):
            a = b.bwd_algorithmic(k, x, b.counts(x, 1))[0]
        else:
            a = b.algorithmic_bytes(k, x, c)
        if not a or a < (1 << 20):
            continue
        assert t <= 1.25 * a, (k, w, t / a)
        checked += 1
    assert checked >= 25


def test_segment_counts_under_both_cutting_rules():
    """The units the roofline numerators count, for a varlen batch cut into
    S = 8 runs: each sequence's own length (ceil(chunks / 8) chunks a run)
    against one common length (ceil(47 / 8) = 6 chunks a run, the tensor-core
    forward), under which sequences of at most 6 chunks stay whole and only
    the 47- and 7-chunk sequences are split (8 + 2 runs)."""
    import torch
    b = _bench()
    lens = [3000, 384, 385, 0, 1, 200]  # 47, 6, 7, 0, 1, 4 chunks
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    x = {"H": 2, "cu_seqlens": cu, "T": sum(lens), "B": 1}
    own = b.counts(x, 8)
    common = b.counts(x, 8, common=True)
    assert own["segments"] == 2 * (8 + 6 + 7 + 0 + 1 + 4)
    assert common["segments"] == 2 * (8 + 2)
    assert common["split_chunk_heads"] == 2 * (47 + 7)
    assert common["split_token_heads"] == 2 * (3000 + 385)
    assert own["split_chunk_heads"] == own["chunk_heads"] == 2 * 65
    assert b.counts(x, 1, common=True)["segments"] == 0
    # the states a composition touches: the split sequences' (common length)
    # or every non-empty one's (own length)
    assert common["split_seq_heads"] == 2 * 2
    assert own["split_seq_heads"] == 2 * 5
