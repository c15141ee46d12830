"""Host logic of bench.py's CPU-oracle record (no GPU): cutting a workload
into independent units and reassembling the units' oracle results gives the
whole-workload oracle result bit for bit, and the two error metrics are the
ones the record states."""
import numpy as np
import pytest

import bench
import oracle
import synth


def _assemble(job):
    ref, secs = job.reference(threads=3)
    assert secs >= 0
    return ref


@pytest.mark.parametrize("T", [1, 37])
def test_scan_units_reassemble_the_whole_oracle_result(T):
    x = synth.scan_inputs(3, T, 300, large=True, cid=41)
    a, b, u, s0 = (x[n].numpy() for n in ("a", "b", "u", "s0"))
    job = bench.scan_job(a, {"fma": b, "gated": u}, s0)
    ref = _assemble(job)
    for form, rhs, fn in (("fma", b, oracle.scan_fma), ("gated", u, oracle.scan_gated)):
        so, sf = fn(a, rhs, s0.astype(np.float64))
        assert np.array_equal(ref[f"s_{form}"], so) and np.array_equal(ref[f"s_final_{form}"], sf)
    assert job.nbytes == 2 * bench.scan_bytes(3, T, 300)


@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "rwkv7"])
@pytest.mark.parametrize("T", [1, 9])
def test_matrix_units_reassemble_the_whole_oracle_result(kind, T):
    B, H = 3, 4
    if kind == "gla":
        x = synth.gla_inputs(B, T, H, 64, 64, cid=42)
        xh = dict(q=x["q"], k=x["k"], v=x["v"], g=x["d"], decay_kind=x["decay_kind"], scale=x["scale"])
        G, mk = H, "diag"
    elif kind == "mamba2":
        x = synth.mamba2_inputs(B, T, H, 2, 64, 64, cid=43)
        xh = dict(q=x["q"], k=x["k"], v=x["v"], g=x["d"], decay_kind=x["decay_kind"], scale=x["scale"])
        G, mk = 2, "diag"
    elif kind == "delta":
        x = synth.deltanet_inputs(B, T, H, 64, 64, cid=44)
        xh = dict(q=x["q"], k=x["k"], v=x["v"], g=x["beta"], scale=x["scale"])
        G, mk = H, "delta"
    else:
        x = synth.rwkv7_inputs(B, T, H, 64, 64, random_state=True, cid=45)
        xh = dict(q=x["q"], k=x["k"], v=x["v"], g=x["w"], S0=x["S0"])
        G, mk = H, "rwkv7"
    xh = {k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in xh.items()}
    job = bench.matrix_job(mk, xh, B, T, H, 64, 64, nbytes=1, G=G)
    ref = _assemble(job)
    S0 = None if xh.get("S0") is None else xh["S0"].astype(np.float64)
    if mk == "diag":
        o, S = oracle.recur_diag(xh["q"], xh["k"], xh["v"], xh["g"], S0, H=H, G=G, decay_kind=xh["decay_kind"],
                                 scale=xh["scale"])
    elif mk == "delta":
        o, S = oracle.recur_delta(xh["q"], xh["k"], xh["v"], xh["g"], S0, scale=xh["scale"])
    else:
        o, S = oracle.recur_rwkv7(xh["q"], xh["k"], xh["v"], xh["g"], S0)
    assert np.array_equal(ref["o"], o) and np.array_equal(ref["S"], S)
    assert job.tok_heads == B * T * H


def test_error_metrics():
    r = np.array([1.0, -2.0, 0.0, 4.0])
    y = r + np.array([0.0, 0.01, 0.002, -0.04])
    nw, ew = bench.err_pair(y, r)
    assert nw == pytest.approx(0.04 / 4.0)
    # elementwise: |dy| / max(|r|, 1e-3 * 4): the zero reference entry uses the floor 0.004
    assert ew == pytest.approx(max(0.01 / 2.0, 0.002 / 0.004, 0.04 / 4.0))
    rec = bench.errors({"s": y}, {"s": r}, tol=0.02)
    assert rec["within_tolerance"] and rec["err_normwise"]["s"] == pytest.approx(0.01)
    assert not bench.errors({"s": y}, {"s": r}, tol=0.001)["within_tolerance"]


def test_cpu_record_reports_all_four_figures():
    x = synth.scan_inputs(2, 16, 256, large=True, cid=46)
    a, b, u, s0 = (x[n].numpy() for n in ("a", "b", "u", "s0"))
    rec, ref = bench.cpu_record(bench.scan_job(a, {"fma": b, "gated": u}, s0), reps_1t=2)
    for key in ("cpu_fp64_all", "cpu_fp32_all", "cpu_fp64_1t", "cpu_fp32_1t"):
        assert rec[key]["GBps"] > 0 and rec[key]["cpu_model"]
    assert rec["cpu_fp64_all"]["threads"] == min(4, bench.host_cores())
    assert rec["cpu_fp64_1t"]["threads"] == 1
    assert set(ref) == {"s_fma", "s_final_fma", "s_gated", "s_final_gated"}
