"""CPU checks of bench.py's host logic: the oracle leg's element-by-element
comparison of one decode step (out within 1e-2 + 1e-2 |ref|, lse within 1e-3),
reported in the JSON line and never fatal to it."""
import json

import numpy as np

import bench
import workloads
from parity import oracle_cache_after_append, oracle_decode


def _reference(inp):
    kc, vc = oracle_cache_after_append(inp)
    return oracle_decode(inp, kc, vc)


def test_matching_step_is_within_tolerance():
    inp = workloads.tiny_decode()
    ref_out, ref_lse = _reference(inp)
    res = bench._cpu_baseline(inp, 0.02, (ref_out.astype(np.float32), ref_lse.astype(np.float32)))
    assert res["kind"] == "oracle" and res["cores"] >= 1 and res["value"] > 0
    assert res["parity"]["within_tolerance"] is True
    assert res["parity"]["rows"] == inp.q.shape[0] * inp.q.shape[1]
    json.dumps(res, allow_nan=False)


def test_errors_and_nans_are_reported_as_outside_tolerance():
    inp = workloads.tiny_decode()
    ref_out, ref_lse = _reference(inp)
    off = ref_out.copy()
    off[0, 0, 0] += 2e-2 + 2e-2 * abs(off[0, 0, 0])
    assert bench._parity_summary((off, ref_lse), ref_out, ref_lse)["within_tolerance"] is False
    lse_off = ref_lse + 2e-3
    assert bench._parity_summary((ref_out, lse_off), ref_out, ref_lse)["within_tolerance"] is False
    nan = ref_out.copy()
    nan[1, 1, 1] = np.nan
    res = bench._parity_summary((nan, ref_lse), ref_out, ref_lse)
    assert res["within_tolerance"] is False
    json.dumps(res, allow_nan=False)  # NaN appears as text, the line stays strict JSON


def test_gpu_failure_is_carried_as_text():
    inp = workloads.tiny_decode()
    res = bench._cpu_baseline(inp, 0.02, "GPU step failed: RuntimeError('x')")
    assert res["parity"] == {"error": "GPU step failed: RuntimeError('x')"}
    assert "parity" not in bench._cpu_baseline(inp, 0.02)
