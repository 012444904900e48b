"""bench.py's parity summary of the sampled heads (no GPU): the reported
max-abs and rel-L2 and the verdict against the GPU tests' bound, on planted
errors."""

import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(spec)
spec.loader.exec_module(bench)


class _Wl:
    def __init__(self, dtype="bf16"):
        self.dtype = dtype


def _refs(rng):
    return {h: {"o": rng.standard_normal((1, 1, 40, 8)), "lse": rng.standard_normal(40),
                "dq": rng.standard_normal((1, 1, 40, 8)), "dk": rng.standard_normal((1, 1, 40, 8)),
                "dv": rng.standard_normal((1, 1, 40, 8))} for h in range(2)}


def test_exact_results_are_within_the_bound():
    rng = np.random.default_rng(0)
    refs = _refs(rng)
    bench._GPU_SAMPLES.clear()
    bench._GPU_SAMPLES.update({h: {n: a.copy() for n, a in r.items()} for h, r in refs.items()})
    out = bench.sample_parity(_Wl(), refs)
    assert out["within_test_bound"] and out["heads"] == [0, 1]
    assert all(out[n]["max_abs"] == 0.0 and out[n]["rel_l2"] == 0.0 for n in ("o", "lse", "dq", "dk", "dv"))


def test_a_planted_error_is_reported_and_fails_the_bound():
    rng = np.random.default_rng(1)
    refs = _refs(rng)
    bench._GPU_SAMPLES.clear()
    bench._GPU_SAMPLES.update({h: {n: a.copy() for n, a in r.items()} for h, r in refs.items()})
    bench._GPU_SAMPLES[1]["dq"][0, 0, 7, 3] += 0.5  # far beyond 2e-2 + half an ulp
    out = bench.sample_parity(_Wl(), refs)
    assert not out["within_test_bound"]
    assert abs(out["dq"]["max_abs"] - 0.5) < 1e-12
    assert out["o"]["max_abs"] == 0.0


def test_rounding_to_bfloat16_stays_within_the_bound():
    rng = np.random.default_rng(2)
    refs = _refs(rng)
    bench._GPU_SAMPLES.clear()
    for h, r in refs.items():
        d = {}
        for n, a in r.items():
            # round to 8 significant bits (bfloat16), the device outputs' precision
            m, e = np.frexp(a)
            d[n] = np.ldexp(np.round(m * 256) / 256, e)
        bench._GPU_SAMPLES[h] = d
    out = bench.sample_parity(_Wl(), refs)
    assert out["within_test_bound"]
    assert 0 < out["o"]["max_abs"] <= 2.0 ** -8 * max(np.abs(r["o"]).max() for r in refs.values())


def test_fully_masked_rows_compare_their_infinities():
    rng = np.random.default_rng(3)
    refs = _refs(rng)
    for r in refs.values():
        r["lse"][5] = -np.inf
    bench._GPU_SAMPLES.clear()
    bench._GPU_SAMPLES.update({h: {n: a.copy() for n, a in r.items()} for h, r in refs.items()})
    assert bench.sample_parity(_Wl(), refs)["within_test_bound"]
    bench._GPU_SAMPLES[0]["lse"][5] = 0.0  # a finite LSE where the oracle has none
    assert not bench.sample_parity(_Wl(), refs)["within_test_bound"]
