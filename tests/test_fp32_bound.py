"""The fp32 tolerance of the GPU parity tests is a derived rounding bound
(tests/gpu_helpers.fp32_error_bound).  Checked here on the CPU: a plain fp32
evaluation of the forward and gradient (torch, float32 throughout, textbook
formulas) must lie within it, and a planted error of a few per cent in one
element must not."""

import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")

from tests import gpu_helpers as gh  # noqa: E402

INF = 2147483647


CASES = {
    "fp32_causal_d64": ("f32", [70, 33], 2, 1, 64, 3, INF, INF, 1.0, False),
    "fp32_band_dropout_sink_d128": ("f32", [140, 65], 2, 2, 128, 4, 30, 5, 0.75, True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_plain_fp32_evaluation_lies_within_the_bound(name):
    dt, sq, nq, nkv, d, mode, pre, nxt, keep, sink = CASES[name]
    wl = workloads.custom(name, dt, sq, sq, nq, nkv, d, keep_prob=keep, pre_tokens=pre, next_tokens=nxt,
                          sparse_mode=mode, has_sink=sink, seed=777)
    inp = workloads.make_inputs(wl)
    ref = gh.oracle_reference(inp)
    bnd = gh.fp32_error_bound(inp, ref)
    got = gh.plain_fp32_eval(inp)
    for n in ("out", "dq", "dk", "dv") + (("dsink",) if sink else ()):
        gh.assert_close(got[n], ref[n], "f32", n, bound=bnd[n])
    # a planted 2 % error in one sizeable element is caught
    bad = got["dq"].copy()
    w = np.unravel_index(np.argmax(np.abs(ref["dq"])), bad.shape)
    bad[w] *= 1.02
    with pytest.raises(AssertionError):
        gh.assert_close(bad, ref["dq"], "f32", "dq", bound=bnd["dq"])
