"""Seeded input generators: determinism, shapes, rounding and keep-bit statistics."""

import numpy as np
import torch

import workloads


def test_named_workloads_shapes():
    shapes = {
        "tiny_varlen_fp16": (101, 2, 2, 64),
        "gqa_causal_bf16": (32768, 32, 8, 128),
        "window_dropout_bf16": (65536, 16, 4, 128),
        "long_causal_sink_bf16": (32768, 8, 8, 128),
    }
    for name, (t, nq, nkv, d) in shapes.items():
        wl = workloads.workload(name)
        assert (wl.tq, wl.nq, wl.nkv, wl.d) == (t, nq, nkv, d)
    wl = workloads.workload("causal_varlen_bf16")
    assert wl.batch == 8 and all(256 <= s <= 2048 for s in wl.seqlens_q)
    assert wl.seqlens_q == workloads.workload("causal_varlen_bf16").seqlens_q
    assert workloads.workload("window_dropout_bf16").mask_bits() == 8 * 16 * 8192 * 8192


def test_generation_is_deterministic():
    wl = workloads.workload("tiny_varlen_fp16")
    a, b = workloads.make_inputs(wl), workloads.make_inputs(wl)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.dy, b.dy)):
        assert x.dtype == np.float16 and np.array_equal(x, y)
    np.testing.assert_array_equal(a.q64, a.q.astype(np.float64))
    assert abs(float(a.q64.std()) - 1.0) < 0.05


def test_bf16_rounding_matches_torch_rne():
    x = np.random.default_rng(0).standard_normal(100000) * 10.0
    x = np.concatenate([x, [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0, -3.4e38, 1e-40]])
    bits, exact = workloads.round_to_dtype(x, "bf16")
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    np.testing.assert_array_equal(bits, ref.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(exact, ref.to(torch.float64).numpy())


def test_dropout_mask_statistics_and_layout():
    m = workloads.dropout_mask(7, 1_000_003, 0.9)
    assert m.size == (1_000_003 + 7) // 8
    frac = np.unpackbits(m, bitorder="little")[:1_000_003].mean()
    assert abs(frac - 0.9) < 0.002
    np.testing.assert_array_equal(m, workloads.dropout_mask(7, 1_000_003, 0.9, chunk_bits=4096))


def test_value_head_dim_and_generated_pse_inputs():
    """A value head dim below D shapes V and dY; a generated pse is fp32 slopes."""
    wl = workloads.custom("dv", "bf16", [5, 9], [5, 9], 4, 2, 64, dv=24, sparse_mode=3,
                          pse_kind="slopes", pse_batch=2, pse_type=2)
    inp = workloads.make_inputs(wl)
    assert wl.dv == 24 and inp.q.shape == (14, 4, 64) and inp.k.shape == (14, 2, 64)
    assert inp.v.shape == (14, 2, 24) and inp.dy.shape == (14, 4, 24)
    assert inp.pse.dtype == np.float32 and inp.pse.shape == (2, 4) and np.all(inp.pse > 0)
    np.testing.assert_array_equal(inp.pse64, inp.pse.astype(np.float64))
    shared = workloads.make_inputs(workloads.custom("dv1", "f16", [5], [5], 3, 1, 32, sparse_mode=2,
                                                    pse_kind="slopes", pse_batch=1, pse_type=3))
    assert shared.pse.shape == (3,) and shared.v.shape == (5, 1, 32)
