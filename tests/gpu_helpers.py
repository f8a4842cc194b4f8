"""Shared helpers of the GPU parity tests: upload seeded inputs, run the
library's forward and gradient through the C ABI, compute oracle references
and compare element by element."""

from __future__ import annotations

import numpy as np
import torch

import attention_backward_tnd_b300 as tnd
import oracle
import workloads

TORCH_DTYPE = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def to_device(arr: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(arr.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(arr).cuda()


def upload(inp: workloads.Inputs):
    wl = inp.wl
    dev = {n: to_device(getattr(inp, n), wl.dtype) for n in ("q", "k", "v", "dy")}
    dev["sink"] = None if inp.sink is None else torch.from_numpy(inp.sink).cuda()
    dev["mask"] = None if inp.mask is None else torch.from_numpy(inp.mask).cuda()
    return dev


def run_library(inp: workloads.Inputs, dev=None, grad_path: int = 0):
    """Forward then gradient through the library; returns device tensors."""
    wl = inp.wl
    dev = dev or upload(inp)
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, grad_path) == tnd.TND_OK
    try:
        out, smax, ssum = tnd.fwd(dev["q"], dev["k"], dev["v"], wl.cu_q, wl.cu_kv, wl.scale, wl.keep_prob,
                                  wl.pre_tokens, wl.next_tokens, wl.sparse_mode, dev["mask"], dev["sink"])
        ws_bytes = tnd.grad_workspace_bytes(dev["q"], dev["k"], wl.cu_q, wl.cu_kv, wl.scale, wl.keep_prob,
                                            wl.pre_tokens, wl.next_tokens, wl.sparse_mode,
                                            dev["mask"] is not None, dev["sink"] is not None)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        dq, dk, dv, dsink = tnd.grad(dev["q"], dev["k"], dev["v"], dev["dy"], out, smax, ssum, wl.cu_q,
                                     wl.cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens, wl.next_tokens,
                                     wl.sparse_mode, dev["mask"], dev["sink"], workspace=ws)
        torch.cuda.synchronize()
        st = tnd.device_status(ws)
        assert st == tnd.TND_OK, f"device status {st}: {tnd.tnd_status_string(st)}"
    finally:
        tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, 0)
    return {"out": out, "smax": smax, "ssum": ssum, "dq": dq, "dk": dk, "dv": dv, "dsink": dsink, "ws": ws}


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_problem(inp: workloads.Inputs, **kw) -> oracle.Problem:
    return oracle.problem_from_workload(inp.wl, drop_mask=inp.mask, sink=inp.sink, **kw)


def oracle_reference(inp: workloads.Inputs, **kw):
    """End-to-end oracle (its own fp64 forward) on the exact stored inputs."""
    p = oracle_problem(inp, **kw)
    out, smax, ssum, dq, dk, dv, dsink = oracle.fwd_grad(p, inp.q64, inp.k64, inp.v64, inp.dy64)
    return {"out": out, "smax": smax, "ssum": ssum, "dq": dq, "dk": dk, "dv": dv, "dsink": dsink}


def tolerance(dtype: str, ref: np.ndarray):
    """Per-element bound: bf16/fp16 |err| <= 1e-2 + 2e-2|ref|; fp32 relative
    1e-4, with an absolute floor of 1e-5 x the tensor's RMS for elements whose
    reference nearly cancels (fp32 sums of O(1) terms carry ~1e-7 absolute
    error however small the result)."""
    if dtype in ("bf16", "f16"):
        return 1e-2 + 2e-2 * np.abs(ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return 1e-4 * np.abs(ref) + 1e-5 * max(rms, 1e-30)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str, mask=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    if got.size == 0:
        return 0.0
    err = np.abs(got - ref)
    tol = tolerance(dtype, ref)
    bad = ~(err <= tol)
    maxnorm = float(np.nanmax(err)) if not np.isnan(err).all() else float("nan")
    if bad.any():
        ratio = np.where(np.isnan(err), np.inf, err / tol).reshape(-1)
        w = int(np.argmax(ratio))
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} elements out of tolerance; max |err| "
                             f"{maxnorm:.3e}; worst at flat {w}: got {got.reshape(-1)[w]:.6g}, ref "
                             f"{ref.reshape(-1)[w]:.6g}, tol {tol.reshape(-1)[w]:.3e}")
    return maxnorm


def stat_lanes_equal(t: torch.Tensor) -> bool:
    h = t.cpu()
    finite = torch.isfinite(h[..., :1])
    same = (h == h[..., :1]) | (~torch.isfinite(h) & ~torch.isfinite(h[..., :1]))
    return bool(same.all()) and finite.numel() > 0


def compare_all(inp: workloads.Inputs, got: dict, ref: dict, q_rows=None, kv_rows=None, heads=None):
    """Compare forward and gradient outputs; q_rows / kv_rows / heads select
    the part the oracle computed (numpy boolean masks over T and N)."""
    wl = inp.wl
    nq, nkv, g = wl.nq, wl.nkv, wl.nq // wl.nkv
    hsel = np.zeros(nq, bool)
    if heads is None:
        hsel[:] = True
    else:
        hsel[heads[0]:heads[1]] = True
    gsel = np.zeros(nkv, bool)
    gsel[np.unique(np.nonzero(hsel)[0] // g)] = True
    qm = np.ones(wl.tq, bool) if q_rows is None else q_rows
    km = np.ones(wl.tkv, bool) if kv_rows is None else kv_rows
    qsel = qm[:, None] & hsel[None, :]
    ksel = km[:, None] & gsel[None, :]
    res = {}
    out = host64(got["out"])
    res["out"] = assert_close(out, ref["out"], wl.dtype, "attention_out", qsel[..., None].repeat(wl.d, -1))
    smax = got["smax"].cpu().numpy().astype(np.float64)
    ssum = got["ssum"].cpu().numpy().astype(np.float64)
    assert stat_lanes_equal(got["smax"]) and stat_lanes_equal(got["ssum"])
    fin = np.isfinite(ref["smax"]) & qsel
    assert np.array_equal(np.isfinite(smax[..., 0]) & qsel, fin), "softmax_max finiteness"
    assert_close(smax[..., 0], ref["smax"], "f32", "softmax_max", fin)
    np.testing.assert_allclose(ssum[..., 0][qsel], ref["ssum"][qsel], rtol=2e-5, atol=1e-6)
    res["dq"] = assert_close(host64(got["dq"]), ref["dq"], wl.dtype, "dq", qsel[..., None].repeat(wl.d, -1))
    res["dk"] = assert_close(host64(got["dk"]), ref["dk"], wl.dtype, "dk", ksel[..., None].repeat(wl.d, -1))
    res["dv"] = assert_close(host64(got["dv"]), ref["dv"], wl.dtype, "dv", ksel[..., None].repeat(wl.d, -1))
    if got["dsink"] is not None:
        ds = got["dsink"].cpu().numpy().astype(np.float64)
        res["dsink"] = assert_close(ds, ref["dsink"], "bf16" if wl.dtype != "f32" else "f32", "dsink", hsel)
    return res
