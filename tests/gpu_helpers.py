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
    dev["amask"] = None if inp.amask is None else torch.from_numpy(inp.amask).cuda()
    if inp.pse is None:
        dev["pse"] = None
    elif wl.pse_kind == "slopes":            # fp32 slopes of a generated pse (pseType 2 / 3)
        dev["pse"] = torch.from_numpy(inp.pse).cuda()
    else:
        dev["pse"] = to_device(inp.pse, wl.dtype)
    return dev


def run_library(inp: workloads.Inputs, dev=None, grad_path: int = 0, deterministic: bool = True):
    """Forward then gradient through the library; returns device tensors."""
    wl = inp.wl
    dev = dev or upload(inp)
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, grad_path) == tnd.TND_OK
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, int(deterministic)) == tnd.TND_OK
    try:
        amask, pse = dev.get("amask"), dev.get("pse")
        out, smax, ssum = tnd.fwd(dev["q"], dev["k"], dev["v"], wl.cu_q, wl.cu_kv, wl.scale, wl.keep_prob,
                                  wl.pre_tokens, wl.next_tokens, wl.sparse_mode, dev["mask"], dev["sink"],
                                  atten_mask=amask, prefix=wl.prefix, pse=pse, pse_type=wl.pse_type)
        ws_bytes = tnd.grad_workspace_bytes(dev["q"], dev["k"], wl.cu_q, wl.cu_kv, wl.scale, wl.keep_prob,
                                            wl.pre_tokens, wl.next_tokens, wl.sparse_mode,
                                            dev["mask"] is not None, dev["sink"] is not None,
                                            amask is not None, wl.prefix, v=dev["v"])
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        dq, dk, dv, dsink = tnd.grad(dev["q"], dev["k"], dev["v"], dev["dy"], out, smax, ssum, wl.cu_q,
                                     wl.cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens, wl.next_tokens,
                                     wl.sparse_mode, dev["mask"], dev["sink"], workspace=ws,
                                     atten_mask=amask, prefix=wl.prefix, pse=pse, pse_type=wl.pse_type)
        torch.cuda.synchronize()
        st = tnd.device_status(ws)
        assert st == tnd.TND_OK, f"device status {st}: {tnd.tnd_status_string(st)}"
    finally:
        tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, 0)
        tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, 1)
    return {"out": out, "smax": smax, "ssum": ssum, "dq": dq, "dk": dk, "dv": dv, "dsink": dsink, "ws": ws}


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_problem(inp: workloads.Inputs, **kw) -> oracle.Problem:
    return oracle.problem_from_workload(inp.wl, drop_mask=inp.mask, sink=inp.sink, atten_mask=inp.amask,
                                        prefix=inp.wl.prefix, pse=inp.pse64, pse_type=inp.wl.pse_type, **kw)


def oracle_reference(inp: workloads.Inputs, **kw):
    """End-to-end oracle (its own fp64 forward) on the exact stored inputs."""
    p = oracle_problem(inp, **kw)
    out, smax, ssum, dq, dk, dv, dsink = oracle.fwd_grad(p, inp.q64, inp.k64, inp.v64, inp.dy64)
    return {"out": out, "smax": smax, "ssum": ssum, "dq": dq, "dk": dk, "dv": dv, "dsink": dsink}


U32 = 2.0 ** -24          # unit roundoff of fp32
EPS_APPROX = 2.0 ** -21   # bound used for the relative error of ex2.approx / lg2.approx.f32 (PTX ISA: ~2 ulp)


def gamma(n):
    """gamma_n = n u / (1 - n u): the standard bound on the relative error of an
    n-term fp32 sum or dot product (|fl(x.y) - x.y| <= gamma_n sum |x_i y_i|)."""
    nu = np.asarray(n, dtype=np.float64) * U32
    return nu / (1.0 - nu)


def pse_matrix(p, b, h, sq, skv):
    """The [sq, skv] pse of (sequence b, head h) as the oracle reads it (zeros without one)."""
    if p.pse is None:
        return np.zeros((sq, skv))
    return np.array([[oracle.pse_at(p, b, h, i, j) for j in range(skv)] for i in range(sq)]).reshape(sq, skv)


def pse_logit(wl, qk, pse):
    """Scores from Q K^T and the pse, in the pse type's order."""
    return wl.scale * (qk + pse) if wl.pse_type == 1 else wl.scale * qk + pse


def fp32_error_bound(inp: workloads.Inputs, ref: dict) -> dict:
    """First-order bound, per output element, on the rounding error of any
    fp32 evaluation of the forward and gradient of this problem.

    Each sum of the method gets the dot-product bound gamma_n * (sum of the
    absolute values of its terms), each exp2 / log2 the fast-approximation
    error EPS_APPROX, each product or subtraction one rounding u; errors are
    carried forward through P, O, D, dP, dS to dQ, dK, dV and dSink.  Inputs
    are the exact stored values, so the arithmetic is the only error source.
    The sum of first-order terms is doubled to cover second-order ones.
    Only for small problems: it forms the dense Sq x Skv matrices."""
    wl = inp.wl
    g = wl.nq // wl.nkv
    d = wl.d
    out = {n: np.zeros_like(ref[n]) for n in ("out", "dq", "dk", "dv")}
    out["dsink"] = np.zeros(wl.nq)
    p = oracle_problem(inp)
    for b in range(wl.batch):
        sq, skv = wl.seqlens_q[b], wl.seqlens_kv[b]
        if sq == 0 or skv == 0:
            continue
        q0, k0 = wl.cu_q[b], wl.cu_kv[b]
        keep = np.array([[oracle.keep_at(p, b, i, j) for j in range(skv)] for i in range(sq)],
                        dtype=bool).reshape(sq, skv)
        nk = keep.sum(axis=1) + (1 if inp.sink is not None else 0)
        base = p.mask_base(b)
        for h in range(wl.nq):
            kv = h // g
            Q, dY = inp.q64[q0:q0 + sq, h], inp.dy64[q0:q0 + sq, h]
            K, V = inp.k64[k0:k0 + skv, kv], inp.v64[k0:k0 + skv, kv]
            O = ref["out"][q0:q0 + sq, h]
            m, l = ref["smax"][q0:q0 + sq, h], ref["ssum"][q0:q0 + sq, h]
            if inp.mask is not None:
                idx = base + (h * sq + np.arange(sq))[:, None] * skv + np.arange(skv)[None, :]
                bits = (inp.mask[idx >> 3] >> (idx & 7)) & 1
                Z = bits / wl.keep_prob
            else:
                Z = np.ones((sq, skv))
            live = l > 0
            PSE = pse_matrix(p, b, h, sq, skv)
            S = pse_logit(wl, Q @ K.T, PSE)
            # |terms| of the score sum; the pse is one more term (one more rounding)
            Sabs = pse_logit(wl, np.abs(Q) @ np.abs(K).T, np.abs(PSE))
            P = np.where(keep & live[:, None], np.exp(S - np.where(live, m, 0)[:, None])
                         / np.where(live, l, 1)[:, None], 0.0)
            smax_abs = np.where(keep, Sabs, 0).max(axis=1)
            epsP = 3 * gamma(d) * smax_abs + 2 * gamma(nk) + 4 * EPS_APPROX + 8 * U32
            PZ = P * np.abs(Z)
            errO = (PZ * (epsP + gamma(nk))[:, None]) @ np.abs(V)
            D = np.sum(dY * O, axis=1)
            errD = gamma(d) * np.sum(np.abs(dY * O), axis=1) + np.sum(np.abs(dY) * errO, axis=1)
            dP = dY @ V.T
            dPabs = np.abs(dY) @ np.abs(V).T
            dS = P * (Z * dP - D[:, None])
            errdS = np.abs(dS) * (epsP + 2 * U32)[:, None] + P * (np.abs(Z) * gamma(d) * dPabs + errD[:, None])
            out["out"][q0:q0 + sq, h] += errO
            out["dq"][q0:q0 + sq, h] += wl.scale * ((errdS + gamma(nk)[:, None] * np.abs(dS)) @ np.abs(K)) \
                + U32 * np.abs(ref["dq"][q0:q0 + sq, h])
            nm = g * sq
            out["dk"][k0:k0 + skv, kv] += wl.scale * ((errdS + gamma(nm) * np.abs(dS)).T @ np.abs(Q))
            out["dv"][k0:k0 + skv, kv] += (PZ * (epsP + gamma(nm))[:, None]).T @ np.abs(dY)
            if inp.sink is not None:
                ps = np.where(live, np.exp(float(inp.sink[h]) - np.where(live, m, 0)) / np.where(live, l, 1), 0.0)
                out["dsink"][h] += np.sum(ps * (np.abs(D) * (epsP + gamma(wl.tq)) + errD))
    for n in ("out", "dq", "dk", "dv", "dsink"):
        out[n] *= 2.0
    out["dk"] += U32 * np.abs(ref["dk"])
    return out


def plain_fp32_eval(inp: workloads.Inputs) -> dict:
    """Textbook fp32 evaluation of the forward and gradient with torch on the
    CPU (float32 throughout, dense masked softmax): the accuracy yardstick
    for the fp32 path.  Small problems only."""
    wl = inp.wl
    g = wl.nq // wl.nkv
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).float()  # noqa: E731
    q, k, v, dy = t(inp.q64), t(inp.k64), t(inp.v64), t(inp.dy64)
    out = torch.zeros_like(dy)   # value head dim
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    dsink = torch.zeros(wl.nq)
    p = oracle_problem(inp)
    for b in range(wl.batch):
        sq, skv = wl.seqlens_q[b], wl.seqlens_kv[b]
        q0, k0 = wl.cu_q[b], wl.cu_kv[b]
        keep = torch.tensor(np.array([[oracle.keep_at(p, b, i, j) for j in range(skv)] for i in range(sq)],
                                     dtype=bool).reshape(sq, skv))
        base = p.mask_base(b)
        for h in range(wl.nq):
            kv = h // g
            Q, dY = q[q0:q0 + sq, h], dy[q0:q0 + sq, h]
            K, V = k[k0:k0 + skv, kv], v[k0:k0 + skv, kv]
            PSE = torch.from_numpy(pse_matrix(p, b, h, sq, skv)).float()
            S = (Q @ K.T + PSE) * wl.scale if wl.pse_type == 1 else (Q @ K.T) * wl.scale + PSE
            S = torch.where(keep, S, torch.tensor(-float("inf")))
            m = S.max(dim=1).values
            if inp.sink is not None:
                m = torch.maximum(m, torch.tensor(float(inp.sink[h])))
            m = torch.where(torch.isfinite(m), m, torch.zeros_like(m))   # rows that keep nothing
            E = torch.exp(S - m[:, None])
            l = E.sum(dim=1) + (torch.exp(torch.tensor(float(inp.sink[h])) - m) if inp.sink is not None else 0)
            P = E / torch.where(l > 0, l, torch.ones_like(l))[:, None]
            if inp.mask is not None:
                idx = base + (h * sq + np.arange(sq))[:, None] * skv + np.arange(skv)[None, :]
                Z = torch.from_numpy(((inp.mask[idx >> 3] >> (idx & 7)) & 1) / wl.keep_prob).float()
            else:
                Z = torch.ones(sq, skv)
            O = (P * Z) @ V
            out[q0:q0 + sq, h] = O
            D = (dY * O).sum(dim=1)
            dS = P * (Z * (dY @ V.T) - D[:, None])
            dq[q0:q0 + sq, h] = (dS @ K) * wl.scale
            dk[k0:k0 + skv, kv] += (dS.T @ Q) * wl.scale
            dv[k0:k0 + skv, kv] += (P * Z).T @ dY
            if inp.sink is not None:
                dsink[h] += -(torch.exp(torch.tensor(float(inp.sink[h])) - m) / l * D).sum()
    return {n: x.double().numpy() for n, x in dict(out=out, dq=dq, dk=dk, dv=dv, dsink=dsink).items()}


def operand_rounding_bound(inp: workloads.Inputs, ref: dict) -> dict:
    """Per-element bound on what the tensor cores' 16-bit operands add to dQ,
    dK and dV.  Before the UMMAs dS (and P z, for dV) are rounded to the input
    dtype (unit roundoff 2^-8 for bf16, 2^-11 for fp16), so to first order an
    element moves by at most that roundoff times the sum of the absolute
    values of its terms: scale sum_j |dS_ij||K_j| for dQ_i, scale sum
    |dS_ij||Q_i| for dK_j and sum |P_ij z_ij||dY_i| for dV_j, over the kv
    head's query heads; the result is doubled to cover the fp32 work around
    the rounding.  The bf16 bar's absolute floor (1e-2) does not grow
    with the number of terms, which is G * Sq for dK and dV: with many query
    heads per kv head a few elements exceed the bar from this rounding alone.
    Small problems only (dense Sq x Skv matrices)."""
    wl = inp.wl
    u = 2.0 ** -8 if wl.dtype == "bf16" else 2.0 ** -11
    g = wl.nq // wl.nkv
    out = {n: np.zeros_like(ref[n]) for n in ("dq", "dk", "dv")}
    p = oracle_problem(inp)
    for b in range(wl.batch):
        sq, skv = wl.seqlens_q[b], wl.seqlens_kv[b]
        if sq == 0 or skv == 0:
            continue
        q0, k0 = wl.cu_q[b], wl.cu_kv[b]
        keep = np.array([[oracle.keep_at(p, b, i, j) for j in range(skv)] for i in range(sq)],
                        dtype=bool).reshape(sq, skv)
        base = p.mask_base(b)
        for h in range(wl.nq):
            kv = h // g
            Q, dY = inp.q64[q0:q0 + sq, h], inp.dy64[q0:q0 + sq, h]
            K, V = inp.k64[k0:k0 + skv, kv], inp.v64[k0:k0 + skv, kv]
            m, l = ref["smax"][q0:q0 + sq, h], ref["ssum"][q0:q0 + sq, h]
            S = pse_logit(wl, Q @ K.T, pse_matrix(p, b, h, sq, skv))
            live = (l > 0)[:, None] & keep
            P = np.where(live, np.exp(np.where(live, S, 0.0) - np.where(l > 0, m, 0.0)[:, None]), 0.0)
            P = P / np.where(l > 0, l, 1.0)[:, None]
            if inp.mask is not None:
                idx = base + (h * sq + np.arange(sq))[:, None] * skv + np.arange(skv)[None, :]
                Z = ((inp.mask[idx >> 3] >> (idx & 7)) & 1) / wl.keep_prob
            else:
                Z = np.ones((sq, skv))
            D = np.sum(dY * ref["out"][q0:q0 + sq, h], axis=1)
            dS = np.abs(P * (Z * (dY @ V.T) - D[:, None]))
            out["dq"][q0:q0 + sq, h] += wl.scale * dS @ np.abs(K)
            out["dk"][k0:k0 + skv, kv] += wl.scale * dS.T @ np.abs(Q)
            out["dv"][k0:k0 + skv, kv] += (P * Z).T @ np.abs(dY)
    return {n: 2.0 * u * x for n, x in out.items()}


def tolerance(dtype: str, ref: np.ndarray, bound=None):
    """Per-element bound.  bf16/fp16: |err| <= 1e-2 + 2e-2|ref|.  fp32: 1e-4
    relative, plus the fp32 rounding bound of that element (fp32_error_bound)
    for elements whose reference nearly cancels: a relative bound alone
    cannot hold where the exact result is far smaller than its terms."""
    if dtype in ("bf16", "f16"):
        # the stated bar; plus, where a caller passes one, the operand-rounding
        # bound of operand_rounding_bound
        return 1e-2 + 2e-2 * np.abs(ref) + (0.0 if bound is None else bound)
    assert bound is not None, "fp32 comparisons need the element-wise rounding bound"
    return 1e-4 * np.abs(ref) + bound


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str, mask=None, bound=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if bound is not None:
        bound = np.broadcast_to(np.asarray(bound, dtype=np.float64), ref.shape)
    if mask is not None:
        got, ref = got[mask], ref[mask]
        bound = None if bound is None else bound[mask]
    if got.size == 0:
        return 0.0
    err = np.abs(got - ref)
    if dtype == "f32":
        # "1e-4 relative" read for the tensor as a whole (norm-wise) ...
        nrm = float(np.linalg.norm(ref))
        assert float(np.linalg.norm(err)) <= 1e-4 * nrm or nrm == 0.0, (
            f"{what}: norm-wise relative error {np.linalg.norm(err) / nrm:.3e} > 1e-4")
    # ... and element by element with the rounding bound where the result cancels
    tol = tolerance(dtype, ref, bound)
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


def smax_bound(inp: workloads.Inputs, ref_smax: np.ndarray) -> np.ndarray:
    """Rounding bound of the forward's softmax max m_i: every logit is an
    fp32 dot product of length D (|error| <= gamma_D scale sum|q||k| <=
    gamma_D scale ||q_i|| ||k_j|| by Cauchy-Schwarz), plus a few roundings
    of the log2 / natural-log unit changes; doubled like fp32_error_bound."""
    wl = inp.wl
    g = wl.nq // wl.nkv
    qn = np.linalg.norm(inp.q64, axis=2)                    # [Tq, Nq]
    kn = np.linalg.norm(inp.k64, axis=2)                    # [Tkv, Nkv]
    bound = np.zeros((wl.tq, wl.nq))
    for b in range(wl.batch):
        q0, q1, k0, k1 = wl.cu_q[b], wl.cu_q[b + 1], wl.cu_kv[b], wl.cu_kv[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        kmax = kn[k0:k1].max(axis=0)                       # [Nkv]
        bound[q0:q1] = wl.scale * qn[q0:q1] * np.repeat(kmax, g)[None, :]
    m = np.where(np.isfinite(ref_smax), np.abs(ref_smax), 0.0)
    return 2.0 * (gamma(wl.d + 2) * bound + 4 * U32 * m)


def ssum_rtol(inp: workloads.Inputs, ref_smax: np.ndarray) -> np.ndarray:
    """Relative rounding bound of the forward's softmax sum l_i: a sum of at
    most Skv_b + 1 positive fp32 terms (|error| <= gamma_n times the sum, in
    any order), each exp(s - m) off by the logit and max errors (smax_bound,
    twice) and the ex2 approximation; doubled like the others."""
    wl = inp.wl
    n = np.zeros((wl.tq, wl.nq))
    for b in range(wl.batch):
        n[wl.cu_q[b]:wl.cu_q[b + 1]] = wl.seqlens_kv[b] + 2
    return 2.0 * (gamma(n) + 2.0 * smax_bound(inp, ref_smax) + 4 * EPS_APPROX)


def compare_all(inp: workloads.Inputs, got: dict, ref: dict, q_rows=None, kv_rows=None, heads=None,
                operand_rounding: bool = False):
    """Compare forward and gradient outputs; q_rows / kv_rows / heads select
    the part the oracle computed (numpy boolean masks over T and N).  fp32
    problems are compared with their element-wise rounding bound, which is
    only formed for small problems.  operand_rounding (16-bit dtypes, small
    problems) widens the dQ / dK / dV bar by operand_rounding_bound."""
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
    bnd = fp32_error_bound(inp, ref) if wl.dtype == "f32" else \
        (operand_rounding_bound(inp, ref) if operand_rounding else {})
    res = {}
    out = host64(got["out"])
    res["out"] = assert_close(out, ref["out"], wl.dtype, "attention_out", qsel[..., None].repeat(wl.dv, -1),
                              bnd.get("out"))
    smax = got["smax"].cpu().numpy().astype(np.float64)
    ssum = got["ssum"].cpu().numpy().astype(np.float64)
    assert stat_lanes_equal(got["smax"]) and stat_lanes_equal(got["ssum"])
    fin = np.isfinite(ref["smax"]) & qsel
    assert np.array_equal(np.isfinite(smax[..., 0]) & qsel, fin), "softmax_max finiteness"
    assert_close(smax[..., 0], ref["smax"], "f32", "softmax_max", fin, smax_bound(inp, ref["smax"]))
    l_tol = ssum_rtol(inp, ref["smax"]) * np.abs(ref["ssum"]) + 1e-6
    l_bad = qsel & ~(np.abs(ssum[..., 0] - ref["ssum"]) <= l_tol)
    assert not l_bad.any(), f"softmax_sum: {int(l_bad.sum())} rows out of their rounding bound"
    res["dq"] = assert_close(host64(got["dq"]), ref["dq"], wl.dtype, "dq", qsel[..., None].repeat(wl.d, -1),
                             bnd.get("dq"))
    res["dk"] = assert_close(host64(got["dk"]), ref["dk"], wl.dtype, "dk", ksel[..., None].repeat(wl.d, -1),
                             bnd.get("dk"))
    res["dv"] = assert_close(host64(got["dv"]), ref["dv"], wl.dtype, "dv", ksel[..., None].repeat(wl.dv, -1),
                             bnd.get("dv"))
    if got["dsink"] is not None:
        ds = got["dsink"].cpu().numpy().astype(np.float64)
        res["dsink"] = assert_close(ds, ref["dsink"], "bf16" if wl.dtype != "f32" else "f32", "dsink", hsel,
                                    bnd.get("dsink"))
    return res
