"""Independent references used to pin the fp64 oracle (CPU only).

Nothing here calls the oracle's arithmetic: masks are built from numpy's
triangle routines, the attention forward is the textbook softmax written with
torch fp64 ops, and gradients come from torch autograd.
"""

from __future__ import annotations

import math

import numpy as np
import torch


def mask_matrix(mode: int, pre: int, nxt: int, sq: int, skv: int, atten_mask=None,
                prefix_n: int = 0) -> np.ndarray:
    """Explicit keep matrix [sq, skv] built from the verbal definitions of
    sparseMode, attenMaskOptional and prefixOptional
    (aclnnFlashAttentionUnpaddingScoreGrad, parameters section)."""
    ones = np.ones((sq, skv), dtype=bool)
    if mode == 0 and atten_mask is not None:   # the matrix, inside the preTokens/nextTokens band
        band = np.tril(ones, k=min(nxt, skv + 1)) & np.triu(ones, k=-min(pre, sq + 1))
        return band & (np.asarray(atten_mask)[:sq, :skv] == 0)
    if mode == 1:                      # the full attention-mask matrix: nonzero masks
        return np.asarray(atten_mask)[:sq, :skv] == 0
    if mode == 6:                      # bottom-right lower triangle, plus the first N columns
        return np.tril(ones, k=skv - sq) | (np.arange(skv)[None, :] < prefix_n)
    if mode == 0:                      # no attention mask: everything takes part
        return ones
    if mode == 2:                      # lower triangle from the top-left vertex
        return np.tril(ones, k=0)
    if mode == 3:                      # lower triangle from the bottom-right vertex
        return np.tril(ones, k=skv - sq)
    if mode == 4:                      # band between preTokens (left) and nextTokens (right)
        return np.tril(ones, k=min(nxt, skv + 1)) & np.triu(ones, k=-min(pre, sq + 1))
    raise ValueError(mode)


def random_bits(rng, shapes, p_keep=0.7):
    """Per-sequence keep-bit tensors [Nq, Sq, Skv] and their packed form,
    flattened in (sequence, head, row, column) order, least significant bit first."""
    tensors = [rng.random(s) < p_keep for s in shapes]
    flat = np.concatenate([t.reshape(-1) for t in tensors]) if tensors else np.zeros(0, bool)
    packed = np.packbits(flat, bitorder="little")
    return tensors, packed


def autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, *, mode=0, pre=2**31 - 1,
                       nxt=2**31 - 1, bits=None, keep_prob=1.0, sink=None, atten_mask=None,
                       prefix=None, bias=None, pse_type=1):
    """Textbook attention per (sequence, head) in torch fp64, differentiated by
    autograd.  Returns dict of numpy arrays: out, smax, ssum, dq, dk, dv, dsink."""
    G = nq // nkv
    Q = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    K = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    V = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    dY = torch.tensor(dy, dtype=torch.float64)
    S_ink = None if sink is None else torch.tensor(np.asarray(sink, np.float64), requires_grad=True)
    out = torch.zeros((Q.shape[0], nq, V.shape[2]), dtype=torch.float64)   # value head dim
    smax = torch.full((Q.shape[0], nq), float("nan"), dtype=torch.float64)
    ssum = torch.full((Q.shape[0], nq), float("nan"), dtype=torch.float64)
    pieces = []
    for b in range(len(cu_q) - 1):
        tq, tk = int(cu_q[b]), int(cu_kv[b])
        sq, skv = int(cu_q[b + 1]) - tq, int(cu_kv[b + 1]) - tk
        if sq == 0:
            continue
        keep = torch.tensor(mask_matrix(mode, pre, nxt, sq, skv, atten_mask,
                                        0 if prefix is None else int(prefix[b])))
        for h in range(nq):
            g = h // G
            qb = Q[tq:tq + sq, h, :]
            kb = K[tk:tk + skv, g, :]
            vb = V[tk:tk + skv, g, :]
            if bias is None:
                logits = scale * qb @ kb.T
            else:   # bias[b]: explicit [Nq, Sq, Skv] pse matrix of the sequence
                pse = torch.tensor(bias[b][h], dtype=torch.float64)
                logits = scale * (qb @ kb.T + pse) if pse_type == 1 else scale * qb @ kb.T + pse
            logits = logits.masked_fill(~keep, float("-inf"))
            if S_ink is not None:
                logits = torch.cat([logits, S_ink[h].expand(sq, 1)], dim=1)
            m = logits.max(dim=1).values if logits.shape[1] else torch.full((sq,), float("-inf"), dtype=torch.float64)
            has = torch.isfinite(m)
            msafe = torch.where(has, m, torch.zeros_like(m))
            e = torch.exp(logits - msafe[:, None])
            e = torch.where(torch.isfinite(logits), e, torch.zeros_like(e))
            l = e.sum(dim=1)
            lsafe = torch.where(l > 0, l, torch.ones_like(l))
            p = e / lsafe[:, None]
            p = p[:, :skv]
            if bits is not None and keep_prob < 1.0:
                z = torch.tensor(bits[b][h].astype(np.float64)) / keep_prob
                p = p * z
            ob = p @ vb
            pieces.append(((tq, h, sq), ob))
            smax[tq:tq + sq, h] = m.detach()
            ssum[tq:tq + sq, h] = l.detach()
    loss = torch.zeros((), dtype=torch.float64)
    for (tq, h, sq), ob in pieces:
        out[tq:tq + sq, h, :] = ob.detach()
        loss = loss + (ob * dY[tq:tq + sq, h, :]).sum()
    grads = torch.autograd.grad(loss, [Q, K, V] + ([S_ink] if S_ink is not None else []),
                                allow_unused=True)
    res = {"out": out.numpy(), "smax": smax.numpy(), "ssum": ssum.numpy(), "loss": float(loss.detach())}
    for name, gr, ref in zip(["dq", "dk", "dv"], grads[:3], [Q, K, V]):
        res[name] = (torch.zeros_like(ref) if gr is None else gr).detach().numpy()
    res["dsink"] = None if S_ink is None else (grads[3] if grads[3] is not None
                                               else torch.zeros(nq, dtype=torch.float64)).detach().numpy()
    return res


def random_problem(seed, seqlens_q, seqlens_kv, nq, nkv, d, dv=None):
    """Random Q, K [.., d] and V, dY [.., dv] (dv = d by default)."""
    rng = np.random.default_rng(seed)
    dv = d if dv is None else dv
    tq, tkv = sum(seqlens_q), sum(seqlens_kv)
    cu_q = np.concatenate([[0], np.cumsum(seqlens_q)]).astype(np.int64)
    cu_kv = np.concatenate([[0], np.cumsum(seqlens_kv)]).astype(np.int64)
    q = rng.standard_normal((tq, nq, d))
    k = rng.standard_normal((tkv, nkv, d))
    v = rng.standard_normal((tkv, nkv, dv))
    dy = rng.standard_normal((tq, nq, dv))
    return rng, cu_q, cu_kv, q, k, v, dy


def scale_for(d):
    return 1.0 / math.sqrt(d)
