"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently: the
closed form of the all-ones sample program on the aclnnFlashAttentionScoreV2
page (example section), torch autograd of the textbook attention forward,
central finite differences, closed forms (Q = 0, causal / band pair counts),
brute-force mask matrices and bit layouts, and exact identities (row sums of
dS, bilinear identities, GQA = repeated MHA, varlen = concatenation).
"""

import json
import math
import os

import numpy as np
import pytest

from tests.oracle_pins_helpers import (autograd_reference, mask_matrix, random_bits,
                                       random_problem, scale_for)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INF = 2147483647


def _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, **kw):
    return ora.Problem(cu_q, cu_kv, nq, nkv, d, scale, **kw)


# --------------------------------------------------------------------------
# worked example of the forward page
# --------------------------------------------------------------------------

def test_allones_sample_forward_and_grad(ora):
    fx = json.load(open(os.path.join(GOLDEN, "scorev2_allones_sample.json")))
    inp, exp_ = fx["inputs"], fx["expected"]
    T, N, D = inp["tnd_relayout"]["T"], inp["tnd_relayout"]["N"], inp["tnd_relayout"]["D"]
    q = np.full((T, N, D), inp["q_value"])
    k = np.full((T, N, D), inp["k_value"])
    v = np.full((T, N, D), inp["v_value"])
    p = _problem(ora, inp["tnd_relayout"]["cu_seqlens"], inp["tnd_relayout"]["cu_seqlens"], N, N, D,
                 inp["scaleValue"], keep_prob=inp["keepProb"], pre_tokens=inp["preTokens"],
                 next_tokens=inp["nextTokens"], sparse_mode=inp["sparseMode"])
    out, smax, ssum = ora.fwd(p, q, k, v)
    np.testing.assert_allclose(smax, exp_["softmax_max"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ssum, exp_["softmax_sum"], rtol=0, atol=1e-9)
    np.testing.assert_allclose(out, exp_["attention_out"], rtol=0, atol=1e-12)
    dy = np.random.default_rng(5).standard_normal((T, N, D))
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    assert np.abs(dq).max() <= 1e-9 and np.abs(dk).max() <= 1e-9
    np.testing.assert_allclose(dv, np.broadcast_to(dy.mean(axis=0), dv.shape), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# masks
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode,pre,nxt", [(0, INF, INF), (2, INF, INF), (3, INF, INF), (4, 3, 0),
                                          (4, 0, 2), (4, 5, 4), (4, 2, -1), (4, -1, 3)])
@pytest.mark.parametrize("sq,skv", [(7, 7), (5, 9), (9, 5), (1, 13), (13, 1), (8, 8)])
def test_mask_predicate_matches_explicit_matrix(ora, mode, pre, nxt, sq, skv):
    ref = mask_matrix(mode, pre, nxt, sq, skv)
    got = np.array([[ora.keep(mode, pre, nxt, sq, skv, i, j) for j in range(skv)] for i in range(sq)],
                   dtype=bool).reshape(sq, skv)
    np.testing.assert_array_equal(got, ref)


def test_mask_pair_counts_closed_forms(ora):
    # causal: S(S+1)/2 kept pairs per (sequence, head)
    for s in (1, 2, 37, 64, 130):
        n = sum(ora.keep(3, INF, INF, s, s, i, j) for i in range(s) for j in range(s))
        assert n == s * (s + 1) // 2
    # band preTokens=W, nextTokens=0 over S rows: sum_i (min(i, W) + 1)
    S, W = 200, 17
    n = sum(ora.keep(4, W, 0, S, S, i, j) for i in range(S) for j in range(S))
    assert n == W * (W + 1) // 2 + (S - W) * (W + 1)
    # the sliding-window workload: 8192 rows, window 1024 back -> 7,872,000 pairs
    S, W = 8192, 1024
    assert W * (W + 1) // 2 + (S - W) * (W + 1) == 7_872_000
    kept_rows = np.array([sum(ora.keep(4, W, 0, S, S, i, j) for j in range(max(0, i - W - 2), i + 3))
                          for i in (0, 1, 500, 1023, 1024, 1025, 5000, 8191)])
    np.testing.assert_array_equal(kept_rows, [1, 2, 501, 1024, 1025, 1025, 1025, 1025])


def test_mask_mode_equivalences(ora):
    for s in (1, 6, 11):
        for i in range(s):
            for j in range(s):
                c3 = ora.keep(3, INF, INF, s, s, i, j)
                assert c3 == ora.keep(2, INF, INF, s, s, i, j) == ora.keep(4, INF, 0, s, s, i, j)
                assert ora.keep(4, s, s, s, s, i, j) == ora.keep(0, INF, INF, s, s, i, j) == 1


# --------------------------------------------------------------------------
# attention-mask matrix (sparseMode 0 / 1) and prefix (sparseMode 6)
# --------------------------------------------------------------------------

def _keep_grid(ora, p, b):
    sq = int(p.cu_q[b + 1] - p.cu_q[b])
    skv = int(p.cu_kv[b + 1] - p.cu_kv[b])
    return np.array([[ora.keep_at(p, b, i, j) for j in range(skv)] for i in range(sq)],
                    dtype=bool).reshape(sq, skv)


@pytest.mark.parametrize("mode,pre,nxt", [(1, INF, INF), (0, INF, INF), (0, 3, 1), (0, 0, 4)])
@pytest.mark.parametrize("sq,skv", [(7, 7), (5, 9), (9, 5), (1, 6)])
def test_atten_mask_predicate_matches_explicit_matrix(ora, mode, pre, nxt, sq, skv):
    rng = np.random.default_rng(sq * 31 + skv)
    # the matrix is [S1Max, S2Max]; the second sequence is the longest one
    amask = (rng.random((sq + 2, skv + 3)) < 0.4).astype(np.uint8) * rng.integers(1, 256, (sq + 2, skv + 3),
                                                                                 dtype=np.uint8)
    cu_q, cu_kv = [0, sq, 2 * sq + 2], [0, skv, 2 * skv + 3]
    p = _problem(ora, cu_q, cu_kv, 1, 1, 4, 1.0, sparse_mode=mode, pre_tokens=pre, next_tokens=nxt,
                 atten_mask=amask)
    for b, (a, c) in enumerate([(sq, skv), (sq + 2, skv + 3)]):
        np.testing.assert_array_equal(_keep_grid(ora, p, b), mask_matrix(mode, pre, nxt, a, c, amask))


@pytest.mark.parametrize("sq,skv", [(7, 7), (5, 9), (9, 5), (4, 1)])
def test_prefix_predicate_matches_explicit_matrix(ora, sq, skv):
    prefixes = [0, 1, skv // 2, skv]
    cu_q = np.arange(len(prefixes) + 1) * sq
    cu_kv = np.arange(len(prefixes) + 1) * skv
    p = _problem(ora, cu_q, cu_kv, 1, 1, 4, 1.0, sparse_mode=6, prefix=prefixes)
    for b, n in enumerate(prefixes):
        np.testing.assert_array_equal(_keep_grid(ora, p, b), mask_matrix(6, INF, INF, sq, skv, prefix_n=n))


def test_atten_mask_and_prefix_special_cases(ora):
    """Degenerate matrices and prefixes reduce to the plain modes."""
    s = 9
    cu = [0, s]
    zero = np.zeros((s, s), np.uint8)
    upper = np.triu(np.ones((s, s), np.uint8), k=1)
    plain = {m: _keep_grid(ora, _problem(ora, cu, cu, 1, 1, 4, 1.0, sparse_mode=m), 0) for m in (0, 3)}
    band = _keep_grid(ora, _problem(ora, cu, cu, 1, 1, 4, 1.0, sparse_mode=4, pre_tokens=2, next_tokens=1), 0)
    grid = lambda **kw: _keep_grid(ora, _problem(ora, cu, cu, 1, 1, 4, 1.0, **kw), 0)
    np.testing.assert_array_equal(grid(sparse_mode=1, atten_mask=zero), plain[0])
    np.testing.assert_array_equal(grid(sparse_mode=1, atten_mask=upper), plain[3])
    np.testing.assert_array_equal(grid(sparse_mode=0, atten_mask=zero, pre_tokens=2, next_tokens=1), band)
    np.testing.assert_array_equal(grid(sparse_mode=0, atten_mask=upper, pre_tokens=INF, next_tokens=INF),
                                  plain[3])
    np.testing.assert_array_equal(grid(sparse_mode=6, prefix=[0]), plain[3])
    np.testing.assert_array_equal(grid(sparse_mode=6, prefix=[s]), plain[0])
    # prefix 3 on a 9 x 9 sequence: the 45 causal pairs plus, in row i, the prefix columns right of i
    n = int(grid(sparse_mode=6, prefix=[3]).sum())
    assert n == s * (s + 1) // 2 + sum(max(0, 3 - (i + 1)) for i in range(s))


MASK_CASES = [
    # seqlens_q, seqlens_kv, nq, nkv, mode, pre, nxt, prefix, dropout, sink
    ([5, 9], [5, 9], 2, 2, 1, INF, INF, None, False, False),
    ([6, 3], [9, 4], 4, 2, 1, INF, INF, None, True, True),
    ([7, 8], [7, 8], 2, 1, 0, 3, 2, None, False, True),
    ([6, 9], [6, 9], 2, 2, 6, INF, INF, [2, 4], False, False),
    ([5, 4, 7], [8, 4, 7], 2, 1, 6, INF, INF, [0, 4, 3], True, True),
]


def _mask_case(ora, ci):
    sq, skv, nq, nkv, mode, pre, nxt, prefix, drop, sink = MASK_CASES[ci]
    d = 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(300 + ci, sq, skv, nq, nkv, d)
    scale = scale_for(d) * 1.7
    amask = None
    if mode in (0, 1):
        amask = (rng.random((max(sq), max(skv))) < 0.35).astype(np.uint8)
        amask[0, :] = 1                         # a fully masked row
    bits, packed, kp = None, None, 1.0
    if drop:
        bits, packed = random_bits(rng, [(nq, a, b) for a, b in zip(sq, skv)], 0.75)
        kp = 0.75
    snk = rng.standard_normal(nq) if sink else None
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, keep_prob=kp, pre_tokens=pre, next_tokens=nxt,
                 sparse_mode=mode, drop_mask=packed, sink=snk, atten_mask=amask, prefix=prefix)
    ref = autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, mode=mode, pre=pre, nxt=nxt,
                             bits=bits, keep_prob=kp, sink=snk, atten_mask=amask, prefix=prefix)
    return p, (q, k, v, dy), ref


@pytest.mark.parametrize("ci", range(len(MASK_CASES)))
def test_masked_forward_and_grad_match_autograd(ora, ci):
    p, (q, k, v, dy), ref = _mask_case(ora, ci)
    out, smax, ssum = ora.fwd(p, q, k, v)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    fin = np.isfinite(ref["smax"])
    np.testing.assert_array_equal(np.isfinite(smax), fin)
    np.testing.assert_allclose(smax[fin], ref["smax"][fin], rtol=1e-13, atol=1e-13)
    dq, dk, dv, dsink = ora.grad(p, q, k, v, dy, out, smax, ssum)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-11, err_msg=name)
    if ref["dsink"] is not None:
        np.testing.assert_allclose(dsink, ref["dsink"], rtol=1e-10, atol=1e-11)


def test_masked_grad_matches_central_differences(ora):
    p, (q, k, v, dy), _ = _mask_case(ora, 1)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, _, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    h, rng = 1e-6, np.random.default_rng(9)
    for name, arr, g in (("q", q, dq), ("k", k, dk)):
        for _ in range(10):
            idx = tuple(rng.integers(0, n) for n in arr.shape)
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            f = lambda a: float(np.sum(ora.fwd(p, *((a, k, v) if name == "q" else (q, a, v)))[0] * dy))
            fd = (f(a1) - f(a2)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


# --------------------------------------------------------------------------
# pse (positional bias), stored as the last 1024 rows of each sequence's bias
# --------------------------------------------------------------------------

def _alibi_full(slopes, sq):
    """Full [Nq, sq, sq] alibi bias slope_h * (j - i): depends only on i - j."""
    ij = np.arange(sq)[None, :] - np.arange(sq)[:, None]
    return np.asarray(slopes, np.float64)[:, None, None] * ij[None]


def _store_last_rows(full, rng):
    """[Nq, 1024, S] store of a full [Nq, sq, S] bias: its last 1024 rows (numpy
    slicing); a shorter bias fills the bottom rows, the rows above hold noise."""
    nq, sq, s = full.shape
    out = rng.standard_normal((nq, 1024, s))
    out[:, max(0, 1024 - sq):, :] = full[:, -1024:, :]
    return out


@pytest.mark.parametrize("pse_type", [0, 1])
@pytest.mark.parametrize("seqs", [[1300, 40], [700]])
def test_alibi_pse_matches_autograd_with_the_full_bias(ora, pse_type, seqs):
    """The stored rows of an alibi bias reproduce the whole [Sq, Sq] bias: rows
    above the last 1024 are read along their diagonal."""
    nq, nkv, d = 2, 1, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(41 + len(seqs), seqs, seqs, nq, nkv, d)
    slopes = [0.05, -0.02]
    s2 = max(seqs)
    store = np.zeros((len(seqs), nq, 1024, s2))
    full = []
    for b, sq in enumerate(seqs):
        f = _alibi_full(slopes, sq)
        full.append(f)
        padded = np.zeros((nq, sq, s2))
        padded[:, :, :sq] = f
        store[b] = _store_last_rows(padded, rng)
    scale = scale_for(d)
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, sparse_mode=3, pse=store, pse_type=pse_type)
    ref = autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, mode=3, bias=full, pse_type=pse_type)
    out, smax, ssum = ora.fwd(p, q, k, v)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(smax, ref["smax"], rtol=1e-12, atol=1e-12)
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("pse_type", [0, 1])
def test_random_pse_short_sequences_match_autograd(ora, pse_type):
    """Sequences shorter than 1024 take the bottom rows of the store as their
    bias, whatever it holds (broadcast over the batch when its first dim is 1)."""
    seqs, nq, nkv, d = [37, 64, 5], 4, 2, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(53, seqs, seqs, nq, nkv, d)
    store = rng.standard_normal((1, nq, 1024, max(seqs)))
    full = [store[0, :, 1024 - sq:, :sq] for sq in seqs]
    scale = scale_for(d) * 1.3
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, sparse_mode=2, pse=store, pse_type=pse_type)
    ref = autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, mode=2, bias=full, pse_type=pse_type)
    out, smax, ssum = ora.fwd(p, q, k, v)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-11, err_msg=name)


def test_pse_special_cases(ora):
    """Zero pse is no pse; a pse constant along each row shifts the max only."""
    seqs, nq, nkv, d = [1100, 30], 2, 2, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(61, seqs, seqs, nq, nkv, d)
    scale = scale_for(d)
    base = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, sparse_mode=3)
    o0, m0, l0 = ora.fwd(base, q, k, v)
    g0 = ora.grad(base, q, k, v, dy, o0, m0, l0)
    zero = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, sparse_mode=3, pse=np.zeros((1, nq, 1024, 1100)))
    o1, m1, l1 = ora.fwd(zero, q, k, v)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(m1, m0)
    # a constant c per (head, stored row) is constant along every row of the full
    # bias (rows above the stored ones read stored row 0); rows shift by c
    # (pseType 0) or scale * c (pseType 1)
    c = rng.standard_normal((2, nq, 1024, 1))
    store = np.broadcast_to(c, (2, nq, 1024, 1100)).copy()
    for pse_type, mul in ((0, 1.0), (1, scale)):
        pp = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, sparse_mode=3, pse=store, pse_type=pse_type)
        o2, m2, l2 = ora.fwd(pp, q, k, v)
        np.testing.assert_allclose(o2, o0, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l2, l0, rtol=1e-12)
        for b, sq in enumerate(seqs):
            rows = np.maximum(np.arange(sq) - (sq - 1024), 0)
            shift = mul * c[b][:, rows, 0].T                  # [sq, nq]
            np.testing.assert_allclose(m2[cu_q[b]:cu_q[b + 1]], m0[cu_q[b]:cu_q[b + 1]] + shift, rtol=1e-12,
                                       atol=1e-12)
        g2 = ora.grad(pp, q, k, v, dy, o2, m2, l2)
        for a_, b_ in zip(g2[:3], g0[:3]):
            np.testing.assert_allclose(a_, b_, rtol=1e-10, atol=1e-12)


def test_pse_grad_matches_central_differences(ora):
    seqs, nq, nkv, d = [1030], 2, 1, 4
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(71, seqs, seqs, nq, nkv, d)
    store = 0.3 * rng.standard_normal((1, nq, 1024, 1030))
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, 0.4, sparse_mode=3, pse=store, pse_type=1)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, _, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    h = 1e-6
    for name, arr, g in (("q", q, dq), ("k", k, dk)):
        for idx in [(0, 0, 1), (5, arr.shape[1] - 1, 3), (1029, 0, 2), (1028, arr.shape[1] - 1, 0)]:
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            f = lambda a: float(np.sum(ora.fwd(p, *((a, k, v) if name == "q" else (q, a, v)))[0] * dy))
            fd = (f(a1) - f(a2)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


# --------------------------------------------------------------------------
# pse generated inside from slopes (pseType 2 / 3), read as alibi
# --------------------------------------------------------------------------

def test_generated_alibi_causal_equals_a_column_bias_in_one_more_dim(ora):
    """pseType 2 under the causal mask: for j <= i the bias -slope (i - j) is
    slope * j plus a constant of the row, which the softmax drops (it only moves
    the max).  slope * j added after the scale is one more feature: Q gets a
    column of ones, K the column slope * j / scale.  The no-pse problem in D + 1
    dims then has the same O, dV, sum, the same dQ and dK in the first D
    columns, and max + slope * i."""
    seqs, nq, d = [37, 130, 1], 3, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(81, seqs, seqs, nq, nq, d)
    slopes = np.array([0.3, -0.15, 0.02])
    scale = scale_for(d) * 1.2
    p = _problem(ora, cu_q, cu_kv, nq, nq, d, scale, sparse_mode=3, pse=slopes, pse_type=2)
    out, smax, ssum, dq, dk, dv, _ = ora.fwd_grad(p, q, k, v, dy)
    jpos = np.concatenate([np.arange(n) for n in seqs]).astype(np.float64)      # in-sequence index
    q1 = np.concatenate([q, np.ones(q.shape[:2] + (1,))], axis=2)
    k1 = np.concatenate([k, (slopes[None, :] * jpos[:, None] / scale)[..., None]], axis=2)
    p1 = _problem(ora, cu_q, cu_kv, nq, nq, d + 1, scale, sparse_mode=3, dv=d)   # V, dY keep d columns
    out1, smax1, ssum1, dq1, dk1, dv1, _ = ora.fwd_grad(p1, q1, k1, v, dy)
    np.testing.assert_allclose(out, out1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ssum, ssum1, rtol=1e-12)
    np.testing.assert_allclose(smax, smax1 - slopes[None, :] * jpos[:, None], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dq, dq1[..., :d], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, dk1[..., :d], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, dv1, rtol=1e-10, atol=1e-12)


def test_generated_alibi_types_agree_at_distances_zero_and_one(ora):
    """sqrt(0) = 0 and sqrt(1) = 1: with sequences of at most two rows the
    sqrt variant (pseType 3) is bitwise the linear one (pseType 2)."""
    seqs, nq, nkv, d = [2, 1, 2, 2], 2, 1, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(83, seqs, seqs, nq, nkv, d)
    slopes = rng.standard_normal((len(seqs), nq))
    r2 = ora.fwd_grad(_problem(ora, cu_q, cu_kv, nq, nkv, d, 0.7, sparse_mode=2, pse=slopes, pse_type=2), q, k, v, dy)
    r3 = ora.fwd_grad(_problem(ora, cu_q, cu_kv, nq, nkv, d, 0.7, sparse_mode=2, pse=slopes, pse_type=3), q, k, v, dy)
    for a_, b_ in zip(r2, r3):
        np.testing.assert_array_equal(a_, b_)


def test_generated_pse_with_zero_slopes_is_no_pse(ora):
    seqs, nq, nkv, d = [40, 9], 2, 2, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(85, seqs, seqs, nq, nkv, d)
    r0 = ora.fwd_grad(_problem(ora, cu_q, cu_kv, nq, nkv, d, 0.3, sparse_mode=3), q, k, v, dy)
    for pse_type in (2, 3):
        r = ora.fwd_grad(_problem(ora, cu_q, cu_kv, nq, nkv, d, 0.3, sparse_mode=3, pse=np.zeros(nq),
                                  pse_type=pse_type), q, k, v, dy)
        for a_, b_ in zip(r, r0):
            np.testing.assert_array_equal(a_, b_)


@pytest.mark.parametrize("pse_type", [2, 3])
@pytest.mark.parametrize("per_batch", [False, True])
def test_generated_alibi_matches_autograd(ora, pse_type, per_batch):
    """The reading written out as explicit [Nq, Sq, Sq] bias matrices, added
    after the scale, through torch autograd; slopes per head ([N]) or per
    sequence and head ([B, N]), GQA and a bias over more than 1024 rows."""
    seqs, nq, nkv, d = [1100, 57, 3], 4, 2, 8
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(87 + pse_type, seqs, seqs, nq, nkv, d)
    slopes = 0.01 * rng.standard_normal((len(seqs), nq) if per_batch else (nq,))
    full = []
    for b, sq in enumerate(seqs):
        sl = slopes[b] if per_batch else slopes
        dist = np.abs(np.arange(sq)[:, None] - np.arange(sq)[None, :]).astype(np.float64)
        full.append(-sl[:, None, None] * (dist if pse_type == 2 else np.sqrt(dist))[None])
    scale = scale_for(d)
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, sparse_mode=3, pse=slopes, pse_type=pse_type)
    ref = autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, mode=3, bias=full, pse_type=0)
    out, smax, ssum = ora.fwd(p, q, k, v)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(smax, ref["smax"], rtol=1e-12, atol=1e-12)
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-11, err_msg=name)


def test_generated_pse_slope_shapes(ora):
    with pytest.raises(ValueError):
        _problem(ora, [0, 3, 5], [0, 3, 5], 2, 1, 8, 0.3, sparse_mode=3, pse=np.zeros((3, 2)), pse_type=2)
    with pytest.raises(ValueError):
        _problem(ora, [0, 3], [0, 3], 2, 1, 8, 0.3, sparse_mode=3, pse=np.zeros(3), pse_type=3)


# --------------------------------------------------------------------------
# dropout keep-bit layout
# --------------------------------------------------------------------------

def test_dropout_bit_layout_bruteforce(ora):
    rng = np.random.default_rng(11)
    seq_q, seq_kv, nq = [3, 0, 5, 9], [7, 4, 0, 13], 3
    shapes = [(nq, a, b) for a, b in zip(seq_q, seq_kv)]
    tensors, packed = random_bits(rng, shapes, 0.5)
    cu_q = np.concatenate([[0], np.cumsum(seq_q)])
    cu_kv = np.concatenate([[0], np.cumsum(seq_kv)])
    p = _problem(ora, cu_q, cu_kv, nq, 1, 4, 1.0, keep_prob=0.5, drop_mask=packed)
    assert p.mask_bits() == sum(int(np.prod(s)) for s in shapes)
    assert packed.size == (p.mask_bits() + 7) // 8
    for b, t in enumerate(tensors):
        base = p.mask_base(b)
        for h in range(nq):
            for i in range(seq_q[b]):
                for j in range(seq_kv[b]):
                    assert ora.keep_bit(packed, base + (h * seq_q[b] + i) * seq_kv[b] + j) == int(t[h, i, j])


def test_all_ones_dropout_mask_scales_by_inverse_keep_prob(ora):
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(3, [5, 7], [6, 7], 2, 1, 8)
    base = _problem(ora, cu_q, cu_kv, 2, 1, 8, 0.3, sparse_mode=3)
    nbits = base.mask_bits()
    ones = np.packbits(np.ones(nbits, bool), bitorder="little")
    kp = 0.8
    drop = _problem(ora, cu_q, cu_kv, 2, 1, 8, 0.3, sparse_mode=3, keep_prob=kp, drop_mask=ones)
    same = _problem(ora, cu_q, cu_kv, 2, 1, 8, 0.3, sparse_mode=3, keep_prob=1.0, drop_mask=ones)
    o0, m0, l0 = ora.fwd(base, q, k, v)
    o1, m1, l1 = ora.fwd(drop, q, k, v)
    o2, _, _ = ora.fwd(same, q, k, v)
    np.testing.assert_allclose(o1, o0 / kp, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(o2, o0)
    np.testing.assert_array_equal(m1, m0)
    np.testing.assert_array_equal(l1, l0)


# --------------------------------------------------------------------------
# forward and gradient against torch autograd of the textbook formula
# --------------------------------------------------------------------------

CASES = [
    # seqlens_q, seqlens_kv, nq, nkv, d, mode, pre, nxt, dropout, sink
    ([5, 9], [5, 9], 2, 2, 8, 0, INF, INF, False, False),
    ([5, 9], [5, 9], 2, 2, 8, 3, INF, INF, False, False),
    ([6, 3], [9, 3], 4, 2, 8, 3, INF, INF, False, False),   # Sq < Skv, GQA
    ([9, 4], [6, 4], 2, 1, 8, 3, INF, INF, False, False),   # Sq > Skv: fully masked rows
    ([7, 0, 5], [7, 3, 5], 2, 2, 4, 2, INF, INF, False, False),
    ([8, 11], [8, 11], 4, 1, 8, 4, 3, 0, False, False),
    ([8, 11], [8, 11], 2, 2, 8, 4, 2, 3, True, False),
    ([6, 5], [6, 5], 2, 2, 8, 3, INF, INF, True, True),
    ([6, 0, 9], [6, 2, 9], 3, 1, 4, 0, INF, INF, False, True),
    ([4, 7], [0, 7], 2, 1, 4, 3, INF, INF, True, True),      # a sequence with no keys
]


def _case(ora, case, seed=0):
    sq, skv, nq, nkv, d, mode, pre, nxt, drop, sink = case
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(100 + seed, sq, skv, nq, nkv, d)
    scale = scale_for(d) * 1.7
    bits, packed, kp = None, None, 1.0
    if drop:
        bits, packed = random_bits(rng, [(nq, a, b) for a, b in zip(sq, skv)], 0.75)
        kp = 0.75
    snk = rng.standard_normal(nq) if sink else None
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, keep_prob=kp, pre_tokens=pre, next_tokens=nxt,
                 sparse_mode=mode, drop_mask=packed, sink=snk)
    ref = autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, mode=mode, pre=pre, nxt=nxt,
                             bits=bits, keep_prob=kp, sink=snk)
    return p, (q, k, v, dy), ref


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_forward_and_grad_match_autograd(ora, ci):
    p, (q, k, v, dy), ref = _case(ora, CASES[ci], ci)
    out, smax, ssum = ora.fwd(p, q, k, v)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    fin = np.isfinite(ref["smax"])
    np.testing.assert_array_equal(np.isfinite(smax), fin)
    np.testing.assert_allclose(smax[fin], ref["smax"][fin], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ssum[~np.isnan(ref["ssum"])], ref["ssum"][~np.isnan(ref["ssum"])],
                               rtol=1e-12, atol=1e-13)
    dq, dk, dv, dsink = ora.grad(p, q, k, v, dy, out, smax, ssum)
    np.testing.assert_allclose(dq, ref["dq"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, ref["dk"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, ref["dv"], rtol=1e-10, atol=1e-11)
    if ref["dsink"] is not None:
        np.testing.assert_allclose(dsink, ref["dsink"], rtol=1e-10, atol=1e-11)
    else:
        assert np.all(dsink == 0)


# --------------------------------------------------------------------------
# value head dim below the query/key head dim (qD == kD >= vD)
# --------------------------------------------------------------------------

DV_CASES = [
    # seqlens_q, seqlens_kv, nq, nkv, d, dv, mode, pre, nxt, dropout, sink
    ([5, 9], [5, 9], 2, 2, 8, 3, 3, INF, INF, False, False),
    ([6, 3], [9, 3], 4, 2, 8, 5, 3, INF, INF, True, True),
    ([8, 11], [8, 11], 2, 1, 6, 1, 4, 3, 1, True, False),
    ([7, 0, 5], [7, 3, 5], 2, 2, 4, 2, 0, INF, INF, False, True),
]


def _dv_case(ora, ci):
    sq, skv, nq, nkv, d, dv, mode, pre, nxt, drop, sink = DV_CASES[ci]
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(600 + ci, sq, skv, nq, nkv, d, dv)
    scale = scale_for(d) * 1.3
    bits, packed, kp = None, None, 1.0
    if drop:
        bits, packed = random_bits(rng, [(nq, a, b) for a, b in zip(sq, skv)], 0.8)
        kp = 0.8
    snk = rng.standard_normal(nq) if sink else None
    kw = dict(keep_prob=kp, pre_tokens=pre, next_tokens=nxt, sparse_mode=mode, drop_mask=packed, sink=snk)
    return (cu_q, cu_kv, nq, nkv, d, dv, scale, kw), (q, k, v, dy), (bits, kp, snk, mode, pre, nxt)


@pytest.mark.parametrize("ci", range(len(DV_CASES)))
def test_unequal_head_dims_match_autograd(ora, ci):
    """Value / dY / O / dV with Dv < D columns (aclnnFlashAttentionUnpaddingScoreGrad,
    constraints: qD == kD >= vD) against autograd of the textbook forward."""
    (cu_q, cu_kv, nq, nkv, d, dv, scale, kw), (q, k, v, dy), (bits, kp, snk, mode, pre, nxt) = _dv_case(ora, ci)
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, dv=dv, **kw)
    ref = autograd_reference(cu_q, cu_kv, nq, nkv, d, scale, q, k, v, dy, mode=mode, pre=pre, nxt=nxt,
                             bits=bits, keep_prob=kp, sink=snk)
    out, smax, ssum = ora.fwd(p, q, k, v)
    assert out.shape == (q.shape[0], nq, dv)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    dq, dk, dvv, dsink = ora.grad(p, q, k, v, dy, out, smax, ssum)
    np.testing.assert_allclose(dq, ref["dq"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, ref["dk"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dvv, ref["dv"], rtol=1e-10, atol=1e-11)
    if snk is not None:
        np.testing.assert_allclose(dsink, ref["dsink"], rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("ci", range(len(DV_CASES)))
def test_unequal_head_dims_equal_zero_padded_value(ora, ci):
    """Appending D - Dv zero columns to V and dY gives the equal-dims problem:
    its O and dV are those of the Dv problem followed by zeros, its dQ, dK, max,
    sum and dSink are the same, bit for bit (the extra terms are exact zeros)."""
    (cu_q, cu_kv, nq, nkv, d, dv, scale, kw), (q, k, v, dy), _ = _dv_case(ora, ci)
    pad = lambda x: np.concatenate([x, np.zeros(x.shape[:2] + (d - dv,))], axis=2)
    p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, dv=dv, **kw)
    pf = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, **kw)
    small = ora.fwd_grad(p, q, k, v, dy)
    full = ora.fwd_grad(pf, q, k, pad(v), pad(dy))
    for n, a, b in zip(("out", "smax", "ssum", "dq", "dk", "dv", "dsink"), small, full):
        if n in ("out", "dv"):
            np.testing.assert_array_equal(b[..., dv:], 0.0, err_msg=n)
            b = b[..., :dv]
        np.testing.assert_array_equal(a, b, err_msg=n)


def test_value_head_dim_bounds(ora):
    with pytest.raises(ValueError):
        _problem(ora, [0, 3], [0, 3], 1, 1, 8, 0.3, dv=9)
    with pytest.raises(ValueError):
        _problem(ora, [0, 3], [0, 3], 1, 1, 8, 0.3, dv=0)


# --------------------------------------------------------------------------
# finite differences of L = sum(dY * O) through the oracle's own forward
# --------------------------------------------------------------------------

@pytest.mark.parametrize("ci", [1, 2, 5, 6, 7, 9])
def test_grad_matches_central_differences(ora, ci):
    p, (q, k, v, dy), _ = _case(ora, CASES[ci], ci)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, dv, dsink = ora.grad(p, q, k, v, dy, out, smax, ssum)
    h = 1e-6
    rng = np.random.default_rng(ci)

    def loss(qq, kk, vv):
        o, _, _ = ora.fwd(p, qq, kk, vv)
        return float(np.sum(o * dy))

    for name, arr, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(rng.integers(0, n) for n in arr.shape)
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            args1 = {"q": q, "k": k, "v": v}
            args2 = dict(args1)
            args1[name], args2[name] = a1, a2
            fd = (loss(args1["q"], args1["k"], args1["v"]) - loss(args2["q"], args2["k"], args2["v"])) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])
    if p.sink is not None:
        for hh in range(p.nq):
            s1, s2 = p.sink.copy(), p.sink.copy()
            s1[hh] += h
            s2[hh] -= h
            p1 = ora.Problem(p.cu_q, p.cu_kv, p.nq, p.nkv, p.d, p._c.scale, p._c.keep_prob,
                             p._c.pre_tokens, p._c.next_tokens, p._c.sparse_mode, p.drop_mask, s1)
            p2 = ora.Problem(p.cu_q, p.cu_kv, p.nq, p.nkv, p.d, p._c.scale, p._c.keep_prob,
                             p._c.pre_tokens, p._c.next_tokens, p._c.sparse_mode, p.drop_mask, s2)
            fd = (np.sum(ora.fwd(p1, q, k, v)[0] * dy) - np.sum(ora.fwd(p2, q, k, v)[0] * dy)) / (2 * h)
            assert abs(fd - dsink[hh]) <= 1e-6 * max(1.0, abs(dsink[hh])), (hh, fd, dsink[hh])


@pytest.mark.parametrize("variant", ["dv_below_d", "alibi_sqrt"])
def test_new_paths_match_central_differences(ora, variant):
    """Central differences of sum(dY * O) through the oracle's own forward, for
    a value head dim below D (with dropout and a sink) and for the generated
    sqrt alibi (pseType 3)."""
    if variant == "dv_below_d":
        (cu_q, cu_kv, nq, nkv, d, dv, scale, kw), (q, k, v, dy), _ = _dv_case(ora, 1)
        p = _problem(ora, cu_q, cu_kv, nq, nkv, d, scale, dv=dv, **kw)
    else:
        seqs, nq, nkv, d = [23, 9], 2, 1, 8
        rng0, cu_q, cu_kv, q, k, v, dy = random_problem(97, seqs, seqs, nq, nkv, d)
        p = _problem(ora, cu_q, cu_kv, nq, nkv, d, 0.4, sparse_mode=3, pse=np.array([0.3, 0.05]), pse_type=3)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, dvv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    h = 1e-6
    rng = np.random.default_rng(5)

    def loss(qq, kk, vv):
        return float(np.sum(ora.fwd(p, qq, kk, vv)[0] * dy))

    for name, arr, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        for _ in range(10):
            idx = tuple(rng.integers(0, n) for n in arr.shape)
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            args1 = {"q": q, "k": k, "v": v}
            args2 = dict(args1)
            args1[name], args2[name] = a1, a2
            fd = (loss(args1["q"], args1["k"], args1["v"]) - loss(args2["q"], args2["k"], args2["v"])) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


# --------------------------------------------------------------------------
# closed forms and exact identities
# --------------------------------------------------------------------------

def test_q_zero_closed_form(ora):
    """Q = 0, no mask, no dropout: every probability is 1/Skv, so
    dV_j = (1/Skv) sum_i dY_i (summed over the group's heads) and dK = 0."""
    seq = [6, 10]
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(7, seq, seq, 4, 2, 8)
    q[:] = 0.0
    p = _problem(ora, cu_q, cu_kv, 4, 2, 8, 0.5)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    assert np.all(dk == 0.0)
    for b in range(2):
        t0, t1 = cu_q[b], cu_q[b + 1]
        for g in range(2):
            expect = dy[t0:t1, 2 * g:2 * g + 2, :].sum(axis=(0, 1)) / seq[b]
            np.testing.assert_allclose(dv[t0:t1, g, :], np.broadcast_to(expect, (seq[b], 8)),
                                       rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(out[t0:t1], np.broadcast_to(
            np.repeat(v[t0:t1].mean(axis=0), 2, axis=0), out[t0:t1].shape), rtol=1e-13, atol=1e-14)


def test_identical_value_rows_give_zero_ds(ora):
    """All V rows equal: dP_ij = D_i, so dS = 0 and dQ = dK = 0 (any mask)."""
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(8, [7, 5], [7, 5], 2, 2, 8)
    v[:] = rng.standard_normal(8)
    p = _problem(ora, cu_q, cu_kv, 2, 2, 8, 0.4, sparse_mode=3)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


@pytest.mark.parametrize("sink", [False, True])
def test_ds_row_sums(ora, sink):
    """Without sink every row of dS sums to 0; with a sink the sum of dS over a
    head plus that head's dSink is 0."""
    seq_q, seq_kv, nq = [6, 9], [8, 9], 2
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(9, seq_q, seq_kv, nq, 1, 8)
    bits, packed = random_bits(rng, [(nq, a, b) for a, b in zip(seq_q, seq_kv)], 0.6)
    snk = rng.standard_normal(nq) if sink else None
    p = _problem(ora, cu_q, cu_kv, nq, 1, 8, 0.35, sparse_mode=3, keep_prob=0.6, drop_mask=packed, sink=snk)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, dv, dsink, ds = ora.grad(p, q, k, v, dy, out, smax, ssum, want_ds=True)
    per_head = np.zeros(nq)
    for b in range(2):
        base = p.mask_base(b)
        blk = ds[base: base + nq * seq_q[b] * seq_kv[b]].reshape(nq, seq_q[b], seq_kv[b])
        if not sink:
            np.testing.assert_allclose(blk.sum(axis=2), 0.0, atol=1e-13)
        per_head += blk.sum(axis=(1, 2))
    if sink:
        np.testing.assert_allclose(per_head + dsink, 0.0, atol=1e-12)
        assert np.abs(dsink).max() > 1e-3


def test_bilinear_identities(ora):
    """<dQ,Q> = <dK,K> (per kv group) and <dV,V> = <dY,O>."""
    p, (q, k, v, dy), _ = _case(ora, CASES[6], 6)
    out, smax, ssum = ora.fwd(p, q, k, v)
    dq, dk, dv, _ = ora.grad(p, q, k, v, dy, out, smax, ssum)
    G = p.nq // p.nkv
    for g in range(p.nkv):
        lhs = np.sum(dq[:, g * G:(g + 1) * G] * q[:, g * G:(g + 1) * G])
        rhs = np.sum(dk[:, g] * k[:, g])
        assert abs(lhs - rhs) < 1e-10 * max(1, abs(lhs))
    assert abs(np.sum(dv * v) - np.sum(dy * out)) < 1e-10 * max(1, abs(np.sum(dy * out)))


def test_gqa_equals_repeated_mha(ora):
    seq = [7, 12]
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(12, seq, seq, 6, 2, 8)
    pg = _problem(ora, cu_q, cu_kv, 6, 2, 8, 0.3, sparse_mode=3)
    pm = _problem(ora, cu_q, cu_kv, 6, 6, 8, 0.3, sparse_mode=3)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    og, mg, lg, dqg, dkg, dvg, _ = ora.fwd_grad(pg, q, k, v, dy)
    om, mm, lm, dqm, dkm, dvm, _ = ora.fwd_grad(pm, q, kr, vr, dy)
    np.testing.assert_allclose(og, om, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dqg, dqm, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dkg, dkm.reshape(-1, 2, 3, 8).sum(axis=2), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dvg, dvm.reshape(-1, 2, 3, 8).sum(axis=2), rtol=1e-12, atol=1e-13)


def test_varlen_equals_concatenated_runs(ora):
    seq_q, seq_kv = [5, 0, 11, 3], [6, 4, 11, 3]
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(13, seq_q, seq_kv, 2, 1, 8)
    snk = rng.standard_normal(2)
    p = _problem(ora, cu_q, cu_kv, 2, 1, 8, 0.3, sparse_mode=3, sink=snk)
    full = ora.fwd_grad(p, q, k, v, dy)
    dsink_total = np.zeros(2)
    for b in range(4):
        a0, a1, c0, c1 = cu_q[b], cu_q[b + 1], cu_kv[b], cu_kv[b + 1]
        pb = _problem(ora, [0, a1 - a0], [0, c1 - c0], 2, 1, 8, 0.3, sparse_mode=3, sink=snk)
        part = ora.fwd_grad(pb, q[a0:a1], k[c0:c1], v[c0:c1], dy[a0:a1])
        np.testing.assert_allclose(full[0][a0:a1], part[0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(full[3][a0:a1], part[3], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(full[4][c0:c1], part[4], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(full[5][c0:c1], part[5], rtol=1e-13, atol=1e-14)
        dsink_total += part[6]
    np.testing.assert_allclose(full[6], dsink_total, rtol=1e-12, atol=1e-14)


def test_very_negative_sink_equals_no_sink(ora):
    seq = [9, 6]
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(14, seq, seq, 2, 2, 8)
    p0 = _problem(ora, cu_q, cu_kv, 2, 2, 8, 0.3, sparse_mode=3)
    p1 = _problem(ora, cu_q, cu_kv, 2, 2, 8, 0.3, sparse_mode=3, sink=np.array([-1e4, -1e4]))
    r0, r1 = ora.fwd_grad(p0, q, k, v, dy), ora.fwd_grad(p1, q, k, v, dy)
    for a, b in zip(r0[:6], r1[:6]):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    assert np.all(r1[6] == 0.0) or np.abs(r1[6]).max() < 1e-300


def test_forward_matches_library_softmax(ora):
    from scipy.special import softmax
    seq = [10]
    rng, cu_q, cu_kv, q, k, v, dy = random_problem(15, seq, seq, 1, 1, 16)
    p = _problem(ora, cu_q, cu_kv, 1, 1, 16, 0.25)
    out, smax, ssum = ora.fwd(p, q, k, v)
    ref = softmax(0.25 * q[:, 0] @ k[:, 0].T, axis=1) @ v[:, 0]
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-13, atol=1e-14)


def test_selection_narrows_without_changing_values(ora):
    p, (q, k, v, dy), _ = _case(ora, CASES[2], 2)
    full = ora.fwd_grad(p, q, k, v, dy)
    sel = ora.Problem(p.cu_q, p.cu_kv, p.nq, p.nkv, p.d, p._c.scale, sparse_mode=3,
                      heads=(2, 4), row_lo=[3, 1])
    out, smax, ssum = ora.fwd(sel, q, k, v)
    dq, dk, dv, _ = ora.grad(sel, q, k, v, dy, full[0], full[1], full[2])
    for b in range(2):
        lo, hi = p.cu_q[b] + [3, 1][b], p.cu_q[b + 1]
        np.testing.assert_array_equal(out[lo:hi, 2:4], full[0][lo:hi, 2:4])
        np.testing.assert_array_equal(dq[lo:hi, 2:4], full[3][lo:hi, 2:4])
    assert np.all(out[:, :2] == 0)
