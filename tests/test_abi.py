"""C ABI checks that need no GPU: the library loads and exports every entry
point the header declares, argument errors are reported before any device
work, and the host-side gradient plan covers every kept tile exactly once in
an order the dQ chain can follow."""

import os
import re

import numpy as np
import pytest

import attention_backward_tnd_b300 as tnd
from attention_backward_tnd_b300 import build as tbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INF = 2147483647


@pytest.fixture(scope="module", autouse=True)
def built():
    tbuild.build()


def header_functions():
    text = open(os.path.join(ROOT, "include", "tnd_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tnd_\w+)\s*\(", text)))


def test_library_exports_every_declared_entry_point():
    names = header_functions()
    assert "tnd_attn_grad" in names and "tnd_attn_fwd" in names
    L = tnd.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(tnd.SYMBOLS) == names


def test_status_strings():
    for s in range(8):
        assert tnd.tnd_status_string(s)
    assert tnd.tnd_status_string(99) == "unknown status"


def ws(dtype=tnd.TND_BF16, batch=2, cu_q=(0, 5, 9), cu_kv=(0, 5, 9), nq=4, nkv=2, d=128, scale=0.1, keep=1.0,
       pre=INF, nxt=INF, mode=3, drop=False, sink=False, amask=False, prefix=None, dv=None):
    return tnd.tnd_attn_grad_workspace_size(dtype, batch, list(cu_q), list(cu_kv), prefix, nq, nkv, d,
                                            d if dv is None else dv, scale, keep, pre, nxt, mode, drop, amask, sink)


def test_workspace_size_accepts_valid_problems():
    st, n = ws()
    assert st == tnd.TND_OK and n > 0
    st2, n2 = ws(cu_q=(0, 500, 900), cu_kv=(0, 500, 900))
    assert st2 == tnd.TND_OK and n2 > n
    assert tnd.tnd_attn_fwd_workspace_size(tnd.TND_F32, 2, [0, 5, 9], [0, 5, 9], None, 4, 2, 64, 64, 0.1, 1.0, INF,
                                           INF, 0, False, False, False)[0] == tnd.TND_OK
    # a value head dim below the query / key one (qD == kD >= vD) runs on the CUDA-core kernels,
    # which take no tensor-core dQ accumulator
    assert ws(dv=64)[0] == tnd.TND_OK and ws(dv=64)[1] < ws()[1]
    assert ws(d=96, dv=1)[0] == tnd.TND_OK
    # the packed matrix of the tensor-core kernels takes workspace
    assert ws(mode=1, amask=True)[1] > ws(mode=0)[1]
    assert ws(mode=6, prefix=[2, 4])[0] == tnd.TND_OK
    assert ws(mode=0, amask=True, pre=2, nxt=0)[0] == tnd.TND_OK
    assert ws(mode=0, amask=True, cu_kv=(0, 7, 9))[0] == tnd.TND_OK       # matrix with Sq != Skv
    assert ws(mode=3, amask=True)[1] == ws(mode=3)[1]                     # not read by index rules


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=7), tnd.TND_ERR_INVALID),
    (dict(batch=0, cu_q=(0,), cu_kv=(0,)), tnd.TND_ERR_INVALID),
    (dict(cu_q=(1, 5, 9)), tnd.TND_ERR_INVALID),
    (dict(cu_q=(0, 6, 5)), tnd.TND_ERR_INVALID),
    (dict(cu_q=(0, 0, 0)), tnd.TND_ERR_INVALID),                  # T = 0
    (dict(cu_q=(0, 1 << 20, (1 << 20) + 1)), tnd.TND_ERR_INVALID),  # T > 1M
    (dict(nq=3, nkv=2), tnd.TND_ERR_INVALID),                     # Nq % Nkv != 0
    (dict(nq=512, nkv=2), tnd.TND_ERR_INVALID),                   # N > 256
    (dict(nq=0), tnd.TND_ERR_INVALID),
    (dict(d=0), tnd.TND_ERR_INVALID),
    (dict(d=1024), tnd.TND_ERR_INVALID),                          # D > 768
    (dict(keep=0.0, drop=True), tnd.TND_ERR_INVALID),
    (dict(keep=1.5), tnd.TND_ERR_INVALID),
    (dict(keep=0.5, drop=False), tnd.TND_ERR_NULLPTR),            # dropMask needed
    (dict(scale=float("nan")), tnd.TND_ERR_INVALID),
    (dict(mode=9), tnd.TND_ERR_INVALID),
    (dict(mode=4, pre=-3, nxt=1), tnd.TND_ERR_INVALID),           # empty band
    (dict(mode=1), tnd.TND_ERR_NULLPTR),                          # the matrix is the mask
    (dict(mode=6), tnd.TND_ERR_NULLPTR),                          # prefix needed
    (dict(mode=6, prefix=[2, 5]), tnd.TND_ERR_INVALID),           # prefix > Skv
    (dict(mode=6, prefix=[-1, 0]), tnd.TND_ERR_INVALID),
    (dict(mode=6, batch=1025, cu_q=tuple(range(1026)), cu_kv=tuple(range(1026)), prefix=[0] * 1025),
     tnd.TND_ERR_INVALID),                                        # B > 1K with prefix
    (dict(mode=0, amask=True, pre=-3, nxt=1), tnd.TND_ERR_INVALID),  # empty band with the matrix
    (dict(mode=5), tnd.TND_ERR_UNSUPPORTED),
    (dict(mode=7), tnd.TND_ERR_UNSUPPORTED),
    (dict(mode=8), tnd.TND_ERR_UNSUPPORTED),
    (dict(mode=4, pre=3, nxt=0, cu_kv=(0, 6, 9)), tnd.TND_ERR_UNSUPPORTED),  # band with Sq != Skv
    (dict(d=769), tnd.TND_ERR_INVALID),                           # D > 768
    (dict(dv=129), tnd.TND_ERR_INVALID),                          # vD > qD
    (dict(dv=0), tnd.TND_ERR_INVALID),
])
def test_workspace_size_rejects(kw, expect):
    assert ws(**kw)[0] == expect


def test_null_workspace_size_pointer_and_seqlens():
    L = tnd.lib()
    assert L.tnd_attn_grad_workspace_size(1, 1, None, None, None, 1, 1, 128, 128, 0.1, 1.0, 0, 0, 0, 0, 0, 0,
                                          None) == \
        tnd.TND_ERR_NULLPTR


def _grad_call(**over):
    """tnd_attn_grad with fake aligned device addresses; only arguments that
    fail validation are used, so nothing is ever dereferenced."""
    args = dict(query=4096, key=4096, value=4096, dy=4096, pse=None, pse_batch=0, pse_type=1, drop_mask=None,
                atten_mask=None, softmax_max=4096,
                softmax_sum=4096, attention_in=4096, sink=None, dtype=tnd.TND_BF16, batch=1, cu_q=[0, 8],
                cu_kv=[0, 8], prefix=None, head_num=2, kv_head_num=1, head_dim=128, value_head_dim=128,
                scale_value=0.1,
                keep_prob=1.0, pre_tokens=INF, next_tokens=INF,
                sparse_mode=3, dq=4096, dk=4096, dv=4096, dsink=None, workspace=None, workspace_size=0, stream=None)
    args.update(over)
    return tnd.tnd_attn_grad(*args.values())


@pytest.mark.parametrize("over,expect", [
    (dict(query=None), tnd.TND_ERR_NULLPTR),
    (dict(dy=None), tnd.TND_ERR_NULLPTR),
    (dict(attention_in=None), tnd.TND_ERR_NULLPTR),
    (dict(dv=None), tnd.TND_ERR_NULLPTR),
    (dict(sink=4096, dsink=None), tnd.TND_ERR_NULLPTR),
    (dict(keep_prob=0.9), tnd.TND_ERR_NULLPTR),
    (dict(sparse_mode=1), tnd.TND_ERR_NULLPTR),                  # no attention-mask matrix
    (dict(sparse_mode=6), tnd.TND_ERR_NULLPTR),                  # no prefix
    (dict(sparse_mode=6, prefix=[9]), tnd.TND_ERR_INVALID),
    (dict(pse=4096, pse_batch=1, sparse_mode=0), tnd.TND_ERR_UNSUPPORTED),   # pse needs a lower triangle
    (dict(pse=4096, pse_batch=1, pse_type=2, sparse_mode=0), tnd.TND_ERR_UNSUPPORTED),  # generated: lower triangle
    (dict(pse=4096, pse_batch=1, pse_type=3, cu_kv=[0, 9]), tnd.TND_ERR_UNSUPPORTED),   # generated: Sq == Skv
    (dict(pse=4096, pse_batch=2, pse_type=2), tnd.TND_ERR_INVALID),                     # slopes [B, N] or [N]
    (dict(pse=4096, pse_batch=1, pse_type=-1), tnd.TND_ERR_INVALID),
    (dict(pse=4096, pse_batch=1, pse_type=5), tnd.TND_ERR_INVALID),
    (dict(pse=4096, pse_batch=3), tnd.TND_ERR_INVALID),                      # first dim is 1 or B
    (dict(pse=4098, pse_batch=1), tnd.TND_ERR_INVALID),                      # misaligned
    (dict(pse=4096, pse_batch=1, cu_kv=[0, 9]), tnd.TND_ERR_UNSUPPORTED),    # Sq != Skv
    (dict(head_num=3, kv_head_num=2), tnd.TND_ERR_INVALID),
    (dict(value_head_dim=256), tnd.TND_ERR_INVALID),             # vD > qD
    (dict(query=4098), tnd.TND_ERR_INVALID),                     # misaligned
    (dict(workspace=None, workspace_size=0), tnd.TND_ERR_WORKSPACE),
    (dict(workspace=4096, workspace_size=16), tnd.TND_ERR_WORKSPACE),
    (dict(workspace=4096 + 16, workspace_size=1 << 30), tnd.TND_ERR_WORKSPACE),  # not 256-aligned
])
def test_grad_rejects_before_device_work(over, expect):
    assert _grad_call(**over) == expect


def test_set_option_checks_values():
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, 5) == tnd.TND_ERR_INVALID
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_WAIT_LIMIT_MS, 0) == tnd.TND_ERR_INVALID
    assert tnd.tnd_attn_set_option(99, 0) == tnd.TND_ERR_INVALID
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, 0) == tnd.TND_OK
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_TEST_SKIP_LOAD, 2) == tnd.TND_ERR_INVALID
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_TEST_SKIP_LOAD, 0) == tnd.TND_OK
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, 2) == tnd.TND_ERR_INVALID
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, 0) == tnd.TND_OK
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, 1) == tnd.TND_OK


# ---------------------------------------------------------------------------
# host-side gradient plan
# ---------------------------------------------------------------------------

def _keep(mode, pre, nxt, sq, skv, i, j, prefix_n=0):
    if mode == 0:
        return True
    if mode == 2:
        return j <= i
    if mode == 3:
        return j <= i + skv - sq
    if mode == 6:
        return j <= i + skv - sq or j < prefix_n
    return -pre <= j - i <= nxt


def _tiles(mode, pre, nxt, sq, skv, prefix_n=0):
    """Brute force: set of (q block, kv block) with a kept pair, and kept pairs."""
    tiles, kept = set(), 0
    for i in range(sq):
        for j in range(skv):
            if _keep(mode, pre, nxt, sq, skv, i, j, prefix_n):
                tiles.add((i // 128, j // 128))
                kept += 1
    return tiles, kept


PLANS = [
    ([300, 129, 1, 0, 700], [300, 129, 1, 5, 700], 4, 2, 3, INF, INF),
    ([400, 50], [100, 600], 2, 2, 3, INF, INF),
    ([700, 257], [700, 257], 2, 1, 4, 200, 0),
    ([700, 257], [700, 257], 2, 1, 4, 30, 150),
    ([130, 65], [500, 7], 2, 2, 0, INF, INF),
    ([260, 90], [130, 300], 2, 1, 2, INF, INF),
    ([300, 129, 200], [300, 400, 100], 2, 1, 6, INF, INF, [170, 390, 0]),
    ([500, 60], [200, 500], 4, 2, 6, INF, INF, [200, 1]),
]


def _plan_case(case):
    sq, skv, nq, nkv, mode, pre, nxt = PLANS[case][:7]
    prefix = PLANS[case][7] if len(PLANS[case]) > 7 else None
    return sq, skv, nq, nkv, mode, pre, nxt, prefix


@pytest.mark.parametrize("case", range(len(PLANS)))
def test_plan_covers_every_kept_tile_once_in_chain_order(case):
    sq, skv, nq, nkv, mode, pre, nxt, prefix = _plan_case(case)
    cu_q = np.concatenate([[0], np.cumsum(sq)])
    cu_kv = np.concatenate([[0], np.cumsum(skv)])
    st, units, kept = tnd.tnd_attn_grad_plan(len(sq), cu_q, cu_kv, nq, nkv, pre, nxt, mode, prefix=prefix)
    assert st == tnd.TND_OK
    seen = {}
    order = {}
    total_kept = 0
    for b in range(len(sq)):
        tiles, k = _tiles(mode, pre, nxt, sq[b], skv[b], 0 if prefix is None else prefix[b])
        total_kept += k * nq
        for g in range(nkv):
            for (qb, j) in tiles:
                seen[(b, g, qb, j)] = 0
    for pos, (b, g, j, lo, hi) in enumerate(units):
        for qb in range(lo, hi):
            key = (b, g, qb, j)
            assert key in seen, f"unit visits an empty tile {key}"
            seen[key] += 1
            order.setdefault((b, g, qb), []).append((pos, j))
    assert all(v == 1 for v in seen.values()), "a kept tile is missed or visited twice"
    assert kept == total_kept
    # every kv block of every (sequence, kv head) is a unit (it writes dK/dV)
    nunits = sum(nkv * ((s + 127) // 128) for s in skv)
    assert len(units) == nunits
    # the dQ chain of a q block runs from its highest kv block down: those
    # units must be taken in that order
    for (b, g, qb), lst in order.items():
        js = [j for _, j in sorted(lst)]
        assert js == sorted(js, reverse=True), (b, g, qb, js)


L2_GROUP_BYTES = 48 << 20       # q-side bytes the units of one head group may sweep (tnd_api.cu)


def _check_unit_order(sq, skv, nq, nkv, mode, pre, nxt, prefix, d=128):
    # per sequence (more tiles first): kv heads in groups sized to the L2
    # share; within a group, kv block by kv block (descending), the group's
    # heads of a block in a row
    cu_q = np.concatenate([[0], np.cumsum(sq)])
    cu_kv = np.concatenate([[0], np.cumsum(skv)])
    st, units, _ = tnd.tnd_attn_grad_plan(len(sq), cu_q, cu_kv, nq, nkv, pre, nxt, mode, prefix=prefix)
    assert st == tnd.TND_OK
    seqs = []
    for u in units:
        if not seqs or seqs[-1][0] != int(u[0]):
            seqs.append((int(u[0]), []))
        seqs[-1][1].append(u)
    assert len({b for b, _ in seqs}) == len(seqs), "a sequence's units are split"
    for b, us in seqs:
        nqblk = (sq[b] + 127) // 128
        per_head = (nq // nkv) * nqblk * 128 * d * 8
        hg = max(1, min(nkv, L2_GROUP_BYTES // max(1, per_head)))
        pos = 0
        for g0 in range(0, nkv, hg):
            heads = list(range(g0, min(nkv, g0 + hg)))
            n_blocks = (skv[b] + 127) // 128
            expect_js = list(range(n_blocks - 1, -1, -1))
            chunk = us[pos:pos + n_blocks * len(heads)]
            pos += n_blocks * len(heads)
            assert [int(u[2]) for u in chunk[::len(heads)]] == expect_js, (b, g0)
            for i in range(0, len(chunk), len(heads)):
                assert [int(u[1]) for u in chunk[i:i + len(heads)]] == heads, (b, g0, i)
                assert len({int(u[2]) for u in chunk[i:i + len(heads)]}) == 1
        assert pos == len(us)
    work = {b: sum(int(u[4] - u[3]) + 1 for u in us if u[1] == 0) for b, us in seqs}
    ws = [work[b] for b, _ in seqs]
    assert ws == sorted(ws, reverse=True), ws
    return seqs


@pytest.mark.parametrize("case", range(len(PLANS)))
def test_plan_hands_out_kv_heads_of_a_block_together(case):
    _check_unit_order(*_plan_case(case))


def test_plan_groups_kv_heads_of_long_sequences():
    # 8192 q rows, 32 query heads on 8 kv heads: one kv head's q-side tiles
    # (4 heads x 64 q blocks x 128 KB = 32 MB) fit the L2 share, two do not
    seqs = _check_unit_order([8192, 1000], [8192, 1000], 32, 8, 3, INF, INF, None)
    long_units = seqs[0][1]
    assert [int(u[1]) for u in long_units[:64]] == [0] * 64
    # the short sequence keeps all its heads together
    assert [int(u[1]) for u in seqs[1][1][:8]] == list(range(8))
