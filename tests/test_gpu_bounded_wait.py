"""Device-side waits end in a timeout status, not a hang.

The pages ask that a run whose device work cannot complete ends with a
timeout or error code ("aclnnFlashAttentionUnpaddingScoreGrad", constraints).
Every wait of the tensor-core gradient has a clock bound.  A test hook that
is off by default (TND_OPT_TEST_SKIP_LOAD) makes the first CTA never load its
first K tile, so the UMMA issuer's wait for it cannot finish: with a 5 ms
bound the call must report TND_ERR_DEVICE_TIMEOUT through
tnd_attn_device_status, and the next call on the same stream and workspace
must run normally and match the oracle (TMEM and the workspace came back
clean).  No fault, trap or unbounded wait is involved.
"""

import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import attention_backward_tnd_b300 as tnd  # noqa: E402
from tests import gpu_helpers as gh  # noqa: E402


def test_expired_wait_reports_timeout_and_next_call_is_clean():
    wl = workloads.custom("bounded_wait_causal", "bf16", [300, 200], [300, 200], 4, 2, 128, sparse_mode=3, seed=41)
    inp = workloads.make_inputs(wl)
    dev = gh.upload(inp)
    out, smax, ssum = tnd.fwd(dev["q"], dev["k"], dev["v"], wl.cu_q, wl.cu_kv, wl.scale, sparse_mode=wl.sparse_mode)
    ws = torch.empty(max(tnd.grad_workspace_bytes(dev["q"], dev["k"], wl.cu_q, wl.cu_kv, wl.scale,
                                                  sparse_mode=wl.sparse_mode), 256), dtype=torch.uint8, device="cuda")
    try:
        assert tnd.tnd_attn_set_option(tnd.TND_OPT_WAIT_LIMIT_MS, 5) == tnd.TND_OK
        assert tnd.tnd_attn_set_option(tnd.TND_OPT_TEST_SKIP_LOAD, 1) == tnd.TND_OK
        tnd.grad(dev["q"], dev["k"], dev["v"], dev["dy"], out, smax, ssum, wl.cu_q, wl.cu_kv, wl.scale,
                 sparse_mode=wl.sparse_mode, workspace=ws)
        st = tnd.device_status(ws)
        assert st == tnd.TND_ERR_DEVICE_TIMEOUT, tnd.tnd_status_string(st)
    finally:
        tnd.tnd_attn_set_option(tnd.TND_OPT_TEST_SKIP_LOAD, 0)
        tnd.tnd_attn_set_option(tnd.TND_OPT_WAIT_LIMIT_MS, 2000)
    dq, dk, dv, _ = tnd.grad(dev["q"], dev["k"], dev["v"], dev["dy"], out, smax, ssum, wl.cu_q, wl.cu_kv, wl.scale,
                             sparse_mode=wl.sparse_mode, workspace=ws)
    torch.cuda.synchronize()
    assert tnd.device_status(ws) == tnd.TND_OK
    ref = gh.oracle_reference(inp)
    got = {"out": out, "smax": smax, "ssum": ssum, "dq": dq, "dk": dk, "dv": dv, "dsink": None}
    gh.compare_all(inp, got, ref)

