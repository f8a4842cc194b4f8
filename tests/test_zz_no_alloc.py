"""The gradient entry point that allocates nothing (tnd_attn_grad_static_ws).

It serves callers that cannot allocate device memory, such as a plug-in that
only gets buffers from its host framework's allocator, or a process that
reserved all device memory at start-up.  Its workspace is a fixed device
array inside the library.  This file is named so that pytest collects it last:
if it fails, a run that stops at the first failure has already run every
other test.
"""

import ctypes

import pytest

import attention_backward_tnd_b300 as tnd
import workloads

INF = 2147483647


def _call_static(dev, wl, outs, stream):
    dq, dk, dv, dsink = outs
    return tnd.tnd_attn_grad_static_ws(
        dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), dev["dy"].data_ptr(),
        None if dev["mask"] is None else dev["mask"].data_ptr(), dev["smax"].data_ptr(), dev["ssum"].data_ptr(),
        dev["out"].data_ptr(), None if dev["sink"] is None else dev["sink"].data_ptr(),
        tnd.dtype_code(dev["q"]), wl.batch, wl.cu_q, wl.cu_kv, wl.nq, wl.nkv, wl.d, wl.scale, wl.keep_prob,
        wl.pre_tokens, wl.next_tokens, wl.sparse_mode, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
        None if dsink is None else dsink.data_ptr(), stream)


def test_static_ws_rejects_problems_beyond_its_capacity():
    # dQ accumulator alone: 40000 x 32 x 128 x 4 B > 32 MiB; checked before any device work
    dummy = ctypes.c_void_p(16)
    st = tnd.tnd_attn_grad_static_ws(dummy, dummy, dummy, dummy, None, dummy, dummy, dummy, None, tnd.TND_BF16, 1,
                                     [0, 40000], [0, 40000], 32, 8, 128, 0.088, 1.0, INF, INF, 3, dummy, dummy,
                                     dummy, None, None)
    assert st == tnd.TND_ERR_WORKSPACE


@pytest.mark.gpu
def test_static_ws_matches_workspace_entry_point_twice():
    """Both entry points run the same deterministic kernels, so their outputs
    must be bit-identical.  Problems run large, small, large again, each call
    twice in a row, so a stale word left in the shared array by a larger or
    an earlier call would show."""
    torch = pytest.importorskip("torch")
    from tests import gpu_helpers as gh

    large = workloads.custom("static_ws_causal_sink", "bf16", [300, 77, 129], [300, 77, 129], 4, 2, 128,
                             sparse_mode=3, has_sink=True, seed=31)
    small = workloads.custom("static_ws_band_dropout", "bf16", [60, 19], [60, 19], 2, 1, 128,
                             keep_prob=0.9, pre_tokens=64, next_tokens=3, sparse_mode=4, seed=32)
    stream = torch.cuda.current_stream().cuda_stream
    prepared = {}
    for wl in (large, small):
        inp = workloads.make_inputs(wl)
        dev = gh.upload(inp)
        dev["out"], dev["smax"], dev["ssum"] = tnd.fwd(dev["q"], dev["k"], dev["v"], wl.cu_q, wl.cu_kv, wl.scale,
                                                       wl.keep_prob, wl.pre_tokens, wl.next_tokens,
                                                       wl.sparse_mode, dev["mask"], dev["sink"])
        ref = tnd.grad(dev["q"], dev["k"], dev["v"], dev["dy"], dev["out"], dev["smax"], dev["ssum"], wl.cu_q,
                       wl.cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens, wl.next_tokens, wl.sparse_mode,
                       dev["mask"], dev["sink"])
        prepared[wl.name] = (dev, ref)
    for wl in (large, small, large):
        dev, ref = prepared[wl.name]
        for _ in range(2):
            outs = (torch.full_like(dev["q"], float("nan")), torch.full_like(dev["k"], float("nan")),
                    torch.full_like(dev["v"], float("nan")),
                    None if dev["sink"] is None else torch.full((wl.nq,), float("nan"), device="cuda"))
            st = _call_static(dev, wl, outs, stream)
            assert st == tnd.TND_OK, tnd.tnd_status_string(st)
            st = tnd.tnd_attn_grad_static_ws_status(stream)
            assert st == tnd.TND_OK, tnd.tnd_status_string(st)
            for name, got, want in zip(("dq", "dk", "dv", "dsink"), outs, ref):
                if want is None:
                    continue
                assert got.dtype == want.dtype
                bits = torch.int16 if got.element_size() == 2 else torch.int32
                assert torch.equal(got.view(bits), want.view(bits)), (wl.name, name)
