"""The failure path of the library, on the GPU, without a GPU fault.

Every device-side wait in the library is bounded; a wait that runs out makes
its kernel record a timeout in the device error word and return, and a range
check that fails records an error and skips the access. The host learns of
either through the word (df_moe_sync), through df_moe_forward_host after its
own synchronisation, or at the next forward call, which then launches nothing.

The timeout is provoked with the library's test hook: the next forward's
gate/up phase leaves one pipeline stage unfilled, so the consumers' bounded
wait (shortened by the hook) runs out. Nothing traps and nothing hangs: the
call ends with wrong results and an error code, and the call after it is
clean and matches the oracle.

The range check is provoked through a single-step entry point that takes the
caller's expert ids: an id outside [0, E) is left out by the grouping kernel
and reported as EDEVICE.
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import Setup, check_ids_weights, check_out, draw_tokens, to_dev_bf16

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS[0]
ETIMEOUT, EDEVICE = -6, -7


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def tiny(torch):
    s = Setup(WL, max_tokens=8)
    yield s
    s.close()


def _host_forward(m, x, T):
    out = np.empty((T, WL.H), dtype=np.uint16)
    out32 = np.empty((T, WL.H), dtype=np.float32)
    ids = np.empty((T, WL.k), dtype=np.int32)
    w = np.empty((T, WL.k), dtype=np.float32)
    m.forward_host(x, T, out, ids=ids, weights=w, out_f32=out32)
    return out32, ids, w


def _check(tiny, x, got):
    out32, ids, w = got
    ref = orc.moe_layer(tiny.layers[0], x)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


@pytest.mark.parametrize("T", [1, 2, 8])
def test_forward_host_reports_its_own_timeout_then_recovers(tiny, torch, T):
    import mxfp4_routed_expert_top_gb300 as dfm
    x = draw_tokens(tiny, T, first_id=20000 + 10 * T)
    tiny.m.test_drop_arrival()
    with pytest.raises(dfm.DfMoeError) as ei:
        _host_forward(tiny.m, x, T)
    assert ei.value.code == ETIMEOUT
    assert "gave up" in str(ei.value)
    # the error was cleared: the next call runs and is right
    _check(tiny, x, _host_forward(tiny.m, x, T))
    tiny.m.sync()  # nothing left in the error word


def test_sync_reports_a_timeout(tiny, torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    x = draw_tokens(tiny, 1, first_id=20100)
    xd = to_dev_bf16(x)
    out = torch.empty((1, WL.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((1, WL.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, WL.k), dtype=torch.float32, device="cuda")
    tiny.m.test_drop_arrival()
    tiny.m.forward(xd, 1, out, ids, w, out_f32=out32)   # enqueued: no error yet
    with pytest.raises(dfm.DfMoeError) as ei:
        tiny.m.sync()
    assert ei.value.code == ETIMEOUT
    tiny.m.forward(xd, 1, out, ids, w, out_f32=out32)
    tiny.m.sync()
    _check(tiny, x, (out32.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()))


def test_next_forward_reports_an_earlier_timeout(tiny, torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    x = draw_tokens(tiny, 1, first_id=20200)
    xd = to_dev_bf16(x)
    out = torch.empty((1, WL.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((1, WL.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, WL.k), dtype=torch.float32, device="cuda")
    tiny.m.test_drop_arrival()
    tiny.m.forward(xd, 1, out, ids, w, out_f32=out32)
    torch.cuda.synchronize()   # the call has ended; its last kernel published the word
    out32.fill_(12345.0)
    with pytest.raises(dfm.DfMoeError) as ei:
        tiny.m.forward(xd, 1, out, ids, w, out_f32=out32)
    assert ei.value.code == ETIMEOUT
    torch.cuda.synchronize()
    assert np.all(out32.cpu().numpy() == 12345.0)   # that call launched nothing
    tiny.m.forward(xd, 1, out, ids, w, out_f32=out32)
    tiny.m.sync()
    _check(tiny, x, (out32.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()))


def test_out_of_range_id_is_skipped_and_reported(tiny, torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    T = 2
    x = draw_tokens(tiny, T, first_id=20300)
    ids = np.array([[1, 5], [WL.E + 3, 2]], dtype=np.int32)   # one id out of range
    hbuf = torch.zeros((T * WL.k, WL.I), dtype=torch.float32, device="cuda")
    tiny.m.step_expert_gateup(0, to_dev_bf16(x), T, torch.from_numpy(ids).cuda(), hbuf)
    with pytest.raises(dfm.DfMoeError) as ei:
        tiny.m.sync()
    assert ei.value.code == EDEVICE
    got = hbuf.cpu().double().numpy()
    # the valid assignments are still computed; the bad one is left untouched
    for t, j in ((0, 0), (0, 1), (1, 1)):
        ref = orc.expert_gateup(tiny._span(0, ids[t, j]), WL.H, WL.I,
                                (x[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        assert np.linalg.norm(got[t * WL.k + j] - ref) <= 1e-5 * np.linalg.norm(ref)
    assert np.all(got[1 * WL.k + 0] == 0.0)
    # and the handle is clean afterwards
    _check(tiny, x, _host_forward(tiny.m, x, T))
