"""mlp_swiglu_forward_host: the layer with x and y in page-locked host memory (on the
decode-size kernels the gate_up launch copies x itself, elsewhere a copy kernel runs first;
the down projection writes y straight into host memory).  Its output must equal the device-buffer
entry point bit for bit, also when consecutive calls chain layers through host memory
(the next call's x is the previous call's y)."""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import assert_close, bits_f64, to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

mse = pytest.importorskip("moe_shared_expert_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_shared_expert_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mse.lib()
    yield
    assert mse.poll_device_error() == 0


def host_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("T,H,I", [(64, 7168, 6144), (7, 384, 320), (300, 512, 256), (5, 40, 24)])
def test_host_io_matches_device_entry_point(T, H, I):
    x = W.make_custom(1500 + T, 0, (T, H))
    wgu = W.make_custom(1500 + T, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(1500 + T, 2, (H, I), 1 / math.sqrt(I))
    dgu, dwd = to_dev(wgu), to_dev(wd)
    ref = mse.mlp_swiglu_forward(to_dev(x), dgu, dwd)
    y = mse.mlp_swiglu_forward_host(host_bf16(x), dgu, dwd)
    torch.cuda.synchronize()
    assert torch.equal(y, ref.cpu())
    if T * H <= 64 * 7168:
        y_ref, _, _ = oracle.mlp_forward(x, wgu, wd)
        assert_close(bits_f64(to_bits(y)), bits_f64(y_ref), "host-buffer layer vs oracle")


def test_host_io_chained_layers_and_back_to_back_calls():
    # four layers chained through host memory (y of one call is x of the next), enqueued
    # back to back without synchronising, then the same chain through device buffers
    T, H, I = 64, 1024, 768
    x0 = W.make_custom(1600, 0, (T, H))
    ws_ = [(to_dev(W.make_custom(1601 + k, 1, (2 * I, H), 1 / math.sqrt(H))),
            to_dev(W.make_custom(1601 + k, 2, (H, I), 1 / math.sqrt(I)))) for k in range(4)]
    bufs = [host_bf16(x0)] + [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    ws = mse.new_host_workspace(T, H, I)
    for k in range(4):
        mse.mlp_swiglu_forward_host(bufs[k], ws_[k][0], ws_[k][1], y_host=bufs[k + 1], workspace=ws)
    torch.cuda.synchronize()
    d = to_dev(x0)
    for k in range(4):
        d = mse.mlp_swiglu_forward(d, ws_[k][0], ws_[k][1])
        torch.cuda.synchronize()
        assert torch.equal(bufs[k + 1], d.cpu()), f"layer {k}"


def test_host_io_pageable_memory_and_overlapping_buffers():
    T, H, I = 16, 384, 320
    x_bits = W.make_custom(1700, 0, (T, H))
    wgu = W.make_custom(1700, 1, (2 * I, H), 1 / math.sqrt(H))
    wd = W.make_custom(1700, 2, (H, I), 1 / math.sqrt(I))
    dgu, dwd = to_dev(wgu), to_dev(wd)
    ws = mse.new_host_workspace(T, H, I)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).clone()   # pageable
    y = torch.zeros((T, H), dtype=torch.bfloat16).pin_memory()
    st = mse.lib().mlp_swiglu_forward_host(x.data_ptr(), T, H, I, dgu.data_ptr(), dwd.data_ptr(), y.data_ptr(),
                                           y.numel(), ws.data_ptr(), ws.numel(),
                                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    # pageable memory is refused where the device cannot reach it, and where it can (e.g.
    # a Grace-based system: the GPU accesses pageable host memory) the result is exact
    assert mse.STATUS[st] in ("MSE_OK", "MSE_ERR_INVALID_ARG")
    if mse.STATUS[st] == "MSE_OK":
        assert torch.equal(y, mse.mlp_swiglu_forward(to_dev(x_bits), dgu, dwd).cpu())
    xy = torch.zeros((2 * T, H), dtype=torch.bfloat16).pin_memory()
    st = mse.lib().mlp_swiglu_forward_host(xy.data_ptr(), T, H, I, dgu.data_ptr(), dwd.data_ptr(),
                                           xy.data_ptr() + T * H, y.numel(), ws.data_ptr(), ws.numel(),
                                           torch.cuda.current_stream().cuda_stream)
    assert mse.STATUS[st] == "MSE_ERR_INVALID_ARG"            # x and y overlap
    torch.cuda.synchronize()


@pytest.mark.parametrize("copiers", [16, 1, 0])
@pytest.mark.parametrize("T", [64, 16])
def test_host_io_early_copies_alternate_buffers(T, copiers):
    """Independent calls streamed back to back: on the decode-size kernels the gate_up launch
    copies x itself, into the other of the workspace's two x buffers than the previous call,
    before the previous layer is complete.  Every call must give what the device entry point
    gives, including calls captured in a CUDA graph (those wait for the previous work) and
    replayed back to back, a change of T on the same workspace, and the calls after them;
    the copy-count words end zero.  copiers = 0: the separate copy kernel."""
    old = mse.set_tuning(mse.TUNE_HOST_X_COPIERS, copiers)
    try:
        _early_copies(T)
    finally:
        mse.set_tuning(mse.TUNE_HOST_X_COPIERS, old)


def _early_copies(T):
    w = W.DECODE_T64
    H, I = w.H, w.I
    wgu, wd = W.make_mlp_weights(w)
    g0, d0 = to_dev(wgu), to_dev(wd)
    gus = [g0, torch.roll(g0, 977, 0).contiguous()]
    wds = [d0, torch.roll(d0, 331, 0).contiguous()]
    xs = [W.make_custom(1800 + k, 0, (T, H)) for k in range(6)]
    refs = [[mse.mlp_swiglu_forward(to_dev(x), gus[c], wds[c]) for c in range(2)] for x in xs]
    xh = [host_bf16(x) for x in xs]
    ws = mse.new_host_workspace(T, H, I)
    ys = [torch.zeros((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(18)]
    for i, y in enumerate(ys):
        mse.mlp_swiglu_forward_host(xh[i % 6], gus[i % 2], wds[i % 2], y_host=y, workspace=ws)
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        assert torch.equal(y, refs[i % 6][i % 2].cpu()), f"call {i}"

    # a smaller T on the same workspace (its buffers move), then T again
    t2 = T // 2
    y2 = mse.mlp_swiglu_forward_host(xh[0][:t2].clone().pin_memory(), gus[0], wds[0], workspace=ws)
    y3 = mse.mlp_swiglu_forward_host(xh[1], gus[1], wds[1], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y2, mse.mlp_swiglu_forward(to_dev(xs[0][:t2]), gus[0], wds[0]).cpu())
    assert torch.equal(y3, refs[1][1].cpu())

    # graph capture: three calls, replayed back to back, then eager calls again
    side = torch.cuda.Stream()
    gy = [torch.zeros((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for k in range(3):
            mse.mlp_swiglu_forward_host(xh[k], gus[k % 2], wds[k % 2], y_host=gy[k], workspace=ws, stream=side)
    for _ in range(3):
        for y in gy:
            y.zero_()
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        for k in range(3):
            assert torch.equal(gy[k], refs[k][k % 2].cpu()), f"graph call {k}"
    for i, y in enumerate(ys[:6]):
        mse.mlp_swiglu_forward_host(xh[(i + 3) % 6], gus[i % 2], wds[i % 2], y_host=y, workspace=ws)
    torch.cuda.synchronize()
    for i, y in enumerate(ys[:6]):
        assert torch.equal(y, refs[(i + 3) % 6][i % 2].cpu()), f"call after graph {i}"
    assert mse.poll_device_error() == 0
    assert int(torch.count_nonzero(ws[:256]).item()) == 0
