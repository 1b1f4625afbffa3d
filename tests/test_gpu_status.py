"""Device-side status reporting: bad indices are skipped and flagged (no
fault), and a device wait that runs out of time gives up with
MOE_ERR_TIMEOUT and leaves the context usable.

The timeout is provoked by shortening the bound on every wait to 1 ns, so the
first wait that is not already satisfied gives up.  The kernel then records
the timeout, drains its own copies and tensor-core work in flight, frees its
tensor memory and returns; the next call with the normal bound must succeed
and match a run made before."""

import pytest
import torch

from mixture_experts_layer_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


def _layer(T=300, d=512, E=16, k=4, I=256):
    w = W.Workload("s", T, d, E, k, I, seed=1)
    return w, W.make_x(w, device="cuda"), W.make_weights(w, device="cuda")


def test_bad_expert_ids_are_flagged(moe):
    ids, _ = W.random_routing(100, 8, 2, seed=2)
    ids[17, 1] = 8          # out of range
    ids[50, 0] = -3
    ws = moe.new_workspace(100, 64, 8, 64, 2)
    moe.moe_permute(ids.cuda(), 8, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert moe.moe_get_device_status(ws) == moe.MOE_OK   # reading clears it


def test_bad_offsets_are_flagged(moe):
    w, x, p = _layer()
    x_perm = torch.zeros((40, w.d), dtype=torch.bfloat16, device="cuda")
    offsets = torch.zeros(w.E + 1, dtype=torch.int32, device="cuda")
    offsets[5:] = 50        # ends past the 40 rows
    ws = moe.new_workspace(40, w.d, w.E, w.I, 1)
    moe.moe_expert_ffn(x_perm, offsets, p["w_gate_up"], p["w_down"], ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    offsets[5:] = 40
    offsets[3] = 45         # goes down
    moe.moe_expert_ffn(x_perm, offsets, p["w_gate_up"], p["w_down"], ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK


def test_bad_slot_positions_are_flagged(moe):
    y = torch.ones((20, 64), dtype=torch.float16, device="cuda")
    slot_pos = torch.arange(20, dtype=torch.int32, device="cuda").view(10, 2).contiguous()
    slot_pos[3, 1] = 20
    gates = torch.full((10, 2), 0.5, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = moe.moe_combine(y, slot_pos, gates, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert out[0].float().eq(1.0).all()


def _control_words_clear(ws):
    """Words 1.. of the status region: the expert GEMMs' tile counters, which
    every launch leaves at zero (moe.h), and the single-launch layer's
    counters, untouched here."""
    return bool(ws[:256].view(torch.int32)[1:].eq(0).all())


# 75 rows per expert: the GEMMs' static tile stride; 8: decode-sized, tiles
# taken from the workspace's counter by a scheduler warp.
@pytest.mark.parametrize("T", [300, 32])
def test_wait_timeout_is_reported_and_recoverable(moe, T):
    w, x, p = _layer(T=T)
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k)
    ref = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert _control_words_clear(ws)
    try:
        moe.moe_set_wait_timeout_ns(1)
        moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k, ws=ws)
        st = moe.moe_get_device_status(ws)
    finally:
        moe.moe_set_wait_timeout_ns(0)
    assert st == moe.MOE_ERR_TIMEOUT
    assert _control_words_clear(ws)   # also after every wait gave up
    again = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert torch.equal(again, ref)
    assert _control_words_clear(ws)


def test_y_outside_fp16_range_saturates_and_is_flagged(moe):
    """y is stored in fp16: finite outputs beyond +-65504 become +-65504 and
    the status word reports MOE_ERR_RANGE; outputs inside the range are
    unaffected.  W_down is scaled by a power of two, which scales the exact
    y by the same factor."""
    import numpy as np
    import oracle
    from tests.gpu_util import ExpertsOnHost, assert_layer_close, f64
    w = W.Workload("r", 48, 256, 2, 1, 128, seed=5)
    p = W.make_weights(w, device="cuda")
    x_perm = W.make_x(w, device="cuda")
    offsets = torch.tensor([0, 20, 48], dtype=torch.int32, device="cuda")
    y_ref = oracle.expert_ffn(f64(x_perm), offsets.cpu().numpy(), ExpertsOnHost(p["w_gate_up"]),
                              ExpertsOnHost(p["w_down"]))
    s = 2.0 ** int(np.ceil(np.log2(4 * 65504 / np.abs(y_ref).max())))  # max |y| in [4, 8) x 65504
    ws = moe.new_workspace(48, 256, 2, 128, 1)
    y = moe.moe_expert_ffn(x_perm, offsets, p["w_gate_up"], p["w_down"] * s, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_RANGE
    ref, got = y_ref * s, f64(y)
    hi = np.abs(ref) > 65504 * (1 + 2.0**-9)
    lo = np.abs(ref) < 65504 * (1 - 2.0**-9)
    assert hi.any() and lo.any()
    assert (got[hi] == np.sign(ref[hi]) * 65504).all()
    assert_layer_close(got[lo], ref[lo], "y inside the fp16 range")
    moe.moe_expert_ffn(x_perm, offsets, p["w_gate_up"], p["w_down"], ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK


def test_y_beyond_fp16_range_with_fp32_y(moe):
    """With y kept in fp32 an expert output beyond the fp16 range is neither
    saturated nor flagged: the whole layer with W_down scaled by a power of
    two (max |y| in [4, 8) x 65504) matches the oracle on the scaled weights,
    while the fp16-y layer reports MOE_ERR_RANGE."""
    import numpy as np
    import oracle
    from tests.gpu_util import ExpertsOnHost, assert_layer_close, f64
    w = W.Workload("r32", 48, 256, 4, 2, 128, seed=9)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    ref1 = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), ExpertsOnHost(p["w_gate_up"]),
                          ExpertsOnHost(p["w_down"]), 2)
    s = 2.0 ** int(np.ceil(np.log2(4 * 65504 / np.abs(ref1["y"]).max())))
    wd = (p["w_down"] * s).contiguous()
    ref = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), ExpertsOnHost(p["w_gate_up"]),
                         ExpertsOnHost(wd), 2)
    assert np.abs(ref["y"]).max() > 65504
    ws = moe.new_workspace(48, 256, 4, 128, 2, y_fp32=True)
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], wd, 2, ws=ws, y_fp32=True)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, 48, 256, 4, 128, 2, y_fp32=True)
    assert_layer_close(f64(v["y"]), ref["y"], "fp32 y beyond the fp16 range")
    assert_layer_close(f64(out), ref["out"], "out")
    ws16 = moe.new_workspace(48, 256, 4, 128, 2)
    moe.moe_forward(x, p["w_router"], p["w_gate_up"], wd, 2, ws=ws16)
    assert moe.moe_get_device_status(ws16) == moe.MOE_ERR_RANGE
