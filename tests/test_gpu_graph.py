"""The layer captured as a CUDA graph (moe_forward_graph / moe_graph_launch):
replays give bit for bit the output of the plain call, follow new contents of
x, and count their kernels in moe_launch_count."""

import pytest
import torch

from mixture_experts_layer_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


def _layer(T, d, E, k, I, I_shared=0, zipf=False, seed=0):
    w = W.Workload("graph", T, d, E, k, I, I_shared=I_shared, zipf_bias=zipf, seed=seed)
    return w, W.make_x(w, device="cuda"), W.make_weights(w, device="cuda")


@pytest.mark.parametrize("T,d,E,k,I,Is,zipf", [(64, 512, 32, 8, 256, 0, False),
                                               (300, 512, 16, 4, 384, 256, True)])
def test_device_graph_matches_plain_call(moe, T, d, E, k, I, Is, zipf):
    w, x, p = _layer(T, d, E, k, I, I_shared=Is, zipf=zipf, seed=T)
    kw = dict(router_bias=p["router_bias"], w_gate_up_shared=p["w_gate_up_shared"],
              w_down_shared=p["w_down_shared"])
    ref = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k, **kw)
    x_in = x.clone()
    out = torch.empty_like(ref)
    ws = moe.new_workspace(T, d, E, I, k, Is)
    g = moe.ForwardGraph(x_in, p["w_router"], p["w_gate_up"], p["w_down"], k, out, ws, **kw)
    n0 = moe.moe_launch_count()
    g.launch()
    g.launch()
    torch.cuda.synchronize()
    per_replay = (moe.moe_launch_count() - n0) // 2
    assert per_replay >= 5
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert torch.equal(out, ref)
    # new contents of x, same graph
    x2 = W.make_x(W.Workload("graph2", T, d, E, k, I, seed=T + 99), device="cuda")
    x_in.copy_(x2)
    g.launch()
    torch.cuda.synchronize()
    ref2 = moe.moe_forward(x2, p["w_router"], p["w_gate_up"], p["w_down"], k, **kw)
    assert torch.equal(out, ref2)
    g.close()


def test_host_graph_matches_plain_call(moe):
    T, d, E, k, I = 64, 1024, 64, 8, 256
    w, x, p = _layer(T, d, E, k, I, seed=5)
    ref = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k)
    x_host = x.cpu().pin_memory()
    out_host = torch.zeros((T, d), dtype=torch.bfloat16).pin_memory()
    ws = moe.new_workspace(T, d, E, I, k)
    g = moe.ForwardGraph(x_host, p["w_router"], p["w_gate_up"], p["w_down"], k, out_host, ws)
    assert (out_host == 0).all()  # capture runs nothing
    g.launch()
    torch.cuda.synchronize()
    assert torch.equal(out_host, ref.cpu())
    g.close()


def test_graph_rejects_bad_arguments(moe):
    w, x, p = _layer(16, 256, 8, 2, 128)
    out = torch.empty((16, 256), dtype=torch.bfloat16)  # host out with device x
    ws = moe.new_workspace(16, 256, 8, 128, 2)
    with pytest.raises(ValueError):
        moe.ForwardGraph(x, p["w_router"], p["w_gate_up"], p["w_down"], 2, out, ws)
