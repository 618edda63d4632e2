"""Graph-safe decode: the fused decode kernel updates the state (and the ring) in place, so a
decode step with stable pointers can be captured once in a CUDA graph and replayed.  In place ==
out of place bit for bit; K graph replays (new token rows copied into the captured input buffers
before each) == K eager one-token calls bit for bit."""

import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

ROWS = ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _call(d, state_in, state_out, ring_in, ring_out, y, N, T, H):
    from gated_delta_rule_scan_gb300 import kda
    kda.kda_decode_fused(d["q_raw"], d["k_raw"], d["v_raw"], d["conv_w"], ring_in, ring_out,
                         d["f_raw"], d["dt_bias"], d["a_log"], d["beta_raw"], state_in, state_out,
                         d["norm_w"], d["gate_raw"], y, N=N, T=T, H=H)


@pytest.mark.parametrize("T", [1, 4])
def test_in_place_equals_out_of_place(T):
    N, H = 8, 16
    d = to_dev(inputs.decode_step(N=N, T=T, H=H, seed=90 + T))
    s_out, r_out = torch.empty_like(d["state_in"]), torch.empty_like(d["ring_in"])
    y1, y2 = torch.empty(N * T, H * 128, device="cuda"), torch.empty(N * T, H * 128, device="cuda")
    _call(d, d["state_in"], s_out, d["ring_in"], r_out, y1, N, T, H)
    s_ip, r_ip = d["state_in"].clone(), d["ring_in"].clone()
    _call(d, s_ip, s_ip, r_ip, r_ip, y2, N, T, H)
    torch.cuda.synchronize()
    assert torch.equal(s_ip, s_out)
    assert torch.equal(r_ip, r_out)
    assert torch.equal(y1, y2)


def test_graph_replay_equals_eager_decode():
    N, H, K = 8, 16, 5
    steps = [to_dev(inputs.decode_step(N=N, T=1, H=H, seed=100 + i)) for i in range(K)]
    first = steps[0]
    # eager reference: K one-token calls from the first step's state and ring
    state, ring = first["state_in"].clone(), first["ring_in"].clone()
    ys = []
    for d in steps:
        y = torch.empty(N, H * 128, device="cuda")
        _call({**d, "conv_w": first["conv_w"], "dt_bias": first["dt_bias"], "a_log": first["a_log"],
               "norm_w": first["norm_w"]}, state, state, ring, ring, y, N, 1, H)
        ys.append(y)
    torch.cuda.synchronize()
    # captured step: static input rows, state and ring updated in place
    static = {k: first[k].clone() for k in ROWS}
    static.update({k: first[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")})
    g_state, g_ring = first["state_in"].clone(), first["ring_in"].clone()
    g_y = torch.empty(N, H * 128, device="cuda")
    warm_s, warm_r = g_state.clone(), g_ring.clone()           # a warm-up call off the graph
    _call(static, warm_s, warm_s, warm_r, warm_r, torch.empty_like(g_y), N, 1, H)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(static, g_state, g_state, g_ring, g_ring, g_y, N, 1, H)
    # capture records without running: the state is still the initial one
    torch.cuda.synchronize()
    assert torch.equal(g_state, first["state_in"])
    for i, d in enumerate(steps):
        for k in ROWS:
            static[k].copy_(d[k])
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(g_y, ys[i]), i
    assert torch.equal(g_state, state)
    assert torch.equal(g_ring, ring)
