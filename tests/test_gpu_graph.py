"""A forward pass captured in a CUDA graph replays with the results of eager calls.

The layer enqueues everything on the caller's stream, keeps the expert counts and the tile
schedule on the device and never synchronises with the host inside a call, so a fixed-shape
pass (the decode-serving form) can be captured once and replayed on new tokens written into
the captured input buffer.  The kernels are deterministic, so replay and eager results must be
identical bit for bit.
"""
import numpy as np
import pytest

import moe_inputs
from moe_inputs.configs import SIGMOID, SOFTMAX, make_shape

from layer_check import gpu_forward, group_args, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_83_b300 as moe
    moe.lib()


CASES = {
    # decode-sized segments (narrow CTA pairs), shared expert, sigmoid + bias
    "bf16_decode_like": make_shape(64, 256, 32, 8, 128, Fs=128, score=SIGMOID, bias_range=0.01,
                                   seed=31),
    # segments of about 256 rows (wide CTA pairs, tall and wide tiles)
    "bf16_prefill_like": make_shape(1024, 256, 8, 2, 256, score=SOFTMAX, seed=32),
    # group-limited routing and an expert capacity inside the captured pass
    "bf16_groups_capacity": dict(make_shape(512, 128, 16, 4, 128, score=SIGMOID,
                                            bias_range=0.01, seed=34, groups=4),
                                 topk_groups=2, capacity_factor=1.0),
    # rerouting of the overflow at an expert capacity: its fixed number of rounds is captured too
    "bf16_reroute": dict(make_shape(400, 128, 16, 2, 128, Fs=64, score=SOFTMAX, seed=35),
                         capacity_factor=1.0, reroute=3),
    # true-fp32 CUDA-core path
    "f32_ragged": make_shape(33, 70, 5, 2, 33, Fs=17, dtype="f32", seed=33),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_replays_from_a_cuda_graph(name):
    import mixture_experts_layer_83_b300 as moe
    cfg = CASES[name]
    T, d, E, k = cfg["T"], cfg["d"], cfg["E"], cfg["k"]
    dev = moe_inputs.upload(cfg, moe_inputs.host_inputs(cfg))
    cfg2 = dict(cfg, seed=cfg["seed"] + 1000)
    x2 = moe_inputs.upload(cfg2, {"x": moe_inputs.host_tensor(cfg2, "x")})["x"]
    ref = [to_host(gpu_forward(cfg, dev)), to_host(gpu_forward(cfg, dict(dev, x=x2)))]

    dt = moe.MOE_DTYPE_BF16 if cfg["dtype"] == "bf16" else moe.MOE_DTYPE_F32
    shape = moe.make_shape(T, d, E, k, cfg["F"], cfg["Fs"], dt)
    ws_bytes = moe.moe_layer_workspace_size(shape)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    x = dev["x"].clone()
    out = torch.empty_like(x)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    tidx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    st = torch.empty(T * k, dtype=torch.int32, device="cuda")
    dropped = torch.zeros(4, dtype=torch.int32, device="cuda")
    shared = (dev["sh_gate_up"], dev["sh_down"]) if cfg["Fs"] > 0 else None
    cf = cfg.get("capacity_factor", 0.0)

    def call():
        moe.moe_layer_forward(shape, x, dev["w_router"], dev["w_gate_up"], dev["w_down"],
                              cfg["score"], dev.get("bias"), shared, out, counts, ws, ws_bytes,
                              None, tidx, tw, st, capacity_factor=cf,
                              dropped=dropped if cf > 0 else None, reroute=cfg.get("reroute", 0),
                              **group_args(cfg))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()   # first call outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()

    for i, xi in enumerate((dev["x"], x2)):
        out.zero_()
        counts.zero_()
        x.copy_(xi)
        graph.replay()
        torch.cuda.synchronize()
        got = {"out": out, "counts": counts, "topk_idx": tidx, "topk_w": tw}
        if cf == 0:
            got["sorted_token"] = st
        for key, v in got.items():
            g = v.float().cpu().numpy().astype(np.float64) if v.dtype == torch.bfloat16 \
                else v.cpu().numpy()
            np.testing.assert_array_equal(g, ref[i][key], err_msg=f"{name} batch {i} {key}")
        if cf > 0:
            R = int(counts.sum().item())
            np.testing.assert_array_equal(st.cpu().numpy()[:R], ref[i]["sorted_token"][:R])
            assert int(dropped[0].item()) == int(ref[i]["dropped"][0])
    assert moe.moe_workspace_status(ws) == (moe.MOE_OK, 0)
