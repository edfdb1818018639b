"""The CUDA twin of the input generator is bit-identical to the numpy twin."""
import numpy as np
import pytest

import moe_inputs
from moe_inputs import configs, host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_device_generator_matches_host_elementwise(dtype):
    cfg = configs.make_shape(1000, 512, 16, 2, 128, Fs=64, dtype=dtype, score=configs.SIGMOID,
                             bias_range=0.01, seed=77)
    for name in moe_inputs.tensor_names(cfg):
        d = moe_inputs.device_tensor(cfg, name)
        h = moe_inputs.host_tensor(cfg, name)
        if d.dtype == torch.bfloat16:
            got = d.view(torch.int16).cpu().numpy().view(np.uint16)
        else:
            got = d.cpu().numpy()
        np.testing.assert_array_equal(got.reshape(h.shape), h, err_msg=name)


def test_device_generator_matches_host_at_large_indices():
    """Samples of a 15 GB tensor (the DeepSeek-V3-shaped gate/up weights)."""
    cfg = configs.CONFIGS[2]
    w = moe_inputs.device_tensor(cfg, "w_gate_up")
    flat = w.view(-1)
    rng = np.random.default_rng(5)
    idx = np.concatenate([rng.integers(0, flat.numel(), 20000), [0, flat.numel() - 1]])
    got = flat[torch.from_numpy(idx).to(w.device)].view(torch.int16).cpu().numpy().view(np.uint16)
    want = host.normal(idx.astype(np.uint64), cfg["seed"], configs.TID_W_GATE_UP,
                       moe_inputs.std_of(cfg, "w_gate_up"), "bf16")
    np.testing.assert_array_equal(got, want)
    del w, flat
    torch.cuda.empty_cache()


def test_zipf_patch_is_identical_on_device():
    cfg = configs.make_shape(64, 128, 128, 8, 64, zipf=dict(s=1.2, scale=2.0), groups=8, seed=4)
    for name in ("x", "w_router"):
        d = moe_inputs.device_tensor(cfg, name).view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(d, moe_inputs.host_tensor(cfg, name))
