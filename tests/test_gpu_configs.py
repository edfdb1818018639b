"""Parity at the five full-size workloads, in the configuration bench.py times (device-resident
seeded inputs, one moe_layer_forward call): routing for every token, dispatch tables
bit-exactly, layer outputs on sampled tokens (all tokens for the tiny and decode layers)."""
import pytest

import moe_inputs
from moe_inputs import configs

from layer_check import sampled_check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SAMPLE = {0: 64, 1: 48, 2: 48, 3: 128, 4: 64}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("cfg_id", [0, 1, 2, 3, 4])
def test_full_size_config(cfg_id):
    c = configs.CONFIGS[cfg_id]
    dev = moe_inputs.device_inputs(c)
    torch.cuda.synchronize()
    stats = sampled_check(c, dev, n_sample=SAMPLE[cfg_id])
    print(c["name"], stats)
    del dev
    torch.cuda.empty_cache()
