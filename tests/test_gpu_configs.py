"""Parity at the five full-size workloads, in the configuration bench.py times (device-resident
seeded inputs, one moe_layer_forward call): routing for every token, dispatch tables
bit-exactly, layer outputs on 1024 sampled tokens plus every token on a tile edge of the
expert GEMMs (all tokens for the tiny and decode layers)."""
import pytest

import moe_inputs
from moe_inputs import configs

from layer_check import sampled_check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SAMPLE = {0: 64, 1: 1024, 2: 1024, 3: 128, 4: 1024}


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
    if SAMPLE[cfg_id] < c["T"] and c["dtype"] == "bf16":
        assert stats["sampled"] >= SAMPLE[cfg_id] and stats["edges"]["tile_rows"] > 0
    del dev
    torch.cuda.empty_cache()


def test_full_size_skewed_layer_with_group_limited_routing():
    """The Zipf-skewed layer (128 experts in its 8 contiguous groups of 16) with each token's
    experts limited to its 4 best groups: routing, dispatch tables and sampled outputs against
    the oracle's group-limited top-k."""
    c = dict(configs.CONFIGS[4], topk_groups=4)
    dev = moe_inputs.device_inputs(c)
    torch.cuda.synchronize()
    stats = sampled_check(c, dev, n_sample=SAMPLE[4])
    print(c["name"], "group-limited", stats)
    del dev
    torch.cuda.empty_cache()


def test_full_size_skewed_layer_with_capacity():
    """The Zipf-skewed layer (hottest experts at about 16x the mean load) with a capacity
    factor of 1.25: the hot experts overflow and their late tokens are dropped; dispatch
    tables and the number dropped bit-exactly, sampled outputs with drops contributing nothing."""
    c = dict(configs.CONFIGS[4], capacity_factor=1.25)
    dev = moe_inputs.device_inputs(c)
    torch.cuda.synchronize()
    stats = sampled_check(c, dev, n_sample=SAMPLE[4])
    print(c["name"], "capacity 1.25", stats)
    assert stats["dropped"] > 0
    del dev
    torch.cuda.empty_cache()


def test_full_size_skewed_layer_with_capacity_and_rerouting():
    """The Zipf-skewed layer with a capacity factor of 1.25 and up to 4 next-best experts per
    token: overflow of the hot experts moves to colder ones; the GPU's assignment is checked
    for validity (serving experts among each token's top-12, capacity, tables) and sampled
    outputs against the oracle under that assignment."""
    c = dict(configs.CONFIGS[4], capacity_factor=1.25, reroute=4)
    dev = moe_inputs.device_inputs(c)
    torch.cuda.synchronize()
    stats = sampled_check(c, dev, n_sample=SAMPLE[4])
    print(c["name"], "capacity 1.25 + reroute 4", stats)
    del dev
    torch.cuda.empty_cache()
