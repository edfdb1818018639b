"""The allocation-free routing entry point, for callers that cannot allocate device memory.

Its results must equal moe_route_from_keys on the same keys, on consecutive calls that share
the library's fixed scratch array.  This file is collected last on purpose.
"""
import numpy as np
import pytest

import mixture_experts_layer_83_b300 as moe

torch = pytest.importorskip("torch")


def _keys(T, E, seed, ties):
    rng = np.random.default_rng(seed)
    key = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        key = (np.round(key * 4) / 4).astype(np.float32)
    score = rng.uniform(0.05, 1.0, (T, E)).astype(np.float32)
    return key, score


def _route(fn, T, E, k, key, score, with_workspace):
    dev = "cuda"
    kk, ss = torch.from_numpy(key).to(dev), torch.from_numpy(score).to(dev)
    out = dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
               w=torch.empty((T, k), dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               off=torch.empty(E + 1, dtype=torch.int32, device=dev),
               st=torch.empty(T * k, dtype=torch.int32, device=dev),
               sp=torch.empty((T, k), dtype=torch.int32, device=dev))
    shape = moe.make_shape(T, 64, E, k, 64)
    args = [shape, kk, ss, out["idx"], out["w"], out["counts"], out["off"], out["st"], out["sp"]]
    if with_workspace:
        ws = torch.empty(moe.moe_layer_workspace_size(shape), dtype=torch.uint8, device=dev)
        fn(*args, ws)
    else:
        fn(*args)
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in out.items()}


def test_oversized_shape_is_rejected_before_any_work():
    # 2^20 assignments over 1024 experts need 1024 x 1024 histogram entries (4 MiB)
    shape = moe.make_shape(131072, 64, 1024, 8, 64)
    fake = 16   # never dereferenced: the size check comes first
    rc = moe.moe_route_from_keys_noalloc(shape, fake, fake, fake, fake, fake, fake, fake, fake,
                                         stream=0, check=False)
    assert rc == moe.MOE_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_routing_equals_workspace_routing_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # a large call first, then a smaller one: the second must not see the first's leftovers
    cases = [(20000, 256, 8, 1, False), (333, 1024, 32, 2, True), (4096, 8, 2, 3, True)]
    for T, E, k, seed, ties in cases:
        key, score = _keys(T, E, seed, ties)
        want = _route(moe.moe_route_from_keys, T, E, k, key, score, True)
        got = _route(moe.moe_route_from_keys_noalloc, T, E, k, key, score, False)
        for name in ("idx", "counts", "off", "st", "sp"):
            np.testing.assert_array_equal(got[name], want[name], err_msg=name)
        np.testing.assert_allclose(got["w"], want["w"], rtol=2e-6, atol=1e-7)
        assert got["off"][-1] == T * k
