"""Host twin of the seeded input generator (CPU only)."""
import numpy as np

import moe_inputs
from moe_inputs import configs, host


def test_counter_based_elements_do_not_depend_on_the_range_requested():
    full = host.normal(np.arange(1000), 3, 7, 0.5, "bf16")
    part = host.normal(np.array([999, 5, 500]), 3, 7, 0.5, "bf16")
    np.testing.assert_array_equal(part, full[[999, 5, 500]])
    assert not np.array_equal(full, host.normal(np.arange(1000), 4, 7, 0.5, "bf16"))
    assert not np.array_equal(full, host.normal(np.arange(1000), 3, 8, 0.5, "bf16"))


def test_log_series_matches_libm():
    s = np.concatenate([np.random.default_rng(0).uniform(1e-300, 1.0, 20000), [0.5, 0.25, 1e-17]])
    np.testing.assert_allclose(host.ln_series(s), np.log(s), rtol=2e-15)


def test_normal_moments():
    z = host.normal_f64(np.arange(400_000), 11, 1)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    assert abs(np.mean(z ** 3)) < 2e-2 and abs(np.mean(z ** 4) - 3) < 5e-2


def test_uniform_range():
    u = host.uniform_f32(np.arange(100_000), 2, 5, -0.01, 0.01)
    assert u.min() >= -0.01 and u.max() <= 0.01 and abs(u.mean()) < 2e-4


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -2.5],
                 dtype=np.float32)
    got = host.bf16_bits_to_f32(host.f32_to_bf16_bits(f))
    np.testing.assert_array_equal(got, [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5])


def test_zipf_offsets_are_a_permuted_power_law():
    off, perm = host.zipf_offsets(128, 4, 1.2, 2.0)
    assert sorted(perm) == list(range(128))
    r = np.arange(1, 129)
    np.testing.assert_allclose(off[perm], (2.0 * -1.2 * np.log(r)).astype(np.float32), rtol=1e-6)


def test_zipf_config_puts_the_offsets_in_the_gate():
    cfg = configs.make_shape(5, 64, 16, 2, 64, zipf=dict(s=1.2, scale=2.0), seed=9)
    x = moe_inputs.host_tensor(cfg, "x")
    wr = moe_inputs.host_tensor(cfg, "w_router")
    off, _ = moe_inputs.zipf(cfg)
    assert np.all(moe_inputs.as_float64(cfg, x[:, 0]) == 1.0)
    np.testing.assert_array_equal(wr[:, 0], host.f32_to_bf16_bits(off))


def test_host_tensor_row_selection_matches_full_tensor():
    cfg = configs.make_shape(7, 64, 4, 2, 64, Fs=64, bias_range=0.01, seed=1)
    full = moe_inputs.host_inputs(cfg)
    np.testing.assert_array_equal(moe_inputs.host_tensor(cfg, "w_gate_up", [3, 1]),
                                  full["w_gate_up"][[3, 1]])
    np.testing.assert_array_equal(moe_inputs.host_tensor(cfg, "x", [6]), full["x"][[6]])
    assert full["bias"].dtype == np.float32 and full["sh_down"].shape == (64, 64)
