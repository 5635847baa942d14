"""The seeded input generator: published SplitMix64 outputs, determinism,
shapes and moments of the drawn values."""
import numpy as np
import torch

import iha_inputs as gi


def test_splitmix64_published_sequence():
    """SplitMix64 seeded with 0 (state advanced by the golden gamma before each
    mix) starts 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, 0x06c45d188009454f
    (Steele, Lea and Flood 2014; the reference generator's first outputs)."""
    gamma = 0x9E3779B97F4A7C15
    states = np.array([0, gamma, (2 * gamma) % 2**64], dtype=np.uint64)
    out = [int(v) for v in gi._splitmix64(states)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_normal_moments_and_determinism():
    a = gi.normal(3, 1, 1 << 18, std=2.0)
    b = gi.normal(3, 1, 1 << 18, std=2.0)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.02 and abs(a.std() - 2.0) < 0.02
    c = gi.normal(4, 1, 1 << 10)
    assert not np.array_equal(a[:1024] / 2.0, c)
    # chunking does not change the stream
    assert np.array_equal(gi.normal(3, 1, 5000, chunk=777), gi.normal(3, 1, 5000))


def test_workload_shapes_and_dtypes():
    w = gi.WORKLOADS["tiny_f32_nomask"]
    inp = gi.make_inputs(w)
    assert inp["X"].shape == (1, 64, 128) and inp["X"].dtype == torch.float32
    assert inp["W_Q"].shape == (128, 128)
    assert inp["alpha_K"].shape == (4, 4, 2) and inp["alpha_K"].dtype == torch.float32
    assert inp["R"].shape == (4, 8)
    w1 = gi.WORKLOADS["bf16_causal_n1024"].with_(N=16, B=1)
    inp1 = gi.make_inputs(w1)
    assert inp1["X"].dtype == torch.bfloat16 and inp1["W_V"].dtype == torch.bfloat16
    # bf16 values are the fp32 draws rounded to nearest even
    ref = torch.from_numpy(gi.normal(w1.seed, gi.TAGS["X"], 16 * w1.D).reshape(1, 16, w1.D))
    assert torch.equal(inp1["X"], ref.to(torch.bfloat16))


def test_every_workload_satisfies_d_equals_h_times_head_dim():
    for w in gi.WORKLOADS.values():
        assert w.D == w.H * w.d
        if w.mask_mode == gi.MASK_WINDOW:
            assert w.window == w.N // (2 * w.P)
