"""Seeded input generators: bf16 rounding, determinism, workload shapes and positions."""

import numpy as np
import torch

from diffusion_transformer_attention_dit_gb300 import inputs


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 100000), rng.normal(0, 1e-30, 1000), rng.normal(0, 1e30, 1000)]).astype(np.float32)
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(ours, ref)
    back = inputs.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_block_draws_independent_of_threads():
    a = inputs.bf16_normal(3 * (1 << 22) + 17, seed=5, threads=1)
    b = inputs.bf16_normal(3 * (1 << 22) + 17, seed=5, threads=4)
    assert np.array_equal(a, b)
    x = inputs.bf16_bits_to_f64(a)
    assert abs(x.mean()) < 1e-3 and abs(x.std() - 1) < 1e-3


def test_workload_shapes_and_positions():
    sizes = {"tiny": 256, "qwen_image": 4312, "qwen_image_edit": 8624, "wan480": 32760, "wan720": 75600}
    for name, S in sizes.items():
        w = inputs.WORKLOADS[name]
        assert w.S == S and sum(w.axis_dims) == w.D
        pos = inputs.positions(w)
        assert pos.shape[0] == S
        c, s = inputs.rope_tables(pos, w.axis_dims)
        assert c.shape == (S, w.D // 2) and c.dtype == np.float32
        np.testing.assert_allclose(c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2, 1.0, atol=1e-6)
    pos = inputs.positions(inputs.WORKLOADS["qwen_image_edit"])
    assert (pos[:512, 0] == np.arange(512)).all()
    assert (pos[512:512 + 4056, 0] == 0).all() and (pos[512 + 4056:, 0] == 1).all()
    assert pos[512 + 4055].tolist() == [0, 77, 51]


def test_chunk_bounds_cover_keys():
    w = inputs.WORKLOADS["wan720"]
    b = w.chunk_bounds()
    assert len(b) == 8 and b[0][0] == 0 and b[-1][1] == w.S
    assert all(hi - lo == 9450 for lo, hi in b)
    assert all(b[i][1] == b[i + 1][0] for i in range(7))
