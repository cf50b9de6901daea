"""The seeded input generators are deterministic and follow the recipe."""
import numpy as np
import torch

from attention_forward_02_gb300 import inputs


def test_same_seed_same_values():
    a = inputs.make_qkv(1, 2, 64, 64, "fp16", (0, 1, 2))
    b = inputs.make_qkv(1, 2, 64, 64, "fp16", (0, 1, 2))
    for x, y in zip(a, b):
        assert x.dtype == torch.float16 and x.is_contiguous()
        assert torch.equal(x, y)
    c = inputs.make_qkv(1, 2, 64, 64, "fp16", (3, 1, 2))
    assert not torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_stress_scaling_is_exact():
    q1, _, _ = inputs.make_qkv(1, 1, 128, 64, "fp16", (5, 6, 7))
    q8, _, _ = inputs.make_qkv(1, 1, 128, 64, "fp16", (5, 6, 7), q_scale=8.0)
    assert torch.equal(q8.double(), q1.double() * 8)


def test_distribution_roughly_standard_normal():
    _, _, v = inputs.make_qkv(1, 4, 1024, 64, "bf16", (0, 1, 2))
    x = v.double()
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02


def test_row_sample_distinct_and_seeded():
    r1 = inputs.sample_rows(1, 8, 65536, 512, 43)
    r2 = inputs.sample_rows(1, 8, 65536, 512, 43)
    assert r1.shape == (8 * 512, 2) and np.array_equal(r1, r2)
    for bh in range(8):
        rows = r1[r1[:, 0] == bh, 1]
        assert len(set(rows.tolist())) == 512 and rows.min() >= 0 and rows.max() < 65536
