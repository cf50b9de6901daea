"""Seeded synthetic inputs for the attention forward workloads.

This module only draws and rounds random numbers; it holds none of the
attention arithmetic.  The tests, the smoke check and the bench take their
inputs from here, so the CUDA path and the fp64 oracle read identical values.

Recipe: Q, K, V are iid N(0, 1) drawn in fp32 by ``torch.Generator`` (CPU,
``manual_seed(seed)``; one seed per tensor), then rounded to the workload's
16-bit dtype.  The stress variant multiplies the rounded Q by 8 (a power of
two, so the product is exact in fp16/bf16), which spreads the scaled scores to
a standard deviation of about 8 so that the running max keeps moving.

The backward pass's upstream gradient dO follows the same recipe with a
seed of its own (``make_dout``); so do the decoding inputs (``make_decode``:
Nq query rows against an Nk-row KV sequence).

Shapes follow the pages' [B, H, N, d] notation (contiguous, row stride d):
"Triton으로 FlashAttention 1·2 forward 구현하기", section "기준 shape", uses
[4, 32, 2048, 64] in fp16, and section "batch 크기에 따른 변화" varies B.
"""
import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}

# name -> (B, H, N, d, dtype, (seed_q, seed_k, seed_v))
WORKLOADS = {
    "tiny": (1, 2, 256, 64, "fp16", (0, 1, 2)),
    "base": (4, 32, 2048, 64, "fp16", (10, 11, 12)),
    "sweep_b1": (1, 32, 2048, 64, "fp16", (21, 22, 23)),
    "sweep_b2": (2, 32, 2048, 64, "fp16", (24, 25, 26)),
    "sweep_b4": (4, 32, 2048, 64, "fp16", (27, 28, 29)),
    "sweep_b8": (8, 32, 2048, 64, "fp16", (50, 51, 52)),
    "d128": (2, 16, 8192, 128, "bf16", (30, 31, 32)),
    "long": (1, 8, 65536, 128, "fp16", (40, 41, 42)),
    # head dims outside the pages' 64 / 128 (the base shape otherwise)
    "hd32": (4, 32, 2048, 32, "fp16", (70, 71, 72)),
    "hd96": (4, 32, 2048, 96, "fp16", (73, 74, 75)),
    # the base shape with a ragged length (2000 = 15 x 128 + 80)
    "ragged": (4, 32, 2000, 64, "fp16", (76, 77, 78)),
}
# seed of the upstream gradient dO per workload (backward pass)
DOUT_SEEDS = {"tiny": 3, "base": 13, "sweep_b1": 33, "sweep_b2": 34, "sweep_b4": 35,
              "sweep_b8": 53, "d128": 36, "long": 44, "hd32": 79, "hd96": 80, "ragged": 81}
# seed of the query rows the oracle checks on the long-context workload
LONG_ROW_SAMPLE_SEED = 43
LONG_ROWS_PER_HEAD = 512


def torch_dtype(name):
    try:
        return DTYPES[name]
    except KeyError:
        raise ValueError("dtype must be one of %s, got %r" % (sorted(DTYPES), name))


def make_qkv(B, H, N, d, dtype="fp16", seeds=(0, 1, 2), q_scale=1.0):
    """Return CPU tensors (q, k, v) of shape [B, H, N, d] in the 16-bit dtype."""
    dt = torch_dtype(dtype) if isinstance(dtype, str) else dtype
    out = []
    for t, seed in enumerate(seeds):
        g = torch.Generator(device="cpu").manual_seed(int(seed))
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(dt)
        if t == 0 and q_scale != 1.0:
            x = x * q_scale
        out.append(x.contiguous())
    return tuple(out)


def make_dout(B, H, N, d, dtype="fp16", seed=3):
    """Upstream gradient dL/dO for the backward pass: iid N(0, 1) in fp32,
    rounded to the 16-bit dtype, [B, H, N, d] on the CPU."""
    dt = torch_dtype(dtype) if isinstance(dtype, str) else dtype
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(dt).contiguous()


# decoding workloads: name -> (B, H, Nq, Nk, d, dtype, (seed_q, seed_k, seed_v), causal)
DECODE_WORKLOADS = {
    "decode": (8, 32, 1, 16384, 128, "fp16", (60, 61, 62), False),
    "decode_spec": (8, 32, 4, 16384, 128, "bf16", (63, 64, 65), True),
    # decode_spec at a quarter of the heads (K/V 0.54 GB, still above L2): for
    # multi-pass profiler captures, which save and restore device memory
    "decode_spec_b2": (2, 32, 4, 16384, 128, "bf16", (69, 70, 71), True),
    # small case for the CPU tests of bench.py's decoding legs
    "decode_small": (1, 4, 2, 1024, 64, "fp16", (66, 67, 68), True),
}


def make_decode(B, H, Nq, Nk, d, dtype="fp16", seeds=(0, 1, 2)):
    """q [B, H, Nq, d] and k, v [B, H, Nk, d] (CPU, 16-bit), same recipe as make_qkv."""
    dt = torch_dtype(dtype) if isinstance(dtype, str) else dtype
    shapes = ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d))
    out = []
    for shape, seed in zip(shapes, seeds):
        g = torch.Generator(device="cpu").manual_seed(int(seed))
        out.append(torch.randn(shape, generator=g, dtype=torch.float32).to(dt).contiguous())
    return tuple(out)


def make_decode_workload(name):
    """(q, k, v, meta) of a named decoding workload."""
    B, H, Nq, Nk, d, dtype, seeds, causal = DECODE_WORKLOADS[name]
    q, k, v = make_decode(B, H, Nq, Nk, d, dtype, seeds)
    return q, k, v, dict(B=B, H=H, Nq=Nq, Nk=Nk, d=d, dtype=dtype, causal=causal)


def make_workload(name, q_scale=1.0):
    """(q, k, v, meta) for a named workload; meta holds B, H, N, d, dtype."""
    B, H, N, d, dtype, seeds = WORKLOADS[name]
    q, k, v = make_qkv(B, H, N, d, dtype, seeds, q_scale=q_scale)
    return q, k, v, dict(B=B, H=H, N=N, d=d, dtype=dtype)


def sample_rows(B, H, N, per_head, seed):
    """Seeded (bh, i) query-row sample: ``per_head`` distinct rows per head."""
    rng = np.random.default_rng(int(seed))
    rows = []
    per = min(per_head, N)
    for bh in range(B * H):
        idx = np.sort(rng.choice(N, size=per, replace=False))
        rows.extend((bh, int(i)) for i in idx)
    return np.array(rows, dtype=np.int64).reshape(-1, 2)
