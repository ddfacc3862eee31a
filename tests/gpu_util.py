"""Shared helpers for the GPU parity tests (inputs, oracle runs, comparisons)."""
import numpy as np

from kv_cache_gb300 import synthetic
from oracle import e4m3

MAX_ABS = 2e-2          # attention output, absolute (fp32 output vs float64 oracle)
MEAN_REL = 5e-3         # sum |diff| / sum |ref|


def chunk_pair(role, idx, T, H, d, outliers=False):
    """(uint16 bf16 bits, float32 values) of one seeded chunk."""
    bits = synthetic.chunk(role, idx, T, H, d, outliers)
    return bits, synthetic.bf16_to_f32(bits)


def to_dev(bits):
    import torch
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def code_ulp_diff(a, b):
    """Per-element |decode(a) - decode(b)| in e4m3 steps at the larger magnitude."""
    x = e4m3.decode(a)
    y = e4m3.decode(b)
    return np.abs(x - y) / e4m3.ulp_at(np.maximum(np.abs(x), np.abs(y)))


def assert_codes_match(gpu, ref, min_identical=0.999, what="codes"):
    same = gpu == ref
    frac = same.mean() if same.size else 1.0
    diff = code_ulp_diff(gpu, ref)
    assert diff.max(initial=0) <= 1.0, f"{what}: max {diff.max()} e4m3 steps apart"
    assert frac >= min_identical, f"{what}: only {frac:.6f} identical"
    return frac


def assert_attention_close(got, ref, what="attention"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs = np.max(np.abs(got - ref))
    mean_rel = np.sum(np.abs(got - ref)) / max(np.sum(np.abs(ref)), 1e-30)
    assert max_abs <= MAX_ABS and mean_rel <= MEAN_REL, f"{what}: max_abs {max_abs:.3e}, mean_rel {mean_rel:.3e}"
    return max_abs, mean_rel
