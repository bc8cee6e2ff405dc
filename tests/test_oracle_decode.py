"""Pins the oracle's exact widening of f16 / bf16 elements to binary64 (all 65536 patterns)."""
import numpy as np
import torch

import oracle


def _same(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_f16_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    assert _same(got, ref)


def test_bf16_all_bit_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode(bits, oracle.BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(got, ref)
