"""The arithmetic premise of the one-query-head KIVI value path, checked on the host.

A b-bit code word holds 32/b codes; channel j of the word's value group sits at bits
[b j, b j + b) of the low half and channel 16/b + j at the same place in the high half (the
4-codes-per-byte packing, channel 4k + i in bits [2i, 2i + 2) of byte k). The kernel masks a
code pair in place and reads each half as an fp16 bit pattern: an integer pattern n < 2^11 is
exactly the fp16 n * 2^-24 (subnormal below 2^10, the first binade above), so the code comes
back as code * 2^(b jj - 24). Codes that would reach bit 11 of a half are taken from the word
shifted right by b * split instead (split = 5 for 2-bit codes, 2 for 4-bit)."""
import numpy as np
import pytest

SPLIT = {2: 5, 4: 2}


def _fp16_of_pattern(x):
    return x.astype(np.uint16).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("bits", [2, 4])
def test_masked_code_pairs_read_back_exactly(bits):
    rng = np.random.default_rng(11)
    words = rng.integers(0, 2**32, size=1 << 14, dtype=np.uint64).astype(np.uint32)
    words[:4] = [0, 0xFFFFFFFF, 0xAAAAAAAA, 0x55555555]
    split, per_half, top = SPLIT[bits], 16 // bits, (1 << bits) - 1
    for j in range(per_half):
        jj = j if j < split else j - split
        src = words if j < split else words >> np.uint32(bits * split)
        m = src & np.uint32((top << (bits * jj)) * 0x10001)
        scale = 2.0 ** (24 - bits * jj)
        code_lo = (words >> np.uint32(bits * j)) & np.uint32(top)
        code_hi = (words >> np.uint32(16 + bits * j)) & np.uint32(top)
        assert np.array_equal(_fp16_of_pattern(m & np.uint32(0xFFFF)) * scale, code_lo)
        assert np.array_equal(_fp16_of_pattern(m >> np.uint32(16)) * scale, code_hi)


@pytest.mark.parametrize("bits", [2, 4])
def test_patterns_stay_linear_only_below_bit_11(bits):
    # every pattern below 2^11 is n * 2^-24 ...
    n = np.arange(1 << 11, dtype=np.uint32)
    assert np.array_equal(_fp16_of_pattern(n), n * 2.0 ** -24)
    # ... and the first code past the split, masked in place, would not be: the split is needed
    j = SPLIT[bits]
    top = (1 << bits) - 1
    pattern = np.array([top << (bits * j)], dtype=np.uint32)
    assert _fp16_of_pattern(pattern)[0] != top * 2.0 ** (bits * j - 24)
