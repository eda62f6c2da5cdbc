"""The scan kernel's decode arithmetic, modelled step by step in numpy and
checked against the oracle's prefix dequantisation (CPU).

The kernel's thread (block b, r in 0..7) takes tokens r + 8m + 32h of the block
(m = 0..3, h = 0 for the low and 1 for the high 32-bit half of each plane
word).  For a channel of depth t it starts from y = 0x01010101 and, for every
plane p < t, rotates the plane's half-word right by (r - (t - p)) mod 32 (token
r + 8m's bit lands on bit t - p of byte m), masks bit t - p of every byte and
ORs it into y; so byte m of y is 1 + sum_p b_p 2^(t - p) = 2 c_t + 1 for token
r + 8m + 32h (at most 31: no carries between bytes).  A byte permute puts byte
m under the exponent of 2^23, and one fp32 subtraction of 2^23 + 2^t leaves
2 (c_t + 1/2 - 2^(t-1)) exactly; the block weight q * a * 2^-t then gives q
times the t-plane value.  This test runs those integer and fp32 steps on real
plane words and compares every token with the oracle's codes and dequantised
values."""
import numpy as np
import pytest

from oracle import oracle as O

MASK = np.uint32(0x01010101)


def rotr32(x, s):
    s = int(s) % 32
    x = int(x)
    return np.uint32(((x >> s) | (x << (32 - s))) & 0xFFFFFFFF) if s else np.uint32(x)


def model_bytes(words_half, r, t):
    """y for one channel: words_half [t] uint32 half-words of planes 0..t-1."""
    y = MASK
    for p in range(t):
        k = t - p
        y = np.uint32(y | (rotr32(words_half[p], (r - k) % 32) & np.uint32(int(MASK) << k)))
    return y


def byte_under_exponent(y, m):
    """The byte permute: byte m of y as the low byte of 0x4B0000xx (2^23 + byte)."""
    bits = np.uint32(0x4B000000) | ((y >> np.uint32(8 * m)) & np.uint32(0xFF))
    return bits.view(np.float32)


@pytest.mark.parametrize("t", [1, 2, 3, 4])
def test_decode_steps_give_the_prefix_value(t):
    rng = np.random.default_rng(40 + t)
    n, D = 512, 8
    keys = (rng.standard_normal((n, D)) * np.exp(rng.standard_normal(D))).astype(np.float32)
    planes, scales, codes = O.quantize_pack(keys)            # [D][4][nb], [D][nb], [n][D]
    K = np.float32(8388608.0 + 2.0 ** t)
    for j in range(D):
        for beta in range(n // 64):
            w = planes[j, :, beta]
            a16 = O.fp16_value(int(scales[j, beta]))
            for half in (0, 1):
                wh = ((w >> np.uint64(32 * half)) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
                for r in range(8):
                    y = model_bytes(wh, r, t)
                    for m in range(4):
                        i = 64 * beta + r + 8 * m + 32 * half
                        c_t = int(codes[i, j]) >> (4 - t)
                        assert int((y >> np.uint32(8 * m)) & np.uint32(0xFF)) == 2 * c_t + 1
                        two_v = np.float32(byte_under_exponent(y, m) - K)      # one fp32 subtraction
                        assert float(two_v) == 2.0 * (c_t + 0.5 - 2.0 ** (t - 1))
                        # times the block weight a * 2^-t: the oracle's t-plane value, exactly
                        val = np.float32(two_v * np.float32(a16 * 2.0 ** -t))
                        assert float(val) == O.dequant(c_t, t, a16)


def test_bytes_never_carry():
    # the largest byte after t = 4 planes is 1 + 2 + 4 + 8 + 16 = 2 * 15 + 1 = 31
    w = np.full(4, 0xFFFFFFFF, np.uint32)
    y = model_bytes(w, 0, 4)
    assert int(y) == 0x1F1F1F1F
