"""Pins of the oracle's block-wise int8 quantization of the parameter shard
for the all-gather (ZeRO++ qwZ: "ZeRO Optimization: Stages 1, 2, and 3
Explained" -- 16-bit parameters sent as 8-bit, a scale per small block --
and "DeepSpeed ZeRO Stages" sec. 5.3, which says it halves the gather
volume).  Block size 256, symmetric absmax scale max|x|/127, ties to even: the
reading, pinned by hand-worked blocks, the error bound and the payload size.
CPU only."""
import numpy as np
import pytest


def _bits(x):
    return np.asarray(x, np.float16).view(np.uint16)


def test_hand_worked_block_scale_one(oracle):
    # amax 127 -> scale exactly 1, so q = rint(x): ties go to the even integer
    x = [127.0, -3.5, 2.5, 0.4, -0.6, 100.5, -127.0, 0.0, 1.5, -2.5]
    codes, scales = oracle.qwz_quantize(_bits(x))
    assert scales.tolist() == [1.0]
    assert codes.tolist() == [127, -4, 2, 0, -1, 100, -127, 0, 2, -2]
    back = oracle.qwz_dequantize(codes, scales).view(np.float16)
    assert back.tolist() == [127.0, -4.0, 2.0, 0.0, -1.0, 100.0, -127.0, 0.0, 2.0, -2.0]


def test_hand_worked_block_scale_two(oracle):
    # amax 254 -> scale 2: x / 2 = 127, 1.5, 2.5, -3.5, 0.5 -> 127, 2, 2, -4, 0
    codes, scales = oracle.qwz_quantize(_bits([254.0, 3.0, 5.0, -7.0, 1.0]))
    assert scales.tolist() == [2.0] and codes.tolist() == [127, 2, 2, -4, 0]


def test_zero_block_and_partial_tail(oracle):
    x = np.zeros(256 * 2 + 37, np.float16)
    x[256 + 5] = -3.0                          # only the second block is non-zero
    x[-1] = 0.5                                # the 37-element tail block
    codes, scales = oracle.qwz_quantize(x.view(np.uint16))
    assert scales.size == 3
    assert scales[0] == 0.0 and not codes[:256].any()
    assert scales[1] == np.float32(3.0) / np.float32(127.0) and codes[256 + 5] == -127
    assert scales[2] == np.float32(0.5) / np.float32(127.0) and codes[-1] == 127
    back = oracle.qwz_dequantize(codes, scales).view(np.float16)
    assert back[256 + 5] == -3.0 and back[-1] == 0.5 and not back[:256].any()


@pytest.mark.parametrize("n", [1, 255, 256, 257, 4096 + 100])
def test_error_bound_and_extremes(oracle, n):
    rng = np.random.Generator(np.random.PCG64(n))
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 2, n)).astype(np.float16)
    codes, scales = oracle.qwz_quantize(x.view(np.uint16))
    assert scales.size == (n + 255) // 256
    assert codes.min() >= -127 and codes.max() <= 127
    xf = x.astype(np.float64)
    back = oracle.qwz_dequantize(codes, scales).view(np.float16).astype(np.float64)
    for b in range(scales.size):
        blk = slice(256 * b, min(n, 256 * (b + 1)))
        amax = np.abs(xf[blk]).max()
        assert scales[b] == np.float32(amax) / np.float32(127)
        # the largest magnitude maps to +-127
        j = int(np.argmax(np.abs(xf[blk])))
        assert abs(int(codes[blk][j])) == 127
        # |x - fp16(q s)| <= s/2 (rounding to the grid) + rounding of q s to fp16
        err = np.abs(back[blk] - xf[blk])
        assert np.all(err <= scales[b] * (0.5 + 1e-6) + np.abs(back[blk]) * 2.0 ** -11 + 1e-12)


def test_blocks_are_independent(oracle):
    rng = np.random.Generator(np.random.PCG64(2))
    x = (rng.standard_normal(1024)).astype(np.float16)
    c0, s0 = oracle.qwz_quantize(x.view(np.uint16))
    y = x.copy()
    y[256:512] *= np.float16(8)                 # rescale block 1 only (exact in fp16)
    c1, s1 = oracle.qwz_quantize(y.view(np.uint16))
    assert np.array_equal(np.delete(c0, np.s_[256:512]), np.delete(c1, np.s_[256:512]))
    assert np.array_equal(c0[256:512], c1[256:512]) and s1[1] == 8 * s0[1]


def test_payload_is_about_half(oracle):
    # int8 codes plus one fp32 scale per 256 parameters vs 2 bytes per fp16
    n = 375_000_064
    qwz_bytes = n + 4 * ((n + 255) // 256)
    assert abs(qwz_bytes / (2 * n) - 0.5078) < 1e-3
