"""The NVFP4 byte format that the GPU tests and the benchmark feed the NVFP4
entry points (CPU, no GPU).

NVFP4 ([MSA-PT] "Kernel open source e MiniMax-M3" lists NVFP4 and FP4 among the
kernel's precisions; the format is the OCP / NVIDIA block format): E2M1 codes
two per byte with the even dimension in the low nibble, one E4M3 scale per 16
consecutive dimensions of a row, value = e2m1(code) * e4m3(scale). The three
quantisers the GPU-side tests and the benchmark use are pinned here against
bytes worked out by hand, so that a nibble order or scale layout shared by them
and by the kernels cannot drift away from the format unnoticed.
"""
import numpy as np
import torch

import bench
import oracle
from tests.nvfp4_inputs import nvfp4_pages, nvfp4_torch

# One row of 48 dimensions = three micro-blocks. Block 0 spans every E2M1
# magnitude with both signs (amax 6: scale 1.0), block 1 is block 0 times 2
# (scale 2.0), block 2 is block 0 / 4 (scale 0.25).
_BLOCK0 = [6.0, -6.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0,
           -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, 0.0, 0.0]
ROW = np.array(_BLOCK0 + [2.0 * v for v in _BLOCK0] + [0.25 * v for v in _BLOCK0])

# Codes of block 0: sign bit 3, magnitude index into {0, .5, 1, 1.5, 2, 3, 4, 6}:
#   6 -> 7, -6 -> F, .5 -> 1, 1 -> 2, 1.5 -> 3, 2 -> 4, 3 -> 5, 4 -> 6,
#   -.5 -> 9, -1 -> A, -1.5 -> B, -2 -> C, -3 -> D, -4 -> E, 0 -> 0, 0 -> 0.
# Bytes: low nibble = even dimension, high nibble = the odd one after it.
_BYTES0 = [0xF7, 0x21, 0x43, 0x65, 0xA9, 0xCB, 0xED, 0x00]
WANT_PACKED = np.array(_BYTES0 * 3, dtype=np.uint8)
# E4M3 (bias 7, three mantissa bits): 1.0 = 0 0111 000, 2.0 = 0 1000 000,
# 0.25 = 0 0101 000.
WANT_SCALES = np.array([0x38, 0x40, 0x28], dtype=np.uint8)


def _bf16_bits(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_hand_worked_bytes_decode_to_the_row():
    """The hand-worked bytes decode back to the row through the oracle's
    E2M1 and E4M3 decoders (themselves pinned to the OCP tables)."""
    lo, hi = WANT_PACKED & 0xF, WANT_PACKED >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(-1)        # even dimension first
    scales = np.repeat([oracle.e4m3_to_f64(int(s)) for s in WANT_SCALES], 16)
    vals = np.array([oracle.e2m1_to_f64(int(c)) for c in codes]) * scales
    assert np.array_equal(vals, ROW)


def test_numpy_packer_matches_hand_worked_bytes():
    packed, scales, bits = nvfp4_pages(_bf16_bits(ROW), None, (1, ROW.size))
    assert np.array_equal(packed.reshape(-1), WANT_PACKED)
    assert np.array_equal(scales.reshape(-1), WANT_SCALES)
    assert np.array_equal(bits.reshape(-1), _bf16_bits(ROW))


def test_torch_packer_matches_hand_worked_bytes():
    x = torch.tensor(ROW, dtype=torch.float32).to(torch.bfloat16).reshape(1, -1)
    packed, scales, dec = nvfp4_torch(x)
    assert np.array_equal(packed.numpy().reshape(-1), WANT_PACKED)
    assert np.array_equal(scales.numpy().reshape(-1), WANT_SCALES)
    assert torch.equal(dec.float().reshape(-1), torch.tensor(ROW, dtype=torch.float32))


def test_bench_quantiser_matches_hand_worked_bytes():
    x = torch.tensor(ROW, dtype=torch.float32).to(torch.bfloat16).reshape(1, -1)
    packed, scales = bench.nvfp4_quantise(x)
    assert np.array_equal(packed.numpy().reshape(-1), WANT_PACKED)
    assert np.array_equal(scales.numpy().reshape(-1), WANT_SCALES)


def test_packers_agree_on_random_rows():
    """Away from the rounding midpoints (where the packers may break ties
    differently) the three quantisers give the same bytes on a random row set."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    bits = _bf16_bits(x)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    p_np, s_np, _ = nvfp4_pages(bits, None, x.shape)
    p_t, s_t, _ = nvfp4_torch(xb)
    p_b, s_b = bench.nvfp4_quantise(xb)
    assert np.array_equal(s_np, s_t.numpy()) and np.array_equal(s_np, s_b.numpy())
    # Where no value of a byte's two dimensions sits at an E2M1 midpoint, all
    # three choose the same codes.
    sc = np.repeat(np.array([oracle.e4m3_to_f64(int(c)) for c in range(256)])[s_np], 16, -1)
    y = np.abs((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)) / sc
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    at_mid = np.isin(y, mids).reshape(x.shape[0], -1, 2).any(-1)
    assert np.array_equal(p_np[~at_mid], p_t.numpy()[~at_mid])
    assert np.array_equal(p_np[~at_mid], p_b.numpy()[~at_mid])
