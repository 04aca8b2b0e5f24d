"""NVFP4 inputs for the tests: E2M1 codes two per byte (even dimension in the
low nibble) and one E4M3 scale per 16 dimensions of a row, built on the host
(numpy) or by torch ops, with the decoded values. Input preparation only: the
values are decoded by the oracle's own E2M1 / E4M3 decoders, and nothing here
runs library code."""
import numpy as np
import torch

import oracle


def bits_f64(b):
    return (np.ascontiguousarray(b).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def nvfp4_pages(x_bits, rng, shape):
    """NVFP4 pages of the given shape [P, H, Bk, d]: E2M1 codes two per byte
    (even dimension low) and one E4M3 scale per 16 dimensions of a row, with the
    decoded values as bf16 bits (exact). With x_bits (bf16 bits of that shape)
    the values are quantised (scale = the E4M3 of amax / 6, at least the
    smallest E4M3 subnormal; codes the nearest E2M1 value); without, codes are
    drawn uniformly and scales from a few powers of two and 1.5 times one."""
    e2m1 = np.array([oracle.e2m1_to_f64(c) for c in range(16)])
    e4m3 = np.array([oracle.e4m3_to_f64(int(c)) for c in range(256)])
    d = shape[-1]
    if x_bits is not None:
        xb = bits_f64(x_bits).reshape(*shape[:-1], d // 16, 16)
        amax = np.abs(xb).max(axis=-1)
        sc_codes = torch.from_numpy((np.maximum(amax, 0.012) / 6.0).astype(np.float32)) \
            .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        y = xb / e4m3[sc_codes][..., None]
        idx = np.abs(np.abs(y)[..., None] - e2m1[:8]).argmin(axis=-1)
        codes = (idx | np.where(y < 0, 8, 0)).astype(np.uint8).reshape(shape)
    else:
        codes = rng.integers(0, 16, size=shape).astype(np.uint8)
        sc_codes = rng.choice(np.array([0x28, 0x30, 0x38, 0x3C, 0x40], dtype=np.uint8),
                              size=(*shape[:-1], d // 16))
    vals = e2m1[codes] * np.repeat(e4m3[sc_codes], 16, axis=-1)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    bits = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bits_f64(bits), vals)                          # exact in bf16
    return packed, sc_codes.astype(np.uint8), bits


def nvfp4_torch(x):
    """NVFP4 quantisation by torch ops, on any device (no library code): per 16
    values one E4M3 scale (amax / 6, at least 2^-9) and the nearest E2M1 code
    of each value over it; returns (codes two per byte, even dimension low;
    scale codes; the decoded values as bf16, exact)."""
    e2m1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device=x.device)
    xb = x.float().reshape(*x.shape[:-1], x.shape[-1] // 16, 16)
    sc = (xb.abs().amax(dim=-1).clamp(min=2.0 ** -9) / 6.0).to(torch.float8_e4m3fn)
    scf = sc.float().unsqueeze(-1)
    y = xb / scf
    mag = (y.abs().unsqueeze(-1) - e2m1).abs().argmin(dim=-1)
    codes = (mag | ((y < 0).to(torch.int64) << 3)).to(torch.uint8).reshape(x.shape)
    dec = (e2m1[mag] * torch.where(y < 0, -1.0, 1.0) * scf).reshape(x.shape)
    dec16 = dec.to(torch.bfloat16)
    assert torch.equal(dec16.float(), dec)  # exact in bf16
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).contiguous()
    return packed, sc.view(torch.uint8).contiguous(), dec16
