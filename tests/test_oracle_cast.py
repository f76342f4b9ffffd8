"""Oracle pins: 16-bit decode and round-to-nearest-even encode against library
conversions (numpy's float32->float16 and torch's float32->bfloat16 are both
IEEE round-to-nearest-even), on every exponent/fraction pattern near a
rounding boundary plus random bit patterns."""
import numpy as np
import torch

from oracle.step import FMT_BF16, FMT_FP16, cast16, decode16


def _structured_f32():
    hi = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(7)
    bits = np.concatenate([bits, rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)])
    # fp16 rounding boundaries: midpoints between neighbouring fp16 values
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    f = h.view(np.float16).astype(np.float64)
    mids = ((f[:-1] + f[1:]) / 2).astype(np.float32)   # exact midpoints where representable
    ext = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    ext = np.concatenate([ext, -ext, np.array([65504, 65519.996, 65520, 65536, np.inf, -np.inf,
                                               2 ** -24, 2 ** -25, 3 * 2 ** -26, 2 ** -14], np.float32)])
    return np.concatenate([bits.view(np.float32), ext.astype(np.float32)])


def _same_bits_or_both_nan(a16: np.ndarray, b16: np.ndarray, fmt: int):
    if fmt == FMT_BF16:
        nan_a = ((a16 & 0x7F80) == 0x7F80) & ((a16 & 0x7F) != 0)
        nan_b = ((b16 & 0x7F80) == 0x7F80) & ((b16 & 0x7F) != 0)
    else:
        nan_a = ((a16 & 0x7C00) == 0x7C00) & ((a16 & 0x3FF) != 0)
        nan_b = ((b16 & 0x7C00) == 0x7C00) & ((b16 & 0x3FF) != 0)
    assert np.array_equal(nan_a, nan_b)
    ok = nan_a | (a16 == b16)
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, (bad[:5], a16[bad[:5]], b16[bad[:5]])


def test_f32_to_f16_matches_numpy_rne():
    x = _structured_f32()
    ours = cast16(x, FMT_FP16)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    _same_bits_or_both_nan(ours, ref, FMT_FP16)


def test_f32_to_bf16_matches_torch_rne():
    x = _structured_f32()
    ours = cast16(x, FMT_BF16)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    _same_bits_or_both_nan(ours, ref, FMT_BF16)


def test_decode_is_exact_for_every_16bit_pattern():
    h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f16 = decode16(h, FMT_FP16)
    ref16 = h.view(np.float16).astype(np.float32)
    both_nan = np.isnan(f16) & np.isnan(ref16)
    assert np.array_equal(f16.view(np.uint32)[~both_nan], ref16.view(np.uint32)[~both_nan])
    bf = decode16(h, FMT_BF16)
    refbf = (h.astype(np.uint32) << 16).view(np.float32)
    both_nan = np.isnan(bf) & np.isnan(refbf)
    assert np.array_equal(bf.view(np.uint32)[~both_nan], refbf.view(np.uint32)[~both_nan])


def test_cast_roundtrip_identity_on_representable_values():
    for fmt in (FMT_BF16, FMT_FP16):
        h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
        f = decode16(h, fmt)
        back = cast16(f, fmt)
        finite = np.isfinite(f)
        assert np.array_equal(back[finite], h[finite])
