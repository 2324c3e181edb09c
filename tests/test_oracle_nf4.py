"""Pins for the oracle's NF4 quantiser (CPU only).

The codebook is checked against the properties the QLoRA construction fixes
(16 sorted levels, exact zero, +-1 ends, 7 negative / 8 positive levels, the
positive and negative levels being normal quantiles on evenly spaced
probability grids, computed here through scipy rather than torch), and the
quantiser against round trips, the nearest-level rule, the tie rule and the
nibble order.
"""

import pytest
import torch

from oracle import nf4

F64 = torch.float64


def test_codebook_shape_and_ends():
    lv = nf4.codebook()
    assert lv.shape == (16,)
    assert torch.all(lv[1:] > lv[:-1])
    assert float(lv[0]) == -1.0 and float(lv[15]) == 1.0
    assert int((lv == 0).sum()) == 1 and float(lv[7]) == 0.0
    assert int((lv < 0).sum()) == 7 and int((lv > 0).sum()) == 8


def test_codebook_is_normal_quantiles():
    stats = pytest.importorskip("scipy.stats")
    lv = nf4.codebook().numpy()
    top = stats.norm.ppf(nf4.OFFSET)
    # Positive levels: quantiles at 8 evenly spaced probabilities from just
    # above 1/2 to OFFSET; negative levels: 7 such probabilities, mirrored.
    p_pos = stats.norm.cdf(lv[8:] * top)
    p_neg = stats.norm.cdf(-lv[:7][::-1] * top)
    step_pos = (nf4.OFFSET - 0.5) / 8
    step_neg = (nf4.OFFSET - 0.5) / 7
    for i, p in enumerate(p_pos):
        assert abs(p - (0.5 + (i + 1) * step_pos)) < 1e-12
    for i, p in enumerate(p_neg):
        assert abs(p - (0.5 + (i + 1) * step_neg)) < 1e-12


def test_round_trip_exact_levels():
    lv = nf4.codebook()
    a = 0.375  # exactly representable in fp16
    row = torch.cat([lv, lv.flip(0), lv, lv.flip(0)]) * a          # 64 values, |max| = a
    w = torch.stack([row, row.roll(5)]).to(torch.float32)
    packed, absmax = nf4.quantize(w)
    assert torch.all(absmax.float() == a)
    codes = nf4.unpack(packed)
    expect = torch.cat([torch.arange(16), torch.arange(15, -1, -1)] * 2)
    assert torch.equal(codes[0].long(), expect)
    # w holds the levels rounded to fp32; dequantised values are the exact ones.
    assert torch.allclose(nf4.dequantize(packed, absmax), w.to(F64), rtol=0, atol=1e-7)


def test_nearest_level_and_ties():
    g = torch.Generator().manual_seed(0)
    w = torch.randn(8, 256, generator=g) * 0.02
    packed, absmax = nf4.quantize(w)
    codes = nf4.unpack(packed).long()
    lv = nf4.codebook()
    x = (w.to(F64) / absmax.to(F64).repeat_interleave(64, 1))
    d_best = (x - lv[codes]).abs()
    d_all = (x[..., None] - lv).abs().min(-1).values
    assert torch.all(d_best <= d_all + 1e-6)
    # A value exactly on an fp32 midpoint takes the lower code.
    mids = nf4.midpoints_f32()
    blk = torch.zeros(1, 64, dtype=torch.float32)
    blk[0, 0] = 1.0                      # absmax 1: x == w
    blk[0, 1] = mids[3]
    blk[0, 2] = torch.nextafter(mids[3], torch.tensor(2.0))
    c = nf4.unpack(nf4.quantize(blk)[0])[0]
    assert int(c[0]) == 15 and int(c[1]) == 3 and int(c[2]) == 4


def test_nibble_order_and_zero_block():
    lv = nf4.codebook().to(torch.float32)
    w = torch.zeros(1, 128, dtype=torch.float32)
    w[0, 0], w[0, 1] = lv[2], lv[15]         # block 0 absmax 1
    packed, absmax = nf4.quantize(w)
    assert int(packed[0, 0]) == (2 | (15 << 4))
    assert float(absmax[0, 1]) == 0.0
    assert torch.all(nf4.unpack(packed)[0, 64:] == 7)     # zero block -> zero level
