"""Pins for the oracle's building blocks and forward pass (CPU only).

Each check ties the oracle to something other than itself: a closed form, an
invariant, or an independent library route to the same mathematics
(torch.nn.functional.rms_norm, scaled_dot_product_attention, complex
multiplication for the rotation, F.silu, F.linear).
"""

import math

import pytest
import torch
import torch.nn.functional as F

from oracle import model as om
from synth import TINY_TARGET, make_weights

F64 = torch.float64


def test_rmsnorm_constant_vector_gives_gain():
    g = torch.linspace(0.5, 2.0, 16, dtype=F64)
    for c in (1e-3, 0.7, -3.0, 250.0):
        y = om.rmsnorm(torch.full((16,), c, dtype=F64), g, 0.0)
        assert torch.allclose(y, g * math.copysign(1.0, c), rtol=0, atol=1e-14)


def test_rmsnorm_hand_value_and_library():
    # x = [3, 4]: mean of squares 12.5.
    x = torch.tensor([3.0, 4.0], dtype=F64)
    g = torch.tensor([1.0, 2.0], dtype=F64)
    eps = 0.5
    y = om.rmsnorm(x, g, eps)
    assert torch.allclose(y, torch.tensor([3.0, 8.0], dtype=F64) / math.sqrt(13.0), atol=1e-15)
    torch.manual_seed(0)
    x = torch.randn(37, dtype=F64)
    g = torch.randn(37, dtype=F64)
    ref = F.rms_norm(x, (37,), weight=g, eps=1e-6)
    assert torch.allclose(om.rmsnorm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_rope_position_zero_is_identity_and_norm_preserved():
    torch.manual_seed(1)
    x = torch.randn(3, 64, dtype=F64)
    assert torch.equal(om.rope(x, 0, 1e6), x)
    for p in (1, 17, 4095):
        y = om.rope(x, p, 1e6)
        assert torch.allclose(y.norm(dim=1), x.norm(dim=1), rtol=1e-13)


def test_rope_head_dim_2_is_rotation_by_position():
    # head_dim 2: a single pair with frequency theta^0 = 1, so the angle is p.
    x = torch.tensor([[1.0, 0.0]], dtype=F64)
    for p in (1, 2, 5):
        y = om.rope(x, p, 10000.0)
        assert torch.allclose(y, torch.tensor([[math.cos(p), math.sin(p)]], dtype=F64), atol=1e-15)


def test_rope_matches_complex_rotation_and_is_relative():
    torch.manual_seed(2)
    hd, theta = 128, 1e6
    half = hd // 2
    q = torch.randn(4, hd, dtype=F64)
    k = torch.randn(4, hd, dtype=F64)
    for p in (3, 1000):
        zc = torch.complex(q[:, :half], q[:, half:])
        freq = theta ** (-(torch.arange(0, hd, 2, dtype=F64)) / hd)
        zc = zc * torch.polar(torch.ones(half, dtype=F64), p * freq)
        ref = torch.cat([zc.real, zc.imag], dim=1)
        assert torch.allclose(om.rope(q, p, theta), ref, rtol=1e-12, atol=1e-12)
    # <rope(q, a), rope(k, b)> depends on a - b only.
    d1 = (om.rope(q, 10, theta) * om.rope(k, 3, theta)).sum(1)
    d2 = (om.rope(q, 507, theta) * om.rope(k, 500, theta)).sum(1)
    assert torch.allclose(d1, d2, rtol=1e-9, atol=1e-10)


def test_silu():
    z = torch.linspace(-20, 20, 101, dtype=F64)
    assert torch.allclose(om.silu(z), F.silu(z), rtol=1e-14, atol=1e-15)
    assert float(om.silu(torch.zeros(1, dtype=F64))) == 0.0


def test_attention_special_cases():
    torch.manual_seed(3)
    nh, nkv, hd = 4, 2, 16
    q = torch.randn(nh, hd, dtype=F64)
    # One slot: the output is that slot's value for every head.
    k = torch.randn(1, nkv, hd, dtype=F64)
    v = torch.randn(1, nkv, hd, dtype=F64)
    out = om.attend(q, k, v, nh // nkv)
    for h in range(nh):
        assert torch.allclose(out[h], v[0, h // 2], atol=1e-15)
    # Equal keys: uniform weights, the output is the mean of the values.
    k = torch.randn(1, nkv, hd, dtype=F64).expand(9, nkv, hd).clone()
    v = torch.randn(9, nkv, hd, dtype=F64)
    out = om.attend(q, k, v, nh // nkv)
    for h in range(nh):
        assert torch.allclose(out[h], v[:, h // 2].mean(0), atol=1e-14)


def test_attention_matches_sdpa_with_gqa():
    torch.manual_seed(4)
    nh, nkv, hd, S = 6, 2, 32, 13
    q = torch.randn(nh, hd, dtype=F64)
    k = torch.randn(S, nkv, hd, dtype=F64)
    v = torch.randn(S, nkv, hd, dtype=F64)
    out = om.attend(q, k, v, nh // nkv)
    kk = k.repeat_interleave(nh // nkv, dim=1).permute(1, 0, 2)  # [nh, S, hd]
    vv = v.repeat_interleave(nh // nkv, dim=1).permute(1, 0, 2)
    ref = F.scaled_dot_product_attention(q[:, None, :], kk, vv)[:, 0, :]
    assert torch.allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_first_argmax_ties_lowest_index():
    l = torch.tensor([0.0, 3.0, -1.0, 3.0, 2.0], dtype=F64)
    assert om.first_argmax(l) == 1
    assert om.first_argmax(torch.tensor([5.0], dtype=F64)) == 0


@pytest.fixture(scope="module")
def tiny():
    w = make_weights(TINY_TARGET, seed=0)
    return TINY_TARGET, w


def test_incremental_equals_one_pass(tiny):
    shape, w = tiny
    m = om.Model(shape, w)
    toks = [5, 900, 17, 17, 3, 1023, 0, 44, 512, 6]
    c1 = m.new_cache()
    one = m.forward(toks, c1)
    c2 = m.new_cache()
    for i, t in enumerate(toks):
        step = m.forward([t], c2)[0]
        assert torch.equal(step, one[i]), f"row {i}"
    for l in range(shape.layers):
        assert torch.equal(c1.keys(l), c2.keys(l))
        assert torch.equal(c1.values(l), c2.values(l))


def _library_forward(shape, w, toks):
    """Same architecture from library routines, all rows of a causal sequence
    at once: F.rms_norm, F.linear, complex rotation, SDPA, F.silu."""
    d = {k: (None if v is None else v.to(F64)) for k, v in w.items()}
    S, hd, half = len(toks), shape.head_dim, shape.head_dim // 2
    x = d["embed"][torch.tensor(toks)]
    pos = torch.arange(S, dtype=F64)
    freq = shape.rope_theta ** (-(torch.arange(0, hd, 2, dtype=F64)) / hd)
    rot = torch.polar(torch.ones(S, half, dtype=F64), pos[:, None] * freq[None, :])

    def rope_all(t):  # t [S, nh, hd]
        z = torch.complex(t[..., :half], t[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    for l in range(shape.layers):
        p = f"layers.{l}."
        h = F.rms_norm(x, (shape.hidden,), weight=d[p + "ln1"], eps=shape.rms_eps)
        q = F.linear(h, d[p + "wq"], d[p + "bq"]).view(S, shape.n_heads, hd)
        k = F.linear(h, d[p + "wk"], d[p + "bk"]).view(S, shape.n_kv_heads, hd)
        v = F.linear(h, d[p + "wv"], d[p + "bv"]).view(S, shape.n_kv_heads, hd)
        q, k = rope_all(q), rope_all(k)
        rep = shape.n_heads // shape.n_kv_heads
        a = F.scaled_dot_product_attention(q.transpose(0, 1), k.repeat_interleave(rep, 1).transpose(0, 1),
                                           v.repeat_interleave(rep, 1).transpose(0, 1), is_causal=True)
        x = x + F.linear(a.transpose(0, 1).reshape(S, -1), d[p + "wo"])
        h2 = F.rms_norm(x, (shape.hidden,), weight=d[p + "ln2"], eps=shape.rms_eps)
        x = x + F.linear(F.silu(F.linear(h2, d[p + "wg"])) * F.linear(h2, d[p + "wu"]), d[p + "wd"])
    xf = F.rms_norm(x, (shape.hidden,), weight=d["norm"], eps=shape.rms_eps)
    return F.linear(xf, d["embed"] if shape.tied else d["lm_head"])


@pytest.mark.parametrize("tied", [True, False])
def test_forward_matches_library_composition(tied):
    shape = TINY_TARGET.with_(tied=tied, vocab=300)
    w = make_weights(shape, seed=7)
    # Non-trivial gains so that a dropped or misplaced gain shows.
    g = torch.Generator().manual_seed(9)
    for k in w:
        if k.endswith("ln1") or k.endswith("ln2") or k == "norm":
            w[k] = (1.0 + 0.5 * torch.randn(w[k].shape, generator=g)).to(torch.bfloat16)
    toks = [3, 250, 7, 7, 99, 0, 1, 299, 42, 5, 6, 13]
    m = om.Model(shape, w)
    out = m.forward(toks, m.new_cache())
    ref = _library_forward(shape, w, toks)
    for i in range(len(toks)):
        assert torch.allclose(out[i], ref[i], rtol=1e-10, atol=1e-12), i


def test_forward_zero_blocks_closed_form():
    # With the attention output and down projections zeroed, every layer
    # leaves the residual untouched: logits = E . rmsnorm(E[t]) * g.
    shape = TINY_TARGET
    w = make_weights(shape, seed=11)
    for l in range(shape.layers):
        w[f"layers.{l}.wo"] = torch.zeros_like(w[f"layers.{l}.wo"])
        w[f"layers.{l}.wd"] = torch.zeros_like(w[f"layers.{l}.wd"])
    m = om.Model(shape, w)
    toks = [1, 2, 1000]
    out = m.forward(toks, m.new_cache())
    E = w["embed"].to(F64)
    for i, t in enumerate(toks):
        e = E[t]
        ref = E @ (e / math.sqrt(float((e * e).mean()) + shape.rms_eps))
        assert torch.allclose(out[i], ref, rtol=1e-12, atol=1e-13)


def test_batched_linear_matches_rowwise(tiny):
    shape, w = tiny
    a = om.Model(shape, w, rowwise=True)
    b = om.Model(shape, w, rowwise=False)
    toks = [9, 8, 7, 6, 5]
    la = a.forward(toks, a.new_cache())
    lb = b.forward(toks, b.new_cache())
    for i in range(len(toks)):
        assert torch.allclose(la[i], lb[i], rtol=1e-11, atol=1e-12)
