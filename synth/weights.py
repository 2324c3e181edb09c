"""Random-init weights for the workloads.

Matrices and biases are drawn from N(0, std) (std 0.02) in fp32 and rounded
to bf16; RMSNorm gains are 1. Each tensor has its own generator, seeded from
(seed, index in the canonical order), so shapes with a common prefix of
tensors never share values by accident and any single tensor can be
regenerated alone.
"""

import torch

from .shapes import ModelShape, weight_names, weight_shape

_GOLDEN = 0x9E3779B97F4A7C15


def _tensor_seed(seed: int, index: int, salt: int = 0) -> int:
    # A plain integer mix of (seed, index, salt) into a 63-bit generator seed.
    x = (seed * 0x100000001B3 + index * _GOLDEN + salt * 0xD1B54A32D192ED03) & ((1 << 64) - 1)
    x ^= x >> 31
    x = (x * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
    x ^= x >> 29
    return x & ((1 << 63) - 1)


def _normal(shape, seed, device, std):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std)


def make_weights(shape: ModelShape, seed: int, device="cpu", dtype=torch.bfloat16,
                 std: float = 0.02) -> dict:
    """All tensors of ``shape`` in the canonical order, values seeded by ``seed``."""
    out = {}
    for i, name in enumerate(weight_names(shape)):
        t = name.split(".")[-1]
        if t in ("bq", "bk", "bv") and not shape.qkv_bias:
            out[name] = None
            continue
        shp = weight_shape(shape, name)
        if t in ("ln1", "ln2", "norm"):
            out[name] = torch.ones(shp, device=device, dtype=dtype)
        else:
            out[name] = _normal(shp, _tensor_seed(seed, i), device, std).to(dtype)
    return out


def _is_gain(name: str) -> bool:
    return name.split(".")[-1] in ("ln1", "ln2", "norm")


def draft_from_target_layer0(target: dict, draft_shape: ModelShape, noise_std: float,
                             seed: int) -> dict:
    """Tiny-workload draft: one layer equal to the target's layer 0 plus
    N(0, noise_std) noise (added in fp32, then rounded to the target's dtype),
    sharing the target's embedding, final norm and LM head.
    """
    assert draft_shape.layers == 1
    out = {"embed": target["embed"], "norm": target["norm"]}
    if not draft_shape.tied:
        out["lm_head"] = target["lm_head"]
    for j, name in enumerate(weight_names(draft_shape)):
        if not name.startswith("layers.0."):
            continue
        src = target[name]
        if src is None or _is_gain(name):
            out[name] = src
            continue
        noise = _normal(tuple(src.shape), _tensor_seed(seed, j, 1), src.device, noise_std)
        out[name] = (src.float() + noise).to(src.dtype)
    return out


def perturbed_copy(weights: dict, sigma: float, seed: int) -> dict:
    """A copy of ``weights`` with N(0, sigma) noise on every random-init tensor
    (norm gains untouched). sigma == 0 returns fresh copies of the tensors."""
    out = {}
    for j, (name, src) in enumerate(weights.items()):
        if src is None:
            out[name] = None
        elif sigma == 0.0 or _is_gain(name):
            out[name] = src.clone()
        else:
            noise = _normal(tuple(src.shape), _tensor_seed(seed, j, 2), src.device, sigma)
            out[name] = (src.float() + noise).to(src.dtype)
    return out


def shared_embedding_draft(draft: dict, target_embed: torch.Tensor, hidden: int) -> dict:
    """Replace the draft's (tied) embedding by the target embedding's first
    ``hidden`` columns: a strided view, row stride = the target's hidden size."""
    out = dict(draft)
    out["embed"] = target_embed[:, :hidden]
    return out


def to_device(weights: dict, device, dtype=None) -> dict:
    """Copy every tensor of a weight dict to ``device`` (optionally casting).
    A strided view is copied as it is; rebuild shared views after the copy."""
    out = {}
    for k, v in weights.items():
        if v is None:
            out[k] = None
        else:
            t = v.to(device)
            out[k] = t if dtype is None else t.to(dtype)
    return out
