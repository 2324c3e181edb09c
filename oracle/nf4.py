"""NormalFloat-4 (NF4) blockwise quantisation (test oracle).

Test infrastructure only (see the package docstring).

The pages name the format only ("Qwen2.5-14B with 4-bit NF4 quantization", I
Got 28 TPS Out of Free Kaggle GPUs, "The Numbers"). Readings:
  * Codebook: the NormalFloat construction of Dettmers et al., "QLoRA:
    Efficient Finetuning of Quantized LLMs" (2023), section 3: quantiles of
    N(0, 1), asymmetric so that zero is exact -- 8 positive levels and 7
    negative ones plus 0, normalised to [-1, 1]. The quantile grid runs from
    probability 1/2 to ``OFFSET`` = ((1 - 1/32) + (1 - 1/30)) / 2, the midpoint
    of the outermost probabilities of a 16- and a 15-point grid, which keeps
    the extreme levels finite.
  * Blocks of 64 consecutive inputs of one output row; the block scale is its
    largest magnitude, stored as fp16 (round to nearest even).
  * A weight w maps to the nearest level of w / scale; the decision is taken
    in fp32 against fp32 midpoints of adjacent fp32 levels, ties going to the
    lower index. Scale 0: every code is the zero level.
  * Two codes per byte: element 2i in the low nibble, 2i+1 in the high one.
  * Dequantised weight = level[code] * scale.
"""

import torch

F64 = torch.float64
BLOCK = 64
OFFSET = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0))


def codebook() -> torch.Tensor:
    """The 16 NF4 levels in increasing order (float64)."""
    pos_p = torch.linspace(OFFSET, 0.5, 9, dtype=F64)[:-1]     # 8 probabilities > 1/2
    neg_p = torch.linspace(OFFSET, 0.5, 8, dtype=F64)[:-1]     # 7 probabilities > 1/2
    pos = torch.special.ndtri(pos_p)
    neg = -torch.special.ndtri(neg_p)
    levels = torch.cat([neg, torch.zeros(1, dtype=F64), pos])
    levels = levels / levels.abs().max()
    return torch.sort(levels).values


def midpoints_f32() -> torch.Tensor:
    """fp32 decision thresholds between adjacent fp32 levels."""
    lv = codebook().to(torch.float32)
    return (lv[:-1] + lv[1:]) * 0.5


def quantize(w: torch.Tensor):
    """w: [rows, cols] (cols a multiple of 64), any float dtype.

    Returns (packed uint8 [rows, cols/2], absmax fp16 [rows, cols/64]).
    """
    rows, cols = w.shape
    assert cols % BLOCK == 0
    wf = w.to(torch.float32).reshape(rows, cols // BLOCK, BLOCK)
    absmax = wf.abs().amax(dim=2).to(torch.float16)
    scale = absmax.to(torch.float32)[..., None]
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    x = wf / safe                                   # fp32 division
    mids = midpoints_f32()
    # code = number of thresholds strictly below x (ties -> lower index)
    codes = (x[..., None] > mids).sum(-1).to(torch.uint8)
    zero_code = int(torch.nonzero(codebook() == 0)[0, 0])
    codes = torch.where(scale > 0, codes, torch.full_like(codes, zero_code))
    codes = codes.reshape(rows, cols)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.contiguous(), absmax.contiguous()


def unpack(packed: torch.Tensor) -> torch.Tensor:
    rows, half = packed.shape
    codes = torch.empty((rows, half * 2), dtype=torch.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    return codes


def dequantize(packed: torch.Tensor, absmax: torch.Tensor) -> torch.Tensor:
    """float64 [rows, cols] = level[code] * scale."""
    codes = unpack(packed.cpu()).long()
    rows, cols = codes.shape
    lv = codebook()
    scale = absmax.cpu().to(F64).repeat_interleave(BLOCK, dim=1)
    return lv[codes] * scale
