"""Model shapes of the workloads (decoder-only, GQA + RoPE + RMSNorm + SwiGLU).

The shapes follow the Qwen2.5 family sizes that the workloads name: a tiny
correctness model, the 0.5B draft, the 7B target and the 14B target.
"""

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class ModelShape:
    layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied: bool = True          # LM head is the embedding matrix
    qkv_bias: bool = True      # Qwen2-style biases on q, k, v
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    embed_ld: int = 0          # row stride of the embedding in elements (0: hidden)

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def with_(self, **kw) -> "ModelShape":
        return replace(self, **kw)

    def n_params(self) -> int:
        h, f = self.hidden, self.ffn
        per_layer = (2 * h + h * self.q_dim + 2 * h * self.kv_dim + self.q_dim * h
                     + 3 * h * f + (self.q_dim + 2 * self.kv_dim if self.qkv_bias else 0))
        emb = self.vocab * h
        return emb + self.layers * per_layer + h + (0 if self.tied else emb)


# Tiny correctness model: 2 layers, hidden 256, 4/2 heads of 64, FFN 688, vocab 1024.
TINY_TARGET = ModelShape(layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
                         ffn=688, vocab=1024, tied=True)
# Its draft: one layer of the same architecture, sharing embedding / LM head.
TINY_DRAFT = TINY_TARGET.with_(layers=1)
# Qwen2.5-0.5B shape (standalone draft decode step).
QWEN05B = ModelShape(layers=24, hidden=896, n_heads=14, n_kv_heads=2, head_dim=64,
                     ffn=4864, vocab=151936, tied=True)
# The 0.5B draft whose embedding is the 7B target's first 896 columns: its
# vocabulary becomes the target's 152064 and its embedding rows are strided.
QWEN05B_SHARED = QWEN05B.with_(vocab=152064, embed_ld=3584)
# Qwen2.5-7B shape target, untied LM head.
QWEN7B = ModelShape(layers=28, hidden=3584, n_heads=28, n_kv_heads=4, head_dim=128,
                    ffn=18944, vocab=152064, tied=False)
# Qwen2.5-14B shape target.
QWEN14B = ModelShape(layers=48, hidden=5120, n_heads=40, n_kv_heads=8, head_dim=128,
                     ffn=13824, vocab=152064, tied=False)


LAYER_TENSORS = ("ln1", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "ln2", "wg", "wu", "wd")


def weight_names(shape: ModelShape) -> list:
    """Canonical tensor order: embed, per layer (ln1, wq, wk, wv, bq, bk, bv, wo,
    ln2, wg, wu, wd), final norm, lm_head (absent when tied).

    Biases are listed even when ``qkv_bias`` is False so that the order never
    shifts; such entries are None.
    """
    names = ["embed"]
    for i in range(shape.layers):
        names += [f"layers.{i}.{t}" for t in LAYER_TENSORS]
    names.append("norm")
    if not shape.tied:
        names.append("lm_head")
    return names


def weight_shape(shape: ModelShape, name: str):
    h = shape.hidden
    if name == "embed" or name == "lm_head":
        return (shape.vocab, h)
    if name == "norm":
        return (h,)
    t = name.split(".")[-1]
    return {
        "ln1": (h,), "ln2": (h,),
        "wq": (shape.q_dim, h), "wk": (shape.kv_dim, h), "wv": (shape.kv_dim, h),
        "bq": (shape.q_dim,), "bk": (shape.kv_dim,), "bv": (shape.kv_dim,),
        "wo": (h, shape.q_dim),
        "wg": (shape.ffn, h), "wu": (shape.ffn, h), "wd": (h, shape.ffn),
    }[t]
