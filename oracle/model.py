"""fp64 forward pass of a Qwen2-style decoder over a KV cache (test oracle).

Test infrastructure only (see the package docstring). The pages fix no model
equations; everything here is the plain textbook definition of the
architecture the workloads name, and each choice that the pages leave open is
marked "reading".

Every row (token) is computed on its own: each linear map is a matrix-vector
product for that row alone, and attention for a row reads only the cache
slots at or before its position. So a row's result does not depend on how
many rows are processed together, which makes "speculative output equals
greedy output" exact inside the oracle.
"""

import math

import torch

F64 = torch.float64


class KVCache:
    """Per-layer keys and values of one sequence: slot j of layer l holds the
    [n_kv_heads, head_dim] float64 key/value of the token at position j.

    Rollback ("in-place KV rewind" in "Why It Kept Breaking (and How I Fixed
    It)") is ``truncate(n)``: the slots at and beyond n stop being part of the
    cache. Storage grows by doubling so that appends stay cheap.
    """

    def __init__(self, layers: int, n_kv_heads: int, head_dim: int, capacity: int = 64):
        self._k = [torch.zeros((capacity, n_kv_heads, head_dim), dtype=F64) for _ in range(layers)]
        self._v = [torch.zeros((capacity, n_kv_heads, head_dim), dtype=F64) for _ in range(layers)]
        self._len = [0] * layers

    @property
    def length(self) -> int:
        return self._len[0]

    def append(self, layer: int, k: torch.Tensor, v: torch.Tensor):
        n = self._len[layer]
        if n == self._k[layer].shape[0]:
            self._k[layer] = torch.cat([self._k[layer], torch.zeros_like(self._k[layer])], 0)
            self._v[layer] = torch.cat([self._v[layer], torch.zeros_like(self._v[layer])], 0)
        self._k[layer][n] = k
        self._v[layer][n] = v
        self._len[layer] = n + 1

    def keys(self, layer: int) -> torch.Tensor:
        return self._k[layer][: self._len[layer]]

    def values(self, layer: int) -> torch.Tensor:
        return self._v[layer][: self._len[layer]]

    def truncate(self, n: int):
        assert 0 <= n <= self.length
        self._len = [n] * len(self._len)


def rmsnorm(x: torch.Tensor, g: torch.Tensor, eps: float) -> torch.Tensor:
    """x / sqrt(mean(x^2) + eps) * g for one row x (reading: standard RMSNorm)."""
    return x / torch.sqrt(torch.mean(x * x) + eps) * g


def rope(x: torch.Tensor, pos: int, theta: float) -> torch.Tensor:
    """Rotary embedding of one row of heads x [n_heads, head_dim] at position pos.

    Reading: rotate-half pairing of element i with i + head_dim/2, angle
    pos * theta^(-2i/head_dim), i.e. x1' = x1 cos - x2 sin, x2' = x2 cos + x1 sin.
    """
    hd = x.shape[-1]
    half = hd // 2
    i = torch.arange(half, dtype=F64)
    ang = float(pos) * torch.pow(torch.tensor(theta, dtype=F64), -2.0 * i / hd)
    c, s = torch.cos(ang), torch.sin(ang)
    x1, x2 = x[:, :half], x[:, half:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=1)


def silu(z: torch.Tensor) -> torch.Tensor:
    """z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + torch.exp(-z))


def attend(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, group: int) -> torch.Tensor:
    """Causal GQA attention of one query row.

    q: [n_heads, hd]; k, v: [n_slots, n_kv_heads, hd] holding exactly the slots
    this row may see (0..its position). Query head h reads KV head h // group
    (reading: grouped-query attention with contiguous groups). Scale 1/sqrt(hd),
    softmax with the maximum subtracted.
    """
    nh, hd = q.shape
    out = torch.empty((nh, hd), dtype=F64)
    scale = 1.0 / math.sqrt(hd)
    for h in range(nh):
        kvh = h // group
        s = torch.mv(k[:, kvh, :], q[h]) * scale
        p = torch.exp(s - torch.max(s))
        p = p / torch.sum(p)
        out[h] = torch.mv(v[:, kvh, :].t(), p)
    return out


def first_argmax(logits: torch.Tensor) -> int:
    """Index of the largest logit; ties go to the lowest index (reading)."""
    m = torch.max(logits)
    return int(torch.nonzero(logits == m)[0, 0])


class Model:
    """One decoder (target or draft) with weights given as a dict of tensors in
    the canonical names (embed, layers.i.{ln1,wq,wk,wv,bq,bk,bv,wo,ln2,wg,wu,wd},
    norm, lm_head). Tensors may be bf16 or fp32; they are widened to fp64 when
    used. ``memoize`` keeps the widened copies (small models only).

    ``rowwise`` (default True) computes every linear map one row at a time
    (torch.mv), so each row's result is independent of the others. With
    ``rowwise=False`` the rows of a call share one matrix product (torch.mm):
    the same mathematics, each weight read once instead of once per row, for
    the full-size shapes where a per-row pass over 60 GB of float64 weights
    would take minutes; rows may then differ from a one-row call in the last
    bits.
    """

    def __init__(self, shape, weights: dict, memoize=None, rowwise=True):
        self.shape = shape
        self.w = weights
        if memoize is None:
            memoize = shape.n_params() < 60_000_000
        self._memo = {} if memoize else None
        self.rowwise = rowwise

    def lin(self, W: torch.Tensor, rows: list) -> list:
        """W @ r for every row r (W is [out, in])."""
        if not rows:
            return []
        if self.rowwise or len(rows) == 1:
            return [torch.mv(W, r) for r in rows]
        y = torch.mm(torch.stack(rows), W.t())
        return [y[i] for i in range(len(rows))]

    def W(self, name: str) -> torch.Tensor:
        if self._memo is not None and name in self._memo:
            return self._memo[name]
        t = self.w[name]
        t = None if t is None else t.detach().to("cpu").to(F64)
        if self._memo is not None:
            self._memo[name] = t
        return t

    def new_cache(self) -> KVCache:
        s = self.shape
        return KVCache(s.layers, s.n_kv_heads, s.head_dim)

    def forward(self, tokens, cache: KVCache, logit_rows=None):
        """Run ``tokens`` (list of ints) at positions cache.length, ... and
        append their keys/values to ``cache``.

        Returns {row: fp64 logits [vocab]} for each row in ``logit_rows``
        (default: every row).
        """
        s = self.shape
        M = len(tokens)
        pos0 = cache.length
        if logit_rows is None:
            logit_rows = range(M)
        group = s.n_heads // s.n_kv_heads
        E = self.W("embed")
        xs = [E[int(t)].clone() for t in tokens]
        for l in range(s.layers):
            p = f"layers.{l}."
            g1, g2 = self.W(p + "ln1"), self.W(p + "ln2")
            wq, wk, wv, wo = self.W(p + "wq"), self.W(p + "wk"), self.W(p + "wv"), self.W(p + "wo")
            bq, bk, bv = self.W(p + "bq"), self.W(p + "bk"), self.W(p + "bv")
            wg, wu, wd = self.W(p + "wg"), self.W(p + "wu"), self.W(p + "wd")
            # Keys and values of all rows first: row m may attend to rows < m.
            hs = [rmsnorm(x, g1, s.rms_eps) for x in xs]
            qs, ks, vs = self.lin(wq, hs), self.lin(wk, hs), self.lin(wv, hs)
            for m in range(M):
                q, k, v = qs[m], ks[m], vs[m]
                if bq is not None:
                    q, k, v = q + bq, k + bk, v + bv
                qs[m] = rope(q.view(s.n_heads, s.head_dim), pos0 + m, s.rope_theta)
                k = rope(k.view(s.n_kv_heads, s.head_dim), pos0 + m, s.rope_theta)
                cache.append(l, k, v.view(s.n_kv_heads, s.head_dim))
            attn = []
            for m in range(M):
                n_vis = pos0 + m + 1
                a = attend(qs[m], cache.keys(l)[:n_vis], cache.values(l)[:n_vis], group)
                attn.append(a.reshape(-1))
            os_ = self.lin(wo, attn)
            xs = [xs[m] + os_[m] for m in range(M)]
            h2 = [rmsnorm(x, g2, s.rms_eps) for x in xs]
            gs, us = self.lin(wg, h2), self.lin(wu, h2)
            ds = self.lin(wd, [silu(gs[m]) * us[m] for m in range(M)])
            xs = [xs[m] + ds[m] for m in range(M)]
            if self._memo is None:
                del wq, wk, wv, wo, wg, wu, wd
        gf = self.W("norm")
        lm = E if s.tied else self.W("lm_head")
        rows = list(logit_rows)
        ls = self.lin(lm, [rmsnorm(xs[m], gf, s.rms_eps) for m in rows])
        return dict(zip(rows, ls))
