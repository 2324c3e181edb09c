"""Helpers shared by the GPU parity tests (imported only by tests)."""

import numpy as np
import torch

from oracle import model as om

LOGIT_TOL_BF16 = 3e-2   # max |gpu - oracle| <= tol * (max - min of the oracle logits), per row


def to_cuda(w: dict) -> dict:
    return {k: (None if v is None else v.to("cuda")) for k, v in w.items()}


def to_cpu(w: dict) -> dict:
    return {k: (None if v is None else v.detach().to("cpu")) for k, v in w.items()}


def logit_err(gpu_row: torch.Tensor, ref_row: torch.Tensor) -> float:
    """max |gpu - oracle| / (max - min of the oracle row)."""
    g = gpu_row.double().cpu()
    r = ref_row.double().cpu()
    return float((g - r).abs().max() / (r.max() - r.min()))


def check_token_against_oracle(tok: int, ref_logits: torch.Tensor, tol: float = LOGIT_TOL_BF16):
    """A GPU token must be the oracle's argmax unless the oracle's own logit
    for it is within tol * range of the best (a near tie: logged, not failed).
    Returns 'exact' or 'near-tie'."""
    best = om.first_argmax(ref_logits)
    if tok == best:
        return "exact"
    rng = float(ref_logits.max() - ref_logits.min())
    gap = float(ref_logits[best] - ref_logits[tok])
    assert gap < tol * rng, f"token {tok} vs oracle {best}: gap {gap:.4g} >= tol {tol * rng:.4g}"
    return "near-tie"


def teacher_forced_stream_check(model: om.Model, prompt, stream, tol=LOGIT_TOL_BF16):
    """Score the GPU's generated stream with the oracle, position by position
    (teacher forcing). Returns the number of near-tie positions."""
    cache = model.new_cache()
    seq = list(prompt)
    model.forward(seq[:-1], cache, logit_rows=[])
    near = 0
    for t in stream:
        ref = model.forward([seq[-1]], cache)[0]
        if check_token_against_oracle(int(t), ref, tol) == "near-tie":
            near += 1
        seq.append(int(t))
    return near


def stream_report(model: om.Model, prompt, stream, tol=LOGIT_TOL_BF16):
    """Teacher-forced comparison of a GPU token stream with the oracle: at
    every position the oracle scores the prefix the GPU committed. Returns
    (positions, flips, near_ties): near_ties counts positions whose oracle
    top-2 gap is below tol * the row's logit range (where the pages allow a
    different choice), flips the positions where the GPU token is not the
    oracle's argmax. Every flip must be a near tie (asserted)."""
    cache = model.new_cache()
    seq = list(prompt)
    model.forward(seq[:-1], cache, logit_rows=[])
    flips = near = 0
    for t in stream:
        ref = model.forward([seq[-1]], cache)[0]
        top = torch.topk(ref, 2).values
        if float(top[0] - top[1]) < tol * float(ref.max() - ref.min()):
            near += 1
        if check_token_against_oracle(int(t), ref, tol) == "near-tie":
            flips += 1
        seq.append(int(t))
    return len(stream), flips, near


def accept_brute(d, t, limit):
    n = 0
    for m in range(limit + 1):
        if all(int(d[j]) == int(t[j]) for j in range(m)):
            n = m
    return n


def np_i32(x):
    return np.asarray(x, dtype=np.int32)
