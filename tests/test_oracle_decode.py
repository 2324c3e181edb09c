"""Pins for the oracle's speculative loop (CPU only).

* Speculative output equals plain greedy decoding token for token (Sangama
  results, "Speculative decoding: correct, but slower (for now)": every
  speculative run produced exactly the same tokens as normal decoding).
* Accept length and the committed tokens against hand cases and a brute
  force.
* N-gram lookup against hand cases and an exhaustive search.
* Rollback: after every round the target cache is exactly the cache a fresh
  pass over the committed prefix produces.
"""

import json
import os
import random

import pytest
import torch

from oracle import decode as od
from oracle import model as om
from synth import (TINY_DRAFT, TINY_TARGET, draft_from_target_layer0, make_weights,
                   ngram_prompt, perturbed_copy, uniform_prompt)

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_accept_golden():
    for c in _load("accept_cases.json")["cases"]:
        n = od.accept_length(c["draft"], c["choice"], c["limit"])
        assert n == c["n"], c
        assert c["draft"][:n] + [c["choice"][n]] == c["committed"]


def _accept_brute(d, t, limit):
    best = 0
    for m in range(limit + 1):
        if all(d[j] == t[j] for j in range(m)):
            best = m
    return best


def test_accept_brute_force():
    rng = random.Random(5)
    for _ in range(3000):
        K = rng.randint(1, 9)
        t = [rng.randint(0, 3) for _ in range(K + 1)]
        d = [t[j] if rng.random() < 0.7 else rng.randint(0, 3) for j in range(K)]
        lim = rng.randint(0, K)
        assert od.accept_length(d, t, lim) == _accept_brute(d, t, lim)


def test_ngram_golden():
    for c in _load("ngram_cases.json")["cases"]:
        assert od.ngram_propose(c["ctx"], c["max_guess"], 2, 4) == c["prop"], c


def _ngram_brute(ctx, max_guess, min_n, max_n):
    T = len(ctx)
    matches = []
    for n in range(min_n, max_n + 1):
        for j in range(0, T - n):
            if all(ctx[j + i] == ctx[T - n + i] for i in range(n)):
                matches.append((n, j))
    if not matches:
        return []
    n, j = max(matches)
    return ctx[j + n: j + n + max_guess]


def test_ngram_brute_force():
    rng = random.Random(6)
    for _ in range(2000):
        T = rng.randint(0, 40)
        V = rng.choice([2, 3, 5, 50])
        ctx = [rng.randrange(V) for _ in range(T)]
        mg = rng.randint(1, 6)
        lo = rng.randint(1, 3)
        hi = rng.randint(lo, 5)
        assert od.ngram_propose(ctx, mg, lo, hi) == _ngram_brute(ctx, mg, lo, hi), (ctx, mg, lo, hi)


@pytest.fixture(scope="module")
def tiny_models():
    tw = make_weights(TINY_TARGET, seed=0)
    dw = draft_from_target_layer0(tw, TINY_DRAFT, 0.005, seed=1)
    return om.Model(TINY_TARGET, tw), om.Model(TINY_DRAFT, dw), tw


@pytest.fixture(scope="module")
def tiny_greedy(tiny_models):
    target, _, _ = tiny_models
    prompt = uniform_prompt(32, 1024, seed=100).tolist()
    return prompt, od.greedy(target, prompt, 64)


@pytest.mark.parametrize("K", [1, 4, 7])
def test_spec_equals_greedy_tiny_draft(tiny_models, tiny_greedy, K):
    target, draft, _ = tiny_models
    prompt, ref = tiny_greedy
    res = od.spec_decode(target, draft, prompt, K, 64)
    assert res["tokens"] == ref
    assert all(0 <= r[0] <= K for r in res["rounds"])


def test_spec_target_copy_accepts_everything(tiny_models, tiny_greedy):
    target, _, tw = tiny_models
    prompt, ref = tiny_greedy
    copy = om.Model(TINY_TARGET, perturbed_copy(tw, 0.0, seed=3))
    K = 4
    res = od.spec_decode(target, copy, prompt, K, 64)
    assert res["tokens"] == ref
    assert all(r[0] == K and len(r[1]) == K + 1 for r in res["rounds"])


def test_spec_unrelated_draft_still_greedy(tiny_models, tiny_greedy):
    target, _, _ = tiny_models
    prompt, ref = tiny_greedy
    other = om.Model(TINY_DRAFT, make_weights(TINY_DRAFT, seed=55))
    res = od.spec_decode(target, other, prompt, 4, 64)
    assert res["tokens"] == ref


def test_spec_ngram_equals_greedy(tiny_models):
    target, _, _ = tiny_models
    prompt, _ = ngram_prompt(96, 0.8, 1024, seed=200, base_len=48, seg_lo=8, seg_hi=16)
    prompt = prompt.tolist()
    ref = od.greedy(target, prompt, 40)
    res = od.spec_decode(target, None, prompt, 4, 40, drafter="ngram")
    assert res["tokens"] == ref
    # The n-gram drafter must have proposed something on this repetitive prompt.
    assert any(any(g != 0 for g in r[2]) for r in res["rounds"])


def test_rollback_cache_equals_fresh_prefix(tiny_models):
    target, draft, _ = tiny_models
    prompt = uniform_prompt(20, 1024, seed=7).tolist()
    K = 4
    seq = list(prompt)
    tc = target.new_cache()
    target.forward(seq[:-1], tc, logit_rows=[])
    for _ in range(6):
        guesses = od.greedy(draft, seq, K)      # any proposals will do here
        logits = target.forward([seq[-1]] + guesses, tc)
        choice = [om.first_argmax(logits[i]) for i in range(K + 1)]
        n = od.accept_length(guesses, choice)
        seq += guesses[:n] + [choice[n]]
        tc.truncate(len(seq) - 1)
        fresh = target.new_cache()
        target.forward(seq[:-1], fresh, logit_rows=[])
        assert tc.length == len(seq) - 1
        for l in range(TINY_TARGET.layers):
            assert torch.equal(tc.keys(l), fresh.keys(l))
            assert torch.equal(tc.values(l), fresh.values(l))


def test_planted_prompts_give_every_accept_length():
    """The prompts the GPU accept tests use: prompt lookup proposes K = 4
    guesses of which exactly the first j agree with greedy decoding, for
    every j in 0..4 (checked against the oracle's own greedy continuation)."""
    from accept_prompts import planted_prompt
    from synth import TINY_TARGET, make_weights
    m = om.Model(TINY_TARGET, make_weights(TINY_TARGET, seed=0))
    for j in range(5):
        P, g = planted_prompt(m, TINY_TARGET.vocab, j, K=4, seed=7 + j, a_len=20 + 3 * j)
        prop = od.ngram_propose(P, 4, 2, 4)
        assert len(prop) == 4
        assert od.accept_length(prop, g + [-1] * (5 - len(g)), 4) == j
        assert g == od.greedy(m, P, j + 1)


def _candidates_by_sorting(ctx, n_cand, max_guess, min_n, max_n):
    """The multi-candidate reading restated another way: every (n, j) match
    sorted by longest n, then rightmost j; duplicates and empty guesses
    dropped; the first n_cand kept."""
    T = len(ctx)
    matches = [(n, j) for n in range(min_n, max_n + 1) if n <= T - 1
               for j in range(0, T - n) if ctx[j:j + n] == ctx[T - n:]]
    matches.sort(key=lambda nj: (-nj[0], -nj[1]))
    out = []
    for n, j in matches:
        g = ctx[j + n: min(j + n + max_guess, T)]
        if g and g not in out:
            out.append(g)
    return out[:n_cand]


def test_ngram_candidates_brute_force():
    rng = random.Random(11)
    for trial in range(400):
        T = rng.randint(1, 24)
        ctx = [rng.randint(0, 3) for _ in range(T)]
        for n_cand in (1, 2, 3, 4):
            for mg in (1, 3, 4):
                got = od.ngram_candidates(ctx, n_cand, mg, 2, 4)
                assert got == _candidates_by_sorting(ctx, n_cand, mg, 2, 4), (ctx, n_cand, mg)
                first = od.ngram_propose(ctx, mg, 2, 4)
                assert (got[:1] == [first]) if first else got == []


def test_tree_accept_cases():
    # candidate 1 agrees further than candidate 0
    assert od.tree_accept([[5, 6], [7, 8, 9]], [[5, 0, 0], [7, 8, 1, 2]]) == (1, 2, [7, 8, 1])
    # ties go to the lowest index; nothing agrees: the target's own token
    assert od.tree_accept([[3], [4]], [[9, 0], [9, 0]]) == (0, 0, [9])
    # a full agreement takes the bonus token after the last guess
    assert od.tree_accept([[1, 2]], [[1, 2, 3]]) == (0, 2, [1, 2, 3])
    # an empty guess list: plain greedy
    assert od.tree_accept([[]], [[42]]) == (0, 0, [42])


def test_tree_accept_brute_force():
    rng = random.Random(5)
    for _ in range(500):
        C = rng.randint(1, 4)
        gs = [[rng.randint(0, 2) for _ in range(rng.randint(0, 4))] for _ in range(C)]
        t0 = rng.randint(0, 2)
        ts = [[t0] + [rng.randint(0, 2) for _ in range(len(g))] for g in gs]
        c, n, com = od.tree_accept(gs, ts)
        ns = [max(m for m in range(len(g) + 1) if all(g[i] == t[i] for i in range(m))) for g, t in zip(gs, ts)]
        assert n == max(ns) and c == ns.index(max(ns))
        assert com == gs[c][:n] + [ts[c][n]]


@pytest.mark.parametrize("n_cand,K", [(1, 4), (2, 8), (3, 6)])
def test_tree_spec_decode_equals_greedy(n_cand, K):
    """Speculation with several guesses per round never changes the output."""
    from synth import ngram_prompt
    m = om.Model(TINY_TARGET, make_weights(TINY_TARGET, seed=0))
    for seed in (200, 201):
        prompt, _ = ngram_prompt(64, 0.8, TINY_TARGET.vocab, seed=seed, base_len=32, seg_lo=6, seg_hi=12)
        prompt = prompt.tolist()
        r = od.spec_decode(m, None, prompt, K, 24, drafter="tree", n_cand=n_cand)
        assert r["tokens"] == od.greedy(m, prompt, 24)
        for n, committed, cands, choices in r["rounds"]:
            assert len(cands) <= n_cand and all(len(g) <= K // n_cand for g in cands)
            assert committed[:n] == cands[[len(g) >= n and g[:n] == committed[:n] for g in cands].index(True)][:n]
