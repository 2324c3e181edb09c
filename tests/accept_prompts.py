"""Prompts that make prompt-lookup drafting propose exactly j correct guesses
(test input construction; uses the oracle only).

A prompt has the form A + s + Y + B + s: its last four tokens s occurred once
before, followed by Y, so the lookup ("Speculative decoding: correct, but
slower (for now)", Sangama page: guess what followed the last 2-4 tokens the
last time they appeared) proposes Y[0..4). Along an accepted prefix the
target's choices are the greedy continuation g of the prompt, so the accept
length is j exactly when Y[0..j) == g[0..j) and Y[j] != g[j]. g depends on Y
(attention reads it), so Y is found as a fixed point: set Y from g, recompute
g, repeat until nothing changes. Prompts whose decisive choices are near ties
of the oracle (top-2 gap below the logit tolerance) are skipped, so the GPU
must make the same choices.
"""

import torch

from oracle import decode as od
from oracle import model as om


def _greedy_margins(model, prompt, n):
    cache = model.new_cache()
    model.forward(prompt[:-1], cache, logit_rows=[])
    seq, out, margins = list(prompt), [], []
    for _ in range(n):
        lg = model.forward([seq[-1]], cache)[0]
        t = om.first_argmax(lg)
        top = torch.topk(lg, 2).values
        margins.append(float((top[0] - top[1]) / (lg.max() - lg.min())))
        out.append(t)
        seq.append(t)
    return out, margins


def planted_prompt(model, vocab, j, K=4, seed=0, a_len=20, tol=3e-2, tries=64):
    """(prompt, greedy continuation of j + 1 tokens) such that the n-gram
    drafter with max_guess K proposes K tokens of which exactly the first j
    are the target's choices."""
    for attempt in range(tries):
        g = torch.Generator().manual_seed(seed * 1000 + attempt)
        rnd = lambda n: torch.randint(0, vocab, (n,), generator=g).tolist()
        A, s, B, Y = rnd(a_len), rnd(4), rnd(6), rnd(K + 1)
        for _ in range(8):
            P = A + s + Y + B + s
            gr, mg = _greedy_margins(model, P, j + 1)
            head = gr[:j]
            if j < K:
                head = head + [Y[j] if Y[j] != gr[j] else (gr[j] + 1) % vocab]
            Yn = head + Y[len(head):]
            if Yn == Y:
                break
            Y = Yn
        else:
            continue
        prop = od.ngram_propose(P, K, 2, 4)
        if prop != Y[:K] or min(mg) <= tol:
            continue
        if od.accept_length(prop, gr + [-1] * (K + 1 - len(gr)), len(prop)) != j:
            continue
        return P, gr
    raise RuntimeError(f"no planted prompt for j={j}")


def planted_tree_prompt(model, vocab, ns, g, seed=0, a_len=20, tol=3e-2, tries=64):
    """(prompt, greedy continuation) such that multi-candidate prompt lookup
    (oracle ngram_candidates with len(ns) candidates of g tokens) proposes
    len(ns) guesses of which guess c starts with exactly ns[c] of the
    target's choices. The prompt is A + (s + Y_c + B_c for c from last to
    first) + s: the most recent occurrence of s is followed by Y_0, the one
    before it by Y_1, and so on; each Y_c is planted by the same fixed point
    as planted_prompt."""
    n_cand = len(ns)
    for attempt in range(tries):
        gen = torch.Generator().manual_seed(seed * 1000 + attempt)
        rnd = lambda n: torch.randint(0, vocab, (n,), generator=gen).tolist()
        A, s = rnd(a_len), rnd(4)
        Bs = [rnd(5) for _ in ns]
        Ys = [rnd(g + 1) for _ in ns]
        for _ in range(8):
            P = list(A)
            for c in reversed(range(n_cand)):
                P += s + Ys[c] + Bs[c]
            P += s
            gr, mg = _greedy_margins(model, P, max(ns) + 1)
            new = []
            for c, n in enumerate(ns):
                head = gr[:n]
                if n < g:
                    head = head + [Ys[c][n] if Ys[c][n] != gr[n] else (gr[n] + 1) % vocab]
                new.append(head + Ys[c][len(head):])
            if new == Ys:
                break
            Ys = new
        else:
            continue
        if od.ngram_candidates(P, n_cand, g, 2, 4) != [y[:g] for y in Ys] or min(mg) <= tol:
            continue
        pad = gr + [-1] * (g + 1 - len(gr))
        if [od.accept_length(y[:g], pad, g) for y in Ys] != list(ns):
            continue
        return P, gr
    raise RuntimeError(f"no planted prompt for accept lengths {ns}")
