"""Greedy decoding and the greedy speculative loop (test oracle).

Test infrastructure only (see the package docstring).

Conventions shared with the engine under test:
  * The committed sequence S has C tokens. Each model's cache holds the keys
    and values of S[0..C-2]; the last token S[C-1] is "pending": it is the
    next input and is not in the target cache yet.
  * One speculative round, per "Speculative Decoding: The Idea" (I Got 28 TPS
    Out of Free Kaggle GPUs): the drafter proposes K tokens d_1..d_K; the
    target runs once over [S[C-1], d_1, ..., d_K] at positions C-1..C+K-1 and
    returns its own greedy choice t_0..t_K at every position ("the last worker
    returns the model's own choice at every position", Sangama results,
    "Speculative decoding: correct, but slower (for now)"); the accepted
    length n is the number of leading guesses that agree with those choices,
    and d_1..d_n plus the target's choice t_n after them are committed
    (reading: the "bonus" token t_n is what plain greedy decoding would emit
    next, so committing it keeps the output equal to greedy decoding).
  * Rollback ("In-place KV rewind", Why It Kept Breaking (and How I Fixed It)):
    the target cache is cut back to the C_new - 1 committed tokens.
"""

from .model import Model, first_argmax


def greedy(model: Model, prompt, n_new: int):
    """Plain greedy decoding: the definition that speculative decoding must
    reproduce token for token. Returns the n_new generated tokens."""
    seq = [int(t) for t in prompt]
    cache = model.new_cache()
    if len(seq) > 1:
        model.forward(seq[:-1], cache, logit_rows=[])
    out = []
    while len(out) < n_new:
        logits = model.forward([seq[-1]], cache)[0]
        t = first_argmax(logits)
        seq.append(t)
        out.append(t)
    return out


def accept_length(draft, target_choice, limit=None) -> int:
    """Longest prefix of guesses that agree with the target: the largest n
    (n <= limit, default len(draft)) with draft[j] == target_choice[j] for all
    j < n. ``target_choice[j]`` is the target's token after the j-th input row,
    i.e. the token it would emit where draft[j] was guessed."""
    n = 0
    lim = len(draft) if limit is None else limit
    while n < lim and int(draft[n]) == int(target_choice[n]):
        n += 1
    return n


def ngram_propose(ctx, max_guess: int = 4, min_n: int = 2, max_n: int = 4):
    """Prompt-lookup guess (Sangama results, "Speculative decoding: correct,
    but slower (for now)": if the last 2-4 tokens appeared earlier, guess what
    followed them then).

    Readings where the page is silent: the longest suffix length n is tried
    first (max_n down to min_n); for that n the rightmost earlier occurrence
    is taken (a start j with j + n < len(ctx), which may overlap the suffix);
    the guess is the up to ``max_guess`` tokens that followed it, cut at the
    end of the context. No occurrence: no guess.
    """
    ctx = [int(t) for t in ctx]
    T = len(ctx)
    for n in range(max_n, min_n - 1, -1):
        if n > T - 1:
            continue
        suffix = ctx[T - n:]
        for j in range(T - n - 1, -1, -1):
            if ctx[j:j + n] == suffix:
                return ctx[j + n: min(j + n + max_guess, T)]
    return []


def ngram_candidates(ctx, n_cand: int, max_guess: int = 4, min_n: int = 2, max_n: int = 4):
    """Several prompt-lookup guesses at once (the Sangama page's "Next":
    better guesses; here several earlier occurrences verified together).

    Readings where the page is silent: the occurrences are visited in the
    order ngram_propose ranks them (longest suffix length n first, max_n down
    to min_n; for each n the rightmost earlier start j < len(ctx) - n first,
    leftward); each gives the up to ``max_guess`` tokens that followed it,
    cut at the end of the context; an empty guess or one equal to a guess
    already taken is skipped; at most ``n_cand`` guesses. The first guess is
    ngram_propose's.
    """
    ctx = [int(t) for t in ctx]
    T = len(ctx)
    out = []
    for n in range(max_n, min_n - 1, -1):
        if n > T - 1:
            continue
        suffix = ctx[T - n:]
        for j in range(T - n - 1, -1, -1):
            if ctx[j:j + n] == suffix:
                g = ctx[j + n: min(j + n + max_guess, T)]
                if g and g not in out:
                    out.append(g)
                    if len(out) == n_cand:
                        return out
    return out


def tree_accept(guesses, choices):
    """Acceptance over several guesses verified in one pass. ``guesses[c]``
    is candidate c's token list; ``choices[c][j]`` is the target's own choice
    after the pending token and guesses[c][:j] (choices[c][0] is the same
    for every c: the choice after the pending token). Candidate c accepts
    n_c = accept_length(guesses[c], choices[c]); the candidate with the
    largest n_c is taken, the lowest index on ties (reading). Returns
    (c, n, committed = guesses[c][:n] + [choices[c][n]])."""
    best_c, best_n = 0, -1
    for c, (g, t) in enumerate(zip(guesses, choices)):
        n = accept_length(g, t, len(g))
        if n > best_n:
            best_c, best_n = c, n
    g, t = guesses[best_c], choices[best_c]
    return best_c, best_n, list(g[:best_n]) + [t[best_n]]


def spec_decode(target: Model, draft, prompt, K: int, n_new: int, drafter: str = "neural",
                min_n: int = 2, max_n: int = 4, n_cand: int = 1):
    """Greedy speculative decoding of n_new tokens after ``prompt``.

    drafter == "neural": ``draft`` is a Model proposing K tokens by its own
    greedy decoding. drafter == "ngram": ``draft`` is unused; up to K tokens
    come from ngram_propose over the committed sequence (unfilled guess slots
    hold token 0 and never count as accepted). drafter == "tree": up to
    ``n_cand`` guesses of up to K // n_cand tokens from ngram_candidates, each
    scored by the target on its own (the pending token and the guess from the
    committed state), the best taken by tree_accept; no guess: the target's
    own next token.

    Returns dict(tokens=[n_new generated tokens], rounds=[(n_accepted,
    committed_tokens, proposals, target_choices), ...]).
    """
    seq = [int(t) for t in prompt]
    C0 = len(seq)
    tcache = target.new_cache()
    if C0 > 1:
        target.forward(seq[:-1], tcache, logit_rows=[])
    dcache, dtoks = None, []
    if drafter == "neural":
        dcache = draft.new_cache()
        if C0 > 1:
            draft.forward(seq[:-1], dcache, logit_rows=[])
        dtoks = seq[:-1]               # tokens whose entries dcache holds
    rounds = []
    while len(seq) - C0 < n_new:
        C = len(seq)
        assert tcache.length == C - 1
        # ---- draft ----
        if drafter == "neural":
            # Keep the draft cache entries that still match the committed
            # sequence, then feed it the committed tokens it has not seen
            # (the pending one, and the last accepted guess when every guess
            # was accepted) and let it decode greedily.
            keep = 0
            while keep < min(len(dtoks), C - 1) and dtoks[keep] == seq[keep]:
                keep += 1
            dcache.truncate(keep)
            dtoks = dtoks[:keep]
            feed = seq[keep:]
            guesses = []
            for _ in range(K):
                logits = draft.forward(feed, dcache, logit_rows=[len(feed) - 1])
                dtoks += feed
                g = first_argmax(logits[len(feed) - 1])
                guesses.append(g)
                feed = [g]
            limit = K
        elif drafter == "tree":
            cands = ngram_candidates(seq, n_cand, K // n_cand, min_n, max_n) or [[]]
            choices = []
            for g in cands:
                lg = target.forward([seq[-1]] + g, tcache)
                choices.append([first_argmax(lg[i]) for i in range(len(g) + 1)])
                tcache.truncate(C - 1)            # each guess is scored from the committed state
            c, n, committed = tree_accept(cands, choices)
            # Keys and values of the pending token and the accepted guesses.
            target.forward([seq[-1]] + cands[c][:n], tcache, logit_rows=[])
            seq += committed
            rounds.append((n, committed, cands, choices))
            continue
        else:
            prop = ngram_propose(seq, K, min_n, max_n)
            limit = len(prop)
            guesses = prop + [0] * (K - len(prop))
        # ---- verify: one target pass over the pending token and the guesses ----
        rows = [seq[-1]] + guesses
        logits = target.forward(rows, tcache)
        choice = [first_argmax(logits[i]) for i in range(K + 1)]
        # ---- accept ----
        n = accept_length(guesses, choice, limit)
        committed = guesses[:n] + [choice[n]]
        seq += committed
        # ---- rollback: the target cache keeps the C_new - 1 committed tokens ----
        tcache.truncate(len(seq) - 1)
        rounds.append((n, committed, guesses, choice))
    return {"tokens": seq[C0:C0 + n_new], "rounds": rounds}
