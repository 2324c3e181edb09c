"""Every accept length 0..K through the GPU's accept kernel, chosen on purpose.

Prompt-lookup drafting proposes the tokens that followed an earlier
occurrence of the context's last tokens; the prompts of accept_prompts.py
plant that earlier occurrence so that exactly j of the K = 4 guesses are the
target's own choices ("Speculative Decoding: The Idea": the target keeps the
guesses it agrees with and adds its own next token). For each j the test
checks, against the oracle and a brute-force prefix compare: the accepted
length, the committed tokens (the first j + 1 tokens of greedy decoding),
both cache lengths after the in-place rollback, and the same through the
graph-replayed round (sf_step). Batch 1 for every j, and batches of four
sequences with a different j each (ragged prompt lengths).
"""

import numpy as np
import pytest
import torch

from oracle import decode as od
from oracle import model as om
from synth import TINY_TARGET, make_weights

from accept_prompts import planted_prompt
from gpu_helpers import accept_brute, to_cuda

pytestmark = pytest.mark.gpu
K = 4


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as p
    return p


@pytest.fixture(scope="module")
def tiny():
    tw = make_weights(TINY_TARGET, seed=0)
    return tw, to_cuda(tw), om.Model(TINY_TARGET, tw)


@pytest.fixture(scope="module")
def planted(tiny):
    """j -> (prompt, greedy continuation); prompt lengths differ per j."""
    m = tiny[2]
    return {j: planted_prompt(m, TINY_TARGET.vocab, j, K=K, seed=7 + j, a_len=20 + 3 * j) for j in range(K + 1)}


def _round_checks(pkg, gt, items):
    B = len(items)
    prompts = [p for p, _ in items]
    eng = pkg.SpecEngine(TINY_TARGET, gt, batch=B, K=K, s_max=256)
    eng.prefill(prompts)
    prop = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
    t_out = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    eng.ngram_draft(K, 2, 4, prop, cnt)
    eng.verify(t_out)
    n_acc, committed = eng.accept_rollback()
    lt, ld = eng.lengths()
    prop_h, cnt_h, t_h = prop.cpu().numpy(), cnt.cpu().numpy(), t_out.cpu().numpy()
    for b, (P, greedy) in enumerate(items):
        j = len(greedy) - 1
        ref = od.ngram_propose(P, K, 2, 4)
        assert int(cnt_h[b]) == len(ref) == K
        assert prop_h[b].tolist() == ref
        n = accept_brute(prop_h[b], t_h[b], int(cnt_h[b]))
        assert int(n_acc[b]) == n == j, (b, j, n)
        assert committed[b] == ref[:j] + [int(t_h[b][j])] == greedy[:j + 1]
        assert int(lt[b]) == len(P) + j and int(ld[b]) == len(P) + j - 1
    hist = eng.accept_hist()
    for b, (_, greedy) in enumerate(items):
        want = np.zeros(K + 1, np.int32)
        want[len(greedy) - 1] = 1
        assert hist[b].tolist() == want.tolist()
    # The same round replayed as one graph from the rewound state.
    eng.reset()
    com = eng.step()
    lt2, _ = eng.lengths()
    for b, (P, greedy) in enumerate(items):
        assert com[b] == greedy
        assert int(lt2[b]) == len(P) + len(greedy) - 1
    eng.close()


@pytest.mark.parametrize("j", list(range(K + 1)))
def test_each_accept_length_batch1(pkg, tiny, planted, j):
    _round_checks(pkg, tiny[1], [planted[j]])


@pytest.mark.parametrize("order", [[3, 0, 4, 1], [2, 4, 1, 0]])
def test_mixed_accept_lengths_batch4(pkg, tiny, planted, order):
    _round_checks(pkg, tiny[1], [planted[j] for j in order])

