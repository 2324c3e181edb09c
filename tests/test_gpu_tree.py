"""Several prompt-lookup guesses verified in one target pass (SF_DRAFT_TREE),
against the oracle's ngram_candidates / tree_accept / spec_decode(drafter="tree").

* Candidates: the GPU lookup kernel's guesses and lengths equal the
  oracle's, bit for bit, on prompts with many repeats (ngram_prompt), an
  all-same-token prompt (every start matches, every guess a duplicate), a
  prompt without any repeat and a two-token prompt.
* One round on planted prompts (accept_prompts.planted_tree_prompt): guess c
  starts with exactly ns[c] of the target's choices. The verify logits of
  each candidate's rows equal the oracle's forward over the pending token
  and that guess alone (the rows of the other guesses are invisible to it);
  the accepted length is max(ns), the winner the first candidate reaching
  it, the committed tokens the greedy continuation; the winner's cache
  entries were moved to the committed slots bit for bit and nothing below
  them changed.
* A 7B-shape two-layer target at a 2-thousand-token context whose guesses
  straddle a 64-slot chunk boundary.
* Whole generations: the token stream is the oracle's greedy stream (flips
  only at near ties), and one candidate of K guesses reproduces the
  single-guess lookup exactly.
"""

import numpy as np
import pytest
import torch

from oracle import decode as od
from oracle import model as om
from synth import QWEN7B, TINY_TARGET, make_weights, uniform_prompt
from synth.prompts import ngram_prompt

from accept_prompts import planted_tree_prompt
from gpu_helpers import LOGIT_TOL_BF16, logit_err, stream_report, to_cpu, to_cuda

pytestmark = pytest.mark.gpu
V = TINY_TARGET.vocab


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


def _lookup_prompts():
    rep = [ngram_prompt(n, 0.8, V, seed=s, base_len=96)[0].tolist() for n, s in ((300, 1), (180, 2), (420, 3))]
    same = [7] * 200
    plain = uniform_prompt(150, V, seed=9).tolist()
    return rep + [same, plain, [3, 3]]


@pytest.mark.parametrize("K,n_cand", [(8, 2), (8, 4), (8, 3), (6, 6)])
def test_tree_candidates_match_oracle(pkg, tiny, K, n_cand):
    tw, gt, m = tiny
    prompts = _lookup_prompts()
    B, g = len(prompts), K // n_cand
    eng = pkg.SpecEngine(TINY_TARGET, gt, batch=B, K=K, s_max=512)
    eng.prefill(prompts)
    prop = torch.full((B, n_cand, g), -1, dtype=torch.int32, device="cuda")
    lens = torch.full((B, n_cand), -1, dtype=torch.int32, device="cuda")
    eng.tree_draft(n_cand, 2, 4, prop, lens)
    torch.cuda.synchronize()
    eng.close()
    for b, p in enumerate(prompts):
        ref = od.ngram_candidates(p, n_cand, g, 2, 4)
        got_len = lens[b].tolist()
        got = [prop[b, c, :got_len[c]].tolist() for c in range(n_cand) if got_len[c] > 0]
        assert got == ref, (b, got, ref)
        assert got_len == [len(x) for x in ref] + [0] * (n_cand - len(ref))
        for c in range(n_cand):
            assert prop[b, c, got_len[c]:].eq(0).all()


def _oracle_rows(m, prompt, guesses):
    """Oracle logits per candidate: the pending token and that guess alone,
    from the committed state."""
    cache = m.new_cache()
    m.forward(prompt[:-1], cache, logit_rows=[])
    base = len(prompt) - 1
    out = []
    for gs in guesses:
        out.append(m.forward([prompt[-1]] + list(gs), cache))
        cache.truncate(base)
    return out


PLANTED = [([1, 3], 4), ([2, 0], 4), ([0, 0], 4), ([4, 2], 4), ([0, 1, 2, 1], 2), ([3, 3], 4)]


@pytest.fixture(scope="module")
def planted(tiny):
    m = tiny[2]
    return [planted_tree_prompt(m, V, ns, g, seed=i + 1, a_len=21 + i) for i, (ns, g) in enumerate(PLANTED)]


def _round(pkg, gt, m, cases, prompts_gr, K):
    """One tree round over a batch; checks everything named in the module
    docstring for each sequence."""
    B = len(cases)
    n_cand = len(cases[0][0])
    g = K // n_cand
    prompts = [p for p, _ in prompts_gr]
    eng = pkg.SpecEngine(TINY_TARGET, gt, batch=B, K=K, s_max=256)
    eng.kv_t.fill_(0xFF)
    eng.prefill(prompts)
    prop = torch.zeros(B, n_cand, g, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, n_cand, dtype=torch.int32, device="cuda")
    t_arg = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    t_log = torch.zeros(B, K + 1, V, dtype=torch.float32, device="cuda")
    eng.tree_draft(n_cand, 2, 4, prop, lens)
    eng.verify(t_arg, t_log)
    torch.cuda.synchronize()
    kv_before = eng.kv_view().clone()
    n_acc, committed = eng.accept_rollback()
    win = eng.tree_winner()
    lt, _ = eng.lengths()
    kv_after = eng.kv_view().clone()
    eng.close()
    worst = 0.0
    for b, ((ns, _), (P, gr)) in enumerate(zip(cases, prompts_gr)):
        guesses = od.ngram_candidates(P, n_cand, g, 2, 4)
        assert [prop[b, c, :len(x)].tolist() for c, x in enumerate(guesses)] == guesses
        refs = _oracle_rows(m, P, guesses)
        for c, ref in enumerate(refs):
            rows = [0] + [c * g + i for i in range(1, len(guesses[c]) + 1)]
            worst = max([worst] + [logit_err(t_log[b, r], ref[i]) for i, r in enumerate(rows)])
        # acceptance: the oracle's rule on the GPU's own choices, and the planted lengths
        ta = t_arg[b].tolist()
        choices = [[ta[0]] + [ta[c * g + i] for i in range(1, g + 1)] for c in range(len(guesses))]
        c_ref, n_ref, com_ref = od.tree_accept(guesses, choices)
        assert (int(win[b]), int(n_acc[b]), committed[b]) == (c_ref, n_ref, com_ref)
        assert n_ref == max(ns) and c_ref == ns.index(max(ns))
        assert committed[b] == gr[:n_ref + 1]
        C = len(P)
        assert int(lt[b]) == C + n_ref
        # cache: slots below C untouched, accepted entries moved down bit for bit
        assert torch.equal(kv_after[:, :, b, :, :C], kv_before[:, :, b, :, :C])
        for i in range(n_ref):
            assert torch.equal(kv_after[:, :, b, :, C + i], kv_before[:, :, b, :, C + c_ref * g + i])
    return worst


@pytest.mark.parametrize("idx", range(len(PLANTED)))
def test_tree_round_planted_batch1(pkg, tiny, planted, idx):
    tw, gt, m = tiny
    worst = _round(pkg, gt, m, [PLANTED[idx]], [planted[idx]], K=8)
    print(f"planted {PLANTED[idx][0]}: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16


def test_tree_round_planted_batch4(pkg, tiny, planted):
    """Four sequences (36 verify rows: the tensor-core GEMM path), ragged
    prompts, different winners per sequence."""
    tw, gt, m = tiny
    sel = [0, 1, 3, 5]
    worst = _round(pkg, gt, m, [PLANTED[i] for i in sel], [planted[i] for i in sel], K=8)
    print(f"planted batch 4: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16


def test_tree_verify_7b_shape_chunk_boundary(pkg):
    """Two layers of the 7B shape, a 2046-token prompt whose last 4 tokens
    occurred twice before with different continuations: the pending token
    sits in slot 2045 (= 31 * 64 + 61), candidate 0's guesses in slots
    2046..2049 across the 64-slot boundary, candidate 1's in 2050..2053."""
    K, n_cand = 8, 2
    g = K // n_cand
    shape = QWEN7B.with_(layers=2)
    tw = make_weights(shape, seed=0, device="cuda")
    base = uniform_prompt(2046, shape.vocab, seed=105).tolist()
    s = base[-4:]
    base[1000:1004] = s
    base[1500:1504] = s
    prompt = base
    guesses = od.ngram_candidates(prompt, n_cand, g, 2, 4)
    assert len(guesses) == 2 and guesses[0] == prompt[1504:1508] and guesses[1] == prompt[1004:1008]
    eng = pkg.SpecEngine(shape, tw, batch=1, K=K, s_max=4096)
    eng.kv_t.fill_(0xFF)
    eng.prefill([prompt])
    t_log = torch.zeros(K + 1, shape.vocab, dtype=torch.float32, device="cuda")
    eng.tree_draft(n_cand, 2, 4)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    eng.accept_rollback()
    eng.close()
    tw_c = to_cpu(tw)
    del tw
    torch.cuda.empty_cache()
    m = om.Model(shape, tw_c, rowwise=False)
    refs = _oracle_rows(m, prompt, guesses)
    worst = 0.0
    for c, ref in enumerate(refs):
        rows = [0] + [c * g + i for i in range(1, g + 1)]
        worst = max([worst] + [logit_err(t_log[r], ref[i]) for i, r in enumerate(rows)])
    print(f"7B shape, tree verify at slot 2045: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16


@pytest.mark.parametrize("n_cand", [2, 4])
def test_tree_generate_is_greedy(pkg, tiny, n_cand):
    tw, gt, m = tiny
    K, n_new = 8, 48
    prompts = [ngram_prompt(160, 0.8, V, seed=20 + b, base_len=64)[0].tolist() for b in range(2)]
    eng = pkg.SpecEngine(TINY_TARGET, gt, batch=2, K=K, s_max=512)
    eng.prefill(prompts)
    eng.set_drafter(pkg.SF_DRAFT_TREE, 2, 4)
    eng.set_tree_candidates(n_cand)
    out, rounds = eng.generate(n_new)
    hist = eng.accept_hist()
    eng.close()
    for b in range(2):
        n, flips, near = stream_report(m, prompts[b], out[b].tolist())
        ref = od.spec_decode(m, None, prompts[b], K, n_new, drafter="tree", n_cand=n_cand)
        ref_hist = np.bincount([r[0] for r in ref["rounds"]], minlength=K + 1)
        print(f"tree n_cand={n_cand} seq {b}: {rounds} rounds, accept histogram {hist[b].tolist()} "
              f"(oracle {ref_hist.tolist()}), {flips} flips, {near} near ties")
        if flips == 0:
            assert out[b].tolist() == ref["tokens"]


def test_tree_one_candidate_is_single_lookup(pkg, tiny):
    """n_cand = 1 (one guess of K tokens, no gap in any row's mask): the same
    rounds, tokens and cache as SF_DRAFT_NGRAM with max_guess K."""
    tw, gt, m = tiny
    K, n_new = 6, 40
    prompts = [ngram_prompt(200, 0.8, V, seed=30 + b, base_len=64)[0].tolist() for b in range(3)]
    res = []
    for mode in ("ngram", "tree"):
        eng = pkg.SpecEngine(TINY_TARGET, gt, batch=3, K=K, s_max=512)
        eng.prefill(prompts)
        if mode == "tree":
            eng.set_drafter(pkg.SF_DRAFT_TREE, 2, 4)
            eng.set_tree_candidates(1)
        else:
            eng.set_drafter(pkg.SF_DRAFT_NGRAM, 2, 4)
        out, rounds = eng.generate(n_new)
        res.append((out.copy(), rounds, eng.accept_hist().copy(), eng.lengths()[0].copy()))
        eng.close()
    (o1, r1, h1, l1), (o2, r2, h2, l2) = res
    assert r1 == r2 and np.array_equal(o1, o2) and np.array_equal(h1, h2) and np.array_equal(l1, l2)


def test_tree_step_graph_equals_manual_round(pkg, tiny, planted):
    """sf_step with SF_DRAFT_TREE (one graph replay, programmatic dependent
    launches) commits what the manual tree_draft / verify / accept sequence
    commits."""
    tw, gt, m = tiny
    P, gr = planted[0]
    got = []
    for manual in (True, False):
        eng = pkg.SpecEngine(TINY_TARGET, gt, batch=1, K=8, s_max=256)
        eng.prefill([P])
        if manual:
            eng.tree_draft(2, 2, 4)
            eng.verify()
            _, com = eng.accept_rollback()
        else:
            eng.set_drafter(pkg.SF_DRAFT_TREE, 2, 4)
            eng.set_tree_candidates(2)
            com = eng.step()
        got.append((com[0], int(eng.tree_winner()[0]), eng.kv_view().clone()))
        eng.close()
    assert got[0][0] == got[1][0] == gr[:len(got[0][0])]
    assert got[0][1] == got[1][1]
    C = len(P) + len(got[0][0]) - 1
    assert torch.equal(got[0][2][:, :, :, :, :C], got[1][2][:, :, :, :, :C])


def test_tree_argument_errors(pkg, tiny):
    tw, gt, m = tiny
    eng = pkg.SpecEngine(TINY_TARGET, gt, batch=1, K=4, s_max=256)
    with pytest.raises(pkg.SFError):
        eng.tree_draft(2)            # no prompt yet
    eng.prefill([[1, 2, 3, 1, 2]])
    for bad in (0, 5):
        with pytest.raises(pkg.SFError):
            eng.tree_draft(bad)
        with pytest.raises(pkg.SFError):
            eng.set_tree_candidates(bad)
    with pytest.raises(pkg.SFError):
        eng.tree_draft(2, 3, 2)      # min_n > max_n
    eng.close()
