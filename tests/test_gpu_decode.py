"""The persistent decode kernel (SF_PERSISTENT=1: forwards of at most four
token rows, two per sequence: the draft's decode steps, a K = 1 verify)
against the oracle and against itself.

* Draft logits of single sequences and of a ragged batch of two, compared
  row by row with the oracle (3e-2 of each row's range), and the batch's
  rows equal to the same sequences run alone bit for bit (the kernel's
  arithmetic does not depend on the other rows of the launch).
* Target as its own draft with K = 1: the draft's two-row step and the
  two-row verify both run on the persistent kernel, so they agree bit for
  bit and every guess is accepted.
* Long contexts: a two-layer 0.5B-shape draft with a ragged batch at 2000 and
  700 tokens (up to 32 attention partials merged per row and head), and a
  two-layer 7B-shape target decoding on its own (head dim 128, seven query
  heads per KV head) at 2047 tokens.
* Against the per-projection kernels (SF_PERSISTENT=0): the same draft logits
  within rounding.
* Token streams of whole generations equal the oracle's greedy stream
  (near ties allowed).
* The error path: SF_TEST_WAIT_EXPIRE=1 makes the first grid barrier report
  an expired wait (it then waits normally); the host sees SF_ERR_DEVICE.
"""

import pytest
import torch

from oracle import decode as od
from oracle import model as om
from synth import (QWEN05B, QWEN05B_SHARED, QWEN7B, TINY_DRAFT, TINY_TARGET, draft_from_target_layer0,
                   make_weights, shared_embedding_draft, uniform_prompt)

from gpu_helpers import LOGIT_TOL_BF16, logit_err, stream_report, to_cpu, to_cuda

pytestmark = pytest.mark.gpu
V = TINY_TARGET.vocab


@pytest.fixture(autouse=True)
def persistent_on(monkeypatch):
    """Every engine of this module runs its small forwards on the persistent
    kernel (SF_PERSISTENT=1; the default is the per-projection kernels)."""
    monkeypatch.setenv("SF_PERSISTENT", "1")


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as p
    return p


@pytest.fixture(scope="module")
def tiny():
    tw = make_weights(TINY_TARGET, seed=0)
    dw = draft_from_target_layer0(tw, TINY_DRAFT, 0.005, seed=1)
    gt, gd = to_cuda(tw), to_cuda(dw)
    gd["embed"], gd["norm"] = gt["embed"], gt["norm"]
    return tw, dw, gt, gd


def _draft_logits(pkg, t_shape, gt, d_shape, gd, prompts, K, s_max=256):
    B = len(prompts)
    eng = pkg.SpecEngine(t_shape, gt, d_shape, gd, batch=B, K=K, s_max=s_max)
    eng.kv_d.fill_(0xFF)
    eng.prefill(prompts)
    d_out = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(B, K, d_shape.vocab, dtype=torch.float32, device="cuda")
    eng.draft(d_out, d_log)
    torch.cuda.synchronize()
    eng.close()
    return d_out.cpu(), d_log


def _oracle_draft_err(dm, prompt, d, d_log):
    c = dm.new_cache()
    dm.forward(prompt[:-1], c, logit_rows=[])
    feed, worst = [prompt[-1]], 0.0
    for i in range(len(d)):
        worst = max(worst, logit_err(d_log[i], dm.forward(feed, c)[0]))
        feed = [int(d[i])]
    return worst


def test_draft_steps_match_oracle_and_single_sequences(pkg, tiny):
    tw, dw, gt, gd = tiny
    K = 4
    prompts = [uniform_prompt(n, V, seed=500 + n).tolist() for n in (37, 90)]
    d2, l2 = _draft_logits(pkg, TINY_TARGET, gt, TINY_DRAFT, gd, prompts, K)
    dm = om.Model(TINY_DRAFT, dw)
    worst = 0.0
    for b, p in enumerate(prompts):
        d1, l1 = _draft_logits(pkg, TINY_TARGET, gt, TINY_DRAFT, gd, [p], K)
        assert torch.equal(l2[b], l1[0]), b
        assert torch.equal(d2[b], d1[0]), b
        worst = max(worst, _oracle_draft_err(dm, p, d2[b].tolist(), l2[b]))
    print(f"persistent draft steps, batch 2: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16


def test_target_as_own_draft_k1(pkg, tiny):
    """K = 1: the prefill, the draft's step (two rows per sequence) and the
    verify (two rows per sequence) all run on the persistent kernel:
    bit-for-bit agreement, every guess accepted, over several rounds and two
    sequences."""
    tw, dw, gt, gd = tiny
    eng = pkg.SpecEngine(TINY_TARGET, gt, TINY_TARGET, gt, batch=2, K=1, s_max=256)
    # Three-token prompts: the prefill (two rows per sequence) runs on the
    # persistent kernel too, so both caches hold the same bits.
    eng.prefill([uniform_prompt(3, V, seed=7).tolist(), uniform_prompt(3, V, seed=8).tolist()])
    d_log = torch.zeros(2, 1, V, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(2, 2, V, dtype=torch.float32, device="cuda")
    for _ in range(6):
        eng.draft(None, d_log)
        eng.verify(None, t_log)
        torch.cuda.synchronize()
        assert torch.equal(d_log[:, 0], t_log[:, 0])
        n_acc, committed = eng.accept_rollback()
        assert [int(n) for n in n_acc] == [1, 1]
    eng.close()


def test_long_context_ragged_batch_05b_shape(pkg):
    K = 4
    t_shape = QWEN7B.with_(layers=1)
    d_shape = QWEN05B_SHARED.with_(layers=2)
    tw = make_weights(t_shape, seed=0, device="cuda")
    dw = shared_embedding_draft(make_weights(QWEN05B.with_(layers=2), seed=2, device="cuda"), tw["embed"],
                                d_shape.hidden)
    prompts = [uniform_prompt(n, t_shape.vocab, seed=600 + n).tolist() for n in (2000, 700)]
    d, l = _draft_logits(pkg, t_shape, tw, d_shape, dw, prompts, K, s_max=4096)
    dw_c = to_cpu(dw)
    del tw, dw
    torch.cuda.empty_cache()
    dm = om.Model(d_shape, dw_c, rowwise=False)
    worst = max(_oracle_draft_err(dm, p, d[b].tolist(), l[b]) for b, p in enumerate(prompts))
    print(f"persistent draft, 0.5B shape (2 layers), contexts 2000 / 700: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16


def test_long_context_7b_shape_two_row_verify(pkg):
    """Plain greedy rounds of a two-layer 7B-shape target (K = 1: two verify
    rows, the pending token and an unused guess slot) at 2047 tokens."""
    shape = QWEN7B.with_(layers=2)
    tw = make_weights(shape, seed=0, device="cuda")
    prompt = uniform_prompt(2047, shape.vocab, seed=106).tolist()
    eng = pkg.SpecEngine(shape, tw, batch=1, K=1, s_max=4096)
    eng.kv_t.fill_(0xFF)
    eng.prefill([prompt])
    eng.set_drafter(pkg.SF_DRAFT_NONE)
    t_log = torch.zeros(2, shape.vocab, dtype=torch.float32, device="cuda")
    eng.ngram_draft(1, 1, 1)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    eng.accept_rollback()
    eng.close()
    tw_c = to_cpu(tw)
    del tw
    torch.cuda.empty_cache()
    m = om.Model(shape, tw_c, rowwise=False)
    c = m.new_cache()
    m.forward(prompt[:-1], c, logit_rows=[])
    ref = m.forward([prompt[-1]], c)
    err = logit_err(t_log[0], ref[0])
    print(f"persistent 2-row verify, 7B shape (2 layers), context 2047: logit error / range = {err:.3e}")
    assert err < LOGIT_TOL_BF16


def test_matches_per_projection_kernels(pkg, tiny, monkeypatch):
    tw, dw, gt, gd = tiny
    prompts = [uniform_prompt(64, V, seed=9).tolist()]
    _, on = _draft_logits(pkg, TINY_TARGET, gt, TINY_DRAFT, gd, prompts, 4)
    monkeypatch.setenv("SF_PERSISTENT", "0")
    _, off = _draft_logits(pkg, TINY_TARGET, gt, TINY_DRAFT, gd, prompts, 4)
    rng = (off.max(dim=-1).values - off.min(dim=-1).values)[..., None]
    diff = float(((on - off).abs() / rng).max())
    print(f"persistent vs per-projection draft logits: max difference / range = {diff:.3e}")
    assert diff < 1.5e-2


@pytest.mark.parametrize("K", [1, 4])
def test_generate_is_greedy(pkg, tiny, K):
    tw, dw, gt, gd = tiny
    prompt = uniform_prompt(32, V, seed=100).tolist()
    eng = pkg.SpecEngine(TINY_TARGET, gt, TINY_DRAFT, gd, batch=1, K=K, s_max=256)
    eng.prefill([prompt])
    out, rounds = eng.generate(48)
    eng.close()
    m = om.Model(TINY_TARGET, tw)
    n, flips, near = stream_report(m, prompt, out[0].tolist())
    print(f"K={K}: 48 tokens in {rounds} rounds, {flips} flips, {near} near ties")
    if flips == 0:
        assert out[0].tolist() == od.greedy(m, prompt, 48)


def test_expired_barrier_is_reported(pkg, tiny, monkeypatch):
    tw, dw, gt, gd = tiny
    from greedy_speculative_decoding_gb300 import SFError
    from greedy_speculative_decoding_gb300._lib import SF_ERR_DEVICE
    prompt = uniform_prompt(20, V, seed=3).tolist()
    monkeypatch.setenv("SF_TEST_WAIT_EXPIRE", "1")
    eng = pkg.SpecEngine(TINY_TARGET, gt, TINY_DRAFT, gd, batch=1, K=1, s_max=256)
    monkeypatch.delenv("SF_TEST_WAIT_EXPIRE")
    eng.prefill([prompt])
    with pytest.raises(SFError) as e:
        eng.step()
    assert e.value.status == SF_ERR_DEVICE
    eng.close()
    eng = pkg.SpecEngine(TINY_TARGET, gt, TINY_DRAFT, gd, batch=1, K=1, s_max=256)
    eng.prefill([prompt])
    assert len(eng.step()[0]) >= 1
    eng.close()
