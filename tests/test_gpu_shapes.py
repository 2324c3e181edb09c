"""GPU parity at the full workload shapes, in the launch configuration the
benchmark uses (K = 8, batch 1, 4096 cache slots), at a short context so the
float64 oracle finishes in about a minute: Qwen2.5-0.5B shape as its own
draft, and the 7B-shape target with the 0.5B-shape shared-embedding draft.
Logit rows of the draft steps and of the verify pass are compared with the
oracle (3e-2 of each row's range); the caches start filled with NaN bytes."""

import pytest
import torch

from oracle import model as om
from synth import QWEN05B, QWEN05B_SHARED, QWEN7B, make_weights, shared_embedding_draft, uniform_prompt

from gpu_helpers import LOGIT_TOL_BF16, accept_brute, logit_err, to_cpu

pytestmark = pytest.mark.gpu
K = 8


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as p
    return p


def _round(eng, vocab):
    d_out = torch.zeros(K, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(K, vocab, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(K + 1, vocab, dtype=torch.float32, device="cuda")
    eng.draft(d_out, d_log)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    return d_out.cpu().tolist(), d_log, t_log


@pytest.mark.parametrize("persistent", [False, True])
def test_05b_shape_self_draft(pkg, monkeypatch, persistent):
    """Without the persistent decode kernel every forward of this engine runs
    on the mma.sync GEMM, so the draft rows equal the verify rows bit for bit
    and every guess is accepted; with it the draft steps run on their own
    arithmetic, equal to the verify rows within rounding, and the accepted
    length is the brute-force prefix compare of the two."""
    monkeypatch.setenv("SF_PERSISTENT", "1" if persistent else "0")
    w = make_weights(QWEN05B, seed=0, device="cuda")
    eng = pkg.SpecEngine(QWEN05B, w, QWEN05B, w, batch=1, K=K, s_max=4096)
    eng.kv_t.fill_(0xFF)
    eng.kv_d.fill_(0xFF)
    prompt = uniform_prompt(16, QWEN05B.vocab, seed=101).tolist()
    eng.prefill([prompt])
    d, d_log, t_log = _round(eng, QWEN05B.vocab)
    n_acc, _ = eng.accept_rollback()
    if not persistent:
        assert torch.equal(d_log, t_log[:K])
        assert int(n_acc[0]) == K
    else:
        rng = (t_log.max(dim=-1).values - t_log.min(dim=-1).values)[:K, None]
        assert bool(((d_log - t_log[:K]).abs() <= 1.5e-2 * rng).all())
        t_arg = t_log.argmax(dim=-1).cpu().tolist()
        assert int(n_acc[0]) == accept_brute(d, t_arg, K)
    m = om.Model(QWEN05B, to_cpu(w), rowwise=False)
    c = m.new_cache()
    m.forward(prompt[:-1], c, logit_rows=[])
    ref = m.forward([prompt[-1]] + d, c)
    worst = max(logit_err(t_log[j], ref[j]) for j in range(K + 1))
    print(f"0.5B shape: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16
    eng.close()


def test_7b_target_with_shared_embedding_draft(pkg):
    tw = make_weights(QWEN7B, seed=0, device="cuda")
    dw = shared_embedding_draft(make_weights(QWEN05B, seed=2, device="cuda"), tw["embed"], QWEN05B_SHARED.hidden)
    eng = pkg.SpecEngine(QWEN7B, tw, QWEN05B_SHARED, dw, batch=1, K=K, s_max=4096)
    eng.kv_t.fill_(0xFF)
    eng.kv_d.fill_(0xFF)
    prompt = uniform_prompt(12, QWEN7B.vocab, seed=102).tolist()
    eng.prefill([prompt])
    d, d_log, t_log = _round(eng, QWEN7B.vocab)
    eng.accept_rollback()
    eng.close()
    tw_c = to_cpu(tw)
    dw_c = to_cpu(dw)
    del tw, dw
    torch.cuda.empty_cache()
    dm = om.Model(QWEN05B_SHARED, dw_c, rowwise=False)
    dc = dm.new_cache()
    dm.forward(prompt[:-1], dc, logit_rows=[])
    feed, worst_d = [prompt[-1]], 0.0
    for i in range(K):
        ref = dm.forward(feed, dc)[0]
        worst_d = max(worst_d, logit_err(d_log[i], ref))
        feed = [d[i]]
    tm = om.Model(QWEN7B, tw_c, rowwise=False)
    tc = tm.new_cache()
    tm.forward(prompt[:-1], tc, logit_rows=[])
    ref = tm.forward([prompt[-1]] + d, tc)
    worst_t = max(logit_err(t_log[j], ref[j]) for j in range(K + 1))
    print(f"0.5B shared draft: {worst_d:.3e}; 7B verify: {worst_t:.3e} (max logit error / range)")
    assert worst_d < LOGIT_TOL_BF16 and worst_t < LOGIT_TOL_BF16
