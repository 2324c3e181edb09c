"""GPU parity on the tiny workload (2-layer target, 1-layer draft, vocab 1024).

Every check runs the CUDA path through the C ABI and compares it with the
CPU oracle on the same seeded inputs:
  * logits of the draft steps and of the verify rows within 3e-2 of each
    row's logit range (bf16 weights), with the actual error reported;
  * token streams equal to the oracle's greedy stream (near ties allowed);
  * accept lengths, committed tokens, cache lengths, n-gram proposals:
    bit-exact integer work;
  * the cache after in-place rollback equals a fresh prefill of the
    committed prefix (bit for bit);
  * batch invariance: a row's logits do not depend on how many rows share
    the launch (draft decode rows == verify rows, bit for bit).
"""

import numpy as np
import pytest
import torch

from oracle import decode as od
from oracle import model as om
from synth import (TINY_DRAFT, TINY_TARGET, draft_from_target_layer0, make_weights, ngram_prompt,
                   uniform_prompt)

from gpu_helpers import (LOGIT_TOL_BF16, accept_brute, check_token_against_oracle, logit_err,
                          teacher_forced_stream_check, to_cuda)

pytestmark = pytest.mark.gpu


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
    gt = to_cuda(tw)
    gd = to_cuda(dw)
    gd["embed"], gd["norm"] = gt["embed"], gt["norm"]
    return tw, dw, gt, gd


def make_engine(pkg, tiny, K=4, s_max=256, draft=True, batch=1):
    tw, dw, gt, gd = tiny
    if draft:
        return pkg.SpecEngine(TINY_TARGET, gt, TINY_DRAFT, gd, batch=batch, K=K, s_max=s_max)
    return pkg.SpecEngine(TINY_TARGET, gt, batch=batch, K=K, s_max=s_max)


def test_draft_and_verify_logits_match_oracle(pkg, tiny):
    tw, dw, _, _ = tiny
    K = 4
    V = TINY_TARGET.vocab
    prompt = uniform_prompt(32, 1024, seed=100).tolist()
    eng = make_engine(pkg, tiny, K=K)
    eng.prefill([prompt])
    d_out = torch.zeros(K, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(K, V, dtype=torch.float32, device="cuda")
    eng.draft(d_out, d_log)
    t_out = torch.zeros(K + 1, dtype=torch.int32, device="cuda")
    t_log = torch.zeros(K + 1, V, dtype=torch.float32, device="cuda")
    eng.verify(t_out, t_log)
    torch.cuda.synchronize()
    d = d_out.cpu().tolist()
    # draft oracle, teacher-forced on the GPU's guesses
    dm = om.Model(TINY_DRAFT, dw)
    dc = dm.new_cache()
    dm.forward(prompt[:-1], dc, logit_rows=[])
    feed = [prompt[-1]]
    worst = 0.0
    for i in range(K):
        ref = dm.forward(feed, dc)[0]
        worst = max(worst, logit_err(d_log[i], ref))
        check_token_against_oracle(d[i], ref)
        feed = [d[i]]
    # target oracle on [pending, d_1..d_K]
    tm = om.Model(TINY_TARGET, tw)
    tc = tm.new_cache()
    tm.forward(prompt[:-1], tc, logit_rows=[])
    ref = tm.forward([prompt[-1]] + d, tc)
    for j in range(K + 1):
        worst = max(worst, logit_err(t_log[j], ref[j]))
    print(f"tiny: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16
    # the argmax kernel picks the first maximum of the logits it produced
    assert t_out.cpu().tolist() == [int(torch.argmax(t_log[j])) for j in range(K + 1)]
    assert d == [int(torch.argmax(d_log[i])) for i in range(K)]
    n_acc, committed = eng.accept_rollback()
    t = t_out.cpu().tolist()
    n = accept_brute(d, t, K)
    assert int(n_acc[0]) == n and committed[0] == d[:n] + [t[n]]
    eng.close()


def test_batch_invariance_target_as_its_own_draft(pkg, tiny, monkeypatch):
    """Draft = the target itself: decode rows (1-2 per launch) and verify rows
    (K+1 per launch) must agree bit for bit, so every guess is accepted. (The
    16-token prompt is prefilled in one 15-row forward, on the same mma.sync
    GEMM as the rounds, so both caches hold the same bits.)"""
    monkeypatch.setenv("SF_PERSISTENT", "0")   # the per-projection kernels' invariant (the persistent decode kernel has its own arithmetic)
    _, _, gt, _ = tiny
    K = 4
    V = TINY_TARGET.vocab
    eng = pkg.SpecEngine(TINY_TARGET, gt, TINY_TARGET, gt, batch=1, K=K, s_max=256)
    eng.prefill([uniform_prompt(16, 1024, seed=5).tolist()])
    d_log = torch.zeros(K, V, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(K + 1, V, dtype=torch.float32, device="cuda")
    for _ in range(5):
        eng.draft(None, d_log)
        eng.verify(None, t_log)
        torch.cuda.synchronize()
        assert torch.equal(d_log, t_log[:K])
        n_acc, committed = eng.accept_rollback()
        assert int(n_acc[0]) == K and len(committed[0]) == K + 1
    eng.close()


def test_batch8_ragged_rows_match_single_sequences(pkg, tiny, monkeypatch):
    """Eight sequences whose prompts differ in length, K=8: every verify
    forward has 72 token rows (the tcgen05 GEMM) and the first draft step 16
    (the mma.sync GEMM). Per sequence, the draft logits equal those of the
    same sequence run alone bit for bit (a row's arithmetic does not depend
    on the other rows or sequences of a <= 16-row launch), the verify logits
    agree with the single sequence's 9-row verify within the bf16 rounding
    of the tensor-core path's activations (1.5e-2 of the row's range); accept
    lengths, committed tokens and cache lengths agree with the batch's own
    guesses and target choices (a brute-force prefix compare); the generated
    streams are the oracle's greedy streams (near ties allowed)."""
    monkeypatch.setenv("SF_PERSISTENT", "0")   # the per-projection kernels' invariant (the persistent decode kernel has its own arithmetic)
    tw = tiny[0]
    K, B, V = 8, 8, TINY_TARGET.vocab
    lens = [20, 33, 47, 12, 60, 25, 8, 41]
    prompts = [uniform_prompt(n, V, seed=300 + i).tolist() for i, n in enumerate(lens)]
    eng = make_engine(pkg, tiny, K=K, batch=B)
    eng.prefill(prompts)
    d_log = torch.zeros(B, K, V, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(B, K + 1, V, dtype=torch.float32, device="cuda")
    eng.draft(None, d_log)
    eng.verify(None, t_log)
    n_acc, committed = eng.accept_rollback()
    lt, ld = eng.lengths()
    torch.cuda.synchronize()
    for b in range(B):
        one = make_engine(pkg, tiny, K=K, batch=1)
        one.prefill([prompts[b]])
        d1 = torch.zeros(1, K, V, dtype=torch.float32, device="cuda")
        t1 = torch.zeros(1, K + 1, V, dtype=torch.float32, device="cuda")
        one.draft(None, d1)
        one.verify(None, t1)
        n1, c1 = one.accept_rollback()
        lt1, ld1 = one.lengths()
        torch.cuda.synchronize()
        one.close()
        assert torch.equal(d_log[b], d1[0]), b
        rng = (t1[0].max(dim=-1).values - t1[0].min(dim=-1).values)[:, None]
        assert bool(((t_log[b] - t1[0]).abs() <= 1.5e-2 * rng).all()), b
        d_b = [int(v) for v in d_log[b].argmax(dim=-1).cpu()]
        t_b = [int(v) for v in t_log[b].argmax(dim=-1).cpu()]
        n = accept_brute(d_b, t_b, K)
        assert int(n_acc[b]) == n and list(committed[b]) == d_b[:n] + [t_b[n]], b
        assert int(lt[b]) == lens[b] + n and int(ld[b]) == lens[b] + n - 1, b
    out, rounds = eng.generate(24)
    eng.close()
    model = om.Model(TINY_TARGET, tw)
    for b in range(B):
        stream = out[b].tolist()
        if stream != od.greedy(model, prompts[b], 24):
            near = teacher_forced_stream_check(model, prompts[b], stream)
            print(f"sequence {b}: {near} near-tie positions")


@pytest.mark.parametrize("K", [1, 4, 7])
def test_generate_matches_oracle_greedy(pkg, tiny, K):
    tw = tiny[0]
    prompt = uniform_prompt(32, 1024, seed=100).tolist()
    eng = make_engine(pkg, tiny, K=K)
    eng.prefill([prompt])
    out, rounds = eng.generate(64)
    hist = eng.accept_hist()
    eng.close()
    stream = out[0].tolist()
    ref = od.greedy(om.Model(TINY_TARGET, tw), prompt, 64)
    if stream != ref:
        near = teacher_forced_stream_check(om.Model(TINY_TARGET, tw), prompt, stream)
        print(f"K={K}: {near} near-tie positions")
    assert rounds >= 64 // (K + 1)
    assert int((hist[0] * (np.arange(K + 1) + 1)).sum()) >= 64


def test_spec_streams_identical_across_drafters(pkg, tiny, monkeypatch):
    """Speculation never changes the output: neural K=1, K=4, K=7 and n-gram
    drafting all give the same tokens bit for bit on the GPU."""
    monkeypatch.setenv("SF_PERSISTENT", "0")   # the per-projection kernels' invariant (the persistent decode kernel has its own arithmetic)
    prompt = uniform_prompt(32, 1024, seed=101).tolist()
    streams = []
    for K in (1, 4, 7):
        eng = make_engine(pkg, tiny, K=K)
        eng.prefill([prompt])
        streams.append(eng.generate(48)[0][0].tolist())
        eng.close()
    eng = make_engine(pkg, tiny, K=4, draft=False)
    eng.prefill([prompt])
    streams.append(eng.generate(48)[0][0].tolist())
    eng.close()
    assert all(s == streams[0] for s in streams)


def test_rounds_integer_state_and_rollback(pkg, tiny):
    K = 4
    prompt = uniform_prompt(24, 1024, seed=102).tolist()
    eng = make_engine(pkg, tiny, K=K)
    eng.prefill([prompt])
    seq = list(prompt)
    d_out = torch.zeros(K, dtype=torch.int32, device="cuda")
    t_out = torch.zeros(K + 1, dtype=torch.int32, device="cuda")
    for _ in range(8):
        eng.draft(d_out)
        eng.verify(t_out)
        n_acc, committed = eng.accept_rollback()
        d, t = d_out.cpu().tolist(), t_out.cpu().tolist()
        n = accept_brute(d, t, K)
        assert int(n_acc[0]) == n
        assert committed[0] == d[:n] + [t[n]]
        seq += committed[0]
        lt, ld = eng.lengths()
        assert int(lt[0]) == len(seq) - 1 and int(ld[0]) == len(seq) - 2
    # The caches below the lengths equal a fresh prefill of the committed
    # prefix: bit for bit where both wrote the entries through the same GEMM
    # kernel, else to one bf16 rounding step (the fresh prefill's chunks of
    # more than 16 rows run on the tcgen05 GEMM, the rounds on mma.sync).
    kv_t = eng.kv_view("target").clone()
    kv_d = eng.kv_view("draft").clone()
    C = len(seq)
    fresh = make_engine(pkg, tiny, K=K)
    fresh.prefill([seq])
    ft, fd = fresh.kv_view("target"), fresh.kv_view("draft")

    def close(a, b):
        # The fresh prefill's QKV projection takes its activations as bf16
        # (tensor-core path): a key or value moves by up to 2^-9 of
        # sum_k |W_nk x_k|, about 1e-2 of the cache's largest entry here.
        a, b = a.float(), b.float()
        return bool(((a - b).abs() <= 2.0 ** -6 * b.abs() + 1e-2 * b.abs().max()).all())
    P = len(prompt)
    assert torch.equal(kv_t[..., : P - 1, :], ft[..., : P - 1, :])
    assert close(kv_t[..., : C - 1, :], ft[..., : C - 1, :])
    assert close(kv_d[..., : C - 2, :], fd[..., : C - 2, :])
    fresh.close()
    eng.close()


def test_rollback_bit_exact_short(pkg, tiny, monkeypatch):
    """Two rounds from a 6-token prompt keep every forward (prefill, draft
    steps, verify, and the fresh prefill of the committed prefix) at 16 rows
    or fewer, so all run on the same GEMM kernel: after the in-place
    rollback both caches below their lengths equal a fresh prefill of the
    committed prefix bit for bit."""
    monkeypatch.setenv("SF_PERSISTENT", "0")   # the per-projection kernels' invariant (the persistent decode kernel has its own arithmetic)
    K = 4
    prompt = uniform_prompt(6, 1024, seed=104).tolist()
    eng = make_engine(pkg, tiny, K=K)
    eng.prefill([prompt])
    seq = list(prompt)
    for _ in range(2):
        eng.draft()
        eng.verify()
        _, committed = eng.accept_rollback()
        seq += committed[0]
    C = len(seq)
    assert C - 1 <= 16
    lt, ld = eng.lengths()
    assert int(lt[0]) == C - 1 and int(ld[0]) == C - 2
    kv_t = eng.kv_view("target").clone()
    kv_d = eng.kv_view("draft").clone()
    fresh = make_engine(pkg, tiny, K=K)
    fresh.prefill([seq])
    assert torch.equal(kv_t[..., : C - 1, :], fresh.kv_view("target")[..., : C - 1, :])
    assert torch.equal(kv_d[..., : C - 2, :], fresh.kv_view("draft")[..., : C - 2, :])
    fresh.close()
    eng.close()


def test_ngram_drafting_matches_oracle(pkg, tiny):
    tw = tiny[0]
    K = 4
    prompt, _ = ngram_prompt(96, 0.8, 1024, seed=200, base_len=48, seg_lo=8, seg_hi=16)
    prompt = prompt.tolist()
    eng = make_engine(pkg, tiny, K=K, draft=False)
    eng.prefill([prompt])
    seq = list(prompt)
    prop = torch.zeros(K, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    t_out = torch.zeros(K + 1, dtype=torch.int32, device="cuda")
    proposed = 0
    for _ in range(12):
        eng.ngram_draft(K, 2, 4, prop, cnt)
        eng.verify(t_out)
        torch.cuda.synchronize()
        ref = od.ngram_propose(seq, K, 2, 4)
        c = int(cnt.item())
        assert c == len(ref) and prop.cpu().tolist()[:c] == ref
        assert all(v == 0 for v in prop.cpu().tolist()[c:])
        proposed += c
        n_acc, committed = eng.accept_rollback()
        t = t_out.cpu().tolist()
        n = accept_brute(ref + [0] * (K - c), t, c)
        assert int(n_acc[0]) == n and committed[0] == ref[:n] + [t[n]]
        seq += committed[0]
    assert proposed > 0
    # and the generated stream is greedy
    teacher_forced_stream_check(om.Model(TINY_TARGET, tw), prompt, seq[len(prompt):])
    eng.close()


@pytest.mark.parametrize("ctx", [[5, 9], [1, 2, 3, 1, 2], [7] * 9])
def test_ngram_edge_cases(pkg, tiny, ctx):
    K = 4
    eng = make_engine(pkg, tiny, K=K, draft=False)
    eng.prefill([ctx])
    prop = torch.zeros(K, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    for mg in (1, 4):
        eng.ngram_draft(mg, 2, 4, prop, cnt)
        ref = od.ngram_propose(ctx, mg, 2, 4)
        assert int(cnt.item()) == len(ref) and prop.cpu().tolist()[:len(ref)] == ref
        eng.verify()
        eng.accept_rollback()
        eng.reset()
    eng.close()


def test_long_context_attention(pkg, tiny):
    """Prompt of 1500 tokens: attention spans 24 cache chunks of 64 slots."""
    tw = tiny[0]
    K = 4
    prompt = uniform_prompt(1500, 1024, seed=103).tolist()
    eng = make_engine(pkg, tiny, K=K, s_max=2048)
    eng.prefill([prompt])
    d_out = torch.zeros(K, dtype=torch.int32, device="cuda")
    t_log = torch.zeros(K + 1, TINY_TARGET.vocab, dtype=torch.float32, device="cuda")
    eng.draft(d_out)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    d = d_out.cpu().tolist()
    tm = om.Model(TINY_TARGET, tw)
    tc = tm.new_cache()
    tm.forward(prompt[:-1], tc, logit_rows=[])
    ref = tm.forward([prompt[-1]] + d, tc)
    worst = max(logit_err(t_log[j], ref[j]) for j in range(K + 1))
    print(f"tiny ctx 1500: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16
    eng.close()


def test_state_and_capacity_errors(pkg, tiny):
    from greedy_speculative_decoding_gb300 import SFError
    from greedy_speculative_decoding_gb300 import _lib as L
    eng = make_engine(pkg, tiny, K=4, s_max=128)
    with pytest.raises(SFError) as e:
        eng.verify()
    assert e.value.status == L.SF_ERR_STATE
    with pytest.raises(SFError) as e:
        eng.prefill([list(range(125))])          # no room for a round
    assert e.value.status == L.SF_ERR_CAPACITY
    eng.prefill([list(range(100))])
    with pytest.raises(SFError) as e:
        eng.accept_rollback()
    assert e.value.status == L.SF_ERR_STATE
    with pytest.raises(SFError) as e:
        eng.generate(64)                          # s_max 128 runs out
    assert e.value.status == L.SF_ERR_CAPACITY
    with pytest.raises(SFError) as e:
        eng.prefill([[3, 2000]])                  # token out of range
    assert e.value.status == L.SF_ERR_ARG
    eng.close()


def test_nonfinite_logits_are_reported(pkg, tiny):
    from greedy_speculative_decoding_gb300 import SFError
    from greedy_speculative_decoding_gb300 import _lib as L
    tw, dw, gt, gd = tiny
    bad = dict(gt)
    bad["norm"] = gt["norm"].clone()
    bad["norm"][3] = float("nan")
    eng = pkg.SpecEngine(TINY_TARGET, bad, batch=1, K=2, s_max=128)
    eng.prefill([[1, 2, 3]])
    with pytest.raises(SFError) as e:
        eng.step()
    assert e.value.status == L.SF_ERR_NONFINITE
    eng.close()


SHAPES = {
    "hd128_g2": TINY_TARGET.with_(n_heads=2, n_kv_heads=1, head_dim=128),
    "hd64_g7": TINY_TARGET.with_(n_heads=14, n_kv_heads=2, head_dim=64),
    "hd128_g7": TINY_TARGET.with_(hidden=384, n_heads=14, n_kv_heads=2, head_dim=128),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_head_shapes_with_poisoned_caches(pkg, name):
    """Other head sizes and GQA group widths, with both caches filled with
    NaN bytes before prefill: every slot the kernels may read is one they
    wrote, and stale slots never leak into a result."""
    shape = SHAPES[name]
    K = 4
    w = make_weights(shape, seed=21)
    g = to_cuda(w)
    eng = pkg.SpecEngine(shape, g, shape, g, batch=1, K=K, s_max=256)
    eng.kv_t.fill_(0xFF)
    eng.kv_d.fill_(0xFF)
    prompt = uniform_prompt(70, shape.vocab, seed=22).tolist()
    eng.prefill([prompt])
    d_out = torch.zeros(K, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(K, shape.vocab, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(K + 1, shape.vocab, dtype=torch.float32, device="cuda")
    eng.draft(d_out, d_log)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    # The draft is the target; the 70-token prompt was prefilled by the
    # tcgen05 GEMM and the first draft step rewrote slot C-2 with the mma.sync
    # GEMM, so draft and verify rows agree within that slot's rounding.
    rng = (t_log.max(dim=-1).values - t_log.min(dim=-1).values)[:, None]
    assert bool(((d_log - t_log[:K]).abs() <= 1.5e-2 * rng[:K]).all())
    d = d_out.cpu().tolist()
    m = om.Model(shape, w)
    c = m.new_cache()
    m.forward(prompt[:-1], c, logit_rows=[])
    ref = m.forward([prompt[-1]] + d, c)
    worst = max(logit_err(t_log[j], ref[j]) for j in range(K + 1))
    print(f"{name}: max logit error / range = {worst:.3e}")
    assert worst < LOGIT_TOL_BF16
    n_acc, _ = eng.accept_rollback()
    assert int(n_acc[0]) == accept_brute(d, t_log.argmax(dim=-1).cpu().tolist(), K)
    eng.close()


@pytest.mark.parametrize("persistent", [False, True])
def test_round_graph_kernel_count(pkg, tiny, monkeypatch, persistent):
    """One replay of the round graph launches: per forward of more than four
    rows (the verify) an embedding, six kernels per layer (QKV, attention
    chunks, merge, O, gate/up, down) and the LM head; per draft step the
    same, or with the persistent decode kernel two launches (the forward and
    the LM head); K draft steps, one verify forward and the acceptance kernel
    (the n-gram round: the lookup kernel instead of the draft steps)."""
    monkeypatch.setenv("SF_PERSISTENT", "1" if persistent else "0")
    K = 4
    eng = make_engine(pkg, tiny, K=K)
    assert eng.round_launches() == 0          # no round graph yet
    eng.prefill([uniform_prompt(32, 1024, seed=100).tolist()])
    eng.step()
    per_fwd = lambda s: 2 + 6 * s.layers
    per_draft = 2 if persistent else per_fwd(TINY_DRAFT)
    assert eng.round_launches() == K * per_draft + per_fwd(TINY_TARGET) + 1
    eng.set_drafter(pkg.SF_DRAFT_NGRAM)
    eng.step()
    assert eng.round_launches() == 1 + per_fwd(TINY_TARGET) + 1
    eng.close()


def test_expired_wait_is_reported(pkg, tiny, monkeypatch):
    """The device error path of the bounded waits: with SF_TEST_WAIT_EXPIRE=1
    every projection's first weight-tile wait gives up at once (and then
    completes normally), the kernels set the wait bit, and the next host
    synchronisation returns SF_ERR_DEVICE; the CUDA context stays usable and
    an engine created without the switch runs a correct round afterwards."""
    from greedy_speculative_decoding_gb300 import SFError
    from greedy_speculative_decoding_gb300 import _lib as L
    prompt = uniform_prompt(32, 1024, seed=100).tolist()
    monkeypatch.setenv("SF_TEST_WAIT_EXPIRE", "1")
    eng = make_engine(pkg, tiny, K=4)
    monkeypatch.delenv("SF_TEST_WAIT_EXPIRE")
    eng.prefill([prompt])
    with pytest.raises(SFError) as e:
        eng.step()
    assert e.value.status == L.SF_ERR_DEVICE
    assert "bounded wait" in str(e.value)
    eng.close()
    ok = make_engine(pkg, tiny, K=4)
    ok.prefill([prompt])
    out, _ = ok.generate(8)
    ok.close()
    assert out[0].tolist() == od.greedy(om.Model(TINY_TARGET, tiny[0]), prompt, 8)


def test_no_drafter_is_plain_greedy(pkg, tiny):
    """SF_DRAFT_NONE: every round proposes nothing, verifies the pending
    token and commits the target's own choice, i.e. plain greedy decoding;
    the round graph is the (empty) lookup, one verify forward and the
    acceptance kernel."""
    tw = tiny[0]
    prompt = uniform_prompt(32, 1024, seed=100).tolist()
    eng = make_engine(pkg, tiny, K=1)
    eng.prefill([prompt])
    eng.set_drafter(pkg.SF_DRAFT_NONE)
    out, rounds = eng.generate(20)
    hist = eng.accept_hist()
    assert rounds == 20 and hist[0].tolist() == [20, 0]
    assert eng.round_launches() == 1 + (2 + 6 * TINY_TARGET.layers) + 1
    eng.close()
    assert out[0].tolist() == od.greedy(om.Model(TINY_TARGET, tw), prompt, 20)


@pytest.mark.parametrize("batch,mode", [(1, "neural"), (4, "neural"), (1, "ngram"), (3, "none")])
def test_device_loop_equals_host_loop(pkg, tiny, monkeypatch, batch, mode):
    """sf_generate's device-resident loop (one graph launch: a WHILE
    conditional node around the round, a control kernel deciding on the
    device) gives the same tokens, round count and accept histogram as the
    host replaying the round graph (SF_HOST_LOOP=1)."""
    lens = [32, 45, 27, 38][:batch]
    prompts = [uniform_prompt(n, 1024, seed=500 + b).tolist() for b, n in enumerate(lens)]
    if mode == "ngram":
        prompts = [ngram_prompt(96, 0.8, 1024, seed=201, base_len=48, seg_lo=8, seg_hi=16)[0].tolist()]
    res = []
    for host in ("1", "0"):
        monkeypatch.setenv("SF_HOST_LOOP", host)
        eng = make_engine(pkg, tiny, K=4, batch=batch, draft=mode == "neural")
        monkeypatch.delenv("SF_HOST_LOOP")
        eng.prefill(prompts)
        if mode == "none":
            eng.set_drafter(pkg.SF_DRAFT_NONE)
        out, rounds = eng.generate(40)
        out2, rounds2 = eng.generate(60)      # continues from 40 tokens
        res.append((out.tolist(), rounds, out2.tolist(), rounds2, eng.accept_hist().tolist(), eng.lengths()))
        eng.close()
    (o1, r1, p1, q1, h1, l1), (o2, r2, p2, q2, h2, l2) = res
    assert o1 == o2 and p1 == p2 and h1 == h2
    assert r1 == r2 and q1 == q2, (r1, r2, q1, q2)
    assert all((a == b).all() for a, b in zip(l1, l2))
    assert r2 > 0 and q2 > 0
