"""GPU parity of the NF4 path (4-bit NormalFloat weights, block 64, fp16
scales, dequantised inside the GEMM).

* The GPU quantiser (sf_nf4_quantize) against the oracle's: codes and
  scales bit-exact (both take the nearest-level decision in fp32).
* NF4 models: the weights are quantised by the oracle (test side) and
  handed to both sides; the oracle runs on the dequantised float64 weights.
  Logits within 6e-2 of each row's range (the NF4 tolerance); draft rows and
  verify rows of the same model bit for bit equal.
* A 14B-shape model (hidden 5120, 40/8 heads, FFN 13824, vocab 152064) with
  two layers: the same matrix shapes, hence the same launch configurations,
  as the 48-layer model.
"""

import pytest
import torch

from oracle import model as om
from oracle import nf4 as onf4
from synth import QWEN14B, TINY_TARGET, make_weights, uniform_prompt

from gpu_helpers import logit_err

pytestmark = pytest.mark.gpu
NF4_TOL = 6e-2
LINEAR = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as p
    return p


@pytest.mark.parametrize("rows,cols,ld", [(64, 64, 64), (300, 896, 896), (128, 5120, 5120), (70, 512, 1024)])
def test_quantizer_matches_oracle(pkg, rows, cols, ld):
    g = torch.Generator().manual_seed(rows + cols)
    full = (torch.randn(rows, ld, generator=g) * 0.02).to(torch.bfloat16)
    full[0, :64] = 0                      # an all-zero block
    full[1, 5] = 0.375                    # an exact level times an fp16 scale
    w = full[:, :cols]
    ref_codes, ref_scales = onf4.quantize(w)
    codes, scales = pkg.nf4_quantize(full.cuda()[:, :cols])
    torch.cuda.synchronize()
    assert torch.equal(codes.cpu(), ref_codes)
    assert torch.equal(scales.cpu()[:, :cols // 64], ref_scales)


def _oracle_nf4(shape, w):
    """(GPU weight dict, oracle weight dict): linear maps quantised by the
    oracle; the GPU gets codes + padded scales, the oracle the dequantised
    float64 matrices."""
    import greedy_speculative_decoding_gb300 as pkg
    gpu, ref = {}, {}
    for k, v in w.items():
        if v is not None and k.split(".")[-1] in LINEAR:
            codes, scales = onf4.quantize(v)
            padded = torch.zeros((scales.shape[0], pkg.nf4_scale_ld(v.shape[1])), dtype=torch.float16)
            padded[:, :scales.shape[1]] = scales
            gpu[k] = codes.cuda()
            gpu[k + ".scales"] = padded.cuda()
            ref[k] = onf4.dequantize(codes, scales)
        else:
            gpu[k] = None if v is None else v.cuda()
            ref[k] = v
    return gpu, ref


def _check_model(pkg, shape, seed, prompt_len, s_max):
    K = 4
    w = make_weights(shape, seed=seed)
    gw, rw = _oracle_nf4(shape, w)
    eng = pkg.SpecEngine(shape, gw, shape, gw, batch=1, K=K, s_max=s_max)
    eng.kv_t.fill_(0xFF)
    eng.kv_d.fill_(0xFF)
    prompt = uniform_prompt(prompt_len, shape.vocab, seed=seed + 1).tolist()
    eng.prefill([prompt])
    d_out = torch.zeros(K, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(K, shape.vocab, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(K + 1, shape.vocab, dtype=torch.float32, device="cuda")
    eng.draft(d_out, d_log)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    n_acc, _ = eng.accept_rollback()
    if prompt_len <= 16:
        # prompt and rounds on the mma.sync GEMM: draft rows equal verify rows
        assert torch.equal(d_log, t_log[:K])
        assert int(n_acc[0]) == K
    else:
        # prompt prefilled on the tcgen05 GEMM (weights dequantised as
        # bf16(level x scale)), slot C-2 rewritten by mma.sync (bf16 levels,
        # scale per chunk): rows agree to one bf16 rounding of the weights
        rng = (t_log.max(dim=-1).values - t_log.min(dim=-1).values)[:, None]
        assert bool(((d_log - t_log[:K]).abs() <= 2e-2 * rng[:K]).all())
        t_arg = t_log.argmax(dim=-1).cpu().tolist()
        d_h = d_out.cpu().tolist()
        n = 0
        while n < K and d_h[n] == t_arg[n]:
            n += 1
        assert int(n_acc[0]) == n
    eng.close()
    d = d_out.cpu().tolist()
    m = om.Model(shape, rw, rowwise=shape.hidden < 1024)
    c = m.new_cache()
    m.forward(prompt[:-1], c, logit_rows=[])
    ref = m.forward([prompt[-1]] + d, c)
    return max(logit_err(t_log[j], ref[j]) for j in range(K + 1))


def test_tiny_nf4_model(pkg):
    shape = TINY_TARGET.with_(ffn=768)
    worst = _check_model(pkg, shape, seed=31, prompt_len=40, s_max=256)
    print(f"tiny NF4: max logit error / range = {worst:.3e}")
    assert worst < NF4_TOL


def test_14b_shape_nf4_two_layers(pkg):
    shape = QWEN14B.with_(layers=2)
    worst = _check_model(pkg, shape, seed=41, prompt_len=12, s_max=1024)
    print(f"14B shape NF4 (2 layers): max logit error / range = {worst:.3e}")
    assert worst < NF4_TOL


@pytest.mark.parametrize("name,B,K,lens", [
    ("tiny", 4, 4, [40, 23, 57, 31]),
    ("14b2", 8, 8, [12, 30, 19, 44, 9, 27, 36, 15]),
])
def test_nf4_row_groups_ragged_batch(pkg, name, B, K, lens):
    """Sequences with prompts of different lengths whose verify forward has
    more than 16 rows (tiny: 20 rows; 14B shape: 72 rows), NF4 weights: the
    verify runs on the tcgen05 GEMM (each weight tile dequantised once into
    bf16 level x scale), the draft steps (at most 16 rows) on the mma.sync
    GEMM (bf16 levels, scale applied per chunk). Target = draft: each draft
    row agrees with its verify row to one bf16 rounding of the weights;
    accept lengths equal the brute-force prefix compare of the two; every
    sequence's verify logits are within the NF4 tolerance of the oracle."""
    shape = TINY_TARGET.with_(ffn=768) if name == "tiny" else QWEN14B.with_(layers=2)
    w = make_weights(shape, seed=51)
    gw, rw = _oracle_nf4(shape, w)
    prompts = [uniform_prompt(n, shape.vocab, seed=60 + b).tolist() for b, n in enumerate(lens)]
    eng = pkg.SpecEngine(shape, gw, shape, gw, batch=B, K=K, s_max=256)
    eng.kv_t.fill_(0xFF)
    eng.kv_d.fill_(0xFF)
    eng.prefill(prompts)
    d_out = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(B, K, shape.vocab, dtype=torch.float32, device="cuda")
    t_log = torch.zeros(B, K + 1, shape.vocab, dtype=torch.float32, device="cuda")
    eng.draft(d_out, d_log)
    eng.verify(None, t_log)
    torch.cuda.synchronize()
    rng = (t_log.max(dim=-1).values - t_log.min(dim=-1).values)[..., None]
    assert bool(((d_log - t_log[:, :K]).abs() <= 2e-2 * rng[:, :K]).all())
    t_arg = t_log.argmax(dim=-1).cpu()
    n_acc, _ = eng.accept_rollback()
    d_h = d_out.cpu()
    for b in range(B):
        n = 0
        while n < K and int(d_h[b, n]) == int(t_arg[b, n]):
            n += 1
        assert int(n_acc[b]) == n, b
    lt, _ = eng.lengths()
    assert [int(x) for x in lt] == [n + int(a) for n, a in zip(lens, n_acc)]
    eng.close()
    m = om.Model(shape, rw, rowwise=shape.hidden < 1024)
    worst = 0.0
    for b in range(B):
        c = m.new_cache()
        m.forward(prompts[b][:-1], c, logit_rows=[])
        ref = m.forward([prompts[b][-1]] + d_out[b].cpu().tolist(), c)
        worst = max(worst, max(logit_err(t_log[b, j], ref[j]) for j in range(K + 1)))
    print(f"{name} NF4 batch {B}: max logit error / range = {worst:.3e}")
    assert worst < NF4_TOL
