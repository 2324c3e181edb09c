"""Benchmark: committed tokens/s of greedy speculative decoding on one GB300,
plus the verify step's and the dominant GEMM's fraction of the HBM roofline.

Workload (default): Qwen2.5-7B-shape bf16 target (random init, seed 0) with
the Qwen2.5-0.5B-shape draft whose embedding is the target's first 896
columns (seed 2), K = 8 guesses per round, batch 1, a 512-token uniform
random prompt (seed 102), 256 generated tokens per step. A step rewinds the
engine to the prompt (sf_reset) and generates 256 tokens with replayed
round graphs (sf_generate). Weights (16 GB) exceed the 129 MB L2, so no
flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs an independent replica (the step has no
cross-sequence exchange); rank 0 prints one JSON line.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "committed tokens/s (greedy spec-decode, 1 GB300); verify-step % HBM roofline"
N_NEW = 256
PROMPT_LEN = 512
VERIFY_CTX = 2048
K_GUESS = 8
S_MAX = 4096


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# the roofline kernel from one ncu capture, valid only for the k_gemm.cu
# source it was taken on (sha256 prefix); reported as null otherwise.
GEMM_TRAFFIC = {"sha": "40337611a5c63c55", "bytes": 274916608}
# Sources the k_gemm kernel is compiled from; the stored traffic applies only
# to the exact sources it was captured with.
GEMM_SOURCES = ("k_gemm.cu", "gemm_epi.cuh", "sf_common.cuh", "sf_kernels.h")


def _gemm_sources_sha():
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "greedy_speculative_decoding_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _gemm_traffic():
    try:
        sha = _gemm_sources_sha()
    except OSError:
        return None
    return GEMM_TRAFFIC["bytes"] if sha == GEMM_TRAFFIC["sha"] else None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        mx.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower().startswith("active"):
                            reasons.add(n)
            os.unlink(self.path)
        except Exception:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0, None
    import torch.distributed as dist
    rank, local = int(os.environ["RANK"]), int(os.environ.get("LOCAL_RANK", "0"))
    dist.init_process_group("gloo")
    return rank, ws, local, dist


def _max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _shapes():
    from synth import QWEN05B_SHARED, QWEN7B
    return QWEN7B, QWEN05B_SHARED


def _weights(device):
    from synth import QWEN05B, make_weights, shared_embedding_draft
    t_shape, d_shape = _shapes()
    tw = make_weights(t_shape, seed=0, device=device)
    dw = make_weights(QWEN05B, seed=2, device=device)
    dw = shared_embedding_draft(dw, tw["embed"], d_shape.hidden)
    return tw, dw


def weight_bytes(shape) -> int:
    h, f = shape.hidden, shape.ffn
    per_layer = 2 * (h * shape.q_dim + 2 * h * shape.kv_dim + shape.q_dim * h + 3 * h * f)
    lm = 2 * shape.vocab * h
    return shape.layers * per_layer + lm


def kv_bytes(shape, ctx_read: int, rows: int) -> int:
    per_slot = shape.layers * 2 * shape.n_kv_heads * shape.head_dim * 2
    return per_slot * (ctx_read + rows)


def launches_per_round(t_shape, d_shape, K) -> int:
    """Upper bound (6 kernels per layer); the engine reports the exact count."""
    per_fwd = lambda s: 2 + 6 * s.layers   # embed, 6 per layer, LM head
    return K * per_fwd(d_shape) + per_fwd(t_shape) + 1


# ---------------------------------------------------------------------------- other workloads
def _timed(fn, stream, reps):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _gen_rate(eng, n_new=256):
    """(committed tokens/s, mean committed per round) of one sf_generate run
    from the prefilled prompt, timed with CUDA events on the engine stream."""
    import torch
    eng.reset()
    eng.generate(8)          # warm: graph captured, clocks up
    eng.reset()
    rounds = [0]

    def run():
        _, r = eng.generate(n_new)
        rounds[0] = r
    ms = _timed(run, eng.stream, 1)
    return n_new / (ms / 1e3), n_new / max(1, rounds[0])


def extra_workloads(pkg, tw, peak):
    """The other workloads of the suite, each bounded to a few seconds:
    the 0.5B-shape draft decode step at context 512 (standalone, vocabulary
    151936), sigma-perturbed target copies as drafts, prompt-lookup drafting
    on repetitive prompts (one guess, and several verified side by side),
    and the 14B-shape NF4 target at batch 1."""
    import torch
    from synth import (QWEN05B, QWEN14B, QWEN7B, make_weights, ngram_prompt, perturbed_copy,
                       repeated_fraction, shared_embedding_draft, uniform_prompt)
    out = {}
    # 0.5B-shape decode step, context 512: the model drafts for itself.
    try:
        w5 = make_weights(QWEN05B, seed=0, device="cuda")
        e5 = pkg.SpecEngine(QWEN05B, w5, QWEN05B, w5, batch=1, K=K_GUESS, s_max=S_MAX)
        e5.prefill([uniform_prompt(512, QWEN05B.vocab, seed=101).numpy()])

        def one():
            e5.draft()
            e5.verify()
            e5.accept_rollback()
        one()
        e5.reset()
        ms = []
        for _ in range(10):
            ms.append(_timed(e5.draft, e5.stream, 1))
            e5.verify()
            e5.accept_rollback()
        step_ms = statistics.median(ms) / K_GUESS
        b = weight_bytes(QWEN05B) + kv_bytes(QWEN05B, 512 + 8, 1)
        out["draft_05b_ctx512"] = {"ms_per_decode_step": round(step_ms, 4), "bytes": b,
                                   "gbs": round(b / step_ms / 1e6, 1), "frac_of_measured_peak": round(b / step_ms / 1e6 / peak, 4),
                                   "frac_of_8TBs": round(b / step_ms / 8e9, 4)}
        e5.close()
        del w5, e5
    except Exception as ex:
        out["draft_05b_ctx512"] = {"error": repr(ex)[:200]}
    torch.cuda.empty_cache()
    # Target copies perturbed by N(0, sigma) as drafts (7B-shape draft).
    prompt = uniform_prompt(PROMPT_LEN, QWEN7B.vocab, seed=102).numpy()
    for sigma in (0.0, 0.002, 0.01):
        try:
            dcopy = perturbed_copy(tw, sigma, seed=3)
            es = pkg.SpecEngine(QWEN7B, tw, QWEN7B, dcopy, batch=1, K=K_GUESS, s_max=S_MAX)
            es.prefill([prompt])
            rate, mean_c = _gen_rate(es)
            out[f"sigma_{sigma}"] = {"tokens_per_s": round(rate, 2), "mean_committed_per_round": round(mean_c, 3),
                                     "accept_hist": es.accept_hist()[0].tolist()}
            es.close()
            del dcopy, es
        except Exception as ex:
            out[f"sigma_{sigma}"] = {"error": repr(ex)[:200]}
        torch.cuda.empty_cache()
    # Prompt lookup on repetitive prompts (K = 4).
    for r in (0.2, 0.5, 0.8):
        try:
            p, mask = ngram_prompt(1024, r, QWEN7B.vocab, seed=200 + int(10 * r))
            en = pkg.SpecEngine(QWEN7B, tw, batch=1, K=4, s_max=S_MAX)
            en.prefill([p.numpy()])
            rate, mean_c = _gen_rate(en)
            out[f"ngram_r{r}"] = {"tokens_per_s": round(rate, 2), "mean_committed_per_round": round(mean_c, 3),
                                  "repeated_fraction": round(repeated_fraction(mask), 3)}
            en.close()
        except Exception as ex:
            out[f"ngram_r{r}"] = {"error": repr(ex)[:200]}
    torch.cuda.empty_cache()
    # Several prompt-lookup guesses per round (K = 8 verify rows after the
    # pending token): one guess of 8, two of 4, four of 2, on the r = 0.8 prompt.
    try:
        p, mask = ngram_prompt(1024, 0.8, QWEN7B.vocab, seed=208)
        for n_cand in (1, 2, 4):
            en = pkg.SpecEngine(QWEN7B, tw, batch=1, K=8, s_max=S_MAX)
            en.set_drafter(pkg.SF_DRAFT_TREE, 2, 4)
            en.set_tree_candidates(n_cand)
            en.prefill([p.numpy()])
            rate, mean_c = _gen_rate(en)
            out[f"ngram_tree_r0.8_c{n_cand}"] = {"tokens_per_s": round(rate, 2),
                                                 "mean_committed_per_round": round(mean_c, 3),
                                                 "candidates": n_cand, "guesses_each": 8 // n_cand}
            en.close()
    except Exception as ex:
        out["ngram_tree_r0.8"] = {"error": repr(ex)[:200]}
    torch.cuda.empty_cache()
    # Plain greedy decoding of the same target (no drafter: each round verifies
    # the pending token and commits the target's own choice), the baseline the
    # speculative rounds are measured against.
    try:
        eg = pkg.SpecEngine(QWEN7B, tw, batch=1, K=1, s_max=S_MAX)
        eg.set_drafter(pkg.SF_DRAFT_NONE)
        eg.prefill([prompt])
        rate, mean_c = _gen_rate(eg)
        out["plain_greedy"] = {"tokens_per_s": round(rate, 2), "mean_committed_per_round": round(mean_c, 3),
                               "what": "7B-shape target alone, one verify forward (2 rows) per token"}
        eg.close()
    except Exception as ex:
        out["plain_greedy"] = {"error": repr(ex)[:200]}
    torch.cuda.empty_cache()
    return out


def nf4_workload(pkg, peak):
    """14B-shape target with NF4 linear maps (quantised on the GPU), batch 1,
    K = 8 with the 0.5B-shape draft on the target's first 896 embedding
    columns: verify step at context 2048 and committed tokens/s."""
    import torch
    from synth import QWEN05B, QWEN14B, make_weights, shared_embedding_draft, uniform_prompt
    tw = make_weights(QWEN14B, seed=0, device="cuda")
    tq = pkg.quantize_model_nf4(QWEN14B, tw)
    for k in list(tw):
        if k.split(".")[-1] in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            tw[k] = None
    torch.cuda.empty_cache()
    d_shape = QWEN05B.with_(vocab=QWEN14B.vocab, embed_ld=QWEN14B.hidden)
    dw = shared_embedding_draft(make_weights(QWEN05B, seed=2, device="cuda"), tq["embed"], QWEN05B.hidden)
    eng = pkg.SpecEngine(QWEN14B, tq, d_shape, dw, batch=1, K=K_GUESS, s_max=S_MAX)
    eng.prefill([uniform_prompt(VERIFY_CTX, QWEN14B.vocab, seed=301).numpy()])
    v = []
    for i in range(8):
        eng.draft()
        v.append(_timed(eng.verify, eng.stream, 1))
        eng.accept_rollback()
    vms = statistics.median(v[2:])
    h, f = QWEN14B.hidden, QWEN14B.ffn
    lin = QWEN14B.layers * (h * QWEN14B.q_dim + 2 * h * QWEN14B.kv_dim + QWEN14B.q_dim * h + 3 * h * f)
    nbytes = lin // 2 + lin // 64 * 2 + 2 * QWEN14B.vocab * h + kv_bytes(QWEN14B, VERIFY_CTX, K_GUESS + 1)
    eng.prefill([uniform_prompt(PROMPT_LEN, QWEN14B.vocab, seed=302).numpy()])
    rate, mean_c = _gen_rate(eng)
    eng.close()
    b1 = {"verify_ms": round(vms, 4), "verify_bytes": nbytes, "verify_gbs": round(nbytes / vms / 1e6, 1),
          "verify_frac_of_measured_peak": round(nbytes / vms / 1e6 / peak, 4), "tokens_per_s": round(rate, 2),
          "mean_committed_per_round": round(mean_c, 3), "batch": 1}
    torch.cuda.empty_cache()
    try:
        b8 = nf4_batch_workload(pkg, peak, tq, d_shape, dw, lin)
    except Exception as ex:  # report, keep the batch-1 figures
        b8 = {"error": repr(ex)[:300]}
    return b1, b8


NF4_B8_SMAX = 8704
NF4_B8_NEW = 32


def nf4_batch_workload(pkg, peak, tq, d_shape, dw, lin):
    """The 14B-shape NF4 target with 8 independent sequences whose contexts
    are drawn uniformly from 1024..8192 tokens (seeded), K = 8 with the
    0.5B-shape draft: every verify forward has 72 token rows. Reports the
    verify step (weights once + each sequence's cache) and committed tokens/s
    over all sequences for NF4_B8_NEW new tokens per sequence."""
    import numpy as np
    import torch
    from synth import QWEN14B, uniform_prompt
    B = 8
    ctx = np.random.default_rng(300).integers(1024, 8193, size=B)
    prompts = [uniform_prompt(int(n), QWEN14B.vocab, seed=310 + b).numpy() for b, n in enumerate(ctx)]
    eng = pkg.SpecEngine(QWEN14B, tq, d_shape, dw, batch=B, K=K_GUESS, s_max=NF4_B8_SMAX)
    t0 = time.time()
    eng.prefill(prompts)
    prefill_s = time.time() - t0
    v = []
    for i in range(6):
        eng.draft()
        v.append(_timed(eng.verify, eng.stream, 1))
        eng.accept_rollback()
    vms = statistics.median(v[2:])
    lt, _ = eng.lengths()
    kv = sum(kv_bytes(QWEN14B, int(n), K_GUESS + 1) for n in lt)   # cache read up to the last verify
    nbytes = lin // 2 + lin // 64 * 2 + 2 * QWEN14B.vocab * QWEN14B.hidden + kv
    eng.reset()
    eng.generate(2)
    eng.reset()
    rounds = [0]

    def run():
        rounds[0] = eng.generate(NF4_B8_NEW)[1]
    ms = _timed(run, eng.stream, 1)
    eng.close()
    return {"batch": B, "contexts": [int(n) for n in ctx], "verify_rows": B * (K_GUESS + 1),
            "verify_ms": round(vms, 4), "verify_bytes": nbytes, "verify_gbs": round(nbytes / vms / 1e6, 1),
            "verify_frac_of_measured_peak": round(nbytes / vms / 1e6 / peak, 4),
            "tokens_per_s": round(B * NF4_B8_NEW / (ms / 1e3), 2), "new_tokens_per_sequence": NF4_B8_NEW,
            "rounds": rounds[0], "prefill_s": round(prefill_s, 2)}


def _kernel_bytes(shape, label, ctx):
    """Algorithmic bytes one launch of a forward kernel moves (weights it
    streams; for attention the keys and values it reads at context ctx). A
    phase of the persistent decode kernel ("d_" + kernel) moves what the
    kernel of that name does."""
    if label.startswith("d_"):
        label = label[2:]
    h, f = shape.hidden, shape.ffn
    w = {"qkv": (shape.q_dim + 2 * shape.kv_dim) * h * 2, "o_proj": h * shape.q_dim * 2,
         "gate_up": 2 * f * h * 2, "down": h * f * 2, "lm_head": shape.vocab * h * 2,
         "attention": 2 * shape.n_kv_heads * shape.head_dim * 2 * ctx}
    # The persistent decode kernel: every layer's projections and cache.
    w["decode"] = shape.layers * (w["qkv"] + w["o_proj"] + w["gate_up"] + w["down"] + w["attention"])
    return w.get(label)


def trace_breakdown(pkg, t_shape, tw, d_shape, dw, rounds=5, ctx=VERIFY_CTX, peak=None):
    """Per (phase, kernel) of replayed rounds: the time each launch adds to the
    dependent chain (gap between consecutive 'producer done' stamps of the
    launch timeline the engine records with SF_TRACE=1) and, for the kernels
    that stream weights or the cache, bytes / that time."""
    import collections
    from synth import uniform_prompt
    old = os.environ.get("SF_TRACE")
    os.environ["SF_TRACE"] = "1"
    try:
        eng = pkg.SpecEngine(t_shape, tw, d_shape, dw, batch=1, K=K_GUESS, s_max=S_MAX)
    finally:
        if old is None:
            del os.environ["SF_TRACE"]
        else:
            os.environ["SF_TRACE"] = old
    eng.prefill([uniform_prompt(ctx, t_shape.vocab, seed=103).numpy()])
    # The round graph is captured on the first step; every replay rewrites the
    # same timeline slots, so the stamps describe the last round replayed.
    first = eng.trace_count()
    for _ in range(rounds):
        eng.step()
    tr = eng.trace(first, eng.trace_count() - first)
    eng.close()
    agg = collections.OrderedDict()
    heads = 0
    for i in range(len(tr) - 1):
        lab, st, wd = tr[i]
        phase = "draft" if heads < K_GUESS else "verify"
        a = agg.setdefault((phase, lab), [0, 0.0, 0.0])
        a[0] += 1
        a[1] += (tr[i + 1][2] - wd) / 1e3
        a[2] += (wd - st) / 1e3
        if lab == "lm_head":
            heads += 1
    rows = []
    for (ph, lab), (n, t, w) in agg.items():
        r = {"phase": ph, "kernel": lab, "launches": n, "total_us": round(t, 1), "avg_us": round(t / n, 2),
             "early_start_us": round(w / n, 2)}
        b = _kernel_bytes(t_shape if ph == "verify" else d_shape, lab, ctx)
        if b:
            r["bytes"] = b
            r["gbs"] = round(b / (t / n) / 1e3, 1)
            if peak:
                r["frac_of_measured_peak"] = round(b / (t / n) / 1e3 / peak, 4)
        rows.append(r)
    return rows, round((tr[-1][2] - tr[0][1]) / 1e3, 1)


def run_trace(args):
    """Launch timeline of replayed rounds at context 2048: per kernel kind,
    the time each launch adds to the dependent chain."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as pkg
    t_shape, d_shape = _shapes()
    tw, dw = _weights("cuda")
    rows, span = trace_breakdown(pkg, t_shape, tw, d_shape, dw, peak=_peaks()[0])
    print(json.dumps({"trace": rows, "round_span_us": span}))


# ---------------------------------------------------------------------------- ours
def run_gemm_only(args):
    """Small case for kernel profiling: the 7B gate+up matrix (271 MB, above
    L2) streamed by sf_linear with --gemm-rows token rows (default 9: the
    mma.sync kernel; above 16: the tcgen05 kernel), a few launches."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as pkg
    t_shape, _ = _shapes()
    N, K, M = 2 * t_shape.ffn, t_shape.hidden, args.gemm_rows
    gen = torch.Generator(device="cuda").manual_seed(0)
    w = (torch.randn(N, K, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    x = torch.randn(M, K, generator=gen, device="cuda")
    y = torch.empty(M, N, device="cuda")
    ws = torch.empty(pkg.load().sf_linear_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    xf = pkg.to_frag(x)
    for _ in range(6):
        pkg.linear_frag(w, xf, M, y, ws)
    torch.cuda.synchronize()
    print(json.dumps({"gemm_only": True, "N": N, "K": K, "M": M}))


def run_nf4_b8_small(args):
    """Small case for kernel profiling of the batch-8 NF4 verify: the 14B
    shape with 2 layers and a 32000-token vocabulary (about 2.5 GB on the
    device), NF4 linear maps, 8 sequences prefilled to the batch-8
    workload's contexts, prompt-lookup rounds (72-row verify forwards); the
    last two rounds run inside the NVTX range "round"."""
    import numpy as np
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as pkg
    from synth import QWEN14B, make_weights, uniform_prompt
    shape = QWEN14B.with_(layers=2, vocab=32000)
    w = pkg.quantize_model_nf4(shape, make_weights(shape, seed=0, device="cuda"))
    B = 8
    ctx = np.random.default_rng(300).integers(1024, 8193, size=B)
    prompts = [uniform_prompt(int(n), shape.vocab, seed=310 + b).numpy() for b, n in enumerate(ctx)]
    eng = pkg.SpecEngine(shape, w, batch=B, K=K_GUESS, s_max=NF4_B8_SMAX)
    eng.prefill(prompts)
    eng.step()
    torch.cuda.synchronize()
    for _ in range(2):
        torch.cuda.nvtx.range_push("round")
        eng.step()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    eng.close()
    print(json.dumps({"nf4_b8_small": True, "contexts": [int(n) for n in ctx]}))


def run_verify_small(args):
    """Small case for kernel profiling of the batch-1 verify: the 7B shape
    with 2 layers (about 2.6 GB on the device), the cache prefilled to 2048
    tokens, prompt-lookup rounds of 9 verify rows; the last two rounds run
    inside the NVTX range "round"."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as pkg
    from synth import QWEN7B, make_weights, uniform_prompt
    shape = QWEN7B.with_(layers=2)
    w = make_weights(shape, seed=0, device="cuda")
    eng = pkg.SpecEngine(shape, w, batch=1, K=K_GUESS, s_max=S_MAX)
    eng.prefill([uniform_prompt(VERIFY_CTX, shape.vocab, seed=103).numpy()])
    eng.step()
    torch.cuda.synchronize()
    for _ in range(2):
        torch.cuda.nvtx.range_push("round")
        eng.step()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    eng.close()
    print(json.dumps({"verify_small": True, "ctx": VERIFY_CTX}))


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local, dist = _dist()
    torch.cuda.set_device(local)
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as pkg
    from synth import uniform_prompt

    t_shape, d_shape = _shapes()
    tw, dw = _weights("cuda")
    torch.cuda.synchronize()
    eng = pkg.SpecEngine(t_shape, tw, d_shape, dw, batch=1, K=K_GUESS, s_max=S_MAX)
    prompt = uniform_prompt(PROMPT_LEN, t_shape.vocab, seed=102).numpy()
    eng.prefill([prompt])
    stream = eng.stream

    for _ in range(args.warmup):
        eng.reset()
        eng.generate(N_NEW)
    torch.cuda.synchronize()
    _barrier(dist)
    rounds_total = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        e0.record(stream)
        for _ in range(args.steps):
            eng.reset()
            _, r = eng.generate(N_NEW)
            rounds_total += r
        e1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    # kernels per round: the node count of the replayed round graph
    round_launches = eng.round_launches() or launches_per_round(t_shape, d_shape, K_GUESS)
    _barrier(dist)
    ms = e0.elapsed_time(e1)
    ms_max = _max_over_ranks(dist, ms)
    hist = eng.accept_hist()[0]
    value = world * args.steps * N_NEW / (ms_max / 1e3)

    # ---- prefill (time to first round): the 512-token prompt and the 2048-token context, both
    # models, chunks of up to 80 rows (host wall clock around the synchronous call)
    prefill = {}
    for n, seed in ((PROMPT_LEN, 102), (VERIFY_CTX, 103)):
        p = uniform_prompt(n, t_shape.vocab, seed=seed).numpy()
        eng.prefill([p])                       # warm
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        eng.prefill([p])
        dt = time.perf_counter() - t0
        prefill[str(n)] = {"ms": round(1e3 * dt, 2), "tokens_per_s": round(n / dt, 1)}

    # ---- verify step and draft step at context 2048 (graph replays, events on the engine stream)
    eng.prefill([uniform_prompt(VERIFY_CTX, t_shape.vocab, seed=103).numpy()])
    v_ms, d_ms = [], []
    for i in range(3 + 10):
        a0, a1, a2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a0.record(stream)
        eng.draft()
        a1.record(stream)
        eng.verify()
        a2.record(stream)
        eng.accept_rollback()
        if i >= 3:
            d_ms.append(a0.elapsed_time(a1))
            v_ms.append(a1.elapsed_time(a2))
    verify_ms = statistics.median(v_ms)
    draft_ms = statistics.median(d_ms) / K_GUESS
    v_bytes = weight_bytes(t_shape) + kv_bytes(t_shape, VERIFY_CTX, K_GUESS + 1)
    d_bytes = weight_bytes(d_shape) + kv_bytes(d_shape, VERIFY_CTX, 1)
    peak, peak_src = _peaks()

    # ---- dominant kernel: the weight-streaming GEMM on the 7B gate/up shape, 9 rows
    N, K, M = 2 * t_shape.ffn, t_shape.hidden, K_GUESS + 1
    wg = torch.cat([tw["layers.0.wg"], tw["layers.0.wu"]], 0)
    x = torch.randn(M, K, device="cuda")
    y = torch.empty(M, N, device="cuda")
    ws = torch.empty(pkg.load().sf_linear_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    xf = pkg.to_frag(x)   # the operand order the GEMM reads; the timed launches are the GEMM alone
    cur = torch.cuda.current_stream()
    for _ in range(3):
        pkg.linear_frag(wg, xf, M, y, ws)
    reps = 20
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(cur)
    for _ in range(reps):
        pkg.linear_frag(wg, xf, M, y, ws)
    g1.record(cur)
    torch.cuda.synchronize()
    gemm_ms = g0.elapsed_time(g1) / reps
    gemm_bytes = N * K * 2 + M * K * 4 + M * N * 4
    gemm_gbs = gemm_bytes / (gemm_ms / 1e3) / 1e9
    # The tcgen05 (TMEM-accumulator) GEMM on the same matrix at 72 token rows,
    # the batch-8 verify's row count: same timing method.
    M72 = 72
    x72 = torch.randn(M72, K, device="cuda")
    y72 = torch.empty(M72, N, device="cuda")
    xf72 = pkg.to_frag(x72)
    for _ in range(3):
        pkg.linear_frag(wg, xf72, M72, y72, ws)
    g0.record(cur)
    for _ in range(reps):
        pkg.linear_frag(wg, xf72, M72, y72, ws)
    g1.record(cur)
    torch.cuda.synchronize()
    tc_ms = g0.elapsed_time(g1) / reps
    tc_bytes = N * K * 2 + M72 * K * 4 + M72 * N * 4
    del wg, x72, y72, xf72

    # ---- end to end through the C ABI with host buffers (prefill from pinned host memory)
    pinned = torch.from_numpy(prompt.astype(np.int32)).pin_memory()
    out = torch.zeros((1, N_NEW), dtype=torch.int32).pin_memory()
    e2e_steps = max(1, min(3, args.steps))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        eng.prefill(pinned.numpy()[None, :])
        eng.generate(N_NEW, out.numpy())
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_value = world * e2e_steps * N_NEW / _max_over_ranks(dist, e2e_s)
    eng.close()

    extra = {}
    if rank == 0 and not args.no_extra:
        extra = extra_workloads(pkg, tw, peak)
        try:
            rows, span = trace_breakdown(pkg, t_shape, tw, d_shape, dw, peak=peak)
            extra["round_kernels"] = {"ctx": VERIFY_CTX, "round_span_us": span, "kernels": rows,
                                      "how": "SF_TRACE=1 launch timeline of one replayed round: time each launch "
                                             "adds to the dependent chain; bytes = weights (attention: KV) per launch"}
        except Exception as ex:
            extra["round_kernels"] = {"error": repr(ex)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del eng
        try:
            cpu = cpu_baseline(tw, dw)
        except Exception as ex:  # report, keep the GPU line
            cpu = {"value": None, "unit": "tokens/s", "kind": "oracle", "error": repr(ex)[:300]}
    if rank == 0 and not args.no_extra:
        del tw, dw
        torch.cuda.empty_cache()
        try:
            extra["nf4_14b_b1"], extra["nf4_14b_b8"] = nf4_workload(pkg, peak)
        except Exception as ex:
            extra["nf4_14b_b1"] = {"error": repr(ex)[:300]}

    if rank == 0:
        mean_commit = float((hist * (np.arange(K_GUESS + 1) + 1)).sum() / max(1, hist.sum()))
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: random-init weights N(0,0.02), uniform random prompt",
            "config": {"workload": "Qwen2.5-7B-shape bf16 target + Qwen2.5-0.5B-shape draft (target's first 896 "
                                   "embedding columns), K=8, batch 1, 512-token prompt, 256 new tokens per step",
                       "global_batch": 1, "seq_len": PROMPT_LEN + N_NEW, "parallelism": f"replicas x{world}",
                       "l2": "no flush: 16 GB of weights stream per round, above the 129 MB L2"},
            "e2e": {"value": round(e2e_value, 3), "unit": "tokens/s", "h2d_bytes_per_step": PROMPT_LEN * 4 + 4,
                    "d2h_bytes_per_step": N_NEW * 4},
            "gpu_launches": rounds_total * round_launches,
            "roofline": {"kernel": "k_gemm (weight-streaming GEMM), 7B gate+up [37888 x 3584] bf16, 9 rows",
                         "bound": "hbm", "achieved": round(gemm_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gemm_gbs / peak, 4), "traffic": _gemm_traffic(), "peak_source": peak_src,
                         "algorithmic_bytes": gemm_bytes, "ms_per_launch": round(gemm_ms, 4)},
            "tc_gemm_72rows": {"kernel": "k_umma (tcgen05, TMEM accumulator), 7B gate+up [37888 x 3584] bf16, "
                                         "72 token rows", "ms_per_launch": round(tc_ms, 4),
                               "gbs": round(tc_bytes / (tc_ms / 1e3) / 1e9, 1),
                               "frac_of_measured_peak": round(tc_bytes / (tc_ms / 1e3) / 1e9 / peak, 4),
                               "tflops": round(2 * N * K * M72 / (tc_ms / 1e3) / 1e12, 1)},
            "verify_step": {"ms": round(verify_ms, 4), "bytes": v_bytes, "ctx": VERIFY_CTX,
                            "gbs": round(v_bytes / (verify_ms / 1e3) / 1e9, 1),
                            "frac_of_measured_peak": round(v_bytes / (verify_ms / 1e3) / 1e9 / peak, 4),
                            "frac_of_8TBs": round(v_bytes / (verify_ms / 1e3) / 8e12, 4)},
            "draft_step": {"ms": round(draft_ms, 4), "bytes": d_bytes, "ctx": VERIFY_CTX,
                           "gbs": round(d_bytes / (draft_ms / 1e3) / 1e9, 1),
                           "frac_of_measured_peak": round(d_bytes / (draft_ms / 1e3) / 1e9 / peak, 4),
                           "frac_of_8TBs": round(d_bytes / (draft_ms / 1e3) / 8e12, 4)},
            "accept": {"mean_committed_per_round": round(mean_commit, 3), "hist": hist.tolist(),
                       "rounds": rounds_total},
            "prefill": {"what": "both models over the prompt, chunks of up to 80 rows", **prefill},
            "clocks": clk.summary(),
        }
        if extra:
            line["workloads"] = extra
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- oracle
def _synthetic_cache(model, n, seed):
    """The oracle's KV cache holding n slots of N(0, 1) keys and values: the
    state a prefill of n tokens leaves, for timing the round after it without
    running that prefill."""
    import torch
    g = torch.Generator().manual_seed(seed)
    s = model.shape
    c = model.new_cache()
    for l in range(s.layers):
        k = torch.randn(n, s.n_kv_heads, s.head_dim, generator=g, dtype=torch.float64)
        v = torch.randn(n, s.n_kv_heads, s.head_dim, generator=g, dtype=torch.float64)
        for j in range(n):
            c.append(l, k[j], v[j])
    return c


class OracleRounds:
    """The CPU oracle on the benchmark's workload: speculative rounds of the
    0.5B-shape draft (K = 8) and the 7B-shape target at the prompt's context
    (512), with both caches holding that context already."""

    def __init__(self, tw_cpu, dw_cpu, ctx=PROMPT_LEN):
        from oracle import model as om
        from synth import uniform_prompt
        t_shape, d_shape = _shapes()
        self.tm = om.Model(t_shape, tw_cpu, memoize=False, rowwise=False)
        self.dm = om.Model(d_shape, dw_cpu, memoize=False, rowwise=False)
        self.seq = uniform_prompt(ctx, t_shape.vocab, seed=102).tolist()
        self.tc = _synthetic_cache(self.tm, ctx - 1, 1)
        self.dc = _synthetic_cache(self.dm, ctx - 1, 2)

    def round(self):
        """One round; returns (committed tokens, seconds, seconds of the draft
        steps, seconds of the verify pass)."""
        from oracle import decode as od
        from oracle import model as om
        t0 = time.perf_counter()
        feed, guesses = [self.seq[-1]], []
        for _ in range(K_GUESS):
            lg = self.dm.forward(feed, self.dc)[0]
            guesses.append(om.first_argmax(lg))
            feed = [guesses[-1]]
        t1 = time.perf_counter()
        lg = self.tm.forward([self.seq[-1]] + guesses, self.tc)
        choice = [om.first_argmax(lg[i]) for i in range(K_GUESS + 1)]
        t2 = time.perf_counter()
        n = od.accept_length(guesses, choice)
        self.seq += guesses[:n] + [choice[n]]
        self.tc.truncate(len(self.seq) - 1)
        self.dc.truncate(min(self.dc.length, len(self.seq) - 1))
        return n + 1, time.perf_counter() - t0, t1 - t0, t2 - t1


def _tiny_end_to_end():
    """The tiny correctness workload end to end on the oracle: prefill of the
    32-token prompt and 64 tokens of speculative decoding (K = 4, one-layer
    draft). Returns (tokens, seconds)."""
    from oracle import decode as od
    from oracle import model as om
    from synth import TINY_DRAFT, TINY_TARGET, draft_from_target_layer0, make_weights, uniform_prompt
    tw = make_weights(TINY_TARGET, seed=0)
    dw = draft_from_target_layer0(tw, TINY_DRAFT, 0.005, seed=1)
    prompt = uniform_prompt(32, TINY_TARGET.vocab, seed=100).tolist()
    t0 = time.perf_counter()
    r = od.spec_decode(om.Model(TINY_TARGET, tw), om.Model(TINY_DRAFT, dw), prompt, 4, 64)
    return len(r["tokens"]), time.perf_counter() - t0


def _cores():
    import torch
    return {"nproc": os.cpu_count(), "torch_threads": torch.get_num_threads()}


def cpu_baseline(tw, dw, rounds=3):
    cpu = lambda w: {k: (None if v is None else v.detach().to("cpu")) for k, v in w.items()}
    orc = OracleRounds(cpu(tw), cpu(dw))
    orc.round()                          # warm: first touch of the weights
    n = s = sd = sv = 0.0
    for _ in range(rounds):
        c, t, td, tv = orc.round()
        n, s, sd, sv = n + c, s + t, sd + td, sv + tv
    tn, ts = _tiny_end_to_end()
    cores = _cores()
    return {"value": round(n / s, 5), "unit": "tokens/s", "cores": cores["torch_threads"], "nproc": cores["nproc"],
            "kind": "oracle",
            "sample": f"{rounds} speculative rounds of the benchmark workload (8 steps of the 0.5B-shape draft, "
                      "one 9-row verify of the 7B-shape target, accept) at the 512-token context, caches holding "
                      "that context already (prefill not run); fp64 torch CPU",
            "seconds": round(s, 2), "committed": int(n),
            "draft_decode_step_s": round(sd / rounds / K_GUESS, 4), "verify_step_s": round(sv / rounds, 3),
            "tiny_end_to_end": {"tokens_per_s": round(tn / ts, 2), "seconds": round(ts, 2),
                                "what": "tiny workload: prefill + 64 tokens, K=4"}}


def run_reference(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    tw, dw = _weights("cpu")
    orc = OracleRounds(tw, dw)
    for _ in range(min(args.warmup, 1)):
        orc.round()
    steps, tot_n, tot_s = args.steps, 0, 0.0
    for _ in range(steps):
        n, s, _, _ = orc.round()
        tot_n += n
        tot_s += s
    value = tot_n / tot_s
    cores = _cores()
    sample = ("one speculative round per step (8 draft steps of the 0.5B-shape draft, one 9-row verify of the "
              "7B-shape target, accept) at the 512-token context, caches holding it already; fp64 torch CPU")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / steps, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic: random-init weights N(0,0.02), uniform prompt",
        "config": {"workload": "Qwen2.5-7B-shape bf16 target + Qwen2.5-0.5B-shape draft, K=8, batch 1, 512-token "
                               "context; each step one speculative round"},
        "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "kind": "oracle",
                         "cores": cores["torch_threads"], "nproc": cores["nproc"], "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--tokens", type=int, default=N_NEW, help="new tokens per step (profiling runs use fewer)")
    ap.add_argument("--gemm-only", action="store_true", help="small case for kernel profiling")
    ap.add_argument("--gemm-rows", type=int, default=K_GUESS + 1, help="token rows of --gemm-only")
    ap.add_argument("--nf4-b8-small", action="store_true", help="small case: 2-layer 14B-shape NF4 batch-8 rounds")
    ap.add_argument("--trace", action="store_true", help="launch timeline of a round (needs SF_TRACE=1)")
    ap.add_argument("--nf4-only", action="store_true", help="only the 14B-shape NF4 workloads (batch 1 and 8)")
    ap.add_argument("--verify-small", action="store_true", help="small case: 2-layer 7B-shape verify rounds at 2048")
    args = ap.parse_args()
    globals()["N_NEW"] = args.tokens
    if args.gemm_only:
        run_gemm_only(args)
        return
    if args.nf4_b8_small:
        run_nf4_b8_small(args)
        return
    if args.verify_small:
        run_verify_small(args)
        return
    if args.nf4_only:
        import torch
        torch.cuda.set_device(0)
        import __graft_entry__ as g
        g.build()
        import greedy_speculative_decoding_gb300 as pkg
        b1, b8 = nf4_workload(pkg, _peaks()[0])
        print(json.dumps({"nf4_14b_b1": b1, "nf4_14b_b8": b8}))
        return
    if args.trace:
        run_trace(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
