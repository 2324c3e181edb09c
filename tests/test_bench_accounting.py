"""The byte counts behind every roofline fraction bench.py prints, checked
on the CPU against independent derivations:

* weight_bytes: the sum of the streamed tensors' sizes as the synthetic
  model defines them (weight_shape), bf16, plus the LM head (the tied
  embedding's first `hidden` columns for the draft);
* the 7B and 0.5B shapes against the published sizes of the models they
  imitate (Qwen2.5-7B: 7.61 B parameters of which 6.53 B outside the
  embeddings; Qwen2.5-0.5B: 0.49 B with tied embeddings), so a wrong
  dimension in a shape cannot hide behind a matching formula;
* kv_bytes: 56 KiB of bf16 keys and values per cached token for the 7B
  shape (28 layers x 4 KV heads x 128 dimensions x 2 tensors x 2 bytes);
* the per-launch bytes of the timeline rows and the verify/draft step totals
  the bench reports (14.26 GB and 1.01 GB at context 2048).
"""

import pytest

import bench
from synth import QWEN05B, QWEN05B_SHARED, QWEN7B, QWEN14B
from synth.shapes import LAYER_TENSORS, weight_shape

LINEAR = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def _streamed_bytes(shape):
    """bf16 bytes one forward streams: every layer's linear maps and the LM
    head (vocab rows of `hidden` features, tied or not)."""
    n = 0
    for t in LAYER_TENSORS:
        if t in LINEAR:
            r, c = weight_shape(shape, f"layers.0.{t}")
            n += r * c
    n *= shape.layers
    v, h = weight_shape(shape, "lm_head")
    return 2 * (n + v * h)


@pytest.mark.parametrize("shape", [QWEN7B, QWEN05B_SHARED, QWEN14B], ids=["7b", "05b_shared", "14b"])
def test_weight_bytes_equal_the_streamed_tensors(shape):
    assert bench.weight_bytes(shape) == _streamed_bytes(shape)


def test_shapes_match_the_published_model_sizes():
    # Qwen2.5-7B: 7.61 B parameters, 6.53 B without the embeddings.
    total = QWEN7B.n_params()
    non_emb = total - 2 * QWEN7B.vocab * QWEN7B.hidden
    assert abs(total / 1e9 - 7.61) < 0.01
    assert abs(non_emb / 1e9 - 6.53) < 0.01
    # Qwen2.5-0.5B: 0.49 B parameters (embedding tied with the LM head).
    assert abs(QWEN05B.n_params() / 1e9 - 0.49) < 0.01


def test_kv_bytes_per_token_and_at_context():
    per_token = 28 * 4 * 128 * 2 * 2
    assert per_token == 56 * 1024
    assert bench.kv_bytes(QWEN7B, 0, 1) == per_token
    assert bench.kv_bytes(QWEN7B, 2048, 9) == per_token * 2057
    # The draft: 24 layers x 2 KV heads x 64 dimensions x 2 tensors x 2 bytes.
    assert bench.kv_bytes(QWEN05B_SHARED, 2048, 1) == 12 * 1024 * 2049


def test_step_totals_as_reported():
    v = bench.weight_bytes(QWEN7B) + bench.kv_bytes(QWEN7B, bench.VERIFY_CTX, bench.K_GUESS + 1)
    d = bench.weight_bytes(QWEN05B_SHARED) + bench.kv_bytes(QWEN05B_SHARED, bench.VERIFY_CTX, 1)
    assert v == 14_258_528_256   # the verify step's 14.26 GB
    assert d == 1_013_329_920    # the draft step's 1.01 GB


def test_kernel_bytes_of_the_timeline_rows():
    kb = bench._kernel_bytes
    gu = 2 * 18944 * 3584 * 2
    assert kb(QWEN7B, "gate_up", 2048) == gu == 271_581_184
    assert kb(QWEN7B, "down", 2048) == gu // 2
    assert kb(QWEN7B, "qkv", 2048) == (3584 + 2 * 512) * 3584 * 2
    assert kb(QWEN7B, "o_proj", 2048) == 3584 * 3584 * 2
    assert kb(QWEN7B, "lm_head", 2048) == 152064 * 3584 * 2
    # One layer's keys and values at context 2048: 4 MiB.
    assert kb(QWEN7B, "attention", 2048) == 4 << 20
    # A phase of the persistent kernel counts like the kernel of its name;
    # the whole persistent forward is every layer's weights and cache.
    assert kb(QWEN05B_SHARED, "d_gate_up", 2048) == kb(QWEN05B_SHARED, "gate_up", 2048)
    per_layer = sum(kb(QWEN05B_SHARED, k, 2048) for k in ("qkv", "o_proj", "gate_up", "down", "attention"))
    assert kb(QWEN05B_SHARED, "decode", 2048) == 24 * per_layer
    assert kb(QWEN7B, "merge", 2048) is None


def test_launch_bound_per_round():
    # K draft forwards and one verify forward (embed + 6 per layer + LM
    # head each) and the acceptance kernel.
    assert bench.launches_per_round(QWEN7B, QWEN05B_SHARED, 8) == 8 * (2 + 6 * 24) + (2 + 6 * 28) + 1
