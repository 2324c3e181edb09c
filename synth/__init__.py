"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This module holds model *shapes*, random weights, prompts and the draft
constructions used by the workloads. It contains none of the decoding
arithmetic: no norm, attention, argmax, acceptance or n-gram rule lives here.
Both sides receive the very same tensors from it.

Random numbers come from torch's seeded generators. One generator is seeded
per tensor (from the workload seed and the tensor's index in the canonical
weight order), so a tensor's values do not depend on which other tensors were
drawn first. Values drawn on the CPU and on a CUDA device differ for the same
seed (different generator algorithms): a test that needs one set of bytes on
both sides draws them once and copies them.
"""

from .shapes import (ModelShape, TINY_TARGET, TINY_DRAFT, QWEN05B, QWEN05B_SHARED,
                     QWEN7B, QWEN14B, weight_names)
from .weights import (make_weights, draft_from_target_layer0, perturbed_copy,
                      shared_embedding_draft, to_device)
from .prompts import uniform_prompt, ngram_prompt, repeated_fraction

__all__ = [
    "ModelShape", "TINY_TARGET", "TINY_DRAFT", "QWEN05B", "QWEN05B_SHARED", "QWEN7B",
    "QWEN14B", "weight_names", "make_weights", "draft_from_target_layer0",
    "perturbed_copy", "shared_embedding_draft", "to_device", "uniform_prompt",
    "ngram_prompt", "repeated_fraction",
]
