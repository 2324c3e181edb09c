"""GB300-native greedy speculative decoding.

One speculative round -- K draft guesses (a small draft model decoding
greedily, or prompt lookup), one causal verify pass of the target over the
pending token and the guesses, acceptance of the longest agreeing prefix plus
the target's bonus token, in-place rollback of both KV caches -- runs as
hand-written sm_103a CUDA kernels behind the C ABI in include/sf.h, replayed
as one CUDA graph per round.

``SpecEngine`` wraps that ABI; PyTorch only provides device memory and the
stream. The library is loaded on first use and its absence raises
ImportError (build it with ``python -m greedy_speculative_decoding_gb300.build``);
there is no fallback path.
"""

from . import _lib
from ._lib import (SF_DRAFT_NEURAL, SF_DRAFT_NGRAM, SF_DRAFT_NONE, SF_DRAFT_TREE, SF_MAX_ROWS, SFError, load)
from .engine import (SpecEngine, linear, linear_frag, model_cfg, nf4_quantize, nf4_scale_ld, quantize_model_nf4,
                     to_frag, weight_order)

__all__ = ["SpecEngine", "SFError", "linear", "linear_frag", "to_frag", "model_cfg", "weight_order",
           "nf4_quantize", "nf4_scale_ld",
           "quantize_model_nf4", "SF_DRAFT_NEURAL",
           "SF_DRAFT_NGRAM", "SF_DRAFT_NONE", "SF_DRAFT_TREE", "SF_MAX_ROWS"]
