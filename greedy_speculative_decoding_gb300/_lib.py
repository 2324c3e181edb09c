"""ctypes binding of libsf.so (the C ABI in include/sf.h).

Argument marshalling only: every step of the decoding path runs in the CUDA
kernels behind this library. If the library is missing the import fails
loudly; there is no fallback.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsf.so")

SF_OK, SF_ERR_ARG, SF_ERR_CAPACITY, SF_ERR_CUDA, SF_ERR_NONFINITE, SF_ERR_STATE, SF_ERR_UNSUPPORTED, \
    SF_ERR_DEVICE = range(8)
SF_WDTYPE_BF16, SF_WDTYPE_NF4, SF_WDTYPE_F32 = 0, 1, 2
SF_DRAFT_NEURAL, SF_DRAFT_NGRAM, SF_DRAFT_NONE, SF_DRAFT_TREE = 0, 1, 2, 3
SF_MAX_ROWS = 80

EXPORTS = (
    "sf_weight_count", "sf_kv_bytes", "sf_workspace_bytes", "sf_create", "sf_prefill", "sf_draft",
    "sf_ngram_draft", "sf_verify", "sf_accept_rollback", "sf_step", "sf_generate", "sf_reset",
    "sf_set_drafter", "sf_get_lengths", "sf_get_accept_hist", "sf_status_str", "sf_last_error",
    "sf_destroy", "sf_nf4_quantize", "sf_linear_workspace_bytes", "sf_linear", "sf_linear_noalloc",
    "sf_trace", "sf_trace_label", "sf_frag_bytes", "sf_to_frag", "sf_linear_frag", "sf_round_launches",
    "sf_tree_draft", "sf_set_tree_candidates", "sf_tree_winner",
)


class ModelCfg(ctypes.Structure):
    _fields_ = [
        ("layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("tied", ctypes.c_int32), ("qkv_bias", ctypes.c_int32),
        ("embed_ld", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
        ("wdtype", ctypes.c_int32),
    ]


class SFError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsf.so (once). Raises if it is missing: build it first."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with `python -m greedy_speculative_decoding_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I32, SZ, ST = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_int
    PI32 = ctypes.POINTER(ctypes.c_int32)
    PCFG = ctypes.POINTER(ModelCfg)
    sig = {
        "sf_weight_count": (I32, [PCFG]),
        "sf_kv_bytes": (SZ, [PCFG, I32, I32]),
        "sf_workspace_bytes": (SZ, [PCFG, PCFG, I32, I32, I32]),
        "sf_create": (ST, [PCFG, P, PCFG, P, I32, I32, I32, P, P, P, P, ctypes.POINTER(P)]),
        "sf_prefill": (ST, [P, PI32, PI32, I32]),
        "sf_draft": (ST, [P, P, P]),
        "sf_ngram_draft": (ST, [P, I32, I32, I32, P, P]),
        "sf_verify": (ST, [P, P, P]),
        "sf_accept_rollback": (ST, [P, PI32, PI32, PI32]),
        "sf_step": (ST, [P, PI32, PI32]),
        "sf_generate": (ST, [P, I32, PI32, PI32]),
        "sf_reset": (ST, [P]),
        "sf_set_drafter": (ST, [P, I32, I32, I32]),
        "sf_get_lengths": (ST, [P, PI32, PI32]),
        "sf_get_accept_hist": (ST, [P, PI32]),
        "sf_status_str": (ctypes.c_char_p, [ST]),
        "sf_last_error": (ctypes.c_char_p, []),
        "sf_destroy": (None, [P]),
        "sf_nf4_quantize": (ST, [P, I32, I32, I32, P, P, P]),
        "sf_linear_workspace_bytes": (SZ, [I32, I32]),
        "sf_linear": (ST, [P, I32, I32, I32, P, I32, P, P, P]),
        "sf_linear_noalloc": (ST, [P, I32, I32, I32, P, I32, P, P]),
        "sf_trace": (I32, [P, ctypes.POINTER(ctypes.c_uint64), I32]),
        "sf_frag_bytes": (SZ, [I32, I32]),
        "sf_to_frag": (ST, [P, I32, I32, I32, P, P]),
        "sf_linear_frag": (ST, [P, I32, I32, I32, P, I32, P, P, P]),
        "sf_trace_label": (ctypes.c_char_p, [P, I32]),
        "sf_round_launches": (ctypes.c_int64, [P]),
        "sf_tree_draft": (ST, [P, I32, I32, I32, P, P]),
        "sf_set_tree_candidates": (ST, [P, I32]),
        "sf_tree_winner": (ST, [P, PI32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int):
    if status != SF_OK:
        lib = load()
        raise SFError(status, f"{lib.sf_status_str(status).decode()}: {lib.sf_last_error().decode()}")
