"""Python face of the engine: argument marshalling over the C ABI.

PyTorch supplies device memory (weights, KV caches, workspace) and the
stream; the library does all the work. Method names follow the C calls.
"""

import ctypes

import numpy as np
import torch

from . import _lib as L

LAYER_TENSORS = ("ln1", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "ln2", "wg", "wu", "wd")
LINEAR = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def model_cfg(shape, wdtype: int = L.SF_WDTYPE_BF16) -> L.ModelCfg:
    """sf_model_cfg from any object with the shape attributes (layers, hidden,
    n_heads, n_kv_heads, head_dim, ffn, vocab, tied, qkv_bias, embed_ld,
    rope_theta, rms_eps)."""
    return L.ModelCfg(
        layers=shape.layers, hidden=shape.hidden, n_heads=shape.n_heads, n_kv_heads=shape.n_kv_heads,
        head_dim=shape.head_dim, ffn=shape.ffn, vocab=shape.vocab, tied=int(bool(shape.tied)),
        qkv_bias=int(bool(shape.qkv_bias)), embed_ld=int(getattr(shape, "embed_ld", 0) or 0),
        rope_theta=float(shape.rope_theta), rms_eps=float(shape.rms_eps), wdtype=wdtype)


def weight_order(shape, nf4: bool = False) -> list:
    """Names in the order of the C ABI's weight pointer array. With NF4 each
    linear map `w` is followed by its block scales `w.scales`."""
    names = ["embed"]
    for i in range(shape.layers):
        for t in LAYER_TENSORS:
            names.append(f"layers.{i}.{t}")
            if nf4 and t in LINEAR:
                names.append(f"layers.{i}.{t}.scales")
    names.append("norm")
    if not shape.tied:
        names.append("lm_head")
    return names


def is_nf4(weights: dict) -> bool:
    return any(k.endswith(".scales") for k in weights)


def is_f32(weights: dict) -> bool:
    e = weights.get("embed")
    return e is not None and e.dtype == torch.float32


def wdtype_of(weights: dict) -> int:
    """SF_WDTYPE_* of a weight dict: NF4 when block scales are present, fp32
    when the tensors are float32, else bf16."""
    if is_nf4(weights):
        return L.SF_WDTYPE_NF4
    return L.SF_WDTYPE_F32 if is_f32(weights) else L.SF_WDTYPE_BF16


def _ptr_array(shape, weights: dict):
    nf4 = is_nf4(weights)
    f32 = is_f32(weights)
    names = weight_order(shape, nf4)
    arr = (ctypes.c_void_p * len(names))()
    keep = []
    for i, n in enumerate(names):
        t = weights.get(n)
        if t is None:
            arr[i] = None
            continue
        want = torch.float32 if f32 else torch.bfloat16
        if nf4 and n.split(".")[-1] in LINEAR:
            want = torch.uint8
        elif n.endswith(".scales"):
            want = torch.float16
        if not t.is_cuda or t.dtype != want:
            raise ValueError(f"{n}: expected a {want} CUDA tensor, got {t.dtype} on {t.device}")
        if t.dim() == 2 and t.stride(1) != 1:
            raise ValueError(f"{n}: rows must be contiguous")
        if n == "embed":
            ld = int(getattr(shape, "embed_ld", 0) or 0) or shape.hidden
            if t.stride(0) != ld:
                raise ValueError(f"embed: row stride {t.stride(0)} != embed_ld {ld}")
        elif not t.is_contiguous():
            raise ValueError(f"{n}: must be contiguous")
        arr[i] = t.data_ptr()
        keep.append(t)
    return arr, keep


def _i32(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class SpecEngine:
    """Greedy speculative decoding engine for one target and an optional
    draft model (without one, prompt lookup drafts).

    Weight dicts map the canonical names (embed, layers.i.*, norm, lm_head)
    to CUDA tensors that must outlive the engine: bf16, fp32 (every tensor),
    or bf16 with NF4 codes + scales for the linear maps.
    """

    def __init__(self, target_shape, target_w: dict, draft_shape=None, draft_w=None, batch: int = 1,
                 K: int = 8, s_max: int = 4096, stream=None):
        self.lib = L.load()
        self.B, self.K, self.s_max = batch, K, s_max
        self.target_shape, self.draft_shape = target_shape, draft_shape
        self.tc = model_cfg(target_shape, wdtype_of(target_w))
        self.dc = None
        if draft_shape is not None:
            self.dc = model_cfg(draft_shape, wdtype_of(draft_w))
        pdc = ctypes.byref(self.dc) if self.dc is not None else None
        ws = self.lib.sf_workspace_bytes(ctypes.byref(self.tc), pdc, batch, K, s_max)
        if ws == 0:
            raise L.SFError(L.SF_ERR_ARG, "sf_workspace_bytes rejected the configuration")
        dev = torch.device("cuda", torch.cuda.current_device())
        self.kv_t = torch.empty(self.lib.sf_kv_bytes(ctypes.byref(self.tc), batch, s_max), dtype=torch.uint8,
                                device=dev)
        self.kv_d = None
        if self.dc is not None:
            self.kv_d = torch.empty(self.lib.sf_kv_bytes(ctypes.byref(self.dc), batch, s_max),
                                    dtype=torch.uint8, device=dev)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        tw, self._keep_t = _ptr_array(target_shape, target_w)
        dw, self._keep_d = (None, [])
        if draft_shape is not None:
            dw, self._keep_d = _ptr_array(draft_shape, draft_w)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = ctypes.c_void_p()
        L.check(self.lib.sf_create(ctypes.byref(self.tc), tw, pdc, dw, batch, K, s_max,
                                   self.kv_t.data_ptr(), None if self.kv_d is None else self.kv_d.data_ptr(),
                                   self.ws.data_ptr(), ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h)))
        self.h = h
        self._tw, self._dw = tw, dw

    # ------------------------------------------------------------ lifecycle
    def close(self):
        if getattr(self, "h", None):
            self.lib.sf_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ the calls
    def prefill(self, prompts):
        """prompts: one token list per sequence; lengths may differ."""
        if len(prompts) != self.B:
            raise ValueError(f"expected {self.B} prompts, got {len(prompts)}")
        lens = np.array([len(q) for q in prompts], dtype=np.int32)
        width = int(lens.max())
        p = np.zeros((self.B, width), np.int32)
        for b, q in enumerate(prompts):
            p[b, :len(q)] = np.asarray(q, dtype=np.int32)
        L.check(self.lib.sf_prefill(self.h, _i32(p), _i32(lens), width))
        self.prompt_len = lens.copy()

    def draft(self, out: torch.Tensor = None, logits: torch.Tensor = None):
        L.check(self.lib.sf_draft(self.h, None if out is None else out.data_ptr(),
                                  None if logits is None else logits.data_ptr()))

    def ngram_draft(self, max_guess: int, min_n: int = 2, max_n: int = 4, prop: torch.Tensor = None,
                    count: torch.Tensor = None):
        L.check(self.lib.sf_ngram_draft(self.h, max_guess, min_n, max_n,
                                        None if prop is None else prop.data_ptr(),
                                        None if count is None else count.data_ptr()))

    def tree_draft(self, n_cand: int, min_n: int = 2, max_n: int = 4, prop: torch.Tensor = None,
                   lens: torch.Tensor = None):
        """Up to n_cand prompt-lookup guesses of K // n_cand tokens, verified
        side by side by the next verify; prop int32 [batch][n_cand][K // n_cand],
        lens int32 [batch][n_cand] (optional device outputs)."""
        L.check(self.lib.sf_tree_draft(self.h, n_cand, min_n, max_n,
                                       None if prop is None else prop.data_ptr(),
                                       None if lens is None else lens.data_ptr()))

    def set_tree_candidates(self, n_cand: int):
        L.check(self.lib.sf_set_tree_candidates(self.h, n_cand))

    def tree_winner(self):
        """The candidate each sequence's last multi-candidate round took."""
        c = np.zeros(self.B, np.int32)
        L.check(self.lib.sf_tree_winner(self.h, _i32(c)))
        return c

    def verify(self, argmax: torch.Tensor = None, logits: torch.Tensor = None):
        L.check(self.lib.sf_verify(self.h, None if argmax is None else argmax.data_ptr(),
                                   None if logits is None else logits.data_ptr()))

    def accept_rollback(self):
        n_acc = np.zeros(self.B, np.int32)
        com = np.zeros((self.B, self.K + 1), np.int32)
        n_com = np.zeros(self.B, np.int32)
        L.check(self.lib.sf_accept_rollback(self.h, _i32(n_acc), _i32(com), _i32(n_com)))
        return n_acc, [com[b, :n_com[b]].tolist() for b in range(self.B)]

    def step(self):
        com = np.zeros((self.B, self.K + 1), np.int32)
        n_com = np.zeros(self.B, np.int32)
        L.check(self.lib.sf_step(self.h, _i32(n_com), _i32(com)))
        return [com[b, :n_com[b]].tolist() for b in range(self.B)]

    def generate(self, n_new: int, out: np.ndarray = None):
        """Returns (tokens int32 [batch][n_new], rounds run)."""
        if out is None:
            out = np.zeros((self.B, n_new), np.int32)
        rounds = ctypes.c_int32(0)
        L.check(self.lib.sf_generate(self.h, n_new, _i32(out), ctypes.byref(rounds)))
        return out, rounds.value

    def reset(self):
        L.check(self.lib.sf_reset(self.h))

    def set_drafter(self, mode: int, min_n: int = 2, max_n: int = 4):
        L.check(self.lib.sf_set_drafter(self.h, mode, min_n, max_n))

    def lengths(self):
        lt = np.zeros(self.B, np.int32)
        ld = np.zeros(self.B, np.int32)
        L.check(self.lib.sf_get_lengths(self.h, _i32(lt), _i32(ld)))
        return lt, ld

    def accept_hist(self):
        hst = np.zeros((self.B, self.K + 1), np.int32)
        L.check(self.lib.sf_get_accept_hist(self.h, _i32(hst)))
        return hst

    def round_launches(self) -> int:
        """Kernel launches in one replay of the round graph (0 before it is built)."""
        return int(self.lib.sf_round_launches(self.h))

    def trace_count(self) -> int:
        """Launches enqueued so far (SF_TRACE=1), the id the next one gets."""
        return self.lib.sf_trace(self.h, None, 0)

    def trace(self, first: int = 0, count: int = None):
        """Launch timeline recorded with SF_TRACE=1 for launch ids first ..
        first + count - 1: list of (label, start_ns, wait_done_ns)."""
        slots = 8192
        buf = (ctypes.c_uint64 * (2 * slots))()
        n = self.lib.sf_trace(self.h, buf, slots)
        if count is None:
            count = min(n, slots)
        out = []
        for i in range(first, first + count):
            j = i % slots
            out.append((self.lib.sf_trace_label(self.h, j).decode(), buf[2 * j], buf[2 * j + 1]))
        return out

    # ------------------------------------------------------------ views
    def kv_view(self, which: str = "target") -> torch.Tensor:
        """[layers][2][batch][n_kv_heads][s_max][head_dim] bf16 view of a cache."""
        shape = self.target_shape if which == "target" else self.draft_shape
        buf = self.kv_t if which == "target" else self.kv_d
        return buf.view(torch.bfloat16).view(shape.layers, 2, self.B, shape.n_kv_heads, self.s_max,
                                              shape.head_dim)


def linear(w: torch.Tensor, x: torch.Tensor, out: torch.Tensor = None, workspace: torch.Tensor = None,
           stream=None) -> torch.Tensor:
    """y = x @ w.T through sf_linear: w bf16 CUDA [N, K] (row stride ld),
    x fp32 CUDA [M, K] with M <= 16. Returns fp32 [M, N]."""
    lib = L.load()
    N, K = w.shape
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(lib.sf_linear_workspace_bytes(N, K), dtype=torch.uint8, device=x.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    L.check(lib.sf_linear(w.data_ptr(), N, K, w.stride(0), x.data_ptr(), M, out.data_ptr(), workspace.data_ptr(),
                          ctypes.c_void_p(st.cuda_stream)))
    return out


def to_frag(x: torch.Tensor, stream=None) -> torch.Tensor:
    """fp32 CUDA rows x [M, K] -> the fragment-ordered bf16 hi/lo copy the
    projections read (uint8 buffer of sf_frag_bytes(K, M) bytes)."""
    lib = L.load()
    M, K = x.shape
    out = torch.empty(lib.sf_frag_bytes(K, M), dtype=torch.uint8, device=x.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    L.check(lib.sf_to_frag(x.data_ptr(), M, K, x.stride(0), out.data_ptr(), ctypes.c_void_p(st.cuda_stream)))
    return out


def linear_frag(w: torch.Tensor, xf: torch.Tensor, M: int, out: torch.Tensor = None,
                workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """y = x @ w.T from the fragment-ordered copy xf = to_frag(x) of M rows."""
    lib = L.load()
    N, K = w.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=w.device)
    if workspace is None:
        workspace = torch.empty(lib.sf_linear_workspace_bytes(N, K), dtype=torch.uint8, device=w.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    L.check(lib.sf_linear_frag(w.data_ptr(), N, K, w.stride(0), xf.data_ptr(), M, out.data_ptr(),
                               workspace.data_ptr(), ctypes.c_void_p(st.cuda_stream)))
    return out


def nf4_scale_ld(cols: int) -> int:
    """Row stride (in scales) of the NF4 block-scale matrix: cols/64 rounded up to 8."""
    return (cols // 64 + 7) // 8 * 8


def nf4_quantize(w: torch.Tensor, stream=None):
    """Blockwise NF4 codes [rows, cols/2] and fp16 scales [rows, nf4_scale_ld(cols)]
    (padding zero) of a bf16 CUDA matrix (cols % 64 == 0)."""
    lib = L.load()
    rows, cols = w.shape
    packed = torch.empty((rows, cols // 2), dtype=torch.uint8, device=w.device)
    scales = torch.zeros((rows, nf4_scale_ld(cols)), dtype=torch.float16, device=w.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    L.check(lib.sf_nf4_quantize(w.data_ptr(), rows, cols, w.stride(0), packed.data_ptr(), scales.data_ptr(),
                                ctypes.c_void_p(st.cuda_stream)))
    return packed, scales


def quantize_model_nf4(shape, weights: dict, stream=None) -> dict:
    """NF4 copy of a bf16 weight dict: every linear map becomes codes + scales
    (quantised on the GPU); embedding, norms, biases and LM head stay bf16."""
    out = {}
    for k, v in weights.items():
        if v is not None and k.split(".")[-1] in LINEAR:
            out[k], out[k + ".scales"] = nf4_quantize(v, stream)
        else:
            out[k] = v
    return out
