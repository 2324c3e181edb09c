"""sf_linear_noalloc: the projection for callers that cannot allocate device
memory (a host framework that owns every allocation, latency-critical loops
that cannot take cudaMalloc's implicit synchronisation). It must give the same result as
sf_linear with a caller-provided workspace, on consecutive calls that reuse
the library's static scratch, and refuse sizes beyond its limit.

Kept in a file of its own that is collected last.
"""

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-4   # of sum_k |x_k w_nk|, as in the sf_linear parity tests


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from greedy_speculative_decoding_gb300 import _lib as L
    return L.load()


def _run(lib, fn, w, x, y, ws=None):
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    N, K = w.shape
    M = x.shape[0]
    if ws is None:
        return fn(w.data_ptr(), N, K, w.stride(0), x.data_ptr(), M, y.data_ptr(), st)
    return fn(w.data_ptr(), N, K, w.stride(0), x.data_ptr(), M, y.data_ptr(), ws.data_ptr(), st)


@pytest.mark.parametrize("N,K,M", [(4608, 3584, 9), (3584, 18944, 1), (1000, 904, 16)])
def test_noalloc_matches_sf_linear_twice(lib, N, K, M):
    from greedy_speculative_decoding_gb300 import _lib as L
    g = torch.Generator(device="cuda").manual_seed(N + K + M)
    w = (torch.randn(N, K, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    x = torch.randn(M, K, generator=g, device="cuda")
    ws = torch.empty(lib.sf_linear_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    ref = torch.empty(M, N, device="cuda")
    assert _run(lib, lib.sf_linear, w, x, ref, ws) == L.SF_OK
    bound = (x.double().abs() @ w.double().abs().t())
    outs = []
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        assert _run(lib, lib.sf_linear_noalloc, w, x, y) == L.SF_OK, lib.sf_last_error()
        torch.cuda.synchronize()
        err = (y.double() - ref.double()).abs()
        assert bool((err <= TOL * bound).all())
        outs.append(y)
    # The second call reuses the scratch left by the first one.
    assert torch.equal(outs[0], outs[1])


def test_noalloc_allocates_nothing_after_first_call(lib):
    from greedy_speculative_decoding_gb300 import _lib as L
    N, K, M = 3584, 3584, 4
    w = torch.randn(N, K, device="cuda").to(torch.bfloat16)
    x = torch.randn(M, K, device="cuda")
    y = torch.empty(M, N, device="cuda")
    assert _run(lib, lib.sf_linear_noalloc, w, x, y) == L.SF_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _run(lib, lib.sf_linear_noalloc, w, x, y) == L.SF_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_sizes_beyond_the_limit(lib):
    from greedy_speculative_decoding_gb300 import _lib as L
    w = torch.zeros(8, 64, device="cuda", dtype=torch.bfloat16)
    x = torch.zeros(1, 64, device="cuda")
    y = torch.zeros(1, 8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.sf_linear_noalloc(w.data_ptr(), (1 << 20) + 1, 64, 64, x.data_ptr(), 1, y.data_ptr(), st)
    assert rc == L.SF_ERR_ARG
    assert b"static scratch" in lib.sf_last_error()
    # N within its limit, but K one 64-wide chunk past what the scratch holds
    # for the operand copy: refused by the byte check (no launch happens).
    rc = lib.sf_linear_noalloc(w.data_ptr(), 1 << 20, 65600, 65600, x.data_ptr(), 1, y.data_ptr(), st)
    assert rc == L.SF_ERR_ARG
    assert b"static scratch" in lib.sf_last_error()
    rc = lib.sf_linear_noalloc(w.data_ptr(), 8, 60, 64, x.data_ptr(), 1, y.data_ptr(), st)
    assert rc == L.SF_ERR_ARG
    assert b"multiple of 8" in lib.sf_last_error()
