"""GPU parity of the weight-streaming GEMM (sf_linear) against a float64
matrix product, over shapes that span several 128-row blocks and 64-wide K
chunks with ragged tails, every row count 1..16 (the mma.sync kernel), row
counts above 16 (the tcgen05 kernel: all rows in one tensor-memory
accumulator), and K splits across CTAs.

Error bound: up to 16 rows the activation is carried as a bf16 pair (hi +
lo, about 16 mantissa bits) and products are summed in fp32, so |y - y_ref|
stays within a small multiple of 2^-16 * sum_k |x_k w_nk|; the test allows
1e-4 of that sum. Above 16 rows the tensor-core kernel takes the activation
as one bf16 (relative rounding <= 2^-9 per element), so the bound is 2^-8 of
the same sum.
"""

TOL_SYNC, TOL_TC = 1e-4, 2.0 ** -8


def tol(M):
    return TOL_TC if M > 16 else TOL_SYNC

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import greedy_speculative_decoding_gb300 as p
    return p


def _check(pkg, N, K, M, ld=None, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    ld = ld or K
    wfull = (torch.randn(N, ld, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w = wfull[:, :K]
    x = torch.randn(M, K, generator=g, device="cuda")
    y = pkg.linear(w, x)
    torch.cuda.synchronize()
    wd, xd = w.double(), x.double()
    ref = xd @ wd.t()
    bound = xd.abs() @ wd.abs().t()
    err = (y.double() - ref).abs()
    assert bool((err <= tol(M) * bound + 1e-30).all()), float((err / bound).max())
    return float((err / bound).max())


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_rows_1_to_16(pkg, M):
    _check(pkg, N=1000, K=904, M=M, seed=M)


@pytest.mark.parametrize("N,K", [(128, 64), (129, 72), (4608, 3584), (3584, 18944), (896, 4864),
                                 (1024, 256), (688 * 2, 256), (256, 688), (5, 8)])
def test_shapes(pkg, N, K):
    _check(pkg, N=N, K=K, M=9)


def test_strided_rows(pkg):
    # rows of a wider matrix: a column slice, as the shared-embedding draft uses
    _check(pkg, N=700, K=896, M=2, ld=3584)


def test_deterministic_and_row_independent(pkg):
    g = torch.Generator(device="cuda").manual_seed(7)
    w = (torch.randn(3584, 18944, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    x = torch.randn(9, 18944, generator=g, device="cuda")
    y1 = pkg.linear(w, x)
    y2 = pkg.linear(w, x)
    assert torch.equal(y1, y2)
    for m in range(9):
        ym = pkg.linear(w, x[m:m + 1].contiguous())
        assert torch.equal(ym[0], y1[m]), m


@pytest.mark.parametrize("M", [17, 24, 33, 40, 72, 80])
def test_rows_above_16(pkg, M):
    _check(pkg, N=1000, K=904, M=M, seed=M)


@pytest.mark.parametrize("N,K,M", [(3584, 18944, 72), (4608, 3584, 40), (129, 72, 80), (896, 4864, 18)])
def test_tensor_core_rows(pkg, N, K, M):
    """Above 16 rows the tcgen05 kernel takes every row in one accumulator.
    Its results are deterministic, a row's bits do not depend on how many
    other rows (above 16) share the launch, and they agree with the 16-row
    mma.sync launches of the same rows within the bf16 rounding of the
    activations."""
    g = torch.Generator(device="cuda").manual_seed(N + K + M)
    w = (torch.randn(N, K, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    x = torch.randn(M, K, generator=g, device="cuda")
    y = pkg.linear(w, x)
    assert torch.equal(y, pkg.linear(w, x))
    assert torch.equal(pkg.linear(w, x[:17].contiguous()), y[:17])
    wd, xd = w.double(), x.double()
    bound = xd.abs() @ wd.abs().t()
    err = (y.double() - xd @ wd.t()).abs()
    assert bool((err <= TOL_TC * bound + 1e-30).all())
    for m0 in range(0, M, 16):
        part = pkg.linear(w, x[m0:m0 + 16].contiguous())
        assert bool(((part.double() - y[m0:m0 + 16].double()).abs() <= TOL_TC * bound[m0:m0 + 16] + 1e-30).all()), m0


def _frag_reference(x):
    """The operand layouts written out element by element (test-side
    restatement of what the header documents), as a uint16 array. Up to 16
    rows: fragment order, bf16 hi/lo pairs of x [M, K]; above 16: the
    tensor-core operand order, bf16 x in 128-byte rows of one token (8
    tokens per 1024-byte tile), piece q (features 8q..8q+7 of a chunk) of row
    m % 8 at position q ^ (m % 8)."""
    M, K = x.shape
    T = (M + 3) // 4 if M <= 16 else (M + 7) // 8
    nch = (K + 63) // 64
    out = torch.zeros(nch * T * 2 * 32 * 8, dtype=torch.int16)
    hi = x.to(torch.bfloat16)
    lo = (x - hi.float()).to(torch.bfloat16)
    hi16, lo16 = hi.view(torch.int16), lo.view(torch.int16)
    for m in range(M):
        for k in range(K):
            j, kk = divmod(k, 64)
            t = m // 4
            if M <= 16:
                c, h, e = kk // 16, (kk // 8) % 2, kk % 8
                col = 2 * (m % 4)
                unit = ((j * T + t) * 2 + h) * 32 + 4 * col + c
                out[unit * 8 + e] = hi16[m, k]
                out[(unit + 4) * 8 + e] = lo16[m, k]
            else:
                q, e, row = kk // 8, kk % 8, m % 8
                byte = (j * T + m // 8) * 1024 + row * 128 + ((q ^ row) << 4)
                out[byte // 2 + e] = hi16[m, k]
    return out


@pytest.mark.parametrize("M,K", [(1, 64), (3, 72), (9, 200), (16, 128), (40, 136), (72, 72)])
def test_to_frag_layout(pkg, M, K):
    g = torch.Generator(device="cuda").manual_seed(M * 1000 + K)
    x = torch.randn(M, K, generator=g, device="cuda")
    xf = pkg.to_frag(x)
    torch.cuda.synchronize()
    ref = _frag_reference(x.cpu())
    assert xf.numel() >= 2 * ref.numel()
    assert torch.equal(xf.cpu().view(torch.int16)[:ref.numel()], ref)


@pytest.mark.parametrize("N,K,M", [(37888, 3584, 9), (1000, 904, 3), (129, 72, 16), (5, 8, 1), (1000, 904, 72)])
def test_linear_frag_equals_linear(pkg, N, K, M):
    g = torch.Generator(device="cuda").manual_seed(N + K + M)
    w = (torch.randn(N, K, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    x = torch.randn(M, K, generator=g, device="cuda")
    ref = pkg.linear(w, x)
    y = pkg.linear_frag(w, pkg.to_frag(x), M)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
