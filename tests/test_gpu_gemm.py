"""tcgen05 GEMM kernel (ttt_k_gemm) against float64 products of the same bf16 inputs.

Covers both operand majors for A and B, ragged M/N/K tails, both tile widths,
the hi/lo split mode and every fused epilogue.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402
from oracle import ttt_oracle as O  # noqa: E402

dev = "cuda"
RNG = np.random.default_rng(7)


def pad8(x):
    """Row-major copy whose row pitch is a multiple of 8 elements (TMA needs 16-B pitches)."""
    x = np.ascontiguousarray(x, np.float32)
    padc = (-x.shape[1]) % 8
    return np.pad(x, ((0, 0), (0, padc))) if padc else x


def bf(x):
    return torch.tensor(pad8(x)).to(dev).to(torch.bfloat16)


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def split(x):
    """fp32 -> (hi, lo) bf16 pair on the device."""
    x32 = torch.tensor(pad8(x), device=dev)
    hi = x32.to(torch.bfloat16)
    lo = (x32 - hi.float()).to(torch.bfloat16)
    return hi, lo


def operands(M, N, K, a_mn, b_mn, scale=1.0):
    A = RNG.standard_normal((M, K)) * scale
    B = RNG.standard_normal((N, K)) * scale
    a = bf(A.T if a_mn else A)
    b = bf(B.T if b_mn else B)
    Aq = f64(a)[:, :M].T if a_mn else f64(a)[:, :K]
    Bq = f64(b)[:, :N].T if b_mn else f64(b)[:, :K]
    return a, b, Aq, Bq


def rel(x, y):
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30))


def errword():
    return torch.zeros(1, dtype=torch.int32, device=dev)


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 200, 200), (1024, 1536, 512), (96, 4608, 160),
                                   (257, 520, 1030), (64, 200, 40)])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_f32_layouts(M, N, K, a_mn, b_mn):
    a, b, Aq, Bq = operands(M, N, K, a_mn, b_mn)
    out = torch.full((M, N + (-N) % 8), float("nan"), dtype=torch.float32, device=dev)
    err = errword()
    T.gemm(T.EPI_F32, M, N, K, a, b, a_mn=a_mn, b_mn=b_mn, out32=out, ldo32=out.shape[1], err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = Aq @ Bq.T
    got = out[:, :N].cpu().numpy().astype(np.float64)
    assert rel(got, ref) < 2e-6, (M, N, K, a_mn, b_mn)


# Shapes of the benchmark's size class, where the tile choice is 256 or 192 wide and each
# persistent CTA takes several tiles (1152 rows: an odd number of row tiles).
@pytest.mark.parametrize("M,N,K", [(1152, 4096, 320), (1024, 6144, 256), (2048, 1536, 1024)])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_wide_tiles(M, N, K, a_mn, b_mn):
    a, b, Aq, Bq = operands(M, N, K, a_mn, b_mn)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    err = errword()
    T.gemm(T.EPI_F32, M, N, K, a, b, a_mn=a_mn, b_mn=b_mn, out32=out, ldo32=N, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert rel(got, Aq @ Bq.T) < 2e-6, (M, N, K, a_mn, b_mn)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 1), (1, 1), (0, 0)])
def test_gemm_split_mode_fp32_accuracy(a_mn, b_mn):
    M, N, K = 200, 320, 384
    A = RNG.standard_normal((M, K))
    B = RNG.standard_normal((N, K))
    ah, al = split(A.T if a_mn else A)
    bh, bl = split(B.T if b_mn else B)
    out = torch.zeros((M, N), dtype=torch.float32, device=dev)
    err = errword()
    T.gemm(T.EPI_F32, M, N, K, ah, bh, a_lo=al, b_lo=bl, a_mn=a_mn, b_mn=b_mn, split=True,
           out32=out, ldo32=N, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    A32 = A.astype(np.float32).astype(np.float64)
    B32 = B.astype(np.float32).astype(np.float64)
    assert rel(out.cpu().numpy(), A32 @ B32.T) < 3e-5


def test_gemm_epilogues():
    M, N, K = 192, 384, 256
    a, b, Aq, Bq = operands(M, N, K, 0, 1, scale=0.5)
    acc = Aq @ Bq.T
    err = errword()
    # OPND (hi/lo)
    oh = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    ol = torch.zeros_like(oh)
    T.gemm(T.EPI_OPND, M, N, K, a, b, b_mn=1, out_hi=oh, out_lo=ol, ldo=N, err=err)
    # RESID in place
    x = torch.tensor(RNG.standard_normal((M, N)), dtype=torch.float32, device=dev)
    x0 = x.cpu().numpy().astype(np.float64)
    T.gemm(T.EPI_RESID, M, N, K, a, b, b_mn=1, out32=x, ldo32=N, resid=x, ldr=N, err=err)
    # GELU
    pre = torch.zeros((M, N), dtype=torch.float32, device=dev)
    gh = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    gl = torch.zeros_like(gh)
    T.gemm(T.EPI_GELU, M, N, K, a, b, b_mn=1, out32=pre, ldo32=N, out_hi=gh, out_lo=gl, ldo=N, err=err)
    # GELU_BWD with aux
    aux = torch.tensor(RNG.standard_normal((M, N)), dtype=torch.float32, device=dev)
    dh = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    dl = torch.zeros_like(dh)
    T.gemm(T.EPI_GELU_BWD, M, N, K, a, b, b_mn=1, aux=aux, ldaux=N, out_hi=dh, out_lo=dl, ldo=N, err=err)
    # SGD
    w = torch.tensor(RNG.standard_normal((M, N)) * 0.02, dtype=torch.float32, device=dev)
    w0 = w.cpu().numpy().astype(np.float64)
    wh = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    wl = torch.zeros_like(wh)
    T.gemm(T.EPI_SGD, M, N, K, a, b, b_mn=1, w32=w, w_hi=wh, w_lo=wl, ldw=N, eta=1e-3, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert rel(f64(oh) + f64(ol), acc) < 1e-5     # hi+lo keeps ~2^-17 of the fp32 value
    assert rel(f64(oh), acc) < 4e-3
    assert rel(x.cpu().numpy(), x0 + acc) < 2e-6
    assert rel(pre.cpu().numpy(), acc) < 2e-6
    assert rel(f64(gh) + f64(gl), O.gelu_tanh(acc)) < 1e-5
    assert rel(f64(dh) + f64(dl), acc * O.gelu_tanh_grad(aux.cpu().numpy().astype(np.float64))) < 1e-5
    wn = w.cpu().numpy().astype(np.float64)
    assert rel(wn, w0 - 1e-3 * acc) < 1e-6
    assert rel(f64(wh) + f64(wl), wn) < 1e-5


@pytest.mark.parametrize("N", [512, 1000])
def test_gemm_cross_entropy_epilogues(N):
    M, K = 300, 128
    a, b, Aq, Bq = operands(M, N, K, 0, 1)
    z = Aq @ Bq.T
    tgt = RNG.integers(0, N, M).astype(np.int32)
    tgt[::7] = -1
    tg = torch.tensor(tgt, device=dev)
    bn = 128 if N <= 128 else 256
    ntiles = max(1, -(-N // 256))
    part = torch.zeros((ntiles + 4) * M * 2, dtype=torch.float32, device=dev)
    zt = torch.zeros(M, dtype=torch.float32, device=dev)
    err = errword()
    T.gemm(T.EPI_CE_FWD, M, N, K, a, b, b_mn=1, tgt=tg, part=part, zt=zt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    p = part.cpu().numpy().reshape(-1, 2)
    # combine the per-tile (max, sum) pairs; the tile width is 128 or 256
    for width in (256, 128):
        nt = -(-N // width)
        pm = p[:nt * M].reshape(nt, M, 2)
        mx = pm[:, :, 0].max(0)
        lse = mx + np.log((pm[:, :, 1] * np.exp(pm[:, :, 0] - mx)).sum(0))
        if np.all(np.isfinite(lse)) and rel(lse, np.log(np.exp(z).sum(1))) < 1e-5:
            break
    else:
        raise AssertionError("partials do not combine to the log-sum-exp")
    ok = tgt >= 0
    assert rel(zt.cpu().numpy()[ok], z[np.nonzero(ok)[0], tgt[ok]]) < 2e-6
    # backward: (softmax - onehot) * scale from a given lse
    lse_t = torch.tensor(np.log(np.exp(z).sum(1)), dtype=torch.float32, device=dev)
    dh = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    dl = torch.zeros_like(dh)
    T.gemm(T.EPI_CE_BWD, M, N, K, a, b, b_mn=1, tgt=tg, lse=lse_t, scale=1.0 / ok.sum(), out_hi=dh, out_lo=dl,
           ldo=N, err=err)
    torch.cuda.synchronize()
    sm = np.exp(z - np.log(np.exp(z).sum(1, keepdims=True)))
    ref = sm.copy()
    ref[np.nonzero(ok)[0], tgt[ok]] -= 1
    ref[~ok] = 0
    ref /= ok.sum()
    assert rel(f64(dh) + f64(dl), ref) < 1e-5


@pytest.mark.parametrize("M,N,K,a_mn", [(1024, 1536, 6144, 0), (1024, 768, 32000, 0), (300, 200, 2048, 1)])
def test_gemm_k_slices_f32_and_residual(M, N, K, a_mn):
    """Under-filled products cut into K slices whose partial sums are added atomically."""
    a, b, Aq, Bq = operands(M, N, K, a_mn, 1, scale=0.25)
    ref = Aq @ Bq.T
    err = errword()
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)   # cleared by the call
    T.gemm(T.EPI_F32, M, N, K, a, b, a_mn=a_mn, b_mn=1, out32=out, ldo32=N, allow_ksplit=1, err=err)
    x = torch.tensor(RNG.standard_normal((M, N)), dtype=torch.float32, device=dev)
    x0 = x.cpu().numpy().astype(np.float64)
    T.gemm(T.EPI_RESID, M, N, K, a, b, a_mn=a_mn, b_mn=1, out32=x, ldo32=N, resid=x, ldr=N, allow_ksplit=1,
           err=err)                                                           # in place
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    T.gemm(T.EPI_RESID, M, N, K, a, b, a_mn=a_mn, b_mn=1, out32=y, ldo32=N, resid=x, ldr=N, allow_ksplit=1,
           err=err)                                                           # out != resid
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    tol = 1e-6 + 6e-10 * K              # fp32 accumulation of K exact bf16 products (TMEM, then slices)
    assert rel(out.cpu().numpy(), ref) < tol
    assert rel(x.cpu().numpy(), x0 + ref) < tol
    assert rel(y.cpu().numpy(), x0 + 2 * ref) < tol
