"""Windowed attention kernels (forward, backward) against the float64 oracle.

Geometries cover: no cache (first chunk), a cache that wraps around its k slots,
chunk starts that are not multiples of 128, ragged query/key tiles, every head
width the kernels support, and the hi/lo split mode.  Cache slots that hold no
visible position are filled with finite garbage so masking errors show.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402
from oracle import ttt_oracle as O  # noqa: E402

dev = "cuda"
LN2 = math.log(2.0)


def to_dev(x, split):
    x32 = torch.tensor(np.ascontiguousarray(x, np.float32), device=dev)
    hi = x32.to(torch.bfloat16)
    lo = (x32 - hi.float()).to(torch.bfloat16) if split else None
    val = hi.double() + (lo.double() if split else 0)
    return hi, lo, val.cpu().numpy()


def heads(x, H):
    n, d = x.shape
    return x.reshape(n, H, d // H).transpose(1, 0, 2)


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


CASES = [  # n, H, dh, window, pos0, split
    (128, 2, 64, 256, 0, False),
    (200, 3, 96, 256, 384, False),
    (256, 2, 128, 512, 1000, False),
    (64, 4, 32, 128, 64, False),
    (64, 4, 32, 128, 448, True),
    (100, 2, 64, 128, 300, True),
    (37, 2, 64, 256, 700, False),
    (512, 2, 96, 1024, 1500, False),   # two 256-query blocks, cache wraps, unaligned start
    (384, 2, 64, 512, 640, False),     # second block half full
    # the benchmark's geometry: a trainable-block step (1024 queries, 72 key tiles per query
    # tile, full 8192-slot cache) at head widths 96 (760M) and 128 (3B), and a frozen-block
    # pass (8192 queries starting at a multiple of the window)
    (1024, 2, 96, 8192, 20000, False),
    (1024, 1, 128, 8192, 20000, False),
    (8192, 1, 96, 8192, 16384, False),
]


@pytest.mark.parametrize("n,H,dh,window,pos0,split", CASES)
def test_attention_forward_backward(n, H, dh, window, pos0, split):
    rng = np.random.default_rng(n * 7 + dh + pos0)
    d = H * dh
    q = rng.standard_normal((n, d))
    ko, vo = rng.standard_normal((2, n, d))
    kc, vc = rng.standard_normal((2, window, d)) * 3.0      # garbage everywhere ...
    cpos = np.arange(max(0, pos0 - window), pos0)            # ... then the visible cache
    kc_true, vc_true = rng.standard_normal((2, len(cpos), d))
    kc[cpos % window] = kc_true
    vc[cpos % window] = vc_true
    dO = rng.standard_normal((n, d))

    dq_, dql, qv = to_dev(q, split)
    kch, kcl, kcv = to_dev(kc, split)
    vch, vcl, vcv = to_dev(vc, split)
    koh, kol, kov = to_dev(ko, split)
    voh, vol, vov = to_dev(vo, split)
    doh, dol, dov = to_dev(dO, split)
    o_hi = torch.zeros((n, d), dtype=torch.bfloat16, device=dev)
    o_lo = torch.zeros_like(o_hi) if split else None
    lse = torch.zeros((H, n), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lo = dict(q=dql, kc=kcl, vc=vcl, ko=kol, vo=vol, o=o_lo, do=dol) if split else None
    T.attn_fwd(n, H, dh, window, pos0, dq_, kch, vch, koh, voh, o_hi, lse, split=split, lo=lo, err=err)

    D = torch.zeros((H, n), dtype=torch.float32, device=dev)
    T.attn_rowdot(n, H, dh, doh, o_hi, D, do_lo=dol, o_lo=o_lo)
    g = [torch.zeros((n, d), dtype=torch.float32, device=dev) for _ in range(3)]
    T.attn_bwd(n, H, dh, window, pos0, dq_, kch, vch, koh, voh, doh, lse, D, *g, split=split, lo=lo, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # oracle on the same (rounded) values
    qpos = pos0 + np.arange(n)
    kpos = np.concatenate([cpos, qpos])
    kall = np.concatenate([kcv[cpos % window], kov])
    vall = np.concatenate([vcv[cpos % window], vov])
    Qh, Kh, Vh = heads(qv, H), heads(kall, H), heads(vall, H)
    o_ref, lse_ref = O.attention(Qh, Kh, Vh, qpos, kpos, window)
    o_got = o_hi.double().cpu().numpy() + (o_lo.double().cpu().numpy() if split else 0)
    tol_o = 3e-5 if split else 6e-3
    assert rel(heads(o_got, H), o_ref) < tol_o
    assert np.max(np.abs(lse.double().cpu().numpy() * LN2 - lse_ref)) < 1e-4

    dq_ref, dk_ref, dv_ref = O.attention_bwd(heads(dov, H), Qh, Kh, Vh, qpos, kpos, window)
    tol_g = 1e-4 if split else 1.5e-2
    got = [heads(t.double().cpu().numpy(), H) for t in g]
    assert rel(got[0], dq_ref) < tol_g, "dq"
    assert rel(got[1], dk_ref[:, -n:]) < tol_g, "dk"
    assert rel(got[2], dv_ref[:, -n:]) < tol_g, "dv"
