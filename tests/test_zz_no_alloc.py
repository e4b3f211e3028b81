"""The allocation-free LM-head cross-entropy entry point (ttt_k_lmhead_ce_static).

Some callers cannot call cudaMalloc: a process whose device memory is owned up
front by another allocator, or a latency-bound caller that cannot take
cudaMalloc's implicit device synchronisation.  For them the library keeps this
variant's scratch in a static device array.  This test checks, through the C
ABI, that two calls in a row give the same per-row log-sum-exp and loss as the
allocating path (ttt_k_gemm with the CE_FWD epilogue into caller scratch, its
partials combined here in float64) and as a float64 numpy computation from the
same bf16 inputs, within the tolerance of the GEMM tests; that the second call
leaves the device's free memory unchanged; and that a size beyond the static
capacity is refused.

The file sorts last so that a run stopping at the first failure has already
run every other test; it passes alone in a fresh process as well.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402

dev = "cuda"


def rel(x, y):
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30))


def reference_from_allocating_path(M, K, V, x, w, tgt):
    """lse / loss from ttt_k_gemm(CE_FWD) with caller-allocated partials.

    The partials are laid out [vocab tile][row]; every pair starts as (-inf, 0),
    so combining over the 128-wide tile count is right whichever tile width
    the library picks (tiles it does not write add exp(-inf) * 0 = 0).
    """
    ntiles = -(-V // 128)
    part = torch.zeros((ntiles * M, 2), dtype=torch.float32, device=dev)
    part[:, 0] = float("-inf")
    zt = torch.zeros(M, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    T.gemm(T.EPI_CE_FWD, M, V, K, x, w, b_mn=1, tgt=tgt, part=part, zt=zt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pm = part.cpu().numpy().astype(np.float64).reshape(ntiles, M, 2)
    t = tgt.cpu().numpy()
    mx = pm[:, :, 0].max(0)
    lse = mx + np.log((pm[:, :, 1] * np.exp(pm[:, :, 0] - mx)).sum(0))
    z_t = zt.cpu().numpy().astype(np.float64)
    loss = np.where(t >= 0, lse - z_t, 0.0)
    return lse, loss


def reference_float64(x, w, tgt):
    """lse = logsumexp(x . W) and loss = lse - z[tgt], in numpy float64 from the bf16 inputs."""
    z = x.double().cpu().numpy() @ w.double().cpu().numpy()
    m = z.max(1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(1))
    t = tgt.cpu().numpy()
    loss = np.where(t >= 0, lse - z[np.arange(len(t)), np.maximum(t, 0)], 0.0)
    return lse, loss


@pytest.mark.parametrize("M,K,V", [(300, 128, 1000), (1024, 768, 32000)])
def test_static_scratch_matches_allocating_path_twice(M, K, V):
    rng = np.random.default_rng(M + K + V)
    x = torch.tensor(rng.standard_normal((M, K)) * 0.5, dtype=torch.float32, device=dev).to(torch.bfloat16)
    w = torch.tensor(rng.standard_normal((K, V)) * 0.05, dtype=torch.float32, device=dev).to(torch.bfloat16)
    t = rng.integers(0, V, M).astype(np.int32)
    t[::7] = -1
    tgt = torch.tensor(t, device=dev)
    lse_ref, loss_ref = reference_from_allocating_path(M, K, V, x, w, tgt)
    lse64, loss64 = reference_float64(x, w, tgt)
    assert rel(lse_ref, lse64) < 1e-5 and rel(loss_ref, loss64) < 1e-5
    for call in range(2):
        free0, _ = torch.cuda.mem_get_info()
        lse = torch.full((M,), float("nan"), dtype=torch.float32, device=dev)
        loss = torch.full((M,), float("nan"), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        T.lmhead_ce_static(M, K, V, x, w, tgt, lse, loss, err=err)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        if call == 1:  # the array is in place after the first call: nothing is allocated any more
            assert free1 == free0, (free0, free1)
        assert int(err.item()) == 0
        got_lse = lse.cpu().numpy().astype(np.float64)
        got_loss = loss.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got_lse)) and np.all(np.isfinite(got_loss)), call
        assert rel(got_lse, lse_ref) < 1e-5, call
        assert rel(got_loss, loss_ref) < 1e-5, call
        assert rel(got_lse, lse64) < 1e-5 and rel(got_loss, loss64) < 1e-5, call
        assert np.all(got_loss[t < 0] == 0.0), call


def test_static_scratch_refuses_sizes_beyond_its_capacity():
    M, K, V = 1024, 64, 65536        # 512 tiles x 1024 rows + 512 > 524288 entries
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((K, V), dtype=torch.bfloat16, device=dev)
    tgt = torch.zeros(M, dtype=torch.int32, device=dev)
    lse = torch.zeros(M, dtype=torch.float32, device=dev)
    loss = torch.zeros(M, dtype=torch.float32, device=dev)
    with pytest.raises(T.TTTError) as e:
        T.lmhead_ce_static(M, K, V, x, w, tgt, lse, loss)
    assert e.value.code == T.TTT_ERR_SCRATCH
    # the largest vocabulary that fits 1024 rows is accepted
    V = 65408
    w = torch.zeros((K, V), dtype=torch.bfloat16, device=dev)
    T.lmhead_ce_static(M, K, V, x, w, tgt, lse, loss)
    torch.cuda.synchronize()
    assert np.allclose(lse.cpu().numpy(), np.log(V), rtol=1e-5)
