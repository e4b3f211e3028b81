"""Failure detection on the GPU without a fault: a bounded wait runs out.

ttt_k_wait_limit_probe makes two threads of one CTA wait on an mbarrier phase
that nothing completes, through the same bounded wait every kernel uses.  The
first waiter must give up after the wait limit, raise the CTA's abort flag and
record its code in the error word; the second, started 100 ms later, must stop
at the flag before its own limit and leave the word alone.  The context must
stay usable afterwards.
"""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402

WAIT_LIMIT_MS = 4000        # the library's bounded-wait limit
TIMEOUT_EPILOGUE = 3        # device error code of an epilogue-side wait that ran out


def test_expired_wait_reports_and_stops_the_cta():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    T.wait_limit_probe(err, status)
    torch.cuda.synchronize()
    ok0, ms0, ok1, ms1 = status.cpu().tolist()
    assert (ok0, ok1) == (0, 0)
    assert int(err.item()) == TIMEOUT_EPILOGUE
    assert WAIT_LIMIT_MS <= ms0 < WAIT_LIMIT_MS + 1000, ms0
    assert ms1 < WAIT_LIMIT_MS, ms1            # stopped by the abort flag, not by its own limit
    # the context is still usable
    x = torch.ones(1 << 20, device="cuda", dtype=torch.float32)
    assert float((2 * x).sum().item()) == float(1 << 21)


def test_null_pointers_are_rejected():
    with pytest.raises(T.TTTError):
        T.wait_limit_probe(None, None)
