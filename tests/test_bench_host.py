"""Host-side arithmetic of bench.py: the FLOP count, the traffic weighting and the
size of the oracle sample.  No GPU needed."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from ttt_inputs import SHAPES  # noqa: E402


def brute_pairs(T, k):
    """Visible (query, key) pairs of a causal window of k keys over T tokens, counted one by one."""
    return sum(1 for p in range(T) for j in range(p + 1) if p - j < k)


@pytest.mark.parametrize("T,k", [(5, 8), (8, 8), (20, 8), (33, 16)])
def test_window_pairs_in_the_flop_count_match_brute_force(T, k):
    s = SHAPES["tiny"].replace(window=k)
    d, L, V = s.d_model, s.n_layers, s.vocab
    # the attention term of the forward is 4 d per visible pair and layer; isolate it by
    # differencing two window sizes that differ only in the pairs
    f_small = bench.algorithmic_flops(s.replace(window=1), T)
    f_k = bench.algorithmic_flops(s, T)
    extra_pairs = brute_pairs(T, k) - brute_pairs(T, 1)
    S = s.n_trainable
    assert f_k - f_small == 4 * d * extra_pairs * L + (S - 1) * 4 * d * extra_pairs
    assert V > 0


def test_attention_traffic_is_weighted_by_the_launch_mix():
    s = SHAPES["760m"]
    nc = s.seq_len // s.chunk
    t = bench.ATTN_FWD_TRAFFIC_760M
    G = min(8192 // s.chunk, s.window // s.chunk)
    passes = -(-nc // G) * (s.n_layers - s.n_trainable)
    steps = nc * s.n_trainable
    assert (passes, steps) == (16 * 18, 128 * 6)
    want = (passes * t["pass"] + steps * t["step"]) / (passes + steps)
    assert bench.attn_fwd_traffic(s, nc) == pytest.approx(want)
    # other shapes have no captured figure
    assert bench.attn_fwd_traffic(SHAPES["125m"], 8) is None


@pytest.mark.parametrize("steps,warmup,want", [(3, 3, 512), (1, 3, 1024), (10, 3, 256), (20, 5, 128),
                                               (200, 5, 64)])
def test_reference_sample_is_a_power_of_two_within_the_budget(steps, warmup, want):
    n = bench.reference_tokens(steps, warmup)
    assert n == want
    assert n & (n - 1) == 0 and 64 <= n <= 1024
    # more samples never get a larger sample
    assert bench.reference_tokens(steps + 10, warmup) <= n


@pytest.mark.parametrize("B,T,b", [(1, 10, 4), (4, 12, 4), (3, 7, 8), (2, 9, 3)])
def test_per_chunk_inputs_walk_every_sequence_chunk_by_chunk(B, T, b):
    import numpy as np
    tokens = np.arange(B * T, dtype=np.int32).reshape(B, T) + 100
    ids, nxt = bench.chunk_major(tokens, b)
    assert ids.size == B * T and nxt.shape == (-(-T // b), B)
    off = 0
    for c, s in enumerate(range(0, T, b)):
        n = min(b, T - s)
        block = ids[off:off + B * n].reshape(B, n)  # what one ttt_prefill_chunk call reads
        off += B * n
        assert (block == tokens[:, s:s + n]).all()
        for q in range(B):
            assert nxt[c, q] == (tokens[q, s + n] if s + n < T else -1)
