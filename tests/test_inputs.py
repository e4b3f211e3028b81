"""Seeded synthetic inputs: determinism, Zipf(1.1) shape, repeated spans, blob layout."""
import numpy as np

from ttt_inputs import SHAPES, blob_layout, blob_size, weight_blob, zipf_tokens, sequence_tokens


def test_tokens_deterministic_in_range_and_prefix_stable():
    s = SHAPES["125m"]
    a = sequence_tokens(s, 0)
    b = sequence_tokens(s, 0)
    assert a.dtype == np.int32 and a.shape == (32768,)
    assert np.array_equal(a, b)
    assert a.min() >= 0 and a.max() < s.vocab
    assert not np.array_equal(a, sequence_tokens(s, 1))
    assert np.array_equal(sequence_tokens(s, 0, T=5000), a[:5000])


def test_zipf_frequencies_follow_pmf():
    V, T = 1000, 200000
    tok = zipf_tokens(T, V, seed=7, copies=0)
    perm = np.random.default_rng(7).permutation(V)
    counts = np.bincount(tok, minlength=V)[perm]          # counts by rank
    pmf = np.arange(1, V + 1) ** -1.1
    pmf /= pmf.sum()
    for r in (0, 1, 9):
        assert abs(counts[r] / T - pmf[r]) < 5 * np.sqrt(pmf[r] / T)


def test_repeated_spans_present():
    tok = zipf_tokens(4096, 32000, seed=3)
    # count 32-grams that appear more than once
    grams = {}
    for i in range(0, 4096 - 32):
        grams.setdefault(tok[i:i + 32].tobytes(), []).append(i)
    assert sum(len(v) > 1 for v in grams.values()) >= 4096 // 128 // 2


def test_blob_layout_and_values():
    s = SHAPES["tiny"]
    lay = blob_layout(s)
    assert lay[0][0] == "E" and lay[-1][0] == "W_lm"
    assert blob_size(s) == sum(int(np.prod(x)) for _, x, _ in lay)
    blob = weight_blob(s)
    assert blob.dtype == np.float32 and blob.size == blob_size(s)
    off = 0
    for name, shp, gain in lay:
        n = int(np.prod(shp))
        seg = blob[off:off + n]
        if gain:
            assert np.all(seg == 1.0), name
        else:
            assert abs(seg.std() - 0.02) < 0.002, name
        off += n
    assert np.array_equal(blob, weight_blob(s))
