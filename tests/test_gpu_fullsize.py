"""Full-size workloads in the benchmark's launch configuration, checked on
outputs the float64 oracle can afford one by one.

Each case runs whole sequences through ttt_prefill_sequence_dev, as the
benchmark does: the frozen blocks run ahead over several chunks, and the
trainable blocks step chunk by chunk. It then checks:

* chunk 0's loss against the oracle's forward of that chunk. The loss comes
  before any update, and for k >= b it does not depend on k. Tolerance is
  2e-2 relative, the bf16 bound.
* the window cache of block 0 after the whole sequence:
  - every slot's absolute position, bit-exact: the latest p < T with
    p mod k == slot;
  - the post-RoPE keys and the values of sampled slots against the oracle's
    block-0 projections of the token at that position. Block 0's keys
    depend on that token and position only.
* every chunk loss is finite; the position is T; the last trainable block's
  fast weights moved, and by a small relative amount.
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402
from oracle import ttt_oracle as O  # noqa: E402
from ttt_inputs import SHAPES, blob_layout, sequence_tokens, weight_blob  # noqa: E402

# 125M, 760M and the 760M-shape window/chunk sweep share blobs in this order; 3B last
CASES = ["125m", "760m"] + sorted(n for n in SHAPES if n.startswith("sweep")) + ["3b"]


class LazyParams(dict):
    """Oracle parameter dict whose float64 arrays are made from the fp32 blob on access.

    The forward reads each weight once per chunk; converting on access keeps
    the float64 copy of a multi-GB blob from existing all at once.
    """

    def __init__(self, blob, shape):
        super().__init__()
        self._blob, self._where, off = blob, {}, 0
        for name, shp, _ in blob_layout(shape):
            n = int(np.prod(shp))
            self._where[name] = (off, shp)
            off += n

    def __getitem__(self, name):
        off, shp = self._where[name]
        n = int(np.prod(shp))
        return self._blob[off:off + n].astype(np.float64).reshape(shp)

    def __contains__(self, name):
        return name in self._where


@functools.lru_cache(maxsize=1)
def blob_for(n_layers, d_model, n_heads, d_ff, vocab):
    s = SHAPES["125m"].replace(n_layers=n_layers, d_model=d_model, n_heads=n_heads, d_ff=d_ff, vocab=vocab)
    return weight_blob(s)


def oracle_chunk0(s, seq, b):
    """Mean loss of chunk 0 (b tokens) by the float64 oracle; independent of k >= b and of eta."""
    return _oracle_chunk0(s.replace(window=max(s.window, b), eta=0.0), seq, b)


@functools.lru_cache(maxsize=None)
def _oracle_chunk0(s, seq, b):
    blob = blob_for(s.n_layers, s.d_model, s.n_heads, s.d_ff, s.vocab)
    cfg = O.Config.from_shape(s.replace(chunk=b))
    tokens = sequence_tokens(s, seq)
    z, _, _ = O.chunk_forward(cfg, LazyParams(blob, s), O.init_state(cfg), tokens[:b], keep=False)
    return O.chunk_loss(z, O.chunk_targets(tokens, 0, b))


def oracle_block0_kv(s, P, tok, pos):
    """Block 0's post-RoPE key and value rows for one token at absolute position pos."""
    x = P["E"][[tok]]
    xn, _ = O.rmsnorm(x, P["g_attn.0"], s.rms_eps)
    H, dh = s.n_heads, s.d_head
    ang = O.rope_angles([pos], dh, s.rope_theta)
    k = (xn @ P["Wk.0"]).reshape(1, H, dh).transpose(1, 0, 2)
    k = O.rope(k, ang).transpose(1, 0, 2).reshape(-1)
    v = (xn @ P["Wv.0"]).reshape(-1)
    return k, v


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("name", CASES)
def test_full_size_sequence(name):
    s = SHAPES[name]
    blob = blob_for(s.n_layers, s.d_model, s.n_heads, s.d_ff, s.vocab)
    Tn, b, B = s.seq_len, s.chunk, s.n_seqs
    nc = -(-Tn // b)
    toks = np.stack([sequence_tokens(s, q) for q in range(B)]).astype(np.int32)
    m = T.TTT.from_shape(s)
    try:
        m.load_weights(blob)
        d_tok = torch.tensor(toks, device="cuda")
        d_loss = torch.zeros((B, nc), dtype=torch.float32, device="cuda")
        m.prefill_sequence_dev(d_tok, Tn, d_loss)
        m.sync()
        losses = d_loss.cpu().numpy().astype(np.float64)
        assert m.position == Tn
        assert np.all(np.isfinite(losses)), name
        kc, vc, pos = m.window(0, 0)
        up, _ = m.fast_weights(0, s.n_trainable - 1)
    finally:
        m.close()

    # chunk 0 against the oracle (sequence 0; also the last one of a multi-sequence run at b = 256)
    for q in sorted({0, B - 1} if b <= 256 else {0}):
        ref = oracle_chunk0(s.replace(window=b), q, b)
        assert abs(losses[q, 0] - ref) / abs(ref) < 2e-2, (name, q, losses[q, 0], ref)

    # window indexing, bit-exact, and block-0 keys/values of sampled slots
    k = s.window
    slots = np.arange(k)
    expect = Tn - 1 - ((Tn - 1 - slots) % k)
    assert np.array_equal(pos, expect)
    P = LazyParams(blob, s)
    small = {n: P[n] for n in ("E", "g_attn.0", "Wk.0", "Wv.0")}
    rng = np.random.default_rng(7)
    for slot in sorted(set(rng.integers(0, k, 12).tolist()) | {int((Tn - 1) % k)}):
        p = int(pos[slot])
        kr, vr = oracle_block0_kv(s, small, int(toks[0, p]), p)
        assert rel(kc[slot], kr) < 1e-2, (name, slot, p)
        assert rel(vc[slot], vr) < 1e-2, (name, slot, p)

    # the last trainable block's W_up moved, and by a small relative amount
    w0 = P[f"W_up.{s.n_layers - 1}"]
    dw = rel(up, w0)
    assert np.all(np.isfinite(up)) and 0.0 < dw < 1.0, dw
    print(f"\n{name}: chunk-0 loss {losses[0, 0]:.5f}, last {losses[0, -1]:.5f}, |dW_up|/|W_up| {dw:.3e}")
