"""The whole inner loop (libttt through its C ABI) against the float64 oracle.

Same seeded tokens and fp32 weights on both sides; per-chunk losses and the
final fast weights are compared with the tolerances of the method's statement:
fp32 compute: loss 1e-4 relative, fast weights 1e-4 relative Frobenius;
bf16 compute (fp32 fast weights): loss 2e-2 relative, fast weights 1e-2.
The update itself is gated too: with dW = W_final - W_0 on each side,
|dW_gpu - dW_ref| / |dW_ref| must stay below 1e-3 (fp32) or 5e-2 (bf16), so a
path that skipped or misscaled the SGD step fails however small the step is
next to W.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402
from oracle import ttt_oracle as O  # noqa: E402
from ttt_inputs import SHAPES, Shape, sequence_tokens, weight_blob, zipf_tokens  # noqa: E402

TOL = {"fp32": (1e-4, 1e-4), "bf16": (2e-2, 1e-2)}
DW_TOL = {"fp32": 1e-3, "bf16": 5e-2}

# small shapes that still span several tiles, wrap the window cache and end in a ragged chunk
SMALL = {
    "dh64": Shape(8, 256, 4, 1024, 1000, 256, 128, 1e4, 1e-2, 1000),
    "dh96": Shape(8, 384, 4, 1536, 2048, 256, 256, 1e6, 1e-2, 900),
    "dh128": Shape(8, 512, 4, 2048, 1024, 512, 256, 1e7, 1e-2, 1100),
    "fp32_dh64": Shape(8, 256, 4, 1024, 512, 128, 128, 1e4, 1e-2, 700, compute="fp32"),
    # the frozen blocks of 4 chunks run as one pass; 10 chunks, the last one ragged
    "dh96_ahead4": Shape(8, 384, 4, 1536, 2048, 512, 128, 1e6, 1e-2, 1200),
    # the dual-MLP variant: two trainable blocks, so the static MLP's gradient path to the
    # block below is exercised; the cache wraps and the last chunk is ragged
    "dual_dh64": Shape(8, 256, 4, 1024, 1000, 256, 128, 1e4, 1e-2, 1000, dual_mlp=True),
    "dual_fp32_dh32": Shape(8, 128, 4, 512, 512, 128, 64, 1e4, 1e-2, 600, compute="fp32", dual_mlp=True),
}


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


def run_gpu(shape, tokens, blob):
    m = T.TTT.from_shape(shape)
    m.load_weights(blob)
    b, Tn = shape.chunk, len(tokens)
    losses = []
    for s in range(0, Tn, b):
        n = min(b, Tn - s)
        nxt = int(tokens[s + n]) if s + n < Tn else -1
        losses.append(float(m.prefill_chunk(tokens[s:s + n], [nxt])[0]))
    fw = [m.fast_weights(0, i) for i in range(shape.n_trainable)]
    pos = m.position
    m.close()
    return losses, fw, pos


def run_gpu_sequence(shape, tokens, blob):
    """Whole sequence through ttt_prefill_sequence_dev (frozen blocks run ahead over several chunks)."""
    m = T.TTT.from_shape(shape)
    m.load_weights(blob)
    Tn, b = len(tokens), shape.chunk
    nc = -(-Tn // b)
    d_tok = torch.tensor(np.asarray(tokens, np.int32), device="cuda")
    d_loss = torch.zeros(nc, dtype=torch.float32, device="cuda")
    m.prefill_sequence_dev(d_tok, Tn, d_loss)
    m.sync()
    losses = [float(x) for x in d_loss.cpu().numpy()]
    fw = [m.fast_weights(0, i) for i in range(shape.n_trainable)]
    pos = m.position
    m.close()
    return losses, fw, pos


def run_gpu_host_sequence(shape, tokens, blob):
    """Whole sequence from host memory through ttt_prefill_sequence (one upload, one download)."""
    m = T.TTT.from_shape(shape)
    m.load_weights(blob)
    losses = [float(x) for x in m.prefill_sequence(np.asarray(tokens, np.int32)[None])[0]]
    fw = [m.fast_weights(0, i) for i in range(shape.n_trainable)]
    pos = m.position
    m.close()
    return losses, fw, pos


def run_gpu_resumed(shape, tokens, blob):
    """The per-chunk API in one context up to the middle chunk boundary, the state moved
    (ttt_export_state / ttt_import_state) into a fresh context, the rest there."""
    b, Tn = shape.chunk, len(tokens)
    cut = (-(-Tn // b) // 2) * b

    def chunks(m, lo, hi):
        out = []
        for s in range(lo, hi, b):
            n = min(b, Tn - s)
            nxt = int(tokens[s + n]) if s + n < Tn else -1
            out.append(float(m.prefill_chunk(tokens[s:s + n], [nxt])[0]))
        return out

    a = T.TTT.from_shape(shape)
    a.load_weights(blob)
    losses = chunks(a, 0, cut)
    state = a.export_state(0)
    a.close()
    m = T.TTT.from_shape(shape)
    m.load_weights(blob)
    m.import_state(state, 0)
    assert m.position == cut
    assert m.export_state(0) == state  # the round trip is bit-exact
    losses += chunks(m, cut, Tn)
    fw = [m.fast_weights(0, i) for i in range(shape.n_trainable)]
    pos = m.position
    m.close()
    return losses, fw, pos


def check(shape, tokens, name, runner=None):
    blob = weight_blob(shape)
    cfg = O.Config.from_shape(shape)
    P = O.unpack(blob, cfg)
    ref_losses, Pf = O.run_sequence(cfg, P, tokens, shape.eta)
    losses, fw, pos = (runner or run_gpu)(shape, tokens, blob)
    assert pos == len(tokens)
    tl, tw = TOL[shape.compute]
    lr = [abs(a - b) / abs(b) for a, b in zip(losses, ref_losses)]
    print(f"\n{name}: loss rel err max {max(lr):.2e}; losses gpu {np.round(losses, 5)} ref {np.round(ref_losses, 5)}")
    assert max(lr) < tl, (losses, ref_losses)
    L, S = shape.n_layers, shape.n_trainable
    for i in range(S):
        l = L - S + i
        for w, key in zip(fw[i], (f"W_up.{l}", f"W_down.{l}")):
            e = rel(w, Pf[key])
            dw = rel(w - P[key], Pf[key] - P[key])
            print(f"  {key}: rel Frobenius {e:.2e}  update rel err {dw:.2e}")
            assert e < tw, key
            assert dw < DW_TOL[shape.compute], (key, dw)


def test_tiny_fp32_full_sequence():
    s = SHAPES["tiny"]
    check(s, sequence_tokens(s), "tiny fp32")


@pytest.mark.parametrize("name", list(SMALL))
def test_small_shapes(name):
    s = SMALL[name]
    check(s, zipf_tokens(s.seq_len, s.vocab, seed=1000), name)


@pytest.mark.parametrize("name", ["dh64", "dh128", "dh96_ahead4", "dual_dh64"])
def test_sequence_api_runs_frozen_blocks_ahead(name):
    s = SMALL[name]
    check(s, zipf_tokens(s.seq_len, s.vocab, seed=1000), name + " (sequence)", runner=run_gpu_sequence)


def test_sequence_api_tiny_fp32():
    s = SHAPES["tiny"]
    check(s, sequence_tokens(s), "tiny fp32 (sequence)", runner=run_gpu_sequence)


@pytest.mark.parametrize("name", ["dh96_ahead4", "fp32_dh64"])
def test_host_sequence_api(name):
    s = SMALL[name]
    check(s, zipf_tokens(s.seq_len, s.vocab, seed=1000), name + " (host sequence)", runner=run_gpu_host_sequence)


def test_eta0_matches_frozen_forward():
    s = SMALL["dh64"].replace(eta=0.0)
    tok = zipf_tokens(s.seq_len, s.vocab, seed=1001)
    cfg = O.Config.from_shape(s)
    P = O.unpack(weight_blob(s), cfg)
    ref = O.dense_forward_losses(cfg, P, tok)
    losses, fw, _ = run_gpu(s, tok, weight_blob(s))
    assert max(abs(a - b) / b for a, b in zip(losses, ref)) < 2e-2
    for i in range(s.n_trainable):
        l = s.n_layers - s.n_trainable + i
        assert np.array_equal(fw[i][0], P[f"W_up.{l}"].astype(np.float32))


def test_bad_token_rejected_and_state_errors():
    s = SMALL["dh64"]
    m = T.TTT.from_shape(s)
    with pytest.raises(T.TTTError) as e:
        m.prefill_chunk(np.zeros(4, np.int32), [-1])
    assert e.value.code == T.TTT_ERR_STATE
    m.load_weights(weight_blob(s))
    with pytest.raises(T.TTTError) as e:
        m.prefill_chunk(np.array([1, 2, s.vocab], np.int32), [-1])
    assert e.value.code == T.TTT_ERR_ARG
    with pytest.raises(T.TTTError) as e:
        m.prefill_chunk(np.zeros(s.chunk + 1, np.int32), [-1])
    assert e.value.code == T.TTT_ERR_ARG
    # the device path reports a bad id at the next sync
    tok = torch.tensor([1, 2, s.vocab + 5], dtype=torch.int32, device="cuda")
    nxt = torch.tensor([-1], dtype=torch.int32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.prefill_chunk_dev(tok, 3, nxt, loss)
    with pytest.raises(T.TTTError) as e:
        m.sync()
    assert e.value.code == T.TTT_ERR_DEVICE
    m.close()


def test_unsupported_shapes_rejected():
    with pytest.raises(T.TTTError) as e:
        T.TTT(T.make_config(4, 200, 4, 800, 512, 128, 64, 1e4, 0.0))      # d_head 50
    assert e.value.code == T.TTT_ERR_UNSUPPORTED
    with pytest.raises(T.TTTError) as e:
        T.TTT(T.make_config(4, 256, 4, 1024, 512, 128, 256, 1e4, 0.0))     # k < b
    assert e.value.code == T.TTT_ERR_ARG


def test_allocation_failure_reports_oom_and_leaves_the_process_usable():
    # a window cache of 2^27 slots x 12 layers x 768 columns (2.4 TB per sequence) cannot be
    # allocated: ttt_create must return TTT_ERR_OOM, free what it took, and leave the device usable
    free0, _ = torch.cuda.mem_get_info()
    with pytest.raises(T.TTTError) as e:
        T.TTT(T.make_config(12, 768, 12, 3072, 32000, 1 << 27, 1024, 1e6, 1e-3))
    assert e.value.code == T.TTT_ERR_OOM
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (64 << 20), (free0, free1)
    s = SHAPES["tiny"]
    tok = sequence_tokens(s)
    check(s.replace(seq_len=256), tok[:256], "tiny fp32 after an allocation failure")


@pytest.mark.parametrize("name", ["dh96_ahead4", "fp32_dh64", "dual_dh64"])
def test_state_export_import_resumes_the_sequence(name):
    s = SMALL[name]
    check(s, zipf_tokens(s.seq_len, s.vocab, seed=1000), name + " (resumed)", runner=run_gpu_resumed)


def test_state_import_rejects_another_shape():
    a = T.TTT.from_shape(SMALL["dh64"])
    a.load_weights(weight_blob(SMALL["dh64"]))
    state = a.export_state(0)
    a.close()
    other = SMALL["dh64"].replace(window=512)
    m = T.TTT.from_shape(other)
    m.load_weights(weight_blob(other))
    with pytest.raises(T.TTTError) as e:
        m.import_state(state + bytes(int(T.ttt_state_bytes(m._h)) - len(state)), 0)
    assert e.value.code == T.TTT_ERR_ARG
    m.close()


# ------------------------------------------------------------------ several sequences per context
def multi_sequence_case(name, n_seqs):
    s = SMALL[name].replace(n_seqs=n_seqs)
    toks = np.stack([zipf_tokens(s.seq_len, s.vocab, seed=2000 + q) for q in range(n_seqs)]).astype(np.int32)
    return s, toks


def run_gpu_multi(shape, toks, blob, api, concurrent):
    B, Tn, b = toks.shape[0], toks.shape[1], shape.chunk
    nc = -(-Tn // b)
    m = T.TTT.from_shape(shape)
    try:
        m.load_weights(blob)
        m.set_concurrency(concurrent)
        if api == "sequence":
            d_tok = torch.tensor(toks, device="cuda")
            d_loss = torch.zeros((B, nc), dtype=torch.float32, device="cuda")
            m.prefill_sequence_dev(d_tok, Tn, d_loss)
            m.sync()
            losses = d_loss.cpu().numpy().astype(np.float64)
        else:
            losses = np.zeros((B, nc))
            for ci, st in enumerate(range(0, Tn, b)):
                n = min(b, Tn - st)
                nxt = toks[:, st + n] if st + n < Tn else np.full(B, -1, np.int32)
                losses[:, ci] = m.prefill_chunk(toks[:, st:st + n], nxt)
        assert m.position == Tn
        fw = [[m.fast_weights(q, i) for i in range(shape.n_trainable)] for q in range(B)]
    finally:
        m.close()
    return losses, fw


@pytest.mark.parametrize("name,n_seqs,api,concurrent", [
    ("dh96_ahead4", 5, "sequence", True),   # five sequences on four lanes: the first lane takes two in turn
    ("dh96_ahead4", 3, "sequence", False),  # one lane, the sequences one after another
    ("dh64", 4, "chunk", True),              # per-chunk calls, every sequence on its own lane
    ("fp32_dh64", 2, "sequence", True),
])
def test_several_sequences_match_the_oracle(name, n_seqs, api, concurrent):
    s, toks = multi_sequence_case(name, n_seqs)
    blob = weight_blob(s)
    cfg = O.Config.from_shape(s)
    P = O.unpack(blob, cfg)
    losses, fw = run_gpu_multi(s, toks, blob, api, concurrent)
    tl, tw = TOL[s.compute]
    L, S = s.n_layers, s.n_trainable
    for q in range(n_seqs):
        ref_losses, Pf = O.run_sequence(cfg, P, toks[q], s.eta)
        lr = np.abs(losses[q] - ref_losses) / np.abs(ref_losses)
        print(f"\n{name} x{n_seqs} {api} seq {q}: loss rel err max {lr.max():.2e}")
        assert lr.max() < tl, (q, losses[q], ref_losses)
        for i in range(S):
            l = L - S + i
            for w, key in zip(fw[q][i], (f"W_up.{l}", f"W_down.{l}")):
                assert rel(w, Pf[key]) < tw, (q, key)
                assert rel(w - P[key], Pf[key] - P[key]) < DW_TOL[s.compute], (q, key)
