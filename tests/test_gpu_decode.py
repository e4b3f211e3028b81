"""Decode-phase TTT (ttt_decode_dev) against the float64 oracle's decode().

The prompt goes through the chunked inner loop; then every generated token is
one forward of one row per block with the current fast weights, and every
complete chunk of b generated tokens takes one inner-loop step.

Token choices are integers decided by floating point, so each side decides
in its own precision and the test checks what is unique:
* every GPU pick is the choice its own logits (returned by the call) make:
  greedy = the first largest logit, bit-exact; sampling = the inverse-CDF
  index at the caller's uniform, valid within fp32 summation error;
* the oracle is then run with the GPU's picks forced (its logits rows, losses
  and fast weights are what the method gives for that token sequence) and
  the GPU's logits rows, prompt-chunk losses, generated-chunk losses and final
  fast weights must match it at the config's tolerances; every GPU pick must
  also be a valid choice for the oracle's logits, within the logits' error.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import test_long_context_02_b300 as T  # noqa: E402
from oracle import ttt_oracle as O  # noqa: E402
from ttt_inputs import SHAPES, Shape, weight_blob, zipf_tokens  # noqa: E402

TOL = {"fp32": (1e-4, 1e-4, 1e-4), "bf16": (2e-2, 1e-2, 2e-2)}   # loss, fast weights, logits rows

# name: shape, prompt length, tokens generated, sample, temperature
CASES = {
    # prompt of 1 full + 1 partial chunk; two complete generated chunks and a partial one
    "tiny_fp32_greedy": (SHAPES["tiny"], 100, 140, False, 1.0),
    "tiny_fp32_sample": (SHAPES["tiny"], 64, 130, True, 0.8),
    # two trainable blocks, the window cache wraps during generation
    "bf16_dh64_greedy": (Shape(8, 256, 4, 1024, 1000, 256, 128, 1e4, 1e-2, 0), 300, 270, False, 1.0),
    "bf16_dual_sample": (Shape(8, 256, 4, 1024, 1000, 256, 128, 1e4, 1e-2, 0, dual_mlp=True), 200, 140, True,
                         1.2),
}


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


def inverse_cdf_ok(z, temp, u, j, eps):
    """j is the first index whose running sum of exp(z/temp - max) exceeds u times the total (within eps)."""
    y = np.asarray(z, np.float64) / temp
    c = np.cumsum(np.exp(y - y.max()))
    t = u * c[-1]
    return c[j] >= t * (1 - eps) and (j == 0 or c[j - 1] <= t * (1 + eps))


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name):
    s, Tp, n_new, sample, temp = CASES[name]
    b, V = s.chunk, s.vocab
    prompt = zipf_tokens(Tp, V, seed=1500)
    blob = weight_blob(s)
    u = np.random.default_rng(7).random(n_new + 1)
    ncp, ncg = -(-Tp // b), n_new // b
    m = T.TTT.from_shape(s)
    try:
        m.load_weights(blob)
        dev = "cuda"
        d_prompt = torch.tensor(prompt[None], dtype=torch.int32, device=dev)
        d_out = torch.full((1, n_new + 1), -1, dtype=torch.int32, device=dev)
        d_pl = torch.zeros((1, ncp), dtype=torch.float32, device=dev)
        d_gl = torch.zeros((1, max(1, ncg)), dtype=torch.float32, device=dev)
        d_z = torch.zeros((1, n_new + 1, V), dtype=torch.float32, device=dev)
        d_u = torch.tensor(u[None], dtype=torch.float32, device=dev)
        m.decode_dev(d_prompt, Tp, n_new, d_out, d_pl, d_gl, sample=sample, temp=temp, d_u=d_u, d_logits=d_z)
        m.sync()
        out = d_out.cpu().numpy()[0]
        zg = d_z.cpu().numpy()[0]
        pl, gl = d_pl.cpu().numpy()[0], d_gl.cpu().numpy()[0][:ncg]
        fw = [m.fast_weights(0, i) for i in range(s.n_trainable)]
        assert m.position == Tp + ncg * b
    finally:
        m.close()

    # every pick follows the GPU's own logits
    u32 = u.astype(np.float32)
    for i in range(n_new + 1):
        assert 0 <= out[i] < V
        if sample:
            assert inverse_cdf_ok(zg[i], np.float32(temp), float(u32[i]), int(out[i]), 1e-4), i
        else:
            assert out[i] == int(np.argmax(zg[i])), i

    # the oracle on the GPU's token sequence
    cfg = O.Config.from_shape(s)
    P0 = O.unpack(blob, cfg)
    res = O.decode(cfg, P0, prompt, n_new, s.eta, lambda z, i: int(out[i]), trace=True)
    tl, tw, tz = TOL[s.compute]
    ez = rel(zg, res["z"])
    print(f"\n{name}: logits rows rel err {ez:.2e}; {n_new} generated, {ncg} generated-chunk steps")
    assert ez < tz
    zerr = float(np.max(np.abs(zg - res["z"])))
    for i in range(n_new + 1):  # the GPU's choice is also a valid one for the oracle's logits
        zr = res["z"][i]
        if sample:
            y = zr / temp
            c = np.cumsum(np.exp(y - y.max()))
            j, t = int(out[i]), u[i] * c[-1]
            slack = np.exp(2 * zerr / temp)  # the logits' error moves every weight by at most this factor
            assert c[j] * slack >= t / slack and (j == 0 or c[j - 1] / slack <= t * slack), i
        else:
            assert zr[out[i]] >= zr.max() - 2 * zerr, i
    lp = np.abs(pl - res["prefill_losses"]) / np.abs(res["prefill_losses"])
    assert lp.max() < tl, (pl, res["prefill_losses"])
    if ncg:
        lg = np.abs(gl - res["gen_losses"]) / np.abs(res["gen_losses"])
        assert lg.max() < tl, (gl, res["gen_losses"])
    L, S = s.n_layers, s.n_trainable
    for i in range(S):
        l = L - S + i
        for w, key in zip(fw[i], (f"W_up.{l}", f"W_down.{l}")):
            e = rel(w, res["P"][key])
            du = rel(w - P0[key], res["P"][key] - P0[key])
            print(f"  {key}: rel Frobenius {e:.2e}, update rel err {du:.2e}")
            assert e < tw, key
            assert du < (1e-3 if s.compute == "fp32" else 5e-2), key


def test_decode_rejects_bad_arguments():
    s = SHAPES["tiny"]
    m = T.TTT.from_shape(s)
    d_prompt = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    d_out = torch.zeros((1, 3), dtype=torch.int32, device="cuda")
    d_pl = torch.zeros((1, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(T.TTTError) as e:          # before any weights
        m.decode_dev(d_prompt, 8, 2, d_out, d_pl)
    assert e.value.code == T.TTT_ERR_STATE
    m.load_weights(weight_blob(s))
    with pytest.raises(T.TTTError) as e:          # sampling without uniforms
        m.decode_dev(d_prompt, 8, 2, d_out, d_pl, sample=True)
    assert e.value.code == T.TTT_ERR_ARG
    with pytest.raises(T.TTTError) as e:          # a generated chunk completes but nowhere to put its loss
        m.decode_dev(d_prompt, 8, s.chunk, torch.zeros((1, s.chunk + 1), dtype=torch.int32, device="cuda"), d_pl)
    assert e.value.code == T.TTT_ERR_ARG
    m.close()
