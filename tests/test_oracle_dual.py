"""Pins of the oracle's dual-MLP variant (a frozen static MLP beside the fast one in
every trainable block) against things other than itself: a torch library model
and its autograd, the reduction to the single-MLP model when the static pair is
zero, the role swap when the fast pair is zero, and the invariants of the loop
(eta = 0 equals one unchunked forward; only the fast pair moves)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ttt_oracle as O
from ttt_inputs import SHAPES, sequence_tokens, weight_blob


@pytest.fixture(autouse=True)
def _float64_default():
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.fixture(scope="module")
def dual():
    """8 layers (2 trainable, so the static MLP's gradient to earlier layers is exercised)."""
    s = SHAPES["tiny"].replace(n_layers=8, dual_mlp=True, chunk=32, window=64)
    cfg = O.Config.from_shape(s)
    assert cfg.dual_mlp and cfg.n_trainable == 2
    P = O.unpack(weight_blob(s), cfg)
    return s, cfg, P, sequence_tokens(s)


def torch_model(cfg, t, tokens, causal_window):
    """Dual-MLP architecture from torch library routines; returns logits."""
    T, H, dh, d, L, S = len(tokens), cfg.n_heads, cfg.d_head, cfg.d_model, cfg.n_layers, cfg.n_trainable
    inv = cfg.rope_theta ** (-2.0 * torch.arange(dh // 2, dtype=torch.float64) / dh)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None]
    cos, sin = torch.cos(ang), torch.sin(ang)
    rot = lambda x: torch.cat([x[..., :dh // 2] * cos - x[..., dh // 2:] * sin,
                               x[..., dh // 2:] * cos + x[..., :dh // 2] * sin], -1)
    qp, kp = np.arange(T)[:, None], np.arange(T)[None, :]
    mask = torch.tensor((kp <= qp) & (kp > qp - causal_window))
    x = t["E"][torch.tensor(np.asarray(tokens), dtype=torch.long)]
    for l in range(L):
        xn = F.rms_norm(x, (d,), t[f"g_attn.{l}"], cfg.rms_eps)
        q, k, v = (F.linear(xn, t[f"W{c}.{l}"].T).view(T, H, dh).transpose(0, 1) for c in "qkv")
        o = F.scaled_dot_product_attention(rot(q), rot(k), v, attn_mask=mask)
        h = x + F.linear(o.transpose(0, 1).reshape(T, d), t[f"Wo.{l}"].T)
        n = F.rms_norm(h, (d,), t[f"g_mlp.{l}"], cfg.rms_eps)
        x = h + F.linear(F.gelu(F.linear(n, t[f"W_up.{l}"].T), approximate="tanh"), t[f"W_down.{l}"].T)
        if l >= L - S:
            x = x + F.linear(F.gelu(F.linear(n, t[f"W_up_s.{l}"].T), approximate="tanh"), t[f"W_down_s.{l}"].T)
    return F.linear(F.rms_norm(x, (d,), t["g_final"], cfg.rms_eps), t["W_lm"].T)


def test_layout_adds_the_static_pair_to_trainable_blocks_only(dual):
    s, cfg, P, _ = dual
    L, S = cfg.n_layers, cfg.n_trainable
    assert all((f"W_up_s.{l}" in P) == (l >= L - S) for l in range(L))
    assert O.trainable_names(cfg) == [n for l in range(L - S, L) for n in (f"W_up.{l}", f"W_down.{l}")]
    assert O.pack(P, cfg).size == weight_blob(s).size


def test_forward_matches_the_torch_library_model(dual):
    _, cfg, P, tok = dual
    T = 96
    z = torch_model(cfg, {k: torch.tensor(v) for k, v in P.items()}, tok[:T], cfg.window)
    per = F.cross_entropy(z[:-1], torch.tensor(tok[1:T], dtype=torch.long), reduction="none").numpy()
    want = [float(per[a:a + cfg.chunk].mean()) for a in range(0, T - 1, cfg.chunk)]
    got = O.dense_forward_losses(cfg, P, tok[:T])
    assert rel(got, want) < 1e-12


def test_gradients_match_torch_autograd(dual):
    _, cfg, P, tok = dual
    n = cfg.chunk
    z, saved, _ = O.chunk_forward(cfg, P, O.init_state(cfg), tok[:n])
    tgt = O.chunk_targets(tok, 0, n)
    tgt[-1] = -1                      # the torch model below has no cross-chunk target
    grads = O.chunk_backward(cfg, P, saved, z, tgt)
    t = {k: torch.tensor(v, requires_grad=k in grads) for k, v in P.items()}
    zz = torch_model(cfg, t, tok[:n], n)
    F.cross_entropy(zz[:-1], torch.tensor(tok[1:n], dtype=torch.long)).backward()
    assert sorted(grads) == sorted(O.trainable_names(cfg))
    for name, g in grads.items():
        assert rel(g, t[name].grad.numpy()) < 1e-11, name


def test_zero_static_pair_reduces_to_the_single_mlp_model(dual):
    s, cfg, P, tok = dual
    Pz = dict(P)
    for l in range(cfg.n_layers - cfg.n_trainable, cfg.n_layers):
        Pz[f"W_down_s.{l}"] = np.zeros_like(P[f"W_down_s.{l}"])
    base_cfg = O.Config(**{**cfg.__dict__, "dual_mlp": False})
    Pb = {k: v for k, v in Pz.items() if "_s." not in k}
    l_dual, P_dual = O.run_sequence(cfg, Pz, tok[:96], 0.05)
    l_base, P_base = O.run_sequence(base_cfg, Pb, tok[:96], 0.05)
    assert rel(l_dual, l_base) < 1e-13
    for k in O.trainable_names(cfg):
        assert rel(P_dual[k], P_base[k]) < 1e-13, k


def test_zero_fast_pair_swaps_roles_with_the_static_pair(dual):
    _, cfg, P, tok = dual
    Pz, Ps = dict(P), dict(P)
    for l in range(cfg.n_layers - cfg.n_trainable, cfg.n_layers):
        Pz[f"W_down.{l}"] = np.zeros_like(P[f"W_down.{l}"])
        Ps[f"W_up.{l}"], Ps[f"W_down.{l}"] = P[f"W_up_s.{l}"], P[f"W_down_s.{l}"]
        Ps[f"W_down_s.{l}"] = np.zeros_like(P[f"W_down_s.{l}"])
    assert rel(O.dense_forward_losses(cfg, Pz, tok[:96]), O.dense_forward_losses(cfg, Ps, tok[:96])) < 1e-13


def test_eta0_chunked_equals_unchunked_and_only_the_fast_pair_moves(dual):
    _, cfg, P, tok = dual
    losses, _ = O.run_sequence(cfg, P, tok[:128], 0.0)
    assert rel(losses, O.dense_forward_losses(cfg, P, tok[:128])) < 1e-12
    _, P2 = O.run_sequence(cfg, P, tok[:128], 0.05)
    fast = set(O.trainable_names(cfg))
    for k in P:
        moved = not np.array_equal(P2[k], P[k])
        assert moved == (k in fast), k
