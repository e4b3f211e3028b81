"""Pins of the float64 oracle against things other than itself.

Library routines (torch float64 rms_norm, gelu(tanh), scaled_dot_product_attention,
cross_entropy, autograd; scipy logsumexp), RoPE closed forms, central finite
differences, and the invariants the TTT-E2E pages fix: eta = 0 reproduces one
unchunked forward of the frozen model, k >= T is full causal attention, only the
last-quarter MLP weights move, one plain SGD step per chunk (linear in eta), and
chunk i depends on chunks < i only through the keys in its window and the fast
weights.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import ttt_oracle as O
from ttt_inputs import SHAPES, sequence_tokens, weight_blob

RNG = np.random.default_rng(1234)


@pytest.fixture(autouse=True)
def _float64_default():
    """torch routines used as pins run in float64; the global default is restored
    afterwards so that tests collected later (GPU buffers) keep float32."""
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def tiny_cfg(**kw):
    s = SHAPES["tiny"]
    c = O.Config.from_shape(s)
    return O.Config(**{**c.__dict__, **kw})


@pytest.fixture(scope="module")
def tiny():
    s = SHAPES["tiny"]
    cfg = O.Config.from_shape(s)
    P = O.unpack(weight_blob(s), cfg)
    tok = sequence_tokens(s)
    return cfg, P, tok


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- components
def test_rmsnorm_matches_torch():
    x = RNG.standard_normal((7, 48)) * 3
    g = RNG.standard_normal(48)
    y, r = O.rmsnorm(x, g, 1e-6)
    ref = F.rms_norm(torch.tensor(x), (48,), torch.tensor(g), 1e-6).numpy()
    assert rel(y, ref) < 1e-14
    assert rel(r[:, 0], 1 / np.sqrt((x ** 2).mean(1) + 1e-6)) < 1e-14


def test_rmsnorm_bwd_matches_autograd():
    x = torch.tensor(RNG.standard_normal((5, 32)), requires_grad=True)
    g = torch.tensor(RNG.standard_normal(32))
    dy = RNG.standard_normal((5, 32))
    F.rms_norm(x, (32,), g, 1e-6).backward(torch.tensor(dy))
    _, r = O.rmsnorm(x.detach().numpy(), g.numpy(), 1e-6)
    dx = O.rmsnorm_bwd(dy, x.detach().numpy(), g.numpy(), r)
    assert rel(dx, x.grad.numpy()) < 1e-13


def test_gelu_tanh_matches_torch_and_autograd():
    a = torch.tensor(np.linspace(-8, 8, 1001), requires_grad=True)
    y = F.gelu(a, approximate="tanh")
    y.sum().backward()
    assert rel(O.gelu_tanh(a.detach().numpy()), y.detach().numpy()) < 1e-15
    assert rel(O.gelu_tanh_grad(a.detach().numpy()), a.grad.numpy()) < 1e-14


def test_rope_closed_forms():
    # d_head = 2: inv_freq_0 = 1, so position p is a plane rotation by p rad.
    x = RNG.standard_normal((3, 2))
    p = np.array([0.0, 1.0, 37.0])
    y = O.rope(x[None], O.rope_angles(p, 2, 1e4))[0]
    ref = np.stack([x[:, 0] * np.cos(p) - x[:, 1] * np.sin(p),
                    x[:, 1] * np.cos(p) + x[:, 0] * np.sin(p)], 1)
    assert rel(y, ref) < 1e-15
    # d_head = 4, theta = 16: pairs (0,2) turn at rate 1, (1,3) at 16^(-1/2) = 1/4.
    x = RNG.standard_normal((1, 4))
    y = O.rope(x[None], O.rope_angles([8.0], 4, 16.0))[0][0]
    c0, s0, c1, s1 = math.cos(8), math.sin(8), math.cos(2), math.sin(2)
    x0, x1, x2, x3 = x[0]
    ref = [x0 * c0 - x2 * s0, x1 * c1 - x3 * s1, x2 * c0 + x0 * s0, x3 * c1 + x1 * s1]
    assert rel(y, ref) < 1e-15


def test_rope_relative_position_and_norm():
    dh = 32
    q, k = RNG.standard_normal((2, 1, dh))
    def dot(p1, p2):
        a = O.rope(q[None], O.rope_angles([p1], dh, 1e4))[0, 0]
        b = O.rope(k[None], O.rope_angles([p2], dh, 1e4))[0, 0]
        return a @ b
    assert abs(dot(5, 2) - dot(105, 102)) < 1e-12
    assert abs(dot(5, 2) - dot(4, 2)) > 1e-6
    y = O.rope(q[None], O.rope_angles([123], dh, 1e4))
    assert abs(np.linalg.norm(y) - np.linalg.norm(q)) < 1e-12
    assert rel(O.rope(q[None], O.rope_angles([0], dh, 1e4))[0], q) == 0.0


def test_rope_bwd_is_adjoint():
    x = RNG.standard_normal((3, 9, 16))
    y = RNG.standard_normal((3, 9, 16))
    ang = O.rope_angles(np.arange(9) * 1000, 16, 1e7)
    lhs = np.sum(O.rope(x, ang) * y)
    rhs = np.sum(x * O.rope_bwd(y, ang))
    assert abs(lhs - rhs) < 1e-12 * np.sum(np.abs(x * y))
    assert rel(O.rope_bwd(O.rope(x, ang), ang), x) < 1e-14


def _band(qpos, kpos, window):
    qp, kp = np.asarray(qpos)[:, None], np.asarray(kpos)[None, :]
    return torch.tensor((kp <= qp) & (kp > qp - window))


@pytest.mark.parametrize("window", [1000, 16, 1])
def test_attention_matches_sdpa(window):
    H, n, dh = 3, 40, 16
    q, k, v = (RNG.standard_normal((H, n, dh)) for _ in range(3))
    pos = np.arange(n)
    o, lse = O.attention(q, k, v, pos, pos, window)
    tq, tk, tv = (torch.tensor(t) for t in (q, k, v))
    if window >= n:
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    else:
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=_band(pos, pos, window))
    assert rel(o, ref.numpy()) < 1e-13
    s = np.einsum("hqd,hkd->hqk", q, k) / math.sqrt(dh)
    s = np.where(_band(pos, pos, window).numpy(), s, -np.inf)
    assert rel(lse, scipy.special.logsumexp(s, axis=-1)) < 1e-14


def test_attention_cached_keys_and_window_brute_force():
    # queries at 100..107, keys 90..107; window 12 -> key j visible iff p-12 < j <= p
    H, dh, window = 2, 8, 12
    qpos, kpos = np.arange(100, 108), np.arange(90, 108)
    q = RNG.standard_normal((H, 8, dh))
    k, v = RNG.standard_normal((2, H, 18, dh))
    o, _ = O.attention(q, k, v, qpos, kpos, window)
    ref = F.scaled_dot_product_attention(*(torch.tensor(t) for t in (q, k, v)),
                                         attn_mask=_band(qpos, kpos, window))
    assert rel(o, ref.numpy()) < 1e-13
    # key 90 lies in the window of p only while p - 12 < 90, i.e. p <= 101:
    # perturbing it moves queries 100, 101 and leaves 102..107 bit-identical
    k2, v2 = k.copy(), v.copy()
    k2[:, 0] += 5.0
    v2[:, 0] -= 3.0
    o2, _ = O.attention(q, k2, v2, qpos, kpos, window)
    assert np.array_equal(o[:, 2:], o2[:, 2:])
    assert not np.allclose(o[:, :2], o2[:, :2])
    # a key after the query (position 107) never reaches query 100..106
    k3 = k.copy()
    k3[:, 17] += 1.0
    o3, _ = O.attention(q, k3, v, qpos, kpos, window)
    assert np.array_equal(o3[:, :7], o[:, :7])
    assert not np.allclose(o3[:, 7], o[:, 7])


def test_attention_bwd_matches_autograd():
    H, n, dh, window = 2, 24, 8, 10
    pos = np.arange(n)
    q, k, v, do = (RNG.standard_normal((H, n, dh)) for _ in range(4))
    tq, tk, tv = (torch.tensor(t, requires_grad=True) for t in (q, k, v))
    F.scaled_dot_product_attention(tq, tk, tv, attn_mask=_band(pos, pos, window)
                                   ).backward(torch.tensor(do))
    dq, dk, dv = O.attention_bwd(do, q, k, v, pos, pos, window)
    assert rel(dq, tq.grad.numpy()) < 1e-12
    assert rel(dk, tk.grad.numpy()) < 1e-12
    assert rel(dv, tv.grad.numpy()) < 1e-12


def test_cross_entropy_matches_torch():
    z = RNG.standard_normal((6, 50)) * 4
    tgt = np.array([3, 0, 49, -1, 7, 7])
    loss, p = O.cross_entropy(z, tgt)
    ok = tgt >= 0
    ref = F.cross_entropy(torch.tensor(z[ok]), torch.tensor(tgt[ok]), reduction="none")
    assert rel(loss[ok], ref.numpy()) < 1e-14
    assert np.isnan(loss[~ok]).all()
    assert rel(p, torch.softmax(torch.tensor(z), -1).numpy()) < 1e-14


# ------------------------------------------------------------- whole model
def _torch_forward_losses(cfg, P, tokens, window):
    """Same architecture assembled from torch library routines (test only)."""
    T, H, dh, d = len(tokens), cfg.n_heads, cfg.d_head, cfg.d_model
    t = {k: torch.tensor(v) for k, v in P.items()}
    pos = torch.arange(T, dtype=torch.float64)
    inv = cfg.rope_theta ** (-2.0 * torch.arange(dh // 2, dtype=torch.float64) / dh)
    ang = pos[:, None] * inv[None]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(x):  # [H, T, dh]
        x1, x2 = x[..., :dh // 2], x[..., dh // 2:]
        return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], -1)

    mask = _band(np.arange(T), np.arange(T), window)
    x = t["E"][torch.tensor(tokens, dtype=torch.long)]
    for l in range(cfg.n_layers):
        xn = F.rms_norm(x, (d,), t[f"g_attn.{l}"], cfg.rms_eps)
        q, k, v = (F.linear(xn, t[f"W{c}.{l}"].T).view(T, H, dh).transpose(0, 1)
                   for c in "qkv")
        o = F.scaled_dot_product_attention(rot(q), rot(k), v, attn_mask=mask)
        h = x + F.linear(o.transpose(0, 1).reshape(T, d), t[f"Wo.{l}"].T)
        hn = F.rms_norm(h, (d,), t[f"g_mlp.{l}"], cfg.rms_eps)
        x = h + F.linear(F.gelu(F.linear(hn, t[f"W_up.{l}"].T), approximate="tanh"),
                         t[f"W_down.{l}"].T)
    z = F.linear(F.rms_norm(x, (d,), t["g_final"], cfg.rms_eps), t["W_lm"].T)
    tg = torch.tensor(np.asarray(tokens[1:]), dtype=torch.long)
    per = F.cross_entropy(z[:-1], tg, reduction="none").numpy()
    per = np.append(per, np.nan)
    out = []
    for s in range(0, T, cfg.chunk):
        seg = per[s:s + cfg.chunk]
        out.append(float(np.nanmean(seg)))
    return out


def test_dense_forward_matches_torch_library_model(tiny):
    cfg, P, tok = tiny
    ref = _torch_forward_losses(cfg, P, tok[:256], cfg.window)
    got = O.dense_forward_losses(cfg, P, tok[:256])
    assert rel(got, ref) < 1e-12


def test_eta0_chunked_equals_unchunked_forward(tiny):
    cfg, P, tok = tiny
    dense = O.dense_forward_losses(cfg, P, tok)
    for b in (64, 48, 128):   # independent of the chunk size, ragged tails too
        c = O.Config(**{**cfg.__dict__, "chunk": b})
        losses, P2 = O.run_sequence(c, P, tok, eta=0.0)
        want = O.dense_forward_losses(c, P, tok)
        assert rel(losses, want) < 1e-12, b
        assert all(np.array_equal(P2[k], P[k]) for k in P)
    assert len(dense) == 8


def test_window_ge_T_is_full_causal(tiny):
    cfg, P, tok = tiny
    c = O.Config(**{**cfg.__dict__, "window": 4096})
    losses, _ = O.run_sequence(c, P, tok[:320], eta=0.0)
    ref = _torch_forward_losses(c, P, tok[:320], 10 ** 9)
    assert rel(losses, ref) < 1e-12


def _state_before(cfg, P, tok, c, eta):
    state = O.init_state(cfg)
    for i in range(c):
        s = i * cfg.chunk
        ids = tok[s:s + cfg.chunk]
        _, P, state, _ = O.ttt_step(cfg, P, state, ids, O.chunk_targets(tok, s, len(ids)), eta)
    return P, state


def test_gradients_match_central_differences(tiny):
    cfg, P, tok = tiny
    c = 3                                     # window full, cache wrapped
    P, state = _state_before(cfg, P, tok, c, cfg_eta := 1e-2)
    s = c * cfg.chunk
    ids, tgt = tok[s:s + cfg.chunk], O.chunk_targets(tok, s, cfg.chunk)
    z, saved, _ = O.chunk_forward(cfg, P, state, ids)
    grads = O.chunk_backward(cfg, P, saved, z, tgt)

    def loss_at(Pp):
        zz, _, _ = O.chunk_forward(cfg, Pp, state, ids, keep=False)
        return O.chunk_loss(zz, tgt)

    # fourth-order central stencil: truncation O(h^4), round-off ~ eps*loss/h
    h = 1e-3

    def fd_along(dirs):
        def at(t):
            Pt = dict(P)
            for n, dd in dirs.items():
                Pt[n] = P[n] + t * dd
            return loss_at(Pt)
        return (-at(2 * h) + 8 * at(h) - 8 * at(-h) + at(-2 * h)) / (12 * h)

    for name in O.trainable_names(cfg):
        W = P[name]
        for _ in range(64):
            ij = tuple(int(RNG.integers(0, n)) for n in W.shape)
            e = np.zeros_like(W)
            e[ij] = 1.0
            fd = fd_along({name: e})
            g = grads[name][ij]
            assert abs(fd - g) <= 1e-6 * max(abs(g), 1e-2 * np.abs(grads[name]).max()), (name, ij, fd, g)
    # one random direction through all fast weights at once
    dirs = {n: RNG.standard_normal(P[n].shape) for n in O.trainable_names(cfg)}
    norm = math.sqrt(sum(np.sum(dd * dd) for dd in dirs.values()))
    dirs = {n: dd / norm for n, dd in dirs.items()}      # unit step in weight space
    fd = fd_along(dirs)
    an = sum(np.sum(grads[n] * dirs[n]) for n in dirs)
    assert abs(fd - an) <= 1e-6 * abs(an)


def test_gradients_match_torch_autograd(tiny):
    """Library cross-check: autograd of the torch-routine model, chunk 0."""
    cfg, P, tok = tiny
    n = cfg.chunk
    z, saved, _ = O.chunk_forward(cfg, P, O.init_state(cfg), tok[:n])
    tgt = O.chunk_targets(tok, 0, n)
    grads = O.chunk_backward(cfg, P, saved, z, tgt)
    t = {k: torch.tensor(v, requires_grad=k in grads) for k, v in P.items()}
    d, H, dh = cfg.d_model, cfg.n_heads, cfg.d_head
    inv = cfg.rope_theta ** (-2.0 * torch.arange(dh // 2, dtype=torch.float64) / dh)
    ang = torch.arange(n, dtype=torch.float64)[:, None] * inv[None]
    cos, sin = torch.cos(ang), torch.sin(ang)
    rot = lambda x: torch.cat([x[..., :dh // 2] * cos - x[..., dh // 2:] * sin,
                               x[..., dh // 2:] * cos + x[..., :dh // 2] * sin], -1)
    x = t["E"][torch.tensor(tok[:n], dtype=torch.long)]
    for l in range(cfg.n_layers):
        xn = F.rms_norm(x, (d,), t[f"g_attn.{l}"], cfg.rms_eps)
        q, k, v = (F.linear(xn, t[f"W{c}.{l}"].T).view(n, H, dh).transpose(0, 1) for c in "qkv")
        o = F.scaled_dot_product_attention(rot(q), rot(k), v, is_causal=True)
        h = x + F.linear(o.transpose(0, 1).reshape(n, d), t[f"Wo.{l}"].T)
        hn = F.rms_norm(h, (d,), t[f"g_mlp.{l}"], cfg.rms_eps)
        x = h + F.linear(F.gelu(F.linear(hn, t[f"W_up.{l}"].T), approximate="tanh"),
                         t[f"W_down.{l}"].T)
    zz = F.linear(F.rms_norm(x, (d,), t["g_final"], cfg.rms_eps), t["W_lm"].T)
    F.cross_entropy(zz[:-1], torch.tensor(tok[1:n], dtype=torch.long)).backward()
    assert tgt[-1] == tok[n]
    # the oracle's chunk 0 also has the cross-chunk target tok[n]; remove it by
    # recomputing the oracle gradient with that target masked
    tgt2 = tgt.copy(); tgt2[-1] = -1
    grads2 = O.chunk_backward(cfg, P, saved, z, tgt2)
    for name in grads2:
        assert rel(grads2[name], t[name].grad.numpy()) < 1e-11, name
    assert any(rel(grads[k], grads2[k]) > 1e-6 for k in grads)


def test_update_support_and_only_fast_weights_move(tiny):
    cfg, P, tok = tiny
    _, P2 = O.run_sequence(cfg, P, tok, eta=1e-2)
    fast = set(O.trainable_names(cfg))
    assert fast == {"W_up.3", "W_down.3"}
    for k in P:
        if k in fast:
            assert not np.array_equal(P2[k], P[k]), k
        else:
            assert np.array_equal(P2[k], P[k]), k


def test_sgd_step_linear_in_eta(tiny):
    cfg, P, tok = tiny
    ids, tgt = tok[:cfg.chunk], O.chunk_targets(tok, 0, cfg.chunk)
    st = O.init_state(cfg)
    l1, P1, _, g = O.ttt_step(cfg, P, st, ids, tgt, 1e-2)
    l2, P2, _, _ = O.ttt_step(cfg, P, st, ids, tgt, 2e-2)
    assert l1 == l2                        # chunk loss is taken before the update
    for k in O.trainable_names(cfg):
        d1, d2 = P1[k] - P[k], P2[k] - P[k]
        assert rel(d2, 2 * d1) < 1e-12
        assert rel(d1, -1e-2 * g[k]) < 1e-12


def test_chunk_causality(tiny):
    cfg, P, tok = tiny
    b = cfg.chunk
    tok2 = tok.copy()
    j = 5
    tok2[j * b + 3] = (tok2[j * b + 3] + 1) % cfg.vocab
    for eta in (0.0, 1e-2):
        la, _ = O.run_sequence(cfg, P, tok, eta)
        lb, _ = O.run_sequence(cfg, P, tok2, eta)
        assert la[:j - 1] == lb[:j - 1]       # earlier chunks untouched
        assert la[j] != lb[j]


def test_far_token_reaches_only_through_fast_weights(tiny):
    """A token beyond the stacked receptive field of chunk i (L*(k-1) positions
    before it: each windowed layer reaches k-1 further back) changes chunk i
    only when eta > 0, i.e. only through the fast weights."""
    cfg, P, tok = tiny
    cfg = O.Config(**{**cfg.__dict__, "window": 32, "chunk": 32})
    i = 10                                  # chunk 10 starts at 320
    assert 10 < i * cfg.chunk - cfg.n_layers * (cfg.window - 1)
    tok2 = tok.copy()
    tok2[10] = (tok2[10] + 7) % cfg.vocab
    la, _ = O.run_sequence(cfg, P, tok, 0.0, n_chunks=i + 1)
    lb, _ = O.run_sequence(cfg, P, tok2, 0.0, n_chunks=i + 1)
    assert la[i] == lb[i]
    la, _ = O.run_sequence(cfg, P, tok, 1e-2, n_chunks=i + 1)
    lb, _ = O.run_sequence(cfg, P, tok2, 1e-2, n_chunks=i + 1)
    assert la[i] != lb[i]


def test_cache_holds_only_window(tiny):
    cfg, P, tok = tiny
    st = O.init_state(cfg)
    for c in range(4):
        s = c * cfg.chunk
        ids = tok[s:s + cfg.chunk]
        _, P, st, _ = O.ttt_step(cfg, P, st, ids, O.chunk_targets(tok, s, len(ids)), 0.0)
        for kc, vc, pc in st["cache"]:
            assert kc.shape[1] == min(st["pos"], cfg.window - 1)
            assert pc.min() > st["pos"] - cfg.window


def test_behaviour_reported(tiny, capsys):
    """Weak behavioural check (reported, not gated): does TTT lower later losses?"""
    cfg, P, tok = tiny
    l0, _ = O.run_sequence(cfg, P, tok, 0.0)
    l1, _ = O.run_sequence(cfg, P, tok, 1e-2)
    print(f"mean loss chunks 4..7: eta=0 {np.mean(l0[4:]):.6f}  eta=1e-2 {np.mean(l1[4:]):.6f}")
    assert np.isfinite(l1).all()
