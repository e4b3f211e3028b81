"""Pins of the oracle's decode-phase TTT against an independent model.

The check model is a dense forward over the whole text, assembled from torch
library routines in float64: no window cache and no chunk loop.  Row t's
trainable MLPs use the fast weights of t's chunk (a weight schedule), which is
what the inner loop means by "keys and values computed with the chunk's
starting weights".  Against it, every generated token must be the pick from
the previous row's logits, every step's update must equal -eta times the torch
autograd gradient of that chunk's mean next-token loss, and every chunk loss
must match.  With eta = 0 greedy decoding must equal plain greedy generation
from the frozen model.
"""
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


def small(chunk=8, window=16):
    s = SHAPES["tiny"]
    c = O.Config.from_shape(s)
    cfg = O.Config(**{**c.__dict__, "chunk": chunk, "window": window})
    return cfg, O.unpack(weight_blob(s), cfg), sequence_tokens(s)


def chunk_rows(T, n_text, b):
    """Row ranges of the prompt's chunks (from 0) and the generation chunks (from T)."""
    out = [(s, min(s + b, T)) for s in range(0, T, b)]
    s = T
    while s < n_text:
        out.append((s, min(s + b, n_text)))
        s += b
    return out


def torch_logits(cfg, P, text, sched, rows):
    """Dense forward over text; rows[c] = (start, end) uses the fast weights sched[c]."""
    T, H, dh, d = len(text), cfg.n_heads, cfg.d_head, cfg.d_model
    L, S = cfg.n_layers, cfg.n_trainable
    t = {k: torch.tensor(v) for k, v in P.items()}
    pos = torch.arange(T, dtype=torch.float64)
    inv = cfg.rope_theta ** (-2.0 * torch.arange(dh // 2, dtype=torch.float64) / dh)
    ang = pos[:, None] * inv[None]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(x):
        x1, x2 = x[..., :dh // 2], x[..., dh // 2:]
        return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], -1)

    qp, kp = np.arange(T)[:, None], np.arange(T)[None, :]
    mask = torch.tensor((kp <= qp) & (kp > qp - cfg.window))
    x = t["E"][torch.tensor(np.asarray(text), dtype=torch.long)]
    for l in range(L):
        xn = F.rms_norm(x, (d,), t[f"g_attn.{l}"], cfg.rms_eps)
        q, k, v = (F.linear(xn, t[f"W{c}.{l}"].T).view(T, H, dh).transpose(0, 1) for c in "qkv")
        o = F.scaled_dot_product_attention(rot(q), rot(k), v, attn_mask=mask)
        h = x + F.linear(o.transpose(0, 1).reshape(T, d), t[f"Wo.{l}"].T)
        hn = F.rms_norm(h, (d,), t[f"g_mlp.{l}"], cfg.rms_eps)
        if l < L - S:
            mlp = F.linear(F.gelu(F.linear(hn, t[f"W_up.{l}"].T), approximate="tanh"), t[f"W_down.{l}"].T)
        else:
            parts = []
            for c, (a, e) in enumerate(rows):
                if a >= T:
                    break
                e = min(e, T)
                up, down = sched[c][f"W_up.{l}"], sched[c][f"W_down.{l}"]
                parts.append(F.linear(F.gelu(F.linear(hn[a:e], up.T), approximate="tanh"), down.T))
            mlp = torch.cat(parts)
        x = h + mlp
    return F.linear(F.rms_norm(x, (d,), t["g_final"], cfg.rms_eps), t["W_lm"].T)


def schedule(cfg, P, hist, n_rows):
    """Fast weights of every chunk: the initial ones, then after each step."""
    names = O.trainable_names(cfg)
    w = [{k: torch.tensor(P[k]) for k in names}]
    w += [{k: torch.tensor(h[k]) for k in names} for h in hist]
    return w + [w[-1]] * max(0, n_rows - len(w))


@pytest.mark.parametrize("T,n_new", [(16, 16), (20, 19), (1, 9), (8, 3)])
def test_eta0_greedy_equals_greedy_generation_of_the_frozen_model(T, n_new):
    cfg, P, tok = small()
    r = O.decode(cfg, P, tok[:T], n_new, 0.0, O.greedy)
    text = list(tok[:T])
    names = O.trainable_names(cfg)
    frozen = [{k: torch.tensor(P[k]) for k in names}] * 64
    for i in range(n_new + 1):
        z = torch_logits(cfg, P, text, frozen, chunk_rows(T, len(text), cfg.chunk))[-1]
        got = r["tokens"][i] if i < n_new else r["next"]
        assert float(z[got]) >= float(z.max()) - 1e-9, i     # the largest logit (ties allowed)
        text.append(got)


@pytest.mark.parametrize("T,n_new", [(16, 16), (20, 19), (5, 17)])
def test_updates_tokens_and_losses_match_the_weight_schedule_model(T, n_new):
    cfg, P, tok = small()
    eta, temp = 0.05, 0.8
    u = np.random.default_rng(T * 31 + n_new).random(n_new + 1)
    r = O.decode(cfg, P, tok[:T], n_new, eta, O.sampler(u, temp), trace=True)
    text = list(tok[:T]) + list(r["tokens"]) + [r["next"]]
    b = cfg.chunk
    rows = chunk_rows(T, T + n_new, b)
    n_pc = len(range(0, T, b))
    n_gc = n_new // b
    assert len(r["hist"]) == n_pc + n_gc
    assert len(r["prefill_losses"]) == n_pc and len(r["gen_losses"]) == n_gc
    sched = schedule(cfg, P, r["hist"], len(rows))

    # the logits behind every pick are the previous row's under the schedule, and every
    # generated token is the inverse-CDF pick from them
    z_all = torch_logits(cfg, P, text[:T + n_new], sched, rows)
    want = z_all[T - 1:T + n_new].detach().numpy()
    assert np.linalg.norm(r["z"] - want) <= 1e-11 * np.linalg.norm(want)
    for i in range(n_new + 1):
        z = z_all[T + i - 1] / temp
        c = torch.cumsum(torch.softmax(z, 0), 0)
        k = text[T + i]
        lo = float(c[k - 1]) if k > 0 else 0.0
        assert lo <= u[i] * float(c[-1]) < float(c[k]) + 1e-12, i

    # every step: W_{c+1} = W_c - eta * d(mean loss of chunk c)/dW_c, and the loss itself
    names = O.trainable_names(cfg)
    losses = list(r["prefill_losses"]) + list(r["gen_losses"])
    for c in range(n_pc + n_gc):
        a, e = rows[c]
        leaf = {k: sched[c][k].clone().requires_grad_(True) for k in names}
        sc = sched[:c] + [leaf] + sched[c + 1:]
        z = torch_logits(cfg, P, text[:e], sc, rows)
        tgt = [text[t + 1] if (t + 1 < len(text) and not (c == n_pc - 1 and t + 1 == T)) else -1
               for t in range(a, e)]
        ok = [i for i, y in enumerate(tgt) if y >= 0]
        loss = F.cross_entropy(z[a:e][ok], torch.tensor([tgt[i] for i in ok], dtype=torch.long))
        loss.backward()
        assert abs(float(loss.detach()) - losses[c]) <= 1e-10 * abs(losses[c]), c
        for k in names:
            want = sched[c][k] - eta * leaf[k].grad
            err = float(torch.linalg.norm(torch.tensor(r["hist"][c][k]) - want) / torch.linalg.norm(want))
            assert err < 1e-12, (c, k, err)


def test_no_step_for_an_incomplete_generation_chunk():
    cfg, P, tok = small()
    r0 = O.decode(cfg, P, tok[:16], 0, 0.05, O.greedy, trace=True)
    r1 = O.decode(cfg, P, tok[:16], cfg.chunk - 1, 0.05, O.greedy, trace=True)
    assert r1["gen_losses"] == [] and len(r1["hist"]) == len(r0["hist"])
    for k in O.trainable_names(cfg):
        assert np.array_equal(r1["P"][k], r0["P"][k])
    assert r1["tokens"][0] == r0["next"]


def test_sampler_limits():
    z = np.array([0.0, 1.0, 2.0])
    assert O.sampler([0.0], 1.0)(z, 0) == 0
    assert O.sampler([1.0 - 1e-15], 1.0)(z, 0) == 2
    # a uniform landing exactly on a cumulative weight picks the next index (weight must exceed it)
    assert O.sampler([0.5], 1.0)(np.zeros(2), 0) == 1
    # a low temperature concentrates the mass on the largest logit
    assert O.sampler([0.5], 1e-3)(z, 0) == 2
