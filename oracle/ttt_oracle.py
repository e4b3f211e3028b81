"""Float64 CPU oracle of the TTT-E2E inner loop (test infrastructure only).

This module is the parity authority for the CUDA path and is used only by the
tests, by ``__graft_entry__.smoke()`` and by the benchmark's CPU-baseline leg.
It shares no code with the CUDA path: plain numpy, float64 throughout, no
blocking, fusion or reordering beyond what the definitions state.

What it computes (pages: "把 Transformer 做成“终身学习者”：TTT-E2E 如何让大模型边用边学？",
§4.2 "推理阶段（Inner Loop 复用）" and §4.4 "伪代码"; "TTT-E2E技术：突破大语言模型上下文限制的新范式",
§2.1 "参数更新机制" and §2.2 "批量更新与稳定性控制"; "测试时训练：长上下文的持续学习",
§2.1.2 "测试时训练目标"):

  for every chunk of b tokens of the text, in order:
    run the decoder forward on the chunk with sliding-window attention whose
        key/value cache holds only the last k positions (k >= b);
    take the mean next-token cross-entropy over the chunk's targets
        (the last input of a chunk predicts the first token of the next one);
    backpropagate through the last quarter of the blocks only, keeping
        gradients for their MLP weights alone;
    take one plain SGD step  W <- W - eta * dW  on those MLP weights
        (all gradients taken at the chunk's starting weights);
    keep this chunk's keys/values (computed with the chunk's starting weights)
        for the windows of later chunks.

Model (pre-norm, row-vector convention y = x.W, no biases, untied LM head):
    h = x + Attn(RMSNorm_a(x));   y = h + GELU_tanh(RMSNorm_m(h).W_up).W_down
    logits = RMSNorm_f(x_L).W_lm
Dual-MLP variant (Config.dual_mlp; "从KV Cache到权重压缩：大模型持续学习的新范式", §2.2,
a static MLP that keeps the pretrained knowledge beside a dynamic one that
adapts): in the trainable blocks
    y = h + GELU_tanh(n.W_up).W_down + GELU_tanh(n.W_up_s).W_down_s,  n = RMSNorm_m(h),
where only W_up, W_down are fast weights and the static pair stays frozen.
RMSNorm eps 1e-6, gains 1 unless loaded; RoPE rotate-half, inv_freq_i =
theta^(-2i/d_head), absolute 0-based positions; attention scale 1/sqrt(d_head);
a query at position p sees keys j with p - k < j <= p.

Pins (each function is checked in tests/test_oracle.py against something other
than itself): library routines (torch float64 rms_norm, gelu(tanh),
scaled_dot_product_attention, cross_entropy, autograd), closed forms of RoPE,
central finite differences of the hand-written backward, and the invariants of
the method (eta=0 equals one unchunked forward, k >= T equals full causal
attention, update support, linearity in eta, chunk causality).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = ["Config", "unpack", "pack", "rmsnorm", "rmsnorm_bwd", "rope_angles",
           "rope", "rope_bwd", "gelu_tanh", "gelu_tanh_grad", "attention",
           "attention_bwd", "cross_entropy", "init_state", "chunk_forward",
           "chunk_backward", "ttt_step", "run_sequence", "dense_forward_losses",
           "trainable_names", "decode", "greedy", "sampler"]


@dataclass(frozen=True)
class Config:
    n_layers: int
    d_model: int
    n_heads: int
    d_ff: int
    vocab: int
    window: int
    chunk: int
    rope_theta: float
    rms_eps: float = 1e-6
    # dual-MLP variant: each trainable block adds a frozen static MLP beside the fast one
    dual_mlp: bool = False

    @property
    def n_trainable(self) -> int:
        # "只改最后 1/4 层的 MLP" (last quarter of the blocks)
        return self.n_layers // 4

    @property
    def d_head(self) -> int:
        return self.d_model // self.n_heads

    @staticmethod
    def from_shape(s) -> "Config":
        return Config(s.n_layers, s.d_model, s.n_heads, s.d_ff, s.vocab,
                      s.window, s.chunk, s.rope_theta, s.rms_eps, getattr(s, "dual_mlp", False))


# ----------------------------------------------------------------------------
# parameter blob  (E; per layer g_attn, Wq, Wk, Wv, Wo, g_mlp, W_up, W_down;
# g_final; W_lm -- all row-major fp32)
# ----------------------------------------------------------------------------
def _layout(cfg: Config):
    d, f, V = cfg.d_model, cfg.d_ff, cfg.vocab
    out = [("E", (V, d))]
    for l in range(cfg.n_layers):
        out += [(f"g_attn.{l}", (d,)), (f"Wq.{l}", (d, d)), (f"Wk.{l}", (d, d)),
                (f"Wv.{l}", (d, d)), (f"Wo.{l}", (d, d)), (f"g_mlp.{l}", (d,)),
                (f"W_up.{l}", (d, f)), (f"W_down.{l}", (f, d))]
        if cfg.dual_mlp and l >= cfg.n_layers - cfg.n_trainable:
            out += [(f"W_up_s.{l}", (d, f)), (f"W_down_s.{l}", (f, d))]
    return out + [("g_final", (d,)), ("W_lm", (d, V))]


def unpack(blob, cfg: Config) -> dict:
    """fp32/fp64 flat blob -> dict of float64 arrays (copies)."""
    blob = np.asarray(blob)
    P, off = {}, 0
    for name, shp in _layout(cfg):
        n = int(np.prod(shp))
        P[name] = blob[off:off + n].astype(np.float64).reshape(shp)
        off += n
    if off != blob.size:
        raise ValueError(f"blob has {blob.size} floats, layout needs {off}")
    return P


def pack(P: dict, cfg: Config) -> np.ndarray:
    return np.concatenate([np.asarray(P[n], np.float64).ravel() for n, _ in _layout(cfg)])


def trainable_names(cfg: Config):
    """W_up / W_down of blocks L-S .. L-1: the fast weights."""
    L, S = cfg.n_layers, cfg.n_trainable
    return [n for l in range(L - S, L) for n in (f"W_up.{l}", f"W_down.{l}")]


# ----------------------------------------------------------------------------
# components
# ----------------------------------------------------------------------------
def rmsnorm(x, g, eps):
    """y = x * g / sqrt(mean(x^2) + eps); also returns r = 1/sqrt(mean(x^2)+eps)."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * g, r


def rmsnorm_bwd(dy, x, g, r):
    """Gradient w.r.t. x of y = x*g*r(x) (g frozen).

    dx_j = r g_j dy_j - x_j r^3 / d * sum_i dy_i g_i x_i
    """
    d = x.shape[-1]
    s = np.sum(dy * g * x, axis=-1, keepdims=True)
    return r * g * dy - x * (r ** 3) * s / d


def rope_angles(pos, d_head, theta):
    """angle[p, i] = pos_p * theta^(-2i/d_head), i < d_head/2 (float64)."""
    i = np.arange(d_head // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d_head)
    return np.asarray(pos, np.float64)[:, None] * inv_freq[None, :]


def rope(x, ang):
    """Rotate-half RoPE on x[..., n, d_head] with pairs (i, i + d_head/2)."""
    h = x.shape[-1] // 2
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_bwd(dy, ang):
    """Transpose of the rotation: gradient of rope() w.r.t. its input."""
    h = dy.shape[-1] // 2
    c, s = np.cos(ang), np.sin(ang)
    d1, d2 = dy[..., :h], dy[..., h:]
    return np.concatenate([d1 * c + d2 * s, d2 * c - d1 * s], axis=-1)


_GC = math.sqrt(2.0 / math.pi)


def gelu_tanh(a):
    """0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3)))."""
    return 0.5 * a * (1.0 + np.tanh(_GC * (a + 0.044715 * a ** 3)))


def gelu_tanh_grad(a):
    t = np.tanh(_GC * (a + 0.044715 * a ** 3))
    return 0.5 * (1.0 + t) + 0.5 * a * (1.0 - t * t) * _GC * (1.0 + 3 * 0.044715 * a * a)


def _window_mask(qpos, kpos, window):
    qp = np.asarray(qpos)[:, None]
    kp = np.asarray(kpos)[None, :]
    return (kp <= qp) & (kp > qp - window)


def attention(q, k, v, qpos, kpos, window):
    """Sliding-window causal attention, one head at a time.

    q [H, n, dh]; k, v [H, m, dh]; key j is visible to query p iff
    p - window < pos_j <= pos_p.  Returns o [H, n, dh] and the per-row
    log-sum-exp lse [H, n] of the scaled scores.
    """
    H, n, dh = q.shape
    scale = 1.0 / math.sqrt(dh)
    mask = _window_mask(qpos, kpos, window)
    o = np.empty_like(q)
    lse = np.empty((H, n))
    for hh in range(H):
        s = (q[hh] @ k[hh].T) * scale
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        o[hh] = (e / l) @ v[hh]
        lse[hh] = (m + np.log(l))[:, 0]
    return o, lse


def attention_bwd(do, q, k, v, qpos, kpos, window):
    """Gradients of attention() w.r.t. q, k, v (all keys), given dO.

    P = softmax(s), dV = P^T dO, dP = dO V^T, dS = P (dP - rowsum(P dP)),
    dQ = dS K / sqrt(dh), dK = dS^T Q / sqrt(dh).
    """
    H, n, dh = q.shape
    scale = 1.0 / math.sqrt(dh)
    mask = _window_mask(qpos, kpos, window)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for hh in range(H):
        s = np.where(mask, (q[hh] @ k[hh].T) * scale, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dv[hh] = p.T @ do[hh]
        dp = do[hh] @ v[hh].T
        ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
        dq[hh] = ds @ k[hh] * scale
        dk[hh] = ds.T @ q[hh] * scale
    return dq, dk, dv


def cross_entropy(z, tgt):
    """Per-row loss lse(z) - z[tgt] (nan where tgt < 0) and softmax(z)."""
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    ssum = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(ssum))[:, 0]
    loss = np.full(z.shape[0], np.nan)
    ok = tgt >= 0
    loss[ok] = lse[ok] - z[np.nonzero(ok)[0], tgt[ok]]
    return loss, e / ssum


# ----------------------------------------------------------------------------
# the chunked inner loop
# ----------------------------------------------------------------------------
def _heads(x, H):
    n, d = x.shape
    return x.reshape(n, H, d // H).transpose(1, 0, 2)


def _merge(x):
    H, n, dh = x.shape
    return x.transpose(1, 0, 2).reshape(n, H * dh)


def init_state(cfg: Config):
    """Per-layer window cache: keys/values (post-RoPE) and their positions."""
    H, dh = cfg.n_heads, cfg.d_head
    return {"pos": 0,
            "cache": [(np.zeros((H, 0, dh)), np.zeros((H, 0, dh)),
                       np.zeros(0, np.int64)) for _ in range(cfg.n_layers)]}


def chunk_forward(cfg: Config, P: dict, state, ids, keep=True):
    """Forward of one chunk; returns (logits z, saved activations, new k/v)."""
    L, H = cfg.n_layers, cfg.n_heads
    n = len(ids)
    pos = state["pos"] + np.arange(n)
    ang = rope_angles(pos, cfg.d_head, cfg.rope_theta)
    x = P["E"][np.asarray(ids)]
    acts, new_kv = [], []
    for l in range(L):
        xn_a, r_a = rmsnorm(x, P[f"g_attn.{l}"], cfg.rms_eps)
        q = rope(_heads(xn_a @ P[f"Wq.{l}"], H), ang)
        k = rope(_heads(xn_a @ P[f"Wk.{l}"], H), ang)
        v = _heads(xn_a @ P[f"Wv.{l}"], H)
        kc, vc, pc = state["cache"][l]
        kall = np.concatenate([kc, k], axis=1)
        vall = np.concatenate([vc, v], axis=1)
        pall = np.concatenate([pc, pos])
        o, _ = attention(q, kall, vall, pos, pall, cfg.window)
        h = x + _merge(o) @ P[f"Wo.{l}"]
        xn_m, r_m = rmsnorm(h, P[f"g_mlp.{l}"], cfg.rms_eps)
        a = xn_m @ P[f"W_up.{l}"]
        u = gelu_tanh(a)
        y = h + u @ P[f"W_down.{l}"]
        a_s = None
        if cfg.dual_mlp and l >= L - cfg.n_trainable:   # static MLP on the same normalised input
            a_s = xn_m @ P[f"W_up_s.{l}"]
            y = y + gelu_tanh(a_s) @ P[f"W_down_s.{l}"]
        if keep and l >= L - cfg.n_trainable:
            acts.append(dict(x=x, r_a=r_a, q=q, kall=kall, vall=vall, pall=pall,
                             h=h, xn_m=xn_m, r_m=r_m, a=a, u=u, a_s=a_s))
        else:
            acts.append(None)
        new_kv.append((k, v))
        x = y
    xf, r_f = rmsnorm(x, P["g_final"], cfg.rms_eps)
    z = xf @ P["W_lm"]
    return z, dict(acts=acts, xL=x, r_f=r_f, pos=pos, ang=ang), new_kv


def chunk_backward(cfg: Config, P: dict, saved, z, tgt):
    """Hand-written backward of the mean chunk loss; grads of fast weights only."""
    L, S, H = cfg.n_layers, cfg.n_trainable, cfg.n_heads
    tgt = np.asarray(tgt)
    ok = tgt >= 0
    nv = int(ok.sum())
    _, p = cross_entropy(z, tgt)
    dz = p.copy()
    dz[np.nonzero(ok)[0], tgt[ok]] -= 1.0
    dz[~ok] = 0.0
    dz /= max(nv, 1)
    dx = rmsnorm_bwd(dz @ P["W_lm"].T, saved["xL"], P["g_final"], saved["r_f"])
    pos, ang = saved["pos"], saved["ang"]
    grads = {}
    for l in range(L - 1, L - S - 1, -1):
        A = saved["acts"][l]
        dy = dx
        du = dy @ P[f"W_down.{l}"].T
        grads[f"W_down.{l}"] = A["u"].T @ dy
        da = du * gelu_tanh_grad(A["a"])
        grads[f"W_up.{l}"] = A["xn_m"].T @ da
        if l == L - S:
            break       # the first trainable block's attention needs no backward
        dxn_m = da @ P[f"W_up.{l}"].T
        if A["a_s"] is not None:   # the static MLP passes gradient to h; its weights stay frozen
            dxn_m = dxn_m + ((dy @ P[f"W_down_s.{l}"].T) * gelu_tanh_grad(A["a_s"])) @ P[f"W_up_s.{l}"].T
        dh = dy + rmsnorm_bwd(dxn_m, A["h"], P[f"g_mlp.{l}"], A["r_m"])
        do = _heads(dh @ P[f"Wo.{l}"].T, H)
        dq, dk, dv = attention_bwd(do, A["q"], A["kall"], A["vall"], pos, A["pall"],
                                   cfg.window)
        n = len(pos)
        dq = rope_bwd(dq, ang)
        dk = rope_bwd(dk[:, -n:], ang)     # cached keys are constants of W_c
        dv = dv[:, -n:]
        dxn = (_merge(dq) @ P[f"Wq.{l}"].T + _merge(dk) @ P[f"Wk.{l}"].T
               + _merge(dv) @ P[f"Wv.{l}"].T)
        dx = dh + rmsnorm_bwd(dxn, A["x"], P[f"g_attn.{l}"], A["r_a"])
    return grads


def _commit(cfg: Config, state, new_kv, n):
    """Append the chunk's k/v; keep only what later windows can still see."""
    end = state["pos"] + n
    pos = state["pos"] + np.arange(n)
    cache = []
    for (kc, vc, pc), (k, v) in zip(state["cache"], new_kv):
        kall = np.concatenate([kc, k], axis=1)
        vall = np.concatenate([vc, v], axis=1)
        pall = np.concatenate([pc, pos])
        keep = pall > end - cfg.window
        cache.append((kall[:, keep], vall[:, keep], pall[keep]))
    return {"pos": end, "cache": cache}


def chunk_targets(tokens, start, n):
    """Next-token targets of positions start..start+n-1 (-1 past the end)."""
    T = len(tokens)
    idx = start + 1 + np.arange(n)
    return np.where(idx < T, np.asarray(tokens)[np.minimum(idx, T - 1)], -1)


def chunk_loss(z, tgt):
    loss, _ = cross_entropy(z, np.asarray(tgt))
    ok = np.asarray(tgt) >= 0
    return float(loss[ok].mean()) if ok.any() else 0.0


def ttt_step(cfg: Config, P: dict, state, ids, tgt, eta):
    """One inner-loop step: forward, loss, suffix backward, SGD, cache commit.

    Returns (loss, new params, new state, grads).
    """
    z, saved, new_kv = chunk_forward(cfg, P, state, ids)
    loss = chunk_loss(z, tgt)
    grads = chunk_backward(cfg, P, saved, z, tgt)
    P2 = dict(P)
    for name, g in grads.items():
        P2[name] = P[name] - eta * g
    return loss, P2, _commit(cfg, state, new_kv, len(ids)), grads


def run_sequence(cfg: Config, P: dict, tokens, eta, n_chunks=None, chunk=None,
                 trace=False):
    """The chunked inner loop over ``tokens``.

    Returns (per-chunk losses, final params[, fast weights after every chunk]).
    """
    b = chunk or cfg.chunk
    T = len(tokens)
    nc = int(math.ceil(T / b)) if n_chunks is None else n_chunks
    state = init_state(cfg)
    losses, hist = [], []
    for c in range(nc):
        s = c * b
        n = min(b, T - s)
        ids = np.asarray(tokens[s:s + n])
        loss, P, state, _ = ttt_step(cfg, P, state, ids, chunk_targets(tokens, s, n), eta)
        losses.append(loss)
        if trace:
            hist.append({k: P[k].copy() for k in trainable_names(cfg)})
    return (losses, P, hist) if trace else (losses, P)


def dense_forward_losses(cfg: Config, P: dict, tokens, chunk=None):
    """Frozen model, whole sequence in one pass (T x T band mask), no cache.

    Returns the per-chunk mean losses the chunked loop must reproduce at eta=0.
    """
    b = chunk or cfg.chunk
    T = len(tokens)
    pos = np.arange(T)
    ang = rope_angles(pos, cfg.d_head, cfg.rope_theta)
    H = cfg.n_heads
    x = P["E"][np.asarray(tokens)]
    for l in range(cfg.n_layers):
        xn, _ = rmsnorm(x, P[f"g_attn.{l}"], cfg.rms_eps)
        q = rope(_heads(xn @ P[f"Wq.{l}"], H), ang)
        k = rope(_heads(xn @ P[f"Wk.{l}"], H), ang)
        v = _heads(xn @ P[f"Wv.{l}"], H)
        o, _ = attention(q, k, v, pos, pos, cfg.window)
        h = x + _merge(o) @ P[f"Wo.{l}"]
        xn_m, _ = rmsnorm(h, P[f"g_mlp.{l}"], cfg.rms_eps)
        y = h + gelu_tanh(xn_m @ P[f"W_up.{l}"]) @ P[f"W_down.{l}"]
        if cfg.dual_mlp and l >= cfg.n_layers - cfg.n_trainable:
            y = y + gelu_tanh(xn_m @ P[f"W_up_s.{l}"]) @ P[f"W_down_s.{l}"]
        x = y
    xf, _ = rmsnorm(x, P["g_final"], cfg.rms_eps)
    loss, _ = cross_entropy(xf @ P["W_lm"], chunk_targets(tokens, 0, T))
    out = []
    for s in range(0, T, b):
        seg = loss[s:s + b]
        seg = seg[~np.isnan(seg)]
        out.append(float(seg.mean()) if seg.size else 0.0)
    return out


# ----------------------------------------------------------------------------
# decode-phase TTT
# ----------------------------------------------------------------------------
def greedy(z_row, i):
    """Pick the first index of the largest logit (the i-th generated token)."""
    return int(np.argmax(z_row))


def sampler(u, temp):
    """Pick the i-th generated token from softmax(z / temp) by inverse CDF at the
    caller's uniform u[i] in [0, 1): the first index whose cumulative weight
    exceeds u[i] times the total."""
    def pick(z_row, i):
        y = np.asarray(z_row, np.float64) / temp
        c = np.cumsum(np.exp(y - y.max()))
        return int(np.searchsorted(c, u[i] * c[-1], side="right"))
    return pick


def decode(cfg: Config, P: dict, prompt, n_new, eta, pick, trace=False):
    """Decode-phase TTT: prefill the prompt with the chunked inner loop, then
    generate n_new tokens, taking one inner-loop step after every chunk of b
    generated tokens (pages: "TTT-E2E技术：突破大语言模型上下文限制的新范式", §2.2
    "批量更新与稳定性控制", one update per 1000 input tokens while prefilling and one
    per 1000 output tokens while generating; "把 Transformer 做成“终身学习者”", §4.2,
    the inner loop reused at inference).

    Readings where the pages are silent:
      * the prompt goes through the chunked inner loop exactly as run_sequence
        does; its last position has no target;
      * the token at position t is picked from the logits of position t - 1, as
        computed by the forward of t - 1's chunk (before that chunk's update); the
        first generated token comes from the prompt's last position;
      * generated tokens form chunks of b starting at the first generated
        position; a complete chunk takes one step (forward, mean next-token
        cross-entropy over its b positions, suffix backward, SGD, cache commit),
        and its last position's target is the token picked after it, from the
        logits of that position before the update; an incomplete last chunk
        takes no step;
      * pick(z_row, i) chooses the i-th generated token (i = 0 for the first);
        random numbers, if any, are the caller's (see sampler).

    Returns a dict: tokens (the n_new generated ids), next (the id picked after
    them), prefill_losses, gen_losses, P (final parameters), state, and with
    trace=True, hist: the fast weights after every step, prompt chunks first,
    and z: the logits row behind every pick (n_new + 1 rows).
    """
    b = cfg.chunk
    prompt = np.asarray(prompt)
    T = len(prompt)
    if T < 1:
        raise ValueError("decode needs a prompt of at least one token")
    state = init_state(cfg)
    names = trainable_names(cfg)
    hist, pre_losses, gen_losses = [], [], []

    def step(P, state, ids, tgt):
        z, saved, new_kv = chunk_forward(cfg, P, state, ids)
        loss = chunk_loss(z, tgt)
        grads = chunk_backward(cfg, P, saved, z, tgt)
        P2 = dict(P)
        for name, g in grads.items():
            P2[name] = P[name] - eta * g
        if trace:
            hist.append({k: P2[k].copy() for k in names})
        return loss, P2, _commit(cfg, state, new_kv, len(ids)), z

    z_last = None
    for s in range(0, T, b):
        n = min(b, T - s)
        loss, P, state, z = step(P, state, prompt[s:s + n], chunk_targets(prompt, s, n))
        pre_losses.append(loss)
        z_last = z[-1]

    out, cur, rows = [], [], []

    def pick_from(z_row, i):
        rows.append(z_row)
        return pick(z_row, i)

    nxt = pick_from(z_last, 0)
    for i in range(n_new):
        out.append(nxt)
        cur.append(nxt)
        # the current chunk so far, with its starting weights: the row of the newest token
        z, _, _ = chunk_forward(cfg, P, state, np.asarray(cur), keep=False)
        nxt = pick_from(z[-1], i + 1)
        if len(cur) == b:
            ids = np.asarray(cur)
            loss, P, state, _ = step(P, state, ids, np.append(ids[1:], nxt))
            gen_losses.append(loss)
            cur = []
    res = dict(tokens=out, next=nxt, prefill_losses=pre_losses, gen_losses=gen_losses, P=P, state=state)
    if trace:
        res["hist"] = hist
        res["z"] = np.stack(rows)
    return res
