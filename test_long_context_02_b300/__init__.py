"""Python binding of libttt (TTT-E2E inner-loop prefill on one B300, sm_103a).

Argument marshalling only: every step of the path runs in the CUDA kernels of
libttt.so, reached through its C ABI (include/ttt.h, include/ttt_kernels.h).
Device buffers are torch CUDA tensors passed by pointer; torch provides memory
and streams, nothing else.  Importing fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libttt.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python test_long_context_02_b300/build.py` "
                      "(there is no fallback implementation)")
lib = ctypes.CDLL(LIB_PATH)

TTT_OK, TTT_ERR_ARG, TTT_ERR_UNSUPPORTED, TTT_ERR_STATE = 0, -1, -2, -3
TTT_ERR_OOM, TTT_ERR_CUDA, TTT_ERR_DEVICE, TTT_ERR_SCRATCH = -4, -5, -6, -7
ERR_NAMES = {0: "OK", -1: "TTT_ERR_ARG", -2: "TTT_ERR_UNSUPPORTED", -3: "TTT_ERR_STATE",
             -4: "TTT_ERR_OOM", -5: "TTT_ERR_CUDA", -6: "TTT_ERR_DEVICE", -7: "TTT_ERR_SCRATCH"}
CE_STATIC_SCRATCH_ENTRIES = 524288

EPI_F32, EPI_OPND, EPI_RESID, EPI_GELU, EPI_GELU_BWD, EPI_SGD, EPI_CE_FWD, EPI_CE_BWD = range(8)

_vp, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float


class TTTError(RuntimeError):
    def __init__(self, code, msg=""):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


class ttt_config(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("n_trainable", _i32), ("d_model", _i32), ("n_heads", _i32),
                ("d_ff", _i32), ("vocab", _i32), ("window", _i32), ("chunk", _i32), ("n_seqs", _i32),
                ("rope_theta", ctypes.c_double), ("rms_eps", _f32), ("eta", _f32), ("compute", _i32),
                ("dual_mlp", _i32)]


class ttt_gemm_epilogue(ctypes.Structure):
    _fields_ = [("out32", _vp), ("ldo32", _i64), ("out_hi", _vp), ("out_lo", _vp), ("ldo", _i64),
                ("resid", _vp), ("ldr", _i64), ("aux", _vp), ("ldaux", _i64),
                ("w32", _vp), ("w_hi", _vp), ("w_lo", _vp), ("ldw", _i64), ("eta", _f32),
                ("tgt", _vp), ("part", _vp), ("zt", _vp), ("lse", _vp), ("scale", _f32),
                ("err", _vp), ("allow_ksplit", _i32)]


def _sig(name, restype, *argtypes):
    f = getattr(lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


ttt_k_gemm = _sig("ttt_k_gemm", ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  _vp, _vp, _i64, ctypes.c_int, _vp, _vp, _i64, ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(ttt_gemm_epilogue), _vp)


def ptr(t):
    """Device (or host) address of a torch tensor / numpy array, 0 for None."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream


def check(code, what=""):
    if code != TTT_OK:
        raise TTTError(code, what)
    return code


def gemm(epi, M, N, K, a, b, *, a_lo=None, b_lo=None, lda=None, ldb=None, a_mn=0, b_mn=0, split=False,
         stream=None, **epilogue):
    """ttt_k_gemm on torch tensors; epilogue fields by name (tensors or scalars)."""
    e = ttt_gemm_epilogue()
    for k, v in epilogue.items():
        if k in ("ldo32", "ldo", "ldr", "ldaux", "ldw", "eta", "scale", "allow_ksplit"):
            setattr(e, k, v)
        else:
            setattr(e, k, ptr(v))
    lda = lda if lda is not None else a.shape[-1]
    ldb = ldb if ldb is not None else b.shape[-1]
    return check(ttt_k_gemm(epi, M, N, K, ptr(a), ptr(a_lo), lda, a_mn, ptr(b), ptr(b_lo), ldb, b_mn,
                            int(split), ctypes.byref(e), _stream(stream)), "ttt_k_gemm")


_attn_ptrs = [_vp] * 10
ttt_k_attn_fwd = _sig("ttt_k_attn_fwd", ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      _i64, ctypes.c_int, *_attn_ptrs, _vp, _vp, _vp, _vp, _vp)
ttt_k_attn_bwd = _sig("ttt_k_attn_bwd", ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      _i64, ctypes.c_int, *_attn_ptrs, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
ttt_k_attn_rowdot = _sig("ttt_k_attn_rowdot", ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                         _vp, _vp, _vp, _vp, _vp, _vp)

# No-allocation variant of the LM-head cross-entropy statistics (scratch in a
# static device array of the library; see include/ttt_kernels.h).
ttt_k_lmhead_ce_static = _sig("ttt_k_lmhead_ce_static", ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              _vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp, _vp)

# A bounded wait that runs out on purpose (failure detection without a fault).
ttt_k_wait_limit_probe = _sig("ttt_k_wait_limit_probe", ctypes.c_int, _vp, _vp, _vp)

ttt_create = _sig("ttt_create", ctypes.c_int, ctypes.POINTER(ttt_config), _vp, ctypes.POINTER(_vp))
ttt_load_weights = _sig("ttt_load_weights", ctypes.c_int, _vp, _vp, ctypes.c_size_t)
ttt_prefill_chunk = _sig("ttt_prefill_chunk", ctypes.c_int, _vp, _vp, _i32, _vp, _vp)
ttt_prefill_chunk_dev = _sig("ttt_prefill_chunk_dev", ctypes.c_int, _vp, _vp, _i32, _vp, _vp)
ttt_prefill_sequence_dev = _sig("ttt_prefill_sequence_dev", ctypes.c_int, _vp, _vp, _i32, _vp)
ttt_prefill_sequence = _sig("ttt_prefill_sequence", ctypes.c_int, _vp, _vp, _i32, _vp)
ttt_decode_dev = _sig("ttt_decode_dev", ctypes.c_int, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _vp)
ttt_sync = _sig("ttt_sync", ctypes.c_int, _vp)
ttt_get_fast_weights = _sig("ttt_get_fast_weights", ctypes.c_int, _vp, _i32, _i32, _vp, _vp)
ttt_position = _sig("ttt_position", _i64, _vp)
ttt_destroy = _sig("ttt_destroy", None, _vp)
ttt_last_error = _sig("ttt_last_error", ctypes.c_char_p, _vp)
ttt_reset = _sig("ttt_reset", ctypes.c_int, _vp)
ttt_get_window = _sig("ttt_get_window", ctypes.c_int, _vp, _i32, _i32, _vp, _vp, _vp)
ttt_launch_count = _sig("ttt_launch_count", _i64, _vp)
ttt_set_concurrency = _sig("ttt_set_concurrency", ctypes.c_int, _vp, _i32)
ttt_state_bytes = _sig("ttt_state_bytes", _i64, _vp)
ttt_export_state = _sig("ttt_export_state", ctypes.c_int, _vp, _i32, _vp, ctypes.c_size_t)
ttt_import_state = _sig("ttt_import_state", ctypes.c_int, _vp, _i32, _vp, ctypes.c_size_t)


class ttt_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", _i64), ("ms", ctypes.c_double),
                ("alg_flops", ctypes.c_double), ("exec_flops", ctypes.c_double), ("bytes", ctypes.c_double)]


ttt_profile = _sig("ttt_profile", ctypes.c_int, _vp, _i64)
ttt_profile_sample = _sig("ttt_profile_sample", ctypes.c_int, _vp, _i32)
ttt_profile_class_name = _sig("ttt_profile_class_name", ctypes.c_char_p, ctypes.c_int)


def profile_classes():
    """Names of the kernel classes, in class-id order (bit i of a profile mask)."""
    out, i = [], 0
    while True:
        n = ttt_profile_class_name(i)
        if n is None:
            return out
        out.append(n.decode())
        i += 1
ttt_profile_read = _sig("ttt_profile_read", ctypes.c_int, _vp, ctypes.POINTER(ttt_kernel_stat), ctypes.c_int,
                        ctypes.POINTER(ctypes.c_int))


def attn_fwd(n, H, dh, window, pos0, q, kc, vc, ko, vo, o, lse=None, *, split=False, lo=None, err=None,
             stream=None):
    """ttt_k_attn_fwd; lo = dict of remainder tensors keyed q, kc, vc, ko, vo, o (split mode)."""
    lo = lo or {}
    return check(ttt_k_attn_fwd(n, H, dh, window, pos0, int(split),
                                ptr(q), ptr(lo.get("q")), ptr(kc), ptr(lo.get("kc")), ptr(vc), ptr(lo.get("vc")),
                                ptr(ko), ptr(lo.get("ko")), ptr(vo), ptr(lo.get("vo")),
                                ptr(o), ptr(lo.get("o")), ptr(lse), ptr(err), _stream(stream)), "ttt_k_attn_fwd")


def attn_bwd(n, H, dh, window, pos0, q, kc, vc, ko, vo, do, lse, D, dq, dk, dv, *, split=False, lo=None,
             err=None, stream=None):
    lo = lo or {}
    return check(ttt_k_attn_bwd(n, H, dh, window, pos0, int(split),
                                ptr(q), ptr(lo.get("q")), ptr(kc), ptr(lo.get("kc")), ptr(vc), ptr(lo.get("vc")),
                                ptr(ko), ptr(lo.get("ko")), ptr(vo), ptr(lo.get("vo")),
                                ptr(do), ptr(lo.get("do")), ptr(lse), ptr(D), ptr(dq), ptr(dk), ptr(dv),
                                ptr(err), _stream(stream)), "ttt_k_attn_bwd")


def attn_rowdot(n, H, dh, do, o, D, *, do_lo=None, o_lo=None, stream=None):
    return check(ttt_k_attn_rowdot(n, H, dh, ptr(do), ptr(do_lo), ptr(o), ptr(o_lo), ptr(D), _stream(stream)),
                 "ttt_k_attn_rowdot")


def wait_limit_probe(err, status, *, stream=None):
    """ttt_k_wait_limit_probe: err [1] and status [4] int32 device tensors."""
    return check(ttt_k_wait_limit_probe(ptr(err), ptr(status), _stream(stream)), "ttt_k_wait_limit_probe")


def lmhead_ce_static(M, K, V, x, w_lm, tgt, lse, loss, *, ldx=None, ldw=None, err=None, stream=None):
    """ttt_k_lmhead_ce_static on torch tensors: lse / loss [M] fp32 from x [M][K] and W_lm [K][V] (bf16)."""
    ldx = ldx if ldx is not None else x.shape[-1]
    ldw = ldw if ldw is not None else w_lm.shape[-1]
    return check(ttt_k_lmhead_ce_static(M, K, V, ptr(x), ldx, ptr(w_lm), ldw, ptr(tgt), ptr(lse), ptr(loss),
                                        ptr(err), _stream(stream)), "ttt_k_lmhead_ce_static")


def make_config(n_layers, d_model, n_heads, d_ff, vocab, window, chunk, rope_theta, eta, n_seqs=1,
                compute="bf16", rms_eps=1e-6, n_trainable=None, dual_mlp=False):
    c = ttt_config()
    c.n_layers, c.d_model, c.n_heads, c.d_ff, c.vocab = n_layers, d_model, n_heads, d_ff, vocab
    c.n_trainable = n_layers // 4 if n_trainable is None else n_trainable
    c.window, c.chunk, c.n_seqs = window, chunk, n_seqs
    c.rope_theta, c.rms_eps, c.eta = float(rope_theta), float(rms_eps), float(eta)
    c.compute = 0 if compute == "fp32" else 1
    c.dual_mlp = 1 if dual_mlp else 0
    return c


class TTT:
    """One libttt context: a model with frozen weights and n_seqs sequences of fast weights."""

    def __init__(self, cfg: ttt_config, stream=None):
        self.cfg = cfg
        self._h = _vp()
        code = ttt_create(ctypes.byref(cfg), _stream(stream), ctypes.byref(self._h))
        if code != TTT_OK:
            raise TTTError(code, "ttt_create")

    @classmethod
    def from_shape(cls, shape, stream=None, **over):
        kw = dict(n_layers=shape.n_layers, d_model=shape.d_model, n_heads=shape.n_heads, d_ff=shape.d_ff,
                  vocab=shape.vocab, window=shape.window, chunk=shape.chunk, rope_theta=shape.rope_theta,
                  eta=shape.eta, n_seqs=shape.n_seqs, compute=shape.compute, rms_eps=shape.rms_eps,
                  dual_mlp=getattr(shape, "dual_mlp", False))
        kw.update(over)
        return cls(make_config(**kw), stream)

    def _check(self, code, what):
        if code != TTT_OK:
            msg = ttt_last_error(self._h)
            raise TTTError(code, f"{what}: {msg.decode() if msg else ''}")
        return code

    def load_weights(self, blob: np.ndarray):
        blob = np.ascontiguousarray(blob, np.float32)
        self._check(ttt_load_weights(self._h, blob.ctypes.data, blob.size), "ttt_load_weights")

    def prefill_chunk(self, tokens, next_tokens) -> np.ndarray:
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(self.cfg.n_seqs, -1)
        nxt = np.ascontiguousarray(next_tokens, np.int32).reshape(self.cfg.n_seqs)
        loss = np.zeros(self.cfg.n_seqs, np.float32)
        self._check(ttt_prefill_chunk(self._h, tokens.ctypes.data, tokens.shape[1], nxt.ctypes.data,
                                      loss.ctypes.data), "ttt_prefill_chunk")
        return loss

    def prefill_chunk_dev(self, d_tokens, n, d_next, d_loss):
        self._check(ttt_prefill_chunk_dev(self._h, ptr(d_tokens), n, ptr(d_next), ptr(d_loss)),
                    "ttt_prefill_chunk_dev")

    def prefill_sequence_dev(self, d_tokens, T, d_losses):
        self._check(ttt_prefill_sequence_dev(self._h, ptr(d_tokens), T, ptr(d_losses)), "ttt_prefill_sequence_dev")

    def prefill_sequence(self, tokens) -> np.ndarray:
        """Whole sequences from host memory: tokens [n_seqs][T] -> chunk losses [n_seqs][ceil(T/b)]."""
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(self.cfg.n_seqs, -1)
        Tn = tokens.shape[1]
        losses = np.zeros((self.cfg.n_seqs, -(-Tn // self.cfg.chunk)), np.float32)
        self._check(ttt_prefill_sequence(self._h, tokens.ctypes.data, Tn, losses.ctypes.data),
                    "ttt_prefill_sequence")
        return losses

    def decode_dev(self, d_prompt, T, n_new, d_out, d_prefill_losses, d_gen_losses=None, *, sample=False,
                   temp=1.0, d_u=None, d_logits=None):
        """ttt_decode_dev on device tensors (see include/ttt.h)."""
        self._check(ttt_decode_dev(self._h, ptr(d_prompt), T, n_new, int(sample), float(temp), ptr(d_u),
                                   ptr(d_out), ptr(d_prefill_losses), ptr(d_gen_losses), ptr(d_logits)),
                    "ttt_decode_dev")

    def sync(self):
        self._check(ttt_sync(self._h), "ttt_sync")

    def fast_weights(self, seq: int, suffix_layer: int):
        d, f = self.cfg.d_model, self.cfg.d_ff
        up = np.zeros((d, f), np.float32)
        down = np.zeros((f, d), np.float32)
        self._check(ttt_get_fast_weights(self._h, seq, suffix_layer, up.ctypes.data, down.ctypes.data),
                    "ttt_get_fast_weights")
        return up, down

    def window(self, seq: int, layer: int):
        """(keys [k][d], values [k][d], positions [k]) of the window cache of one block."""
        k, d = self.cfg.window, self.cfg.d_model
        ko = np.zeros((k, d), np.float32)
        vo = np.zeros((k, d), np.float32)
        po = np.zeros(k, np.int64)
        self._check(ttt_get_window(self._h, seq, layer, ko.ctypes.data, vo.ctypes.data, po.ctypes.data),
                    "ttt_get_window")
        return ko, vo, po

    def export_state(self, seq: int = 0) -> bytes:
        """Position, fast weights and window cache of one sequence as bytes (ttt_export_state)."""
        buf = np.zeros(int(ttt_state_bytes(self._h)), np.uint8)
        self._check(ttt_export_state(self._h, seq, buf.ctypes.data, buf.size), "ttt_export_state")
        return buf.tobytes()

    def import_state(self, state: bytes, seq: int = 0):
        buf = np.frombuffer(state, np.uint8)
        self._check(ttt_import_state(self._h, seq, buf.ctypes.data, buf.size), "ttt_import_state")

    def set_concurrency(self, on: bool):
        """Side streams and side-by-side sequences inside the context (on by default); off runs in issue order."""
        self._check(ttt_set_concurrency(self._h, 1 if on else 0), "ttt_set_concurrency")

    def reset(self):
        self._check(ttt_reset(self._h), "ttt_reset")

    @property
    def launches(self) -> int:
        return int(ttt_launch_count(self._h))

    def profile(self, enable=True, classes=None, every=1):
        """Start (enable) or stop event timing; `classes` limits it to those class names,
        `every` to one launch in that many of each class."""
        mask = 0
        if enable:
            names = profile_classes()
            mask = -1 if classes is None else sum(1 << names.index(c) for c in classes)
        self._check(ttt_profile(self._h, mask), "ttt_profile")
        self._check(ttt_profile_sample(self._h, every), "ttt_profile_sample")

    def profile_read(self):
        """{class name: dict(launches, ms, alg_flops, exec_flops, bytes)} since ttt_profile(1)."""
        arr = (ttt_kernel_stat * 64)()
        n = ctypes.c_int()
        self._check(ttt_profile_read(self._h, arr, 64, ctypes.byref(n)), "ttt_profile_read")
        return {arr[i].name.decode(): dict(launches=arr[i].launches, ms=arr[i].ms, alg_flops=arr[i].alg_flops,
                                           exec_flops=arr[i].exec_flops, bytes=arr[i].bytes)
                for i in range(min(n.value, 64))}

    @property
    def position(self) -> int:
        return int(ttt_position(self._h))

    def close(self):
        if self._h:
            ttt_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
