"""The C ABI of libttt without a GPU: every declared symbol is exported, the
ctypes mirrors of the public structs match the C layout, and the host-side
argument checks reject bad input before any CUDA call is made.
"""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import test_long_context_02_b300 as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def declared_symbols():
    names = []
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            src = open(os.path.join(INCLUDE, h)).read()
            names += re.findall(r"TTT_API\s+[\w\s\*]+?\b(ttt_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 18
    missing = [n for n in names if not hasattr(T.lib, n)]
    assert not missing, missing


def test_exports_are_exactly_the_declared_api():
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", T.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if len(l.split()) == 3 and l.split()[1] == "T"}
    ttt = {n for n in exported if n.startswith("ttt_")}
    assert ttt == set(declared_symbols())
    assert exported == ttt, sorted(exported - ttt)  # nothing else leaks out of the library


LAYOUT_PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "ttt.h"
#include "ttt_kernels.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("ttt_config %zu\n", sizeof(ttt_config));
  F(ttt_config, n_layers) F(ttt_config, window) F(ttt_config, n_seqs) F(ttt_config, rope_theta)
  F(ttt_config, rms_eps) F(ttt_config, eta) F(ttt_config, compute) F(ttt_config, dual_mlp)
  printf("ttt_kernel_stat %zu\n", sizeof(ttt_kernel_stat));
  F(ttt_kernel_stat, launches) F(ttt_kernel_stat, ms) F(ttt_kernel_stat, bytes)
  printf("ttt_gemm_epilogue %zu\n", sizeof(ttt_gemm_epilogue));
  F(ttt_gemm_epilogue, ldo) F(ttt_gemm_epilogue, eta) F(ttt_gemm_epilogue, tgt) F(ttt_gemm_epilogue, scale)
  F(ttt_gemm_epilogue, err) F(ttt_gemm_epilogue, allow_ksplit)
  return 0;
}
"""


def test_ctypes_structs_match_c_layout():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "probe.c"), os.path.join(d, "probe")
        open(src, "w").write(LAYOUT_PROBE)
        subprocess.run([cc, "-I", INCLUDE, src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    c = {k: int(v) for k, v in (l.split() for l in out.splitlines())}
    mirrors = {"ttt_config": T.ttt_config, "ttt_kernel_stat": T.ttt_kernel_stat,
               "ttt_gemm_epilogue": T.ttt_gemm_epilogue}
    for key, val in c.items():
        if "." in key:
            sname, field = key.split(".")
            assert getattr(mirrors[sname], field).offset == val, key
        else:
            assert ctypes.sizeof(mirrors[key]) == val, key


def _create(cfg):
    h = ctypes.c_void_p()
    return T.ttt_create(ctypes.byref(cfg), None, ctypes.byref(h)), h


@pytest.mark.parametrize("bad", [
    dict(chunk=256, window=128),          # k < b
    dict(n_layers=0),
    dict(d_model=130, n_heads=4),         # d not divisible by H
    dict(n_seqs=0),
    dict(compute=2),
    dict(dual_mlp=2),
])
def test_create_rejects_inconsistent_configs_before_any_cuda_call(bad):
    cfg = T.make_config(4, 128, 4, 512, 512, 128, 64, 1e4, 1e-2)
    for k, v in bad.items():
        setattr(cfg, k, v)
    code, h = _create(cfg)
    assert code == T.TTT_ERR_ARG and not h.value


@pytest.mark.parametrize("bad", [
    dict(d_model=200, n_heads=4),         # d_head 50
    dict(d_model=256, n_heads=2),         # d_head 128 in the fp32 (split) mode
    dict(window=192, chunk=64),           # window not a multiple of 128
    dict(vocab=515),
])
def test_create_rejects_unsupported_shapes(bad):
    cfg = T.make_config(4, 128, 4, 512, 512, 128, 64, 1e4, 1e-2, compute="fp32")
    for k, v in bad.items():
        setattr(cfg, k, v)
    code, h = _create(cfg)
    assert code == T.TTT_ERR_UNSUPPORTED and not h.value


def test_kernel_entry_points_reject_bad_arguments():
    e = T.ttt_gemm_epilogue()
    # null operand, negative size, pitch not a multiple of 8
    assert T.ttt_k_gemm(0, 8, 8, 8, None, None, 8, 0, 1, None, 8, 0, 0, ctypes.byref(e), None) == T.TTT_ERR_ARG
    assert T.ttt_k_gemm(0, -1, 8, 8, 1, None, 8, 0, 1, None, 8, 0, 0, ctypes.byref(e), None) == T.TTT_ERR_ARG
    assert T.ttt_k_gemm(0, 8, 8, 8, 1, None, 12, 0, 1, None, 8, 0, 0, ctypes.byref(e), None) == T.TTT_ERR_ARG
    # split mode without remainders
    assert T.ttt_k_gemm(0, 8, 8, 8, 1, None, 8, 0, 1, None, 8, 0, 1, ctypes.byref(e), None) == T.TTT_ERR_ARG
    p = [1] * 10
    # n > window, window not a multiple of 128, unsupported head width
    assert T.ttt_k_attn_fwd(300, 2, 64, 256, 0, 0, *p, 1, None, None, None, None) == T.TTT_ERR_ARG
    assert T.ttt_k_attn_fwd(64, 2, 64, 200, 0, 0, *p, 1, None, None, None, None) == T.TTT_ERR_ARG
    assert T.ttt_k_attn_fwd(64, 2, 48, 256, 0, 0, *p, 1, None, None, None, None) == T.TTT_ERR_UNSUPPORTED
    assert T.ttt_k_attn_fwd(64, 2, 96, 256, 0, 1, *p, 1, None, None, None, None) == T.TTT_ERR_UNSUPPORTED
    assert T.ttt_k_attn_rowdot(0, 2, 64, 1, None, 1, None, 1, None) == T.TTT_ERR_ARG


def test_context_calls_reject_null_context():
    assert T.ttt_load_weights(None, 1, 10) == T.TTT_ERR_ARG
    assert T.ttt_prefill_chunk(None, 1, 1, 1, 1) == T.TTT_ERR_ARG
    assert T.ttt_prefill_sequence(None, 1, 1, 1) == T.TTT_ERR_ARG
    assert T.ttt_get_fast_weights(None, 0, 0, None, None) == T.TTT_ERR_ARG
    assert T.ttt_reset(None) == T.TTT_ERR_ARG
    assert T.ttt_launch_count(None) == -1
    assert T.ttt_state_bytes(None) == -1
    assert T.ttt_set_concurrency(None, 1) == T.TTT_ERR_ARG
    assert T.ttt_profile_sample(None, 8) == T.TTT_ERR_ARG
    assert T.ttt_export_state(None, 0, 1, 48) == T.TTT_ERR_ARG
    assert T.ttt_import_state(None, 0, 1, 48) == T.TTT_ERR_ARG
    assert T.ttt_position(None) == -1
    assert T.ttt_last_error(None) == b"null context"
    T.ttt_destroy(None)


def test_host_blob_size_matches_layout():
    from ttt_inputs import SHAPES, blob_size
    s = SHAPES["760m"]
    d, f, V, L = s.d_model, s.d_ff, s.vocab, s.n_layers
    assert blob_size(s) == V * d + L * (2 * d + 4 * d * d + 2 * d * f) + d + d * V
    assert np.dtype(np.float32).itemsize * blob_size(s) < 3.5e9
