"""liblcsw.so builds, loads without a GPU, exports every symbol include/lcsw.h
declares, matches the header's struct layouts, and rejects bad arguments on the
host (no CUDA call is made for any of these)."""
import ctypes
import os
import re
import subprocess

import pytest

import long_context_sparse_weighted_b300 as lcsw
from long_context_sparse_weighted_b300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return lcsw.lib()


def _header_functions():
    src = open(lcsw.HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lcsw_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _header_functions()
    assert len(names) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", lcsw.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (lcsw_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)
    assert set(lcsw._SIGNATURES) == set(names)


def _c_layout(struct, fields, tmp_path):
    prog = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{lcsw.HEADER}"',
            'int main(void) {', f'printf("size %zu\\n", sizeof({struct}));']
    for f in fields:
        prog.append(f'printf("{f} %zu\\n", offsetof({struct}, {f}));')
    prog.append("return 0; }")
    c = tmp_path / f"{struct}.c"
    c.write_text("\n".join(prog))
    exe = tmp_path / struct
    subprocess.run(["gcc", "-o", str(exe), str(c)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}


@pytest.mark.parametrize("cls,struct", [(lcsw.DecodeArgs, "lcsw_decode_args"),
                                        (lcsw.PrefillArgs, "lcsw_prefill_args")])
def test_struct_layout_matches_header(cls, struct, tmp_path):
    names = [f[0] for f in cls._fields_]
    c = _c_layout(struct, names, tmp_path)
    assert c["size"] == ctypes.sizeof(cls)
    for n in names:
        assert c[n] == getattr(cls, n).offset, n


def _err(L):
    return L.lcsw_last_error().decode()


def test_version_and_empty_error(L):
    assert "sm_103a" in lcsw.version()


def test_pool_keys_rejects_bad_arguments(L):
    p = ctypes.c_void_p(256)
    # P not in {1,2,4,8}
    assert L.lcsw_pool_keys(p, 0, p, 0, p, None, 1, 4, 64, 3, p, 0, None) == lcsw.ERR_INVALID_ARG
    assert "P must be" in _err(L)
    # null pointer
    assert L.lcsw_pool_keys(None, 0, p, 0, p, None, 1, 4, 64, 4, p, 0, None) == lcsw.ERR_INVALID_ARG
    # misaligned bf16 rows
    q = ctypes.c_void_p(258)
    assert L.lcsw_pool_keys(q, 0, p, 0, p, None, 1, 4, 64, 4, p, 0, None) == lcsw.ERR_INVALID_ARG
    assert "aligned" in _err(L)
    # empty work is fine and launches nothing
    assert L.lcsw_pool_keys(None, 0, None, 0, None, None, 0, 4, 64, 4, None, 0, None) == lcsw.OK


def test_index_scores_rejects_bad_arguments(L):
    p = ctypes.c_void_p(256)
    assert L.lcsw_index_scores(p, p, p, 0, p, None, 1, 1, 8, 32, 4, 16, p, None) == lcsw.ERR_INVALID_ARG
    assert "d_idx" in _err(L)
    assert L.lcsw_index_scores(p, p, p, 0, p, None, 1, 1, 17, 64, 4, 16, p, None) == lcsw.ERR_INVALID_ARG
    assert "H_i" in _err(L)


def test_topk_and_attention_reject_bad_arguments(L):
    p = ctypes.c_void_p(256)
    assert L.lcsw_topk_groups(p, p, 1, 16, 0, p, None, 0, None) == lcsw.ERR_INVALID_ARG
    assert "k must be" in _err(L)
    # unsupported head count
    assert L.lcsw_sparse_attn(p, p, 0, p, 0, p, p, 1, 1, 48, 128, 128, 4, 8, 0.1, p, None, None,
                              0, None) == lcsw.ERR_INVALID_ARG
    # workspace too small (rows=1 -> several splits -> partials needed)
    need = L.lcsw_sparse_attn_workspace_size(1, 1, 64, 128, 512, 4)
    assert need > 0
    assert L.lcsw_sparse_attn(p, p, 0, p, 0, p, p, 1, 1, 64, 128, 128, 4, 512, 0.1, p, None, p,
                              need - 1, None) == lcsw.ERR_WORKSPACE


def test_decode_workspace_and_validation(L):
    a = lcsw.DecodeArgs()
    a.B, a.G_max, a.H_i, a.d_idx, a.P, a.k = 1, 262144, 8, 64, 4, 512
    a.H_q, a.d_qk, a.d_v, a.scale = 64, 128, 128, 0.088
    n = L.lcsw_decode_workspace_size(ctypes.byref(a))
    assert n >= 262144 * 4 + 512 * 4
    # null tensors -> invalid argument before any device work
    assert L.lcsw_decode_fused(ctypes.byref(a), ctypes.c_void_p(256), n, None) == lcsw.ERR_INVALID_ARG
    a.d_idx = 32
    assert L.lcsw_decode_fused(ctypes.byref(a), None, 0, None) == lcsw.ERR_INVALID_ARG
    assert L.lcsw_decode_fused(None, None, 0, None) == lcsw.ERR_INVALID_ARG


def test_prefill_workspace_and_validation(L):
    a = lcsw.PrefillArgs()
    p = 256  # non-null, 256-byte aligned stand-ins: no call below reaches the device
    for name in ("q_idx", "w_head", "k_pooled", "k_idx", "pool_w", "q", "K", "V", "seq_len",
                 "out", "lse"):
        setattr(a, name, p)
    G, L_tok = 66560, 266240
    a.sp_b, a.sk_b, a.sw_b, a.sK_b, a.sV_b = G * 64, L_tok * 64, G * 4, L_tok * 128, L_tok * 128
    a.B, a.T, a.G_max, a.H_i, a.d_idx, a.P, a.k = 1, 4096, G, 8, 64, 4, 512
    a.H_q, a.d_qk, a.d_v, a.scale = 32, 128, 128, 0.088
    n = L.lcsw_prefill_workspace_size(ctypes.byref(a))
    assert n > 4096 * G * 4  # room for dense scores of rows that take the fallback
    assert L.lcsw_prefill(ctypes.byref(a), ctypes.c_void_p(256), n - 1, None) == lcsw.ERR_WORKSPACE
    a.H_q = 20  # head counts are 16, 32 or multiples of 64
    assert L.lcsw_prefill(ctypes.byref(a), ctypes.c_void_p(256), n, None) == lcsw.ERR_INVALID_ARG


def test_prefill_binding_rejects_a_small_workspace(L):
    import torch
    B, T, H_i, G, P, k, H_q = 1, 64, 8, 256, 4, 16, 16
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lcsw.prefill(bf(B, T, H_i, 64), torch.zeros(B, T, H_i), bf(B, G, 64), bf(B, G * P, 64),
                     torch.zeros(B, G, P), bf(B, T, H_q, 128), bf(B, G * P, 128),
                     bf(B, G * P, 128), torch.full((B,), G * P, dtype=torch.int32), P, k, 0.1,
                     ws=torch.zeros(16, dtype=torch.uint8))


def test_product_package_does_not_reach_the_oracle():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "long_context_sparse_weighted_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_decode_reuse_validates_arguments(L):
    import ctypes

    import long_context_sparse_weighted_b300 as lcsw
    a = lcsw.DecodeArgs()
    a.B, a.P, a.k, a.H_q, a.d_qk, a.d_v, a.scale = 2, 4, 16, 32, 128, 128, 0.1
    a.q, a.K, a.V, a.seq_len, a.out = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    a.sK_b = a.sV_b = 128 * 64
    ws = 0x100000
    assert L.lcsw_decode_reuse(ctypes.byref(a), None, ws, 1 << 30, None) == lcsw.ERR_INVALID_ARG
    assert L.lcsw_decode_reuse(ctypes.byref(a), 0x60002, ws, 1 << 30, None) == lcsw.ERR_INVALID_ARG
    a.H_q = 48
    assert L.lcsw_decode_reuse(ctypes.byref(a), 0x60000, ws, 1 << 30, None) == lcsw.ERR_INVALID_ARG
    a.H_q = 32
    assert L.lcsw_decode_reuse(ctypes.byref(a), 0x60000, ws, 16, None) == lcsw.ERR_WORKSPACE


def test_kda_step_validates_arguments(L):
    import long_context_sparse_weighted_b300 as lcsw
    p = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000]
    # head width other than 128 is a valid shape the kernel does not cover
    assert L.lcsw_kda_step(*p, 2, 1, 64, 64, None) == lcsw.ERR_UNSUPPORTED
    assert L.lcsw_kda_step(*p, -1, 1, 64, 128, None) == lcsw.ERR_INVALID_ARG
    assert L.lcsw_kda_step(*p, 2, 1, 0, 128, None) == lcsw.ERR_INVALID_ARG
    # empty batch or no tokens: nothing to do, nothing dereferenced
    assert L.lcsw_kda_step(None, None, None, None, None, None, None, 0, 1, 64, 128, None) == lcsw.OK
    assert L.lcsw_kda_step(None, None, None, None, None, None, None, 2, 0, 64, 128, None) == lcsw.OK
    assert L.lcsw_kda_step(*p[:6], None, 2, 1, 64, 128, None) == lcsw.ERR_INVALID_ARG
    bad = list(p)
    bad[5] = 0x60004                       # state not 16-byte aligned
    assert L.lcsw_kda_step(*bad, 2, 1, 64, 128, None) == lcsw.ERR_INVALID_ARG


def test_int8_cache_entries_validate_arguments(L):
    import long_context_sparse_weighted_b300 as lcsw
    x, codes, scales = 0x10000, 0x20000, 0x30000
    # width must be a multiple of 16; codes and their stride 16-byte aligned
    assert L.lcsw_quantize_rows_i8(x, 24, None, 2, 3, 24, codes, 32, scales, 3, None) == \
        lcsw.ERR_INVALID_ARG
    assert L.lcsw_quantize_rows_i8(x, 64, None, 2, 3, 64, codes + 8, 64, scales, 3, None) == \
        lcsw.ERR_INVALID_ARG
    assert L.lcsw_quantize_rows_i8(x, 64, None, 2, 3, 64, None, 64, scales, 3, None) == \
        lcsw.ERR_INVALID_ARG
    assert L.lcsw_quantize_rows_i8(None, 64, None, 0, 3, 64, None, 64, None, 3, None) == lcsw.OK
    p = [0x10000, 0x20000, 64 * 128, 0x30000, 64, 0x40000, 64 * 128, 0x50000, 64, 0x60000,
         0x70000]
    # an unsupported attention shape, then a missing workspace
    assert L.lcsw_sparse_attn_kvi8(*p, 1, 1, 48, 128, 128, 4, 16, 0.1, 0x80000, None, None, 0,
                                   None) == lcsw.ERR_INVALID_ARG
    ws = L.lcsw_sparse_attn_kv8_workspace_size(1, 1, 64, 128, 512, 4)
    if ws:
        assert L.lcsw_sparse_attn_kvi8(*p, 1, 1, 64, 128, 128, 4, 512, 0.1, 0x80000, None, None,
                                       0, None) == lcsw.ERR_WORKSPACE
    assert L.lcsw_sparse_attn_kvi8(*p, 0, 1, 64, 128, 128, 4, 512, 0.1, 0x80000, None, None, 0,
                                   None) == lcsw.OK


def test_append_token_validates_arguments(L):
    import long_context_sparse_weighted_b300 as lcsw
    r, s, k, K, V = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    bad_width = (r, 320, s, 2, k, 64 * 100, 60, K, 128 * 100, 128, V, 128 * 100, 128, None)
    assert L.lcsw_append_token(*bad_width) == lcsw.ERR_INVALID_ARG
    short_row = (r, 256, s, 2, k, 64 * 100, 64, K, 128 * 100, 128, V, 128 * 100, 128, None)
    assert L.lcsw_append_token(*short_row) == lcsw.ERR_INVALID_ARG
    v_mismatch = (r, 320, s, 2, k, 64 * 100, 64, K, 128 * 100, 128, None, 0, 128, None)
    assert L.lcsw_append_token(*v_mismatch) == lcsw.ERR_INVALID_ARG
    misaligned = (r + 8, 320, s, 2, k, 64 * 100, 64, K, 128 * 100, 128, V, 128 * 100, 128, None)
    assert L.lcsw_append_token(*misaligned) == lcsw.ERR_INVALID_ARG
    empty = (None, 320, None, 0, None, 0, 64, None, 0, 128, None, 0, 0, None)
    assert L.lcsw_append_token(*empty) == lcsw.OK
