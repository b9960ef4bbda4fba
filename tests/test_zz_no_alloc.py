"""lcsw_sparse_attn_noalloc: the attention entry point that takes no workspace.

The file is named to be collected last: the entry point must pass after every
other test has used the library in the same process, and alone in a fresh
process.  The GPU test checks it against lcsw_sparse_attn (the entry point with a
caller workspace) and against the CPU oracle on two calls in a row; the CPU
tests check that its arguments are validated as lcsw_sparse_attn validates
them, and that a valid shape whose split-K scratch would not fit is rejected
before any device work.
"""
import os
import re

import numpy as np
import pytest

import long_context_sparse_weighted_b300 as lcsw
import synth

HEADER = os.path.join(os.path.dirname(__file__), "..", "include", "lcsw.h")


def _scratch_bytes():
    with open(HEADER) as f:
        m = re.search(r"#define\s+LCSW_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", f.read())
    assert m, "LCSW_NOALLOC_SCRATCH_BYTES not found in the header"
    return int(m.group(1)) << int(m.group(2))


def _case(seed, B, lengths, H_q, d_qk, d_v, k, P):
    spec = synth.Spec(B=B, lengths=lengths, T=1, H_q=H_q, d_qk=d_qk, d_v=d_v, P=P, k=k,
                      seed=seed)
    c = synth.generate(spec)
    rng = np.random.default_rng(seed)
    idx = np.full((B, 1, k), -1, np.int32)
    for b in range(B):
        G = lengths[b] // P
        n = min(k - 2, G)  # two -1 pads per row
        idx[b, 0, :n] = np.sort(rng.choice(G, size=n, replace=False))
    return c, idx


# Stand-in device addresses: the host checks only look at their alignment and
# reject the call before anything would dereference them.
_FAKE = [0x10000 * (i + 1) for i in range(6)]


def test_noalloc_rejects_oversized_shape():
    L = lcsw.lib()
    B, T, H_q, d_qk, d_v, k, P = 4, 1, 128, 128, 128, 2048, 4
    need = L.lcsw_sparse_attn_workspace_size(B, T, H_q, d_v, k, P)
    assert need > _scratch_bytes()
    q, K, V, seq, idx, out = _FAKE
    st = L.lcsw_sparse_attn_noalloc(q, K, 0, V, 0, seq, idx, B, T, H_q, d_qk, d_v,
                                    P, k, 1.0, out, None, None)
    assert st == lcsw.ERR_UNSUPPORTED
    msg = L.lcsw_last_error().decode()
    assert "split-K scratch" in msg and str(need) in msg


@pytest.mark.parametrize("bad", ["null", "heads", "P", "misaligned"])
def test_noalloc_validates_arguments_first(bad):
    """An invalid call is an argument error, as from lcsw_sparse_attn, even
    when its shape would also overflow the fixed scratch."""
    L = lcsw.lib()
    B, T, H_q, d_qk, d_v, k, P = 4, 1, 128, 128, 128, 2048, 4
    q, K, V, seq, idx, out = _FAKE
    if bad == "null":
        q = None
    elif bad == "heads":
        H_q = 48
    elif bad == "P":
        P = 3
    else:
        K += 2
    st = L.lcsw_sparse_attn_noalloc(q, K, 0, V, 0, seq, idx, B, T, H_q, d_qk, d_v,
                                    P, k, 1.0, out, None, None)
    assert st == lcsw.ERR_INVALID_ARG, L.lcsw_last_error().decode()
    st_ws = L.lcsw_sparse_attn(q, K, 0, V, 0, seq, idx, B, T, H_q, d_qk, d_v, P, k, 1.0, out,
                               None, None, 0, None)
    assert st_ws == lcsw.ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_two_calls(cuda_device):
    import torch

    import oracle
    from gpu_util import assert_attn_close, assert_lse_close, dev, host_bits, upload_case

    L = lcsw.lib()
    cases = [
        (_case(901, 8, [16384] * 8, 32, 192, 128, 512, 4), 4),
        (_case(902, 2, [32768, 20000], 64, 128, 128, 512, 4), 4),
    ]
    for (c, idx), P in cases:  # two calls in a row: the second reuses the scratch
        B, _, k = idx.shape
        H_q, d_v = c["q"].shape[2], c["V"].shape[2]
        need = L.lcsw_sparse_attn_workspace_size(B, 1, H_q, d_v, k, P)
        assert 0 < need <= _scratch_bytes()  # split-K really goes through the scratch
        d = upload_case(c)
        di = dev(idx)
        ref_out, ref_lse = lcsw.sparse_attn(d["q"], d["K"], d["V"], d["seq_len"], di, P,
                                            c["scale"])
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        lcsw.sparse_attn_noalloc(d["q"], d["K"], d["V"], d["seq_len"], di, P, c["scale"], out,
                                 lse)
        torch.cuda.synchronize()
        assert_attn_close(host_bits(out), host_bits(ref_out))
        assert_lse_close(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64))
        o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, P,
                                          c["scale"])
        assert_attn_close(host_bits(out), o_ref)
        assert_lse_close(lse.cpu().numpy(), l_ref)
