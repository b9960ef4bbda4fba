"""The decode steps exactly as bench.py times them, against the oracle.

bench.py builds one Decoder per rotated input copy (append on: k_idx and
pool_w given; no index or score output, which switch the kernel to other
internal paths) and replays the steps from captured CUDA graphs.  Here the
same helpers build and replay them, and every copy's output and lse, read
after the graph replays, are compared with the oracle element by element at
the attention tolerance.
"""
import numpy as np
import pytest
import torch

import bench
import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import assert_attn_close, assert_lse_close, host_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name", ["decode_1m", "decode_b8"])
def test_benchmarked_decode_call_matches_oracle(name):
    spec = synth.named(name)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    P, k, B = spec.P, spec.k, spec.B
    copies, _ = bench.workload_config(spec, name, bench.l2_bytes())

    def kp_builder(k_idx, pool_w, seq):
        kp = torch.zeros(B, spec.G_max, spec.d_idx, dtype=torch.bfloat16, device="cuda")
        lcsw.pool_keys(k_idx, pool_w, seq, P, kp)
        return kp

    decs, keep = bench.make_decoders(lcsw, torch, c, copies, P, k, kp_builder)
    assert all(d.args.idx_out is None and d.args.scores_out is None for d in decs)
    assert all(d.args.k_idx is not None for d in decs)
    # warm-up, graph capture and replay of 3 rounds of the rotation, as timed
    bench.time_graph_steps(torch, decs, 3 * copies, 3, 1)
    torch.cuda.synchronize()
    decs[0].status()
    for d in decs:
        d.status()
        assert_attn_close(host_bits(d.out), ref["out"][:, 0])
        assert_lse_close(d.lse.cpu().numpy(), ref["lse"][:, 0])
    # the appended group was re-pooled in place, bit for bit
    kp0 = keep["kp0"]
    for b in range(B):
        g = int(c["seq_len"][b]) // P - 1
        got = kp0[b, g].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ref["k_pooled"][b, g])
