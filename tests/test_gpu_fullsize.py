"""The four larger named workloads at full size, through the same C-ABI calls
and launch configuration the benchmark times.  Decode workloads are checked in
full; chunked prefill on sampled query rows (the oracle scores every group for
each sampled row in fp64)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_attn_close, assert_lse_close, selection_diff
from test_gpu_decode import check_against_oracle, run_decode, run_prefill, _cached_part

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name", ["decode_b8", "decode_1m", "ragged_b64"])
def test_decode_full_size(name):
    c = synth.generate(synth.named(name))
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"], append=True, corrupt_last=True)
    assert np.array_equal(got["k_pooled"], ref["k_pooled"])
    check_against_oracle(c, got, ref)


def test_prefill_4k_sampled_rows():
    c = synth.generate(synth.named("prefill_4k"))
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], c["P"])
    got = run_prefill(c, _cached_part(kp, c))
    assert np.array_equal(got["k_pooled"], kp)
    rng = np.random.default_rng(4)
    ts = np.unique(np.concatenate([[0, 1, 2, 3, 4095], rng.choice(4096, 59, replace=False)]))
    ref = oracle.retrieval_step(c["q_idx"][:, ts], c["w_head"][:, ts], kp, c["q"][:, ts],
                                c["K"], c["V"], c["seq_len"], c["P"], c["k"], c["scale"],
                                q_pos=c["q_pos"][:, ts])
    nd = selection_diff(got["idx"][:, ts], ref["idx"], ref["scores"])
    assert nd == 0, f"{nd} sampled rows differ by near-ties"
    assert_attn_close(got["out"][:, ts], ref["out"])
    assert_lse_close(got["lse"][:, ts], ref["lse"])
