"""Host-side arithmetic of bench.py, pinned on the CPU.

The algorithmic bytes of a decode step (the roofline's numerator) against the
values the baseline notes give from their formula
Σ_b [G_b·64·2 + 4k·(d_qk+d_v)·2 + H_q·(d_qk+d_v)·2 + H_i·(64·2+4)]:
270,864 B (tiny), 44,212,480 B (decode_b8), 34,636,832 B (decode_1m), and
about 135.3 MB for decode_1m with IndexPool off (P = 1, k = 2,048 groups).
"""
import bench
import synth


def _ab(spec, P=None, k=None):
    return bench.alg_bytes(spec.lengths, P or spec.P, spec.H_i, spec.d_idx, k or spec.k, spec.H_q,
                           spec.d_qk, spec.d_v)


def test_decode_step_bytes_match_the_published_figures():
    assert _ab(synth.named("tiny")) == 270_864
    assert _ab(synth.named("decode_b8")) == 44_212_480
    assert _ab(synth.named("decode_1m")) == 34_636_832


def test_indexpool_off_ablation_bytes():
    ab1 = _ab(synth.named("decode_1m"), P=1, k=2048)
    assert round(ab1 / 1e6, 1) == 135.3
    # the same token budget: 2,048 single-token groups against 512 of four
    assert ab1 - _ab(synth.named("decode_1m")) == 1_048_576 * 64 * 2 - 262_144 * 64 * 2


def test_replica_value_counts_every_sequence_over_the_slowest_rank():
    assert bench.replica_value(1, 1, 20000, 572.9) == 20000 / 0.5729
    assert bench.replica_value(4, 8, 100, 10.0) == 4 * 8 * 100 / 0.01
