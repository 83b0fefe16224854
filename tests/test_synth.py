"""The seeded input generator: published SplitMix64 values, determinism, distributions."""
import numpy as np

from int4_routed_expert_05_b300 import synth


def test_splitmix64_published_values():
    # the reference sequence of SplitMix64 (Steele, Lea, Flood 2014) from state 0 and 1234567
    assert int(synth.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF
    assert [int(v) for v in synth.splitmix64(1234567, 5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    # counter-based: any window of the stream can be drawn on its own
    assert np.array_equal(synth.splitmix64(99, 4, start=3), synth.splitmix64(99, 7)[3:])


def test_determinism_and_independence():
    a = synth.expert_tensors(synth.TINY, 5, 2, 3)
    b = synth.expert_tensors(synth.TINY, 5, 2, 3)
    c = synth.expert_tensors(synth.TINY, 5, 2, 4)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["gate_q"], c["gate_q"])


def test_distributions():
    sh = synth.S80
    t = synth.expert_tensors(sh, 0, 0, 0)
    q = t["gate_q"]
    assert q.shape == (sh.inter, sh.hidden) and q.min() == 0 and q.max() == 15
    hist = np.bincount(q.ravel(), minlength=16) / q.size
    assert np.all(np.abs(hist - 1 / 16) < 0.003)
    s = synth.bf16_value(t["gate_s"])
    b = synth.bf16_value(t["gate_b"])
    assert s.min() >= 0.0049 and s.max() <= 0.0201
    assert np.array_equal(b, -8 * s)
    t8 = synth.expert_tensors(sh.with_bits(8), 0, 0, 0)
    assert t8["down_q"].max() == 255
    assert np.array_equal(synth.bf16_value(t8["up_b"]), -128 * synth.bf16_value(t8["up_s"]))
    n = synth.normal(synth.stream_key(1, 2), 200000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    Wr = synth.bf16_value(synth.router_bits(synth.TINY, 0, 0))
    assert abs(Wr.std() - 0.02) < 0.001


def test_bf16_bits_roundtrip():
    x = np.float32([1.0, -2.5, 0.1, 3.14159])
    v = synth.bf16_value(synth.bf16_bits(x))
    assert np.all(np.abs(v - x) <= np.abs(x) * 2 ** -8)
    assert np.array_equal(synth.bf16_bits(v), synth.bf16_bits(x))


def test_expert_map_is_per_layer_permutation():
    m = synth.expert_map(synth.S80, 0, 3, 512)
    assert sorted(m) == list(range(512))
    m2 = synth.expert_map(synth.S80, 0, 4, 512)
    assert not np.array_equal(m, m2)
    m3 = synth.expert_map(synth.S80, 0, 4, 64)
    assert m3.max() < 64
