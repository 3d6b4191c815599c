"""The seeded input generator: published hash, determinism, distributions."""
import numpy as np

from skinny_gemm_gb300 import synth

MASK = (1 << 64) - 1


def _mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_python_splitmix64_matches_published_vector():
    # splitmix64 started at state 0: first three outputs
    s, out = 0, []
    for _ in range(3):
        s = (s + 0x9E3779B97F4A7C15) & MASK
        out.append(_mix(s))
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_hash_is_splitmix64_stream():
    for seed, tid in [(0, 1), (7, 2), (2**63 + 5, 5)]:
        key = _mix(seed ^ ((tid * 0xD1B54A32D192ED03) & MASK))
        want = [_mix((key + (i + 1) * 0x9E3779B97F4A7C15) & MASK) for i in range(10, 20)]
        got = synth.hashes(seed, tid, 10, offset=10)
        assert [int(v) for v in got] == want


def test_deterministic_and_offset_consistent():
    a = synth.make_x(3, 4, 256)
    b = synth.make_x(3, 4, 256)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.make_x(3, 2, 256, row0=2), a[2:])
    w1 = synth.make_weights(5, 300, 128)
    w2 = synth.make_weights(5, 300, 128)
    assert np.array_equal(w1.Wq, w2.Wq) and np.array_equal(w1.scales, w2.scales)
    assert not np.array_equal(synth.make_weights(6, 300, 128).Wq, w1.Wq)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_distributions():
    x = _f(synth.make_x(0, 1, 1 << 20))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    w = synth.make_weights(0, 1024, 2048)
    nib = np.stack([(w.Wq >> (4 * i)) & 0xF for i in range(8)]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert np.all(np.abs(counts / nib.size - 1 / 16) < 0.002)
    s, b = _f(w.scales), _f(w.biases)
    assert s.min() >= 0.00199 and s.max() <= 0.0201
    assert abs(s.mean() - 0.011) < 0.0005
    noise = b + 8 * s
    assert abs(noise.mean()) < 1e-4 and 0.9e-3 < noise.std() < 1.2e-3
    ids = synth.make_ids(0, 80000, 8)
    assert ids.min() == 0 and ids.max() == 7
    assert np.all(np.abs(np.bincount(ids) / ids.size - 1 / 8) < 0.01)


def test_experts_are_distinct_draws():
    w = synth.make_weights(0, 64, 128, E=3)
    assert w.Wq.shape == (3, 64, 16) and w.scales.shape == (3, 64, 2)
    assert not np.array_equal(w.Wq[0], w.Wq[1])


def test_stq1_blocks_and_f32_activations():
    b = synth.make_stq1(3, 64, 2048)
    assert b.shape == (64, 8, 42) and np.array_equal(b, synth.make_stq1(3, 64, 2048))
    assert np.array_equal(synth.make_stq1(3, 64, 2048, E=2)[0], b)
    d = b[:, :, 40:].copy().view(np.float16).astype(np.float64)
    assert np.all(np.isfinite(d)) and d.min() >= 0.00199 and d.max() <= 0.0201
    codes = np.concatenate([b[:, :, :32] & 0xF, b[:, :, :32] >> 4]).ravel()
    assert np.all(np.abs(np.bincount(codes, minlength=16) / codes.size - 1 / 16) < 0.01)
    signs = np.unpackbits(b[:, :, 32:40])
    assert abs(signs.mean() - 0.5) < 0.01
    x = synth.make_x_f32(0, 3, 512)
    bits = (x.view(np.uint32).astype(np.uint64) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16
    assert np.array_equal(bits.astype(np.uint16), synth.make_x(0, 3, 512)), "bf16 x is the rounded f32 x"
    for v in (1.0, 0.002, 0.02, 1e-5, 65504.0, -3.25):
        assert synth.fp16_bits(v) == int(np.array([v], np.float32).astype(np.float16).view(np.uint16)[0])
