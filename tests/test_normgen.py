"""The seeded input generator: published known answers, determinism, sub-range and
thread-count independence, and the moments of its draws."""
import math

import numpy as np
import pytest

import normgen


def test_splitmix64_known_answers():
    # First two outputs of SplitMix64 seeded with 0, as published with the
    # reference C implementation of the generator.
    assert normgen.splitmix64_output(0, 0) == 0xE220A8397B1DCDAF
    assert normgen.splitmix64_output(0, 1) == 0x6E789E6AA1B965F4


def test_same_seed_same_bytes_and_threads_do_not_matter():
    a = normgen.normal(300_001, seed=7, tensor_id=0, threads=1)
    b = normgen.normal(300_001, seed=7, tensor_id=0, threads=5)
    c = normgen.normal(300_001, seed=7, tensor_id=0, threads=16)
    assert a.tobytes() == b.tobytes() == c.tobytes()


def test_streams_differ_by_seed_and_tensor():
    a = normgen.normal(1000, seed=0, tensor_id=0)
    assert not np.array_equal(a, normgen.normal(1000, seed=1, tensor_id=0))
    assert not np.array_equal(a, normgen.normal(1000, seed=0, tensor_id=1))


@pytest.mark.parametrize("start,n", [(0, 1), (1, 1), (3, 10), (12345, 1001), (70000, 70001)])
def test_subrange_matches_full_stream(start, n):
    full = normgen.normal(start + n + 3, seed=3, tensor_id=2)
    part = normgen.normal(n, seed=3, tensor_id=2, start=start)
    assert part.tobytes() == full[start:start + n].tobytes()
    fu = normgen.uniform(start + n, seed=3, tensor_id=2)
    pu = normgen.uniform(n, seed=3, tensor_id=2, start=start)
    assert pu.tobytes() == fu[start:start + n].tobytes()


def test_normal_moments():
    n = 2_000_000
    x = normgen.normal(n, mean=1000.0, std=1e-2, seed=0).astype(np.float64)
    # sample mean within 6 standard errors, sample variance within 6 of its standard errors
    assert abs(x.mean() - 1000.0) < 6 * 1e-2 / math.sqrt(n)
    z = normgen.normal(n, seed=11).astype(np.float64)
    assert abs(z.var() - 1.0) < 6 * math.sqrt(2.0 / n)
    assert abs(np.mean(z ** 3)) < 6 * math.sqrt(15.0 / n)
    assert abs(np.mean(z ** 4) - 3.0) < 6 * math.sqrt(96.0 / n)


def test_uniform_range_and_mean():
    u = normgen.uniform(1_000_000, 0.0, 1.0, seed=5).astype(np.float64)
    assert u.min() >= 0.0 and u.max() <= 1.0
    assert abs(u.mean() - 0.5) < 6 * math.sqrt(1 / 12 / u.size)


def test_into_existing_buffer():
    buf = np.zeros(4097, dtype=np.float32)
    out = normgen.normal(4097, seed=9, out=buf)
    assert out is buf
    assert buf.tobytes() == normgen.normal(4097, seed=9).tobytes()


def test_bf16_rounding_known_values():
    import normgen
    vals = np.array([1.0, -2.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-20, 0.0, -0.0, 3.0e38, 1e-40],
                    dtype=np.float32)
    want = [0x3F80, 0xC000, 0x3F80, 0x3F82, 0x3F81, 0x0000, 0x8000, 0x7F62, 0x0001]
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even 0x3F80;
    # 1 + 3*2^-8 ties to 0x3F82; just above the tie rounds up; 1e-40 is subnormal
    assert list(normgen.bf16_bits(vals)) == want
    assert np.array_equal(normgen.bf16_to_f32(normgen.bf16_bits(vals[:2])), vals[:2])


def test_bf16_rounding_matches_torch():
    import normgen
    torch = pytest.importorskip("torch")
    x = normgen.normal(100_000, 0.0, 100.0, seed=3)
    t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(normgen.bf16_bits(x), t)
    r = normgen.round_bf16(x)
    assert np.array_equal(normgen.bf16_bits(r), t)  # representable values map to themselves
    assert np.all(np.abs(r - x) <= 2.0**-8 * np.abs(x))
