"""Host-side input generators: Philox known answers, dtype rounding, shapes."""
import os

import numpy as np

import workloads as W
from workloads.philox import philox4x32_10

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    n = 0
    for line in open(os.path.join(GOLD, "philox4x32_10_kat.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        w = [int(t, 16) for t in line.split()]
        ctr, key, want = w[0:4], w[4:6], w[6:10]
        got = philox4x32_10(np.array([ctr], np.uint32), key)[0]
        assert [int(v) for v in got] == want
        n += 1
    assert n == 3


def test_uniforms_are_exact_24_bit_grid():
    u = W.uniform_grid(123, 1, 50, 7)
    assert u.dtype == np.float32 and u.shape == (50, 7)
    assert np.all((u >= 0) & (u < 1))
    k = u.astype(np.float64) * 2 ** 24
    assert np.all(k == np.floor(k))
    assert np.array_equal(u, W.uniform_grid(123, 1, 50, 7))
    assert not np.array_equal(u, W.uniform_grid(124, 1, 50, 7))


def test_bf16_rounding_round_trip():
    x = np.array([1.0, 1.00390625, 1.005859375, -3.14159, 0.0, 65504.0], np.float32)
    h = W.f32_to_bf16_bits(x)
    y = W.bf16_bits_to_f32(h)
    assert y[0] == 1.0
    assert y[1] == 1.0            # tie rounds to even
    assert y[2] == 1.0078125      # above the tie rounds up
    assert np.all(np.abs(y - x) <= np.abs(x) * 2 ** -8)
    assert np.array_equal(W.f32_to_bf16_bits(y), h)


def test_host_workload_shapes_and_tokens():
    inp = W.make_host(5, np.array([1, 3, 0, 2, 3], np.int32), 100, "bf16", 2.0, 1.0,
                      np.array([1, 0, 1, 0.7, 0], np.float32), seed=8)
    assert inp["target"].shape == (5, 4, 100) and inp["target"].dtype == np.uint16
    assert inp["draft"].shape == (5, 3, 100)
    assert inp["tokens"].shape == (5, 3) and inp["uniforms"].shape == (5, 4)
    d = W.as_f32(inp["draft"], "bf16")
    # greedy sequences propose the draft argmax
    for b in (1, 4):
        for i in range(inp["K"][b]):
            assert inp["tokens"][b, i] == int(np.argmax(d[b, i]))
    assert np.all((inp["tokens"] >= 0) & (inp["tokens"] < 100))


def test_ragged_k_range_and_determinism():
    k = W.configs.ragged_k(1004, 1024)
    assert k.min() == 1 and k.max() == 8
    assert np.array_equal(k, W.configs.ragged_k(1004, 1024))


def test_byte_accounting():
    K = np.array([2, 3], np.int64)
    T = np.array([1.0, 0.0])
    allb = W.bytes_all_rows(K, T, 10, "bf16", 3)
    rows = (3 + 4) + 2          # target rows K+1 each, draft rows only for sampling
    assert allb == rows * 10 * 2 + 2 * 3 * 4 + 2 * 4 * 4 + 2 * 5 * 4
    need = W.bytes_needed(K, T, np.array([0, 3]), 10, "bf16", 3)
    rows_n = (1 + 4) + 1
    assert need == rows_n * 10 * 2 + 2 * 3 * 4 + 2 * 4 * 4 + 2 * 5 * 4
