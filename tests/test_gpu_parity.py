"""GPU parity: libspecverify (through its C ABI) against the fp64 oracle.

Token outputs and num_accepted must be bit-exact except for sequences the
oracle flags as ties (a uniform within 1e-6 of an acceptance threshold or of
a CDF boundary on the path it walks); those are counted.  Per-position
probabilities must agree within 1e-5 relative error.
"""
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import speculative_decoding_verification_04_gb300 as sv  # noqa: E402
import workloads as W  # noqa: E402
from helpers import (compare, dtype_code, oracle_ref, oracle_ref_threaded, rows_to_host,  # noqa: E402
                     run_gpu, to_device)  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _check(inp, dev, mode="ws", **kw):
    ref = oracle_ref(inp)
    got_t, got_n = run_gpu(to_device(inp, dev), mode, **kw)
    return ref, got_t, got_n, compare(ref, got_t, got_n, inp=inp)


# ---------------------------------------------------------------------------
# small and tiny workloads, element by element
# ---------------------------------------------------------------------------
def test_workload0_b64_k4_v5(dev):
    _, _, _, c = _check(W.make_spec_host(0), dev)
    assert c["n"] == 64


def test_toy_pair_200k(dev):
    inp = W.make_toy(200_000, seed=1000)
    ref, got_t, got_n, c = _check(inp, dev)
    assert abs(got_n.mean() - 0.78) < 4 * np.sqrt(0.78 * 0.22 / 200_000)
    freq = np.bincount(got_t[:, 0], minlength=5) / 200_000
    assert np.all(np.abs(freq - W.TOY_P) < 0.005)


SMALL = [
    # name, B, K, V, dtype, temps
    ("f32_v5003_mixed", 12, [0, 1, 2, 3, 4, 5, 5, 4, 3, 2, 1, 0], 5003, "f32",
     [1.0, 0.0, 0.7, 2.0, 1.0, 0.0, 1.0, 0.5, 0.0, 1.0, 1.0, 0.0]),
    ("bf16_v5003_mixed", 12, [0, 1, 2, 3, 4, 5, 5, 4, 3, 2, 1, 0], 5003, "bf16",
     [1.0, 0.0, 0.7, 2.0, 1.0, 0.0, 1.0, 0.5, 0.0, 1.0, 1.0, 0.0]),
    ("f32_v4999_unaligned", 9, 3, 4999, "f32", 1.0),
    ("bf16_v4097_unaligned", 9, 3, 4097, "bf16", 0.8),
    ("bf16_v3", 40, 4, 3, "bf16", 1.0),
    ("f32_v1", 5, 2, 1, "f32", 1.0),
    ("f32_v300", 30, 6, 300, "f32", 1.2),
    ("bf16_v33000_k8", 8, 8, 33000, "bf16", 1.0),
    ("bf16_v700_k32", 3, 32, 700, "bf16", 1.0),
    ("f32_v20000_greedy", 10, 5, 20000, "f32", 0.0),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_workloads_match_oracle(dev, case):
    name, B, K, V, dtype, temps = case
    inp = W.make_host(B, K, V, dtype, 2.0, 1.0, temps, seed=zlib.crc32(name.encode()) % 10000)
    _check(inp, dev)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_largest_vocabulary(dev, dtype):
    """The largest V the library accepts (a row of target and draft resident
    in one cluster of 16 CTAs): greedy and sampling rows against the oracle."""
    V = sv.sv_max_vocab(dtype_code(dtype))
    B = 6
    temps = np.array([1.0, 0.0, 0.7, 1.0, 0.0, 1.3], np.float32)
    inp = W.make_host(B, [3, 2, 3, 1, 3, 2], V, dtype, 2.0, 1.0, temps, seed=V % 997)
    _check(inp, dev)


def test_high_acceptance_reaches_bonus_rows(dev):
    inp = W.make_host(24, 6, 9000, "bf16", 2.0, 0.02, 1.0, seed=5)
    ref, got_t, got_n, _ = _check(inp, dev)
    assert np.mean(got_n == 6) > 0.5


@pytest.mark.parametrize("dtype,V", [("bf16", 3001), ("f32", 2500), ("bf16", 700), ("f32", 600)])
def test_longest_walks_reach_position_32(dev, dtype, V):
    """K = 32 (the most a call takes) with drafts close to the target, so
    that walks run through all 32 tests to the bonus row at position 32:
    the last lane's token and uniform, the final uniform in slot 32 and a
    33-token output row (V = 700 and 600 take the small-vocabulary kernel)."""
    T = np.where(np.arange(8) % 4 == 0, 0.0, 1.0).astype(np.float32)
    inp = W.make_host(8, 32, V, dtype, 2.0, 0.01, T, seed=V + 32)
    ref, got_t, got_n, _ = _check(inp, dev)
    assert np.any(got_n == 32)


def test_greedy_ties_lowest_index(dev):
    inp = W.make_host(16, 4, 6000, "bf16", 2.0, 1.0, 0.0, seed=6)
    # coarse logits: many exact ties at the row maximum
    for k in ("target", "draft"):
        f = np.round(W.as_f32(inp[k], "bf16"))
        inp[k] = W.f32_to_bf16_bits(f)
    d = W.as_f32(inp["draft"], "bf16")
    inp["tokens"] = np.argmax(d, axis=-1).astype(np.int32)
    _check(inp, dev)


def test_special_uniforms(dev):
    """Uniforms at the ends of [0, 1): a final uniform of 0 or 1 - 2^-24 lies
    within 1e-6 of the first or last CDF boundary, so every sequence here is
    a tie by the oracle's definition; the GPU must still give the oracle's
    results (the first and the last token with mass), bit for bit."""
    inp = W.make_host(32, 3, 2000, "f32", 2.0, 1.0, 1.0, seed=8)
    inp["uniforms"][:8] = 0.0
    inp["uniforms"][8:16] = np.float32(1 - 2 ** -24)
    inp["uniforms"][16:24, -1] = 0.0
    inp["uniforms"][24:, -1] = np.float32(1 - 2 ** -24)
    ref = oracle_ref(inp)
    got_t, got_n = run_gpu(to_device(inp, dev), "ws")
    c = compare(ref, got_t, got_n, inp=inp, max_ties=32)
    assert c["tie_mismatch"] == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_proposals_far_below_the_row_max(dev, dtype):
    """Weights taken against the proposal's own logit overflow when that logit
    lies far below the row's maximum (or is -inf); such rows are weighed again
    against their maxima and must still match the oracle."""
    B, K, V = 24, 3, 3000
    inp = W.make_host(B, K, V, "f32", 2.0, 1.0, 1.0, seed=21)
    tgt, drf, tok = inp["target"], inp["draft"], inp["tokens"]
    for b in range(B):
        for i in range(K):
            x = tok[b, i]
            if b % 4 == 0:    # target logit at x 200 below a spike: exp2 of ~288 overflows
                tgt[b, i, (x + 7) % V] = 150.0
                tgt[b, i, x] = -50.0
            elif b % 4 == 1:  # draft logit at x far below its own spike
                drf[b, i, (x + 11) % V] = 150.0
                drf[b, i, x] = -60.0
            elif b % 4 == 2:  # -inf at the proposal in the target row: p(x) = 0
                tgt[b, i, x] = -np.inf
    if dtype == "bf16":
        for k in ("target", "draft"):
            inp[k] = W.configs.f32_to_bf16_bits(inp[k])
        inp["dtype"] = "bf16"
    _check(inp, dev)


def test_workload1_full_size(dev):
    _check(W.make_spec_host(1), dev)


def test_workload2_full_size_host_generated(dev):
    _check(W.make_spec_host(2), dev)


# ---------------------------------------------------------------------------
# invalid device data and degenerate inputs
# ---------------------------------------------------------------------------
def test_invalid_inputs_give_minus_one(dev):
    B, K, V = 10, 3, 1500
    inp = W.make_host(B, K, V, "f32", 2.0, 1.0, 1.0, seed=9)
    inp["tokens"][:, 0] = np.argmax(W.as_f32(inp["target"], "f32")[:, 0], axis=-1)
    inp["target"][0, 0, 7] = np.nan          # tested row
    inp["target"][1, 0, 9] = np.inf
    inp["tokens"][2, 0] = V                  # token out of range
    inp["uniforms"][3, 0] = 1.0              # uniform out of range
    inp["temperature"][4] = -1.0
    inp["temperature"][5] = np.nan
    inp["draft"][6, 0, :] = -np.inf          # draft row with no finite entry
    inp["uniforms"][7, 3] = 2.0              # final-draw uniform out of range
    # sequence 8: reject at position 0 for sure, NaN in the rows after it
    inp["tokens"][8, 0] = int(np.argmin(W.as_f32(inp["target"], "f32")[8, 0]))
    inp["draft"][8, 0, inp["tokens"][8, 0]] = 50.0
    inp["uniforms"][8, 0] = 0.999
    inp["target"][8, 1:, :] = np.nan
    inp["draft"][8, 1:, :] = np.nan
    ref, got_t, got_n, _ = _check(inp, dev)
    assert list(got_n[:8]) == [-1] * 8
    assert np.all(got_t[:8] == -1)
    assert got_n[8] == 0 and got_t[8, 0] >= 0


def test_missing_draft_logits(dev):
    inp = W.make_host(6, 3, 800, "bf16", 2.0, 1.0, [0, 0, 1, 0, 1, 0], seed=10)
    d = to_device(inp, dev)
    ref = oracle.verify(inp["target"], None, "bf16", inp["tokens"], inp["uniforms"],
                        inp["temperature"], inp["K"])
    K = inp["K"]
    t, n = sv.spec_verify(d["target"], None, d["tokens"], d["uniforms"], d["temperature"], K)
    torch.cuda.synchronize()
    compare(ref, t.cpu().numpy(), n.cpu().numpy())
    assert n.cpu().numpy()[2] == -1 and n.cpu().numpy()[0] >= 0


def test_empty_batch_is_noop(dev):
    t = torch.zeros((0, 1, 10), device=dev)
    out_t, out_n = sv.spec_verify(t, None, None, torch.zeros((0, 1), device=dev),
                                  torch.zeros(0, device=dev), np.zeros(0, np.int32))
    assert out_t.shape == (0, 1) and out_n.shape == (0,)


# ---------------------------------------------------------------------------
# entry points, options, determinism
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def mixed(dev):
    inp = W.make_host(40, W.configs.ragged_k(3, 40), 12345, "bf16", 2.0, 1.0,
                      np.where(np.arange(40) % 3 == 0, 0.0, 0.9).astype(np.float32), seed=12)
    return inp, to_device(inp, dev), oracle_ref(inp)


def test_entry_points_agree(dev, mixed):
    inp, d, ref = mixed
    base = run_gpu(d, "ws")
    compare(ref, *base, inp=inp)
    for mode in ("alloc", "ex"):
        got = run_gpu(d, mode)
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1]), mode
    staging = torch.empty(sv.sv_host_staging_size(inp["B"], inp["Kmax"], inp["V"],
                                                  sv.SV_DTYPE_BF16), dtype=torch.uint8, device=dev)
    ht = torch.from_numpy(inp["target"].view(np.int16)).view(torch.bfloat16)
    hd = torch.from_numpy(inp["draft"].view(np.int16)).view(torch.bfloat16)
    t, n = sv.spec_verify_host(ht, hd, torch.from_numpy(inp["tokens"]),
                               torch.from_numpy(inp["uniforms"]),
                               torch.from_numpy(inp["temperature"]), inp["K"], staging)
    assert np.array_equal(t.numpy(), base[0]) and np.array_equal(n.numpy(), base[1])
    # page-locked logits are read in place by the kernel: the same results
    t, n = sv.spec_verify_host(ht.pin_memory(), hd.pin_memory(), torch.from_numpy(inp["tokens"]),
                               torch.from_numpy(inp["uniforms"]),
                               torch.from_numpy(inp["temperature"]), inp["K"], staging)
    assert np.array_equal(t.numpy(), base[0]) and np.array_equal(n.numpy(), base[1])


@pytest.mark.parametrize("idx", [3, 4])
def test_host_logits_read_in_place_full_size(dev, idx):
    """Full-size workloads from page-locked host logits (read in place over
    the host link, bf16 and fp32, greedy and sampling rows): the device
    results, bit for bit."""
    d = W.make_device(idx, dev)
    B, Kmax, V = d["B"], d["Kmax"], d["V"]
    base = run_gpu(d, "ws")
    code = dtype_code(d["dtype"])
    staging = torch.empty(sv.sv_host_staging_size(B, Kmax, V, code), dtype=torch.uint8, device=dev)
    host = [d[k].cpu().pin_memory() for k in ("target", "draft", "tokens", "uniforms", "temperature")]
    t, n = sv.spec_verify_host(*host, d["K"], staging)
    assert np.array_equal(t.numpy(), base[0]) and np.array_equal(n.numpy(), base[1])


def test_verify_all_gives_identical_outputs(dev, mixed):
    inp, d, ref = mixed
    base = run_gpu(d, "ws")
    got = run_gpu(d, "ex", verify_all=True)
    assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1])


GEOMETRIES = [dict(chunks_per_cta=1), dict(chunks_per_cta=2), dict(chunks_per_cta=5),
              dict(chunks_per_cta=13), dict(chunks_per_cta=4, chunks_per_warp=4),
              dict(chunks_per_cta=13, chunks_per_warp=1), dict(chunks_per_cta=3, chunks_per_warp=3),
              dict(chunks_per_cta=8, chunks_per_warp=2),
              dict(verify_all=True, chunks_per_cta=5, chunks_per_warp=2)]


@pytest.mark.parametrize("kw", GEOMETRIES, ids=[str(sorted(g.items())) for g in GEOMETRIES])
def test_launch_geometries_match_oracle(dev, mixed, kw):
    """Tuning options change only the fp32 summation grouping: every geometry
    agrees with the oracle outside its tie band, and a geometry reproduces
    itself bit for bit."""
    inp, d, ref = mixed
    got = run_gpu(d, "ex", **kw)
    compare(ref, *got, inp=inp)
    again = run_gpu(d, "ex", **kw)
    assert np.array_equal(got[0], again[0]) and np.array_equal(got[1], again[1])


# chunks per CTA, chunks per warp: one to sixteen CTAs per row, one to eight
# warps per CTA, one to twenty chunks per warp, up to 64 warp ranges per row
# (two partials per lane in the combines)
LARGE_GEOMETRIES = [("bf16", 128256, 16, 4), ("bf16", 128256, 8, 2), ("bf16", 128256, 21, 2),
                    ("bf16", 128256, 32, 8), ("bf16", 128256, 20, 20), ("f32", 151936, 21, 2),
                    ("f32", 151936, 38, 10), ("f32", 151936, 20, 20),
                    ("bf16", 128256, 16, 2), ("bf16", 128256, 9, 1), ("f32", 151936, 50, 7)]


@pytest.mark.parametrize("dtype,V,ncpc,cpw", LARGE_GEOMETRIES)
def test_large_vocab_geometries_match_oracle(dev, dtype, V, ncpc, cpw):
    B = 12
    inp = W.make_host(B, W.configs.ragged_k(7, B), V, dtype, 2.0, 1.0,
                      np.where(np.arange(B) % 2 == 0, 0.0, 1.0).astype(np.float32), seed=ncpc * 31 + cpw)
    ref = oracle_ref(inp)
    got = run_gpu(to_device(inp, dev), "ex", chunks_per_cta=ncpc, chunks_per_warp=cpw)
    compare(ref, *got, inp=inp)


def test_deterministic_across_runs(dev, mixed):
    inp, d, ref = mixed
    a = run_gpu(d, "ws")
    for _ in range(3):
        b = run_gpu(d, "ws")
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_no_device_errors_recorded(dev, mixed):
    inp, d, ref = mixed
    ws = sv.Workspace(inp["B"], inp["Kmax"], inp["V"], sv.SV_DTYPE_BF16, dev)
    run_gpu(d, "ws", workspace=ws)
    assert sv.sv_workspace_errors(ws) == 0


# ---------------------------------------------------------------------------
# per-position probabilities (diagnostics) within 1e-5 relative
# ---------------------------------------------------------------------------
# the last case runs the kernel variant with more than 32 warp ranges per row
@pytest.mark.parametrize("dtype,V,T", [("f32", 7001, 0.7), ("bf16", 12345, 1.0), ("f32", 5, 1.0),
                                       ("f32", 151936, 0.7)])
def test_position_probabilities(dev, dtype, V, T):
    B, K = 16, 5
    inp = W.make_host(B, K, V, dtype, 2.0, 1.0, T, seed=V)
    d = to_device(inp, dev)
    px = torch.full((B, K), -7.0, device=dev)
    qx = torch.full((B, K), -7.0, device=dev)
    rm = torch.full((B, K), -7.0, device=dev)
    fr = torch.full((B,), -7, dtype=torch.int32, device=dev)
    got_t, got_n = run_gpu(d, "ex", diag=dict(p_x=px, q_x=qx, resid_mass=rm, final_row=fr))
    ref = oracle_ref(inp)
    compare(ref, got_t, got_n, inp=inp)
    opx, oqx, orm = oracle.position_probs(inp["target"], inp["draft"], dtype, inp["tokens"],
                                          inp["temperature"], inp["K"])
    for g, o in ((px, opx), (qx, oqx)):
        g = g.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g))
        assert np.max(np.abs(g - o) / o) < 1e-5
    g = rm.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(g - orm)) < 1e-5
    assert np.array_equal(fr.cpu().numpy(), got_n)


# ---------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration: every sequence
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_workloads_every_sequence(dev, idx):
    """Workloads 1-4 at full size, generated on the device as the benchmark
    does and verified in its launch geometry: every sequence against the
    oracle (run over all host cores), bit-exact outside the counted ties."""
    d = W.make_device(idx, dev)
    B = d["B"]
    K = np.asarray(d["K"])
    # the draft rows carry the workload's noise (they are not the target rows)
    noise = (d["draft"][:, 0].float() - d["target"][:, 0].float()).std().item()
    assert abs(noise - W.SPECS[idx].sigma_d) < 0.05 * W.SPECS[idx].sigma_d + 0.01
    ws = sv.Workspace(B, d["Kmax"], d["V"], dtype_code(d["dtype"]), dev)
    got_t, got_n = run_gpu(d, "ws", workspace=ws)
    assert sv.sv_workspace_errors(ws) == 0
    assert np.all((got_n >= 0) & (got_n <= K))
    host = rows_to_host(d, np.arange(B))
    ref = oracle_ref_threaded(host)
    c = compare(ref, got_t, got_n, inp=host)
    assert c["n"] == B


@pytest.mark.parametrize("dtype,V,ncpc,cpw,parts", [("bf16", 128256, 16, 2, 64), ("bf16", 128256, 9, 1, 56),
                                                     ("f32", 151936, 50, 7, 48)])
def test_wide_geometries_use_more_than_32_ranges(dev, dtype, V, ncpc, cpw, parts):
    """The overrides above really cut a row into more than 32 warp ranges."""
    code = sv.SV_DTYPE_BF16 if dtype == "bf16" else sv.SV_DTYPE_F32
    g = sv.sv_geometry(12, 7, V, code, ncpc, cpw)
    assert g["cluster_ctas"] * g["warps"] == parts == g["warp_ranges"]
