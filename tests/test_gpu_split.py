"""Split launches: the temperature hint (sv_options.temperature_host), and
batches of K = 0 sequences, which split every cluster without a hint.

With a host copy of the temperatures the launch may split some clusters in
two halves that walk the greedy sequences, while the whole clusters take the
sampling sequences first.  The outputs must not change: every hinted call
here is compared with the unhinted call on the same batch, and with the
oracle.  A hint that calls a sampling sequence greedy is caught by the half
that takes it: that sequence's outputs are -1 and the workspace error word
says so.  In these batches the split happens: the wrong hint's sequence has
the longest K of the greedy queue and the lowest index, so the first split
cluster's first half takes it (which the -1 shows).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_04_gb300 as sv  # noqa: E402
import workloads as W  # noqa: E402
from helpers import (compare, dtype_code, oracle_ref_threaded, rows_to_host,  # noqa: E402
                     run_gpu, to_device)  # noqa: E402

pytestmark = pytest.mark.gpu

HINT_BIT = 2   # bit 1 of the workspace error word


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _split_clusters(B, Kmax, V, dtype, temps):
    """How many clusters a hinted call of this batch splits (the library's
    rule, restated so that each test can first check that it splits)."""
    temps = np.asarray(temps)
    g = sv.sv_geometry(B, Kmax, V, dtype_code(dtype))
    nv4 = V >= (2048 if dtype == "bf16" else 1024)
    if V <= 1024 or not nv4 or g["warps"] % 2 or g["warp_ranges"] > 32 or g["clusters"] < 2:
        return 0
    ng = int(np.sum(temps == 0.0))
    ns = B - ng
    cg = min(g["clusters"] * ng // (ng + 6 * ns), g["clusters"] - 1, ng // 2)
    ok = cg >= 1 and ns >= 2 * (g["clusters"] - cg) and g["clusters"] + cg <= 256
    return cg if ok else 0


def _check_splits(d):
    th = d["temperature"].cpu().numpy()
    bad = th.copy()
    bad[0] = 0.0
    for t in (th, bad):
        assert _split_clusters(d["B"], d["Kmax"], d["V"], d["dtype"], t) > 0, \
            "this batch would not split: the test would not reach the split kernel"


def _hinted_equals_unhinted(d, ws, sample=None):
    th = d["temperature"].cpu().numpy()
    t0, n0 = run_gpu(d, "ws", workspace=ws)
    t1, n1 = run_gpu(d, "ex", workspace=ws, temperature_host=th)
    assert sv.sv_workspace_errors(ws) == 0
    assert np.array_equal(t0, t1) and np.array_equal(n0, n1)
    seqs = np.arange(d["B"]) if sample is None else np.asarray(sample)
    host = rows_to_host(d, seqs)
    c = compare(oracle_ref_threaded(host), t1[seqs], n1[seqs], inp=host)
    assert c["n"] == len(seqs)
    return th, t0, n0


def _wrong_hint(d, ws, th, t0, n0):
    """Sequence 0 (K = Kmax, sampling) hinted greedy: -1 and the flag; every
    other sequence as before."""
    K = np.asarray(d["K"])
    assert K[0] == d["Kmax"] and th[0] != 0.0
    bad = th.copy()
    bad[0] = 0.0
    t2, n2 = run_gpu(d, "ex", workspace=ws, temperature_host=bad)
    assert sv.sv_workspace_errors(ws) == HINT_BIT
    assert n2[0] == -1 and np.all(t2[0] == -1)
    assert np.array_equal(t2[1:], t0[1:]) and np.array_equal(n2[1:], n0[1:])
    # the flag was cleared by the read: the next call reports nothing
    run_gpu(d, "ex", workspace=ws, temperature_host=th)
    assert sv.sv_workspace_errors(ws) == 0


def _sampling_first(d):
    """Make sequence 0 a sampling sequence with the longest K (the device
    batch's temperature and K arrays are edited in place)."""
    d["temperature"][0] = 1.0
    K = np.asarray(d["K"], np.int32).copy()
    K[0] = d["Kmax"]
    d["K"] = K
    return d


def test_benchmark_batch_hinted(dev):
    """Workload 4 at full size (B = 1024, half greedy, V = 128256 bf16): the
    hinted call equals the unhinted one on every sequence, and the oracle on
    a sample of 128 of them."""
    d = _sampling_first(W.make_device(4, dev))
    _check_splits(d)
    ws = sv.Workspace(d["B"], d["Kmax"], d["V"], dtype_code(d["dtype"]), dev)
    rng = np.random.default_rng(4)
    sample = np.unique(np.concatenate([[0], rng.choice(d["B"], 127, replace=False)]))
    th, t0, n0 = _hinted_equals_unhinted(d, ws, sample)
    _wrong_hint(d, ws, th, t0, n0)


@pytest.mark.parametrize("greedy_frac,B", [(0.5, 260), (0.7, 400), (0.3, 300)])
def test_mixes_bf16(dev, greedy_frac, B):
    """Other greedy shares and batch sizes (V = 128256 bf16, ragged K):
    every sequence against the oracle."""
    d = _sampling_first(W.make_device(4, dev, B=B))
    rng = np.random.default_rng(int(greedy_frac * 10) + B)
    temps = np.where(rng.random(B) < greedy_frac, 0.0, 1.0).astype(np.float32)
    temps[0] = 1.0
    d["temperature"].copy_(torch.from_numpy(temps))
    _check_splits(d)
    ws = sv.Workspace(B, d["Kmax"], d["V"], dtype_code(d["dtype"]), dev)
    th, t0, n0 = _hinted_equals_unhinted(d, ws)
    _wrong_hint(d, ws, th, t0, n0)


def test_mix_f32(dev):
    """fp32 logits (the first of a few vocabularies near 50000 whose geometry
    splits; K ~ U{0..6}, temperatures 0 / 0.7 / 1.3)."""
    B = 600
    rng = np.random.default_rng(77)
    K = rng.integers(0, 7, size=B).astype(np.int32)
    K[0] = 6
    temps = rng.choice(np.array([0.0, 0.0, 0.7, 1.3], np.float32), size=B)
    temps[0] = 1.3
    bad = temps.copy()
    bad[0] = 0.0
    V = next((v for v in (50000, 48000, 56000, 40000, 64000, 32000, 80000, 24000, 100000)
              if _split_clusters(B, 6, v, "f32", temps) and _split_clusters(B, 6, v, "f32", bad)),
             None)
    assert V is not None, "no fp32 vocabulary of the list splits"
    inp = W.make_host(B, K, V, "f32", 2.0, 1.0, temps, seed=77)
    d = to_device(inp, dev)
    ws = sv.Workspace(B, int(K.max()), V, dtype_code("f32"), dev)
    th, t0, n0 = _hinted_equals_unhinted(d, ws)
    _wrong_hint(d, ws, th, t0, n0)


def test_ragged_k_with_zeros_and_three_temperatures(dev):
    """K drawn from 0..8 (K = 0: the bonus draw alone, greedy or sampling),
    temperatures 0 / 0.8 / 1.5, bf16 logits of the first vocabulary in a
    short list whose geometry splits: every sequence against the oracle."""
    B = 500
    rng = np.random.default_rng(123)
    K = rng.integers(0, 9, size=B).astype(np.int32)
    K[0] = 8
    assert np.sum(K == 0) > 20
    temps = rng.choice(np.array([0.0, 0.0, 0.8, 1.5], np.float32), size=B)
    temps[0] = 1.5
    bad = temps.copy()
    bad[0] = 0.0
    V = next((v for v in (128256, 100000, 64000, 50000, 32000)
              if _split_clusters(B, 8, v, "bf16", temps) and _split_clusters(B, 8, v, "bf16", bad)),
             None)
    assert V is not None, "no bf16 vocabulary of the list splits"
    inp = W.make_host(B, K, V, "bf16", 2.0, 1.0, temps, seed=123)
    d = to_device(inp, dev)
    ws = sv.Workspace(B, 8, V, dtype_code("bf16"), dev)
    th, t0, n0 = _hinted_equals_unhinted(d, ws)
    _wrong_hint(d, ws, th, t0, n0)


def _all_k0_splits(B, V, dtype):
    """Whether a batch of K = 0 sequences splits every cluster (the library's
    rule, restated)."""
    g = sv.sv_geometry(B, 0, V, dtype_code(dtype))
    nv4 = V >= (2048 if dtype == "bf16" else 1024)
    return (V > 1024 and nv4 and g["warps"] % 2 == 0 and g["warp_ranges"] <= 32 and
            B >= 2 * g["clusters"] and 2 * g["clusters"] <= 256)


@pytest.mark.parametrize("dtype,vocabs,B", [("bf16", (128256,), 400),
                                            ("f32", (50000, 40000, 64000, 32000, 24000), 500)])
def test_k0_batches_split_every_cluster(dev, dtype, vocabs, B):
    """A batch of K = 0 sequences (the draft model's sampling step) runs on
    half clusters with no hint: spec_sample and a K = 0 verification give
    the oracle's draws for every row (temperatures 0, 0.7, 1 and 1.6)."""
    V = next((v for v in vocabs if _all_k0_splits(B, v, dtype)), None)
    assert V is not None, "no vocabulary of the list splits"
    temps = np.array([0.0, 0.7, 1.0, 1.6], np.float32)[np.arange(B) % 4]
    inp = W.make_host(B, 0, V, dtype, 2.0, 1.0, temps, seed=B + 7)
    ref = oracle_ref_threaded(inp)
    d = to_device(inp, dev)
    out = sv.spec_sample(d["target"].view(B, V), d["uniforms"].view(B), d["temperature"])
    got = out.cpu().numpy().astype(np.int32).reshape(B, 1)
    c = compare(ref, got, np.zeros(B, np.int32), inp=inp)
    assert c["n"] == B
    ws = sv.Workspace(B, 0, V, dtype_code(dtype), dev)
    t, n = run_gpu(d, "ws", workspace=ws)
    assert sv.sv_workspace_errors(ws) == 0
    assert np.array_equal(t, got) and np.all(n == 0)


def test_hint_ignored_where_it_does_not_apply(dev):
    """All-sampling and all-greedy batches, a small vocabulary, verify-all:
    no split, the same outputs, no flag."""
    for temps in (1.0, 0.0):
        inp = W.make_host(64, 5, 20000, "bf16", 2.0, 1.0, temps, seed=5)
        d = to_device(inp, dev)
        ws = sv.Workspace(64, 5, 20000, dtype_code("bf16"), dev)
        th = np.full(64, temps, np.float32)
        t0, n0 = run_gpu(d, "ws", workspace=ws)
        t1, n1 = run_gpu(d, "ex", workspace=ws, temperature_host=th)
        t2, n2 = run_gpu(d, "ex", workspace=ws, temperature_host=th, verify_all=True)
        assert sv.sv_workspace_errors(ws) == 0
        assert np.array_equal(t0, t1) and np.array_equal(n0, n1)
        assert np.array_equal(t0, t2) and np.array_equal(n0, n2)
    inp = W.make_host(40, 4, 700, "f32", 2.0, 1.0, np.where(np.arange(40) % 2, 0.0, 1.0), seed=6)
    d = to_device(inp, dev)
    ws = sv.Workspace(40, 4, 700, dtype_code("f32"), dev)
    t0, n0 = run_gpu(d, "ws", workspace=ws)
    t1, n1 = run_gpu(d, "ex", workspace=ws, temperature_host=np.zeros(40, np.float32))
    assert sv.sv_workspace_errors(ws) == 0
    assert np.array_equal(t0, t1) and np.array_equal(n0, n1)


def test_hint_shape_is_checked():
    """The binding refuses a hint of the wrong length before any call."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    dev = torch.device("cuda:0")
    inp = W.make_host(4, 2, 3000, "bf16", 2.0, 1.0, 1.0, seed=1)
    d = to_device(inp, dev)
    ws = sv.Workspace(4, 2, 3000, dtype_code("bf16"), dev)
    with pytest.raises(ValueError):
        run_gpu(d, "ex", workspace=ws, temperature_host=np.zeros(3, np.float32))


def test_hint_with_packed_logits_counters_kv_and_graph(dev):
    """Packed logits, the counters and the KV-length commit under a split
    launch give the unhinted call's results; a hinted call captured into a
    CUDA graph replays them."""
    B = 300
    d = _sampling_first(W.make_device(4, dev, B=B))
    _check_splits(d)
    K = np.asarray(d["K"], np.int32)
    th = d["temperature"].cpu().numpy()
    ws = sv.Workspace(B, d["Kmax"], d["V"], dtype_code(d["dtype"]), dev)
    tp = torch.cat([d["target"][b, : K[b] + 1] for b in range(B)]).contiguous()
    dp = torch.cat([d["draft"][b, : K[b]] for b in range(B)]).contiguous()
    res = []
    for hint in (None, th):
        st = sv.Stats()
        kv = torch.arange(B, dtype=torch.int32, device=dev)
        t, n = sv.spec_verify_ex(tp, dp, d["tokens"], d["uniforms"], d["temperature"], K, ws,
                                 packed=True, stats=st, kv_len=kv, temperature_host=hint)
        torch.cuda.synchronize()
        res.append((t.cpu().numpy(), n.cpu().numpy(), st.read(), kv.cpu().numpy()))
        assert sv.sv_workspace_errors(ws) == 0
    (t0, n0, s0, k0), (t1, n1, s1, k1) = res
    assert np.array_equal(t0, t1) and np.array_equal(n0, n1)
    assert s0 == s1 and np.array_equal(k0, k1)
    assert s0["sequences"] == B
    # captured after one ordinary call of the shape (which reserves the
    # graph's header slot), replayed into cleared outputs
    ot = torch.empty((B, d["Kmax"] + 1), dtype=torch.int32, device=dev)
    on = torch.empty((B,), dtype=torch.int32, device=dev)
    args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    sv.spec_verify_ex(*args, ws, out_tokens=ot, out_num_accepted=on, temperature_host=th)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sv.spec_verify_ex(*args, ws, out_tokens=ot, out_num_accepted=on, temperature_host=th)
    ot.fill_(-7)
    on.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(ot.cpu().numpy(), t0) and np.array_equal(on.cpu().numpy(), n0)
    assert sv.sv_workspace_errors(ws) == 0
