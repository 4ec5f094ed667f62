"""Small vocabularies (V <= 1024) take a warp-per-sequence kernel: every
output against the oracle, element by element, with the cluster sweep (forced
by a tuning option) giving the oracle's results on the same inputs; the
options (packed layout, counters, KV lengths, diagnostics) and unusable
inputs as in the sweep."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_04_gb300 as sv  # noqa: E402
import workloads as W  # noqa: E402
from helpers import compare, dtype_code, oracle_ref, run_gpu, to_device  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _mixed(B, V, dtype, seed):
    K = (W.configs.ragged_k(seed, B, 1, 9) - 1).astype(np.int32)   # 0..8
    temps = np.where(np.arange(B) % 3 == 0, 0.0, np.where(np.arange(B) % 3 == 1, 1.0, 0.7)).astype(np.float32)
    return W.make_host(B, K, V, dtype, 2.0, 1.0, temps, seed=seed)


@pytest.mark.parametrize("V", [1, 5, 32, 33, 100, 257, 700, 1024])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_vocab_matches_oracle(dev, V, dtype):
    inp = _mixed(90, V, dtype, seed=V * 7 + len(dtype))
    ref = oracle_ref(inp)
    d = to_device(inp, dev)
    compare(ref, *run_gpu(d, "ws"), inp=inp)
    # the cluster sweep on the same inputs (a tuning option selects it)
    compare(ref, *run_gpu(d, "ex", chunks_per_cta=1), inp=inp)


def test_small_vocab_unusable_inputs(dev):
    B, K, V = 10, 3, 300
    inp = W.make_host(B, K, V, "f32", 2.0, 1.0, 1.0, seed=9)
    inp["tokens"][:, 0] = np.argmax(W.as_f32(inp["target"], "f32")[:, 0], axis=-1)
    inp["target"][0, 0, 7] = np.nan
    inp["target"][1, 0, 9] = np.inf
    inp["tokens"][2, 0] = V
    inp["uniforms"][3, 0] = 1.0
    inp["temperature"][4] = -1.0
    inp["temperature"][5] = np.nan
    inp["draft"][6, 0, :] = -np.inf
    inp["uniforms"][7, 3] = 2.0
    inp["tokens"][8, 0] = int(np.argmin(W.as_f32(inp["target"], "f32")[8, 0]))
    inp["draft"][8, 0, inp["tokens"][8, 0]] = 50.0
    inp["uniforms"][8, 0] = 0.999
    inp["target"][8, 1:, :] = np.nan
    inp["draft"][8, 1:, :] = np.nan
    ref = oracle_ref(inp)
    t, n = run_gpu(to_device(inp, dev), "ws")
    compare(ref, t, n, inp=inp)
    assert list(n[:8]) == [-1] * 8 and np.all(t[:8] == -1)
    assert n[8] == 0 and t[8, 0] >= 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_vocab_options(dev, dtype):
    """Packed logits, counters and KV lengths give what the padded, plain
    call and the oracle's walk give."""
    B, V = 70, 200
    inp = _mixed(B, V, dtype, seed=3)
    d = to_device(inp, dev)
    k = np.asarray(inp["K"])
    ws = sv.Workspace(B, int(k.max()), V, dtype_code(dtype), dev)
    st = sv.Stats(dev)
    kv = torch.arange(B, dtype=torch.int32, device=dev) * 10
    base = kv.clone()
    t0, n0 = run_gpu(d, "ex", workspace=ws, stats=st, kv_len=kv)
    ref = oracle_ref(inp)
    compare(ref, t0, n0, inp=inp)
    got = st.read()
    valid = n0 >= 0
    assert got["sequences"] == int(valid.sum()) and got["invalid"] == int((~valid).sum())
    assert got["committed"] == int((n0[valid] + 1).sum()) and got["accepted"] == int(n0[valid].sum())
    assert got["tested"] == int(np.where(valid, n0 + (n0 < k), 0).sum())
    assert np.array_equal(kv.cpu().numpy()[valid], base.cpu().numpy()[valid] + 1 + n0[valid])
    tp = torch.cat([d["target"][b, : k[b] + 1] for b in range(B)]).contiguous()
    dp = torch.cat([d["draft"][b, : max(k[b], 0)] for b in range(B)]).contiguous()
    t1, n1 = sv.spec_verify_ex(tp, dp, d["tokens"], d["uniforms"], d["temperature"], k, ws, packed=True)
    torch.cuda.synchronize()
    assert np.array_equal(t1.cpu().numpy(), t0) and np.array_equal(n1.cpu().numpy(), n0)


@pytest.mark.parametrize("V,dtype", [(5, "f32"), (257, "bf16"), (1024, "f32"), (1024, "bf16")])
def test_small_vocab_diagnostics_and_verify_all(dev, V, dtype):
    """Diagnostics (which force verify_all) on the warp kernel: p(x_i), q(x_i)
    within 1e-5 relative and the residual mass within 1e-5 at every sampling
    position below K_b, rows after the stop included; NaN where the oracle has
    none (greedy sequences, positions past K_b); outputs unchanged."""
    import oracle
    B = 40
    inp = _mixed(B, V, dtype, seed=V + 11)
    d = to_device(inp, dev)
    Kmax = int(inp["Kmax"])
    bufs = [torch.full((B, Kmax), -7.0, device=dev) for _ in range(3)]
    fr = torch.full((B,), -7, dtype=torch.int32, device=dev)
    t0, n0 = run_gpu(d, "ws")
    t1, n1 = run_gpu(d, "ex", diag=dict(p_x=bufs[0], q_x=bufs[1], resid_mass=bufs[2], final_row=fr))
    assert np.array_equal(t0, t1) and np.array_equal(n0, n1)
    compare(oracle_ref(inp), t1, n1, inp=inp)
    opx, oqx, orm = oracle.position_probs(inp["target"], inp["draft"], dtype, inp["tokens"],
                                          inp["temperature"], inp["K"])
    gpx, gqx, grm = (b.cpu().numpy().astype(np.float64) for b in bufs)
    want = np.isfinite(opx)
    assert want.sum() > B            # rows after the stop are among them
    assert np.array_equal(np.isnan(gpx), ~want) and np.array_equal(np.isnan(gqx), ~want)
    for g, o in ((gpx, opx), (gqx, oqx)):
        assert np.max(np.abs(g[want] - o[want]) / o[want]) < 1e-5
    assert np.max(np.abs(grm[want] - orm[want])) < 1e-5
    assert np.array_equal(fr.cpu().numpy(), n1)


def test_toy_pair_through_the_small_kernel_is_fast(dev):
    """The pages' V = 5 pair replicated 200,000 times: the oracle's results,
    and the whole batch in well under a millisecond (the cluster sweep took
    2.4 ms)."""
    inp = W.make_toy(200_000, seed=1000)
    d = to_device(inp, dev)
    ws = sv.Workspace(200_000, 1, 5, sv.SV_DTYPE_F32, dev)
    compare(oracle_ref(inp), *run_gpu(d, "ws", workspace=ws), inp=inp)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K = np.asarray(inp["K"], np.int32)
    args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    sv.spec_verify_ws(*args, ws)
    e0.record()
    for _ in range(5):
        sv.spec_verify_ws(*args, ws)
    e1.record()
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) / 5 < 1.0
