"""GPU tests of the entry points beside verification: the draft-side sampler
(spec_sample), the per-call counters (sv_stats) and the on-device KV-length
commit (kv_len).  Each is checked against the oracle or against what the
verified outputs imply."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import speculative_decoding_verification_04_gb300 as sv  # noqa: E402
import workloads as W  # noqa: E402
from helpers import compare, dtype_code, oracle_ref, run_gpu, to_device  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.mark.parametrize("dtype,V,B", [("bf16", 9000, 64), ("f32", 7001, 40), ("bf16", 128256, 48),
                                       ("f32", 151936, 16), ("bf16", 3, 32)])
def test_spec_sample_is_the_oracles_draw_from_p(dev, dtype, V, B):
    """One token per row from softmax(l / T) (argmax at T = 0): the final draw
    of a K = 0 verification, which the oracle defines; bit-exact outside the
    oracle's tie band."""
    temps = np.where(np.arange(B) % 4 == 0, 0.0, np.where(np.arange(B) % 4 == 1, 0.7, 1.0))
    inp = W.make_host(B, 0, V, dtype, 2.0, 1.0, temps.astype(np.float32), seed=V % 1000 + B)
    ref = oracle_ref(inp)
    d = to_device(inp, dev)
    logits = d["target"].view(B, V)
    out = sv.spec_sample(logits, d["uniforms"].view(B), d["temperature"])
    got = out.cpu().numpy().astype(np.int32)
    compare(ref, got.reshape(B, 1), np.zeros(B, np.int32), inp=inp)


def test_spec_sample_marks_unusable_rows(dev):
    """A NaN logit or a uniform outside [0, 1) gives -1 for that row only."""
    import torch
    B, V = 8, 4000
    inp = W.make_host(B, 0, V, "f32", 2.0, 1.0, 1.0, seed=11)
    ref = oracle_ref(inp)
    d = to_device(inp, dev)
    logits = d["target"].view(B, V).clone()
    logits[2, 17] = float("nan")
    uni = d["uniforms"].view(B).clone()
    uni[5] = 1.0
    got = sv.spec_sample(logits, uni, d["temperature"]).cpu().numpy()
    assert got[2] == -1 and got[5] == -1
    keep = [b for b in range(B) if b not in (2, 5)]
    ok = ~ref["tie"][keep]
    assert np.array_equal(got[keep][ok], ref["out_tokens"][keep, 0][ok])


def _oracle_counts(inp: dict, ref: dict) -> dict:
    """The sv_stats counters the oracle's walk implies.  tested: the positions
    up to and including the first rejection (n_b, plus one when n_b < K_b);
    accepted: sum n_b; committed: sum (n_b + 1); over valid sequences.
    near_ties: the walked sampling tests whose uniform lies within 1e-6 of
    p(x)/q(x), from the oracle's per-position probabilities (fp64)."""
    K = np.asarray(inp["K"])
    n = ref["num_accepted"]
    valid = n >= 0
    tested = np.where(valid, n + (n < K), 0)
    px, qx, _ = oracle.position_probs(inp["target"], inp["draft"], inp["dtype"], inp["tokens"],
                                      inp["temperature"], inp["K"])
    near = 0
    for b in np.flatnonzero(valid & (np.asarray(inp["temperature"]) > 0)):
        for i in range(int(tested[b])):
            if qx[b, i] > 0 and abs(float(inp["uniforms"][b, i]) - px[b, i] / qx[b, i]) < 1e-6:
                near += 1
    return dict(sequences=int(valid.sum()), invalid=int((~valid).sum()), tested=int(tested.sum()),
                accepted=int(np.where(valid, n, 0).sum()), committed=int(np.where(valid, n + 1, 0).sum()),
                near_ties=near)


def test_stats_match_the_oracles_walk(dev):
    """The per-call counters equal what the oracle's walk implies (counts of
    tested and accepted positions as the acceptance rate is counted on the
    pages: r-jc.jp, section 投機的デコーディングを実装して受理率と速度を実測,
    decisions after the first rejection are not taken).  Uniforms are planted
    5e-7 below or above p/q at position 0 of the sampling sequences whose p/q
    lies below 1, so near_ties is nonzero, and must be exact; the planted
    sequences are the oracle's ties.  The counts are the same under
    verify_all (rows after the stop do not count), and a second call
    accumulates."""
    B, V = 48, 6000
    temps = np.where(np.arange(B) % 3 == 0, 0.0, 1.0).astype(np.float32)
    inp = W.make_host(B, W.configs.ragged_k(5, B), V, "bf16", 2.0, 0.6, temps, seed=17)
    px, qx, _ = oracle.position_probs(inp["target"], inp["draft"], "bf16", inp["tokens"],
                                      inp["temperature"], inp["K"])
    planted = []
    for b in np.flatnonzero(temps > 0):
        ratio = px[b, 0] / qx[b, 0]
        if 1e-3 < ratio < 1 - 1e-3:
            inp["uniforms"][b, 0] = np.float32(ratio + (5e-7 if len(planted) % 2 else -5e-7))
            planted.append(b)
    assert len(planted) >= 8
    ref = oracle_ref(inp)
    assert ref["tie"][planted].all()
    want = _oracle_counts(inp, ref)
    assert want["near_ties"] >= len(planted)
    d = to_device(inp, dev)
    ws = sv.Workspace(B, int(inp["Kmax"]), V, dtype_code("bf16"), dev)
    st = sv.Stats(dev)
    t, n = run_gpu(d, "ex", workspace=ws, stats=st)
    # the walks agree everywhere, the planted decisions included (5e-7 is far
    # beyond the fp32 rounding of p/q at this size)
    assert np.array_equal(n, ref["num_accepted"]) and np.array_equal(t, ref["out_tokens"])
    got = st.read()
    for k, v in want.items():
        assert got[k] == v, (k, got[k], v)
    st_all = sv.Stats(dev)
    t2, n2 = run_gpu(d, "ex", workspace=ws, stats=st_all, verify_all=True)
    assert np.array_equal(n, n2) and st_all.read() == got
    run_gpu(d, "ex", workspace=ws, stats=st)   # accumulates
    again = st.read()
    for k in want:
        assert again[k] == 2 * got[k]


def _draw_rows(inp: dict, ref: dict, b: int):
    """The oracle's final-draw distribution of sequence b (fp64, normalised)
    and its CDF, or None when the draw is not a sampling draw with mass."""
    K = int(inp["K"][b])
    n = int(ref["num_accepted"][b])
    T = float(inp["temperature"][b])
    if n < 0 or T == 0.0:
        return None
    drow = inp["draft"][b, n] if n < K else None
    r, code = oracle.final_distribution(inp["target"][b, n], drow, inp["dtype"], T)
    if code == 0:   # (2: no residual mass, r is p: the distribution drawn from all the same)
        return None
    return np.cumsum(r)


def _draw_tie_counts(inp: dict, ref: dict):
    """(draws within 1e-6 of a bound of the drawn token's CDF interval, draws
    whose distance lies in [0.8e-6, 1.2e-6], where fp32 rounding may decide
    either way), from the oracle's fp64 CDF."""
    near = amb = 0
    for b in range(inp["B"]):
        C = _draw_rows(inp, ref, b)
        if C is None:
            continue
        K, n = int(inp["K"][b]), int(ref["num_accepted"][b])
        j = int(ref["out_tokens"][b, n])
        u = float(inp["uniforms"][b, K])
        lo = C[j - 1] if j > 0 else 0.0
        dist = min(abs(u - lo), abs(C[j] - u))
        near += dist < 1e-6
        amb += 0.8e-6 <= dist <= 1.2e-6
    return near, amb


@pytest.mark.parametrize("dtype,V", [("bf16", 6000), ("f32", 5003), ("f32", 700), ("bf16", 257)])
def test_draw_near_ties_match_the_oracle(dev, dtype, V):
    """sv_stats.draw_near_ties counts the final draws whose point lies within
    1e-6 of a bound of the drawn token's interval, as the oracle flags them
    (V = 700 and 257 take the small-vocabulary kernel).  The final uniforms
    of most sampling sequences are planted 5e-7 below or above a CDF bound
    in the middle of the distribution (the tokens on both sides with mass
    above 1e-5), so the count is large; draws that fall near the band's own edge
    by chance are the only slack allowed."""
    B = 40
    temps = np.where(np.arange(B) % 4 == 0, 0.0, 1.0).astype(np.float32)
    inp = W.make_host(B, W.configs.ragged_k(7, B), V, dtype, 2.0, 0.6, temps, seed=V + 5)
    ref = oracle_ref(inp)
    planted = 0
    for b in range(B):
        C = _draw_rows(inp, ref, b)
        if C is None or b % 5 == 4:   # leave some draws as they are
            continue
        j = int(np.searchsorted(C, 0.5))
        r = np.diff(np.concatenate([[0.0], C]))
        after = np.flatnonzero(r[j + 1:] > 0)   # the next token with mass starts at C_j
        if r[j] < 1e-5 or len(after) == 0 or r[j + 1 + after[0]] < 1e-5:
            continue
        u = np.float32(C[j] + (5e-7 if planted % 2 else -5e-7))
        if abs(float(u) - C[j]) >= 9e-7:   # the float32 grid near C_j is coarser than the band
            continue
        inp["uniforms"][b, int(inp["K"][b])] = u
        planted += 1
    assert planted >= 10
    ref = oracle_ref(inp)   # the walks are unchanged; the draws moved
    want, amb = _draw_tie_counts(inp, ref)
    assert want >= planted
    d = to_device(inp, dev)
    ws = sv.Workspace(B, int(inp["Kmax"]), V, dtype_code(dtype), dev)
    st = sv.Stats(dev)
    t, n = run_gpu(d, "ex", workspace=ws, stats=st)
    # every planted draw is a tie: only the counted ties may differ
    compare(ref, t, n, inp=inp, max_ties=B)
    got = st.read()["draw_near_ties"]
    assert abs(got - want) <= amb, (got, want, amb)


def test_kv_len_advances_by_committed_tokens(dev):
    """kv_len[b] += 1 + n_b for valid sequences, unchanged for invalid ones."""
    import torch
    B = 24
    inp = W.make_host(B, 4, 5000, "f32", 2.0, 0.5, 1.0, seed=23)
    inp["target"][3, 0, 10] = np.nan          # sequence 3 is invalid
    d = to_device(inp, dev)
    base = torch.arange(B, dtype=torch.int32, device=dev) * 100
    kv = base.clone()
    st = sv.Stats(dev)
    t, n = run_gpu(d, "ex", kv_len=kv, stats=st)
    kvh, bh = kv.cpu().numpy(), base.cpu().numpy()
    assert n[3] == -1 and kvh[3] == bh[3]
    valid = n >= 0
    assert np.array_equal(kvh[valid], bh[valid] + 1 + n[valid])
    assert st.read()["invalid"] == 1
    compare(oracle_ref(inp), t, n, inp=inp)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_packed_logits_give_the_padded_results(dev, dtype):
    """Logits packed by K (sequence b's rows from row sum_{c<b}(K_c + 1) of the
    target and sum_{c<b} K_c of the draft) verify exactly as the padded
    layout, and match the oracle."""
    B, V = 30, 7000
    K = W.configs.ragged_k(6, B)
    inp = W.make_host(B, K, V, dtype, 2.0, 0.7,
                      np.where(np.arange(B) % 4 == 0, 0.0, 0.9).astype(np.float32), seed=31)
    d = to_device(inp, dev)
    k = np.asarray(inp["K"])
    tp = torch.cat([d["target"][b, : k[b] + 1] for b in range(B)]).contiguous()
    dp = torch.cat([d["draft"][b, : k[b]] for b in range(B)]).contiguous()
    assert tp.shape[0] == int((k + 1).sum()) and dp.shape[0] == int(k.sum())
    ws = sv.Workspace(B, int(k.max()), V, dtype_code(dtype), dev)
    args = (d["tokens"], d["uniforms"], d["temperature"], k)
    t1, n1 = sv.spec_verify_ex(tp, dp, *args, ws, packed=True)
    t0, n0 = sv.spec_verify_ex(d["target"], d["draft"], *args, ws)
    torch.cuda.synchronize()
    assert torch.equal(t1, t0) and torch.equal(n1, n0)
    compare(oracle_ref(inp), t1.cpu().numpy(), n1.cpu().numpy(), inp=inp)


@pytest.mark.parametrize("V", [12345, 700])
def test_cuda_graph_replays_the_verification(dev, V):
    """A verification captured into a CUDA graph (after one ordinary call of
    its shape) replays on whatever the captured buffers hold: the oracle's
    results for the inputs at capture time and for new inputs copied into the
    same buffers, with ordinary calls of other shapes in between (which reuse
    the library's rotating header slots, not the graph's).  V = 700 takes
    the small-vocabulary kernel."""
    import torch
    B = 48
    K = W.configs.ragged_k(5, B)
    temps = np.where(np.arange(B) % 3 == 0, 0.0, 1.0).astype(np.float32)
    inp1 = W.make_host(B, K, V, "bf16", 2.0, 1.0, temps, seed=71)
    inp2 = W.make_host(B, K, V, "bf16", 2.0, 1.0, temps, seed=72)
    d = to_device(inp1, dev)
    Kmax = int(np.max(K))
    ws = sv.Workspace(B, Kmax, V, sv.SV_DTYPE_BF16)
    ot = torch.empty((B, Kmax + 1), dtype=torch.int32, device=dev)
    on = torch.empty((B,), dtype=torch.int32, device=dev)
    args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    sv.spec_verify_ws(*args, ws, out_tokens=ot, out_num_accepted=on)   # reserves the graph's header
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sv.spec_verify_ws(*args, ws, out_tokens=ot, out_num_accepted=on)
    ot.fill_(-7)
    on.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    compare(oracle_ref(inp1), ot.cpu().numpy(), on.cpu().numpy(), inp=inp1)
    # new inputs in the captured buffers; other calls churn the header slots
    d2 = to_device(inp2, dev)
    for key in ("target", "draft", "tokens", "uniforms", "temperature"):
        d[key].copy_(d2[key])
    other = W.make_host(16, 3, 9000, "bf16", 2.0, 1.0, 1.0, seed=73)
    for _ in range(20):
        run_gpu(to_device(other, dev), "ws")
    g.replay()
    torch.cuda.synchronize()
    compare(oracle_ref(inp2), ot.cpu().numpy(), on.cpu().numpy(), inp=inp2)


def test_host_entry_point_is_refused_under_capture(dev):
    """The host entry point synchronises: refused on a capturing stream, with
    the capture left intact."""
    import torch
    inp = W.make_host(4, 2, 3000, "bf16", 2.0, 1.0, 1.0, seed=74)
    staging = torch.empty(sv.sv_host_staging_size(4, 2, 3000, sv.SV_DTYPE_BF16), dtype=torch.uint8,
                          device=dev)
    ht = torch.from_numpy(inp["target"].view(np.int16)).view(torch.bfloat16)
    hd = torch.from_numpy(inp["draft"].view(np.int16)).view(torch.bfloat16)
    g = torch.cuda.CUDAGraph()
    x = torch.zeros(4, device=dev)
    with torch.cuda.graph(g):
        x += 1
        with pytest.raises(RuntimeError):
            sv.spec_verify_host(ht, hd, torch.from_numpy(inp["tokens"]), torch.from_numpy(inp["uniforms"]),
                                torch.from_numpy(inp["temperature"]), inp["K"], staging)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(x, torch.ones(4, device=dev))
