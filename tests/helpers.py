"""Shared helpers for the GPU parity tests: move seeded workloads to the
device, call the library through its C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import speculative_decoding_verification_04_gb300 as sv


def to_device(inp: dict, dev="cuda") -> dict:
    import torch
    out = dict(inp)
    for k in ("target", "draft"):
        a = inp[k]
        if inp["dtype"] == "bf16":
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        out[k] = t.to(dev)
    out["tokens"] = torch.from_numpy(np.ascontiguousarray(inp["tokens"], np.int32)).to(dev)
    out["uniforms"] = torch.from_numpy(np.ascontiguousarray(inp["uniforms"], np.float32)).to(dev)
    out["temperature"] = torch.from_numpy(
        np.ascontiguousarray(inp["temperature"], np.float32)).to(dev)
    return out


def rows_to_host(dinp: dict, seqs) -> dict:
    """Copy the rows of the chosen sequences of a device workload to numpy."""
    import torch
    idx = torch.as_tensor(np.asarray(seqs), device=dinp["target"].device, dtype=torch.long)

    def host(t):
        t = t.index_select(0, idx).cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    seqs = np.asarray(seqs)
    return dict(target=host(dinp["target"]), draft=host(dinp["draft"]), dtype=dinp["dtype"],
                tokens=host(dinp["tokens"]), uniforms=host(dinp["uniforms"]),
                temperature=host(dinp["temperature"]), K=np.asarray(dinp["K"])[seqs],
                B=len(seqs), Kmax=dinp["Kmax"], V=dinp["V"])


def dtype_code(dtype: str) -> int:
    return sv.SV_DTYPE_BF16 if dtype == "bf16" else sv.SV_DTYPE_F32


def run_gpu(d: dict, mode: str = "ws", **kw):
    """Verify a device workload; returns numpy (out_tokens, num_accepted)."""
    import torch
    K = np.asarray(d["K"], np.int32)
    args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    if mode == "alloc":
        t, n = sv.spec_verify(*args)
    else:
        ws = kw.pop("workspace", None) or sv.Workspace(len(K), int(K.max()) if len(K) else 0,
                                                       d["V"], dtype_code(d["dtype"]),
                                                       d["target"].device)
        if mode == "ws":
            t, n = sv.spec_verify_ws(*args, ws)
        else:
            t, n = sv.spec_verify_ex(*args, ws, **kw)
    torch.cuda.synchronize()
    return t.cpu().numpy(), n.cpu().numpy()


def tie_bound(n: int, V: int = 1, n_draws: int = 0, n_tests: int = 0) -> int:
    """Most oracle-flagged ties a random batch may hold (5 sigma above an upper
    bound of their expected number).  An accept test is flagged when its
    uniform lies within 1e-6 of p/q: probability 2e-6.  A draw is flagged when
    its uniform lies within 1e-6 of either end of the drawn token's interval:
    probability sum_j min(r_j, 2e-6) <= min(1, 2e-6 V), which is not small
    for large vocabularies (the intervals are about 1/V wide).  n sequences
    taking n_draws sampling draws and n_tests sampling accept tests in all; a
    flag set too often (a wider band, a flag that ignores the distance) fails
    this, bad luck does not."""
    mean = n_draws * min(1.0, 2e-6 * V) + n_tests * 2e-6
    return int(mean + 5.0 * np.sqrt(mean) + 2)


def tie_bound_for(inp: dict) -> int:
    """tie_bound for a workload dict: its sampling sequences each take one draw
    and at most K_b accept tests."""
    K = np.asarray(inp["K"])
    samp = np.asarray(inp["temperature"]) > 0
    return tie_bound(len(K), int(inp["V"]) if "V" in inp else int(np.shape(inp["target"])[-1]),
                     int(samp.sum()), int(K[samp].sum()))


def _flipped_matches(inp: dict, b: int, got_t: np.ndarray, got_n: int) -> tuple[bool, str]:
    """Whether the GPU's result for sequence b of `inp` is the oracle's with
    one decision flipped.  Either the walk is the oracle's and only the drawn
    token differs: its interval in the oracle's fp64 CDF of the distribution
    drawn from must lie within 1e-6 of the final uniform (a flagged draw has
    the uniform within 1e-6 of a boundary, and at large V several tokens of
    mass below 1e-6 may sit inside that band).  Or an accept test flipped:
    one uniform slot of the walk (0..K_b) moved 1.1e-6 to 3e-6 either way
    makes the oracle reproduce the GPU's outputs."""
    one = {k: (inp[k][b:b + 1] if k in ("target", "draft", "tokens", "uniforms", "temperature", "K")
               else inp[k]) for k in inp}
    one["uniforms"] = np.array(one["uniforms"], np.float32, copy=True)
    ref = oracle.verify_inputs(one)
    n_ref, Kb, T = int(ref["num_accepted"][0]), int(one["K"][0]), float(one["temperature"][0])
    why = f"oracle n={n_ref} tokens={ref['out_tokens'][0].tolist()} gpu n={got_n} tokens={got_t.tolist()}"
    if got_n == n_ref >= 0 and T > 0 and np.array_equal(got_t[:got_n], ref["out_tokens"][0, :got_n]) \
            and np.all(got_t[got_n + 1:] == -1):
        drow = one["draft"][0, got_n] if got_n < Kb else None
        r, code = oracle.final_distribution(one["target"][0, got_n], drow, one["dtype"], T)
        t = int(got_t[got_n])
        if code and 0 <= t < len(r) and r[t] > 0:
            C = np.cumsum(r)
            lo, hi = (C[t - 1] if t > 0 else 0.0), C[t]
            u = float(one["uniforms"][0, Kb])
            dist = max(lo - u, u - hi, 0.0)
            if dist < 1.05e-6:
                return True, ""
            why += f"; drawn token's interval [{lo:.9f}, {hi:.9f}) lies {dist:.3g} from u={u:.9f}"
    for j in range(Kb + 1):
        for delta in (1.1e-6, -1.1e-6, 1.5e-6, -1.5e-6, 2e-6, -2e-6, 3e-6, -3e-6):
            u = one["uniforms"].copy()
            u[0, j] = np.float32(min(max(float(u[0, j]) + delta, 0.0), 1.0 - 2.0 ** -24))
            alt = oracle.verify_inputs(dict(one, uniforms=u))
            if alt["num_accepted"][0] == got_n and np.array_equal(alt["out_tokens"][0], got_t):
                return True, ""
    return False, why


def compare(ref: dict, got_t: np.ndarray, got_n: np.ndarray, seqs=None, inp=None,
            max_ties=None) -> dict:
    """Bit-exact comparison outside oracle-flagged ties.  Returns counts.

    `ref` is the oracle's result on the sequences `seqs` (all when None) of
    the GPU outputs.  The number of flagged sequences must stay within
    `max_ties` (by default tie_bound_for(inp); with no `inp`, tie_bound(n),
    the bound of a batch that takes no draws).  With `inp`, the workload `ref` was computed
    from, every flagged sequence on which the GPU differs must be the
    oracle's result with that one decision flipped."""
    if seqs is not None:
        got_t, got_n = got_t[seqs], got_n[seqs]
    tie = ref["tie"]
    bad_n = got_n != ref["num_accepted"]
    bad_t = np.any(got_t != ref["out_tokens"], axis=1)
    bad = bad_n | bad_t
    hard = bad & ~tie
    if np.any(hard):
        i = int(np.flatnonzero(hard)[0])
        raise AssertionError(
            f"{int(hard.sum())} sequence(s) differ from the oracle outside ties; first b={i}: "
            f"gpu n={got_n[i]} tokens={got_t[i].tolist()} oracle n={ref['num_accepted'][i]} "
            f"tokens={ref['out_tokens'][i].tolist()}")
    n, ties, tm = len(tie), int(tie.sum()), int((bad & tie).sum())
    print(f"parity: sequences={n} ties={ties} tie_mismatch={tm}")
    if max_ties is not None:
        limit = max_ties
    elif inp is not None:
        limit = tie_bound_for(inp)
    else:
        limit = tie_bound(n)
    assert ties <= limit, f"{ties} oracle-flagged ties in {n} sequences (bound {limit})"
    if inp is not None:
        for i in np.flatnonzero(bad & tie):
            ok, why = _flipped_matches(inp, int(i), got_t[i], int(got_n[i]))
            assert ok, f"sequence {int(i)}: the GPU result is not the oracle's with one decision flipped: {why}"
    return dict(n=n, ties=ties, tie_mismatch=tm)


def oracle_ref(inp: dict, seqs=None) -> dict:
    return oracle.verify_inputs(inp, seqs)


def oracle_ref_threaded(inp: dict, threads: int | None = None) -> dict:
    """The oracle over every sequence of `inp`, the batch cut into contiguous
    shards run at once on host threads (the oracle's C loop runs outside
    Python's lock); the same results as oracle_ref, shard by shard."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    B = len(inp["K"])
    if threads is None:
        try:
            threads = len(os.sched_getaffinity(0))
        except AttributeError:
            threads = os.cpu_count() or 1
    cuts = np.linspace(0, B, max(1, min(threads, B)) + 1).astype(int)
    keys = ("target", "draft", "tokens", "uniforms", "temperature", "K")
    shards = [dict({k: inp[k][a:b] for k in keys}, dtype=inp["dtype"])
              for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    with ThreadPoolExecutor(max_workers=len(shards)) as ex:
        parts = list(ex.map(oracle.verify_inputs, shards))
    return dict(out_tokens=np.concatenate([p["out_tokens"] for p in parts]),
                num_accepted=np.concatenate([p["num_accepted"] for p in parts]),
                tie=np.concatenate([p["tie"] for p in parts]),
                final_row=np.concatenate([p["final_row"] for p in parts]),
                fallbacks=sum(p["fallbacks"] for p in parts))
