"""Seeded random configurations against the oracle: batch size, ragged K
(including K = 0), vocabulary sizes on both sides of the small-vocabulary
limit and around chunk boundaries, dtype, temperature mix and noise level
are drawn per case; every output is compared with the oracle, and the
packed layout and the verify-all mode must give the padded call's outputs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_04_gb300 as sv  # noqa: E402
import workloads as W  # noqa: E402
from helpers import compare, dtype_code, oracle_ref, run_gpu, to_device  # noqa: E402

pytestmark = pytest.mark.gpu

# the small-vocabulary limit (1024), one chunk of fp32 (512) and of bf16
# (1024), and sizes a few elements past them
VOCABS = [2, 31, 511, 512, 513, 1023, 1024, 1025, 1031, 2047, 2049, 4100, 9999]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _case(seed: int) -> dict:
    rng = np.random.default_rng(9000 + seed)
    B = int(rng.integers(1, 90))
    V = int(rng.choice(VOCABS))
    dtype = "bf16" if rng.random() < 0.5 else "f32"
    Kmax = int(rng.integers(1, 13))
    K = rng.integers(0, Kmax + 1, size=B).astype(np.int32)
    K[0] = Kmax   # the padded layout has Kmax + 1 target rows
    temps = rng.choice(np.array([0.0, 0.5, 1.0, 1.7], np.float32), size=B)
    sigma_t = float(rng.choice([0.5, 2.0, 4.0]))
    sigma_d = float(rng.choice([0.05, 0.5, 1.5]))
    return W.make_host(B, K, V, dtype, sigma_t, sigma_d, temps, seed=9000 + seed)


@pytest.mark.parametrize("seed", range(16))
def test_random_configuration_matches_oracle(dev, seed):
    inp = _case(seed)
    B, V, k = inp["B"], inp["V"], np.asarray(inp["K"])
    d = to_device(inp, dev)
    ws = sv.Workspace(B, int(inp["Kmax"]), V, dtype_code(inp["dtype"]), dev)
    t0, n0 = run_gpu(d, "ws", workspace=ws)
    c = compare(oracle_ref(inp), t0, n0, inp=inp)
    assert c["n"] == B
    assert sv.sv_workspace_errors(ws) == 0
    # verify-all reads every row and must not change any output
    t1, n1 = run_gpu(d, "ex", workspace=ws, verify_all=True)
    assert np.array_equal(t0, t1) and np.array_equal(n0, n1)
    # the same batch packed by K
    tp = torch.cat([d["target"][b, : k[b] + 1] for b in range(B)]).contiguous()
    dp = torch.cat([d["draft"][b, : k[b]] for b in range(B)]).contiguous()
    t2, n2 = sv.spec_verify_ex(tp, dp, d["tokens"], d["uniforms"], d["temperature"], k, ws, packed=True)
    torch.cuda.synchronize()
    assert np.array_equal(t2.cpu().numpy(), t0) and np.array_equal(n2.cpu().numpy(), n0)
