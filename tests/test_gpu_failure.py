"""Failure detection on the GPU without a fault: a bounded device wait that
gives up must be reported, poison only the affected sequences' outputs, and
leave the context and the workspace usable.

The wait is made to run out by the library's test-only option
expire_copy_waits (every wait for a row's copy into shared memory gives up
before its first poll).  The copies themselves are legitimate and still land;
the kernel waits for them, with the normal bound, before it exits.  Nothing
here traps, faults or hangs the GPU."""
import ctypes

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


@pytest.mark.parametrize("dtype,V", [("bf16", 12345), ("f32", 151936)])
def test_expired_copy_waits_are_reported_and_recovered_from(dev, dtype, V):
    B = 24
    temps = np.where(np.arange(B) % 3 == 0, 0.0, 1.0).astype(np.float32)
    inp = W.make_host(B, W.configs.ragged_k(9, B), V, dtype, 2.0, 1.0, temps, seed=V % 101)
    d = to_device(inp, dev)
    ws = sv.Workspace(B, int(inp["Kmax"]), V, dtype_code(dtype), dev)
    t, n = run_gpu(d, "ex", workspace=ws, expire_copy_waits=True)
    # the call returned and the device still answers; every cluster's first
    # wait gave up, so every sequence's outputs are poisoned
    assert np.all(n == -1) and np.all(t == -1)
    flags = ctypes.c_uint32(0)
    stream = torch.cuda.current_stream()
    st = sv.library().sv_workspace_errors(ws.ptr, ctypes.byref(flags), ctypes.c_void_p(stream.cuda_stream))
    assert st == sv.SV_ERR_TIMEOUT and flags.value & 1
    # the error word was cleared by the read; an ordinary call on the same
    # workspace gives the oracle's results and records no error
    t2, n2 = run_gpu(d, "ws", workspace=ws)
    compare(oracle_ref(inp), t2, n2, inp=inp)
    assert sv.sv_workspace_errors(ws) == 0
    # a stats-counting call with expired waits counts every sequence invalid
    stats = sv.Stats(dev)
    run_gpu(d, "ex", workspace=ws, expire_copy_waits=True, stats=stats)
    got = stats.read()
    assert got["invalid"] == B and got["sequences"] == 0 and got["tested"] == 0
    assert sv.sv_workspace_errors(ws) == 1
