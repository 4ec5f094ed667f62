"""spec_verify_noalloc: the same verification as spec_verify_ws, computed in
the library's fixed device scratch array instead of a workspace.  This file
is collected last so that it also runs after every other test in one
process; it passes on its own as well."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import workloads as W
import speculative_decoding_verification_04_gb300 as sv
from helpers import compare, oracle_ref, to_device


def test_shape_beyond_static_scratch_is_rejected():
    """A shape needing more than SV_STATIC_SCRATCH_BYTES of scratch returns
    SV_ERR_NO_MEMORY before any CUDA call (so this runs without a GPU)."""
    B, V = 4 << 20, 128256
    K = np.full(B, 2, np.int32)
    need = sv.sv_workspace_size(B, 2, V, sv.SV_DTYPE_BF16)
    assert need > sv.SV_STATIC_SCRATCH_BYTES
    dummy = ctypes.c_void_p(256)
    st = sv.library().spec_verify_noalloc(dummy, dummy, sv.SV_DTYPE_BF16, dummy, dummy, dummy, B,
                                          K.ctypes.data_as(ctypes.c_void_p), V, dummy, dummy, None)
    assert st == sv.SV_ERR_NO_MEMORY


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["mixed_bf16", "f32_large_vocab"])
def test_noalloc_matches_workspace_entry_point(case):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if case == "mixed_bf16":
        B = 40
        inp = W.make_host(B, W.configs.ragged_k(3, B), 12345, "bf16", 2.0, 1.0,
                          np.where(np.arange(B) % 3 == 0, 0.0, 0.9).astype(np.float32), seed=12)
        code = sv.SV_DTYPE_BF16
    else:
        B = 8
        inp = W.make_host(B, 8, 151936, "f32", 2.0, 1.5, 0.7, seed=77)
        code = sv.SV_DTYPE_F32
    assert sv.sv_workspace_size(B, inp["Kmax"], inp["V"], code) <= sv.SV_STATIC_SCRATCH_BYTES
    d = to_device(inp, dev)
    K = np.asarray(inp["K"], np.int32)
    args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    ws = sv.Workspace(B, inp["Kmax"], inp["V"], code, dev)
    ref_t, ref_n = sv.spec_verify_ws(*args, ws)
    ref_t, ref_n = ref_t.cpu().numpy(), ref_n.cpu().numpy()
    compare(oracle_ref(inp), ref_t, ref_n, inp=inp)
    out_t = torch.full((B, inp["Kmax"] + 1), -9, dtype=torch.int32, device=dev)
    out_n = torch.full((B,), -9, dtype=torch.int32, device=dev)
    for _ in range(2):   # two calls in a row: the second reuses the scratch the first left
        t, n = sv.spec_verify_noalloc(*args, out_t, out_n)
        torch.cuda.synchronize()
        assert t.data_ptr() == out_t.data_ptr() and n.data_ptr() == out_n.data_ptr()
        assert np.array_equal(t.cpu().numpy(), ref_t) and np.array_equal(n.cpu().numpy(), ref_n)
        out_t.fill_(-9)
        out_n.fill_(-9)
