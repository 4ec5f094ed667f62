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


def compare(ref: dict, got_t: np.ndarray, got_n: np.ndarray, seqs=None) -> dict:
    """Bit-exact comparison outside oracle-flagged ties.  Returns counts."""
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
    return dict(n=len(tie), ties=int(tie.sum()), tie_mismatch=int((bad & tie).sum()))


def oracle_ref(inp: dict, seqs=None) -> dict:
    return oracle.verify_inputs(inp, seqs)
