"""fp64 CPU oracle for batched draft-token verification (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The GPU library shares no code with
it and never calls it.

The arithmetic lives in ``oracle.c`` (plain C, fp64); this module compiles it
with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

DTYPES = {"f32": 0, "bf16": 1}


def build_command() -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (idempotent)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.run(build_command(), check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.oracle_verify.argtypes = [P, P, ctypes.c_int, P, P, P, i32, P, i32, i32, P, P, P, P]
        lib.oracle_verify.restype = ctypes.c_int
        lib.oracle_position_probs.argtypes = [P, P, ctypes.c_int, P, P, i32, P, i32, i32, P, P, P]
        lib.oracle_position_probs.restype = ctypes.c_int
        lib.oracle_final_distribution.argtypes = [P, P, ctypes.c_int, i32, ctypes.c_float, P]
        lib.oracle_final_distribution.restype = ctypes.c_int
        lib.oracle_tree_verify.argtypes = [P, P, ctypes.c_int, P, P, P, P, i32, P, i32, i32, P, P, P, P]
        lib.oracle_tree_verify.restype = ctypes.c_int
        lib.oracle_abi_version.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a, dtype):
    if a is None:
        return None
    want = np.uint16 if dtype == "bf16" else np.float32
    return np.ascontiguousarray(a, dtype=want)


def verify(target, draft, dtype, tokens, uniforms, temperature, K, V=None):
    """Run the oracle over a batch.

    Returns a dict with out_tokens [B, Kmax+1], num_accepted [B], tie [B]
    (bool: a decision lies within 1e-6 of its threshold), final_row [B] and
    fallbacks (count of zero-residual fallbacks).
    """
    lib = _load()
    tgt = _logits(target, dtype)
    drf = _logits(draft, dtype)
    K = np.ascontiguousarray(K, dtype=np.int32)
    B = int(K.shape[0])
    Kmax = int(tgt.shape[1]) - 1
    V = int(tgt.shape[2]) if V is None else int(V)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, Kmax) if Kmax else \
        np.zeros((B, 0), np.int32)
    uni = np.ascontiguousarray(uniforms, dtype=np.float32)
    tmp = np.ascontiguousarray(temperature, dtype=np.float32)
    out_tok = np.empty((B, Kmax + 1), np.int32)
    out_n = np.empty(B, np.int32)
    tie = np.empty(B, np.uint8)
    frow = np.empty(B, np.int32)
    rc = lib.oracle_verify(_ptr(tgt), _ptr(drf), DTYPES[dtype], _ptr(tok), _ptr(uni), _ptr(tmp),
                           B, _ptr(K), Kmax, V, _ptr(out_tok), _ptr(out_n), _ptr(tie), _ptr(frow))
    if rc < 0:
        raise ValueError("oracle_verify rejected its arguments")
    return dict(out_tokens=out_tok, num_accepted=out_n, tie=tie.astype(bool),
                final_row=frow, fallbacks=rc)


def position_probs(target, draft, dtype, tokens, temperature, K):
    """p_i(x_i), q_i(x_i) and residual mass at every draft position, [B, Kmax]."""
    lib = _load()
    tgt = _logits(target, dtype)
    drf = _logits(draft, dtype)
    K = np.ascontiguousarray(K, dtype=np.int32)
    B = int(K.shape[0])
    Kmax = int(tgt.shape[1]) - 1
    V = int(tgt.shape[2])
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    tmp = np.ascontiguousarray(temperature, dtype=np.float32)
    px = np.empty((B, Kmax), np.float64)
    qx = np.empty((B, Kmax), np.float64)
    rm = np.empty((B, Kmax), np.float64)
    rc = lib.oracle_position_probs(_ptr(tgt), _ptr(drf), DTYPES[dtype], _ptr(tok), _ptr(tmp),
                                   B, _ptr(K), Kmax, V, _ptr(px), _ptr(qx), _ptr(rm))
    if rc < 0:
        raise ValueError("oracle_position_probs rejected its arguments")
    return px, qx, rm


def final_distribution(target_row, draft_row, dtype, T):
    """Normalised distribution of the final draw for one row; (r, code)."""
    lib = _load()
    t = _logits(np.asarray(target_row).reshape(-1), dtype)
    d = None if draft_row is None else _logits(np.asarray(draft_row).reshape(-1), dtype)
    r = np.empty(t.shape[0], np.float64)
    code = lib.oracle_final_distribution(_ptr(t), _ptr(d), DTYPES[dtype], t.shape[0],
                                         float(T), _ptr(r))
    return r, code


def verify_inputs(inp: dict, seqs=None):
    """Convenience: run ``verify`` on a workload dict (numpy arrays).  ``seqs``
    optionally restricts to a subset of sequence indices."""
    if seqs is None:
        return verify(inp["target"], inp["draft"], inp["dtype"], inp["tokens"],
                      inp["uniforms"], inp["temperature"], inp["K"])
    seqs = np.asarray(seqs)
    return verify(inp["target"][seqs], inp["draft"][seqs], inp["dtype"], inp["tokens"][seqs],
                  inp["uniforms"][seqs], inp["temperature"][seqs], inp["K"][seqs])


def tree_verify(target, draft, dtype, tokens, parent, uniforms, temperature, n_nodes):
    """Token-tree verification (``oracle_tree_verify`` in oracle.c).

    target / draft logits [B, Nmax, V] (row n: the distribution after node n),
    tokens / parent / uniforms [B, Nmax] (uniforms[:, 0] is the final draw),
    temperature [B], n_nodes [B].  Returns out_tokens, out_path [B, Nmax],
    out_len [B] and tie [B] (bool).
    """
    lib = _load()
    tgt = _logits(target, dtype)
    drf = _logits(draft, dtype)
    B, Nmax, V = (int(x) for x in tgt.shape)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    par = np.ascontiguousarray(parent, dtype=np.int32)
    uni = np.ascontiguousarray(uniforms, dtype=np.float32)
    tmp = np.ascontiguousarray(temperature, dtype=np.float32)
    nn = np.ascontiguousarray(n_nodes, dtype=np.int32)
    out_tok = np.empty((B, Nmax), np.int32)
    out_path = np.empty((B, Nmax), np.int32)
    out_len = np.empty(B, np.int32)
    tie = np.empty(B, np.uint8)
    rc = lib.oracle_tree_verify(_ptr(tgt), _ptr(drf), DTYPES[dtype], _ptr(tok), _ptr(par), _ptr(uni),
                                _ptr(tmp), B, _ptr(nn), Nmax, V, _ptr(out_tok), _ptr(out_path),
                                _ptr(out_len), _ptr(tie))
    if rc < 0:
        raise ValueError("oracle_tree_verify rejected its arguments")
    return dict(out_tokens=out_tok, out_path=out_path, out_len=out_len, tie=tie.astype(bool))


def library_path() -> str:
    return _LIB

