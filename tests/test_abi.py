"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before queueing any work."""
import ctypes
import os
import re

import numpy as np
import pytest

import speculative_decoding_verification_04_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported():
    lib = sv.library()
    names = _declared_functions()
    assert {"spec_verify", "spec_verify_ws", "spec_verify_ex", "spec_verify_host",
            "sv_workspace_size", "sv_status_string"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings_and_version():
    for code, name in [(0, "SV_OK"), (1, "SV_ERR_INVALID_ARG"), (2, "SV_ERR_CUDA"),
                       (3, "SV_ERR_UNSUPPORTED"), (4, "SV_ERR_NO_MEMORY"), (5, "SV_ERR_TIMEOUT")]:
        assert sv.sv_status_string(code) == name
    assert sv.sv_status_string(99) == "SV_UNKNOWN_STATUS"
    assert sv.sv_abi_version() == 5


def test_limits_and_workspace_sizes():
    assert sv.sv_max_vocab(sv.SV_DTYPE_F32) >= 262144
    assert sv.sv_max_vocab(sv.SV_DTYPE_BF16) >= 2 * 262144
    assert sv.sv_max_vocab(7) == 0
    w1 = sv.sv_workspace_size(64, 5, 128256, sv.SV_DTYPE_BF16)
    w2 = sv.sv_workspace_size(128, 5, 128256, sv.SV_DTYPE_BF16)
    assert 0 < w1 < w2 and w1 % 256 == 0
    assert sv.sv_workspace_size(-1, 5, 100, 0) == 0
    assert sv.sv_workspace_size(4, 33, 100, 0) == 0
    assert sv.sv_workspace_size(4, 3, 0, 0) == 0
    assert sv.sv_workspace_size(4, 3, 100, 9) == 0
    assert sv.sv_host_staging_size(4, 3, 100, 0) > 4 * 4 * 100 * 4


def _call(B=2, K=(1, 2), V=10, dtype=0, tgt=1, drf=1, tok=1, uni=1, tmp=1, out_t=1, out_n=1):
    """spec_verify with fake (never dereferenced) pointers: host checks only."""
    lib = sv.library()
    k = None if K is None else np.asarray(K, np.int32)
    kp = None if k is None else k.ctypes.data_as(ctypes.c_void_p)
    P = lambda f: ctypes.c_void_p(0x1000) if f else None  # noqa: E731
    return lib.spec_verify(P(tgt), P(drf), dtype, P(tok), P(uni), P(tmp), B, kp, V, P(out_t),
                           P(out_n), None)


def test_host_argument_validation():
    assert _call(B=0, K=None) == sv.SV_OK            # empty batch is a no-op
    assert _call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert _call(V=0) == sv.SV_ERR_INVALID_ARG
    assert _call(dtype=5) == sv.SV_ERR_INVALID_ARG
    assert _call(K=(1, 33)) == sv.SV_ERR_INVALID_ARG
    assert _call(K=(-1, 2)) == sv.SV_ERR_INVALID_ARG
    assert _call(K=None) == sv.SV_ERR_INVALID_ARG
    assert _call(tgt=0) == sv.SV_ERR_INVALID_ARG
    assert _call(uni=0) == sv.SV_ERR_INVALID_ARG
    assert _call(tmp=0) == sv.SV_ERR_INVALID_ARG
    assert _call(out_t=0) == sv.SV_ERR_INVALID_ARG
    assert _call(out_n=0) == sv.SV_ERR_INVALID_ARG
    assert _call(tok=0) == sv.SV_ERR_INVALID_ARG      # tokens required when Kmax > 0
    assert _call(V=sv.sv_max_vocab(0) + 1) == sv.SV_ERR_UNSUPPORTED


def test_workspace_and_host_entry_validation():
    lib = sv.library()
    k = np.array([1, 2], np.int32)
    kp = k.ctypes.data_as(ctypes.c_void_p)
    f = ctypes.c_void_p(0x1000)
    # a workspace that is too small (or missing) is refused before any CUDA call
    st = lib.spec_verify_ws(f, f, 0, f, f, f, 2, kp, 10, f, f, None, 0, None)
    assert st == sv.SV_ERR_NO_MEMORY
    st = lib.spec_verify_host(f, f, 0, f, f, f, -3, kp, 10, f, f, f, 1 << 20, None)
    assert st == sv.SV_ERR_INVALID_ARG
    st = lib.spec_verify_host(f, f, 0, f, f, f, 2, kp, 10, f, f, None, 0, None)
    assert st == sv.SV_ERR_NO_MEMORY
    flags = ctypes.c_uint32(0)
    assert lib.sv_workspace_errors(None, ctypes.byref(flags), None) == sv.SV_ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    t = torch.zeros((1, 2, 4))
    with pytest.raises(ValueError):
        sv.spec_verify(t, t[:, :1], torch.zeros((1, 1), dtype=torch.int32),
                       torch.zeros((1, 2)), torch.ones(1), [1])


def test_sample_entry_validation():
    """spec_sample rejects bad arguments on the host (fake, never dereferenced
    pointers), and its workspace size follows from B, V and dtype."""
    lib = sv.library()
    P = lambda f: ctypes.c_void_p(0x1000) if f else None  # noqa: E731

    def call(B=4, V=10, dtype=0, lg=1, uni=1, tmp=1, out=1, ws=1, nbytes=1 << 20):
        w = ctypes.c_void_p(0x100000) if ws else None
        return lib.spec_sample(P(lg), dtype, P(uni), P(tmp), B, V, P(out), w, nbytes, None)

    assert call(B=0) == sv.SV_OK
    assert call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert call(V=0) == sv.SV_ERR_INVALID_ARG
    assert call(dtype=3) == sv.SV_ERR_INVALID_ARG
    assert call(lg=0) == sv.SV_ERR_INVALID_ARG
    assert call(uni=0) == sv.SV_ERR_INVALID_ARG
    assert call(tmp=0) == sv.SV_ERR_INVALID_ARG
    assert call(out=0) == sv.SV_ERR_INVALID_ARG
    assert call(ws=0) == sv.SV_ERR_NO_MEMORY
    assert call(nbytes=16) == sv.SV_ERR_NO_MEMORY
    n = sv.sv_sample_workspace_size(64, 128256, sv.SV_DTYPE_BF16)
    assert n > sv.sv_workspace_size(64, 0, 128256, sv.SV_DTYPE_BF16) and n % 256 == 0
    assert sv.sv_sample_workspace_size(-1, 10, 0) == 0
    assert sv.sv_sample_workspace_size(4, 0, 0) == 0


def test_option_pointer_alignment_is_checked():
    """sv_stats holds 64-bit counters and kv_len 32-bit lengths: misaligned
    option pointers are refused before any work, as are flag options outside
    {0, 1}."""
    lib = sv.library()
    P = lambda: ctypes.c_void_p(0x1000)  # noqa: E731
    k = np.asarray([1, 2], np.int32)
    for field, addr in (("stats", 0x1004), ("kv_len", 0x1002)):
        opt = sv.SVOptions()
        setattr(opt, field, addr)
        st = lib.spec_verify_ex(P(), P(), 0, P(), P(), P(), 2, k.ctypes.data_as(ctypes.c_void_p), 10,
                                P(), P(), ctypes.byref(opt), ctypes.c_void_p(0x100000), 1 << 20, None)
        assert st == sv.SV_ERR_INVALID_ARG, field
    for field, value in (("packed_logits", 2), ("expire_copy_waits", -1), ("expire_copy_waits", 2)):
        opt = sv.SVOptions()
        setattr(opt, field, value)
        st = lib.spec_verify_ex(P(), P(), 0, P(), P(), P(), 2, k.ctypes.data_as(ctypes.c_void_p), 10,
                                P(), P(), ctypes.byref(opt), ctypes.c_void_p(0x100000), 1 << 20, None)
        assert st == sv.SV_ERR_INVALID_ARG, (field, value)


def test_tree_entry_validation():
    """spec_verify_tree rejects bad arguments on the host (fake, never
    dereferenced pointers) before any device work."""
    lib = sv.library()
    P = lambda f: ctypes.c_void_p(0x1000) if f else None  # noqa: E731
    assert sv.library().sv_tree_workspace_size() >= 16

    def call(B=4, Nmax=7, V=10, dtype=0, tgt=1, tok=1, par=1, uni=1, tmp=1, nn=1, out=1, ws=1, nbytes=256):
        w = ctypes.c_void_p(0x100000) if ws else None
        return lib.spec_verify_tree(P(tgt), P(1), dtype, P(tok), P(par), P(uni), P(tmp), B, Nmax, P(nn), V,
                                    P(out), P(out), P(out), w, nbytes, None)

    assert call(B=0) == sv.SV_OK
    assert call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert call(V=0) == sv.SV_ERR_INVALID_ARG
    assert call(Nmax=0) == sv.SV_ERR_INVALID_ARG
    assert call(Nmax=33) == sv.SV_ERR_INVALID_ARG
    assert call(dtype=5) == sv.SV_ERR_INVALID_ARG
    for k in ("tgt", "tok", "par", "uni", "tmp", "nn", "out"):
        assert call(**{k: 0}) == sv.SV_ERR_INVALID_ARG, k
    assert call(ws=0) == sv.SV_ERR_NO_MEMORY
    assert call(nbytes=8) == sv.SV_ERR_NO_MEMORY
    assert call(V=sv.sv_max_vocab(0) + 1) == sv.SV_ERR_UNSUPPORTED


def test_binding_structs_match_the_header(tmp_path):
    """The ctypes structs of the binding have the C header's layout: a small C
    program built with gcc against include/specverify.h prints each field's
    offset and each struct's size, and the binding's must agree (a field added
    on one side only would shift every field after it)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("needs gcc and the CUDA headers")
    fields = {
        "sv_diag": ["p_x", "q_x", "resid_mass", "final_row"],
        "sv_options": [n for n, _ in sv.SVOptions._fields_],
        "sv_stats": list(sv.STATS_FIELDS),
    }
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "specverify.h"', "int main(void) {"]
    for st, names in fields.items():
        lines.append(f'  printf("{st} size %zu\\n", sizeof({st}));')
        for n in names:
            lines.append(f'  printf("{st} {n} %zu\\n", offsetof({st}, {n}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    c = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    assert c[("sv_diag", "size")] == ctypes.sizeof(sv.SVDiag)
    for n in fields["sv_diag"]:
        assert c[("sv_diag", n)] == getattr(sv.SVDiag, n).offset
    assert c[("sv_options", "size")] == ctypes.sizeof(sv.SVOptions)
    for n in fields["sv_options"]:
        assert c[("sv_options", n)] == getattr(sv.SVOptions, n).offset, n
    # the counters are read back as consecutive unsigned 64-bit words
    assert c[("sv_stats", "size")] == 8 * len(sv.STATS_FIELDS)
    for k, n in enumerate(sv.STATS_FIELDS):
        assert c[("sv_stats", n)] == 8 * k, n
