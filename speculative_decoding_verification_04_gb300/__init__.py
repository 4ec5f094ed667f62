"""Python binding of libspecverify (argument marshalling only).

Every step of the verification path runs in the CUDA library; this module
turns torch tensors and host sequences into the pointers and sizes that the
C ABI in ``include/specverify.h`` takes, and raises on a non-OK status.  If
the shared library has not been built the import of any entry point raises:
there is no CPU fallback.

Entry points (same names as the C ABI):
  spec_verify, spec_verify_ws, spec_verify_ex, spec_verify_host, spec_sample,
  sv_workspace_size, sv_sample_workspace_size, sv_host_staging_size,
  sv_max_vocab, sv_status_string, sv_abi_version, sv_workspace_errors
plus ``Workspace`` (a device buffer of sv_workspace_size bytes), ``Stats``
(a device sv_stats) and ``SVOptions`` / ``SVDiag`` (the ctypes mirrors of
sv_options / sv_diag).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SV_OK = 0
SV_ERR_INVALID_ARG = 1
SV_ERR_CUDA = 2
SV_ERR_UNSUPPORTED = 3
SV_ERR_NO_MEMORY = 4
SV_ERR_TIMEOUT = 5
SV_DTYPE_F32 = 0
SV_DTYPE_BF16 = 1
SV_K_MAX = 32

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {sv_status_string(status)} ({status})")


class SVDiag(ctypes.Structure):
    _fields_ = [("p_x", ctypes.c_void_p), ("q_x", ctypes.c_void_p),
                ("resid_mass", ctypes.c_void_p), ("final_row", ctypes.c_void_p)]


class SVOptions(ctypes.Structure):
    _fields_ = [("diag", SVDiag), ("verify_all", ctypes.c_int32),
                ("chunks_per_cta", ctypes.c_int32), ("chunks_per_warp", ctypes.c_int32),
                ("stats", ctypes.c_void_p), ("kv_len", ctypes.c_void_p),
                ("packed_logits", ctypes.c_int32), ("expire_copy_waits", ctypes.c_int32),
                ("temperature_host", ctypes.c_void_p)]


STATS_FIELDS = ("sequences", "invalid", "tested", "accepted", "committed", "near_ties", "draw_near_ties")


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libspecverify is not built ({LIB_PATH} missing); "
                           "run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    common = [P, P, ctypes.c_int, P, P, P, i32, P, i32, P, P]
    lib.spec_verify.argtypes = common + [P]
    lib.spec_verify_noalloc.argtypes = common + [P]
    lib.spec_verify_noalloc.restype = ctypes.c_int
    lib.spec_verify_ws.argtypes = common + [P, sz, P]
    lib.spec_verify_ex.argtypes = common + [ctypes.POINTER(SVOptions), P, sz, P]
    lib.spec_verify_host.argtypes = common + [P, sz, P]
    lib.spec_sample.argtypes = [P, ctypes.c_int, P, P, i32, i32, P, P, sz, P]
    lib.spec_sample.restype = ctypes.c_int
    lib.spec_verify_tree.argtypes = [P, P, ctypes.c_int, P, P, P, P, i32, i32, P, i32, P, P, P, P, sz, P]
    lib.spec_verify_tree.restype = ctypes.c_int
    lib.sv_tree_workspace_size.argtypes = []
    lib.sv_tree_workspace_size.restype = sz
    lib.sv_sample_workspace_size.argtypes = [i32, i32, ctypes.c_int]
    lib.sv_sample_workspace_size.restype = sz
    for f in (lib.spec_verify, lib.spec_verify_ws, lib.spec_verify_ex, lib.spec_verify_host):
        f.restype = ctypes.c_int
    lib.sv_workspace_size.argtypes = [i32, i32, i32, ctypes.c_int]
    lib.sv_workspace_size.restype = sz
    lib.sv_host_staging_size.argtypes = [i32, i32, i32, ctypes.c_int]
    lib.sv_host_staging_size.restype = sz
    lib.sv_max_vocab.argtypes = [ctypes.c_int]
    lib.sv_max_vocab.restype = i32
    lib.sv_status_string.argtypes = [ctypes.c_int]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_abi_version.restype = i32
    lib.sv_workspace_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.sv_workspace_errors.restype = ctypes.c_int
    lib.sv_geometry.argtypes = [i32, i32, i32, ctypes.c_int, i32, i32, P]
    lib.sv_geometry.restype = ctypes.c_int
    _lib = lib
    return lib


def library():
    """The loaded ctypes CDLL (raises if the library is not built)."""
    return _load()


def sv_status_string(status: int) -> str:
    return _load().sv_status_string(int(status)).decode()


def sv_abi_version() -> int:
    return int(_load().sv_abi_version())


def sv_max_vocab(dtype: int) -> int:
    return int(_load().sv_max_vocab(int(dtype)))


GEOMETRY_FIELDS = ("cluster_ctas", "warps", "chunks_per_warp", "clusters", "threads",
                   "smem_bytes", "warp_ranges", "chunks")


def sv_geometry(B: int, Kmax: int, V: int, dtype: int, chunks_per_cta: int = 0,
                chunks_per_warp: int = 0) -> dict:
    """Launch geometry a call of this shape would use on the current device."""
    out = (ctypes.c_int32 * 8)()
    st = _load().sv_geometry(int(B), int(Kmax), int(V), int(dtype), int(chunks_per_cta),
                             int(chunks_per_warp), out)
    _check(st, "sv_geometry")
    return dict(zip(GEOMETRY_FIELDS, [int(v) for v in out]))


def sv_workspace_size(B: int, Kmax: int, V: int, dtype: int) -> int:
    return int(_load().sv_workspace_size(int(B), int(Kmax), int(V), int(dtype)))


def sv_host_staging_size(B: int, Kmax: int, V: int, dtype: int) -> int:
    return int(_load().sv_host_staging_size(int(B), int(Kmax), int(V), int(dtype)))


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SV_DTYPE_BF16
    if t.dtype == torch.float32:
        return SV_DTYPE_F32
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _dptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host_k(K):
    k = np.ascontiguousarray(np.asarray(K.cpu() if hasattr(K, "cpu") else K, dtype=np.int32))
    return k, k.ctypes.data_as(ctypes.c_void_p)


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream), s


def _check(status: int, where: str):
    if status != SV_OK:
        raise SpecVerifyError(status, where)


def _require(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _outputs(B, Kmax, device, out_tokens, out_num_accepted):
    import torch
    if out_tokens is None:
        out_tokens = torch.empty((B, Kmax + 1), dtype=torch.int32, device=device)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=device)
    return out_tokens, out_num_accepted


def _common(target, draft, draft_tokens, uniforms, temperature, K):
    import torch
    _require(target, "target_logits")
    _require(draft, "draft_logits", target.dtype)
    _require(draft_tokens, "draft_tokens", torch.int32)
    _require(uniforms, "uniforms", torch.float32)
    _require(temperature, "temperature", torch.float32)
    k, kp = _host_k(K)
    B = int(k.shape[0])
    Kmax = int(k.max()) if B else 0
    V = int(target.shape[-1])
    return k, kp, B, Kmax, V


class Workspace:
    """A device buffer sized by sv_workspace_size for one batch shape."""

    def __init__(self, B: int, Kmax: int, V: int, dtype: int, device="cuda"):
        import torch
        self.nbytes = sv_workspace_size(B, Kmax, V, dtype)
        if self.nbytes == 0:
            raise ValueError("invalid workspace shape")
        # 256-byte alignment: the caching allocator hands out 512-byte aligned blocks
        self.buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        assert self.buffer.data_ptr() % 256 == 0

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buffer.data_ptr())


class Stats:
    """A device sv_stats (seven 64-bit counters), zeroed; calls accumulate into it."""

    def __init__(self, device="cuda"):
        import torch
        self.buffer = torch.zeros(len(STATS_FIELDS), dtype=torch.int64, device=device)

    @property
    def ptr(self):
        return self.buffer.data_ptr()

    def zero(self):
        self.buffer.zero_()

    def read(self) -> dict:
        """The counters (synchronises), plus the acceptance rate and tokens per round."""
        v = [int(x) for x in self.buffer.cpu().tolist()]
        d = dict(zip(STATS_FIELDS, v))
        d["alpha"] = d["accepted"] / d["tested"] if d["tested"] else float("nan")
        d["tokens_per_round"] = d["committed"] / d["sequences"] if d["sequences"] else float("nan")
        return d


def sv_sample_workspace_size(B: int, V: int, dtype: int) -> int:
    return int(_load().sv_sample_workspace_size(int(B), int(V), int(dtype)))


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def spec_verify(target, draft, draft_tokens, uniforms, temperature, K, out_tokens=None,
                out_num_accepted=None, stream=None):
    """spec_verify on torch CUDA tensors; scratch from the stream-ordered allocator."""
    k, kp, B, Kmax, V = _common(target, draft, draft_tokens, uniforms, temperature, K)
    out_tokens, out_num_accepted = _outputs(B, Kmax, target.device, out_tokens, out_num_accepted)
    sp, _ = _stream(stream)
    st = _load().spec_verify(_dptr(target), _dptr(draft), _dtype_code(target), _dptr(draft_tokens),
                             _dptr(uniforms), _dptr(temperature), B, kp, V, _dptr(out_tokens),
                             _dptr(out_num_accepted), sp)
    _check(st, "spec_verify")
    return out_tokens, out_num_accepted


def spec_verify_noalloc(target, draft, draft_tokens, uniforms, temperature, K, out_tokens,
                        out_num_accepted, stream=None):
    """spec_verify for callers that cannot allocate device memory per call.

    Works in the library's fixed device scratch array (SV_STATIC_SCRATCH_BYTES,
    16 MiB per device) instead of a workspace, so nothing is allocated: not by
    the library and not here (the outputs are the caller's).  Overlapping calls
    share that array and race; order them on one stream from one thread.  The
    first call on a device resolves the array's address and should come before
    any stream capture.  Shapes needing more scratch raise SpecVerifyError
    with SV_ERR_NO_MEMORY."""
    import torch
    if out_tokens is None or out_num_accepted is None:
        raise ValueError("spec_verify_noalloc writes into caller-provided outputs")
    k, kp, B, Kmax, V = _common(target, draft, draft_tokens, uniforms, temperature, K)
    _require(out_tokens, "out_tokens", torch.int32)
    _require(out_num_accepted, "out_num_accepted", torch.int32)
    if tuple(out_tokens.shape) != (B, Kmax + 1) or tuple(out_num_accepted.shape) != (B,):
        raise ValueError("out_tokens must be [B, Kmax+1] and out_num_accepted [B]")
    sp, _ = _stream(stream)
    st = _load().spec_verify_noalloc(_dptr(target), _dptr(draft), _dtype_code(target),
                                     _dptr(draft_tokens), _dptr(uniforms), _dptr(temperature), B,
                                     kp, V, _dptr(out_tokens), _dptr(out_num_accepted), sp)
    _check(st, "spec_verify_noalloc")
    return out_tokens, out_num_accepted


SV_STATIC_SCRATCH_BYTES = 16 << 20


def spec_verify_ws(target, draft, draft_tokens, uniforms, temperature, K, workspace: Workspace,
                   out_tokens=None, out_num_accepted=None, stream=None):
    """spec_verify with a caller-provided Workspace (no allocation per call)."""
    k, kp, B, Kmax, V = _common(target, draft, draft_tokens, uniforms, temperature, K)
    out_tokens, out_num_accepted = _outputs(B, Kmax, target.device, out_tokens, out_num_accepted)
    sp, _ = _stream(stream)
    st = _load().spec_verify_ws(_dptr(target), _dptr(draft), _dtype_code(target),
                                _dptr(draft_tokens), _dptr(uniforms), _dptr(temperature), B, kp, V,
                                _dptr(out_tokens), _dptr(out_num_accepted), workspace.ptr,
                                workspace.nbytes, sp)
    _check(st, "spec_verify_ws")
    return out_tokens, out_num_accepted


def spec_verify_ex(target, draft, draft_tokens, uniforms, temperature, K, workspace: Workspace,
                   diag: dict | None = None, verify_all: bool = False, chunks_per_cta: int = 0,
                   chunks_per_warp: int = 0, out_tokens=None,
                   out_num_accepted=None, stream=None, stats: "Stats | None" = None,
                   kv_len=None, packed: bool = False, expire_copy_waits: bool = False,
                   temperature_host=None):
    """spec_verify_ex; ``diag`` maps p_x / q_x / resid_mass / final_row to tensors,
    ``stats`` accumulates the call's counters, ``kv_len`` (int32 [B] CUDA
    tensor) is advanced in place by 1 + n_b for every valid sequence; ``packed``
    takes target [sum(K+1), V] and draft [sum(K), V] packed by K;
    ``expire_copy_waits`` (testing only) makes every bounded copy wait give up
    at once, to exercise the timeout path; ``temperature_host`` (a host copy
    of ``temperature``, anything numpy turns into float32 [B]) lets the
    launch give the greedy sequences to split clusters."""
    k, kp, B, Kmax, V = _common(target, draft, draft_tokens, uniforms, temperature, K)
    out_tokens, out_num_accepted = _outputs(B, Kmax, target.device, out_tokens, out_num_accepted)
    opt = SVOptions()
    if diag:
        for name in ("p_x", "q_x", "resid_mass", "final_row"):
            t = diag.get(name)
            if t is not None:
                _require(t, name)
                setattr(opt.diag, name, t.data_ptr())
    opt.verify_all = 1 if verify_all else 0
    opt.chunks_per_cta = int(chunks_per_cta)
    opt.chunks_per_warp = int(chunks_per_warp)
    if stats is not None:
        opt.stats = stats.ptr
    if kv_len is not None:
        _require(kv_len, "kv_len")
        opt.kv_len = kv_len.data_ptr()
    opt.packed_logits = 1 if packed else 0
    opt.expire_copy_waits = 1 if expire_copy_waits else 0
    th = None
    if temperature_host is not None:
        import numpy as np
        th = np.ascontiguousarray(np.asarray(temperature_host, dtype=np.float32))
        if th.shape != (B,):
            raise ValueError("temperature_host must have shape [B]")
        opt.temperature_host = th.ctypes.data
    sp, _ = _stream(stream)
    st = _load().spec_verify_ex(_dptr(target), _dptr(draft), _dtype_code(target),
                                _dptr(draft_tokens), _dptr(uniforms), _dptr(temperature), B, kp, V,
                                _dptr(out_tokens), _dptr(out_num_accepted), ctypes.byref(opt),
                                workspace.ptr, workspace.nbytes, sp)
    _check(st, "spec_verify_ex")
    return out_tokens, out_num_accepted


def spec_sample(logits, uniforms, temperature, workspace=None, out_tokens=None, stream=None):
    """spec_sample on torch CUDA tensors: one token per row of ``logits`` [B, V]
    from softmax(logits / T) at ``uniforms`` [B] (argmax where T == 0); -1 for
    a row with unusable data.  ``workspace``: a uint8 CUDA tensor of at least
    sv_sample_workspace_size bytes (allocated here when omitted)."""
    import torch
    if logits.dim() != 2:
        raise ValueError("logits must be [B, V]")
    B, V = int(logits.shape[0]), int(logits.shape[1])
    code = _dtype_code(logits)
    for t, n in ((logits, "logits"), (uniforms, "uniforms"), (temperature, "temperature")):
        _require(t, n)
    if out_tokens is None:
        out_tokens = torch.empty(B, dtype=torch.int32, device=logits.device)
    if workspace is None:
        workspace = torch.empty(max(1, sv_sample_workspace_size(B, V, code)), dtype=torch.uint8,
                                device=logits.device)
    sp, _ = _stream(stream)
    st = _load().spec_sample(_dptr(logits), code, _dptr(uniforms), _dptr(temperature), B, V,
                             _dptr(out_tokens), ctypes.c_void_p(workspace.data_ptr()),
                             workspace.numel(), sp)
    _check(st, "spec_sample")
    return out_tokens


def spec_verify_tree(target, draft, tokens, parent, uniforms, temperature, n_nodes, workspace=None,
                     out_tokens=None, out_path=None, out_len=None, stream=None):
    """spec_verify_tree on torch CUDA tensors: target / draft logits [B, Nmax, V]
    (row n: the distribution after node n), tokens / parent (int32) and
    uniforms (float32) [B, Nmax], temperature [B], n_nodes (int32) [B].
    Returns (out_tokens, out_path, out_len).  ``workspace``: a uint8 CUDA
    tensor of at least sv_tree_workspace_size() bytes (allocated when omitted)."""
    import torch
    if target.dim() != 3:
        raise ValueError("target logits must be [B, Nmax, V]")
    B, Nmax, V = (int(x) for x in target.shape)
    _require(target, "target_logits")
    if draft is not None:
        _require(draft, "draft_logits", target.dtype)
    _require(tokens, "tokens", torch.int32)
    _require(parent, "parent", torch.int32)
    _require(uniforms, "uniforms", torch.float32)
    _require(temperature, "temperature", torch.float32)
    _require(n_nodes, "n_nodes", torch.int32)
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, Nmax), dtype=torch.int32, device=dev)
    if out_path is None:
        out_path = torch.empty((B, Nmax), dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(int(_load().sv_tree_workspace_size()), dtype=torch.uint8, device=dev)
    sp, _ = _stream(stream)
    st = _load().spec_verify_tree(_dptr(target), _dptr(draft) if draft is not None else None,
                                  _dtype_code(target), _dptr(tokens), _dptr(parent), _dptr(uniforms),
                                  _dptr(temperature), B, Nmax, _dptr(n_nodes), V, _dptr(out_tokens),
                                  _dptr(out_path), _dptr(out_len), ctypes.c_void_p(workspace.data_ptr()),
                                  workspace.numel(), sp)
    _check(st, "spec_verify_tree")
    return out_tokens, out_path, out_len


def spec_verify_host(target, draft, draft_tokens, uniforms, temperature, K, staging,
                     out_tokens=None, out_num_accepted=None, stream=None):
    """spec_verify_host on HOST tensors: pinned (page-locked, device-mapped)
    logits are read in place by the kernel, only the rows the method reaches;
    pageable logits are copied into ``staging`` first.

    ``staging`` is a uint8 CUDA tensor of at least sv_host_staging_size bytes.
    Returns (out_tokens, out_num_accepted) as CPU tensors.
    """
    import torch
    if target.is_cuda:
        raise ValueError("spec_verify_host takes host tensors")
    k, kp = _host_k(K)
    B = int(k.shape[0])
    Kmax = int(k.max()) if B else 0
    V = int(target.shape[-1])
    code = _dtype_code(target)
    if out_tokens is None:
        out_tokens = torch.empty((B, Kmax + 1), dtype=torch.int32)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32)
    sp, _ = _stream(stream)
    st = _load().spec_verify_host(_dptr(target), _dptr(draft), code, _dptr(draft_tokens),
                                  _dptr(uniforms), _dptr(temperature), B, kp, V,
                                  _dptr(out_tokens), _dptr(out_num_accepted),
                                  ctypes.c_void_p(staging.data_ptr()), staging.numel(), sp)
    _check(st, "spec_verify_host")
    return out_tokens, out_num_accepted


def sv_workspace_errors(workspace: Workspace, stream=None) -> int:
    """Device-side error flags of the last call on ``workspace`` (synchronises):
    bit 0 a bounded wait gave up, bit 1 a wrong temperature hint."""
    flags = ctypes.c_uint32(0)
    sp, _ = _stream(stream)
    st = _load().sv_workspace_errors(workspace.ptr, ctypes.byref(flags), sp)
    # the status only restates the flags (timeout: bit 0; invalid argument: bit 1)
    if st not in (SV_OK, SV_ERR_TIMEOUT) and not (st == SV_ERR_INVALID_ARG and flags.value & 2):
        _check(st, "sv_workspace_errors")
    return int(flags.value)
