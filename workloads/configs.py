"""Seeded synthetic inputs for batched draft-token verification.

This module only *generates inputs*; it holds none of the verification
arithmetic (no softmax, ratio test, residual or inverse-CDF step of the
method).  Draft tokens are drawn with the Gumbel-max trick
(argmax of l/T + Gumbel noise), which samples exactly from softmax(l/T)
without forming it, or, for the fixed toy pairs whose draft distribution is
given as probabilities, with a searchsorted draw on the given vector.

Shapes follow the library's layout:
  target   [B, Kmax+1, V]   float32 or bfloat16 (numpy: uint16 bit patterns)
  draft    [B, Kmax,   V]   same dtype
  tokens   [B, Kmax]        int32 (padding slots i >= K_b hold 0)
  uniforms [B, Kmax+1]      float32, Philox4x32-10, slot i < K_b = accept
                            test i, slot K_b = final sample
  temperature [B]           float32, 0 = greedy
  K        [B]              int32, per-sequence draft count

Workloads (the speculative-decoding verification benchmark set):
  0  B=64, K=4, V=5, fp32 logits ~N(0,1), draft = target + N(0,1), T=1
  0t the fixed p/q toy pair replicated 200,000 times, K=1, V=5
  1  B=1, K=4, V=32000, bf16 ~N(0,2^2), draft noise N(0,1), T=1
  2  B=64, K=5, V=128256, bf16 ~N(0,3^2), draft noise N(0,0.5^2), T=1
  3  B=256, K=8, V=151936, fp32 ~N(0,2^2), draft noise N(0,1.5^2), T=0.7
  4  B=1024, K_b ~ U{1..8}, V=128256, bf16 ~N(0,2^2), noise N(0,1);
     sequences 0..511 at T=1, 512..1023 greedy (T=0)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .philox import STREAM_DRAFT, STREAM_LOGITS, STREAM_UNIFORMS, uniform_grid

# The toy pair printed with the 200k-draw simulation (target p, draft q).
TOY_P = np.array([0.40, 0.25, 0.15, 0.12, 0.08])
TOY_Q = np.array([0.20, 0.40, 0.20, 0.10, 0.10])


@dataclass(frozen=True)
class Spec:
    name: str
    B: int
    K: object            # int, or "ragged" (K_b ~ U{1..8})
    V: int
    dtype: str           # "f32" or "bf16"
    sigma_t: float
    sigma_d: float
    temp: object         # float, or "mixed" (first half 1.0, second half 0)
    seed: int
    extra: dict = field(default_factory=dict)


SPECS = {
    0: Spec("b64_k4_v5_f32", 64, 4, 5, "f32", 1.0, 1.0, 1.0, 1000),
    1: Spec("b1_k4_v32000_bf16", 1, 4, 32000, "bf16", 2.0, 1.0, 1.0, 1001),
    2: Spec("b64_k5_v128256_bf16", 64, 5, 128256, "bf16", 3.0, 0.5, 1.0, 1002),
    3: Spec("b256_k8_v151936_f32_t0.7", 256, 8, 151936, "f32", 2.0, 1.5, 0.7, 1003),
    4: Spec("b1024_raggedk1-8_v128256_bf16_halfgreedy", 1024, "ragged", 128256,
            "bf16", 2.0, 1.0, "mixed", 1004),
}


# ----------------------------------------------------------------------------
# dtype helpers
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(arr) if dtype == "bf16" else np.asarray(arr, dtype=np.float32)


def quantize(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == "bf16" else np.asarray(x32, dtype=np.float32)


# ----------------------------------------------------------------------------
# per-sequence K and temperature
# ----------------------------------------------------------------------------
def ragged_k(seed: int, B: int, kmin: int = 1, kmax: int = 8) -> np.ndarray:
    u = uniform_grid(seed, STREAM_LOGITS ^ 0x4B, B, 1)[:, 0].astype(np.float64)
    return (kmin + np.floor(u * (kmax - kmin + 1))).astype(np.int32)


def k_array(spec_k, B: int, seed: int) -> np.ndarray:
    if isinstance(spec_k, str):
        return ragged_k(seed, B)
    return np.full(B, int(spec_k), dtype=np.int32)


def temp_array(spec_t, B: int) -> np.ndarray:
    if isinstance(spec_t, str):          # "mixed": first half sampling, second half greedy
        t = np.ones(B, dtype=np.float32)
        t[B // 2:] = 0.0
        return t
    return np.full(B, float(spec_t), dtype=np.float32)


# ----------------------------------------------------------------------------
# Gumbel-max draft sampling on the host (small inputs)
# ----------------------------------------------------------------------------
def _gumbel_rows(seed: int, nrows: int, V: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, STREAM_DRAFT]))
    return rng.gumbel(size=(nrows, V))


def draft_tokens_host(draft32: np.ndarray, K: np.ndarray, temps: np.ndarray,
                      seed: int) -> np.ndarray:
    """Tokens x_i: Gumbel-max sample of softmax(l_d/T) (T>0) or argmax (T=0)."""
    B, Kmax, V = draft32.shape
    tok = np.zeros((B, Kmax), dtype=np.int32)
    if Kmax == 0:
        return tok
    g = _gumbel_rows(seed, B * Kmax, V).reshape(B, Kmax, V)
    T = np.asarray(temps, np.float64).reshape(B, 1, 1)
    d = draft32.astype(np.float64)
    samp = np.argmax(d / np.where(T > 0, T, 1.0) + g, axis=-1)
    greedy = np.argmax(d, axis=-1)
    tok = np.where(T.reshape(B, 1) > 0, samp, greedy).astype(np.int32)
    pad = np.arange(Kmax)[None, :] >= np.asarray(K).reshape(B, 1)
    tok[pad] = 0
    return tok


def categorical_draws(probs: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Draw from a *given* probability vector with uniforms u (searchsorted)."""
    cdf = np.cumsum(np.asarray(probs, dtype=np.float64))
    cdf /= cdf[-1]
    idx = np.searchsorted(cdf, np.asarray(u, dtype=np.float64), side="right")
    return np.minimum(idx, len(cdf) - 1).astype(np.int32)


# ----------------------------------------------------------------------------
# numpy generation (sizes the oracle finishes in seconds)
# ----------------------------------------------------------------------------
def make_host(B: int, K, V: int, dtype: str, sigma_t: float, sigma_d: float,
              temps, seed: int) -> dict:
    K = np.asarray(K, dtype=np.int32) if not np.isscalar(K) else np.full(B, int(K), np.int32)
    temps = np.asarray(temps, dtype=np.float32) if not np.isscalar(temps) else \
        np.full(B, float(temps), np.float32)
    Kmax = int(K.max()) if B else 0
    rng = np.random.Generator(np.random.PCG64(seed))
    t32 = rng.standard_normal((B, Kmax + 1, V), dtype=np.float32) * np.float32(sigma_t)
    tgt = quantize(t32, dtype)
    tq = as_f32(tgt, dtype)
    noise = rng.standard_normal((B, Kmax, V), dtype=np.float32) * np.float32(sigma_d)
    drf = quantize(tq[:, :Kmax] + noise, dtype)
    dq = as_f32(drf, dtype)
    tok = draft_tokens_host(dq, K, temps, seed)
    uni = uniform_grid(seed, STREAM_UNIFORMS, B, Kmax + 1)
    return dict(target=tgt, draft=drf, dtype=dtype, tokens=tok, uniforms=uni,
                temperature=temps, K=K, B=B, Kmax=Kmax, V=V)


def make_spec_host(idx: int, B: int | None = None, V: int | None = None) -> dict:
    """A workload of the benchmark set generated on the host, optionally shrunk."""
    s = SPECS[idx]
    B = s.B if B is None else B
    V = s.V if V is None else V
    K = k_array(s.K, B, s.seed)
    return make_host(B, K, V, s.dtype, s.sigma_t, s.sigma_d, temp_array(s.temp, B), s.seed)


def make_pair_batch(p: np.ndarray, q: np.ndarray, B: int, K: int, seed: int,
                    bonus_p: np.ndarray | None = None) -> dict:
    """Every sequence sees the same target p and draft q at each of K positions.

    Logits are log p / log q in float32 (zeros map to -inf); x_i ~ q is drawn
    with Philox uniforms.  The bonus row (position K) is log(bonus_p or p).
    """
    p = np.asarray(p, np.float64)
    q = np.asarray(q, np.float64)
    V = len(p)
    with np.errstate(divide="ignore"):
        lp = np.log(p).astype(np.float32)
        lq = np.log(q).astype(np.float32)
        lb = np.log(p if bonus_p is None else np.asarray(bonus_p, np.float64)).astype(np.float32)
    tgt = np.empty((B, K + 1, V), np.float32)
    tgt[:, :K] = lp
    tgt[:, K] = lb
    drf = np.empty((B, K, V), np.float32)
    drf[:] = lq
    ud = uniform_grid(seed, STREAM_DRAFT, B, max(K, 1))[:, :K]
    tok = categorical_draws(q, ud.reshape(-1)).reshape(B, K)
    uni = uniform_grid(seed, STREAM_UNIFORMS, B, K + 1)
    return dict(target=tgt, draft=drf, dtype="f32", tokens=tok.astype(np.int32),
                uniforms=uni, temperature=np.ones(B, np.float32),
                K=np.full(B, K, np.int32), B=B, Kmax=K, V=V)


def make_toy(B: int = 200_000, seed: int = 1000) -> dict:
    """The fixed V=5 toy pair replicated B times, K=1, T=1."""
    return make_pair_batch(TOY_P, TOY_Q, B, 1, seed)


def make_geometric(alpha: float, B: int, K: int, seed: int) -> dict:
    """V=2 pair with acceptance probability exactly alpha at every position.

    p = [alpha/2, 1 - alpha/2], q = [1 - alpha/2, alpha/2]: sum_x min(p, q) = alpha.
    """
    p = np.array([alpha / 2, 1 - alpha / 2])
    q = np.array([1 - alpha / 2, alpha / 2])
    return make_pair_batch(p, q, B, K, seed)


# ----------------------------------------------------------------------------
# torch generation on the device (full-size workloads)
# ----------------------------------------------------------------------------
def make_device(idx: int, device="cuda", B: int | None = None, V: int | None = None,
                batch: int = 32) -> dict:
    """Full-size workload generated on the device with torch's seeded RNG.

    Logits come from torch.randn on a seeded device generator; draft tokens
    are Gumbel-max samples (argmax of l/T - log E, E ~ Exp(1)); the uniforms
    are Philox4x32-10 from the host, uploaded.
    """
    import torch
    s = SPECS[idx]
    B = s.B if B is None else B
    V = s.V if V is None else V
    K = k_array(s.K, B, s.seed)
    temps = temp_array(s.temp, B)
    Kmax = int(K.max())
    tdt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(s.seed)
    tgt = torch.empty((B, Kmax + 1, V), dtype=tdt, device=device)
    drf = torch.empty((B, Kmax, V), dtype=tdt, device=device)
    tok = torch.zeros((B, Kmax), dtype=torch.int32, device=device)
    temps_d = torch.from_numpy(temps).to(device)
    for b0 in range(0, B, batch):
        b1 = min(B, b0 + batch)
        t32 = torch.randn((b1 - b0, Kmax + 1, V), generator=g, device=device,
                          dtype=torch.float32).mul_(s.sigma_t)
        tgt[b0:b1] = t32.to(tdt)
        # explicit copy: for fp32 logits .float() would alias the target rows
        d32 = tgt[b0:b1, :Kmax].to(torch.float32, copy=True)
        d32.add_(torch.randn((b1 - b0, Kmax, V), generator=g, device=device,
                             dtype=torch.float32).mul_(s.sigma_d))
        drf[b0:b1] = d32.to(tdt)
        dq = drf[b0:b1].float()
        tb = temps_d[b0:b1].view(-1, 1, 1)
        e = torch.empty_like(dq).exponential_(generator=g)
        samp = torch.argmax(dq / tb.clamp_min(1e-30) - torch.log(e), dim=-1)
        greedy = torch.argmax(dq, dim=-1)
        tok[b0:b1] = torch.where(tb.view(-1, 1) > 0, samp, greedy).to(torch.int32)
        del t32, d32, dq, e
    # padding slots (i >= K_b) are never read; keep them at token 0
    pad = torch.arange(Kmax, device=device).view(1, -1) >= torch.from_numpy(K).to(device).view(-1, 1)
    tok[pad] = 0
    uni = uniform_grid(s.seed, STREAM_UNIFORMS, B, Kmax + 1)
    return dict(target=tgt, draft=drf, dtype=s.dtype, tokens=tok,
                uniforms=torch.from_numpy(uni).to(device), temperature=temps_d,
                K=K, B=B, Kmax=Kmax, V=V, uniforms_host=uni, temperature_host=temps)


def bytes_all_rows(K: np.ndarray, temps: np.ndarray, V: int, dtype: str, Kmax: int) -> int:
    """One read of every logit row a verify-all-positions pass touches, plus the
    small per-sequence arrays (tokens, uniforms, outputs)."""
    s = 2 if dtype == "bf16" else 4
    K = np.asarray(K, np.int64)
    samp = np.asarray(temps) > 0
    rows = int(np.sum(K + 1) + np.sum(np.where(samp, K, 0)))
    B = len(K)
    return rows * V * s + B * Kmax * 4 + B * (Kmax + 1) * 4 + B * (Kmax + 2) * 4


def bytes_needed(K: np.ndarray, temps: np.ndarray, nacc: np.ndarray, V: int, dtype: str,
                 Kmax: int) -> int:
    """One read of every logit row the method reads: target rows 0..n_b and draft
    rows 0..min(n_b, K_b - 1) (sampling sequences), where n_b = num_accepted;
    rows past the first rejection are never looked at."""
    s = 2 if dtype == "bf16" else 4
    K = np.asarray(K, np.int64)
    n = np.asarray(nacc, np.int64)
    n = np.where(n < 0, K, n)            # invalid sequences: count every row
    samp = np.asarray(temps) > 0
    rows = int(np.sum(n + 1) + np.sum(np.where(samp, np.minimum(n + 1, K), 0)))
    B = len(K)
    return rows * V * s + B * Kmax * 4 + B * (Kmax + 1) * 4 + B * (Kmax + 2) * 4
