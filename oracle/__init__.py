"""fp64 CPU oracle for the batched speculative-sampling verify step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The
product path (the CUDA library of the package) never calls it and shares no
code with it.

This module is argument marshalling over ``liboracle.so`` (plain C, fp64,
single-threaded); every step of the arithmetic lives in ``oracle.c``.
bf16 inputs are passed as ``uint16`` bit patterns, fp32 inputs as ``float32``.
"""
from __future__ import annotations

import ctypes as C
import math
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
DRAFT_LOGITS, DRAFT_PROBS = 0, 1
ROW_OK, ROW_BAD_TOKEN, ROW_BAD_K, ROW_NONFINITE, ROW_ZERO_RESIDUAL = 0, 1, 2, 3, 4

_lib = None


class _RowInfo(C.Structure):
    _fields_ = [("M", C.c_double), ("S", C.c_double), ("topp_margin", C.c_double),
                ("n_kept", C.c_int32), ("nonfinite", C.c_int32)]


class _VerifyIn(C.Structure):
    _fields_ = [("B", C.c_int32), ("K_max", C.c_int32), ("V", C.c_int32),
                ("target_dtype", C.c_int32), ("target", C.c_void_p),
                ("draft_kind", C.c_int32), ("draft_dtype", C.c_int32),
                ("draft", C.c_void_p), ("draft_tokens", C.c_void_p),
                ("k_per_row", C.c_void_p)]


class _Sampling(C.Structure):
    _fields_ = [("temperature", C.c_double), ("top_k", C.c_int32), ("top_p", C.c_double),
                ("seed", C.c_uint64), ("round", C.c_uint64), ("delta", C.c_double)]


class _VerifyOut(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("num_accepted", C.c_void_p),
                ("row_status", C.c_void_p), ("p_t_at_draft", C.c_void_p),
                ("p_d_at_draft", C.c_void_p), ("residual_mass", C.c_void_p),
                ("target_lse", C.c_void_p), ("alpha", C.c_void_p),
                ("margin_accept", C.c_void_p), ("margin_topp", C.c_void_p),
                ("margin_cdf", C.c_void_p), ("cdf_lo", C.c_void_p), ("cdf_hi", C.c_void_p),
                ("topp_margin_t", C.c_void_p), ("topp_margin_d", C.c_void_p)]


def lib() -> C.CDLL:
    """Load (building first if needed) liboracle.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.orc_philox_batch.argtypes = [C.c_uint64, C.c_void_p, C.c_int64, C.c_void_p]
        L.orc_u24.argtypes = [C.c_uint32]
        L.orc_u24.restype = C.c_double
        L.orc_row_dist.argtypes = [C.c_void_p, C.c_int32, C.c_double, C.c_int32, C.c_double,
                                   C.c_void_p, C.POINTER(_RowInfo)]
        L.orc_row_probs.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_double, C.c_int32,
                                    C.c_double, C.c_void_p, C.POINTER(_RowInfo)]
        L.orc_inverse_cdf.argtypes = [C.c_void_p, C.c_int32, C.c_double, C.c_double,
                                      C.POINTER(C.c_double), C.POINTER(C.c_double),
                                      C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
        L.orc_inverse_cdf.restype = C.c_int32
        L.orc_residual.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]
        L.orc_residual.restype = C.c_double
        L.orc_verify.argtypes = [C.POINTER(_VerifyIn), C.POINTER(_Sampling),
                                 C.POINTER(_VerifyOut), C.c_int32, C.c_int32]
        L.orc_draft_sample.argtypes = [C.POINTER(_VerifyIn), C.POINTER(_Sampling), C.c_void_p,
                                       C.c_void_p, C.c_int32, C.c_int32]
        L.orc_lmhead.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                 C.c_int32, C.c_void_p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle inputs are float32 or bf16 bits (uint16), got {a.dtype}")


# --------------------------------------------------------------------------- #
# Philox
# --------------------------------------------------------------------------- #
def philox_batch(seed: int, ctrs: np.ndarray) -> np.ndarray:
    """Philox4x32-10 of every counter row of ``ctrs`` ([n, 4] uint32)."""
    ctrs = np.ascontiguousarray(ctrs, dtype=np.uint32).reshape(-1, 4)
    out = np.empty_like(ctrs)
    lib().orc_philox_batch(C.c_uint64(seed), _ptr(ctrs), ctrs.shape[0], _ptr(out))
    return out


def u24(word: int) -> float:
    return lib().orc_u24(C.c_uint32(word))


# --------------------------------------------------------------------------- #
# rows
# --------------------------------------------------------------------------- #
@dataclass
class RowInfo:
    M: float
    S: float
    topp_margin: float
    n_kept: int
    nonfinite: bool


def row_dist(l: np.ndarray, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """Knobs + softmax of one row of double logits. Returns (P or None, RowInfo)."""
    l = np.ascontiguousarray(l, dtype=np.float64)
    P = np.zeros_like(l)
    info = _RowInfo()
    rc = lib().orc_row_dist(_ptr(l), l.size, float(temperature), int(top_k), float(top_p),
                            _ptr(P), C.byref(info))
    ri = RowInfo(info.M, info.S, info.topp_margin, info.n_kept, bool(info.nonfinite))
    return (None if rc else P), ri


def row_probs(row: np.ndarray, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """Knobs + softmax of one row given as float32 or bf16 bits."""
    row = np.ascontiguousarray(row)
    P = np.zeros(row.size, dtype=np.float64)
    info = _RowInfo()
    rc = lib().orc_row_probs(_ptr(row), _dtype_code(row), row.size, float(temperature),
                             int(top_k), float(top_p), _ptr(P), C.byref(info))
    ri = RowInfo(info.M, info.S, info.topp_margin, info.n_kept, bool(info.nonfinite))
    return (None if rc else P), ri


def inverse_cdf(R: np.ndarray, u: float, delta: float = 0.0):
    """Returns (token, Z, margin, v_lo, v_hi)."""
    R = np.ascontiguousarray(R, dtype=np.float64)
    Z, m = C.c_double(), C.c_double()
    lo, hi = C.c_int32(), C.c_int32()
    t = lib().orc_inverse_cdf(_ptr(R), R.size, float(u), float(delta), C.byref(Z), C.byref(m),
                              C.byref(lo), C.byref(hi))
    return t, Z.value, m.value, lo.value, hi.value


def residual(Pt: np.ndarray, Pd: np.ndarray):
    Pt = np.ascontiguousarray(Pt, dtype=np.float64)
    Pd = np.ascontiguousarray(Pd, dtype=np.float64)
    R = np.empty_like(Pt)
    Z = lib().orc_residual(_ptr(Pt), _ptr(Pd), Pt.size, _ptr(R))
    return R, Z


# --------------------------------------------------------------------------- #
# batch verify / draft sampler
# --------------------------------------------------------------------------- #
def _make_in(target, draft, draft_tokens, k_per_row, draft_kind):
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    B, K1, V = target.shape
    K = K1 - 1
    if draft.shape != (B, K, V):
        raise ValueError(f"draft shape {draft.shape} != {(B, K, V)}")
    if draft_kind == DRAFT_PROBS and draft.dtype != np.float32:
        raise TypeError("draft probabilities are float32")
    toks = np.ascontiguousarray(
        draft_tokens if draft_tokens is not None else np.full((B, K), -1, np.int32),
        dtype=np.int32)
    kpr = None if k_per_row is None else np.ascontiguousarray(k_per_row, dtype=np.int32)
    vin = _VerifyIn(B, K, V, _dtype_code(target), _ptr(target), draft_kind,
                    _dtype_code(draft), _ptr(draft), _ptr(toks), _ptr(kpr))
    return vin, (target, draft, toks, kpr), (B, K, V)


def verify(target, draft, draft_tokens, k_per_row=None, *, draft_kind=DRAFT_LOGITS,
           temperature=1.0, top_k=0, top_p=1.0, seed=0, round=0, delta=1e-6,
           b_begin=0, b_end=None):
    """Verify sequences [b_begin, b_end); returns a dict of numpy outputs."""
    vin, keep, (B, K, V) = _make_in(target, draft, draft_tokens, k_per_row, draft_kind)
    b_end = B if b_end is None else b_end
    out = dict(
        tokens=np.full((B, K + 1), -1, np.int32), num_accepted=np.full(B, -1, np.int32),
        row_status=np.zeros(B, np.int32), p_t_at_draft=np.full((B, K), np.nan),
        p_d_at_draft=np.full((B, K), np.nan), residual_mass=np.zeros(B),
        target_lse=np.full((B, K + 1), np.nan), alpha=np.full((B, K), np.nan),
        margin_accept=np.full(B, np.inf), margin_topp=np.full(B, np.inf),
        margin_cdf=np.full(B, np.inf), cdf_lo=np.full(B, -1, np.int32),
        cdf_hi=np.full(B, -1, np.int32), topp_margin_t=np.full((B, K + 1), np.inf),
        topp_margin_d=np.full((B, K), np.inf))
    vout = _VerifyOut(*[_ptr(out[f]) for f, _ in _VerifyOut._fields_])
    s = _Sampling(float(temperature), int(top_k), float(top_p), int(seed), int(round),
                  float(delta))
    rc = lib().orc_verify(C.byref(vin), C.byref(s), C.byref(vout), int(b_begin), int(b_end))
    if rc:
        raise MemoryError("oracle verify failed to allocate")
    del keep
    return out


def draft_sample(draft, k_per_row=None, *, draft_kind=DRAFT_LOGITS, temperature=1.0,
                 top_k=0, top_p=1.0, seed=0, round=0, delta=1e-6, b_begin=0, b_end=None):
    """Draft tokens x[b, j] ~ P_d[b, j] with Philox tag 1; returns (tokens, margin)."""
    draft = np.ascontiguousarray(draft)
    B, K, V = draft.shape
    dummy_target = np.zeros((1, 1, 1), dtype=draft.dtype if draft.dtype == np.uint16 else np.float32)
    toks = np.full((B, K), -1, np.int32)
    margin = np.full((B, K), np.inf)
    kpr = None if k_per_row is None else np.ascontiguousarray(k_per_row, dtype=np.int32)
    vin = _VerifyIn(B, K, V, _dtype_code(dummy_target), _ptr(dummy_target), draft_kind,
                    _dtype_code(draft), _ptr(draft), None, _ptr(kpr))
    s = _Sampling(float(temperature), int(top_k), float(top_p), int(seed), int(round),
                  float(delta))
    b_end = B if b_end is None else b_end
    rc = lib().orc_draft_sample(C.byref(vin), C.byref(s), _ptr(toks), _ptr(margin),
                                int(b_begin), int(b_end))
    if rc:
        raise MemoryError("oracle draft sampler failed to allocate")
    return toks, margin


def lmhead(H_bits: np.ndarray, W_bits: np.ndarray, m0: int = 0, m1: int | None = None):
    """fp64 logits rows [m0, m1) of H (bf16 bits [M, K]) x W (bf16 bits [K, N])."""
    H_bits = np.ascontiguousarray(H_bits, dtype=np.uint16)
    W_bits = np.ascontiguousarray(W_bits, dtype=np.uint16)
    M, K = H_bits.shape
    K2, N = W_bits.shape
    assert K == K2
    m1 = M if m1 is None else m1
    out = np.empty((m1 - m0, N), dtype=np.float64)
    lib().orc_lmhead(_ptr(H_bits), _ptr(W_bits), N, K, m0, m1, _ptr(out))
    return out


def near_tie(out: dict, delta: float) -> np.ndarray:
    """Rows whose decision margins fall inside the window ``delta``."""
    return ((out["margin_accept"] < delta) | (out["margin_topp"] < delta)
            | (out["margin_cdf"] < delta))


def cores_used() -> int:
    """The oracle is single-threaded."""
    return 1


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("C", "math", "os", "np",
                                                                    "dataclass")]
