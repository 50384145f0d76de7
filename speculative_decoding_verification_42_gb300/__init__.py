"""Batched speculative-sampling verify step for GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libspec_verify.so`` (declared in
``include/spec_verify.h``).  The functions keep the ABI's names and only
marshal arguments: every step of the verify runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing, loading it
raises.

``Verifier`` is a convenience wrapper that takes torch tensors (device memory
and the current CUDA stream come from PyTorch) and calls the same entry points.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspec_verify.so")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_OOM, SPEC_ERR_CUDA, \
    SPEC_ERR_TIMEOUT = range(6)
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_TARGET_LOGITS, SPEC_TARGET_HIDDEN_LMHEAD = 0, 1
SPEC_DRAFT_LOGITS, SPEC_DRAFT_PROBS = 0, 1
SPEC_ROW_OK, SPEC_ROW_BAD_TOKEN, SPEC_ROW_BAD_K, SPEC_ROW_NONFINITE, \
    SPEC_ROW_ZERO_RESIDUAL = range(5)

# every function the header declares (checked by the tests)
ABI_FUNCTIONS = ("spec_verify_create", "spec_verify_run", "spec_draft_sample",
                 "spec_verify_destroy", "spec_verify_status_string", "spec_verify_run_noalloc",
                 "spec_verify_set_profiling", "spec_lmhead_logits", "spec_verify_run_early_exit",
                 "spec_verify_check", "spec_verify_inject_fault", "spec_verify_set_allocator")
SPEC_FAULT_NONE, SPEC_FAULT_STALL_STREAM = 0, 1

# spec_alloc_fn / spec_release_fn of spec_verify_set_allocator
SPEC_ALLOC_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_uint64, C.c_int32, C.POINTER(C.c_void_p))
SPEC_RELEASE_FN = C.CFUNCTYPE(None, C.c_void_p, C.c_void_p, C.c_int32)
SPEC_NOALLOC_SCRATCH_BYTES = 16 << 20


class spec_verify_config(C.Structure):
    _fields_ = [("device", C.c_int32), ("max_batch", C.c_int32), ("max_k", C.c_int32),
                ("vocab", C.c_int32), ("hidden", C.c_int32), ("target_kind", C.c_int32),
                ("target_dtype", C.c_int32), ("draft_kind", C.c_int32),
                ("draft_dtype", C.c_int32)]


class spec_sampling(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_k", C.c_int32), ("top_p", C.c_float),
                ("reserved", C.c_int32), ("seed", C.c_uint64), ("round", C.c_uint64)]


class spec_verify_inputs(C.Structure):
    _fields_ = [("target", C.c_void_p), ("w_vocab", C.c_void_p), ("draft", C.c_void_p),
                ("draft_tokens", C.c_void_p), ("k_per_row", C.c_void_p),
                ("batch", C.c_int32), ("k_max", C.c_int32)]


class spec_verify_outputs(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("num_accepted", C.c_void_p),
                ("row_status", C.c_void_p), ("p_t_at_draft", C.c_void_p),
                ("p_d_at_draft", C.c_void_p), ("residual_mass", C.c_void_p),
                ("target_lse", C.c_void_p), ("alpha", C.c_void_p)]


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {spec_verify_status_string(code)} ({code})")
        self.code = code


_lib = None


def load_library(path: str | None = None) -> C.CDLL:
    """Load libspec_verify.so (raises OSError when it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError(f"{p} is missing: build it with "
                      "speculative_decoding_verification_42_gb300.build.build()")
    L = C.CDLL(p)
    L.spec_verify_create.argtypes = [C.POINTER(spec_verify_config), C.POINTER(C.c_void_p)]
    L.spec_verify_create.restype = C.c_int
    L.spec_verify_run.argtypes = [C.c_void_p, C.POINTER(spec_verify_inputs),
                                  C.POINTER(spec_sampling), C.POINTER(spec_verify_outputs),
                                  C.c_void_p]
    L.spec_verify_run.restype = C.c_int
    L.spec_draft_sample.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                    C.POINTER(spec_sampling), C.c_void_p, C.c_void_p,
                                    C.c_void_p]
    L.spec_draft_sample.restype = C.c_int
    L.spec_verify_destroy.argtypes = [C.c_void_p]
    L.spec_verify_destroy.restype = C.c_int
    L.spec_verify_status_string.argtypes = [C.c_int]
    L.spec_verify_status_string.restype = C.c_char_p
    L.spec_verify_run_noalloc.argtypes = [C.POINTER(spec_verify_config), C.POINTER(spec_verify_inputs),
                                          C.POINTER(spec_sampling), C.POINTER(spec_verify_outputs),
                                          C.c_void_p]
    L.spec_verify_run_noalloc.restype = C.c_int
    L.spec_verify_set_profiling.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p,
                                            C.POINTER(C.c_int32)]
    L.spec_verify_set_profiling.restype = C.c_int
    L.spec_lmhead_logits.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                     C.c_void_p, C.c_void_p]
    L.spec_lmhead_logits.restype = C.c_int
    L.spec_verify_check.argtypes = [C.c_void_p, C.c_void_p]
    L.spec_verify_check.restype = C.c_int
    L.spec_verify_inject_fault.argtypes = [C.c_void_p, C.c_int32]
    L.spec_verify_inject_fault.restype = C.c_int
    L.spec_verify_set_allocator.argtypes = [SPEC_ALLOC_FN, SPEC_RELEASE_FN, C.c_void_p]
    L.spec_verify_set_allocator.restype = C.c_int
    if path is None:
        _lib = L
    return L


# --------------------------------------------------------------------------- #
# the C entry points, same names                                              #
# --------------------------------------------------------------------------- #
def spec_verify_status_string(code: int) -> str:
    return load_library().spec_verify_status_string(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != SPEC_OK:
        raise SpecVerifyError(code, what)


def spec_verify_create(cfg: spec_verify_config) -> C.c_void_p:
    h = C.c_void_p()
    _check(load_library().spec_verify_create(C.byref(cfg), C.byref(h)), "spec_verify_create")
    return h


def spec_verify_run(h, inputs: spec_verify_inputs, sampling: spec_sampling,
                    outputs: spec_verify_outputs, stream: int = 0) -> None:
    _check(load_library().spec_verify_run(h, C.byref(inputs), C.byref(sampling),
                                          C.byref(outputs), C.c_void_p(stream)),
           "spec_verify_run")


def spec_verify_run_early_exit(h, inputs: spec_verify_inputs, sampling: spec_sampling,
                               outputs: spec_verify_outputs, stream: int = 0) -> None:
    """The verify reading each sequence's rows only up to its first rejection."""
    _check(load_library().spec_verify_run_early_exit(h, C.byref(inputs), C.byref(sampling),
                                                     C.byref(outputs), C.c_void_p(stream)),
           "spec_verify_run_early_exit")


def spec_draft_sample(h, draft: int, k_per_row: int | None, batch: int, k_max: int,
                      sampling: spec_sampling, draft_tokens: int, draft_probs: int | None,
                      stream: int = 0) -> None:
    _check(load_library().spec_draft_sample(h, C.c_void_p(draft), C.c_void_p(k_per_row or 0),
                                            int(batch), int(k_max), C.byref(sampling),
                                            C.c_void_p(draft_tokens),
                                            C.c_void_p(draft_probs or 0), C.c_void_p(stream)),
           "spec_draft_sample")


def spec_verify_run_noalloc(cfg: spec_verify_config, inputs: spec_verify_inputs,
                            sampling: spec_sampling, outputs: spec_verify_outputs,
                            stream: int = 0) -> None:
    """The verify step with the library's static workspace: no handle, no
    allocation (for callers that cannot allocate device memory)."""
    _check(load_library().spec_verify_run_noalloc(C.byref(cfg), C.byref(inputs), C.byref(sampling),
                                                  C.byref(outputs), C.c_void_p(stream)),
           "spec_verify_run_noalloc")


def spec_verify_set_profiling(h, ev_begin: int | None, ev_end: int | None,
                              launches_out=None) -> None:
    """Events (cudaEvent_t handles as ints) around the stage-1 stream kernel of
    later runs, and a ctypes int32 that receives each run's kernel count."""
    ptr = C.byref(launches_out) if launches_out is not None else None
    _check(load_library().spec_verify_set_profiling(h, C.c_void_p(ev_begin or 0),
                                                    C.c_void_p(ev_end or 0), ptr),
           "spec_verify_set_profiling")


def spec_lmhead_logits(hidden: int, w_vocab: int, m: int, hidden_dim: int, vocab: int,
                       logits: int, stream: int = 0) -> None:
    _check(load_library().spec_lmhead_logits(C.c_void_p(hidden), C.c_void_p(w_vocab), int(m),
                                             int(hidden_dim), int(vocab), C.c_void_p(logits),
                                             C.c_void_p(stream)),
           "spec_lmhead_logits")


def spec_verify_check(h, stream: int = 0) -> int:
    """Wait for `stream`, then read and clear the handle's device-side failure
    record: SPEC_OK, or SPEC_ERR_TIMEOUT when a bounded wait of a run ran out
    (returned, not raised; other errors raise)."""
    code = load_library().spec_verify_check(h, C.c_void_p(stream))
    if code not in (SPEC_OK, SPEC_ERR_TIMEOUT):
        _check(code, "spec_verify_check")
    return code


def spec_verify_inject_fault(h, fault: int) -> None:
    _check(load_library().spec_verify_inject_fault(h, int(fault)), "spec_verify_inject_fault")


def spec_verify_set_allocator(alloc, release, ctx: int | None = None) -> None:
    """alloc / release: SPEC_ALLOC_FN / SPEC_RELEASE_FN objects (keep them
    alive while handles created with them exist), or None for both."""
    _check(load_library().spec_verify_set_allocator(alloc or SPEC_ALLOC_FN(),
                                                    release or SPEC_RELEASE_FN(),
                                                    C.c_void_p(ctx or 0)),
           "spec_verify_set_allocator")


def spec_verify_destroy(h) -> None:
    _check(load_library().spec_verify_destroy(h), "spec_verify_destroy")


# --------------------------------------------------------------------------- #
# torch convenience wrapper (marshalling only)                                #
# --------------------------------------------------------------------------- #
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


class Verifier:
    """One library handle (its workspace sized for max_batch x max_k x vocab)."""

    def __init__(self, *, vocab: int, max_batch: int, max_k: int, dtype, draft_kind: str =
                 "logits", device: int | None = None, hidden: int = 0):
        """hidden > 0: the fused LM head (targets are bf16 hidden states, draft
        probabilities)."""
        import torch
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.vocab, self.max_batch, self.max_k = vocab, max_batch, max_k
        dt = SPEC_BF16 if dtype in ("bf16", torch.bfloat16) else SPEC_F32
        dk = SPEC_DRAFT_PROBS if draft_kind == "probs" else SPEC_DRAFT_LOGITS
        kind = SPEC_TARGET_HIDDEN_LMHEAD if hidden else SPEC_TARGET_LOGITS
        self.cfg = spec_verify_config(self.device, max_batch, max_k, vocab, int(hidden),
                                      kind, dt, dk,
                                      SPEC_F32 if dk == SPEC_DRAFT_PROBS else dt)
        self.h = spec_verify_create(self.cfg)

    def close(self):
        if self.h is not None and self.h.value:
            spec_verify_destroy(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def sampling(temperature=1.0, top_k=0, top_p=1.0, seed=0, round=0) -> spec_sampling:
        return spec_sampling(float(temperature), int(top_k), float(top_p), 0, int(seed),
                             int(round))

    def run(self, target, draft, draft_tokens, k_per_row=None, *, temperature=1.0, top_k=0,
            top_p=1.0, seed=0, round=0, out: dict | None = None, debug: bool = True,
            stream=None, w_vocab=None, alpha: bool = False, early_exit: bool = False) -> dict:
        """Verify a batch; returns (and fills) a dict of output tensors.  With the
        LM head, ``target`` is the hidden states [B * (K + 1), H] and ``w_vocab``
        the [H, V] matrix.  alpha: also the acceptance statistic of every slot.
        early_exit: read each sequence's rows only up to its first rejection."""
        import torch
        if w_vocab is not None:
            B, K = draft_tokens.shape[0], draft_tokens.shape[1]
            V = w_vocab.shape[1]
        else:
            B, K1, V = target.shape
            K = K1 - 1
        dev = target.device
        if out is None:
            out = dict(tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                       num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                       row_status=torch.empty(B, dtype=torch.int32, device=dev))
            if debug:
                out.update(p_t_at_draft=torch.empty((B, K), dtype=torch.float32, device=dev),
                           p_d_at_draft=torch.empty((B, K), dtype=torch.float32, device=dev),
                           residual_mass=torch.empty(B, dtype=torch.float32, device=dev),
                           target_lse=torch.empty((B, K + 1), dtype=torch.float32,
                                                  device=dev))
            if alpha:
                out.update(alpha=torch.empty((B, K), dtype=torch.float32, device=dev))
        ins = spec_verify_inputs(_ptr(target), _ptr(w_vocab), _ptr(draft), _ptr(draft_tokens),
                                 _ptr(k_per_row), B, K)
        outs = spec_verify_outputs(*[_ptr(out.get(f)) for f, _ in spec_verify_outputs._fields_])
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        run = spec_verify_run_early_exit if early_exit else spec_verify_run
        run(self.h, ins, self.sampling(temperature, top_k, top_p, seed, round), outs, s.cuda_stream)
        return out

    def draft_sample(self, draft, k_per_row=None, *, temperature=1.0, top_k=0, top_p=1.0,
                     seed=0, round=0, probs: bool = False, stream=None):
        """Draft tokens x ~ P_d (tag-1 uniforms); optionally the dense P_d too."""
        import torch
        B, K, V = draft.shape
        toks = torch.empty((B, K), dtype=torch.int32, device=draft.device)
        pr = torch.zeros((B, K, V), dtype=torch.float32, device=draft.device) if probs else None
        s = stream if stream is not None else torch.cuda.current_stream(draft.device)
        spec_draft_sample(self.h, _ptr(draft), _ptr(k_per_row), B, K,
                          self.sampling(temperature, top_k, top_p, seed, round), _ptr(toks),
                          _ptr(pr), s.cuda_stream)
        return (toks, pr) if probs else toks


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("C", "os")]
