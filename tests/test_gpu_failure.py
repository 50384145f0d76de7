"""Failure reporting through the C ABI, with every fault made on the host
(no kernel is broken and nothing waits forever):

* a stalled stream (spec_verify_inject_fault): the stream kernel's producer
  issues no copy, its consumers' bounded waits run out after 4096 polls, the
  kernel records it and returns; spec_verify_check reports SPEC_ERR_TIMEOUT
  once, and the next run on the same handle matches the oracle;
* an allocator that fails: spec_verify_create returns SPEC_ERR_OOM and no
  handle;
* a caller's allocator: create takes the workspace from it, destroy gives it
  back, and runs in between are correct."""
import ctypes as C

import numpy as np
import pytest

from parity_util import compare, oracle_tokens, run_gpu, run_oracle
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_42_gb300 import build
    build.build()
    import speculative_decoding_verification_42_gb300 as m
    m.load_library()
    return m


def _workload():
    return make_workload("failure", B=8, K_max=4, V=4096, dtype="bf16", target_std=2.0,
                         draft_noise_std=0.5, temperature=0.9, top_k=50, seed=11)


def test_stalled_stream_reports_timeout_then_recovers(sv, orc):
    import torch
    w = _workload()
    toks, _ = oracle_tokens(orc, w)
    ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype="bf16")
    stream = torch.cuda.current_stream().cuda_stream
    assert sv.spec_verify_check(ver.h, stream) == sv.SPEC_OK
    sv.spec_verify_inject_fault(ver.h, sv.SPEC_FAULT_STALL_STREAM)
    run_gpu(w, toks, verifier=ver)          # launches only the stalled stream kernel
    assert sv.spec_verify_check(ver.h, stream) == sv.SPEC_ERR_TIMEOUT
    assert sv.spec_verify_check(ver.h, stream) == sv.SPEC_OK  # the record was cleared
    # the fault lasted one run: the next run is correct
    g = run_gpu(w, toks, verifier=ver)
    assert sv.spec_verify_check(ver.h, stream) == sv.SPEC_OK
    ver.close()
    assert compare(g, run_oracle(orc, w, toks), w, toks) <= 1


def test_fault_arguments(sv):
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_inject_fault(None, sv.SPEC_FAULT_STALL_STREAM)
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG
    ver = sv.Verifier(vocab=4096, max_batch=1, max_k=1, dtype="bf16")
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_inject_fault(ver.h, 99)
    ver.close()


def test_failing_allocator_gives_oom(sv):
    calls = []

    @sv.SPEC_ALLOC_FN
    def alloc(ctx, nbytes, device, ptr):
        calls.append(nbytes)
        return 1  # out of memory

    @sv.SPEC_RELEASE_FN
    def release(ctx, ptr, device):
        raise AssertionError("nothing was allocated")

    sv.spec_verify_set_allocator(alloc, release)
    try:
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.Verifier(vocab=32000, max_batch=8, max_k=4, dtype="bf16")
        assert e.value.code == sv.SPEC_ERR_OOM
        assert len(calls) == 1 and calls[0] > 0
    finally:
        sv.spec_verify_set_allocator(None, None)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_set_allocator(alloc, None)
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG


def test_caller_allocator_is_used(sv, orc):
    import torch
    held = {}

    @sv.SPEC_ALLOC_FN
    def alloc(ctx, nbytes, device, ptr):
        t = torch.empty(int(nbytes), dtype=torch.uint8, device=f"cuda:{device}")
        held[t.data_ptr()] = t
        ptr[0] = t.data_ptr()
        return 0

    released = []

    @sv.SPEC_RELEASE_FN
    def release(ctx, p, device):
        released.append(p)
        held.pop(p)

    sv.spec_verify_set_allocator(alloc, release)
    try:
        w = _workload()
        ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype="bf16")
    finally:
        sv.spec_verify_set_allocator(None, None)  # the handle keeps its own functions
    assert len(held) == 1
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks, verifier=ver)
    ver.close()
    assert len(released) == 1 and not held
    assert compare(g, run_oracle(orc, w, toks), w, toks) <= 1
