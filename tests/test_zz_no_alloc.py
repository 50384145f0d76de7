"""spec_verify_run_noalloc: the verify step for callers that cannot allocate
device memory (a plugin handed only a stream at enqueue time, a serving loop
whose memory is a fixed arena, code that must avoid the device synchronisation
an allocation can cause).  It takes no handle and works in the library's one
static device array.

Its outputs must equal those of the handle entry point on the same inputs, on
two calls in a row (the second call reuses the array the first one left
behind).  This file is collected last on purpose, and it must pass both after
the other tests and alone in a fresh process."""
import ctypes as C

import numpy as np
import pytest

from parity_util import PROB_RTOL, compare, oracle_tokens, run_oracle, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu

OUT_FIELDS = ("tokens", "num_accepted", "row_status", "p_t_at_draft", "p_d_at_draft",
              "residual_mass", "target_lse")


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_42_gb300 import build
    build.build()
    import speculative_decoding_verification_42_gb300 as sv
    sv.load_library()
    return sv


def _empty_outputs(torch, B, K):
    dev = torch.device("cuda")
    return dict(tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
                num_accepted=torch.full((B,), -7, dtype=torch.int32, device=dev),
                row_status=torch.full((B,), -7, dtype=torch.int32, device=dev),
                p_t_at_draft=torch.zeros((B, K), dtype=torch.float32, device=dev),
                p_d_at_draft=torch.zeros((B, K), dtype=torch.float32, device=dev),
                residual_mass=torch.zeros((B,), dtype=torch.float32, device=dev),
                target_lse=torch.zeros((B, K + 1), dtype=torch.float32, device=dev))


def _run_noalloc(sv, torch, w, target, draft, toks, kpr, round_):
    dt = sv.SPEC_BF16 if w.dtype == "bf16" else sv.SPEC_F32
    cfg = sv.spec_verify_config(torch.cuda.current_device(), 0, 0, w.V, 0, sv.SPEC_TARGET_LOGITS,
                                dt, sv.SPEC_DRAFT_LOGITS, dt)
    ins = sv.spec_verify_inputs(target.data_ptr(), None, draft.data_ptr(), toks.data_ptr(),
                                kpr.data_ptr(), w.B, w.K_max)
    s = sv.spec_sampling(w.temperature, w.top_k, w.top_p, 0, w.seed, round_)
    out = _empty_outputs(torch, w.B, w.K_max)
    outs = sv.spec_verify_outputs(*[out[f].data_ptr() for f in OUT_FIELDS])
    sv.spec_verify_run_noalloc(cfg, ins, s, outs, torch.cuda.current_stream().cuda_stream)
    return out


@pytest.mark.parametrize("knobs,dtype,V", [
    (dict(top_k=50, temperature=0.8), "bf16", 32000),   # kept lists: decided in stage 1
    (dict(temperature=1.0), "f32", 20000),              # full rows: the stage-2 sampler
    (dict(top_p=0.9), "bf16", 32768),                   # key histograms in the array, ring sampler
])
def test_noalloc_equals_handle_entry_point_twice(orc, lib, knobs, dtype, V):
    import torch
    sv = lib
    w = make_workload("noalloc", B=16, K_max=5, V=V, dtype=dtype, ragged_k=(0, 5), seed=V,
                      **knobs)
    toks_np, _ = oracle_tokens(orc, w)
    target, draft = to_device(w.target), to_device(w.draft)
    toks = torch.from_numpy(toks_np).cuda()
    kpr = torch.from_numpy(w.k_per_row).cuda()
    ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype=dtype)
    for round_ in (3, 4):  # two calls in a row
        want = ver.run(target, draft, toks, kpr, temperature=w.temperature, top_k=w.top_k,
                       top_p=w.top_p, seed=w.seed, round=round_)
        got = _run_noalloc(sv, torch, w, target, draft, toks, kpr, round_)
        torch.cuda.synchronize()
        for f in ("tokens", "num_accepted", "row_status"):
            np.testing.assert_array_equal(got[f].cpu().numpy(), want[f].cpu().numpy(),
                                          err_msg=f"{f}, call with round {round_}")
        for f in ("p_t_at_draft", "p_d_at_draft", "residual_mass", "target_lse"):
            np.testing.assert_allclose(got[f].cpu().numpy(), want[f].cpu().numpy(),
                                       rtol=PROB_RTOL, atol=1e-9, equal_nan=True,
                                       err_msg=f"{f}, call with round {round_}")
        assert (got["num_accepted"] >= 0).all()
        # and against the fp64 oracle on the same bytes
        w.round = round_
        g = {f: got[f].cpu().numpy() for f in OUT_FIELDS}
        assert compare(g, run_oracle(orc, w, toks_np), w, toks_np) <= 1
    ver.close()


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    import torch
    sv = lib
    L = sv.load_library()
    cfg = sv.spec_verify_config(torch.cuda.current_device(), 0, 0, 128256, 0,
                                sv.SPEC_TARGET_LOGITS, sv.SPEC_BF16, sv.SPEC_DRAFT_LOGITS,
                                sv.SPEC_BF16)
    # 4096 x 17 row slots at V = 128256 need far more than the array holds;
    # the call is refused on the host before any pointer is touched
    ins = sv.spec_verify_inputs(16, None, 16, 16, None, 4096, 8)
    s = sv.spec_sampling(1.0, 50, 1.0, 0, 0, 0)
    outs = sv.spec_verify_outputs(16, 16, None, None, None, None, None)
    rc = L.spec_verify_run_noalloc(C.byref(cfg), C.byref(ins), C.byref(s), C.byref(outs), None)
    assert rc == sv.SPEC_ERR_INVALID_ARG
    # the fused LM head is not served without a workspace of its own
    cfg.target_kind, cfg.target_dtype, cfg.hidden = sv.SPEC_TARGET_HIDDEN_LMHEAD, sv.SPEC_BF16, 64
    cfg.draft_kind, cfg.draft_dtype = sv.SPEC_DRAFT_PROBS, sv.SPEC_F32
    ins = sv.spec_verify_inputs(16, 16, 16, 16, None, 1, 1)
    rc = L.spec_verify_run_noalloc(C.byref(cfg), C.byref(ins), C.byref(s), C.byref(outs), None)
    assert rc == sv.SPEC_ERR_UNSUPPORTED
