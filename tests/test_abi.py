"""The C-ABI library builds, loads and exports every function include/*.h
declares; host-side argument checks (no GPU needed for these)."""
import ctypes as C
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                             r"(spec_[a-z0-9_]+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_42_gb300 import build
    path = build.build()
    import speculative_decoding_verification_42_gb300 as sv
    return sv, sv.load_library(path)


def test_header_declares_the_abi():
    import speculative_decoding_verification_42_gb300 as sv
    names = _declared_functions()
    assert names == set(sv.ABI_FUNCTIONS), names


def test_library_exports_every_declared_symbol(lib):
    sv, L = lib
    out = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_status_strings(lib):
    sv, _ = lib
    assert sv.spec_verify_status_string(sv.SPEC_OK) == "ok"
    assert "invalid" in sv.spec_verify_status_string(sv.SPEC_ERR_INVALID_ARG)
    assert sv.spec_verify_status_string(99) == "unknown status"


def test_create_rejects_bad_configs_without_touching_a_gpu(lib):
    sv, L = lib
    h = C.c_void_p()
    assert L.spec_verify_create(None, C.byref(h)) == sv.SPEC_ERR_INVALID_ARG
    bad = [
        dict(max_batch=0), dict(vocab=0), dict(max_k=-1), dict(device=-1),
        dict(target_dtype=7), dict(draft_kind=5),
        dict(draft_kind=sv.SPEC_DRAFT_LOGITS, draft_dtype=sv.SPEC_F32),   # mixed dtypes
        dict(draft_kind=sv.SPEC_DRAFT_PROBS, draft_dtype=sv.SPEC_BF16),   # probs are f32
    ]
    for change in bad:
        cfg = dict(device=0, max_batch=4, max_k=3, vocab=100, hidden=0,
                   target_kind=sv.SPEC_TARGET_LOGITS, target_dtype=sv.SPEC_BF16,
                   draft_kind=sv.SPEC_DRAFT_LOGITS, draft_dtype=sv.SPEC_BF16)
        cfg.update(change)
        c = sv.spec_verify_config(**cfg)
        rc = L.spec_verify_create(C.byref(c), C.byref(h))
        assert rc == sv.SPEC_ERR_INVALID_ARG, (change, rc)
        assert not h.value


def test_run_rejects_null_handle(lib):
    sv, L = lib
    s = sv.spec_sampling(1.0, 0, 1.0, 0, 0, 0)
    ins = sv.spec_verify_inputs()
    outs = sv.spec_verify_outputs()
    assert L.spec_verify_run(None, C.byref(ins), C.byref(s), C.byref(outs), None) == \
        sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_destroy(None) == sv.SPEC_ERR_INVALID_ARG
