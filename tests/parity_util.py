"""Helpers of the GPU parity tests: run the library through the C ABI on a
workload and compare it with the fp64 oracle on the same input bytes.

Bar: row_status, num_accepted and every emitted token bit-exact, except rows
where the oracle reports a decision margin below the near-tie window DELTA
(|u - ratio|, a CDF gap relative to Z, or a top-p prefix gap); those are
counted, and their outputs are checked for validity (accepted prefix equals
the drafts, the final token inside the oracle's near-tie neighbourhood when
the accepted length agrees).  Probabilities at the drafted tokens agree within
PROB_RTOL relative (+ PROB_ATOL absolute for tiny values).
"""
from __future__ import annotations

import numpy as np

DELTA = 1e-6          # near-tie window of the decisions
PROB_RTOL = 1e-5      # probabilities at the drafted tokens, fp32 path
PROB_ATOL = 1e-9
LSE_ATOL = 2e-5
LSE_RTOL = 2.0 ** -22  # the output is fp32: two units in the last place at |lse|

SUMMARY = []  # lines repeated in the session summary (conftest)


def report(line: str):
    """Print a result line now and again at the end of the session."""
    print(line)
    SUMMARY.append(line)


def to_device(arr: np.ndarray):
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(
            torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def oracle_tokens(orc, w, *, draft_kind=None, delta=DELTA):
    """Drafted tokens from the oracle's draft-side sampler (tag-1 uniforms)."""
    dk = orc.DRAFT_PROBS if (draft_kind or w.draft_kind) == "probs" else orc.DRAFT_LOGITS
    toks, margin = orc.draft_sample(w.draft, w.k_per_row, draft_kind=dk,
                                    temperature=abi_float(w.temperature), top_k=w.top_k,
                                    top_p=abi_float(w.top_p), seed=w.seed, round=w.round,
                                    delta=delta)
    return toks, margin


def run_gpu(w, toks, *, verifier=None, seed=None, round=None, repeat=1, early_exit=False):
    import torch
    import speculative_decoding_verification_42_gb300 as sv
    target = to_device(w.target)
    draft = to_device(w.draft)
    xt = torch.from_numpy(np.ascontiguousarray(toks, dtype=np.int32)).cuda()
    kpr = torch.from_numpy(np.ascontiguousarray(w.k_per_row, dtype=np.int32)).cuda()
    own = verifier is None
    if own:
        verifier = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max,
                               dtype="bf16" if w.target.dtype == np.uint16 else "f32",
                               draft_kind=w.draft_kind)
    outs = []
    for _ in range(repeat):
        out = verifier.run(target, draft, xt, kpr, temperature=w.temperature, top_k=w.top_k,
                           top_p=w.top_p, seed=w.seed if seed is None else seed,
                           round=w.round if round is None else round, alpha=True,
                           early_exit=early_exit)
        torch.cuda.synchronize()
        outs.append({k: v.cpu().numpy() for k, v in out.items()})
    if own:
        verifier.close()
    return outs[0] if repeat == 1 else outs


def abi_float(x: float) -> float:
    """A knob as the C ABI carries it: spec_sampling holds temperature and
    top_p as fp32, so the oracle is given the same (fp32-rounded) numbers."""
    return float(np.float32(x))


def run_oracle(orc, w, toks, b_begin=0, b_end=None, delta=DELTA):
    dk = orc.DRAFT_PROBS if w.draft_kind == "probs" else orc.DRAFT_LOGITS
    return orc.verify(w.target, w.draft, toks, w.k_per_row, draft_kind=dk,
                      temperature=abi_float(w.temperature), top_k=w.top_k,
                      top_p=abi_float(w.top_p), seed=w.seed, round=w.round, delta=delta,
                      b_begin=b_begin, b_end=b_end)


def run_oracle_parallel(orc, w, toks, delta=DELTA, chunk=4, workers=None):
    """The oracle over every sequence, split into ranges of ``chunk`` sequences
    verified by a pool of threads.  Each call is the single-threaded C oracle
    (ctypes releases the interpreter lock while it runs, and the oracle keeps
    no global state), so the ranges run in parallel on the host cores; the
    outputs of each range are copied into one result."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    ranges = [(b, min(w.B, b + chunk)) for b in range(0, w.B, chunk)]
    n = workers or max(1, min(len(ranges), os.cpu_count() or 1))
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda r: (r, run_oracle(orc, w, toks, r[0], r[1], delta=delta)),
                            ranges))
    out = {k: v.copy() for k, v in parts[0][1].items()}
    for (b0, b1), part in parts[1:]:
        for k in out:
            out[k][b0:b1] = part[k][b0:b1]
    return out


def compare(g, o, w, toks, rows=None, delta=DELTA, prob_rtol=PROB_RTOL, early_exit=False,
            delta_topp=None):
    """Assert parity on the sequences ``rows``; returns the near-tie count.
    early_exit: the per-slot outputs exist only for the positions read (up to
    the first rejection): they are compared there and must be NaN beyond;
    alpha is not computed.  delta_topp: the window of the top-p prefix gaps
    when the path's nucleus arithmetic allows a narrower one than delta."""
    import oracle as O
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    dtp = delta if delta_topp is None else delta_topp
    near = (o["margin_accept"] < delta) | (o["margin_topp"] < dtp) | (o["margin_cdf"] < delta)
    n_near = 0
    for b in rows:
        st_o, st_g = int(o["row_status"][b]), int(g["row_status"][b])
        kb = int(w.k_per_row[b])
        if near[b]:
            n_near += 1
            assert st_g in (O.ROW_OK, O.ROW_ZERO_RESIDUAL) or st_g == st_o, (b, st_g, st_o)
            n = int(g["num_accepted"][b])
            assert 0 <= n <= kb, (b, n)
            np.testing.assert_array_equal(g["tokens"][b, :n], toks[b, :n])
            assert 0 <= g["tokens"][b, n] < w.V
            assert np.all(g["tokens"][b, n + 1:] == -1)
            if n == o["num_accepted"][b] and o["cdf_lo"][b] >= 0:
                assert o["cdf_lo"][b] <= g["tokens"][b, n] <= o["cdf_hi"][b], (
                    b, g["tokens"][b, n], o["cdf_lo"][b], o["cdf_hi"][b])
            continue
        assert st_g == st_o, (b, st_g, st_o)
        assert g["num_accepted"][b] == o["num_accepted"][b], (
            b, g["num_accepted"][b], o["num_accepted"][b], o["margin_accept"][b])
        np.testing.assert_array_equal(g["tokens"][b], o["tokens"][b], err_msg=f"sequence {b}")
        if st_o in (O.ROW_OK, O.ROW_ZERO_RESIDUAL) and early_exit:
            n = int(o["num_accepted"][b])  # positions 0..n were read
            last = min(n + 1, kb)          # drafted slots with p_t / p_d
            for name in ("p_t_at_draft", "p_d_at_draft"):
                np.testing.assert_allclose(g[name][b, :last], o[name][b, :last], rtol=prob_rtol,
                                           atol=PROB_ATOL, err_msg=f"{name} sequence {b}")
                assert np.all(np.isnan(g[name][b, last:])), (name, b)
            np.testing.assert_allclose(g["target_lse"][b, :n + 1], o["target_lse"][b, :n + 1],
                                       rtol=LSE_RTOL, atol=LSE_ATOL, err_msg=f"lse sequence {b}")
            assert np.all(np.isnan(g["target_lse"][b, n + 1:]))
            np.testing.assert_allclose(g["residual_mass"][b], o["residual_mass"][b],
                                       rtol=prob_rtol, atol=1e-7)
            assert np.all(np.isnan(g["alpha"][b]))
        elif st_o in (O.ROW_OK, O.ROW_ZERO_RESIDUAL):
            if "p_t_at_draft" in g:
                # a row whose nucleus boundary lies inside the window may keep one
                # boundary token more or less: its probabilities are not compared
                sure_t = o["topp_margin_t"][b, :kb + 1] >= dtp
                sure = sure_t[:kb] & (o["topp_margin_d"][b, :kb] >= dtp)
                for name in ("p_t_at_draft", "p_d_at_draft"):
                    np.testing.assert_allclose(g[name][b, :kb][sure], o[name][b, :kb][sure],
                                               rtol=prob_rtol, atol=PROB_ATOL,
                                               err_msg=f"{name} sequence {b}")
                    assert np.all(np.isnan(g[name][b, kb:]))
                np.testing.assert_allclose(g["target_lse"][b, :kb + 1][sure_t],
                                           o["target_lse"][b, :kb + 1][sure_t], rtol=LSE_RTOL,
                                           atol=LSE_ATOL, err_msg=f"lse sequence {b}")
                np.testing.assert_allclose(g["residual_mass"][b], o["residual_mass"][b],
                                           rtol=prob_rtol, atol=1e-7,
                                           err_msg=f"residual mass sequence {b}")
            if "alpha" in g:
                # alpha_j = sum_v min(p_t, p_d): each term in fp32, summed exactly
                sure = (o["topp_margin_t"][b, :kb] >= dtp) & (o["topp_margin_d"][b, :kb] >= dtp)
                np.testing.assert_allclose(g["alpha"][b, :kb][sure], o["alpha"][b, :kb][sure],
                                           rtol=prob_rtol, atol=1e-7, err_msg=f"alpha sequence {b}")
                assert np.all(np.isnan(g["alpha"][b, kb:]))
    return n_near
