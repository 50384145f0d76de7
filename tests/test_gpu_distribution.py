"""The emitted token's distribution on the device (losslessness, run on the
GPU): one set of V = 16 target and draft logits repeated over 2^18
sequences, each with its own Philox counters, verified in four rounds
(2^20 draws in all).  Drafted tokens come from the library's draft-side
sampler.  By the rejection rule the first emitted token is distributed as the
target's post-knob distribution p_t(row 0), and, given that the draft was
accepted, the second as p_t(row 1) ("57 Speculative Decoding", Acceptance,
and why the distribution is NOT distorted; "Accelerating Large Language
Model Decoding with Speculative Sampling", Why the output distribution is
exactly the target's).  A chi-square test of the counts against p_t (from the
fp64 oracle's row softmax) must not reject at the pre-registered p = 1e-3."""
import numpy as np
import pytest

from parity_util import report

pytestmark = pytest.mark.gpu


def _chi2_sf(x, dof):
    from scipy.stats import chi2
    return float(chi2.sf(x, dof))


def _chisq(counts, p):
    n = counts.sum()
    keep = p > 0
    assert counts[~keep].sum() == 0, "a token outside the kept set was emitted"
    e = n * p[keep]
    return float(((counts[keep] - e) ** 2 / e).sum()), int(keep.sum()) - 1


@pytest.mark.parametrize("knobs", [dict(temperature=1.0), dict(temperature=0.8, top_k=6),
                                   dict(temperature=1.0, top_p=0.7)])
def test_emitted_token_follows_target(orc, knobs):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_42_gb300 import build
    build.build()
    import speculative_decoding_verification_42_gb300 as sv
    V, B, K = 16, 1 << 18, 1
    rng = np.random.default_rng(7)
    tl = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    dl = (tl[:K] + rng.standard_normal((K, V)).astype(np.float32) * 1.0).astype(np.float32)
    dev = torch.device("cuda")
    target = torch.from_numpy(tl).to(dev).expand(B, K + 1, V).contiguous()
    draft = torch.from_numpy(dl).to(dev).expand(B, K, V).contiguous()
    kpr = torch.full((B,), K, dtype=torch.int32, device=dev)
    ver = sv.Verifier(vocab=V, max_batch=B, max_k=K, dtype="f32")
    c0 = np.zeros(V, np.int64)
    c1 = np.zeros(V, np.int64)
    for rnd in range(4):
        toks = ver.draft_sample(draft, kpr, seed=123, round=rnd, **knobs)
        out = ver.run(target, draft, toks, kpr, seed=123, round=rnd, debug=False, **knobs)
        torch.cuda.synchronize()
        t = out["tokens"].cpu().numpy()
        n = out["num_accepted"].cpu().numpy()
        assert (out["row_status"].cpu().numpy() == 0).all()
        c0 += np.bincount(t[:, 0], minlength=V)
        acc = n == 1
        c1 += np.bincount(t[acc, 1], minlength=V)
    ver.close()
    p0 = orc.row_probs(tl[0], **knobs)[0]
    p1 = orc.row_probs(tl[1], **knobs)[0]
    for counts, p in ((c0, p0), (c1, p1)):
        x, dof = _chisq(counts, p)
        pv = _chi2_sf(x, dof)
        report(f"{knobs}: n = {counts.sum()}, chi2 = {x:.1f} on {dof} dof, p = {pv:.3g}")
        assert pv > 1e-3, (knobs, x, dof, pv)
