"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Tokens, accepted lengths and status are bit-exact except
reported near-tie rows; probabilities at the drafted tokens within 1e-5
relative (see parity_util)."""
import numpy as np
import pytest

from parity_util import (DELTA, compare, oracle_tokens, run_gpu, run_oracle, run_oracle_parallel,
                         to_device, report)
from workloads import make_config, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_42_gb300 import build
    build.build()


def _check(orc, w, rows=None, max_near_frac=0.05, min_exact=None):
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks)
    if rows is None:
        o = run_oracle(orc, w, toks)
    else:
        o = {}
        parts = [run_oracle(orc, w, toks, b, b + 1) for b in rows]
        for k in parts[0]:
            o[k] = parts[0][k].copy()
            for b, part in zip(rows, parts):
                o[k][b] = part[k][b]
    n_near = compare(g, o, w, toks, rows)
    n = w.B if rows is None else len(rows)
    idx = np.arange(w.B) if rows is None else np.asarray(rows)
    why = {k: int((o[k][idx] < DELTA).sum()) for k in ("margin_accept", "margin_topp",
                                                         "margin_cdf")}
    report(f"{w.name}: {n - n_near} of {n} sequences compared bit-exactly; near-ties {why}")
    assert n_near <= max(1, max_near_frac * n), f"{n_near} near-tie rows of {n}: {why}"
    if min_exact is not None:
        assert n - n_near >= min_exact
    return g, o, n_near


# ----------------------------------------------------------- small shapes --
SMALL = [
    # (V, dtype, knobs)
    (2, "f32", dict()), (3, "bf16", dict(temperature=0.6)), (16, "f32", dict(top_k=1)),
    (16, "bf16", dict(top_k=2)), (1000, "f32", dict(top_k=50, temperature=0.7)),
    (1000, "bf16", dict(top_p=0.9)), (4097, "bf16", dict(top_k=50)),
    (4097, "f32", dict(top_p=0.5, temperature=1.3)), (4097, "bf16", dict(top_k=4096)),
    (4097, "f32", dict(top_p=1e-6)), (4097, "bf16", dict(top_k=300, top_p=0.8)),
    (4097, "f32", dict()), (1000, "bf16", dict(top_k=999, top_p=0.95)),
]


@pytest.mark.parametrize("V,dtype,knobs", SMALL)
def test_small_shapes(orc, V, dtype, knobs):
    w = make_workload(f"V={V}", B=24, K_max=4, V=V, dtype=dtype, target_std=2.5,
                      draft_scale=0.9, draft_noise_std=1.0, ragged_k=(0, 4), seed=V + 7,
                      **knobs)
    _check(orc, w)


@pytest.mark.parametrize("V,dtype,knobs", [
    (40000, "bf16", dict()),                       # 3 segments, ragged tail
    (70000, "f32", dict(temperature=0.8)),         # 9 segments, vector path
    (20001, "f32", dict(top_k=50)),                # odd V: scalar path, chunk path
    (50001, "bf16", dict(top_p=0.9)),              # odd V, several segments, nucleus
    (131072, "bf16", dict(top_k=50, top_p=0.9)),
    (65536, "f32", dict(top_k=2000)),              # k above the list capacity
])
def test_several_segments(orc, V, dtype, knobs):
    w = make_workload(f"V={V}", B=6, K_max=3, V=V, dtype=dtype, target_std=3.0, peaks=5,
                      peak_height=6.0, draft_noise_std=1.0, ragged_k=(0, 3), seed=V,
                      **knobs)
    _check(orc, w)


# ------------------------------------------------------- top-k row merge --
# Top-k rows (k <= 128, 16-byte rows) are streamed for their 16-bit chunk
# keys, then one CTA per row takes the k-th largest chunk key as the bound,
# re-reads the chunks reaching it and ranks their logits exactly; rows with
# more candidates than the CTA stages (ties) go to the decision grid's block
# merge.  f32 rows have 32-element chunks; the last chunk of a row may be
# short.
@pytest.mark.parametrize("V,dtype,B,K,knobs", [
    (128256, "bf16", 16, 8, dict(top_k=50, temperature=0.7)),
    (128256, "f32", 8, 8, dict(top_k=50)),                  # last segment: 40 chunks < k
    (100000, "bf16", 12, 6, dict(top_k=128, top_p=0.95)),   # largest k of the path
    (65536, "bf16", 16, 4, dict(top_k=1, temperature=1.5)),
    (40000, "f32", 24, 5, dict(top_k=7, temperature=0.5)),
])
def test_topk_merge(orc, V, dtype, B, K, knobs):
    w = make_workload(f"cand V={V}", B=B, K_max=K, V=V, dtype=dtype, target_std=3.0, peaks=20,
                      peak_height=8.0, draft_noise_std=1.0, ragged_k=(0, K), seed=V + B,
                      **knobs)
    _check(orc, w)


def test_long_drafts(orc):
    """K_b up to 20: sequences with 2 K_b + 1 > 32 rows are decided by the
    general (looping) warp decision, shorter ones one row per lane."""
    w = make_workload("long K", B=10, K_max=20, V=8192, dtype="bf16", target_std=2.5,
                      draft_noise_std=0.8, ragged_k=(0, 20), seed=123, top_k=40, temperature=0.9)
    assert (w.k_per_row >= 16).any() and (w.k_per_row < 16).any()
    _check(orc, w)


def test_topk_merge_heavy_ties(orc):
    """Logits rounded to integers: many chunks and logits tie at the bound,
    so rows overflow the CTA's staging and take the block merge; ties keep
    the lowest ids either way."""
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    w = make_workload("ties-int", B=8, K_max=4, V=50000, dtype="bf16", target_std=1.5,
                      draft_noise_std=0.7, seed=41, top_k=60)
    w.target = f32_to_bf16_bits(np.round(bf16_bits_to_f32(w.target)))
    w.draft = f32_to_bf16_bits(np.round(bf16_bits_to_f32(w.draft)))
    _check(orc, w)


def test_topk_merge_spike(orc):
    """A few logits far above the rest: the largest chunk key is more than
    the histogram window above the k-th, so the bound falls back to the first
    (thread-maximum) bound or to every chunk; the result is the same."""
    w = make_workload("spike", B=6, K_max=3, V=32768, dtype="bf16", target_std=2.0,
                      peaks=3, peak_height=3000.0, draft_noise_std=0.5, seed=77, top_k=40)
    _check(orc, w)


def test_topk_merge_clustered_chunks(orc):
    """Tokens 0..4095 all far above the rest: eight of the row merge's threads
    own every hot chunk, so the first bound (the k-th largest thread maximum)
    lies among the cold logits.  Its ~110 chunks fit one gather but hold
    ~4100 candidates, more than the staging; the bound is raised to the k-th
    largest chunk key and the chunks read again (~100 candidates)."""
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    w = make_workload("clustered", B=4, K_max=3, V=65536, dtype="bf16", target_std=1.0,
                      draft_noise_std=0.5, seed=91, top_k=50)
    rng = np.random.default_rng(5)
    for name in ("target", "draft"):
        a = bf16_bits_to_f32(getattr(w, name))
        a[..., :4096] = 6.0 + 4.0 * rng.random(a[..., :4096].shape)
        setattr(w, name, f32_to_bf16_bits(a))
    _check(orc, w)


def test_topk_merge_draft_probs(orc):
    """Top-k target rows through the row merge, draft given as f32
    probabilities (not streamed)."""
    w = make_workload("cand-probs", B=10, K_max=5, V=40960, dtype="f32", ragged_k=(0, 5),
                      seed=52, temperature=0.9, top_k=20)
    q = np.empty_like(w.draft)
    for b in range(w.B):
        for j in range(w.K_max):
            q[b, j] = orc.row_probs(w.draft[b, j], 0.9, 20)[0].astype(np.float32)
    w.draft, w.draft_kind = q, "probs"
    _check(orc, w)


# ---------------------------------------------------- greedy verify (T = 0) --
# Temperature 0: the kept set of a row is its argmax (lowest id on ties); a
# draft is accepted iff it is the target's argmax, and the emitted token is the
# target's argmax at the first mismatch (or at K_b).  No draft row is read.
@pytest.mark.parametrize("V,dtype,B,K,tied", [
    (128256, "bf16", 16, 8, False),
    (32000, "f32", 12, 5, True),
    (1000, "bf16", 24, 6, True),
    (2, "f32", 8, 3, True),
    (130, "bf16", 8, 4, False),      # rows not on 16 bytes: the per-segment path
])
def test_greedy_verify(orc, V, dtype, B, K, tied):
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    w = make_workload(f"greedy V={V}", B=B, K_max=K, V=V, dtype=dtype, target_std=2.0,
                      draft_scale=1.0, draft_noise_std=0.3, ragged_k=(0, K), seed=V + 7,
                      temperature=0.0, top_k=5, top_p=0.5)
    if tied:  # integer logits: equal maxima in most rows
        if dtype == "bf16":
            w.target = f32_to_bf16_bits(np.round(bf16_bits_to_f32(w.target)))
            w.draft = f32_to_bf16_bits(np.round(bf16_bits_to_f32(w.draft)))
        else:
            w.target, w.draft = np.round(w.target), np.round(w.draft)
    toks, _ = oracle_tokens(orc, w)  # the draft's argmax
    rng = np.random.default_rng(V)
    flip = rng.random(toks.shape) < 0.15
    toks = np.where(flip & (toks >= 0), rng.integers(0, V, toks.shape), toks).astype(np.int32)
    g = run_gpu(w, toks)
    o = run_oracle(orc, w, toks)
    assert compare(g, o, w, toks) == 0  # greedy has no near-ties
    assert (o["num_accepted"] > 0).any() and (o["num_accepted"] < w.k_per_row).any()


def test_greedy_without_draft(orc):
    """Greedy verify reads no draft row: a NULL draft gives the same result."""
    import torch
    import speculative_decoding_verification_42_gb300 as sv
    w = make_workload("greedy no draft", B=6, K_max=4, V=4096, dtype="bf16", seed=5,
                      temperature=0.0)
    toks, _ = oracle_tokens(orc, w)
    ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype="bf16")
    out = ver.run(to_device(w.target), None, torch.from_numpy(toks).cuda(),
                  torch.from_numpy(w.k_per_row).cuda(), temperature=0.0)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}
    ver.close()
    o = run_oracle(orc, w, toks)
    assert compare(g, o, w, toks) == 0


def test_greedy_draft_sampler(orc):
    """The draft-side sampler at temperature 0 returns each draft row's argmax."""
    import torch
    import speculative_decoding_verification_42_gb300 as sv
    w = make_workload("greedy drafts", B=8, K_max=5, V=20000, dtype="f32", seed=6,
                      ragged_k=(0, 5), temperature=0.0)
    ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype="f32")
    g = ver.draft_sample(to_device(w.draft), torch.from_numpy(w.k_per_row).cuda(),
                         temperature=0.0).cpu().numpy()
    ver.close()
    want, _ = oracle_tokens(orc, w)
    np.testing.assert_array_equal(g, want)


# ------------------------------------------------------ early-exit verify --
# The rows after the first rejection are not read: the same tokens, lengths
# and statuses as the full verify; p_t / p_d / lse only at the positions read.
@pytest.mark.parametrize("V,dtype,B,K,knobs", [
    (128256, "bf16", 24, 8, dict(top_k=50, temperature=0.7)),
    (32000, "f32", 40, 6, dict(top_k=20, top_p=0.9)),
    (50000, "bf16", 30, 5, dict(top_k=1, temperature=1.3)),
    (20000, "bf16", 20, 7, dict(temperature=0.0)),           # greedy: no draft row read
])
def test_early_exit(orc, V, dtype, B, K, knobs):
    w = make_workload(f"exit V={V}", B=B, K_max=K, V=V, dtype=dtype, target_std=3.0, peaks=10,
                      peak_height=6.0, draft_noise_std=1.0, ragged_k=(0, K), seed=V + 3, **knobs)
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks, early_exit=True)
    o = run_oracle(orc, w, toks)
    n_near = compare(g, o, w, toks, early_exit=True)
    assert n_near <= max(1, 0.05 * w.B)
    assert (o["num_accepted"] < w.k_per_row).any()  # some sequences stop early


def test_early_exit_matches_full(orc):
    """Early exit and the full verify take the same decisions (heavy ties
    included: rows whose candidates overflow send the batch through the
    regular pipeline)."""
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    for tied in (False, True):
        w = make_workload("exit vs full", B=16, K_max=6, V=30000, dtype="bf16", target_std=1.5,
                          draft_noise_std=0.7, seed=61, top_k=60, ragged_k=(0, 6))
        if tied:
            w.target = f32_to_bf16_bits(np.round(bf16_bits_to_f32(w.target)))
            w.draft = f32_to_bf16_bits(np.round(bf16_bits_to_f32(w.draft)))
        toks, _ = oracle_tokens(orc, w)
        e = run_gpu(w, toks, early_exit=True)
        f = run_gpu(w, toks)
        for k in ("tokens", "num_accepted", "row_status"):
            np.testing.assert_array_equal(e[k], f[k], err_msg=f"{k} tied={tied}")


def test_early_exit_refusals(orc):
    """Bad K, bad tokens and a non-finite row before the first rejection."""
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    w = make_workload("exit refusals", B=6, K_max=4, V=8192, dtype="bf16", seed=62, top_k=30)
    toks, _ = oracle_tokens(orc, w)
    toks[1, 0] = w.V                  # a token outside the vocabulary
    w.k_per_row[2] = w.K_max + 1      # K_b out of range
    t = bf16_bits_to_f32(w.target)
    t[3, 0, 17] = np.nan              # position 0 of sequence 3 is always read
    w.target = f32_to_bf16_bits(t)
    g = run_gpu(w, toks, early_exit=True)
    o = run_oracle(orc, w, toks)
    assert list(g["row_status"][1:4]) == [orc.ROW_BAD_TOKEN, orc.ROW_BAD_K, orc.ROW_NONFINITE]
    assert compare(g, o, w, toks, early_exit=True) <= 1


# ------------------------------------------------------ the five workloads --
def test_config1_tiny(orc):
    _check(orc, make_config(1))


def test_config2(orc):
    _check(orc, make_config(2))


def test_config3_full_size(orc):
    """Every one of the 64 sequences (576 target and 512 draft rows) against
    the oracle, which runs on the host cores in parallel ranges."""
    w = make_config(3)
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks)
    o = run_oracle_parallel(orc, w, toks)
    n_near = compare(g, o, w, toks)
    why = {k: int((o[k] < DELTA).sum()) for k in ("margin_accept", "margin_topp", "margin_cdf")}
    report(f"{w.name}: {w.B - n_near} of {w.B} sequences bit-exact; near-ties {why}")
    assert n_near <= max(1, 0.05 * w.B), why


# Nucleus window of the key-histogram path (bf16 rows with top-p alone).  The
# GPU weighs each bf16 key by exp2f of an exponent exact to ~2^-40 (<= 2 ulp,
# 1.2e-7 relative, independent from key to key) and sums the per-key masses in
# fp64; the tokens below the two-binade key window (a few % of the mass) are
# summed in fp32 by the stream (relative error <= 4e-6 on that part).  Its
# prefix mass at the cut is then within ~5e-8 of the exact one; the window is
# four times that.
DELTA_TOPP_HIST = 2e-7


def test_config4_full_size(orc):
    """Every one of the 256 sequences of the top-p workload against the oracle.
    Top-p 0.9 over V = 152064 keeps ~6000 tokens whose boundary tokens carry
    ~3e-5 of mass each; a row whose prefix mass at the boundary lies within
    the window of top_p is a near-tie.  The expected share of such rows is
    about 2 delta / 3e-5 (1.3% at delta = 2e-7), and a sequence reads ~10 rows;
    the bound is 1.5 times the expected count, plus two."""
    w = make_config(4)
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks)
    o = run_oracle_parallel(orc, w, toks)
    n_near = compare(g, o, w, toks, delta_topp=DELTA_TOPP_HIST)
    why = {"margin_accept": int((o["margin_accept"] < DELTA).sum()),
           "margin_topp": int((o["margin_topp"] < DELTA_TOPP_HIST).sum()),
           "margin_cdf": int((o["margin_cdf"] < DELTA).sum())}
    rows_read = float(np.mean(2 * w.k_per_row + 1))
    expect = w.B * (1.0 - (1.0 - 2 * DELTA_TOPP_HIST / 3e-5) ** rows_read)
    # the GPU's nucleus error, measured: a row whose kept set differs from the
    # oracle's by a boundary token has its P(x_j) off by that token's share of
    # the kept mass (>= 1e-6 relative here), a row with the same set agrees
    # to ~1e-7; the largest oracle prefix margin among the differing rows
    # bounds the GPU's prefix-mass error from below, and the window must hold it
    diff_margins = []
    for b in range(w.B):
        kb = int(w.k_per_row[b])
        if g["row_status"][b] != 0 or o["row_status"][b] != 0:
            continue
        for name, mname in (("p_t_at_draft", "topp_margin_t"), ("p_d_at_draft", "topp_margin_d")):
            pg, po = g[name][b, :kb].astype(np.float64), o[name][b, :kb]
            live = po > 0
            rel = np.abs(pg[live] / po[live] - 1.0)
            diff_margins += list(o[mname][b, :kb][live][rel > 1e-6])
    worst = max(diff_margins) if diff_margins else 0.0
    report(f"{w.name}: {w.B - n_near} of {w.B} sequences bit-exact; near-ties {why}; "
          f"expected about {expect:.0f}; rows with another nucleus: {len(diff_margins)}, "
          f"largest oracle prefix margin among them {worst:.3g} (window {DELTA_TOPP_HIST:g})")
    assert worst < DELTA_TOPP_HIST, (worst, len(diff_margins))
    assert n_near <= 1.5 * expect + 2, (n_near, expect, why)


# ----------------------------------------------------------------- edges --
def test_ties_fall_back_and_keep_lowest_ids(orc):
    """All-equal logits: the chunk bound admits every token, so the fast top-k
    gather overflows and the radix descent takes over; the tie rule keeps the
    lowest ids."""
    w = make_workload("ties", B=4, K_max=2, V=70000, dtype="bf16", target_std=0.0,
                      draft_noise_std=0.0, seed=5, top_k=50)
    _check(orc, w)


def _shift_bf16(w, delta):
    """Every logit of a bf16 workload moved by delta (rounded back to bf16)."""
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    w.target = f32_to_bf16_bits(bf16_bits_to_f32(w.target) + np.float32(delta))
    w.draft = f32_to_bf16_bits(bf16_bits_to_f32(w.draft) + np.float32(delta))
    return w


@pytest.mark.parametrize("case", ["negative", "all-equal", "flat", "over-32-segments"])
def test_key_histogram_edges(orc, case):
    """The nucleus of bf16 rows with top-p alone comes from per-segment key
    histograms; each case takes a path the workloads do not:
    negative: every logit below 0, so a segment's key window reaches zero and
      the general (non-positive) counting loop runs;
    all-equal: every token of a segment shares one key, the u8 bins saturate
      and the block merge recomputes the row (ties keep the lowest ids);
    flat: top-p 0.999 over N(0, 0.4^2) logits puts the cut more than 256 keys
      below the max, outside the window: the radix descent finds it (each
      token carries ~6e-5 of the mass, so a few rows are near-ties);
    over-32-segments: V = 300000 has 37 segments, more than a warp stages, so
      the block merge takes the histograms."""
    if case == "negative":
        w = _shift_bf16(make_workload(case, B=6, K_max=3, V=40000, dtype="bf16", target_std=2.0,
                                      draft_noise_std=1.0, ragged_k=(0, 3), seed=41, top_p=0.9), -30.0)
    elif case == "all-equal":
        # (V = 19992: top_p V is far from an integer, so no prefix sits on top_p)
        w = make_workload(case, B=4, K_max=2, V=19992, dtype="bf16", target_std=0.0,
                          draft_noise_std=0.0, seed=43, top_p=0.9)
    elif case == "flat":
        w = make_workload(case, B=12, K_max=3, V=16384, dtype="bf16", target_std=0.4,
                          draft_noise_std=0.2, ragged_k=(0, 3), seed=45, top_p=0.999)
    else:
        # (std 6: a nucleus of a few tokens, each carrying much of the mass,
        # so no row of 300000 tokens sits within 1e-6 of top_p)
        w = make_workload(case, B=4, K_max=2, V=300000, dtype="bf16", target_std=6.0,
                          draft_noise_std=1.0, seed=47, top_p=0.9)
    _check(orc, w, max_near_frac=0.34)


def test_masked_and_invalid_rows(orc):
    import oracle as O
    w = make_workload("edge", B=10, K_max=3, V=3000, dtype="f32", ragged_k=(0, 3), seed=9,
                      top_k=40)
    toks, _ = oracle_tokens(orc, w)
    w.target[0, :, 1000:] = -np.inf                  # masked tokens
    w.draft[0, :, 1500:] = -np.inf
    w.target[1, 0, 7] = np.nan                       # NaN in a read row
    w.target[2, w.K_max, 3] = np.inf                 # +inf (read only if K_b == K_max)
    w.draft[3, 0, :] = -np.inf                       # no finite logit
    w.k_per_row[4] = -1                              # bad K
    w.k_per_row[5] = w.K_max + 1
    toks[6, 0] = w.V                                 # bad token
    toks[7, :] = 0
    w.k_per_row[7] = 0                               # K_b = 0: bonus only
    toks, _ = orc.draft_sample(w.draft, w.k_per_row, temperature=w.temperature,
                               top_k=w.top_k, seed=w.seed)
    toks[6, 0] = w.V
    g = run_gpu(w, toks)
    o = run_oracle(orc, w, toks)
    compare(g, o, w, toks)
    assert g["row_status"][1] == O.ROW_NONFINITE
    assert g["row_status"][4] == O.ROW_BAD_K and g["row_status"][5] == O.ROW_BAD_K
    assert g["row_status"][6] == O.ROW_BAD_TOKEN


def test_draft_probabilities_input(orc):
    """The draft given as f32 probabilities (used as given)."""
    import oracle as O
    rng = np.random.default_rng(3)
    w = make_workload("probs", B=12, K_max=4, V=5000, dtype="f32", ragged_k=(0, 4), seed=31,
                      temperature=0.8)
    q = np.empty_like(w.draft)
    for b in range(w.B):
        for j in range(w.K_max):
            q[b, j] = orc.row_probs(w.draft[b, j], 0.8)[0].astype(np.float32)
    w.draft, w.draft_kind = q, "probs"
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks)
    o = run_oracle(orc, w, toks)
    compare(g, o, w, toks)


def test_deterministic_and_reusable(orc):
    w = make_config(2)
    toks, _ = oracle_tokens(orc, w)
    a, b = run_gpu(w, toks, repeat=2)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    # a different round gives different draws but still matches the oracle
    w.round = 5
    g = run_gpu(w, toks)
    o = run_oracle(orc, w, toks)
    compare(g, o, w, toks)


def test_invariants_random(orc):
    """1 <= emitted <= K_b + 1, accepted prefix equals the drafts, -1 padding."""
    w = make_workload("inv", B=64, K_max=6, V=2048, dtype="bf16", ragged_k=(0, 6), seed=77,
                      top_p=0.95)
    toks, _ = oracle_tokens(orc, w)
    g = run_gpu(w, toks)
    for b in range(w.B):
        n, kb = g["num_accepted"][b], w.k_per_row[b]
        assert 0 <= n <= kb
        np.testing.assert_array_equal(g["tokens"][b, :n], toks[b, :n])
        assert 0 <= g["tokens"][b, n] < w.V
        assert np.all(g["tokens"][b, n + 1:] == -1)


# ------------------------------------------------------ draft-side sampler --
@pytest.mark.parametrize("V,dtype,knobs", [
    (1000, "f32", dict()), (32000, "bf16", dict(top_k=50, temperature=0.7)),
    (4097, "bf16", dict(top_p=0.9)), (20001, "f32", dict(top_k=3000)),
])
def test_draft_sampler_parity(orc, V, dtype, knobs):
    import torch
    import speculative_decoding_verification_42_gb300 as sv
    from parity_util import to_device
    w = make_workload("draft", B=16, K_max=4, V=V, dtype=dtype, ragged_k=(0, 4), seed=V + 1,
                      **knobs)
    want, margin = oracle_tokens(orc, w)
    ver = sv.Verifier(vocab=V, max_batch=w.B, max_k=w.K_max, dtype=dtype)
    kpr = torch.from_numpy(w.k_per_row).cuda()
    got, probs = ver.draft_sample(to_device(w.draft), kpr, temperature=w.temperature,
                                  top_k=w.top_k, top_p=w.top_p, seed=w.seed, probs=True)
    torch.cuda.synchronize()
    got, probs = got.cpu().numpy(), probs.cpu().numpy()
    ver.close()
    ok = margin >= DELTA
    np.testing.assert_array_equal(got[ok], want[ok])
    assert (~ok & (want >= 0)).sum() <= max(1, 0.05 * ok.size)
    for b in range(w.B):
        for j in range(w.k_per_row[b]):
            P = orc.row_probs(w.draft[b, j], w.temperature, w.top_k, w.top_p)[0]
            np.testing.assert_allclose(probs[b, j], P, rtol=1e-5, atol=1e-9)


def test_handle_reuse_across_paths(orc):
    """One handle serving, in turn, the verify of top-k rows, the draft-side
    sampler, the early-exit verify and a tie-heavy batch whose rows go to the
    block merge of the decision grid: every verify matches the oracle (no run
    depends on what an earlier one left in the workspace)."""
    import torch
    import speculative_decoding_verification_42_gb300 as sv
    from workloads.synth import bf16_bits_to_f32, f32_to_bf16_bits
    w = make_workload("reuse", B=16, K_max=6, V=30000, dtype="bf16", target_std=1.5,
                      draft_noise_std=0.7, seed=62, top_k=60, ragged_k=(0, 6))
    wt = make_workload("reuse, tied", B=16, K_max=6, V=30000, dtype="bf16", target_std=1.5,
                       draft_noise_std=0.7, seed=63, top_k=60, ragged_k=(0, 6))
    wt.target = f32_to_bf16_bits(np.round(bf16_bits_to_f32(wt.target)))
    wt.draft = f32_to_bf16_bits(np.round(bf16_bits_to_f32(wt.draft)))
    toks = {id(w): oracle_tokens(orc, w)[0], id(wt): oracle_tokens(orc, wt)[0]}
    ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype="bf16")
    kpr = torch.from_numpy(w.k_per_row).cuda()
    plan = [("verify", w), ("draft", w), ("verify", w), ("exit", w), ("verify", wt), ("verify", w),
            ("verify", wt), ("verify", w)]
    for kind, wk in plan:
        if kind == "draft":
            ver.draft_sample(to_device(wk.draft), kpr, temperature=wk.temperature,
                             top_k=wk.top_k, seed=wk.seed)
            continue
        tk = toks[id(wk)]
        g = run_gpu(wk, tk, verifier=ver, early_exit=kind == "exit")
        o = run_oracle(orc, wk, tk)
        assert compare(g, o, wk, tk, early_exit=kind == "exit") <= 1, (kind, wk.name)
    ver.close()
