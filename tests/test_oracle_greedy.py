"""Pins of the oracle's greedy verify (temperature 0).

Greedy speculative decoding ("Speculative Decoding from Scratch", How much
faster in practice? (3.3, 4.1): the "argmax" setting) accepts drafted tokens
while they equal the target's argmax and then emits the target's argmax.  The
pins: numpy's argmax (first maximum: the lowest id on ties) driving the
textbook loop, the top-k = 1 case of the sampling path, the draft-side
sampler, and the refusals."""
import numpy as np
import pytest

import oracle as orc
from workloads.synth import f32_to_bf16_bits, bf16_bits_to_f32

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _tied_rows(rng, B, K, V):
    """Integer-valued logits in [-3, 3]: equal maxima in most rows."""
    tgt = rng.integers(-3, 4, size=(B, K + 1, V)).astype(np.float32)
    drf = rng.integers(-3, 4, size=(B, K, V)).astype(np.float32)
    return tgt, drf


def _textbook(tgt, toks, kpr):
    """The greedy loop written with numpy's argmax."""
    B, K1, V = tgt.shape
    K = K1 - 1
    tokens = np.full((B, K + 1), -1, np.int32)
    nacc = np.zeros(B, np.int32)
    for b in range(B):
        kb = int(kpr[b])
        j = 0
        while j < kb and toks[b, j] == int(np.argmax(tgt[b, j])):
            tokens[b, j] = toks[b, j]
            j += 1
        tokens[b, j] = int(np.argmax(tgt[b, j]))
        nacc[b] = j
    return tokens, nacc


@pytest.mark.parametrize("V", [2, 5, 64, 1000])
def test_greedy_is_the_argmax_loop(V):
    rng = np.random.default_rng(V)
    B, K = 40, 6
    tgt, drf = _tied_rows(rng, B, K, V)
    kpr = rng.integers(0, K + 1, size=B).astype(np.int32)
    # half the drafts are the target's argmax (long accepted runs), half random
    toks = rng.integers(0, V, size=(B, K)).astype(np.int32)
    am = np.argmax(tgt[:, :K], axis=2).astype(np.int32)
    take = rng.random((B, K)) < 0.7
    toks = np.where(take, am, toks).astype(np.int32)
    out = orc.verify(tgt, drf, toks, kpr, temperature=0.0, top_k=5, top_p=0.3, seed=9)
    want_t, want_n = _textbook(tgt, toks, kpr)
    np.testing.assert_array_equal(out["num_accepted"], want_n)
    np.testing.assert_array_equal(out["tokens"], want_t)
    assert (out["row_status"] == 0).all()
    # p_t at the draft is the one-hot argmax distribution; p_d is not read
    for b in range(B):
        for j in range(K):
            v = out["p_t_at_draft"][b, j]
            if j < kpr[b]:
                assert v == (1.0 if toks[b, j] == am[b, j] else 0.0)
            else:
                assert np.isnan(v)
    assert np.isnan(out["p_d_at_draft"]).all()
    assert (out["residual_mass"] == 0.0).all()
    assert np.isnan(out["target_lse"]).all()


def test_greedy_equals_top1_sampling():
    """With top-k = 1 on both sides and the drafts taken as the draft's
    argmax, the sampling path makes the same decisions as greedy verify."""
    rng = np.random.default_rng(3)
    B, K, V = 30, 5, 300
    tgt, drf = _tied_rows(rng, B, K, V)
    tgt += rng.normal(0, 0.01, tgt.shape).astype(np.float32)  # few exact ties
    drf += rng.normal(0, 0.01, drf.shape).astype(np.float32)
    kpr = rng.integers(0, K + 1, size=B).astype(np.int32)
    toks = np.argmax(drf, axis=2).astype(np.int32)
    g = orc.verify(tgt, drf, toks, kpr, temperature=0.0, seed=4)
    s = orc.verify(tgt, drf, toks, kpr, temperature=1.3, top_k=1, seed=4)
    np.testing.assert_array_equal(g["tokens"], s["tokens"])
    np.testing.assert_array_equal(g["num_accepted"], s["num_accepted"])
    np.testing.assert_array_equal(g["row_status"], s["row_status"])


def test_greedy_draft_sampler_is_argmax():
    rng = np.random.default_rng(8)
    B, K, V = 12, 4, 77
    _, drf = _tied_rows(rng, B, K, V)
    kpr = rng.integers(0, K + 1, size=B).astype(np.int32)
    toks, _ = orc.draft_sample(drf, kpr, temperature=0.0, seed=1)
    for b in range(B):
        for j in range(K):
            assert toks[b, j] == (int(np.argmax(drf[b, j])) if j < kpr[b] else -1)


def test_greedy_refusals_and_bf16():
    rng = np.random.default_rng(5)
    B, K, V = 6, 3, 50
    tgt, drf = _tied_rows(rng, B, K, V)
    tgt = f32_to_bf16_bits(tgt)
    drf = f32_to_bf16_bits(drf)
    toks = np.argmax(bf16_bits_to_f32(tgt)[:, :K], axis=2).astype(np.int32)
    kpr = np.full(B, K, np.int32)
    toks[1, 1] = V          # a token outside the vocabulary
    t32 = bf16_bits_to_f32(tgt)
    t32[2, 3, 7] = np.nan   # the bonus row of sequence 2 is not finite
    tgt = f32_to_bf16_bits(t32)
    kpr[3] = K + 1          # K_b out of range
    out = orc.verify(tgt, drf, toks, kpr, temperature=0.0)
    assert list(out["row_status"][:4]) == [0, orc.ROW_BAD_TOKEN, orc.ROW_NONFINITE, orc.ROW_BAD_K]
    assert out["num_accepted"][0] == K        # every draft is the argmax: the bonus follows
    assert out["tokens"][0, K] == int(np.argmax(bf16_bits_to_f32(tgt)[0, K]))
