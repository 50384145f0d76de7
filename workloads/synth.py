"""Synthetic workloads of the batched verify step.

Every random draw comes from numpy's Philox bit generator, seeded per row by a
``SeedSequence([seed, stream, ...indices])``, so each row is reproducible on
its own and the result does not depend on the thread count.

Streams: 0 target row (b, j); 1 draft noise row (b, j); 2 peaked ids of target
row (b, j); 3 per-row K; 4 hidden row m; 5 W_vocab row k; 6 LM-head draft
noise row (b, j).

Values are drawn in fp32 and, where the workload says bf16, rounded to bf16 by
round-to-nearest-even; the draft is formed from the unrounded fp32 target.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

F32, BF16 = "f32", "bf16"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence(list(key))))


def _normal(n: int, *key: int) -> np.ndarray:
    return _rng(*key).standard_normal(n, dtype=np.float32)


def _pool_map(fn, items):
    workers = max(1, min(len(items), os.cpu_count() or 1))
    if workers == 1 or len(items) < 4:
        return [fn(i) for i in items]
    with ThreadPoolExecutor(workers) as ex:
        return list(ex.map(fn, items))


@dataclass
class Workload:
    """One verify batch: B sequences, per-row K, vocabulary V."""
    name: str
    B: int
    K_max: int
    V: int
    k_per_row: np.ndarray                 # int32 [B]
    dtype: str                            # element type of the logits
    target: np.ndarray | None             # [B, K_max+1, V] (bf16 bits or float32)
    draft: np.ndarray | None              # [B, K_max, V] draft logits, or None
    draft_kind: str = "logits"            # "logits" or "probs"
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    seed: int = 0
    round: int = 0
    hidden: np.ndarray | None = None      # LM-head workload: [B*(K_max+1), H] bf16 bits
    w_vocab: np.ndarray | None = None     # LM-head workload: [H, V] bf16 bits
    draft_noise: np.ndarray | None = None  # LM-head workload: [B, K_max, V] float32
    meta: dict = field(default_factory=dict)

    @property
    def uniform_k(self) -> bool:
        return bool(np.all(self.k_per_row == self.K_max))

    def rows(self) -> int:
        """Verify rows B*(K+1) summed over sequences: sum_b (K_b + 1)."""
        return int(np.sum(self.k_per_row.astype(np.int64) + 1))

    def logit_bytes(self) -> int:
        """Bytes of every valid target and draft row, each read once."""
        es = 2 if self.dtype == BF16 else 4
        kb = self.k_per_row.astype(np.int64)
        t = int(np.sum(kb + 1)) * self.V * es
        d_es = 4 if self.draft_kind == "probs" else es
        d = int(np.sum(kb)) * self.V * d_es
        return t + d


def make_workload(name: str, B: int, K_max: int, V: int, *, dtype: str = BF16,
                  target_std: float = 3.0, draft_scale: float = 1.0,
                  draft_noise_std: float = 1.0, peaks: int = 0, peak_height: float = 0.0,
                  k_per_row: np.ndarray | None = None, ragged_k: tuple[int, int] | None = None,
                  temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                  seed: int = 0, round: int = 0) -> Workload:
    """Target ~ N(0, target_std^2) (+ peak_height on ``peaks`` distinct ids per
    row); draft = draft_scale * target + N(0, draft_noise_std^2)."""
    if k_per_row is None:
        if ragged_k is not None:
            lo, hi = ragged_k
            k_per_row = _rng(seed, 3).integers(lo, hi + 1, size=B).astype(np.int32)
        else:
            k_per_row = np.full(B, K_max, np.int32)
    k_per_row = np.asarray(k_per_row, dtype=np.int32)

    def target_row_f32(bj):
        b, j = bj
        x = _normal(V, seed, 0, b, j) * np.float32(target_std)
        if peaks:
            ids = _rng(seed, 2, b, j).choice(V, size=peaks, replace=False)
            x[ids] += np.float32(peak_height)
        return x

    conv = f32_to_bf16_bits if dtype == BF16 else (lambda a: a.astype(np.float32))
    store = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((B, K_max + 1, V), dtype=store)
    draft = np.empty((B, K_max, V), dtype=store)

    def fill(b):
        for j in range(K_max + 1):
            t = target_row_f32((b, j))
            target[b, j] = conv(t)
            if j < K_max:
                d = np.float32(draft_scale) * t + _normal(V, seed, 1, b, j) * np.float32(
                    draft_noise_std)
                draft[b, j] = conv(d)
        return b

    _pool_map(fill, list(range(B)))
    return Workload(name=name, B=B, K_max=K_max, V=V, k_per_row=k_per_row, dtype=dtype,
                    target=target, draft=draft, temperature=temperature, top_k=top_k,
                    top_p=top_p, seed=seed, round=round)


def make_lmhead_workload(name: str, B: int, K_max: int, V: int, H: int, *,
                         temperature: float = 0.8, seed: int = 4, hidden_std: float = 1.0,
                         w_std: float = 0.02, draft_noise_std: float = 1.0) -> Workload:
    """Hidden ~ N(0, hidden_std^2) [B*(K+1), H] bf16, W ~ N(0, w_std^2) [H, V] bf16,
    plus the fp32 draft-logit noise N(0, draft_noise_std^2) [B, K, V].  The draft
    probabilities (softmax((target logits + noise) / T)) are made by a sampler."""
    M = B * (K_max + 1)
    hidden = np.empty((M, H), np.uint16)
    w = np.empty((H, V), np.uint16)
    noise = np.empty((B, K_max, V), np.float32)

    def fill_h(m):
        hidden[m] = f32_to_bf16_bits(_normal(H, seed, 4, m) * np.float32(hidden_std))

    def fill_w(k):
        w[k] = f32_to_bf16_bits(_normal(V, seed, 5, k) * np.float32(w_std))

    def fill_n(bj):
        b, j = bj
        noise[b, j] = _normal(V, seed, 6, b, j) * np.float32(draft_noise_std)

    _pool_map(fill_h, list(range(M)))
    _pool_map(fill_w, list(range(H)))
    _pool_map(fill_n, [(b, j) for b in range(B) for j in range(K_max)])
    return Workload(name=name, B=B, K_max=K_max, V=V,
                    k_per_row=np.full(B, K_max, np.int32), dtype=F32, target=None, draft=None,
                    draft_kind="probs", temperature=temperature, seed=seed, hidden=hidden,
                    w_vocab=w, draft_noise=noise, meta={"H": H})


# The five workloads of the verify step (sizes, value distributions, knobs, seeds).
CONFIGS = {
    1: dict(name="tiny: B=1 K=4 V=1000 fp32", B=1, K_max=4, V=1000, dtype=F32,
            target_std=2.0, draft_scale=1.0, draft_noise_std=0.5, temperature=1.0, seed=0),
    2: dict(name="B=8 K=5 V=32000 bf16", B=8, K_max=5, V=32000, dtype=BF16,
            target_std=3.0, draft_scale=0.8, draft_noise_std=0.6 * 3.0, temperature=1.0,
            seed=1),
    3: dict(name="B=64 K=8 V=128256 bf16 T=0.7 top-k=50", B=64, K_max=8, V=128256,
            dtype=BF16, target_std=3.0, peaks=20, peak_height=8.0, draft_scale=1.0,
            draft_noise_std=1.0, temperature=0.7, top_k=50, seed=2),
    4: dict(name="B=256 ragged K=1..8 V=152064 bf16 top-p=0.9", B=256, K_max=8, V=152064,
            dtype=BF16, target_std=3.0, draft_scale=0.9, draft_noise_std=1.5,
            ragged_k=(1, 8), temperature=1.0, top_p=0.9, seed=3),
    5: dict(name="fused LM head: B=32 K=7 H=8192 V=128256", B=32, K_max=7, V=128256,
            H=8192, temperature=0.8, seed=4),
}


def make_config(n: int, **override) -> Workload:
    """Workload ``n`` (1..5) of the verify step; keyword overrides shrink it."""
    spec = dict(CONFIGS[n])
    spec.update(override)
    if n == 5:
        H = spec.pop("H")
        return make_lmhead_workload(spec.pop("name"), spec.pop("B"), spec.pop("K_max"),
                                    spec.pop("V"), H, **spec)
    return make_workload(spec.pop("name"), spec.pop("B"), spec.pop("K_max"), spec.pop("V"),
                         **spec)
