"""Benchmark of the batched speculative-sampling verify step on GB300.

One step = one ``spec_verify_run`` over one batch (every stage of the verify
path), on inputs already resident in HBM.  Default workload: B = 64 sequences,
K = 8 drafts, V = 128256, bf16 logits, temperature 0.7, top-k 50 on both
distributions.  The metric is verify rows/s (rows = sum_b (K_b + 1)) with the
achieved HBM bandwidth of the dominant kernel against the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3]
  python bench.py --impl reference ...   # the fp64 CPU oracle, same workload

Multi-GPU (torchrun, one rank per GPU): every rank verifies its own batch
(weak scaling, no collective on the data path); a barrier brackets the timed
region and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify rows/s (B·(K+1)) and achieved HBM GB/s vs GB300 peak, speculative sampling"
UNIT = "rows/s"
ROTATE = 3  # input copies cycled between steps (3 x 279 MB > L2)
E2E_STREAMS = 4  # copy streams of the end-to-end measurement


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def _stage1_kernel(w) -> str:
    """The kernel that streams the logits for this workload's knobs."""
    row_bytes = w.V * (2 if w.dtype == "bf16" else 4)
    if row_bytes % 16:
        return "k_rows"
    return "k_stream"


def _traffic(kernel: str, w):
    """DRAM bytes per launch of the kernel from the committed ncu capture of
    this workload (one record, or a list of records, per kernel), or None when
    there is none or it is of an older kernel source."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        recs = d[kernel]
        for e in (recs if isinstance(recs, list) else [recs]):
            if e["workload"] != w.name:
                continue
            src = os.path.join(ROOT, "speculative_decoding_verification_42_gb300", "csrc", e["source"])
            with open(src, "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()
            return float(e["dram_bytes_per_launch"]) if sha == e["source_sha256"] else None
        return None
    except (OSError, KeyError, ValueError, TypeError):
        return None


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, steps: int, world: int, ms: float) -> float:
    """Units per second of the whole job: every rank verifies its own batch
    (replicas, weak scaling) and the job takes the slowest rank's time."""
    return units_per_rank * steps * world / (ms / 1e3)


def _workload(n: int, batch: int | None = None):
    from workloads import make_config
    return make_config(n) if not batch else make_config(n, B=batch)


def _wl_config(w, n_rot):
    cfg = {
        "workload": w.name, "config_id": None, "B": w.B, "K": w.K_max, "V": w.V,
        "input_dtype": w.dtype, "temperature": w.temperature, "top_k": w.top_k,
        "top_p": w.top_p, "rows_per_step": w.rows(), "logit_bytes_per_step": w.logit_bytes(),
        "l2": f"{n_rot} rotating input copies ({n_rot * w.logit_bytes() / 1e6:.0f} MB) > L2",
        "parallelism": "replicas (one batch per GPU)",
    }
    if w.hidden is not None:
        wb = w.w_vocab.size * 2
        cfg.update(H=int(w.hidden.shape[1]), input_dtype="bf16 hidden states, bf16 W_vocab, "
                   "f32 draft probabilities", logit_bytes_per_step=None,
                   l2=f"every step reads W_vocab ({wb / 1e9:.2f} GB) > L2")
    return cfg


# --------------------------------------------------------------------------- #
# clocks sampled during the timed region                                      #
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 0.5 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(busy), "power_w_max": max(r["power"] for r in rows)}


# --------------------------------------------------------------------------- #
# CPU baseline: the fp64 oracle as it stands, on a bounded sample             #
# --------------------------------------------------------------------------- #
def cpu_baseline(w, toks, seconds_target: float = 15.0, max_seq: int | None = None):
    import oracle
    dk = oracle.DRAFT_PROBS if w.draft_kind == "probs" else oracle.DRAFT_LOGITS
    t0 = time.perf_counter()
    rows = 0
    nseq = 0
    while True:
        b = nseq % w.B
        oracle.verify(w.target, w.draft, toks, w.k_per_row, draft_kind=dk,
                      temperature=w.temperature, top_k=w.top_k, top_p=w.top_p, seed=w.seed,
                      round=w.round, b_begin=b, b_end=b + 1)
        rows += int(w.k_per_row[b]) + 1
        nseq += 1
        el = time.perf_counter() - t0
        if el >= seconds_target or (max_seq and nseq >= max_seq):
            break
    return {"value": rows / el, "unit": UNIT, "cores": oracle.cores_used(), "kind": "oracle",
            "sample": f"{nseq} sequences ({rows} verify rows) of the same workload, "
                      f"{el:.1f} s single-threaded fp64",
            "host": _host()}


def _fused_seq(oracle, w, probs, toks, b):
    """One sequence of the fused round on the host: the fp64 LM head of its
    K+1 hidden rows, then the verify against its draft probabilities."""
    K1 = w.K_max + 1
    lg = oracle.lmhead(w.hidden, w.w_vocab, b * K1, (b + 1) * K1).astype(np.float32)
    return oracle.verify(lg.reshape(1, K1, w.V), probs[b:b + 1], toks[b:b + 1],
                         w.k_per_row[b:b + 1], draft_kind=oracle.DRAFT_PROBS,
                         temperature=w.temperature, top_k=w.top_k, top_p=w.top_p,
                         seed=w.seed, round=w.round)


def cpu_baseline_fused(w, probs, toks, seconds_target: float = 15.0):
    import oracle
    t0 = time.perf_counter()
    rows = nseq = 0
    while True:
        b = nseq % w.B
        _fused_seq(oracle, w, probs, toks, b)
        rows += int(w.k_per_row[b]) + 1
        nseq += 1
        el = time.perf_counter() - t0
        if el >= seconds_target:
            break
    return {"value": rows / el, "unit": UNIT, "cores": oracle.cores_used(), "kind": "oracle",
            "sample": f"{nseq} sequences ({rows} rows) of the same workload: fp64 LM head "
                      f"of the sequence's hidden rows + the verify, {el:.1f} s single-threaded",
            "host": _host()}


def _host():
    try:
        model = ""
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        return f"{os.cpu_count()} cores {model}".strip()
    except OSError:
        return f"{os.cpu_count()} cores"


# --------------------------------------------------------------------------- #
# the reference arm: the oracle on the host cores                             #
# --------------------------------------------------------------------------- #
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = _workload(args.config, args.batch)
    fused = w.hidden is not None
    per_step = max(1, args.ref_seq)
    if fused:
        # per sequence, untimed: the draft probabilities softmax((target
        # logits + noise) / T) and the drafted tokens; timed: the LM head of
        # the sequence's rows and its verify
        cache = {}

        def prep(b):
            if b not in cache:
                K1 = w.K_max + 1
                lg = oracle.lmhead(w.hidden, w.w_vocab, b * K1, b * K1 + w.K_max)
                q = np.stack([oracle.row_probs((lg[j] + w.draft_noise[b, j]).astype(np.float32),
                                               w.temperature)[0] for j in range(w.K_max)])
                q = q.astype(np.float32)[None]
                t, _ = oracle.draft_sample(q, w.k_per_row[b:b + 1], draft_kind=oracle.DRAFT_PROBS,
                                           temperature=w.temperature, seed=w.seed, round=w.round)
                cache.clear()
                cache[b] = (q, t)
            return cache[b]

        def one(b):
            q, t = prep(b)
            t0 = time.perf_counter()
            _fused_seq(oracle, w, q, t, 0)
            return time.perf_counter() - t0
    else:
        dk = oracle.DRAFT_PROBS if w.draft_kind == "probs" else oracle.DRAFT_LOGITS
        toks, _ = oracle.draft_sample(w.draft, w.k_per_row, draft_kind=dk,
                                      temperature=w.temperature, top_k=w.top_k, top_p=w.top_p,
                                      seed=w.seed, round=w.round)

        def one(b):
            t0 = time.perf_counter()
            oracle.verify(w.target, w.draft, toks, w.k_per_row, draft_kind=dk,
                          temperature=w.temperature, top_k=w.top_k, top_p=w.top_p,
                          seed=w.seed, round=w.round, b_begin=b, b_end=b + 1)
            return time.perf_counter() - t0

    for i in range(min(args.warmup, 1 if fused else 3)):
        one(i % w.B)
    el = 0.0
    rows = 0
    steps = 0
    for s in range(args.steps):
        for q in range(per_step):
            b = (s * per_step + q) % w.B
            el += one(b)
            rows += int(w.k_per_row[b]) + 1
        steps += 1
        if el >= args.ref_seconds:
            break  # a bounded sample: the oracle is slow by design
    value = rows / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _wl_config(w, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.cores_used(),
                         "kind": "oracle",
                         "sample": f"{steps} step(s) of {per_step} sequence(s) of the same "
                                   f"workload ({rows} rows, {el:.1f} s timed)"
                                   + ("; each: fp64 LM head + verify" if fused else ""),
                         "host": _host()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    line["config"]["l2"] = "n/a: host memory"
    line["config"]["config_id"] = args.config
    line["config"]["note"] = ("reference arm: the fp64 CPU oracle (this project's checker) on "
                              "the host cores; the pages ship no implementation; the timed "
                              f"loop stops after {args.ref_seconds:.0f} s of oracle time")
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# the GB300 arm                                                               #
# --------------------------------------------------------------------------- #
L2_BYTES = 129 * 2**20      # GB300 L2, for the rotation / flush decision


class Arm:
    """One workload resident on the device, ready to run verify steps."""

    def __init__(self, sv, torch, w, dev, local, early_exit=False, min_rot=ROTATE):
        self.sv, self.torch, self.w, self.dev = sv, torch, w, dev
        self.early_exit = early_exit
        self.stream = torch.cuda.current_stream(dev)
        self.kpr = torch.from_numpy(w.k_per_row).to(dev)
        self.knobs = dict(temperature=w.temperature, top_k=w.top_k, top_p=w.top_p, seed=w.seed)
        self.fused = w.hidden is not None
        self.wv = None

        def to_dev(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)

        if self.fused:
            # the fused round: hidden states x W_vocab, then the verify against
            # draft probabilities softmax((target logits + noise) / T) (the
            # workload's recipe, prepared once here); W (2.1 GB) exceeds L2
            H = w.hidden.shape[1]
            self.H = H
            hid = to_dev(w.hidden)
            self.wv = to_dev(w.w_vocab)
            logits = torch.empty((w.B * (w.K_max + 1), w.V), dtype=torch.float32, device=dev)
            sv.spec_lmhead_logits(hid.data_ptr(), self.wv.data_ptr(), logits.shape[0], H, w.V,
                                  logits.data_ptr(), self.stream.cuda_stream)
            lg = logits.view(w.B, w.K_max + 1, w.V)[:, :w.K_max]
            probs = torch.softmax((lg + to_dev(w.draft_noise)) / w.temperature, dim=-1).contiguous()
            del logits, lg
            self.ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype="bf16",
                                   device=local, draft_kind="probs", hidden=H)
            # drafted tokens x ~ P_d: inputs of the round, drawn once by torch
            gen = torch.Generator(device=dev)
            gen.manual_seed(w.seed)
            toks = torch.multinomial(probs.view(-1, w.V), 1, generator=gen)
            self.toks = toks.view(w.B, w.K_max).to(torch.int32).contiguous()
            self.n_rot = 1
            self.target, self.draft = [hid], [probs]
            self.l2 = f"every step reads W_vocab ({w.w_vocab.size * 2 / 1e9:.2f} GB) > L2"
        else:
            self.target, self.draft = [to_dev(w.target)], [to_dev(w.draft)]
            step_bytes = w.logit_bytes()
            # enough copies to exceed L2 twice over, unless that would be absurd
            # (the tiny workloads take an L2 flush between steps instead)
            n_rot = max(min_rot, -(-2 * L2_BYTES // step_bytes))
            self.n_rot = n_rot if n_rot <= 64 else 1
            for _ in range(self.n_rot - 1):
                self.target.append(self.target[0].clone())
                self.draft.append(self.draft[0].clone())
            self.ver = sv.Verifier(vocab=w.V, max_batch=w.B, max_k=w.K_max, dtype=w.dtype,
                                   device=local, draft_kind=w.draft_kind)
            # drafted tokens: the library's draft-side sampler (tag-1 uniforms)
            self.toks = self.ver.draft_sample(self.draft[0], self.kpr, **self.knobs)
            rb = self.n_rot * step_bytes
            self.l2 = (f"{self.n_rot} rotating input copies ({rb / 1e6:.0f} MB) > L2"
                       if self.n_rot > 1 else
                       "L2 flushed between steps (a 256 MB write outside the per-step events)")
        self.flush = None
        if self.n_rot == 1 and not self.fused:
            self.flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
        self.out = None
        torch.cuda.synchronize()
        self.out = self.step(0)

    def step(self, i):
        c = i % self.n_rot
        return self.ver.run(self.target[c], self.draft[c], self.toks, self.kpr, out=self.out,
                            debug=False, w_vocab=self.wv, early_exit=self.early_exit,
                            **self.knobs)

    def kernel_and_bytes(self):
        """The dominant kernel, its algorithmic bytes per launch, flops (or None)."""
        w = self.w
        if self.fused:
            M = w.B * (w.K_max + 1)
            return ("k_lmhead", (w.hidden.size + w.w_vocab.size) * 2 + M * w.V * 4,
                    2.0 * M * self.H * w.V)
        if self.early_exit:
            # the rows actually read: target rows 0..j*, draft rows 0..min(j*, K_b - 1)
            na = self.out["num_accepted"].cpu().numpy().astype(np.int64)
            kb = w.k_per_row.astype(np.int64)
            es = 2 if w.dtype == "bf16" else 4
            d_rows = 0 if (w.draft_kind == "probs" or w.temperature == 0) else \
                int(np.minimum(na + 1, kb).sum())
            return "k_verify_exit", int((na + 1).sum() + d_rows) * w.V * es, None
        return _stage1_kernel(w), w.logit_bytes(), None

    def close(self):
        self.ver.close()


def timed_loop(arm, K, W, dist=None, per_step=False, sample_every=None):
    """W warm-up steps, then exactly K timed steps between a barrier and a
    synchronize on both sides.  The library's events around its stage-1
    kernel go on every sample_every-th step from step 1 on (at least 16 of
    them when K allows).  per_step: an event pair around every step and an L2
    flush between steps, outside the pairs (inputs smaller than L2)."""
    import ctypes
    import torch
    sv = arm.sv
    stream = arm.stream
    for i in range(max(3, W)):
        arm.step(i)
    if sample_every is None:
        sample_every = max(1, (K - 1) // 16)
    kev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for i in range(1 if K > 1 else 0, K, sample_every)}
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)] if per_step else []
    for a, b in list(kev.values()) + sev:  # torch creates the CUDA events on first record
        a.record(stream)
        b.record(stream)
    n_launch = ctypes.c_int32(0)
    sv.spec_verify_set_profiling(arm.ver.h, None, None, n_launch)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    launches = 0
    h0 = time.perf_counter()
    t_start.record(stream)
    for i in range(K):
        pair = kev.get(i)
        if per_step:
            arm.flush.zero_()
            sev[i][0].record(stream)
        if pair:
            sv.spec_verify_set_profiling(arm.ver.h, pair[0].cuda_event, pair[1].cuda_event, n_launch)
        arm.step(i)
        if pair:
            sv.spec_verify_set_profiling(arm.ver.h, None, None, n_launch)
        if per_step:
            sev[i][1].record(stream)
        launches += n_launch.value
    t_end.record(stream)
    host_s = time.perf_counter() - h0
    torch.cuda.synchronize()
    sv.spec_verify_set_profiling(arm.ver.h, None, None, None)
    if dist:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    if per_step:
        step_ms = [a.elapsed_time(b) for a, b in sev]
        total_ms = sum(step_ms)
    kern_ms = [a.elapsed_time(b) for a, b in kev.values()]
    return {"total_ms": total_ms, "kern_ms": kern_ms, "launches": launches,
            "host_us_per_step": 1e6 * host_s / K}


def _kstats(kern_ms):
    ks = sorted(kern_ms)
    return {"median_us": 1e3 * statistics.median(ks), "mean_us": 1e3 * statistics.fmean(ks),
            "min_us": 1e3 * ks[0], "max_us": 1e3 * ks[-1], "n": len(ks)}


def workload_summary(sv, torch, n, dev, local, steps, warmup, peak):
    """value, ms_per_step and the stage-1 kernel's fraction of one workload,
    timed like the headline (its own arm, warm-up and K steps)."""
    w = _workload(n)
    arm = Arm(sv, torch, w, dev, local)
    r = timed_loop(arm, steps, warmup, per_step=arm.flush is not None)
    kernel, bytes_step, flops = arm.kernel_and_bytes()
    ks = _kstats(r["kern_ms"])
    step_us = 1e3 * r["total_ms"] / steps
    d = {"workload": w.name, "value": w.rows() / (step_us * 1e-6), "unit": UNIT,
         "ms_per_step": step_us / 1e3, "kernel": kernel,
         "kernel_us_median": ks["median_us"], "launches_timed": ks["n"],
         "algorithmic_bytes_per_launch": bytes_step,
         "frac": bytes_step / (ks["median_us"] * 1e-6) / 1e9 / peak,
         "step_frac": bytes_step / (step_us * 1e-6) / 1e9 / peak, "l2": arm.l2,
         "gpu_launches": r["launches"]}
    if flops:
        d["tensor_frac"] = flops / (ks["median_us"] * 1e-6) / 1e12 / _tensor_peak()
        d.update(_verify_stage(arm, step_us, ks["median_us"], peak))
    arm.close()
    del arm
    torch.cuda.empty_cache()
    return d


def _verify_stage(arm, step_us, lm_us, peak):
    """The fused round's verify stage (the step without the LM head) against
    the bytes it reads: the LM head's softmax partials, the logits and draft
    probabilities at the drafted tokens, and the rows the sample reads (the
    target row j* and the draft row j* after a rejection, the bonus row
    otherwise)."""
    w = arm.w
    na = arm.out["num_accepted"].cpu().numpy().astype(np.int64)
    kb = w.k_per_row.astype(np.int64)
    rej = na < kb
    rows_read = int((1 + rej).sum())
    nseg = -(-w.V // 256)
    stats = int((kb + 1).sum()) * nseg * 16
    at_tokens = int(kb.sum()) * 2 * 4
    vb = rows_read * w.V * 4 + stats + at_tokens
    v_us = step_us - lm_us
    return {"verify_stage": {
        "us": v_us, "bytes_read": vb, "achieved_gbs": vb / (v_us * 1e-6) / 1e9,
        "frac": vb / (v_us * 1e-6) / 1e9 / peak,
        "note": "step minus the LM head's median launch; bytes: the LM head's softmax partials, "
                "the values at the drafted tokens and the sampled rows (latency-bound)"}}


def run_gpu(args):
    import torch
    import speculative_decoding_verification_42_gb300 as sv

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    sv.load_library()
    w = _workload(args.config, args.batch)
    try:
        gpu_sel = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_sel = str(local)
    # the clock sampler starts before the warm-up, so that no idle gap sits
    # between the warm-up and the timed steps
    sampler = ClockSampler(gpu_sel) if rank == 0 else None
    if sampler:
        sampler.start()
    arm = Arm(sv, torch, w, dev, local, early_exit=args.early_exit)
    K = args.steps
    r = timed_loop(arm, K, args.warmup, dist=dist)
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(r["total_ms"], dist, dev)
    kern_ms = r["kern_ms"]
    ks = _kstats(kern_ms)
    mean_step_ms = r["total_ms"] / K
    rows = w.rows()
    value = whole_job_rate(rows, K, world, total_ms)
    peak, peak_src = _peaks()
    kernel, bytes_step, flops = arm.kernel_and_bytes()
    achieved = bytes_step / (ks["median_us"] * 1e-6) / 1e9

    # end to end: host buffers through the same call, copies inside the timed
    # region; the inputs go in as E2E_STREAMS slices of each tensor on as many
    # copy streams (several copy engines at once), the compute stream waits
    # for all of them
    e2e = None
    if args.e2e_steps > 0:
        out = arm.out
        target, draft, toks, kpr = arm.target, arm.draft, arm.toks, arm.kpr
        stream = arm.stream
        h_target = torch.empty(target[0].shape, dtype=target[0].dtype, pin_memory=True)
        h_draft = torch.empty(draft[0].shape, dtype=draft[0].dtype, pin_memory=True)
        h_target.copy_(target[0])
        h_draft.copy_(draft[0])
        h_toks = toks.cpu().pin_memory()
        h_kpr = kpr.cpu().pin_memory()
        h_out_t = torch.empty(out["tokens"].shape, dtype=torch.int32, pin_memory=True)
        h_out_n = torch.empty(out["num_accepted"].shape, dtype=torch.int32, pin_memory=True)
        d_toks = torch.empty_like(toks)
        d_kpr = torch.empty_like(kpr)
        cs = [torch.cuda.Stream(dev) for _ in range(E2E_STREAMS)]
        nrot = max(2, arm.n_rot)
        tgt = target if len(target) >= 2 else target * 2
        drf = draft if len(draft) >= 2 else draft * 2
        ready = [torch.cuda.Event() for _ in range(E2E_STREAMS)]
        done = [torch.cuda.Event() for _ in range(nrot)]

        def slices(t):
            flat = t.reshape(-1)
            n = -(-flat.numel() // E2E_STREAMS)
            return [flat[k * n:(k + 1) * n] for k in range(E2E_STREAMS)]

        h_slices = list(zip(slices(h_target), slices(h_draft)))
        d_slices = [list(zip(slices(tgt[c]), slices(drf[c]))) for c in range(nrot)]

        def e2e_step(i):
            c = i % nrot
            # the copies into buffer c wait for the step that last read it
            for k, s in enumerate(cs):
                s.wait_event(done[c])
                with torch.cuda.stream(s):
                    for dst, src in zip(d_slices[c][k], h_slices[k]):
                        dst.copy_(src, non_blocking=True)
                    if k == 0:
                        d_toks.copy_(h_toks, non_blocking=True)
                        d_kpr.copy_(h_kpr, non_blocking=True)
                ready[k].record(s)
            for ev in ready:
                stream.wait_event(ev)
            o = arm.ver.run(tgt[c], drf[c], d_toks, d_kpr, out=out, debug=False,
                            w_vocab=arm.wv, **arm.knobs)
            done[c].record(stream)
            h_out_t.copy_(o["tokens"], non_blocking=True)
            h_out_n.copy_(o["num_accepted"], non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for s in cs:
            s.wait_event(a)
        for i in range(args.e2e_steps):
            e2e_step(i)
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        h2d = (h_target.numel() * h_target.element_size() + h_draft.numel() * h_draft.element_size()
               + h_toks.numel() * 4 + h_kpr.numel() * 4)
        d2h = h_out_t.numel() * 4 + h_out_n.numel() * 4
        e2e = {"value": whole_job_rate(rows, args.e2e_steps, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps, "ms_per_step": e_ms / args.e2e_steps,
               "copies": f"target and draft in {E2E_STREAMS} slices each on {E2E_STREAMS} copy streams, "
                         f"{nrot} device buffers"}

    fused = arm.fused
    verify_stage = _verify_stage(arm, 1e3 * mean_step_ms, ks["median_us"], peak) if fused else {}
    toks_np = arm.toks.cpu().numpy()
    draft0 = arm.draft[0].cpu().numpy() if fused else None
    l2_note = arm.l2
    arm.close()
    del arm
    torch.cuda.empty_cache()

    others = None
    if rank == 0 and world == 1 and not args.no_others and not args.batch and not args.early_exit:
        others = {}
        for n in (1, 2, 3, 4, 5):
            if n == args.config:
                continue
            others[str(n)] = workload_summary(sv, torch, n, dev, local, K, args.warmup, peak)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        if fused:
            cpu = cpu_baseline_fused(w, draft0, toks_np, seconds_target=args.cpu_seconds)
        else:
            cpu = cpu_baseline(w, toks_np, seconds_target=args.cpu_seconds)
    cfg = _wl_config(w, ROTATE)
    cfg["config_id"] = args.config
    cfg["l2"] = l2_note
    if args.batch:
        cfg["workload"] += f" (B overridden to {w.B})"
    if args.early_exit:
        cfg["mode"] = ("early exit: rows read only up to each sequence's first rejection; "
                       "roofline bytes are the rows read")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        # the arithmetic type of the path (bf16 inputs are widened exactly);
        # the inputs' type is config.input_dtype
        "dtype": "f32",
        "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "traffic": _traffic(kernel, w),
                     "algorithmic_bytes_per_launch": bytes_step,
                     "launch_us": ks,
                     "launches_timed": ks["n"],
                     "step_us": mean_step_ms * 1e3,
                     "step_frac": bytes_step / (mean_step_ms / 1e3) / 1e9 / peak,
                     "host_enqueue_us_per_step": r["host_us_per_step"]},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": r["launches"],
        "clocks": clocks,
    }
    line.update(verify_stage)
    if flops:
        tf = _tensor_peak()
        line["roofline"]["tensor"] = {
            "achieved_tflops": flops / (ks["median_us"] * 1e-6) / 1e12, "peak_tflops": tf,
            "frac": flops / (ks["median_us"] * 1e-6) / 1e12 / tf if tf else None,
            "flops_per_launch": flops,
            "peak_source": "measured bf16_tflops (MEASURED_PEAKS.json), burst"}
    if others is not None:
        line["workloads"] = others
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seq", type=int, default=1,
                    help="reference arm: sequences verified by the oracle per step")
    ap.add_argument("--early-exit", action="store_true",
                    help="time spec_verify_run_early_exit (top-k rows of logits)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's B")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the per-workload summaries of the other four workloads")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: stop the timed loop after this much oracle time")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
