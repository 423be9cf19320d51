"""Benchmark of the quantized-KV decode layer-step on GB300.

Headline workload (N=1, the largest single-GPU configuration): Llama-3-8B-
shaped grouped-query decode layer, batch 64, 32 query / 8 KV heads,
head_dim 128, 32768 cached tokens, K2V2 (keys per channel over 32-token
groups, values per token over 32-channel groups), fp16 residual R = 128,
one seeded key channel per kv head x15.  One step = one layer-step of the
whole hot path:
  a2  kv_quant_value  on the B*Hkv value tokens leaving the fp16 window,
  a1  kv_quant_key    on the amortized key flush (1/R of the (b, kv head)
                      pairs flush their R/G groups each step),
  a3  decode stage 1  (split-KV attention over quantized + fp16 segments),
  a4  decode merge    (LSE merge, fp16 out).
`value` is microseconds per layer-step (whole job: time / (steps * N)),
inputs resident in HBM, the K steps captured into a CUDA graph and timed
over one replay; the roofline's stage-1 time comes from the same kind of
replay of a graph of K stage-1 launches.  `e2e` is the same metric through
the C ABI with the step's inputs copied from pinned host memory and the
output copied back inside the timed region, the copies launched per step
from the host and each step's kernels replayed as one CUDA graph.  At N=1
the other workloads (the MHA layer, the mixed-key layer in both boost
selections, the INT8 dither layer, the tiny case) are measured the same way
and reported under `configs`.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from bit_kv_cache_keyquant_gb300 import inputs as I  # noqa: E402

METRIC = "quantized-KV decode attention: us/layer-step and HBM GB/s (% of GB300 peak)"
UNIT = "us/layer-step"


# Pure Philox4x32-10 throughput of this GPU (blocks of 4 words per second): a probe kernel running the
# decode kernels' Philox form (round keys precomputed, 32x32->64 products) over 152 x 8 CTAs x 256 threads
# x 4 independent streams, CUDA events, 2070 MHz: 519.2 G blocks/s, i.e. 1.65 blocks (33 wide products)
# per clock per SM.  The INT8 decode paths are bound by this arithmetic, not by HBM.
PHILOX_PEAK_GBLOCKS = 519.2


def philox_blocks(w, lens) -> int:
    """Philox4x32-10 blocks one INT8 decode launch must run: one per (quantized token, kv head, side,
    4 channels)."""
    if w.variant == "int8":
        T = 256
        nq = sum(int(L) - ((int(L) - 1) % T + 1) for L in lens)
    else:
        nq = sum(int(L) for L in lens)
    return nq * w.n_kv_heads * 2 * (128 // 4)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _workload_desc(w):
    base = f"{w.name}: batch {w.batch}, {w.n_q_heads} query / {w.n_kv_heads} KV heads, head_dim 128, "
    if w.variant == "kivi":
        return base + (f"{w.seq_len} cached tokens, K{w.bits_k}V{w.bits_v} (key per-channel G=32, value per-token "
                       f"Gv=32), R=128" + (", paged: 128-token pages in a hashed order from a shared pool"
                                           if w.paged else ""))
    if w.variant == "kitty":
        sel = "by variance over the page (score_mode 1)" if w.score_mode else "by the Eq. 2 sum of |x| (score_mode 0)"
        return base + (f"{w.seq_len} cached tokens, Kitty pages G=128, 16 of 128 key channels boosted to 4 bit "
                       f"{sel} (two 2-bit planes), value 2 bit, sink 32, local 128")
    if w.variant == "int8t":
        return base + (f"lengths U[{w.min_seq_len}, {w.seq_len}], token-granular INT8 slot pool (scattered 16-slot "
                       f"pages), fp16 scale per token and 32 channels, Philox4x32-10 dither keyed by slot, "
                       f"one token appended per request per step")
    return base + (f"lengths U[{w.min_seq_len}, {w.seq_len}], INT8 K and V with Philox4x32-10 subtractive dither, "
                   f"fp16 scale per 256-token block and channel, fp16 active block")


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for ln in out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
_PAIRS = {}     # per process: (workload, batch row, kv head) -> the pair's quantized cache, built once


def _pair(w, b, h):
    """The oracle's cache of one (batch row, kv head) of workload w and the value token that leaves the fp16
    window this step (built on first use, outside any timing)."""
    from oracle import oracle as O
    key = (w, b, h)
    if key not in _PAIRS:
        L = w.seq_len
        K = I.gen_kv_np(w, I.T_K, b, h, L)
        V = I.gen_kv_np(w, I.T_V, b, h, L)
        _PAIRS[key] = (V[L - 129:L - 128].copy(), O.kivi_build_one(K, V, bits_k=w.bits_k, bits_v=w.bits_v))
    return _PAIRS[key]


def oracle_step_seconds(w, budget_s: float, min_pairs: int = 4, seed: int = 0):
    """Time the oracle's layer-step on a bounded sample of (b, kv head) pairs.

    Per pair: quantize the value token leaving the fp16 window, then split-free
    fp64 attention of the pair's query heads over the quantized cache and the
    fp16 residual.  The sample is the seed's shuffle of the pairs; each pair's
    cache is built once per process.  Returns (seconds per pair, pairs timed)."""
    from oracle import oracle as O
    O.build()
    g = w.n_q_heads // w.n_kv_heads
    q = I.gen_q_np(w)
    L = w.seq_len
    pairs = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    rng = np.random.default_rng(seed)
    rng.shuffle(pairs)
    spent, n = 0.0, 0
    for b, h in pairs:
        vtok, parts = _pair(w, b, h)
        t0 = time.perf_counter()
        O.kivi_quant_value(vtok, 32, w.bits_v)
        O.kivi_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, bits_k=w.bits_k, bits_v=w.bits_v)
        spent += time.perf_counter() - t0
        n += 1
        if n >= min_pairs and spent >= budget_s:
            break
    return spent / n, n


def _oracle_worker(job):
    """One host process of the all-cores CPU leg (a spawned process: it never touches the GPU)."""
    w, budget_s, min_pairs, seed = job
    return oracle_step_seconds(w, budget_s, min_pairs, seed)


def oracle_pool(procs: int = 0):
    """A pool of spawned host processes for the all-cores CPU leg (spawned, not forked: the parent
    may already hold a CUDA context)."""
    import multiprocessing as mp
    from oracle import oracle as O
    O.build()                                          # once, before the workers load it
    procs = procs or (os.cpu_count() or 1)
    return mp.get_context("spawn").Pool(procs), procs


def oracle_step_seconds_all_cores(w, budget_s: float, pool, procs: int, seed: int = 1):
    """The oracle on every host core at once: `procs` processes, each timing its own shuffled sample of
    (b, kv head) pairs for about budget_s / procs seconds.  Returns (layer-step seconds at the aggregate
    throughput, pairs timed)."""
    jobs = [(w, budget_s / procs, 2, seed + i) for i in range(procs)]
    res = pool.map(_oracle_worker, jobs, chunksize=1)
    rate = sum(1.0 / per_pair for per_pair, _ in res)  # pairs per second, all processes together
    return w.batch * w.n_kv_heads / rate, sum(n for _, n in res)


def run_reference(args, w):
    """The oracle on every host core: one pool of spawned processes, warm-up steps, then K timed steps,
    each a bounded sample of the workload's (b, kv head) pairs at the processes' summed throughput."""
    pool, procs = oracle_pool()
    with pool:
        # the warm-up steps build every process's sample pairs; the timed steps time the same samples
        for i in range(max(1, args.warmup)):
            oracle_step_seconds_all_cores(w, 0.0, pool, procs, seed=1)
        times, npairs = [], 0
        for i in range(args.steps):
            step_s, n = oracle_step_seconds_all_cores(w, 0.1 * procs, pool, procs, seed=1)
            times.append(step_s)
            npairs += n
    us = statistics.median(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(w), "batch": w.batch, "seq_len": w.seq_len},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": procs, "kind": "oracle",
                         "sample": f"{npairs} (batch row, kv head) pairs over {args.steps} steps on {procs} spawned "
                                   f"processes at once; each step is the median step's layer-step at the processes' "
                                   f"summed throughput ({w.batch * w.n_kv_heads} pairs per layer-step)"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def build_state(w, device, appends: int = 1024):
    """Device-resident cache of the workload plus the per-step write-side inputs."""
    import torch
    from bit_kv_cache_keyquant_gb300 import cache as C
    from bit_kv_cache_keyquant_gb300 import kvq
    lens = I.seq_lens(w)
    Lmax = int(lens.max())
    if w.variant == "kivi" and w.paged:
        cfg = kvq.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, bits_k=w.bits_k, bits_v=w.bits_v)
        n_pages = int(sum((int(L) + 127) // 128 for L in lens)) + 64
        cache = C.KiviPagedCache(cfg, w.batch, Lmax, n_pages, device=device)
        cache.shuffle_free(I.page_permutation(w, n_pages))
        variant = kvq.KVQ_VARIANT_KIVI_PAGED
    elif w.variant == "kivi":
        cfg = kvq.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, bits_k=w.bits_k, bits_v=w.bits_v)
        cache = C.KiviCache(cfg, w.batch, Lmax, device=device)
        variant = kvq.KVQ_VARIANT_KIVI
    elif w.variant == "kitty":
        cfg = kvq.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, group_k=128, sink=32, residual=128,
                              boost_k=16)
        cache = C.KittyCache(cfg, w.batch, Lmax, device=device)
        variant = kvq.KVQ_VARIANT_KITTY
    elif w.variant == "int8t":
        cfg = kvq.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, int8_group=32)
        margin = (appends + 15) // 16 * 16                                  # tokens appended per request, at most
        n_slots = (int(lens.sum()) + w.batch * margin + 15) // 16 * 16
        cache = C.Int8TokenCache(cfg, w.batch, Lmax + margin, n_slots, layer=5, seed=w.seed, device=device)
        cache.shuffle_free(I.page_permutation(w, n_slots // 16), 16)
        variant = kvq.KVQ_VARIANT_INT8_TOKEN
    else:
        cfg = kvq.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads)
        cache = C.Int8Cache(cfg, w.batch, Lmax, layer=5, seed=w.seed, device=device)
        variant = kvq.KVQ_VARIANT_INT8
    reqs = I.request_ids(w)
    for b in range(w.batch):
        if w.variant == "int8t" or (w.variant == "kivi" and w.paged):
            L = int(lens[b])
            if w.variant == "kivi":
                cache.fill(b, torch.stack([I.gen_kv_torch(w, I.T_K, b, h, L, device) for h in range(w.n_kv_heads)]),
                           torch.stack([I.gen_kv_torch(w, I.T_V, b, h, L, device) for h in range(w.n_kv_heads)]))
                continue
            cache.fill(b, torch.stack([I.gen_kv_torch(w, I.T_K, b, h, L, device) for h in range(w.n_kv_heads)], 1),
                       torch.stack([I.gen_kv_torch(w, I.T_V, b, h, L, device) for h in range(w.n_kv_heads)], 1))
            continue
        L = int(lens[b])
        for h in range(w.n_kv_heads):
            K = I.gen_kv_torch(w, I.T_K, b, h, L, device)
            V = I.gen_kv_torch(w, I.T_V, b, h, L, device)
            if w.variant == "int8":
                cache.fill(b, h, K, V, int(reqs[b]))
            elif w.variant == "kitty":
                cache.fill(b, h, K, V, score_mode=w.score_mode)
            else:
                cache.fill(b, h, K, V)
    q = I.gen_q_torch(w, device)
    pairs = w.batch * w.n_kv_heads
    st = dict(w=w, cfg=cfg, cache=cache, desc=cache.desc(), q=q, lens=lens, variant=variant)
    # per-step write-side inputs (the amortized quantization work of one decode step)
    if w.variant == "kivi":
        n_vtok = pairs                                                      # one value token per (b, kv head)
        n_kgrp = max(1, pairs * (cfg.residual // cfg.group_k) // cfg.residual)   # 1/R of the key flushes
        st.update(n_vtok=n_vtok, n_kgrp=n_kgrp,
                  vnew=I.gen_slice_torch(w.seed, I.T_V, 9999, 0, n_vtok, 128, device),
                  knew=I.gen_slice_torch(w.seed, I.T_K, 9999, 1, n_kgrp * cfg.group_k, 128, device),
                  scratch=[torch.empty(((n_vtok + 31) // 32 * 32, 128 * w.bits_v // 8), dtype=torch.uint8, device=device),
                           torch.empty((n_vtok, 128 // cfg.group_v), dtype=torch.int32, device=device),
                           torch.empty((n_kgrp, cfg.group_k * 128 * w.bits_k // 8), dtype=torch.uint8,
                                       device=device),
                           torch.empty((n_kgrp, 128), dtype=torch.int32, device=device)])
    elif w.variant == "kitty":
        n_pg = max(1, pairs // 128)                                         # 1/G of the page flushes
        st.update(n_pg=n_pg, knew=I.gen_slice_torch(w.seed, I.T_K, 9999, 1, n_pg * 128, 128, device),
                  vnew=I.gen_slice_torch(w.seed, I.T_V, 9999, 0, n_pg * 128, 128, device),
                  scratch=[torch.empty((n_pg, kvq.kvq_kitty_key_page_bytes(cfg)), dtype=torch.uint8, device=device),
                           torch.empty((n_pg, kvq.kvq_kitty_value_page_bytes(cfg)), dtype=torch.uint8,
                                       device=device)])
    elif w.variant == "int8t":
        # one new token per request, appended (slot from the pool, quantized) before the attention reads it
        st.update(pool=cache.pool(),
                  knew=I.gen_slice_torch(w.seed, I.T_K, 9999, 1, pairs, 128, device).view(w.batch, w.n_kv_heads, 128),
                  vnew=I.gen_slice_torch(w.seed, I.T_V, 9999, 0, pairs, 128, device).view(w.batch, w.n_kv_heads, 128))
    else:
        n_blk = max(1, (pairs + 255) // 256)                                # 1/T of the block flushes, rounded up
        st.update(n_blk=n_blk, knew=I.gen_slice_torch(w.seed, I.T_K, 9999, 1, n_blk * 256, 128, device),
                  vnew=I.gen_slice_torch(w.seed, I.T_V, 9999, 0, n_blk * 256, 128, device),
                  blk_meta=[torch.zeros(n_blk, dtype=torch.int32, device=device) for _ in range(3)],
                  scratch=[torch.empty((n_blk, 256, 128), dtype=torch.int8, device=device),
                           torch.empty((n_blk, 128), dtype=torch.float16, device=device)])
    n_splits, wsb = kvq.kv_decode_attn_plan(cfg, variant, w.batch, Lmax)
    st.update(ws=torch.empty(wsb, dtype=torch.uint8, device=device), wsb=wsb, n_splits=n_splits,
              out=torch.empty((w.batch, w.n_q_heads, 128), dtype=torch.float16, device=device), Lmax=Lmax)
    torch.cuda.synchronize()
    return st


def quant_step(st, stream, vnew=None, knew=None):
    """The step's write-side kernels (amortized quantization of the new tokens)."""
    from bit_kv_cache_keyquant_gb300 import kvq
    w, cfg, sc = st["w"], st["cfg"], st.get("scratch")
    vnew = st["vnew"] if vnew is None else vnew
    knew = st["knew"] if knew is None else knew
    if w.variant == "kivi":
        kvq.kv_quant_value(cfg, vnew, st["n_vtok"], sc[0], sc[1], stream)
        kvq.kv_quant_key(cfg, knew, st["n_kgrp"], sc[2], sc[3], stream)
    elif w.variant == "kitty":
        kvq.kv_quant_key_kitty(cfg, knew, st["n_pg"], w.score_mode, sc[0], stream)
        kvq.kv_quant_value_kitty(cfg, vnew, st["n_pg"], sc[1], stream)
    elif w.variant == "int8t":
        kvq.kv_append_int8_token(cfg, st["desc"], st["pool"], knew, vnew, stream)
    else:
        m = st["blk_meta"]
        for sel, x in ((0, knew), (1, vnew)):
            kvq.kv_quant_int8_dither(cfg, x, st["n_blk"], m[0], m[1], m[2], 5, sel, w.seed, sc[0], sc[1], stream)


def decode_step(st, stream, ev=None, q=None, vnew=None, knew=None, out=None):
    """One layer-step.  The write side (quantizing the tokens that leave the
    fp16 window) runs on a second stream beside the attention: in the
    insert -> attend -> quantize order it reads only the new tokens and writes
    cache slots that this step's attention does not read.  It is forked at the
    start of the step but enqueued after stage 1, so that stage 1's persistent
    grid takes every SM first and the small write-side grids run on SMs as
    stage-1 CTAs drain (enqueued first, they held some SMs while stage 1
    started, and the CTAs that started late ended the kernel late: 4 us per
    step on the MHA layer, 4-19 us on the grouped-query one).  The
    token-granular INT8 cache quantizes on insert: its append precedes the
    attention on the same stream."""
    from bit_kv_cache_keyquant_gb300 import kvq
    cfg, side = st["cfg"], st["side"]
    insert_first = st["w"].variant == "int8t"
    if insert_first:
        side = stream

    def write_side():
        if ev is not None:
            ev[0].record(side)
        quant_step(st, side, vnew, knew)
        if ev is not None:
            ev[1].record(side)
        st["join"].record(side)

    st["fork"].record(stream)
    side.wait_event(st["fork"])
    if insert_first:
        write_side()
    if ev is not None:
        ev[2].record(stream)
    kvq.kv_decode_attn_stage1(cfg, st["variant"], st["desc"], st["q"] if q is None else q, st["ws"], st["wsb"],
                              stream)
    if ev is not None:
        ev[3].record(stream)
    if not insert_first:
        write_side()
    kvq.kv_decode_attn_merge(cfg, st["variant"], st["cache"].batch, st["cache"].max_seq_len, st["ws"], st["wsb"],
                             st["out"] if out is None else out, stream)
    if ev is not None:
        ev[4].record(stream)
    stream.wait_event(st["join"])


def quant_kernels_bench(w, cfg, dev, stream, reps: int = 10):
    """The workload's quantization kernels on their own, outside the timed step, at 256 MB of fp16 input
    per call (twice the L2): us per call, HBM GB/s of the bytes each call must move (fp16 input read,
    codes and scales written) against the measured copy peak, and the call's time amortized over a
    layer-step: the units one decode step needs on average (one value token per (row, kv head); a key
    flush of R/G groups every R steps; a Kitty key and value page every 128 steps; an INT8 block per side
    every 256 steps), times the time per unit."""
    import torch
    from bit_kv_cache_keyquant_gb300 import kvq
    peak, _ = _peaks()
    total = 256 << 20
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    pairs = w.batch * w.n_kv_heads

    def entry(us, units, unit, nbytes, per_step):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us_per_call": us, "units": units, "unit": unit, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak,
                "units_per_step": per_step, "amortized_us_per_step": us * per_step / units}

    x = torch.randn(total // 2, generator=gen, device=dev).half()
    out = {}
    with torch.cuda.stream(stream):
        if w.variant == "kivi":
            G, Gv = cfg.group_k, cfg.group_v
            ng = total // (G * 128 * 2)
            kc = torch.empty(ng * G * 128 * w.bits_k // 8, dtype=torch.uint8, device=dev)
            ks = torch.empty((ng, 128), dtype=torch.int32, device=dev)
            us = timed(lambda: kvq.kv_quant_key(cfg, x, ng, kc, ks, stream))
            out["kv_quant_key"] = entry(us, ng, f"{G}-token key groups", total + kc.numel() + ks.numel() * 4,
                                        pairs / G)
            nt = total // 256
            vc = torch.empty((nt + 31) // 32 * 32 * 128 * w.bits_v // 8, dtype=torch.uint8, device=dev)   # whole tiles
            vs = torch.empty((nt, 128 // Gv), dtype=torch.int32, device=dev)
            us = timed(lambda: kvq.kv_quant_value(cfg, x, nt, vc, vs, stream))
            out["kv_quant_value"] = entry(us, nt, "value tokens", total + vc.numel() + vs.numel() * 4, pairs)
        elif w.variant == "kitty":
            npg = total // (128 * 128 * 2)
            kp = torch.empty(npg * kvq.kvq_kitty_key_page_bytes(cfg), dtype=torch.uint8, device=dev)
            us = timed(lambda: kvq.kv_quant_key_kitty(cfg, x, npg, w.score_mode, kp, stream))
            out["kv_quant_key_kitty"] = entry(us, npg, "128-token key pages", total + kp.numel(), pairs / 128)
            out["kv_quant_key_kitty"]["score_mode"] = w.score_mode
            vp = torch.empty(npg * kvq.kvq_kitty_value_page_bytes(cfg), dtype=torch.uint8, device=dev)
            us = timed(lambda: kvq.kv_quant_value_kitty(cfg, x, npg, vp, stream))
            out["kv_quant_value_kitty"] = entry(us, npg, "128-token value pages", total + vp.numel(), pairs / 128)
        elif w.variant == "int8":
            nb = total // (256 * 128 * 2)
            blk = torch.arange(nb, dtype=torch.int32, device=dev)
            meta = [blk // w.n_kv_heads, blk % w.n_kv_heads, 256 * (blk // w.n_kv_heads)]   # request, kv head, tok0
            codes = torch.empty(nb * 256 * 128, dtype=torch.int8, device=dev)
            scale = torch.empty((nb, 128), dtype=torch.float16, device=dev)
            us = timed(lambda: kvq.kv_quant_int8_dither(cfg, x, nb, meta[0], meta[1], meta[2], 5, 0, w.seed, codes,
                                                        scale, stream))
            out["kv_quant_int8_dither"] = entry(us, nb, "256-token blocks", total + codes.numel() + scale.numel() * 2,
                                                2 * pairs / 256)
    torch.cuda.synchronize()
    return out


def launches_per_step(w) -> int:
    return {"kivi": 4, "kitty": 4, "int8": 4, "int8t": 4}[w.variant]


def job_time_ms(local_ms: float, world: int, device=None) -> float:
    """The job's timed-region length: the max over ranks of each rank's (one collective, the only one)."""
    if world == 1:
        return local_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_step(job_ms: float, steps: int, world: int) -> float:
    """us per layer-step of the whole job: `world` replicas each ran `steps` layer-steps in job_ms."""
    return job_ms * 1e3 / (steps * world)


def measure(args, w, rank, world, local_rank, steps: int, want_quant: bool = True, want_cpu: bool = True):
    """Time workload w on this rank: the step, its stage 1 and the write side, e2e through host buffers.
    Returns the measurement (rank 0; None on the other ranks)."""
    import torch
    import torch.distributed as dist
    from bit_kv_cache_keyquant_gb300 import kvq

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    st = build_state(w, dev, appends=2 * args.warmup + 4 * steps + 16)
    stream = torch.cuda.current_stream(dev)
    st["side"] = torch.cuda.Stream(device=dev)
    st["fork"], st["join"] = torch.cuda.Event(), torch.cuda.Event()

    # ---- kernel-only timing: inputs resident in HBM (every workload but the tiny one reads more than the
    #      129 MB L2 per step) ----
    for _ in range(args.warmup):
        decode_step(st, stream)
    torch.cuda.synchronize()
    # The K timed steps are captured once into a CUDA graph and replayed, as a serving loop would run
    # them: the library's calls are stream-ordered, allocate nothing and never synchronize, so they
    # capture as they are (the merge's programmatic early launch becomes a programmatic graph edge).
    # One untimed replay uploads the graph; the timed replay runs exactly K steps with no host launch
    # between them and no event between their kernels.  A second graph holds K stage-1 launches alone:
    # its replay, timed the same way, gives the stage-1 duration of the roofline.
    gs = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for i in range(steps):
            decode_step(st, gs)
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=gs):
        for i in range(steps):
            kvq.kv_decode_attn_stage1(st["cfg"], st["variant"], st["desc"], st["q"], st["ws"], st["wsb"], gs)
    with torch.cuda.stream(gs):
        graph.replay()
        g1.replay()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with Clocks(local_rank) as clk:
        ev[0].record(gs)
        with torch.cuda.stream(gs):
            graph.replay()
        ev[1].record(gs)
        torch.cuda.synchronize()
        ev[2].record(gs)
        with torch.cuda.stream(gs):
            g1.replay()
        ev[3].record(gs)
        torch.cuda.synchronize()
        # a third pass of K steps, launched one by one with events around every kernel: the per-kernel
        # breakdown (the write side's span and the merge)
        for i in range(steps):
            decode_step(st, stream, evs[i])
        torch.cuda.synchronize()
    total_ms = ev[0].elapsed_time(ev[1])
    s1 = ev[2].elapsed_time(ev[3]) / steps
    stage1_evt_ms = [e[2].elapsed_time(e[3]) for e in evs]
    quant_ms = [e[0].elapsed_time(e[1]) for e in evs]
    merge_ms = [e[3].elapsed_time(e[4]) for e in evs]
    assert kvq.kvq_get_device_error() == 0
    total_ms = job_time_ms(total_ms, world, dev)
    ms_per_step = total_ms / steps

    # ---- end to end through the C ABI with host buffers: every step copies its inputs from pinned host
    #      memory and reads its output back; a serving loop overlaps these copies with the neighbouring
    #      steps' compute (inputs of step i+1 and the output of step i on two copy streams, two device
    #      buffer sets) ----
    qh = st["q"].cpu().pin_memory()
    vh = st["vnew"].cpu().pin_memory()
    kh = st["knew"].cpu().pin_memory()
    outh = [torch.empty(st["out"].shape, dtype=torch.float16).pin_memory() for _ in range(2)]
    bufs = [dict(q=torch.empty_like(st["q"]), v=torch.empty_like(st["vnew"]), k=torch.empty_like(st["knew"]),
                 out=torch.empty_like(st["out"])) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_free = [torch.cuda.Event() for _ in range(2)]      # the step that read buffer set s has finished
    in_ready = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer set s copied
    out_free = [torch.cuda.Event() for _ in range(2)]     # output of buffer set s read back

    # each buffer set's decode step is captured once into a CUDA graph (kernels only; the copies stay on
    # the copy streams, launched per step from the host)
    step_graphs = []
    for kk in range(2):
        gk = torch.cuda.CUDAGraph()
        bk = bufs[kk]
        with torch.cuda.graph(gk, stream=gs):
            decode_step(st, gs, q=bk["q"], vnew=bk["v"], knew=bk["k"], out=bk["out"])
        step_graphs.append(gk)
    torch.cuda.synchronize()

    def e2e_step(i):
        k = i % 2
        b = bufs[k]
        h2d_s.wait_event(in_free[k])
        with torch.cuda.stream(h2d_s):
            b["q"].copy_(qh, non_blocking=True)
            b["v"].copy_(vh, non_blocking=True)
            b["k"].copy_(kh, non_blocking=True)
        in_ready[k].record(h2d_s)
        stream.wait_event(in_ready[k])
        stream.wait_event(out_free[k])
        with torch.cuda.stream(stream):
            step_graphs[k].replay()
        in_free[k].record(stream)
        d2h_s.wait_event(in_free[k])
        with torch.cuda.stream(d2h_s):
            outh[k].copy_(b["out"], non_blocking=True)
        out_free[k].record(d2h_s)

    # the copies launched step by step from the host (a graph of the K steps with their copies measured
    # 7-35 us per step slower on the large workloads: its copies did not overlap the neighbouring steps'
    # kernels as the stream-launched ones do; on the tiny workload 1, whose steps are host-launch bound,
    # it gave 17 us per step, the per-step graphs 57 and step-by-step launches 78)
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    for i in range(steps):
        e2e_step(i)
    stream.wait_event(out_free[(steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = job_time_ms(e0.elapsed_time(e1), world, dev)
    h2d = qh.numel() * 2 + vh.numel() * 2 + kh.numel() * 2
    d2h = outh[0].numel() * 2

    quant = quant_kernels_bench(w, st["cfg"], dev, stream) if (rank == 0 and want_quant) else None
    if rank != 0:
        return None
    lens = st["lens"]
    if w.variant == "int8t":       # one token appended per request before every attention
        lens = lens + args.warmup + steps                                  # at the stage-1 graph's replay
    cache_bytes = st["cache"].nbytes_read(lens)
    q_bytes = w.batch * w.n_q_heads * 128 * 2
    alg_bytes_stage1 = cache_bytes + q_bytes
    achieved = alg_bytes_stage1 / (s1 * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    traffic = None
    kname, kfiles = stage1_kernel(w)
    if os.path.exists(prof):
        tr = json.load(open(prof)).get(f"{kname}@workload{w.index}")
        if tr and tr.get("source_hash") == kernel_source_hash(kfiles):
            traffic = tr["bytes_per_launch"]
    timing = f"a CUDA graph of {steps} stage-1 launches, one timed replay (CUDA events on its stream)"
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_kind": peak_kind, "kernel": kname + " (stage 1)",
            "alg_bytes_per_launch": alg_bytes_stage1, "stage1_us": 1e3 * s1, "stage1_timing": timing}
    if w.variant in ("int8", "int8t"):
        nb = philox_blocks(w, lens)
        ach = nb / (s1 * 1e-3) / 1e9
        roof = {"bound": "alu", "achieved": ach, "peak": PHILOX_PEAK_GBLOCKS, "unit": "G Philox4x32-10 blocks/s",
                "frac": ach / PHILOX_PEAK_GBLOCKS, "traffic": traffic,
                "peak_kind": "measured (pure Philox4x32-10 probe kernel on this GPU)",
                "kernel": kname + " (stage 1)", "alg_philox_blocks_per_launch": nb,
                "alg_bytes_per_launch": alg_bytes_stage1, "hbm_gbs": achieved, "hbm_frac": achieved / peak,
                "stage1_us": 1e3 * s1, "stage1_timing": timing}
    cpu = None
    if world == 1 and want_cpu and not args.no_cpu and w.variant == "kivi":
        # the oracle on every host core (the reference arm's form), and on one thread
        pool, procs = oracle_pool()
        with pool:
            step_s, n_all = oracle_step_seconds_all_cores(w, args.cpu_budget, pool, procs)
        per_pair, n = oracle_step_seconds(w, args.cpu_budget / 2)
        cpu = {"value": step_s * 1e6, "unit": UNIT, "cores": procs, "kind": "oracle",
               "sample": f"{n_all} (batch row, kv head) pairs of the workload over {procs} spawned processes "
                         f"running at once, each timing its own pairs; the layer-step ({w.batch * w.n_kv_heads} "
                         f"pairs) at their summed throughput",
               "single_thread": {"value": per_pair * w.batch * w.n_kv_heads * 1e6, "unit": UNIT, "cores": 1,
                                 "sample": f"{n} pairs, one thread, scaled by {w.batch * w.n_kv_heads} pairs"}}
    out = {
        "value": whole_job_us_per_step(total_ms, steps, world), "unit": UNIT, "ms_per_step": ms_per_step,
        "steps": steps,
        "dtype": DTYPE["kivi4" if w.variant == "kivi" and w.bits_k == 4 else w.variant],
        "config": {"workload": _workload_desc(w), "batch": w.batch, "q_heads": w.n_q_heads,
                   "kv_heads": w.n_kv_heads, "head_dim": 128, "seq_len": w.seq_len, "parallelism": f"replicas x{world}",
                   "splits": st["n_splits"],
                   "l2": (f"inputs larger than L2 ({cache_bytes / 1e6:.0f} MB read per step vs 129 MB L2)"
                          if cache_bytes > 129e6 else
                          f"L2-resident ({cache_bytes / 1e6:.2f} MB read per step): launch-latency bound"),
                   "timed": "K steps captured once into a CUDA graph; one untimed replay, then one timed replay"},
        "breakdown_us": {("append_before_attention" if w.variant == "int8t" else "quant_writes_side_stream_span"):
                         1e3 * statistics.mean(quant_ms), "decode_stage1": 1e3 * s1,
                         "decode_stage1_launched_one_by_one": 1e3 * statistics.mean(stage1_evt_ms),
                         "merge": 1e3 * statistics.mean(merge_ms),
                         "timing": "stage 1 from the stage-1 graph; the write side, the merge and the "
                                   "one-by-one stage 1 from a pass of the K steps with events around every kernel"},
        "hbm_gbs_step": (alg_bytes_stage1 + d2h) / (ms_per_step * 1e-3) / 1e9,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_us_per_step(e2e_ms, steps, world), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "every step's inputs from pinned host memory and its output back, on two copy streams "
                          "overlapping the neighbouring steps (two device buffer sets), launched per step from "
                          "the host; each step's kernels one CUDA graph replay"},
        "quant_kernels": quant,
        "gpu_launches": launches_per_step(w) * steps,
        "clocks": clk.summary(),
    }
    del st, graph, g1, step_graphs, bufs
    torch.cuda.empty_cache()
    return out


# The other workloads measured beside the headline at N=1: (key, workload index, field overrides)
EXTRA_CONFIGS = (
    ("2", 2, {}),
    ("4", 4, {}),
    ("4_variance", 4, {"score_mode": 1}),
    ("5", 5, {}),
    ("1", 1, {}),
)


def run_gpu(args, w, rank, world, local_rank):
    head = measure(args, w, rank, world, local_rank, args.steps)
    extras = None
    if world == 1 and not args.only and args.batch == 0:
        extras = {}
        for key, idx, over in EXTRA_CONFIGS:
            if idx == args.workload and not over:
                continue
            wk = dataclasses.replace(I.WORKLOADS[idx], **over)
            m = measure(args, wk, rank, world, local_rank, min(args.steps, 20), want_quant=True, want_cpu=False)
            m.pop("cpu_baseline", None)
            extras[key] = m
    if rank != 0:
        return
    line = {"metric": METRIC, "value": head.pop("value"), "unit": head.pop("unit"), "n_gpus": world,
            "steps": head.pop("steps"), "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "data": "synthetic"}
    line.update(head)
    if extras is not None:
        line["configs"] = extras
    print(json.dumps(line))


def stage1_kernel(w):
    """Name and source files of the stage-1 kernel the library runs for workload w."""
    g = w.n_q_heads // w.n_kv_heads
    gqa = 2 <= g <= 4 or (4 < g <= 8 and g % 2 == 0)        # up to 4 heads per unit, two units per kv head beyond
    if w.variant == "kivi" and gqa:
        return "kivi_decode_gqa_kernel", ("kvq_decode_kivi_gqa.cu", "kvq_kivi.cuh", "kvq_mma.cuh", "kvq_device.cuh")
    if w.variant == "kivi":
        return "kivi_decode_kernel", ("kvq_decode_kivi.cu", "kvq_kivi.cuh", "kvq_device.cuh")
    if w.variant == "kitty" and gqa:
        return "kitty_decode_gqa_kernel", ("kvq_decode_kitty_gqa.cu", "kvq_kitty.cuh", "kvq_mma.cuh", "kvq_device.cuh")
    if w.variant == "kitty":
        return "kitty_decode_kernel", ("kvq_decode_kitty.cu", "kvq_kitty.cuh", "kvq_device.cuh")
    if w.variant == "int8t":
        return "int8_token_decode_kernel", ("kvq_decode_int8.cu", "kvq_device.cuh")
    return f"{w.variant}_decode_kernel", (f"kvq_decode_{w.variant}.cu", "kvq_device.cuh")
DTYPE = {"kivi": "u2 codes + fp16 scales, fp32 accumulate", "kivi4": "u4 codes + fp16 scales, fp32 accumulate", "kitty": "u2 planes + fp16 scales, fp32 accumulate",
         "int8": "s8 codes + Philox dither + fp16 scales, fp32 accumulate",
         "int8t": "s8 codes + Philox dither + fp16 token scales, fp32 accumulate"}


def kernel_source_hash(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "bit_kv_cache_keyquant_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9, 10],
                    help="3 (default: the headline line, the largest single-GPU workload); 1, 2, 4, 5 are the "
                         "other synthetic workloads, 6-10 the variants (token-granular INT8, KIVI-4, paged KIVI, "
                         "KIVI-4 grouped-query, 64q/8kv grouped-query)")
    ap.add_argument("--score-mode", type=int, default=0, choices=[0, 1],
                    help="Kitty boost selection of workload 4: 0 = Eq. 2 sum of |x|, 1 = variance")
    ap.add_argument("--only", action="store_true",
                    help="measure the chosen workload alone (no `configs` entries for the other workloads)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller captures for profiling; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = dataclasses.replace(I.WORKLOADS[args.workload], score_mode=args.score_mode)
    if args.batch > 0:
        w = dataclasses.replace(w, batch=args.batch)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            if w.variant != "kivi":
                print(json.dumps({"impl": "reference", "unavailable": "the reference leg times the KIVI workloads"}))
            else:
                run_reference(args, w)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    from bit_kv_cache_keyquant_gb300 import build
    build.build()
    run_gpu(args, w, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
