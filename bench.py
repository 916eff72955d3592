"""Benchmark: committed tokens/sec of the block-diffusion denoise loop.

Default workload (one GPU, the largest single-GPU configuration): the
long-context decode in bf16, batch 8, prefix 16384 (visual + prompt tokens)
in a paged KV cache (64-token pages, randomly permuted), 16 successive
blocks of L'=32 masked tokens through a 28-layer random-init decoder of
SDAR-1.7B shapes (hidden 2048, 16 query / 8 KV heads, head_dim 128), LM head
151936 x 2048 ~ N(0,0.02); the commit reads planted hidden states
h = a W[t]/|W[t]| + N(0,1) with a ~ U(0,12) redrawn per step; T = 0.95.
`--workload sdar_b1` (and the other names) select the single-layer cases.

One bench step = one full pass of the hot path over one block: denoise steps
(every layer's projections and block attention, then the LM head /
confidence / commit) until no position is masked, then the pass over the
committed tokens that appends every layer's K/V.  value = committed tokens /
second.

Arms:
  default            the CUDA library (libbd.so) through its C ABI
  --impl reference   the CPU oracle on the host cores (rank 0 only), the same
                     metric on a bounded sample of the same workload
Under torchrun with N > 1 GPUs every rank decodes its own replica of the
workload (no collective on the data path); timing takes the max over ranks.
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

METRIC = "committed tokens/sec per denoise loop"
# DRAM bytes (read + write) of one lmhead_tc_kernel launch at sdar_b1
# (32 positions, h read in place, two CTAs per SM): the mean over 26 launches
# of an ncu launch list of the current kernel, dram__bytes_read.sum 622.55 MB
# + dram__bytes_write.sum 0.23 MB.
LMHEAD_TRAFFIC_BYTES = 622_550_725 + 225_526
# DRAM bytes (read + write) of one attn_pair_kernel launch at longctx_b8 (8
# sequences x 16384 cached tokens, one layer), from an ncu capture of the
# current kernel: dram__bytes_read.sum 539.87 MB + dram__bytes_write.sum
# 5.02 MB, against 540.02 MB of algorithmic bytes for that launch; the decode
# line scales it by its calls' algorithmic bytes (the context grows by one
# block per block).
LONGCTX_ATTN_TRAFFIC = (539_869_440 + 5_019_136, 540_016_640)
UNIT = "tokens/s"
WORKLOAD = "longctx_b8"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--check-every", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", default=None,
                    help="comma-separated thresholds: run the multi-block threshold sweep")
    ap.add_argument("--regions", default=None,
                    help="region thresholds by block position, e.g. 0.99:8,0.7:16,0.9:8 "
                         "(T:positions, summing to the block length): one more sweep line")
    ap.add_argument("--blocks", type=int, default=0, help="blocks per sweep decode")
    ap.add_argument("--mlp", action="store_true",
                    help="longctx_b8: add the gated MLP (SwiGLU, intermediate 6144) to every "
                         "decoder layer")
    ap.add_argument("--ar-compare", action="store_true",
                    help="block diffusion vs token-by-token decoding on the same shapes")
    ap.add_argument("--ar-threshold", type=float, default=0.95)
    ap.add_argument("--a-max", type=float, default=None,
                    help="planted amplitude bound (the workload's own by default)")
    ap.add_argument("--temperature", type=float, default=None,
                    help="decode with sampled tokens (bd_sample_commit) at this temperature")
    ap.add_argument("--top-k", type=int, default=0,
                    help="with --temperature: keep the k most likely tokens (0: all)")
    ap.add_argument("--top-p", type=float, default=1.0,
                    help="with --temperature: nucleus truncation at this mass (1: none)")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch every kernel from the host instead of replaying CUDA graphs")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name (the headline line uses longctx_b8)")
    ap.add_argument("--kernel", default=None, choices=["lmhead", "attention", "proj", "step"],
                    help="time one call alone (per-call us, GB/s, TFLOP/s) instead of decoding; "
                         "'step': one eager denoise step of the decoder workload (for a launch "
                         "list of exactly one step)")
    ap.add_argument("--rows", type=int, default=None,
                    help="--kernel lmhead: masked rows of the call (default: all of the workload's)")
    ap.add_argument("--iters", type=int, default=20, help="--kernel: timed calls")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _whole_job_rate(units_per_rank: float, ms_local: float, world: int, device):
    """Whole-job throughput of `world` replicas that each processed
    units_per_rank in ms_local: the slowest rank's time sets the clock.
    Returns (units per second over all ranks, that time in ms)."""
    ms = _max_over_ranks(ms_local, device)
    return units_per_rank * world / (ms / 1e3), ms


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _inputs(w, seed=0):
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    W = wl.lm_head(w, seed)
    plen = wl.prefix_lengths(w, seed)
    kv = [wl.prefix_kv(w, b, int(plen[b]), seed) for b in range(w.batch)]
    q, kb, vb = wl.block_qkv(w, 0, seed)
    h, _ = wl.planted_hidden(w, W, 0, seed)
    return W, plen, kv, q, kb, vb, h


def _config(w, a):
    """The workload this line measures.  Both arms print exactly this dict for
    the same flags; what is specific to one run goes to the line's "run"."""
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    shape = "layer" if w.num_layers == 1 else f"{w.num_layers}-layer decoder"
    c = {"workload": f"{w.name}: SDAR-1.7B-shaped {shape}, batch {w.batch}, prefix {w.prefix}, "
                     f"block {w.block_len}, Hq {w.num_q_heads}/Hkv {w.num_kv_heads}, "
                     f"D {w.head_dim}, LM head {w.vocab}x{w.hidden}, T={w.threshold}, "
                     f"planted a~U(0,{w.a_max:g})",
         "batch": w.batch, "prefix": w.prefix, "prefix_min": w.prefix_min,
         "block_len": w.block_len, "vocab": w.vocab, "hidden": w.hidden,
         "threshold": w.threshold, "a_max": w.a_max,
         "paged_kv": "64-token pages, permuted page table",
         "decoding": _decoding(a)}
    if w.num_layers > 1:
        c.update({"layers": w.num_layers, "blocks": w.num_blocks,
                  "mlp": (f"SwiGLU, intermediate {wl.MLP_INTER}" if getattr(a, "mlp", False)
                          else "none (the plainest reading)"),
                  "l2": "inputs larger than L2: 15.5 GB of per-layer KV cache streamed by "
                        "every denoise step"})
    else:
        c["l2"] = ("inputs larger than L2: the 622 MB LM head is streamed every denoise step "
                   "(evicting the KV cache between steps)")
    return c


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_block(w, W64, kv, q, kb, vb, h, step_lo=0, step_hi=None, tokens=None):
    """Run denoise steps [step_lo, step_hi) of the block on the CPU oracle.

    Every step runs the oracle's block attention (all sequences), confidence,
    commit; the append runs when the block finishes.  Returns
    (tokens, committed count, denoise steps run)."""
    import oracle
    B, L = w.batch, w.block_len
    tokens = np.full((B, L), -1, np.int64) if tokens is None else tokens
    committed, s = 0, step_lo
    step_hi = L if step_hi is None else step_hi
    while (tokens == -1).any() and s < step_hi:
        for b in range(B):
            oracle.current_block_attention(q[b], kv[b][0], kv[b][1], kb[b], vb[b])
        new, *_ = oracle.denoise_step(tokens, h[s].astype(np.float64), W64, w.threshold)
        committed += int((new != tokens).sum())
        tokens = new
        s += 1
    if not (tokens == -1).any():
        ps = 64
        for b in range(B):
            n = kv[b][0].shape[0]
            table = np.arange((n + L + ps - 1) // ps)
            pool = np.zeros((len(table), w.num_kv_heads, ps, w.head_dim))
            oracle.append_block(pool, table[None], [n], kb[b:b + 1], [True], ps)
    return tokens, committed, s - step_lo


def cpu_baseline(w, W, kv, q, kb, vb, h, budget_s=25.0):
    """Time the oracle on a bounded sample: whole blocks while the budget lasts."""
    W64 = W.astype(np.float64)
    t0 = time.perf_counter()
    tokens_done, blocks, steps = 0, 0, 0
    while True:
        _, c, s = oracle_block(w, W64, kv, q, kb, vb, h)
        tokens_done += c
        steps += s
        blocks += 1
        if time.perf_counter() - t0 > budget_s / 2 or blocks >= 4:
            break
    dt = time.perf_counter() - t0
    return {"value": tokens_done / dt, "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{blocks} full block(s) of {w.name} ({steps} denoise steps, "
                      f"{tokens_done} committed tokens) in {dt:.1f} s, numpy fp64"}


class DecoderOracle:
    """The oracle's decode of one sequence of the decoder workload, one denoise
    step at a time: every step runs the layer stack over the block's current
    tokens, then the confidence and commit of that sequence's planted hidden
    states; a finished block is run through the stack once more with its
    committed tokens and every layer's K/V is appended before the next block
    (after the last block the decode starts over from the prefix)."""

    def __init__(self, w, b=0, keep=None, mlp=False, temperature=None, seed=1,
                 top_k=0, top_p=1.0):
        from block_diffusion_decoding_denoise_gb300 import workload as wl
        self.w, self.b, self.wl = w, b, wl
        plen = wl.prefix_lengths(w)
        self.prefix = (keep if keep is not None else
                       [wl.prefix_kv(w, b, int(plen[b]), 0, l) for l in range(w.num_layers)])
        W = wl.lm_head(w)
        self.W, self.W64 = W, W.astype(np.float64)
        self.E, self.em = wl.embed_table(w), wl.mask_embedding(w)
        lw = [wl.layer_weights(w, l) for l in range(w.num_layers)]
        if mlp:
            lw = [t + wl.mlp_weights(w, l) for l, t in enumerate(lw)]
        self.layers = lw
        self.temperature, self.seed, self.top_k, self.top_p = temperature, seed, top_k, top_p
        self.draws = 0
        self._start(0)

    def _start(self, blk):
        if blk == 0:
            self.caches = [(k, v) for k, v in self.prefix]
        self.blk = blk
        self.h = self.wl.planted_hidden(self.w, self.W, blk)[0][:, self.b:self.b + 1]
        self.tokens = np.full((1, self.w.block_len), -1, np.int64)
        self.s = 0

    def step(self):
        """One denoise step (preceded by the append pass when the previous block
        finished); returns the number of tokens it committed."""
        import oracle
        w = self.w
        if not (self.tokens == -1).any():
            _, ks, vs = oracle.decoder_forward(self.tokens[0], self.E, self.em, self.layers,
                                               self.caches, w.num_q_heads, w.num_kv_heads)
            self.caches = [(np.concatenate([kc, k.astype(np.float32)]),
                            np.concatenate([vc, v.astype(np.float32)]))
                           for (kc, vc), k, v in zip(self.caches, ks, vs)]
            self._start((self.blk + 1) % w.num_blocks)
        oracle.decoder_forward(self.tokens[0], self.E, self.em, self.layers, self.caches,
                               w.num_q_heads, w.num_kv_heads)
        h = self.h[self.s].astype(np.float64)
        if self.temperature is None:
            new, *_ = oracle.denoise_step(self.tokens, h, self.W64, w.threshold)
        else:
            new, *_ = oracle.denoise_step_sampled(self.tokens, h, self.W64, w.threshold,
                                                  self.temperature, self.seed, self.draws,
                                                  top_k=self.top_k, top_p=self.top_p)
            self.draws += 1
        c = int((new != self.tokens).sum())
        self.tokens = new
        self.s += 1
        return c


def _reference_steps(a, w):
    """(one reference step, its description) for workload w."""
    if w.num_layers > 1:
        ref = DecoderOracle(w, 0, mlp=a.mlp, temperature=a.temperature, top_k=a.top_k,
                            top_p=a.top_p)
        return ref.step, (f"each step = one denoise step of sequence 0 of {w.name} on the fp64 "
                          f"oracle: the {w.num_layers}-layer stack over the block, confidence "
                          f"over the full vocabulary and commit (the append pass when a block "
                          f"finishes)")
    W, plen, kv, q, kb, vb, h = _inputs(w)
    W64 = W.astype(np.float64)
    chunk = 8                       # one reference step = 8 denoise steps of the block
    state = {"tokens": None, "s": 0}

    def ref_step():
        if state["tokens"] is None or not (state["tokens"] == -1).any():
            state["tokens"], state["s"] = None, 0
        tok, c, n = oracle_block(w, W64, kv, q, kb, vb, h, state["s"], state["s"] + chunk,
                                 state["tokens"])
        state["tokens"], state["s"] = tok, state["s"] + n
        return c
    return ref_step, (f"each step = {chunk} denoise steps of one {w.name} block (all "
                      f"{w.batch} sequences) on the fp64 oracle: attention, full-logit "
                      f"confidence, commit, append at block end")


def run_reference(a):
    rank, world, _ = _dist()
    if rank != 0:
        return
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    w = wl.WORKLOADS[a.workload]
    if a.a_max is not None:
        w = w.with_(a_max=a.a_max)
    ref_step, sample = _reference_steps(a, w)
    for _ in range(a.warmup):
        ref_step()
    t0 = time.perf_counter()
    committed = sum(ref_step() for _ in range(a.steps))
    dt = time.perf_counter() - t0
    value = committed / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt * 1e3 / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w, a),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": f"{sample}; {a.steps} steps, {committed} committed tokens "
                                   f"in {dt:.1f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------------------
# CUDA leg
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def run_cuda(a):
    import torch
    rank, world, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA arm has no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from block_diffusion_decoding_denoise_gb300 import bd, build
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    from block_diffusion_decoding_denoise_gb300.engine import DenoiseEngine, PagedCache
    if not os.path.exists(bd.LIB_PATH):
        build.build()
    bd.load()

    w = wl.WORKLOADS[a.workload]
    if a.a_max is not None:
        w = w.with_(a_max=a.a_max)
    W, plen, kv, q, kb, vb, h = _inputs(w)
    table, npg = wl.page_tables(w, plen + w.block_len)
    cache = PagedCache(npg, w.num_kv_heads, w.head_dim, torch.bfloat16, table)
    for b in range(w.batch):
        cache.load_prefix(b, torch.from_numpy(kv[b][0]), torch.from_numpy(kv[b][1]))
    Wd = torch.from_numpy(W).to("cuda", torch.bfloat16)
    qd = torch.from_numpy(q).to("cuda", torch.bfloat16)
    kbd = torch.from_numpy(kb).to("cuda", torch.bfloat16)
    vbd = torch.from_numpy(vb).to("cuda", torch.bfloat16)
    hd = torch.from_numpy(h).to("cuda", torch.bfloat16)
    max_ctx = int(plen.max()) + w.block_len
    eng = DenoiseEngine(Wd, cache, plen, batch=w.batch, block_len=w.block_len,
                        num_q_heads=w.num_q_heads, threshold=w.threshold, max_ctx=max_ctx,
                        temperature=a.temperature, seed=1, top_k=a.top_k, top_p=a.top_p)
    ctx0 = eng.ctx_len.clone()
    stream = torch.cuda.current_stream()

    # per-call CUDA events around both calls of every denoise step.  With CUDA
    # graphs the events are captured as event-record nodes, so every replay
    # re-records them; they are read after each chunk (the engine syncs there).
    use_graphs = not a.no_graphs
    ev_kw = {"enable_timing": True}
    if use_graphs:
        try:
            torch.cuda.Event(enable_timing=True, external=True)
            ev_kw["external"] = True
        except TypeError:
            use_graphs = False           # this torch cannot time inside a graph
    orig_step = eng.step
    step_events = {}
    attn_ms, conf_ms, rows_seen = [], [], []
    stride = eng.n_committed.stride(0) * eng.n_committed.element_size()

    def timed_step(hh, qq, kk, vv, ncom=None, layer=0):
        s = (ncom.data_ptr() - eng.n_committed.data_ptr()) // stride
        ea = [torch.cuda.Event(**ev_kw) for _ in range(3)]
        ea[0].record(torch.cuda.current_stream())
        bd.bd_block_attention(eng.caches[layer].kv, eng.ctx_len, eng.tokens, qq, kk, vv,
                              eng.attn_out, eng.attn_ws, eng.max_ctx, dev_status=eng.dev_status)
        ea[1].record(torch.cuda.current_stream())
        eng.commit(hh, ncom)
        ea[2].record(torch.cuda.current_stream())
        step_events[s] = ea

    recording = [False]

    def on_chunk(s0, s1):
        if recording[0]:
            for s in range(s0, s1):
                ea = step_events[s]
                attn_ms.append(ea[0].elapsed_time(ea[1]))
                conf_ms.append(ea[1].elapsed_time(ea[2]))
                rows_seen.append(s)

    def block():
        eng.ctx_len.copy_(ctx0)
        return eng.decode_block(hd, qd, kbd, vbd, check_every=a.check_every, graphs=use_graphs,
                                on_chunk=on_chunk)

    # warm-up of both variants (the first block of each captures its graphs):
    # the plain step, timed for `value`, and the step with per-call events,
    # run afterwards for the per-call rooflines (the event nodes cost a few
    # percent of throughput, so they stay out of the timed region)
    for variant in (timed_step, orig_step):
        eng.step = variant
        for _ in range(max(3, a.warmup)):
            block()
    torch.cuda.synchronize()
    eng.check_status()

    # timed region (device-resident inputs)
    steps_issued = 0
    l0 = bd.bd_kernel_launches()
    g0 = eng.graph_kernel_launches
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(a.steps):
            steps_issued += block()
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches = (bd.bd_kernel_launches() - l0) + (eng.graph_kernel_launches - g0)
    ms = t0.elapsed_time(t1)
    eng.check_status()
    committed_per_block = int((eng.tokens != -1).sum().item())
    tokens_total = committed_per_block * a.steps
    steps_per_seq = eng.steps_per_sequence()

    # per-call durations: the same blocks again with CUDA events around each call
    eng.step = timed_step
    recording[0] = True
    for _ in range(min(a.steps, 20)):
        block()
    torch.cuda.synchronize()
    recording[0] = False
    eng.step = orig_step
    eng.check_status()
    value, ms = _whole_job_rate(tokens_total, ms, world, "cuda")

    # roofline of the dominant call: bd_confidence_commit
    # algorithmic bytes per call: W once, plus the masked rows of h (read) and
    # the per-position outputs; masked rows per step follow the commit trace
    masked_rows = []
    rem = w.batch * w.block_len
    nc = eng.n_committed.cpu().numpy()
    for s in range(nc.shape[0]):
        masked_rows.append(max(rem, 0))
        rem -= int(nc[s].sum())
    rows_per_call = [masked_rows[s] for s in rows_seen]
    bytes_w = w.vocab * w.hidden * 2
    alg = [bytes_w + r * w.hidden * 2 + w.batch * w.block_len * 12 for r in rows_per_call]
    peak, peak_kind = _peaks()
    active = [(b, t) for b, t, r in zip(alg, conf_ms, rows_per_call) if r > 0]
    achieved = sum(b for b, _ in active) / (sum(t for _, t in active) / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": LMHEAD_TRAFFIC_BYTES if a.workload == "sdar_b1" else None,
                "kernel": "bd_confidence_commit (masked-row compaction + LM head with online "
                          "max/sum-exp/argmax + commit)",
                "peak_source": f"{peak_kind} hbm_gbs"}
    # block attention: K/V of cache + block once per KV head, Q read, O written
    ctx_tot = int(plen.sum())
    attn_bytes = (2 * (ctx_tot + w.batch * w.block_len) * w.num_kv_heads * w.head_dim * 2
                  + 2 * w.batch * w.block_len * w.num_q_heads * w.head_dim * 2)
    act = [t for t, r in zip(attn_ms, rows_per_call) if r > 0]
    attn_gbs = attn_bytes * len(act) / (sum(act) / 1e3) / 1e9 if act else None
    roofline_attn = {"bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s",
                     "frac": attn_gbs / peak if attn_gbs else None,
                     "bytes_per_call": attn_bytes,
                     "us_per_call": 1e3 * statistics.mean(act) if act else None}

    e2e = None
    if not a.no_e2e:
        e2e = _e2e(a, eng, w, h, q, kb, vb, hd, qd, kbd, vbd, ctx0, stream, committed_per_block,
                   world, use_graphs)
    if rank != 0:
        return
    cpu = None
    if not a.no_cpu_baseline:
        cpu = cpu_baseline(w, W, kv, q, kb, vb, h)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": max(3, a.warmup), "ms_per_step": ms / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(w, a),
        "run": {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "denoise_steps_per_block": [int(x) for x in steps_per_seq],
                "denoise_steps_issued": steps_issued // a.steps,
                "check_every": a.check_every, "cuda_graphs": use_graphs,
                "per_call_timing": f"CUDA events around every call in {min(a.steps, 20)} "
                                   f"further blocks after the timed region (event nodes "
                                   f"slow the graphs)"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches), "clocks": clk.summary(),
        "conf_call_us_mean": 1e3 * statistics.mean(conf_ms) if conf_ms else None,
        "roofline_attention": roofline_attn,
    }
    print(json.dumps(line))


def _e2e(a, eng, w, h, q, kb, vb, hd, qd, kbd, vbd, ctx0, stream, committed_per_block, world,
         use_graphs):
    """Same metric through the public API with host buffers: every block copies its
    inputs from pinned host memory and reads the committed tokens back."""
    import torch
    h_host = torch.from_numpy(h).to(torch.bfloat16).pin_memory()
    q_host = torch.from_numpy(q).to(torch.bfloat16).pin_memory()
    k_host = torch.from_numpy(kb).to(torch.bfloat16).pin_memory()
    v_host = torch.from_numpy(vb).to(torch.bfloat16).pin_memory()
    tok_host = torch.empty(w.batch, w.block_len, dtype=torch.int32).pin_memory()
    h_in = torch.empty_like(hd)
    q_in, k_in, v_in = torch.empty_like(qd), torch.empty_like(kbd), torch.empty_like(vbd)
    h2d = sum(t.numel() * t.element_size() for t in (h_host, q_host, k_host, v_host))
    d2h = tok_host.numel() * tok_host.element_size()
    def one():
        h_in.copy_(h_host, non_blocking=True)
        q_in.copy_(q_host, non_blocking=True)
        k_in.copy_(k_host, non_blocking=True)
        v_in.copy_(v_host, non_blocking=True)
        eng.ctx_len.copy_(ctx0)
        eng.decode_block(h_in, q_in, k_in, v_in, check_every=a.check_every, graphs=use_graphs)
        tok_host.copy_(eng.tokens, non_blocking=True)

    one()                                  # captures the graphs over these buffers
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    return {"value": committed_per_block * a.steps * world / (e2e_ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def _decoding(a):
    if a.temperature is None:
        return "greedy"
    d = f"sampled, temperature {a.temperature}"
    if a.top_k > 0:
        d += f", top-k {a.top_k}"
    if a.top_p < 1.0:
        d += f", top-p {a.top_p}"
    return d


def run_sweep(a):
    """Threshold sweep: full multi-block decodes (each finished block's K/V is
    appended before the next block) at every T, one JSON line per T with the
    denoise steps per block and committed tokens/s.  Not the headline line."""
    import torch
    from block_diffusion_decoding_denoise_gb300 import bd, build
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    from block_diffusion_decoding_denoise_gb300.engine import DenoiseEngine, PagedCache
    if not os.path.exists(bd.LIB_PATH):
        build.build()
    bd.load()
    w = wl.WORKLOADS[a.workload]
    nblk = a.blocks or w.num_blocks
    a_max = w.a_max if a.a_max is None else a.a_max
    W = wl.lm_head(w)
    Wd = torch.from_numpy(W).to("cuda", torch.bfloat16)
    plen = wl.prefix_lengths(w)
    cap = plen + nblk * w.block_len
    table, npg = wl.page_tables(w, cap)
    blocks = []
    for blk in range(nblk):
        q, kb, vb = wl.block_qkv(w, blk)
        h, _ = wl.planted_hidden(w, W, blk, a_max=a_max)
        blocks.append(tuple(torch.from_numpy(x).to("cuda", torch.bfloat16) for x in (h, q, kb, vb)))
    kvs = [wl.prefix_kv(w, b, int(plen[b])) for b in range(w.batch)]
    entries = [({"threshold": float(x)}, float(x)) for x in a.sweep.split(",")] if a.sweep else []
    if a.regions:
        row = []
        for part in a.regions.split(","):
            t, n = part.split(":")
            row += [float(t)] * int(n)
        if len(row) != w.block_len:
            raise SystemExit(f"--regions covers {len(row)} positions, the block has {w.block_len}")
        entries.append(({"region_thresholds": a.regions},
                         np.tile(np.asarray(row, np.float32), (w.batch, 1))))
    for label, T in entries:
        cache = PagedCache(npg, w.num_kv_heads, w.head_dim, torch.bfloat16, table)
        for b in range(w.batch):
            cache.load_prefix(b, torch.from_numpy(kvs[b][0]), torch.from_numpy(kvs[b][1]))
        eng = DenoiseEngine(Wd, cache, plen, batch=w.batch, block_len=w.block_len,
                            num_q_heads=w.num_q_heads, threshold=T, max_ctx=int(cap.max()))
        ctx0 = eng.ctx_len.clone()
        for _ in range(2):                      # warm-up decodes (capture the graphs)
            eng.ctx_len.copy_(ctx0)
            for (h, q, kb, vb) in blocks:
                eng.decode_block(h, q, kb, vb, check_every=a.check_every,
                                 graphs=not a.no_graphs)
        torch.cuda.synchronize()
        eng.ctx_len.copy_(ctx0)
        steps = []
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for (h, q, kb, vb) in blocks:
            eng.decode_block(h, q, kb, vb, check_every=a.check_every, graphs=not a.no_graphs)
            steps.append(eng.steps_per_sequence())
        e1.record()
        torch.cuda.synchronize()
        eng.check_status()
        ms = e0.elapsed_time(e1)
        tokens = w.batch * w.block_len * nblk
        st = np.array(steps)
        print(json.dumps({
            "sweep": True, "metric": METRIC, "unit": UNIT, **label,
            "value": tokens / (ms / 1e3), "ms": ms, "blocks": nblk,
            "denoise_steps_per_block_mean": float(st.mean()),
            "denoise_steps_per_block_min": int(st.min()),
            "denoise_steps_per_block_max": int(st.max()),
            "config": _config(w.with_(a_max=a_max), a),
            "run": {"blocks": nblk, "prefix_after": int(eng.ctx_len.max().item())}}),
              flush=True)


def _decode_tokens_per_s(w, W, Wd, a_max, T, ntok, check_every, graphs):
    """Decode ntok tokens per sequence in blocks of w.block_len (appending each
    finished block), twice; returns (tokens/s of the second pass, mean denoise
    steps per block)."""
    import torch
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    from block_diffusion_decoding_denoise_gb300.engine import DenoiseEngine, PagedCache
    nblk = ntok // w.block_len
    plen = wl.prefix_lengths(w)
    cap = plen + ntok
    table, npg = wl.page_tables(w, cap)
    cache = PagedCache(npg, w.num_kv_heads, w.head_dim, torch.bfloat16, table)
    for b in range(w.batch):
        k, v = wl.prefix_kv(w, b, int(plen[b]))
        cache.load_prefix(b, torch.from_numpy(k), torch.from_numpy(v))
    blocks = []
    for blk in range(nblk):
        q, kb, vb = wl.block_qkv(w, blk)
        h, _ = wl.planted_hidden(w, W, blk, a_max=a_max)
        blocks.append(tuple(torch.from_numpy(x).to("cuda", torch.bfloat16) for x in (h, q, kb, vb)))
    eng = DenoiseEngine(Wd, cache, plen, batch=w.batch, block_len=w.block_len,
                        num_q_heads=w.num_q_heads, threshold=T, max_ctx=int(cap.max()))
    ctx0 = eng.ctx_len.clone()
    if w.block_len == 1:
        return _ar_tokens_per_s(eng, blocks, ctx0, w.batch * ntok, graphs), 1.0
    ms = steps = 0.0
    for rep in range(2):
        eng.ctx_len.copy_(ctx0)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        tot = 0
        for (h, q, kb, vb) in blocks:
            eng.decode_block(h, q, kb, vb, check_every=min(check_every, w.block_len),
                             graphs=graphs)
            tot += float(eng.steps_per_sequence().mean())
        e1.record()
        torch.cuda.synchronize()
        eng.check_status()
        ms, steps = e0.elapsed_time(e1), tot / nblk
    return w.batch * ntok / (ms / 1e3), steps


def _ar_tokens_per_s(eng, blocks, ctx0, ntok_total, graphs):
    """Token-by-token decoding: with one position per block every step
    commits it, so the loop needs no host check at all.  Each token is
    reset-mask + attention + confidence/commit + append; with `graphs` the
    whole token sequence is one CUDA graph.  Returns tokens/s of the second
    pass."""
    import torch
    from block_diffusion_decoding_denoise_gb300 import bd

    def one_pass():
        for (h, q, kb, vb) in blocks:
            eng.tokens.fill_(bd.BD_MASK)
            eng.step(h[0], q, kb, vb, eng.n_committed[0])
            bd.bd_append_block_kv(eng.caches[0].kv, kb, vb, eng.ctx_len, eng.n_masked,
                                  eng.dev_status)

    g = None
    if graphs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one_pass()
    ms = 0.0
    for rep in range(2):
        eng.ctx_len.copy_(ctx0)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        if g is not None:
            g.replay()
        else:
            one_pass()
        e1.record()
        torch.cuda.synchronize()
        eng.check_status()
        ms = e0.elapsed_time(e1)
    assert int((eng.ctx_len - ctx0).min().item()) == len(blocks)   # every token appended
    return ntok_total / (ms / 1e3)


def run_ar_compare(a):
    """Block diffusion (blocks of 32) against token-by-token decoding (blocks of
    1, i.e. causal AR decoding on the same kernels) on the same shapes: the
    synthetic counterpart of the pages' decoding-speedup comparison."""
    import torch
    from block_diffusion_decoding_denoise_gb300 import bd, build
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    if not os.path.exists(bd.LIB_PATH):
        build.build()
    bd.load()
    w = wl.WORKLOADS[a.workload]
    a_max = w.a_max if a.a_max is None else a.a_max
    T = float(a.ar_threshold)
    W = wl.lm_head(w)
    Wd = torch.from_numpy(W).to("cuda", torch.bfloat16)
    ntok = 32 * max(1, a.blocks or 1)
    res = {}
    for L in (w.block_len, 1):
        wb = w.with_(block_len=L)
        res[L] = _decode_tokens_per_s(wb, W, Wd, a_max, T, ntok, a.check_every,
                                      not a.no_graphs)
    print(json.dumps({
        "ar_compare": True, "metric": METRIC, "unit": UNIT, "threshold": T, "a_max": a_max,
        "tokens_per_sequence": ntok,
        "block_diffusion": {"block_len": w.block_len, "value": res[w.block_len][0],
                            "denoise_steps_per_block": res[w.block_len][1]},
        "autoregressive": {"block_len": 1, "value": res[1][0]},
        "speedup": res[w.block_len][0] / res[1][0],
        "config": _config(w.with_(a_max=a_max), a)}))


# ---------------------------------------------------------------------------
# decoder workload (28-layer stack, successive blocks)
# ---------------------------------------------------------------------------
def _decoder_inputs(w, plen, seed=0, keep_seq=None):
    """Per-layer prefix K/V generator: yields (layer, b, k, v); the caller loads
    them.  Sequences of a layer are drawn in parallel threads."""
    import concurrent.futures as cf
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    with cf.ThreadPoolExecutor(min(w.batch, _cores())) as ex:
        for l in range(w.num_layers):
            futs = [ex.submit(wl.prefix_kv, w, b, int(plen[b]), seed, l) for b in range(w.batch)]
            for b, f in enumerate(futs):
                k, v = f.result()
                yield l, b, k, v


def run_decoder(a):
    """The long-context workload: a 28-layer decoder stack in front of every
    denoise step's commit, successive blocks of one decode (each finished
    block is run through the stack once more and its K/V appended to every
    layer before the next block)."""
    import torch
    rank, world, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA arm has no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from block_diffusion_decoding_denoise_gb300 import bd, build
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    from block_diffusion_decoding_denoise_gb300.engine import (DecoderStack, DenoiseEngine,
                                                               PagedCache)
    if not os.path.exists(bd.LIB_PATH):
        build.build()
    bd.load()
    w = wl.WORKLOADS[a.workload]
    if a.a_max is not None:
        w = w.with_(a_max=a.a_max)
    L, nb = w.block_len, w.num_blocks
    plen = wl.prefix_lengths(w)
    cap = plen + nb * L
    table, npg = wl.page_tables(w, cap)
    bf = torch.bfloat16
    caches = [PagedCache(npg, w.num_kv_heads, w.head_dim, bf, table) for _ in range(w.num_layers)]
    keep = [] if rank == 0 and not a.no_cpu_baseline else None
    t_gen = time.perf_counter()
    for l, b, k, v in _decoder_inputs(w, plen):
        caches[l].load_prefix(b, torch.from_numpy(k), torch.from_numpy(v))
        if keep is not None and b == 0:
            keep.append((k, v))
    W = wl.lm_head(w)
    E = wl.embed_table(w)
    em = wl.mask_embedding(w)
    lw = [wl.layer_weights(w, l) for l in range(w.num_layers)]
    if a.mlp:
        lw = [t + wl.mlp_weights(w, l) for l, t in enumerate(lw)]
    dev = lambda x: torch.from_numpy(x).to("cuda", bf)
    ctx = torch.from_numpy(plen.astype(np.int32)).cuda()
    max_ctx = int(cap.max())
    stack = DecoderStack(dev(E), dev(em), [tuple(dev(x) for x in t) for t in lw], caches, ctx,
                         batch=w.batch, block_len=L, num_q_heads=w.num_q_heads, max_ctx=max_ctx)
    eng = DenoiseEngine(dev(W), caches, plen, batch=w.batch, block_len=L,
                        num_q_heads=w.num_q_heads, threshold=w.threshold, max_ctx=max_ctx,
                        temperature=a.temperature, seed=1, decoder=stack,
                        top_k=a.top_k, top_p=a.top_p)
    h_host = [wl.planted_hidden(w, W, blk)[0] for blk in range(nb)]
    del W, E, em, lw
    h_dev = [dev(h) for h in h_host]
    h_cur = torch.empty_like(h_dev[0])
    dummy = torch.empty(1, dtype=bf, device="cuda")
    gen_s = time.perf_counter() - t_gen
    ctx0 = ctx.clone()
    use_graphs = not a.no_graphs
    ev_kw = {"enable_timing": True}
    if use_graphs:
        try:
            torch.cuda.Event(enable_timing=True, external=True)
            ev_kw["external"] = True
        except TypeError:
            use_graphs = False

    # per-call events (attention of every layer, the commit) inside every
    # denoise step, captured into the step graphs as event nodes and read
    # after each chunk; these graphs run only after the timed region
    orig_forward = stack.forward
    orig_commit = eng.commit
    events = {}
    attn_ms, conf_ms = [], []
    stride = eng.n_committed.stride(0) * eng.n_committed.element_size()
    cur_step = [None]

    def timed_forward(tokens, attn_tokens=None):
        if attn_tokens is None:
            return orig_forward(tokens, None)
        evs = events.setdefault(cur_step[0], {"attn": [], "conf": None})
        evs["attn"] = []
        stack_attn = bd.bd_block_attention

        def attn_wrap(*args, **kw):
            e0, e1 = torch.cuda.Event(**ev_kw), torch.cuda.Event(**ev_kw)
            e0.record(torch.cuda.current_stream())
            stack_attn(*args, **kw)
            e1.record(torch.cuda.current_stream())
            evs["attn"].append((e0, e1))
        bd.bd_block_attention = attn_wrap
        try:
            orig_forward(tokens, attn_tokens)
        finally:
            bd.bd_block_attention = stack_attn

    def timed_commit(h, ncom):
        cur = (ncom.data_ptr() - eng.n_committed.data_ptr()) // stride
        e0, e1 = torch.cuda.Event(**ev_kw), torch.cuda.Event(**ev_kw)
        e0.record(torch.cuda.current_stream())
        orig_commit(h, ncom)
        e1.record(torch.cuda.current_stream())
        events.setdefault(cur, {"attn": [], "conf": None})["conf"] = (e0, e1)

    orig_step = eng.step

    def timed_step(hh, qq, kk, vv, ncom=None, layer=0):
        cur_step[0] = (ncom.data_ptr() - eng.n_committed.data_ptr()) // stride
        stack.forward = timed_forward
        eng.commit = timed_commit
        try:
            orig_step(hh, qq, kk, vv, ncom, layer)
        finally:
            stack.forward = orig_forward
            eng.commit = orig_commit

    recording = [False]

    def on_chunk(s0, s1):
        if recording[0]:
            for s in range(s0, s1):
                ev = events.get(s)
                if ev is None:
                    continue
                for e0, e1 in ev["attn"]:
                    attn_ms.append(e0.elapsed_time(e1))
                if ev["conf"] is not None:
                    conf_ms.append(ev["conf"][0].elapsed_time(ev["conf"][1]))

    blk_ctr = [0]

    def block():
        blk = blk_ctr[0] % nb
        if blk == 0:
            ctx.copy_(ctx0)
        blk_ctr[0] += 1
        h_cur.copy_(h_dev[blk])
        return eng.decode_block(h_cur, dummy, dummy, dummy, check_every=a.check_every,
                                graphs=use_graphs, on_chunk=on_chunk)

    # warm-up of both step variants (the first block of each captures its
    # graphs): the plain step, timed for `value`, then the step with events
    warm = max(3, a.warmup)
    for variant in (timed_step, orig_step):
        eng.step = variant
        blk_ctr[0] = 0
        for _ in range(warm):
            block()
    torch.cuda.synchronize()
    eng.check_status()
    blk_ctr[0] = 0
    ctx_at = ctx0.clone()
    steps_issued = committed = 0
    l0 = bd.bd_kernel_launches()
    g0 = eng.graph_kernel_launches
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(a.steps):
            steps_issued += block()
            committed += w.batch * L
        t1.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    eng.check_status()
    launches = (bd.bd_kernel_launches() - l0) + (eng.graph_kernel_launches - g0)
    value, ms = _whole_job_rate(committed, ms, world, "cuda")

    # per-call durations: the same blocks again (from block 0) with events
    eng.step = timed_step
    blk_ctr[0] = 0
    recording[0] = True
    for _ in range(min(a.steps, nb)):
        block()
    torch.cuda.synchronize()
    recording[0] = False
    eng.step = orig_step
    eng.check_status()

    # attention roofline: K/V of the cache + block once per KV head, Q read, O
    # written; the context grows by one block per block, so take the mean
    # context of the blocks timed per call
    nper = min(a.steps, nb)
    ctx_mean = float(ctx_at.float().mean().item()) + L * (nper - 1) / 2.0
    attn_bytes = (2 * w.batch * (ctx_mean + L) * w.num_kv_heads * w.head_dim * 2
                  + 2 * w.batch * L * w.num_q_heads * w.head_dim * 2)
    peak, peak_kind = _peaks()
    attn_us = 1e3 * statistics.mean(attn_ms) if attn_ms else None
    achieved = attn_bytes / (attn_us / 1e6) / 1e9 if attn_us else None
    traffic = None
    if a.workload == "longctx_b8":
        traffic = LONGCTX_ATTN_TRAFFIC[0] * attn_bytes / LONGCTX_ATTN_TRAFFIC[1]
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak if achieved else None, "traffic": traffic,
                "kernel": f"bd_block_attention (one call per layer, {w.num_layers} per "
                          f"denoise step: attn_pair_kernel + attn_pair_merge_kernel)",
                "bytes_per_call": attn_bytes, "us_per_call": attn_us,
                "calls_timed": len(attn_ms), "peak_source": f"{peak_kind} hbm_gbs"}
    breakdown = {
        "denoise_steps_per_block": steps_issued / a.steps,
        "ms_per_denoise_step": ms / steps_issued if steps_issued else None,
        "attention_us_per_layer_call": attn_us,
        "attention_share_of_step": (attn_us * w.num_layers / 1e3) / (ms / steps_issued)
                                   if attn_us and steps_issued else None,
        "commit_us_per_call": 1e3 * statistics.mean(conf_ms) if conf_ms else None,
    }

    # e2e: the same blocks through the public API, planted h copied from pinned
    # host memory per block and the committed tokens read back
    e2e = None
    if not a.no_e2e:
        hp = [torch.from_numpy(h).to(bf).pin_memory() for h in h_host]
        tok_host = torch.empty(w.batch, L, dtype=torch.int32).pin_memory()
        ctx.copy_(ctx0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for j in range(a.steps):
            blk = j % nb
            if blk == 0:
                ctx.copy_(ctx0)
            h_cur.copy_(hp[blk], non_blocking=True)
            eng.decode_block(h_cur, dummy, dummy, dummy, check_every=a.check_every,
                             graphs=use_graphs)
            tok_host.copy_(eng.tokens, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        eng.check_status()
        e2e_ms = _max_over_ranks(e0.elapsed_time(e1), "cuda")
        e2e = {"value": committed * world / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": hp[0].numel() * hp[0].element_size(),
               "d2h_bytes_per_step": tok_host.numel() * 4}
    if rank != 0:
        return
    cpu = None
    if keep is not None:
        ref = DecoderOracle(w, 0, keep=keep, mlp=a.mlp, temperature=a.temperature,
                            top_k=a.top_k, top_p=a.top_p)
        t0c = time.perf_counter()
        st = c = 0
        while True:
            c += ref.step()
            st += 1
            if time.perf_counter() - t0c > 20.0 or st >= w.block_len:
                break
        dt = time.perf_counter() - t0c
        cpu = {"value": c / dt, "unit": UNIT, "cores": _cores(), "kind": "oracle",
               "sample": f"sequence 0 of block 0: {st} denoise step(s) of the {w.num_layers}-"
                         f"layer stack + confidence + commit ({c} committed tokens) in "
                         f"{dt:.1f} s, numpy fp64"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": warm, "ms_per_step": ms / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(w, a),
        "run": {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "blocks_timed": a.steps, "denoise_steps_issued": steps_issued // a.steps,
                "check_every": a.check_every, "cuda_graphs": use_graphs,
                "input_generation_s": gen_s,
                "per_call_timing": f"CUDA events around every attention and commit call in "
                                   f"{nper} further blocks after the timed region (event "
                                   f"nodes slow the graphs)"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches), "clocks": clk.summary(),
        "step_breakdown": breakdown,
    }
    print(json.dumps(line))


def run_kernel(a):
    """One library call timed alone: the LM head + confidence/commit call at a
    given number of masked rows, or the block attention at a workload's prefix
    lengths.  Inputs are seeded synthetic tensors of the workload's shapes;
    a 256 MB buffer is rewritten between calls so no call starts with the
    previous call's data in L2."""
    import torch
    from block_diffusion_decoding_denoise_gb300 import bd, build
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    from block_diffusion_decoding_denoise_gb300.engine import PagedCache
    if not os.path.exists(bd.LIB_PATH):
        build.build()
    bd.load()
    w = wl.WORKLOADS[a.workload]
    g = torch.Generator(device="cuda").manual_seed(0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L, H, V = w.block_len, w.hidden, w.vocab
    if a.kernel == "lmhead":
        rows = a.rows or w.batch * L
        B = (rows + L - 1) // L
        W = torch.from_numpy(wl.lm_head(w)).to("cuda", torch.bfloat16)
        h = torch.randn(B, L, H, device="cuda", generator=g).to(torch.bfloat16)
        ws = torch.empty(bd.bd_confidence_commit_workspace(bd.BD_BF16, B, L, H, V),
                         dtype=torch.uint8, device="cuda")
        tok = torch.empty(B, L, dtype=torch.int32, device="cuda")
        pm = torch.empty(B, L, device="cuda")
        am = torch.empty_like(tok)
        nc = torch.empty(B, dtype=torch.int32, device="cuda")
        nm = torch.empty_like(nc)

        def call():
            tok.fill_(7)
            tok.view(-1)[:rows] = -1
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            bd.bd_confidence_commit(h, W, w.threshold, tok, pm, am, nc, nm, ws, dev_status=st)
            e1.record()
            return e0, e1
        flops = 2.0 * rows * H * V
        byts = V * H * 2 + rows * H * 2
        what = f"bd_confidence_commit, {rows} masked rows, LM head {V}x{H}"
    elif a.kernel == "proj":
        # the decoder's QKV projection and output projection + residual + RMSNorm
        # of one layer over the workload's block rows
        rows = a.rows or w.batch * L
        Fq = (w.num_q_heads + 2 * w.num_kv_heads) * w.head_dim
        Fi = w.num_q_heads * w.head_dim
        wqkv, wo = (torch.from_numpy(x).to("cuda", torch.bfloat16) for x in wl.layer_weights(w, 0))
        xn = torch.randn(rows, H, device="cuda", generator=g).to(torch.bfloat16)
        att = torch.randn(rows, Fi, device="cuda", generator=g).to(torch.bfloat16)
        x = torch.randn(rows, H, device="cuda", generator=g)
        q = torch.empty(rows, w.num_q_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
        k = torch.empty(rows, w.num_kv_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        ws = torch.empty(max(bd.bd_qkv_projection_workspace(rows, H, w.num_q_heads,
                                                            w.num_kv_heads, w.head_dim),
                             bd.bd_out_projection_workspace(rows, Fi, H)),
                         dtype=torch.uint8, device="cuda")

        def call():
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            bd.bd_qkv_projection(xn, wqkv, q, k, v, ws, dev_status=st)
            bd.bd_out_projection_residual(att, wo, x, xn, ws, dev_status=st)
            e1.record()
            return e0, e1
        flops = 2.0 * rows * H * (Fq + Fi)
        byts = (Fq + H) * H * 2 + rows * (H + Fi) * 2 + rows * (Fq + H) * 2 + rows * H * 8
        what = f"bd_qkv_projection + bd_out_projection_residual, {rows} rows, {Fq}x{H} + {H}x{Fi}"
    else:
        plen = wl.prefix_lengths(w)
        table, npg = wl.page_tables(w, plen + L)
        cache = PagedCache(npg, w.num_kv_heads, w.head_dim, torch.bfloat16, table)
        cache.k.normal_(generator=g)
        cache.v.normal_(generator=g)
        ctx = torch.from_numpy(plen.astype(np.int32)).cuda()
        q = torch.randn(w.batch, L, w.num_q_heads, w.head_dim, device="cuda",
                        generator=g).to(torch.bfloat16)
        kb = torch.randn(w.batch, L, w.num_kv_heads, w.head_dim, device="cuda",
                         generator=g).to(torch.bfloat16)
        vb = torch.randn(kb.shape, device="cuda", generator=g).to(torch.bfloat16)
        out = torch.empty_like(q)
        mc = int(plen.max()) + L
        ws = torch.zeros(max(1, bd.bd_block_attention_workspace(
            w.batch, L, w.num_q_heads, w.num_kv_heads, w.head_dim, mc)), dtype=torch.uint8,
            device="cuda")

        def call():
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            bd.bd_block_attention(cache.kv, ctx, None, q, kb, vb, out, ws, mc, dev_status=st)
            e1.record()
            return e0, e1
        nk = int(plen.sum()) + w.batch * L
        byts = 2 * nk * w.num_kv_heads * w.head_dim * 2 + 2 * w.batch * L * w.num_q_heads * w.head_dim * 2
        flops = 4.0 * nk * L * w.num_q_heads * w.head_dim
        what = f"bd_block_attention, {w.name} prefixes (sum {int(plen.sum())}, max {int(plen.max())})"
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(a.iters):
        e0, e1 = call()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    if int(st.item()) != 0:
        raise SystemExit(f"device status {bd.STATUS.get(int(st.item()))}")
    us = statistics.median(ts)
    peak, kind = _peaks()
    print(json.dumps({"kernel": a.kernel, "call": what, "us_median": us, "us_min": min(ts),
                      "gb_s": byts / us / 1e3, "hbm_frac": byts / us / 1e3 / peak,
                      "tflop_s": flops / us / 1e6, "iters": a.iters,
                      "peak_source": f"{kind} hbm_gbs"}))


def run_step(a):
    """One denoise step of the decoder workload launched eagerly, after one
    warm-up step: every layer's projections and block attention, then the
    confidence/commit.  Prints the step's duration; under a profiler the
    second step's launches are exactly one step."""
    import torch
    from block_diffusion_decoding_denoise_gb300 import bd, build
    from block_diffusion_decoding_denoise_gb300 import workload as wl
    from block_diffusion_decoding_denoise_gb300.engine import (DecoderStack, DenoiseEngine,
                                                               PagedCache)
    if not os.path.exists(bd.LIB_PATH):
        build.build()
    bd.load()
    w = wl.WORKLOADS[a.workload]
    if w.num_layers == 1:
        raise SystemExit("--kernel step needs a decoder workload (longctx_b8)")
    L = w.block_len
    plen = wl.prefix_lengths(w)
    cap = plen + L
    table, npg = wl.page_tables(w, cap)
    bf = torch.bfloat16
    caches = [PagedCache(npg, w.num_kv_heads, w.head_dim, bf, table) for _ in range(w.num_layers)]
    for l, b, k, v in _decoder_inputs(w, plen):
        caches[l].load_prefix(b, torch.from_numpy(k), torch.from_numpy(v))
    dev = lambda x: torch.from_numpy(x).to("cuda", bf)
    W = wl.lm_head(w)
    lw = [tuple(dev(x) for x in wl.layer_weights(w, l)) for l in range(w.num_layers)]
    ctx = torch.from_numpy(plen.astype(np.int32)).cuda()
    stack = DecoderStack(dev(wl.embed_table(w)), dev(wl.mask_embedding(w)), lw, caches, ctx,
                         batch=w.batch, block_len=L, num_q_heads=w.num_q_heads,
                         max_ctx=int(cap.max()))
    eng = DenoiseEngine(dev(W), caches, plen, batch=w.batch, block_len=L,
                        num_q_heads=w.num_q_heads, threshold=w.threshold, max_ctx=int(cap.max()),
                        decoder=stack)
    h = dev(wl.planted_hidden(w, W, 0, steps=2)[0])
    dummy = torch.empty(1, dtype=bf, device="cuda")
    ts = []
    for s in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push(f"step{s}")
        e0.record()
        eng.step(h[s], dummy, dummy, dummy, eng.n_committed[s])
        e1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    eng.check_status()
    print(json.dumps({"kernel": "step", "workload": w.name, "us": ts}))


def main():
    a = _args()
    if a.kernel == "step":
        run_step(a)
        return
    if a.kernel:
        run_kernel(a)
        return
    if a.impl == "reference":
        run_reference(a)
    elif a.sweep or a.regions:
        run_sweep(a)
    elif a.ar_compare:
        run_ar_compare(a)
    else:
        from block_diffusion_decoding_denoise_gb300 import workload as wl
        if wl.WORKLOADS[a.workload].num_layers > 1:
            run_decoder(a)
        else:
            run_cuda(a)


if __name__ == "__main__":
    main()
