"""Benchmark of the paged KV-cache decode step on GB300.

Workload: GQA 32 q / 8 kv heads, head_dim 128, bf16, block size 16, 256
sequences with context lengths clip(round(LogNormal(ln 4096, 1)), 64, 32768),
K/V/Q ~ N(0,1), blocks drawn from a shuffled pool sized to fit.  One step is
the whole decode step: host ledger (on-demand blocks, block table, slot
mapping) -> block table / lengths / slots to the GPU -> cache write of the new
token's K/V -> paged decode attention over every sequence.

Metric: KV GB/s of the decode-attention step (algorithmic bytes: K and V of
every context token + q + out + table entries, per step, over step time), with
seq-tokens/s (context tokens attended per second, one layer) beside it.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun each rank runs its own batch of 256 sequences (weak scaling, no
collective on the data path; only a barrier and a max over ranks of the time).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV GB/s as % of GB300 HBM peak; seq-tokens/s"
LENGTHS = {
    "gqa_long": "clip(round(LogNormal(ln 4096, 1)), 64, 32768)",
    "gqa_long_q8": "clip(round(LogNormal(ln 4096, 1)), 64, 32768)",
    "tiny": "{1, 17, 100, 33} + steps",
    "opt13b": "U[128, 2048]",
    "shared_prefix": "1024 shared + U[64, 512] private",
}
DECODE_WORKLOADS = tuple(LENGTHS)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


DECODE_SOURCES = ("decode_params.h", "paged_decode.cu", "pkv_device.cuh")
PREFILL_SOURCES = ("paged_prefill.cu", "tc_device.cuh", "pkv_device.cuh")


def decode_source_hash(sources=DECODE_SOURCES) -> str:
    """First 16 hex digits of the SHA-256 of the code the kernels compile from
    (the 16-bit decode kernels by default; comments removed and whitespace
    collapsed, so a comment edit does not count as a kernel change)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_146_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str = "gqa_long", summary: str | None = None,
                     sources=None):
    """DRAM bytes (read + write) per attention call from the committed ncu
    launch-list summary of the workload (at its default size), or None when there
    is none or the kernel sources changed since it was taken."""
    prof = os.path.join(ROOT, "profiles", summary or f"paged_decode_{workload}_launches.md")
    if sources is None:     # the shared-prefix path also runs the tcgen05 kernel
        sources = DECODE_SOURCES + (PREFILL_SOURCES[:2] if workload == "shared_prefix" else ())
    try:
        fields = dict(line.split(": ", 1) for line in open(prof).read().splitlines()
                      if line.startswith(("attention_traffic_bytes_per_launch:", "source_sha256_16:")))
        current = decode_source_hash(sources)
        if fields.get("source_sha256_16", "").strip() != current:
            return None
        return int(fields["attention_traffic_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.lines = []
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sms, maxes, watts, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                maxes.append(float(parts[1]))
            except ValueError:
                continue
            try:
                watts.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        out = {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
               "reasons": sorted(reasons), "samples": len(sms)}
        if watts:
            out["power_w"] = statistics.median(watts)
        return out


# ------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl != "reference" else "gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """Slowest rank's time: the job is done when every rank is."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(seed: int, rank: int, num_seqs: int, growth_tokens: int):
    """Each rank decodes its own batch of sequences (weak scaling): rank r draws
    the batch with seed + r, so ranks hold disjoint, independent work."""
    from paged_kv_cache_146_gb300 import workloads
    return workloads.gqa_long(seed + rank, num_seqs=num_seqs, growth_tokens=growth_tokens)


def job_rate(bytes_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: bytes of all ranks over the slowest rank's time."""
    return bytes_per_rank * world / (max_ms * 1e-3) / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- oracle arm
class OracleSample:
    """The oracle (fp64 C, all host cores) on the first ``k`` sequences of the
    named decode workload: the same length law, shapes and dtype, bounded in
    size.  A shared prefix is stored with each sampled sequence (the oracle
    gathers every sequence's context on its own, so the work is the same)."""

    def __init__(self, seed: int, k: int, q8: bool = False, workload: str = "gqa_long"):
        import dataclasses

        import oracle
        from oracle.allocator_model import BlockLedger
        from paged_kv_cache_146_gb300 import workloads

        self.o = oracle.load()
        self.threads = self.o.max_threads()
        if workload in ("gqa_long", "gqa_long_q8"):
            w = workloads.gqa_long(seed, num_seqs=k, growth_tokens=16)
            full = 256
        else:
            wf = workloads.CONFIGS[workload](seed)
            full = wf.num_seqs
            k = min(k, full)
            prior, new = wf.prior_lens[:k].copy(), wf.new_tokens[:k].copy()
            need = int(sum(-(-int(a + b) // 16) for a, b in zip(prior, new)))
            w = dataclasses.replace(
                wf, prior_lens=prior, new_tokens=new, num_blocks=need,
                free_order=np.random.default_rng(seed + 7).permutation(need).astype(np.int32))
        v = workloads.host_values(w)
        k_prompt, v_prompt = v["k_prompt"], v["v_prompt"]
        if w.shared_prefix_tokens:          # rows of every cached token, sequence after sequence
            P, off, ks, vs = w.shared_prefix_tokens, 0, [], []
            for s in range(k):
                n = int(w.prior_lens[s]) - P
                ks += [v["k_shared"], k_prompt[off:off + n]]
                vs += [v["v_shared"], v_prompt[off:off + n]]
                off += n
            k_prompt, v_prompt = np.concatenate(ks), np.concatenate(vs)
        led = BlockLedger(w.num_blocks, 16, w.free_order)
        tables = [[-1] * w.max_blocks_per_seq for _ in range(k)]
        slots_p = led.append([0] * k, [int(x) for x in w.prior_lens], tables)
        slots_n = led.append([int(x) for x in w.prior_lens], [1] * k, tables)
        shape = (w.num_blocks, w.num_kv_heads, 16, w.head_dim)
        self.q8 = q8
        if q8:      # 8-bit cache: codes and fp16 scales written by the oracle's quantiser
            nb, hkv, d = w.num_blocks, w.num_kv_heads, w.head_dim
            self.pools = (np.zeros(shape, np.int8), np.zeros((nb, hkv, d, 16), np.int8),
                          np.zeros((nb, hkv, 16, d // 32), np.uint16),
                          np.zeros((nb, hkv, 16, d // 32), np.uint16))
            for kr, vr, sl in ((k_prompt, v_prompt, slots_p), (v["k_new"], v["v_new"], slots_n)):
                self.o.cache_write_q8(kr, vr, np.array(sl, dtype=np.int64), self.pools, 16, True)
        else:
            self.kp = np.zeros(shape, dtype=np.uint16)
            self.vp = np.zeros(shape, dtype=np.uint16)
            self.o.cache_write(k_prompt, v_prompt, np.array(slots_p, dtype=np.int64),
                               self.kp, self.vp, 16)
            self.o.cache_write(v["k_new"], v["v_new"], np.array(slots_n, dtype=np.int64),
                               self.kp, self.vp, 16)
        self.w, self.q = w, v["q"]
        self.tables = np.array(tables, dtype=np.int32)
        self.lens = (w.prior_lens + 1).astype(np.int32)
        self.tokens = int(self.lens.astype(np.int64).sum())
        per_head = 2 * (w.head_dim + w.head_dim // 16) if q8 else w.head_dim * 2 * 2
        self.nbytes = self.tokens * w.num_kv_heads * per_head + \
            2 * k * w.num_q_heads * w.head_dim * 2 + \
            4 * int(sum(-(-int(n) // 16) for n in self.lens)) + 4 * k
        self.desc = (f"first {k} of {full} sequences of {workload} ({self.tokens} context tokens"
                     + (", each storing the shared prefix itself" if w.shared_prefix_tokens else "")
                     + "), one decode call")

    def run(self) -> float:
        t0 = time.perf_counter()
        if self.q8:
            self.o.paged_decode_q8(self.q, self.pools, self.tables, self.lens, self.w.scale, True,
                                   self.threads)
        else:
            self.o.paged_decode(self.q, self.kp, self.vp, self.tables, self.lens, self.w.scale,
                                self.w.is_bf16, self.threads)
        return time.perf_counter() - t0


def oracle_calibrated(seed: int, target_s: float, q8: bool = False,
                      workload: str = "gqa_long", threads: int | None = None) -> OracleSample:
    """An oracle sample whose one call takes about ``target_s`` seconds on
    ``threads`` host threads (default: all)."""
    probe = OracleSample(seed, 2, q8, workload)
    if threads:
        probe.threads = threads
    dt = probe.run()
    k = int(min(256, max(2, round(2 * target_s / max(dt, 1e-3)))))
    sample = OracleSample(seed, k, q8, workload)
    if threads:
        sample.threads = threads
    return sample


def reference_arm(args, world, rank):
    """The oracle as the reference implementation, timed on the host cores."""
    if rank != 0:
        return
    per_step = min(args.ref_seconds, 150.0 / (args.steps + args.warmup))
    if args.workload not in DECODE_WORKLOADS:
        print(json.dumps({"impl": "reference", "unavailable":
                          f"the oracle baseline covers the decode workloads, not {args.workload}"}),
              flush=True)
        return
    from paged_kv_cache_146_gb300 import workloads
    q8 = args.workload == "gqa_long_q8"
    sample = oracle_calibrated(args.seed, per_step, q8, args.workload)
    w = sample.w
    w_full_seqs = (workloads.CONFIGS[args.workload](args.seed).num_seqs
                   if args.workload in workloads.CONFIGS and args.workload != "gqa_long" else 256)
    for _ in range(args.warmup):
        sample.run()
    secs = [sample.run() for _ in range(args.steps)]
    value = sample.nbytes / statistics.median(secs) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.median(secs), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload,
                       "num_seqs": args.num_seqs if args.workload in ("gqa_long", "gqa_long_q8")
                       else w_full_seqs,
                       "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                       "head_dim": w.head_dim, "block_size": 16,
                       "kv_dtype": "q8_bf16" if q8 else w.dtype, "lengths": LENGTHS[args.workload],
                       "shared_prefix_tokens": w.shared_prefix_tokens},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": sample.threads,
                             "kind": "oracle", "sample": sample.desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def decode_run(args, workload: str, world: int, rank: int, dev, steps: int, warmup: int,
               repeats: int = 1, e2e_steps: int = 0, prompt_write: bool = False,
               clocks: "ClockSampler | None" = None) -> dict:
    """Decode steps of one workload through DecodeEngine: ``warmup`` untimed
    steps, then ``repeats`` timed regions of ``steps`` steps each (barrier and
    synchronisation on both sides of every region), optionally ``e2e_steps``
    steps through the host-buffer call and one write of every prompt token."""
    import torch
    from paged_kv_cache_146_gb300 import KVPool, default_split, workloads
    from paged_kv_cache_146_gb300.engine import DecodeEngine

    e2e_warmup = 3 if e2e_steps > 0 else 0
    n_steps = warmup + steps * repeats + e2e_warmup + e2e_steps
    q8 = workload == "gqa_long_q8"
    if workload in ("gqa_long", "gqa_long_q8"):
        w = rank_workload(args.seed, rank, args.num_seqs, n_steps + 16)
    else:
        w = workloads.CONFIGS[workload](args.seed + rank)
        # room for the timed steps' growth
        need_b = -(-(int(w.prior_lens.max()) + n_steps + 16) // 16)
        if need_b > w.max_blocks_per_seq:
            w.max_blocks_per_seq = need_b
        need = sum(-(-(int(x) + n_steps + 16) // 16) for x in w.prior_lens) + 64
        if need > w.num_blocks:
            w.num_blocks = need
            w.free_order = np.random.default_rng(args.seed + 11).permutation(need).astype(np.int32)
    S, hq, hkv, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    vals = workloads.device_values(w, dev)
    pool = KVPool(w.num_blocks, hkv, d, "q8_" + w.dtype if q8 else w.dtype,
                  free_order=w.free_order, device=dev)
    eng = DecodeEngine(pool, S, hq, w.max_blocks_per_seq, w.scale, dev,
                       plan_on_host=not args.device_plan)
    if w.shared_prefix_tokens:
        first = np.zeros(S, dtype=np.int32)
        first[0] = w.shared_prefix_tokens
        eng.prefill(vals["k_shared"], vals["v_shared"], first)
        eng.share_prefix(w.shared_prefix_tokens)
        slots_p = eng.prefill(vals["k_prompt"], vals["v_prompt"],
                              w.prior_lens - w.shared_prefix_tokens)
    else:
        slots_p = eng.prefill(vals["k_prompt"], vals["v_prompt"], w.prior_lens)
    prompt_rows = (vals["k_prompt"], vals["v_prompt"], torch.from_numpy(slots_p).to(dev))
    vals.clear()
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 7 + rank)
    tdt = torch.bfloat16 if w.is_bf16 else torch.float16

    def draw(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(tdt)

    n_draw = warmup + steps          # the repeats cycle through the same step inputs
    qs = [draw(S, hq, d) for _ in range(n_draw)]
    ks = [draw(S, hkv, d) for _ in range(n_draw)]
    vs = [draw(S, hkv, d) for _ in range(n_draw)]
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        eng.host_step()
        if ev:
            ev[2].record(stream)
        eng.write(ks[i % n_draw], vs[i % n_draw])
        if ev:
            ev[0].record(stream)
        eng.attend(qs[i % n_draw])
        if ev:
            ev[1].record(stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    rc, word = eng.check()
    if rc != 0:
        raise SystemExit(f"device status {rc} word {word:#x} after warm-up ({workload})")

    ev = lambda: torch.cuda.Event(enable_timing=True)    # noqa: E731
    region_ms, region_bytes, region_toks, attn_ms, cw_ms = [], [], [], [], []
    if clocks is not None:
        clocks.start()
        time.sleep(0.25)
    i = warmup
    for _ in range(repeats):
        attn_ev = [(ev(), ev(), ev()) for _ in range(steps)]
        start, stop = ev(), ev()
        nbytes, toks = 0, 0
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(steps):
            step(i, attn_ev[k])
            i += 1
            nbytes += eng.step_bytes()
            toks += int(eng.lens.astype(np.int64).sum())
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        region_ms.append(max_over_ranks(start.elapsed_time(stop), world))
        region_bytes.append(nbytes)
        region_toks.append(toks)
        attn_ms += [a.elapsed_time(b) for a, b, _ in attn_ev]
        cw_ms += [c.elapsed_time(a) for a, _, c in attn_ev]
    clk = clocks.stop() if clocks is not None else None
    rc, word = eng.check()
    if rc != 0:
        raise SystemExit(f"device status {rc} word {word:#x} in the timed steps ({workload})")
    rates = [job_rate(b, world, t) for b, t in zip(region_bytes, region_ms)]
    med = sorted(range(repeats), key=lambda r: rates[r])[repeats // 2]
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    bytes_per_launch = sum(region_bytes) / (steps * repeats)
    res = {"w": w, "pool": pool, "q8": q8, "S": S, "hq": hq, "hkv": hkv, "d": d,
           "value": rates[med], "repeat_values": [round(r, 2) for r in rates],
           "ms_per_step": region_ms[med] / steps, "region_toks": region_toks[med],
           "region_ms": region_ms[med], "bytes_per_launch": bytes_per_launch,
           "attn_avg_ms": attn_avg_ms, "attn_median_ms": statistics.median(attn_ms),
           "toks_per_step": region_toks[med] / steps, "clocks": clk,
           # cache write, then: planned call -- [shared-prefix kernel] + main
           # [+ merge]; otherwise prep + main [+ merge] (the merge kernel runs
           # when a sequence may have several pieces)
           "launches_per_step": 1 + (1 + (eng.plan_prefix_items > 0) if eng.planned else 2)
           + (1 if eng.maxb > default_split() or (eng.planned and eng.plan_prefix_items > 0)
              else 0)}

    # ---- end to end through the public API with host buffers
    if e2e_steps > 0:
        n_e = e2e_warmup + e2e_steps
        hq_h = [qs[j % n_draw].cpu().pin_memory() for j in range(n_e)]
        hk_h = [ks[j % n_draw].cpu().pin_memory() for j in range(n_e)]
        hv_h = [vs[j % n_draw].cpu().pin_memory() for j in range(n_e)]
        out_h = [torch.empty_like(eng.out, device="cpu").pin_memory() for _ in range(n_e)]
        for j in range(e2e_warmup):      # untimed: copy streams and buffers come up here
            eng.decode_step_host(hq_h[j], hk_h[j], hv_h[j], out_h[j])
        eng.join_copies()
        hq_h, hk_h, hv_h, out_h = (x[e2e_warmup:] for x in (hq_h, hk_h, hv_h, out_h))
        e_start, e_stop = ev(), ev()
        e_bytes = 0
        barrier(world)
        torch.cuda.synchronize()
        e_start.record(stream)
        eng.copies_after(e_start)
        for j in range(e2e_steps):
            # inputs from pinned host memory, output back to it: transfers overlap
            # the neighbouring steps' kernels and stay inside the timed region
            eng.decode_step_host(hq_h[j], hk_h[j], hv_h[j], out_h[j])
            e_bytes += eng.step_bytes()
        eng.join_copies()
        e_stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = max_over_ranks(e_start.elapsed_time(e_stop), world)
        h2d = (hq_h[0].numel() + hk_h[0].numel() + hv_h[0].numel()) * 2 + \
            eng.h_tables.numel() * 4 + eng.h_lens.numel() * 4 + eng.h_slots.numel() * 8
        res["e2e"] = {"value": round(e_bytes * world / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(out_h[0].numel() * 2),
                      "ms_per_step": round(e_ms / e2e_steps, 4)}
        rc, word = eng.check()
        if rc != 0:
            raise SystemExit(f"device status {rc} word {word:#x} in the e2e steps")

    if prompt_write:
        # the cache write, reported on its own: the decode step's (one token per
        # sequence, timed above) and the prompts' (every prompt token, written
        # again into the same slots -- the cache is unchanged -- and timed once)
        k_pr, v_pr, d_slots_pr = prompt_rows
        c0, c1 = ev(), ev()
        torch.cuda.synchronize()
        c0.record(stream)
        eng.write(k_pr, v_pr, d_slots_pr)
        c1.record(stream)
        torch.cuda.synchronize()
        rc, word = eng.check()
        if rc != 0:
            raise SystemExit(f"device status {rc} word {word:#x} in the prompt write")
        row_out = (2 * (d + d // 32 * 2) if q8 else 2 * d * 2) * hkv   # K+V bytes stored per token
        row_in = 2 * d * 2 * hkv                                        # K+V bytes read per token
        T_pr = int(d_slots_pr.shape[0])
        cw_step_ms = sum(cw_ms) / len(cw_ms)
        res["cache_write"] = {
            "bytes": "T x (K+V row bytes read + stored) + 8 T",
            "step_tokens": S, "step_us": round(1e3 * cw_step_ms, 2),
            "step_gbs": round(S * (row_in + row_out + 8) / (cw_step_ms * 1e-3) / 1e9, 2),
            "prompt_tokens": T_pr, "prompt_ms": round(c0.elapsed_time(c1), 4),
            "prompt_gbs": round(T_pr * (row_in + row_out + 8) / (c0.elapsed_time(c1) * 1e-3) / 1e9,
                                2)}
    # the attention call alone on the final state, replayed back to back from a
    # CUDA graph on the engine's current buffers: one launch per call, so the
    # host's Python and launch overhead leaves no gaps in short calls
    from paged_kv_cache_146_gb300 import CapturedDecode
    qbuf = qs[0].clone()
    cap = CapturedDecode(pool, qbuf, eng.d_tables, eng.d_lens, w.scale, eng.workspace,
                         eng.status, eng.out,
                         planned_prefix_items=eng.plan_prefix_items if eng.planned else None)
    for _ in range(3):
        cap.replay()
    gev = [(ev(), ev()) for _ in range(20)]
    torch.cuda.synchronize()
    for a, b in gev:
        a.record(stream)
        cap.replay()
        b.record(stream)
    torch.cuda.synchronize()
    rc, word = eng.check()
    if rc != 0:
        raise SystemExit(f"device status {rc} word {word:#x} in the graph replays")
    res["graph_ms"] = statistics.median(a.elapsed_time(b) for a, b in gev)
    res["graph_bytes"] = eng.step_bytes()
    del prompt_rows, qs, ks, vs, eng, cap
    return res


def config_summary(args, workload: str, world: int, rank: int, dev) -> dict:
    """Attention-call rate of a further decode workload (20 timed steps after 3
    warm-ups), for the ``configs`` object of the headline line."""
    import torch
    r = decode_run(args, workload, world, rank, dev, steps=20, warmup=3)
    peak, _ = peaks()
    gms = r["graph_ms"]
    achieved = r["graph_bytes"] / (gms * 1e-3) / 1e9
    out = {"attention_gbs": round(achieved, 2), "pct_of_peak": round(100 * achieved / peak, 2),
           "attention_ms": round(gms, 4),
           "attention": "the call replayed back to back from a CUDA graph on the final state "
                        "(median of 20); attention_ms_in_step: the direct call inside the timed "
                        "steps, host launch gaps included",
           "attention_ms_in_step": round(r["attn_avg_ms"], 4),
           "step_gbs": round(r["value"], 2),
           "seq_tokens_per_s": round(r["toks_per_step"] / (gms * 1e-3), 1),
           "bytes_per_call": int(r["graph_bytes"]),
           "num_seqs": r["S"], "q_heads": r["hq"], "kv_heads": r["hkv"], "head_dim": r["d"],
           "kv_dtype": r["pool"].dtype, "lengths": LENGTHS[workload]}
    if workload == "shared_prefix":
        traffic = profiled_traffic(workload) if args.seed == 0 else None
        out["dram_bytes_per_call"] = traffic
        if traffic:
            out["dram_gbs"] = round(traffic / (gms * 1e-3) / 1e9, 2)
            out["dram_pct_of_peak"] = round(100 * out["dram_gbs"] / peak, 2)
    del r
    torch.cuda.empty_cache()
    return out


def our_arm(args, world, rank, local):
    import torch

    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_uuid)
    r = decode_run(args, args.workload, world, rank, dev, args.steps, args.warmup,
                   repeats=args.repeats, e2e_steps=args.e2e_steps, prompt_write=True,
                   clocks=clocks)
    w, q8, S, hq, hkv, d = r["w"], r["q8"], r["S"], r["hq"], r["hkv"], r["d"]
    peak, peak_kind = peaks()
    value = r["value"]
    attn_avg_ms = r["attn_avg_ms"]
    bytes_per_launch = r["bytes_per_launch"]
    achieved = bytes_per_launch / (attn_avg_ms * 1e-3) / 1e9
    dtype_name, pool_dtype = w.dtype, r["pool"].dtype
    e2e, cache_write_line = r.get("e2e"), r.get("cache_write")
    toks_region, region_ms = r["region_toks"], r["region_ms"]
    graph = {"ms": round(r["graph_ms"], 4),
             "gbs": round(r["graph_bytes"] / (r["graph_ms"] * 1e-3) / 1e9, 2),
             "what": "the attention call replayed back to back from a CUDA graph on the final "
                     "state, median of 20"}
    clk, repeat_values, launches = r["clocks"], r["repeat_values"], r["launches_per_step"]
    del r
    torch.cuda.empty_cache()

    # the other decode configurations, after the headline's timed regions
    configs = None
    if args.configs and args.workload == "gqa_long" and args.num_seqs == 256:
        configs = {}
        for wl in ("opt13b", "shared_prefix", "gqa_long_q8", "tiny"):
            configs[wl] = config_summary(args, wl, world, rank, dev)
        configs["trace"] = trace_summary(args, world, rank, dev)

    if rank != 0:
        return
    cpu = None
    if args.cpu_seconds > 0 and world == 1:
        sample = oracle_calibrated(args.seed, args.cpu_seconds, q8, args.workload)
        dt = sample.run()
        cpu = {"value": round(sample.nbytes / dt / 1e9, 4), "unit": "GB/s",
               "cores": sample.threads, "kind": "oracle", "sample": sample.desc,
               "seconds": round(dt, 2)}
        one = oracle_calibrated(args.seed, args.cpu_seconds / 2, q8, args.workload, threads=1)
        dt1 = one.run()
        cpu["single_thread"] = {"value": round(one.nbytes / dt1 / 1e9, 4), "unit": "GB/s",
                                "cores": 1, "sample": one.desc, "seconds": round(dt1, 2)}
    traffic = args.traffic
    if traffic is None and args.num_seqs == 256 and args.seed == 0 and not q8:
        traffic = profiled_traffic(args.workload)
    # where cached bytes are shared (a common prefix read by many sequences)
    # DRAM moves fewer bytes than the algorithmic count: report both
    dram = None
    if traffic is not None and args.workload == "shared_prefix":
        dram = {"bytes_per_launch": int(traffic),
                "gbs": round(traffic / (attn_avg_ms * 1e-3) / 1e9, 2),
                "pct_of_peak": round(100.0 * traffic / (attn_avg_ms * 1e-3) / 1e9 / peak, 2)}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(region_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name, "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs": S, "q_heads": hq, "kv_heads": hkv,
                   "head_dim": d, "block_size": 16, "kv_dtype": pool_dtype,
                   "lengths": LENGTHS[args.workload],
                   "shared_prefix_tokens": w.shared_prefix_tokens,
                   "mean_context": round(toks_region / args.steps / S, 1),
                   "pool_blocks": w.num_blocks,
                   "l2": ("inputs larger than L2 (KV per step ~%.1f GB vs 129 MB L2)"
                          % (bytes_per_launch / 1e9)
                          if not w.shared_prefix_tokens else
                          "unique KV larger than L2; the shared prefix (%d tokens) is re-read from L2"
                          % w.shared_prefix_tokens),
                   "timed": (f"{args.repeats} regions of {args.steps} steps, each bracketed by a "
                             "barrier and a synchronisation; value, ms_per_step = the median "
                             "region"),
                   "step": "host ledger + table/lens/slots H2D + cache_write + paged attention"},
        "seq_tokens_per_s": round(toks_region * world / (region_ms * 1e-3), 1),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "pct_of_nominal_8tbs": round(100.0 * value / 8000.0, 2),
        "repeat_values": repeat_values,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
                     "kernel": ("paged_decode_attention_q8" if q8 else "paged_decode_attention")
                     + (" (main kernel; work plan built on the host)" if not q8 else
                        " (prep + main + merge kernels)"),
                     "bytes_per_launch": int(bytes_per_launch),
                     "launch_ms": round(attn_avg_ms, 4)},
        "attention_graph": graph,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "cache_write": cache_write_line,
        **({"dram": dram} if dram else {}),
        **({"configs": configs} if configs else {}),
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def prefill_arm(args, world, rank, local):
    """Chunked-prefill attention: 16 prompts of 2048 tokens (GQA 32/8, D 128,
    bf16, or fp16 with --kv-dtype f16) whose K/V are cached, attended in one
    call; causal flops over time."""
    import torch
    from paged_kv_cache_146_gb300 import (KVPool, cache_write, paged_prefill_attention,
                                          prefill_workspace_bytes, workloads)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    S, P, hq, hkv, d = 16, 2048, 32, 8, 128
    T = S * P
    maxb = P // 16
    rng = np.random.default_rng(args.seed + rank)
    order = rng.permutation(S * maxb + 16).astype(np.int32)
    kvd = args.kv_dtype
    tdt = torch.bfloat16 if kvd == "bf16" else torch.float16
    pool = KVPool(S * maxb + 16, hkv, d, kvd, free_order=order, device=dev)
    tables = np.full((S, maxb), -1, dtype=np.int32)
    slots = pool.append_slots(np.zeros(S, np.int32), np.full(S, P, np.int32), tables)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 17 + rank)
    k = torch.randn(T, hkv, d, generator=gen, device=dev).to(tdt)
    v = torch.randn(T, hkv, d, generator=gen, device=dev).to(tdt)
    q = torch.randn(T, hq, d, generator=gen, device=dev).to(tdt)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cache_write(pool, k, v, torch.from_numpy(slots).to(dev), status)
    d_tables = torch.from_numpy(tables).to(dev)
    qs = torch.from_numpy(np.arange(0, T + 1, P, dtype=np.int32)).to(dev)
    lens = torch.full((S,), P, dtype=torch.int32, device=dev)
    # bf16 pools: room for the fp16 copy of V (made inside every timed call)
    # unless --prefill-plain asks for P V with two bf16 parts of P
    staged = kvd == "bf16" and not args.prefill_plain
    extra = (d, maxb) if staged else ()
    ws = torch.empty(prefill_workspace_bytes(S, T, hq, hkv, *extra), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    scale = 1.0 / math.sqrt(d)

    def call():
        paged_prefill_attention(pool, q, d_tables, qs, lens, scale, ws, status, out=out)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_uuid)     # a timed region of ~0.65 ms per step: pass --steps 300+
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    clocks.start()
    start.record()
    for _ in range(args.steps):
        call()
    stop.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(start.elapsed_time(stop) / args.steps, world)
    rc, word = __import__("paged_kv_cache_146_gb300").status_check(status)
    if rc != 0:
        raise SystemExit(f"device status {rc} word {word:#x}")
    if rank != 0:
        return
    # causal attention: each query at position p does 2*D flops per key for QK and
    # for PV over p + 1 keys
    flops = S * hq * 4 * d * (P * (P + 1) // 2)
    tflops = flops * world / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        tpeak, tkind = float(pk["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        tpeak, tkind = 1900.0, "fallback"
    line = {"metric": "chunked-prefill attention TFLOP/s", "value": round(tflops, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": kvd, "data": "synthetic",
            "config": {"workload": "prefill", "num_seqs": S, "prompt_tokens": P,
                       "q_heads": hq, "kv_heads": hkv, "head_dim": d, "block_size": 16},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak,
                         "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4),
                         "traffic": (profiled_traffic(summary="paged_prefill_tc_launches.md",
                                                      sources=PREFILL_SOURCES)
                                     if staged and args.seed == 0 else None),
                         "peak_kind": tkind,
                         "note": "tcgen05.mma kind::f16 (TMEM accumulators), two query tiles of "
                                 "128 rows per CTA, "
                                 + ("128-key tiles, P as one fp16 part, V copied to fp16 (scaled per "
                                    "sequence and kv head) by two kernels inside each call" if staged else
                                    "64-key tiles, "
                                    + ("P as bf16 high + low parts" if kvd == "bf16" else "P as one fp16 part"))},
            "gpu_launches": (4 if staged else 2) * args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def blocks_arm(args, world, rank, local):
    """Block movement for copy-on-write and swap, GQA 8 kv heads x 128, bf16 (64 KiB of K+V
    per block): ``cow`` -- one kv_block_copy call copying 8,192 random blocks
    into 8,192 others (copy-on-write of many forks at once); ``swap`` -- a
    2,048-block sequence (32K tokens) packed into staging (kv_gather_blocks),
    copied to pinned host memory and back, unpacked into fresh blocks
    (kv_scatter_blocks).  Kernel GB/s count bytes read + written."""
    import torch
    from paged_kv_cache_146_gb300 import (KVPool, block_copy, gather_blocks, scatter_blocks,
                                          status_check)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    hkv, d, bs = 8, 128, 16
    blk = 2 * hkv * bs * d * 2                         # K + V bytes of one block
    n = 8192 if args.workload == "cow" else 2048
    nb = 2 * n + 16
    rng = np.random.default_rng(args.seed + 31 + rank)
    pool = KVPool(nb, hkv, d, "bf16", device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 37 + rank)
    pool.k_pool.copy_(torch.randn(pool.k_pool.shape, generator=gen, device=dev))
    pool.v_pool.copy_(torch.randn(pool.v_pool.shape, generator=gen, device=dev))
    perm = rng.permutation(nb).astype(np.int32)
    src = torch.from_numpy(perm[:n]).to(dev)
    dst = torch.from_numpy(perm[n:2 * n]).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        barrier(world)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b) / args.steps, world)

    peak, peak_kind = peaks()
    extra = {}
    if args.workload == "cow":
        ms = timed(lambda: block_copy(pool, src, dst, status))
        nbytes = 2 * n * blk
        ok = torch.equal(pool.k_pool[dst.long()], pool.k_pool[src.long()]) and \
            torch.equal(pool.v_pool[dst.long()], pool.v_pool[src.long()])
        metric, kern = "kv_block_copy GB/s (bytes read + written)", "kv_block_copy"
        cfg = {"workload": "cow", "block_pairs": n, "kv_heads": hkv, "head_dim": d,
               "block_size": bs, "kv_dtype": "bf16", "bytes_per_call": nbytes}
    else:
        staging = torch.empty((n, 2, hkv, bs, d), dtype=torch.bfloat16, device=dev)
        host = torch.empty(staging.shape, dtype=torch.bfloat16, pin_memory=True)
        ms = timed(lambda: gather_blocks(pool, src, staging, status))
        ms_sc = timed(lambda: scatter_blocks(pool, dst, staging, status))
        ms_d2h = timed(lambda: host.copy_(staging, non_blocking=True))
        ms_h2d = timed(lambda: staging.copy_(host, non_blocking=True))
        nbytes = 2 * n * blk
        gather_blocks(pool, src, staging, status)
        scatter_blocks(pool, dst, staging, status)
        ok = torch.equal(pool.k_pool[dst.long()], pool.k_pool[src.long()])
        extra = {"scatter_gbs": round(nbytes / (ms_sc * 1e-3) / 1e9, 2),
                 "d2h_gbs": round(n * blk / (ms_d2h * 1e-3) / 1e9, 2),
                 "h2d_gbs": round(n * blk / (ms_h2d * 1e-3) / 1e9, 2),
                 "swap_out_ms": round(ms + ms_d2h, 4), "swap_in_ms": round(ms_h2d + ms_sc, 4)}
        metric, kern = "kv_gather_blocks GB/s (bytes read + written)", "kv_gather_blocks"
        cfg = {"workload": "swap", "blocks": n, "tokens": n * bs, "kv_heads": hkv, "head_dim": d,
               "block_size": bs, "kv_dtype": "bf16", "bytes_per_call": nbytes}
    rc, word = status_check(status)
    if rc != 0 or not ok:
        raise SystemExit(f"device status {rc} word {word:#x}, copies equal: {ok}")
    if rank != 0:
        return
    gbs = nbytes * world / (ms * 1e-3) / 1e9
    line = {"metric": metric, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 2),
                         "peak": peak, "unit": "GB/s",
                         "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "traffic": None,
                         "peak_kind": peak_kind, "kernel": kern},
            "gpu_launches": args.steps, **extra}
    print(json.dumps(line), flush=True)


def _pct(xs, q):
    xs = sorted(xs)
    return xs[int(q * (len(xs) - 1))]


def trace_run(args, world, rank, dev, steps: int | None = None) -> dict:
    """The continuous-batching trace (500 steps of FCFS admission, prefill,
    decode and release), the host enqueueing step after step with no
    synchronisation in between, so the host side of step t + 1 overlaps the
    GPU work of step t.  Per step: host seconds of each phase (perf_counter)
    and device milliseconds of each phase (CUDA events)."""
    import torch
    from paged_kv_cache_146_gb300 import workloads
    from paged_kv_cache_146_gb300.trace import TraceRunner
    sched = workloads.trace(seed=5 + args.seed + rank,
                            pool_bytes=int(args.pool_gib * 2**30) if args.pool_gib else 40 * 2**30)
    steps = sched.steps if steps is None else min(steps, sched.steps)
    order = np.random.default_rng(sched.seed).permutation(sched.num_blocks).astype(np.int32)
    run = TraceRunner(sched, dev, free_order=order)
    recs = []
    torch.cuda.synchronize()
    barrier(world)
    t_all = time.perf_counter()
    for t in range(steps):
        rec = run.step(t)
        recs.append((rec.kv_bytes, rec.extra["host_s"]))
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t_all
    barrier(world)
    device = run.finish()
    rc, word = run.check()
    if rc != 0:
        raise SystemExit(f"device status {rc} word {word:#x}")
    rates, attn, h2d, cw = [], [], [], []
    host = [[], [], [], []]
    for t, (kv_bytes, hs) in enumerate(recs):
        h2d_ms, cw_ms, ms = device[t]
        h2d.append(1e3 * h2d_ms)
        cw.append(1e3 * cw_ms)
        for i in range(4):
            host[i].append(1e6 * hs[i])
        if ms and kv_bytes:
            attn.append(ms)
            rates.append(kv_bytes / (ms * 1e-3) / 1e9)
    peak, _ = peaks()
    names = ("schedule_and_ledger", "wait_for_previous_handoff", "enqueue_device_work",
             "release_finished")

    def dist(xs):
        return {"median": round(statistics.median(xs), 2), "p90": round(_pct(xs, 0.9), 2)}

    res = {"steps": steps, "pool_blocks": sched.num_blocks,
           "attention_gbs_median": round(statistics.median(rates), 2),
           "attention_gbs_p90": round(_pct(rates, 0.9), 2),
           "attention_gbs_p10": round(_pct(rates, 0.1), 2),
           "pct_of_peak_median": round(100 * statistics.median(rates) / peak, 2),
           "attention_ms_median": round(statistics.median(attn), 4),
           "step_ms_pipelined": round(1e3 * wall_s / steps, 4),
           "phases": {"unit": "host phases in us (perf_counter), device phases in us "
                              "(CUDA events): median and p90 over steps",
                      "host": {n: dist(x) for n, x in zip(names, host)},
                      "device": {"h2d_tables_lens_slots": dist(h2d),
                                 "cache_write": dist(cw),
                                 "attention": dist([1e3 * a for a in attn])}},
           "swapped_gb": round(run.swapped_bytes / 1e9, 3),
           "total_s": round(wall_s, 2)}
    del run, recs
    torch.cuda.empty_cache()
    return res


def trace_summary(args, world, rank, dev) -> dict:
    return trace_run(args, world, rank, dev)


def trace_arm(args, world, rank, local):
    """Continuous-batching trace: 500 steps (or --steps) of FCFS admission,
    prefill, decode and release; per-step attention GB/s (CUDA events around the
    attention call), the pipelined step time and the per-phase split."""
    import torch
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    r = trace_run(args, world, rank, dev, steps=None if args.steps == 20 else args.steps)
    if rank != 0:
        return
    line = {"metric": METRIC, "value": r["attention_gbs_median"], "unit": "GB/s",
            "n_gpus": world, "steps": r["steps"], "warmup": 0,
            "ms_per_step": r["step_ms_pipelined"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "trace", "arrivals_per_step": 8, "prompt": "U[64,1024]",
                       "output": "Geometric(1/200) capped at 2048", "max_running": 512,
                       "pool_blocks": r["pool_blocks"],
                       "value": "median over steps of attention GB/s",
                       "ms_per_step": "wall time of the whole run / steps, host and GPU "
                                      "pipelined (no synchronisation between steps)"},
            **{k: v for k, v in r.items() if k not in ("steps", "pool_blocks")}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workload", default="gqa_long",
                    choices=["gqa_long", "gqa_long_q8", "tiny", "opt13b", "shared_prefix", "trace",
                             "prefill", "cow", "swap"],
                    help="gqa_long is the headline line; the others report their own config")
    ap.add_argument("--pool-gib", type=float, default=0.0,
                    help="trace only: pool size (default 40 GiB); small pools force swapping")
    ap.add_argument("--num-seqs", type=int, default=256,
                    help="sequences per GPU (256 is the workload; fewer only for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--device-plan", action="store_true",
                    help="decode workloads: the attention call plans its work on the device "
                         "(prep kernel) instead of taking the engine's host-built plan")
    ap.add_argument("--repeats", type=int, default=10,
                    help="timed regions of --steps steps each; the median region is reported")
    ap.add_argument("--configs", type=int, default=1,
                    help="1: the headline line also carries the other decode configurations")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "f16"],
                    help="cache dtype of the prefill workload")
    ap.add_argument("--prefill-plain", action="store_true",
                    help="prefill on a bf16 pool without the fp16 copy of V")
    ap.add_argument("--ref-seconds", type=float, default=8.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per attention launch from an ncu capture, if current")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        reference_arm(args, world, rank)
    elif args.workload == "trace":
        trace_arm(args, world, rank, local)
    elif args.workload == "prefill":
        prefill_arm(args, world, rank, local)
    elif args.workload in ("cow", "swap"):
        blocks_arm(args, world, rank, local)
    else:
        our_arm(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
