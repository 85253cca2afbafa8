"""Benchmark: one decode step (paged KV append + paged decode attention) of one layer.

Default workload: the Llama-3-8B-shaped decode layer (batch 64, context lengths uniform
in [512, 4096], Hq 32 / Hkv 8, D 128, 16-token blocks, bf16 KV, shuffled pool, 64 new
tokens appended before attention).  Every value is seeded synthetic data.

Metric: achieved HBM GB/s of the step = algorithmic bytes / device time, where the
algorithmic bytes are the unique valid KV bytes the attention must read (shared blocks
once) plus q, the output, the block tables and lengths, and the append's reads and writes.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
Under torchrun each rank runs its own replica (independent sequences, no collective on the
data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged decode attention achieved HBM GB/s (fraction of 8 TB/s); µs/decode step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20  # about twice the 129 MB L2
HOST_LEAD_CYCLES = 500_000  # about 0.25 ms of GPU spin at 2 GHz, untimed (see lead())


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="llama3_8b", choices=W.ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="step", choices=["step", "copy_blocks"],
                    help="step: append + decode attention (the headline); copy_blocks: the copy-on-write "
                         "block copy alone")
    ap.add_argument("--layout", default="shuffled", choices=["shuffled", "contiguous"],
                    help="physical block order of the pool (contiguous = each sequence's blocks in order)")
    ap.add_argument("--copy-pairs", type=int, default=4096, help="(src, dst) pairs per copy_blocks launch")
    ap.add_argument("--cascade", action="store_true",
                    help="decode through the cascade call: shared prefixes once for all their members "
                         "(tensor cores), each sequence's own blocks by the decode kernel")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--l2", choices=("flushed", "warm"), default="flushed",
                    help="flushed (default): L2 flushed between timed steps; warm: no flush, a diagnostic of "
                         "the reuse the shared-prefix and fork workloads get when a step follows a step")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time only the --config workload, not the other target workloads next to it")
    ap.add_argument("--no-read-ceiling", action="store_true",
                    help="skip the read-only checksum pass that gives the ceiling of the decode's reads")
    ap.add_argument("--no-clock-fill", action="store_true",
                    help="do not run the untimed clock-sampling loop when the timed region is too short "
                         "(for profiler runs)")
    return ap.parse_args()


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest of every rank's x (timings: the job is as slow as its slowest rank); one
    all-reduce outside the data path, and nothing to do for a single rank."""
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ byte accounting

def step_bytes(w: W.Workload) -> dict:
    """Algorithmic bytes of one step (the roofline numerator)."""
    c = w.cfg
    B = w.batch
    kv = w.unique_kv_bytes()
    q = B * c.hq * c.d * 2
    out = B * c.hq * c.d * 2
    meta = sum((s.length + 15) // 16 for s in w.seqs) * 4 + B * 4 + (2 * c.hkv * 4 if w.scales is not None else 0)
    T = w.slot_mapping.numel()
    append = T * c.hkv * c.d * 2 * 2 + T * c.hkv * c.d * c.elem_bytes * 2 + T * 8
    decode = kv + q + out + meta
    return {"decode": decode, "append": append, "step": decode + append, "unique_kv": kv,
            "logical_kv": w.logical_kv_bytes()}


def decode_kernel_name(cfg, cascade: bool, w=None) -> str:
    """The kernels inside the decode call's timed interval (the merge runs for split
    sequences, and for cascades, whose prefix records it merges).  A cascade's prefix pass
    runs on mma.sync for groups of at most 32 query rows over an E4M3 pool, else on tcgen05."""
    tc = os.environ.get("PKV_DECODE_CUDA_CORES") != "1"  # both pool types run the tensor-core form
    core = "paged_decode_mma_kernel (tensor cores)" if tc else "paged_decode_kernel (CUDA cores)"
    name = core + " + merge_partitions_kernel"
    if not cascade:
        return name
    small = False
    if w is not None and w.scales is not None:
        c = w.cascade()
        small = c.max_members * (cfg.hq // cfg.hkv) <= 32
    if not small or os.environ.get("PKV_PREFIX_PASS") == "tc":
        return "cascade_prefix_tc_kernel (tcgen05) + " + name
    return "cascade_prefix_mma_kernel (mma.sync) + " + name


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_17_gb300", "csrc")
    for name in ("decode_kernel.cuh", "decode_mma.cuh", "mma_ops.cuh", "pkv_device.cuh", "decode_launch.cuh",
                 "merge_partitions.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(config: str):
    """DRAM bytes per decode launch from the committed ncu summary of this workload, if it
    was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"decode_{config}_ncu.md")
    if not os.path.exists(p):
        return None
    digest, traffic = None, None
    with open(p) as f:
        for line in f:
            if line.startswith("kernel_source_digest:"):
                digest = line.split(":", 1)[1].strip()
            if line.startswith("dram_bytes_per_launch:"):
                traffic = int(line.split(":", 1)[1].strip())
    return traffic if digest == kernel_source_digest() else None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict:
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(sms)
        loaded = [s for s in sms if s >= 0.5 * top] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------ CPU baseline (the oracle)

def oracle_sample(w: W.Workload, budget_s: float, threads: int):
    """Time the fp64 CPU oracle on whole (sequence, kv head) groups of this workload -- a
    prefix of the groups if the whole step takes longer than budget_s, else whole steps
    repeated until about budget_s seconds; returns (GB/s of unique KV, seconds,
    description, bytes)."""
    import oracle

    a = w.np()
    c = w.cfg
    g = c.g
    per_tok = 2 * c.d * c.elem_bytes  # K+V bytes of one token of one kv head
    b0 = 0
    pairs = np.array([(b0, hq) for hq in range(g)], dtype=np.int32)
    t0 = time.perf_counter()
    oracle.decode_pairs(a["q"], a["k_cache"], a["v_cache"], w.kv_dtype_code, a["block_tables"], a["context_lens"],
                        c.softmax_scale, pairs, scales=a["scales"], nthreads=1)
    sec_per_tok = (time.perf_counter() - t0) / max(1, w.seqs[b0].length)
    target_tok = budget_s * threads / max(sec_per_tok, 1e-12)
    groups, tok = [], 0
    for b in range(w.batch):
        for h in range(c.hkv):
            if tok >= target_tok:
                break
            groups.append((b, h))
            tok += w.seqs[b].length
    pairs = np.array([(b, h * g + i) for (b, h) in groups for i in range(g)], dtype=np.int32)
    reps, dt = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.decode_pairs(a["q"], a["k_cache"], a["v_cache"], w.kv_dtype_code, a["block_tables"],
                            a["context_lens"], c.softmax_scale, pairs, scales=a["scales"], nthreads=threads)
        dt += time.perf_counter() - t0
        reps += 1
        if dt >= 0.8 * budget_s or len(groups) < w.batch * c.hkv:
            break
    nbytes = tok * per_tok * reps
    whole = len(groups) == w.batch * c.hkv
    desc = (f"{'the whole step' if whole else f'{len(groups)} of {w.batch * c.hkv} (sequence, kv head) groups'}"
            f" x {reps} ({tok} tokens, {tok * per_tok / 1e6:.1f} MB of KV per pass), all {g} query heads of "
            f"each group; fp64 C oracle on {threads} threads")
    one_core = per_tok / max(sec_per_tok, 1e-12) / 1e9  # the first (sequence, kv head) group, one thread
    return nbytes / dt / 1e9, dt, desc, nbytes, one_core


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ our arm

# the workloads timed next to the headline one, each with the decode call that suits it
EXTRA_CONFIGS = (("long_context_70b", False), ("prefix_shared", True), ("fp8_fork", True))


def config_dict(cfg, w: W.Workload, layout: str, cascade: bool, ws: int, cold: bool = True) -> dict:
    """The workload description both arms print (nothing in it depends on the GPU)."""
    B = w.batch
    lens = cfg.len_range if cfg.kind == "uniform" else "mixed"
    return {"workload": f"{cfg.name}: batch {B}, context {lens}, Hq {cfg.hq}, Hkv {cfg.hkv}, D {cfg.d}, block 16, "
                        f"{cfg.kv_dtype} KV, append {w.slot_mapping.numel()} tokens",
            "batch": B, "num_q_heads": cfg.hq, "num_kv_heads": cfg.hkv, "head_dim": cfg.d, "kv_dtype": cfg.kv_dtype,
            "max_context_len": int(w.context_lens.max()), "total_context_tokens": w.total_tokens(),
            "layout": layout, "decode_call": "cascade" if cascade else "paged",
            "l2": ("flushed between timed steps: 256 MiB write, then a 256 MiB read of another buffer "
                   "(both untimed; the read writes the dirty lines back before the step)") if cold else
                  "warm: no flush between steps (diagnostic; each step finds the previous step's lines)",
            "parallelism": f"replicas x{ws}"}


class Timed:
    """One workload resident on the device, its step (append + decode) and the timed loops
    every measurement here shares: an untimed L2 flush and host-lead spin before each timed
    step, CUDA events on the launching stream around it."""

    def __init__(self, pkv, args, cfg, w: W.Workload, dev, cascade: bool):
        self.pkv, self.args, self.cfg, self.w, self.dev = pkv, args, cfg, w, dev
        B, hq, hkv, d = w.batch, cfg.hq, cfg.hkv, cfg.d
        self.max_len = int(w.context_lens.max())
        self.t = {k: (v.to(dev) if v is not None else None) for k, v in
                  dict(q=w.q, k_cache=w.k_cache, v_cache=w.v_cache, k_new=w.k_new, v_new=w.v_new,
                       slots=w.slot_mapping, tables=w.block_tables, lens=w.context_lens, scales=w.scales).items()}
        self.out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=dev)
        self.cas = w.cascade() if cascade else None
        if self.cas is not None:
            self.ct = {k: getattr(self.cas, k).to(dev) for k in ("prefix_tables", "prefix_lens", "member_indptr",
                                                                 "member_seqs", "seq_prefix", "block_tables",
                                                                 "context_lens")}
            self.dec_len = max(16, int(self.cas.context_lens.max()))
            need = pkv.cascade_workspace_size(B, hq, hkv, d, self.dec_len, self.cas.prefix_tables.shape[0],
                                              self.cas.max_members, self.cas.max_prefix_len)
        else:
            self.dec_len = self.max_len
            need = pkv.workspace_size(B, hq, hkv, d, self.max_len)
        self.wsbuf = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        self.sums = torch.empty((B, hkv, 2), dtype=torch.int32, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.scrub = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()
        self.cold = args.l2 == "flushed"

    def decode(self, q, tables, lens, ctabs=None, out=None):
        pkv, t, cfg = self.pkv, self.t, self.cfg
        out = self.out if out is None else out
        if self.cas is None:
            pkv.paged_decode_attention(q, t["k_cache"], t["v_cache"], tables, lens, cfg.softmax_scale, out,
                                       scales=t["scales"], max_context_len=self.max_len, workspace=self.wsbuf)
        else:
            c2 = ctabs or self.ct
            pkv.cascade_decode_attention(q, t["k_cache"], t["v_cache"], c2["prefix_tables"], c2["prefix_lens"],
                                         c2["member_indptr"], c2["member_seqs"], c2["seq_prefix"],
                                         c2["block_tables"], c2["context_lens"], cfg.softmax_scale, out,
                                         max_members=self.cas.max_members, max_prefix_len=self.cas.max_prefix_len,
                                         max_context_len=self.dec_len, scales=t["scales"], workspace=self.wsbuf)

    def step(self, mark=None):
        t = self.t
        self.pkv.paged_kv_append(t["k_new"], t["v_new"], t["slots"], t["k_cache"], t["v_cache"], scales=t["scales"])
        if mark is not None:
            mark.record(self.stream)
        self.decode(t["q"], t["tables"], t["lens"])

    def fused_step(self, inputs=None, out=None):
        """The step in one call (append fused into the decode; plain decode only)."""
        t = self.t
        i = inputs or dict(k_new=t["k_new"], v_new=t["v_new"], slots=t["slots"], q=t["q"], tables=t["tables"],
                           lens=t["lens"])
        out = self.out if out is None else out
        self.pkv.paged_append_decode(i["k_new"], i["v_new"], i["slots"], i["q"], t["k_cache"], t["v_cache"],
                                     i["tables"], i["lens"], self.cfg.softmax_scale, out, scales=t["scales"],
                                     max_context_len=self.max_len, workspace=self.wsbuf)

    def user_step(self):
        """The step as a user runs it: the fused call for the plain decode, append then the
        cascade call for shared prefixes."""
        if self.cas is None:
            self.fused_step()
        else:
            self.step()

    def read_pass(self):
        t = self.t
        self.pkv.kv_checksum(t["k_cache"], t["v_cache"], t["tables"], t["lens"], self.sums, scales=t["scales"],
                             max_context_len=self.max_len)

    def evict(self, i):
        if self.cold:
            self.flush.fill_(i & 0xFF)  # evict the previous step's lines from L2 (not timed)

    def lead(self):
        # Untimed, between the L2 flush and the step: a read of a second buffer larger than
        # L2, which writes back the flush's dirty lines and leaves L2 holding clean, unrelated
        # lines (the timed kernel then pays for its own traffic only, as under ncu's cache
        # control), then a GPU spin long enough for this Python host loop to queue the whole
        # step before the GPU reaches it.
        if self.cold:
            self.scrub.amax()
        torch.cuda._sleep(HOST_LEAD_CYCLES)

    def warm(self, n):
        for _ in range(n):
            self.flush.fill_(1)
            self.step()
            if self.cas is None:
                self.fused_step()
        torch.cuda.synchronize()
        assert self.pkv.check_device_status() == 0

    def timed(self, n, body, split_mark=False):
        """Per-step milliseconds of `body` over n timed steps; with split_mark, the time from
        a mark that the body records (between the append and the decode) to its end."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            self.evict(i)
            self.lead()
            if split_mark:
                body(evs[i][0])
            else:
                evs[i][0].record(self.stream)
                body()
            evs[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for (a, b) in evs]


def summary_entry(tm: Timed, step_ms, dec_ms, read_ms, peak: float, ws: int, dev) -> dict:
    """The per-workload figures: step and decode time, unique-byte GB/s and roofline
    fractions, sequence-steps per second, and the read-only ceiling when it was timed."""
    nb = step_bytes(tm.w)
    B = tm.w.batch
    step_tot = max_over_ranks(sum(step_ms), ws, dev)
    dec_tot = max_over_ranks(sum(dec_ms), ws, dev)
    n = len(step_ms)
    dec_avg = dec_tot / n
    achieved = nb["decode"] / (dec_avg * 1e-3) / 1e9
    e = {"decode_call": "cascade" if tm.cas is not None else "paged", "batch": B,
         "total_context_tokens": tm.w.total_tokens(), "unique_kv_bytes": nb["unique_kv"],
         "kernel": decode_kernel_name(tm.cfg, tm.cas is not None, tm.w),
         "decode_bytes": nb["decode"], "step_us": round(step_tot / n * 1e3, 2), "decode_us": round(dec_avg * 1e3, 2),
         "decode_us_p10_p50_p90": [round(float(x) * 1e3, 2) for x in np.percentile(dec_ms, [10, 50, 90])],
         "unique_kv_gbs": round(nb["unique_kv"] / (dec_avg * 1e-3) / 1e9, 1),
         "decode_gbs": round(achieved, 1), "roofline_frac": round(achieved / peak, 4),
         "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
         "seq_steps_per_s": round(B * ws * n / (step_tot * 1e-3), 1),
         "decode_seq_steps_per_s": round(B * ws * n / (dec_tot * 1e-3), 1)}
    if read_ms:
        rd = max_over_ranks(sum(read_ms), ws, dev) / len(read_ms)
        rbytes = nb["unique_kv"] + sum((s.length + 15) // 16 for s in tm.w.seqs) * 4 + B * 4
        e["read_ceiling"] = {"us": round(rd * 1e3, 2), "gbs": round(rbytes / (rd * 1e-3) / 1e9, 1),
                             "frac": round(rbytes / (rd * 1e-3) / 1e9 / peak, 4),
                             "kernel": "kv_checksum_kernel (the decode's TMA gather, no arithmetic)"}
    return e


def run_ours(args):
    import paged_kv_cache_17_gb300 as pkv

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = W.get(args.config)
    w = W.make_workload(cfg, seed=cfg.seed + 1000 * rank, layout=args.layout)
    tm = Timed(pkv, args, cfg, w, dev, args.cascade)
    nb = step_bytes(w)
    B, hq, hkv, d = w.batch, cfg.hq, cfg.hkv, cfg.d
    max_len = tm.max_len
    cas = tm.cas
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS

    tm.warm(args.warmup)
    with ClockSampler(dev.index) as clk:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        # the step as a user runs it: one call that appends each sequence's new token and
        # decodes (the cascade: append, then the cascade call)
        step_ms = tm.timed(args.steps, tm.user_step)
        # the decode alone (the roofline figure): the two calls with an event between them
        dec_ms = tm.timed(args.steps, lambda mark: tm.step(mark=mark), split_mark=True)
        # the two calls back to back, for comparison with the fused step
        two_call_ms = tm.timed(args.steps, tm.step) if cas is None else step_ms
        if ws > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - wall0
    clocks = clk.summary()
    if clocks.get("samples", 0) < 3 and not args.no_clock_fill:
        # the timed region was shorter than the sampler's period: sample the same step loop
        # for another half second (untimed) and say so
        with ClockSampler(dev.index) as clk2:
            t_end = time.perf_counter() + 0.5
            while time.perf_counter() < t_end:
                for _ in range(50):
                    tm.flush.fill_(3)
                    tm.user_step()
                torch.cuda.synchronize()
        clocks = clk2.summary()
        clocks["window"] = "same step loop, 0.5 s right after the timed region (timed region too short)"
    else:
        clocks["window"] = "timed region"
    # the read-only ceiling of the same gather (untimed warm-up, then the same protocol)
    read_ms = []
    if not args.no_read_ceiling and cas is None:
        tm.read_pass()
        torch.cuda.synchronize()
        read_ms = tm.timed(args.steps, tm.read_pass)
    assert pkv.check_device_status() == 0
    tot_ms = max_over_ranks(sum(step_ms), ws, dev)
    value = nb["step"] * ws * args.steps / (tot_ms * 1e-3) / 1e9
    ms_per_step = tot_ms / args.steps
    head = summary_entry(tm, step_ms, dec_ms, read_ms, peak, ws, dev)
    dec_avg_ms = head["decode_us"] * 1e-3
    achieved = head["decode_gbs"]

    # our kernels per step: append, [prefix pass], decode, [merge: of split sequences, or of
    # the prefix records, which the tensor-core decode leaves to it]; the fused step has no
    # separate append (the CUDA-core form runs the two calls)
    dec_len = tm.dec_len
    has_prefix = cas is not None and cas.prefix_tables.shape[0] > 0
    tensor_core = os.environ.get("PKV_DECODE_CUDA_CORES") != "1"
    deferred = has_prefix and tensor_core and os.environ.get("PKV_CASCADE_DEFER", "1") == "1"
    split = dec_len > pkv.partition_tokens(B, hkv, dec_len)
    launches_per_step = 2 + (1 if has_prefix else 0) + (1 if split or deferred else 0)
    user_launches = launches_per_step - (1 if cas is None and tensor_core else 0)
    launches = user_launches * args.steps + launches_per_step * args.steps + len(read_ms)
    if cas is None:
        launches += launches_per_step * args.steps  # the two-call comparison pass

    # ---- end to end through the public API with host buffers (pinned), H2D + D2H timed
    e2e = None
    if not args.no_e2e:
        inputs = dict(q=w.q, k_new=w.k_new, v_new=w.v_new, slots=w.slot_mapping, tables=w.block_tables,
                      lens=w.context_lens)
        if cas is not None:
            inputs.update({"c_" + k: getattr(cas, k) for k in tm.ct})
        # the step's inputs staged in one pinned host buffer (256-byte aligned fields), copied
        # to the device in one transfer per step by the SMs (pkv_stage_copy: a copy-engine
        # transfer of this size costs about 10 us of latency); the calls take device views
        # into it, and the output comes back the same way
        offs, total = {}, 0
        for k, v in inputs.items():
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
        d_pack = torch.empty(total, dtype=torch.uint8, device=dev)
        dev_in = {}
        for k, v in inputs.items():
            n = v.numel() * v.element_size()
            h_pack[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8))
            dev_in[k] = d_pack[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
        h_out = torch.empty((B, hq, d), dtype=torch.bfloat16).pin_memory()
        h2d = total
        d2h = h_out.numel() * h_out.element_size()

        def user_call(ins, out):
            """The step through the public API on device views of the staged inputs."""
            if cas is None:
                tm.fused_step(ins, out=out)
            else:
                pkv.paged_kv_append(ins["k_new"], ins["v_new"], ins["slots"], tm.t["k_cache"], tm.t["v_cache"],
                                    scales=tm.t["scales"])
                ctabs = {k[2:]: v for k, v in ins.items() if k.startswith("c_")}
                tm.decode(ins["q"], ins["tables"], ins["lens"], ctabs, out=out)

        # (1) one step at a time: the H2D copy, the step and the D2H copy back to back on one
        # stream (the SMs copy: pkv_stage_copy), each step behind the untimed L2 flush
        def e2e_step():
            pkv.stage_copy(d_pack, h_pack)
            user_call(dev_in, tm.out)
            pkv.stage_copy(h_out, tm.out)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        serial_ms = max_over_ranks(sum(tm.timed(args.steps, e2e_step)), ws, dev)
        launches += (user_launches + 2) * args.steps  # the step and its two staging copies

        # (2) as a serving loop runs it: step i + 1's inputs go up and step i - 1's output
        # comes back on a second stream (copy engines) while step i computes; two input packs
        # and two outputs alternate.  The pool is larger than L2, so no flush runs between
        # these steps and one pair of events brackets all of them, after an untimed spin that
        # lets the host queue the whole loop first.
        packs = [d_pack, torch.empty_like(d_pack)]
        ins2 = {k: packs[1][offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                for k, v in inputs.items()}
        ins_of = [dev_in, ins2]
        outs = [tm.out, torch.empty_like(tm.out)]
        h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
        comp = torch.cuda.current_stream(dev)
        cs = torch.cuda.Stream(device=dev)

        def pipelined(n, timed, copies=True):
            in_ready = [torch.cuda.Event(), torch.cuda.Event()]
            pack_free = [torch.cuda.Event(), torch.cuda.Event()]
            out_ready = [torch.cuda.Event(), torch.cuda.Event()]
            out_free = [torch.cuda.Event(), torch.cuda.Event()]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(cs):
                torch.cuda._sleep(HOST_LEAD_CYCLES * 4 * (n + 2))  # untimed: the host queues the loop
                t0.record(cs)
                if copies:
                    packs[0].copy_(h_pack, non_blocking=True)
                in_ready[0].record(cs)
            for i in range(n):
                j = i % 2
                comp.wait_event(in_ready[j])
                if i >= 2:
                    comp.wait_event(out_free[j])  # the D2H of step i - 2 has read outs[j]
                user_call(ins_of[j], outs[j])
                out_ready[j].record(comp)
                pack_free[j].record(comp)
                with torch.cuda.stream(cs):
                    if i + 1 < n:
                        jn = (i + 1) % 2
                        if i >= 1:
                            cs.wait_event(pack_free[jn])  # step i - 1 is done with packs[jn]
                        if copies:
                            packs[jn].copy_(h_pack, non_blocking=True)
                        in_ready[jn].record(cs)
                    cs.wait_event(out_ready[j])
                    if copies:
                        h_outs[j].copy_(outs[j], non_blocking=True)
                    out_free[j].record(cs)
            t1.record(cs)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) if timed else 0.0

        pipelined(max(args.warmup, 3), False)
        assert pkv.check_device_status() == 0
        e2e_ms = max_over_ranks(pipelined(args.steps, True), ws, dev)
        # the same loop with the copies left out: the device-only step in this steady state
        loop_ms = max_over_ranks(pipelined(args.steps, True, copies=False), ws, dev)
        e2e = {"value": round(nb["step"] * ws * args.steps / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_ms / args.steps, 4),
               "seq_steps_per_s": round(B * ws * args.steps / (e2e_ms * 1e-3), 1),
               "pipelined": True, "copies": "copy engines, on a second stream",
               "l2": "not flushed between steps (the KV pool is larger than L2)",
               "same_loop_without_copies_ms_per_step": round(loop_ms / args.steps, 4),
               "serial": {"value": round(nb["step"] * ws * args.steps / (serial_ms * 1e-3) / 1e9, 2),
                          "unit": "GB/s", "ms_per_step": round(serial_ms / args.steps, 4),
                          "seq_steps_per_s": round(B * ws * args.steps / (serial_ms * 1e-3), 1),
                          "copies": "SMs (pkv_stage_copy), on the step's stream",
                          "l2": "flushed before every step (untimed)"}}
        launches += 2 * user_launches * args.steps  # the pipelined loop, with and without its copies
    head_partition = pkv.partition_tokens(B, hkv, max_len)
    del tm
    torch.cuda.empty_cache()

    # ---- the other target workloads, the same protocol (decode call as suits each)
    extras = {}
    if not args.no_extra_configs:
        for name, cascade in EXTRA_CONFIGS:
            if name == args.config and cascade == args.cascade:
                continue
            xc = W.get(name)
            xw = W.make_workload(xc, seed=xc.seed + 1000 * rank, layout=args.layout)
            xt = Timed(pkv, args, xc, xw, dev, cascade)
            xt.warm(args.warmup)
            with ClockSampler(dev.index) as xclk:
                x_step = xt.timed(args.steps, xt.user_step)
                x_dec = xt.timed(args.steps, lambda mark: xt.step(mark=mark), split_mark=True)
            x_read = []
            if not args.no_read_ceiling and not cascade:
                xt.read_pass()
                torch.cuda.synchronize()
                x_read = xt.timed(args.steps, xt.read_pass)
            assert pkv.check_device_status() == 0
            entry = summary_entry(xt, x_step, x_dec, x_read, peak, ws, dev)
            entry["config"] = config_dict(xc, xw, args.layout, cascade, ws, xt.cold)
            entry["partition_tokens"] = pkv.partition_tokens(xw.batch, xc.hkv, xt.dec_len)
            xs = xclk.summary()
            entry["clocks"] = {k: xs.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")}
            xsplit = xt.dec_len > entry["partition_tokens"]
            xprefix = xt.cas is not None and xt.cas.prefix_tables.shape[0] > 0
            xdefer = xprefix and tensor_core and os.environ.get("PKV_CASCADE_DEFER", "1") == "1"
            x_per_step = 2 + (1 if xprefix else 0) + (1 if xsplit or xdefer else 0)
            x_user = x_per_step - (1 if xt.cas is None and tensor_core else 0)
            launches += (x_user + x_per_step) * args.steps + len(x_read)
            extras[name + ("_cascade" if cascade else "")] = entry
            del xt
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        thr = host_threads()
        gbs, dt, desc, _, one = oracle_sample(w, args.cpu_seconds, thr)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2), "value_one_core": round(one, 4)}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg.kv_dtype == "bf16" else "e4m3",
        "data": f"synthetic (seeded N(0,1) bf16 q/K/V, {args.layout} 16-token block pool)",
        "config": config_dict(cfg, w, args.layout, args.cascade, ws, args.l2 == "flushed"),
        "partition_tokens": head_partition,
        "us_per_step": round(ms_per_step * 1e3, 2),
        "step_call": "paged_append_decode (one call: the append fused into the decode)" if cas is None else
                     "paged_kv_append + cascade_decode_attention",
        "two_call_step_us": round(max_over_ranks(sum(two_call_ms), ws, dev) / args.steps * 1e3, 2),
        "seq_steps_per_s": round(B * ws * args.steps / (tot_ms * 1e-3), 1),
        "frac_of_8tbs": round(value / NOMINAL_HBM_GBS, 4),
        "bytes_per_step": nb,
        "decode_us": head["decode_us"],
        "decode_us_p10_p50_p90": head["decode_us_p10_p50_p90"],
        "decode_seq_steps_per_s": head["decode_seq_steps_per_s"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None if cas is not None else ncu_traffic(cfg.name),
                     "kernel": decode_kernel_name(cfg, cas is not None, w),
                     "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)},
        "read_ceiling": head.get("read_ceiling"),
        "configs": extras,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": launches,
        "timing": "step: events around the step as a user runs it (the fused append + decode call; cascades: "
                  "append, then the cascade call); two_call_step_us: events around append + decode as two calls; "
                  "decode_us: events around the decode alone (the two calls with an event between them); read_ceiling: events around the read-only checksum pass over the "
                  "same tables; e2e: the public API with host buffers as a serving loop runs it: one pair of "
                  "events around all steps, each step's inputs (one pinned buffer) copied H2D on a second stream "
                  "(copy engines) while the previous step computes and its output copied D2H while the next one "
                  "computes, two input packs and two outputs alternating, no L2 flush between these steps (the "
                  "pool is larger than L2); e2e.serial: events around one H2D copy of the step's inputs (copied "
                  "by the SMs: pkv_stage_copy) + the step + the D2H of the output (the same way); every other "
                  "timed step, e2e.serial's included, follows an untimed L2 flush and an untimed GPU spin that "
                  "lets the host queue the step first; configs: the other target workloads under the same "
                  "protocol",
        "clocks": clocks,
        "wall_s": round(wall, 3),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ copy-on-write block copy

def copy_pairs(num_blocks: int, n: int, seed: int) -> torch.Tensor:
    """n (src, dst) pairs over disjoint random blocks (no dst is also a src)."""
    n = min(n, num_blocks // 2)
    perm = torch.randperm(num_blocks, generator=torch.Generator().manual_seed(seed))
    return torch.stack([perm[:n], perm[n:2 * n]], dim=1).contiguous()


def oracle_copy_sample(w: W.Workload, pairs: torch.Tensor, budget_s: float):
    """Time the oracle's block copy (one host thread) on the same pool and pairs."""
    import oracle

    a = w.np()
    kc, vc = a["k_cache"], a["v_cache"]
    pr = pairs.numpy()
    moved = 2 * 2 * pr.shape[0] * kc[0].nbytes  # K and V, read + write
    reps, dt = 0, 0.0
    while dt < budget_s:
        t0 = time.perf_counter()
        oracle.copy_blocks(kc, vc, pr)
        dt += time.perf_counter() - t0
        reps += 1
    return moved * reps / dt / 1e9, dt, reps


def run_copy_blocks(args):
    import paged_kv_cache_17_gb300 as pkv

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = W.get(args.config)
    w = W.make_workload(cfg, seed=cfg.seed + 1000 * rank, layout=args.layout)
    pairs_h = copy_pairs(w.num_blocks, args.copy_pairs, cfg.seed + 77 + 1000 * rank)
    n = pairs_h.shape[0]
    block_bytes = 16 * cfg.hkv * cfg.d * cfg.elem_bytes
    moved = 2 * 2 * n * block_bytes  # K and V blocks, each read once and written once
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    sc = None if w.scales is None else w.scales.to(dev)
    pairs = pairs_h.to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scrub = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.fill_(1)
        pkv.copy_blocks(pairs, kc, vc, scales=sc)
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            scrub.amax()  # untimed: write the flush's dirty lines back before the launch
            torch.cuda._sleep(HOST_LEAD_CYCLES)  # untimed: the host queues the launch first
            evs[i][0].record(stream)
            pkv.copy_blocks(pairs, kc, vc, scales=sc)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
    clocks = clk.summary()
    clocks["window"] = "timed region"
    tot_ms = sum(a.elapsed_time(b) for a, b in evs)
    tot_ms = max_over_ranks(tot_ms, ws, dev)
    assert pkv.check_device_status() == 0
    achieved = moved * args.steps / (tot_ms * 1e-3) / 1e9
    # end to end: the pair list comes from pinned host memory every step
    host_pairs = pairs_h.pin_memory()
    dev_pairs = torch.empty_like(pairs)
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ee[i][0].record(stream)
        dev_pairs.copy_(host_pairs, non_blocking=True)
        pkv.copy_blocks(dev_pairs, kc, vc, scales=sc)
        ee[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in ee)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        gbs, dt, reps = oracle_copy_sample(w, pairs_h, min(args.cpu_seconds, 5.0))
        cpu = {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"the same {n} pairs x {reps} passes (memcpy per block, one thread)",
               "seconds": round(dt, 2)}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    line = {
        "metric": "copy-on-write block copy achieved HBM GB/s (bytes read + written)", "value": round(achieved * ws, 2),
        "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8" if cfg.kv_dtype == "e4m3" else "bf16 (bit copy)",
        "data": f"synthetic (seeded pool of {args.config}, {n} disjoint random block pairs)",
        "config": {"workload": f"copy {n} blocks of {block_bytes} B (K and V) in the {args.config} pool "
                               f"({w.num_blocks} blocks)", "pairs": n, "block_bytes": block_bytes,
                   "l2": "flushed between timed launches: 256 MiB write, then a 256 MiB read of another "
                         "buffer (both untimed)", "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "kernel": "copy_blocks_kernel",
                     "peak_source": f"{peak_src} hbm_gbs (copy)"},
        "e2e": {"value": round(moved * ws * args.steps / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(n * 16), "d2h_bytes_per_step": 0},
        "cpu_baseline": cpu,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return  # the oracle runs on rank 0 only
    cfg = W.get(args.config)
    w = W.make_workload(cfg, layout=args.layout)
    thr = host_threads()
    per_step = max(1.0, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step, thr)
    total_b, total_s, desc = 0, 0.0, ""
    for _ in range(args.steps):
        _, dt, desc, nbytes, _ = oracle_sample(w, per_step, thr)
        total_b += nbytes
        total_s += dt
    value = total_b / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic (seeded N(0,1) bf16 q/K/V, {args.layout} 16-token block pool)",
        "config": config_dict(cfg, w, args.layout, args.cascade, ws, args.l2 == "flushed"),
        "timing": "the fp64 oracle on the host cores; each step a bounded sample of (sequence, kv head) groups "
                  "of the workload (its attention is the same for the paged and the cascade call)",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        import __graft_entry__

        __graft_entry__.build()
        if args.op == "copy_blocks":
            run_copy_blocks(args)
        else:
            run_ours(args)


if __name__ == "__main__":
    main()
