"""Benchmark of the attention hot path on GB300; prints ONE JSON line.

A step is one pass of the whole hot path over one batch of synthetic input:
  * bf16 causal MHA prefill, B=4, H=16, N=4096, D=128 (attn_fwd), then
  * bf16 MLA absorbed decode, batch 64, Hq=128, seq 4096 (mla_decode).
`value` is the prefill's algorithmic TFLOP/s (the first half of the metric);
the decode's KV-cache GB/s is reported under `decode`.  Kernel times come
from CUDA events on the launching stream; an L2 flush (a 512 MiB write)
separates timed steps.  `--workload` selects another single path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload step|prefill|prefill_noncausal|decode|decode_paged|
                              decode_b16|decode_b128|decode_b256|mla_layer|fp32|fp32_causal|
                              fp32_tc|fp32_tc_causal]

Multi-GPU: the path shards into independent problems, and every box here has
one GPU, so N ranks run N independent replicas (weak scaling); value sums
over ranks and the step time is the max over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from online_softmax_attention_attn_gb300 import inputs as I  # noqa: E402
from online_softmax_attention_attn_gb300 import metrics  # noqa: E402

METRIC = "prefill attention TFLOPS (% bf16 peak); MLA decode KV-cache GB/s (% HBM)"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "online_softmax_attention_attn_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str, sha: str):
    """DRAM bytes per launch from a committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("source_sha") == sha:
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t_start = self.t_end = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        # the load lasts most of the sampled window: report the busy half
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- workloads

# The pages' own figure for exactly this metric and workload, where they print
# one: the FA2-v2 blog's section 4.1 table (fp32 v2 kernel, RTX 5080).  Other
# workloads have none, so their vs_baseline stays null.
PAGE_TFLOPS = {I.FP32_PAGE2.name: 14.45, I.FP32_PAGE2_CAUSAL.name: 12.87}


class PrefillLeg:
    kernel = "prefill_bf16_kernel"

    def __init__(self, cfg: I.MHAConfig, dev):
        import online_softmax_attention_attn_gb300 as pkg
        self.pkg, self.cfg, self.dev = pkg, cfg, dev
        self.q, self.k, self.v = I.mha_config_inputs(cfg)
        self.dq, self.dk, self.dv = (t.to(dev) for t in (self.q, self.k, self.v))
        self.o = torch.empty_like(self.dq)
        self.lse = torch.empty(cfg.B, cfg.H, cfg.N, dtype=torch.float32, device=dev)
        self.flops = metrics.mha_flops(cfg.B, cfg.H, cfg.N, cfg.D, cfg.causal)
        eb = 2 if cfg.dtype == torch.bfloat16 else 4
        self.bytes = metrics.mha_bytes(cfg.B, cfg.H, cfg.N, cfg.D, eb)
        self.launches_per_call = 1
        self.host_entry = True  # e2e through attn_fwd_host
        self.bound = "tensor" if cfg.dtype == torch.bfloat16 else "alu"
        self.kernel = "prefill_bf16_kernel" if cfg.dtype == torch.bfloat16 else "prefill_f32_kernel"
        self.src = ("prefill_bf16.cu",) if cfg.dtype == torch.bfloat16 else ("prefill_f32.cu",)

    def run(self):
        self.pkg.attn_fwd(self.dq, self.dk, self.dv, self.o, self.lse, causal=self.cfg.causal,
                          scale=self.cfg.scale)

    # host buffers for the end-to-end number
    def e2e_setup(self):
        self.hq, self.hk, self.hv = (t.pin_memory() for t in (self.q, self.k, self.v))
        self.ho = torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory()
        self.hl = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        self.hws = None
        if self.host_entry:
            c = self.cfg
            code = (self.pkg.ATTN_DTYPE_F32 if c.dtype == torch.float32
                    else self.pkg.ATTN_DTYPE_BF16)
            need = self.pkg.attn_fwd_host_workspace_size(c.B, c.H, c.N, c.D, code)
            raw = torch.empty(need + 256, dtype=torch.uint8, device=self.dev)
            off = (-raw.data_ptr()) % 256
            self.hws = raw[off:off + need]
        self.h2d = sum(t.numel() * t.element_size() for t in (self.hq, self.hk, self.hv))
        self.d2h = self.ho.numel() * self.ho.element_size() + self.hl.numel() * 4

    def e2e_run(self):
        # the host-buffer entry point: copies in, attention, copies out, with
        # the copies of one chunk of heads overlapping another's attention
        if self.hws is None:
            self._e2e_run_copies()
            return
        self.pkg.attn_fwd_host(self.hq, self.hk, self.hv, self.ho, self.hl,
                               causal=self.cfg.causal, scale=self.cfg.scale, workspace=self.hws)

    def _e2e_run_copies(self):
        self.dq.copy_(self.hq, non_blocking=True)
        self.dk.copy_(self.hk, non_blocking=True)
        self.dv.copy_(self.hv, non_blocking=True)
        self.run()
        self.ho.copy_(self.o, non_blocking=True)
        self.hl.copy_(self.lse, non_blocking=True)

    def value(self, seconds):
        return self.flops / seconds / 1e12, "TFLOP/s"

    def workload_name(self):
        c = self.cfg
        return c.name

    def oracle_sample(self, budget_s: float, threads: int):
        """Time the oracle on a bounded sample of rows; returns (TFLOP/s, desc, s)."""
        import numpy as np
        import oracle
        c = self.cfg
        rng = np.random.default_rng(0)
        total_rows = c.B * c.H * c.N

        def rows_flops(rows):
            i = rows % c.N
            keys = (i + 1) if c.causal else np.full_like(i, c.N)
            return float((4.0 * c.D * keys).sum())

        n = 64
        while True:
            rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False))
            t0 = time.perf_counter()
            ro, rl = oracle.mha(self.q, self.k, self.v, c.causal, c.scale, rows=rows,
                                threads=threads)
            dt = time.perf_counter() - t0
            if dt >= budget_s or n >= total_rows:
                break
            n = int(min(total_rows, n * max(2.0, 1.2 * budget_s / max(dt, 1e-3))))
        desc = f"{len(rows)} random query rows of {total_rows} ({c.name})"
        self.sample_err = None
        if getattr(self, "o", None) is not None:
            # the timed runs' output on the same rows, against the oracle
            go = self.o.float().cpu().numpy().reshape(-1, c.D)[rows]
            gl = self.lse.cpu().numpy().reshape(-1)[rows]
            self.sample_err = {"o": float(np.abs(go - ro).max()),
                               "lse": float(np.abs(gl - rl).max()), "rows": int(len(rows))}
        return rows_flops(rows) / dt / 1e12, desc, dt


class Tf32x3Leg(PrefillLeg):
    """fp32 prefill on the tensor cores (three-product TF32 split): the call
    is the split pre-pass plus the attention kernel, both inside the timing."""

    def __init__(self, cfg: I.MHAConfig, dev):
        super().__init__(cfg, dev)
        need = self.pkg.attn_fwd_tf32x3_workspace_size(cfg.B, cfg.H, cfg.N, cfg.D)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.bound = "tensor_tf32"
        self.host_entry = False  # no host-buffer entry: copies around the device call
        self.kernel = "prefill_tf32x3_kernel"
        self.src = ("prefill_tf32x3.cu",)
        self.launches_per_call = 2

    def run(self):
        self.pkg.attn_fwd_tf32x3(self.dq, self.dk, self.dv, self.o, self.lse,
                                 causal=self.cfg.causal, scale=self.cfg.scale, workspace=self.ws)

    def workload_name(self):
        return self.cfg.name + " on tensor cores (3xTF32)"


class DecodeLeg:
    kernel = "mla_decode_kernel"

    def __init__(self, cfg: I.MLAConfig, dev):
        import online_softmax_attention_attn_gb300 as pkg
        self.pkg, self.cfg, self.dev = pkg, cfg, dev
        self.q, self.kv, self.table, self.sl = I.mla_config_inputs(cfg)
        self.dq, self.dkv, self.dtable, self.dsl = (t.to(dev) for t in
                                                    (self.q, self.kv, self.table, self.sl))
        B = cfg.batch
        self.o = torch.empty(B, cfg.Hq, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B, cfg.Hq, dtype=torch.float32, device=dev)
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        ws = pkg.mla_decode_workspace_size(B, cfg.Hq, self.table.shape[1], nsm)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.bytes = metrics.mla_bytes(self.sl.tolist(), cfg.Hq, max_blocks=self.table.shape[1])
        self.flops = metrics.mla_flops(self.sl.tolist(), cfg.Hq)
        self.bound = "hbm"
        self.src = ("mla_decode.cu",)
        self.launches_per_call = None  # filled by the library's own count

    def run(self):
        self.pkg.mla_decode(self.dq, self.dkv, self.dtable, self.dsl, self.o, self.lse,
                            scale=self.cfg.scale, workspace=self.ws)

    def e2e_setup(self):
        self.hq, self.hkv, self.htable, self.hsl = (t.pin_memory() for t in
                                                    (self.q, self.kv, self.table, self.sl))
        self.ho = torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory()
        self.hl = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in
                       (self.hq, self.hkv, self.htable, self.hsl))
        self.d2h = self.ho.numel() * 2 + self.hl.numel() * 4
        nsm = torch.cuda.get_device_properties(self.dev).multi_processor_count
        need = self.pkg.mla_decode_host_workspace_size(self.cfg.batch, self.cfg.Hq,
                                                       self.table.shape[1], self.kv.shape[0], nsm)
        raw = torch.empty(need + 256, dtype=torch.uint8, device=self.dev)
        off = (-raw.data_ptr()) % 256
        self.hws = raw[off:off + need]

    def e2e_run(self):
        # the host-buffer entry point: copies in, plan + decode + combine,
        # copies out, in order on the stream
        self.pkg.mla_decode_host(self.hq, self.hkv, self.htable, self.hsl, self.ho, self.hl,
                                 scale=self.cfg.scale, workspace=self.hws)

    def value(self, seconds):
        return self.bytes / seconds / 1e9, "GB/s"

    def workload_name(self):
        return self.cfg.name

    def oracle_sample(self, budget_s: float, threads: int):
        import numpy as np
        import oracle
        c = self.cfg
        total = c.batch * c.Hq
        rng = np.random.default_rng(0)
        n = 16
        while True:
            rows = np.sort(rng.choice(total, size=min(n, total), replace=False))
            t0 = time.perf_counter()
            ro, rl = oracle.mla(self.q, self.kv, self.table, self.sl, c.scale, rows=rows,
                                threads=threads)
            dt = time.perf_counter() - t0
            if dt >= budget_s or n >= total:
                break
            n = int(min(total, n * max(2.0, 1.2 * budget_s / max(dt, 1e-3))))
        sample_bytes = self.bytes * (len(rows) / total)
        desc = f"{len(rows)} of {total} (sequence, head) rows ({c.name})"
        self.sample_err = None
        if getattr(self, "o", None) is not None and not isinstance(self, LayerLeg):
            go = self.o.float().cpu().numpy().reshape(-1, 512)[rows]
            gl = self.lse.cpu().numpy().reshape(-1)[rows]
            self.sample_err = {"o": float(np.abs(go - ro).max()),
                               "lse": float(np.abs(gl - rl).max()), "rows": int(len(rows))}
        return sample_bytes / dt / 1e9, desc, dt


class LayerLeg(DecodeLeg):
    """One MLA attention layer: the absorbed query (q_nope W_UK | q_rope), the
    latent decode, and each head's value projection O_latent W_UV.  Weights
    stay resident; the bytes count the cache, both weight sets and every
    activation read or written once."""

    def __init__(self, cfg: I.MLAConfig, dev):
        super().__init__(cfg, dev)
        B, Hq = cfg.batch, cfg.Hq
        (self.qn, self.qr, self.wk, self.wv, _, _, _) = I.mla_layer_inputs(
            B, Hq, self.sl, seed=cfg.seed)
        self.dqn, self.dqr, self.dwk, self.dwv = (t.to(dev) for t in
                                                  (self.qn, self.qr, self.wk, self.wv))
        self.qa = torch.empty(B, Hq, 576, dtype=torch.bfloat16, device=dev)
        self.out = torch.empty(B, Hq, I.MLA_DVHEAD, dtype=torch.bfloat16, device=dev)
        e = 2
        proj = (self.wk.numel() + self.wv.numel() + self.qn.numel() + self.qr.numel()
                + self.qa.numel() + self.o.numel() + self.out.numel()) * e
        self.bytes = self.bytes + proj
        self.flops = self.flops + 2.0 * B * Hq * (I.MLA_DNOPE * 512 + 512 * I.MLA_DVHEAD)

    def run(self):
        self.pkg.mla_absorb_q(self.dqn, self.dqr, self.dwk, q_out=self.qa)
        self.pkg.mla_decode(self.qa, self.dkv, self.dtable, self.dsl, self.o, self.lse,
                            scale=self.cfg.scale, workspace=self.ws)
        self.pkg.mla_project_out(self.o, self.dwv, out=self.out)

    def e2e_setup(self):
        super().e2e_setup()
        self.hqn, self.hqr = (t.pin_memory() for t in (self.qn, self.qr))
        self.hout = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.h2d = (self.h2d - self.hq.numel() * 2 + self.hqn.numel() * 2 + self.hqr.numel() * 2)
        self.d2h = self.hout.numel() * 2 + self.hl.numel() * 4

    def e2e_run(self):
        self.dqn.copy_(self.hqn, non_blocking=True)
        self.dqr.copy_(self.hqr, non_blocking=True)
        self.dkv.copy_(self.hkv, non_blocking=True)
        self.dtable.copy_(self.htable, non_blocking=True)
        self.dsl.copy_(self.hsl, non_blocking=True)
        self.run()
        self.hout.copy_(self.out, non_blocking=True)
        self.hl.copy_(self.lse, non_blocking=True)

    def workload_name(self):
        return "bf16 MLA layer (absorb + decode + project) batch64 Hq128 seq4096"

    def oracle_sample(self, budget_s: float, threads: int):
        import oracle
        c = self.cfg
        n, t0 = 0, time.perf_counter()
        while True:
            oracle.mla_decompressed(self.qn[n:n + 1], self.qr[n:n + 1], self.wk, self.wv,
                                    self.kv, self.table[n:n + 1], self.sl[n:n + 1], c.scale)
            n += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s or n >= c.batch:
                break
        desc = f"{n} of {c.batch} sequences, all {c.Hq} heads, keys and values decompressed"
        return self.bytes * (n / c.batch) / dt / 1e9, desc, dt


def make_leg(name, dev):
    if name == "prefill":
        return PrefillLeg(I.BF16_PREFILL, dev)
    if name == "prefill_noncausal":
        return PrefillLeg(I.BF16_PREFILL_NONCAUSAL, dev)
    if name == "fp32":
        return PrefillLeg(I.FP32_PAGE2, dev)
    if name == "fp32_causal":
        return PrefillLeg(I.FP32_PAGE2_CAUSAL, dev)
    if name == "fp32_tc":
        return Tf32x3Leg(I.FP32_PAGE2, dev)
    if name == "fp32_tc_causal":
        return Tf32x3Leg(I.FP32_PAGE2_CAUSAL, dev)
    if name == "decode":
        return DecodeLeg(I.MLA_B64, dev)
    if name == "decode_paged":
        return DecodeLeg(I.MLA_B256_PAGED, dev)
    if name == "mla_layer":
        return LayerLeg(I.MLA_B64, dev)
    if name == "decode_b16":
        return DecodeLeg(I.MLA_B16, dev)
    if name == "decode_b128":
        return DecodeLeg(I.MLA_B128, dev)
    if name == "decode_b256":
        return DecodeLeg(I.MLA_B256, dev)
    raise ValueError(name)


# ----------------------------------------------------------------- main

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world, dev):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle
    threads = oracle.num_threads(0)
    legs = ["prefill", "decode"] if args.workload == "step" else [args.workload]
    cpu = torch.device("cpu")
    main = None
    results = {}
    for name in legs:
        leg = make_leg_cpu(name)
        per = max(2.0, 20.0 / max(1, args.steps) / len(legs))
        vals = []
        for _ in range(args.warmup):
            leg.oracle_sample(0.2, threads)
        for _ in range(args.steps):
            v, desc, dt = leg.oracle_sample(per, threads)
            vals.append(v)
        results[name] = (statistics.median(vals), desc, leg)
        if main is None:
            main = name
    v, desc, leg = results[main]
    unit = "TFLOP/s" if isinstance(leg, PrefillLeg) else "GB/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload, leg),
        "cpu_baseline": {"value": v, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if "decode" in results and main != "decode":
        dv, ddesc, _ = results["decode"]
        line["decode"] = {"value": dv, "unit": "GB/s", "sample": ddesc}
    print(json.dumps(line))


def make_leg_cpu(name):
    """Legs for the reference arm: host tensors only, no GPU needed."""
    class _P(PrefillLeg):
        def __init__(self, cfg):
            self.cfg = cfg
            self.q, self.k, self.v = I.mha_config_inputs(cfg)
    class _D(DecodeLeg):
        def __init__(self, cfg):
            self.cfg = cfg
            self.q, self.kv, self.table, self.sl = I.mla_config_inputs(cfg)
            self.bytes = metrics.mla_bytes(self.sl.tolist(), cfg.Hq,
                                           max_blocks=self.table.shape[1])
    if name in ("prefill", "prefill_noncausal", "fp32", "fp32_causal", "fp32_tc",
                "fp32_tc_causal"):
        cfg = {"prefill": I.BF16_PREFILL, "prefill_noncausal": I.BF16_PREFILL_NONCAUSAL,
               "fp32": I.FP32_PAGE2, "fp32_causal": I.FP32_PAGE2_CAUSAL,
               "fp32_tc": I.FP32_PAGE2, "fp32_tc_causal": I.FP32_PAGE2_CAUSAL}[name]
        return _P(cfg)
    return _D(I.MLA_B64 if name == "decode" else I.MLA_B256_PAGED)


def config_of(workload, leg):
    if isinstance(leg, PrefillLeg):
        c = leg.cfg
        cfg = {"workload": c.name, "B": c.B, "H": c.H, "N": c.N, "D": c.D, "causal": c.causal,
               "dtype": "bf16" if c.dtype == torch.bfloat16 else "fp32"}
    else:
        c = leg.cfg
        cfg = {"workload": leg.workload_name(), "batch": c.batch, "Hq": c.Hq, "seq_min": c.seq_min,
               "seq_max": c.seq_max, "page": 64, "paged_random": c.paged_random}
    if workload == "step":
        cfg["workload"] = ("step = " + I.BF16_PREFILL.name + " + " + I.MLA_B64.name)
    cfg["l2"] = "flushed between steps (512 MiB write)"
    cfg["parallelism"] = "replicas"
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="step",
                    choices=["step", "prefill", "prefill_noncausal", "decode", "decode_paged",
                             "decode_b16", "decode_b128", "decode_b256", "mla_layer", "fp32",
                             "fp32_causal", "fp32_tc", "fp32_tc_causal"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import online_softmax_attention_attn_gb300 as pkg
    pkg.lib()  # fail loudly if the CUDA library is missing
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    names = ["prefill", "decode"] if args.workload == "step" else [args.workload]
    legs = []
    for n in names:
        try:
            legs.append(make_leg(n, dev))
        except pkg.AttnError as e:
            print(f"# leg {n} unavailable: {e}", file=sys.stderr)
    legs = [lg for lg in legs if _leg_works(lg, pkg)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # warm-up
    for _ in range(args.warmup):
        for lg in legs:
            flush.zero_()
            lg.run()
    pkg.attn_device_status()

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3)
    ev = {id(lg): [] for lg in legs}
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for lg in legs:
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            lg.run()
            b.record(stream)
            ev[id(lg)].append((a, b))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    if sampler:
        sampler.mark_end()
    status = pkg.attn_device_status(raise_on_error=False)
    if status != 0:
        raise SystemExit(f"device error during timing: {pkg.attn_last_error()}")
    clocks = sampler.stop() if sampler else None

    leg_ms = {id(lg): statistics.fmean(a.elapsed_time(b) for a, b in ev[id(lg)]) for lg in legs}
    step_ms = sum(leg_ms.values())
    step_ms_max = allreduce_max(step_ms, world, dev)
    wall_max = allreduce_max(wall, world, dev)

    # end to end through the public API with pinned host buffers: each leg in
    # its own loop (inputs copied in, the call, outputs read back, a sync)
    e2e_steps = max(3, min(args.steps, 20))
    e2e_s = {}
    for lg in legs:
        lg.e2e_setup()
        for _ in range(3):
            lg.e2e_run()
        torch.cuda.synchronize()
        barrier(world)
        t1 = time.perf_counter()
        for _ in range(e2e_steps):
            lg.e2e_run()
            torch.cuda.synchronize()
        e2e_s[id(lg)] = allreduce_max((time.perf_counter() - t1) / e2e_steps, world, dev)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    main_leg = legs[0]
    main_ms = leg_ms[id(main_leg)]
    v1, unit = main_leg.value(main_ms * 1e-3)
    value = v1 * world
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / PAGE_TFLOPS[main_leg.cfg.name]
                        if isinstance(main_leg, PrefillLeg) and len(legs) == 1
                        and main_leg.cfg.name in PAGE_TFLOPS else None),
        "dtype": "bf16" if main_leg.bound in ("tensor", "hbm") else "f32", "data": "synthetic",
        "config": config_of(args.workload, main_leg),
        "wall_ms_per_step": wall_max / args.steps * 1e3,
    }
    # roofline of the dominant kernel
    if main_leg.bound == "tensor":
        peak = peaks.get("bf16_tflops")
        achieved = main_leg.flops / (main_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    elif main_leg.bound == "tensor_tf32":
        # tf32 dense peak: the measured bf16 peak x the nominal tf32 / bf16
        # ratio (1.1 / 2.25 PFLOP/s); three MMAs per product cap frac at 1/3
        peak = peaks.get("bf16_tflops") * (1.1 / 2.25)
        achieved = main_leg.flops / (main_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "peak_dtype": "tf32 (measured bf16 x 1.1/2.25)", "mma_per_product": 3}
        props = torch.cuda.get_device_properties(dev)
        smax = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
        roof["ffma_peak"] = props.multi_processor_count * 128 * 2 * smax * 1e6 / 1e12
    elif main_leg.bound == "hbm":
        peak = peaks.get("hbm_gbs")
        achieved = main_leg.bytes / (main_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    else:
        # fp32 FFMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock
        props = torch.cuda.get_device_properties(dev)
        smax = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
        peak = props.multi_processor_count * 128 * 2 * smax * 1e6 / 1e12
        achieved = main_leg.flops / (main_ms * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["peak"] else None
    roof["peak_source"] = peak_src
    # the spec denominators beside the measured ones: dense bf16 = SMs x 8192
    # FLOP/clk x max SM clock (tf32 half of it), HBM 8 TB/s
    props = torch.cuda.get_device_properties(dev)
    smax_mhz = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    bf16_spec = props.multi_processor_count * 8192 * smax_mhz * 1e6 / 1e12
    spec = {"tensor": bf16_spec, "tensor_tf32": bf16_spec / 2, "hbm": 8000.0,
            "alu": roof["peak"]}.get(main_leg.bound)
    if spec:
        roof["peak_spec"] = spec
        roof["frac_spec"] = roof["achieved"] / spec
    sha = source_sha(*main_leg.src)
    roof["traffic"] = committed_traffic(main_leg.kernel, main_leg.workload_name(), sha)
    roof["kernel"] = main_leg.kernel
    line["roofline"] = roof

    # end-to-end number of the main leg
    e2e_val, e2e_unit = main_leg.value(e2e_s[id(main_leg)])
    line["e2e"] = {"value": e2e_val * world, "unit": e2e_unit,
                   "h2d_bytes_per_step": main_leg.h2d, "d2h_bytes_per_step": main_leg.d2h,
                   "ms_per_step": e2e_s[id(main_leg)] * 1e3}

    # secondary legs (decode inside a full step)
    for lg in legs[1:]:
        ms = leg_ms[id(lg)]
        v, u = lg.value(ms * 1e-3)
        ev_, eu_ = lg.value(e2e_s[id(lg)])
        line["decode"] = {"value": v * world, "unit": u, "ms": ms, "workload": lg.workload_name(),
                          "frac_of_hbm": v / peaks.get("hbm_gbs"),
                          "e2e": {"value": ev_ * world, "unit": eu_,
                                  "h2d_bytes_per_step": lg.h2d, "d2h_bytes_per_step": lg.d2h,
                                  "ms_per_step": e2e_s[id(lg)] * 1e3}}
    line["gpu_launches"] = args.steps * sum(_launches(lg, pkg) for lg in legs)
    line["clocks"] = clocks

    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.num_threads(0)
        v, desc, dt = main_leg.oracle_sample(12.0, threads)
        line["cpu_baseline"] = {"value": v, "unit": unit, "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": dt}
        err = getattr(main_leg, "sample_err", None)
        if err is not None:
            # the timed GPU output on the sampled rows against the oracle
            tol = ({"o": 1e-4, "lse": 1e-4} if main_leg.bound in ("alu", "tensor_tf32")
                   else {"o": 2e-2, "lse": 1e-3})
            line["cpu_baseline"]["max_abs_err"] = dict(err, tolerance=tol)
    print(json.dumps(line))


def _leg_works(leg, pkg):
    try:
        leg.run()
        torch.cuda.synchronize()
        return True
    except pkg.AttnError as e:
        print(f"# leg {type(leg).__name__} skipped: {e}", file=sys.stderr)
        return False


def _launches(leg, pkg):
    if isinstance(leg, PrefillLeg):
        return getattr(leg, "launches_per_call", 1)
    return 3  # plan, decode, combine


if __name__ == "__main__":
    main()
