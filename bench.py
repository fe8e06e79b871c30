"""Benchmark of the attention hot path on GB300; prints ONE JSON line.

A step is one pass of the whole hot path over one batch of synthetic input:
  * bf16 causal MHA prefill, B=4, H=16, N=4096, D=128 (attn_fwd), then
  * bf16 MLA absorbed decode, batch 64, Hq=128, seq 4096 (mla_decode).
`value` is the prefill's algorithmic TFLOP/s (the first half of the metric),
from the median of the per-step CUDA-event times; the decode's KV-cache GB/s
is reported under `decode`.  Kernel times come from CUDA events on the
launching stream; an L2 flush (a 512 MiB write) separates timed calls.

The default run also reports
  * `sustained`: each leg of the step back to back for two seconds, with the
    SM clock and power sampled inside that window and time x clock;
  * `configs`: every other workload of the target list (the fp32 small causal
    case and the fp32 B4 H8 N8192 D64 case, both masks, on the CUDA cores and
    on the tensor cores; the non-causal bf16 prefill; the paged batch-256
    decode; the decode batch sweep), each with its median time (at least 50
    L2-flushed calls after 10 warm-up calls), throughput,
    fractions of the measured and spec peaks, and its output checked against
    the fp64 oracle (every row, or a seeded sample of rows for the largest);
  * `cpu_baseline`: the oracle's own time on every row of the step's prefill,
    on the host cores, beside its check of the timed GPU output.
`--workload` selects one path alone.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload step|prefill|prefill_noncausal|decode|decode_paged|
                              decode_b16|decode_b128|decode_b256|mla_layer|fp32|fp32_causal|
                              fp32_tc|fp32_tc_causal|fp32_small|fp32_small_tc]
                  [--no-configs] [--no-sustained] [--no-cpu-baseline]

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
    """nvidia-smi clocks, power and throttle reasons sampled every 100 ms, with
    the box's timestamp on every sample, so that each load window (the timed
    steps, each sustained run) gets the samples taken inside it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.rows = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            self.rows = []
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        rows = []
        for line in out.strip().splitlines():
            r = [x.strip() for x in line.split(",")]
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax, pw = float(r[2]), float(r[3]), float(r[4])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.REASONS, r[6:10]) if v.lower() == "active"}
            rows.append((ts, sm, smax, pw, reasons))
        self.rows = rows

    def window(self, windows):
        """Clock statistics of the samples taken inside any of the (t0, t1) windows."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples_under_load": 0}
        inside = [r for r in self.rows if any(t0 <= r[0] <= t1 for t0, t1 in windows)]
        sm = [r[1] for r in inside]
        reasons = sorted(set().union(*[r[4] for r in inside])) if inside else []
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max((r[2] for r in self.rows), default=None),
                "power_w_max": max((r[3] for r in inside), default=None),
                "reasons": reasons, "samples_under_load": len(sm)}


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
        return rows_flops(rows) / dt / 1e12, desc, dt


    def tolerance(self):
        return ({"o": 1e-4, "lse": 1e-4} if self.cfg.dtype == torch.float32
                else {"o": 2e-2, "lse": 1e-3})

    def oracle_check(self, threads: int, max_rows: int):
        """The last call's output against the fp64 oracle on every query row, or
        on a seeded random sample of max_rows rows (plus each head's first and
        last row) when there are more."""
        import numpy as np
        import oracle
        c = self.cfg
        total = c.B * c.H * c.N
        if total <= max_rows:
            rows = np.arange(total)
        else:
            rng = np.random.default_rng(c.seed)
            edge = np.concatenate([np.arange(c.B * c.H) * c.N, np.arange(c.B * c.H) * c.N + c.N - 1])
            rows = np.unique(np.concatenate([rng.choice(total, size=max_rows, replace=False),
                                             edge]))
        t0 = time.perf_counter()
        ro, rl = oracle.mha(self.q, self.k, self.v, c.causal, c.scale,
                            rows=None if len(rows) == total else rows, threads=threads)
        dt = time.perf_counter() - t0
        go = self.o.float().cpu().numpy().reshape(-1, c.D)[rows]
        gl = self.lse.cpu().numpy().reshape(-1)[rows]
        i = rows % c.N
        keys = (i + 1) if c.causal else np.full_like(i, c.N)
        flops = float((4.0 * c.D * keys).sum())
        return {"o": float(np.abs(go - ro.reshape(go.shape)).max()),
                "lse": float(np.abs(gl - rl.reshape(gl.shape)).max()),
                "rows": int(len(rows)), "of_rows": int(total), "tolerance": self.tolerance(),
                "oracle_s": dt, "oracle_tflops": flops / dt / 1e12}


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
        return sample_bytes / dt / 1e9, desc, dt


    def tolerance(self):
        return {"o": 2e-2, "lse": 1e-3}

    def oracle_check(self, threads: int, max_rows: int):
        """The last call's output against the fp64 oracle on every (sequence,
        head) row, or on a seeded random sample of max_rows rows (plus the
        first and last rows) when there are more."""
        import numpy as np
        import oracle
        c = self.cfg
        total = c.batch * c.Hq
        if total <= max_rows:
            rows = np.arange(total)
        else:
            rng = np.random.default_rng(c.seed)
            rows = np.unique(np.concatenate([rng.choice(total, size=max_rows, replace=False),
                                             [0, c.Hq - 1, total - 1]]))
        t0 = time.perf_counter()
        ro, rl = oracle.mla(self.q, self.kv, self.table, self.sl, c.scale,
                            rows=None if len(rows) == total else rows, threads=threads)
        dt = time.perf_counter() - t0
        ro = ro.reshape(len(rows), 512)
        rl = rl.reshape(len(rows))
        go = self.o.float().cpu().numpy().reshape(-1, 512)[rows]
        gl = self.lse.cpu().numpy().reshape(-1)[rows]
        fin = np.isfinite(rl)
        lens = self.sl.numpy()[rows // c.Hq].astype(np.float64)
        return {"o": float(np.abs(go - ro).max()),
                "lse": float(np.abs(gl[fin] - rl[fin]).max()) if fin.any() else 0.0,
                "lse_inf_match": bool(np.array_equal(np.isneginf(gl), np.isneginf(rl))),
                "rows": int(len(rows)), "of_rows": int(total), "tolerance": self.tolerance(),
                "oracle_s": dt,
                "oracle_gbs": float((lens * 1152.0).sum()) / dt / 1e9}


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

    def tolerance(self):
        # the layer's bounds: the absorbed query is itself rounded to bf16
        # before the decode reads it, and the value projection rescales O
        return {"o_rel_to_max_ref": 2e-2, "lse": 5e-3}

    def oracle_check(self, threads: int, max_rows: int):
        """The layer's output against attention over explicitly decompressed
        keys and values (the definition before any absorption), on the first
        two sequences, all heads: the fp64 oracle takes seconds per sequence."""
        import numpy as np
        import oracle
        c = self.cfg
        n = 2
        t0 = time.perf_counter()
        ref, rl = oracle.mla_decompressed(self.qn[:n], self.qr[:n], self.wk, self.wv, self.kv,
                                          self.table[:n], self.sl[:n], c.scale)
        dt = time.perf_counter() - t0
        got = self.out[:n].float().cpu().numpy()
        gl = self.lse[:n].cpu().numpy()
        rel = float(np.abs(got - ref).max() / np.abs(ref).max())
        return {"o": rel, "lse": float(np.abs(gl - rl).max()), "rows": n * c.Hq,
                "of_rows": c.batch * c.Hq, "tolerance": {"o": 2e-2, "lse": 5e-3},
                "o_is_relative_to_max_ref": True, "oracle_s": dt,
                "oracle_gbs": self.bytes * (n / c.batch) / dt / 1e9}

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


WORKLOADS = ["prefill", "prefill_noncausal", "decode", "decode_paged", "decode_b16",
             "decode_b128", "decode_b256", "mla_layer", "fp32", "fp32_causal", "fp32_tc",
             "fp32_tc_causal", "fp32_small", "fp32_small_tc"]


def make_leg(name, dev):
    if name == "fp32_small":
        return PrefillLeg(I.FP32_SMALL_CAUSAL, dev)
    if name == "fp32_small_tc":
        return Tf32x3Leg(I.FP32_SMALL_CAUSAL, dev)
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
    mha = {"prefill": I.BF16_PREFILL, "prefill_noncausal": I.BF16_PREFILL_NONCAUSAL,
           "fp32": I.FP32_PAGE2, "fp32_causal": I.FP32_PAGE2_CAUSAL,
           "fp32_tc": I.FP32_PAGE2, "fp32_tc_causal": I.FP32_PAGE2_CAUSAL,
           "fp32_small": I.FP32_SMALL_CAUSAL, "fp32_small_tc": I.FP32_SMALL_CAUSAL}
    if name in mha:
        return _P(mha[name])
    mla = {"decode": I.MLA_B64, "decode_paged": I.MLA_B256_PAGED, "decode_b16": I.MLA_B16,
           "decode_b128": I.MLA_B128, "decode_b256": I.MLA_B256, "mla_layer": I.MLA_B64}
    return _D(mla[name])


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


# Every workload of the target list, measured and checked in the default
# run: (leg name, rows the oracle checks at most: all rows when there are
# fewer).  The two legs of the step itself are taken from the step's timing.
CONFIG_LEGS = [
    ("fp32_small", 1 << 30), ("fp32_small_tc", 1 << 30),
    ("fp32", 4096), ("fp32_causal", 4096), ("fp32_tc", 4096), ("fp32_tc_causal", 4096),
    ("prefill", 1 << 30), ("prefill_noncausal", 32768),
    ("decode", 1 << 30), ("decode_paged", 1 << 30),
    ("decode_b16", 1 << 30), ("decode_b128", 4096), ("decode_b256", 4096),
]
SUSTAINED_S = 2.0
TABLE_WARMUP = 10   # per-workload table: warm-up calls, then the median of
TABLE_REPS = 50     # at least this many L2-flushed calls


def time_calls(leg, reps, flush, stream):
    """CUDA-event time (ms) of each of `reps` calls, L2 flushed before each."""
    evs = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        leg.run()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def peak_of(leg, peaks, props, smax_mhz):
    """(measured peak, spec peak, unit) of the roofline that bounds the leg."""
    bf16_spec = props.multi_processor_count * 8192 * smax_mhz * 1e6 / 1e12
    ffma = props.multi_processor_count * 128 * 2 * smax_mhz * 1e6 / 1e12
    if leg.bound == "tensor":
        return peaks.get("bf16_tflops"), bf16_spec, "TFLOP/s"
    if leg.bound == "tensor_tf32":
        # tf32 dense peak: the measured bf16 peak x the nominal tf32 / bf16
        # ratio (1.1 / 2.25 PFLOP/s); three MMAs per product cap frac at 1/3
        return peaks.get("bf16_tflops") * (1.1 / 2.25), bf16_spec / 2, "TFLOP/s"
    if leg.bound == "hbm":
        return peaks.get("hbm_gbs"), 8000.0, "GB/s"
    return ffma, ffma, "TFLOP/s"  # fp32 FFMA on the CUDA cores


def achieved_of(leg, ms):
    if leg.bound == "hbm":
        return leg.bytes / (ms * 1e-3) / 1e9
    return leg.flops / (ms * 1e-3) / 1e12


def config_entry(leg, times, peaks, props, smax_mhz, check):
    ms = statistics.median(times)
    v, unit = leg.value(ms * 1e-3)
    peak, spec, _ = peak_of(leg, peaks, props, smax_mhz)
    ach = achieved_of(leg, ms)
    e = {"workload": leg.workload_name(), "kernel": leg.kernel, "ms": ms,
         "ms_mean": statistics.fmean(times), "reps": len(times), "value": v, "unit": unit,
         "frac": ach / peak if peak else None, "frac_spec": ach / spec if spec else None,
         "bound": leg.bound,
         "traffic": committed_traffic(leg.kernel, leg.workload_name(), source_sha(*leg.src))}
    if leg.bound == "tensor_tf32":
        e["ffma_peak_tflops"] = props.multi_processor_count * 128 * 2 * smax_mhz * 1e6 / 1e12
    if isinstance(leg, PrefillLeg) and leg.cfg.name in PAGE_TFLOPS:
        e["page_tflops_rtx5080"] = PAGE_TFLOPS[leg.cfg.name]
    if check is not None:
        e["max_abs_err"] = check
        tol = check["tolerance"]
        e["parity_ok"] = bool(check["o"] <= tol["o"] and check["lse"] <= tol["lse"]
                              and check.get("lse_inf_match", True))
    return e


def sustained_run(leg, seconds, flush, stream):
    """The same call back to back (L2 flushed between calls) for >= `seconds`;
    returns (per-call ms list, (t0, t1) wall window)."""
    times = []
    t0 = time.time()
    while time.time() - t0 < seconds:
        times += time_calls(leg, 25, flush, stream)
    return times, (t0, time.time())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="step", choices=["step"] + WORKLOADS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table (the default step measures every one)")
    ap.add_argument("--no-sustained", action="store_true")
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
    props = torch.cuda.get_device_properties(dev)

    names = ["prefill", "decode"] if args.workload == "step" else [args.workload]
    legs = []
    for n in names:
        try:
            legs.append(make_leg(n, dev))
        except pkg.AttnError as e:
            print(f"# leg {n} unavailable: {e}", file=sys.stderr)
    legs = [lg for lg in legs if _leg_works(lg, pkg)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3)

    # warm-up
    for _ in range(args.warmup):
        for lg in legs:
            flush.zero_()
            lg.run()
    pkg.attn_device_status()

    # ---- the timed steps: K steps, each leg bracketed by CUDA events
    ev = {id(lg): [] for lg in legs}
    barrier(world)
    torch.cuda.synchronize()
    t_main0 = time.time()
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
    t_main1 = time.time()
    barrier(world)
    status = pkg.attn_device_status(raise_on_error=False)
    if status != 0:
        raise SystemExit(f"device error during timing: {pkg.attn_last_error()}")
    times = {id(lg): [a.elapsed_time(b) for a, b in ev[id(lg)]] for lg in legs}
    leg_ms = {k: statistics.median(v) for k, v in times.items()}
    step_ms = sum(leg_ms.values())
    step_ms_max = allreduce_max(step_ms, world, dev)
    wall_max = allreduce_max(wall, world, dev)

    # ---- sustained: each leg back to back for a few seconds, its own clocks
    sus = {}
    if not args.no_sustained:
        for lg in legs:
            sus[id(lg)] = sustained_run(lg, SUSTAINED_S, flush, stream)
        if pkg.attn_device_status(raise_on_error=False) != 0:
            raise SystemExit(f"device error in the sustained runs: {pkg.attn_last_error()}")

    # ---- the per-workload table wants the median of at least TABLE_REPS calls
    # after TABLE_WARMUP; the step's legs get extra reps when K is smaller
    table_times = {}
    if args.workload == "step" and not args.no_configs:
        for lg in legs:
            tt = times[id(lg)]
            if len(tt) < TABLE_REPS:
                tt = time_calls(lg, TABLE_REPS, flush, stream)
            table_times[id(lg)] = tt
        if pkg.attn_device_status(raise_on_error=False) != 0:
            raise SystemExit(f"device error in the table reps: {pkg.attn_last_error()}")

    # ---- end to end through the public API with pinned host buffers: each leg in
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
    import oracle
    threads = oracle.num_threads(0)
    peaks, peak_src = load_peaks()
    # the timed GPU outputs of the step's legs against the oracle (before the
    # per-workload table reuses the device)
    checks = {}
    if not args.no_cpu_baseline:
        for lg in legs:
            checks[id(lg)] = lg.oracle_check(threads, 1 << 30)

    # ---- every other workload of the target list: median of max(K, TABLE_REPS) calls, the
    # roofline fractions, and the output against the oracle
    configs = {}
    if args.workload == "step" and not args.no_configs:
        main_names = {n: lg for n, lg in zip(names, legs)}
        for name, max_rows in CONFIG_LEGS:
            if name in main_names:
                continue
            try:
                lg = make_leg(name, dev)
            except pkg.AttnError as e:
                configs[name] = {"unavailable": str(e)}
                continue
            if not _leg_works(lg, pkg):
                configs[name] = {"unavailable": pkg.attn_last_error()}
                continue
            for _ in range(max(args.warmup, TABLE_WARMUP)):
                flush.zero_()
                lg.run()
            tt = time_calls(lg, max(args.steps, TABLE_REPS), flush, stream)
            if pkg.attn_device_status(raise_on_error=False) != 0:
                raise SystemExit(f"device error in {name}: {pkg.attn_last_error()}")
            chk = None if args.no_cpu_baseline else lg.oracle_check(threads, max_rows)
            configs[name] = (lg, tt, chk)
            del lg
            torch.cuda.empty_cache()
    if sampler:
        sampler.stop()
    windows = [(t_main0, t_main1)] + [w for _, w in sus.values()]
    clocks = sampler.window(windows) if sampler else None
    smax_mhz = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)

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
        "timing": "median of the per-step CUDA-event times",
        "median_ms": main_ms,
        "mean_ms": statistics.fmean(times[id(main_leg)]),
        "wall_ms_per_step": wall_max / args.steps * 1e3,
    }
    # roofline of the dominant kernel
    peak, spec, runit = peak_of(main_leg, peaks, props, smax_mhz)
    achieved = achieved_of(main_leg, main_ms)
    roof = {"bound": "tensor" if main_leg.bound.startswith("tensor") else main_leg.bound,
            "achieved": achieved, "peak": peak, "unit": runit,
            "frac": achieved / peak if peak else None, "peak_source": peak_src,
            "peak_spec": spec, "frac_spec": achieved / spec if spec else None}
    if main_leg.bound == "tensor_tf32":
        roof.update(peak_dtype="tf32 (measured bf16 x 1.1/2.25)", mma_per_product=3)
    if main_leg.bound == "alu":
        roof["bound"] = "alu"
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
        pk, sp, _ = peak_of(lg, peaks, props, smax_mhz)
        line["decode"] = {"value": v * world, "unit": u, "ms": ms, "workload": lg.workload_name(),
                          "frac_of_hbm": v / pk, "frac_of_spec_hbm": v / sp,
                          "traffic": committed_traffic(lg.kernel, lg.workload_name(),
                                                       source_sha(*lg.src)),
                          "e2e": {"value": ev_ * world, "unit": eu_,
                                  "h2d_bytes_per_step": lg.h2d, "d2h_bytes_per_step": lg.d2h,
                                  "ms_per_step": e2e_s[id(lg)] * 1e3}}

    # sustained figures with the clocks seen under that load
    if sus:
        line["sustained"] = {}
        for lg in legs:
            tt, w = sus[id(lg)]
            ck = sampler.window([w]) if sampler else None
            ms = statistics.median(tt)
            v, u = lg.value(ms * 1e-3)
            pk, sp, _ = peak_of(lg, peaks, props, smax_mhz)
            ach = achieved_of(lg, ms)
            entry = {"workload": lg.workload_name(), "seconds": w[1] - w[0], "calls": len(tt),
                     "median_ms": ms, "value": v, "unit": u, "frac": ach / pk if pk else None,
                     "frac_spec": ach / sp if sp else None, "clocks": ck}
            if ck and ck.get("sm_mhz"):
                # time x clock: millions of SM cycles per call, which stays put
                # when only the clock moves
                entry["mcycles_per_call"] = ms * ck["sm_mhz"] / 1e3
            line["sustained"]["prefill" if isinstance(lg, PrefillLeg) else "decode"] = entry

    line["gpu_launches"] = args.steps * sum(_launches(lg, pkg) for lg in legs)
    line["clocks"] = clocks

    # per-workload table: the step's own legs from the timed steps (or their
    # extra reps), the rest measured above
    if configs or (args.workload == "step" and not args.no_configs):
        table = {}
        for name, max_rows in CONFIG_LEGS:
            if name in names:
                lg = legs[names.index(name)]
                table[name] = config_entry(lg, table_times.get(id(lg), times[id(lg)]),
                                           peaks, props, smax_mhz,
                                           checks.get(id(lg)))
            elif name in configs:
                c = configs[name]
                table[name] = c if isinstance(c, dict) else config_entry(
                    c[0], c[1], peaks, props, smax_mhz, c[2])
        line["configs"] = table

    if checks:
        chk = checks[id(main_leg)]
        rate = (chk["oracle_tflops"] if "oracle_tflops" in chk else chk["oracle_gbs"])
        line["cpu_baseline"] = {
            "value": rate, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"all {chk['rows']} query rows of {main_leg.workload_name()}"
            if chk["rows"] == chk["of_rows"] else
            f"{chk['rows']} of {chk['of_rows']} rows of {main_leg.workload_name()}",
            "seconds": chk["oracle_s"],
            "max_abs_err": {k: chk[k] for k in ("o", "lse", "rows", "tolerance")}}
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
