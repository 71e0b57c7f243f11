"""Benchmark: paged decode over a paged KV cache on GB300.

One step = one pass of the whole hot path over one batch:
  llama8b_layer (default): the append of each sequence's newest token and
      the decode of 64 sequences x 32 query heads at context 4096, in one
      append_and_decode call
      (8 KV heads, head_dim 128, block 16, bf16) -- 1 GiB of KV read;
  long_b4_32k / long_b1_128k: paged_decode, 64 q / 8 KV heads, block 32;
  mixed_prefix: 256 sequences, log-uniform lengths, shared prefix blocks;
  fp8_shared: four layer calls that read one E4M3 cache (shared-with pointer);
  int8_shared: the same with an INT8 cache, per-page (scale, zero) pairs;
  spec_verify_tN (N = 4 .. 128): the Llama-8B layer scoring N draft tokens
      per sequence (append N tokens, then one multi-token decode, causal
      among them); spec_verify_t32_fp8 / _int8: the same with an E4M3 or an
      asymmetric INT8 cache;
  prefill_t256 / prefill_t512: chunked prefill, windows of 256 / 512 new
      tokens per sequence over the same layer.

Metric: KV bytes read per step / step time (GB/s, 1e9), with % of the
measured HBM peak and decode steps/s beside it.  Inputs (>= 512 MiB of KV)
are larger than L2, so L2 is not flushed between steps.

Each step is issued through prepared library calls (the step's arguments
checked and marshalled once, every kernel launched anew each step);
`--eager-calls` uses the plain calls, `--graph` replays a captured step.
The e2e leg adds the pinned-host uploads of each step's inputs and the
download of its output, pipelined on two copy streams.

`--impl reference` times the CPU float64 oracle on a bounded sample of the
same workload instead (the only place besides the cpu_baseline leg where
this script runs the oracle).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s and % of GB300 HBM peak; decode steps/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
WORKLOADS = ("llama8b_layer", "long_b4_32k", "long_b1_128k", "mixed_prefix", "fp8_shared",
             "int8_shared", "spec_verify_t4", "spec_verify_t8", "spec_verify_t16", "spec_verify_t32",
             "spec_verify_t64", "spec_verify_t128", "prefill_t256", "prefill_t512",
             "spec_verify_t32_fp8", "spec_verify_t32_int8", "tiny", "copy_blocks")


def query_tokens_of(name):
    """Query tokens per sequence of a workload (1: single-token decode)."""
    for prefix in ("spec_verify_t", "prefill_t"):
        if name.startswith(prefix):
            return int(name[len(prefix):].split("_")[0])
    return 1


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="llama8b_layer")
    ap.add_argument("--math", choices=("auto", "mma", "ffma", "tc"), default="auto")
    ap.add_argument("--partition-blocks", type=int, default=0)
    ap.add_argument("--warps", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one step captured in a CUDA graph (launch-bound small steps)")
    ap.add_argument("--eager-calls", action="store_true",
                    help="issue each step through the plain calls (argument checks and marshalling every "
                         "step) instead of prepared calls")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# environment: ranks, peaks, clocks, profile summaries
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_device():
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def max_over_ranks(x, world):
    """Largest value over ranks (a step time: the slowest replica sets it)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    """Sum over ranks (bytes every replica processed)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_gbs(bytes_per_rank, ms_per_rank, world):
    """Weak-scaling throughput: all ranks' bytes over the slowest rank's time."""
    total = sum_over_ranks(float(bytes_per_rank), world)
    ms = max_over_ranks(float(ms_per_rank), world)
    return total / (ms * 1e-3) / 1e9, ms, total


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 (= f16) tensor-core TFLOP/s: the burst figure, for a kernel
    timed on its own."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def attention_flops_of(c, T):
    """Algorithmic FLOPs of one call: 2 D for q.k and 2 D for p.v per
    (query row, attended key); query token t of a sequence with context
    length L attends to its first L - T + 1 + t keys."""
    ctx = np.asarray(c.context_lens, dtype=np.int64)
    keys = int((T * ctx - T * (T - 1) // 2).sum())
    return 4 * c.D * c.Hq * keys


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for r in csv.reader(io.StringIO(getattr(self, "text", "") or "")):
            if len(r) < 9:
                continue
            try:
                rows.append([x.strip() for x in r])
            except Exception:
                pass
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def profile_traffic(workload, math="mma"):
    """Per-launch DRAM bytes of the workload's kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    name = "copy_blocks_llama8b_pool" if workload == "copy_blocks" else f"paged_decode_{workload}"
    if math in ("ffma", "tc"):
        name += "_" + math
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    from paged_kv_cache_274_gb300 import _build
    if h.group(1) != _build.kernel_digest():
        return None
    return int(m.group(1))


# ---------------------------------------------------------------------------
# workloads (inputs resident in HBM before timing starts)
# ---------------------------------------------------------------------------
def structure(name):
    """Block tables, lengths, queries, append slots (no cache contents)."""
    from workloads import gen
    if name == "llama8b_layer" or query_tokens_of(name) > 1:
        c = gen.llama8b_layer_case(fill=False)
        if name.endswith("_fp8"):      # the same layer with an E4M3 cache
            c.kv_dtype = "fp8"
        elif name.endswith("_int8"):   # ... or an asymmetric INT8 cache
            c.kv_dtype = "int8a"
        return c
    if name.startswith("long_"):
        return gen.long_context_case(name[len("long_"):], fill=False)
    if name == "mixed_prefix":
        return gen.mixed_prefix_case(fill=False)
    if name == "fp8_shared":
        return gen.fp8_shared_case(fill=False)
    if name == "int8_shared":
        return gen.fp8_shared_case(fill=False, kv_dtype="int8a")
    return gen.tiny_case()


def kv_bytes_of(c, seqs=None, layers=None):
    """Algorithmic KV bytes one decode call reads: every real token's K and V
    row of its KV heads (no tail padding), plus per-page E4M3 scales or
    INT8 (scale, zero) pairs."""
    one_byte = c.kv_dtype != "bf16"
    elem = 1 if one_byte else 2
    idx = range(c.B) if seqs is None else seqs
    ctx = np.asarray(c.context_lens, dtype=np.int64)[list(idx)]
    b = int(ctx.sum()) * 2 * c.Hkv * c.D * elem
    if one_byte:
        per_page = 4 if c.kv_dtype == "fp8" else 8
        b += int(((ctx + c.bs - 1) // c.bs).sum()) * 2 * c.Hkv * per_page
    n_layers = len(layers) if layers is not None else c.L
    return b * n_layers


def unique_kv_bytes_of(c, layers=None):
    """KV bytes one decode call must bring from HBM: each (physical block, KV
    head) page once, however many sequences' tables alias it, with the rows
    up to the most that any sequence reads from it (plus its page
    parameters for one-byte caches).  Equal to kv_bytes_of when no block is
    shared; smaller for the prefix-sharing batch, whose aliased prefix pages
    are read by many sequences but stored once ("KV Cache Engineering:
    PagedAttention, Continuous Batching, Attention Variants, and the
    Bandwidth Wall", "PagedAttention": block sharing)."""
    one_byte = c.kv_dtype != "bf16"
    elem = 1 if one_byte else 2
    rows = {}
    for b in range(c.B):
        n = int(c.context_lens[b])
        for j in range((n + c.bs - 1) // c.bs):
            blk = int(c.block_tables[b, j])
            rows[blk] = max(rows.get(blk, 0), min(c.bs, n - j * c.bs))
    nbytes = sum(rows.values()) * 2 * c.Hkv * c.D * elem
    if one_byte:
        nbytes += len(rows) * 2 * c.Hkv * (4 if c.kv_dtype == "fp8" else 8)
    n_layers = len(layers) if layers is not None else c.L
    return nbytes * n_layers


def cpu_model():
    """Host CPU model name (lscpu, else /proc/cpuinfo), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


class DeviceWorkload:
    def __init__(self, name, rank, opts_kw):
        import paged_kv_cache_274_gb300 as pkv
        self.pkv = pkv
        self.name = name
        self.c = c = structure(name)
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        shape = (c.S, c.NB, c.Hkv, c.bs, c.D)
        g = torch.Generator(device=dev)
        g.manual_seed(7919 * (rank + 1) + len(name))
        if c.kv_dtype == "fp8":
            self.k = torch.empty(shape, dtype=torch.uint8, device=dev)
            self.v = torch.empty(shape, dtype=torch.uint8, device=dev)
            self.ks = torch.empty(shape[:3], dtype=torch.float32, device=dev)
            self.vs = torch.empty(shape[:3], dtype=torch.float32, device=dev)
            self._fill_fp8(g)
        elif c.kv_dtype.startswith("int8"):
            self.k = torch.empty(shape, dtype=torch.int8, device=dev)
            self.v = torch.empty(shape, dtype=torch.int8, device=dev)
            self.ks = torch.empty(shape[:3] + (2,), dtype=torch.float32, device=dev)
            self.vs = torch.empty(shape[:3] + (2,), dtype=torch.float32, device=dev)
            self._fill_int8(g)
        else:
            self.k = torch.randn(shape, generator=g, device=dev, dtype=torch.bfloat16)
            self.v = torch.randn(shape, generator=g, device=dev, dtype=torch.bfloat16)
            self.ks = self.vs = None
        self.q = torch.from_numpy(c.q).view(torch.bfloat16).to(dev)          # [L][B][Hq][D]
        self.bt = torch.from_numpy(c.block_tables).to(dev)
        self.cl = torch.from_numpy(c.context_lens).to(dev)
        self.out = torch.empty((c.L, c.B, c.Hq, c.D), dtype=torch.bfloat16, device=dev)
        self.append = c.k_new is not None
        if self.append:
            self.k_new = torch.from_numpy(c.k_new).view(torch.bfloat16).to(dev)
            self.v_new = torch.from_numpy(c.v_new).view(torch.bfloat16).to(dev)
            self.slots = torch.from_numpy(c.slot_mapping).to(dev)
        self.append_every_layer = False
        self.opts_kw = opts_kw
        self.opts = pkv.decode_opts(**opts_kw)
        T = query_tokens_of(name)
        self.ws = pkv.new_decode_workspace(self.k, c.B, c.Hq, c.MB, self.opts, T)
        self.plan = pkv.decode_plan(self.k, c.B, c.Hq, c.MB, self.opts, T)
        self.layers = list(range(c.L))
        self.kv_bytes_logical = kv_bytes_of(c)
        self.kv_bytes = unique_kv_bytes_of(c)
        self.launches_per_step = len(self.layers) * self.plan["kernels_per_call"]
        torch.cuda.synchronize()

    def prepare(self, stream=None):
        """The step as prepared library calls (one per layer), bound to the
        tensors the workload holds now (and to `stream`, if given): what a
        serving loop with fixed step buffers calls each step."""
        pkv, c = self.pkv, self.c
        calls = []
        for i, layer in enumerate(self.layers):
            app = self.append and (i == 0 or self.append_every_layer)
            calls.append(pkv.PreparedDecode(
                self.q[layer], self.k, self.v, self.bt, self.cl, c.kv_group_ptr.tolist(), layer, c.scale,
                out=self.out[layer], workspace=self.ws, k_scale=self.ks, v_scale=self.vs, opts=self.opts,
                k_new=self.k_new if app else None, v_new=self.v_new if app else None,
                slot_mapping=self.slots if app else None, stream=stream))
        return calls

    def _fill_fp8(self, g):
        """E4M3 cache from bf16 N(0,1) data through the library's own append,
        with per-(block, KV head) scales amax / 448 chosen by the caller."""
        c, pkv = self.c, self.pkv
        chunk = 2048  # blocks per append call
        for b0 in range(0, c.NB, chunk):
            nb = min(chunk, c.NB - b0)
            toks = []
            for sc in (self.ks, self.vs):
                src = torch.randn((nb, c.Hkv, c.bs, c.D), generator=g, device=self.dev, dtype=torch.bfloat16)
                amax = src.float().abs().amax(dim=(2, 3))
                s = amax / 448.0
                s[amax == 0] = 1.0
                sc[0, b0:b0 + nb] = s
                toks.append(src.permute(0, 2, 1, 3).reshape(nb * c.bs, c.Hkv, c.D).contiguous())
            slots = torch.arange(b0 * c.bs, (b0 + nb) * c.bs, device=self.dev, dtype=torch.int64)
            pkv.kv_append(toks[0], toks[1], slots, self.k, self.v, self.ks, self.vs)
        torch.cuda.synchronize()

    def _fill_int8(self, g):
        """INT8 cache from bf16 N(0,1) data through the library's append, with
        asymmetric per-(block, KV head) parameters: scale (max - min) / 255,
        zero point round(-128 - min / scale)."""
        c, pkv = self.c, self.pkv
        chunk = 2048
        for b0 in range(0, c.NB, chunk):
            nb = min(chunk, c.NB - b0)
            toks = []
            for prm in (self.ks, self.vs):
                src = torch.randn((nb, c.Hkv, c.bs, c.D), generator=g, device=self.dev, dtype=torch.bfloat16)
                lo = src.float().amin(dim=(2, 3))
                hi = src.float().amax(dim=(2, 3))
                s = (hi - lo) / 255.0
                s[s == 0] = 1.0
                prm[0, b0:b0 + nb, :, 0] = s
                prm[0, b0:b0 + nb, :, 1] = torch.round(-128.0 - lo / s).clamp(-128, 127)
                toks.append(src.permute(0, 2, 1, 3).reshape(nb * c.bs, c.Hkv, c.D).contiguous())
            slots = torch.arange(b0 * c.bs, (b0 + nb) * c.bs, device=self.dev, dtype=torch.int64)
            pkv.kv_append(toks[0], toks[1], slots, self.k, self.v, self.ks, self.vs)
        torch.cuda.synchronize()

    def step(self, events=None):
        """One decode step; `events`: optional list of (start, end) per layer
        call.  The step's append rides in the first layer call's planner
        launch (append_and_decode)."""
        pkv, c = self.pkv, self.c
        for i, layer in enumerate(self.layers):
            opts = self.opts
            if events is not None:
                opts = pkv.decode_opts(**self.opts_kw, event_start=events[i][0], event_end=events[i][1])
            args = (self.q[layer], self.k, self.v, self.bt, self.cl, c.kv_group_ptr.tolist(), layer, c.scale)
            kw = dict(out=self.out[layer], workspace=self.ws, k_scale=self.ks, v_scale=self.vs, opts=opts)
            if self.append and i == 0:
                pkv.append_and_decode(self.k_new, self.v_new, self.slots, *args, **kw)
            else:
                pkv.paged_decode(*args, **kw)


class VerifyWorkload(DeviceWorkload):
    """Speculative-decoding verification on the Llama-3.1-8B decode layer:
    each step appends T draft tokens per sequence (positions ctx-T .. ctx-1)
    and scores them with one multi-token decode (64 sequences x T query
    tokens x 32 heads over context 4096; the T x 4 rows of a KV head share
    one read of its pages)."""

    def __init__(self, name, rank, opts_kw):
        super().__init__(name, rank, opts_kw)
        c, pkv, dev = self.c, self.pkv, self.dev
        self.T = T = query_tokens_of(name)
        g = torch.Generator(device=dev)
        g.manual_seed(15485863 * (rank + 1) + T)
        self.q = torch.randn((c.L, c.B, T, c.Hq, c.D), generator=g, device=dev, dtype=torch.bfloat16)
        self.out = torch.empty_like(self.q)
        pos = c.context_lens.astype(np.int64)[:, None] - T + np.arange(T)[None, :]
        blk = c.block_tables[np.arange(c.B)[:, None], pos // c.bs].astype(np.int64)
        self.slots = torch.from_numpy((blk * c.bs + pos % c.bs).reshape(-1)).to(dev)
        self.k_new = torch.randn((c.B * T, c.Hkv, c.D), generator=g, device=dev, dtype=torch.bfloat16)
        self.v_new = torch.randn((c.B * T, c.Hkv, c.D), generator=g, device=dev, dtype=torch.bfloat16)
        self.append = True
        self.append_every_layer = True
        self.launches_per_step = len(self.layers) * self.plan["kernels_per_call"]
        torch.cuda.synchronize()

    def step(self, events=None):
        pkv, c = self.pkv, self.c
        for i, layer in enumerate(self.layers):
            opts = self.opts
            if events is not None:
                opts = pkv.decode_opts(**self.opts_kw, event_start=events[i][0], event_end=events[i][1])
            pkv.append_and_decode(self.k_new, self.v_new, self.slots, self.q[layer], self.k, self.v, self.bt,
                                  self.cl, c.kv_group_ptr.tolist(), layer, c.scale, out=self.out[layer],
                                  workspace=self.ws, k_scale=self.ks, v_scale=self.vs, opts=opts)


class CopyWorkload:
    """Block copy (copy-on-write / swap): 4096 random blocks of the
    Llama-3.1-8B layer pool (8 KV heads x 16 tokens x 128 x bf16, K and V:
    64 KiB a block) to 4096 other blocks of the same pool, HBM to HBM.
    Bytes per step = read + write = 2 x 4096 x 64 KiB."""

    def __init__(self, rank):
        import paged_kv_cache_274_gb300 as pkv
        self.pkv = pkv
        self.c = c = structure("llama8b_layer")
        dev = torch.device("cuda", torch.cuda.current_device())
        g = torch.Generator(device=dev)
        g.manual_seed(104729 * (rank + 1))
        shape = (c.NB, c.Hkv, c.bs, c.D)
        self.k = torch.randn(shape, generator=g, device=dev, dtype=torch.bfloat16)
        self.v = torch.randn(shape, generator=g, device=dev, dtype=torch.bfloat16)
        rng = np.random.Generator(np.random.PCG64(1000 * 6 + 9))
        ids = rng.permutation(c.NB)[:8192]
        self.pairs = torch.from_numpy(np.stack([ids[:4096], ids[4096:]], axis=1).astype(np.int32)).to(dev)
        block = c.Hkv * c.bs * c.D * 2 * 2
        self.kv_bytes = self.kv_bytes_logical = 2 * 4096 * block
        self.layers = [0]
        self.append = False
        self.plan = {"kernels_per_call": 1, "math": 0, "partition_blocks": 0, "max_partitions": 0,
                     "warps_per_cta": 8, "stages": 0}
        self.launches_per_step = 1
        torch.cuda.synchronize()

    def step(self, events=None):
        if events is not None:
            events[0][0].record()
        self.pkv.copy_blocks(self.k, self.v, self.k, self.v, self.pairs)
        if events is not None:
            events[0][1].record()


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------
def step_launch_mode(w, args):
    if args.graph:
        return "graph"
    return "eager" if args.eager_calls or not hasattr(w, "prepare") else "prepared"


STEP_LAUNCH_DESC = {"graph": "CUDA graph replay",
                    "prepared": "prepared library calls (programmatic dependent launch)",
                    "eager": "plain library calls (programmatic dependent launch)"}


def time_device(w, steps, warmup, world, mode="eager"):
    """Device-resident inputs.  Loop 1 times K steps between CUDA events on
    the launching stream (the headline), issued as `mode` says: "eager",
    the plain calls; "prepared", the step's prepared calls (arguments checked
    and marshalled once, the kernels launched anew every step); "graph", one
    step captured in a CUDA graph after the warm-up and replayed.  Loop 2 repeats
    K eager steps with the decode kernel bracketed by events the library
    records around it (the roofline's kernel time; those events keep the
    planner and the decode from overlapping, so loop 2 is not used for the
    step time)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        w.step()
    torch.cuda.synchronize()
    run_step = w.step
    if mode == "prepared":
        calls = w.prepare(stream)

        def run_step():
            for f in calls:
                f()
        run_step()
    if mode == "graph":
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            w.step()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            w.step()
        g.replay()
        torch.cuda.synchronize()
        run_step = g.replay

    def made_event():
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)   # torch creates the CUDA event lazily, on first record
        return ev
    kev = [[(made_event(), made_event()) for _ in w.layers] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        start.record(stream)
        for _ in range(steps):
            run_step()
        end.record(stream)
        torch.cuda.synchronize()
        for i in range(steps):
            w.step(events=kev[i])
        torch.cuda.synchronize()
    barrier(world)
    total_ms = start.elapsed_time(end)
    kernel_ms = [a.elapsed_time(b) for evs in kev for (a, b) in evs]
    return total_ms, kernel_ms, clk.summary()


TC_PAIR_WARPS = 11  # warps of the tile-pair tcgen05 kernel (the plan's warps_per_cta)


def read_probe_gbs(nbytes=1 << 30, iters=10):
    """The read-only HBM rate of this device: the library's read probe
    streaming an `nbytes` buffer (larger than L2) once per launch, timed with
    CUDA events around each launch after three warm-up launches.  Taken at
    the decode's own byte count, it carries the same launch, ramp-up and
    drain as the decode: the rate a one-pass read of that many bytes can
    reach on this device."""
    import paged_kv_cache_274_gb300 as pkv
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(3):
        pkv.read_probe(buf, out)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        pkv.read_probe(buf, out)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    del buf
    return nbytes / (ms * 1e-3) / 1e9, ms


def time_e2e(w, steps, warmup, world, prepared=True):
    """Through the public API from pinned host memory, pipelined as a serving
    loop would be: each step's inputs (queries, new tokens and slots, block
    tables, lengths) go host->device as one packed staging buffer on a copy
    stream while the previous step computes, and each step's output goes
    device->host on a second copy stream while the next step computes (two
    streams, so that no upload queues behind a download).  Staging
    and output buffers are double-buffered; events order every copy against
    the compute that produces or consumes it.  With `prepared`, each buffer
    set's step is prepared once and called every step; otherwise the plain
    calls run with the buffers of the step.  The timed region spans the
    first upload to the last download."""
    names = ["q", "bt", "cl"] + (["k_new", "v_new", "slots"] if w.append else [])
    tensors = [getattr(w, n) for n in names]
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host_blob = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_blobs = [torch.empty(off, dtype=torch.uint8, device=w.dev) for _ in range(2)]
    views = [{}, {}]
    for n, t, o in zip(names, tensors, offs):
        nbytes = t.numel() * t.element_size()
        for k in range(2):
            v = dev_blobs[k][o:o + nbytes].view(t.dtype).view(t.shape)
            v.copy_(t)
            views[k][n] = v
        host_blob[o:o + nbytes].copy_(views[0][n].view(torch.uint8).reshape(-1).cpu())
    outs = [w.out, torch.empty_like(w.out)]
    out_host = torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory()
    h2d = off
    d2h = out_host.numel() * out_host.element_size()
    compute = torch.cuda.current_stream()
    up = torch.cuda.Stream(device=w.dev)     # host -> device (next step's inputs)
    down = torch.cuda.Stream(device=w.dev)   # device -> host (previous step's output)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer k uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]   # step on buffer k done (inputs read, out written)
    ev_out = [torch.cuda.Event() for _ in range(2)]    # out of buffer k downloaded
    for k in range(2):
        for e in (ev_used[k], ev_out[k]):
            e.record(compute)

    def bind(k):
        for n_, v in views[k].items():
            setattr(w, n_, v)
        w.out = outs[k]
    calls = []
    if prepared:
        for k in range(2):
            bind(k)
            calls.append(w.prepare(compute))
    set_stream = torch.cuda.set_stream

    def run(n):
        for i in range(n):
            k = i & 1
            up.wait_event(ev_used[k])                   # buffer k no longer read by step i-2
            set_stream(up)
            dev_blobs[k].copy_(host_blob, non_blocking=True)
            ev_in[k].record(up)
            set_stream(compute)
            compute.wait_event(ev_in[k])
            compute.wait_event(ev_out[k])               # out buffer k downloaded (step i-2)
            if prepared:
                for f in calls[k]:
                    f()
            else:
                bind(k)
                w.step()
            ev_used[k].record(compute)
            down.wait_event(ev_used[k])
            set_stream(down)
            out_host.copy_(outs[k], non_blocking=True)
            ev_out[k].record(down)
            set_stream(compute)

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    start.record(compute)
    up.wait_event(start)
    down.wait_event(start)
    run(steps)
    compute.wait_stream(up)
    compute.wait_stream(down)
    end.record(compute)
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3
    barrier(world)
    return max(start.elapsed_time(end), wall_ms), h2d, d2h


def oracle_sample(name, target_s):
    """Time the CPU oracle (as it stands) on a bounded sample of the workload:
    the first n sequences of one decode call, all query heads, layer 0.
    Returns (GB/s, seconds, threads, description)."""
    import oracle
    from workloads import normal_bf16_bits
    c = structure(name)
    shape = (c.S, c.NB, c.Hkv, c.bs, c.D)
    fp8 = c.kv_dtype == "fp8"
    int8 = c.kv_dtype.startswith("int8")
    dt = np.uint8 if fp8 else np.int8 if int8 else np.uint16
    k = np.zeros(shape, dtype=dt)
    v = np.zeros(shape, dtype=dt)
    ks = vs = None
    if fp8:
        ks = np.ones(shape[:3], np.float32)
        vs = np.ones(shape[:3], np.float32)
    if int8:
        ks = np.zeros(shape[:3] + (2,), np.float32)
        ks[..., 0] = 0.02
        ks[..., 1] = 3.0
        vs = ks.copy()
    rng = np.random.Generator(np.random.PCG64(11))
    order = list(range(c.B))
    filled = set()

    def fill(upto):
        for b in order[:upto]:
            if b in filled:
                continue
            n = (int(c.context_lens[b]) + c.bs - 1) // c.bs
            blks = c.block_tables[b, :n]
            for arr, seed in ((k, 2), (v, 3)):
                if fp8:
                    arr[0, blks] = rng.integers(0, 0x7E, size=(n,) + shape[2:], dtype=np.uint8)
                elif int8:
                    arr[0, blks] = rng.integers(-128, 128, size=(n,) + shape[2:], dtype=np.int8)
                else:
                    arr[0, blks] = normal_bf16_bits(1000 * seed + b, (n,) + shape[2:])
            filled.add(b)

    T = query_tokens_of(name)
    qm = normal_bf16_bits(17, (c.B, T, c.Hq, c.D)) if T > 1 else None

    def run(nseq):
        fill(nseq)
        t0 = time.perf_counter()
        if T > 1:
            rows = np.array([(b, t, h) for b in order[:nseq] for t in range(T) for h in range(c.Hq)])
            oracle.paged_decode_multi(qm, k, v, c.block_tables, c.context_lens, c.kv_group_ptr, 0,
                                      c.scale, k_scale=ks, v_scale=vs, rows=rows)
        else:
            pairs = np.array([(b, h) for b in order[:nseq] for h in range(c.Hq)], np.int32)
            oracle.paged_decode(c.q[0], k, v, c.block_tables, c.context_lens, c.kv_group_ptr, 0,
                                c.scale, k_scale=ks, v_scale=vs, pairs=pairs)
        return time.perf_counter() - t0

    t1 = run(1)
    nseq = int(min(c.B, max(1, math.floor(target_s / max(t1, 1e-6)))))
    secs = run(nseq) if nseq > 1 else t1
    reps = 1
    while secs * (reps + 1) / reps < target_s and secs / reps < target_s / 2 and reps < 64:
        secs += run(nseq)
        reps += 1
    nbytes = kv_bytes_of(c, seqs=order[:nseq], layers=[0]) * reps
    desc = (f"{name}: sequences 0..{nseq - 1} of {c.B} (all {c.Hq} query heads"
            f"{f' x {T} query tokens' if T > 1 else ''}, one layer call), "
            f"{reps} repetition(s), {nbytes / 1e9:.3f} GB of KV")
    return nbytes / secs / 1e9, secs, oracle.num_threads(), desc


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def config_of(name, c, extra=None):
    cfg = {"workload": name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv, "head_dim": c.D,
           "block_size": c.bs, "kv_dtype": c.kv_dtype, "layer_calls_per_step": c.L,
           "context_lens": ("uniform %d" % int(c.context_lens[0]) if len(set(c.context_lens.tolist())) == 1
                            else "mixed %d..%d (mean %.0f)" % (int(c.context_lens.min()),
                                                                int(c.context_lens.max()),
                                                                float(c.context_lens.mean()))),
           "pool_blocks": c.NB, "l2": "inputs larger than L2 (129 MB); no flush between steps"}
    if query_tokens_of(name) > 1:
        cfg["query_tokens_per_seq"] = query_tokens_of(name)
    if extra:
        cfg.update(extra)
    return cfg


def run_reference(args, rank, world):
    if rank != 0:
        return
    c = structure(args.workload)
    per_step_s = min(2.0, max(0.2, 150.0 / max(1, args.steps + args.warmup)))
    samples = []
    for i in range(args.warmup + args.steps):
        gbs, secs, threads, desc = oracle_sample(args.workload, per_step_s)
        if i >= args.warmup:
            samples.append((gbs, secs))
    value = statistics.median(g for g, _ in samples)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(s for _, s in samples),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(args.workload, c),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc, "cpu_model": cpu_model(), "nproc": os.cpu_count()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world):
    import paged_kv_cache_274_gb300 as pkv
    pkv.load()   # fails loudly if the CUDA library is missing
    opts_kw = dict(partition_blocks=args.partition_blocks,
                   math={"auto": pkv.MATH_AUTO, "mma": pkv.MATH_MMA, "ffma": pkv.MATH_FFMA, "tc": pkv.MATH_TC}[args.math],
                   warps=args.warps, stages=args.stages)
    copy = args.workload == "copy_blocks"
    if copy:
        w = CopyWorkload(rank)
    elif query_tokens_of(args.workload) > 1:
        w = VerifyWorkload(args.workload, rank, opts_kw)
    else:
        w = DeviceWorkload(args.workload, rank, opts_kw)
    c = w.c
    mode = step_launch_mode(w, args)
    total_ms, kernel_ms, clocks = time_device(w, args.steps, args.warmup, world, mode=mode)
    assert pkv.read_device_error() == 0, "device error word set during the benchmark"
    value, ms, kv_total = whole_job_gbs(w.kv_bytes, total_ms / args.steps, world)
    logical_total = sum_over_ranks(float(w.kv_bytes_logical), world)
    peak, peak_kind = hbm_peak()
    per_call_bytes = w.kv_bytes if copy else unique_kv_bytes_of(c, layers=[0])
    per_call_logical = w.kv_bytes_logical if copy else kv_bytes_of(c, layers=[0])
    k_ms = statistics.mean(kernel_ms)
    achieved = per_call_bytes / (k_ms * 1e-3) / 1e9
    probe_bytes = (per_call_bytes // 4096) * 4096 if per_call_bytes >= (256 << 20) else (1 << 30)
    probe_gbs, probe_ms = read_probe_gbs(probe_bytes)
    e2e = None
    if not args.no_e2e and not copy:
        # enough steps that the pipeline's fill and drain (one upload, one
        # download) weigh little: at least K, and at least ~50 ms of steps
        e_steps = min(4000, max(args.steps, int(math.ceil(50.0 / (total_ms / args.steps)))))
        e_ms, h2d, d2h = time_e2e(w, e_steps, max(3, args.warmup), world, prepared=mode != "eager")
        e_ms = max_over_ranks(e_ms / e_steps, world)
        e2e = {"value": kv_total / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e_ms, "steps": e_steps,
               "step_launch": STEP_LAUNCH_DESC["eager" if mode == "eager" else "prepared"],
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not copy:
        gbs, secs, threads, desc = oracle_sample(args.workload, args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": secs, "cpu_model": cpu_model(), "nproc": os.cpu_count()}
    # The dominant roof: HBM bytes or tensor-core FLOPs (multi-token calls
    # with many query rows per KV head do ~4 D T G flops per K/V byte pair).
    tpeak, tpeak_kind = tensor_peak()
    flops = 0 if copy else attention_flops_of(c, query_tokens_of(args.workload))
    tflops = flops / (k_ms * 1e-3) / 1e12
    hbm = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
           "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s"}
    tensor = {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
              "peak_kind": f"{tpeak_kind} (MEASURED_PEAKS.json bf16_tflops, burst)" if tpeak_kind == "measured"
              else "fallback 1.9 PFLOP/s bf16"}
    t_hbm = per_call_bytes / (peak * 1e9)
    t_tensor = flops / (tpeak * 1e12)
    bound_fields = dict(tensor if t_tensor > t_hbm else hbm)
    bound_fields.update({"hbm_frac": hbm["frac"], "tensor_frac": tensor["frac"],
                         "algorithmic_flops_per_launch": flops})
    if rank == 0:
        plan = w.plan
        line = {
            "metric": "paged KV block copy GB/s (read + write bytes)" if copy else METRIC,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {"fp8": "fp8-e4m3 kv, f16 mma, fp32 accumulate",
                                           "bf16": "bf16 kv, bf16 mma, fp32 accumulate"}.get(
                c.kv_dtype, "int8 kv (scale, zero per page), f16 mma, fp32 accumulate"),
            "data": "synthetic (seeded N(0,1) K/V/q, seeded block permutations)",
            "config": config_of(args.workload, c, {
                "parallelism": "replicas" if world > 1 else "single GPU",
                "step_launch": STEP_LAUNCH_DESC[mode],
                "math": {0: "-", 1: "ffma", 2: "mma", 3: "tcgen05"}[plan["math"]],
                "partition_blocks": plan["partition_blocks"], "max_partitions": plan["max_partitions"],
                "warps_per_cta": plan["warps_per_cta"], "stages": plan["stages"]}),
            "kv_bytes_per_step": w.kv_bytes,
            "kv_bytes_accounting": "unique physical pages read (aliased prefix pages counted once)",
            "kv_bytes_logical_per_step": w.kv_bytes_logical,
            "logical_gbs": logical_total / (ms * 1e-3) / 1e9,
            "decode_steps_per_s": 1e3 / ms,
            "pct_of_hbm_peak": 100.0 * value / peak,
            "pct_of_nominal_8tbs": 100.0 * value / 8000.0,
            "roofline": {**bound_fields, "kernel": "copy_blocks_kernel" if copy else
                         (("paged_decode_tc2_kernel" if plan["warps_per_cta"] == TC_PAIR_WARPS else "paged_decode_tc_kernel")
                          if plan["math"] == 3 else "paged_decode_kernel"),
                         "traffic": profile_traffic(args.workload, {1: "ffma", 2: "mma", 3: "tc"}.get(plan["math"], "mma")),
                         "algorithmic_bytes_per_launch": per_call_bytes,
                         "logical_bytes_per_launch": per_call_logical,
                         "logical_gbs": per_call_logical / (k_ms * 1e-3) / 1e9,
                         "kernel_ms_mean": k_ms, "kernel_ms_median": statistics.median(kernel_ms)},
            "hbm_read_probe": {"gbs": probe_gbs, "ms": probe_ms, "bytes": probe_bytes, "kernel": "read_probe_kernel",
                               "frac_of_copy_peak": probe_gbs / peak,
                               "kernel_frac_of_read_probe": achieved / probe_gbs,
                               "note": "read-only streaming rate of this device over the decode's own byte count "
                                       "(same launch, ramp-up and drain: the decode's own ceiling); "
                                       "the roofline peak stays the measured copy rate"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": w.launches_per_step * args.steps,
            "gpu_launches_note": "kernels of the headline loop per layer call: planner (with the step's append on extra CTAs), decode, merge when more than 4 partitions",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, _ = dist_setup(args.gpus)
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
