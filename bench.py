"""Benchmark: packed-state AdamW on GB300 (one JSON line on rank 0).

Workload (default): the Llama-70B depth slice, 8 decoder layers (h 8,192, 64
heads / 8 key-value heads, SwiGLU FFN 28,672; 855,654,400 parameters each,
6,845,235,200 in all) in the 12 B/param layout (bf16 G | bf16 W | fp32 m |
fp32 v), 82.1 GB of state; AdamW lr 1e-4, betas 0.9/0.999, eps 1e-8, wd 0.01.
Inputs: the seeded synthetic generator (synth), step t starting at 1 with zero
moments; the gradient of step t is drawn with seed + t.

  value     params/s of the device-resident step (lst_adamw_step, one
            multi-block launch per step) with all 82 GB of state resident in
            HBM (larger than the L2, so no flush is needed).
  e2e       params/s of the streamed step (lst_stream_step) over pinned host
            blocks for t = 1..3 from the initial state, a fresh gradient per
            step: every step copies the fields the update reads host ->
            device and the fields it writes device -> host.
  e2e_before_heal  the same call on the pinned blocks as first allocated,
            before the bench replaces slow pinned allocations.
  roofline  the fused update kernel against the measured HBM copy bandwidth.
  stream    pinned host-link bandwidth measured in the same run (H2D, D2H,
            both at once) and the streamed step against it.
  zero_copy the same step with the update kernel reading and writing the
            pinned host blocks directly (lst_zero_copy_step), against the
            same link roofline.
  stream_devgrad  the streamed step with the gradients already on the device
            (lst_stream_step_devgrad): 10 B/param inbound instead of 12.
  configs   the device-resident step (plain, per-block options, SGD form) on
            the other workloads: one TinyLlama-1.1B layer, the full
            TinyLlama-1.1B mixed layout, the TinyLlama LoRA adapters (L2
            flushed) and LLaMA-7B.
  cpu_baseline  the oracle (plain C, all host cores) on a bounded sample.
  parity    one block stepped by the product kernel and by the oracle, and
            sampled elements of the streamed t = 1..3 result followed through
            the three steps by the oracle.

`--impl reference` times the oracle alone on the host, on the same workload.
Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (weak scaling, no collective on the data path); value is the sum over
ranks of parameters updated divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "AdamW params/s/GPU; HBM GB/s % of peak; streamed host-link GB/s % of measured"
WORKLOADS = {
    # name: (shape function name, format, description)
    "tinyllama_full_l16m": ("tinyllama_full", "L16M",
                            "TinyLlama-1.1B full shape, 16 B/param mixed (fp32 master), 24 blocks"),
    "tinyllama_layer_l12": ("tinyllama_layer", "L12", "one TinyLlama-1.1B decoder layer, 12 B/param"),
    "tinyllama_lora_l16f": ("tinyllama_lora", "L16F", "TinyLlama-1.1B LoRA r=8 adapters, fp32, 22 blocks"),
    "llama7b_l12": ("llama7b", "L12", "LLaMA-7B shape, 12 B/param, 34 blocks"),
    "llama70b_slice8_l12": ("llama70b_slice", "L12", "Llama-70B depth slice, 8 decoder layers, 12 B/param"),
}
# Algorithmic bytes per parameter of one device-resident step (reads + writes).
ALG_BYTES = {"L12": 22, "L16M": 28, "L16F": 28}
# ... and of one SGD step (G and W read, W written; the mixed layout reads the
# fp32 master and writes it and the bf16 W; m and v are untouched)
SGD_BYTES = {"L12": 6, "L16M": 12, "L16F": 12}
# algorithmic bytes below which the launch path uses lst_update_small_kernel
# (kSmallLaunchBytes in lst_kernels.cu: about twice the 129 MB L2)
SMALL_LAUNCH_BYTES = 256 << 20
HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
HP_LORA = dict(lr=2e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
# The largest workload that fits one GPU: the Llama-70B depth slice (82.1 GB).
DEFAULT_WORKLOAD = "llama70b_slice8_l12"
# Workloads whose gradient is drawn afresh for every step t (seed + t), and
# the streamed steps t = 1..n they are measured over from the initial state.
FRESH_GRAD_STEPS = {"llama70b_slice8_l12": 3}
# The other workloads, measured device-resident in the same run (configs).
CONFIG_LEGS = ("tinyllama_layer_l12", "tinyllama_full_l16m", "tinyllama_lora_l16f", "llama7b_l12")


# ---------------------------------------------------------------------------
# distributed helpers (host logic; covered by the gloo tests)
# ---------------------------------------------------------------------------
def dist_env():
    """(rank, local_rank, world) from torchrun's environment, (0, 0, 1) otherwise."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def dist_init(backend: str):
    """Joins the process group when launched by torchrun (any world size, so
    the same path runs with one process as with eight)."""
    import torch.distributed as dist
    rank, _, world = dist_env()
    if "RANK" in os.environ and "MASTER_ADDR" in os.environ and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_blocks(block_bytes, world: int):
    """Contiguous block ranges [start, stop) of one model for `world` ranks,
    balanced by bytes: rank r's range ends at the block boundary nearest to
    (r + 1) / world of the model's bytes (every rank gets at least one block
    while there are blocks enough; ranges may be empty when there are fewer
    blocks than ranks). The update needs no exchange between ranks."""
    n = len(block_bytes)
    total = float(sum(block_bytes))
    cum = [0.0]
    for b in block_bytes:
        cum.append(cum[-1] + b)
    cuts = [0]
    for r in range(1, world):
        target = total * r / world
        k = min(range(cuts[-1], n + 1), key=lambda j: (abs(cum[j] - target), j))
        # leave at least one block for each remaining rank when possible
        k = max(k, min(cuts[-1] + 1, n))
        k = min(k, max(n - (world - r), cuts[-1]))
        cuts.append(k)
    cuts.append(n)
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def replica_seed(seed: int, rank: int) -> int:
    """Each rank's replica draws its own state (weak scaling: a disjoint shard
    of an N-times larger job)."""
    return seed + 1_000_003 * rank


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks, utilisation and throttle reasons, sampled every
    200 ms; the SM clock is summarised over the samples taken under load
    (utilisation of at least 50 %, all samples if none is)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def snapshot(self):
        """Summary of the samples so far (the sampler keeps running)."""
        return self.summary(list(self.lines))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        return self.summary(self.lines)

    @staticmethod
    def summary(lines):
        rows, mx = [], None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm = float(p[1])
                mx = float(p[2])
            except ValueError:
                continue
            try:
                util = float(p[9]) if len(p) > 9 else None
            except ValueError:
                util = None
            rows.append((sm, util, {n for n, v in zip(names, p[5:9]) if v.lower() == "active"}))
        loaded = [r for r in rows if r[1] is not None and r[1] >= 50.0] or rows
        reasons = set()
        for r in loaded:
            reasons |= r[2]
        return {"sm_mhz": statistics.median([r[0] for r in loaded]) if loaded else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_sha() -> str:
    """Hash of the device code of the update kernels: lst_device.cuh and the
    part of lst_kernels.cu before its host-side launch section."""
    csrc = os.path.join(ROOT, "optimizer_update_gb300", "csrc")
    h = hashlib.sha256()
    h.update(open(os.path.join(csrc, "lst_device.cuh"), "rb").read())
    k = open(os.path.join(csrc, "lst_kernels.cu"), "rb").read()
    h.update(k.split(b"// ---- launch ----")[0])
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str, fmt: str, params: int):
    """DRAM bytes per launch of `kernel` on format `fmt` from the committed ncu
    summary (bytes per parameter of a captured case), scaled to `params`; None
    if that pair was not captured or the kernels' device code changed since."""
    summ = os.path.join(ROOT, "profiles", "lst_update_kernel_traffic.txt")
    if not os.path.exists(summ):
        return None
    sha, per_param = None, None
    for line in open(summ):
        p = line.split()
        if not p or line.startswith("#"):
            continue
        if p[0] == "kernel_source_sha256_16":
            sha = p[1]
        elif p[0] == "traffic" and p[1] == kernel and p[2] == fmt:
            per_param = float(p[3])
    if sha != kernel_source_sha() or per_param is None:
        return None
    return per_param * params


def workload_specs(workload: str, max_blocks: int = 0):
    """(tensor name, shape, block) of the workload; max_blocks > 0 keeps only
    its first blocks (a smaller case of the same kernel, e.g. for profiling)."""
    from synth import shapes
    fn, _, _ = WORKLOADS[workload]
    specs = getattr(shapes, fn)()
    if max_blocks > 0:
        specs = [s for s in specs if s[2] < max_blocks]
    return specs


def build_layout(workload: str, max_blocks: int = 0):
    from optimizer_update_gb300 import Layout
    return Layout(workload_specs(workload, max_blocks), WORKLOADS[workload][1])


def host_mem_available() -> int:
    """MemAvailable of /proc/meminfo in bytes (0 if it cannot be read)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def replicas_fit(state_bytes: int, local_ranks: int, available: int, heal_extra: int = 40 << 30) -> bool:
    """Whether one pinned copy of the state per rank on this host, plus the
    health check's allowance for replacing slow allocations, fits in 3/4 of
    the host's available memory (unknown availability: assume it does)."""
    if available <= 0:
        return True
    per_rank = state_bytes + min(heal_extra, state_bytes // 2)
    return local_ranks * per_rank <= 0.75 * available


def rank_layout(workload: str, max_blocks: int, shard: bool, rank: int, world: int):
    """The layout this rank updates and the model index of its first block:
    the whole model (a replica), or with `shard` its contiguous range of the
    model's blocks (shard_blocks)."""
    from optimizer_update_gb300 import Layout
    full = build_layout(workload, max_blocks)
    if not shard or world == 1:
        return full, 0
    a, b = shard_blocks([full.block_bytes(i) for i in range(full.n_layers)], world)[rank]
    if a == b:
        raise SystemExit(f"--shard: {full.n_layers} blocks cannot give rank {rank} of {world} a block")
    specs = [(n, sh, blk - a) for (n, sh, blk) in workload_specs(workload, max_blocks) if a <= blk < b]
    return Layout(specs, full.fmt), a


def anon_huge_page_bytes() -> int:
    """Bytes of this process's anonymous memory backed by transparent huge
    pages (Linux /proc/self/smaps_rollup), 0 where unavailable."""
    try:
        for line in open("/proc/self/smaps_rollup"):
            if line.startswith("AnonHugePages:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def grad_seed(workload: str, seed: int, t: int):
    """Seed of step t's gradient: seed + t for the workloads that draw a fresh
    gradient per step, None (the state's own seed) for the others."""
    return seed + t if workload in FRESH_GRAD_STEPS else None


def fill_blocks_parallel(jobs, workers: int = 8):
    """Run fill jobs (callables) on a thread pool: the generator and numpy's
    zero-fill release the GIL, so blocks fill in parallel."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=max(1, min(workers, len(jobs)))) as ex:
        for f in [ex.submit(j) for j in jobs]:
            f.result()


def draw_state(L, arrs, workload: str, seed: int, first_block: int = 0):
    """Every block of the state as at step t = 1 (zero moments), the
    gradient of step 1; block i of L is block first_block + i of the model."""
    import synth
    fill_blocks_parallel([
        (lambda i=i: synth.fill_block(L.numpy_views(i, arrs[i]), L.spans(i), first_block + i, workload, L.fmt,
                                      t=1, seed=seed, g_seed=grad_seed(workload, seed, 1), threads=4))
        for i in range(L.n_layers)])


def redraw_gradients(L, arrs, workload: str, seed: int, t: int, first_block: int = 0):
    """Step t's gradient (seed + t) into every block's G segment."""
    import synth
    gs = grad_seed(workload, seed, t)
    fill_blocks_parallel([
        (lambda i=i: synth.fill_field(L.numpy_views(i, arrs[i])["G"], "G", L.fmt, L.spans(i), first_block + i,
                                      workload, t, gs, threads=4))
        for i in range(L.n_layers)])


def alloc_pinned_state(L, workload: str, seed: int, first_block: int = 0):
    """Pinned host blocks (lst_host_alloc) holding the state at t = 1."""
    import ctypes
    import numpy as np
    from optimizer_update_gb300 import lst
    ptrs, arrs = [], []
    for i in range(L.n_layers):
        n = L.block_bytes(i)
        p = lst.lst_host_alloc(n)
        ptrs.append(p)
        arrs.append(np.ctypeslib.as_array((ctypes.c_uint8 * n).from_address(p)))
    draw_state(L, arrs, workload, seed, first_block)
    return ptrs, arrs


def cpu_oracle_rate(L, arrs, hp_kw, budget_s: float, threads: int):
    """Oracle throughput (params/s) over the state, whole passes until the time
    budget is used (at least one block)."""
    import oracle
    done, t_start, step = 0, time.perf_counter(), 1
    blocks = 0
    while True:
        for i in range(L.n_layers):
            oracle.step(L.fmt, L.numpy_views(i, arrs[i]), oracle.hparams(step=step, **hp_kw), threads=threads)
            done += L.block(i)[1]
            blocks += 1
            if time.perf_counter() - t_start >= budget_s:
                el = time.perf_counter() - t_start
                return done / el, done, el, blocks
        step += 1


def parity_sample(L, arrs, hp_kw, device, threads: int, t: int = 7):
    """One block of the current state stepped once by the product kernel (a
    one-block layout with the block's geometry, lst_adamw_step) and once by
    the oracle on a host copy: the largest fp32 relative error, the largest
    bf16 distance in ulps, and whether every byte matches. Part of the CPU
    baseline leg (the one place the bench may run the oracle besides the
    reference arm)."""
    import numpy as np
    import torch
    import oracle
    from optimizer_update_gb300 import Layout, lst
    i = max(range(L.n_layers), key=lambda k: (L.block(k)[1] if k else -1))  # the largest block but the first
    if L.n_layers == 1:
        i = 0
    Li = Layout([(name, (n,), 0) for (name, _off, n) in L.spans(i)], L.fmt)
    if Li.block_bytes(0) != L.block_bytes(i):
        return None
    host = arrs[i].copy()
    dev = torch.from_numpy(host).to(device)
    lst.lst_adamw_step(Li.handle, [dev.data_ptr()], lst.adamw_hparams(step=t, **hp_kw),
                       torch.cuda.current_stream(device).cuda_stream)
    got = dev.cpu().numpy()
    del dev
    oracle.step(L.fmt, Li.numpy_views(0, host), oracle.hparams(step=t, **hp_kw), threads=threads)
    gv, ev = Li.numpy_views(0, got), Li.numpy_views(0, host)
    out = {"block": i, "elements": int(Li.block(0)[1]), "step": t, "bit_exact": bool(np.array_equal(got, host))}
    out.update(field_errors(L.fmt, gv, ev, Li.fields()))
    return out


def field_errors(fmt, got, exp, fields):
    """Largest fp32 relative error, largest bf16 distance in ulps and the
    number of NaN outputs over the written fields (G excluded)."""
    import numpy as np
    rel, ulp, nans = 0.0, 0, 0

    def order(x):  # bf16 bit patterns in monotone integer order
        x = x.view(np.uint16).astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), x + 0x8000)

    for f, dt in fields.items():
        if f == "G":
            continue
        a, b = got[f], exp[f]
        if dt == "f32":
            an, bn = np.isnan(a), np.isnan(b)
        else:
            an, bn = (a.view(np.uint16) & 0x7FFF) > 0x7F80, (b.view(np.uint16) & 0x7FFF) > 0x7F80
        nans += int(bn.sum())
        if not np.array_equal(an, bn):  # NaN on one side only
            rel, ulp = float("inf"), 1 << 16
            continue
        a, b = a[~an], b[~bn]
        if not a.size:
            continue
        if dt == "f32":
            d = np.abs(a.astype(np.float64) - b.astype(np.float64)) / np.maximum(np.abs(b.astype(np.float64)), 1e-30)
            rel = max(rel, float(np.max(d)))
        else:
            ulp = max(ulp, int(np.max(np.abs(order(a) - order(b)))))
    return {"max_rel_err_fp32": rel, "max_ulp_bf16": ulp, "nan_outputs": nans}


def stream_samples(L, arrs, rng_seed: int = 11, n_random: int = 4096):
    """Indices of every block (both ends, tensor boundaries, a random sample)
    and the host state's values there: taken right after the streamed steps,
    checked against the oracle later (parity_stream)."""
    import numpy as np
    rng = np.random.default_rng(rng_seed)
    out = []
    for i in range(L.n_layers):
        p = L.padded(i)
        idx = [np.arange(min(256, p)), np.arange(max(0, p - 256), p), rng.integers(0, p, n_random)]
        for (_, off, n) in L.spans(i):
            idx.append(np.array([e for e in (off, off + n - 1) if 0 <= e < p], dtype=np.int64))
        idx = np.unique(np.concatenate(idx).astype(np.int64))
        v = L.numpy_views(i, arrs[i])
        out.append((idx, {f: v[f][idx].copy() for f in L.fields()}))
    return out


def parity_stream(L, samples, workload: str, seed: int, hp_kw, steps: int, first_block: int = 0):
    """The oracle follows the sampled elements from the generator's inputs at
    t = 1 through steps t = 1..steps (step t's gradient drawn with
    grad_seed(t)) and compares them with what the streamed steps left in the
    host blocks: every byte, or the error figures."""
    import numpy as np
    import oracle
    import synth
    fields = L.fields()
    n, exact, worst = 0, True, {"max_rel_err_fp32": 0.0, "max_ulp_bf16": 0, "nan_outputs": 0}
    for i, (idx, got) in enumerate(samples):
        blk = first_block + i
        cur = {f: np.ascontiguousarray(synth.gather_block(f, L.fmt, L.spans(i), blk, workload, 1, idx, seed,
                                                          grad_seed(workload, seed, 1))) for f in fields}
        for t in range(1, steps + 1):
            if t > 1:
                cur["G"] = np.ascontiguousarray(synth.gather_block("G", L.fmt, L.spans(i), blk, workload, t, idx,
                                                                   seed, grad_seed(workload, seed, t)))
            oracle.step(L.fmt, cur, oracle.hparams(step=t, **hp_kw))
        n += idx.size
        for f in fields:
            if f != "G" and not np.array_equal(got[f].view(np.uint8), cur[f].view(np.uint8)):
                exact = False
        e = field_errors(L.fmt, got, cur, fields)
        worst = {k: max(worst[k], e[k]) if k != "nan_outputs" else worst[k] + e[k] for k in worst}
    return dict({"steps": steps, "elements": n, "bit_exact": exact}, **worst)


# ---------------------------------------------------------------------------
def run_reference(args):
    """The oracle alone, on the host cores: each step a bounded sample of the
    workload. Geometry, inputs and arithmetic come from oracle/ and synth/
    only; the product library is never loaded in this process."""
    import numpy as np
    import oracle
    from oracle import layout as olayout
    import synth
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    fmt = WORKLOADS[args.workload][1]
    plan = olayout.plan(workload_specs(args.workload, args.max_blocks), fmt)
    hp_kw = HP_LORA if fmt == "L16F" else HP
    threads = os.cpu_count() or 1
    # The sample: blocks from the start of the model, about 2 GiB of state at
    # most (so the run leaves the host's memory much as it found it); a block
    # larger than what is left contributes its first elements (the update is
    # elementwise, so a prefix of every segment is a smaller block of the same
    # kind). Stops early once a step would take --ref-step-s.
    budget = args.ref_sample_bytes
    sample, state, step_est = [], 0, 0.0
    for b in plan.blocks:
        if state >= budget or step_est >= args.ref_step_s:
            break
        per_elem = b.nbytes // max(1, b.padded)
        if sample and budget - state < 2048 * per_elem:
            break
        n = b.padded if state + b.nbytes <= budget else max(2048, (budget - state) // per_elem // 2048 * 2048)
        n = min(n, b.padded)
        spans = [(name, off, max(0, min(cnt, n - off))) for (name, off, cnt) in b.spans if off < n]
        fields = {f: np.zeros(n, olayout.field_dtype(fmt, f)) for f, _ in olayout.FORMATS[fmt]}
        synth.fill_block(fields, spans, b.layer, args.workload, fmt, t=1, seed=args.seed,
                         g_seed=grad_seed(args.workload, args.seed, 1))
        t0 = time.perf_counter()
        oracle.step(fmt, fields, oracle.hparams(step=1, **hp_kw), threads=threads)
        step_est += time.perf_counter() - t0
        sample.append((b.layer, n, fields, sum(c for (_, _, c) in spans)))
        state += n * per_elem
    sample_params = sum(s[3] for s in sample)
    for w in range(args.warmup):
        for (_, _, fields, _) in sample:
            oracle.step(fmt, fields, oracle.hparams(step=2 + w, **hp_kw), threads=threads)
    t0 = time.perf_counter()
    for k in range(args.steps):
        for (_, _, fields, _) in sample:
            oracle.step(fmt, fields, oracle.hparams(step=2 + args.warmup + k, **hp_kw), threads=threads)
    el = time.perf_counter() - t0
    value = sample_params * args.steps / el
    last = sample[-1]
    desc = (f"blocks {sample[0][0]}..{last[0]} of {len(plan.blocks)}"
            + (f" (block {last[0]}: its first {last[1]} of {plan.blocks[last[0]].padded} elements)"
               if last[1] < plan.blocks[last[0]].padded else "")
            + f", {sample_params} of {plan.n_params} params per step, oracle on {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_for(fmt, plan.n_params, [b.nbytes for b in plan.blocks], args.workload, world,
                             args.max_blocks),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_note(state_bytes: int) -> str:
    return ("inputs larger than twice the L2 (no flush)" if state_bytes >= 2 * (132 << 20) else
            "L2 flushed before every timed launch (a write of twice its size, then a read of another such buffer)")


def config_for(fmt, n_params, block_bytes, workload, world, max_blocks=0, shard=False, params_job=None):
    desc = WORKLOADS[workload][2]
    if max_blocks > 0:
        desc += f", first {max_blocks} blocks only"
    state = sum(block_bytes)
    sharded = shard and world > 1
    cfg = {"workload": desc, "name": workload, "layout": fmt,
           "params": int(params_job) if sharded and params_job else int(n_params),
           "blocks": len(block_bytes), "state_bytes": int(state), "l2": l2_note(state),
           "parallelism": (f"blocks sharded x{world} (rank 0: {len(block_bytes)} blocks, {n_params} params)"
                           if sharded else f"replicas x{world}"),
           "hparams": HP_LORA if fmt == "L16F" else HP}
    if workload in FRESH_GRAD_STEPS:
        cfg["gradient"] = "drawn afresh for every step t with seed + t"
        cfg["stream_steps"] = f"t = 1..{FRESH_GRAD_STEPS[workload]} from the initial state"
    return cfg


def layout_config(L, workload, world, max_blocks=0, shard=False, params_job=None):
    return config_for(L.fmt, L.n_params, [L.block_bytes(i) for i in range(L.n_layers)], workload, world,
                      max_blocks, shard, params_job)


def block_link_rates(torch, arrs, dev):
    """Host-to-device and device-to-host rate of each pinned block, one
    whole-block copy each way (GB/s, CUDA events on one stream; the copy back
    writes the bytes the first copy just read): on a host where some pinned
    allocations are slow, in either direction, this names them. Returns
    (h2d rates, d2h rates)."""
    s = torch.cuda.Stream()
    h2d, d2h = [], []
    for a in arrs:
        n = a.size
        h = torch.from_numpy(a)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        with torch.cuda.stream(s):
            e[0].record(s)
            dev[:n].copy_(h, non_blocking=True)
            e[1].record(s)
            h.copy_(dev[:n], non_blocking=True)
            e[2].record(s)
        e[2].synchronize()
        h2d.append(n / (e[0].elapsed_time(e[1]) / 1e3) / 1e9)
        d2h.append(n / (e[1].elapsed_time(e[2]) / 1e3) / 1e9)
    return h2d, d2h


def slow_block_flags(rates, frac: float = 0.85):
    """Per block: is either direction under `frac` of the best block's rate?"""
    h2d, d2h = rates
    return [r < frac * max(h2d) or q < frac * max(d2h) for r, q in zip(h2d, d2h)]


def heal_pinned_state(torch, L, ptrs, arrs, dev, tries: int = 3, max_extra_bytes: int = 40 << 30,
                      frac: float = 0.85, rates=None):
    """Health check of the pinned state blocks. On the GB300 hosts here, some
    pinned allocations are moved by the copy engines at a fraction of the link
    rate (a few GB/s to about half), for their whole lifetime (more of them
    after other processes have pinned and freed a lot of memory), and the
    slowest block sets the pace of a streamed step. A block whose
    host-to-device or device-to-host rate is under `frac` of the best block's
    in that direction is copied into a fresh allocation, up to `tries` times;
    replaced allocations stay pinned until the caller frees them (returned),
    so the allocator does not hand the same pages straight back. Returns (slow
    blocks before, blocks replaced, allocations to free)."""
    import ctypes
    import numpy as np
    from optimizer_update_gb300 import lst
    rates = rates if rates is not None else block_link_rates(torch, arrs, dev)
    best_h2d, best_d2h = max(rates[0]), max(rates[1])
    slow = slow_block_flags(rates, frac)
    slow_before = sum(slow)
    retired, healed, extra = [], 0, 0
    for i in range(len(arrs)):
        k = 0
        bad = slow[i]
        while bad and k < tries:
            n = arrs[i].size
            if extra + n > max_extra_bytes:
                break
            p = lst.lst_host_alloc(n)
            a = np.ctypeslib.as_array((ctypes.c_uint8 * n).from_address(p))
            a[:] = arrs[i]
            retired.append(ptrs[i])
            ptrs[i], arrs[i] = p, a
            extra += n
            h, d = block_link_rates(torch, [a], dev)
            bad = h[0] < frac * best_h2d or d[0] < frac * best_d2h
            k += 1
        if k:
            healed += 1
    return slow_before, healed, retired


def link_bandwidth(torch, host_ptr_arrs, dev_a, dev_b, nbytes: int, reps: int = 5):
    """Pinned host <-> device copy bandwidth: H2D alone, D2H alone, both at once
    (each direction timed on its own stream with CUDA events), on the given
    host arrays (blocks of the state: the rate is the one the state's own
    memory gets). The device-to-host direction writes back into the state, so
    dev_b first receives a copy of exactly those bytes: every timed copy
    rewrites the bytes that are already there."""
    h_in = torch.from_numpy(host_ptr_arrs[0][:nbytes])
    h_out = torch.from_numpy(host_ptr_arrs[1][:nbytes])
    dev_b[:nbytes].copy_(h_out)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(h2d: bool, d2h: bool):
        best = [float("inf"), float("inf")]
        for _ in range(reps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            torch.cuda.synchronize()
            if h2d:
                e[0].record(s1)
                with torch.cuda.stream(s1):
                    dev_a[:nbytes].copy_(h_in, non_blocking=True)
                e[1].record(s1)
            if d2h:
                e[2].record(s2)
                with torch.cuda.stream(s2):
                    h_out.copy_(dev_b[:nbytes], non_blocking=True)
                e[3].record(s2)
            torch.cuda.synchronize()
            if h2d:
                best[0] = min(best[0], e[0].elapsed_time(e[1]) / 1e3)
            if d2h:
                best[1] = min(best[1], e[2].elapsed_time(e[3]) / 1e3)
        return [nbytes / t / 1e9 if t < float("inf") else None for t in best]

    h2d_alone, _ = timed(True, False)
    _, d2h_alone = timed(False, True)
    h2d_conc, d2h_conc = timed(True, True)
    return {"h2d_gbs": h2d_alone, "d2h_gbs": d2h_alone, "h2d_concurrent_gbs": h2d_conc,
            "d2h_concurrent_gbs": d2h_conc, "bytes": nbytes}


def copy_choice_summary(L):
    """What the streamed steps' default copy mode (LST_COPY_AUTO) has learned:
    sub-chunks timed, how many of them later steps move with the copy kernel
    each way, and the slowest copy-engine sub-chunk rates it timed."""
    cs = [L.stream_copy_choice(i) for i in range(L.n_layers)]
    m = [c for c in cs if c["measured"]]
    out = {"blocks_measured": len(m), "chunks": sum(c["chunks"] for c in m),
           "kernel_in_chunks": sum(c["kernel_in_chunks"] for c in m),
           "kernel_out_chunks": sum(c["kernel_out_chunks"] for c in m)}
    h = [c["engine_h2d_gbs_min"] for c in m if c["engine_h2d_gbs_min"] > 0]
    d = [c["engine_d2h_gbs_min"] for c in m if c["engine_d2h_gbs_min"] > 0]
    out["engine_h2d_gbs_min"] = min(h) if h else None
    out["engine_d2h_gbs_min"] = min(d) if d else None
    return out


def timed_launches(torch, stream, launch, steps, flush, flush_rd):
    """Per-launch device times (s) of `steps` launches, CUDA events on the
    launching stream around each, the L2 flushed before each when a flush
    buffer is given (outside the event pair)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
                flush_rd.sum()
        starts[k].record(stream)
        launch()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return [starts[k].elapsed_time(ends[k]) / 1e3 for k in range(steps)]


def l2_flush_buffers(torch, device, state_bytes: int):
    """For a state under twice the L2: a buffer of twice the L2 to write (the
    flush) and one to read (which writes the flush's dirty lines back), so a
    timed launch starts cold and clean. (None, None) otherwise."""
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (132 << 20))
    if state_bytes >= 2 * l2:
        return None, None
    return (torch.empty(2 * l2, dtype=torch.uint8, device=device),
            torch.zeros(2 * l2 // 4, dtype=torch.int32, device=device))


def device_leg(args, L, dptrs, hp_kw, stream, device, world, P_job, peak, t0_step: int = 1):
    """The device-resident lst_adamw_step: warm-up, then args.steps timed
    launches (one multi-block launch per step). Returns (result dict, next t,
    per-launch times, flush buffers)."""
    import torch
    from optimizer_update_gb300 import lst
    state_bytes = sum(L.block_bytes(i) for i in range(L.n_layers))
    flush, flush_rd = l2_flush_buffers(torch, device, state_bytes)
    ptr_arr = lst._ptr_array(dptrs)
    hp = lst.adamw_hparams(step=t0_step, **hp_kw)
    call = lst.lib().lst_adamw_step
    t = [t0_step]

    def launch():
        hp.step = t[0]
        st = call(L.handle, ptr_arr, ctypes.byref(hp), stream.cuda_stream)
        if st != lst.LST_OK:
            raise lst.LstError(st, lst.lst_last_error())
        t[0] += 1

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize(device)
    barrier(device)
    torch.cuda.synchronize(device)
    per_launch = timed_launches(torch, stream, launch, args.steps, flush, flush_rd)
    torch.cuda.synchronize(device)
    barrier(device)
    torch.cuda.synchronize(device)
    t_dev = sum(per_launch)
    t_dev_max = max_over_ranks(t_dev, device)
    avg = t_dev / args.steps
    alg_bytes = ALG_BYTES[L.fmt] * L.n_params
    # the launch path picks the cross-run kernel below about twice the L2
    kname = "lst_update_small_kernel" if alg_bytes < SMALL_LAUNCH_BYTES else "lst_update_kernel"
    res = {"value": P_job * args.steps / t_dev_max, "t_dev_max": t_dev_max, "avg_launch": avg,
           "achieved_gbs": alg_bytes / avg / 1e9, "frac_of_hbm_peak": alg_bytes / avg / 1e9 / peak,
           "alg_bytes": alg_bytes, "kernel": kname, "per_launch": per_launch}
    # state under twice the L2: also back to back without the flush (the
    # launches then find part of the state in L2), beside the cold figure
    if flush is not None:
        wk = max(3, args.steps // 2)
        wms = timed_launches(torch, stream, launch, wk, None, None)
        res["back_to_back_l2_warm"] = {"median_launch_ms": 1e3 * statistics.median(wms), "launches": wk,
                                       "algorithmic_gbs": alg_bytes / statistics.median(wms) / 1e9}
    else:
        res["back_to_back_l2_warm"] = None
    return res, t[0], flush, flush_rd


def device_blocks_from_generator(torch, L, workload, seed, device, first_block=0):
    """Device blocks holding the state at t = 1, drawn block by block on the
    host into one pinned staging buffer and copied over."""
    import ctypes
    import numpy as np
    import synth
    from optimizer_update_gb300 import lst
    stage_p = lst.lst_host_alloc(max(1, L.max_block_bytes))
    try:
        stage = np.ctypeslib.as_array((ctypes.c_uint8 * max(1, L.max_block_bytes)).from_address(stage_p))
        dev = []
        for i in range(L.n_layers):
            n = L.block_bytes(i)
            synth.fill_block(L.numpy_views(i, stage[:n]), L.spans(i), first_block + i, workload, L.fmt, t=1,
                             seed=seed, g_seed=grad_seed(workload, seed, 1))
            d = torch.empty(n, dtype=torch.uint8, device=device)
            d.copy_(torch.from_numpy(stage[:n]))
            dev.append(d)
        torch.cuda.synchronize(device)
    finally:
        lst.lst_host_free(stage_p)
    return dev


def configs_leg(args, device, world, seed, peak):
    """The device-resident step (plain, per-block options, SGD form) on the
    other workloads, each timed like the main device-resident leg."""
    import torch
    out = {}
    for name in CONFIG_LEGS:
        if name == args.workload:
            continue
        try:
            L = build_layout(name)
            hp_kw = HP_LORA if L.fmt == "L16F" else HP
            dev = device_blocks_from_generator(torch, L, name, seed, device)
            dptrs = [d.data_ptr() for d in dev]
            stream = torch.cuda.Stream(device=device)
            P_job = sum_over_ranks(L.n_params, device)
            state = sum(L.block_bytes(i) for i in range(L.n_layers))
            # steps of tens of microseconds (a state under a few hundred MB)
            # vary by a microsecond or two from launch to launch: time at
            # least 200 of them
            cargs = argparse.Namespace(**vars(args))
            if state < (512 << 20):
                cargs.steps = max(args.steps, 200)
            res, t, flush, flush_rd = device_leg(cargs, L, dptrs, hp_kw, stream, device, world, P_job, peak)
            opt = time_options_leg(cargs, L, dptrs, hp_kw, stream, device, world, t, flush, flush_rd, peak)
            sgd = time_sgd_leg(cargs, L, dptrs, hp_kw, stream, device, world, flush, flush_rd, peak)
            out[name] = {"workload": WORKLOADS[name][2], "layout": L.fmt, "params": L.n_params,
                         "blocks": L.n_layers, "state_bytes": state, "l2": l2_note(state),
                         "value": res["value"], "unit": "params/s", "kernel": f"{res['kernel']}<{L.fmt}>",
                         "achieved_gbs": res["achieved_gbs"], "frac_of_hbm_peak": res["frac_of_hbm_peak"],
                         "avg_launch_ms": 1e3 * res["avg_launch"],
                         "median_launch_ms": 1e3 * statistics.median(res["per_launch"]), "steps": cargs.steps,
                         "back_to_back_l2_warm": res["back_to_back_l2_warm"],
                         "options": {k: opt[k] for k in ("value", "frac_of_hbm_peak", "avg_launch_ms",
                                                         "grad_sq_all_positive_finite")},
                         "sgd": {k: sgd[k] for k in ("value", "frac_of_hbm_peak", "avg_launch_ms")}}
            del dev, flush, flush_rd
        except Exception as e:  # recorded in the line; the main result stands
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import numpy as np
    import torch
    from optimizer_update_gb300 import lst

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init("nccl")
    # Replicas pin one copy of the state per rank; where the ranks on this
    # host could not all hold one (82 GB each for the Llama-70B slice), they
    # split the model's blocks instead (strong scaling). Decided together:
    # any rank short of memory makes every rank shard.
    auto_shard = False
    if world > 1 and not args.shard:
        full = build_layout(args.workload, args.max_blocks)
        state = sum(full.block_bytes(i) for i in range(full.n_layers))
        local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", world))
        short = 0 if replicas_fit(state, local_ranks, host_mem_available()) else 1
        if sum_over_ranks(short, device) > 0:
            args.shard = auto_shard = True
    # replicas draw their own state; shards are parts of one model (one seed)
    seed = args.seed if args.shard else replica_seed(args.seed, rank)

    L, first_block = rank_layout(args.workload, args.max_blocks, args.shard, rank, world)
    hp_kw = HP_LORA if L.fmt == "L16F" else HP
    P = L.n_params
    P_job = sum_over_ranks(P, device)  # parameters all ranks update per step
    chunk = 1 << 24  # 16 Mi elements per sub-chunk (the library default)
    L.set_stream_chunk(chunk)
    state_bytes = sum(L.block_bytes(i) for i in range(L.n_layers))
    ptrs, arrs = alloc_pinned_state(L, args.workload, seed, first_block)
    huge_bytes = anon_huge_page_bytes()  # the pinned blocks' share of huge pages
    peak, peak_kind = measured_peaks()
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(vis[local] if local < len(vis) else str(local))
    clocks.start()

    # ---- device-resident leg -------------------------------------------------
    dev = []
    for i in range(L.n_layers):
        d = torch.empty(L.block_bytes(i), dtype=torch.uint8, device=device)
        d.copy_(torch.from_numpy(arrs[i]), non_blocking=False)
        dev.append(d)
    dptrs = [d.data_ptr() for d in dev]
    stream = torch.cuda.Stream(device=device)
    time.sleep(0.3)
    res, t, flush, flush_rd = device_leg(args, L, dptrs, hp_kw, stream, device, world, P_job, peak)
    clk = clocks.snapshot()
    value, t_dev_max = res["value"], res["t_dev_max"]
    avg_launch, per_launch, alg_bytes, kname = res["avg_launch"], res["per_launch"], res["alg_bytes"], res["kernel"]
    achieved = res["achieved_gbs"]
    traffic = kernel_traffic(kname, L.fmt, P)
    # ---- per-block options leg: lst_adamw_step_ex with a step counter per
    # block (staggered, as after progressive locking) and every block's
    # sum of g^2 returned by the same pass ---------------------------------------
    options = time_options_leg(args, L, dptrs, hp_kw, stream, device, world, t, flush, flush_rd, peak)
    sgd = time_sgd_leg(args, L, dptrs, hp_kw, stream, device, world, flush, flush_rd, peak)
    del dev, flush, flush_rd
    torch.cuda.empty_cache()

    # ---- host link, measured in this run -------------------------------------
    buf0 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device=device)
    buf1 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device=device)
    big = [i for i in range(L.n_layers) if L.block_bytes(i) >= min(1 << 30, L.max_block_bytes)]
    nb = min(arrs[big[0] if big else 0].size, arrs[big[-1] if len(big) > 1 else -1].size, buf0.numel(), 1 << 30)

    def probe_pair():
        return (arrs[big[0]] if big else arrs[0]), (arrs[big[-1]] if len(big) > 1 else arrs[-1])

    h2d_b = sum(L.transfer(i)[1] for i in range(L.n_layers))
    d2h_b = sum(L.transfer(i)[3] for i in range(L.n_layers))
    n_stream = FRESH_GRAD_STEPS.get(args.workload, max(1, min(args.steps, args.e2e_steps)))

    def stream_call(tt):
        lst.lst_stream_step(L.handle, ptrs, buf0.data_ptr(), buf1.data_ptr(), lst.adamw_hparams(step=tt, **hp_kw),
                            600_000)

    # ---- the streamed step as a caller gets it: the pinned blocks as first
    # allocated, before the health check below replaces slow allocations -------
    link_before = link_bandwidth(torch, list(probe_pair()), buf0, buf1, nb)
    pre = []
    for k in range(3):
        t0w = time.perf_counter()
        stream_call(t)
        t += 1
        pre.append(time.perf_counter() - t0w)
    choice_before = copy_choice_summary(L)
    # the same three steps with every sub-chunk on the copy engines (the mode
    # that learns nothing), on the same allocations, for comparison
    L.set_stream_copy(lst.LST_COPY_ENGINE, lst.LST_COPY_ENGINE)
    pre_engine = []
    for k in range(3):
        t0w = time.perf_counter()
        stream_call(t)
        t += 1
        pre_engine.append(time.perf_counter() - t0w)
    L.set_stream_copy(lst.LST_COPY_AUTO, lst.LST_COPY_AUTO)
    rates_before = block_link_rates(torch, arrs, buf0)
    roof_before = max(h2d_b / (link_before["h2d_concurrent_gbs"] * 1e9),
                      d2h_b / (link_before["d2h_concurrent_gbs"] * 1e9))
    e2e_before_heal = {"value": P_job / statistics.median(pre), "unit": "params/s", "call": "lst_stream_step",
                       "step_ms": [1e3 * x for x in pre], "median_step_ms": 1e3 * statistics.median(pre),
                       "frac_of_link_roofline": roof_before / statistics.median(pre),
                       "note": "first three calls on the pinned blocks as allocated (lst_host_alloc), "
                               "before slow allocations are replaced",
                       "copy_choice": choice_before,
                       "copy_engines_only": {"step_ms": [1e3 * x for x in pre_engine],
                                             "median_step_ms": 1e3 * statistics.median(pre_engine),
                                             "frac_of_link_roofline": roof_before / statistics.median(pre_engine)},
                       "block_h2d_gbs_min": min(rates_before[0]), "block_d2h_gbs_min": min(rates_before[1]),
                       "slow_blocks": sum(slow_block_flags(rates_before))}
    heal_budget = min(40 << 30, state_bytes // 2)  # as replicas_fit allows for
    slow_before_heal, healed, retired = heal_pinned_state(torch, L, ptrs, arrs, buf0, max_extra_bytes=heal_budget)
    a0, a1 = probe_pair()
    link = link_bandwidth(torch, [a0, a1], buf0, buf1, nb)

    # ---- streamed leg (the public end-to-end call) ------------------------------
    # On the shared hosts here, host-link throughput also varies from moment
    # to moment (besides the slow allocations the health check above
    # replaces), so the streamed legs warm up until two steps agree; the link
    # is measured again after the streamed legs.
    stream_warm, t = warm_until_stable(stream_call, t)
    # The timed steps start from the initial state: t = 1 with zero moments
    # and step 1's gradient, each later step's gradient drawn before the step
    # (outside the timed region, standing in for the backward pass).
    if args.workload in FRESH_GRAD_STEPS:
        draw_state(L, arrs, args.workload, seed, first_block)
        t_first = 1
    else:
        t_first = t
    # every block's own rates both ways, right before the timed steps (a
    # slow pinned allocation holds up the pipeline): a block that has become
    # slow since the health check is replaced as well
    block_rates = block_link_rates(torch, arrs, buf0)
    slow_late, healed_late, retired_late = heal_pinned_state(torch, L, ptrs, arrs, buf0, rates=block_rates,
                                                             max_extra_bytes=heal_budget)
    retired += retired_late
    if healed_late:
        block_rates = block_link_rates(torch, arrs, buf0)
    step_times = []
    # sub-chunks the timed steps move with the SM copy kernel (what the
    # default copy mode learned so far): one copy-kernel launch per run of
    # equal-width segments (two per direction, one for the fp32 layout)
    cc_timed = copy_choice_summary(L)
    sm_launches = (1 if L.fmt == "L16F" else 2) * (cc_timed["kernel_in_chunks"] + cc_timed["kernel_out_chunks"])
    for k in range(n_stream):
        tt = t_first + k
        if args.workload in FRESH_GRAD_STEPS and k > 0:
            redraw_gradients(L, arrs, args.workload, seed, tt, first_block)
        torch.cuda.synchronize(device)
        barrier(device)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        stream_call(tt)
        torch.cuda.synchronize(device)
        step_times.append(time.perf_counter() - t0)
    t = max(t, t_first + n_stream)
    samples = stream_samples(L, arrs) if (rank == 0 and args.workload in FRESH_GRAD_STEPS) else None
    t_e2e = sum(step_times)
    t_e2e_max = max_over_ranks(t_e2e, device)
    e2e_value = P_job * n_stream / t_e2e_max
    chunks = sum((L.padded(i) + chunk - 1) // chunk for i in range(L.n_layers))
    roof_t = max(h2d_b / (link["h2d_concurrent_gbs"] * 1e9), d2h_b / (link["d2h_concurrent_gbs"] * 1e9))
    # the same bytes with the two directions one after the other (each at its
    # measured bandwidth alone): what the three-stream overlap saves
    serial_t = h2d_b / (link["h2d_gbs"] * 1e9) + d2h_b / (link["d2h_gbs"] * 1e9)
    stream_info = dict(link, step_ms=1e3 * t_e2e / n_stream, step_ms_each=[1e3 * x for x in step_times],
                       steps=n_stream, t_first=t_first, serial_copies_ms=1e3 * serial_t,
                       achieved_h2d_gbs=h2d_b * n_stream / t_e2e / 1e9,
                       achieved_d2h_gbs=d2h_b * n_stream / t_e2e / 1e9,
                       roofline_ms=1e3 * roof_t, frac_of_link_roofline=roof_t / (t_e2e / n_stream),
                       chunk_elems=chunk, warmup_steps=stream_warm,
                       host_huge_page_bytes=huge_bytes, host_state_bytes=state_bytes,
                       block_h2d_gbs_min=min(block_rates[0]), block_h2d_gbs_median=statistics.median(block_rates[0]),
                       block_d2h_gbs_min=min(block_rates[1]), block_d2h_gbs_median=statistics.median(block_rates[1]),
                       slow_blocks=sum(slow_block_flags(block_rates)),
                       slow_blocks_before_heal=slow_before_heal, healed_blocks=healed,
                       copy_choice=copy_choice_summary(L),
                       last_step=L.stream_last_stats(),
                       slow_blocks_before_timed_steps=slow_late, healed_before_timed_steps=healed_late,
                       link_before_heal={k: link_before[k] for k in ("h2d_gbs", "d2h_gbs", "h2d_concurrent_gbs",
                                                                     "d2h_concurrent_gbs")})

    # ---- streamed leg with the gradients produced on the device by a
    # backward stand-in (the generator's GPU twin), block by block last to
    # first, each block released by its Backward-Done event: only the state
    # crosses the link inbound, and the step overlaps the production ---------
    stream_devgrad = devgrad_leg(args, L, ptrs, buf0, buf1, hp_kw, device, P_job, link, d2h_b, seed, first_block,
                                 t)
    t = stream_devgrad.pop("next_t")

    # ---- zero-copy leg: the update kernel directly on the pinned host blocks ----
    zstream = torch.cuda.Stream(device=device)
    def zc_call(tt):
        lst.lst_zero_copy_step(L.handle, ptrs, lst.adamw_hparams(step=tt, **hp_kw), zstream.cuda_stream)
        torch.cuda.synchronize(device)
    zc_warm, t = warm_until_stable(zc_call, t)
    e_steps = n_stream
    barrier(device)
    zs, ze = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    zs.record(zstream)
    for _ in range(e_steps):
        lst.lst_zero_copy_step(L.handle, ptrs, lst.adamw_hparams(step=t, **hp_kw), zstream.cuda_stream)
        t += 1
    ze.record(zstream)
    torch.cuda.synchronize(device)
    t_zc = max_over_ranks(zs.elapsed_time(ze) / 1e3, device)
    link_after = link_bandwidth(torch, [a0, a1], buf0, buf1, nb)
    stream_info["link_after"] = {k: link_after[k] for k in ("h2d_gbs", "d2h_gbs", "h2d_concurrent_gbs",
                                                             "d2h_concurrent_gbs")}
    zero_copy = {"value": P_job * e_steps / t_zc, "unit": "params/s", "call": "lst_zero_copy_step",
                 "step_ms": 1e3 * t_zc / e_steps, "link_bytes_per_step": h2d_b + d2h_b,
                 "frac_of_link_roofline": roof_t / (t_zc / e_steps), "steps": e_steps, "warmup_steps": zc_warm}

    # ---- file-backed store leg (opt-in: writes the state to disk) ---------------
    store = None
    if args.store_dir:
        store = run_store_leg(args, L, ptrs, buf0, buf1, hp_kw, device, world, rank)
    del buf0, buf1
    torch.cuda.empty_cache()

    # ---- CPU baseline: the oracle on the host cores, bounded sample ------------
    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        rate, done, el, nblocks = cpu_oracle_rate(L, arrs, hp_kw, args.cpu_budget_s, threads)
        cpu = {"value": rate, "unit": "params/s", "cores": threads, "kind": "oracle",
               "sample": f"{nblocks} block updates ({done} params) of this workload's state in {el:.1f} s"}
        parity = parity_sample(L, arrs, hp_kw, device, threads)
        if samples is not None and parity is not None:
            parity["stream"] = parity_stream(L, samples, args.workload, seed, hp_kw, n_stream, first_block)

    for p in ptrs + retired:
        lst.lst_host_free(p)
    arrs = []

    # ---- the other workloads, device-resident --------------------------------
    configs = configs_leg(args, device, world, seed, peak) if not args.no_configs else None
    clk_all = clocks.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_dev_max / args.steps, "higher_is_better": True,
            "scaling": "strong" if (args.shard and world > 1) else "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": dict(layout_config(L, args.workload, world, args.max_blocks, args.shard, P_job),
                           **({"sharded_because": "a pinned replica per rank would not fit in host memory"}
                              if auto_shard else {})),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": f"{kname}<{L.fmt}>", "alg_bytes_per_launch": alg_bytes,
                         "avg_launch_ms": 1e3 * avg_launch, "median_launch_ms": 1e3 * statistics.median(per_launch),
                         "min_launch_ms": 1e3 * min(per_launch), "peak_source": f"{peak_kind} hbm_gbs",
                         "back_to_back_l2_warm": res["back_to_back_l2_warm"]},
            "e2e": {"value": e2e_value, "unit": "params/s", "h2d_bytes_per_step": h2d_b,
                    "d2h_bytes_per_step": d2h_b, "steps": n_stream, "call": "lst_stream_step",
                    "gpu_launches": n_stream * (chunks + sm_launches)},
            "e2e_before_heal": e2e_before_heal,
            "options": options,
            "sgd": sgd,
            "stream": stream_info,
            "zero_copy": zero_copy,
            "stream_devgrad": stream_devgrad,
            **({"store": store} if store is not None else {}),
            "configs": configs,
            "cpu_baseline": cpu,
            "parity": parity,
            "clocks": clk,
            "clocks_whole_run": clk_all,
            "gpu_launches": args.steps,
        }
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


def warm_until_stable(call, t: int, lo: int = 3, hi: int = 12, tol: float = 0.05):
    """Untimed calls call(t), call(t + 1), ... until two in a row take times
    within `tol` of each other (at least `lo` calls, at most `hi`). Returns
    (calls made, the next step counter)."""
    prev, n = None, 0
    while True:
        t0 = time.perf_counter()
        call(t)
        t += 1
        n += 1
        dt = time.perf_counter() - t0
        if (n >= lo and prev is not None and abs(dt - prev) <= tol * prev) or n >= hi:
            return n, t
        prev = dt


def devgrad_leg(args, L, ptrs, buf0, buf1, hp_kw, device, P_job, link, d2h_b, seed, first_block, t):
    """lst_stream_step_devgrad_events fed by a gradient producer on the
    device (synth.device_fill_field: the generator's values, written block by
    block in backward order, n-1 .. 0, on its own stream, an event recorded
    after each block). The timed region of a step holds the production and
    the streamed step: from before the producer is enqueued until the call
    returns. Step t's gradient is drawn with grad_seed(t). The roofline is
    max(producer alone, the link time of the bytes moved). A second
    measurement slows the producer (extra hash rounds per element, calibrated
    to about 0.8 of the link time) to show the two overlapping: the step then
    takes about the larger of the two, not their sum."""
    import torch
    import synth
    from optimizer_update_gb300 import lst
    n = L.n_layers
    order = list(reversed(range(n)))
    grads = [torch.empty(L.segment(i, "G")[1], dtype=torch.uint8, device=device) for i in range(n)]
    gptrs = [g.data_ptr() for g in grads]
    producer = torch.cuda.Stream(device=device)
    dg_h2d = sum(L.transfer(i)[1] - L.segment(i, "G")[1] for i in range(n))
    roof_link = max(dg_h2d / (link["h2d_concurrent_gbs"] * 1e9), d2h_b / (link["d2h_concurrent_gbs"] * 1e9))

    def produce(tt, passes, events=None):
        gs = grad_seed(args.workload, seed, tt)
        for i in order:
            synth.device_fill_field(gptrs[i], "G", L.fmt, L.spans(i), L.padded(i), first_block + i, args.workload,
                                    tt, seed if gs is None else gs, producer.cuda_stream, passes)
            if events is not None:
                events[i].record(producer)

    def producer_alone(tt, passes, reps=2):
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(device)
            e0.record(producer)
            produce(tt, passes)
            e1.record(producer)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        return best

    def overlapped(tt, passes):
        """One step: enqueue the producer (async), then the synchronous
        streamed step; wall time of both."""
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        events = [torch.cuda.Event() for _ in range(n)]
        produce(tt, passes, events)
        lst.lst_stream_step_devgrad_events(L.handle, ptrs, gptrs, [e.cuda_event for e in events], order,
                                           buf0.data_ptr(), buf1.data_ptr(), lst.adamw_hparams(step=tt, **hp_kw),
                                           None, 600_000)
        torch.cuda.synchronize(device)
        return time.perf_counter() - t0

    def serial(tt, passes):
        """The same work without overlap: produce every gradient, wait, then
        the streamed step with the gradients complete."""
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        produce(tt, passes)
        producer.synchronize()
        lst.lst_stream_step_devgrad(L.handle, ptrs, gptrs, buf0.data_ptr(), buf1.data_ptr(),
                                    lst.adamw_hparams(step=tt, **hp_kw), None, 600_000)
        torch.cuda.synchronize(device)
        return time.perf_counter() - t0

    prod_s = producer_alone(t, 1)
    n_warm, t = warm_until_stable(lambda tt: overlapped(tt, 1), t)
    e_steps = FRESH_GRAD_STEPS.get(args.workload, max(1, min(args.steps, args.e2e_steps)))
    barrier(device)
    times = []
    for _ in range(e_steps):
        times.append(overlapped(t, 1))
        t += 1
    t_dg = max_over_ranks(sum(times), device)
    roof = max(prod_s, roof_link)
    out = {"value": P_job * e_steps / t_dg, "unit": "params/s", "call": "lst_stream_step_devgrad_events",
           "producer": "synth.device_fill_field, blocks n-1..0, one Backward-Done event per block",
           "step_ms": 1e3 * t_dg / e_steps, "producer_alone_ms": 1e3 * prod_s, "link_roofline_ms": 1e3 * roof_link,
           "roofline_ms": 1e3 * roof, "frac_of_roofline": roof / (t_dg / e_steps),
           "h2d_bytes_per_step": dg_h2d, "d2h_bytes_per_step": d2h_b, "steps": e_steps, "warmup_steps": n_warm}
    # the step with the gradients complete before the call (no producer in
    # the timed region), for comparison
    t0 = time.perf_counter()
    lst.lst_stream_step_devgrad(L.handle, ptrs, gptrs, buf0.data_ptr(), buf1.data_ptr(),
                                lst.adamw_hparams(step=t, **hp_kw), None, 600_000)
    out["gradients_ready_step_ms"] = 1e3 * (time.perf_counter() - t0)
    t += 1
    # a producer as slow as a backward pass: calibrate its extra rounds
    p_cal = 32
    c_cal = producer_alone(t, p_cal, reps=1)
    per_pass = max(1e-9, (c_cal - prod_s) / (p_cal - 1))
    passes = int(max(1, min(20000, 1 + (0.8 * roof_link - prod_s) / per_pass)))
    heavy_prod = producer_alone(t, passes, reps=1)
    ov = overlapped(t, passes)
    t += 1
    se = serial(t, passes)
    t += 1
    stream_only = out["gradients_ready_step_ms"] / 1e3
    out["heavy_producer"] = {"passes": passes, "producer_alone_ms": 1e3 * heavy_prod,
                             "overlapped_step_ms": 1e3 * ov, "serial_ms": 1e3 * se,
                             "max_ms": 1e3 * max(heavy_prod, roof_link),
                             "sum_ms": 1e3 * (heavy_prod + stream_only),
                             "frac_of_max": max(heavy_prod, roof_link) / ov}
    del grads
    out["next_t"] = t
    return out


def time_options_leg(args, L, dptrs, hp_kw, stream, device, world, t, flush, flush_rd, peak):
    """Device-resident lst_adamw_step_ex, timed like the main leg (CUDA events
    around each launch on the launching stream, L2 flushed before each when the
    state is under twice the L2): per-block step counters t + (block mod 4) and
    grad_sq for every block, so the extended kernel runs with its reduction."""
    import torch
    from optimizer_update_gb300 import lst
    n = L.n_layers
    gsq = torch.zeros(n, dtype=torch.float64, device=device)
    ws = torch.empty(lst.lst_workspace_bytes(), dtype=torch.uint8, device=device)
    opts = lst.step_options(block_steps=[t] * n, grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
    steps_arr = opts._keep[0]
    ptr_arr = lst._ptr_array(dptrs)
    hp = lst.adamw_hparams(step=t, **hp_kw)
    call = lst.lib().lst_adamw_step_ex
    k_steps = max(3, args.steps // 2)

    def launch(tt):
        for i in range(n):
            steps_arr[i] = tt + (i % 4)
        hp.step = tt
        st = call(L.handle, ptr_arr, ctypes.byref(hp), ctypes.byref(opts), stream.cuda_stream)
        if st != lst.LST_OK:
            raise lst.LstError(st, lst.lst_last_error())

    for _ in range(3):
        launch(t)
        t += 1
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(k_steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(k_steps)]
    torch.cuda.synchronize(device)
    barrier(device)
    for k in range(k_steps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
                flush_rd.sum()
        starts[k].record(stream)
        launch(t)
        t += 1
        ends[k].record(stream)
    torch.cuda.synchronize(device)
    per = [starts[k].elapsed_time(ends[k]) / 1e3 for k in range(k_steps)]
    t_max = max_over_ranks(sum(per), device)
    avg = sum(per) / k_steps
    achieved = ALG_BYTES[L.fmt] * L.n_params / avg / 1e9
    finite = bool(torch.isfinite(gsq).all().item()) and bool((gsq > 0).all().item())
    return {"value": sum_over_ranks(L.n_params, device) * k_steps / t_max, "unit": "params/s", "call": "lst_adamw_step_ex",
            "per_block_steps": True, "grad_sq": True, "achieved_gbs": achieved, "frac_of_hbm_peak": achieved / peak,
            "avg_launch_ms": 1e3 * avg, "median_launch_ms": 1e3 * statistics.median(per), "steps": k_steps,
            "grad_sq_all_positive_finite": finite}


def time_sgd_leg(args, L, dptrs, hp_kw, stream, device, world, flush, flush_rd, peak):
    """Device-resident lst_sgd_step (W += -lr*g), timed like the main leg."""
    import torch
    from optimizer_update_gb300 import lst
    ptr_arr = lst._ptr_array(dptrs)
    call = lst.lib().lst_sgd_step
    lr = ctypes.c_float(hp_kw["lr"])
    k_steps = max(3, args.steps // 2)

    def launch():
        st = call(L.handle, ptr_arr, lr, stream.cuda_stream)
        if st != lst.LST_OK:
            raise lst.LstError(st, lst.lst_last_error())

    for _ in range(3):
        launch()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(k_steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(k_steps)]
    torch.cuda.synchronize(device)
    barrier(device)
    for k in range(k_steps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
                flush_rd.sum()
        starts[k].record(stream)
        launch()
        ends[k].record(stream)
    torch.cuda.synchronize(device)
    per = [starts[k].elapsed_time(ends[k]) / 1e3 for k in range(k_steps)]
    t_max = max_over_ranks(sum(per), device)
    avg = sum(per) / k_steps
    achieved = SGD_BYTES[L.fmt] * L.n_params / avg / 1e9
    return {"value": sum_over_ranks(L.n_params, device) * k_steps / t_max, "unit": "params/s", "call": "lst_sgd_step",
            "alg_bytes_per_param": SGD_BYTES[L.fmt], "achieved_gbs": achieved, "frac_of_hbm_peak": achieved / peak,
            "avg_launch_ms": 1e3 * avg, "median_launch_ms": 1e3 * statistics.median(per), "steps": k_steps}


def disk_bandwidth(directory: str, nbytes: int, req: int = 64 << 20):
    """Sequential direct-I/O write (then fsync) and read bandwidth of the file
    system under `directory`, GB/s, over one `nbytes` file in `req` requests
    (the access the block store makes); buffered I/O where O_DIRECT is refused."""
    import mmap
    path = os.path.join(directory, "disk_probe.bin")
    buf = mmap.mmap(-1, req)
    buf.write(bytes(range(256)) * (req // 256))
    direct = getattr(os, "O_DIRECT", 0)
    try:
        fd = os.open(path, os.O_WRONLY | os.O_CREAT | os.O_TRUNC | direct, 0o644)
    except OSError:
        direct = 0
        fd = os.open(path, os.O_WRONLY | os.O_CREAT | os.O_TRUNC, 0o644)
    nbytes -= nbytes % req
    t0 = time.perf_counter()
    for off in range(0, nbytes, req):
        os.pwrite(fd, buf, off)
    os.fsync(fd)
    tw = time.perf_counter() - t0
    os.close(fd)
    fd = os.open(path, os.O_RDONLY | direct)
    t0 = time.perf_counter()
    for off in range(0, nbytes, req):
        os.preadv(fd, [buf], off)
    tr = time.perf_counter() - t0
    os.close(fd)
    os.remove(path)
    return nbytes / tw / 1e9, nbytes / tr / 1e9, bool(direct)


def run_store_leg(args, L, ptrs, buf0, buf1, hp_kw, device, world, rank):
    """lst_store_step over this workload's blocks in files under a fresh
    directory inside --store-dir: the disk's own bandwidth measured first in
    the same place, then one untimed and --store-steps timed store steps (each
    reads every block file, runs the streamed step and commits every block
    through a shadow file). Everything it writes is removed afterwards."""
    import shutil
    import tempfile
    from optimizer_update_gb300 import lst
    state = sum(L.block_bytes(i) for i in range(L.n_layers))
    os.makedirs(args.store_dir, exist_ok=True)
    free = shutil.disk_usage(args.store_dir).free
    probe_bytes = min(4 << 30, max(256 << 20, state))
    if free < 2 * state + probe_bytes + (1 << 30):
        return {"skipped": f"{free} bytes free under the store directory, {2 * state + probe_bytes} needed"}
    top = tempfile.mkdtemp(prefix=f"lst_store_r{rank}_", dir=args.store_dir)
    staging = []
    S = None
    try:
        w_gbs, r_gbs, direct = disk_bandwidth(top, probe_bytes)
        S = lst.lst_store_create(L.handle, os.path.join(top, "blocks"), ptrs, 0)
        staging = [lst.lst_host_alloc(L.max_block_bytes) for _ in range(3)]
        lst.lst_store_step(S, staging, buf0.data_ptr(), buf1.data_ptr(), lst.adamw_hparams(step=1, **hp_kw), 600_000)
        k = max(1, args.store_steps)
        barrier(device)
        t0 = time.perf_counter()
        for t in range(2, 2 + k):
            lst.lst_store_step(S, staging, buf0.data_ptr(), buf1.data_ptr(), lst.adamw_hparams(step=t, **hp_kw), 600_000)
        dt = max_over_ranks(time.perf_counter() - t0, device) / k
    finally:
        if S is not None:
            lst.lst_store_close(S)
        for p in staging:
            lst.lst_host_free(p)
        shutil.rmtree(top, ignore_errors=True)
    serial = state / (w_gbs * 1e9) + state / (r_gbs * 1e9)
    return {"value": sum_over_ranks(L.n_params, device) / dt, "unit": "params/s", "call": "lst_store_step", "step_s": dt,
            "file_read_bytes_per_step": state, "file_write_bytes_per_step": state,
            "disk_write_gbs": w_gbs, "disk_read_gbs": r_gbs, "direct_io": direct,
            "disk_serial_s": serial, "frac_of_disk_serial": serial / dt,
            "frac_of_disk_write": state / (w_gbs * 1e9) / dt, "steps": k, "warmup_steps": 1}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0x5EED)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--ref-sample-bytes", type=int, default=2 << 30,
                    help="state the reference arm's sample holds at most")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the device-resident legs on the other workloads (configs object)")
    ap.add_argument("--shard", action="store_true",
                    help="with N > 1: each rank updates a contiguous range of the model's blocks (strong scaling) "
                         "instead of a replica of the whole model (weak scaling, the default)")
    ap.add_argument("--store-dir", default=None,
                    help="also time lst_store_step with the blocks in files under this directory (writes twice "
                         "the state to disk, removed afterwards)")
    ap.add_argument("--store-steps", type=int, default=2)
    ap.add_argument("--max-blocks", type=int, default=0,
                    help="keep only the first N blocks of the workload (a smaller case)")
    args = ap.parse_args(argv)
    # at least three untimed warm-up steps, whatever is asked; the line reports
    # the number actually run
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
