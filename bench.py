#!/usr/bin/env python
"""Benchmark of fused nested 4-bit dequantization on GB300; prints one JSON line.

A step is one fused dequantization (`dq4_nested`, one kernel launch) of the
28672x8192 NF4-style weight (234,881,024 values; blocksize 64, nested
blocksize 256, FP16 out) with its inputs resident in HBM.  Metric:
dequantized elements/s, with effective HBM GB/s (algorithmic bytes / time)
against the measured GB300 copy bandwidth as the roofline.

Timing (CUDA events on the launching stream; protocol of "Fuse nested scale
reconstruction into SM103 4-bit dequantization", section "B300 evidence
plan": warm-ups, >= 7 timed batches, every batch sample with median / p10 /
p90, unfused sequence timed interleaved as the comparison):
  * W untimed warm-up steps, then exactly K steps between barrier +
    synchronize on both sides; the time is the max over ranks.
  * every step uses the next of 4 rotating buffer sets (2.36 GB in all, each
    larger than L2), so no step finds the previous steps' lines in L2.
  * nvidia-smi samples SM clocks and throttle reasons during the timed region.

Other legs: `e2e` (the same metric with host buffers: one dq4_nested_host call
per step, which copies the step's inputs from pinned host memory and the
output back to pinned host memory chunk by chunk, all timed), `cpu_baseline`
(the CPU oracle on the host cores), and `--impl reference` (the CPU oracle
as the reference arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dq4_inputs as gen  # noqa: E402

METRIC = "dequantized elements/s and effective HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "elements/s"
DEFAULT_CELL = "C4a"
# Every cell of the >= 80 % bar (the >= 4096x11008 weights: C3, C4, and C5 at each block size,
# whose four offsets change arithmetic, not traffic, so each block size is timed at one of
# them) and the smaller C1 / C2 cells, timed one by one for the `cells` record.
DEFAULT_CELLS = (["C1", "C2a", "C2b", "C3a", "C3b", "C3c", "C3d", "C4a", "C4b", "C4c", "C4d"]
                 + [f"C5-bs{bs}-off{off:+g}" for bs, off in
                    zip((32, 64, 128, 256, 512, 1024, 2048, 4096),
                        (-1.0, -1e-3, 1e-3, 1.0, -1.0, -1e-3, 1e-3, 1.0))])
BAR_CELL_PREFIXES = ("C3", "C4", "C5")
# cells also timed through dq4_nested_transposed (W^T out) in the default run, so the
# transposed path's record comes from the same run as the headline
DEFAULT_T_CELLS = ["C1", "C3a", "C3c", "C4a", "C4b", "C5-bs64-off-0.001"]
N_SETS = 4  # rotating buffer sets of the timed region (each larger than L2)
E2E_WINDOWS = 5  # the e2e steps are timed in this many windows (median window reported)
HOLD_CYCLES = 2_000_000  # the pre-region spin: ~1 ms at the 2.07 GHz SM clock
FALLBACK_HBM_GBS = 6800.0
# the sources of the flat dequantization kernels (the ncu traffic record is tied to them)
KERNEL_SRCS = [os.path.join(ROOT, "quantized_weight_dequantization_gb300", "csrc", f)
               for f in ("common.cuh", "flat.cu")]
PROFILES = os.path.join(ROOT, "profiles")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cell", default=DEFAULT_CELL, choices=sorted(gen.CELLS))
    ap.add_argument("--op", choices=["nested", "transposed", "int8prep", "outprod", "linear",
                                     "grad_a", "pair"],
                    default="nested",
                    help="nested: dq4_nested (flat output); transposed: dq4_nested_transposed "
                         "(W^T output of the rows x cols weight); int8prep: LLM.int8 "
                         "correction-operand preparation (--m, --kn, --l)")
    ap.add_argument("--m", type=int, default=2048, help="int8prep: activation rows M")
    ap.add_argument("--kn", type=int, default=14336, help="int8prep: K = N")
    ap.add_argument("--l", type=int, default=64, help="int8prep: outlier columns L")
    ap.add_argument("--int8-grid", action="store_true",
                    help="int8prep: the page's preparation grid, one launch against the eager "
                         "gather/multiply/cast/transpose sequence")
    ap.add_argument("--rows", type=int, default=600000, help="outprod: rows of W (summed over)")
    ap.add_argument("--cols", type=int, default=256, help="outprod: columns of W")
    ap.add_argument("--ncols", type=int, default=256, help="outprod: columns of G")
    ap.add_argument("--transient-mib", type=int, default=256, help="outprod: transient bound")
    ap.add_argument("--grad-m", default="2048,8192",
                    help="grad_a: rows M of dY (tokens) for the grad_A = dY W shapes")
    ap.add_argument("--lin-m", default="16,128,512,2048,4096",
                    help="linear: comma-separated M values (activation rows)")
    ap.add_argument("--lin-n", type=int, default=11008, help="linear: N (weight rows)")
    ap.add_argument("--lin-k", type=int, default=4096, help="linear: K")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--compare-batches", type=int, default=7)
    ap.add_argument("--sets", type=int, default=N_SETS,
                    help="rotating device buffer sets (each larger than L2)")
    ap.add_argument("--isolated-launches", type=int, default=100,
                    help="launches timed one by one (own event pair) after the timed region")
    ap.add_argument("--cells", default=",".join(DEFAULT_CELLS),
                    help="cells timed one by one into the `cells` record (empty: none)")
    ap.add_argument("--t-cells", default=",".join(DEFAULT_T_CELLS),
                    help="cells timed through the transposed entry point into the "
                         "`transposed_cells` record (--op nested only; empty: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-compare", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-hold", action="store_true",
                    help="open the timed region on an idle device (no pre-region spin)")
    return ap.parse_args()


# ------------------------------------------------------------ utilities
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Ranks:
    """The ranks of a run: one process per GPU under torchrun, each a replica of the
    workload (no data-path collective).  The only cross-rank traffic is the barrier that
    brackets the timed region and the max of the ranks' times.  `backend` is "nccl" on
    the GPUs; the multi-rank CPU tests run the same code over "gloo"."""

    def __init__(self, backend: str = "nccl", device=None):
        self.rank, self.world, self.local = dist_env()
        self.device = device
        self._dist = None
        if self.world > 1:
            import torch.distributed as dist
            kw = {"device_id": device} if backend == "nccl" else {}
            dist.init_process_group(backend, **kw)
            self._dist = dist

    def barrier(self):
        if self._dist is not None:
            self._dist.barrier()

    def max_over_ranks(self, x: float) -> float:
        if self._dist is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self._dist.all_reduce(t, op=self._dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self._dist is not None:
            self._dist.destroy_process_group()
            self._dist = None


def whole_job_rate(world: int, units_per_rank: float, elapsed_ms: float) -> float:
    """Units all ranks processed per second of the slowest rank's time (weak scaling:
    every rank processes the same units)."""
    return world * units_per_rank / (elapsed_ms / 1e3)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_sha256() -> str:
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_record(cell: str):
    """ncu DRAM bytes per launch from a committed summary, if it matches this source."""
    sha = source_sha256()
    if not os.path.isdir(PROFILES):
        return None
    for fn in sorted(os.listdir(PROFILES)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(PROFILES, fn)) as f:
            for line in f:
                m = re.match(r"\s*traffic_record:\s*(\{.*\})\s*$", line)
                if not m:
                    continue
                rec = json.loads(m.group(1))
                if rec.get("cell") == cell and rec.get("src_sha256") == sha:
                    return rec
    return None


def pct(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None
        self.error = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError as e:
            self.error = str(e)
        time.sleep(0.5)

    def stop(self):
        if self.proc is None:
            return {"error": self.error or "nvidia-smi not started"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.tmp.name)
        if not rows:
            return {"error": "no nvidia-smi samples"}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if re.match(r"^\s*[\d.]+\s*$", r[3])]
        reasons = sorted({name for r in rows for name, v in zip(self.REASONS, r[5:9])
                          if v.strip().lower() == "active"})
        # samples under load: power above the midpoint of the observed range
        if power and len(power) == len(sm):
            thr = (min(power) + max(power)) / 2
            loaded = [s for s, p in zip(sm, power) if p >= thr] or sm
        else:
            loaded = sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(power) if power else None}


def cell_config(cell, op: str, world: int, n_sets: int) -> dict:
    """The workload description both arms print (same dict, so the two lines compare)."""
    transposed = op == "transposed"
    alg_bytes = cell.algorithmic_bytes()
    return {
        "workload": f"{cell.rows}x{cell.cols} {cell.fmt.upper()}-style nested 4-bit dequant, "
                    f"blocksize {cell.blocksize}, nested blocksize {cell.nested_blocksize}, "
                    f"{cell.out.upper()} out ({cell.name})"
                    + (", transposed output" if transposed else ""),
        "op": op,
        "n_values": cell.n, "blocksize": cell.blocksize,
        "nested_blocksize": cell.nested_blocksize, "format": cell.fmt,
        "out_dtype": cell.out, "offset": cell.offset,
        "algorithmic_bytes_per_step": alg_bytes,
        "l2": f"inputs larger than L2: {alg_bytes / 1e6:.1f} MB per step, {n_sets} rotating "
              "buffer sets",
        "parallelism": f"replicas x{world}",
    }


# -------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    import quantized_weight_dequantization_gb300 as dq

    _, _, local = dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    ranks = Ranks("nccl", dev)
    rank, world = ranks.rank, ranks.world
    barrier, max_over_ranks = ranks.barrier, ranks.max_over_ranks

    cell = gen.CELLS[args.cell]
    p = cell.problem()
    out_dtype = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[cell.out]
    n = p.n
    alg_bytes = cell.algorithmic_bytes()
    host = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k)))
            for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook",
                      "value_codebook")}
    scb = host["scale_codebook"].to(dev)
    vcb = host["value_codebook"].to(dev)
    n_sets = max(1, args.sets)
    sets = []
    for _ in range(n_sets):
        sets.append(dict(packed=host["packed"].to(dev), codes=host["scale_codes"].to(dev),
                         absmax=host["nested_absmax"].to(dev),
                         out=torch.empty(n, dtype=out_dtype, device=dev),
                         scratch=torch.empty(p.nblocks, dtype=torch.float32, device=dev)))
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    L = dq.lib
    code = {torch.float16: dq.OUT_F16, torch.bfloat16: dq.OUT_BF16,
            torch.float32: dq.OUT_F32}[out_dtype]
    ptrs = [(s["packed"].data_ptr(), s["codes"].data_ptr(), s["absmax"].data_ptr(),
             s["out"].data_ptr(), s["scratch"].data_ptr()) for s in sets]
    off = float(p.offset)
    bs, nbs = p.blocksize, p.nested_blocksize
    scb_p, vcb_p = scb.data_ptr(), vcb.data_ptr()

    transposed = args.op == "transposed"
    rows, cols = cell.rows, cell.cols

    def fused(i):
        pk, cd, am, o, _ = ptrs[i % n_sets]
        if not transposed:
            return L.dq4_nested(pk, cd, am, scb_p, vcb_p, off, n, bs, nbs, code, o, sh)
        return L.dq4_nested_transposed(pk, cd, am, scb_p, vcb_p, off, rows, cols, bs, nbs, code,
                                       o, sh)

    def unfused(i):
        pk, cd, am, o, sc = ptrs[i % n_sets]
        return L.dq4_nested_unfused(pk, cd, am, scb_p, vcb_p, off, n, bs, nbs, code, o, sc, sh)

    # correctness gate before timing: first and last 64 Ki values of the fused
    # output vs the unfused sequence (bit-identical by construction); for the
    # transposed op, its first 64 rows vs the flat output's first 64 columns
    if transposed:
        ref = torch.empty_like(sets[0]["out"])
        pk, cd, am, _, _ = ptrs[0]
        assert fused(0) == 0
        assert L.dq4_nested(pk, cd, am, scb_p, vcb_p, off, n, bs, nbs, code, ref.data_ptr(),
                            sh) == 0
        torch.cuda.synchronize(dev)
        iv = torch.int32 if ref.element_size() == 4 else torch.int16
        t_rows = sets[0]["out"].view(cols, rows)[:64].view(iv)
        f_cols = ref.view(rows, cols)[:, :64].t().contiguous().view(iv)
        if not torch.equal(t_rows, f_cols):
            raise SystemExit("transposed and flat outputs differ; refusing to time")
        del ref, t_rows, f_cols
    assert fused(0) == 0
    torch.cuda.synchronize(dev)
    a = sets[0]["out"].clone()
    assert (unfused(0) if not transposed else fused(0)) == 0
    torch.cuda.synchronize(dev)
    b = sets[0]["out"]
    if not (torch.equal(a[:65536].view(torch.int16 if a.element_size() == 2 else torch.int32),
                        b[:65536].view(torch.int16 if b.element_size() == 2 else torch.int32))
            and torch.equal(a[-65536:].view(torch.int16 if a.element_size() == 2 else torch.int32),
                            b[-65536:].view(torch.int16 if b.element_size() == 2
                                            else torch.int32))):
        raise SystemExit("fused and unfused outputs differ; refusing to time")

    # ---- warm-up, then exactly K timed steps.  The clock sampler starts first (it takes
    # half a second to come up), so the warm-up launches run right before the timed region
    # and the GPU does not idle in between.
    K, W = args.steps, args.warmup
    gpu_uuid = None
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    clocks = None if args.no_clocks else ClockSampler(gpu_uuid)
    if clocks:
        clocks.start()
    for i in range(W):
        if fused(i):
            raise SystemExit("dq4_nested failed in warm-up")
    # batch boundaries (>= 7 batches); the launches run back to back
    nb = max(1, min(K, max(7, min(20, K // 50))))
    edges = sorted(set(np.linspace(0, K, nb + 1).astype(int).tolist()))
    ev_b = {e: torch.cuda.Event(enable_timing=True) for e in edges}
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    # The device is held in torch's fixed-length spin kernel (~1 ms, before the start
    # event, so untimed) while the host queues the start event and the first launches:
    # the timed region then opens on a queue of launches, as with a blocking kernel in
    # nvbench, instead of on the host's latency to its first call.
    hold_cycles = 0 if args.no_hold else HOLD_CYCLES
    if hold_cycles:
        torch.cuda._sleep(hold_cycles)
    wall0 = time.perf_counter()
    bad = 0
    for i in range(K):
        if i in ev_b:
            ev_b[i].record(stream)
        bad |= fused(W + i)
    ev_b[K].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if clocks else {"error": "not sampled (--no-clocks)"}
    if bad:
        raise SystemExit(f"dq4_nested returned status {bad} in the timed region")
    elapsed_ms = max_over_ranks(ev_b[0].elapsed_time(ev_b[K]))
    # The timed region launches this one kernel and nothing else (one launch per
    # step; the ncu launch list of this command shows a 100 % share), so its
    # average launch duration is the region's time over K.
    share = 1.0
    avg_launch_ms = elapsed_ms * share / K
    batch_ms = [ev_b[a].elapsed_time(ev_b[b]) / (b - a) for a, b in zip(edges[:-1], edges[1:])]

    # launches timed one by one (each between its own events, so no overlap with
    # a neighbour): not part of the timed region
    iso_ms = []
    for i in range(max(0, args.isolated_launches)):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fused(i)
        e1.record(stream)
        iso_ms.append((e0, e1))
    torch.cuda.synchronize(dev)
    iso_ms = [a.elapsed_time(b) for a, b in iso_ms]

    # ---- interleaved fused / unfused comparison (not part of the timed region)
    cmp_f, cmp_u = [], []
    per = 200
    for j in range(0 if (args.no_compare or transposed) else args.compare_batches):
        for fn, acc in ((fused, cmp_f), (unfused, cmp_u)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(per):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            acc.append(e0.elapsed_time(e1) / per * 1e3)

    # ---- end to end with host buffers (pinned H2D of the inputs, call, D2H of the output)
    pin = {k: v.pin_memory() for k, v in host.items()} if not args.no_e2e else dict(host)
    host_out = torch.empty(n if not args.no_e2e else 0, dtype=out_dtype)
    if not args.no_e2e:
        host_out = host_out.pin_memory()
    s0 = sets[0]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = host_out.numel() * host_out.element_size()
    E = max(3, args.e2e_steps)

    def e2e_step():
        if not transposed:
            # the host-to-host API: inputs from pinned host memory, output to pinned host
            # memory, chunks pipelined through device scratch (copies inside the call)
            dq.dq4_nested_host(pin["packed"], pin["scale_codes"], pin["nested_absmax"],
                               pin["scale_codebook"], pin["value_codebook"], off, n, bs, nbs,
                               out=host_out, device=dev, stream=stream)
            return
        s0["packed"].copy_(pin["packed"], non_blocking=True)
        s0["codes"].copy_(pin["scale_codes"], non_blocking=True)
        s0["absmax"].copy_(pin["nested_absmax"], non_blocking=True)
        scb.copy_(pin["scale_codebook"], non_blocking=True)
        vcb.copy_(pin["value_codebook"], non_blocking=True)
        if transposed:
            dq.dq4_nested_transposed(s0["packed"], s0["codes"], s0["absmax"], scb, vcb, off,
                                     rows, cols, bs, nbs, out_dtype, out=s0["out"],
                                     stream=stream)
        else:
            dq.dq4_nested(s0["packed"], s0["codes"], s0["absmax"], scb, vcb, off, n, bs, nbs,
                          out_dtype, out=s0["out"], stream=stream)
        host_out.copy_(s0["out"], non_blocking=True)

    e2e_ms = None
    e2e_windows = []
    if not args.no_e2e:
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        # the E steps in E2E_WINDOWS windows of back-to-back steps, events between windows;
        # the step time is the median window's (one window slowed by the host, e.g. page
        # locking or another tenant, cannot decide the record), and every window is kept
        nwin = min(E2E_WINDOWS, E)
        per_win = [E // nwin + (1 if w < E % nwin else 0) for w in range(nwin)]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nwin + 1)]
        ev[0].record(stream)
        for w in range(nwin):
            for _ in range(per_win[w]):
                e2e_step()
            ev[w + 1].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_windows = [max_over_ranks(ev[w].elapsed_time(ev[w + 1])) / per_win[w]
                       for w in range(nwin)]
        e2e_ms = pct(e2e_windows, 50) * E  # E steps at the median window's step time
        # the copied-back output must equal the device result
        if not torch.equal(host_out.view(torch.uint8), s0["out"].cpu().view(torch.uint8)):
            raise SystemExit("e2e output mismatch")

    peak, peak_kind = read_peaks()
    # the host link alone for the e2e step's bytes, and every listed cell timed on its own
    link = link_bound(h2d, d2h, dev) if e2e_ms is not None else None
    names = [c for c in args.cells.split(",") if c]
    cells_rec = time_cells(names, dev, stream, transposed, peak) if names else None
    t_names = [c for c in args.t_cells.split(",") if c] if not transposed else []
    t_cells_rec = time_cells(t_names, dev, stream, True, peak) if t_names else None
    ms_per_step = elapsed_ms / K
    value = whole_job_rate(world, K * n, elapsed_ms)
    achieved_gbs = alg_bytes / (avg_launch_ms / 1e3) / 1e9
    rec = traffic_record(args.cell)
    out = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cell.out,
        "data": "synthetic (seeded splitmix64 codes, lognormal nested absmax)",
        "config": cell_config(cell, args.op, world, n_sets),
        "effective_gbs": alg_bytes / (ms_per_step / 1e3) / 1e9,
        "roofline": {
            "bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
            "frac": achieved_gbs / peak,
            "traffic": rec["bytes_per_launch"] if rec else None,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "frac_of_nominal_8tbs": achieved_gbs / 8000.0,
            "kernel": (f"dq4_transposed_kernel<{cell.out}>" if transposed
                       else f"dq4_vec_kernel<{cell.out},nested>"),
            "avg_launch_us": avg_launch_ms * 1e3,
            "share_of_timed_region": share,
            "isolated_launch_us": {"median": pct(iso_ms, 50) * 1e3, "p10": pct(iso_ms, 10) * 1e3,
                                   "p90": pct(iso_ms, 90) * 1e3, "count": len(iso_ms)}
            if iso_ms else None,
        },
        "batches_us_per_step": [round(x * 1e3, 3) for x in batch_ms],
        "batch_stats_us": {"median": pct(batch_ms, 50) * 1e3, "p10": pct(batch_ms, 10) * 1e3,
                           "p90": pct(batch_ms, 90) * 1e3},
        "fused_vs_unfused": None if not cmp_f else {
            "fused_us": {"median": pct(cmp_f, 50), "p10": pct(cmp_f, 10), "p90": pct(cmp_f, 90),
                         "samples": [round(x, 3) for x in cmp_f]},
            "unfused_us": {"median": pct(cmp_u, 50), "p10": pct(cmp_u, 10),
                           "p90": pct(cmp_u, 90), "samples": [round(x, 3) for x in cmp_u]},
            "speedup": pct(cmp_u, 50) / pct(cmp_f, 50),
            "launches": {"fused": 1, "unfused": 3},
        },
        "e2e": None if e2e_ms is None else {
            "value": whole_job_rate(world, E * n, e2e_ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
            "ms_per_step": e2e_ms / E,
            "windows_ms_per_step": [round(x, 4) for x in e2e_windows],
            # the roofline of this leg is the host link: the step's copies alone, both
            # directions at once, against the whole step
            "link_gbs": link, "link_bound_ms": link["both_directions_ms"],
            "frac": link["both_directions_ms"] / (e2e_ms / E)},
        "cells": cells_rec,
        "transposed_cells": t_cells_rec,
        "gpu_launches": K,
        "timed_region_start": (f"launch queue filled behind a {hold_cycles}-cycle spin kernel "
                               f"(untimed)" if hold_cycles else "idle device"),
        "clocks": clk,
        "wall_s_timed": wall,
        "gpu": torch.cuda.get_device_name(dev),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(p, cell, transposed)
    ranks.close()
    if rank == 0:
        print(json.dumps(out), flush=True)


def time_cells(names, dev, stream, transposed: bool, peak: float, batches: int = 7):
    """Each named cell timed as back-to-back launches on `stream` over >= 4 rotating buffer sets
    (together more than twice the L2, so no launch finds its inputs there): >= 20 warm-up
    launches, then one batch of >= 2 ms of launches captured in a CUDA graph and replayed
    `batches` times, so that the record is the device's time per call and not the gaps
    between Python launches (which exceed the kernel at the 42 MB cells); per call the
    median, p10 and p90 over the replays, the effective GB/s and its fraction of `peak`."""
    import torch

    import quantized_weight_dequantization_gb300 as dq

    L = dq.lib
    stream = torch.cuda.Stream(dev)  # graphs are captured on a stream of their own
    sh = stream.cuda_stream
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    codes = {"f16": dq.OUT_F16, "bf16": dq.OUT_BF16, "f32": dq.OUT_F32}
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    rec = {}
    for name in names:
        cell = gen.CELLS[name]
        p = cell.problem()
        alg = cell.algorithmic_bytes()
        n_sets = max(4, -(-2 * l2 // alg) + 1)
        first = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
                 for k in ("packed", "scale_codes", "nested_absmax")}
        scb = torch.from_numpy(p.scale_codebook).to(dev)
        vcb = torch.from_numpy(p.value_codebook).to(dev)
        sets = [{k: (v if i == 0 else v.clone()) for k, v in first.items()}
                for i in range(n_sets)]
        for s in sets:
            s["out"] = torch.empty(p.n, dtype=tdt[cell.out], device=dev)
        ptrs = [(s["packed"].data_ptr(), s["scale_codes"].data_ptr(),
                 s["nested_absmax"].data_ptr(), s["out"].data_ptr()) for s in sets]
        off, bs, nbs, code = float(p.offset), p.blocksize, p.nested_blocksize, codes[cell.out]

        def call(i):
            pk, cd, am, o = ptrs[i % n_sets]
            if transposed:
                return L.dq4_nested_transposed(pk, cd, am, scb.data_ptr(), vcb.data_ptr(), off,
                                               cell.rows, cell.cols, bs, nbs, code, o, sh)
            return L.dq4_nested(pk, cd, am, scb.data_ptr(), vcb.data_ptr(), off, p.n, bs, nbs,
                                code, o, sh)

        est_us = alg / (peak * 1e3)
        iters = max(20, int(2000.0 / est_us) + 1)
        for i in range(max(20, n_sets)):
            if call(i):
                raise SystemExit(f"{name}: launch failed")
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for j in range(iters):
                if call(j):
                    raise SystemExit(f"{name}: launch failed during capture")
        graph.replay()  # one untimed replay
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(batches + 1)]
        with torch.cuda.stream(stream):
            for b in range(batches):
                ev[b].record(stream)
                graph.replay()
            ev[batches].record(stream)
        torch.cuda.synchronize(dev)
        del graph
        us = [ev[b].elapsed_time(ev[b + 1]) / iters * 1e3 for b in range(batches)]
        med = pct(us, 50)
        gbs = alg / (med * 1e-6) / 1e9
        rec[name] = {"us": round(med, 3), "p10_us": round(pct(us, 10), 3),
                     "p90_us": round(pct(us, 90), 3), "gbs": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "in_bar": name.startswith(BAR_CELL_PREFIXES),
                     "algorithmic_bytes": alg, "sets": n_sets, "calls_per_batch": iters,
                     "batches": batches}
        del sets, first
    bar = [v["frac"] for v in rec.values() if v["in_bar"]]
    return {"cells": rec, "bar_min_frac": min(bar) if bar else None,
            "protocol": f"per cell: >= 4 rotating buffer sets (> 2x L2 in all), >= 20 warm-up "
                        f"launches, >= 2 ms of back-to-back launches captured in one CUDA "
                        f"graph and replayed {batches} times, median / p10 / p90 per call "
                        f"over the replays"}


def link_bound(h2d_bytes: int, d2h_bytes: int, dev, reps: int = 7):
    """The host link alone for one e2e step's byte counts: one pinned H2D and one pinned
    D2H cudaMemcpyAsync timed apart (GB/s) and at once on two streams (ms, the e2e step's
    floor: its pipeline overlaps the two directions).  Each is the fastest of `reps`
    repetitions after one untimed: a floor, which a slowed repetition must not raise."""
    import torch

    hin = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dout = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    hout = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(h2d: bool, d2h: bool) -> float:
        ts = []
        for _ in range(reps + 1):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if h2d:
                with torch.cuda.stream(s1):
                    din.copy_(hin, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    hout.copy_(dout, non_blocking=True)
            torch.cuda.synchronize(dev)
            ts.append(time.perf_counter() - t0)
        return min(ts[1:]) * 1e3

    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_gbs": round(h2d_bytes / (t_in * 1e-3) / 1e9, 1),
            "d2h_gbs": round(d2h_bytes / (t_out * 1e-3) / 1e9, 1),
            "both_directions_ms": round(t_both, 4)}


def run_pair(args):
    """One fused call and one unfused sequence per step, untimed, for a profiler's launch
    list: `--warmup` pairs, then `--steps` pairs (1 + 3 launches each)."""
    import torch

    import quantized_weight_dequantization_gb300 as dq

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cell = gen.CELLS[args.cell]
    p = cell.problem()
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[cell.out]
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    out = torch.empty(p.n, dtype=tdt, device=dev)
    scratch = torch.empty(p.nblocks, dtype=torch.float32, device=dev)
    args_ = (t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
             t["value_codebook"], float(p.offset), p.n, p.blocksize, p.nested_blocksize, tdt)
    for _ in range(args.warmup + args.steps):
        dq.dq4_nested(*args_, out=out)
        dq.dq4_nested_unfused(*args_, out=out, scale_scratch=scratch)
    torch.cuda.synchronize(dev)
    print(json.dumps({"op": "pair", "cell": cell.name, "pairs": args.warmup + args.steps,
                      "launches_per_pair": {"fused": 1, "unfused": 3},
                      "scale_scratch_bytes": p.nblocks * 4}), flush=True)


# --------------------------------------------------------- CPU baseline
def cpu_baseline(p, cell, transposed: bool = False, repeats: int = 3):
    """The CPU oracle, as it stands, over the whole workload on all host cores."""
    import oracle

    threads = os.cpu_count() or 1
    oracle.dq4_nested(gen.make_problem(1 << 16, 64, 256), "f16")  # build + load
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        if transposed:
            oracle.dq4_nested_transposed(p, cell.rows, cell.cols, cell.out, threads=threads)
        else:
            oracle.dq4_nested(p, cell.out, threads=threads)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    out = {"value": p.n / t, "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": f"the whole {cell.name} workload ({p.n} values), median of {repeats} runs, "
                     f"{threads} threads over nested-group-aligned chunks",
           "gbs": cell.algorithmic_bytes() / t / 1e9}
    if not transposed:
        # one thread, on a prefix of whole nested groups (bounded: 2^24 values)
        unit = p.blocksize * p.nested_blocksize
        n1 = max(unit, min(p.n, 1 << 24) // unit * unit) if p.n >= unit else p.n
        p1 = gen.Problem(p.packed[:(n1 + 1) // 2], p.scale_codes[:-(-n1 // p.blocksize)],
                         p.nested_absmax[:-(-n1 // unit)], p.scale_codebook, p.value_codebook,
                         p.offset, n1, p.blocksize, p.nested_blocksize)
        t1 = []
        for _ in range(repeats):
            t0 = time.perf_counter()
            oracle.dq4_nested(p1, cell.out, threads=1)
            t1.append(time.perf_counter() - t0)
        out["single_thread"] = {"value": n1 / statistics.median(t1), "unit": UNIT,
                                "sample": f"the first {n1} values of {cell.name}, median of "
                                          f"{repeats} runs, one thread"}
    try:
        info = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        model = next((ln.split(":", 1)[1].strip() for ln in info.splitlines()
                      if ln.startswith("Model name")), None)
    except (OSError, subprocess.SubprocessError):
        model = None
    out["cpu_model"] = model
    return out


# ------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: K steps, each a bounded sample of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    cell = gen.CELLS[args.cell]
    p = cell.problem()
    threads = os.cpu_count() or 1
    unit = p.blocksize * p.nested_blocksize
    # calibrate: rate on one nested-group-aligned slice
    probe = min(p.n, 1 << 22)

    def sub(lo, hi):
        return gen.Problem(p.packed[lo // 2:(hi + 1) // 2],
                           p.scale_codes[lo // p.blocksize:-(-hi // p.blocksize)],
                           p.nested_absmax[lo // unit:-(-hi // unit)], p.scale_codebook,
                           p.value_codebook, p.offset, hi - lo, p.blocksize, p.nested_blocksize)

    oracle.dq4_nested(sub(0, probe), cell.out, threads=threads)
    t0 = time.perf_counter()
    oracle.dq4_nested(sub(0, probe), cell.out, threads=threads)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    budget_s = 60.0
    K, W = args.steps, args.warmup
    sample = int(min(p.n, max(unit, budget_s * rate / max(K + W, 1))))
    sample = max(unit, (sample // unit) * unit)
    nsub = max(1, p.n // sample)
    for i in range(W):
        lo = (i % nsub) * sample
        oracle.dq4_nested(sub(lo, min(p.n, lo + sample)), cell.out, threads=threads)
    done = 0
    t0 = time.perf_counter()
    for i in range(K):
        lo = (i % nsub) * sample
        hi = min(p.n, lo + sample)
        oracle.dq4_nested(sub(lo, hi), cell.out, threads=threads)
        done += hi - lo
    el = time.perf_counter() - t0
    value = done / el
    desc = (f"{sample} consecutive values of {cell.name} per step (of {p.n}), "
            f"{threads} threads over nested-group-aligned chunks")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cell.out,
        "data": "synthetic (seeded splitmix64 codes, lognormal nested absmax)",
        "config": cell_config(cell, args.op, world, max(1, args.sets)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_int8_grid(args):
    """dq4_int8_correction_prep against the eager torch sequence it replaces, over the
    preparation grid of "Fuse LLM.int8 correction operand preparation into one CUDA kernel"
    (section "B300 benchmark plan": M in {1, 8, 64, 512, 2048}, K = N in {3584, 4096, 8192,
    14336}, L in {1, 5, 16, 64}).  Eager: gather A's columns; gather CB's columns, FP32
    multiply by SCB, FP32 multiply by RN32(1/127), FP16, transpose (section "Exact
    correctness oracle" fixes that order).  Both produce the same bits, checked per cell.
    Inputs are drawn on the device from a seeded generator (CB is up to 205 MB per cell).
    Times: CUDA events around `reps` back-to-back calls, interleaved over `samples` rounds,
    median per cell, twice: called from Python (host dispatch included: five torch ops
    against one ctypes call) and replayed from a CUDA graph (device time alone)."""
    import torch

    import quantized_weight_dequantization_gb300 as dq

    dev = torch.device("cuda:0")
    L_ = dq.get_lib()
    r127 = torch.tensor(1.0 / 127.0, dtype=torch.float32, device=dev)
    g = torch.Generator(device=dev)
    samples, reps = 30, 10
    cells = []
    for KN in (3584, 4096, 8192, 14336):
        g.manual_seed(KN)
        CB = torch.randint(-127, 128, (KN, KN), dtype=torch.int8, device=dev, generator=g)
        SCB = torch.rand(KN, dtype=torch.float32, device=dev, generator=g) * 8.0
        for M in (1, 8, 64, 512, 2048):
            A = torch.randn(M, KN, dtype=torch.float16, device=dev, generator=g)
            for L in (1, 5, 16, 64):
                cols = torch.sort(torch.randperm(KN, device=dev, generator=g)[:L]).values
                subA = torch.empty((M, L), dtype=torch.float16, device=dev)
                subB = torch.empty((L, KN), dtype=torch.float16, device=dev)

                def ours():
                    return L_.dq4_int8_correction_prep(
                        A.data_ptr(), CB.data_ptr(), SCB.data_ptr(), cols.data_ptr(), M, KN, KN,
                        L, subA.data_ptr(), subB.data_ptr(), None,
                        torch.cuda.current_stream(dev).cuda_stream)

                def eager():
                    ea = A.index_select(1, cols)
                    eb = ((CB.index_select(1, cols).float() * SCB.view(-1, 1)) * r127)
                    return ea, eb.half().t().contiguous()

                if ours() != 0:
                    raise SystemExit(f"status error at M={M} K=N={KN} L={L}")
                ea, eb = eager()
                torch.cuda.synchronize(dev)
                if not (torch.equal(ea.view(torch.int16), subA.view(torch.int16)) and
                        torch.equal(eb.view(torch.int16), subB.view(torch.int16))):
                    raise SystemExit(f"eager and fused differ at M={M} K=N={KN} L={L}")
                for _ in range(max(3, args.warmup)):
                    ours()
                    eager()
                t_o, t_e = [], []
                for _ in range(samples):
                    for fn, acc in ((ours, t_o), (eager, t_e)):
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        for _ in range(reps):
                            fn()
                        e1.record()
                        torch.cuda.synchronize(dev)
                        acc.append(e0.elapsed_time(e1) / reps * 1e3)
                # device time alone: each arm's `reps` calls captured in a CUDA graph
                graphs = []
                for fn in (ours, eager):
                    s_ = torch.cuda.Stream(dev)
                    s_.wait_stream(torch.cuda.current_stream(dev))
                    with torch.cuda.stream(s_):
                        fn()
                    torch.cuda.current_stream(dev).wait_stream(s_)
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr):
                        for _ in range(reps):
                            fn()
                    graphs.append(gr)
                d_o, d_e = [], []
                for _ in range(samples):
                    for gr, acc in zip(graphs, (d_o, d_e)):
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        gr.replay()
                        e1.record()
                        torch.cuda.synchronize(dev)
                        acc.append(e0.elapsed_time(e1) / reps * 1e3)
                del graphs
                cells.append({"M": M, "KN": KN, "L": L,
                              "fused_us": pct(t_o, 50), "eager_us": pct(t_e, 50),
                              "speedup": pct(t_e, 50) / pct(t_o, 50),
                              "fused_device_us": pct(d_o, 50), "eager_device_us": pct(d_e, 50),
                              "speedup_device": pct(d_e, 50) / pct(d_o, 50)})
            del A
        del CB, SCB
    sp = [c["speedup"] for c in cells]
    spd = [c["speedup_device"] for c in cells]
    print(json.dumps({
        "metric": "LLM.int8 correction-operand preparation: eager torch time / fused time",
        "value": pct(spd, 50), "unit": "x (median over cells, device time)",
        "higher_is_better": True,
        "n_gpus": 1, "dtype": "f32", "data": "synthetic (seeded device generator)",
        "config": {"workload": "int8 correction prep grid M {1,8,64,512,2048} x K=N "
                               "{3584,4096,8192,14336} x L {1,5,16,64}",
                   "timing": f"CUDA events, {samples} interleaved samples of {reps} calls, "
                             "median per cell; inputs resident; device time from CUDA-graph "
                             "replay, host-driven time from Python calls"},
        "speedup_device_min": min(spd), "speedup_device_median": pct(spd, 50),
        "speedup_device_max": max(spd),
        "speedup_host_min": min(sp), "speedup_host_median": pct(sp, 50),
        "speedup_host_max": max(sp),
        "cells": cells,
    }), flush=True)


def run_int8prep(args):
    """Time dq4_int8_correction_prep on one (M, K = N, L) cell of the preparation grid."""
    if args.int8_grid:
        return run_int8_grid(args)
    import torch

    import quantized_weight_dequantization_gb300 as dq

    dev = torch.device("cuda:0")
    M, KN, L = args.m, args.kn, args.l
    sets = []
    for k in range(3):  # the gathered CB sectors (N * L * 32 B) would otherwise stay in L2
        p = gen.make_int8_problem(M, KN, KN, L, seed=100 + k)
        sets.append(dict(p=p, A=torch.from_numpy(p.A_bits).to(dev).view(torch.float16),
                         CB=torch.from_numpy(p.CB).to(dev), SCB=torch.from_numpy(p.SCB).to(dev),
                         cols=torch.from_numpy(p.cols).to(dev),
                         subA=torch.empty((M, L), dtype=torch.float16, device=dev),
                         subB=torch.empty((L, KN), dtype=torch.float16, device=dev)))
    L_ = dq.get_lib()
    sh = torch.cuda.current_stream(dev).cuda_stream

    def call(i):
        t = sets[i % 3]
        return L_.dq4_int8_correction_prep(t["A"].data_ptr(), t["CB"].data_ptr(),
                                           t["SCB"].data_ptr(), t["cols"].data_ptr(), M, KN, KN,
                                           L, t["subA"].data_ptr(), t["subB"].data_ptr(), None, sh)

    # correctness gate
    import oracle
    assert call(0) == 0
    torch.cuda.synchronize(dev)
    p0 = sets[0]["p"]
    wa, wb = oracle.int8_correction_prep(p0.A_bits, p0.CB, p0.SCB, p0.cols)
    ga = sets[0]["subA"].cpu().view(torch.int16).numpy().view(np.uint16)
    gb = sets[0]["subB"].cpu().view(torch.int16).numpy().view(np.uint16)
    if not (np.array_equal(ga, wa) and np.array_equal(gb, wb)):
        raise SystemExit("int8 preparation differs from the oracle; refusing to time")
    for i in range(args.warmup):
        call(i)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record()
    bad = 0
    for i in range(args.steps):
        bad |= call(i)
    e1.record()
    torch.cuda.synchronize(dev)
    if bad:
        raise SystemExit(f"status {bad}")
    us = e0.elapsed_time(e1) / args.steps * 1e3
    outs = M * L + L * KN
    alg = M * L * 2 * 2 + KN * L * 1 + KN * 4 + L * 8 + L * KN * 2
    sector = M * L * 32 + M * L * 2 + KN * L * 32 + KN * 4 + L * 8 + L * KN * 2
    t0 = time.perf_counter()
    for _ in range(3):
        oracle.int8_correction_prep(p0.A_bits, p0.CB, p0.SCB, p0.cols)
    cpu_s = (time.perf_counter() - t0) / 3
    print(json.dumps({
        "metric": "LLM.int8 correction-operand preparation (subA + subB outputs/s)",
        "value": outs / (us / 1e6), "unit": "outputs/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "us_per_call": us,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"int8 correction prep M={M} K=N={KN} L={L}", "M": M, "K": KN,
                   "N": KN, "L": L, "l2": "3 rotating input sets"},
        "algorithmic_gbs": alg / (us / 1e6) / 1e9,
        "sector_gbs": sector / (us / 1e6) / 1e9,
        "gpu_launches": args.steps,
        "cpu_baseline": {"value": outs / cpu_s, "unit": "outputs/s", "cores": 1,
                         "kind": "oracle", "sample": "the same cell, median of 3"},
    }), flush=True)


def run_outprod(args):
    """Time dq4_nested_out_prod (W decoded in row blocks inside a tcgen05 GEMM with FP32
    accuracy) against the page's unfused sequence (row blocks dequantized into a bounded FP32
    transient, each accumulated by a cuBLAS FP32 GEMM) and against dequantizing all of W."""
    import torch

    import quantized_weight_dequantization_gb300 as dq

    torch.backends.cuda.matmul.allow_tf32 = False  # the comparison GEMMs in true FP32
    dev = torch.device("cuda:0")
    rows, cols, ncols = args.rows, args.cols, args.ncols
    p = gen.make_problem(rows * cols, 64, 256, "nf4", 0.5, 0.0371, seed=7)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    G = torch.from_numpy(gen.make_normal_g(rows, ncols, seed=8)).to(dev)
    dst = torch.empty((cols, ncols), dtype=torch.float32, device=dev)
    args_w = (t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
              t["value_codebook"], float(p.offset))

    def fused():
        dq.out_prod(*args_w, rows, cols, G, dst=dst)

    # the page's sequence: row blocks of at most --transient-mib MiB of FP32, each block
    # starting on a nested-group boundary (16384 values), beta 0 for the first GEMM, 1 after
    unit = 64 * 256
    rb = max(1, min(rows, (args.transient_mib << 20) // (4 * cols)))
    align = unit // int(np.gcd(cols, unit))
    if rb >= align:
        rb -= rb % align
    transient = torch.empty(rb * cols, dtype=torch.float32, device=dev)

    def blocked_unfused():
        for r0 in range(0, rows, rb):
            nr = min(rb, rows - r0)
            first = r0 * cols
            w = dq.dq4_nested(t["packed"][first // 2:], t["scale_codes"][first // 64:],
                              t["nested_absmax"][first // unit:], t["scale_codebook"],
                              t["value_codebook"], float(p.offset), nr * cols, 64, 256,
                              torch.float32, out=transient[:nr * cols])
            torch.addmm(dst, w.view(nr, cols).t(), G[r0:r0 + nr], beta=0.0 if r0 == 0 else 1.0,
                        out=dst)

    full = torch.empty((rows, cols), dtype=torch.float32, device=dev)

    def whole():  # dequantize all of W to FP32, then one GEMM
        dq.dq4_nested(*args_w, rows * cols, 64, 256, torch.float32, out=full.view(-1))
        torch.mm(full.t(), G, out=dst)

    def timeit(fn, k):
        for _ in range(max(3, args.warmup)):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(k):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / k

    k = max(1, args.steps)
    fused()
    torch.cuda.synchronize(dev)
    ref = dst.clone()
    blocked_unfused()
    torch.cuda.synchronize(dev)
    rel = float((ref - dst).abs().max() / dst.abs().max())
    if not rel < 1e-4:
        raise SystemExit(f"fused and unfused out_prod differ (max relative {rel}); refusing to time")
    ms_fused = timeit(fused, k)
    ms_blocked = timeit(blocked_unfused, k)
    ms_whole = timeit(whole, k)
    flops = 2.0 * rows * cols * ncols
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    bf16 = float(peaks.get("bf16_tflops", 1900.0))
    # the two bounds of one call: its algorithmic bytes (packed W, codes, absmax, G read once,
    # dst written once) at the copy bandwidth, and its tensor work (six BF16 products per
    # FP32 multiply-add) at the BF16 peak
    alg_bytes = rows * cols // 2 + rows * cols // 64 + 4 * (rows * cols // unit) + \
        4 * rows * ncols + 4 * cols * ncols
    hbm_ms = alg_bytes / (hbm * 1e9) * 1e3
    tensor_ms = 6 * flops / (bf16 * 1e12) * 1e3
    bound = "tensor" if tensor_ms >= hbm_ms else "hbm"
    nws = int(dq.lib.dq4_nested_out_prod_workspace_bytes(rows, cols, ncols))
    print(json.dumps({
        "metric": "row-blocked dequant + GEMM (dst = W^T G) time",
        "value": ms_fused, "unit": "ms", "higher_is_better": False, "n_gpus": 1,
        "steps": k, "warmup": args.warmup, "ms_per_step": ms_fused, "dtype": "f32",
        "config": {"workload": f"out_prod rows={rows} cols={cols} ncols={ncols}, NF4-style "
                               f"nested (bs 64, nested 256), FP32 G and dst",
                   "l2": f"G alone is {4 * rows * ncols / 1e6:.0f} MB per call"},
        "fp32_equivalent_tflops": flops / (ms_fused / 1e3) / 1e12,
        "roofline": {"bound": bound, "hbm_ms": hbm_ms, "tensor_ms_6_bf16_products": tensor_ms,
                     "frac": max(hbm_ms, tensor_ms) / ms_fused, "peaks": "measured"
                     if peaks else "fallback"},
        "unfused_blocked_ms": ms_blocked,
        "unfused_blocked_transient_bytes": rb * cols * 4,
        "unfused_blocks": -(-rows // rb),
        "whole_copy_ms": ms_whole, "whole_copy_bytes": rows * cols * 4,
        "speedup_vs_unfused_blocked": ms_blocked / ms_fused,
        "workspace_bytes": nws,
        "fused_vs_unfused_max_rel_diff": rel,
        "gpu_launches_per_step": 2 if nws > 0 else 1,
    }), flush=True)


def run_linear(args):
    """Fused nested dequant + tcgen05 GEMM against dequantize-then-cuBLAS, over M.

    Weight sets rotate (more bytes than L2 holds), so every call streams its
    packed weight from HBM.  Per M the line gives both times, the cuBLAS GEMM
    alone, and a roofline: the lower bound is the larger of the tensor time
    (2 M N K at the measured bf16 peak) and the HBM time (packed weight, codes,
    absmax, X and Y at the measured copy bandwidth).
    """
    import torch

    import quantized_weight_dequantization_gb300 as dq

    dev = torch.device("cuda:0")
    N, K = args.lin_n, args.lin_k
    peaks = {"hbm_gbs": 6676.8, "bf16_tflops": 1900.0}
    peak_src = "fallback"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mp = json.load(f)
        peaks = {"hbm_gbs": float(mp["hbm_gbs"]), "bf16_tflops": float(mp["bf16_tflops"])}
        peak_src = "measured"
    except (OSError, KeyError, ValueError):
        pass
    wbytes = (N * K) // 2 + N * K // 64 + 4 * -(-(N * K // 64) // 256)
    nsets = max(2, -(-(160 << 20) // wbytes) + 1)
    sets = []
    for i in range(nsets):
        p = gen.make_problem(N * K, 64, 256, "nf4", 1.0, 0.0371, seed=31 + i) if i < 2 else None
        src = p if p is not None else sets[i % 2]["p"]
        sets.append({"p": src, **{k: torch.from_numpy(np.ascontiguousarray(getattr(src, k))).to(dev)
                                  for k in ("packed", "scale_codes", "nested_absmax",
                                            "scale_codebook", "value_codebook")}})
    Wd = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    cells = []
    for M in [int(x) for x in args.lin_m.split(",")]:
        X = torch.from_numpy(gen.make_normal_g(M, K, seed=32)).to(torch.bfloat16).to(dev)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        state = {"i": 0}

        def nxt():
            state["i"] = (state["i"] + 1) % nsets
            return sets[state["i"]]

        def fused():
            t = nxt()
            dq.linear(X, t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                      t["value_codebook"], float(t["p"].offset), N, 64, 256, Y=Y)

        def unfused():
            t = nxt()
            dq.dq4_nested(t["packed"], t["scale_codes"], t["nested_absmax"],
                          t["scale_codebook"], t["value_codebook"], float(t["p"].offset), N * K,
                          64, 256, torch.bfloat16, out=Wd.view(-1))
            torch.matmul(X, Wd.t(), out=Y)

        def gemm_only():
            torch.matmul(X, Wd.t(), out=Y)

        # each arm is captured as 2 x nsets back-to-back calls in a CUDA graph and timed
        # from its replays (host overhead excluded); the fused arm is also timed eagerly
        res = {}
        for name, fn in (("fused", fused), ("unfused", unfused), ("cublas_gemm_only", gemm_only)):
            stream = torch.cuda.Stream(dev)
            with torch.cuda.stream(stream):
                for _ in range(max(3, args.warmup)):
                    fn()
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                if name == "fused":
                    k = max(1, args.steps)
                    e0.record()
                    for _ in range(k):
                        fn()
                    e1.record()
                    torch.cuda.synchronize(dev)
                    res["fused_eager"] = e0.elapsed_time(e1) / k * 1e3
                calls = 2 * nsets
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for _ in range(calls):
                        fn()
                for _ in range(2):
                    graph.replay()
                torch.cuda.synchronize(dev)
                reps = max(1, args.steps // calls + 1)
                e0.record()
                for _ in range(reps):
                    graph.replay()
                e1.record()
                torch.cuda.synchronize(dev)
                res[name] = e0.elapsed_time(e1) / (reps * calls) * 1e3
        flops = 2.0 * M * N * K
        nbytes = wbytes + 2 * M * K + 2 * M * N
        t_tensor = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        tensor_bound = t_tensor >= t_hbm
        us = res["fused"]
        cells.append({
            "M": M, "fused_us": us, "fused_eager_us": res["fused_eager"],
            "unfused_us": res["unfused"],
            "cublas_gemm_only_us": res["cublas_gemm_only"],
            "speedup_vs_unfused": res["unfused"] / us,
            "roofline": {"bound": "tensor" if tensor_bound else "hbm",
                         "achieved": flops / us / 1e6 if tensor_bound else nbytes / us / 1e3,
                         "peak": peaks["bf16_tflops"] if tensor_bound else peaks["hbm_gbs"],
                         "unit": "TFLOP/s" if tensor_bound else "GB/s",
                         "frac": max(t_tensor, t_hbm) / us,
                         "traffic": None},
            "weight_bytes": wbytes, "algorithmic_bytes": nbytes, "flops": flops})
    print(json.dumps({
        "metric": "fused nested dequant + tcgen05 GEMM (Y = X W^T) time", "unit": "us",
        "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"linear N={N} K={K} NF4-style nested (bs 64, nested 256), "
                               "BF16 X and Y",
                   "l2": f"{nsets} rotating weight sets of {wbytes} bytes (> L2)",
                   "timing": "CUDA-graph replay of back-to-back calls (host overhead "
                             "excluded); fused_eager_us through the Python binding",
                   "peaks": peak_src, **peaks},
        "gpu_launches_per_step": 1,
        "cells": cells}), flush=True)


def graph_time_us(fn, dev, warmup: int, steps: int, calls: int) -> float:
    """Time per call of `fn`: `calls` back-to-back calls captured in a CUDA graph, replayed
    until about `steps` calls ran (host overhead excluded)."""
    import torch

    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(calls):
                fn()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)
        reps = max(1, steps // calls + 1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / (reps * calls) * 1e3


def run_grad_a(args):
    """grad_A = dY W for a nested 4-bit weight W (N x K): the weight dequantized to BF16 and a
    cuBLAS GEMM, with the fused dequantization (dq4_nested, one launch) against the unfused
    three-launch sequence (dq4_nested_unfused, caller-owned FP32 scratch, so no allocator work
    is timed).  "Fuse nested scale reconstruction into SM103 4-bit dequantization", section
    "Problem", names this path (the backward of the 4-bit matmul takes grad_A through the
    dequantization), and section "B300 evidence plan" lists it as a public-path control for
    training shapes.  At those M the weight is dequantized once per call and the GEMM
    dominates; the line reports both the whole step and the dequantization alone.  The two
    arms' dequantized weights and grad_A are checked equal bit for bit first."""
    import torch

    import quantized_weight_dequantization_gb300 as dq

    dev = torch.device("cuda:0")
    cells = []
    for N, K in ((11008, 4096), (4096, 11008)):
        wbytes = (N * K) // 2 + N * K // 64 + 4 * -(-(N * K // 64) // 256)
        nsets = max(2, -(-(160 << 20) // wbytes) + 1)
        p0 = gen.make_problem(N * K, 64, 256, "nf4", 1.0, 0.0371, seed=61)
        sets = []
        for i in range(nsets):
            sets.append({k: torch.from_numpy(np.ascontiguousarray(getattr(p0, k))).to(dev)
                         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook",
                                   "value_codebook")})
        nb = N * K // 64
        scratch = torch.empty(nb, dtype=torch.float32, device=dev)
        Wd = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
        state = {"i": 0}

        def nxt():
            state["i"] = (state["i"] + 1) % nsets
            return sets[state["i"]]

        def deq_fused():
            t = nxt()
            dq.dq4_nested(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                          t["value_codebook"], float(p0.offset), N * K, 64, 256,
                          torch.bfloat16, out=Wd.view(-1))

        def deq_unfused():
            t = nxt()
            dq.dq4_nested_unfused(t["packed"], t["scale_codes"], t["nested_absmax"],
                                  t["scale_codebook"], t["value_codebook"], float(p0.offset),
                                  N * K, 64, 256, torch.bfloat16, out=Wd.view(-1),
                                  scale_scratch=scratch)

        for M in [int(x) for x in args.grad_m.split(",")]:
            dY = torch.from_numpy(gen.make_normal_g(M, N, seed=62)).to(torch.bfloat16).to(dev)
            GA = torch.empty((M, K), dtype=torch.bfloat16, device=dev)

            def fused():
                deq_fused()
                torch.matmul(dY, Wd, out=GA)

            def unfused():
                deq_unfused()
                torch.matmul(dY, Wd, out=GA)

            fused()
            torch.cuda.synchronize(dev)
            w_f, g_f = Wd.clone(), GA.clone()
            unfused()
            torch.cuda.synchronize(dev)
            if not (torch.equal(w_f.view(torch.int16), Wd.view(torch.int16)) and
                    torch.equal(g_f.view(torch.int16), GA.view(torch.int16))):
                raise SystemExit(f"fused and unfused grad_A differ at M={M} N={N} K={K}")
            calls = 2 * nsets
            t = {name: graph_time_us(fn, dev, args.warmup, args.steps, calls)
                 for name, fn in (("fused", fused), ("unfused", unfused),
                                  ("dequant_fused", deq_fused), ("dequant_unfused", deq_unfused))}
            cells.append({"M": M, "N": N, "K": K, "fused_us": t["fused"],
                          "unfused_us": t["unfused"], "speedup": t["unfused"] / t["fused"],
                          "dequant_fused_us": t["dequant_fused"],
                          "dequant_unfused_us": t["dequant_unfused"],
                          "dequant_speedup": t["dequant_unfused"] / t["dequant_fused"]})
        del sets, Wd, scratch
    print(json.dumps({
        "metric": "grad_A = dY W time: fused nested dequant + cuBLAS GEMM", "unit": "us",
        "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "grad_A = dY W, W = N x K NF4-style nested (bs 64, nested 256), "
                               "BF16 dY and grad_A",
                   "l2": "rotating weight sets of more bytes than L2",
                   "timing": "CUDA-graph replay of back-to-back calls (host overhead "
                             "excluded)"},
        "cells": cells}), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "int8prep":
        run_int8prep(args)
    elif args.op == "outprod":
        run_outprod(args)
    elif args.op == "linear":
        run_linear(args)
    elif args.op == "grad_a":
        run_grad_a(args)
    elif args.op == "pair":
        run_pair(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
