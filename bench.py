#!/usr/bin/env python3
"""Throughput of the GB300 error-feedback gradient compressor.

Default workload (--workload layers): the gradient set of a 32-layer
transformer, each layer {4096x4096 x4, 4096x11008 x2, 11008x4096, 4096},
6,476,136,448 fp32 elements (25.9 GB) drawn N(0, (1e-3/sqrt(fan_in))^2) per
tensor, with temporally correlated steps g_t = 0.9 g_{t-1} + 0.436 fresh_t.
One step is one pass of the whole compressor over every tensor: error
feedback + Top-K 1 % of the tensor + 8-bit QSGD (groups of 64, stochastic
rounding) on the kept values + dequantisation + residual write-back, each
of the 256 tensors its own bucket of one gc_ef_topk_quant_buckets call
(every tensor in one launch per pass).  --path per-bucket calls
gc_ef_topk_quant once per tensor, spread over several contexts / CUDA
streams.  --workload buckets runs the same compressor on a flat gradient of
134,217,728 Student-t (nu = 3) elements cut into 25 MiB buckets; the other
workloads are the other compressors of the library.

The metric is fp32 gradient GB/s through the compressor (4 bytes per
gradient element per step), whole job over all GPUs.  Also reported: the
roofline fraction of the dominant kernel (CUDA-event durations of every
launch, measured in a second pass over the same steps), an end-to-end
number through the C ABI with host buffers (pinned H2D of the gradient and
D2H of the compressed result inside the timed region), the single-threaded
CPU oracle on a bounded sample, and SM clocks sampled during the timed
region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    torchrun --nproc-per-node N bench.py --gpus N ...   (one rank per GPU)
"""
import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gradient_compression_ef_gb300 import inputs  # noqa: E402

METRIC = "fp32 gradient GB/s through EF+Top-K+quant compressor; % of GB300 HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gc", "reference"], default="gc")
    p.add_argument("--streams", type=int, default=4, help="contexts/streams for the buckets")
    p.add_argument("--ratio", type=int, default=10, help="Top-K ratio in per mille")
    p.add_argument("--distinct", type=int, default=None,
                   help="distinct correlated gradients (default 2 for layers, else 3)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--diag", action="store_true",
                   help="buckets workload: also compute the fused per-bucket diagnostics")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--residual", choices=["deferred", "immediate"], default="deferred",
                   help="buckets workload: kept entries' residuals applied by the next step's "
                        "read of e (one flush per timed run) or stored by every step")
    p.add_argument("--eager", action="store_true",
                   help="time eager launches instead of CUDA-graph replay")
    p.add_argument("--path", choices=["buckets", "per-bucket"], default="buckets",
                   help="one bucketed call per step, or one call per bucket")
    p.add_argument("--elems", type=int, default=None,
                   help="gradient elements (default: the workload's own size; for buckets a "
                        "smaller value cuts the same 25 MiB buckets from a shorter gradient)")
    p.add_argument("--layers", type=int, default=inputs.TRANSFORMER_LAYERS,
                   help="layers workloads: transformer layers in the gradient set")
    p.add_argument("--workload", choices=["layers", "buckets", "topk", "demo", "quant", "tern",
                                          "powersgd", "aggregate", "randk", "diff"],
                   default="layers",
                   help="layers: EF + Top-K 1%% + 8-bit QSGD per tensor of the 32-layer "
                        "transformer gradient set (the headline); buckets: the same "
                        "compressor per 25 MiB bucket of a flat gradient; topk: EF + Top-K only "
                        "per 25 MiB bucket (--ratio per mille); demo: the error-compensation "
                        "demo (1e6 elements, two EF Top-K 1%% steps, min-max 8-bit); quant: "
                        "EF + group quantisation of 2^30 elements; tern: EF + TernGrad per "
                        "tensor of the transformer layer set; powersgd: rank-4 PowerSGD on one "
                        "layer's matrix shapes; aggregate: 8 ranks' Top-K + QSGD outputs summed "
                        "into one dense gradient; randk: EF + random sparsification at 1%%; "
                        "diff: EF + 4-bit min-max differential quantisation of the "
                        "correlated 134M-element gradient")
    p.add_argument("--mode", choices=["minmax", "qsgd", "log"], default="qsgd",
                   help="quant workload: quantisation rule")
    p.add_argument("--bits", type=int, default=8, help="quant workload: bits per code")
    p.add_argument("--rounding", choices=["nearest_even", "stochastic"], default="stochastic",
                   help="quant workload: rounding")
    args = p.parse_args()
    if args.elems is None:
        args.elems = inputs.GROUP_ELEMS if args.workload == "quant" else inputs.FLAT_ELEMS
    if args.distinct is None:
        # two correlated gradients of the layer set are 52 GB already
        args.distinct = 2 if args.workload in ("layers", "tern") else 3
    return args


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; reads only)
# ---------------------------------------------------------------------------
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    """Polls the SM clock and clock-event reasons of one GPU every ~2 ms."""

    def __init__(self, pci_bus_id):
        self.samples, self.reasons = [], 0
        self.max_mhz = None
        self.ok = False
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nvml.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.nvml, self.h = nvml, h
            self.reason_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _run(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(int(mhz.value))
            if self.reason_fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "source": "unavailable"}
        names = [v for b, v in REASON_BITS.items() if self.reasons & b and b != 0x1]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples),
                "source": "nvml"}


# DRAM traffic of the dominant kernel from one ncu capture:
# dram__bytes_read.sum + dram__bytes_write.sum of bk_hist (the variant that
# applies the previous step's deferred residuals) on 65,536,000 elements, per
# element; the pass streams each element once, so it scales with the
# elements.  Valid only for the kernel source it was taken on (first 16 hex
# digits of the SHA-256 of the file), else the bench reports null.
# DRAM bytes (read + write) of one launch of a workload's dominant kernel
# from a one-kernel ncu capture (profiles/), per element of the launch, with
# a hash of the kernel's source at the time of the capture.
TRAFFIC = {
    ("layers", "bk_hist"): {"bytes_per_elem": (1639.077e6 + 886.405e6) / 202379264,
                            "source": "gradient_compression_ef_gb300/csrc/gc_buckets.cu",
                            "sha256_16": "684a39e10dd37a08",
                            "captured_on": "one transformer layer, 202,379,264 elements"},
    ("buckets", "bk_hist"): {"bytes_per_elem": (530.639e6 + 220.218e6) / 65536000,
                             "source": "gradient_compression_ef_gb300/csrc/gc_buckets.cu",
                             "sha256_16": "684a39e10dd37a08",
                             "captured_on": "65,536,000 elements"},
    # pass 1 is the same as at this capture; the file has since changed in
    # the loaders of passes 2 and 3 only (a proxy fence before each refill)
    ("powersgd", "psgd_mq"): {"bytes_per_elem": (361.22e6 + 134.55e6) / 45088768,
                              "source": "gradient_compression_ef_gb300/csrc/gc_powersgd.cu",
                              "sha256_16": "cd2e0a7cc238c40b",
                              "captured_on": "one 4096 x 11008 matrix, 45,088,768 elements"},
    # the full workload (one pass: both metrics); the output's last tens of
    # MB are still in L2 when the kernel ends, so the writes read below 4 B
    # per output element.  The file has changed since in the bounds kernel
    # only (eight positions a step).
    ("aggregate", "agg_accumulate"): {"bytes_per_elem": (59.95e6 + 471.76e6) / 134217728,
                                      "source": "gradient_compression_ef_gb300/csrc/gc_aggregate.cu",
                                      "sha256_16": "174459dedb864e6b",
                                      "captured_on": "the full workload, 8 ranks x 134,217,728 "
                                                     "elements"},
}


def kernel_traffic(workload, name, elems):
    import hashlib
    t = TRAFFIC.get((workload, name))
    if t is None:
        return None, "no ncu capture for this kernel"
    try:
        digest = hashlib.sha256(open(os.path.join(ROOT, t["source"]), "rb").read()).hexdigest()
    except OSError:
        return None, "kernel source missing"
    if digest[:16] != t["sha256_16"]:
        return None, "kernel changed since the ncu capture"
    return t["bytes_per_elem"] * elems, ("ncu dram bytes of one launch on %s, scaled by "
                                         "elements" % t["captured_on"])


# GB300's nominal HBM3e bandwidth (7.9 TB/s), reported beside the measured peak
NOMINAL_HBM_GBS = 7900.0


def dist_env():
    """(world, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank):
    """Each rank compresses its own gradient replica: a seed of its own."""
    return 42 + rank


def max_over_ranks(torch, value, world, device):
    """The largest of every rank's value (a step time): the job is as slow
    as its slowest rank.  One all-reduce on a one-element tensor; no
    collective touches the gradients."""
    if world <= 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, elems_per_rank, ms_per_step):
    """fp32 gradient GB/s of the whole job: every rank processes
    elems_per_rank elements per step in ms_per_step (the max over ranks)."""
    return world * 4.0 * elems_per_rank / (ms_per_step * 1e-3) / 1e9


def pin_host_near_gpu(torch, dev):
    """Restricts this process to the host CPUs local to the GPU (from the
    PCI device's local_cpulist), so that pinned host buffers are allocated on
    the GPU's own memory node; returns the CPU list, or None when the
    topology is not available (the affinity is then left alone)."""
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        text = open("/sys/bus/pci/devices/%s/local_cpulist" % bus).read().strip()
        cpus = set()
        for part in text.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return text
    except (AttributeError, OSError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# the default workload
# ---------------------------------------------------------------------------
class BucketWorkload:
    """One step = EF + Top-K (+ 8-bit QSGD of the kept values unless
    quant=False) over every bucket: either the 134,217,728-element flat
    gradient in 25 MiB buckets, or (layers) the transformer layer set with
    one bucket per tensor.

    path "buckets": one bucket plan on one context, the whole step is one
    gc_ef_topk_quant_buckets call (one launch per pass over all buckets).
    path "per-bucket": one gc_ef_topk_quant call per bucket, spread over
    several contexts / CUDA streams."""

    BITS, GROUP, SEED = 8, 64, 1000

    def __init__(self, torch, gc, dev, ratio_per_mille, streams, distinct, seed, path,
                 n=inputs.FLAT_ELEMS, diag=False, residual="immediate", layers=None,
                 quant=True):
        self.torch, self.gc, self.dev, self.path = torch, gc, dev, path
        self.quant = quant
        if layers is None:
            # the flat gradient cut into 25 MiB buckets
            self.n = n
            self.bounds = inputs.bucket_bounds(self.n)
            self.grads = inputs.correlated_steps_device(self.n, distinct, dev, seed=seed)
        else:
            # one bucket per tensor of the transformer layer set
            sizes = [n_ for n_, _ in inputs.transformer_set_sizes(layers)]
            self.n = sum(sizes)
            starts = np.concatenate([[0], np.cumsum(sizes)]).tolist()
            self.bounds = [(int(a), int(l)) for a, l in zip(starts, sizes)]
            self.grads = inputs.transformer_set_device(layers, distinct, dev, seed=seed)
        self.ks = [inputs.ratio_k(length, ratio_per_mille, 1000) for _, length in self.bounds]
        self.err = torch.zeros(self.n, dtype=torch.float32, device=dev)
        # outputs of all buckets in three contiguous buffers (16-byte aligned slices)
        self.oi, self.oc, self.os = gc.bucket_offsets(self.ks, self.BITS, self.GROUP)
        self.idx = torch.empty(self.oi[-1], dtype=torch.int32, device=dev)
        self.codes = torch.empty(self.oc[-1], dtype=torch.uint8, device=dev)
        self.scales = torch.empty(self.os[-1], dtype=torch.float32, device=dev)
        # Top-K only: the kept values themselves
        self.val = torch.empty(self.oi[-1], dtype=torch.float32, device=dev) if not quant else None
        # per-bucket diagnostics (sum c^2, sum g_hat^2, sum e'^2), bucketed path only
        self.diag = (torch.zeros(3 * len(self.bounds), dtype=torch.float64, device=dev)
                     if diag and path == "buckets" else None)
        self.main = torch.cuda.current_stream(dev)
        if path == "buckets":
            self.streams = [self.main]
            self.ctxs = [gc.Context(0, stream=self.main)]
            self.ctxs[0].set_buckets([length for _, length in self.bounds], self.ks)
        else:
            self.streams = [torch.cuda.Stream(device=dev) for _ in range(streams)]
            self.ctxs = [gc.Context(max(l for _, l in self.bounds), stream=s)
                         for s in self.streams]
        # deferred: each step keeps its kept entries' residuals aside and the
        # next step applies them while it reads e; finish() flushes the last
        self.deferred = residual == "deferred" and path == "buckets"
        if self.deferred:
            self.ctxs[0].set_deferred_residual(True)

    def out_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.outputs())

    def outputs(self):
        """Device tensors holding one step's compressed result."""
        main = [self.idx, self.codes, self.scales] if self.quant else [self.idx, self.val]
        return main + ([self.diag] if self.diag is not None else [])

    def algorithmic_bytes(self):
        """Bytes the method must move per step: read g and e, write e' (12 B
        per element) plus, per kept entry, its index (4 B) and either its
        code (b/8 B), sign (1/8 B) and 4/64 B of scale, or its value (4 B)."""
        kept = sum(self.ks)
        per_kept = 4 + (self.BITS / 8 + 1 / 8 + 4 / self.GROUP if self.quant else 4)
        return 12 * self.n + kept * per_kept

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        """Enqueues one step on `main` (default: the current stream)."""
        torch, gc = self.torch, self.gc
        main = self.main if main is None else main
        g = self.grads[t % len(self.grads)] if grad is None else grad
        if self.path == "buckets":
            ctx = self.ctxs[0] if ctxs is None else ctxs[0]
            if ctx._stream_ref is not main:
                ctx.set_stream(main)
            if self.quant:
                gc.ef_topk_quant_buckets(ctx, g, self.err, self.BITS, self.GROUP, "stochastic",
                                         self.SEED, t, self.idx, self.codes, self.scales,
                                         diag=self.diag)
            else:
                gc.ef_topk_buckets(ctx, g, self.err, self.idx, self.val, diag=self.diag)
            return
        ctxs = self.ctxs if ctxs is None else ctxs
        streams = [c._stream_ref for c in ctxs]
        fork = torch.cuda.Event()
        fork.record(main)
        for s in streams:
            s.wait_event(fork)
        oi, oc, os_ = self.oi, self.oc, self.os
        for b, ((start, length), k) in enumerate(zip(self.bounds, self.ks)):
            ctx = ctxs[b % len(ctxs)]
            if not self.quant:
                gc.ef_topk(ctx, g[start:start + length], self.err[start:start + length], k,
                           self.idx[oi[b]:oi[b] + k], self.val[oi[b]:oi[b] + k], n=length)
                continue
            gc.ef_topk_quant(ctx, g[start:start + length], self.err[start:start + length], k,
                             self.BITS, self.GROUP, "stochastic", gc.bucket_seed(self.SEED, b), t,
                             self.idx[oi[b]:oi[b] + k], self.codes[oc[b]:oc[b + 1]],
                             self.scales[os_[b]:os_[b + 1]], n=length)
        for s in streams:
            j = torch.cuda.Event()
            j.record(s)
            main.wait_event(j)

    def finish(self):
        """Enqueues what completes the last step's results: with deferred
        residuals, the flush of the last step's kept-entry residuals into e.
        Returns the launches it made."""
        if not self.deferred:
            return 0
        ctx = self.ctxs[0]
        if ctx._stream_ref is not self.main:
            ctx.set_stream(self.main)
        ctx.bucket_flush()
        return 1

    def capture(self):
        """One CUDA graph per distinct gradient buffer, each holding a whole
        step.  Returns (graphs, launches/step).  With deferred residuals one
        eager step first leaves residuals pending, so that every captured
        step applies the ones the step before it left."""
        torch = self.torch
        if self.deferred:
            self.launch_step(0)
        graphs = []
        cap = torch.cuda.Stream(device=self.dev)
        before = self.launches()
        for d in range(len(self.grads)):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(self.main)
            with torch.cuda.graph(g, stream=cap):
                self.launch_step(d, main=cap)
            graphs.append(g)
        self.main.wait_stream(cap)
        if self.path == "buckets":
            self.ctxs[0].set_stream(self.main)
        return graphs, (self.launches() - before) // len(self.grads)

    def algorithmic_bytes_per_launch(self):
        """Bytes each kernel must move per launch.  Bucketed path (one launch
        covers every bucket): hist reads g, e and writes c (12 B/element);
        collect and refine walk the candidate lists (scratch, no gradient
        bytes); write stores each kept index (4 B) and, Top-K only, its value
        (4 B); the QSGD pass writes code, sign, 1/64 of a scale and the
        residual of each kept entry (4 B).  Per-bucket path: the same per
        bucket."""
        kept = sum(self.ks)
        q = kept * (self.BITS / 8 + 1 / 8 + 4 / self.GROUP + 4)
        if self.path == "buckets":
            out = {"bk_hist": 12.0 * self.n, "bk_collect": 0.0, "bk_refine": 0.0,
                   "bk_write": (4.0 if self.quant else 8.0) * kept}
            if self.quant:
                out["bk_quant"] = q
            return out
        nb = len(self.bounds)
        n = self.n / nb
        return {"ef_hist": 12.0 * n, "collect": 4.0 * n, "refine": 0.0,
                "write": 4.0 * n + 12.0 * kept / nb,
                "quant_fused": kept / nb * (8 + self.BITS / 8 + 1 / 8 + 4 / self.GROUP + 4)}

    def launches(self):
        return sum(c.launch_count() for c in self.ctxs)

    def check(self):
        for c in self.ctxs:
            c.check()


class _SimpleWorkload:
    """Shared plumbing of the single-context workloads: one context on the
    main stream, whole steps captured in CUDA graphs."""

    def _init_common(self, torch, gc, dev, max_n):
        self.torch, self.gc, self.dev = torch, gc, dev
        self.main = torch.cuda.current_stream(dev)
        self.streams = [self.main]
        self.ctxs = [gc.Context(max_n, stream=self.main)]

    def out_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.outputs())

    def _ctx_on(self, main, ctxs):
        ctx = self.ctxs[0] if ctxs is None else ctxs[0]
        if ctx._stream_ref is not main:
            ctx.set_stream(main)
        return ctx

    def _init_streams(self, count, make_ctx):
        """count > 1: one context per CUDA stream, the first the common one,
        the others made by make_ctx(stream)."""
        if count <= 1:
            return
        self.streams = [self.torch.cuda.Stream(device=self.dev) for _ in range(count)]
        self.ctxs = [self.ctxs[0]] + [make_ctx(st) for st in self.streams[1:]]
        self.ctxs[0].set_stream(self.streams[0])

    def _fork(self, main, ctxs):
        """The contexts a step uses in turn and the streams to join back:
        one context on `main` when given `ctxs` (the per-kernel timing) or
        when there is only one, else every context, forked from `main`."""
        if ctxs is not None or len(self.ctxs) == 1:
            return [self._ctx_on(main, ctxs)], []
        fork = self.torch.cuda.Event()
        fork.record(main)
        for c in self.ctxs:
            c._stream_ref.wait_event(fork)
        return self.ctxs, [c._stream_ref for c in self.ctxs]

    def _join(self, main, streams):
        for st in streams:
            j = self.torch.cuda.Event()
            j.record(st)
            main.wait_event(j)

    def finish(self):
        return 0

    def capture(self):
        torch = self.torch
        graphs = []
        cap = torch.cuda.Stream(device=self.dev)
        before = self.launches()
        for d in range(len(self.grads)):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(self.main)
            with torch.cuda.graph(g, stream=cap):
                self.launch_step(d, main=cap)
            graphs.append(g)
        self.main.wait_stream(cap)
        self.ctxs[0].set_stream(self.main)
        return graphs, (self.launches() - before) // len(self.grads)

    def launches(self):
        return sum(c.launch_count() for c in self.ctxs)

    def check(self):
        for c in self.ctxs:
            c.check()


class QuantWorkload(_SimpleWorkload):
    """Group-wise quantisation with error feedback: 2^30 fp32 N(0, 0.01^2)
    with 0.1 % distinct positions x 100, groups of 64; one step is one
    gc_ef_quant call over the whole array (the fused single-pass kernel)."""

    GROUP, SEED = 64, 77

    def __init__(self, torch, gc, dev, args, seed):
        self.n = args.elems
        self.bits, self.mode, self.rounding = args.bits, args.mode, args.rounding
        self._init_common(torch, gc, dev, 0)
        self.grads = [inputs.outlier_gradient_device(self.n, dev, seed + d)
                      for d in range(args.distinct)]
        self.err = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.codes = torch.empty(gc.codes_bytes(self.n, self.bits, self.mode),
                                 dtype=torch.uint8, device=dev)
        self.scales = torch.empty(gc.scales_floats(self.n, self.GROUP, self.mode),
                                  dtype=torch.float32, device=dev)

    def outputs(self):
        return [self.codes, self.scales]

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        main = self.main if main is None else main
        ctx = self._ctx_on(main, ctxs)
        g = self.grads[t % len(self.grads)] if grad is None else grad
        self.gc.ef_quant(ctx, g, self.err, self.bits, self.GROUP, self.mode, self.rounding,
                         self.SEED, t, self.codes, self.scales)

    def algorithmic_bytes(self):
        """Read g and e, write e' (12 B per element), the packed codes and
        the scales."""
        return 12 * self.n + self.codes.numel() + 4 * self.scales.numel()

    def algorithmic_bytes_per_launch(self):
        return {"quant_fused": float(self.algorithmic_bytes())}


class TernWorkload(_SimpleWorkload):
    """TernGrad with error feedback on the transformer layer set (--layers
    layers of 4 x 4096^2, 2 x 4096 x 11008, 11008 x 4096, 4096), one scale
    per tensor (max |c|), stochastic rounding: one gc_ef_quant call per
    tensor, tensor t keyed by gc_bucket_seed(SEED, t).  The tensors go round
    robin to --streams contexts, each on its own CUDA stream, as layer-wise
    compression would be issued: a tensor's statistics pass (memory-bound)
    then overlaps another tensor's apply pass (issue-bound)."""

    SEED = 91

    def __init__(self, torch, gc, dev, args, seed):
        sizes = [n_ for n_, _ in inputs.transformer_set_sizes(args.layers)]
        self.sizes = sizes
        self.n = sum(sizes)
        self._init_common(torch, gc, dev, max(sizes))
        self._init_streams(args.streams, lambda st: gc.Context(max(sizes), stream=st))
        self.starts = np.concatenate([[0], np.cumsum(sizes)]).tolist()
        self.grads = inputs.transformer_set_device(args.layers, args.distinct, dev, seed=seed)
        self.err = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.cb = [gc.codes_bytes(n_, 2, "tern") for n_ in sizes]
        self.coff = np.concatenate([[0], np.cumsum(self.cb)]).tolist()
        self.codes = torch.empty(self.coff[-1], dtype=torch.uint8, device=dev)
        self.scales = torch.empty(4 * len(sizes), dtype=torch.float32, device=dev)

    def outputs(self):
        return [self.codes, self.scales]

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        main = self.main if main is None else main
        g = self.grads[t % len(self.grads)] if grad is None else grad
        ctxs, join = self._fork(main, ctxs)
        for w_, (a, b) in enumerate(zip(self.starts, self.starts[1:])):
            self.gc.ef_quant(ctxs[w_ % len(ctxs)], g[a:b], self.err[a:b], 2, 0, "tern",
                             "stochastic", self.gc.bucket_seed(self.SEED, w_), t,
                             self.codes[self.coff[w_]:self.coff[w_ + 1]],
                             self.scales[4 * w_:4 * w_ + 4])
        self._join(main, join)

    def algorithmic_bytes(self):
        """Read g and e, write e' (12 B per element) and 2-bit codes; the
        per-tensor max needs the whole tensor before any element can be
        coded, so the kernels read c once more (16 B per element)."""
        return 12 * self.n + self.codes.numel() + 4 * len(self.sizes)

    def algorithmic_bytes_per_launch(self):
        """quant_stats reads g, e and writes c (12 B per element); quant_apply
        reads c, writes e' and the codes (8.25 B per element); averaged over
        the set's tensors."""
        k = len(self.sizes)
        return {"quant_stats": 12.0 * self.n / k,
                "quant_apply": (8.0 * self.n + self.codes.numel()) / k}


class PowerSGDWorkload(_SimpleWorkload):
    """Rank-4 PowerSGD with error feedback on the matrices of the transformer
    layers: --layers x {4096 x 4096, 4096 x 11008, 11008 x 4096} (96
    matrices for 32 layers), each a rank-16 signal plus N(0, 1e-4^2) noise
    with its own start Q: one gc_powersgd_step per matrix per step, every
    matrix's Q carried from step to step.  The matrices go round robin to
    --streams contexts on their own CUDA streams (each with its own
    PowerSGD scratch), so one matrix's short passes and kernel tails overlap
    another's streaming passes."""

    R = 4

    def __init__(self, torch, gc, dev, args, seed):
        shapes = list(inputs.POWERSGD_SHAPES) * args.layers
        self.shapes = shapes
        self.n = sum(m * n_ for m, n_ in shapes)
        self._init_common(torch, gc, dev, 0)
        mm, mn = max(m for m, _ in shapes), max(n_ for _, n_ in shapes)

        def make_ctx(st):
            c = gc.Context(0, stream=st)
            c.reserve_powersgd(mm, mn, self.R)
            return c
        self.ctxs[0].reserve_powersgd(mm, mn, self.R)
        self._init_streams(args.streams, make_ctx)
        self.starts = np.concatenate([[0], np.cumsum([m * n_ for m, n_ in shapes])]).tolist()
        flat = torch.empty(self.n, dtype=torch.float32, device=dev)
        self.Q = []
        for i, (m, n_) in enumerate(shapes):
            M, Q0 = inputs.low_rank_matrix_device(m, n_, dev, seed=seed * 1000 + i, r=self.R)
            flat[self.starts[i]:self.starts[i + 1]] = M.reshape(-1)
            self.Q.append(Q0.contiguous())
            del M
        self.grads = [flat]
        self.err = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.P = [torch.empty(m * self.R, dtype=torch.float32, device=dev) for m, _ in shapes]

    def outputs(self):
        return self.P + self.Q

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        main = self.main if main is None else main
        g = self.grads[t % len(self.grads)] if grad is None else grad
        ctxs, join = self._fork(main, ctxs)
        for i, (m, n_) in enumerate(self.shapes):
            a, b = self.starts[i], self.starts[i + 1]
            self.gc.powersgd_step(ctxs[i % len(ctxs)], g[a:b], self.err[a:b], m, n_, self.R,
                                  self.P[i], self.Q[i])
        self._join(main, join)

    def algorithmic_bytes(self):
        """The minimum: read G and E, write E' (12 B per element)."""
        return 12 * self.n

    def algorithmic_bytes_per_launch(self):
        """Per matrix: pass 1 reads G, E and writes M into E (12 B per
        element), pass 2 reads M (4 B), pass 3 reads M and writes E' (8 B);
        averaged over the three matrices."""
        k = len(self.shapes)
        return {"psgd_mq": 12.0 * self.n / k, "psgd_mtp": 4.0 * self.n / k,
                "psgd_resid": 8.0 * self.n / k}


class AggregateWorkload(_SimpleWorkload):
    """The step after compression: W = 8 simulated ranks' Top-K 1 % + 8-bit
    QSGD outputs (groups of 64) over the 134,217,728-element gradient,
    aggregated into one dense fp32 gradient in rank order by one
    gc_topk_quant_aggregate call.  Each rank's outputs come from the hybrid
    compressor on its own Student-t gradient; all of a step's compressed
    inputs sit in one byte buffer (indices, codes, scales)."""

    W, BITS, GROUP = 8, 8, 64

    def __init__(self, torch, gc, dev, args, seed):
        self.n = args.elems
        n, W = self.n, self.W
        self.k = k = inputs.ratio_k(n, 1, 100)
        K = -(-k // 4) * 4
        self.cb = gc.codes_bytes(k, self.BITS, "qsgd")
        self.sf = -(-gc.scales_floats(k, self.GROUP, "qsgd") // 4) * 4
        self._init_common(torch, gc, dev, n)
        # byte offsets of the three arrays inside one step's input buffer
        self.o_idx, self.o_codes = 0, 4 * W * K
        self.o_scales = self.o_codes + -(-(W * self.cb) // 16) * 16
        total = self.o_scales + 4 * W * self.sf
        self.grads = []
        ctx = self.ctxs[0]
        e = torch.zeros(n, dtype=torch.float32, device=dev)
        for d in range(args.distinct):
            buf = torch.zeros(total, dtype=torch.uint8, device=dev)
            idx, codes, scales = self._views(buf)
            for w in range(W):
                g = inputs.student_t_device(n, dev, seed=seed * 100 + d * W + w)
                e.zero_()
                gc.ef_topk_quant(ctx, g, e, k, self.BITS, self.GROUP, "stochastic", 5 + w, d,
                                 idx[w * K:w * K + k], codes[w * self.cb:(w + 1) * self.cb],
                                 scales[w * self.sf:w * self.sf +
                                        gc.scales_floats(k, self.GROUP, "qsgd")])
            self.grads.append(buf)
        ctx.check()
        del e
        self.out = torch.empty(n, dtype=torch.float32, device=dev)

    def _views(self, buf):
        W, K = self.W, -(-self.k // 4) * 4
        idx = buf[self.o_idx:self.o_idx + 4 * W * K].view(self.torch.int32)
        codes = buf[self.o_codes:self.o_codes + W * self.cb]
        scales = buf[self.o_scales:self.o_scales + 4 * W * self.sf].view(self.torch.float32)
        return idx, codes, scales

    def outputs(self):
        return [self.out]

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        main = self.main if main is None else main
        ctx = self._ctx_on(main, ctxs)
        buf = self.grads[t % len(self.grads)] if grad is None else grad
        idx, codes, scales = self._views(buf)
        self.gc.topk_quant_aggregate(ctx, self.W, self.k, idx, codes, scales, self.BITS,
                                     self.GROUP, self.n, self.out)

    def input_bytes(self):
        return self.grads[0].numel()

    def algorithmic_bytes(self):
        """Write the dense gradient (4 B per element) and read every rank's
        indices, codes, signs and scales once."""
        return 4 * self.n + self.W * (4 * self.k + self.cb + 4 * self.sf)

    def algorithmic_bytes_per_launch(self):
        """bounds reads the indices (4 B per entry); accumulate reads indices,
        codes and scales and writes the dense output."""
        return {"agg_bounds": 4.0 * self.W * self.k,
                "agg_accumulate": float(self.algorithmic_bytes())}


class RandKWorkload(_SimpleWorkload):
    """Error feedback + random sparsification (keep each element with
    probability 1 %) over the 134,217,728-element gradient: one gc_ef_randk
    call per step."""

    P, SEED = 0.01, 31

    def __init__(self, torch, gc, dev, args, seed):
        self.n = args.elems
        self._init_common(torch, gc, dev, self.n)
        self.grads = inputs.correlated_steps_device(self.n, args.distinct, dev, seed=seed)
        self.err = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.cap = -(-int(self.n * self.P * 1.1 + 1024) // 4) * 4
        self.idx = torch.empty(self.cap, dtype=torch.int32, device=dev)
        self.val = torch.empty(self.cap, dtype=torch.float32, device=dev)
        self.count = torch.zeros(2, dtype=torch.int64, device=dev)

    def outputs(self):
        return [self.idx, self.val, self.count]

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        main = self.main if main is None else main
        ctx = self._ctx_on(main, ctxs)
        g = self.grads[t % len(self.grads)] if grad is None else grad
        self.gc.ef_randk(ctx, g, self.err, self.P, self.SEED, t, self.idx, self.val, self.count)

    def algorithmic_bytes(self):
        """Read g and e, write e' (12 B per element) and the kept (index,
        value) pairs (8 B per kept entry)."""
        return 12 * self.n + 8 * self.n * self.P

    def algorithmic_bytes_per_launch(self):
        """mark reads g, e and writes e' (12 B per element); write stores the
        kept pairs (8 B each)."""
        return {"randk_mark": 12.0 * self.n, "randk_write": 8.0 * self.n * self.P}


class DiffWorkload(_SimpleWorkload):
    """Error feedback + differential quantisation of the correlated
    134,217,728-element gradient: the change from the history is quantised
    in 4-bit min-max groups of 64 with stochastic rounding; one
    gc_ef_diff_quant call per step (the first call of the run refreshes)."""

    BITS, GROUP, MODE, SEED = 4, 64, "minmax", 53

    def __init__(self, torch, gc, dev, args, seed):
        self.n = args.elems
        self._init_common(torch, gc, dev, 0)
        self.grads = inputs.correlated_steps_device(self.n, args.distinct, dev, seed=seed)
        self.err = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.ref = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.codes = torch.empty(gc.codes_bytes(self.n, self.BITS, self.MODE),
                                 dtype=torch.uint8, device=dev)
        self.scales = torch.empty(gc.scales_floats(self.n, self.GROUP, self.MODE),
                                  dtype=torch.float32, device=dev)
        self.first = True

    def outputs(self):
        return [self.codes, self.scales]

    def launch_step(self, t, grad=None, main=None, ctxs=None):
        main = self.main if main is None else main
        ctx = self._ctx_on(main, ctxs)
        g = self.grads[t % len(self.grads)] if grad is None else grad
        refresh, self.first = self.first, False
        self.gc.ef_diff_quant(ctx, g, self.err, self.ref, self.BITS, self.GROUP, self.MODE,
                              "stochastic", self.SEED, t, refresh, self.codes, self.scales)

    def algorithmic_bytes(self):
        """Read g, e and the history, write e' and the history (20 B per
        element), the packed codes and the scales."""
        return 20 * self.n + self.codes.numel() + 4 * self.scales.numel()

    def algorithmic_bytes_per_launch(self):
        return {"quant_fused": float(self.algorithmic_bytes())}


class DemoWorkload(_SimpleWorkload):
    """The Python demo of "梯度聚合通信优化实战方案" (Python 演示) replayed on
    the GPU: a 1,000,000-element N(0, 1) gradient (numpy seed 42), zero
    residual; one step is the demo's sequence -- EF + Top-K 1 % (k =
    10,000) on g, EF + Top-K 1 % on fl(0.9 g) with the residual the first
    call left, and whole-tensor min-max 8-bit quantisation of g (round half
    to even) with its dequantisation.  Every step starts the demo again from
    a zero residual (cleared inside the step).  The 4 MB arrays stay in L2."""

    K, N = 10_000, 1_000_000

    def __init__(self, torch, gc, dev, args, seed):
        n = self.N
        self.n = 3 * n  # gradient elements one step runs through the compressor
        self._init_common(torch, gc, dev, n)
        g = inputs.demo_gradient(n)
        self.g1 = torch.from_numpy(g).to(dev)
        self.g2 = torch.from_numpy((g * np.float32(0.9)).astype(np.float32)).to(dev)
        self.grads = [self.g1]
        self.err = torch.zeros(n, dtype=torch.float32, device=dev)
        self.idx = [torch.empty(self.K, dtype=torch.int32, device=dev) for _ in range(2)]
        self.val = [torch.empty(self.K, dtype=torch.float32, device=dev) for _ in range(2)]
        self.codes = torch.empty(gc.codes_bytes(n, 8, "minmax"), dtype=torch.uint8, device=dev)
        self.scales = torch.empty(gc.scales_floats(n, 0, "minmax"), dtype=torch.float32,
                                  device=dev)
        self.deq = torch.empty(n, dtype=torch.float32, device=dev)

    def outputs(self):
        return self.idx + self.val + [self.codes, self.scales]

    def launch_step(self, t, grad=None, main=None, ctxs=None, energies=None):
        main = self.main if main is None else main
        ctx = self._ctx_on(main, ctxs)
        g1 = self.g1 if grad is None else grad
        self.err.zero_()
        self.gc.ef_topk(ctx, g1, self.err, self.K, self.idx[0], self.val[0])
        if energies is not None:
            energies.append(float((self.err.double() ** 2).sum()))
        self.gc.ef_topk(ctx, self.g2, self.err, self.K, self.idx[1], self.val[1])
        if energies is not None:
            energies.append(float((self.err.double() ** 2).sum()))
        self.gc.quant(ctx, g1, 8, 0, "minmax", "nearest_even", 0, 0, self.codes, self.scales)
        self.gc.dequant(ctx, self.codes, self.scales, self.N, 8, 0, "minmax", self.deq)

    def input_bytes(self):
        return 4 * self.N

    def algorithmic_bytes(self):
        """Two EF Top-K calls (read g and e, write e': 12 B per element, 8 B
        per kept entry), the quantisation (read g, write 1 B codes) and the
        dequantisation (read codes, write 4 B)."""
        return 2 * (12 * self.N + 8 * self.K) + 5 * self.N + 5 * self.N

    def algorithmic_bytes_per_launch(self):
        return {"ef_hist": 12.0 * self.N, "quant_apply": 5.0 * self.N,
                "dequant": 5.0 * self.N}


WORKLOADS = {"demo": DemoWorkload, "quant": QuantWorkload, "tern": TernWorkload, "powersgd": PowerSGDWorkload,
             "aggregate": AggregateWorkload, "randk": RandKWorkload, "diff": DiffWorkload}


def kernel_timing(wl, steps, warmup_step, launches_per_step):
    """Per-phase CUDA-event durations over `steps` more steps run with all
    buckets on one context / stream, so that each kernel runs alone and its
    events bracket its own execution (room for every launch of the steps)."""
    ctx = wl.ctxs[0]
    ctx.enable_timing(max(64, launches_per_step + 8) * steps)
    for t in range(steps):
        wl.launch_step(warmup_step + t, ctxs=[ctx])
    wl.finish()
    phases = {name: [ms, cnt] for name, (ms, cnt) in ctx.read_timing().items()}
    ctx.enable_timing(0)
    return phases


def cpu_sample(args, seed=7):
    """One bounded sample of the workload for the oracle: returns
    (callable running the oracle on it once, fp32 gradient elements it
    covers, description)."""
    import oracle
    r = inputs.rng(seed)
    if args.workload == "quant":
        n = 1 << 22
        g = r.standard_normal(n).astype(np.float32) * np.float32(0.01)
        e = np.zeros(n, np.float32)
        return (lambda: oracle.ef_quant(g, e, args.bits, 64, args.mode, args.rounding, 77, 0),
                n, "4,194,304 elements of the 2^30-element gradient, EF + %s %d-bit g64 %s"
                % (args.mode, args.bits, args.rounding))
    if args.workload == "tern":
        g = inputs.transformer_tensor(0, 0)  # one 4096 x 4096 tensor
        e = np.zeros_like(g)
        return (lambda: oracle.ef_quant(g, e, 2, 0, "tern", "stochastic", 91, 0), g.size,
                "one 4096 x 4096 tensor of the layer set, EF + TernGrad per tensor")
    if args.workload == "diff":
        n = 1 << 22
        g = inputs.student_t(r, n)
        e = np.zeros(n, np.float32)
        ref = (0.9 * g + 0.1 * inputs.student_t(r, n)).astype(np.float32)
        return (lambda: oracle.ef_diff_quant(g, e, ref, 4, 64, "minmax", "stochastic", 53, 1),
                n, "4,194,304 elements, EF + 4-bit min-max differential quantisation g64")
    if args.workload == "randk":
        n = 1 << 22
        g = inputs.student_t(r, n)
        e = (0.1 * inputs.student_t(r, n)).astype(np.float32)
        return (lambda: oracle.ef_randk(g, e.copy(), 0.01, 31, 0), n,
                "4,194,304 elements, EF + random sparsification at 1%")
    if args.workload == "aggregate":
        n, W = 1 << 22, 8
        k = inputs.ratio_k(n, 1, 100)
        idx, codes, scales = [], [], []
        for w in range(W):
            g = inputs.student_t(inputs.rng(seed + w), n)
            i_, c_, s_, _ = oracle.ef_topk_quant(g, np.zeros(n, np.float32), k, 8, 64,
                                                 "stochastic", 5 + w, 0)
            idx.append(i_)
            codes.append(c_)
            s4 = np.zeros(-(-s_.size // 4) * 4, np.float32)
            s4[:s_.size] = s_
            scales.append(s4)
        idx, codes, scales = np.stack(idx), np.concatenate(codes), np.concatenate(scales)
        return (lambda: oracle.topk_quant_aggregate(idx, codes, scales, W, k, 8, 64, n), n,
                "8 ranks' Top-K 1%% + 8-bit QSGD outputs over 4,194,304 elements, aggregated")
    if args.workload == "powersgd":
        M, Q0 = inputs.low_rank_matrix(4096, 4096, seed=seed, r=4)
        E = np.zeros_like(M)
        return (lambda: oracle.powersgd_step(M, E, Q0, 4), M.size,
                "one 4096 x 4096 matrix of the layer, rank-4 PowerSGD step (fp64)")
    if args.workload == "demo":
        g = inputs.demo_gradient()
        g2 = (g * np.float32(0.9)).astype(np.float32)

        def run():
            _, _, e = oracle.ef_topk(g, np.zeros_like(g), 10_000)
            oracle.ef_topk(g2, e, 10_000)
            codes, scales = oracle.quant(g, 8, 0, "minmax", "nearest_even")
            oracle.dequant(codes, scales, g.size, 8, 0, "minmax")
        return (run, 3 * g.size, "the whole demo: two EF + Top-K 1% calls on 1,000,000 elements "
                "and whole-tensor min-max 8-bit quantisation and dequantisation")
    if args.workload == "topk":
        length = inputs.BUCKET_ELEMS
        k = inputs.ratio_k(length, args.ratio, 1000)
        g = inputs.student_t(r, length)
        e = (0.1 * inputs.student_t(r, length)).astype(np.float32)
        return (lambda: oracle.ef_topk(g, e, k), length,
                "one 6,553,600-element bucket, EF + Top-K %g%%" % (args.ratio / 10))
    if args.workload == "layers":
        g = inputs.transformer_tensor(0, 0)
        e = (0.1 * inputs.transformer_tensor(1, 0)).astype(np.float32)
        k = inputs.ratio_k(g.size, args.ratio, 1000)
        return (lambda: oracle.ef_topk_quant(g, e, k, 8, 64, "stochastic", 1000, 0), g.size,
                "one 4096 x 4096 tensor of the layer set, EF + Top-K %g%% + 8-bit QSGD"
                % (args.ratio / 10))
    length = inputs.BUCKET_ELEMS
    k = inputs.ratio_k(length, args.ratio, 1000)
    g = inputs.student_t(r, length)
    e = (0.1 * inputs.student_t(r, length)).astype(np.float32)
    return (lambda: oracle.ef_topk_quant(g, e, k, 8, 64, "stochastic", 1000, 0), length,
            "one 6,553,600-element bucket, EF + Top-K %g%% + 8-bit QSGD" % (args.ratio / 10))


def cpu_baseline(args, budget_s=12.0):
    """The oracle (single-threaded C) on a bounded sample of the workload,
    repeated until about budget_s seconds (at most 8 runs); GB/s of fp32
    gradient."""
    run, n, what = cpu_sample(args)
    elapsed, runs = 0.0, 0
    while runs == 0 or (elapsed < budget_s and runs < 8):
        t0 = time.perf_counter()
        run()
        elapsed += time.perf_counter() - t0
        runs += 1
    return {"value": 4.0 * n * runs / elapsed / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%s, %d run(s), %.1f s single-threaded" % (what, runs, elapsed)}


def config(args, wl=None):
    n = args.elems
    l2 = {"l2": "inputs larger than L2: each step reads a {0} MiB gradient and the {0} MiB "
                "residual, no flush", "parallelism": "dp%d" % args.gpus}
    if args.workload == "quant":
        cfg = {"workload": "flat fp32 gradient {:,} elements N(0, 0.01^2) with 0.1% distinct "
                           "positions x 100; EF + {} {}-bit quantisation, groups of 64, {} "
                           "rounding".format(n, args.mode, args.bits, args.rounding),
               "total_elems": n, "group": 64, "mode": args.mode, "bits": args.bits,
               "rounding": args.rounding}
    elif args.workload == "tern":
        sizes = [n_ for n_, _ in inputs.transformer_set_sizes(args.layers)]
        n = sum(sizes)
        cfg = {"workload": "transformer gradient set, {} layers x {{4096x4096 x4, 4096x11008 x2, "
                           "11008x4096, 4096}} = {:,} fp32 elements, N(0, (1e-3/sqrt(fan_in))^2), "
                           "correlated steps; EF + TernGrad per tensor (scale = max|c| of the "
                           "tensor), stochastic, 2-bit codes".format(args.layers, n),
               "total_elems": n, "layers": args.layers, "tensors": len(sizes)}
    elif args.workload == "diff":
        cfg = {"workload": "flat fp32 gradient {:,} elements, Student-t nu=3 x 1e-3, correlated "
                           "steps; EF + differential quantisation against the reconstructed "
                           "history, 4-bit min-max groups of 64, stochastic".format(n),
               "total_elems": n, "bits": 4, "group": 64, "mode": "minmax"}
    elif args.workload == "randk":
        cfg = {"workload": "flat fp32 gradient {:,} elements, Student-t nu=3 x 1e-3, correlated "
                           "steps; EF + random sparsification keeping each element with "
                           "probability 1% (Philox draws)".format(n),
               "total_elems": n, "keep_probability": 0.01}
    elif args.workload == "aggregate":
        cfg = {"workload": "8 simulated ranks' Top-K 1% + 8-bit QSGD (groups of 64) outputs over "
                           "a {:,}-element Student-t gradient, summed in rank order into one "
                           "dense fp32 gradient".format(n),
               "total_elems": n, "ranks": 8, "topk_percent": 1, "quant": "qsgd 8-bit g64"}
    elif args.workload == "demo":
        cfg = {"workload": "error-compensation demo: 1,000,000 fp32 N(0,1) (numpy seed 42), zero "
                           "residual; EF + Top-K 1% (k = 10,000), EF + Top-K 1% on 0.9 g with "
                           "the residual, whole-tensor min-max 8-bit quantisation (round half to "
                           "even) and dequantisation; the residual restarts at 0 every step",
               "total_elems": 3 * 1_000_000, "gradient_elems": 1_000_000, "k": 10_000}
    elif args.workload == "topk":
        bounds = inputs.bucket_bounds(n)
        cfg = {"workload": "flat fp32 gradient {:,} elements in 25 MiB buckets ({} buckets), "
                           "Student-t nu=3 x 1e-3, correlated steps; per bucket EF + Top-K {:g}% "
                           "only, (index, value) outputs".format(n, len(bounds), args.ratio / 10),
               "total_elems": n, "bucket_elems": inputs.BUCKET_ELEMS, "buckets": len(bounds),
               "topk_per_mille": args.ratio, "path": args.path}
        if args.path == "buckets":
            cfg["residual"] = ("deferred: each step's kept entries are cleared in e by the next "
                               "step's read of e; the last step's are flushed inside the timed "
                               "region" if args.residual == "deferred" else
                               "immediate: every step clears its kept entries in e")
    elif args.workload == "layers":
        sizes = [n_ for n_, _ in inputs.transformer_set_sizes(args.layers)]
        n = sum(sizes)
        cfg = {"workload": "transformer gradient set, {} layers x {{4096x4096 x4, 4096x11008 x2, "
                           "11008x4096, 4096}} = {:,} fp32 elements, N(0, (1e-3/sqrt(fan_in))^2), "
                           "correlated steps; per tensor (one bucket each) EF + Top-K {:g}% + 8-bit "
                           "QSGD (groups of 64, stochastic) on the kept values".format(
                               args.layers, n, args.ratio / 10),
               "total_elems": n, "layers": args.layers, "tensors": len(sizes),
               "topk_per_mille": args.ratio, "quant": "qsgd 8-bit g64 stochastic",
               "path": args.path}
        if args.path == "buckets":
            cfg["residual"] = ("deferred: each step's kept-entry residuals are applied by the "
                               "next step's read of e; the last step's are flushed into e inside "
                               "the timed region" if args.residual == "deferred" else
                               "immediate: every step stores its kept-entry residuals into e")
    elif args.workload == "powersgd":
        n = sum(m * n_ for m, n_ in inputs.POWERSGD_SHAPES) * args.layers
        cfg = {"workload": "PowerSGD rank 4 with error feedback on {} matrices ({} layers x "
                           "{{4096x4096, 4096x11008, 11008x4096}}), each a rank-16 signal "
                           "(singular values 1 .. 0.05 geometric) + N(0, 1e-4^2) noise with its "
                           "own N(0,1) start Q; every step runs each matrix once and carries "
                           "its Q to the next step".format(3 * args.layers, args.layers),
               "total_elems": n, "rank": 4, "matrices": 3 * args.layers,
               "gemm_path": "P = M Q on tcgen05 kind::tf32 (3-term split, fp32 accumulate); "
                            "Q' = M^T P_hat and E' on CUDA-core fp32 FMAs"}
    else:
        bounds = inputs.bucket_bounds(n)
        sizes = "%d x %s" % (len([1 for _, l in bounds if l == inputs.BUCKET_ELEMS]),
                             "6,553,600")
        if bounds[-1][1] != inputs.BUCKET_ELEMS:
            sizes += " + {:,}".format(bounds[-1][1])
        cfg = {"workload": "flat fp32 gradient {:,} elements in 25 MiB buckets ({}), Student-t "
                           "nu=3 x 1e-3, correlated steps; per bucket EF + Top-K {:g}% + 8-bit "
                           "QSGD (groups of 64, stochastic) on the kept values".format(
                               n, sizes, args.ratio / 10),
               "total_elems": n, "bucket_elems": inputs.BUCKET_ELEMS,
               "buckets": len(bounds), "topk_per_mille": args.ratio,
               "quant": "qsgd 8-bit g64 stochastic", "path": args.path}
        if args.diag:
            cfg["diagnostics"] = "per-bucket sum c^2, sum g_hat^2, sum e'^2 fused into the passes"
        if args.path == "buckets":
            cfg["residual"] = ("deferred: each step's kept-entry residuals are applied by the "
                               "next step's read of e; the last step's are flushed into e inside "
                               "the timed region" if args.residual == "deferred" else
                               "immediate: every step stores its kept-entry residuals into e")
    cfg["l2"] = l2["l2"].format(4 * n >> 20)
    cfg["parallelism"] = l2["parallelism"]
    if wl is not None:
        cfg["streams"] = len(wl.streams)
        cfg["distinct_gradients"] = len(wl.grads)
    return cfg


# ---------------------------------------------------------------------------
def run_reference(args):
    """The reference arm: the oracle (single-threaded C, the pages'
    definitions), each step one bounded sample of the workload."""
    rank = dist_env()[1]
    if rank != 0:
        return 0
    run, n, what = cpu_sample(args, seed=11)
    times = []
    for t in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        if t >= args.warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    value = 4.0 * n / sec / 1e9
    sample = what + ", single-threaded C oracle, one sample per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config(args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    host_cpus = pin_host_near_gpu(torch, dev)
    from gradient_compression_ef_gb300 import gc

    if args.workload in ("buckets", "layers", "topk"):
        wl = BucketWorkload(torch, gc, dev, args.ratio, args.streams, args.distinct,
                            seed=rank_seed(rank), path=args.path, n=args.elems, diag=args.diag,
                            residual=args.residual,
                            layers=args.layers if args.workload == "layers" else None,
                            quant=args.workload != "topk")
    else:
        wl = WORKLOADS[args.workload](torch, gc, dev, args, seed=rank_seed(rank))
    torch.cuda.synchronize(dev)
    for t in range(args.warmup):
        wl.launch_step(t)
    wl.check()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    def timed(run_step, steps, side_streams=()):
        barrier()
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(wl.main)
        for s_ in side_streams:
            s_.wait_event(start)
        for t in range(steps):
            run_step(t)
        wl.finish()  # inside the timed region
        stop.record(wl.main)
        torch.cuda.synchronize(dev)
        barrier()
        ms_ = max_over_ranks(torch, start.elapsed_time(stop), world, dev)
        return ms_ / steps

    props = torch.cuda.get_device_properties(dev)
    pci = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0),
                                 getattr(props, "pci_bus_id", 0),
                                 getattr(props, "pci_device_id", 0))
    sampler = ClockSampler(pci)

    # eager launches through the C ABI
    launches0 = wl.launches()
    eager_ms = timed(lambda t: wl.launch_step(args.warmup + t), args.steps)
    eager_launches = wl.launches() - launches0
    wl.check()
    # CUDA-graph replay of whole steps (the same kernels, launched by the graph)
    graphs, per_step_launches = wl.capture()
    for t in range(args.warmup):
        graphs[t % len(graphs)].replay()
    wl.check()
    with sampler:
        graph_ms = timed(lambda t: graphs[t % len(graphs)].replay(), args.steps)
    wl.check()
    if args.eager:
        ms_per_step, launches, launch_mode = eager_ms, eager_launches, "eager"
    else:
        ms_per_step, launch_mode = graph_ms, "cuda_graph"
        launches = per_step_launches * args.steps + (1 if getattr(wl, "deferred", False) else 0)
    value = whole_job_value(world, wl.n, ms_per_step)
    eager_value = whole_job_value(world, wl.n, eager_ms)

    # per-kernel durations (second pass over the same kind of steps)
    phases = kernel_timing(wl, args.steps, args.warmup + args.steps, per_step_launches)
    # dominant kernel: the largest total time among kernels that move
    # gradient bytes (the selection passes in between move almost none)
    algo = wl.algorithmic_bytes_per_launch()
    top = max(((k_, v) for k_, v in phases.items() if algo.get(k_)), key=lambda kv: kv[1][0])
    peak, peak_src = measured_peaks()
    kernels = {}
    for name, (ms_, cnt) in phases.items():
        avg_s = ms_ / cnt * 1e-3
        kernels[name] = {"launches": cnt, "total_ms": ms_, "avg_us": avg_s * 1e6,
                         "algorithmic_bytes_per_launch": algo.get(name),
                         "achieved_gbs": algo[name] / avg_s / 1e9 if algo.get(name) else None}
    # elements of one launch of the dominant kernel: the whole gradient for
    # the bucketed passes, one matrix on average for PowerSGD
    launch_elems = wl.n / len(wl.shapes) if hasattr(wl, "shapes") else wl.n
    traffic, traffic_src = kernel_traffic(args.workload, top[0], launch_elems) \
        if args.path == "buckets" else (None, "no ncu capture")
    roofline = {"bound": "hbm", "kernel": top[0], "achieved": kernels[top[0]]["achieved_gbs"],
                "peak": peak, "unit": "GB/s", "peak_source": peak_src,
                "frac": kernels[top[0]]["achieved_gbs"] / peak, "traffic": traffic,
                "traffic_source": traffic_src,
                "frac_of_nominal": kernels[top[0]]["achieved_gbs"] / NOMINAL_HBM_GBS}
    step_achieved = wl.algorithmic_bytes() / (ms_per_step * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: every step copies its
    # gradient from pinned host memory (overlapped with the previous step on a
    # copy stream) and reads the compressed result back
    e2e = None
    if not args.no_e2e:
        T = len(wl.grads)
        # one pinned host copy per distinct gradient; above 8 GB of gradient
        # one host buffer serves every step (the bytes copied are the same)
        nh = T if 4 * wl.n * T <= (8 << 30) else 1
        hosts = []
        for g in wl.grads[:nh]:
            h_ = torch.empty(g.numel(), dtype=g.dtype, pin_memory=True)
            h_.copy_(g)
            hosts.append(h_)
        outs_h = [torch.empty(t.numel(), dtype=t.dtype).pin_memory() for t in wl.outputs()]
        copy_s = torch.cuda.Stream(device=dev)
        ready = [torch.cuda.Event() for _ in range(T)]
        done = [torch.cuda.Event() for _ in range(T)]
        e2e_steps = max(3, min(args.steps, 30))

        def e2e_step(t):
            d = t % T
            if t >= T:
                copy_s.wait_event(done[d])
            with torch.cuda.stream(copy_s):
                wl.grads[d].copy_(hosts[d % nh], non_blocking=True)
            ready[d].record(copy_s)
            wl.main.wait_event(ready[d])
            if args.eager:
                wl.launch_step(d)
            else:
                graphs[d].replay()
            done[d].record(wl.main)
            for h_, t_ in zip(outs_h, wl.outputs()):
                h_.copy_(t_.view(-1), non_blocking=True)

        e_ms = timed(e2e_step, e2e_steps, side_streams=(copy_s,))
        h2d = wl.input_bytes() if hasattr(wl, "input_bytes") else 4 * wl.n
        e2e = {"value": whole_job_value(world, wl.n, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": wl.out_bytes(),
               "ms_per_step": e_ms, "launch": launch_mode,
               "host_cpus": host_cpus if host_cpus else "affinity unchanged"}
        wl.check()

    if args.workload == "demo":
        # the demo prints the residual's energy after each step
        energies = []
        wl.launch_step(0, energies=energies)
        wl.check()
        roofline["note"] = ("the demo's 4 MB arrays stay in the 129 MB L2: the HBM roofline does "
                            "not bound it; reported, not claimed")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config(args, wl), "roofline": roofline,
            "step_roofline": {"algorithmic_bytes_per_step": wl.algorithmic_bytes(),
                              "achieved": step_achieved, "peak": peak, "unit": "GB/s",
                              "frac": step_achieved / peak},
            "kernels": kernels,
            "e2e": e2e, "clocks": sampler.summary(), "gpu_launches": launches,
            "launch": launch_mode, "eager": {"value": eager_value, "ms_per_step": eager_ms}}
    if args.workload == "demo":
        line["demo"] = {"error_energy_after_step1": energies[0],
                        "error_energy_after_step2": energies[1]}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
