#!/usr/bin/env python3
"""Benchmark of the fused randomized-Hadamard + bitshift-trellis GEMV.

Metric: fused trellis GEMV weights/s (and effective HBM GB/s, and the
fraction of the roofline) at batch 1.

Default workload: the Llama-3-8B-shaped decoder layer set -- q/o 4096x4096,
k/v 1024x4096, gate/up 14336x4096, down 4096x14336, each at K = 2, 3, 4 with
both computed codes (1MAD, 3INST): 42 GEMVs, 1.309 G weights and 490 MB of
packed codes per step, all resident in HBM.  A step runs every GEMV once, each
on its own x.  The step is captured once in a CUDA graph and replayed; the
490 MB working set is larger than L2, so every weight is re-read from HBM.

Other workloads (--workload): single (4096x4096 K2 1MAD), llama70b (32 layers
of Llama-3-70B shapes, K2 3INST, 6.85 GB packed), mixed (80-layer 2.9 bpw stack
+ K6 lm_head, 25 GB packed), sweep (14336x4096 and 4096x14336 K3 1MAD at a
batch given by --batch).

Roofline: per launch T_roof = max(packed+vector bytes / HBM bandwidth,
decode integer ops / INT32 peak), integer ops per weight 4 (3INST: window
funnel + mask, LCG multiply-add, mask/XOR; MCG the same with a multiply), 5
(1MAD: window funnel + mask, LCG, byte sum, int-to-float) or 6 (mul1: as 1MAD
plus the six-bit byte mask).  The HBM bandwidth is the measured copy bandwidth
of this GPU model; the INT32 peak is SMs x 128 integer lanes per clock (4
schedulers x 32 lanes) x the maximum SM clock.

--impl reference times the CPU oracle (test infrastructure) on a bounded
sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

# The oracle's float64 matmuls run single-threaded so the CPU figure states its
# thread count honestly.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from trellis_decode_gemv_gb300 import synth  # noqa: E402

METRIC = "fused trellis GEMV weights/s & effective HBM GB/s, batch 1, % of roofline"
L2_BYTES = 129 * 1024 * 1024
MAX_GROUP = 64  # layers per grouped call (EXL3_MAX_GROUP in include/exl3.h)
SM_COUNT_NOMINAL = 152
SM_MAX_MHZ_NOMINAL = 2070.0
INT_LANES_PER_SM_CLK = 128
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
# MCG: as 3INST (a multiply instead of the multiply-add); mul1: as 1MAD plus
# the six-bit byte mask
OPS_PER_WEIGHT = {synth.CB_3INST: 4, synth.CB_1MAD: 5, synth.CB_MCG: 4, synth.CB_MUL1: 6}
# the int8-activation path: window, generator, (mul1: six-bit mask), one dp4a
# that both sums the bytes and multiplies by the activation
OPS_PER_WEIGHT_INT8 = {synth.CB_1MAD: 3, synth.CB_MUL1: 4}
# DRAM traffic / algorithmic bytes of the dominant kernel, from the ncu
# captures of those kernels (dram__bytes_read.sum +
# dram__bytes_write.sum of the captured launches over their algorithmic bytes).
TRAFFIC_RATIO = {
    # DRAM reads + writes against the algorithmic bytes of one grouped launch
    # over the 7 Llama-3-8B projections (218 M weights): (54.881 + 0.029) /
    # 54.940 MB at K2 3INST, (109.415 + 3.208) / 109.466 MB at K4 1MAD (x and
    # the signs come from L2; the writes are the fp32 row-sum atomics)
    "shuffle": ((54.881 + 0.029) / 54.940, "the ncu capture of layer_kernel (32-tile sub-units) on one grouped "
                                           "call over the 7 Llama-3-8B projections, K2 3INST"),
    "tensor": (23.12 / 22.15, "the ncu capture of tc_layer_kernel on 14336x4096 K3 1MAD at batch 16"),
    "dense": (None, None),
    # DRAM reads 26.0 + 26.6 MB against 2 x 23.86 MB of algorithmic bytes; the
    # packed codes are most of both, so the ratio holds for tiles up to 128 rows
    "mv": (22.830 / 22.655, "the ncu capture of mv_kernel on 4096x14336 K3 1MAD at batch 16"),
    "fused": ((26.0 + 26.6) / (2 * 23.86),
              "the ncu capture of the fused dense_kernel (128-row tiles) on 14336x4096 and 4096x14336 K3 1MAD "
              "at batch 48"),
    # the int8-activation layer kernel on the same call at K2 1MAD:
    # (54.889 + 0.029) / 54.940 MB
    "int8": ((54.889 + 0.029) / 54.940, "the ncu capture of i8_kernel (32-tile sub-units) on one grouped "
                                        "int8-activation call over the 7 Llama-3-8B projections, K2 1MAD"),
    # the one-K kernels (classes of one K in one launch) over the 7 projections
    # at two codes of K2, 436 M weights: reads + writes against 109.88 MB
    "kset": ((109.782 + 3.208) / 109.879, "the ncu capture of layer_kernel_kset<2> on one multi-code call over "
                                          "the 7 Llama-3-8B projections at 3INST and 1MAD"),
    "int8kset": ((109.791 + 3.569) / 109.879, "the ncu capture of i8_kernel_kset<2> on one multi-code call over "
                                              "the 7 Llama-3-8B projections at 1MAD and mul1"),
}


def measured_peaks():
    """(HBM GB/s, max SM MHz, dense bf16 TFLOP/s burst, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL)),
                float(d.get("bf16_tflops", BF16_FALLBACK_TFLOPS)), "measured")
    except Exception:
        return HBM_FALLBACK_GBS, SM_MAX_MHZ_NOMINAL, BF16_FALLBACK_TFLOPS, "fallback"


def workload(name: str, batch: int):
    if name == "llama8b":
        desc = ("Llama-3-8B-shaped layer set at batch 1: q/o 4096x4096, k/v 1024x4096, "
                "gate/up 14336x4096, down 4096x14336, each at K=2,3,4 x {1MAD,3INST}")
        return desc, 1, synth.llama8b_layer_set(), 1
    if name == "llama8b-mcg-mul1":
        desc = ("Llama-3-8B-shaped layer set at batch 1 with the MCG and mul1 codes: q/o 4096x4096, "
                "k/v 1024x4096, gate/up 14336x4096, down 4096x14336, each at K=2,3,4")
        return desc, 5, synth.llama8b_layer_set((synth.CB_MCG, synth.CB_MUL1)), 1
    if name == "prefill":
        M = batch if batch > 32 else 512
        return (f"14336x4096 and 4096x14336, K=3, 1MAD, prefill batch {M}, 4 distinct instances of each"), 6, \
            synth.BATCH_SWEEP_SHAPES * 4, M
    if name == "single":
        # 32 distinct 4096x4096 layers (128 MB of codes) so that the timed
        # steps stream from HBM rather than L2
        return ("4096x4096 layer, K=2, 1MAD, batch 1, 32 distinct instances per step"), 0, \
            synth.SINGLE_4096 * 32, 1
    if name == "llama70b":
        return ("Llama-3-70B-shaped layers (q/o 8192x8192, k/v 1024x8192, gate/up 28672x8192, "
                "down 8192x28672) x 32 layers resident, K=2, 3INST, batch 1"), 2, synth.llama70b_stack(), 1
    if name == "mixed":
        return ("80-layer mixed-width stack (attn 8192x8192 K4; MLP 28672x8192 / 8192x28672, "
                "K in {2,3,4}, 2.90 bpw body) + lm_head 128256x8192 K6, 3INST, batch 1"), 4, synth.mixed_stack(), 1
    if name in ("int8", "mad-mul1"):
        how = ("int8 activations (exl3_gemm_int8act: rotation + per-128-block int8 quantization, "
               "one dp4a per weight)") if name == "int8" else "binary16 activations (the fused layer)"
        return (f"Llama-3-8B-shaped layer set with the byte-sum codes 1MAD and mul1 at K=2,3,4, {how}, "
                f"batch {batch}"), 9, synth.llama8b_layer_set((synth.CB_1MAD, synth.CB_MUL1)), batch
    if name == "whole":
        # QTIP's whole-vector rotations need power-of-two dimensions: the
        # attention projections of a Llama-3-70B-shaped model, 8 layers
        # resident (1.21 G weights, 302 MB of codes at K=2, more than L2)
        return (f"Llama-3-70B attention shapes (q/o 8192x8192, k/v 1024x8192) x 8 layers, K=2, 3INST, "
                f"whole-vector rotations on both sides, batch {batch}"), 7, synth.whole_attention_stack(), batch
    if name == "sweep":
        # four distinct instances of each shape (176 MB of codes, more than L2)
        return (f"14336x4096 and 4096x14336, K=3, 1MAD, batch {batch}, 4 distinct instances of each"), 3, \
            synth.BATCH_SWEEP_SHAPES * 4, batch
    raise SystemExit(f"unknown workload {name}")


def uses_shuffle(path: str, M: int) -> bool:
    """The kernel family of a call of M <= 32 rows (exl3_set_path): the
    warp-shuffle kernels at M <= 2 under AUTO, the decode-MMA kernel above."""
    return path == "shuffle" or (path == "auto" and M <= 2)


def kernels_per_call(path: str, M: int, m: int, n: int, sms: int) -> int:
    """Kernel launches of one exl3_gemm_small call.  Decode-MMA kernel (every
    path but the warp-shuffle one): one launch at M <= 2, plus the
    operand-image kernel above.  Warp-shuffle path, per batch chunk of 8, 4, 2
    or 1 rows: layer kernel and output kernel, plus the x-pair kernel when the
    chunk runs the sub-unit kernel (chunks above 2 rows, or at least 1024
    tiles per SM)."""
    if M > 32:
        from trellis_decode_gemv_gb300 import binding as B
        return B.exl3_gemm_launches(m, n, M)
    if not uses_shuffle(path, M):
        return 1 if M <= 2 else 2
    tiles_per_sm = (m // 16) * (n // 16) // sms
    launches, rem = 0, M
    for c in (8, 4, 2, 1):
        while rem >= c:
            rem -= c
            launches += 3 if (c > 2 or tiles_per_sm >= 1024) else 2
    return launches


def multi_layer_launches(mb: int, classes: dict, sms: int) -> int:
    """Sub-unit kernel launches of one batch chunk of an exl3_gemm_multi call:
    one per (K, code) class, except at chunks of one row, where the classes of
    one K whose tiles give every SM at least 2048 (32-tile sub-units) share
    one launch."""
    if mb != 1:
        return len(classes)
    by_k = {}
    for (K, _cb), shs in classes.items():
        by_k.setdefault(K, []).append(sum((m // 16) * (n // 16) for m, n in shs))
    n = 0
    for tiles in by_k.values():
        n += 1 if (len(tiles) > 1 and sum(tiles) // sms >= 2048) else len(tiles)
    return n


def int8_chunks(M: int) -> int:
    """Layer-kernel launches of one int8-activation call: one per batch chunk
    of 8, 4, 2 or 1 rows (plus the preparation and output kernels)."""
    n, rem = 0, M
    for c in (8, 4, 2, 1):
        while rem >= c:
            rem -= c
            n += 1
    return n


def decoder_groups(gemvs, grouped: bool = True):
    """Calls of one step: lists of GEMV indices.  A decoder applies q, k and v
    (and gate and up) to the same step, so consecutive projections of one of
    those families that share K and the code go into one exl3_gemm_grouped
    call; everything else is one exl3_gemm_small call."""
    def base(name):
        parts = name.split(".")
        return parts[1] if parts[0].startswith("L") and len(parts) > 1 else parts[0]

    families = ({"q", "k", "v"}, {"gate", "up"})
    out, i = [], 0
    while i < len(gemvs):
        fam = next((f for f in families if base(gemvs[i][0]) in f), None) if grouped else None
        j = i + 1
        if fam is not None:
            seen = {base(gemvs[i][0])}
            while (j < len(gemvs) and base(gemvs[j][0]) in fam and base(gemvs[j][0]) not in seen
                   and gemvs[j][3] == gemvs[i][3] and gemvs[j][4] == gemvs[i][4]):
                seen.add(base(gemvs[j][0]))
                j += 1
        out.append(list(range(i, j)))
        i = j
    return out


def class_groups(gemvs, max_group: int):
    """Calls of one step when every GEMV of the step that shares K and the code
    goes into one exl3_gemm_grouped call (at most max_group layers each): the
    GEMVs of a step are independent, each on its own x, so one kernel chain
    serves a whole class."""
    order, by = [], {}
    for i, g in enumerate(gemvs):
        key = (g[3], g[4])
        if key not in by:
            by[key] = []
            order.append(key)
        by[key].append(i)
    out = []
    for key in order:
        idx = by[key]
        out += [idx[s:s + max_group] for s in range(0, len(idx), max_group)]
    return out


def step_groups(gemvs, max_group: int):
    """Calls of one step when every GEMV of the step goes into exl3_gemm_multi
    calls of at most max_group layers (mixed K and code)."""
    idx = list(range(len(gemvs)))
    return [idx[s:s + max_group] for s in range(0, len(idx), max_group)]


GROUPING_CALLS = {
    "step": "every GEMV of the step in multi-code calls of up to 64 layers (mixed K and code: one input "
            "kernel, a layer kernel per (K, code) class, at batch 1 one per K, one output kernel)",
    "class": "every GEMV of the step that shares K and the code in one grouped call",
    "decoder": "q/k/v and gate/up grouped per call (the projections a decoder applies to one step), "
               "the rest one call each",
    "none": "one call per GEMV",
}


def kernels_per_group(path: str, M: int, shapes, sms: int) -> int:
    """Kernel launches of one grouped call over layers of the given (m, n):
    one decode-MMA launch over every layer (after one operand-image launch for
    every layer above batch 2); on the warp-shuffle path three per batch chunk
    (x pairs, one sub-unit kernel over every layer, output transform)."""
    if len(shapes) == 1:
        return kernels_per_call(path, M, shapes[0][0], shapes[0][1], sms)
    if not uses_shuffle(path, M):
        return 1 if M <= 2 else 2  # one operand-image launch for every layer, one decode-MMA launch
    chunks, rem = 0, M
    for c in (8, 4, 2, 1):
        while rem >= c:
            rem -= c
            chunks += 1
    return 3 * chunks


def algorithmic(m, n, K, cb, M, path="auto", int8=False):
    """Weights, algorithmic bytes and decode integer ops of one call; above 32
    batch rows the dense prefill decodes every tile once per call, the
    tensor-memory passes once per 128-row pass."""
    weights = m * n
    nbytes = m * n * K // 8 + 2 * m + 2 * (m + n) + 2 * M * n + 2 * M * m
    passes = (M + 127) // 128 if (M > 32 and path == "tensor") else 1
    ops = weights * (OPS_PER_WEIGHT_INT8 if int8 else OPS_PER_WEIGHT)[cb] * passes
    return weights, nbytes, ops


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of the SM clock, power and throttle reasons every
    50 ms while the benchmark runs; statistics over the samples taken since
    the last mark (one timed region) or over the whole run."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.proc = None
        self.bus_id = bus_id
        self.path = None
        self._mark = 0

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50", "-f", self.path]
            if self.bus_id:
                cmd[1:1] = ["-i", self.bus_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            # nvidia-smi takes a moment to start: wait (at most 10 s) for its
            # first samples, so that the first timed region is covered
            t0 = time.time()
            while len(self._rows()) < 2 and time.time() - t0 < 10.0 and self.proc.poll() is None:
                time.sleep(0.05)
        except Exception:
            self.proc = None

    def _rows(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        except Exception:
            pass
        return rows

    @staticmethod
    def _stats(rows):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": len(rows)}
        if not rows:
            out["reasons"] = ["unsampled"]
            return out
        num = lambda v: v.replace(".", "").isdigit()  # noqa: E731
        sm = [float(r[0]) for r in rows if num(r[0])]
        mx = [float(r[1]) for r in rows if num(r[1])]
        pw = [float(r[2]) for r in rows if num(r[2])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        out.update(sm_mhz=float(np.median(sm)) if sm else None, sm_max_mhz=max(mx) if mx else None,
                   reasons=sorted(reasons), power_w_max=max(pw) if pw else None)
        return out

    def mark(self):
        # the last sample before the region counts too: regions shorter than
        # the 50 ms sampling interval still get the samples around them
        if self.proc is not None:
            self._mark = max(0, len(self._rows()) - 1)

    def since_mark(self):
        if self.proc is None:
            return self._stats([])
        time.sleep(0.12)  # the sample covering the region's end
        return self._stats(self._rows()[self._mark:])

    def stop(self):
        if self.proc is None:
            return self._stats([])
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        rows = self._rows()
        try:
            os.unlink(self.path)
        except Exception:
            pass
        return self._stats(rows)


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_timed(gemvs, M, cfg, sel, blocks=1, target_s=None, whole=False, cache=None):
    """Time only the oracle (input generation excluded) on `blocks` 128-row
    output blocks of each selected GEMV.  With target_s, a one-block pass
    calibrates and a second pass takes as many blocks as fill about target_s
    seconds; both passes count.  With whole, the whole-vector layer of each
    selected GEMV instead (its output transform mixes every row).  `cache`
    (a dict) keeps the generated inputs of each GEMV for later calls."""
    from oracle import exl3_oracle as O
    inputs = []
    for i in sel:
        name, m, n, K, cb = gemvs[i]
        if cache is not None and i in cache:
            inp = cache[i]
        else:
            inp = synth.layer_inputs(m, n, K, M, config=cfg, index=i)
            if cache is not None:
                cache[i] = inp
        inputs.append((inp, gemvs[i], i))

    def one_pass(nblk, first):
        w = 0
        t0 = time.perf_counter()
        for inp, (name, m, n, K, cb), i in inputs:
            if whole:
                O.layer_forward_whole(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"],
                                      inp["x"])
                w += m * n * M
                continue
            nb = m // 128
            rbs = sorted({(i + first + 7 * j) % nb for j in range(nblk)})
            O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"],
                                      inp["scales"], inp["x"], rbs)
            w += 128 * len(rbs) * n * M
        return w, time.perf_counter() - t0

    weights, dt = one_pass(blocks, 0)
    if target_s is not None and dt < target_s and not whole:
        more = max(1, int((target_s - dt) / dt))
        w2, dt2 = one_pass(more, 1)
        weights, dt = weights + w2, dt + dt2
    return weights, dt


# ---------------------------------------------------------------------------
# multi-rank host logic (one replica per GPU; no collective on the data path)
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself when
    no process group runs."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def whole_job_rate(units_per_rank_step: float, world: int, steps: int, seconds: float) -> float:
    """Units per second of the whole job: every rank processes its own
    units_per_rank_step per step (weak scaling); seconds is the slowest rank's
    time for `steps` steps."""
    return units_per_rank_step * world * steps / seconds


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # the default run's headline is the Llama-3-8B layer set
    wl = "llama8b" if args.workload == "all" else args.workload
    desc, cfg, gemvs, M = workload(wl, args.batch)
    whole = wl == "whole"
    # the GPU arm's grouping for this workload (its line's `config`)
    ref_grouping = resolve_grouping(args.grouping, M, whole)
    per_step = 1 if whole else min(6, len(gemvs))
    # the whole-vector oracle runs full layers: take the smallest GEMVs
    pool = [i for i, g in enumerate(gemvs) if g[1] * g[2] == min(h[1] * h[2] for h in gemvs)] if whole \
        else list(range(len(gemvs)))
    # every GEMV's inputs are generated once (outside the timed oracle calls)
    cache = {}
    if not whole:
        # 128-row blocks per step: up to 6, fewer when the run has many steps,
        # so that the oracle's time stays near a minute and a half on this host
        # (one untimed step of 6 blocks gives the time of a block)
        _w, dt = oracle_sample_timed(gemvs, M, cfg, pool[:per_step], whole=False, cache=cache)
        per_block = max(dt / per_step, 1e-4)
        per_step = max(1, min(per_step, int(90.0 / (max(args.steps + args.warmup, 1) * per_block))))
    for s in range(args.warmup):
        oracle_sample_timed(gemvs, M, cfg, [pool[(s * per_step + i) % len(pool)] for i in range(per_step)],
                            whole=whole, cache=cache)
    tw, tt = 0, 0.0
    for s in range(args.steps):
        sel = [pool[((args.warmup + s) * per_step + i) % len(pool)] for i in range(per_step)]
        w, dt = oracle_sample_timed(gemvs, M, cfg, sel, whole=whole, cache=cache)
        tw += w
        tt += dt
    value = tw / tt
    sample = (f"per step: one 128-row output block of {per_step} of the {len(gemvs)} GEMVs "
              f"(round-robin), oracle layer forward (decode + float64 product + transforms)") if not whole else \
        (f"per step: one of the smallest GEMVs of the workload in full (round-robin), oracle whole-vector "
         f"layer forward")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "weights/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tt / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(args, desc, gemvs, M, ref_grouping,
                              groups_of([(g[0], g[1], g[2], g[3], g[4]) for g in gemvs], ref_grouping, MAX_GROUP),
                              args.path),
        "cpu_baseline": {"value": value, "unit": "weights/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "weights/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def int_peak_probe(B, torch, dev, stream, sms, clocks_mhz):
    """The integer-throughput probe (exl3_probe_int): ops per clock per SM of
    each instruction kind and of the two mixes, timed with CUDA events on the
    stream; the measured INT32 peak is the best mix in ops/s."""
    blocks, iters = 8 * sms, 256
    out = torch.empty(blocks * 256, dtype=torch.int32, device=dev)
    res = {}
    with torch.cuda.stream(stream):
        for kind in sorted(B.PROBE_KINDS):
            B.exl3_probe_int(kind, out, blocks, iters)  # warm-up
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 5
            e0.record(stream)
            for _ in range(reps):
                ops = B.exl3_probe_int(kind, out, blocks, iters)
            e1.record(stream)
            stream.synchronize()
            sec = e0.elapsed_time(e1) * 1e-3
            rate = ops * reps / sec
            res[B.PROBE_KINDS[kind]] = {"ops_per_s": rate, "ops_per_clk_sm": rate / (sms * clocks_mhz * 1e6)}
    best = max(("IMAD+LOP3", "IMAD+IDP4A+LOP3+SHF"), key=lambda k: res[k]["ops_per_s"])
    return {"kinds": res, "peak_ops_per_s": res[best]["ops_per_s"], "peak_kind": best,
            "clock_mhz_assumed": clocks_mhz,
            "how": (f"exl3_probe_int: {blocks} CTAs x 256 threads x 8 independent chains x {4 * iters} "
                    "instructions, 5 launches per kind, CUDA events; ops/clk/SM at the stated clock")}


def launches_of_group(B, path, M, shapes, sms, whole, int8, kcs=None):
    """Kernel launches of one call of the step (a single layer or a group)."""
    if whole:
        if len(shapes) == 1:
            return B.exl3_gemm_launches(shapes[0][0], shapes[0][1], M) + 2
        return kernels_per_group(path, M, shapes, sms) + 2
    if int8:  # one activation kernel, the layer kernels of each batch chunk, one output kernel
        if kcs is None:
            return 2 + int8_chunks(M)
        classes = {}
        for sh, kc in zip(shapes, kcs):
            classes.setdefault(kc, []).append(sh)
        total, rem = 2, M
        for c in (8, 4, 2, 1):
            while rem >= c:
                rem -= c
                total += multi_layer_launches(c, classes, sms)
        return total
    if kcs is not None and len(shapes) > 1:  # exl3_gemm_multi: one chain per batch chunk
        classes = {}
        for sh, kc in zip(shapes, kcs):
            classes.setdefault(kc, []).append(sh)
        if uses_shuffle(path, M):
            total, rem = 0, M
            for c in (8, 4, 2, 1):
                while rem >= c:
                    rem -= c
                    total += 2 + multi_layer_launches(c, classes, sms)
            return total
        return sum(1 if M <= 2 else 2 for shs in classes.values())
    return kernels_per_group(path, M, shapes, sms)


def resolve_grouping(grouping, M, whole):
    """The grouping a workload's step runs with: grouped calls take at most 32
    batch rows, and the whole-vector variant has no multi-code call."""
    if M > 32:
        return "none"
    if grouping == "step" and whole:
        return "class"
    return grouping


def groups_of(shapes_kc, grouping, max_group):
    if grouping == "step":
        return step_groups(shapes_kc, max_group)
    if grouping == "class":
        return class_groups(shapes_kc, max_group)
    return decoder_groups(shapes_kc, grouped=grouping == "decoder")


def step_config(args, desc, gemvs, M, grouping, groups, path, cuda_graph=True):
    """The `config` of a workload's line: what the step computes and how it is
    called (the same for the GPU arm and the reference arm)."""
    whole, int8 = args_workload_kind(desc)
    alg = [algorithmic(m, n, K, cb, M, path, int8) for _, m, n, K, cb in gemvs]
    packed = sum(m * n * K // 8 for _, m, n, K, _ in gemvs)
    l2_note = (f"inputs larger than L2: {packed / 1e6:.0f} MB of packed codes per step "
               f"vs {L2_BYTES / 1e6:.0f} MB L2") if packed > L2_BYTES else "L2 NOT exceeded"
    return {"workload": desc, "gemvs_per_step": len(gemvs), "batch": M,
            "weights_per_step": sum(a[0] for a in alg), "packed_bytes_per_step": packed,
            "algorithmic_bytes_per_step": sum(a[1] for a in alg), "l2": l2_note,
            "cuda_graph": cuda_graph, "kernel_path": path, "prefill": args.prefill,
            "grouping": grouping,
            "calls": GROUPING_CALLS[grouping] + (
                " (exl3_gemm, prefill)" if M > 32 and not whole else
                " (exl3_gemm_whole_grouped / exl3_gemm_whole)" if whole else
                " (exl3_gemm_int8act_multi / exl3_gemm_int8act)" if int8 and grouping == "step" else
                " (exl3_gemm_int8act_grouped / exl3_gemm_int8act)" if int8 else
                " (exl3_gemm_multi / exl3_gemm_small)" if grouping == "step" else
                " (exl3_gemm_grouped / exl3_gemm_small)") + f"; {len(groups)} calls per step"}


def args_workload_kind(desc):
    """(whole-vector variant, int8 activations) of a workload, from its description."""
    return "whole-vector rotations" in desc, "int8 activations" in desc


def measure_workload(ctx, args, wl, batch, steps, warmup, want_e2e=True, want_cpu=False, grouping=None):
    """One workload: resident inputs, warm-up, graph capture, `steps` timed
    graph replays (CUDA events on the launch stream), per-call apportioning,
    roofline terms, the end-to-end leg and (optionally) the oracle baseline."""
    torch, B, dev, stream = ctx["torch"], ctx["B"], ctx["dev"], ctx["stream"]
    sms, world, rank = ctx["sms"], ctx["world"], ctx["rank"]
    hbm_gbs, bf16_tflops, peak_src, p_int = ctx["hbm_gbs"], ctx["bf16_tflops"], ctx["peak_src"], ctx["p_int"]
    desc, cfg, gemvs, M = workload(wl, batch)

    # ---- resident inputs ------------------------------------------------
    # Codes are uniform random words drawn on the device (torch's Philox
    # generator, seeded per tensor from the same seed table as the host
    # generator): tens of GB for the largest stacks.  Signs, scales and x come
    # from the host generator.
    total_n = sum(g[2] for g in gemvs) * M
    total_m = sum(g[1] for g in gemvs) * M
    X = torch.empty(total_n, dtype=torch.float16, device=dev)
    Y = torch.empty(total_m, dtype=torch.float16, device=dev)
    calls = []
    xo = yo = 0
    whole = wl == "whole"
    int8 = wl == "int8"
    ws_of = (B.exl3_gemm_whole_workspace_bytes if whole else B.exl3_gemm_i8_workspace_bytes if int8
             else B.exl3_gemm_workspace_bytes)
    ws_bytes = max(ws_of(m, n, M) for _, m, n, _, _ in gemvs)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    packed = 0
    gen = torch.Generator(device=dev)
    for i, (name, m, n, K, cb) in enumerate(gemvs):
        words = (m // 16) * (n // 16) * 8 * K
        gen.manual_seed(synth.seed_for(cfg, 10 * i) & ((1 << 63) - 1))
        codes = torch.randint(-(1 << 31), 1 << 31, (words,), generator=gen, device=dev, dtype=torch.int64).to(
            torch.int32)
        b = 10 * i
        s_in = torch.from_numpy(synth.sign_vector(n, synth.seed_for(cfg, b + 1))).to(dev)
        s_out = torch.from_numpy(synth.sign_vector(m, synth.seed_for(cfg, b + 2))).to(dev)
        scales = torch.from_numpy(synth.channel_scales(m, synth.seed_for(cfg, b + 3))).to(dev)
        X[xo:xo + M * n] = torch.from_numpy(synth.activations(M, n, synth.seed_for(cfg, b + 4)).reshape(-1)).to(dev)
        x = X[xo:xo + M * n].view(M, n)
        y = Y[yo:yo + M * m].view(M, m)
        calls.append(dict(name=name, m=m, n=n, K=K, cb=cb, codes=codes, s_in=s_in, s_out=s_out,
                          scales=scales, x=x, y=y))
        packed += codes.numel() * 4
        xo += M * n
        yo += M * m
    torch.cuda.synchronize(dev)

    grouping = resolve_grouping(grouping or args.grouping, M, whole)
    shapes_kc = [(c["name"], c["m"], c["n"], c["K"], c["cb"]) for c in calls]
    groups = groups_of(shapes_kc, grouping, MAX_GROUP)
    gws_of = (B.exl3_group_i8_workspace_bytes if int8 else B.exl3_gemm_whole_grouped_workspace_bytes if whole
              else B.exl3_group_workspace_bytes)
    gws = max([gws_of([(calls[i]["m"], calls[i]["n"]) for i in g], M)
               for g in groups if len(g) > 1] + [0])
    if gws > ws.numel():
        ws = torch.zeros(gws, dtype=torch.uint8, device=dev)

    def run_group(g):
        if len(g) == 1:
            c = calls[g[0]]
            fn = (B.exl3_gemm_whole if whole else B.exl3_gemm_int8act if int8 else B.exl3_gemm if M > 32
                  else B.exl3_gemm_small)
            fn(c["codes"], c["K"], c["cb"], c["m"], c["n"], c["s_in"], c["s_out"],
               c["scales"], c["x"], y=c["y"], workspace=ws)
        elif grouping == "step":
            (B.exl3_gemm_int8act_multi if int8 else B.exl3_gemm_multi)([calls[i] for i in g], workspace=ws)
        else:
            c0 = calls[g[0]]
            gfn = (B.exl3_gemm_int8act_grouped if int8 else B.exl3_gemm_whole_grouped if whole
                   else B.exl3_gemm_grouped)
            gfn([calls[i] for i in g], c0["K"], c0["cb"], workspace=ws)

    def step():
        for g in groups:
            run_group(g)

    # Decode work (weights, integer ops) does not grow with the batch; the
    # multiply-accumulates do (macs = weights * M).
    alg = [algorithmic(c["m"], c["n"], c["K"], c["cb"], M, args.path, int8) for c in calls]
    weights_step = sum(a[0] for a in alg)
    bytes_step = sum(a[1] for a in alg)
    ops_step = sum(a[2] for a in alg)

    # ---- warm-up + graph capture ----------------------------------------
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
    torch.cuda.synchronize(dev)
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        graph = g
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize(dev)
    except Exception as e:  # capture unsupported: time eager launches
        print(f"[bench] graph capture failed ({e}); timing eager launches", file=sys.stderr)
        graph = None

    def replay():
        if graph is not None:
            graph.replay()
        else:
            step()

    # ---- timed region: `steps` steps ----------------------------------------
    ctx["clocks"].mark()
    barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = ctx["clocks"].since_mark()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_step = ms_total / steps
    value = whole_job_rate(weights_step, world, steps, ms_total / 1e3)

    # ---- per-launch durations (events around every launch) ---------------
    nrep = max(3, min(steps, 20))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(groups) + 1)]
    gdur = np.zeros(len(groups))
    with torch.cuda.stream(stream):
        for r in range(nrep + 1):
            torch.cuda._sleep(int(2e6 + 4e4 * len(groups)))  # keep the queue ahead of the host
            evs[0].record(stream)
            for i, g in enumerate(groups):
                run_group(g)
                evs[i + 1].record(stream)
            torch.cuda.synchronize(dev)
            if r > 0:
                gdur += np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(len(groups))]) * 1e-3
    # a group's time is shared among its GEMVs in proportion to their weights
    dur = np.zeros(len(calls))
    for g, d in zip(groups, gdur):
        w = np.array([calls[i]["m"] * calls[i]["n"] for i in g], dtype=np.float64)
        dur[g] = d * w / w.sum()
    dur /= nrep
    # The eager per-call durations (events between calls) lose the overlap that
    # programmatic dependent launch gives inside the graph, so they only
    # apportion the graph-timed step time among the GEMVs.
    t_step = ms_step / 1e3
    t_call = dur * (t_step / dur.sum())
    t_hbm = np.array([a[1] / (hbm_gbs * 1e9) for a in alg])
    t_int = np.array([a[2] / p_int for a in alg])
    # tensor-core term: 2 M m n flops at the measured dense bf16 (= fp16) peak
    # (above 32 rows only: below, the MMAs' flops are far under the peak)
    flops_step = 2.0 * M * sum(c["m"] * c["n"] for c in calls) if (M > 32 and not int8) else 0.0
    p_tensor = bf16_tflops * 1e12
    t_tc = np.array([2.0 * M * c["m"] * c["n"] / p_tensor if (M > 32 and not int8) else 0.0 for c in calls])
    t_roof = np.maximum(np.maximum(t_hbm, t_int), t_tc)
    terms = {"alu": t_int.sum(), "hbm": t_hbm.sum(), "tensor": t_tc.sum()}
    bound = max(terms, key=terms.get)
    if bound == "alu":
        achieved, peak, unit = ops_step / t_step / 1e12, p_int / 1e12, "Tops/s"
    elif bound == "tensor":
        achieved, peak, unit = flops_step / t_step / 1e12, bf16_tflops, "TFLOP/s"
    else:
        achieved, peak, unit = bytes_step / t_step / 1e9, hbm_gbs, "GB/s"
    shuffle = uses_shuffle(args.path, M) and M <= 32
    dense = M > 32 and args.path != "tensor"
    passes = M > 32 and args.path == "tensor"
    fused = dense and (args.prefill == "fused" or (args.prefill == "auto" and M <= 256))
    # batch 1 with every GEMV of a step in multi-code calls: do classes of one K
    # share a launch (the one-K kernel)?
    kset = False
    if grouping == "step" and M == 1 and uses_shuffle(args.path, M):
        for g in groups:
            classes = {}
            for i in g:
                classes.setdefault((calls[i]["K"], calls[i]["cb"]), []).append((calls[i]["m"], calls[i]["n"]))
            kset = kset or multi_layer_launches(1, classes, sms) < len(classes)
    if int8:
        kname = ("i8_kernel (window, generator, one dp4a per weight into int32 tile sums) + activation "
                 "rotation/quantization and output kernels")
        tkey = "int8kset" if kset else "int8"
        if kset:
            kname = ("i8_kernel_kset (one launch per K over its byte-sum codes: window, generator, one dp4a per "
                     "weight into int32 tile sums) + activation rotation/quantization and output kernels")
    elif fused:
        kname = ("dense_kernel, fused (sixteen warps decode each stage's codes into the operand-A image in shared "
                 "memory; tcgen05 128xNx16 MMAs, N = 64/128/256 by batch) + operand-B kernel")
        tkey = "fused" if M <= 128 else "dense"
    elif dense:
        kname = ("dense_kernel (tcgen05 128xNx16 MMAs, N = 64/128/256 by batch, both operands in shared memory) + "
                 "decode-to-operand-image, operand-B and output kernels")
        tkey = "dense"
    elif passes:
        kname = "tc_layer_kernel (128-row passes: decoded tiles in TMEM -> tcgen05 MMAs) + operand and output kernels"
        tkey = "tensor"
    elif shuffle:
        kname = "layer_kernel / seg_layer_kernel (trellis decode + HFMA2 + warp shuffles) + x-pair and output kernels"
        tkey = "kset" if kset else "shuffle"
        if kset:
            kname = ("layer_kernel_kset (one launch per K over its codes: trellis decode + HFMA2 + warp shuffles) + "
                     "x-pair and output kernels")
    else:
        kname = ("mv_kernel (decode into TMEM, tcgen05 128xNx16 MMAs; input RHT by in-kernel x warps at M <= 2, "
                 "output RHT by the CTA completing each 128-row block)" + (" + operand-image kernel" if M > 2 else ""))
        tkey = "mv"
    ratio, ratio_src = TRAFFIC_RATIO[tkey]
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": None if ratio is None else ratio * bytes_step,
                "traffic_note": ("no ncu DRAM capture of this kernel yet" if ratio is None else
                                 f"bytes per step: algorithmic bytes x {ratio:.3f}, the DRAM/algorithmic "
                                 f"ratio of {ratio_src}"),
                "peak_source": (f"INT32: {sms} SMs x {INT_LANES_PER_SM_CLK} lanes/clk x "
                                f"{ctx['sm_max_mhz']:.0f} MHz (derived)") if bound == "alu"
                else (f"dense bf16 GEMM ({peak_src}; fp16 MMAs run at the same rate)" if bound == "tensor"
                      else f"HBM copy bandwidth ({peak_src})"),
                "kernel": kname,
                "timing": "algorithmic ops (bytes) per step / graph-timed step, CUDA events on the launch stream",
                "per_call_us_mean": 1e6 * t_step / len(groups),
                "eager_call_us_mean": 1e6 * dur.sum() / len(groups),
                "calls_per_step": len(groups)}
    if bound == "alu" and ctx.get("probe"):
        pm = ctx["probe"]["peak_ops_per_s"] / 1e12
        roofline.update(peak_measured=pm, frac_measured=achieved / pm,
                        peak_measured_source=f"exl3_probe_int, {ctx['probe']['peak_kind']} chains (measured)")
    hbm = {"achieved_gbs": bytes_step / t_step / 1e9, "peak_gbs": hbm_gbs, "peak_source": peak_src,
           "frac": bytes_step / t_step / 1e9 / hbm_gbs}
    roof_pct = 100.0 * t_roof.sum() / t_step

    # per-(K, code) summary
    per = {}
    for c, d, a, th, ti in zip(calls, t_call, alg, t_hbm, t_int):
        key = f"K{c['K']}.{synth.CODE_NAMES[c['cb']]}"
        e = per.setdefault(key, [0.0, 0, 0.0])
        e[0] += d
        e[1] += a[0]
        e[2] += max(th, ti)
    per_summary = {k: {"weights_per_s": v[1] / v[0], "roofline_pct": 100 * v[2] / v[0]}
                   for k, v in sorted(per.items())}

    # ---- e2e: host buffers, copies inside the timed region ---------------
    e2e = None
    if want_e2e:
        e2e = measure_e2e(ctx, calls, groups, M, ws, whole, int8, total_n, total_m, X, Y, weights_step, steps,
                          grouping)

    # ---- CPU oracle baseline (rank 0, N=1 only) --------------------------
    cpu = None
    if want_cpu and rank == 0 and world == 1 and not args.no_cpu_baseline:
        nsel = len(gemvs) if wl == "llama8b" else min(len(gemvs), 8)
        sel = list(range(nsel)) if nsel == len(gemvs) else list(range(0, len(gemvs), max(1, len(gemvs) // nsel)))[:nsel]
        if whole:  # full layers: the three smallest (k/v) GEMVs
            sel = sorted(range(len(gemvs)), key=lambda i: gemvs[i][1] * gemvs[i][2])[:3]
        w, dt = oracle_sample_timed(gemvs, M, cfg, sel, target_s=12.0, whole=whole)
        cpu = {"value": w / dt, "unit": "weights/s", "cores": 1, "kind": "oracle",
               "sample": (f"{len(sel)} whole GEMVs (the smallest of the workload; {w / 1e6:.1f} M weights, "
                          f"{dt:.1f} s), oracle whole-vector layer forward") if whole else
                         (f"128-row output blocks of each of {len(sel)} GEMVs of the workload "
                          f"({w / 1e6:.1f} M weights, {dt:.1f} s), oracle layer forward")}

    launches_step = sum(launches_of_group(B, args.path, M, [(calls[i]["m"], calls[i]["n"]) for i in g], sms,
                                          whole, int8,
                                          [(calls[i]["K"], calls[i]["cb"]) for i in g] if grouping == "step"
                                          else None) for g in groups)
    res = {
        "value": value, "unit": "weights/s", "steps": steps, "warmup": warmup, "ms_per_step": ms_step,
        "config": step_config(args, desc, gemvs, M, grouping, groups, args.path, cuda_graph=graph is not None),
        "effective_gbs": bytes_step * world / (ms_step / 1e3) / 1e9,
        "macs_per_s": value * M,
        "roofline_pct": roof_pct,
        "roofline": roofline, "hbm": hbm, "per_code": per_summary,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": steps * launches_step, "launches_per_step": launches_step,
        "clocks": clk,
    }
    del calls, X, Y, ws, graph
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def measure_e2e(ctx, calls, groups, M, ws, whole, int8, total_n, total_m, X, Y, weights_step, steps,
                grouping="class"):
    """The same workload through the binding's public per-layer objects,
    eager, with the step's x copied in from pinned host memory and y copied
    back inside the timed region."""
    torch, B, dev, stream, world = ctx["torch"], ctx["B"], ctx["dev"], ctx["stream"], ctx["world"]
    layer_objs = []
    for g in groups:
        if int8 and grouping == "step" and len(g) > 1:  # the mixed-code layer object
            layer_objs.append(B.Exl3LinearMulti([calls[i] for i in g], int8=True))
        elif int8 and len(g) > 1:  # the public calls themselves
            c0 = calls[g[0]]
            layer_objs.append(lambda g=g, c0=c0: B.exl3_gemm_int8act_grouped(
                [calls[i] for i in g], c0["K"], c0["cb"], workspace=ws))
        elif int8:
            c = calls[g[0]]
            layer_objs.append(lambda c=c: B.exl3_gemm_int8act(
                c["codes"], c["K"], c["cb"], c["m"], c["n"], c["s_in"], c["s_out"], c["scales"], c["x"],
                y=c["y"], workspace=ws))
        elif whole and len(g) > 1:  # no layer object for the whole-vector variant: the public calls
            c0 = calls[g[0]]
            layer_objs.append(lambda g=g, c0=c0: B.exl3_gemm_whole_grouped(
                [calls[i] for i in g], c0["K"], c0["cb"], workspace=ws))
        elif whole:
            c = calls[g[0]]
            layer_objs.append(lambda c=c: B.exl3_gemm_whole(
                c["codes"], c["K"], c["cb"], c["m"], c["n"], c["s_in"], c["s_out"], c["scales"], c["x"],
                y=c["y"], workspace=ws))
        elif grouping == "step" and len(g) > 1:  # the mixed-code layer object
            layer_objs.append(B.Exl3LinearMulti([calls[i] for i in g]))
        elif len(g) == 1:
            c = calls[g[0]]
            lin = B.Exl3Linear(c["codes"], c["K"], c["cb"], c["m"], c["n"], c["s_in"], c["s_out"],
                               c["scales"], max_batch=M)
            layer_objs.append(lambda lin=lin, c=c: lin(c["x"], c["y"]))
        else:
            c0 = calls[g[0]]
            grp = B.Exl3LinearGroup([calls[i] for i in g], c0["K"], c0["cb"])
            layer_objs.append(grp)

    def step_public():
        for f in layer_objs:
            f()

    Xh = torch.empty(total_n, dtype=torch.float16, pin_memory=True)
    Xh.copy_(X.cpu())
    Yh = torch.empty(total_m, dtype=torch.float16, pin_memory=True)
    e2e_steps = max(3, min(steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(2):
            X.copy_(Xh, non_blocking=True)
            step_public()
            Yh.copy_(Y, non_blocking=True)
        stream.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            X.copy_(Xh, non_blocking=True)
            step_public()
            Yh.copy_(Y, non_blocking=True)
            stream.synchronize()
        t_e2e = time.perf_counter() - t0
    t_e2e = max_over_ranks(t_e2e, dev)
    return {"value": whole_job_rate(weights_step, world, e2e_steps, t_e2e), "unit": "weights/s",
            "steps": e2e_steps, "h2d_bytes_per_step": total_n * 2, "d2h_bytes_per_step": total_m * 2,
            "path": ("binding layer objects (Exl3Linear / Exl3LinearGroup / Exl3LinearMulti), eager calls; "
                     "pinned host x -> "
                     "device, y -> pinned host, inside the timed region")}


# The configurations of the default run: the headline (the Llama-3-8B layer
# set at batch 1) first, then the other four, each timed with the same steps
# and warm-up.  C3 is the batch sweep on the two MLP shapes.
ALL_CONFIGS = [("C1", "llama8b", 1), ("C0", "single", 1), ("C2", "llama70b", 1)] + \
    [(f"C3.M{M}", "sweep", M) for M in synth.BATCH_SWEEP] + [("C4", "mixed", 1)]


def _summary(r):
    """The per-config record of the default run."""
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "effective_gbs", "macs_per_s", "roofline_pct",
            "gpu_launches", "launches_per_step")
    out = {k: r[k] for k in keep}
    out["workload"] = r["config"]["workload"]
    out["batch"] = r["config"]["batch"]
    out["weights_per_step"] = r["config"]["weights_per_step"]
    out["l2"] = r["config"]["l2"]
    ro = r["roofline"]
    out["roofline"] = {k: ro[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic") if k in ro}
    for k in ("peak_measured", "frac_measured"):
        if k in ro:
            out["roofline"][k] = ro[k]
    out["hbm_frac"] = r["hbm"]["frac"]
    out["e2e"] = None if r["e2e"] is None else {"value": r["e2e"]["value"], "unit": r["e2e"]["unit"]}
    out["per_code"] = r["per_code"]
    out["clocks"] = r["clocks"]
    out["grouping"] = r["config"]["grouping"]
    if "decoder_grouping" in r:
        out["decoder_grouping"] = r["decoder_grouping"]
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    from trellis_decode_gemv_gb300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    B.load_library()
    B.exl3_set_path({"auto": B.PATH_AUTO, "shuffle": B.PATH_SHUFFLE, "tensor": B.PATH_TENSOR}[args.path])
    B.exl3_set_prefill({"auto": B.PREFILL_AUTO, "fused": B.PREFILL_FUSED,
                        "decode_once": B.PREFILL_DECODE_ONCE}[args.prefill])
    hbm_gbs, sm_max_mhz, bf16_tflops, peak_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    bus = getattr(props, "pci_bus_id", None)
    clocks = ClockSampler(bus if isinstance(bus, str) else None)
    clocks.start()
    stream = torch.cuda.Stream(dev)
    ctx = dict(torch=torch, B=B, dev=dev, stream=stream, sms=sms, world=world, rank=rank, hbm_gbs=hbm_gbs,
               bf16_tflops=bf16_tflops, peak_src=peak_src, sm_max_mhz=sm_max_mhz,
               p_int=sms * INT_LANES_PER_SM_CLK * sm_max_mhz * 1e6, clocks=clocks)
    ctx["probe"] = int_peak_probe(B, torch, dev, stream, sms, sm_max_mhz)

    def with_decoder_grouping(res, wl, M):
        # the same workload with only the decoder's own groups (q/k/v,
        # gate/up): every other GEMV of the step waits for its predecessor
        if args.grouping not in ("step", "class") or M > 32 or wl in ("encode",):
            return res
        d = measure_workload(ctx, args, wl, M, min(args.steps, 300), args.warmup, want_e2e=False,
                             want_cpu=False, grouping="decoder")
        res["decoder_grouping"] = {"value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"],
                                   "roofline_frac": d["roofline"]["frac"], "calls": d["config"]["calls"],
                                   "steps": d["steps"]}
        return res

    if args.workload == "all":
        runs = {}
        for key, wl, M in ALL_CONFIGS:
            runs[key] = with_decoder_grouping(measure_workload(ctx, args, wl, M, args.steps, args.warmup,
                                                               want_e2e=True, want_cpu=(key == "C1")), wl, M)
        head = runs["C1"]
    else:
        head = with_decoder_grouping(measure_workload(ctx, args, args.workload, args.batch, args.steps,
                                                      args.warmup, want_e2e=True, want_cpu=True),
                                     args.workload, args.batch)
        runs = None
    clk_all = clocks.stop()
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "weights/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16",
            "arith": ("binary16 products of the weights and x-tilde, accumulated in binary16 over each tile row "
                      "(16 columns, HFMA2), fp32 beyond (warp-shuffle kernels, batch <= 2)")
                     if uses_shuffle(args.path, head["config"]["batch"]) else
                     ("binary16 weights x binary16 x-tilde on tcgen05 MMAs, fp32 accumulation in TMEM and fp32 "
                      "split-K reductions; y rounded once to binary16"),
            "data": "synthetic",
            "config": head["config"],
            "effective_gbs": head["effective_gbs"], "macs_per_s": head["macs_per_s"],
            "roofline_pct": head["roofline_pct"], "roofline": head["roofline"], "hbm": head["hbm"],
            "per_code": head["per_code"], "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "decoder_grouping": head.get("decoder_grouping"),
            "int_peak_probe": ctx["probe"],
            "clocks": clk_all,
        }
        if runs is not None:
            line["configs"] = {k: _summary(v) for k, v in runs.items()}
            line["configs_note"] = ("every config timed in this run with the same --steps/--warmup: C1 the "
                                    "headline (top-level fields), C0 single 4096x4096, C2 Llama-3-70B stack, "
                                    "C3 batch sweep M=1..32, C4 mixed 2.9 bpw stack + lm_head")
            line["gpu_launches_all_configs"] = sum(v["gpu_launches"] for v in runs.values())
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


ENCODE_METRIC = "tail-biting Viterbi encode, weights (trellis steps) encoded per second"
ENCODE_TILES = 1216  # 8 tiles per SM of a GB300


def code_rms(cb: int) -> float:
    """Closed-form rms value of a code's weights over uniform states.  The
    byte-sum codes are centred and scaled to unit variance by definition.  A
    three-instruction weight is the sum of two independent binary16 halves of
    random sign, biased exponent uniform in 12..15 and a uniform 10-bit
    mantissa: E[w^2] = 2 * (1/4) * sum_e 4^(e-15) * mean_k (1 + k/1024)^2."""
    if cb in (synth.CB_1MAD, synth.CB_MUL1):
        return 1.0
    k = np.arange(1024, dtype=np.float64)
    m2 = float(np.mean((1.0 + k / 1024.0) ** 2))
    return float(np.sqrt(2.0 * 0.25 * sum(4.0 ** (e - 15) for e in range(12, 16)) * m2))


def encode_inputs(K: int, cb: int, tiles: int):
    """Unit-Gaussian sequences scaled by the code's rms value (code units),
    binary32 [tiles][256], and that rms value."""
    sigma = code_rms(cb)
    g = synth.activations(tiles, 256, synth.seed_for(8, 0)).astype(np.float64)
    return (g * sigma).astype(np.float32), sigma


def encode_oracle_timed(target, K, cb, target_s):
    """The oracle's binary32 encoder on whole tiles until about target_s
    seconds; returns (tiles, seconds)."""
    from oracle import exl3_encoder as E
    from oracle import exl3_oracle as O
    raw = O.decode_states(np.arange(1 << 16, dtype=np.uint32), cb).astype(np.float32)
    n, t0 = 0, time.perf_counter()
    while n < len(target):
        E.encode_tile(target[n], raw, K, dtype=np.float32)
        n += 1
        if time.perf_counter() - t0 >= target_s:
            break
    return n, time.perf_counter() - t0


def run_encode(args):
    """The encoder leg: every step encodes ENCODE_TILES tiles of a unit
    Gaussian source (K = 2, 3INST) with exl3_encode_tiles."""
    K, cb = 2, 0
    rank = int(os.environ.get("RANK", "0"))
    desc = (f"tail-biting two-pass Viterbi encode of {ENCODE_TILES} tiles (256 steps each) of a unit "
            f"Gaussian source, K={K}, 3INST, binary32 path costs")
    target, sigma = encode_inputs(K, cb, ENCODE_TILES)
    weights_step = ENCODE_TILES * 256
    if args.impl == "reference":
        if rank != 0:
            return 0
        tw, tt = 0, 0.0
        steps = max(1, min(args.steps, 20))  # a bounded sample: about a minute in all
        for _ in range(steps):
            n, dt = encode_oracle_timed(target, K, cb, target_s=60.0 / steps)
            tw += n * 256
            tt += dt
        value = tw / tt
        print(json.dumps({
            "impl": "reference", "metric": ENCODE_METRIC, "value": value, "unit": "weights/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tt / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": {"workload": desc},
            "cpu_baseline": {"value": value, "unit": "weights/s", "cores": 1, "kind": "oracle",
                             "sample": "whole tiles of the workload per step, oracle binary32 encoder"},
            "e2e": {"value": value, "unit": "weights/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return 0
    import torch
    import torch.distributed as dist
    from trellis_decode_gemv_gb300 import binding as B
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:  # one replica per GPU; the ranks meet only at the barriers
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    hbm_gbs, sm_max_mhz, _, peak_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    t_dev = torch.from_numpy(target).to(dev)
    words = torch.empty((ENCODE_TILES, 8 * K), dtype=torch.int32, device=dev)
    cost = torch.empty(ENCODE_TILES, dtype=torch.float32, device=dev)
    ws = torch.empty(B.exl3_encode_workspace_bytes(K, sms), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    steps = max(1, min(args.steps, 50))

    def step():
        B.exl3_encode_tiles(t_dev, K, cb, words=words, cost=cost, workspace=ws)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(getattr(props, "pci_bus_id", None) if isinstance(getattr(props, "pci_bus_id", None), str)
                          else None)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_step = ms_total / steps
    value = whole_job_rate(weights_step, world, steps, ms_total / 1e3)
    mse = float(cost.double().sum()) / weights_step / sigma ** 2
    # FP32 candidate work: 2 passes x 256 steps x 2^16 states x (sub, mul, add, compare)
    ops_step = ENCODE_TILES * 2 * 256 * (1 << 16) * 4
    p_fp32 = sms * 128 * sm_max_mhz * 1e6
    achieved = ops_step / (ms_step / 1e3)
    # end to end: pinned host target in, words and costs out, every step
    th = torch.from_numpy(target).pin_memory()
    wh = torch.empty_like(words, device="cpu").pin_memory()
    ch = torch.empty_like(cost, device="cpu").pin_memory()
    e2e_steps = max(3, min(steps, 20))
    with torch.cuda.stream(stream):
        t_dev.copy_(th, non_blocking=True)
        step()
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            t_dev.copy_(th, non_blocking=True)
            step()
            wh.copy_(words, non_blocking=True)
            ch.copy_(cost, non_blocking=True)
            stream.synchronize()
        t_e2e = time.perf_counter() - t0
    t_e2e = max_over_ranks(t_e2e, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, dt = encode_oracle_timed(target, K, cb, target_s=12.0)
        cpu = {"value": n * 256 / dt, "unit": "weights/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} whole tiles of the workload ({dt:.1f} s), oracle binary32 encoder"}
    if rank != 0:
        return 0
    print(json.dumps({
        "metric": ENCODE_METRIC, "value": value, "unit": "weights/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc, "tiles": ENCODE_TILES,
                   "l2": "each step writes 4 MB of predecessor choices per tile (4.9 GB), far more than L2"},
        "mse_unit_variance": mse,
        "roofline": {"bound": "alu", "achieved": achieved / 1e12, "peak": p_fp32 / 1e12, "unit": "Tops/s",
                     "frac": achieved / p_fp32, "traffic": None,
                     "peak_source": f"FP32: {sms} SMs x 128 lanes/clk x {sm_max_mhz:.0f} MHz (derived)",
                     "kernel": "encode_kernel (one CTA per tile, binary32 path costs)",
                     "ops_note": "2 passes x 256 steps x 65536 states x 4 ops (sub, mul, add, compare) per tile"},
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(weights_step, world, e2e_steps, t_e2e), "unit": "weights/s",
                "h2d_bytes_per_step": target.nbytes, "d2h_bytes_per_step": words.numel() * 4 + cost.numel() * 4},
        "clocks": clk, "gpu_launches": steps}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    choices=["all", "llama8b", "llama8b-mcg-mul1", "single", "llama70b", "mixed", "sweep", "prefill",
                             "whole", "encode", "int8", "mad-mul1"],
                    help="all (default): every config, the Llama-3-8B layer set at batch 1 as the headline")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--grouping", choices=["step", "class", "decoder", "none"], default="step",
                    help="step: every GEMV of a step in exl3_gemm_multi calls (mixed K and code); class: every "
                         "GEMV of a step sharing K and the code in one grouped call; decoder: q/k/v and gate/up "
                         "grouped; none: one call per GEMV")
    ap.add_argument("--ungrouped", action="store_true", help="same as --grouping none")
    ap.add_argument("--path", choices=["auto", "shuffle", "tensor"], default="auto",
                    help="kernel family of the fused layer (exl3_set_path)")
    ap.add_argument("--prefill", choices=["auto", "fused", "decode_once"], default="auto",
                    help="prefill strategy above 32 batch rows (exl3_set_prefill)")
    args = ap.parse_args()
    if args.ungrouped:
        args.grouping = "none"
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "encode":
        return run_encode(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
