#!/usr/bin/env python
"""Throughput of the TurboQuant_prod score path (query transform + scoring) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c2] [--path auto]
    python bench.py --impl reference ...      # the CPU oracle on the host cores
    python bench.py --config c2 --s-sweep 32768,131072,524288,2097152   # fixed + per-key fit

One step = one pass of the whole hot path over one workload through the fused
public entry (tq_solve / tq_solve_packed): the query transform A = Pi q,
T = S_mat q for every query, then every raw score read from the compressed
cache.  Inputs are synthetic (the ``synth`` draws), compressed on the GPU by
libtq's own compressor before timing starts; nothing on the timed path touches
the CPU oracle.  Prints one JSON line (rank 0).

The default workload is c2, single-query decode over 131072 bit-packed 3-bit keys.

Timing: the timed region replays CUDA graphs that hold 8 consecutive steps each
(one graph per step for a remainder), exactly K steps, bracketed by CUDA events
on the launching stream; the region is repeated (at least 5 times and for at least
half a second, so the clock sampler sees it) and the median repeat is reported.  Steps rotate over enough independent input/output
copies that their union is more than twice the L2, so every step reads its
cache from HBM.  The roofline's kernel time is the mean of back-to-back
launches of the dominant kernel (the scoring kernel, or the single fused
kernel when the step is one launch) over the same copies.  Under torchrun every
rank runs its own replica of the workload (weak scaling, no data-path
collective); the timed region is bracketed by a barrier and the max over ranks
is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "scores/sec and achieved HBM GB/s (fraction of ~8 TB/s) at 1 GB300"
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the scoring kernel, from
# the ncu captures summarised under profiles/, keyed by (workload, path, fingerprint of
# that kernel's sources).  A changed kernel source makes the figure stale: it is
# reported null.
# Writes that were still in L2 when the kernel ended are not in the figure.
NCU_TRAFFIC = {
    ("c1", "bf16_mma", "d0448b366b12"): 8586496,      # scores_mma_kernel, unpacked, lite
    ("c2", "fp32", "cb02f6e173b7"): 6714368,          # solve_packed_lut_kernel, cluster of 8
    ("c3", "fp32", "cb02f6e173b7"): 255750912,        # scores_packed_lut8_kernel, stream-K, 4 queries
    ("c4", "bf16_mma", "d0448b366b12"): 89109760,     # scores_mma_kernel, packed 3-bit, full
    ("m1", "fp32", "294cce443cd0"): 6573312,          # scores_mse_lut_kernel, stream-K
    ("d1", "fp32", "584008419dc3"): 13317888,         # decode_split_kernel + decode_combine_kernel
    ("d2", "fp32", "584008419dc3"): 13324032,         # the same, product keys
    ("k1", "compress", "3cf3e4fc3955"): 16954880,     # compress_tile_kernel, packed output
    ("s1", "split", "a002a5eeb0d2"): 5281280,         # split_scores_kernel
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(synth.WORKLOADS), default="c2")
    ap.add_argument("--path", choices=["auto", "fp32", "bf16_mma"], default="auto")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-one-core", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--s-sweep", default="",
                    help="comma-separated key counts: time the step of this workload at each S "
                         "(keys tiled from the workload's own cache) and fit fixed + S x per-key")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------

def key_bytes(w) -> int:
    if w.layout == "unpacked":
        return 2 * w.D + (4 if w.gamma_dtype == "f32" else 2)
    if w.layout == "mse":                 # code plane + norm, no sign plane
        return w.D * w.mse_bits // 8 + (4 if w.gamma_dtype == "f32" else 2)
    if w.layout == "decode":              # the key's and the value's code plane + norm
        return 2 * (w.D * w.mse_bits // 8 + 2)
    if w.layout == "split":               # both instances' code planes + two fp16 norms
        return (w.n_out * (w.mse_bits + 1) + (w.D - w.n_out) * w.mse_bits) // 8 + 4
    if w.layout == "decode_prod":         # product key (codes, signs, gamma) + value (codes, norm)
        return w.D * w.mse_bits // 8 + w.D // 8 + 2 + w.D * w.v_bits // 8 + 2
    return w.D * w.mse_bits // 8 + w.D // 8 + (4 if w.gamma_dtype == "f32" else 2)


def score_kernel_bytes(w) -> int:
    """Algorithmic bytes of one scoring launch: the compressed cache once, the
    scores once, A and T once (A only for the MSE-only scorer), the codebook."""
    if w.layout == "decode":
        # cache once, A and the outputs once, Pi_v once, both codebooks
        return (w.P * w.S * key_bytes(w) + 2 * 4 * w.P * w.B * w.D + 4 * w.H * w.D * w.D + 8 * w.C)
    if w.layout == "decode_prod":
        # cache once, A, T and the outputs once, Pi_v once, both codebooks
        return (w.P * w.S * key_bytes(w) + 3 * 4 * w.P * w.B * w.D + 4 * w.H * w.D * w.D
                + 4 * w.C + 4 * (1 << w.v_bits))
    if w.layout == "split":
        # cache once, scores once, A_out and A_reg once, both codebooks
        return (w.P * w.S * key_bytes(w) + 4 * w.P * w.B * w.S + 4 * w.P * w.B * w.D
                + 4 * ((1 << (w.mse_bits + 1)) + (1 << w.mse_bits)))
    n_at = 1 if w.layout == "mse" else 2
    return (w.P * w.S * key_bytes(w) + 4 * w.P * w.B * w.S + n_at * 4 * w.P * w.B * w.D + 4 * w.C)


def fused_kernel_extra_bytes(w) -> int:
    """Inputs the single fused kernel also reads once: the queries and Pi, S_mat."""
    return w.P * w.B * w.D * (2 if w.q_dtype == "bf16" else 4) + 2 * 4 * w.H * w.D * w.D - 8 * w.P * w.B * w.D


def step_input_bytes(w) -> int:
    qbytes = w.P * w.B * w.D * (2 if w.q_dtype == "bf16" else 4)
    return qbytes + w.P * w.S * key_bytes(w) + 2 * 4 * w.H * w.D * w.D + 4 * w.C


def rank_workload(w, rank: int):
    """The workload rank `rank` scores under torchrun: the same shape, its own seed, so
    that every rank processes distinct problems (weak scaling; no data is exchanged)."""
    import dataclasses
    return dataclasses.replace(w, seed=w.seed + 7919 * rank)


def max_over_ranks(value: float, dist, device) -> float:
    """Maximum of `value` over all ranks (the slowest rank bounds the job); identity when
    not distributed."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources each kind of dominant kernel is built from: a traffic figure goes stale
# only when one of its own kernel's sources changes.
KERNEL_SOURCES = {
    "mma": ("tq_scores_mma.cu", "tq_internal.cuh"),
    "simt": ("tq_scores_simt.cu", "tq_lut.cuh", "tq_internal.cuh"),
    "mse": ("tq_scores_mse.cu", "tq_lut.cuh", "tq_internal.cuh"),
    "decode": ("tq_decode.cu", "tq_lut.cuh", "tq_internal.cuh"),
    "split": ("tq_split.cu", "tq_internal.cuh"),
    "compress": ("tq_compress.cu", "tq_internal.cuh"),
}


def kernel_family(w, path) -> str:
    if w.layout in ("mse", "decode"):
        return w.layout
    if w.layout == "decode_prod":
        return "decode"
    if w.layout == "split":
        return "split"
    return "mma" if path == "bf16_mma" else "simt"


def kernel_fingerprint(family: str) -> str:
    import hashlib
    h = hashlib.sha1()
    for name in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "compressed_kv_cache_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:12]


def staging_pair(torch, dev, tensors):
    """One pinned host buffer and one device buffer holding `tensors` (name -> host
    tensor) back to back at 256-byte aligned offsets, so that a step's inputs travel in
    one host-to-device copy; returns (host, device, {name: device view})."""
    offs, off = {}, 0
    for k, t in tensors.items():
        offs[k] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(off, dtype=torch.uint8).pin_memory()
    devb = torch.empty(off, dtype=torch.uint8, device=dev)
    views = {}
    for k, t in tensors.items():
        nb = t.numel() * t.element_size()
        host[offs[k]:offs[k] + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
        views[k] = devb[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    return host, devb, views


def time_e2e(torch, dev, streams, step, n, warmup):
    """Times n end-to-end steps (step(k) issues step k, copies in, call, read-back, on
    streams[k % 2]) two ways: issued from Python call by call, and captured once as a
    CUDA graph and replayed.  Returns (graph_ms, eager_ms) for the n steps."""
    def body(m):
        streams[1].wait_stream(streams[0])          # the second stream forks from the first
        for k in range(m):
            step(k)
        streams[0].wait_stream(streams[1])          # and joins it at the end

    def timed(fn, reps=1):
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(streams[0]):
            es.record()
            for _ in range(reps):
                fn()
            ee.record()
        torch.cuda.synchronize(dev)
        return es.elapsed_time(ee) / reps

    with torch.cuda.stream(streams[0]):
        body(max(2, warmup))
    torch.cuda.synchronize(dev)
    eager_ms = timed(lambda: body(n))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=streams[0]):
        body(n)
    with torch.cuda.stream(streams[0]):
        for _ in range(max(1, warmup)):
            g.replay()
    torch.cuda.synchronize(dev)
    return timed(g.replay, reps=5), eager_ms


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling every 50 ms in the background.  Each line is stamped with its
    arrival time; the timed region is bracketed by samples (the sampler is running
    before the region starts and has delivered a line after it ends), so even a region
    shorter than the sampling interval gets the samples nearest to it."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import threading
        self.proc = None
        self.lines = []
        self.cv = threading.Condition()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        self._wait_for(lambda: len(self.lines) > 0, 10.0)

    def _read(self):
        for line in self.proc.stdout:
            with self.cv:
                self.lines.append((time.time(), line))
                self.cv.notify_all()

    def _wait_for(self, pred, timeout):
        deadline = time.time() + timeout
        with self.cv:
            while not pred() and time.time() < deadline:
                self.cv.wait(timeout=0.05)

    def stop(self, region):
        empty = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_in_region": 0}
        if self.proc is None:
            return empty
        t_lo, t_hi = region
        self._wait_for(lambda: any(t >= t_hi for t, _ in self.lines), 2.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with self.cv:
            stamped = list(self.lines)
        rows = []
        for t, line in stamped:
            parts = [q.strip() for q in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return empty
        inside = [r for r in rows if t_lo <= r[0] <= t_hi]
        before = [r for r in rows if r[0] < t_lo][-1:]
        after = [r for r in rows if r[0] > t_hi][:1]
        use = inside + before + after if inside else before + after
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": reasons, "samples": len(use), "samples_in_region": len(inside)}


# ---------------------------------------------------------------------------
# workload on the device (product code only)
# ---------------------------------------------------------------------------

def build_split_workload(w, tq, torch, dev):
    """The outlier-split cache on the device: the n_out channels with the largest mean |k|
    over problem 0's keys, then each instance's unit sub-vectors compressed by libtq's
    compressor (its codes are the MSE codes of a unit vector) and their lengths as fp16."""
    n_out, n_reg = w.n_out, w.D - w.n_out
    bo, br = w.mse_bits + 1, w.mse_bits
    keys = torch.from_numpy(np.stack([synth.unit_keys(w.seed, p, 0, w.S, w.D) for p in range(w.P)])
                            .astype(np.float32)).to(dev)
    ch = torch.sort(torch.topk(keys[0].abs().mean(dim=0), n_out).indices).values.to(torch.int32)
    mask = torch.ones(w.D, dtype=torch.bool, device=dev)
    mask[ch.long()] = False
    reg = torch.nonzero(mask).flatten()
    sub = {"out": (keys[:, :, ch.long()], n_out, bo), "reg": (keys[:, :, reg], n_reg, br)}
    cache = {"channels": ch}
    rot = {}
    for name, (x, n, b) in sub.items():
        cb = torch.from_numpy(tq.lloyd_max_codebook(n, b)).to(dev)
        Pi = torch.from_numpy(np.stack([tq.haar_rotation(synth.rotation_seed_matrix(w.seed + n, h, n))
                                        for h in range(w.H)])).to(dev)
        Sx = torch.from_numpy(np.stack([synth.s_matrix(w.seed + n, h, n) for h in range(w.H)])).to(dev)
        nrm = torch.linalg.vector_norm(x, dim=2)
        unit = (x / nrm[:, :, None]).contiguous()
        idx = torch.empty((w.P, w.S, n), dtype=torch.uint8, device=dev)
        for p in range(w.P):
            idx[p].copy_(tq.compress_keys(unit[p], Pi[p % w.H], Sx[p % w.H], cb, torch.float16)[0])
        cache[name + "_plane"] = tq.pack_indices(idx, b)
        cache[name + "_norm"] = nrm.to(torch.float16)
        cache[name + "_cb"] = cb
        rot[name] = Pi
    Q = torch.from_numpy(np.stack([synth.queries(w.seed, p, w.B, w.D, "f32")[0] for p in range(w.P)])).to(dev)
    torch.cuda.synchronize(dev)
    return Q, rot["out"], rot["reg"], cache


def split_call(tq, w, Q, Pi_out, Pi_reg, cache, Ao, Ar, out):
    """One step of the split path: both rotated queries, then the scores."""
    tq.prepare_queries_split(Q, cache["channels"], Pi_out, Pi_reg, out=(Ao, Ar))
    return tq.scores_split(Ao, Ar, cache["out_plane"], cache["out_norm"], cache["out_cb"], w.mse_bits + 1,
                           cache["reg_plane"], cache["reg_norm"], cache["reg_cb"], w.mse_bits, out=out)


def build_device_workload(w, tq, torch, dev):
    cb = torch.from_numpy(tq.lloyd_max_codebook(w.D, w.mse_bits)).to(dev)
    Pi = torch.from_numpy(np.stack([tq.haar_rotation(synth.rotation_seed_matrix(w.seed, h, w.D))
                                    for h in range(w.H)])).to(dev)
    S_mat = torch.from_numpy(np.stack([synth.s_matrix(w.seed, h, w.D) for h in range(w.H)])).to(dev)
    gdt = torch.float32 if w.gamma_dtype == "f32" else torch.float16
    idx = torch.empty((w.P, w.S, w.D), dtype=torch.uint8, device=dev)
    sg = torch.empty((w.P, w.S, w.D), dtype=torch.int8, device=dev)
    gamma = torch.empty((w.P, w.S), dtype=gdt, device=dev)
    for p in range(w.P):
        keys = torch.from_numpy(synth.unit_keys(w.seed, p, 0, w.S, w.D).astype(np.float32)).to(dev)
        i_, s_, g_ = tq.compress_keys(keys, Pi[p % w.H], S_mat[p % w.H], cb, gdt)
        idx[p].copy_(i_)
        sg[p].copy_(s_)
        gamma[p].copy_(g_)
    if w.q_dtype == "bf16":
        Q = torch.from_numpy(np.stack([synth.queries(w.seed, p, w.B, w.D, "bf16")[1]
                                       for p in range(w.P)]).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        Q = torch.from_numpy(np.stack([synth.queries(w.seed, p, w.B, w.D, "f32")[0]
                                       for p in range(w.P)])).to(dev)
    cache = {"gamma": gamma}
    if w.layout == "unpacked":
        cache["idx"], cache["signs"] = idx, sg
    elif w.layout in ("mse", "decode"):
        # unit keys: the codes of TurboQuant_prod's MSE stage are the MSE-only codes
        # (same rotation, codebook and cells) and every stored norm is 1
        cache = {"idx": tq.pack_indices(idx, w.mse_bits),
                 "norm": torch.ones((w.P, w.S), dtype=torch.float16, device=dev)}
        if w.layout == "decode":
            # unit values of their own, with their own rotation per head
            Pi_v = torch.from_numpy(np.stack([tq.haar_rotation(synth.rotation_seed_matrix(w.seed + 1, h, w.D))
                                              for h in range(w.H)])).to(dev)
            vidx = torch.empty((w.P, w.S, w.D), dtype=torch.uint8, device=dev)
            for p in range(w.P):
                vals = torch.from_numpy(synth.unit_keys(w.seed + 1, p, 0, w.S, w.D).astype(np.float32)).to(dev)
                vidx[p].copy_(tq.compress_keys(vals, Pi_v[p % w.H], S_mat[p % w.H], cb, gdt)[0])
            cache.update({"vidx": tq.pack_indices(vidx, w.mse_bits), "Pi_v": Pi_v,
                          "vnorm": torch.ones((w.P, w.S), dtype=torch.float16, device=dev),
                          # outputs and split-KV scratch of the decode (not inputs)
                          "dout": torch.empty((w.P, w.B, w.D), device=dev),
                          "dws": torch.empty(max(16, int(tq.lib().tq_decode_workspace_bytes(w.P, w.B, w.S, w.D))),
                                             dtype=torch.uint8, device=dev)})
    else:
        cache["idx"] = tq.pack_indices(idx, w.mse_bits)
        cache["signs"] = tq.pack_signs(sg)
        if w.layout == "decode_prod":
            # unit values of their own, with their own rotation per head and codebook
            vcb = torch.from_numpy(tq.lloyd_max_codebook(w.D, w.v_bits)).to(dev)
            Pi_v = torch.from_numpy(np.stack([tq.haar_rotation(synth.rotation_seed_matrix(w.seed + 1, h, w.D))
                                              for h in range(w.H)])).to(dev)
            vidx = torch.empty((w.P, w.S, w.D), dtype=torch.uint8, device=dev)
            for p in range(w.P):
                vals = torch.from_numpy(synth.unit_keys(w.seed + 1, p, 0, w.S, w.D).astype(np.float32)).to(dev)
                vidx[p].copy_(tq.compress_keys(vals, Pi_v[p % w.H], S_mat[p % w.H], vcb, gdt)[0])
            cache.update({"vidx": tq.pack_indices(vidx, w.v_bits), "Pi_v": Pi_v, "vcb": vcb,
                          "vnorm": torch.ones((w.P, w.S), dtype=torch.float16, device=dev),
                          "dout": torch.empty((w.P, w.B, w.D), device=dev),
                          "dws": torch.empty(max(16, int(tq.lib().tq_decode_workspace_bytes(w.P, w.B, w.S, w.D))),
                                             dtype=torch.uint8, device=dev)})
    torch.cuda.synchronize(dev)
    return Q, Pi, S_mat, cb, cache


def score_call(tq, w, path, A, T, cache, cb, out):
    if w.layout == "decode_prod":
        return tq.decode_prod(A, T, cache["idx"], cache["signs"], cache["gamma"], cb, w.mse_bits, cache["vidx"],
                              cache["vnorm"], cache["vcb"], w.v_bits, cache["Pi_v"], workspace=cache["dws"],
                              out=cache["dout"])
    if w.layout == "decode":
        return tq.decode_mse(A, cache["idx"], cache["norm"], cb, w.mse_bits, cache["vidx"], cache["vnorm"], cb,
                             w.mse_bits, cache["Pi_v"], workspace=cache["dws"], out=cache["dout"])
    if w.layout == "mse":
        return tq.scores_mse(A, cache["idx"], cache["norm"], cb, w.mse_bits, norm_correction=True, out=out)
    if w.layout == "unpacked":
        return tq.scores(A, T, cache["idx"], cache["signs"], cache["gamma"], cb, path=path, out=out)
    return tq.scores_packed(A, T, cache["idx"], cache["signs"], cache["gamma"], cb, w.mse_bits,
                            path=path, out=out)


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and --impl reference only)
# ---------------------------------------------------------------------------

def oracle_sample(w, n_keys):
    import oracle
    cb = oracle.lloyd_max_sphere(w.D, w.mse_bits)[0].astype(np.float32)
    Pi = oracle.haar_rotation(synth.rotation_seed_matrix(w.seed, 0, w.D)).astype(np.float32)
    S_mat = synth.s_matrix(w.seed, 0, w.D)
    keys = synth.unit_keys(w.seed, 0, 0, n_keys, w.D)
    Q = synth.queries(w.seed, 0, w.B, w.D, w.q_dtype)[0]
    if w.layout == "decode":
        Pi_v = oracle.haar_rotation(synth.rotation_seed_matrix(w.seed + 1, 0, w.D)).astype(np.float32)
        ki, kn = oracle.compress_mse(keys, Pi, cb)
        vi, vn = oracle.compress_mse(synth.unit_keys(w.seed + 1, 0, 0, n_keys, w.D), Pi_v, cb)

        def run_decode():
            A, _ = oracle.prepare_queries(Q, Pi, Pi)
            return oracle.decode_mse(A, ki, kn, cb, vi, vn, cb, Pi_v, 1.0 / np.sqrt(w.D))
        return run_decode
    if w.layout == "mse":
        idx, nrm = oracle.compress_mse(keys, Pi, cb)

        def run():
            A, _ = oracle.prepare_queries(Q, Pi, Pi)
            return oracle.scores_mse(A, idx, nrm, cb, norm_correction=True)
        return run
    idx, sg, gamma = oracle.compress_prod(keys, Pi, S_mat, cb, w.gamma_dtype)
    if w.layout == "decode_prod":
        vcb = oracle.lloyd_max_sphere(w.D, w.v_bits)[0].astype(np.float32)
        Pi_v = oracle.haar_rotation(synth.rotation_seed_matrix(w.seed + 1, 0, w.D)).astype(np.float32)
        vi, vn = oracle.compress_mse(synth.unit_keys(w.seed + 1, 0, 0, n_keys, w.D), Pi_v, vcb)

        def run_decode_prod():
            A, T = oracle.prepare_queries(Q, Pi, S_mat)
            return oracle.decode_prod(A, T, idx, sg, gamma, cb, vi, vn, vcb, Pi_v, 1.0 / np.sqrt(w.D))
        return run_decode_prod
    return lambda: oracle.scores_from_queries(Q, Pi, S_mat, idx, sg, gamma, cb)


def time_oracle(w, seconds, n_keys=None):
    """Scores/s of the oracle (query transform + scoring of B queries over a key sample)."""
    n_keys = n_keys or min(w.S, 4096)
    run = oracle_sample(w, n_keys)
    t0 = time.perf_counter()
    reps = 0
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": reps * w.B * n_keys / el, "unit": "scores/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x (query transform + {w.B} queries x {n_keys} keys of problem 0), "
                      f"{el:.1f} s, float64 NumPy (BLAS threads = host cores)"}


def time_oracle_one_core(config, seconds):
    """The same oracle timing in a child process pinned to one core with one BLAS thread
    (the variables must be set before NumPy loads its BLAS).  Returns scores/s or None."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-one-core", "--config", config,
           "--cpu-seconds", str(seconds)]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=10 * seconds + 120)
        return json.loads(res.stdout.strip().splitlines()[-1])["value"]
    except (subprocess.SubprocessError, ValueError, IndexError, KeyError):
        return None


def oracle_one_core_child(args, w):
    if hasattr(os, "sched_setaffinity"):
        cpu = min(os.sched_getaffinity(0))
        os.sched_setaffinity(0, {cpu})
    print(json.dumps(time_oracle(w, args.cpu_seconds)), flush=True)


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if w.layout in ("compress", "split"):
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the scoring path of "
                          "the page configurations; this workload's CPU baseline is in its own line"}), flush=True)
        return
    n_keys = min(w.S, 4096)
    run = oracle_sample(w, n_keys)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = args.steps * w.B * n_keys / el
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "scores/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample_keys": n_keys, "B": w.B, "D": w.D},
            "cpu_baseline": {"value": value, "unit": "scores/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: query transform + {w.B} queries x {n_keys} keys "
                                       f"(a bounded sample of the workload), float64 NumPy"},
            "e2e": {"value": value, "unit": "scores/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# S-sweep: the per-call time of one workload as the cache grows
# ---------------------------------------------------------------------------

def run_s_sweep(args, w, tq, torch, dev, path):
    """Times one step (the fused public entry) of workload `w` at each S of --s-sweep and
    fits t(S) = fixed + S * per_key by least squares.  The cache at each S repeats the
    workload's own compressed keys; every launch reads its inputs from HBM (rotating
    copies larger than twice the L2).  Prints one JSON line."""
    Q0, Pi, S_mat, cb, cache0 = build_device_workload(w, tq, torch, dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(dev)
    rows = []
    for S in [int(x) for x in args.s_sweep.split(",") if x]:
        reps_ = -(-S // w.S)
        cache = {k: v.repeat_interleave(1, dim=0).repeat(*([1, reps_] + [1] * (v.dim() - 2)))[:, :S].contiguous()
                 for k, v in cache0.items()}
        ws = dataclasses_replace(w, S=S)
        per_copy = score_kernel_bytes(ws)
        R = max(2, min(64, math.ceil(2.2 * l2 / per_copy)))
        copies = [{"cache": {k: v.clone() for k, v in cache.items()}, "Q": Q0.clone(),
                   "out": torch.empty((w.P, w.B, S), device=dev),
                   "ws": torch.empty(tq.workspace_bytes(w.P, w.B, w.D), dtype=torch.uint8, device=dev)}
                  for _ in range(R)]
        del cache

        def call(cp):
            c = cp["cache"]
            if w.layout == "unpacked":
                tq.solve(cp["Q"], c["idx"], c["signs"], c["gamma"], Pi, S_mat, cb, path=path,
                         workspace=cp["ws"], out=cp["out"])
            else:
                tq.solve_packed(cp["Q"], c["idx"], c["signs"], c["gamma"], Pi, S_mat, cb, w.mse_bits,
                                path=path, workspace=cp["ws"], out=cp["out"])
        with torch.cuda.stream(stream):
            for cp in copies:
                call(cp)
        torch.cuda.synchronize(dev)
        n = max(R, 32)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                call(copies[k % R])
        times = []
        for _ in range(6):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record()
                g.replay()
                e1.record()
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) / n)
        ms = statistics.median(times[1:])
        nbytes = score_kernel_bytes(ws) + fused_kernel_extra_bytes(ws)
        rows.append({"S": S, "ms_per_call": ms, "bytes": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9,
                     "copies": R})
        del copies, g
        torch.cuda.empty_cache()
    xs = np.array([r["S"] for r in rows], dtype=np.float64)
    ys = np.array([r["ms_per_call"] for r in rows], dtype=np.float64)
    fit = None
    if len(rows) >= 2:
        slope, icpt = np.polyfit(xs, ys, 1)
        per_key_bytes = key_bytes(w) + 4 * w.B
        fit = {"fixed_us": icpt * 1e3, "per_key_ns": slope * 1e6,
               "streaming_gbs": per_key_bytes / (slope * 1e-3) / 1e9 if slope > 0 else None}
    peak, _ = hbm_peak()
    for r in rows:
        r["frac"] = r["gbs"] / peak
    print(json.dumps({"sweep": w.name, "path": path, "peak_gbs": peak, "rows": rows, "fit": fit}), flush=True)


def fma_peak_tflops():
    """fp32 FMA-pipe peak: 152 SMs x 128 FMA lanes x 2 FLOP x the maximum SM clock
    (MEASURED_PEAKS.json sm_max_mhz, else 2070 MHz)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        mhz = 2070.0
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def run_compress(args, w, tq, torch, dev):
    """The write side: tq_compress_keys_packed over P x S fp32 keys (rotating copies larger
    than twice the L2), timed like the scoring steps; one JSON line."""
    cb = torch.from_numpy(tq.lloyd_max_codebook(w.D, w.mse_bits)).to(dev)
    Pi = torch.from_numpy(np.stack([tq.haar_rotation(synth.rotation_seed_matrix(w.seed, h, w.D))
                                    for h in range(w.H)])).to(dev)
    S_mat = torch.from_numpy(np.stack([synth.s_matrix(w.seed, h, w.D) for h in range(w.H)])).to(dev)
    keys0 = torch.from_numpy(np.stack([synth.unit_keys(w.seed, p, 0, w.S, w.D) for p in range(w.P)])
                             .astype(np.float32)).to(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    key_b = 4 * w.D
    out_b = w.D * w.mse_bits // 8 + w.D // 8 + 2
    per_copy = w.P * w.S * (key_b + out_b)
    R = max(2, min(64, math.ceil(2.2 * l2 / per_copy)))
    copies = [{"k": keys0.clone(), "out": (torch.empty((w.P, w.S, w.D * w.mse_bits // 8), dtype=torch.uint8, device=dev),
                                           torch.empty((w.P, w.S, w.D // 8), dtype=torch.uint8, device=dev),
                                           torch.empty((w.P, w.S), dtype=torch.float16, device=dev))}
              for _ in range(R)]
    stream = torch.cuda.Stream(dev)

    def call(cp):
        tq.compress_keys_packed(cp["k"], Pi, S_mat, cb, w.mse_bits, out=cp["out"])
    with torch.cuda.stream(stream):
        for cp in copies:
            call(cp)
    torch.cuda.synchronize(dev)
    G = 8
    graphs = []
    for b in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(G):
                call(copies[(b + j) % R])
        graphs.append(g)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            graphs[k % R].replay()
    torch.cuda.synchronize(dev)
    steps = -(-args.steps // G) * G

    def region():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            for k in range(steps // G):
                graphs[k % R].replay()
            e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)
    t0 = time.time()
    regions = [region()]
    n_rep = int(min(200, max(5, math.ceil(500.0 / max(regions[0], 1e-3)))))
    while len(regions) < n_rep:
        regions.append(region())
    t1 = time.time()
    clk = clocks.stop((t0, t1))
    ms = statistics.median(regions) / steps
    nkeys = w.P * w.S
    flops = 3 * 2 * w.D * w.D * nkeys                  # three D x D products per key
    achieved = flops / (ms / 1e3) / 1e12
    peak = fma_peak_tflops()
    # end to end: keys in from pinned host memory, the packed cache out, two streams
    hk = keys0.cpu().pin_memory()
    e_streams = [stream, torch.cuda.Stream(dev)]
    e_bufs = [{"k": torch.empty_like(keys0), "out": copies[i]["out"],
               "h": tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in copies[i]["out"])}
              for i in range(2)]

    def e2e_step(k):
        eb = e_bufs[k % 2]
        with torch.cuda.stream(e_streams[k % 2]):
            eb["k"].copy_(hk, non_blocking=True)
            tq.compress_keys_packed(eb["k"], Pi, S_mat, cb, w.mse_bits, out=eb["out"])
            for h_, d_ in zip(eb["h"], eb["out"]):
                h_.copy_(d_, non_blocking=True)
    n_e = max(4, min(args.steps, 48)) // 2 * 2
    e_ms, eager_ms = time_e2e(torch, dev, e_streams, e2e_step, n_e, args.warmup)
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        n = min(w.S, 2048)
        k_np = synth.unit_keys(w.seed, 0, 0, n, w.D)
        cb_np, Pi_np, S_np = cb.cpu().numpy(), Pi[0].cpu().numpy(), S_mat[0].cpu().numpy()
        t_0, reps = time.perf_counter(), 0
        while time.perf_counter() - t_0 < args.cpu_seconds:
            oracle.compress_prod(k_np, Pi_np, S_np, cb_np, "f16")
            reps += 1
        el = time.perf_counter() - t_0
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        cpu = {"value": reps * n / el, "unit": "keys/s", "cores": cores, "kind": "oracle",
               "hardware_concurrency": os.cpu_count(),
               "sample": f"{reps} x compress_prod of {n} keys, {el:.1f} s, float64 NumPy"}
    line = {"metric": "compressed keys/s (fp32 keys in, packed TurboQuant_prod cache out) at 1 GB300",
            "value": nkeys / (ms / 1e3), "unit": "keys/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "P": w.P, "H": w.H, "S": w.S, "D": w.D, "idx_bits": w.mse_bits,
                       "l2": f"{R} rotating key/output copies, {R * per_copy / 1e6:.0f} MB > 2x L2"},
            "key_gbs": nkeys * key_b / (ms / 1e3) / 1e9,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "traffic": NCU_TRAFFIC.get((args.config, "compress", kernel_fingerprint("compress"))),
                         "kernel": "compress_tile_kernel", "kernel_fingerprint": kernel_fingerprint("compress"),
                         "kernel_ms": ms, "flops_per_launch": flops,
                         "peak_source": "152 SMs x 128 fp32 FMA lanes x 2 FLOP x max SM clock"},
            "timed_region": {"repeats": len(regions), "median_ms": statistics.median(regions)},
            "cpu_baseline": cpu,
            "e2e": {"value": nkeys * n_e / (e_ms / 1e3), "unit": "keys/s",
                    "h2d_bytes_per_step": nkeys * key_b, "d2h_bytes_per_step": nkeys * out_b,
                    "steps": n_e, "streams": 2, "graph": True,
                    "eager_value": nkeys * n_e / (eager_ms / 1e3)},
            "gpu_launches": steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def run_split(args, w, tq, torch, dev):
    """The outlier-split decode: one step = the split query transform and the split scorer
    over P x S keys (rotating copies larger than twice the L2); one JSON line."""
    Q0, Pi_out, Pi_reg, cache0 = build_split_workload(w, tq, torch, dev)
    n_reg = w.D - w.n_out
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = score_kernel_bytes(w)
    R = max(2, min(64, math.ceil(2.2 * l2 / per_copy)))
    G = 8
    R = -(-R // G) * G
    copies = [{"Q": Q0.clone(), "c": {k: v.clone() for k, v in cache0.items()},
               "Ao": torch.empty((w.P, w.B, w.n_out), device=dev), "Ar": torch.empty((w.P, w.B, n_reg), device=dev),
               "out": torch.empty((w.P, w.B, w.S), device=dev)} for _ in range(R)]
    stream = torch.cuda.Stream(dev)

    def step(cp):
        split_call(tq, w, cp["Q"], Pi_out, Pi_reg, cp["c"], cp["Ao"], cp["Ar"], cp["out"])

    def score_only(cp):
        c = cp["c"]
        tq.scores_split(cp["Ao"], cp["Ar"], c["out_plane"], c["out_norm"], c["out_cb"], w.mse_bits + 1,
                        c["reg_plane"], c["reg_norm"], c["reg_cb"], w.mse_bits, out=cp["out"])
    with torch.cuda.stream(stream):
        for cp in copies:
            step(cp)
    torch.cuda.synchronize(dev)

    def graphs_of(fn):
        gs = []
        for b in range(R // G):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for j in range(G):
                    fn(copies[b * G + j])
            gs.append(g)
        return gs
    steps_g, score_g = graphs_of(step), graphs_of(score_only)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    with torch.cuda.stream(stream):
        for k in range(max(1, args.warmup // G + 1)):
            steps_g[k % len(steps_g)].replay()
    torch.cuda.synchronize(dev)
    steps = -(-args.steps // G) * G

    def region(gs, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            for k in range(n // G):
                gs[k % len(gs)].replay()
            e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)
    t0 = time.time()
    regions = [region(steps_g, steps)]
    n_rep = int(min(500, max(5, math.ceil(500.0 / max(regions[0], 1e-3)))))
    while len(regions) < n_rep:
        regions.append(region(steps_g, steps))
    t1 = time.time()
    clk = clocks.stop((t0, t1))
    ms = statistics.median(regions) / steps
    kernel_ms = statistics.median([region(score_g, 3 * R) for _ in range(5)]) / (3 * R)
    kbytes = score_kernel_bytes(w)
    achieved = kbytes / (kernel_ms / 1e3) / 1e9
    peak, peak_src = hbm_peak()
    # end to end: the query, the cache and the rotations in from pinned host memory, the
    # scores out, two streams
    hQ = Q0.cpu().pin_memory()
    hc = {k: v.cpu().pin_memory() for k, v in cache0.items()}
    hPo, hPr = Pi_out.cpu().pin_memory(), Pi_reg.cpu().pin_memory()
    h2d = (hQ.numel() * 4 + sum(v.numel() * v.element_size() for v in hc.values()) + (hPo.numel() + hPr.numel()) * 4)
    e_streams = [stream, torch.cuda.Stream(dev)]
    e_bufs = [{"Q": torch.empty_like(Q0), "c": {k: torch.empty_like(v) for k, v in cache0.items()},
               "Po": torch.empty_like(Pi_out), "Pr": torch.empty_like(Pi_reg), "Ao": copies[i]["Ao"],
               "Ar": copies[i]["Ar"], "out": copies[i]["out"],
               "h": torch.empty((w.P, w.B, w.S), dtype=torch.float32).pin_memory()} for i in range(2)]

    def e2e_step(k):
        eb = e_bufs[k % 2]
        with torch.cuda.stream(e_streams[k % 2]):
            eb["Q"].copy_(hQ, non_blocking=True)
            for key in hc:
                eb["c"][key].copy_(hc[key], non_blocking=True)
            eb["Po"].copy_(hPo, non_blocking=True)
            eb["Pr"].copy_(hPr, non_blocking=True)
            split_call(tq, w, eb["Q"], eb["Po"], eb["Pr"], eb["c"], eb["Ao"], eb["Ar"], eb["out"])
            eb["h"].copy_(eb["out"], non_blocking=True)
    n_e = max(4, min(args.steps, 48)) // 2 * 2
    e_ms, eager_ms = time_e2e(torch, dev, e_streams, e2e_step, n_e, args.warmup)
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        n = min(w.S, 4096)
        keys = synth.unit_keys(w.seed, 0, 0, n, w.D)
        ch = cache0["channels"].cpu().numpy().astype(np.int64)
        Po, Pr = Pi_out[0].cpu().numpy(), Pi_reg[0].cpu().numpy()
        co, cr = cache0["out_cb"].cpu().numpy(), cache0["reg_cb"].cpu().numpy()
        io, no, ir, nr = oracle.compress_split(keys, ch, Po, Pr, co, cr)
        Qs = Q0[0].cpu().numpy()
        t_0, reps = time.perf_counter(), 0
        while time.perf_counter() - t_0 < args.cpu_seconds:
            Ao, Ar = oracle.prepare_queries_split(Qs, ch, Po, Pr)
            oracle.scores_split(Ao, Ar, io, no, co, ir, nr, cr)
            reps += 1
        el = time.perf_counter() - t_0
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        cpu = {"value": reps * w.B * n / el, "unit": "scores/s", "cores": cores, "kind": "oracle",
               "hardware_concurrency": os.cpu_count(),
               "sample": f"{reps} x (split query transform + {w.B} queries x {n} keys), {el:.1f} s, float64 NumPy"}
    fp = kernel_fingerprint("split")
    line = {"metric": METRIC, "value": w.P * w.B * w.S / (ms / 1e3), "unit": "scores/s", "n_gpus": 1,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "P": w.P, "H": w.H, "B": w.B, "S": w.S, "D": w.D,
                       "n_out": w.n_out, "out_bits": w.mse_bits + 1, "reg_bits": w.mse_bits,
                       "l2": f"{R} rotating copies, {R * per_copy / 1e6:.0f} MB > 2x L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": NCU_TRAFFIC.get((args.config, "split", fp)),
                         "kernel": "split_scores_kernel",
                         "kernel_ms": kernel_ms, "bytes_per_launch": kbytes,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                         "kernel_fingerprint": fp},
            "timed_region": {"repeats": len(regions), "median_ms": statistics.median(regions)},
            "cpu_baseline": cpu,
            "e2e": {"value": w.P * w.B * w.S * n_e / (e_ms / 1e3), "unit": "scores/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4 * w.P * w.B * w.S,
                    "steps": n_e, "streams": 2, "graph": True,
                    "eager_value": w.P * w.B * w.S * n_e / (eager_ms / 1e3)},
            "gpu_launches": 2 * steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def dataclasses_replace(w, **kw):
    import dataclasses
    return dataclasses.replace(w, **kw)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def main():
    args = parse_args()
    w = synth.WORKLOADS[args.config]
    if args.oracle_one_core:
        oracle_one_core_child(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    from compressed_kv_cache_gb300 import tq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = rank_workload(w, rank)

    tq.lib()
    path = args.path if args.path != "auto" else tq.auto_path(w.B, w.D)
    if args.s_sweep:
        run_s_sweep(args, w, tq, torch, dev, path)
        return
    if w.layout == "compress":
        run_compress(args, w, tq, torch, dev)
        return
    if w.layout == "split":
        run_split(args, w, tq, torch, dev)
        return
    Q0, Pi, S_mat, cb, cache0 = build_device_workload(w, tq, torch, dev)

    # rotating copies: their union exceeds twice the L2 so that every step reads HBM;
    # R is a multiple of G, the number of consecutive steps one timed graph holds
    G = 8
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = score_kernel_bytes(w)
    R = max(1, math.ceil(2.2 * l2 / per_copy))
    R = min(R, max(1, int(40e9 // per_copy)))
    R = math.ceil(R / G) * G if R > 1 else 1
    copies = []
    for r in range(R):
        c = {k: v.clone() for k, v in cache0.items()}
        copies.append({
            "Q": Q0.clone(), "cache": c,
            "A": torch.empty((w.P, w.B, w.D), device=dev), "T": torch.empty((w.P, w.B, w.D), device=dev),
            "ws": torch.empty(tq.workspace_bytes(w.P, w.B, w.D), dtype=torch.uint8, device=dev),
            "out": torch.empty((w.P, w.B, w.S), device=dev)})

    stream = torch.cuda.Stream(dev)
    # tq_solve_packed runs one fused kernel for the fp32 path when D = 128, B <= 8 and
    # the problems fill fewer than half the SMs; otherwise the transform and the scorer
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fused_single = (w.layout == "packed" and path == "fp32" and w.D == 128 and w.B <= 8
                    and 2 * w.P < sms)

    def solve_call(cp):
        # one step = the fused public entry over the whole workload (for the MSE-only
        # variant, which has no fused entry: the query transform and the MSE scorer)
        if w.layout in ("mse", "decode"):
            tq.prepare_queries(cp["Q"], Pi, Pi, out=(cp["A"], cp["T"]))
            score_call(tq, w, path, cp["A"], cp["T"], cp["cache"], cb, cp["out"])
        elif w.layout == "decode_prod":
            tq.prepare_queries(cp["Q"], Pi, S_mat, out=(cp["A"], cp["T"]))
            score_call(tq, w, path, cp["A"], cp["T"], cp["cache"], cb, cp["out"])
        elif w.layout == "unpacked":
            tq.solve(cp["Q"], cp["cache"]["idx"], cp["cache"]["signs"], cp["cache"]["gamma"], Pi, S_mat, cb,
                     path=path, workspace=cp["ws"], out=cp["out"])
        else:
            tq.solve_packed(cp["Q"], cp["cache"]["idx"], cp["cache"]["signs"], cp["cache"]["gamma"], Pi, S_mat,
                            cb, w.mse_bits, path=path, workspace=cp["ws"], out=cp["out"])

    with torch.cuda.stream(stream):
        for cp in copies:          # eager pass over every copy before capture
            solve_call(cp)
    torch.cuda.synchronize(dev)
    single, chunk = [], []
    for cp in copies:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            solve_call(cp)
        single.append(g)
    nG = G if R >= G else 1
    for b in range(R // nG):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(nG):
                solve_call(copies[b * nG + j])
        chunk.append(g)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for k in range(args.warmup):          # the least recently used copies are the first timed ones
            single[(R - 1 - k) % R].replay()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    def timed_region():
        """Exactly K steps on the launching stream between two CUDA events (ms)."""
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record()
            k = 0
            while k < args.steps:                 # exactly K steps; step k uses copy k mod R
                if k % nG == 0 and k + nG <= args.steps:
                    chunk[(k % R) // nG].replay()
                    k += nG
                else:
                    single[k % R].replay()
                    k += 1
            end.record()
        torch.cuda.synchronize(dev)
        return start.elapsed_time(end)

    # The K-step region is repeated (at least 5 times and for at least half a second, so
    # that the clock sampler sees it) and the median repeat is reported.
    t_wall0 = time.time()
    regions = [timed_region()]
    n_rep = int(min(500, max(5, math.ceil(500.0 / max(regions[0], 1e-3)))))
    while len(regions) < n_rep:
        regions.append(timed_region())
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    elapsed_ms = max_over_ranks(statistics.median(regions), dist, dev)
    clk = clocks.stop((t_wall0, t_wall1))

    # Dominant-kernel duration: the mean of back-to-back launches in one graph over the
    # rotating copies (CUDA events on the launching stream, launch gaps included).
    gk = torch.cuda.CUDAGraph()
    reps = max(R, 16)
    with torch.cuda.stream(stream):      # A, T of every copy for the scoring-only launches
        for cp in copies:
            tq.prepare_queries(cp["Q"], Pi, S_mat, out=(cp["A"], cp["T"]))
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(gk, stream=stream):
        for k in range(reps):
            cp = copies[k % R]
            if fused_single:      # the step is this one kernel (transform + scoring)
                solve_call(cp)
            else:
                score_call(tq, w, path, cp["A"], cp["T"], cp["cache"], cb, cp["out"])
    with torch.cuda.stream(stream):
        gk.replay()
    torch.cuda.synchronize(dev)
    ks, ke = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ks.record()
        for _ in range(3):
            gk.replay()
        ke.record()
    torch.cuda.synchronize(dev)
    kernel_ms = ks.elapsed_time(ke) / (3 * reps)
    ktiming = (f"mean of {3 * reps} back-to-back launches in one graph over the {R} rotating copies "
               f"(CUDA events on the launching stream)")

    def graph_ms(fn):
        """Mean time of one call of fn(copy) over back-to-back launches in one graph."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(reps):
                fn(copies[k % R])
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(3):
                g.replay()
            e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / (3 * reps)

    # the query transform alone, the scoring alone (from precomputed A and T) and the
    # fused call, each as back-to-back launches over the rotating copies
    split_ms = {"prepare_ms": graph_ms(lambda cp: tq.prepare_queries(cp["Q"], Pi, S_mat, out=(cp["A"], cp["T"]))),
                "score_only_ms": graph_ms(lambda cp: score_call(tq, w, path, cp["A"], cp["T"], cp["cache"], cb,
                                                                cp["out"])),
                "fused_ms": graph_ms(solve_call)}

    scores_per_step = w.P * w.B * w.S
    value = world * scores_per_step * args.steps / (elapsed_ms / 1e3)
    peak, peak_src = hbm_peak()
    kbytes = score_kernel_bytes(w) + (fused_kernel_extra_bytes(w) if fused_single else 0)
    achieved = kbytes / (kernel_ms / 1e3) / 1e9
    fp = kernel_fingerprint(kernel_family(w, path))
    traffic = NCU_TRAFFIC.get((args.config, path, fp))

    # end to end through the public fused API with host buffers: every step copies its
    # inputs in from pinned host memory and its result out.  Steps alternate between two
    # streams with their own device buffers, so one step's device-to-host read overlaps
    # the next step's host-to-device copies (the two directions use separate engines).
    if True:
        hostQ = Q0.cpu().pin_memory()
        scratch = ("dout", "dws")             # decode outputs and workspace: not copied in
        hcache = {k: v.cpu().pin_memory() for k, v in cache0.items() if k not in scratch}
        hPi, hS, hcb = Pi.cpu().pin_memory(), S_mat.cpu().pin_memory(), cb.cpu().pin_memory()
        mse = w.layout in ("mse", "decode")   # no S_mat: the MSE-only paths need Pi alone
        out_shape = (w.P, w.B, w.D) if w.layout in ("decode", "decode_prod") else (w.P, w.B, w.S)
        h2d = (hostQ.numel() * hostQ.element_size() + sum(v.numel() * v.element_size() for v in hcache.values())
               + (hPi.numel() + (0 if mse else hS.numel()) + hcb.numel()) * 4)
        d2h = int(np.prod(out_shape)) * 4
        e_streams = [stream, torch.cuda.Stream(device=dev)]

        # every step's inputs (query, cache, rotation, projection, codebook) sit back to
        # back in one pinned buffer and travel in one host-to-device copy
        staged = {"Q": hostQ, "Pi": hPi, "cb": hcb, **{"c_" + k: v for k, v in hcache.items()}}
        if not mse:
            staged["S"] = hS

        def e2e_buffers():
            hbuf, dbuf, v = staging_pair(torch, dev, staged)
            cache = {k: v["c_" + k] for k in hcache}
            cache.update({k: torch.empty_like(cache0[k]) for k in scratch if k in cache0})
            return {"hbuf": hbuf, "dbuf": dbuf, "Q": v["Q"], "cache": cache, "Pi": v["Pi"],
                    "S": v.get("S", v["Pi"]), "cb": v["cb"],
                    "out": torch.empty((w.P, w.B, w.S), device=dev),
                    "ws": torch.empty(tq.workspace_bytes(w.P, w.B, w.D), dtype=torch.uint8, device=dev),
                    "A": torch.empty((w.P, w.B, w.D), device=dev), "T": torch.empty((w.P, w.B, w.D), device=dev),
                    "hout": torch.empty(out_shape, dtype=torch.float32).pin_memory()}
        e_bufs = [e2e_buffers(), e2e_buffers()]
        h2d = e_bufs[0]["hbuf"].numel()         # the bytes copied in each step, alignment included

        def e2e_step(k):
            eb = e_bufs[k % 2]
            with torch.cuda.stream(e_streams[k % 2]):
                eb["dbuf"].copy_(eb["hbuf"], non_blocking=True)
                dc, dA, dT, dout = eb["cache"], eb["A"], eb["T"], eb["out"]
                if w.layout in ("decode", "decode_prod"):
                    tq.prepare_queries(eb["Q"], eb["Pi"], eb["Pi"] if mse else eb["S"], out=(dA, dT))
                    score_call(tq, w, path, dA, dT, dc, eb["cb"], None)
                    eb["hout"].copy_(dc["dout"], non_blocking=True)
                    return
                if mse:
                    tq.prepare_queries(eb["Q"], eb["Pi"], eb["Pi"], out=(dA, dT))
                    tq.scores_mse(dA, dc["idx"], dc["norm"], eb["cb"], w.mse_bits, norm_correction=True,
                                  out=dout)
                elif w.layout == "unpacked":
                    tq.solve(eb["Q"], dc["idx"], dc["signs"], dc["gamma"], eb["Pi"], eb["S"], eb["cb"],
                             path=path, workspace=eb["ws"], out=dout)
                else:
                    tq.solve_packed(eb["Q"], dc["idx"], dc["signs"], dc["gamma"], eb["Pi"], eb["S"],
                                    eb["cb"], w.mse_bits, path=path, workspace=eb["ws"], out=dout)
                eb["hout"].copy_(dout, non_blocking=True)

        e_steps = max(4, min(args.steps, 48)) // 2 * 2
        e_ms, eager_ms = time_e2e(torch, dev, e_streams, e2e_step, e_steps, args.warmup)
        e2e = {"value": scores_per_step * e_steps / (e_ms / 1e3), "unit": "scores/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e_steps,
               "streams": 2, "graph": True,
               "eager_value": scores_per_step * e_steps / (eager_ms / 1e3)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, args.cpu_seconds)
        cpu["hardware_concurrency"] = os.cpu_count()
        cpu["value_1core"] = time_oracle_one_core(args.config, max(2.0, args.cpu_seconds / 3))
        cpu["sample"] += "; value_1core: the same sample on one pinned core, one BLAS thread"

    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "scores/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if path == "fp32" else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "P": w.P, "H": w.H, "B": w.B, "S": w.S, "D": w.D,
                   "idx_bits": w.mse_bits, "layout": w.layout, "gamma": w.gamma_dtype,
                   "queries": w.q_dtype, "path": path,
                   "l2": f"{R} rotating input/output copies, {R * per_copy / 1e6:.0f} MB > 2x L2 "
                         f"({l2 / 1e6:.0f} MB); every step reads its cache from HBM",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": ("fused transform+scoring kernel" if fused_single else
                                "decode split + combine kernels" if w.layout in ("decode", "decode_prod")
                                else "scoring kernel"),
                     "kernel_ms": kernel_ms, "bytes_per_launch": kbytes,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s",
                     "timing": ktiming, "kernel_fingerprint": fp},
        "split_ms": split_ms,
        "timed_region": {"repeats": len(regions), "median_ms": statistics.median(regions),
                         "min_ms": min(regions), "max_ms": max(regions)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (1 if fused_single else (3 if w.layout in ("decode", "decode_prod") else 2)) * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
