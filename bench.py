"""Benchmark: decode-attention throughput of libfd on GB300.

One step = one decode-attention call (every row of the hot path that the
workload uses: split planning, the per-chunk partial pass, the merge; for the
sparse workloads the fused 2-bit scan / top-delta / residual / attention pass)
over one batch of synthetic inputs already resident in HBM.

Default workload: million-token decode, B=1, Hq=32, Hkv=8, d=128,
L=1048576, bf16 KV cache with attention sinks (4 GiB of K+V per call, larger
than the 129 MB L2, so no flush is needed between calls), the largest of the
workloads that fits one GPU.  Its JSON line also carries `ffd_compare`: the
dense pass and the top-delta pass at delta 5 and 7 timed in the same process
on the same FFD cache (B=4, Hq=32, Hkv=8, d=128, L=131072), interleaved, each
arm --steps calls after --warmup calls per round.  Other workloads:
--workload tiny|mha32k|gqa_paged|million|ffd_dense|ffd_topdelta5|
ffd_topdelta7, and mha32k_fp8|million_fp8|ffd_dense_fp8|gqa_paged_fp8 (the same
caches in the fp8 e4m3 encoding, per-row f32 scales), the *_fp4 variants
(e2m1 codes with power-of-two scales per 32 channels), the *_unified variants
(one fixed max value --phi for every chunk), ffd_topdelta{5,7}_union (one
candidate set per KV group) and ffd_sparse_{dense,topdelta5[_union]} (a
sparser FFD cache: --plant-frac of the tokens and the anchors far above the
rest).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fd|reference]

With N > 1 (torchrun) every rank runs an independent replica of the
workload on its own GPU (the path has no exchange step): weak scaling.
--impl reference times the CPU oracle (the plain fp64 restatement) on the
host cores, on a bounded sample of the same workload per step.
Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention tokens/s and µs/call at 1 GB300; achieved HBM GB/s vs 8 TB/s"
NOMINAL_HBM_GBS = 8000.0  # nominal GB300 HBM3e bandwidth, the denominator of frac_of_8tbs
FALLBACK_HBM_GBS = 6800.0

DEFAULT_STEPS = {"tiny": 20000, "mha32k": 20000, "gqa_paged": 3000, "million": 3000,
                 "ffd_dense": 4000, "ffd_topdelta5": 4000, "ffd_topdelta7": 4000,
                 "mha32k_fp8": 20000, "million_fp8": 4000, "ffd_dense_fp8": 6000, "gqa_paged_fp8": 4000,
                 "mha32k_fp4": 20000, "million_fp4": 4000, "ffd_dense_fp4": 6000, "gqa_paged_fp4": 4000,
                 "mha32k_unified": 20000, "million_unified": 3000, "gqa_paged_unified": 3000,
                 "ffd_topdelta5_union": 4000, "ffd_topdelta7_union": 4000,
                 "ffd_sparse_dense": 4000, "ffd_sparse_topdelta5": 4000, "ffd_sparse_topdelta5_union": 4000,
                 "ladder": 50}
# The sparse FFD cache: anchors and planted tokens boosted by 20 along q_hat
# (a ~13-unit score lead at G=4), --plant-frac of the tokens planted.
SPARSE_BOOST = 20.0
WORKLOADS = list(DEFAULT_STEPS)


# ----------------------------------------------------------------- helpers

def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    for key in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
        if key in d:
            return float(d[key]), d
    return None


class _Nvml:
    """Read-only clock queries through the driver's NVML library (ctypes; the
    call releases the GIL), for sampling inside timed regions shorter than
    nvidia-smi's period.  Raises OSError when NVML or the device is missing."""

    CLOCK_SM = 1  # NVML_CLOCK_SM
    # clocks event reason bits (nvml.h): the four the timing rules name
    REASONS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"), (0x20, "sw_thermal_slowdown"),
               (0x4, "sw_power_cap"))

    def __init__(self, cuda_index):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        found = False
        try:  # the CUDA device's own UUID: immune to CUDA_VISIBLE_DEVICES renumbering
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
            found = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
        except Exception:
            found = False
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        self.lib, self.h = lib, h
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if self.sample() is None:
            raise OSError("NVML queries failed")

    def sample(self):
        ct = self.ct
        sm, mx, r = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(sm)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ct.byref(mx)) != 0 or
                self.reasons_fn(self.h, ct.byref(r)) != 0):
            return None
        return float(sm.value), float(mx.value), [n for bit, n in self.REASONS if r.value & bit]


class ClockSampler:
    """SM clocks and throttle reasons sampled in a thread: every 2 ms through
    NVML when the driver's library answers (so that even a timed region of a
    few milliseconds holds samples), else every 200 ms from nvidia-smi."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NVML_PERIOD_S = 0.002

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []  # (t, sm, max_sm, reasons)
        self.proc = None
        self.thread = None
        self.source = None
        self._halt = threading.Event()

    def start(self):
        try:
            nvml = _Nvml(self.gpu)
        except Exception:
            nvml = None
        if nvml is not None:
            self.source = "NVML every 2 ms"
            self.thread = threading.Thread(target=self._poll, args=(nvml,), daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi every 200 ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self, nvml):
        while not self._halt.is_set():
            s = nvml.sample()
            if s is not None:
                self.samples.append((time.time(),) + s)
            time.sleep(self.NVML_PERIOD_S)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        self._halt.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        where = "timed region"
        if not inside:
            inside = list(self.samples)
            where = "whole run (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "neither NVML nor nvidia-smi answered"}
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": where, "source": self.source}


# --------------------------------------------------------------- workloads

class Workload:
    """Resident inputs plus a `call()` that runs one decode through the C ABI."""

    def __init__(self, name, seed, device, batch=None, seq_len=None, num_splits=None, n_sink=4, window=64,
                 problem=None, encoded_keys=None, phi=6.5, plant_frac=0.001):
        """`problem` (and, for top-delta, `encoded_keys`) reuse another
        workload's resident inputs instead of generating them again."""
        import torch

        import long_context_decode_split_gb300 as fd
        import workloads as W

        self.name = name
        self.fd = fd
        self.device = device
        self.topdelta = None
        self.fp8 = name.endswith("_fp8")
        self.fp4 = name.endswith("_fp4")
        self.unified = name.endswith("_unified")
        self.group_union = name.endswith("_union")
        if self.fp8 or self.fp4:
            name = name[:-4]
        if self.unified:
            name = name[:-len("_unified")]
        if self.group_union:
            name = name[:-len("_union")]
        self.sparse = name.startswith("ffd_sparse")
        self.phi = phi
        self.n_sink, self.window = n_sink, window
        over = {}
        if seq_len is not None:
            over["L"] = seq_len
        if problem is not None:
            p = problem
            if name.startswith("ffd_top"):
                self.topdelta = 5.0 if name.endswith("5") else 7.0
        elif name == "tiny":
            p = W.tiny(seed=seed, device=device)
        elif name == "mha32k":
            p = W.mha32k(seed=seed, device=device, **over)
        elif name == "million":
            p = W.million(seed=seed, device=device, **over)
        elif name == "ladder":
            p = W.ladder(B=batch or 1, seed=seed, device=device, **over)
        elif name == "gqa_paged":
            kw = {"B": batch} if batch is not None else {}
            if seq_len is not None:
                kw.update(L_min=max(64, seq_len // 8), L_max=seq_len)
            p = W.gqa_paged(seed=seed, device=device, **kw)
        elif name.startswith("ffd"):
            if batch is not None:
                over["B"] = batch
            if self.sparse:
                over.update(anchor_boost=SPARSE_BOOST, plant_mean=SPARSE_BOOST, plant_frac=plant_frac)
            p = W.ffd(seed=seed, device=device, **over)
            if not name.endswith("_dense"):
                self.topdelta = 5.0 if name.endswith("5") else 7.0
        else:
            raise ValueError(name)
        if num_splits is not None and problem is None:
            p.num_splits = num_splits
        self.p = p
        # a dense cache smaller than L2 is rotated through enough copies that
        # consecutive calls read from HBM (the ladder's short rungs)
        self.copies = [p]
        if name == "ladder":
            for _ in range(ladder_copies(p.B, p.kv_tokens() // max(1, p.B), p.Hkv, p.d) - 1):
                self.copies.append(dataclasses.replace(p, k=p.k.clone(), v=p.v.clone()))
        self._turn = 0
        self.paged = p.paged
        self.out_dtype = p.out_dtype
        B, Hq, Hkv, d = p.B, p.Hq, p.Hkv, p.d
        # out and lse share one device buffer, so a step's result leaves the GPU in one copy
        out_t = torch.float32 if p.out_dtype == "f32" else torch.bfloat16
        n_out = B * Hq * d * (4 if p.out_dtype == "f32" else 2)
        lse_at = (n_out + 15) // 16 * 16
        self.io = torch.empty(lse_at + B * Hq * 4, dtype=torch.uint8, device=device)
        self.out = self.io[:n_out].view(out_t).view(B, Hq, d)
        self.lse = self.io[lse_at:].view(torch.float32).view(B, Hq)
        self.sel_stats = None
        if self.fp8 or self.fp4:
            # encode the cache once (outside the timed region); keep the bf16 copy for e2e rows
            enc = fd.fd_quantize_kv_fp8 if self.fp8 else fd.fd_quantize_kv_fp4
            venc = fd.fd_quantize_kv_fp8 if self.fp8 else fd.fd_quantize_v_fp4  # fp4 values: token pairs
            if self.paged:
                self.kv8 = enc(p.k_pages) + venc(p.v_pages)
            else:
                self.kv8 = enc(p.k) + venc(p.v)
            n_copies = 1 if self.paged else encoded_copies(name, p.B, p.L_max, p.Hkv, p.d)
            self.kv8_copies = [self.kv8] + [tuple(t.clone() for t in self.kv8) for _ in range(n_copies - 1)]
            torch.cuda.synchronize()
            if self.fp8:
                need = fd.fd_decode_fp8_workspace_size(B, Hq, Hkv, p.L_max, d, p.num_splits, self.paged)
                self.splits = fd.fd_num_splits_fp8(B, Hq, Hkv, p.L_max, d, p.num_splits, self.paged)
            else:
                need = fd.fd_decode_fp4_workspace_size(B, Hq, Hkv, p.L_max, d, p.num_splits, self.paged)
                self.splits = fd.fd_num_splits_fp4(B, Hq, Hkv, p.L_max, d, p.num_splits, self.paged)
        elif self.topdelta is not None:
            self.qk = encoded_keys if encoded_keys is not None else fd.fd_quantize_keys(p.k, p.seq_lens)
            need = fd.fd_topdelta_workspace_size(B, Hq, Hkv, p.L_max, d, p.num_splits)
            self.splits = None
            self.sel_stats = self._selection_stats()
        else:
            need = fd.fd_decode_workspace_size(B, Hq, Hkv, p.L_max, d, p.num_splits, self.paged)
            self.splits = fd.fd_num_splits(B, Hq, Hkv, p.L_max, d, p.num_splits, self.paged)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.kv_tokens = p.kv_tokens()

    def _selection_stats(self):
        """One inspection call: candidate counts per query head, their union per
        KV head (what the method must read residual + V for) and the 64-token
        tiles that hold any candidate (what the kernel actually loads)."""
        import numpy as np
        import torch

        p, fd = self.p, self.fd
        c, ms, r, rs = self.qk
        out_s, lse_s, mask, cnt = fd.fd_decode_topdelta(p.q, c, ms, r, rs, p.v, p.seq_lens, p.scale, self.topdelta,
                                                        self.n_sink, self.window, p.num_splits,
                                                        out_dtype=self.out_dtype, want_selection=True,
                                                        group_union=self.group_union)
        # quality proxy: the dense softmax mass the candidate set captures, exp(lse_sel - lse_dense),
        # and the largest output deviation from dense attention over the bf16 keys
        out_d, lse_d = fd.fd_decode_dense(p.q, p.k, p.v, p.seq_lens, p.scale, out_dtype=self.out_dtype)
        mass = torch.exp(lse_s - lse_d)
        dev = (out_s.float() - out_d.float()).abs().max().item()
        m = mask.cpu().numpy().view(np.uint32)
        B, Hq, W_ = m.shape
        G = Hq // p.Hkv
        union = np.bitwise_or.reduce(m.reshape(B, p.Hkv, G, W_), axis=2)       # [B, Hkv, words]
        ubits = np.unpackbits(union.view(np.uint8), bitorder="little").reshape(B, p.Hkv, -1)
        pad = (-ubits.shape[-1]) % 64
        tiles = np.pad(ubits, ((0, 0), (0, 0), (0, pad))).reshape(B, p.Hkv, -1, 64).any(axis=-1)
        L = p.kv_tokens() / B
        # the key quantization's share of that deviation: attention with the bf16 keys over the same
        # candidate sets (KV head 0 and its query heads; plain fp32 torch, informational only)
        bits_h = np.unpackbits(m[:, :G].view(np.uint8), bitorder="little").reshape(B, G, -1)[:, :, :p.L_max]
        sel_h = torch.from_numpy(bits_h.astype(bool)).to(p.q.device)
        s_h = torch.einsum("bgd,bld->bgl", p.q[:, :G].float(), p.k[:, 0].float()) * p.scale
        s_h = s_h.masked_fill(~sel_h, -math.inf)
        w_h = torch.softmax(s_h, dim=-1).nan_to_num(0.0)
        o_h = torch.einsum("bgl,bld->bgd", w_h, p.v[:, 0].float())
        dev_q = (out_s[:, :G].float() - o_h).abs().max().item()
        return {"selected_per_query": float(cnt.float().mean().item()) / L,
                "attended": "group union" if self.group_union else "per query head",
                "captured_mass_min": float(mass.min().item()), "captured_mass_mean": float(mass.mean().item()),
                "max_abs_dev_vs_dense": dev,
                "max_abs_dev_vs_bf16_keys_same_selection": dev_q,
                "union_per_kv_head": float(ubits.sum()) / (B * p.Hkv * L),
                "union_tokens": int(ubits.sum()), "tiles_loaded": int(tiles.sum()),
                "tiles_total": int(tiles.size)}

    def call(self, stream=None, q=None, rotate=True):
        """One decode call; with `rotate` consecutive calls read the cache's
        copies in turn (the end-to-end step, which writes the newest row into
        the cache it then reads, passes rotate=False)."""
        fd = self.fd
        turn = self._turn if rotate else 0
        self._turn += 1 if rotate else 0
        p = self.copies[turn % len(self.copies)]
        q = p.q if q is None else q
        if self.fp8 or self.fp4:
            kc, ks, vc, vs = self.kv8_copies[turn % len(self.kv8_copies)]
            if self.paged:
                paged = fd.fd_decode_paged_fp8 if self.fp8 else fd.fd_decode_paged_fp4
                paged(q, kc, ks, vc, vs, p.page_table, p.num_pages, p.seq_lens, p.scale, p.num_splits,
                      out=self.out, lse=self.lse, out_dtype=self.out_dtype, workspace=self.ws, stream=stream)
            else:
                dense = fd.fd_decode_dense_fp8 if self.fp8 else fd.fd_decode_dense_fp4
                dense(q, kc, ks, vc, vs, None, p.scale, p.num_splits, out=self.out, lse=self.lse,
                      out_dtype=self.out_dtype, workspace=self.ws, stream=stream)
        elif self.topdelta is not None:
            c, ms, r, rs = self.qk
            fd.fd_decode_topdelta(q, c, ms, r, rs, p.v, p.seq_lens, p.scale, self.topdelta, self.n_sink,
                                  self.window, p.num_splits, out=self.out, lse=self.lse, out_dtype=self.out_dtype,
                                  workspace=self.ws, stream=stream, group_union=self.group_union)
        elif self.unified and self.paged:
            fd.fd_decode_paged_unified(q, p.k_pages, p.v_pages, p.page_table, p.num_pages, p.seq_lens, p.scale,
                                       self.phi, p.num_splits, out=self.out, lse=self.lse, out_dtype=self.out_dtype,
                                       workspace=self.ws, stream=stream)
        elif self.unified:
            fd.fd_decode_dense_unified(q, p.k, p.v, None, p.scale, self.phi, p.num_splits, out=self.out, lse=self.lse,
                                       out_dtype=self.out_dtype, workspace=self.ws, stream=stream)
        elif self.paged:
            fd.fd_decode_paged(q, p.k_pages, p.v_pages, p.page_table, p.num_pages, p.seq_lens, p.scale,
                               p.num_splits, out=self.out, lse=self.lse, out_dtype=self.out_dtype,
                               workspace=self.ws, stream=stream)
        else:
            fd.fd_decode_dense(q, p.k, p.v, None, p.scale, p.num_splits, out=self.out, lse=self.lse,
                               out_dtype=self.out_dtype, workspace=self.ws, stream=stream)

    def launches_per_call(self):
        if self.topdelta is not None:
            return 2  # fused pass + merge
        return 1 if self.splits == 1 else 2

    def algorithmic_bytes(self, topdelta_union=None):
        """HBM bytes the method must move per call (K/V or 2-bit body + residual + V,
        plus q in and out/lse out)."""
        p = self.p
        B, Hq, Hkv, d = p.B, p.Hq, p.Hkv, p.d
        io = B * Hq * d * 2 + B * Hq * d * (4 if p.out_dtype == "f32" else 2) + B * Hq * 4
        if self.fp8:
            return self.kv_tokens * Hkv * (d + 4) * 2 + io  # K and V codes + their row scales
        if self.fp4:
            return self.kv_tokens * Hkv * (d // 2 + d // 32) * 2 + io  # codes + block exponents
        if self.topdelta is None:
            return self.kv_tokens * Hkv * d * 2 * 2 + io
        scan = self.kv_tokens * Hkv * (d // 4 + (d // 32) * 4)
        union = topdelta_union if topdelta_union is not None else self.sel_stats["union_tokens"]
        detail = union * (d + (d // 32) * 2 + d * 2)
        return scan + detail + io

    def algorithmic_flops(self):
        """Floating-point operations the method performs per call: 4d per (query
        head, attended token) for q.k and p.v, plus 2d per (query head, scanned
        token) for the top-delta 2-bit scan."""
        p = self.p
        if self.topdelta is None:
            return self.kv_tokens * p.Hq * 4 * p.d
        st = self.sel_stats
        if self.group_union:
            attended = st["union_tokens"] * (p.Hq // p.Hkv)
        else:
            attended = st["selected_per_query"] * self.kv_tokens * p.Hq
        return self.kv_tokens * p.Hq * 2 * p.d + attended * 4 * p.d

    def plan(self):
        """What this run's inputs and the library's planner made of the workload
        (known only once the inputs exist and the device is queried)."""
        p = self.p
        c = {"kv_tokens": self.kv_tokens,
             "chunks_per_sequence": self.splits if self.splits is not None else
             ("planner (top-delta)" if not p.num_splits else p.num_splits),
             "launches_per_call": self.launches_per_call()}
        if self.topdelta is not None:
            c.update(selection=self.sel_stats, dense_equivalent_bytes=self.kv_tokens * p.Hkv * p.d * 4)
        return c


L2_BYTES = 129 * 1024 * 1024


def ladder_copies(B, L, Hkv, d):
    """Copies of a ladder cache that together exceed three times the L2."""
    return max(1, -(-3 * L2_BYTES // (B * L * Hkv * d * 4)))


def encoded_copies(name, B, L, Hkv, d):
    """Copies of an fp8/fp4 cache read in turn: a cache less than twice the L2
    could partly stay resident from one call to the next, so it gets enough
    copies to exceed three times the L2 together."""
    if not name.endswith(("_fp8", "_fp4")) or not isinstance(L, int):
        return 1
    per_token = 2 * (d + 4) if name.endswith("_fp8") else 2 * (d // 2 + d // 32)
    nbytes = B * L * Hkv * per_token
    return 1 if nbytes >= 2 * L2_BYTES else -(-3 * L2_BYTES // nbytes)


def workload_config(args):
    """The workload as the command line names it: the same dict in the GPU
    arm and in the reference arm (nothing here depends on the device)."""
    name = args.workload
    base = name[:-4] if name.endswith(("_fp8", "_fp4")) else name
    base = base[:-len("_unified")] if base.endswith("_unified") else base
    B, Hq, Hkv, L, d = FULL_SHAPES[name]
    if args.batch is not None and (base in ("gqa_paged", "ladder") or base.startswith("ffd")):
        B = args.batch
    if base == "gqa_paged":
        hi = args.seq_len if args.seq_len is not None else 131072
        lo = max(64, hi // 8) if args.seq_len is not None else 16384
        L = f"U{{{lo}..{hi}}} per sequence"
    elif args.seq_len is not None and base in ("mha32k", "million", "ladder"):
        L = args.seq_len
    kv = ("e4m3 codes + f32 row scales" if name.endswith("_fp8") else
          "e2m1 codes + power-of-two scales per 32 channels" if name.endswith("_fp4") else "bf16")
    c = {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d, "L": L,
         "cache": "paged-64" if base == "gqa_paged" else "contiguous",
         "out_dtype": "f32" if base == "tiny" else "bf16", "kv_dtype": kv,
         "num_splits": "planner" if not args.num_splits else args.num_splits,
         **({"split_sweep": True} if getattr(args, "split_sweep", False) else {}),
         "l2": "inputs smaller than L2: a 512 MiB write before each call, outside its CUDA events"
               if base == "tiny" else "inputs larger than L2",
         **({"l2": f"{ladder_copies(B, L, Hkv, d)} copies of the cache read in turn (together larger than L2)"}
            if base == "ladder" and ladder_copies(B, L, Hkv, d) > 1 else {}),
         **({"l2": f"{encoded_copies(name, B, L, Hkv, d)} copies of the encoded cache read in turn "
                   f"(together more than three times the L2)"}
            if encoded_copies(name, B, L, Hkv, d) > 1 else {}),
         "parallelism": f"replicas x{args.gpus}"}
    if base == "tiny":
        c["num_splits"] = args.num_splits or 4
    top = base[:-len("_union")] if base.endswith("_union") else base
    if top.startswith("ffd") and not top.endswith("_dense"):
        c.update(delta=5.0 if top.endswith("5") else 7.0, n_sink=args.n_sink, window=args.window,
                 selection="group union" if base.endswith("_union") else "per query head")
    if base.startswith("ffd_sparse"):
        c["keys"] = (f"sparse FFD cache: sinks, last 64 tokens and {args.plant_frac:g} of the tokens "
                     f"+{SPARSE_BOOST:g} q_hat")
    if name.endswith("_unified"):
        c["softmax"] = f"unified max value phi={args.phi} (FlashDecoding++), running-max fallback"
    if args.graph:
        c["timing"] = f"CUDA graph of {args.graph} calls, replayed"
    return c


# ------------------------------------------------------------------ timing

FLUSH_BYTES = 512 * 1024 * 1024


def time_device_flushed(wl, steps, warmup, dist_ctx):
    """For inputs smaller than L2: each call timed alone with CUDA events,
    a 512 MiB write before it (outside its events) so that it reads its
    inputs from HBM.  The host enqueues the next call while the device is
    still writing, so the events bracket device time only.  Returns the sum
    of the calls' times (ms), as time_device does for its steps."""
    import torch

    stream = torch.cuda.current_stream()
    scratch = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=wl.device)
    for _ in range(warmup):
        wl.call()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t_wall0 = time.time()
    for a, b in evs:
        scratch.fill_(1.0)
        a.record(stream)
        wl.call()
        b.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    dist_ctx.barrier()
    ms = sum(a.elapsed_time(b) for a, b in evs)
    return dist_ctx.max(ms), (t_wall0, t_wall1), steps


def time_device(wl, steps, warmup, dist_ctx, graph=0):
    """CUDA-event time of `steps` calls on the current stream.  With graph > 0
    the calls are captured `graph` at a time into a CUDA graph and replayed,
    so host-side overhead (Python, argument checks) leaves the measurement."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        wl.call()
    torch.cuda.synchronize()
    g = None
    if graph > 0:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(graph):
                    wl.call()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        steps = max(graph, steps // graph * graph)
    dist_ctx.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    if g is not None:
        for _ in range(steps // graph):
            g.replay()
    else:
        for _ in range(steps):
            wl.call()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    dist_ctx.barrier()
    ms = ev0.elapsed_time(ev1)
    return dist_ctx.max(ms), (t_wall0, t_wall1), steps


def time_e2e(wl, steps, warmup, dist_ctx):
    """Same call through the public API, with this step's new inputs copied
    from pinned host memory and the result read back, inside the timed
    region.  Per step: one host->device copy of the query and the newest
    token's K/V rows (packed in one pinned buffer), the rows written into the
    cache in the form the decode reads (bf16 rows; fp8/fp4 codes and scales
    from the cache encoder; for top-delta the key encoding from
    fd_quantize_keys plus the bf16 V row), the decode call on the copied
    query, and one device->host copy of out and lse."""
    import torch

    p = wl.p
    fd = wl.fd
    dev = wl.device
    # newest token of every sequence: (page, row) in the paged pool, else position L_max - 1
    if wl.paged:
        lens = p.seq_lens.cpu().tolist()
        tgt = [(int(p.page_table[b, (L - 1) // 64]), (L - 1) % 64) for b, L in enumerate(lens) if L > 0]
        pg = torch.tensor([t[0] for t in tgt], dtype=torch.long, device=dev)
        rr = torch.tensor([t[1] for t in tgt], dtype=torch.long, device=dev)
        k_rows, v_rows = p.k_pages[pg, :, rr], p.v_pages[pg, :, rr]  # [n, Hkv, d]
    else:
        k_rows, v_rows = p.k[:, :, p.L_max - 1], p.v[:, :, p.L_max - 1]  # [B, Hkv, d]
    n, H, dd = k_rows.shape
    nq, nr = p.q.numel() * 2, k_rows.numel() * 2
    host = torch.empty(nq + 2 * nr, dtype=torch.uint8).pin_memory()
    host[:nq].view(torch.bfloat16).copy_(p.q.reshape(-1).cpu())
    host[nq:nq + nr].view(torch.bfloat16).copy_(k_rows.reshape(-1).cpu())
    host[nq + nr:].view(torch.bfloat16).copy_(v_rows.reshape(-1).cpu())
    staged = torch.empty_like(host, device=dev)
    q_d = staged[:nq].view(torch.bfloat16).view(p.q.shape)
    k_d = staged[nq:nq + nr].view(torch.bfloat16).view(n, H, dd)
    v_d = staged[nq + nr:].view(torch.bfloat16).view(n, H, dd)
    kv_d = staged[nq:].view(torch.bfloat16).view(2 * n, H, 1, dd)  # K rows, then V rows, as one-token caches
    result = torch.empty(wl.io.shape, dtype=torch.uint8).pin_memory()

    if wl.fp8:
        c_new = torch.empty((2 * n, H, 1, dd), dtype=torch.uint8, device=dev)
        s_new = torch.empty((2 * n, H, 1), dtype=torch.float32, device=dev)
        encode = fd.fd_quantize_kv_fp8
    elif wl.fp4:
        # keys: one row; values: the newest token's pair (tokens 2j, 2j + 1) encoded again, its
        # partner read from the bf16 cache when the newest token is the second of the pair
        kc_new = torch.empty((n, H, 1, dd // 2), dtype=torch.uint8, device=dev)
        ks_new = torch.empty((n, H, 1, dd // 32), dtype=torch.uint8, device=dev)
        vc_new = torch.empty((n, H, 1, dd), dtype=torch.uint8, device=dev)
        vs_new = torch.empty((n, H, 2, dd // 32), dtype=torch.uint8, device=dev)
        if wl.paged:
            odd = (rr % 2) == 1
            prev = p.v_pages[pg, :, torch.clamp(rr - 1, min=0)]
        else:
            odd = torch.full((n,), (p.L_max - 1) % 2 == 1, device=dev)
            prev = p.v[:, :, max(p.L_max - 2, 0)]
        # the partner of an odd newest token is already in the cache: place it once; each step
        # writes the newest row into its slot of the pair (1 when odd, 0 when even)
        pair_x = torch.zeros((n, H, 2, dd), dtype=torch.bfloat16, device=dev)
        pair_x[:, :, 0] = torch.where(odd.view(n, 1, 1), prev, torch.zeros_like(prev))
        pair_len = torch.where(odd, 2, 1).to(torch.int32)
        slot = odd.long()
        ar = torch.arange(n, device=dev)
    elif wl.topdelta is not None:
        k_one = staged[nq:nq + nr].view(torch.bfloat16).view(n, H, 1, dd)
        enc_new = (torch.empty((n, H, 1, dd // 4), dtype=torch.uint8, device=dev),
                   torch.empty((n, H, 1, dd // 32, 2), dtype=torch.float16, device=dev),
                   torch.empty((n, H, 1, dd), dtype=torch.int8, device=dev),
                   torch.empty((n, H, 1, dd // 32), dtype=torch.float16, device=dev))

    def put(cache, rows, pairs=False):
        """Write one row per (sequence, head) at the newest token's position
        (with pairs: at its pair row)."""
        if wl.paged:
            cache[pg, :, rr // 2 if pairs else rr] = rows
        else:
            cache[:, :, (p.L_max - 1) // 2 if pairs else p.L_max - 1] = rows

    def step():
        staged.copy_(host, non_blocking=True)
        if wl.fp8:
            encode(kv_d, codes=c_new, scales=s_new)
            kc, ks, vc, vs = wl.kv8
            put(kc, c_new[:n, :, 0])
            put(ks, s_new[:n, :, 0])
            put(vc, c_new[n:, :, 0])
            put(vs, s_new[n:, :, 0])
        elif wl.fp4:
            kc, ks, vc, vs = wl.kv8
            fd.fd_quantize_kv_fp4(k_d.view(n, H, 1, dd), codes=kc_new, scales=ks_new)
            put(kc, kc_new[:, :, 0])
            put(ks, ks_new[:, :, 0])
            pair_x[ar, :, slot] = v_d
            fd.fd_quantize_v_fp4(pair_x, pair_len, codes=vc_new, scales=vs_new)
            put(vc, vc_new[:, :, 0], pairs=True)
            put(vs, vs_new[ar, :, slot])
        elif wl.topdelta is not None:
            fd.fd_quantize_keys(k_one, None, *enc_new)
            for cache, row in zip(wl.qk, enc_new):
                put(cache, row[:, :, 0])
            put(p.v, v_d)
        elif wl.paged:
            put(p.k_pages, k_d)
            put(p.v_pages, v_d)
        else:
            put(p.k, k_d)
            put(p.v, v_d)
        wl.call(q=q_d, rotate=False)
        result.copy_(wl.io, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    dist_ctx.barrier()
    return dist_ctx.max((t1 - t0) * 1e3), host.numel(), result.numel()


def split_sweep(args, wl, ctx):
    """Chunk counts around the planner's choice for the same inputs: median
    and spread of --rounds rounds of --steps calls each (dense bf16 only)."""
    p = wl.p
    planned = wl.splits
    cands = sorted({max(1, int(round(planned * f))) for f in (0.5, 0.75, 1.0, 1.25, 1.5, 2.0)})
    res = []
    for S in cands:
        w = Workload(wl.name, 0, wl.device, problem=dataclasses.replace(p, num_splits=S))
        us = []
        for _ in range(max(1, args.rounds)):
            ms, _, steps = time_device(w, args.steps, args.warmup, ctx)
            us.append(ms * 1e3 / steps)
        res.append({"num_splits": S, "planner": S == planned, "median_us": statistics.median(us),
                    "min_us": min(us), "max_us": max(us),
                    "gbs": w.algorithmic_bytes() / (statistics.median(us) * 1e-6) / 1e9})
    return res


def ffd_compare(args, ctx, sampler, dev):
    """Dense pass vs top-delta at delta 5 and 7 on one FFD cache (B=4, Hq=32,
    Hkv=8, d=128, L=131072; the same K/V, the keys encoded once): `rounds`
    interleaved rounds, in each every arm times --steps calls after --warmup
    calls with CUDA events; medians over the rounds."""
    seed = args.seed + ctx.rank
    dense = Workload("ffd_dense", seed, dev)
    td5 = Workload("ffd_topdelta5", seed, dev, problem=dense.p)
    td7 = Workload("ffd_topdelta7", seed, dev, problem=dense.p, encoded_keys=td5.qk)
    arms = (("dense", dense), ("topdelta5", td5), ("topdelta7", td7))
    rounds = 3
    us = {n: [] for n, _ in arms}
    t0 = time.time()
    for _ in range(rounds):
        for n, wl in arms:
            ms, _, steps = time_device(wl, args.steps, args.warmup, ctx)
            us[n].append(ms * 1e3 / steps)
    t1 = time.time()
    med = {n: statistics.median(v) for n, v in us.items()}
    res = {"workload": "ffd: B=4, Hq=32, Hkv=8, d=128, L=131072, sinks and last 64 tokens +2.5 q_hat, "
                       "1% of tokens +N(2,0.5) q_hat; n_sink=4, window=64",
           "rounds": rounds, "steps_per_round": args.steps, "warmup_per_round": args.warmup,
           "us_per_call": med, "us_per_call_rounds": us,
           "achieved_gbs": {n: wl.algorithmic_bytes() / (med[n] * 1e-6) / 1e9 for n, wl in arms},
           "algorithmic_bytes": {n: wl.algorithmic_bytes() for n, wl in arms},
           "topdelta5_speedup_vs_dense": med["dense"] / med["topdelta5"],
           "topdelta7_speedup_vs_dense": med["dense"] / med["topdelta7"],
           "selection": {"topdelta5": td5.sel_stats, "topdelta7": td7.sel_stats},
           "clocks": sampler.summary(t0, t1)}
    return res


# ------------------------------------------------------------ CPU oracle

FULL_SHAPES = {"tiny": (1, 1, 1, 1024, 64), "mha32k": (1, 32, 32, 32768, 128),
               "million": (1, 32, 8, 1 << 20, 128), "gqa_paged": (8, 64, 8, 73728, 128),
               "ffd_dense": (4, 32, 8, 131072, 128), "ffd_topdelta5": (4, 32, 8, 131072, 128),
               "ffd_topdelta7": (4, 32, 8, 131072, 128)}
FULL_SHAPES.update({k + "_fp8": FULL_SHAPES[k] for k in ("mha32k", "million", "gqa_paged", "ffd_dense")})
FULL_SHAPES.update({k + "_fp4": FULL_SHAPES[k] for k in ("mha32k", "million", "gqa_paged", "ffd_dense")})
FULL_SHAPES.update({k + "_unified": FULL_SHAPES[k] for k in ("mha32k", "million", "gqa_paged")})
FULL_SHAPES.update({k: FULL_SHAPES["ffd_dense"] for k in WORKLOADS if k.startswith("ffd")})
FULL_SHAPES["ladder"] = (1, 32, 8, 32768, 128)


class OracleSample:
    """A bounded slice of a workload for the CPU oracle: the first `heads` KV
    heads (with their query groups) and the first `Ls` tokens of every
    sequence.  `frac` is the slice's share of one full call's work.  For the
    ragged paged batch the full call is taken at the mean length."""

    def __init__(self, name, seed, target_s, plant_frac=0.001, batch=None, seq_len=None):
        import numpy as np
        import torch

        import oracle
        import workloads as W

        self.name = name
        self.oracle = oracle
        B, Hq, Hkv, L, d = FULL_SHAPES[name]
        if batch is not None and (name == "ladder" or name.startswith("ffd")):
            B = batch
        if seq_len is not None and name.split("_")[0] in ("mha32k", "million", "ladder"):
            L = seq_len
        self.fp8 = name.endswith("_fp8")
        self.fp4 = name.endswith("_fp4")
        G = Hq // Hkv
        self.B = B
        self.delta = None
        self.union = name.endswith("_union")
        top = name[:-len("_union")] if self.union else name
        if top.startswith("ffd") and not top.endswith("_dense"):
            self.delta = 5.0 if top.endswith("5") else 7.0

        def bits(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)

        heads, Ls = 1, min(L, 2048)
        while True:
            if name.startswith("ffd_sparse"):
                p = W.ffd(seed=seed, B=B, L=Ls, Hq=heads * G, Hkv=heads, d=d, anchor_boost=SPARSE_BOOST,
                          plant_mean=SPARSE_BOOST, plant_frac=plant_frac)
            elif name.startswith("ffd"):
                p = W.ffd(seed=seed, B=B, L=Ls, Hq=heads * G, Hkv=heads, d=d)
            else:
                p = W.random_problem(B, heads * G, heads, Ls, d, seed=seed)
            self.args = (bits(p.q), bits(p.k), bits(p.v), p.scale)
            if self.delta is not None:
                self.enc = oracle.quantize_keys(self.args[1])
            if self.fp8:
                self.enc = oracle.quantize_kv_fp8(self.args[1]) + oracle.quantize_kv_fp8(self.args[2])
            if self.fp4:  # values in the token-pair layout the fp4 decode reads
                self.enc = oracle.quantize_kv_fp4(self.args[1]) + oracle.quantize_v_fp4(self.args[2])
            t0 = time.perf_counter()
            self.run()
            dt = time.perf_counter() - t0
            if dt >= target_s / 2 or (heads == Hkv and Ls == L):
                break
            grow = max(2, min(8, int(target_s / max(dt, 1e-4))))
            if Ls < L:
                Ls = min(L, Ls * grow)
            else:
                heads = min(Hkv, heads * 2)
        self.frac = (heads / Hkv) * (Ls / L)
        self.desc = (f"{heads} of {Hkv} KV heads (with their query heads) x first {Ls} of {L} tokens, "
                     f"B={B}, d={d}: {self.frac:.4g} of one full call")
        self.threads = oracle.max_threads()

    def run(self, n_threads=0):
        """One pass of the oracle over the sample (n_threads 0: every core)."""
        q, k, v, scale = self.args
        if self.fp8:
            kc, ks, vc, vs = self.enc
            self.oracle.decode_dense_fp8(q, kc, ks, vc, vs, None, scale, n_threads=n_threads)
        elif self.fp4:
            kc, ks, vc, vs = self.enc
            self.oracle.decode_dense_fp4(q, kc, ks, vc, vs, None, scale, n_threads=n_threads)
        elif self.delta is not None:
            c, ms, r, rs = self.enc
            fn = self.oracle.decode_topdelta_group_union if self.union else self.oracle.decode_topdelta
            fn(q, c, ms, r, rs, v, None, scale, self.delta, n_threads=n_threads)
        else:
            self.oracle.decode_dense(q, k, v, None, scale, n_threads=n_threads)


def time_oracle(sample, steps, warmup):
    """Returns (tokens/s of full calls, seconds per step)."""
    for _ in range(warmup):
        sample.run()
    t0 = time.perf_counter()
    for _ in range(steps):
        sample.run()
    dt = time.perf_counter() - t0
    per_call = dt / steps / sample.frac
    return sample.B / per_call, dt / steps


# ---------------------------------------------------------------- context

class DistCtx:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x):
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([float(x)], device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x):
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([float(x)], device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------- main

def run_reference(args, ctx):
    """The oracle as it stands, on the host cores: W warm-up and K timed
    steps, each one bounded sample of the workload; value in the fd arm's unit."""
    if ctx.rank != 0:
        return
    per_step = max(0.002, min(2.0, 90.0 / max(1, args.steps + args.warmup)))
    sample = OracleSample(args.workload, args.seed, per_step, args.plant_frac, args.batch, args.seq_len)
    value, s_per_step = time_oracle(sample, args.steps, args.warmup)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": sample.threads, "kind": "oracle",
                             "sample": sample.desc + " per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--workload", default="million", choices=WORKLOADS)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=None, help="override B (gqa_paged, ffd_*)")
    ap.add_argument("--seq-len", type=int, default=None, help="override L (L_max for gqa_paged)")
    ap.add_argument("--num-splits", type=int, default=None, help="chunks per sequence (0 = planner)")
    ap.add_argument("--graph", type=int, default=0, help="replay calls from a CUDA graph of this many calls")
    ap.add_argument("--n-sink", type=int, default=4, help="top-delta: attention-sink anchors")
    ap.add_argument("--window", type=int, default=64, help="top-delta: local-window anchors")
    ap.add_argument("--phi", type=float, default=6.5, help="*_unified: the fixed max value (natural-log units)")
    ap.add_argument("--plant-frac", type=float, default=0.001, help="ffd_sparse_*: fraction of planted tokens")
    ap.add_argument("--rounds", type=int, default=1, help="timed rounds of --steps calls (value = median)")
    ap.add_argument("--split-sweep", action="store_true",
                    help="also time chunk counts around the planner's (0.5x..2x), --rounds rounds each")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ffd-compare", choices=["auto", "on", "off"], default="auto",
                    help="time dense vs top-delta 5/7 on the FFD cache in the same run (auto: with million)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]
    args.warmup = max(3, args.warmup)

    ctx = DistCtx()
    if args.impl == "reference":
        ctx.init("gloo")
        run_reference(args, ctx)
        ctx.close()
        return

    import torch

    torch.cuda.set_device(ctx.local_rank)
    ctx.init("nccl")
    import long_context_decode_split_gb300 as fd

    fd.load()
    dev = f"cuda:{ctx.local_rank}"
    wl = Workload(args.workload, args.seed + ctx.rank, dev, batch=args.batch, seq_len=args.seq_len,
                  num_splits=args.num_splits, n_sink=args.n_sink, window=args.window, phi=args.phi,
                  plant_frac=args.plant_frac)

    sampler = ClockSampler(ctx.local_rank)
    sampler.start()
    time.sleep(0.3)
    rounds_ms = []
    for _ in range(max(1, args.rounds)):
        if args.workload == "tiny" and not args.graph:
            ms_r, (tw0_r, tw1), steps_r = time_device_flushed(wl, min(args.steps, 2000), args.warmup, ctx)
        else:
            ms_r, (tw0_r, tw1), steps_r = time_device(wl, args.steps, args.warmup, ctx, graph=args.graph)
        rounds_ms.append(ms_r)
        tw0 = tw0_r if len(rounds_ms) == 1 else tw0
    args.steps = steps_r
    ms = statistics.median(rounds_ms)
    sampler_summary = sampler.summary(tw0, tw1)
    sweep = None
    if args.split_sweep:
        sweep = split_sweep(args, wl, ctx)
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 2000))
        ms_e2e, h2d, d2h = time_e2e(wl, e2e_steps, args.warmup, ctx)
    compare = None
    if args.ffd_compare == "on" or (args.ffd_compare == "auto" and args.workload == "million"):
        compare = ffd_compare(args, ctx, sampler, dev)
    sampler.stop()

    status = fd.fd_device_status(clear=True)
    B = wl.p.B
    n = ctx.world
    per_call_s = ms / 1e3 / args.steps
    value = n * B * args.steps / (ms / 1e3)
    algo = wl.algorithmic_bytes()
    flops = wl.algorithmic_flops()
    achieved_gbs = algo / per_call_s / 1e9
    peak = measured_peaks()
    if peak is not None:
        peak_gbs, peak_src = peak[0], "measured (MEASURED_PEAKS.json hbm copy)"
    else:
        peak_gbs, peak_src = FALLBACK_HBM_GBS, "fallback (6.8 TB/s, no MEASURED_PEAKS.json)"
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        try:
            with open(tfile) as f:
                tj = json.load(f)
            ent = tj.get(args.workload)
            if ent and ent.get("source_sha") == source_digest(args.workload):
                traffic = ent.get("dram_bytes_per_launch")
        except (OSError, ValueError):
            traffic = None
    if not args.no_e2e:
        e2e = {"value": n * B * e2e_steps / (ms_e2e / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "note": "per step: one host->device copy (query + newest token's K/V rows), the rows written "
                       "into the cache in the form the decode reads (encoded for fp8/fp4/top-delta), the "
                       "decode, one device->host copy (out + lse)"}
    cpu = None
    if ctx.rank == 0 and n == 1 and not args.no_cpu_baseline:
        sample = OracleSample(args.workload, args.seed, 1.0, args.plant_frac, args.batch, args.seq_len)
        t0 = time.perf_counter()
        sample.run()
        reps = max(1, int(args.cpu_budget / max(time.perf_counter() - t0, 1e-3)))
        v, s_rep = time_oracle(sample, reps, 1)
        cpu = {"value": v, "unit": "tokens/s", "cores": sample.threads, "kind": "oracle",
               "sample": f"{sample.desc}; {reps} timed runs of {s_rep * 1e3:.1f} ms"}
        if args.workload in ("tiny", "mha32k"):
            # the same sample on one core, once
            t0 = time.perf_counter()
            sample.run(n_threads=1)
            dt1 = time.perf_counter() - t0
            cpu["single_thread"] = {"value": sample.B / (dt1 / sample.frac), "unit": "tokens/s", "cores": 1,
                                    "seconds": dt1}
    if ctx.rank == 0:
        cfg = workload_config(args)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "kv_dtype": "e4m3" if wl.fp8 else "e2m1" if wl.fp4 else "bf16",
            "data": "synthetic", "config": cfg, "plan": wl.plan(),
            "us_per_call": per_call_s * 1e6,
            "kv_tokens_per_s": wl.kv_tokens * n / per_call_s,
            "achieved_hbm_gbs": achieved_gbs,
            "frac_of_8tbs": achieved_gbs / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
                         "frac": achieved_gbs / peak_gbs, "traffic": traffic, "peak_source": peak_src,
                         "kernel": "split partial pass + merge (whole call)",
                         "algorithmic_bytes_per_launch": algo},
            "compute": {"algorithmic_flops_per_call": flops, "achieved_tflops": flops / per_call_s / 1e12,
                        "flop_per_byte": flops / algo},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * wl.launches_per_call(),
            "clocks": sampler_summary,
            "device_status": fd.fd_status_string(status),
        }
        if compare is not None:
            line["ffd_compare"] = compare
        if args.rounds > 1:
            line["rounds"] = {"n": len(rounds_ms), "us_per_call": [r * 1e3 / args.steps for r in rounds_ms],
                              "median_us": ms * 1e3 / args.steps,
                              "spread_us": (max(rounds_ms) - min(rounds_ms)) * 1e3 / args.steps}
        if sweep is not None:
            line["split_sweep"] = sweep
        print(json.dumps(line), flush=True)
    ctx.close()


KERNEL_SOURCES = {"bf16": "fd_decode.cu", "topdelta": "fd_topdelta.cu", "fp8": "fd_fp8.cu", "fp4": "fd_fp4.cu"}


def kernel_family(workload):
    if workload.endswith("_fp8"):
        return "fp8"
    if workload.endswith("_fp4"):
        return "fp4"
    if workload.startswith("ffd") and not workload.endswith("_dense"):
        return "topdelta"
    return "bf16"


def source_digest(workload):
    """Digest of the sources that define a workload's kernels and their launch
    plan: the kernel's translation unit, the shared device/host headers and
    the C-ABI layer (which picks the chunk count)."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "long_context_decode_split_gb300", "csrc")
    files = sorted(f for f in os.listdir(csrc) if f.endswith((".cuh", ".h")))
    files += ["fd_api.cu", KERNEL_SOURCES[kernel_family(workload)]]
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
