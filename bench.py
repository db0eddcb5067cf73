#!/usr/bin/env python3
"""Benchmark of the FP8 fine-grained-scaled GEMM library on GB300.

`python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                 [--workload all|dense_tiny|dense_decode|dense_prefill|
                             grouped_contiguous|grouped_masked|...]
                 [--case I]`

Prints one JSON line.  By default (`--workload all`) every workload of the
method's benchmark runs in one process: the dense tiny case, the dense decode
sweep (M in {64, 128}), the dense prefill sweep (M = 4096) over six (N, K)
pairs of the DeepSeek-V3/R1 inference shapes, the contiguous M-grouped MoE
GEMM and the masked M-grouped MoE GEMM.  A step of a workload is one pass of
the GEMM over every case of that workload, with all inputs resident in HBM and
the step captured once in a CUDA graph; each workload's K steps are timed with
CUDA events on the launching stream.

The line's headline (`value`, `unit`, `roofline`, `cpu_baseline`, `e2e`) is the
largest of the workloads, the contiguous MoE GEMM (4 experts, about 32768
rows), in TFLOP/s; `per_config` holds the same record for every workload:
GB/s and TFLOP/s, the fraction of the roofline of each case's binding roof
(the ideal time of a case is the larger of bytes / HBM peak and FLOPs / FP8
peak), the same against the nominal 8 TB/s and 4.5 PFLOP/s, the CPU oracle on
a bounded sample and the end-to-end figure through the C ABI with the inputs
copied from pinned host memory and the outputs copied back inside every step.

`--impl reference` times the CPU oracle (the plain C reference) on this
machine's host cores instead, on a bounded sample of the headline workload.

Under torchrun (N > 1) every rank runs the whole workload on its own GPU
(replicas, no collective on the data path); timing is the max over ranks.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "FP8 block-scaled GEMM TFLOPS & HBM GB/s, % of GB300 FP8/HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0       # GB300 HBM3e, nominal
NOMINAL_FP8_TFLOPS = 4500.0    # GB300 dense FP8 tensor rate, nominal
L2_BYTES = 129 * 1024 * 1024
#: the workloads of the default run, in the order they are timed
ALL_WORKLOADS = ("dense_tiny", "dense_decode", "dense_prefill", "grouped_contiguous",
                 "grouped_masked")
#: the headline: the largest single-GPU workload
HEADLINE = "grouped_contiguous"


# ------------------------------------------------------------- workloads ---
class Case:
    """One GEMM call of a workload: its host inputs and algorithmic counts."""

    def __init__(self, kind, prob, label):
        self.kind = kind
        self.p = prob
        self.label = label
        K = prob["K"]
        if kind == "quantize":
            # bf16 read, e4m3 written, one fp32 scale per 128 elements
            M = prob["M"]
            self.m_valid = M
            self.flops = 0.0
            self.bytes = 2 * M * K + M * K + 4 * M * (K // 128)
            return
        kb = K // 128
        N = prob["N"]
        nb = (N + 127) // 128
        if kind == "k_grouped":
            # K = all groups' K rows; every group writes a full [M, N] output
            M, G = prob["M"], prob["G"]
            self.m_valid = M
            self.flops = 2.0 * M * N * K
            self.bytes = K * M + K * N + 4 * M * kb + 4 * nb * kb + 2 * G * M * N
            return
        if kind == "dense":
            mv, gu = prob["M"], 1
        elif kind == "contiguous":
            mv, gu = int((prob["m_indices"] >= 0).sum()), prob["G"]
        else:
            mv, gu = int(prob["masked_m"].sum()), int((prob["masked_m"] > 0).sum())
        self.m_valid = mv
        # algorithmic work counts valid rows only (padding and masked rows excluded)
        self.flops = 2.0 * mv * N * K
        self.bytes = mv * K + gu * N * K + 4 * mv * kb + 4 * gu * nb * kb + 2 * mv * N


def make_cases(name, only=None, add_c=False, layout="nt", ue8m0=False):
    cfg = W.CONFIGS[name]
    out = []
    if layout != "nt":
        assert cfg["kind"] == "dense", "--layout is for the dense workloads"
    if cfg["kind"] == "quantize":
        for (M, K) in cfg["cases"]:
            out.append(("quantize", lambda M=M, K=K: W.activation_problem(M, K, seed=cfg["seed"]),
                        f"{M}x{K}"))
    elif cfg["kind"] == "dense":
        for (M, N, K) in cfg["cases"]:
            out.append(("dense", lambda M=M, N=N, K=K: W.dense_problem(M, N, K, seed=cfg["seed"]),
                        f"{M}x{N}x{K}"))
    elif cfg["kind"] == "k_grouped":
        for i, (M, N) in enumerate(cfg["mn"]):
            ks = W.random_ks(cfg["groups"], *cfg["k_range"], seed=cfg["seed"] + i)
            out.append(("k_grouped", lambda ks=ks, M=M, N=N: W.k_grouped_problem(
                ks, M, N, seed=cfg["seed"]), f"G{cfg['groups']}x{M}x{N}xK{int(ks.sum())}"))
    elif cfg["kind"] == "contiguous":
        for (N, K) in cfg["nk"]:
            out.append(("contiguous", lambda N=N, K=K: W.contiguous_problem(
                cfg["groups"], N, K, *cfg["m_range"], seed=cfg["seed"]),
                f"G{cfg['groups']}x{N}x{K}"))
    else:
        for G in cfg["groups"]:
            for (N, K) in cfg["nk"]:
                out.append(("masked", lambda G=G, N=N, K=K: W.masked_problem(
                    G, cfg["max_m"], N, K, cfg["expected_m"], seed=cfg["seed"] + G),
                    f"G{G}x{cfg['max_m']}x{N}x{K}"))
    if only is not None:
        out = [out[only]]
    cases = [Case(kind, make(), label) for kind, make, label in out]
    if add_c:
        assert cfg["kind"] in ("dense", "k_grouped"), "--add-c is for the dense and K-grouped workloads"
        for c in cases:
            M, N = c.p["M"], c.p["N"]
            shape = (c.p["G"], M, N) if c.kind == "k_grouped" else (M, N)
            g = np.random.default_rng(c.p["K"] + M + N)
            c.p["C"] = (g.standard_normal(shape).astype(np.float32).view(np.uint32) >>
                        16).astype(np.uint16)   # bf16 bits (truncated N(0,1))
            c.bytes += 2 * int(np.prod(shape))
            c.label += "+C"
    for c in cases:
        c.layout = layout
        if layout != "nt":
            c.label += "+" + layout
    if ue8m0:
        assert cfg["kind"] in ("dense", "contiguous", "masked") and layout == "nt" and not add_c, \
            "--ue8m0 is for the nt dense / contiguous / masked workloads"
        for c in cases:
            # packed UE8M0 scales; the oracle sample reads their fp32 values
            c.p["sfa"], c.p["sfb"], c.p["sa"], c.p["sb"] = W.ue8m0_packed_scales(c.p["sa"], c.p["sb"])
            kb, nb = c.p["K"] // 128, (c.p["N"] + 127) // 128
            gu = (1 if c.kind == "dense" else c.p["G"] if c.kind == "contiguous"
                  else int((c.p["masked_m"] > 0).sum()))
            c.bytes -= 3 * (c.m_valid * kb + gu * nb * kb)   # 1 byte per scale, not 4
            c.label += "+ue8m0"
    return cases


def describe(name):
    cfg = W.CONFIGS[name]
    if name == "dense_decode":
        return ("dense decode sweep: M in {64,128} x (N,K) in "
                + ",".join(f"({n},{k})" for n, k in W.DENSE_NK))
    if name == "dense_prefill":
        return "dense prefill sweep: M=4096 x (N,K) in " + ",".join(
            f"({n},{k})" for n, k in W.DENSE_NK)
    if name == "quantize_act":
        return ("per-token 1x128 FP8 quantisation of bf16 activations [M,K]: M in {64,128,4096} "
                "x K in {512,1536,2048,7168,16384}")
    if name == "dense_tiny":
        return "dense M=128, N=256, K=512"
    if name == "grouped_contiguous":
        return (f"contiguous M-grouped MoE GEMM: {cfg['groups']} experts, m_e~U[{cfg['m_range'][0]},"
                f"{cfg['m_range'][1]}] padded to 128, (N,K) in {cfg['nk']}")
    if name == "k_grouped_wgrad":
        return (f"K-grouped tn (MoE weight gradient): {cfg['groups']} experts, tokens per expert "
                f"K_g~U[{cfg['k_range'][0]},{cfg['k_range'][1]}] rounded down to 128, "
                f"(M,N) in {cfg['mn']}, A [K,M] and B [K,N] stored MN-major")
    return (f"masked M-grouped MoE GEMM: G in {cfg['groups']}, max_m={cfg['max_m']}, "
            f"masked_m~U[1,{2 * cfg['expected_m']}], (N,K) in {cfg['nk']}")


def data_desc(name):
    if name == "quantize_act":
        return "synthetic (seeded N(0,1) bf16 activations)"
    return "synthetic (seeded N(0,1), 1x128 / 128x128 fp32-scaled e4m3)"


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class Peaks:
    """Roofline denominators: the measured HBM copy bandwidth and the dense FP8
    tensor rate taken as 2x the measured bf16 cuBLAS burst (the nominal
    fp8 / bf16 ratio, 4.5 / 2.25 PFLOP/s)."""

    def __init__(self):
        self.hbm, bf16, _, self.src = measured_peaks()
        self.fp8 = 2.0 * bf16

    def ideal_s(self, c, hbm=None, fp8=None):
        """Seconds of case c at its binding roof."""
        return max(c.bytes / ((hbm or self.hbm) * 1e9), c.flops / ((fp8 or self.fp8) * 1e12))

    def bound(self, cases):
        """The roof that binds a whole step: the one its cases spend more
        ideal time against."""
        t_mem = sum(c.bytes for c in cases) / (self.hbm * 1e9)
        t_cmp = sum(c.flops for c in cases) / (self.fp8 * 1e12)
        return "hbm" if t_mem >= t_cmp else "tensor"


def _code_only(text):
    """C++ source without its comments and blank space (the sources hold no
    string literal with a comment marker), so that editing a comment does not
    count as a change of the kernels."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(workload):
    """Hash of the code a workload's kernels and launch choices come from:
    the quantiser's own files for quantize_act, every other file for the
    GEMM workloads (the host code, which plans and launches both, in each);
    comments and blank space do not count."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_grouped_gemm_bf16_gb300", "csrc")
    quant = workload == "quantize_act"
    for f in sorted(os.listdir(csrc)):
        if f != "dg_host.cu" and f.startswith("dg_quant") != quant:
            continue
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/<workload>_traffic.txt), if it was taken on the current kernel
    sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{workload}_traffic.txt")
    try:
        kv = {}
        with open(path) as fh:
            for line in fh:
                if line.startswith("#") or ":" not in line:
                    continue
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_hash") == kernel_source_hash(workload):
            return float(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def roofline(name, cases, seconds, peaks, launches):
    """The roofline record of one workload's step: achieved rate against the
    binding roof of the step, the fraction of each case's own binding roof
    (sum of the cases' ideal times over the measured time) and the same
    against the nominal peaks."""
    bound = peaks.bound(cases)
    B = sum(c.bytes for c in cases)
    F = sum(c.flops for c in cases)
    ideal = sum(peaks.ideal_s(c) for c in cases)
    ideal_nom = sum(peaks.ideal_s(c, NOMINAL_HBM_GBS, NOMINAL_FP8_TFLOPS) for c in cases)
    per_launch_s = seconds / max(1, launches)
    if bound == "hbm":
        achieved = B / launches / per_launch_s / 1e9
        peak, unit, nominal = peaks.hbm, "GB/s", NOMINAL_HBM_GBS
        src = ("measured HBM copy, MEASURED_PEAKS.json hbm_gbs" if peaks.src == "measured"
               else "fallback 6.8 TB/s")
    else:
        achieved = F / launches / per_launch_s / 1e12
        peak, unit, nominal = peaks.fp8, "TFLOP/s", NOMINAL_FP8_TFLOPS
        src = f"{peaks.src} bf16 cuBLAS burst x 2 (fp8/bf16 nominal ratio)"
    n_hbm = sum(1 for c in cases if c.bytes / peaks.hbm / 1e9 >= c.flops / peaks.fp8 / 1e12)
    return {"bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4),
            "frac_binding": round(ideal / seconds, 4),
            "frac_nominal": round(achieved / nominal, 4),
            "frac_binding_nominal": round(ideal_nom / seconds, 4),
            "cases_hbm_bound": n_hbm, "cases_tensor_bound": len(cases) - n_hbm,
            "traffic": recorded_traffic(name), "peak_source": src}


def value_of(cases, seconds, unit):
    if unit == "GB/s":
        return sum(c.bytes for c in cases) / seconds / 1e9
    return sum(c.flops for c in cases) / seconds / 1e12


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region.
    Each sample carries nvidia-smi's own timestamp, so the samples of a region
    are found by time even when the tool's output arrives late (buffered)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=3.0):
        """Block until the first sample has arrived (or `timeout` seconds)."""
        t = time.time()
        while self.proc is not None and not self.lines and time.time() - t < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.lines

    @staticmethod
    def summarize(lines, t0=None, t1=None):
        """Median SM clock, max clock and the throttle reasons seen in the
        samples taken in [t0, t1] (wall-clock seconds; all samples when not
        given)."""
        if not lines:
            return None
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, power, reasons = [], [], [], set()
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if ts is not None and ((t0 is not None and ts < t0) or (t1 is not None and ts > t1)):
                continue
            parts = parts[1:]
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


class NvmlSampler:
    """Reads of SM clock, clock-event reasons and power through NVML (the
    driver's libnvidia-ml, called with ctypes; reads only) every ~1 ms on a
    thread, so that a timed region of a few tens of milliseconds still gets
    tens of samples.  Same record as ClockSampler.summarize; None when NVML
    cannot be loaded."""

    # clock-event reason bits (nvml.h): SW power cap, HW slowdown, SW thermal, HW thermal
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index, period_s=0.001):
        self.gpu = gpu_index
        self.period = period_s
        self.samples = []          # (time, sm_mhz, reasons, power_mw)
        self.run = False
        self.thread = None
        self.lib = None
        self.dev = None
        self.max_mhz = None

    def start(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            dev = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(dev)) != 0:
                return False
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(dev, ctypes.c_int(1), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except Exception:
            return False
        self.lib, self.dev, self.ct = lib, dev, ctypes
        self.run = True
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()
        return True

    def _loop(self):
        ct, lib, dev = self.ct, self.lib, self.dev
        mhz, rs, mw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        while self.run:
            ok = lib.nvmlDeviceGetClockInfo(dev, ct.c_int(1), ct.byref(mhz)) == 0  # NVML_CLOCK_SM
            r = rs.value if self.reasons_fn(dev, ct.byref(rs)) == 0 else 0
            p = mw.value if lib.nvmlDeviceGetPowerUsage(dev, ct.byref(mw)) == 0 else None
            if ok:
                self.samples.append((time.time(), float(mhz.value), r, p))
            time.sleep(self.period)

    def stop(self):
        self.run = False
        if self.thread:
            self.thread.join(timeout=2)
        return self.samples

    def summarize(self, t0=None, t1=None):
        sel = [s for s in self.samples
               if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        if not sel:
            return None
        reasons = sorted({nm for s in sel for nm, b in self.BITS.items() if s[2] & b})
        pw = [s[3] / 1000.0 for s in sel if s[3] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in sel),
                "sm_max_mhz": self.max_mhz or max(s[1] for s in sel),
                "reasons": reasons, "samples": len(sel),
                "power_w_max": round(max(pw), 1) if pw else None,
                "source": f"NVML every {self.period * 1e3:.0f} ms"}


# --------------------------------------------------------------- GPU arm ---
class DeviceCase:
    """A case's tensors resident on the GPU and the library call on them."""

    def __init__(self, c, torch, dg):
        self.c = c
        self.dg = dg
        p = c.p
        dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
        if c.kind == "quantize":
            self.X = dev(p["X"].view(np.int16))
            self.D = torch.empty((p["M"], p["K"]), dtype=torch.uint8, device="cuda")   # codes
            self.sa = torch.zeros((p["K"] // 128, p["ld_sa"]), dtype=torch.float32,
                                  device="cuda")
            self.idx = None
            self.inputs = [self.X]
            return
        A, B = p["A"], p["B"]
        if getattr(c, "layout", "nt")[0] == "t":   # the stored forms of the other layouts
            A = np.ascontiguousarray(A.T)
        if getattr(c, "layout", "nt")[1] == "n":
            B = np.ascontiguousarray(B.T)
        self.ue8m0 = "sfa" in p
        self.A, self.B = dev(A), dev(B)
        self.sa = dev(p["sfa"]) if self.ue8m0 else dev(p["sa"])
        self.sb = dev(p["sfb"]) if self.ue8m0 else dev(p["sb"])
        self.idx = None
        self.C = dev(p["C"].view(np.int16)) if "C" in p else None
        if c.kind == "k_grouped":
            self.idx = dev(p["ks"])
            self.D = torch.zeros((p["G"], p["M"], p["N"]), dtype=torch.bfloat16, device="cuda")
        elif c.kind == "dense":
            self.D = torch.zeros((p["M"], p["N"]), dtype=torch.bfloat16, device="cuda")
        elif c.kind == "contiguous":
            self.idx = dev(p["m_indices"])
            self.D = torch.zeros((p["M"], p["N"]), dtype=torch.bfloat16, device="cuda")
        else:
            self.idx = dev(p["masked_m"])
            self.D = torch.zeros((p["G"], p["max_m"], p["N"]), dtype=torch.bfloat16,
                                 device="cuda")
        self.inputs = [self.A, self.sa, self.B, self.sb] + (
            [self.idx] if self.idx is not None else []) + ([self.C] if self.C is not None else [])

    def footprint(self):
        return sum(t.numel() * t.element_size() for t in self.inputs) + \
            self.D.numel() * self.D.element_size()

    def call(self, stream):
        p, dg = self.c.p, self.dg
        if self.c.kind == "quantize":
            dg.quantize_fp8_1x128(self.X, self.D, self.sa, 1, p["M"], p["K"], p["ld_sa"], stream)
        elif self.c.kind == "k_grouped":
            dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(
                self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D, self.idx, p["G"],
                p["M"], p["N"], p["K"], C=self.C, stream=stream)
        elif self.c.kind == "dense" and self.c.layout != "nt":
            getattr(dg, "gemm_fp8_fp8_bf16_" + self.c.layout)(
                self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D, p["M"], p["N"],
                p["K"], C=self.C, stream=stream)
        elif self.ue8m0 and self.c.kind == "dense":
            dg.gemm_fp8_fp8_bf16_nt_ue8m0(self.A, self.sa, self.sa.shape[-1], self.B, self.sb,
                                          self.D, p["M"], p["N"], p["K"], stream)
        elif self.ue8m0 and self.c.kind == "contiguous":
            dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(
                self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D, self.idx, p["M"],
                p["N"], p["K"], p["G"], stream)
        elif self.ue8m0:
            em = W.CONFIGS["grouped_masked"]["expected_m"]
            dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(
                self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D, self.idx, p["G"],
                p["max_m"], p["N"], p["K"], em, stream)
        elif self.c.kind == "dense" and self.C is not None:
            dg.gemm_fp8_fp8_bf16_nt_add_c(self.A, self.sa, self.sa.shape[-1], self.B, self.sb,
                                          self.C, self.D, p["M"], p["N"], p["K"], stream)
        elif self.c.kind == "dense":
            dg.gemm_fp8_fp8_bf16_nt(self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D,
                                    p["M"], p["N"], p["K"], stream)
        elif self.c.kind == "contiguous":
            dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous(
                self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D, self.idx, p["M"],
                p["N"], p["K"], p["G"], stream)
        else:
            em = W.CONFIGS["grouped_masked"]["expected_m"]
            dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked(
                self.A, self.sa, self.sa.shape[-1], self.B, self.sb, self.D, self.idx, p["G"],
                p["max_m"], p["N"], p["K"], em, stream)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, x):
    if pg is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


class Workload:
    """One workload on the device: its cases, their resident tensors and the
    CUDA graph of one step (every case once)."""

    def __init__(self, name, args, torch, dg, stream):
        self.name = name
        self.cases = make_cases(name, args.case, add_c=args.add_c, layout=args.layout,
                                ue8m0=args.ue8m0)
        self.dcs = [DeviceCase(c, torch, dg) for c in self.cases]
        self.footprint = sum(d.footprint() for d in self.dcs)
        with torch.cuda.stream(stream):
            # eager warm-up (device set-up, occupancy queries), then graph capture
            for _ in range(2):
                for d in self.dcs:
                    d.call(stream.cuda_stream)
            stream.synchronize()
            if dg.get_device_status(stream.cuda_stream) != 0:
                raise RuntimeError(f"{name}: device status set during warm-up")
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                for d in self.dcs:
                    d.call(stream.cuda_stream)
        self.launches = len(self.dcs)
        self.ms = None

    def describe(self, args):
        desc = describe(self.name)
        if args.add_c:
            desc += "; D = C + A B with a bf16 addend C read per call"
        if args.layout != "nt":
            desc += f"; operands stored as the {args.layout} layout"
        if args.ue8m0:
            desc += "; packed UE8M0 scales (the fp32 scales rounded up to powers of two)"
        if args.case is not None:
            desc += f" (case {args.case} only: {self.cases[0].label})"
        return desc

    def l2_note(self):
        if self.footprint > 2 * L2_BYTES:
            return (f"inputs larger than L2: step footprint {self.footprint / 1e6:.0f} MB vs "
                    f"129 MB L2; each case's buffers are evicted by the other cases before it "
                    f"runs again")
        return (f"step footprint {self.footprint / 1e6:.0f} MB: NOT larger than L2, repeats may "
                f"hit L2")


def time_steps(w, torch, stream, steps, pg):
    """K graph replays of a workload between CUDA events on the launching
    stream, with a barrier and a device synchronisation on both sides; the
    max over ranks of the elapsed milliseconds."""
    barrier(pg)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(steps):
            w.graph.replay()
        t1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(pg)
    return max_over_ranks(pg, t0.elapsed_time(t1))


def run_ours(args):
    import torch

    import moe_grouped_gemm_bf16_gb300 as dg
    from moe_grouped_gemm_bf16_gb300 import _build

    world, rank, local, pg = dist_setup()
    torch.cuda.set_device(local)
    _build.build()
    dg.lib()
    names = ALL_WORKLOADS if args.workload == "all" else (args.workload,)
    head = HEADLINE if args.workload == "all" else args.workload
    peaks = Peaks()
    stream = torch.cuda.Stream()
    log = (lambda *a: print(*a, file=sys.stderr, flush=True)) if rank == 0 else (lambda *a: None)

    t_gen = time.perf_counter()
    wls = []
    for nm in names:
        wls.append(Workload(nm, args, torch, dg, stream))
        log(f"[bench] {nm}: {len(wls[-1].cases)} cases ready "
            f"({time.perf_counter() - t_gen:.1f} s)")

    steps = args.steps
    if steps is None:
        # default: about two seconds of the slowest workload's steps
        per = max(time_steps(w, torch, stream, 3, None) / 3.0 for w in wls)
        steps = int(max(20, min(20000, 2000.0 / max(per, 1e-3))))
        steps = int(max_over_ranks(pg, steps))

    # warm-up, then the timed regions back to back (clocks sampled throughout)
    with torch.cuda.stream(stream):
        for w in wls:
            for _ in range(args.warmup):
                w.graph.replay()
    stream.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        sampler.wait_first()
    nvml = NvmlSampler(local) if rank == 0 else None
    if nvml and not nvml.start():
        nvml = None
    spans, exact = {}, {}
    for w in wls:
        a = time.time()
        w.ms = time_steps(w, torch, stream, steps, pg)
        b = time.time()
        exact[w.name] = (a, b)
        # (a region shorter than nvidia-smi's interval still gets its nearest samples)
        spans[w.name] = (a - 0.06, b + 0.06)
    if sampler:
        time.sleep(0.15)
    samples = sampler.stop() if sampler else None
    if nvml:
        nvml.stop()

    def clocks_of(t0, t1, s0, s1):
        """The clock record of a region: NVML's 1 ms reads inside it when
        there are any, with nvidia-smi's samples around it beside them."""
        smi = ClockSampler.summarize(samples, s0, s1) if samples else None
        rec = nvml.summarize(t0, t1) if nvml else None
        if rec is None:
            return smi
        rec["nvidia_smi"] = smi
        return rec
    status = dg.get_device_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed regions")

    detail = {}
    for w in wls:
        rec = {"steps": steps, "ms_per_step": round(w.ms / steps, 5), "cases": len(w.cases),
               "gpu_launches": steps * w.launches}
        secs = w.ms / 1e3 / steps
        roof = roofline(w.name, w.cases, secs, peaks, w.launches)
        rec["unit"] = roof["unit"]
        rec["value"] = round(value_of(w.cases, secs, roof["unit"]), 1)
        rec["gbs"] = round(value_of(w.cases, secs, "GB/s"), 1)
        rec["tflops"] = round(value_of(w.cases, secs, "TFLOP/s"), 1)
        rec["roofline"] = roof
        rec["workload"] = w.describe(args)
        rec["l2"] = w.l2_note()
        if samples:
            rec["clocks"] = clocks_of(*exact[w.name], *spans[w.name])
        detail[w.name] = rec
    for w in wls:
        if rank == 0 and not args.quick:
            detail[w.name]["per_case"] = per_case_cold(w.dcs, torch, stream, peaks)
        detail[w.name]["e2e"] = run_e2e(w.dcs, w.cases, torch, stream,
                                        min(steps, args.e2e_steps), pg, world,
                                        detail[w.name]["unit"])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        orc = oracle.Oracle()
        for w in wls:
            detail[w.name]["cpu_baseline"] = cpu_baseline(
                orc, w.cases, detail[w.name]["unit"],
                args.cpu_budget if w.name == head else args.cpu_budget / 2)
    if rank != 0:
        return None

    h = detail[head]
    hw = next(w for w in wls if w.name == head)
    value = world * h["value"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": h["unit"], "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": h["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if head == "quantize_act" else "e4m3",
        "data": data_desc(head),
        "config": {"workload": h["workload"], "cases": h["cases"],
                   "launch": "one CUDA graph per step (all cases of the workload), inputs "
                             "resident in HBM",
                   "l2": h["l2"], "parallelism": f"replicas x{world}",
                   "other_workloads": [n for n in names if n != head]},
        "tflops": round(world * h["tflops"], 1), "gbs": round(world * h["gbs"], 1),
        "roofline": h["roofline"],
        "cpu_baseline": h.get("cpu_baseline"),
        "e2e": h["e2e"],
        "gpu_launches": h["gpu_launches"],
        "gpu_launches_all_workloads": sum(detail[n]["gpu_launches"] for n in names),
        "clocks": clocks_of(exact[names[0]][0], exact[names[-1]][1], spans[names[0]][0],
                            spans[names[-1]][1]),
        "cases": h.get("per_case"),
    }
    if len(names) > 1:
        line["per_config"] = detail
    if hw.footprint <= 2 * L2_BYTES:
        line["config"]["note"] = "footprint not larger than L2"
    return line


def per_case_cold(dcs, torch, stream, peaks, reps=10):
    """Per-case kernel time with a cold L2, free of host launch overhead: a
    graph [write a 256 MB buffer, GEMM] and a graph [write the buffer] are each
    replayed `reps` times between CUDA events, and the difference is the
    GEMM's time.  Runs after the timed regions; reported as detail, each case
    with the fraction of its own binding roof."""
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    out = []

    def timed(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    with torch.cuda.stream(stream):
        g0 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g0, stream=stream):
            flush.zero_()
        t_flush = min(timed(g0) for _ in range(3))
        for d in dcs:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=stream):
                flush.zero_()
                d.call(stream.cuda_stream)
            us = max(1e-3, min(timed(g1) for _ in range(3)) - t_flush)
            c = d.c
            out.append({"case": c.label, "us": round(us, 2),
                        "gbs": round(c.bytes / (us * 1e-6) / 1e9, 1),
                        "tflops": round(c.flops / (us * 1e-6) / 1e12, 1),
                        "bound": ("hbm" if c.bytes / peaks.hbm / 1e9 >= c.flops / peaks.fp8 / 1e12
                                  else "tensor"),
                        "frac_binding": round(peaks.ideal_s(c) / (us * 1e-6), 4)})
            del g1
    del flush
    return out


def run_e2e(dcs, cases, torch, stream, steps, pg, world, unit="GB/s"):
    """The same metric through the C ABI, with every step's inputs copied from
    pinned host memory and every output read back to the host."""
    steps = max(3, int(steps))
    host_in = [[t.cpu().pin_memory() for t in d.inputs] for d in dcs]
    host_out = [torch.empty(d.D.shape, dtype=d.D.dtype).pin_memory() for d in dcs]
    h2d = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    # Three streams, chained by events and never synchronised inside the timed
    # region: inputs host -> device on s_in, the GEMMs on `stream`, results
    # device -> host on s_out.  So the inputs of the next case (and of the next
    # step) travel while a case computes and an earlier result travels back:
    # the two directions of the link run at once.  A case's input buffers are
    # refilled only after its previous kernel ended, and its output buffer is
    # rewritten only after the previous read-back of it ended.
    s_in = torch.cuda.Stream()
    s_out = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in dcs]
    ev_done = [torch.cuda.Event() for _ in dcs]
    ev_out = [torch.cuda.Event() for _ in dcs]
    started = [False]

    def one_step():
        for i, (d, hs, ho) in enumerate(zip(dcs, host_in, host_out)):
            with torch.cuda.stream(s_in):
                if started[0]:
                    s_in.wait_event(ev_done[i])
                for dev_t, h in zip(d.inputs, hs):
                    dev_t.copy_(h, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[i])
                if started[0]:
                    stream.wait_event(ev_out[i])
                d.call(stream.cuda_stream)
                ev_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                ho.copy_(d.D, non_blocking=True)
                ev_out[i].record(s_out)
        started[0] = True

    def sync_all():
        for st in (s_in, stream, s_out):
            st.synchronize()

    one_step()
    sync_all()
    barrier(pg)
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    sync_all()
    dt = max_over_ranks(pg, time.perf_counter() - t0)
    per = dt / steps
    return {"value": round(world * value_of(cases, per, unit), 2), "unit": unit,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": round(per * 1e3, 4),
            "copies": "pinned host buffers; inputs, kernels and read-backs on three streams "
                      "chained by events (every step copies all its inputs in and all its "
                      "outputs out; the next inputs travel while earlier results return), one "
                      "synchronisation at the end of the timed steps"}


# -------------------------------------------------------- CPU oracle arm ---
def _oracle_sample(orc, c, rows, ncols, threads):
    """Time the oracle on `rows` output rows x the first `ncols` output columns
    of case c.  Returns (seconds, sampled output elements, output elements of
    the whole case)."""
    p = c.p
    if c.kind == "quantize":
        # `rows` whole rows (the quantiser has no output columns to sample)
        r = np.linspace(0, p["M"] - 1, num=min(rows, p["M"])).astype(np.int64)
        t = time.perf_counter()
        orc.quantize_1x128(p["X"][r], nthreads=threads)
        return time.perf_counter() - t, r.size * p["K"], p["M"] * p["K"]
    ncols = min(ncols, p["N"])
    nbs = (ncols + 127) // 128
    if c.kind == "k_grouped":
        # the same sampled rows of every group's output, through the K-grouped oracle
        r = np.linspace(0, p["M"] - 1, num=min(rows, p["M"])).astype(np.int64)
        A, sa = np.ascontiguousarray(p["A"][:, r]), np.ascontiguousarray(p["sa"][:, r])
        B, sb = np.ascontiguousarray(p["B"][:, :ncols]), np.ascontiguousarray(p["sb"][:nbs])
        t = time.perf_counter()
        orc.k_grouped_tn(A, sa, B, sb, p["ks"], nthreads=threads)
        return time.perf_counter() - t, p["G"] * r.size * ncols, p["G"] * p["M"] * p["N"]
    if c.kind == "dense":
        r = np.linspace(0, p["M"] - 1, num=min(rows, p["M"])).astype(np.int64)
        t = time.perf_counter()
        orc.gemm_nt_rows(p["A"], p["sa"], p["B"][:ncols], p["sb"][:nbs], r, nthreads=threads)
        return time.perf_counter() - t, r.size * ncols, c.m_valid * p["N"]
    if c.kind == "contiguous":
        valid = np.nonzero(p["m_indices"] >= 0)[0]
        r = valid[np.linspace(0, valid.size - 1, num=min(rows, valid.size)).astype(np.int64)]
        t = time.perf_counter()
        orc.grouped_contiguous(p["A"], p["sa"], p["B"][:, :ncols], p["sb"][:, :nbs],
                               p["m_indices"], rows=r, nthreads=threads)
        return time.perf_counter() - t, r.size * ncols, c.m_valid * p["N"]
    G = p["G"]
    per = max(1, rows // G)
    secs, done = 0.0, 0
    for g in range(G):
        v = int(p["masked_m"][g])
        if v == 0:
            continue
        r = np.linspace(0, v - 1, num=min(per, v)).astype(np.int64)
        t = time.perf_counter()
        orc.gemm_nt_rows(p["A"][g], p["sa"][g], p["B"][g][:ncols], p["sb"][g][:nbs], r,
                         nthreads=threads)
        secs += time.perf_counter() - t
        done += r.size * ncols
    return secs, done, c.m_valid * p["N"]


def macs_per_output(c):
    """Multiply-adds per output element (K-grouped: the average group's K)."""
    return c.p["K"] / c.p["G"] if c.kind == "k_grouped" else c.p["K"]


def _sample_shape(c, budget_s, rate, cores):
    """Rows and columns of a case's oracle sample sized to take about
    `budget_s` seconds at `rate` output-element MACs per second."""
    if c.kind == "quantize":
        return max(1, min(c.m_valid, int(budget_s * rate / c.p["K"]))), 0
    per_out = macs_per_output(c) * (c.p["G"] if c.kind == "k_grouped" else 1)
    rows = min(max(cores, c.p["G"]) if c.kind == "masked" else cores, c.m_valid)
    cols = int(budget_s * rate / (rows * per_out))
    if cols >= c.p["N"]:
        # whole rows: as many (a multiple of the core count) as the budget allows
        rows = int(budget_s * rate / (c.p["N"] * per_out)) // cores * cores
        rows = max(1, min(c.m_valid, max(rows, cores)))
    return rows, max(16, min(c.p["N"], cols // 16 * 16))


def _calibrate(orc, c, cores):
    """Output-element MACs (quantiser: elements) per second of the oracle on
    this host, from a small sample of case c."""
    s, done, _ = _oracle_sample(orc, c, cores, 128, cores)
    return done * (1 if c.kind == "quantize" else macs_per_output(c)) / max(s, 1e-6)


def cpu_baseline(orc, cases, unit, budget_s):
    """The oracle as it stands, on this host's cores, on a bounded sample of
    every case of a workload (about `budget_s` seconds in all): each case's
    sample is sized from a calibration run, and its time scaled to the whole
    case by the ratio of output elements."""
    cores = len(os.sched_getaffinity(0))
    rate = _calibrate(orc, cases[0], cores)
    t_full, wall, shapes = 0.0, 0.0, []
    for c in cases:
        rows, cols = _sample_shape(c, budget_s / len(cases), rate, cores)
        secs, done, full = _oracle_sample(orc, c, rows, cols, cores)
        wall += secs
        t_full += secs * full / done
        shapes.append(f"{rows}x{cols or c.p['K']}")
    return {"value": round(value_of(cases, t_full, unit), 5), "unit": unit, "cores": cores,
            "kind": "oracle",
            "sample": (f"per case a block of output rows x columns sized for ~{budget_s:.0f} s "
                       f"in all ({', '.join(shapes)}); time scaled to the whole case by "
                       f"output elements; {wall:.1f} s wall"),
            "seconds": round(wall, 2)}


def run_reference(args):
    """The CPU oracle timed on this host's cores on the headline workload;
    step i samples case i mod n, each step sized so the whole run takes about
    two minutes."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return None
    import oracle
    orc = oracle.Oracle()
    cores = len(os.sched_getaffinity(0))
    name = HEADLINE if args.workload == "all" else args.workload
    cases = make_cases(name, args.case, add_c=args.add_c, layout=args.layout,
                       ue8m0=args.ue8m0)
    peaks = Peaks()
    unit = "GB/s" if peaks.bound(cases) == "hbm" else "TFLOP/s"
    steps = args.steps if args.steps is not None else 2 * len(cases)
    warm = args.warmup
    budget = 120.0 / max(1, steps + warm)
    rate = _calibrate(orc, cases[0], cores)
    t_full, wall = 0.0, 0.0
    done_cases = []
    for i in range(warm + steps):
        c = cases[i % len(cases)]
        rows, cols = _sample_shape(c, budget, rate, cores)
        secs, done, full = _oracle_sample(orc, c, rows, cols, cores)
        if i >= warm:
            wall += secs
            t_full += secs * full / done
            done_cases.append(c)
    value = value_of(done_cases, t_full, unit)
    sample = (f"per step one case (round robin over {len(cases)}), a block of output rows x "
              f"columns sized for a ~2 minute run; time scaled to the whole case by output "
              f"elements")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
        "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": round(wall / steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if name == "quantize_act" else "f64",
        "data": data_desc(name),
        "config": {"workload": describe(name), "cases": len(cases),
                   "parallelism": "host cores (OpenMP over output rows)"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps per workload (default: about two seconds of steps)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all"] + sorted(W.CONFIGS), default="all")
    ap.add_argument("--case", type=int, default=None,
                    help="run only case I of the workload (profiling one shape)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the headline's CPU baseline (half that for "
                         "each other workload)")
    ap.add_argument("--add-c", action="store_true",
                    help="dense workloads: D = C + A B^T through dg_gemm_fp8_fp8_bf16_nt_add_c "
                         "(a seeded bf16 addend C; its 2*M*N bytes count as read)")
    ap.add_argument("--layout", choices=["nt", "nn", "tn", "tt"], default="nt",
                    help="dense workloads: store A and B as this layout names and call "
                         "dg_gemm_fp8_fp8_bf16_<layout> (the same logical problem)")
    ap.add_argument("--ue8m0", action="store_true",
                    help="nt dense / grouped workloads: packed UE8M0 scales through the _ue8m0 "
                         "entry points (scale bytes counted at 1 byte each)")
    ap.add_argument("--quick", action="store_true",
                    help="skip the per-case cold-L2 detail (profiling runs)")
    args = ap.parse_args(argv)
    if args.impl == "ours" and args.warmup < 3:
        args.warmup = 3
    if args.workload == "all" and (args.add_c or args.layout != "nt" or args.case is not None):
        ap.error("--add-c, --layout and --case need a single --workload")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
