#!/usr/bin/env python
"""Benchmark: CSA + HCA decode queries/s and achieved HBM GB/s at 1M context on one B300.

Workload (default ``decode_1m_b32_csa_hca``): 32 sequences with seeded lengths in
[524288, 1048576]; one decode step = for every sequence, one new token through a CSA layer
(m=4, lightning indexer over FP4 e2m1 keys with UE8M0/32 scales, top-1024, window 128) and an
HCA layer (m=128, dense over every compressed entry plus the window 128); 64 query heads over
one shared KV stream of d=128, bf16.  Inputs are synthetic, seeded; caches are built before the
timed region.  A query = one sequence's one-token decode step through both layers.

Arms:  ``--impl ours`` (default) times the CUDA library; each step is one CUDA graph of the
C-ABI calls with in-graph timing events between them.  ``--impl reference`` times the CPU
oracle on the host cores on a bounded sample of the same workload.

Under torchrun (N > 1) every rank runs an independent replica (the batch is the unit of work,
no collective on the data path); the time is the max over ranks and the value counts every
rank's queries.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "CSA+HCA decode queries/s and achieved HBM GB/s at 1M ctx on 1 B300"
UNIT = "queries/s"
L2_BYTES = 126 * 1000 * 1000      # B300 L2
# layers of a decode step per workload kind
DEFAULT_LAYERS = {"hybrid_decode": "both", "csa_decode": "csa", "hca_decode": "hca"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_1m_b32_csa_hca")
    ap.add_argument("--cpu-seqs", type=int, default=0, help="sequences in the CPU-baseline sample (0 = auto)")
    ap.add_argument("--cpu-rows", type=int, default=64, help="query rows in the prefill CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", default=None, choices=["both", "csa", "hca", "index"],
                    help="restrict the step (profiling): csa / hca layer only, or the CSA indexer + top-k only "
                         "(default: the workload's layers)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- dist utils
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------- clock sampler
class ClockSampler:
    """Samples SM clock, max clock, power and clock-event reasons during the timed region:
    NVML when the Python binding is importable, else ``nvidia-smi -lms`` in a subprocess."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
        "sync_boost": 0x10, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80, "display_clock_setting": 0x100,
    }
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active"]

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples = []
        self.period = period_s
        self.index = index
        self.mode = None
        self.max_mhz = None
        self.err = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err = f"nvml: {e}"
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "smi"

    def _run_nvml(self):
        nv, h = self.nv, self.h
        while not self._stop.is_set():
            try:
                sm = nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM)
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(h)
                pw = nv.nvmlDeviceGetPowerUsage(h) / 1000.0
                self.samples.append((sm, rs, pw))
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.mode == "nvml":
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        elif self.mode == "smi":
            import subprocess
            self._p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.SMI_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            time.sleep(0.3)   # let the first sample land before the timed work starts
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self._t.join()
        elif self.mode == "smi":
            time.sleep(0.05)
            self._p.terminate()
            out, _ = self._p.communicate(timeout=10)
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(f[0]), int(f[3], 16), float(f[2])))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    continue

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "error": self.err or "no samples"}
        sm = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[1]
        reasons = [k for k, v in self.REASONS.items() if bits & v and k != "gpu_idle"]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "power_w_max": round(max(s[2] for s in self.samples), 1), "source": self.mode}


# ---------------------------------------------------------------------------- ours
def algorithmic_bytes(w, lens_csa_nvis, lens_hca_nvis, layers="both"):
    """Minimum bytes one decode step must move (per the method): all visible CSA index keys
    (+ scales), the k selected + W window K/V rows, all visible HCA entries + window, and the
    queries/outputs -- of the layers the step runs.  Returns dict of per-part bytes."""
    d, H, B = w.d, w.H, w.B
    key_row = {"f32": 4 * w.d_I, "bf16": 2 * w.d_I, "e4m3": w.d_I + 4, "e2m1": w.d_I // 2 + w.d_I // 32}[w.key_fmt]
    # one K row + one V row: bf16, or FP8 (K: 64 codes + a scale byte + 64 bf16 RoPE dims; V: 128
    # codes + 2 scale bytes; the rows' zero padding is not counted)
    kv_row = 2 * d * 2 if w.kv_cache == "bf16" else (64 + 1 + 128) + (128 + 2)
    csa = layers in ("both", "csa", "index")
    hca = layers in ("both", "hca")
    parts = {
        "csa_index_keys": int(sum(lens_csa_nvis)) * key_row if csa else 0,
        "csa_gather": B * (w.k + w.W) * kv_row if layers in ("both", "csa") else 0,
        "hca_entries": int(sum(lens_hca_nvis)) * kv_row if hca else 0,
        "hca_window": B * w.W * kv_row if hca else 0,
        "q_o": B * ((4 * H * d * 2 if layers in ("both", "csa") else 0) + (4 * H * d * 2 if hca else 0)
                    + (w.H_I * w.d_I * 2 + w.H_I * 4 if csa else 0)),
    }
    parts["total"] = sum(parts.values())
    return parts


class StepInputs:
    """All inputs of one decode step packed in one contiguous buffer (so that the end-to-end
    run can move them with a single host->device copy)."""

    def __init__(self, w, B, device, pin=False):
        d, H, H_I, d_I = w.d, w.H, w.H_I, w.d_I
        bf = torch.bfloat16
        spec = [("pos", (B,), torch.int64), ("nvis", (B,), torch.int64),
                ("c_k", (B, 1, d), bf), ("c_v", (B, 1, d), bf), ("c_g", (B, 1), torch.float32),
                ("c_kidx", (B, 1, d_I), bf), ("c_q", (B, 1, H, d), bf), ("c_qi", (B, 1, H_I, d_I), bf),
                ("c_w", (B, 1, H_I), torch.float32),
                ("h_k", (B, 1, d), bf), ("h_v", (B, 1, d), bf), ("h_g", (B, 1), torch.float32),
                ("h_q", (B, 1, H, d), bf)]
        offs, off = {}, 0
        for name, shape, dt in spec:
            nb = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
            offs[name] = (off, shape, dt, nb)
            off += (nb + 255) // 256 * 256
        self.nbytes = off
        self.buf = torch.empty(off, dtype=torch.uint8, device=device, pin_memory=pin)
        self.t = {}
        for name, (o, shape, dt, nb) in offs.items():
            self.t[name] = self.buf[o:o + nb].view(dt).view(shape)


def make_step_inputs(w, step: int, lens, device, m_csa):
    """Seeded inputs of decode step `step` (the token at position L_b - 1 + step)."""
    B = w.B
    si = StepInputs(w, B, device)
    t = si.t
    pos = torch.tensor([L - 1 + step for L in lens], dtype=torch.int64)
    t["pos"].copy_(pos)
    t["nvis"].copy_((pos + 1) // m_csa)
    tag = f"step{step}"
    for layer, pre in (("csa", "c_"), ("hca", "h_")):
        k = wl.normal((B, w.d), 1.0, device, w.seed, f"{layer}/{tag}/k", 0)
        v = wl.normal((B, w.d), 1.0, device, w.seed, f"{layer}/{tag}/v", 0)
        if w.outlier_frac > 0:
            rows = wl.outlier_rows(B, w.outlier_frac * 3, device, w.seed, f"{layer}/{tag}/out", 0)
            k[rows] *= w.outlier_mult
            v[rows] *= w.outlier_mult
        t[pre + "k"].copy_(k.to(torch.bfloat16)[:, None])
        t[pre + "v"].copy_(v.to(torch.bfloat16)[:, None])
        t[pre + "g"].copy_(wl.normal((B, 1), 1.0, device, w.seed, f"{layer}/{tag}/g", 0))
        t[pre + "q"].copy_(wl.normal((B, 1, w.H, w.d), 1.0, device, w.seed, f"{layer}/{tag}/q", 0).to(torch.bfloat16))
    t["c_kidx"].copy_(wl.normal((B, 1, w.d_I), 1.0, device, w.seed, f"csa/{tag}/kidx", 0).to(torch.bfloat16))
    t["c_qi"].copy_(wl.normal((B, 1, w.H_I, w.d_I), 1.0, device, w.seed, f"csa/{tag}/qi", 0).to(torch.bfloat16))
    t["c_w"].copy_(wl.uniform((B, 1, w.H_I), device, w.seed, f"csa/{tag}/w", 0))
    return si


class DecodeBench:
    """Caches + per-step calls of the CSA layer then the HCA layer."""

    SUBSTEPS = ["csa_cache_append", "csa_index_topk", "csa_attend", "hca_cache_append", "hca_attend"]

    def __init__(self, w, device, total_steps, layers="both"):
        import types
        import long_context_sparse_28_b300 as L
        from long_context_sparse_28_b300.layers import CSACache, HCACache
        self.L, self.w, self.dev = L, w, device
        self.lens = w.lengths()
        B = w.B
        grow = total_steps + 8
        self.Ncap_c = ((max(self.lens) + grow) // w.m_csa + 1 + 255) // 256 * 256
        self.Ncap_h = (max(self.lens) + grow) // w.m_hca + 1
        fmt = L.KEY_FMT[w.key_fmt]
        self.active = {"both": [0, 1, 2, 3, 4], "csa": [0, 1, 2], "hca": [3, 4], "index": [1]}[layers]
        self.cb = wl.layer_bias(w, "csa", w.m_csa, device)
        self.hb = wl.layer_bias(w, "hca", w.m_hca, device)
        if layers in ("both", "csa"):
            self.csa = CSACache(B, self.Ncap_c, w.d, w.W, w.d_I, fmt, torch.bfloat16, device, m=w.m_csa,
                                kv_fp8=w.kv_cache == "fp8")
        elif layers == "index":            # index keys only (no compressed K/V)
            codes, scale = L.key_storage(B, self.Ncap_c, w.d_I, fmt, device)
            self.csa = types.SimpleNamespace(k_codes=codes.zero_(), k_scale=scale.zero_(), key_fmt=fmt, m=w.m_csa)
        if layers in ("both", "hca"):
            self.hca = HCACache(B, self.Ncap_h, w.d, w.W, torch.bfloat16, device, m=w.m_hca, kv_fp8=w.kv_cache == "fp8")
        for b, Lb in enumerate(self.lens):
            if layers in ("both", "csa"):
                k, v, g = wl.raw_tokens(w, "csa", b, Lb - 1, device)
                kin = wl.index_key_inputs(w, "csa", b, Lb // w.m_csa + 1, device)
                self.csa.build_seq(b, k, v, g, self.cb, kin, Lb - 1)
                del k, v, g, kin
            elif layers == "index":
                n = (Lb - 1) // w.m_csa
                kin = wl.index_key_inputs(w, "csa", b, n, device)
                L.csa_index_key_quantize(kin, fmt, self.csa.k_codes[b, :n], self.csa.k_scale[b, :n])
                del kin
            if layers in ("both", "hca"):
                k, v, g = wl.raw_tokens(w, "hca", b, Lb - 1, device)
                self.hca.build_seq(b, k, v, g, self.hb, Lb - 1)
                del k, v, g
        torch.cuda.synchronize()
        self.scores = torch.empty(B, 1, self.Ncap_c, dtype=torch.float32, device=device)
        self.idx = torch.empty(B, 1, w.k, dtype=torch.int32, device=device)
        self.out_c = torch.empty(B, 1, w.H, w.d, dtype=torch.bfloat16, device=device)
        self.out_h = torch.empty(B, 1, w.H, w.d, dtype=torch.bfloat16, device=device)
        self.lse_c = torch.empty(B, 1, w.H, dtype=torch.float32, device=device)
        self.lse_h = torch.empty(B, 1, w.H, dtype=torch.float32, device=device)
        self.ws_topk = torch.zeros(L.csa_index_topk_workspace(B, 1, self.Ncap_c, w.k), dtype=torch.uint8,
                                   device=device)
        if w.index_q == "e2m1":          # FP4 indexer queries: quantised every step
            self.q4c = torch.empty(B, 1, w.H_I, w.d_I // 2, dtype=torch.uint8, device=device)
            self.q4s = torch.empty(B, 1, w.H_I, w.d_I // 32, dtype=torch.uint8, device=device)
        self.ws_ca = torch.zeros(max(256, L.csa_attend_workspace(B, 1, w.H, w.d, w.k, w.W)), dtype=torch.uint8,
                                 device=device)
        self.ws_ha = torch.zeros(max(256, L.hca_attend_workspace(B, 1, w.H, w.d, self.Ncap_h, w.W, 0)),
                                 dtype=torch.uint8, device=device)
        self.scale = 1.0 / math.sqrt(w.d)

    def substep(self, i, t):
        L, w, c, h = self.L, self.w, getattr(self, "csa", None), getattr(self, "hca", None)
        if i == 0:
            L.csa_cache_append(t["c_k"], t["c_v"], t["c_g"], t["c_kidx"], t["pos"], self.cb, c.m, c.ring_k,
                               c.ring_v, c.ring_gate, c.ck, c.cv, c.k_codes, c.k_scale, c.key_fmt)
        elif i == 1 and w.index_q == "e2m1":
            L.csa_index_key_quantize(t["c_qi"], L.E2M1_UE8M0, self.q4c, self.q4s)
            L.csa_index_topk_fp4(self.q4c, self.q4s, t["c_w"], c.k_codes, c.k_scale, t["pos"], c.m, w.k, self.idx,
                                 workspace=self.ws_topk)
        elif i == 1:
            L.csa_index_topk(t["c_qi"], t["c_w"], c.k_codes, c.k_scale, c.key_fmt, t["pos"], c.m, w.k, self.idx,
                             workspace=self.ws_topk)
        elif i == 2:
            L.csa_attend(t["c_q"], self.scale, c.ck, c.cv, self.idx, c.ring_k, c.ring_v, w.W, t["pos"], self.out_c,
                         self.lse_c, workspace=self.ws_ca)
        elif i == 3:
            L.hca_cache_append(t["h_k"], t["h_v"], t["h_g"], t["pos"], self.hb, h.m, h.ring_k, h.ring_v,
                               h.ring_gate, h.ck, h.cv)
        else:
            L.hca_attend(t["h_q"], self.scale, h.ck, h.cv, h.m, h.ring_k, h.ring_v, w.W, t["pos"], self.out_h,
                         self.lse_h, workspace=self.ws_ha)

    def step(self, t):
        for i in self.active:
            self.substep(i, t)


def _events(n):
    from cuda.bindings import runtime as rt
    evs = []
    for _ in range(n):
        err, ev = rt.cudaEventCreate()
        assert err == rt.cudaError_t.cudaSuccess
        evs.append(ev)
    return evs


def _record_external(ev, stream):
    from cuda.bindings import runtime as rt
    err, = rt.cudaEventRecordWithFlags(ev, stream.cuda_stream, rt.cudaEventRecordExternal)
    assert err == rt.cudaError_t.cudaSuccess, err


def _record(ev, stream):
    from cuda.bindings import runtime as rt
    err, = rt.cudaEventRecord(ev, stream.cuda_stream)
    assert err == rt.cudaError_t.cudaSuccess, err


def _elapsed_ms(a, b):
    from cuda.bindings import runtime as rt
    err, ms = rt.cudaEventElapsedTime(a, b)
    assert err == rt.cudaError_t.cudaSuccess, err
    return ms


# Sources each timed call's kernels are compiled from (its own files plus the shared headers and
# the launch helpers); a DRAM-traffic figure stays valid while these files are unchanged.
_SHARED_SOURCES = ["common.cuh", "tc_ptx.cuh", "tmap.cuh", "tmap.cu", "runtime.cu"]
CALL_SOURCES = {
    "csa_index_topk": ["indexer.cu", "indexer_tc.cu", "topk.cu", "quant.cuh"] + _SHARED_SOURCES,
    "hca_attend": ["attend.cu", "attend_tc.cu", "attend.cuh", "quant.cuh"] + _SHARED_SOURCES,
    "csa_attend": ["attend.cu", "attend_tc.cu", "attend.cuh", "quant.cuh"] + _SHARED_SOURCES,
}


def kernel_source_hash(call: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "long_context_sparse_28_b300", "csrc")
    for f in sorted(CALL_SOURCES[call]):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of a call's kernels from the committed ncu summary, if it was taken
    on this workload and on the call's current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        e = d.get(kernel)
        if (e and kernel in CALL_SOURCES and e.get("workload") == workload and
                e.get("source_hash") == kernel_source_hash(kernel)):
            return e
    except Exception:
        pass
    return None


def _oracle_caches(oracle, K, V, G, bias, m, kv_cache):
    """The oracle's compressed caches: bf16, or FP8 (dequantised, fp64)."""
    if kv_cache == "fp8":
        c = oracle.compress_kv_fp8(K, V, G, bias, m)
        return c["ck"], c["cv"]
    return oracle.compress(K, V, G, bias, m, oracle.BF16)


def cpu_baseline_decode(w, seqs: int, device, layers="both"):
    """The oracle (as it stands) on `seqs` sequences of the workload: one decode query per
    sequence through the step's layers.  Cache construction is setup and not timed."""
    import oracle
    lens = w.lengths()
    order = list(range(w.B))[:seqs]
    fmt = {"f32": oracle.KEY_F32, "bf16": oracle.KEY_BF16, "e4m3": oracle.KEY_E4M3, "e2m1": oracle.KEY_E2M1}[w.key_fmt]
    ctx = []
    for b in order:
        Lb = lens[b]
        K = V = ck = cv = codes = sc = HK = HV = hck = hcv = None
        if layers in ("both", "csa"):
            k, v, g = wl.raw_tokens(w, "csa", b, Lb, device)
            kin = wl.index_key_inputs(w, "csa", b, Lb // w.m_csa + 1, device)
            K, V, G, KIN = (wl.to_numpy(x) for x in (k, v, g, kin))
            cb = wl.to_numpy(wl.layer_bias(w, "csa", w.m_csa, device))
            ck, cv = _oracle_caches(oracle, K, V, G, cb, w.m_csa, w.kv_cache)
            codes, sc = oracle.quantize_keys(KIN[: Lb // w.m_csa], fmt)
            del k, v, g, kin
        if layers in ("both", "hca"):
            hk, hv, hg = wl.raw_tokens(w, "hca", b, Lb, device)
            HK, HV, HG = (wl.to_numpy(x) for x in (hk, hv, hg))
            hb = wl.to_numpy(wl.layer_bias(w, "hca", w.m_hca, device))
            hck, hcv = _oracle_caches(oracle, HK, HV, HG, hb, w.m_hca, w.kv_cache)
            del hk, hv, hg
        q = wl.to_numpy(wl.queries(w, "csa", b, 1, device))
        qh = wl.to_numpy(wl.queries(w, "hca", b, 1, device))
        qi, ww = (wl.to_numpy(x) for x in wl.indexer_queries(w, "csa", b, 1, device))
        ctx.append((Lb, K, V, ck, cv, codes, sc, HK, HV, hck, hcv, q, qh, qi, ww))
    t0 = time.perf_counter()
    for (Lb, K, V, ck, cv, codes, sc, HK, HV, hck, hcv, q, qh, qi, ww) in ctx:
        if layers in ("both", "csa"):
            oracle.csa_queries(q, qi, ww, [Lb - 1], ck, cv, codes, sc, fmt, K, V, 0, w.m_csa, w.k, w.W, w.scale,
                               q_fp4=w.index_q == "e2m1")
        if layers in ("both", "hca"):
            oracle.hca_queries(qh, [Lb - 1], hck, hcv, HK, HV, 0, w.m_hca, w.W, w.scale)
    dt = time.perf_counter() - t0
    names = {"both": "the CSA and HCA layers", "csa": "the CSA layer", "hca": "the HCA layer"}[layers]
    return dict(value=len(ctx) / dt, unit=UNIT, cores=oracle.num_threads(), kind="oracle",
                sample=f"{len(ctx)} of {w.B} sequences, one decode query each through {names} "
                       f"(fp64 C oracle, OpenMP); cache construction untimed; {dt:.2f} s")


def run_ours(args, dist):
    import long_context_sparse_28_b300 as L
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    w = wl.shrink(wl.WORKLOADS[args.workload], seed=dist.rank) if dist.world > 1 else wl.WORKLOADS[args.workload]
    full = DEFAULT_LAYERS[w.kind]
    layers = args.layers or full
    K, Wm = args.steps, args.warmup
    total = K + Wm
    e2e_steps = 0 if args.no_e2e else min(K, 20)
    if layers != full:
        e2e_steps = 0
    bench = DecodeBench(w, dev, total + e2e_steps + 2, layers)
    lens = bench.lens
    stream = torch.cuda.Stream(device=dev)
    inputs = [make_step_inputs(w, s, lens, dev, w.m_csa) for s in range(total)]
    torch.cuda.synchronize()

    # One graph per decode step, as a serving loop replays it: `graphs` holds the library calls
    # only (their kernels chain with programmatic dependent launch across calls); `graphs_ev`
    # the same calls with timing events between them, replayed in a second pass over the same
    # steps for the per-call durations (an event node ends the programmatic overlap at its
    # place, so it stays out of the headline pass).  Launches per step are counted during capture.
    active = bench.active
    nsub = len(active)
    evs = [_events(nsub + 1) for _ in range(total)]
    graphs, graphs_ev = [], []
    launches_per_step = None
    with torch.cuda.stream(stream):
        for s in range(total):
            g = torch.cuda.CUDAGraph()
            c0 = L.launch_count()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(nsub):
                    bench.substep(active[i], inputs[s].t)
            if launches_per_step is None:
                launches_per_step = L.launch_count() - c0
            graphs.append(g)
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream, capture_error_mode="relaxed"):
                for i in range(nsub):
                    _record_external(evs[s][i], stream)
                    bench.substep(active[i], inputs[s].t)
                _record_external(evs[s][nsub], stream)
            graphs_ev.append(ge)
    torch.cuda.synchronize()
    assert L.device_status() == 0

    # algorithmic bytes (average over timed steps)
    nv_c = [[min(bench.Ncap_c, (L0 + s) // w.m_csa) for L0 in lens] for s in range(Wm, total)]
    nv_h = [[min(bench.Ncap_h, (L0 + s) // w.m_hca) for L0 in lens] for s in range(Wm, total)]
    parts_list = [algorithmic_bytes(w, a, b, layers) for a, b in zip(nv_c, nv_h)]
    parts = {k: statistics.mean(p[k] for p in parts_list) for k in parts_list[0]}
    # Steps that read less than twice the L2 (126 MB) would find their caches there on the next
    # step: L2 is flushed (a 256 MB write) before every timed step, and each step is timed alone
    # between CUDA events that exclude the flush.
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if parts["total"] < 2 * L2_BYTES else None

    # warmup
    with torch.cuda.stream(stream):
        for s in range(Wm):
            graphs[s].replay()
    stream.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    with sampler:
        with torch.cuda.stream(stream):
            start.record(stream)
            for s in range(Wm, total):
                if flush_buf is not None:
                    flush_buf.fill_(s & 255)
                    step_ev[s - Wm][0].record(stream)
                graphs[s].replay()
                if flush_buf is not None:
                    step_ev[s - Wm][1].record(stream)
            stop.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    dist.barrier()
    if flush_buf is not None:
        ms_total = sum(a.elapsed_time(b) for a, b in step_ev)
    else:
        ms_total = start.elapsed_time(stop)
    ms_total = dist.max(ms_total)
    ms_per_step = ms_total / K
    st = L.device_status(stream)
    assert st == 0, f"device status {st}"

    # per-call durations: the same K steps again, from the graphs with events
    with torch.cuda.stream(stream):
        for s in range(Wm, total):
            if flush_buf is not None:
                flush_buf.fill_(s & 255)
            graphs_ev[s].replay()
    stream.synchronize()
    ms_per_step_ev = sum(_elapsed_ms(evs[s][0], evs[s][nsub]) for s in range(Wm, total)) / K
    sub_ms = [statistics.mean(_elapsed_ms(evs[s][i], evs[s][i + 1]) for s in range(Wm, total)) for i in range(nsub)]

    queries = w.B * dist.world
    value = queries / (ms_per_step / 1e3)
    step_gbs = parts["total"] / (ms_per_step / 1e3) / 1e9

    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6400.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    # dominant kernel with a defined algorithmic byte count
    kern_bytes = {"csa_index_topk": parts["csa_index_keys"], "hca_attend": parts["hca_entries"] + parts["hca_window"],
                  "csa_attend": parts["csa_gather"]}
    per = {DecodeBench.SUBSTEPS[a]: sub_ms[i] for i, a in enumerate(active)}
    dom = max((n for n in kern_bytes if n in per), key=lambda n: per[n])
    dom_gbs = kern_bytes[dom] / (per[dom] / 1e3) / 1e9
    traffic = load_traffic(dom, w.name)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(dom_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(dom_gbs / hbm_peak, 4), "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                "algorithmic_bytes_per_launch": int(kern_bytes[dom]), "avg_launch_ms": round(per[dom], 5),
                "peak_source": peak_src}

    # end-to-end through the public API with host buffers
    e2e = None
    if e2e_steps:
        # short steps: one graph per step with its copies (host issue would bound them); long
        # steps: the double-buffered stream loop (graph boundaries would cut the launch chain)
        e2e_fn = run_e2e_graphs if ms_per_step < 0.1 else run_e2e
        e2e = (run_e2e_graphs(bench, w, lens, total, e2e_steps, dev, dist, flush_buf) if e2e_fn is run_e2e_graphs
               else run_e2e(bench, w, lens, total, e2e_steps, dev, dist))

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and layers == full:
        cpu = cpu_baseline_decode(w, args.cpu_seqs or min(w.B, 6), dev, layers)

    clocks = sampler.summary()
    key_desc = {"e2m1": "e2m1+ue8m0/32", "e4m3": "e4m3+f32 row scale", "bf16": "bf16", "f32": "f32"}[w.key_fmt]
    cfg = {"workload": w.name, "B": w.B,
           "L": f"U[{w.L_range[0]},{w.L_range[1]}] seeded" if w.L_range else w.L[0] if len(set(w.L)) == 1 else list(w.L),
           "H": w.H, "d": w.d, "layers": layers,
           "kv_cache": "bf16" if w.kv_cache == "bf16" else "e4m3+ue8m0/64, K RoPE dims 64..127 bf16"}
    if layers in ("both", "csa", "index"):
        cfg["csa"] = {"m": w.m_csa, "k": w.k, "W": w.W, "H_I": w.H_I, "d_I": w.d_I, "index_keys": key_desc,
                      "index_queries": "e2m1+ue8m0/32" if w.index_q == "e2m1" else "bf16"}
    if layers in ("both", "hca"):
        cfg["hca"] = {"m": w.m_hca, "W": w.W}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world, "steps": K, "warmup": Wm,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {**cfg, "parallelism": f"replicas x{dist.world}",
                   "l2": ("L2 flushed (256 MB write) before each timed step, steps timed alone: %.0f MB read per "
                          "step" if flush_buf is not None else "inputs larger than L2: %.0f MB read per step")
                         % (parts["total"] / 1e6),
                   "hbm_gbs_step": round(step_gbs, 1), "algorithmic_bytes_per_step": int(parts["total"]),
                   "substep_ms": {n: round(v, 5) for n, v in per.items()},
                   "substep_pass_ms_per_step": round(ms_per_step_ev, 5)},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches_per_step * K),
        "clocks": clocks,
    }
    return line


def run_e2e(bench, w, lens, first_step, n, dev, dist):
    """The public API end to end, as a serving loop would drive it: every step's inputs are
    copied from pinned host memory and both layers' outputs read back into pinned host memory,
    all inside the timed region.  Inputs and outputs are double-buffered: the copy-in of step
    i+1 and the read-back of step i-1 run on their own streams (copy engines) while step i
    computes (the step's C-ABI calls replayed as one CUDA graph per buffer)."""
    L = bench.L
    warm = 3
    steps = [first_step + s for s in range(warm + n)]
    host = []
    for s in steps:
        si = make_step_inputs(w, s, lens, "cpu", w.m_csa)
        pinned = StepInputs(w, w.B, "cpu", pin=True)
        pinned.buf.copy_(si.buf)
        host.append(pinned)
    slabs = [StepInputs(w, w.B, dev) for _ in range(2)]
    outs = [(torch.empty_like(bench.out_c), torch.empty_like(bench.out_h)) for _ in range(2)]
    out_host = [torch.empty(2, w.B, 1, w.H, w.d, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    cs, hs, ds = (torch.cuda.Stream(device=dev) for _ in range(3))
    graphs = []
    saved = (bench.out_c, bench.out_h)
    with torch.cuda.stream(cs):
        for b in range(2):
            bench.out_c, bench.out_h = outs[b]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
                bench.step(slabs[b].t)
            graphs.append(g)
    bench.out_c, bench.out_h = saved
    torch.cuda.synchronize()
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def run(i0, i1, start_ev):
        hs.wait_event(start_ev)
        for i in range(i0, i1):
            b = i & 1
            if i - i0 >= 2:
                hs.wait_event(comp_done[b])            # step i-2 has consumed this input buffer
            with torch.cuda.stream(hs):
                slabs[b].buf.copy_(host[i].buf, non_blocking=True)
                h2d_done[b].record(hs)
            cs.wait_event(h2d_done[b])
            if i - i0 >= 2:
                cs.wait_event(d2h_done[b])             # step i-2's outputs have been read back
            graphs[b].replay()
            comp_done[b].record(cs)
            ds.wait_event(comp_done[b])
            with torch.cuda.stream(ds):
                out_host[b][0].copy_(outs[b][0], non_blocking=True)
                out_host[b][1].copy_(outs[b][1], non_blocking=True)
                d2h_done[b].record(ds)
        cs.wait_event(d2h_done[(i1 - 1) & 1])
        cs.wait_event(d2h_done[(i1 - 2) & 1])

    with torch.cuda.stream(cs):
        ev = torch.cuda.Event()
        ev.record(cs)
        run(0, warm, ev)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        t0.record(cs)
        run(warm, warm + n, t0)
        t1.record(cs)
    torch.cuda.synchronize()
    ms = dist.max(t0.elapsed_time(t1)) / n
    assert L.device_status() == 0
    return {"value": round(w.B * dist.world / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(slabs[0].nbytes), "d2h_bytes_per_step": int(out_host[0].numel() * 2),
            "path": "per step: H2D copy from pinned host memory, the C-ABI calls (one CUDA graph), D2H copy of "
                    "both layers' outputs; inputs and outputs double-buffered on copy streams"}


def run_e2e_graphs(bench, w, lens, first_step, n, dev, dist, flush_buf=None):
    """The same end-to-end steps for short decode steps, where issuing a dozen stream operations
    per step from Python would set the pace: each step is ONE CUDA graph with three independent
    branches -- the step's C-ABI calls on its input buffer, the copy-in of the next step's inputs
    from pinned host memory into the other buffer, and the read-back of the previous step's
    outputs -- so the host issues one replay per step.  A timed sequence starts with its first
    step's copy-in and ends with its last step's read-back, so every timed step's copies are
    inside the timed region.  With `flush_buf` each graph first overwrites L2 and is timed between
    CUDA events after the flush and at its end; the first graph then also copies its own step's
    inputs in before computing, and the last one reads its own outputs back."""
    L = bench.L
    warm = 3
    steps = [first_step + s for s in range(warm + n)]
    host = []
    for s in steps:
        si = make_step_inputs(w, s, lens, "cpu", w.m_csa)
        pinned = StepInputs(w, w.B, "cpu", pin=True)
        pinned.buf.copy_(si.buf)
        host.append(pinned)
    slabs = [StepInputs(w, w.B, dev) for _ in range(2)]
    outs = [(torch.empty_like(bench.out_c), torch.empty_like(bench.out_h)) for _ in range(2)]
    out_host = [torch.empty(2, w.B, 1, w.H, w.d, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    cs, hs, ds = (torch.cuda.Stream(device=dev) for _ in range(3))
    saved = (bench.out_c, bench.out_h)

    evs = {}

    def chain(i0, i1):
        """Graphs of steps i0..i1-1 (buffer i & 1 for step i)."""
        gs = []
        with torch.cuda.stream(cs):
            for i in range(i0, i1):
                b = i & 1
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
                    if flush_buf is not None:
                        flush_buf.fill_(i & 255)
                        evs[i] = _events(2)
                        _record_external(evs[i][0], cs)
                        if i == i0:
                            slabs[b].buf.copy_(host[i].buf, non_blocking=True)
                    hs.wait_stream(cs)
                    ds.wait_stream(cs)
                    if i + 1 < i1:
                        with torch.cuda.stream(hs):
                            slabs[(i + 1) & 1].buf.copy_(host[i + 1].buf, non_blocking=True)
                    if i > i0:
                        with torch.cuda.stream(ds):
                            out_host[(i - 1) & 1][0].copy_(outs[(i - 1) & 1][0], non_blocking=True)
                            out_host[(i - 1) & 1][1].copy_(outs[(i - 1) & 1][1], non_blocking=True)
                    bench.out_c, bench.out_h = outs[b]
                    bench.step(slabs[b].t)
                    cs.wait_stream(hs)
                    cs.wait_stream(ds)
                    if flush_buf is not None:
                        if i == i1 - 1:
                            out_host[b][0].copy_(outs[b][0], non_blocking=True)
                            out_host[b][1].copy_(outs[b][1], non_blocking=True)
                        _record_external(evs[i][1], cs)
                gs.append(g)
        bench.out_c, bench.out_h = saved
        return gs

    def run(gs, i0, i1):
        if flush_buf is not None:                    # (the first and last copies are in the graphs)
            for g in gs:
                g.replay()
            return
        slabs[i0 & 1].buf.copy_(host[i0].buf, non_blocking=True)
        for g in gs:
            g.replay()
        last = (i1 - 1) & 1
        out_host[last][0].copy_(outs[last][0], non_blocking=True)
        out_host[last][1].copy_(outs[last][1], non_blocking=True)

    g_warm, g_timed = chain(0, warm), chain(warm, warm + n)
    torch.cuda.synchronize()
    with torch.cuda.stream(cs):
        run(g_warm, 0, warm)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        t0.record(cs)
        run(g_timed, warm, warm + n)
        t1.record(cs)
    torch.cuda.synchronize()
    if flush_buf is not None:
        ms = dist.max(sum(_elapsed_ms(evs[i][0], evs[i][1]) for i in range(warm, warm + n))) / n
    else:
        ms = dist.max(t0.elapsed_time(t1)) / n
    assert L.device_status() == 0
    # the copies moved the data: the input buffers hold the last two steps' inputs and the last
    # read-back holds the last step's outputs
    last = warm + n - 1
    assert torch.equal(slabs[last & 1].buf.cpu(), host[last].buf)
    assert n < 2 or torch.equal(slabs[(last - 1) & 1].buf.cpu(), host[last - 1].buf)
    assert torch.equal(out_host[last & 1][0], outs[last & 1][0].cpu())
    assert torch.equal(out_host[last & 1][1], outs[last & 1][1].cpu())
    return {"value": round(w.B * dist.world / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(slabs[0].nbytes), "d2h_bytes_per_step": int(out_host[0].numel() * 2),
            "path": "per step one CUDA graph: the C-ABI calls, the H2D copy of the next step's inputs from "
                    "pinned host memory and the D2H copy of the previous step's outputs as parallel branches "
                    "(the sequence's first copy-in and last read-back inside the timed region too)"
                    + ("; L2 flushed before each step, steps timed alone" if flush_buf is not None else "")}


# --------------------------------------------------------------------- chunked prefill
PREFILL_METRIC = "CSA+HCA chunked-prefill query tokens/s on 1 B300"


def prefill_flops(w):
    """Tensor-core work of one chunk (multiply-adds x 2): the indexer over every causally visible
    CSA entry, CSA attention over k selected entries + W window keys (QK and PV), HCA attention over
    every visible HCA entry + W window keys."""
    o, T = w.offset, w.T
    p = np.arange(o, o + T, dtype=np.int64)
    nv_c = (p + 1) // w.m_csa
    nv_h = (p + 1) // w.m_hca
    index = 2.0 * float(nv_c.sum()) * w.H_I * w.d_I
    csa = 2.0 * 2.0 * T * (w.k + w.W) * w.H * w.d
    hca = 2.0 * 2.0 * float((nv_h + w.W).sum()) * w.H * w.d
    return {"csa_index_topk": index, "csa_attend": csa, "hca_attend": hca, "total": index + csa + hca}


class PrefillBench:
    """A CSA and an HCA layer cache holding a synthetic prior state (entries, index keys and the
    window ring before the chunk, as drawn by the workload), and the chunk's inputs; a step = one
    chunk through both layers.  Every timed step re-processes the same chunk at the same position
    (identical work)."""

    SUBSTEPS = ["compress+quantise", "csa_index_topk", "csa_attend", "hca_attend", "ring_write"]

    def __init__(self, w, device):
        import long_context_sparse_28_b300 as L
        from long_context_sparse_28_b300.layers import CSACache, HCACache, HybridPrefill
        self.L, self.w = L, w
        x = wl.prefill_inputs(w, device)
        o, T, W = w.offset, w.T, w.W
        n_csa, n_hca = o // w.m_csa, o // w.m_hca
        self.csa = CSACache(1, (o + T) // w.m_csa, w.d, W, w.d_I, L.KEY_FMT[w.key_fmt], torch.bfloat16, device)
        self.hca = HCACache(1, (o + T) // w.m_hca, w.d, W, torch.bfloat16, device)
        self.csa.ck[0, :n_csa] = x["csa_ck"]
        self.csa.cv[0, :n_csa] = x["csa_cv"]
        L.csa_index_key_quantize(x["csa_kidx"], self.csa.key_fmt, self.csa.k_codes[0, :n_csa],
                                 None if self.csa.k_scale is None else self.csa.k_scale[0, :n_csa])
        self.hca.ck[0, :n_hca] = x["hca_ck"]
        self.hca.cv[0, :n_hca] = x["hca_cv"]
        pos_ring = torch.tensor([o - W], dtype=torch.int64, device=device)
        for c in (self.csa, self.hca):
            L.swa_ring_write(x["ring_k"][None], x["ring_v"][None], x["ring_gate"][None], pos_ring, W, c.ring_k,
                             c.ring_v, c.ring_gate)
        self.x = x
        self.step_ = HybridPrefill(self.csa, self.hca, T, w.H, w.k, x["csa_bias"], x["hca_bias"], H_I=w.H_I,
                                   q_fp4=w.index_q == "e2m1")
        self.step_.set_position(o)
        self.args = (x["chunk_k"][None], x["chunk_v"][None], x["chunk_gate"][None], x["chunk_kidx"][None],
                     x["q_csa"][None], x["q_idx"][None], x["w"][None], x["q_hca"][None])

    def step(self, args=None):
        return self.step_.step(*(args or self.args))


def cpu_baseline_prefill(w, rows: int):
    """The oracle (as it stands) on `rows` seeded query rows of the chunk (CSA: indexer, top-k and
    attention; HCA: dense attention), scaled to query tokens/s.  Pooling the chunk's blocks is
    included; building the prior state is setup."""
    import oracle
    x = {k: wl.to_numpy(v) for k, v in wl.prefill_inputs(w, "cpu").items()}
    o, T, W = w.offset, w.T, w.W
    fmt = {"f32": oracle.KEY_F32, "bf16": oracle.KEY_BF16, "e4m3": oracle.KEY_E4M3, "e2m1": oracle.KEY_E2M1}[w.key_fmt]
    sel = np.sort(np.random.default_rng(0).choice(T, rows, replace=False))
    t0 = time.perf_counter()
    cck, ccv = oracle.compress(x["chunk_k"], x["chunk_v"], x["chunk_gate"], x["csa_bias"], w.m_csa, oracle.BF16)
    hck, hcv = oracle.compress(x["chunk_k"], x["chunk_v"], x["chunk_gate"], x["hca_bias"], w.m_hca, oracle.BF16)
    ck, cv = np.concatenate([x["csa_ck"], cck]), np.concatenate([x["csa_cv"], ccv])
    codes, sc = oracle.quantize_keys(np.concatenate([x["csa_kidx"], x["chunk_kidx"]]), fmt)
    rawk, rawv = np.concatenate([x["ring_k"], x["chunk_k"]]), np.concatenate([x["ring_v"], x["chunk_v"]])
    pos = o + sel
    oracle.csa_queries(x["q_csa"][sel], x["q_idx"][sel], x["w"][sel], pos, ck, cv, codes, sc, fmt, rawk, rawv, o - W,
                       w.m_csa, w.k, W, w.scale, q_fp4=w.index_q == "e2m1")
    oracle.hca_queries(x["q_hca"][sel], pos, np.concatenate([x["hca_ck"], hck]), np.concatenate([x["hca_cv"], hcv]),
                       rawk, rawv, o - W, w.m_hca, W, w.scale)
    dt = time.perf_counter() - t0
    return dict(value=rows / dt, unit="query tokens/s", cores=oracle.num_threads(), kind="oracle",
                sample=f"{rows} of {T} query rows of the chunk through both layers (fp64 C oracle, OpenMP), the "
                       f"chunk's pooling included, scaled by rows; {dt:.2f} s")


def run_prefill(args, dist):
    import long_context_sparse_28_b300 as L
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    w = wl.shrink(wl.WORKLOADS[args.workload], seed=dist.rank) if dist.world > 1 else wl.WORKLOADS[args.workload]
    K, Wm = args.steps, args.warmup
    bench = PrefillBench(w, dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    # one graph of the chunk's calls; a second one with timing events between the calls
    nsub = 5
    evs = [_events(nsub + 1) for _ in range(K)]
    g = torch.cuda.CUDAGraph()
    c0 = L.launch_count()
    with torch.cuda.stream(stream):
        bench.step()                                   # first run outside capture (per-device set-up)
        stream.synchronize()
        c0 = L.launch_count()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            bench.step()
        launches = L.launch_count() - c0
    torch.cuda.synchronize()
    assert L.device_status() == 0
    with torch.cuda.stream(stream):
        for _ in range(Wm):
            g.replay()
    stream.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    with sampler:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(K):
                g.replay()
            stop.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    dist.barrier()
    ms_per_step = dist.max(start.elapsed_time(stop)) / K
    assert L.device_status(stream) == 0
    # per-call durations, the calls run eagerly between events on the same stream
    st = bench.step_
    csa, hca = bench.csa, bench.hca
    a = bench.args
    calls = [
        lambda: (L.csa_compress(a[0], a[1], a[2], st.p0, st.nT, st.csa_bias, csa.m, csa.ck, csa.cv),
                 L.hca_compress(a[0], a[1], a[2], st.p0, st.nT, st.hca_bias, hca.m, hca.ck, hca.cv),
                 L.csa_index_key_quantize(a[3][0, :w.T // w.m_csa], csa.key_fmt,
                                          csa.k_codes[0, st.pos0 // csa.m:st.pos0 // csa.m + w.T // csa.m],
                                          None if csa.k_scale is None else
                                          csa.k_scale[0, st.pos0 // csa.m:st.pos0 // csa.m + w.T // csa.m])),
        lambda: st.index_topk(a[5], a[6]),
        lambda: L.csa_attend(a[4], st.scale, csa.ck, csa.cv, st.idx, csa.ring_k, csa.ring_v, csa.W, st.q_pos, st.out_c,
                             st.lse_c, chunk_k=a[0], chunk_v=a[1], chunk_pos0=st.p0, workspace=st.ws_ca),
        lambda: L.hca_attend(a[7], st.scale, hca.ck, hca.cv, hca.m, hca.ring_k, hca.ring_v, hca.W, st.q_pos, st.out_h,
                             st.lse_h, chunk_k=a[0], chunk_v=a[1], chunk_pos0=st.p0, workspace=st.ws_ha),
        lambda: (L.swa_ring_write(a[0], a[1], a[2], st.p0, w.T, csa.ring_k, csa.ring_v, csa.ring_gate),
                 L.swa_ring_write(a[0], a[1], a[2], st.p0, w.T, hca.ring_k, hca.ring_v, hca.ring_gate)),
    ]
    with torch.cuda.stream(stream):
        for s in range(K):
            for i in range(nsub):
                _record(evs[s][i], stream)
                calls[i]()
            _record(evs[s][nsub], stream)
    stream.synchronize()
    sub_ms = [statistics.mean(_elapsed_ms(evs[s][i], evs[s][i + 1]) for s in range(K)) for i in range(nsub)]
    per = dict(zip(PrefillBench.SUBSTEPS, sub_ms))
    fl = prefill_flops(w)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    tf_peak = peaks.get("bf16_tflops_sustained", 1400.0)
    dom = max(("csa_index_topk", "csa_attend", "hca_attend"), key=lambda n: per[n])
    # FP4 x FP4 indexer MMAs (kind::mxf8f6f4) run at the 8-bit rate: 2x bf16 (the nominal 4.5 / 2.25
    # ratio); with more than 256 query rows the FP4 operands are expanded exactly to bf16 and scored
    # on the bf16 MMA, so the bf16 peak applies
    fp4_idx = dom == "csa_index_topk" and w.index_q == "e2m1" and w.T <= 256
    if fp4_idx:
        tf_peak = tf_peak * 2
    ach = fl[dom] / (per[dom] / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 1), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(ach / tf_peak, 4), "traffic": None, "algorithmic_flops_per_launch": fl[dom],
                "avg_launch_ms": round(per[dom], 4),
                "peak_source": ("measured (sustained)" if "bf16_tflops_sustained" in peaks else "fallback") +
                               (": bf16 x 2, the 8-bit MMA rate" if fp4_idx else ""),
                "step_tflops": round(fl["total"] / (ms_per_step / 1e3) / 1e12, 1)}
    e2e = None if args.no_e2e else run_e2e_prefill(bench, w, K, dev, dist)
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(w, args.cpu_rows)
    return {
        "metric": PREFILL_METRIC, "value": round(w.T * dist.world / (ms_per_step / 1e3), 1), "unit": "query tokens/s",
        "n_gpus": dist.world, "steps": K, "warmup": Wm, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "offset": w.offset, "H": w.H, "d": w.d,
                   "csa": {"m": w.m_csa, "k": w.k, "W": w.W, "H_I": w.H_I, "d_I": w.d_I, "index_keys": w.key_fmt,
                           "index_queries": "e2m1+ue8m0/32" if w.index_q == "e2m1" else "bf16"},
                   "hca": {"m": w.m_hca, "W": w.W}, "parallelism": f"replicas x{dist.world}",
                   "l2": "scores (1.09 GB) and gathered keys larger than L2; no flush",
                   "tflop_per_step": round(fl["total"] / 1e12, 4),
                   "substep_ms": {n: round(v, 4) for n, v in per.items()}},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches * K),
        "clocks": sampler.summary(),
    }


def run_e2e_prefill(bench, w, n, dev, dist):
    """The public API end to end, as a serving loop would drive it: each step copies the chunk's
    inputs from pinned host memory, runs the chunk's calls (one CUDA graph per buffer) and reads
    both layers' outputs back into pinned host memory, all inside the timed region.  Inputs and
    outputs are double-buffered: the copy-in of step i+1 and the read-back of step i-1 run on their
    own streams (copy engines) while step i computes."""
    L = bench.L
    st = bench.step_
    host = [t.to("cpu").pin_memory() for t in bench.args]          # the chunk, re-sent every step
    dev_in = [[torch.empty_like(t) for t in bench.args] for _ in range(2)]
    outs = [(torch.empty_like(st.out_c), torch.empty_like(st.out_h)) for _ in range(2)]
    out_host = [[torch.empty(st.out_c.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
                for _ in range(2)]
    cs, hs, ds = (torch.cuda.Stream(device=dev) for _ in range(3))
    saved = (st.out_c, st.out_h)
    graphs = []
    with torch.cuda.stream(cs):
        for b in range(2):
            for d_, h_ in zip(dev_in[b], host):
                d_.copy_(h_)
            st.out_c, st.out_h = outs[b]
            bench.step(dev_in[b])
            cs.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
                bench.step(dev_in[b])
            graphs.append(g)
    st.out_c, st.out_h = saved
    torch.cuda.synchronize()
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def run(i0, i1, start_ev):
        hs.wait_event(start_ev)
        for i in range(i0, i1):
            b = i & 1
            if i - i0 >= 2:
                hs.wait_event(comp_done[b])            # step i-2 has consumed this input buffer
            with torch.cuda.stream(hs):
                for d_, h_ in zip(dev_in[b], host):
                    d_.copy_(h_, non_blocking=True)
                h2d_done[b].record(hs)
            cs.wait_event(h2d_done[b])
            if i - i0 >= 2:
                cs.wait_event(d2h_done[b])             # step i-2's outputs have been read back
            graphs[b].replay()
            comp_done[b].record(cs)
            ds.wait_event(comp_done[b])
            with torch.cuda.stream(ds):
                out_host[b][0].copy_(outs[b][0], non_blocking=True)
                out_host[b][1].copy_(outs[b][1], non_blocking=True)
                d2h_done[b].record(ds)
        cs.wait_event(d2h_done[(i1 - 1) & 1])
        cs.wait_event(d2h_done[(i1 - 2) & 1])

    with torch.cuda.stream(cs):
        ev = torch.cuda.Event()
        ev.record(cs)
        run(0, 2, ev)
    torch.cuda.synchronize()
    dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        t0.record(cs)
        run(2, 2 + n, t0)
        t1.record(cs)
    torch.cuda.synchronize()
    ms = dist.max(t0.elapsed_time(t1)) / n
    assert L.device_status() == 0
    return {"value": round(w.T * dist.world / (ms / 1e3), 1), "unit": "query tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host)),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in out_host[0])),
            "path": "per step: H2D copy of the chunk's inputs from pinned host memory, the chunk's C-ABI calls "
                    "(one CUDA graph per buffer), D2H copy of both layers' outputs; inputs and outputs "
                    "double-buffered on copy streams"}


# ------------------------------------------------------------------------- bulk pooling
POOL_METRIC = "CSA+HCA bulk pooling of a 1M-token sequence: raw tokens/s on 1 B300"


def run_pool(args, dist):
    """Both compressors over one sequence's raw K/V/gates (m = 4 and m = 128), the caches written;
    value = raw tokens pooled per second (each token through both compressors)."""
    import long_context_sparse_28_b300 as L
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    n = w.L[0]
    k, v, g = wl.raw_tokens(w, "pool", 0, n, dev)
    k, v, g = k[None].contiguous(), v[None].contiguous(), g[None].contiguous()
    cb, hb = wl.layer_bias(w, "csa", w.m_csa, dev), wl.layer_bias(w, "hca", w.m_hca, dev)
    n_c, n_h = n // w.m_csa, n // w.m_hca
    ck = torch.empty(1, n_c, w.d, dtype=torch.bfloat16, device=dev)
    cv = torch.empty_like(ck)
    hk = torch.empty(1, n_h, w.d, dtype=torch.bfloat16, device=dev)
    hv = torch.empty_like(hk)
    p0 = torch.zeros(1, dtype=torch.int64, device=dev)
    nr = torch.full((1,), n, dtype=torch.int64, device=dev)
    K, Wm = args.steps, args.warmup
    stream = torch.cuda.Stream(device=dev)

    def call(i):
        if i == 0:
            L.csa_compress(k, v, g, p0, nr, cb, w.m_csa, ck, cv)
        else:
            L.hca_compress(k, v, g, p0, nr, hb, w.m_hca, hk, hv)

    with torch.cuda.stream(stream):
        for _ in range(Wm):
            call(0)
            call(1)
    stream.synchronize()
    c0 = L.launch_count()
    evs = [_events(3) for _ in range(K)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    dist.barrier()
    with sampler:
        with torch.cuda.stream(stream):
            for s in range(K):
                _record(evs[s][0], stream)
                call(0)
                _record(evs[s][1], stream)
                call(1)
                _record(evs[s][2], stream)
        stream.synchronize()
    launches = L.launch_count() - c0
    ms_c = statistics.mean(_elapsed_ms(evs[s][0], evs[s][1]) for s in range(K))
    ms_h = statistics.mean(_elapsed_ms(evs[s][1], evs[s][2]) for s in range(K))
    ms_step = dist.max(statistics.mean(_elapsed_ms(evs[s][0], evs[s][2]) for s in range(K)))
    assert L.device_status(stream) == 0
    row = w.d * 2
    bytes_c = n * (2 * row + 4) + n_c * 2 * row          # raw K, V, gates read; entries written
    bytes_h = n * (2 * row + 4) + n_h * 2 * row
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    hbm = peaks.get("hbm_gbs", 6400.0)
    dom, ms_dom, b_dom = ("csa_compress", ms_c, bytes_c) if ms_c >= ms_h else ("hca_compress", ms_h, bytes_h)
    ach = b_dom / (ms_dom / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": None, "algorithmic_bytes_per_launch": int(b_dom),
                "avg_launch_ms": round(ms_dom, 4), "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"}
    e2e = None
    if not args.no_e2e:
        hk_, hv_, hg_ = (t.to("cpu").pin_memory() for t in (k, v, g))
        out_h = torch.empty(ck.shape, dtype=torch.bfloat16, pin_memory=True)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nrep = max(1, min(K, 5))
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(nrep):
                k.copy_(hk_, non_blocking=True)
                v.copy_(hv_, non_blocking=True)
                g.copy_(hg_, non_blocking=True)
                call(0)
                call(1)
                out_h.copy_(ck, non_blocking=True)
            t1.record(stream)
        stream.synchronize()
        ms_e = dist.max(t0.elapsed_time(t1)) / nrep
        e2e = {"value": round(n / (ms_e / 1e3), 1), "unit": "raw tokens/s", "ms_per_step": round(ms_e, 4),
               "h2d_bytes_per_step": int(hk_.numel() * 2 + hv_.numel() * 2 + hg_.numel() * 4),
               "d2h_bytes_per_step": int(out_h.numel() * 2),
               "path": "per step: H2D copy of the raw K, V and gates from pinned host memory, both compressors, "
                       "D2H copy of the CSA keys' cache"}
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        nb = 2048                                     # a bounded sample: the first 2048 x 128 tokens
        K_, V_, G_ = (wl.to_numpy(t[0, :nb * w.m_hca]) for t in (k, v, g))
        t0c = time.perf_counter()
        oracle.compress(K_, V_, G_, wl.to_numpy(cb), w.m_csa, oracle.BF16)
        oracle.compress(K_, V_, G_, wl.to_numpy(hb), w.m_hca, oracle.BF16)
        dt = time.perf_counter() - t0c
        cpu = {"value": round(nb * w.m_hca / dt, 1), "unit": "raw tokens/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": f"the first {nb * w.m_hca} of {n} tokens through both compressors "
                                           f"(fp64 C oracle, OpenMP); {dt:.2f} s"}
    return {"metric": POOL_METRIC, "value": round(n * dist.world / (ms_step / 1e3), 1), "unit": "raw tokens/s",
            "n_gpus": dist.world, "steps": K, "warmup": Wm, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "L": n, "d": w.d, "m": [w.m_csa, w.m_hca],
                       "parallelism": f"replicas x{dist.world}",
                       "l2": "inputs (516 MB) larger than L2; no flush",
                       "substep_ms": {"csa_compress": round(ms_c, 4), "hca_compress": round(ms_h, 4)},
                       "algorithmic_bytes": {"csa_compress": int(bytes_c), "hca_compress": int(bytes_h)}},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": sampler.summary()}


# ------------------------------------------------------------------------ reference arm
def run_reference(args, dist):
    """The CPU oracle as it stands, on the host cores, on a bounded sample of the workload:
    each step = one sequence's decode query through both layers."""
    import oracle
    w = wl.WORKLOADS[args.workload]
    if not w.kind.endswith("_decode"):
        return {"impl": "reference", "unavailable": f"the reference arm times the oracle on the decode workloads; "
                                                    f"{w.name} is a {w.kind} workload"}
    layers = DEFAULT_LAYERS[w.kind]
    fmt = {"f32": oracle.KEY_F32, "bf16": oracle.KEY_BF16, "e4m3": oracle.KEY_E4M3, "e2m1": oracle.KEY_E2M1}[w.key_fmt]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    nseq = min(2, w.B)
    lens = w.lengths()
    ctx = []
    for b in range(nseq):
        Lb = lens[b]
        K = V = ck = cv = codes = sc = HK = HV = hck = hcv = None
        if layers in ("both", "csa"):
            k, v, g = wl.raw_tokens(w, "csa", b, Lb, dev)
            kin = wl.index_key_inputs(w, "csa", b, Lb // w.m_csa + 1, dev)
            K, V, G, KIN = (wl.to_numpy(x) for x in (k, v, g, kin))
            ck, cv = _oracle_caches(oracle, K, V, G, wl.to_numpy(wl.layer_bias(w, "csa", w.m_csa, dev)), w.m_csa,
                                    w.kv_cache)
            codes, sc = oracle.quantize_keys(KIN[: Lb // w.m_csa], fmt)
        if layers in ("both", "hca"):
            hk, hv, hg = wl.raw_tokens(w, "hca", b, Lb, dev)
            HK, HV, HG = (wl.to_numpy(x) for x in (hk, hv, hg))
            hck, hcv = _oracle_caches(oracle, HK, HV, HG, wl.to_numpy(wl.layer_bias(w, "hca", w.m_hca, dev)),
                                      w.m_hca, w.kv_cache)
        q = wl.to_numpy(wl.queries(w, "csa", b, 1, dev))
        qh = wl.to_numpy(wl.queries(w, "hca", b, 1, dev))
        qi, ww = (wl.to_numpy(x) for x in wl.indexer_queries(w, "csa", b, 1, dev))
        ctx.append((Lb, K, V, ck, cv, codes, sc, HK, HV, hck, hcv, q, qh, qi, ww))

    def step(i):
        (Lb, K, V, ck, cv, codes, sc, HK, HV, hck, hcv, q, qh, qi, ww) = ctx[i % len(ctx)]
        if layers in ("both", "csa"):
            oracle.csa_queries(q, qi, ww, [Lb - 1], ck, cv, codes, sc, fmt, K, V, 0, w.m_csa, w.k, w.W, w.scale,
                               q_fp4=w.index_q == "e2m1")
        if layers in ("both", "hca"):
            oracle.hca_queries(qh, [Lb - 1], hck, hcv, HK, HV, 0, w.m_hca, w.W, w.scale)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cpu = {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"each step = one of {nseq} sequences of {w.name}, one decode query through the workload's "
                     f"layers ({layers}; fp64 C oracle, OpenMP); cache construction untimed"}
    return {"metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "sample_sequences": nseq},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            if dist.rank != 0:
                return
            line = run_reference(args, dist)
        elif wl.WORKLOADS[args.workload].kind == "hybrid_prefill":
            line = run_prefill(args, dist)
        elif wl.WORKLOADS[args.workload].kind == "pool":
            line = run_pool(args, dist)
        else:
            line = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
