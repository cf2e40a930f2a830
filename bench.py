#!/usr/bin/env python
"""Throughput of the TokenGate gated-prefill step on B300.

One step = the whole hot path on one synthetic prompt already resident in
HBM: gate MLP over all N tokens -> top-K select over the document span ->
gather of the kept rows -> QKV projection -> key-bias causal attention over
the kept rows.  Default workload: Qwen3-1.7B shapes at N = 131072 (document
130816, question 256, 6.25% of the document kept), the long-context end of
the 16k-128k range; the 16k, 32k and 64k workloads run with --workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-graph]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own copy
of the workload (independent prompts, no data-path collective) and the
reported value is the tokens of all ranks over the slowest rank's time.
`--impl reference` times the fp64 CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import tg_inputs as TI  # noqa: E402

METRIC = "gated-prefill tokens/s at 16k–128k; key-bias attn TFLOP/s and % of roofline"
DEFAULT_WORKLOAD = "qwen3_1p7b_n128k_keep6p25"
# the hybrid model's gated layer is reported on a 32k prompt; 10% kept
DELTANET_WORKLOAD = "qwen3_1p7b_n32k_sweep"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNELS = ("gate_score", "select_topk", "gather_rows", "qkv_proj", "keybias_attn")
PIPELINE = ("gate_score", "select_topk", "gather_rows")  # the HBM-bound front of the step
# the sources each kernel's code comes from (the attention dispatcher and
# its short-sequence kernel live in keybias_attn_1h.cu)
KERNEL_SOURCES = {"gate_score": ("gemm_tc.cu",), "select_topk": ("select_topk.cu",),
                  "gather_rows": ("rows.cu",), "qkv_proj": ("gemm_tc.cu",),
                  "keybias_attn": ("keybias_attn.cu", "keybias_attn_1h.cu"),
                  "keybias_bias_grad": ("attn_bwd.cu",),
                  "gated_delta_rule": ("deltanet.cu", "deltanet_tc.cu")}
# DRAM bytes per launch from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by workload/kernel, with the sha256 (first 16
# hex) of the kernel's source at capture time; a stale hash reports null.
NCU_TRAFFIC: dict[str, dict] = {
    # Qwen3-1.7B shapes, N = 16384, 10% of the document kept (M = 1868)
    "qwen3_1p7b_n16k_keep10/gate_score": {"bytes_per_launch": 68190720 + 17920,
                                          "source_sha": "0f25d4a8caaef008"},
    "qwen3_1p7b_n16k_keep10/select_topk": {"bytes_per_launch": 130304,
                                           "source_sha": "60fe527eba4acb2d"},
    "qwen3_1p7b_n16k_keep10/gather_rows": {"bytes_per_launch": 7729152,
                                           "source_sha": "27ffa82b44661223"},
    "qwen3_1p7b_n16k_keep10/qkv_proj": {"bytes_per_launch": 24450304,
                                        "source_sha": "0f25d4a8caaef008"},
    "qwen3_1p7b_n16k_keep10/keybias_attn": {"bytes_per_launch": 15368192,
                                            "source_sha": "1c005f0c3228e382"},
    # N = 131072, 6.25% of the document kept (M = 8432)
    "qwen3_1p7b_n128k_keep6p25/gate_score": {"bytes_per_launch": 537975808 + 367616,
                                             "source_sha": "0f25d4a8caaef008"},
    "qwen3_1p7b_n128k_keep6p25/select_topk": {"bytes_per_launch": 588800,
                                              "source_sha": "60fe527eba4acb2d"},
    "qwen3_1p7b_n128k_keep6p25/gather_rows": {"bytes_per_launch": 35035136 + 19968,
                                              "source_sha": "27ffa82b44661223"},
    "qwen3_1p7b_n128k_keep6p25/qkv_proj": {"bytes_per_launch": 51419648 + 20432896,
                                           "source_sha": "0f25d4a8caaef008"},
    "qwen3_1p7b_n128k_keep6p25/keybias_attn": {"bytes_per_launch": 69526784 + 6329600,
                                               "source_sha": "1c005f0c3228e382"},
    # the backward's bias-gradient kernel at M = 8432
    "qwen3_1p7b_n128k_keep6p25/keybias_bias_grad": {"bytes_per_launch": 137630464 + 3417344,
                                                    "source_sha": "3d91e7a27c9845f8"},
    # the delta rule over the 3507 kept tokens of the 32k prompt (10% budget),
    # both kernels of one call: chunk preparation + state scan
    "qwen3_1p7b_n32k_sweep/gated_delta_rule": {
        "bytes_per_launch": (29930240 + 3514368) + (72087296 + 1188864),
        "source_sha": "8d0ec53ce4a61ce6"},
}


# --------------------------------------------------------------- workloads --
def algorithmic_work(w: TI.Workload, K: int) -> dict:
    """Algorithmic bytes / flops of each kernel for one step (no re-reads)."""
    N, D, d, Hg = w.N, w.D, w.d, w.Hg
    M = w.M(K)
    cols = w.qkv_cols
    e = 2  # bf16 bytes
    return {
        "gate_score": {"bytes": N * d * e + Hg * d * e + 2 * Hg * 4 + N * 4,
                       "flops": 2 * N * d * Hg, "bound": "hbm"},
        "select_topk": {"bytes": 4 * D + 4 * M, "flops": 0, "bound": "hbm"},
        "gather_rows": {"bytes": 2 * M * d * e + 3 * 4 * M, "flops": 0, "bound": "hbm"},
        "qkv_proj": {"bytes": M * d * e + cols * d * e + M * cols * e,
                     "flops": 2 * M * d * cols, "bound": "tensor"},
        # causal half of the 4 M^2 dh Hq of dense attention
        "keybias_attn": {"bytes": M * cols * e + M * 4 + M * w.Hq * w.dh * e,
                         "flops": 2 * M * M * w.dh * w.Hq, "bound": "tensor"},
    }


def tensor_peak(peaks: dict, clocks: dict | None) -> tuple[float, str]:
    """The bf16 denominator for a contraction timed in this run: the burst
    figure while the SMs held their clock, the sustained one (a seconds-long
    GEMM loop under the power cap) when the run was power-capped or its
    median SM clock fell below 97% of the maximum."""
    capped = False
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        capped = ("sw_power_cap" in (clocks.get("reasons") or [])
                  or clocks["sm_mhz"] < 0.97 * clocks["sm_max_mhz"])
    if capped:
        return peaks["bf16_tflops_sustained"], (
            f"bf16 sustained: this run was power-capped, median SM clock "
            f"{clocks['sm_mhz']:.0f} of {clocks['sm_max_mhz']:.0f} MHz")
    return peaks["bf16_tflops"], "bf16 burst"


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(fnames) -> str:
    """sha256 (first 16 hex) of the named csrc files, concatenated in order."""
    h = hashlib.sha256()
    for fname in ([fnames] if isinstance(fnames, str) else fnames):
        with open(os.path.join(ROOT, "learned_token_pruning_residual_b300", "csrc", fname),
                  "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` at `workload` from the ncu table, or
    None when there is no capture or the kernel's source changed since."""
    trf = NCU_TRAFFIC.get(f"{workload}/{kernel}")
    if trf and kernel in KERNEL_SOURCES and trf.get("source_sha") == \
            source_hash(KERNEL_SOURCES[kernel]):
        return trf["bytes_per_launch"]
    return None


# ------------------------------------------------------------ distribution --
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank: int, world: int, max_ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (max_ms_per_step * 1e-3)


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons,
    kept only while `active` is set (the timed region)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples: list[list[str]] = []
        self.active = False
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.samples.append([x.strip() for x in line.split(",")])

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sms = [float(s[0]) for s in self.samples if len(s) >= 8 and s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if len(s) >= 8 and s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i - 4] for s in self.samples if len(s) >= 8
                          for i in range(4, 8) if s[i].lower() == "active"})
        return {"sm_mhz": float(np.median(sms)) if sms else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sms)}


# ------------------------------------------------------------- oracle arm --
def oracle_sample_step(w, K, host, full, f: float, rng) -> tuple[float, float]:
    """One step of the fp64 oracle, charged against f * N prompt tokens:
    the row-wise stages (gate rows, QKV rows, attention query rows) run on a
    uniform row sample of fraction f; select and gather need the whole
    prompt, so they run once on it and f of their time is charged (their
    cost is linear in the prompt, so f of it is the sampled tokens' share).
    Returns (seconds charged, tokens covered)."""
    import oracle as O
    X, gp, Wqkv, ap = host["X"], host["gp"], host["Wqkv"], host["ap"]
    M = w.M(K)
    t0 = time.perf_counter()
    idx = O.select_topk(full["s32"], w.doc_begin, w.doc_end, K)
    Xk, ls = O.gather_rows(X, idx, full["s32"])
    t_whole = time.perf_counter() - t0
    t1 = time.perf_counter()
    rows = np.sort(rng.choice(w.N, size=max(1, int(round(f * w.N))), replace=False))
    O.gate_score(X[rows], gp["W1"], gp["b1"], gp["w2"], gp["b2"])
    qrows = np.sort(rng.choice(M, size=max(1, int(round(f * M))), replace=False))
    O.qkv_proj(Xk[qrows], Wqkv)
    O.keybias_attn(full["qkv"], w.Hq, w.Hkv, w.dh, ls, ap["gain"], ap["temperature"], rows=qrows)
    t_rows = time.perf_counter() - t1
    return t_rows + f * t_whole, f * w.N


def oracle_setup(w, K):
    import oracle as O
    host = {"X": TI.residual(w), "gp": TI.gate_params(w), "Wqkv": TI.qkv_weight(w),
            "ap": TI.attn_params(w)}
    s = O.gate_score(host["X"], host["gp"]["W1"], host["gp"]["b1"], host["gp"]["w2"],
                     host["gp"]["b2"])
    s32 = s.astype(np.float32)
    idx = O.select_topk(s32, w.doc_begin, w.doc_end, K)
    Xk, _ = O.gather_rows(host["X"], idx, s32)
    return host, {"s32": s32, "qkv": O.qkv_proj(Xk, host["Wqkv"])}


def cudart():
    """The CUDA runtime library this process already loaded (through torch)."""
    with open("/proc/self/maps") as f:
        for line in f:
            if "libcudart" in line:
                L = ctypes.CDLL(line.split()[-1])
                break
        else:
            L = ctypes.CDLL("libcudart.so")
    L.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    L.cudaEventRecordWithFlags.restype = ctypes.c_int
    return L


def blas_threads() -> int:
    """Threads the oracle's BLAS calls use (its matmuls, which dominate its
    time); its elementwise numpy steps run on one thread."""
    try:
        import threadpoolctl
        info = [i for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    return host_cores()


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_fraction(w, K, host, full, budget_s: float, steps: int) -> float:
    """Row fraction so that `steps` sampled steps take about budget_s."""
    rng = np.random.default_rng(0)
    f0 = 1.0 / 16
    t, _ = oracle_sample_step(w, K, host, full, f0, rng)
    per_full = t / f0
    return float(min(1.0, max(1.0 / 256, budget_s / max(steps, 1) / per_full)))


def cpu_baseline(w, K, budget_s: float = 15.0) -> dict:
    host, full = oracle_setup(w, K)
    f = oracle_fraction(w, K, host, full, budget_s, steps=4)
    rng = np.random.default_rng(1)
    secs, toks, n = 0.0, 0.0, 0
    while secs < budget_s * 0.66 or n < 2:
        t, tk = oracle_sample_step(w, K, host, full, f, rng)
        secs += t
        toks += tk
        n += 1
    return {"value": toks / secs, "unit": "tokens/s", "cores": blas_threads(),
            "host_cores": host_cores(), "kind": "oracle",
            "sample": (f"{n} fp64 oracle steps, each on a uniform {f:.4f} row sample of gate rows, "
                       f"QKV rows and attention query rows of {w.name}; select and gather run on "
                       f"the whole prompt and {f:.4f} of their time is charged; {secs:.1f} s of "
                       f"CPU work; tokens/s = sampled tokens / charged time")}


def workload_config(w, K: int, world: int) -> dict:
    """The `config` of the JSON line: the workload, as both arms report it."""
    return {"workload": w.name, "N": w.N, "doc": [w.doc_begin, w.doc_end], "K": K, "M": w.M(K),
            "d_model": w.d, "gate_hidden": w.Hg, "heads_q": w.Hq, "heads_kv": w.Hkv,
            "head_dim": w.dh, "parallelism": f"replicas x{world}",
            "l2": "flushed between steps (256 MiB write), outside the timed events"}


def run_reference(args, w, K, rank, world):
    if rank != 0:
        return 0
    host, full = oracle_setup(w, K)
    steps = args.steps + args.warmup
    f = oracle_fraction(w, K, host, full, budget_s=150.0, steps=steps)
    rng = np.random.default_rng(2)
    for _ in range(args.warmup):
        oracle_sample_step(w, K, host, full, f, rng)
    secs, toks = 0.0, 0.0
    for _ in range(args.steps):
        t, tk = oracle_sample_step(w, K, host, full, f, rng)
        secs += t
        toks += tk
    value = toks / secs
    sample = (f"fp64 oracle, each step a uniform {f:.4f} row sample of gate rows, QKV rows and "
              f"attention query rows of {w.name}; select and gather on the whole prompt, "
              f"{f:.4f} of their time charged")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, K, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                             "host_cores": host_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm --
def run_gpu(args, w, K, rank, world, local_rank):
    import torch

    import learned_token_pruning_residual_b300 as tg

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = dist_init(world, "nccl")
    L = tg.lib()

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    X_host = TI.residual(w)
    gp, Wqkv_h, ap = TI.gate_params(w), TI.qkv_weight(w), TI.attn_params(w)
    M = w.M(K)
    W1, b1, w2 = to_dev(gp["W1"]), to_dev(gp["b1"]), to_dev(gp["w2"])
    Wqkv, gain = to_dev(Wqkv_h), to_dev(ap["gain"])
    bf = torch.bfloat16

    def make_bufs(X=None):
        """One prompt's device buffers: the residual and every step output."""
        return {"X": X if X is not None else torch.empty(w.N, w.d, dtype=bf, device=dev),
                "s": torch.empty(w.N, dtype=torch.float32, device=dev),
                "idx": torch.empty(M, dtype=torch.int32, device=dev),
                "Xk": torch.empty(M, w.d, dtype=bf, device=dev),
                "ls": torch.empty(M, dtype=torch.float32, device=dev),
                "qkv": torch.empty(M, w.qkv_cols, dtype=bf, device=dev),
                "out": torch.empty(M, w.Hq * w.dh, dtype=bf, device=dev),
                "ws": tg.new_select_workspace(dev)}

    A = make_bufs(to_dev(X_host))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    m_out = ctypes.c_int64(0)
    ws_bytes = tg.tg_select_workspace_bytes()
    t = ap["temperature"]
    wp = {"W1": W1.data_ptr(), "b1": b1.data_ptr(), "w2": w2.data_ptr(),
          "Wqkv": Wqkv.data_ptr(), "gain": gain.data_ptr()}

    def check(st):
        if st != 0:
            raise tg.TokenGateError(st, L.tg_last_error_message().decode())

    def make_calls(bufs, sh):
        """The five C-ABI calls of one step on stream handle sh, with raw
        pointers (no per-call marshalling)."""
        p = {k: v.data_ptr() for k, v in bufs.items()}
        return [
            lambda: check(L.tg_gate_score(p["X"], 1, w.N, w.d, wp["W1"], wp["b1"], w.Hg,
                                          wp["w2"], gp["b2"], p["s"], p["ws"], w.doc_begin,
                                          w.doc_end, sh)),
            lambda: check(L.tg_select_topk(p["s"], w.N, w.doc_begin, w.doc_end, K, p["idx"],
                                           ctypes.byref(m_out), p["ws"], ws_bytes, sh)),
            lambda: check(L.tg_gather_rows(p["X"], 1, w.N, w.d, p["idx"], M, p["Xk"], 1,
                                           p["s"], p["ls"], sh)),
            lambda: check(L.tg_qkv_proj(p["Xk"], 1, M, w.d, wp["Wqkv"], w.Hq, w.Hkv, w.dh,
                                        p["qkv"], sh)),
            lambda: check(L.tg_keybias_attn(p["qkv"], 1, M, w.Hq, w.Hkv, w.dh, p["ls"],
                                            wp["gain"], t, p["out"], None, sh)),
        ]

    def run_calls(calls, evs=None, record=None):
        if evs is not None:
            record(evs[0])
        for i, c in enumerate(calls):
            c()
            if evs is not None:
                record(evs[i + 1])

    calls_direct = make_calls(A, stream.cuda_stream)
    nev = len(KERNELS) + 1
    graph, graph_inst, gev = None, None, None
    side = torch.cuda.Stream(dev)
    plan_args = (W1, b1, w2, gp["b2"], w.doc_begin, w.doc_end, K, Wqkv, w.Hq, w.Hkv, w.dh, gain,
                 t)

    def make_plan(bufs):
        """The library's CUDA graph of the five calls on one buffer set."""
        return tg.GatedLayerPlan(bufs["X"], *plan_args,
                                 bufs={"scores": bufs["s"], "select_ws": bufs["ws"],
                                       "idx": bufs["idx"], "Xk": bufs["Xk"],
                                       "logsig": bufs["ls"], "qkv": bufs["qkv"],
                                       "out": bufs["out"]})

    if not args.no_graph:
        # The step is the library's plan (tg_gated_layer_plan_create: the five
        # calls captured into one CUDA graph), timed by events around each
        # launch.  A second copy with an event-record node before and after
        # every call, captured here and replayed separately, gives the
        # per-kernel device times; the record nodes serialise the kernels
        # (their prologues can no longer overlap the previous kernel's
        # tail), so they stay out of the timed step.
        run_calls(calls_direct)  # load modules / set attributes outside capture
        torch.cuda.synchronize()
        graph = make_plan(A)
        graph_inst = torch.cuda.CUDAGraph()
        gev = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
        for ev in gev:  # torch creates the event handle on its first record
            ev.record(stream)
        torch.cuda.synchronize()
        rt = cudart()

        def record_node(ev):  # cudaEventRecordExternal: a real record node in the graph
            rc = rt.cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event),
                                             ctypes.c_void_p(side.cuda_stream), 1)
            if rc != 0:
                raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")

        calls_side = make_calls(A, side.cuda_stream)
        with torch.cuda.graph(graph_inst, stream=side):
            run_calls(calls_side, gev, record_node)

    def step():
        if graph is None:
            run_calls(calls_direct)
        else:
            graph.launch(stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if tg.tg_get_device_status(raise_on_error=False) != 0:
        raise RuntimeError("device status set during warm-up")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    if sampler:
        sampler.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev if graph is None else 2)]
           for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.active = True
    torch.cuda._sleep(50_000_000)  # let the host queue run ahead of the device
    for k in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the timed events
        if graph is None:
            run_calls(calls_direct, evs[k], lambda ev: ev.record(stream))
        else:
            evs[k][0].record(stream)
            graph.launch(stream.cuda_stream)
            evs[k][1].record(stream)
    torch.cuda.synchronize()
    clocks = None
    if sampler:
        sampler.active = False
        clocks = sampler.stop()
    if dist:
        dist.barrier()
    st = tg.tg_get_device_status(raise_on_error=False)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    step_ms = np.array([e[0].elapsed_time(e[-1]) for e in evs])
    if graph is None:
        per = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(len(KERNELS))] for e in evs])
        inst_ms = None
    else:
        # per-kernel device times from the instrumented copy of the step
        n_inst = max(1, min(args.steps, 200))
        for _ in range(3):
            flush.zero_()
            graph_inst.replay()
        torch.cuda.synchronize()
        per = np.zeros((n_inst, len(KERNELS)))
        inst_ms = np.zeros(n_inst)
        for k in range(n_inst):
            flush.zero_()
            graph_inst.replay()
            gev[-1].synchronize()  # read this step's event nodes before the next replay
            per[k] = [gev[i].elapsed_time(gev[i + 1]) for i in range(len(KERNELS))]
            inst_ms[k] = gev[0].elapsed_time(gev[-1])
    ms_per_step = reduce_max(float(step_ms.mean()), dist, dev)
    value = aggregate_tokens_per_s(w.N, world, ms_per_step)

    # ---- clocks over a longer stretch of the same step (the timed region
    # above can be a few milliseconds, shorter than the 50 ms sampling
    # period): the graph replayed back to back for about a second
    soak = None
    if rank == 0 and not args.no_clock_soak:
        soak_sampler = ClockSampler(uuid)
        soak_sampler.start()
        n_soak = int(min(20000, max(50, 1000.0 / max(ms_per_step, 1e-3))))
        soak_sampler.active = True
        for _ in range(n_soak):
            step()
        torch.cuda.synchronize()
        soak_sampler.active = False
        soak = soak_sampler.stop()
        soak["steps"] = n_soak

    # ---- end to end through the C ABI from pinned host memory, every step:
    # H2D of the prompt's residual, the five calls, D2H of the attention
    # output and the kept indices.  Two buffer sets alternate, so the copies
    # of one prompt overlap the kernels of the other (copy stream + events);
    # the time is the whole run over the number of prompts.
    X_pin = torch.from_numpy(X_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    B = make_bufs()
    sets = [A, B]
    outs_pin = [(torch.empty(M, w.Hq * w.dh, dtype=bf).pin_memory(),
                 torch.empty(M, dtype=torch.int32).pin_memory()) for _ in sets]
    copy = torch.cuda.Stream(dev)
    set_plans = [graph, make_plan(B)] if graph is not None else None
    set_calls = [make_calls(b, stream.cuda_stream) for b in sets]
    h2d_done = [torch.cuda.Event() for _ in sets]
    comp_done = [torch.cuda.Event() for _ in sets]
    d2h_done = [torch.cuda.Event() for _ in sets]
    for e in d2h_done:
        e.record(copy)
    e2e_steps = max(4, min(args.steps, 100))
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(-2, e2e_steps):
        if k == 0:
            torch.cuda.synchronize()
            e_start.record(copy)
        j = k % 2
        b = sets[j]
        with torch.cuda.stream(copy):
            copy.wait_event(d2h_done[j])  # this set's previous result has left the device
            b["X"].copy_(X_pin, non_blocking=True)
            h2d_done[j].record(copy)
        stream.wait_event(h2d_done[j])
        if set_plans is not None:
            set_plans[j].launch(stream.cuda_stream)
        else:
            run_calls(set_calls[j])
        comp_done[j].record(stream)
        with torch.cuda.stream(copy):
            copy.wait_event(comp_done[j])
            outs_pin[j][0].copy_(b["out"], non_blocking=True)
            outs_pin[j][1].copy_(b["idx"], non_blocking=True)
            d2h_done[j].record(copy)
    e_end.record(copy)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e_start.elapsed_time(e_end) / e2e_steps, dist, dev)
    # both sets ran the same prompt: their outputs must agree bit for bit
    assert torch.equal(outs_pin[0][1], outs_pin[1][1])
    assert torch.equal(outs_pin[0][0].view(torch.int16), outs_pin[1][0].view(torch.int16))
    assert np.isfinite(outs_pin[0][0][:4].float().numpy()).all()
    h2d_bytes = int(A["X"].numel() * 2)
    d2h_bytes = int(A["out"].numel() * 2 + A["idx"].numel() * 4)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    work = algorithmic_work(w, K)
    peaks, peak_src = load_peaks()
    kernels = {}
    for i, name in enumerate(KERNELS):
        ms = float(per[:, i].mean())
        wk = work[name]
        kernels[name] = {"ms": ms, "GB/s": wk["bytes"] / ms / 1e6,
                         "TFLOP/s": wk["flops"] / ms / 1e9 if wk["flops"] else None}
    dom = max(KERNELS, key=lambda n: kernels[n]["ms"])
    wk = work[dom]
    ms = kernels[dom]["ms"]
    tpeak, tpeak_kind = tensor_peak(peaks, clocks)
    if wk["bound"] == "tensor":
        ach, peak, unit = wk["flops"] / ms / 1e9, tpeak, "TFLOP/s"
    else:
        ach, peak, unit = wk["bytes"] / ms / 1e6, peaks["hbm_gbs"], "GB/s"
    roofline = {"kernel": dom, "bound": wk["bound"], "achieved": ach, "peak": peak,
                "unit": unit, "frac": ach / peak, "traffic": ncu_traffic(w.name, dom),
                "algorithmic": wk["flops"] if wk["bound"] == "tensor" else wk["bytes"],
                "peak_source": f"{peak_src} ({tpeak_kind if unit == 'TFLOP/s' else 'HBM copy'})"}
    pipe_bytes = sum(work[n]["bytes"] for n in PIPELINE)
    pipe_ms = sum(kernels[n]["ms"] for n in PIPELINE)
    pipeline = {"kernels": list(PIPELINE), "bytes": pipe_bytes, "ms": pipe_ms,
                "GB/s": pipe_bytes / pipe_ms / 1e6, "peak": peaks["hbm_gbs"],
                "frac": pipe_bytes / pipe_ms / 1e6 / peaks["hbm_gbs"],
                "peak_source": f"{peak_src} (HBM copy)"}
    attn = kernels["keybias_attn"]
    e2e_s = e2e_ms * 1e-3
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, K, world),
        "timing": ("one launch per step of the library's plan (the five calls as one CUDA "
                   "graph, tg_gated_layer_plan_create), timed by events around each launch; "
                   "per-kernel times from a separately replayed copy with an event-record node "
                   "around every call" if graph is not None else "direct C-ABI calls"),
        "roofline": roofline,
        "pipeline": pipeline,
        "attn_tflops": attn["TFLOP/s"],
        "attn_frac_bf16_peak": attn["TFLOP/s"] / tpeak,
        "kernels": kernels,
        "instrumented_ms_per_step": float(inst_ms.mean()) if inst_ms is not None else None,
        "e2e": {"value": aggregate_tokens_per_s(w.N, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "ms_per_step": e2e_ms,
                "host_link_gbs": (h2d_bytes + d2h_bytes) / e2e_s / 1e9,
                "how": ("two buffer sets alternate: the H2D copy of one prompt and the D2H "
                        "copy of the other's result run on a copy stream while the kernels "
                        "run; time = whole run / prompts")},
        "gpu_launches": len(KERNELS) * args.steps,
        "clocks": clocks,
        "clocks_soak": soak,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, K)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------- gated vs full ----
def run_compare(args, w, K, rank, world, local_rank):
    """The pages' comparison at one workload: the gated path (gate, select,
    gather, then the pruned layers on the M kept rows) against full prefill
    (the same layers on all N rows, no bias), on the same kernels.  A
    one-layer workload runs one attention layer; the 20-layer workload runs
    x <- x + attn(qkv(RMSNorm(x))) per layer on an fp32 residual stream.
    Reports tokens/s of both and the peak device memory each path allocates
    (inputs and weights included)."""
    import torch

    import learned_token_pruning_residual_b300 as tg

    if rank != 0:
        return 0
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    qwen3 = args.decoder == "qwen3"
    stack = w.layers > 1 or qwen3
    M = w.M(K)
    X_host = TI.residual(w)
    gp = TI.gate_params(w)
    W1, b1, w2 = to_dev(gp["W1"]), to_dev(gp["b1"]), to_dev(gp["w2"])
    if qwen3:
        # full Qwen3 decoder layers (q/k norm, rotary embedding at the prompt
        # positions, o-projection, SwiGLU MLP); weights moved to the device one
        # layer at a time
        layers = []
        for i in range(w.layers):
            P = TI.qwen3_layer_params(w, layer=i)
            layers.append({k: (to_dev(v) if isinstance(v, np.ndarray) else v) for k, v in P.items()})
    else:
        layers_h = [{"Wqkv": TI.qkv_weight(w, layer=i), "gamma": TI.rms_gamma(w, layer=i),
                     **TI.attn_params(w, layer=i)} for i in range(w.layers)]
        layers = [{"Wqkv": to_dev(L["Wqkv"]), "gamma": to_dev(L["gamma"]),
                   "gain": to_dev(L["gain"]), "temperature": L["temperature"]} for L in layers_h]
    X = to_dev(X_host)
    bf, f32 = torch.bfloat16, torch.float32

    def gated_bufs():
        b = {"scores": torch.empty(w.N, dtype=f32, device=dev),
             "idx": torch.empty(M, dtype=torch.int32, device=dev),
             "logsig": torch.empty(M, dtype=f32, device=dev),
             "qkv": torch.empty(M, w.qkv_cols, dtype=bf, device=dev),
             "ws": tg.new_select_workspace(dev)}
        if stack:
            b["x"] = torch.empty(M, w.d, dtype=f32, device=dev)
            b["xn"] = torch.empty(M, w.d, dtype=bf, device=dev)
        else:
            b["Xk"] = torch.empty(M, w.d, dtype=bf, device=dev)
            b["out"] = torch.empty(M, w.Hq * w.dh, dtype=bf, device=dev)
        return b

    def full_bufs():
        b = {"qkv": torch.empty(w.N, w.qkv_cols, dtype=bf, device=dev)}
        if stack:
            b["x"] = torch.empty(w.N, w.d, dtype=f32, device=dev)
            b["xn"] = torch.empty(w.N, w.d, dtype=bf, device=dev)
        else:
            b["out"] = torch.empty(w.N, w.Hq * w.dh, dtype=bf, device=dev)
        return b

    def gated(b):
        s = tg.tg_gate_score(X, W1, b1, w2, gp["b2"], out=b["scores"], select_ws=b["ws"],
                             doc_begin=w.doc_begin, doc_end=w.doc_end)
        idx = tg.tg_select_topk(s, w.doc_begin, w.doc_end, K, out=b["idx"], workspace=b["ws"])
        if qwen3:
            tg.tg_gather_rows(X, idx, s, out=b["x"], logsig_out=b["logsig"])
            tg.qwen3_pruned_stack(b["x"], idx, layers, w.Hq, w.Hkv, w.dh, b["logsig"],
                                  bufs={"xn": b["xn"], "qkv": b["qkv"]})
        elif stack:
            tg.tg_gather_rows(X, idx, s, out=b["x"], logsig_out=b["logsig"])
            tg.pruned_stack(b["x"], layers, w.Hq, w.Hkv, w.dh, b["logsig"],
                            bufs={"xn": b["xn"], "qkv": b["qkv"]})
        else:
            L0 = layers[0]
            Xk, ls = tg.tg_gather_rows(X, idx, s, out=b["Xk"], logsig_out=b["logsig"])
            tg.tg_qkv_proj(Xk, L0["Wqkv"], w.Hq, w.Hkv, w.dh, out=b["qkv"])
            tg.tg_keybias_attn(b["qkv"], w.Hq, w.Hkv, w.dh, ls, L0["gain"], L0["temperature"],
                               out=b["out"])

    positions_all = torch.arange(w.N, dtype=torch.int32, device=dev)

    def full(b):
        if qwen3:
            tg.tg_gather_rows(X, None, out=b["x"])  # widen the residual to fp32
            tg.qwen3_pruned_stack(b["x"], positions_all, layers, w.Hq, w.Hkv, w.dh, None,
                                  bufs={"xn": b["xn"], "qkv": b["qkv"]})
        elif stack:
            tg.tg_gather_rows(X, None, out=b["x"])  # widen the residual to fp32
            tg.pruned_stack(b["x"], layers, w.Hq, w.Hkv, w.dh, None,
                            bufs={"xn": b["xn"], "qkv": b["qkv"]})
        else:
            L0 = layers[0]
            tg.tg_qkv_proj(X, L0["Wqkv"], w.Hq, w.Hkv, w.dh, out=b["qkv"])
            tg.tg_keybias_attn(b["qkv"], w.Hq, w.Hkv, w.dh, None, None, L0["temperature"],
                               out=b["out"])

    def measure(fn, make_bufs, steps, warmup):
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        b = make_bufs()
        for _ in range(warmup):
            fn(b)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            e0.record()
            fn(b)
            e1.record()
        torch.cuda.synchronize()
        if tg.tg_get_device_status(raise_on_error=False) != 0:
            raise RuntimeError("device status set")
        ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
        peak = torch.cuda.max_memory_allocated(dev) - base
        del b
        return ms, peak

    weights = sum(t.numel() * t.element_size() for t in [X, W1, b1, w2] +
                  [v for L in layers for v in L.values() if isinstance(v, torch.Tensor)])
    steps, warmup = max(1, args.steps), max(3, args.warmup)
    g_ms, g_peak = measure(gated, gated_bufs, steps, warmup)
    f_ms, f_peak = measure(full, full_bufs, max(1, min(steps, 5)), 1)
    attn_flops_full = 2.0 * w.N * w.N * w.dh * w.Hq * w.layers
    line = {
        "metric": (f"{w.layers}-layer Qwen3 decoder prefill tokens/s, gated vs full" if qwen3 else
                   "20-layer pruned-stack prefill tokens/s, gated vs full" if stack else
                   "one-layer prefill tokens/s, gated vs full-context attention"),
        "decoder": ("full Qwen3 layers: RMSNorm, QKV + q/k RMSNorm + rotary embedding at the "
                    "prompt positions, token-gated attention, o-projection, RMSNorm, SwiGLU MLP "
                    "(width 6144)" if qwen3 else "x <- x + attn(qkv(RMSNorm(x)))"),
        "value": w.N / (g_ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": g_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "mode": "compare",
        "config": {"workload": w.name, "N": w.N, "doc": [w.doc_begin, w.doc_end], "K": K, "M": M,
                   "layers": w.layers, "l2": "not flushed (inputs larger than L2)"},
        "gated": {"ms": g_ms, "tokens_per_s": w.N / (g_ms * 1e-3),
                  "peak_mem_bytes": int(g_peak + weights)},
        "full": {"ms": f_ms, "tokens_per_s": w.N / (f_ms * 1e-3),
                 "peak_mem_bytes": int(f_peak + weights),
                 "attn_tflops_incl_other_calls": attn_flops_full / (f_ms * 1e-3) / 1e12},
        "speedup": f_ms / g_ms,
        "mem_ratio": (f_peak + weights) / (g_peak + weights),
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------- the gradient path to the scorer
BWD_KERNELS = ("attn_bwd_delta", "keybias_bias_grad", "bias_grad_reduce")


def backward_work(w: TI.Workload, M: int) -> dict:
    """Algorithmic bytes / flops of the three backward calls at M kept rows."""
    Hq, dh, e = w.Hq, w.dh, 2
    return {
        "attn_bwd_delta": {"bytes": 2 * M * Hq * dh * e + Hq * M * 4, "flops": 0,
                           "bound": "hbm"},
        # S^T = K Q^T and dP^T = V dO^T over the causal half: 2 x 2 dh flops
        # per (query, key) pair with key <= query, per q head
        "keybias_bias_grad": {"bytes": M * w.qkv_cols * e + M * Hq * dh * e + 3 * Hq * M * 4
                              + M * 4, "flops": 2 * M * M * dh * Hq, "bound": "tensor"},
        "bias_grad_reduce": {"bytes": Hq * M * 4 + 3 * M * 4 + 2 * Hq * 4, "flops": 0,
                             "bound": "hbm"},
    }


def run_backward(args, w, K, rank, world, local_rank):
    """The gradient path from the attention output back to the scorer at the
    workload's kept-row count M: D = dO . O, dL/db on the tensor cores, and
    the reduction to dL/dlogsig, dL/dgain and dL/dscore.  Inputs are seeded
    q|k|v, logsig, gain and an upstream gradient dO of the workload's shapes;
    the forward (which writes O and lse) runs once, untimed.  Each timed step
    is the three C-ABI calls with an event before and after each, and the L2
    flushed between steps."""
    import torch

    import learned_token_pruning_residual_b300 as tg

    if rank != 0:
        return 0
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    L = tg.lib()
    M = w.M(K)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    qkv = to_dev(TI.random_qkv(M, w.Hq, w.Hkv, w.dh, seed=w.seed))
    ls = to_dev(TI.random_logsig(M, seed=w.seed))
    ap = TI.attn_params(w)
    gain, t = to_dev(ap["gain"]), ap["temperature"]
    dO = to_dev(TI.random_dout(M, w.Hq, w.dh, seed=w.seed))
    out, lse = tg.tg_keybias_attn_lse(qkv, w.Hq, w.Hkv, w.dh, ls, gain, t)
    f32 = torch.float32
    delta = torch.empty(w.Hq, M, dtype=f32, device=dev)
    dbias = torch.empty(w.Hq, M, dtype=f32, device=dev)
    dls = torch.empty(M, dtype=f32, device=dev)
    dgain = torch.empty(w.Hq, dtype=f32, device=dev)
    dscore = torch.empty(M, dtype=f32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=f32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    P = {k: v.data_ptr() for k, v in dict(qkv=qkv, ls=ls, gain=gain, dO=dO, out=out, lse=lse,
                                         delta=delta, dbias=dbias, dls=dls, dgain=dgain,
                                         dscore=dscore).items()}

    def check(st):
        if st != 0:
            raise tg.TokenGateError(st, L.tg_last_error_message().decode())

    calls = [
        lambda: check(L.tg_attn_bwd_delta(P["dO"], P["out"], 1, M, w.Hq, w.dh, P["delta"], sh)),
        lambda: check(L.tg_keybias_attn_bias_grad(P["qkv"], P["dO"], 1, M, w.Hq, w.Hkv, w.dh,
                                                  P["ls"], P["gain"], t, P["lse"], P["delta"],
                                                  P["dbias"], sh)),
        lambda: check(L.tg_bias_grad_reduce(P["dbias"], M, w.Hq, P["ls"], P["gain"], P["dls"],
                                            P["dgain"], P["dscore"], sh)),
    ]
    steps, warmup = max(1, args.steps), max(3, args.warmup)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
           for _ in range(steps)]
    for _ in range(warmup):
        flush.zero_()
        for c in calls:
            c()
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    sampler.active = True
    torch.cuda._sleep(50_000_000)
    for k in range(steps):
        flush.zero_()
        evs[k][0].record(stream)
        for i, c in enumerate(calls):
            c()
            evs[k][i + 1].record(stream)
    torch.cuda.synchronize()
    sampler.active = False
    clocks = sampler.stop()
    if tg.tg_get_device_status(raise_on_error=False) != 0:
        raise RuntimeError("device status set during the backward")
    per = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(len(calls))] for e in evs])
    step_ms = float(np.mean([e[0].elapsed_time(e[-1]) for e in evs]))
    work = backward_work(w, M)
    peaks, peak_src = load_peaks()
    kernels = {}
    for i, name in enumerate(BWD_KERNELS):
        ms = float(per[:, i].mean())
        wk = work[name]
        kernels[name] = {"ms": ms, "GB/s": wk["bytes"] / ms / 1e6,
                         "TFLOP/s": wk["flops"] / ms / 1e9 if wk["flops"] else None}
    wk, ms = work["keybias_bias_grad"], kernels["keybias_bias_grad"]["ms"]
    ach = wk["flops"] / ms / 1e9
    traffic = ncu_traffic(w.name, "keybias_bias_grad")
    tpeak, tpeak_kind = tensor_peak(peaks, clocks)
    line = {
        "metric": "token-gated attention backward to the scorer: prompt tokens/s",
        "value": w.N / (step_ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "mode": "backward",
        "config": {"workload": w.name, "N": w.N, "K": K, "M": M, "heads_q": w.Hq,
                   "heads_kv": w.Hkv, "head_dim": w.dh,
                   "l2": "flushed between steps (256 MiB write), outside the timed events",
                   "launch": "direct C-ABI calls, an event before and after each"},
        "roofline": {"kernel": "keybias_bias_grad", "bound": "tensor", "achieved": ach,
                     "peak": tpeak, "unit": "TFLOP/s",
                     "frac": ach / tpeak, "traffic": traffic,
                     "algorithmic": wk["flops"], "peak_source": f"{peak_src} ({tpeak_kind})"},
        "kernels": kernels,
        "gpu_launches": len(calls) * steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0



DN_CHUNK = 64  # tokens per chunk of the chunked delta rule


def deltanet_flops(T: int, H: int, dk: int, dv: int) -> dict:
    """Products of the chunked form per chunk of C tokens and head: K K^T and
    Q K^T (2 C^2 dk each), W = T diag(g) K (2 C^2 dk), U^T = V^T T^T (2 C^2 dv),
    S W^T, S (diag(g) Q)^T and the update U^T K' (2 C dk dv each), and
    U^T P^T (2 C^2 dv); plus, for reference, the recurrence's own count
    (S k, the rank-one update and S q: 6 dk dv per token and head)."""
    C = DN_CHUNK
    chunks = -(-T // C)
    per = 6 * C * C * dk + 4 * C * C * dv + 6 * C * dk * dv
    return {"chunked": chunks * H * per, "recurrence": 6 * T * H * dk * dv}


def run_deltanet(args, w, K, rank, world, local_rank):
    """The gated delta rule (the recurrence of a hybrid model's Gated-DeltaNet
    layers) over the M kept tokens of the workload's prompt, against the same
    recurrence over all N tokens (full prefill of that layer).  Inputs are
    seeded q, k, v of the DeltaNet head shape (bf16) and fp32 decay and write
    strength; the kept tokens are a seeded sorted subset of M positions.  Each
    timed step is one C-ABI call (two kernels), the L2 flushed between steps
    outside the events."""
    import torch

    import learned_token_pruning_residual_b300 as tg

    if rank != 0:
        return 0
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    L = tg.lib()
    M, N = w.M(K), w.N
    H, dk, dv = TI.DELTANET_SHAPE["H"], TI.DELTANET_SHAPE["dk"], TI.DELTANET_SHAPE["dv"]
    x = TI.deltanet_inputs(N, H, dk, dv, seed=w.seed, dtype="bf16")
    idx = np.sort(np.random.default_rng(w.seed).choice(N, M, replace=False))

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    def bufs(rows):
        b = {n: to_dev(x[n] if rows is None else x[n][rows]) for n in ("q", "k", "v", "alpha",
                                                                      "beta")}
        T = b["q"].shape[0]
        b["o"] = torch.empty(T, H, dv, dtype=torch.bfloat16, device=dev)
        nb = int(L.tg_gated_delta_rule_workspace_bytes(T, H))
        b["ws"] = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
        b["T"] = T
        return b

    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    steps, warmup = max(1, args.steps), max(3, args.warmup)

    def call(b):
        st = L.tg_gated_delta_rule(b["q"].data_ptr(), b["k"].data_ptr(), b["v"].data_ptr(), 1,
                                   b["alpha"].data_ptr(), b["beta"].data_ptr(), b["T"], H, dk,
                                   dv, None, b["o"].data_ptr(), None, b["ws"].data_ptr(),
                                   b["ws"].numel(), sh)
        if st != 0:
            raise tg.TokenGateError(st, L.tg_last_error_message().decode())

    def measure(b, n_steps, sampler=None):
        for _ in range(warmup):
            flush.zero_()
            call(b)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_steps)]
        if sampler:
            sampler.active = True
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            call(b)
            e1.record(stream)
        torch.cuda.synchronize()
        if sampler:
            sampler.active = False
        return float(np.mean([a.elapsed_time(c) for a, c in evs]))

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    kept, full = bufs(idx), bufs(None)
    sampler = ClockSampler(uuid)
    sampler.start()
    ms_kept = measure(kept, steps, sampler)
    clocks = sampler.stop()
    ms_full = measure(full, max(1, min(steps, 20)))
    if tg.tg_get_device_status(raise_on_error=False) != 0:
        raise RuntimeError("device status set during the delta rule")
    peaks, peak_src = load_peaks()
    tpeak, tpeak_kind = tensor_peak(peaks, clocks)
    fl = deltanet_flops(M, H, dk, dv)
    ach = fl["chunked"] / ms_kept / 1e9
    line = {
        "metric": "Gated-DeltaNet layer over the kept tokens: prompt tokens/s",
        "value": N / (ms_kept * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_kept, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "mode": "deltanet",
        "config": {"workload": f"gated delta rule, {H} heads of dk = dv = {dk}, over the kept "
                               f"tokens of {w.name}", "N": N, "K": K, "M": M, "heads": H,
                   "dk": dk, "dv": dv, "inputs": "q, k, v bf16; alpha, beta fp32",
                   "l2": "flushed between steps (256 MiB write), outside the timed events",
                   "launch": "direct C-ABI call (chunk preparation + state scan)"},
        "full": {"ms": ms_full, "tokens_per_s": N / (ms_full * 1e-3), "T": N},
        "speedup": ms_full / ms_kept,
        "roofline": {"kernel": "gated_delta_rule (both kernels)", "bound": "tensor",
                     "achieved": ach, "peak": tpeak, "unit": "TFLOP/s",
                     "frac": ach / tpeak,
                     "traffic": ncu_traffic(w.name, "gated_delta_rule"),
                     "algorithmic": fl["chunked"], "recurrence_flops": fl["recurrence"],
                     "peak_source": f"{peak_src} ({tpeak_kind})",
                     "note": "the state scan is sequential over chunks, one CTA per head: "
                             f"{H} of the SMs"},
        "gpu_launches": 2 * steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=None, choices=sorted(TI.WORKLOADS),
                    help=f"default {DEFAULT_WORKLOAD}; {DELTANET_WORKLOAD} for --mode deltanet")
    ap.add_argument("--budget", type=int, default=None,
                    help="index into the workload's budgets (default 0; 1, i.e. 10%%, for "
                         "--mode deltanet)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the five calls directly instead of replaying one CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clock-soak", action="store_true",
                    help="skip the one-second replay that samples clocks under load")
    ap.add_argument("--decoder", default="attention", choices=["attention", "qwen3"],
                    help="--mode compare: layers of the stack, attention only (the workload's "
                         "definition) or full Qwen3 decoder layers")
    ap.add_argument("--mode", default="step", choices=["step", "compare", "backward", "deltanet"],
                    help="step: the timed gated-prefill step (default); compare: gated path vs "
                         "full prefill on the same kernels, with peak device memory; backward: "
                         "the gradient path from the attention bias to the scorer; deltanet: the "
                         "gated delta rule over the kept tokens vs over the whole prompt")
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    dn = args.mode == "deltanet"
    if args.workload is None:
        args.workload = DELTANET_WORKLOAD if dn else DEFAULT_WORKLOAD
    if args.budget is None:
        args.budget = 1 if dn and args.workload == DELTANET_WORKLOAD else 0
    w = TI.WORKLOADS[args.workload]
    K = w.Ks()[args.budget]
    if args.impl == "reference":
        return run_reference(args, w, K, rank, world)
    if args.mode == "compare":
        return run_compare(args, w, K, rank, world, local_rank)
    if args.mode == "backward":
        return run_backward(args, w, K, rank, world, local_rank)
    if args.mode == "deltanet":
        return run_deltanet(args, w, K, rank, world, local_rank)
    return run_gpu(args, w, K, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
