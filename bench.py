"""Benchmark: KDA chunk_fwd tokens/s on one GB300, with roofline fraction.

One step = one kda_chunk_fwd over the whole packed batch of the chosen workload
(default ``prefill_4k``: 4 sequences x 4096 tokens, H=32, dk=dv=128, bf16,
fp32 initial and final states), inputs resident in HBM.  ``value`` counts
sequence tokens (heads not multiplied in) per second over all ranks.

Multi-GPU: (sequence, head) chains are independent, so each rank runs its own
copy of the batch (weak scaling, no collective on the data path); the timed
region is bracketed by barriers and the max over ranks is taken.

``--prep`` runs the same workload on raw inputs (un-normalised q / k, raw gate and
beta logits) through kda_chunk_fwd_prep with every preprocessing flag, so the
normalisation, sigmoid gate and sigmoid beta are fused into the kernels.

``--impl reference`` times the fp64 CPU oracle (the correctness reference, a
deliberately slow program) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "KDA chunk_fwd tokens/s at T=4K-128K (1 GB300) and % of roofline"
UNIT = "tokens/s"

# DRAM bytes (read + write) of one launch of the chunked kernel on prefill_4k, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum), with the first 16 hex digits of the
# sha256 of the kernel's source file at the time of the capture: the figure is reported only
# while that file is unchanged, and as null otherwise (until it is captured again).
DOMINANT_TRAFFIC = {"prefill_4k": (664636416, "12719058f1916c60")}
DOMINANT_SRC = os.path.join(ROOT, "gated_linear_attention_chunk_gb300", "csrc", "kda_chunk_tc.cu")


def source_sha16(path: str) -> str:
    import hashlib
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def dominant_traffic(workload: str):
    entry = DOMINANT_TRAFFIC.get(workload)
    if not entry:
        return None
    nbytes, sha = entry
    return nbytes if source_sha16(DOMINANT_SRC) == sha else None


# every preprocessing flag (KDA_PREP_L2NORM_Q | _L2NORM_K | _SIGMOID_GATE | _SIGMOID_BETA)
PREP_ALL, PREP_EPS = 15, 1e-6


# ------------------------------------------------------------------------------------------------
# algorithmic work (per step)
# ------------------------------------------------------------------------------------------------

def algorithmic_bytes(case) -> int:
    """Bytes a perfect kernel moves: every input once, o once, states in and out once."""
    T, H, dk, dv = case.T_total, case.H, case.dk, case.dv
    es = case.q.element_size()
    b = T * H * (3 * dk + dv) * es          # q, k, g, v
    b += T * H * es                         # beta
    b += T * H * dv * es                    # o
    b += case.N * H * dk * dv * 4           # final state
    if case.init_state is not None:
        b += case.N * H * dk * dv * 4       # initial state
    b += (case.N + 1) * 4                   # cu_seqlens
    return int(b)


def algorithmic_flops(case, C: int = 64) -> int:
    """6 d^2 + 5 C d flop per token-head for dk = dv = d (triangular halves counted once)."""
    d = case.dk
    return int(case.T_total * case.H * (6 * d * d + 5 * C * d))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------------------------
# distributed helpers (host logic; covered by gloo tests)
# ------------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(max_elapsed_ms: float, world: int, tokens_per_rank_step: int, steps: int):
    """Whole-job throughput: every rank's tokens over the slowest rank's time.
    Returns (tokens/s, ms per step)."""
    return world * tokens_per_rank_step * steps / (max_elapsed_ms / 1e3), max_elapsed_ms / steps


def max_over_ranks(value: float, device=None) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------

class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, power, clock-event reasons)."""
    SW_POWER_CAP, HW_SLOWDOWN, SW_THERMAL, HW_THERMAL = 0x4, 0x8, 0x20, 0x40

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        props = torch.cuda.get_device_properties(device_index)
        self.handle = ctypes.c_void_p()
        ok = False
        for fmt in ("{:08X}:{:02X}:{:02X}.0", "{:04X}:{:02X}:{:02X}.0"):
            bus = fmt.format(props.pci_domain_id, props.pci_bus_id, props.pci_device_id).encode()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.handle)) == 0:
                ok = True
                break
        if not ok:
            raise RuntimeError("no NVML handle for this device")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        m = ctypes.c_uint()
        self.sm_max = float(m.value) if lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(m)) == 0 else None

    def sample(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(clk)) != 0:  # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(pw))
        self.reasons_fn(self.handle, ct.byref(rs))
        names = []
        for bit, name in ((self.HW_SLOWDOWN, "hw_slowdown"), (self.HW_THERMAL, "hw_thermal_slowdown"),
                          (self.SW_THERMAL, "sw_thermal_slowdown"), (self.SW_POWER_CAP, "sw_power_cap")):
            if rs.value & bit:
                names.append(name)
        return float(clk.value), self.sm_max, pw.value / 1e3, names


class ClockSampler:
    """SM clocks, power and clock-event reasons sampled while the GPU works: NVML (read-only
    queries, through ctypes) about every millisecond, so that even a few-millisecond timed region
    holds samples; nvidia-smi every 100 ms where NVML cannot be loaded.  ``summary(t0, t1)``
    keeps the samples taken between two wall-clock times."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int = 0, period_s: float = 0.001):
        self.samples = []  # (time, sm_mhz, sm_max_mhz, power_w, reasons)
        self.proc = None
        self.source = None
        self._stop = threading.Event()
        try:
            nv = _Nvml(device_index)
            self.source = "nvml"

            def loop():
                while not self._stop.is_set():
                    r = nv.sample()
                    if r is not None:
                        self.samples.append((time.time(), *r))
                    time.sleep(period_s)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
        except Exception:
            self._start_smi(device_index)

    def _start_smi(self, device_index):
        sel = []
        try:
            p = torch.cuda.get_device_properties(device_index)
            sel = ["-i", "{:08X}:{:02X}:{:02X}.0".format(p.pci_domain_id, p.pci_bus_id, p.pci_device_id)]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
                pw = float(parts[2]) if parts[2] not in ("", "[N/A]") else None
            except ValueError:
                continue
            rs = [n for n, v in zip(names, parts[4:8]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, smax, pw, rs))

    def wait_first(self, timeout_s: float = 3.0):
        t = time.time()
        while not self.samples and time.time() - t < timeout_s:
            time.sleep(0.005)

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [r for r in list(self.samples) if t0 <= r[0] <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        sm = sorted(r[1] for r in rows)
        reasons = sorted({n for r in rows for n in r[4]})
        pw = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": sm[len(sm) // 2], "sm_mhz_min": sm[0], "sm_max_mhz": rows[-1][2], "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None, "source": self.source,
                "region_s": t1 - t0}


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (bounded sample)
# ------------------------------------------------------------------------------------------------

def oracle_sample_rate(case, budget_s: float = 10.0, prep: int = 0):
    """Oracle tokens/s on a bounded sample of the workload, sized to about ``budget_s`` of
    CPU work: whole sequences (all heads), repeated, when one sequence takes less than
    the budget; otherwise a prefix of sequence 0 (all heads)."""
    import oracle
    threads = max(1, min(os.cpu_count() or 1, case.N * case.H))
    cu = case.cu_seqlens.tolist()

    def run_prefix(L):
        sl = slice(0, L)
        t = time.perf_counter()
        oracle.forward(case.q[sl], case.k[sl], case.v[sl], case.g[sl], case.beta[sl],
                       torch.tensor([0, L], dtype=torch.int64),
                       None if case.init_state is None else case.init_state[:1],
                       scale=case.scale, threads=threads, prep_flags=prep, prep_eps=PREP_EPS)
        return time.perf_counter() - t

    def run_seqs(m):
        T = cu[m]
        t = time.perf_counter()
        oracle.forward(case.q[:T], case.k[:T], case.v[:T], case.g[:T], case.beta[:T],
                       torch.tensor(cu[:m + 1], dtype=torch.int64),
                       None if case.init_state is None else case.init_state[:m],
                       scale=case.scale, threads=threads, prep_flags=prep, prep_eps=PREP_EPS)
        return time.perf_counter() - t

    L0 = min(case.lengths[0], 16)
    t0 = run_prefix(L0)
    per_token = t0 / max(L0, 1)
    if per_token * case.lengths[0] > budget_s:
        L = int(max(L0, min(case.lengths[0], budget_s / max(per_token, 1e-9))))
        t = run_prefix(L) if L > L0 else t0
        return {"value": L / t, "unit": UNIT, "cores": threads, "kind": "oracle", "seconds": t,
                "sample": f"first {L} tokens of sequence 0, all {case.H} heads (fp64, {threads} threads), {t:.1f} s"}
    # whole sequences: as many as fit the budget, then repeats of that batch
    m = 1
    while m < case.N and per_token * cu[m + 1] <= budget_s:
        m += 1
    tokens, total, reps = 0, 0.0, 0
    while total < budget_s and reps < 50:
        total += run_seqs(m)
        tokens += cu[m]
        reps += 1
    return {"value": tokens / total, "unit": UNIT, "cores": threads, "kind": "oracle", "seconds": total,
            "sample": f"{reps} x the first {m} sequences ({cu[m]} tokens), all {case.H} heads (fp64, {threads} "
                      f"threads), {total:.1f} s"}


# ------------------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    case = workloads.named_case(args.workload, raw=args.prep)
    prep = PREP_ALL if args.prep else 0
    # the whole run (warm-up + timed samples) stays within about three minutes
    budget = min(args.ref_budget, 150.0 / (args.steps + args.warmup))
    per_step = []
    for _ in range(args.warmup):
        oracle_sample_rate(case, budget_s=budget, prep=prep)
    for _ in range(args.steps):
        per_step.append(oracle_sample_rate(case, budget_s=budget, prep=prep))
    vals = [r["value"] for r in per_step]
    v = sum(vals) / len(vals)
    cb = dict(per_step[-1])
    cb["value"] = v
    cb["sample"] = f"{args.steps} timed samples; last: " + cb["sample"]
    ms = 1e3 * sum(r["seconds"] for r in per_step) / len(per_step)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(args, case), "cpu_baseline": cb,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(args, case):
    return {"workload": args.workload, "desc": workloads.NAMED_WORKLOADS[args.workload]["desc"],
            "global_batch": case.N * max(1, args.gpus), "seq_len": max(case.lengths) if case.lengths else 0,
            "tokens_per_step_per_gpu": case.T_total, "heads": case.H, "dk": case.dk, "dv": case.dv,
            "parallelism": f"dp{max(1, args.gpus)} (independent replicas)",
            "l2": "inputs larger than L2 (no flush needed)" if algorithmic_bytes(case) > 256e6
                  else "L2 flushed between steps",
            "workspace": "minimum (no T-segment split)" if getattr(args, "plain_workspace", False) else "full",
            "inputs": ("raw: L2 norm of q / k rows (eps 1e-6), sigmoid gate, sigmoid beta fused"
                       " (kda_chunk_fwd_prep)") if getattr(args, "prep", False) else "preprocessed"}


def measure_state_kernels(kda, dev, hbm_peak, n_seq=128, H=32, d=128, reps=50):
    """Achieved HBM bandwidth of kda_decode_step and kda_replay on a pool of n_seq x H
    128x128 fp32 states (256 MiB, larger than L2): the state read + write per call is the
    algorithmic traffic; replay applies 4 accepted tokens per sequence."""
    pool = torch.randn(n_seq, H, d, d, device=dev) * 0.02
    q, k, v, g, b = (x.to(dev) for x in workloads.make_decode_tokens(4 * n_seq, H, d, d, torch.bfloat16, seed=77))
    ws = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, dev)
    o = torch.empty(n_seq, H, d, dtype=torch.bfloat16, device=dev)
    cu = torch.arange(0, 4 * n_seq + 1, 4, dtype=torch.int32, device=dev)
    state_bytes = 2 * pool.numel() * 4
    out = {}
    # the same with the short convolution fused (raw projections, every preprocessing flag)
    cw = torch.randn(H, 3 * d, kda.KDA_CONV_WIDTH, device=dev) * 0.5
    cpool = torch.zeros(n_seq, kda.KDA_CONV_WIDTH - 1, H, 3 * d, device=dev)
    for name in ("decode", "replay", "replay_prep", "decode_conv", "replay_conv"):
        def call():
            if name == "decode":
                kda.kda_decode_step(q[:n_seq], k[:n_seq], v[:n_seq], g[:n_seq], b[:n_seq], pool, o=o, workspace=ws)
            elif name == "replay":
                kda.kda_replay(pool, k, v, g, b, cu, workspace=ws)
            elif name == "replay_prep":  # every preprocessing flag, no convolution
                kda.kda_replay_prep(pool, k, v, g, b, cu, prep=15, workspace=ws)
            elif name == "decode_conv":
                kda.kda_decode_step_conv(q[:n_seq], k[:n_seq], v[:n_seq], g[:n_seq], b[:n_seq], pool, cw, cpool,
                                         prep=15, o=o, workspace=ws)
            else:
                kda.kda_replay_conv(pool, q, k, v, g, b, cu, cw, cpool, prep=15, workspace=ws)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            call()
        e1.record(st)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        ntok = n_seq if name.startswith("decode") else 4 * n_seq
        tok_bytes = ntok * H * (4 * d * 2 + 2) + (ntok * H * d * 2 if name == "replay_conv" else 0)  # + q
        conv_bytes = 2 * cpool.numel() * 4 if name.endswith("conv") else 0
        gbs = (state_bytes + conv_bytes + tok_bytes) / (ms / 1e3) / 1e9
        out[name] = {"ms_per_call": ms, "achieved_GBs": gbs, "frac_of_hbm": gbs / hbm_peak,
                     "states": n_seq * H, "tokens_per_seq": 1 if name.startswith("decode") else 4}
    # state-pool operations on the same pool: fork half the slots onto the other half
    # (read + write of 64 states x H heads), offload them to pinned host memory (write)
    half = n_seq // 2
    src = torch.arange(0, half, dtype=torch.int32, device=dev)
    dst = torch.arange(half, 2 * half, dtype=torch.int32, device=dev)
    host = torch.empty(half, H, d, d, dtype=torch.float32).pin_memory()
    slot_bytes = H * d * d * 4
    for name, call, nbytes in (("fork", lambda: kda.kda_state_fork(pool, src, dst, workspace=ws), 2 * half * slot_bytes),
                               ("offload", lambda: kda.kda_state_offload(pool, src, host, workspace=ws),
                                half * slot_bytes)):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            call()
        e1.record(st)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms_per_call": ms, "achieved_GBs": gbs, "states": half * H,
                     "frac_of_hbm": gbs / hbm_peak if name == "fork" else None,
                     "bytes": "HBM read + write" if name == "fork" else "bytes written to pinned host memory"}
    if kda.kda_device_status(ws) != kda.KDA_OK:
        raise RuntimeError("decode/replay/pool device status")
    return out


def measure_conv(kda, case, dev, hbm_peak, reps=20):
    """kda_conv_fwd (short convolution + SiLU of q, k, v) on the same workload: q, k, v
    read and written once, plus the convolution states read and written."""
    q, k, v = (x.to(dev) for x in (case.q, case.k, case.v))
    cu = case.cu_seqlens.to(dev)
    H, dk, dv = case.H, case.dk, case.dv
    w = torch.randn(H, 2 * dk + dv, kda.KDA_CONV_WIDTH, device=dev) * 0.5
    st = torch.zeros(case.N, kda.KDA_CONV_WIDTH - 1, H, 2 * dk + dv, device=dev)
    ws = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, dev)
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))

    def call():
        lib = kda.load_library()
        rc = lib.kda_conv_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), 0 if q.dtype == torch.bfloat16 else 1,
                              w.data_ptr(), kda.KDA_CONV_WIDTH, st.data_ptr(), cu.data_ptr(), case.N, case.T_total,
                              H, dk, dv, outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), st.data_ptr(),
                              ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
        if rc != 0:
            raise RuntimeError(f"kda_conv_fwd: {kda.kda_status_string(rc)}")

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    st_ = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st_)
    for _ in range(reps):
        call()
    e1.record(st_)
    torch.cuda.synchronize()
    if kda.kda_device_status(ws) != kda.KDA_OK:
        raise RuntimeError("conv device status")
    ms = e0.elapsed_time(e1) / reps
    nbytes = 2 * case.T_total * H * (2 * dk + dv) * q.element_size() + 2 * st.numel() * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"ms_per_call": ms, "achieved_GBs": gbs, "frac_of_hbm": gbs / hbm_peak, "algorithmic_bytes": nbytes,
            "launches_per_call": 2}


def measure_backward(kda, case, dev, hbm_peak, reps=3):
    """kda_chunk_bwd on the same workload: d_o ~ N(0, 1), no final-state gradient.
    Algorithmic bytes per token-head: q, k, v, g, d_o and beta read, dq, dk, dv, dg and
    dbeta written (10 d + 2 values of the input dtype), plus the initial state read and
    its gradient written per (sequence, head)."""
    q, k, v, g, b = (x.to(dev) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = case.cu_seqlens.to(dev)
    s0 = None if case.init_state is None else case.init_state.to(dev)
    d_o = torch.randn(case.T_total, case.H, case.dv, generator=torch.Generator().manual_seed(9)).to(q.dtype).to(dev)
    ws = kda.new_workspace(kda.kda_chunk_bwd_workspace_size(case.N, case.T_total, case.H, case.dk, case.dv), dev)

    def call():
        kda.kda_chunk_bwd(q, k, v, g, b, d_o, cu_seqlens=cu, init_state=s0, scale=case.scale, workspace=ws)

    call()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        call()
    e1.record(st)
    torch.cuda.synchronize()
    if kda.kda_device_status(ws) != kda.KDA_OK:
        raise RuntimeError("backward device status")
    ms = e0.elapsed_time(e1) / reps
    es = q.element_size()
    nbytes = case.T_total * case.H * (10 * case.dk + 2) * es + 2 * case.N * case.H * case.dk * case.dv * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"ms_per_call": ms, "tokens_per_s": case.T_total / (ms / 1e3), "achieved_GBs": gbs,
            "frac_of_hbm": gbs / hbm_peak, "algorithmic_bytes": nbytes, "calls": reps,
            "launches_per_call": 4}


def _median_ms(call, reps: int, warm: int = 3) -> float:
    """Median per-call CUDA-event time of ``call`` on the current stream."""
    for _ in range(warm):
        call()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(st)
        call()
        b.record(st)
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    return ms[len(ms) // 2]


def host_link_peak(dev, nbytes=512 << 20, reps=5):
    """GB/s of one large pinned host -> device copy, of one device -> host copy, and of both
    at once on two streams (total bytes over the time both take; best of ``reps``, CUDA
    events): the link bounds the end-to-end pipeline is measured against."""
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    devb = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    host2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    devb2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", devb, host), ("d2h", host, devb)):
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        out[name] = nbytes / (best / 1e3) / 1e9
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    cur = torch.cuda.current_stream(dev)
    best = None
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for s_ in (s_in, s_out):
            s_.wait_stream(cur)
        with torch.cuda.stream(s_in):
            devb.copy_(host, non_blocking=True)
        with torch.cuda.stream(s_out):
            host2.copy_(devb2, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)
        b.record(cur)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    out["both"] = 2 * nbytes / (best / 1e3) / 1e9
    del host, devb, host2, devb2
    torch.cuda.empty_cache()
    return out


def measure_workload(kda, name, dev, hbm_peak, tf_peak, reps=10):
    """kda_chunk_fwd tokens/s and roofline fraction on another named prefill workload (inputs
    drawn on the device with the same recipe; full workspace, so every path of the call is
    enabled: the T-segment split for few long chains, the longest-first launch order for
    more chains than one wave)."""
    case = workloads.named_case(name, device=dev)
    N, T, H, dk, dv = case.N, case.T_total, case.H, case.dk, case.dv
    o = torch.empty(T, H, dv, dtype=case.q.dtype, device=dev)
    fs = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(N, T, H, dk, dv), dev)

    def call():
        kda.kda_chunk_fwd(case.q, case.k, case.v, case.g, case.beta, cu_seqlens=case.cu_seqlens,
                          init_state=case.init_state, scale=case.scale, o=o, final_state=fs, workspace=ws)

    ms = _median_ms(call, reps)
    if kda.kda_device_status(ws) != kda.KDA_OK:
        raise RuntimeError(f"{name}: device status")
    nbytes, flops = algorithmic_bytes(case), algorithmic_flops(case)
    roof_ms = 1e3 * max(nbytes / (hbm_peak * 1e9), flops / (tf_peak * 1e12))
    gbs = nbytes / (ms / 1e3) / 1e9
    out = {"tokens_per_s": T / (ms / 1e3), "ms_per_call": ms, "tokens": T, "sequences": N, "heads": H,
           "achieved_GBs": gbs, "frac_of_hbm": gbs / hbm_peak, "roofline_ms": roof_ms, "frac": roof_ms / ms,
           "algorithmic_bytes": nbytes, "calls": reps,
           "inputs": "drawn on the device (same recipe, CUDA generator)", "desc": workloads.NAMED_WORKLOADS[name]["desc"]}
    del case, o, fs, ws
    torch.cuda.empty_cache()
    return out


def measure_spec_rollout(kda, dev, hbm_peak, steps=64, loops=3):
    """The speculative rollout loop: a 2048-token prefill of 128 sequences into a state pool,
    then ``steps`` x (4-token verify kda_chunk_fwd from the committed states, no final state
    + kda_replay of the accepted prefix, U{1..4} tokens per sequence).  Every step's tokens,
    accept lengths and packed accepted tokens are prepared before the timed loop (inputs
    resident in HBM); the pool is reset to the prefill's states before each timed loop."""
    case = workloads.named_case("spec_rollout", device=dev)
    N, T, H, dk, dv = case.N, case.T_total, case.H, case.dk, case.dv
    pool = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    o_p = torch.empty(T, H, dv, dtype=case.q.dtype, device=dev)
    ws_p = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(N, T, H, dk, dv), dev)

    def prefill():
        kda.kda_chunk_fwd(case.q, case.k, case.v, case.g, case.beta, cu_seqlens=case.cu_seqlens, init_state=None,
                          scale=case.scale, o=o_p, final_state=pool, workspace=ws_p)

    prefill_ms = _median_ms(prefill, 5)
    pool0 = pool.clone()
    del case, o_p, ws_p
    q, k, v, g, b = workloads.make_decode_tokens(4 * N * steps, H, dk, dv, torch.bfloat16, seed=4004, device=dev)
    q, k, v, g, b = (x.view(steps, 4 * N, *x.shape[1:]) for x in (q, k, v, g, b))
    acc = workloads.make_accept_lengths(steps, N, 4, seed=404)
    packed = []
    for s in range(steps):
        a = acc[s]
        sel = torch.cat([torch.arange(4 * i, 4 * i + int(a[i])) for i in range(N)]).to(dev)
        cu_a = torch.zeros(N + 1, dtype=torch.int32)
        cu_a[1:] = torch.cumsum(a, 0)
        packed.append((k[s][sel].contiguous(), v[s][sel].contiguous(), g[s][sel].contiguous(),
                       b[s][sel].contiguous(), cu_a.to(dev)))
    cu4 = torch.arange(0, 4 * N + 1, 4, dtype=torch.int32, device=dev)
    o_v = torch.empty(4 * N, H, dv, dtype=torch.bfloat16, device=dev)
    ws_v = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(N, 4 * N, H, dk, dv), dev)
    ws_r = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, dev)

    def loop():
        for s in range(steps):
            kda.kda_chunk_fwd(q[s], k[s], v[s], g[s], b[s], cu_seqlens=cu4, init_state=pool, output_final_state=False,
                              o=o_v, workspace=ws_v)
            ka, va, ga, ba, cua = packed[s]
            kda.kda_replay(pool, ka, va, ga, ba, cua, workspace=ws_r)

    pool.copy_(pool0)
    loop()
    torch.cuda.synchronize()
    if kda.kda_device_status(ws_v) != kda.KDA_OK or kda.kda_device_status(ws_r) != kda.KDA_OK:
        raise RuntimeError("spec rollout: device status")
    st = torch.cuda.current_stream()
    times = []
    for _ in range(loops):
        pool.copy_(pool0)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(st)
        loop()
        b_.record(st)
        torch.cuda.synchronize()
        times.append(a_.elapsed_time(b_))
    ms = sorted(times)[len(times) // 2]
    accepted = int(acc.sum())
    state = N * H * dk * dv * 4
    tok_v = 4 * N * H * ((3 * dk + dv + 1) * 2 + dv * 2)          # q, k, g, v, beta in; o out
    tok_r = accepted * H * (2 * dk + dv + 1) * 2                 # k, g, v, beta of accepted tokens
    nbytes = steps * (state + 2 * state) + steps * tok_v + tok_r
    roof_ms = 1e3 * nbytes / (hbm_peak * 1e9)
    out = {"accepted_tokens_per_s": accepted / (ms / 1e3), "ms_per_loop": ms, "steps": steps,
           "ms_per_step": ms / steps, "accepted_tokens": accepted, "sequences": N, "heads": H,
           "prefill_ms": prefill_ms, "prefill_tokens_per_s": T / (prefill_ms / 1e3),
           "algorithmic_bytes_per_loop": nbytes, "achieved_GBs": nbytes / (ms / 1e3) / 1e9,
           "roofline_ms_per_step": roof_ms / steps, "frac": roof_ms / ms, "loops_timed": loops,
           "launches_per_step": 4,  # verify: launch order, chunked, token-sequential; replay: token-sequential
           "inputs": "drawn on the device (same recipe, CUDA generator); accept lengths U{1..4}, seed 404"}
    del q, k, v, g, b, packed, pool, pool0, o_v, ws_v
    torch.cuda.empty_cache()
    return out


def run_gpu(args, world, rank, local):
    import gated_linear_attention_chunk_gb300 as kda

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import torch.distributed as dist
    distributed = world > 1
    if distributed:
        dist.init_process_group("nccl", device_id=dev)

    case = workloads.named_case(args.workload, raw=args.prep)
    prep = PREP_ALL if args.prep else 0
    q, k, v, g, b = (x.to(dev) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = case.cu_seqlens.to(dev)
    s0 = None if case.init_state is None else case.init_state.to(dev)
    N, T, H, dk, dv = case.N, case.T_total, case.H, case.dk, case.dv
    o = torch.empty(T, H, dv, dtype=q.dtype, device=dev)
    fs = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    # The full workspace enables every path of the call (the T-segment split for batches with
    # few chains and long sequences); --plain-workspace gives only the minimum (unsplit).
    plain_bytes = kda.KDA_WS_HEADER_BYTES
    full_bytes = kda.kda_chunk_fwd_workspace_size(N, T, H, dk, dv)
    # the T-segment split runs for few long chains (N * H <= 48, T >= 4096, dk = dv = 128)
    split = (not args.plain_workspace) and dk == 128 and dv == 128 and N * H <= 48 and T >= 4096
    ws = kda.new_workspace(plain_bytes if args.plain_workspace else full_bytes, dev)
    flush = None
    if algorithmic_bytes(case) <= 256e6:
        flush = torch.empty(int(256e6), dtype=torch.uint8, device=dev)

    def call(q, k, v, g, b, cu, s0):
        if prep:
            kda.kda_chunk_fwd_prep(q, k, v, g, b, prep, PREP_EPS, cu_seqlens=cu, init_state=s0, scale=case.scale,
                                   o=o, final_state=fs, workspace=ws)
        else:
            kda.kda_chunk_fwd(q, k, v, g, b, cu_seqlens=cu, init_state=s0, scale=case.scale, o=o,
                              final_state=fs, workspace=ws)

    def step():
        call(q, k, v, g, b, cu, s0)

    # kernels of ours per kda_chunk_fwd: the chunked tensor-core kernel (when it serves this shape)
    # plus the token-sequential partial-chunk kernel
    # (with the T-segment split, also the two merge kernels)
    # (and, for more chains than one wave of CTAs, the kernel that orders the sequences longest first)
    uses_tc = bool(kda.kda_chunk_fwd_uses_tensor_cores(dk, dv, q.dtype))
    ordered = uses_tc and not split and not args.plain_workspace and 2 <= N <= 8192 and N * H > 152
    launches_per_step = 1 + int(uses_tc) + (2 if split else 0) + int(ordered)
    clocks = ClockSampler(local)
    clocks.wait_first()
    for _ in range(args.warmup):
        step()
    st = kda.kda_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"device status {kda.kda_status_string(st)}")
    torch.cuda.synchronize()
    if distributed:
        dist.barrier()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if distributed:
        dist.barrier()
    step_ms = [a.elapsed_time(bb) for a, bb in ev]
    total_ms = sum(step_ms)
    clk = clocks.summary(wall0, wall1)
    clocks.stop()
    total_ms = max_over_ranks(total_ms, dev)
    value, ms_per_step = aggregate(total_ms, world, T, args.steps)
    st = kda.kda_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"device status {kda.kda_status_string(st)}")

    # End to end through the public API with host buffers: every step copies the inputs in from
    # pinned host memory and o and the final states out, with the copies of one sequence group
    # overlapping the other pieces' compute (HostPrefill: one kda_chunk_fwd per piece; a long
    # sequence is cut into chunk-aligned parts whose state carries in device memory).
    from gated_linear_attention_chunk_gb300.host_pipeline import HostPrefill
    pipe = HostPrefill(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                       scale=case.scale, groups=16, device=dev)
    if prep:
        pipe = None  # the pipelined helper runs the plain call; --prep reports no end-to-end number
    e2e = None
    if pipe is not None:
        e2e_steps = max(1, min(args.steps, 20))
        pipe.run()
        torch.cuda.synchronize()
        if pipe.status() != kda.KDA_OK:
            raise RuntimeError("e2e device status")
        if distributed:
            dist.barrier()
        # three timed loops, the median one reported: the host link is shared with the node's
        # other jobs, so a single loop can land in someone else's burst
        loop_ms = []
        for _ in range(3):
            a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(e2e_steps):
                pipe.run()
            bb.record(stream)
            torch.cuda.synchronize()
            loop_ms.append(a.elapsed_time(bb))
        e2e_ms = max_over_ranks(sorted(loop_ms)[1], dev)
        h2d, d2h = pipe.h2d_bytes, pipe.d2h_bytes
        e2e = {"value": world * T * e2e_steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
               "host_link_GBs": (h2d + d2h) * e2e_steps / (e2e_ms / 1e3) / 1e9,
               "host_link_peak_GBs": host_link_peak(dev),
               "pipeline": f"{len(pipe.groups)} pieces (sequence groups, long sequences cut at chunk"
                           " boundaries); H2D, compute and D2H on three streams",
               "loops_ms": loop_ms, "timing": "median of 3 timed loops"}
        # a step can be no shorter than either direction's copy alone, nor than all of its bytes
        # at the rate the two directions reach together (where they share the link)
        pk = e2e["host_link_peak_GBs"]
        e2e["link_bound_ms_per_step"] = max(h2d / pk["h2d"], d2h / pk["d2h"], (h2d + d2h) / pk["both"]) / 1e6
        del pipe
        torch.cuda.empty_cache()

    hbm_peak, tf_peak, peak_src = measured_peaks()
    nbytes = algorithmic_bytes(case)
    flops = algorithmic_flops(case)
    kern_ms = sorted(step_ms)[len(step_ms) // 2]
    t_hbm = nbytes / (hbm_peak * 1e9)
    t_tc = flops / (tf_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = None if prep else dominant_traffic(args.workload)  # captured on preprocessed inputs
    if bound == "hbm":
        achieved = nbytes / (kern_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic}
    else:
        achieved = flops / (kern_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": achieved / tf_peak, "traffic": traffic}
    roof.update({"peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else peak_src,
                 "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                 "kernel_ms_median": kern_ms, "roofline_ms": 1e3 * max(t_hbm, t_tc),
                 "timing": "median per-step CUDA-event time of kda_chunk_fwd (includes the status-word memset"
                           " and the partial-chunk launch)"})

    # the rest of the metric's 4K-128K range, 64-wide heads and the speculative rollout loop
    # (default workload only)
    workloads_sub = None
    if args.workload == "prefill_4k" and not (args.prep or args.no_sub_workloads):
        workloads_sub = {name: measure_workload(kda, name, dev, hbm_peak, tf_peak)
                         for name in ("long_128k", "varlen_64", "prefill_4k_d64", "prefill_4k_fp32")}
        workloads_sub["spec_rollout"] = measure_spec_rollout(kda, dev, hbm_peak)
    state_kernels = measure_state_kernels(kda, dev, hbm_peak) if not args.no_state_kernels else None
    backward = measure_backward(kda, case, dev, hbm_peak) if not (args.no_backward or args.prep) else None
    conv = measure_conv(kda, case, dev, hbm_peak) if not (args.no_state_kernels or args.prep) else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample_rate(case, budget_s=args.ref_budget, prep=prep)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if q.dtype == torch.bfloat16 else "f32",
                "data": "synthetic", "config": config_dict(args, case), "roofline": roof,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
                "clocks": clk, "workloads": workloads_sub, "state_kernels": state_kernels, "backward": backward,
                "conv_fwd": conv}
        print(json.dumps(line), flush=True)
    if distributed:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["libkda", "reference"], default="libkda")
    ap.add_argument("--workload", default="prefill_4k", choices=sorted(workloads.NAMED_WORKLOADS))
    ap.add_argument("--ref-budget", type=float, default=10.0, help="seconds of oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-state-kernels", action="store_true", help="skip the decode/replay bandwidth check")
    ap.add_argument("--plain-workspace", action="store_true",
                    help="minimum workspace: kda_chunk_fwd runs without the T-segment split")
    ap.add_argument("--no-backward", action="store_true", help="skip the kda_chunk_bwd measurement")
    ap.add_argument("--no-sub-workloads", action="store_true",
                    help="skip the long_128k / varlen_64 / spec_rollout sub-records")
    ap.add_argument("--state-kernels-only", action="store_true",
                    help="only the decode / replay / pool measurements (a short command for profiling them)")
    ap.add_argument("--state-reps", type=int, default=50, help="timed calls per state kernel")
    ap.add_argument("--prep", action="store_true",
                    help="raw inputs through kda_chunk_fwd_prep with every preprocessing flag")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.state_kernels_only:
        import gated_linear_attention_chunk_gb300 as kda
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        out = measure_state_kernels(kda, dev, measured_peaks()[0], reps=args.state_reps)
        print(json.dumps({"state_kernels": out}), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
