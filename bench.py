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

# DRAM bytes (read + write) of one kda_chunk_tc_kernel launch on prefill_4k, from the
# ncu capture summarised in profiles/kda_chunk_tc_prefill_4k.md (546.59 MB read +
# 118.15 MB written).  Reset to None whenever that kernel changes until it is re-captured.
DOMINANT_TRAFFIC = {"prefill_4k": 664739328}

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

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int = 0):
        self.samples = []
        self.proc = None
        sel = []
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            if bus:
                sel = ["-i", str(bus)]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for ts, s in self.samples if t0 <= ts <= t1]
        if not rows and self.samples:  # region shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            rows = [min(self.samples, key=lambda x: abs(x[0] - mid))[1]]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


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
    for name in ("decode", "replay", "decode_conv", "replay_conv"):
        def call():
            if name == "decode":
                kda.kda_decode_step(q[:n_seq], k[:n_seq], v[:n_seq], g[:n_seq], b[:n_seq], pool, o=o, workspace=ws)
            elif name == "replay":
                kda.kda_replay(pool, k, v, g, b, cu, workspace=ws)
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
    split = (not args.plain_workspace) and full_bytes > plain_bytes + N * H * dk * dv * 4
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

    # end to end through the public API with host buffers: H2D inputs, call, D2H outputs
    e2e = None
    host = {n: x.pin_memory() for n, x in (("q", case.q), ("k", case.k), ("v", case.v), ("g", case.g),
                                           ("beta", case.beta), ("cu", case.cu_seqlens))}
    if case.init_state is not None:
        host["s0"] = case.init_state.pin_memory()
    host_o = torch.empty(T, H, dv, dtype=q.dtype).pin_memory()
    host_fs = torch.empty(N, H, dk, dv, dtype=torch.float32).pin_memory()
    dq, dk_, dvv, dg, db = (torch.empty_like(x) for x in (q, k, v, g, b))
    dcu = torch.empty_like(cu)
    ds0 = None if s0 is None else torch.empty_like(s0)
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = host_o.numel() * host_o.element_size() + host_fs.numel() * 4
    e2e_steps = max(1, min(args.steps, 20))

    def e2e_step():
        dq.copy_(host["q"], non_blocking=True)
        dk_.copy_(host["k"], non_blocking=True)
        dvv.copy_(host["v"], non_blocking=True)
        dg.copy_(host["g"], non_blocking=True)
        db.copy_(host["beta"], non_blocking=True)
        dcu.copy_(host["cu"], non_blocking=True)
        if ds0 is not None:
            ds0.copy_(host["s0"], non_blocking=True)
        call(dq, dk_, dvv, dg, db, dcu, ds0)
        host_o.copy_(o, non_blocking=True)
        host_fs.copy_(fs, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if distributed:
        dist.barrier()
    a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    bb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(bb), dev)
    e2e = {"value": world * T * e2e_steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    hbm_peak, tf_peak, peak_src = measured_peaks()
    nbytes = algorithmic_bytes(case)
    flops = algorithmic_flops(case)
    kern_ms = sorted(step_ms)[len(step_ms) // 2]
    t_hbm = nbytes / (hbm_peak * 1e9)
    t_tc = flops / (tf_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = None if prep else (DOMINANT_TRAFFIC or {}).get(args.workload)  # captured on preprocessed inputs
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
                "clocks": clk, "state_kernels": state_kernels, "backward": backward, "conv_fwd": conv}
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
    ap.add_argument("--prep", action="store_true",
                    help="raw inputs through kda_chunk_fwd_prep with every preprocessing flag")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
