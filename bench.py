"""Benchmark of the KDA forward hot path on GB300.

Default line: chunkwise prefill of the largest single-GPU workload, 64 packed
sequences of seeded lengths uniform in [512, 16384] (about 540 K tokens), H=32,
d_k=d_v=128, chunk 64, bf16 I/O with fp32 state; one step = one kda_chunk_fwd
call over the whole batch.  The same run times the other prefill workloads
(4 x 4096 tokens with H=16, and 1 x 65536 tokens with H=32) under their own names,
the decode workload (256 sequences x 32 heads, 128 consecutive steps, 512 MiB state
updated in place) under "decode", and a 4-token speculative verification under
"verify".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload varlen_prefill_bf16|prefill_bf16|long_prefill_bf16|decode_bf16]

Under torchrun each rank runs its own copy of the workload on its own GPU
(independent problems, no collective on the data path); the timing is the max
over ranks and `value` counts the tokens of all ranks.  `--impl reference`
times the fp64 CPU oracle (the only other implementation of this method) on the
host cores, on rank 0 only.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA tokens/sec on 1 GB300 (prefill & decode) and % of roofline"
D_FLOP_CONST = 180_224          # 6 d^2 + 10 C d flops per token-head at d=128, C=64
PREFILL_KERNELS = ("kda_chunk_tc_kernel", "kda_chunk_simt_kernel")
DEFAULT_WORKLOAD = "varlen_prefill_bf16"  # the largest workload that fits one GPU


# ----------------------------------------------------------------- helpers
def gate_elems(gate: str, d_k: int) -> int:
    """Elements of g read per token-head: one per key channel, one, or none."""
    return {"channel": d_k, "scalar": 1, "none": 0}[gate]


def algorithmic_prefill(token_heads: int, pairs: int, d_k: int, d_v: int, io_bytes: int, C=64,
                        gate: str = "channel"):
    """Algorithmic bytes and flops of one prefill launch.
    bytes: q, k (d_k each), g (see gate_elems) and v (d_v) read, beta read, o (d_v)
    written per token-head, plus the fp32 state read and written once per
    (sequence, head).
    flops: 3 state-sized GEMMs (2 d_k d_v each) + 5 chunk products (2 C d each)
    per token-head, the accounting 2Ld^2 + 2LCd of the chunked-attention cost."""
    per_tok = io_bytes * (2 * d_k + gate_elems(gate, d_k) + 2 * d_v) + io_bytes
    state = 2 * 4 * d_k * d_v
    flops_tok = 2 * (d_k * d_v) * 3 + 2 * C * d_k * 5
    return token_heads * per_tok + pairs * state, token_heads * flops_tok


def algorithmic_decode(pairs: int, d_k: int, d_v: int, io_bytes: int):
    per_tok = io_bytes * (3 * d_k + 2 * d_v) + io_bytes
    return pairs * (per_tok + 2 * 4 * d_k * d_v)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash(kind: str) -> str:
    name = {"tensor": "kda_chunk_tc.cu", "simt": "kda_chunk_simt.cu", "decode": "kda_decode.cu",
            "recurrent": "kda_decode.cu"}[kind]
    p = os.path.join(ROOT, "kimi_delta_attention_fwd_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(f"{kind}:{workload}")
    if not rec or rec.get("source_sha256_16") != kernel_source_hash(kind):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """Samples SM clock and clock-event reasons with NVML (via ctypes on
    libnvidia-ml), falling back to nvidia-smi, while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks",
               0x1: "gpu_idle"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period = period_s
        self._stop = threading.Event()
        self._nvml = None
        self._handle = None
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                raise OSError("handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._handle = nv, h
        except Exception:
            self._nvml = None
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        if self._nvml is None:
            return
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(c)) == 0:
            self.samples.append(c.value)
        if self._nvml.nvmlDeviceGetCurrentClocksEventReasons(self._handle, ctypes.byref(r)) == 0:
            for bit, name in self.REASONS.items():
                if r.value & bit and name != "gpu_idle":
                    self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def __enter__(self):
        self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thread.join()

    def summary(self):
        if self._nvml is None:
            return self._smi_fallback()
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": "nvml"}

    @staticmethod
    def _smi_fallback():
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm", "--format=csv,noheader,nounits"],
                                 capture_output=True, text=True, timeout=20).stdout.split("\n")[0]
            cur, mx = (float(x) for x in out.split(","))
            return {"sm_mhz": cur, "sm_max_mhz": mx, "reasons": [], "samples": 1,
                    "source": "nvidia-smi after the timed region"}
        except Exception:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "none"}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own independent problem (weak scaling, no data exchange)."""
    return seed + 1000 * rank


def max_over_ranks(value: float, ws: int, device) -> float:
    """The job's time is the slowest rank's (all_reduce MAX; a no-op on one rank)."""
    if ws <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: int, ws: int, ms_per_step: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * ws / (ms_per_step * 1e-3)


def oracle_cpu_baseline(x, pairs_limit=None):
    """Times the oracle, as it stands, on the host cores.  Returns (seconds,
    tokens processed, token-heads processed, threads, sample description)."""
    import oracle
    import numpy as np
    import torch
    q, k, v, g, beta, cu, init = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"].cpu(),
                                  x["init_state"])
    # the oracle takes one log alpha per key channel: repeat a per-token one, or zeros
    if g is None:
        g = torch.zeros_like(q)
    elif g.dim() == 2:
        g = g.unsqueeze(-1).expand_as(q)
    H = q.shape[1]
    if pairs_limit is not None and pairs_limit < H:
        q, k, v, g, beta = (t[:, :pairs_limit] for t in (q, k, v, g, beta))
        init = None if init is None else init[:, :pairs_limit]
    # widen once outside the timed call (the oracle's input is fp64)
    q, k, v, g, beta = (t.float().cpu().numpy().astype(np.float64) for t in (q, k, v, g, beta))
    init = None if init is None else init.cpu().numpy().astype(np.float64)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.kda_fwd(q, k, v, g, beta, cu.numpy(), init_state=init, threads=threads)
    dt = time.perf_counter() - t0
    tokens = int(cu[-1])
    heads = q.shape[1]
    return dt, tokens, tokens * heads, threads, heads


# ------------------------------------------------------------- our arm
def run_prefill(args, ws, rank, dev, workload, e2e=True, steps=None):
    """Times `steps` kda_chunk_fwd calls on the named workload (inputs resident in HBM),
    and with e2e=True the same calls end to end from pinned host memory.  Returns the
    result block and the inputs (for the CPU baseline)."""
    import torch
    from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd, kda_chunk_fwd_workspace_bytes
    from kimi_delta_attention_fwd_gb300 import workloads as W
    from kimi_delta_attention_fwd_gb300 import kda as K

    steps = args.steps if steps is None else steps
    spec = W.named(workload)
    spec = W.PrefillSpec(spec.seqlens, spec.num_heads, spec.d_k, spec.d_v, spec.io_dtype, spec.gate,
                         spec.init, rank_seed(spec.seed, rank))
    big = spec.total_tokens * spec.num_heads > 4_000_000
    # --prep: q, k and beta as drawn before the input steps, which the kernels then apply
    x = W.prefill_inputs(spec, device=("cuda" if big else "cpu"), raw=args.prep)
    prep = dict(qk_silu=args.prep, qk_l2norm=args.prep, beta_sigmoid=args.prep)
    if args.gate == "scalar":    # Gated DeltaNet: one log alpha per (token, head)
        x["g"] = x["g"][..., 0].contiguous()
    elif args.gate == "none":    # DeltaNet: alpha = 1, no g at all
        x["g"] = None
    d = {kk: (vv.to(dev) if vv is not None else None) for kk, vv in x.items()}
    T, H, dk, dv, N = spec.total_tokens, spec.num_heads, spec.d_k, spec.d_v, spec.num_seqs
    io_bytes = 2 if spec.io_dtype == "bf16" else 4
    out = torch.empty((T, H, dv), dtype=d["q"].dtype, device=dev)
    fin = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    wsb = kda_chunk_fwd_workspace_bytes(N, T, H, dk, dv, d["q"].dtype, args.algo)
    work = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    tensor_path = K.kda_chunk_fwd_selected_algo(N, T, H, dk, dv, d["q"].dtype, args.algo) == "tensor"
    # kernels one call launches: the prefill kernel; on the tensor-core path with a decay the
    # check-and-recompute kernel of the exact fallback; and, when the plain schedule takes
    # more than one wave, the launch-order kernel (the workspace here always has room)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    per_call = 1 + (1 if tensor_path and args.gate != "none" else 0) + \
        (1 if tensor_path and N * H > max(76, sms) and 2 <= N <= 2048 else 0)

    def step(o=out, f=fin):
        kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"],
                      out=o, final_state=f, workspace=work, algo=args.algo, stream=stream, **prep)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    from kimi_delta_attention_fwd_gb300 import kda_workspace_status, workspace_status_words
    status = kda_workspace_status(work, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    # the tensor-core schedule that ran (status word 2): the segment-parallel scan of one
    # sequence launches the run tables, the start states, the first pass, the combine, the
    # second pass and the final-state copy in place of the one prefill kernel
    schedule = {1: "plain", 2: "solve helpers", 3: "segments"}.get(
        int(workspace_status_words(work)[2]), "none") if tensor_path else "none"
    if schedule == "segments":
        per_call += 5

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms_step = max_over_ranks(total_ms / steps, ws, dev)
    hbm, tflops, peak_src = measured_peaks()
    alg_bytes, alg_flops = algorithmic_prefill(T * H, N * H, dk, dv, io_bytes, gate=args.gate)
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    kind = "tensor" if tensor_path else "simt"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm,
                "traffic": recorded_traffic(kind, (workload if args.gate == "channel" else
                                                   f"{workload}:{args.gate}")
                                            + (":prep" if args.prep else "")),
                "peak_source": f"{peak_src} hbm_gbs",
                "tensor_tflops_algorithmic": alg_flops / (launch_ms * 1e-3) / 1e12,
                "tensor_peak_tflops": tflops,
                "kernel_ms": launch_ms,
                "roofline_ms": max(alg_bytes / (hbm * 1e9), alg_flops / (tflops * 1e12)) * 1e3}
    config = {"workload": workload, "num_seqs": N, "total_tokens": T, "num_heads": H,
              "d_k": dk, "d_v": dv, "chunk": 64, "io_dtype": spec.io_dtype, "gate": args.gate,
              "prep": "silu + l2norm of q, k; sigmoid of beta" if args.prep else "none",
              "kernel": kind, "schedule": schedule, "l2": "inputs larger than L2 (%.0f MB read+written per step)" % (alg_bytes / 1e6),
              "parallelism": f"replicas x{ws} (independent sequences per GPU)"}
    if not e2e:
        del d, out, fin, work
        return {"workload": workload, "value": aggregate_throughput(T, ws, ms_step), "unit": "tokens/s",
                "ms_per_step": ms_step, "steps": steps, "config": config, "roofline": roofline,
                "gpu_launches": steps * per_call, "clocks": clk.summary()}, x

    # e2e through the public API: every step copies its inputs from pinned host memory,
    # runs kda_chunk_fwd and reads its outputs and final states back.  Steps are
    # double-buffered on three streams (copy in, compute, copy out), so step i + 1's
    # inputs cross the host link while step i computes and its results come back.
    e2e_steps = max(2, min(steps, 10))
    host_in = {kk: (vv.to("cpu").pin_memory() if vv is not None else None) for kk, vv in x.items()}
    h2d = sum(vv.numel() * vv.element_size() for vv in host_in.values() if vv is not None)
    sets = []
    for _ in range(2):
        sets.append(dict(
            din={kk: (torch.empty_like(vv, device=dev) if vv is not None else None) for kk, vv in x.items()},
            out=torch.empty_like(out), fin=torch.empty_like(fin),
            hout=torch.empty_like(out, device="cpu").pin_memory(),
            hfin=torch.empty_like(fin, device="cpu").pin_memory(),
            work=torch.zeros_like(work)))
    d2h = sets[0]["hout"].numel() * sets[0]["hout"].element_size() + \
        sets[0]["hfin"].numel() * sets[0]["hfin"].element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_cmp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            b = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])  # step i - 2 has read this input set
                for kk, vv in host_in.items():
                    if vv is not None:
                        b["din"][kk].copy_(vv, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])  # step i - 2's results have left this set
                di = b["din"]
                kda_chunk_fwd(di["q"], di["k"], di["v"], di["g"], di["beta"], di["cu_seqlens"],
                              di["init_state"], out=b["out"], final_state=b["fin"], workspace=b["work"],
                              algo=args.algo, stream=s_cmp, **prep)
                ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                b["hout"].copy_(b["out"], non_blocking=True)
                b["hfin"].copy_(b["fin"], non_blocking=True)
                ev_out[i].record(s_out)
        return ev_out[n - 1]

    e2e_run(2)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    last = e2e_run(e2e_steps)
    b_end = torch.cuda.Event(enable_timing=True)
    s_out.wait_event(last)
    b_end.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b_end) / e2e_steps, ws, dev)

    res = {
        "metric": METRIC, "value": aggregate_throughput(T, ws, ms_step), "unit": "tokens/s", "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if tensor_path else "f32", "data": "synthetic",
        "config": config, "roofline": roofline,
        "e2e": {"value": aggregate_throughput(T, ws, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "schedule": "double-buffered: a step's host-to-device copies overlap the previous step's kernel and device-to-host copies"},
        "gpu_launches": steps * per_call,
        "clocks": clk.summary(),
    }
    del sets, host_in, d, out, fin, work
    return res, x


def run_decode(args, ws, rank, dev, name="decode_bf16"):
    import torch
    from kimi_delta_attention_fwd_gb300 import kda_decode_step
    from kimi_delta_attention_fwd_gb300 import workloads as W
    spec = W.named(name)
    spec = W.DecodeSpec(spec.num_seqs, spec.num_heads, spec.d_k, spec.d_v, spec.steps, spec.io_dtype,
                        spec.gate, rank_seed(spec.seed, rank))
    y = W.decode_inputs(spec, device=str(dev))
    st = y["state"].clone()
    outs = torch.empty((spec.steps, spec.num_seqs, spec.num_heads, spec.d_v), dtype=y["q"].dtype, device=dev)
    stream = torch.cuda.current_stream()

    def run_all():
        for t in range(spec.steps):
            kda_decode_step(y["q"][t], y["k"][t], y["v"][t], y["g"][t], y["beta"][t], st, out=outs[t],
                            stream=stream)

    for _ in range(max(1, args.warmup)):
        run_all()
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 5))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        a.record(stream)
        for _ in range(reps):
            run_all()
        b.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / (reps * spec.steps), ws, dev)  # per decode step
    io_bytes = 2 if spec.io_dtype == "bf16" else 4
    by = algorithmic_decode(spec.num_seqs * spec.num_heads, spec.d_k, spec.d_v, io_bytes)
    hbm, _, src = measured_peaks()
    ach = by / (ms * 1e-3) / 1e9
    return {"workload": name, "value": aggregate_throughput(spec.num_seqs, ws, ms), "unit": "tokens/s",
            "ms_per_decode_step": ms, "steps_per_rep": spec.steps, "reps": reps,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": recorded_traffic("decode", name), "peak_source": f"{src} hbm_gbs"},
            "gpu_launches": reps * spec.steps, "clocks": clk.summary()}


def run_verify(args, ws, rank, dev, drafts=4, name="decode_bf16"):
    """Speculative verification on the decode workload's sequences: `drafts`
    consecutive tokens per sequence through kda_recurrent_fwd in one call (outputs
    of every token, the state advanced in place), against `drafts` decode steps."""
    import torch
    from kimi_delta_attention_fwd_gb300 import kda_recurrent_fwd
    from kimi_delta_attention_fwd_gb300 import workloads as W
    spec = W.named(name)
    spec = W.DecodeSpec(spec.num_seqs, spec.num_heads, spec.d_k, spec.d_v, drafts, spec.io_dtype,
                        spec.gate, rank_seed(spec.seed, rank))
    y = W.decode_inputs(spec, device=str(dev))
    N, H = spec.num_seqs, spec.num_heads
    pack = lambda t: t.transpose(0, 1).reshape(N * drafts, *t.shape[2:]).contiguous()
    q, k, v, g, beta = (pack(y[n]) for n in ("q", "k", "v", "g", "beta"))
    cu = torch.arange(N + 1, dtype=torch.int32, device=dev) * drafts
    st = y["state"].clone()
    out = torch.empty((N * drafts, H, spec.d_v), dtype=q.dtype, device=dev)
    stream = torch.cuda.current_stream()
    call = lambda: kda_recurrent_fwd(q, k, v, g, beta, cu, st, out=out, final_state=st, stream=stream)
    for _ in range(max(1, args.warmup)):
        call()
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 10))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        a.record(stream)
        for _ in range(reps):
            call()
        b.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / reps, ws, dev)
    io_bytes = 2 if spec.io_dtype == "bf16" else 4
    per_tok = io_bytes * (3 * spec.d_k + 2 * spec.d_v) + io_bytes
    by = N * H * (drafts * per_tok + 2 * 4 * spec.d_k * spec.d_v)
    hbm, _, src = measured_peaks()
    ach = by / (ms * 1e-3) / 1e9
    return {"workload": f"{name} sequences, {drafts} draft tokens each (kda_recurrent_fwd)",
            "value": aggregate_throughput(N * drafts, ws, ms), "unit": "tokens/s", "ms_per_call": ms,
            "reps": reps,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": recorded_traffic("recurrent", f"verify{drafts}:{name}"),
                         "peak_source": f"{src} hbm_gbs"},
            "gpu_launches": reps, "clocks": clk.summary()}


def main_ours(args):
    import torch
    ws, rank, local = dist_info()
    if ws > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from kimi_delta_attention_fwd_gb300 import build as kbuild
    if not kbuild.up_to_date():
        kbuild.build()
    if args.workload == "decode_bf16":
        dec = run_decode(args, ws, rank, dev)
        res = {"metric": METRIC, "value": dec["value"], "unit": "tokens/s", "n_gpus": ws,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": dec["ms_per_decode_step"],
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
               "data": "synthetic", "config": {"workload": "decode_bf16", "l2": "state 512 MiB > L2"},
               "roofline": dec["roofline"], "gpu_launches": dec["gpu_launches"], "clocks": dec["clocks"]}
        x = None
    else:
        res, x = run_prefill(args, ws, rank, dev, args.workload)
    if rank == 0 and not args.no_cpu_baseline and not args.prep and x is not None:
        # a bounded sample: on the largest workloads (over 4 M token-heads) an eighth
        # of the heads, so that one oracle run stays within seconds
        limit = args.cpu_heads
        if limit is None and x["q"].shape[0] * x["q"].shape[1] > 4_000_000:
            limit = max(1, x["q"].shape[1] // 8)
        # repeat the sample until about --cpu-seconds of oracle time have accumulated
        reps, total = 0, 0.0
        while True:
            dt, tokens, th, threads, heads = oracle_cpu_baseline(x, pairs_limit=limit)
            reps, total = reps + 1, total + dt
            if total >= args.cpu_seconds or reps >= 50:
                break
        dt = total / reps
        res["cpu_baseline"] = {"value": th / dt / x["q"].shape[1],
                               "unit": "tokens/s", "cores": threads, "kind": "oracle",
                               "sample": f"{args.workload}: all {tokens} tokens of {heads} of {x['q'].shape[1]} heads "
                                         f"({th} token-heads per run, {reps} runs, {total:.1f} s in all), "
                                         f"scaled to tokens/s over all heads"}
    x = None
    torch.cuda.empty_cache()
    if args.workload == DEFAULT_WORKLOAD and not args.prep:
        # the other prefill workloads, each timed the same way on the device (no e2e leg)
        if not args.no_extra:
            for name in ("prefill_bf16", "long_prefill_bf16"):
                blk, _ = run_prefill(args, ws, rank, dev, name, e2e=False, steps=min(args.steps, 10))
                res[name] = blk
                torch.cuda.empty_cache()
        if not args.no_decode:
            res["decode"] = run_decode(args, ws, rank, dev)
            res["verify"] = run_verify(args, ws, rank, dev)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


# ------------------------------------------------------- reference arm
def main_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import torch
    from kimi_delta_attention_fwd_gb300 import workloads as W
    spec_name = args.workload if args.workload != "decode_bf16" else DEFAULT_WORKLOAD
    spec = W.named(spec_name)
    H = spec.num_heads
    # each step runs a bounded sample: every token of `heads` heads (one head on the
    # workloads over 4 M token-heads, all heads otherwise)
    heads = args.cpu_heads or (1 if spec.total_tokens * H > 4_000_000 else H)
    if torch.cuda.is_available():
        # the same inputs as our arm, drawn on the device; the sampled heads go to the host
        x = W.prefill_inputs(spec, device="cuda")
        drawn = "the workload's own inputs"
    else:
        # no device to draw the whole workload on: the same recipe and lengths, drawn
        # for the sampled heads only
        spec = W.PrefillSpec(spec.seqlens, heads, spec.d_k, spec.d_v, spec.io_dtype, spec.gate,
                             spec.init, spec.seed)
        x = W.prefill_inputs(spec)
        drawn = "inputs of the same recipe drawn for the sampled heads"
    if args.gate == "scalar":
        x["g"] = x["g"][..., 0].contiguous()
    elif args.gate == "none":
        x["g"] = None
    times = []
    for i in range(args.warmup + args.steps):
        dt, tokens, th, threads, used = oracle_cpu_baseline(x, pairs_limit=heads)
        if i >= args.warmup:
            times.append(dt)
    dt = statistics.mean(times)
    value = tokens * (used / H) / dt  # tokens/s over all heads, from a sample of heads
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 * H / used,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": spec_name, "num_seqs": spec.num_seqs,
                      "total_tokens": spec.total_tokens, "num_heads": H, "d_k": spec.d_k,
                      "d_v": spec.d_v, "gate": args.gate},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                            "sample": f"{used} of {H} heads, all {tokens} tokens per step ({drawn}), "
                                      f"scaled to tokens/s over all heads"},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["prefill_bf16", "long_prefill_bf16", "long_prefill_16k_bf16",
                             "varlen_prefill_bf16", "decode_bf16"])
    ap.add_argument("--algo", default="auto", choices=["auto", "tensor", "simt"])
    ap.add_argument("--gate", default="channel", choices=["channel", "scalar", "none"],
                    help="decay per key channel (KDA), per token (Gated DeltaNet) or none (DeltaNet)")
    ap.add_argument("--cpu-heads", type=int, default=None,
                    help="heads of the workload the CPU oracle runs (default: all; an eighth on "
                         "workloads over 4 M token-heads)")
    ap.add_argument("--prep", action="store_true",
                    help="raw q, k and beta logits; the kernels apply silu and the L2 norm to q, k "
                         "and the sigmoid to beta (no CPU baseline, no decode block)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the 4 x 4096 and 1 x 65536 prefill blocks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle time to accumulate for the CPU baseline (whole runs of the sample)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
