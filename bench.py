"""Benchmark of the TTT layer forward on GB300: tokens/s (B*H*T per second).

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl ours|reference]

One step = one forward of the whole layer (one kernel launch) over one batch of
synthetic inputs already resident in HBM; the L2 is flushed before every timed
step (a 256 MiB write, larger than the 129 MB L2, then a 256 MiB read so the L2
holds clean lines).  Device time comes from CUDA
events on the launching stream.  Rank 0 prints one JSON line.

Under torchrun every rank runs the same workload on its own GPU (independent
(batch, head) chains, no data-path collective: weak scaling); the step time is the
maximum over ranks.

--impl reference times the fp64 CPU oracle (the only reference this method has)
on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "TTT layer fwd tokens/s (B·H·T) and TFLOP/s vs GB300 bf16 dense peak, 1 GPU"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- work model


def flops_per_token_head(inp):
    """Algorithmic FLOPs of one token-head (masked products counted exactly:
    (b+1)/2 visible pairs per token in a causal block of b)."""
    d, m, b = inp.d, inp.m, inp.b
    o = inp.options
    if inp.kind == "gate":  # theta_h . x_t over the layer width H d, then the sigmoid
        return 2 * inp.H * d
    if inp.kind == "dwconv":
        # per channel and epoch: residual 9 FMAs (none for the dot loss), gradient 9
        # FMAs; output 9 FMAs
        per_epoch = 18 * d + (18 * d if o.get("loss", "mse") == "mse" else 0)
        return o.get("epochs", 1) * per_epoch + 18 * d
    if inp.kind == "linear" and o.get("gate"):
        # the rate gate: theta_h . x_t over the model width H d (2 H d), then the layer
        return 2 * inp.H * d + 6 * d * d + (2 * (b + 1) * d if inp.causal else 0)
    if inp.kind == "linear" and o.get("ln"):
        # plus the inner norm: statistics, normalisation and its backward on k W (about
        # 12 d) and on q W (about 6 d)
        return 6 * d * d + (2 * (b + 1) * d if inp.causal else 0) + 18 * d
    if inp.kind == "linear" and (o.get("loss") == "dot" or o.get("epochs", 1) > 1):
        # dot loss: no K W product; epochs: the E / update pass repeats
        upd = (2 if o.get("loss") == "dot" else 4) * d * d
        return o.get("epochs", 1) * upd + 2 * d * d + (2 * (b + 1) * d if inp.causal else 0)
    if inp.kind == "linear":
        # E = K W, update K^T Et, Q W (2d^2 each); causal: masked (Q K^T) and its product
        # with Et over (b+1)/2 visible pairs (2d each); non-causal: Z = Q W_end
        return 6 * d * d + (2 * (b + 1) * d if inp.causal else 0)
    # MLP: 7 products of 2dm (K W1, A W2, E W2^T, two updates, Q W1, A_q W2) + masked terms
    # (+ about 18 d for the inner norm: statistics, normalisation and its backward)
    if inp.causal:
        return 14 * d * m + 2 * (b + 1) * (d + m) + (18 * d if o.get("ln") else 0)
    return 14 * d * m + 2 * (d + m)


def bytes_per_launch(inp):
    """Algorithmic HBM bytes of one launch: q, k, v read once, z written once,
    per-token eta read, initial weights read once per head, final weights written."""
    es = inp.q.element_size()
    BH, T, d = inp.B * inp.H, inp.T, inp.d
    if inp.kind == "gate":  # x read once, the gate vectors, the rates written
        return inp.q.numel() * es + inp.gate_theta.numel() * 2 + BH * T * 4
    n = BH * T * d * es * 4
    if inp.eta is not None:
        n += BH * T * 4
    nparam = sum(p.numel() for p in inp.params.values()) // inp.H  # one head's set
    n += inp.H * nparam * 4 + BH * nparam * 4
    if inp.gate_x is not None:
        # the gate reads x and its vectors once and writes the rates, which the layer reads
        n += inp.gate_x.numel() * 2 + inp.gate_theta.numel() * 2 + 2 * BH * T * 4
    return n


def roofline_bound(flops, nbytes, ms, peaks):
    """The attainable bound min(tensor peak, AI x HBM bandwidth): the launch is
    HBM-bound when its algorithmic bytes take longer at the copy bandwidth than its
    algorithmic FLOPs at the bf16 tensor peak, else tensor-bound.  The fraction is
    achieved / peak of that resource."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "bound_ms": t_hbm * 1e3}
    tf = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tf / peaks["bf16_tflops"], "bound_ms": t_tc * 1e3}


def kernel_name(inp):
    """The kernel the library dispatches this workload to (mirrors the C ABI's choice)."""
    if inp.kind == "gate":
        return "ttt_eta_gate_kernel"
    if inp.kind == "dwconv":
        return "ttt_dwconv_kernel"
    if inp.q.element_size() == 4:
        return "ttt_linear_f32_kernel" if inp.kind == "linear" else "ttt_mlp_f32_kernel"
    if inp.kind == "linear":
        if not inp.causal and inp.b >= inp.T and inp.d == 64 and inp.T <= 256:
            return "ttt_linear_fb_tc_kernel" if inp.options.get("epochs", 1) == 1 else "ttt_linear_fb_kernel"
        if inp.b == 1 and inp.options.get("epochs", 1) == 1 and not inp.options.get("ln"):
            # the delta rule: 16-token chunks on the b = 16 kernel (d <= 64, MSE), else the
            # column-parallel kernel
            dot = inp.options.get("loss", "mse") == "dot"
            return "ttt_linear_b16_kernel" if inp.d <= 64 and not dot else "ttt_linear_b1_kernel"
        return "ttt_linear_b16_kernel" if min(inp.b, inp.T) == 16 and inp.d <= 64 else "ttt_linear_bf16_kernel"
    if inp.d == 64 and not inp.causal and inp.b >= inp.T:
        return "ttt_mlp_fb_tc_kernel"
    if inp.d == 64 and min(inp.b, inp.T) <= 16:
        return "ttt_mlp_w8_ln_kernel" if inp.options.get("ln") else "ttt_mlp_w8_kernel"
    return "ttt_mlp_bf16_kernel"


def recorded_traffic(workload):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json), or
    None when there is no record or the kernel sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(workload)
    if not rec:
        return None
    m = hashlib.sha256()
    for name in rec["sources"]:
        with open(os.path.join(ROOT, "test_sequence_layers_gb300", "csrc", name), "rb") as f:
            m.update(f.read())
    return rec["dram_bytes_per_launch"] if m.hexdigest() == rec["sources_sha256"] else None


# --------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle sampling; summary() keeps the samples taken
    inside the timed region [t0, t1] (host wall clock)."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = ""

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    @staticmethod
    def _ts(s):
        import datetime
        try:
            return datetime.datetime.strptime(s.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self, t0, t1, spin0=None):
        """Clocks over the timed region [t0, t1]; when the region is too short for the
        sampler to land in it, over the untimed spin [spin0, t0) that ran the same
        step back to back just before it (labelled in "source")."""
        rows = [r for r in csv.reader(io.StringIO(self.out)) if len(r) >= 9]
        within = lambda a, b: [r for r in rows if (lambda t: t is not None and a <= t <= b)(self._ts(r[0]))]
        inside = within(t0, t1)
        spin = within(spin0, t0) if spin0 is not None else []
        use = inside or spin or rows
        source = ("timed region" if inside else
                  "same-load spin just before the timed region (the region is shorter than the "
                  "sampling interval)" if spin else "whole run")
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        num = lambda x: float(x) if x.strip().replace(".", "", 1).isdigit() else None
        sm = [v for v in (num(r[1]) for r in use) if v is not None]
        mx = [v for v in (num(r[2]) for r in use) if v is not None]
        pw = [v for v in (num(r[3]) for r in use) if v is not None]
        reasons = sorted({n for r in use for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None,
                "samples": len(use), "samples_in_timed_region": len(inside), "source": source}


# ------------------------------------------------------------------ our arm


def allreduce_max(x, dev):
    """Maximum of a host float over ranks (device tensor for NCCL, host for gloo)."""
    on = dev if torch.distributed.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=on)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


E2E_STREAMS = 3


def run_ours(args, rank, world, inp, peaks):
    from test_sequence_layers_gb300 import abi, build
    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    q, k, v = (x.to(dev) if x is not None else None for x in (inp.q, inp.k, inp.v))
    # the per-token input of the rate: eta itself, or the layer input x of the gate
    gate = inp.gate_x is not None
    eta_src = inp.gate_x if gate else inp.eta
    eta = eta_src.to(dev) if eta_src is not None else None
    theta = inp.gate_theta.to(dev) if inp.gate_theta is not None else None
    params = {n: p.to(dev) for n, p in inp.params.items()}
    z = torch.empty_like(q) if inp.kind != "gate" else None
    B, H, d = inp.B, inp.H, inp.d
    if inp.kind == "linear":
        outs = torch.empty((B, H, d, d), device=dev)
        # fewer chains than SMs: the sequence-parallel entry point (affine maps of
        # segments, scan, segment outputs), with its workspace allocated once
        need = 0 if args.no_seqpar else abi.ttt_linear_seqpar_workspace(
            B, H, inp.T, d, inp.b, inp.causal, dtype=inp.q.dtype)
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None

        loss, epochs = inp.options.get("loss", "mse"), inp.options.get("epochs", 1)
        if loss != "mse" or epochs != 1 or "ln_gamma" in params:
            ws = None

        def new_outs():
            return [torch.empty((B, H, d, d), device=dev)]

        def step(qq=q, kk=k, vv=v, ee=eta, zz=z, oo=(outs,), wsp=ws):
            if gate:  # ee holds x: the rates come from the gate, every step
                ee = abi.ttt_eta_gate(ee, theta, inp.eta_scalar)
            if wsp is not None:
                abi.ttt_linear_fwd_seqpar(qq, kk, vv, params["W0"], inp.b, inp.causal, eta=ee,
                                          eta_scalar=inp.eta_scalar, z=zz, W_out=oo[0], workspace=wsp)
            else:
                abi.ttt_linear_fwd(qq, kk, vv, params["W0"], inp.b, inp.causal, eta=ee,
                                   eta_scalar=inp.eta_scalar, z=zz, W_out=oo[0], loss=loss,
                                   epochs=epochs, ln_gamma=params.get("ln_gamma"),
                                   ln_beta=params.get("ln_beta"))
        out_bytes = [z, outs]
    elif inp.kind == "gate":  # the rates alone, from x (held in q)
        outs = torch.empty((B, H, inp.T), device=dev)
        ws = None

        def new_outs():
            return [torch.empty((B, H, inp.T), device=dev)]

        def step(qq=q, kk=None, vv=None, ee=None, zz=None, oo=(outs,), wsp=None):
            abi.ttt_eta_gate(qq, theta, inp.eta_scalar, eta=oo[0])
        out_bytes = [outs]
    elif inp.kind == "dwconv":
        outs = torch.empty((B, H, 9, d), device=dev)
        o = inp.options
        ws = None

        def new_outs():
            return [torch.empty((B, H, 9, d), device=dev)]

        def step(qq=q, kk=k, vv=v, ee=eta, zz=z, oo=(outs,), wsp=None):
            abi.ttt_dwconv_fwd(qq, kk, vv, params["W0"], o["height"], o["width"], eta=ee,
                               eta_scalar=inp.eta_scalar, loss=o.get("loss", "mse"),
                               epochs=o.get("epochs", 1), z=zz, W_out=oo[0])
        out_bytes = [z, outs]
    else:
        m = inp.m
        ws = None

        def new_outs():
            return [torch.empty((B, H, d, m), device=dev), torch.empty((B, H, m), device=dev),
                    torch.empty((B, H, m, d), device=dev), torch.empty((B, H, d), device=dev)]
        outs = tuple(new_outs())

        def step(qq=q, kk=k, vv=v, ee=eta, zz=z, oo=outs, wsp=None):
            abi.ttt_mlp_fwd(qq, kk, vv, params["W1"], params["c1"], params["W2"], params["c2"],
                            inp.b, inp.causal, eta=ee, eta_scalar=inp.eta_scalar, z=zz, outs=tuple(oo),
                            activation=inp.options.get("activation", "silu"),
                            ln_gamma=params.get("ln_gamma"), ln_beta=params.get("ln_beta"))
        out_bytes = [z, *outs]

    flush_w = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.zeros((), dtype=torch.float32, device=dev)

    def l2_flush():
        # write a buffer larger than L2, then read another one so the L2 holds clean
        # lines (no write-back of the flush traffic inside the timed launch)
        flush_w.add_(1.0)
        flush_out.copy_(flush_r.sum())

    for _ in range(args.warmup):
        l2_flush()
        step()
    abi.ttt_sync_status()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clk = ClockSampler(dev.index)
    if not args.quick:
        clk.start()
    # keep the GPU busy (untimed) while the sampler starts up; its samples stand in
    # for a timed region shorter than the sampling interval
    spin_wall0 = time.time()
    t_spin = time.perf_counter()
    while not args.quick and time.perf_counter() - t_spin < 0.6:
        l2_flush()
        step()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n0 = abi.ttt_launch_count()
    w0 = time.time()
    for i in range(args.steps):
        l2_flush()  # evict the inputs from L2 (outside the timed events)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    launches = abi.ttt_launch_count() - n0
    clk.stop()
    abi.ttt_sync_status()
    if world > 1:
        torch.distributed.barrier()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = statistics.mean(times)
    if world > 1:
        ms = allreduce_max(ms, dev)

    # end to end through the same call with host buffers: pinned host -> device
    # copies of the step's inputs, the forward, device -> host copies of z and the
    # final weights, all inside the timed region.  Steps go round-robin over E2E_STREAMS
    # streams, each with its own device buffers (and split-path workspace), so one
    # step's copies overlap another step's compute, as a serving loop would run them;
    # every step still moves its own inputs and outputs.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (x.pin_memory() if x is not None else None for x in (inp.q, inp.k, inp.v))
        he = eta_src.pin_memory() if eta_src is not None else None
        lanes = []
        for _ in range(E2E_STREAMS):
            like = lambda t: torch.empty_like(t) if t is not None else None
            ln = {"s": torch.cuda.Stream(device=dev), "q": like(q), "k": like(k),
                  "v": like(v), "e": like(eta),
                  "z": like(z), "o": new_outs(),
                  "ws": torch.empty_like(ws) if ws is not None else None}
            ln["h"] = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in [ln["z"], *ln["o"]]
                       if t is not None]
            lanes.append(ln)

        def e2e_step(i):
            ln = lanes[i % E2E_STREAMS]
            with torch.cuda.stream(ln["s"]):
                for dst, src in ((ln["q"], hq), (ln["k"], hk), (ln["v"], hv)):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
                if ln["e"] is not None:
                    ln["e"].copy_(he, non_blocking=True)
                step(ln["q"], ln["k"], ln["v"], ln["e"], ln["z"], ln["o"], ln["ws"])
                for h, t in zip(ln["h"], [t for t in [ln["z"], *ln["o"]] if t is not None]):
                    h.copy_(t, non_blocking=True)
        for i in range(E2E_STREAMS):
            e2e_step(i)
        torch.cuda.synchronize()
        ne = max(3 * E2E_STREAMS, min(args.steps, 12))
        t0 = time.perf_counter()
        for i in range(ne):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / ne
        if world > 1:
            e2e_ms = allreduce_max(e2e_ms, dev)
        h2d = sum(x.numel() * x.element_size() for x in (inp.q, inp.k, inp.v) if x is not None)
        h2d += eta_src.numel() * eta_src.element_size() if eta_src is not None else 0
        d2h = sum(t.numel() * t.element_size() for t in out_bytes)
        e2e = {"value": world * inp.token_heads / (e2e_ms / 1e3), "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    clocks = clk.summary(w0, w1, spin_wall0)
    return ms, times, launches, e2e, clocks


# -------------------------------------------------------------- CPU baseline


def oracle_sample(inp, budget_s):
    """Times the fp64 oracle on whole (batch, head) chains of the workload, adding
    chains until about budget_s of CPU work; returns (token-heads/s, threads, desc)."""
    import numpy as np
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    if inp.kind == "gate":  # slices of 1024 tokens of the layer input, every head
        done, elapsed, S = 0, 0.0, 1024
        while elapsed < budget_s and done < inp.B * inp.T:
            b, t = divmod(done, inp.T)
            t0 = time.perf_counter()
            oracle.eta_gate(inp.q[b:b + 1, t:t + S], inp.gate_theta, inp.eta_scalar)
            elapsed += time.perf_counter() - t0
            done += min(S, inp.T - t)
        return done * inp.H / elapsed, 1, f"{done} of {inp.B * inp.T} tokens x {inp.H} heads, " \
                                           f"{elapsed:.1f} s of oracle time (one thread)"
    BH = inp.B * inp.H
    n = min(BH, threads)
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < BH:
        take = min(n, BH - done)
        sel = list(range(done, done + take))
        flat = lambda x: x.reshape(-1, *x.shape[2:])[sel].unsqueeze(0)
        q, k, v = flat(inp.q), flat(inp.k), flat(inp.v)
        eta = flat(inp.eta) if inp.eta is not None else None
        t0 = time.perf_counter()
        o = inp.options
        if inp.gate_x is not None:  # the rates of the sampled chains from the gate
            eta = torch.from_numpy(np.stack([oracle.eta_gate(inp.gate_x[c // inp.H:c // inp.H + 1],
                                                             inp.gate_theta[c % inp.H:c % inp.H + 1],
                                                             inp.eta_scalar)[0, 0] for c in sel]))[None]
        if inp.kind == "linear":
            W0 = torch.stack([inp.params["W0"][c % inp.H] for c in sel]).unsqueeze(0)
            ln = {}
            if "ln_gamma" in inp.params:
                ln = {"ln_gamma": torch.stack([inp.params["ln_gamma"][c % inp.H] for c in sel]),
                      "ln_beta": torch.stack([inp.params["ln_beta"][c % inp.H] for c in sel])}
            oracle.linear(q, k, v, W0, inp.b, inp.causal, eta=eta, eta_scalar=inp.eta_scalar,
                          threads=threads, loss=o.get("loss", "mse"), epochs=o.get("epochs", 1), **ln)
        elif inp.kind == "dwconv":
            W0 = torch.stack([inp.params["W0"][c % inp.H] for c in sel]).unsqueeze(0)
            oracle.dwconv(q, k, v, W0, o["height"], o["width"], eta=eta, eta_scalar=inp.eta_scalar,
                          loss=o.get("loss", "mse"), epochs=o.get("epochs", 1), threads=threads)
        else:
            P = [torch.stack([inp.params[nm][c % inp.H] for c in sel]).unsqueeze(0)
                 for nm in ("W1", "c1", "W2", "c2")]
            ln = {}
            if "ln_gamma" in inp.params:
                ln = {"ln_gamma": torch.stack([inp.params["ln_gamma"][c % inp.H] for c in sel]),
                      "ln_beta": torch.stack([inp.params["ln_beta"][c % inp.H] for c in sel])}
            oracle.mlp(q, k, v, *P, inp.b, inp.causal, eta=eta, eta_scalar=inp.eta_scalar,
                       threads=threads, activation=o.get("activation", "silu"), **ln)
        elapsed += time.perf_counter() - t0
        done += take
        n = min(2 * n, BH)
    th = done * inp.T
    return th / elapsed, threads, f"{done} of {BH} (batch, head) chains, full T={inp.T}, " \
                                  f"{elapsed:.1f} s of oracle time"


# ---------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="linear_125m")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-seqpar", action="store_true",
                    help="TTT-Linear: always one CTA per chain (no sequence-parallel split)")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only (no clock spin, e2e or CPU baseline); "
                         "used for profiler captures")
    args = ap.parse_args()
    if args.quick:
        args.no_e2e = args.no_cpu_baseline = True
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend)

    from test_sequence_layers_gb300 import synth
    inp = synth.workload(args.workload)
    peaks = load_peaks()
    flops = flops_per_token_head(inp) * inp.token_heads
    config = {"workload": args.workload, "kind": inp.kind, "B": inp.B, "H": inp.H, "T": inp.T,
              "d": inp.d, "m": inp.m or None, "mini_batch": inp.b, "causal": inp.causal,
              "eta": ("per-token sigmoid(g)" if inp.eta is not None else
                      f"per-token {inp.eta_scalar} sigmoid(theta_h . x_t), x of width {inp.H * inp.d} (ttt_eta_gate)"
                      if inp.gate_x is not None else inp.eta_scalar),
              "io_dtype": str(inp.q.dtype).replace("torch.", ""),
              "state_dtype": "float32", "l2": "flushed before every timed step (256 MiB write + 256 MiB read)",
              "parallelism": f"weak: every rank runs its own {inp.B}x{inp.H} chains"}

    if args.impl == "reference":
        if rank != 0:
            return
        steps = []
        threads, desc = 0, ""
        for _ in range(args.warmup + args.steps):
            v, threads, desc = oracle_sample(inp, budget_s=max(0.5, args.cpu_budget / 10))
            steps.append(v)
        val = statistics.mean(steps[args.warmup:])
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": inp.token_heads / val * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    ms, times, launches, e2e, clocks = run_ours(args, rank, world, inp, peaks)
    value = world * inp.token_heads / (ms / 1e3)
    tflops = flops / (ms * 1e-3) / 1e12
    nbytes = bytes_per_launch(inp)
    gbs = nbytes / (ms * 1e-3) / 1e9
    roof = roofline_bound(flops, nbytes, ms, peaks)
    roof.update({"traffic": recorded_traffic(args.workload), "peak_source": peaks["source"],
                 "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
                 "kernel": kernel_name(inp),
                 "launch_ms_mean": ms, "launch_ms_min": min(times)})
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if inp.q.dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded N(0,1) q,k,v with unit-norm q,k; N(0,0.02^2) weights)",
            "config": config, "tflops": tflops,
            "tflops_frac_of_bf16_peak": tflops / peaks["bf16_tflops"], "hbm_gbs": gbs,
            "roofline": roof, "gpu_launches": launches, "clocks": clocks}
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        v, threads, desc = oracle_sample(inp, args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
