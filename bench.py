"""Benchmark of resident-prefix replay attention (forward + backward).

One step = one replay of the response through the whole hot path with
the prompt already resident in HBM: write the response's K/V pages, then
for every response block (last block first) the forward partials, the
LSE merge and the backward (D, dQ over prompt+response, dQ reduction,
response-only dK/dV).  The prompt capture happens once, before timing.

Default workload: the 2M-position one (P = 2,093,056 prompt keys, R = 4096
response rows, 32 query heads / 8 kv heads, head_dim 128, pages of 256
shuffled, 8 prompt shards, 0.1% of prompt keys x8).  Prompt K/V are 8.6 GB
of bf16, far larger than L2, so no L2 flush is needed between steps.

Prints one JSON line.  ``--impl reference`` times the CPU fp64 oracle on a
bounded sample of the same workload instead (host cores only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from resident_prefix_attention_gb300 import workloads as W  # noqa: E402

METRIC = ("response-replay attention fwd+bwd TFLOP/s at 2M-pos prefix; "
          "% of bf16 peak")


def metric_for(cfg) -> str:
    """The headline metric names the 2M workload; other workloads name
    their own prefix length."""
    if cfg.name == "2M":
        return METRIC
    if is_latent(cfg):
        return (f"latent-page replay attention fwd+bwd TFLOP/s, {cfg.name} "
                f"workload ({cfg.P}-pos prefix, d_c={cfg.d_c}, "
                f"d_r={cfg.d_r}); % of bf16 peak")
    return (f"response-replay attention fwd+bwd TFLOP/s, {cfg.name} workload "
            f"({cfg.P}-pos prefix); % of bf16 peak")
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
                "clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


# ------------------------------------------------------------------ flops
def block_list(R: int, blocks: int):
    base = R // blocks
    out = []
    for b in range(blocks):
        n = base if b < blocks - 1 else R - base * (blocks - 1)
        out.append((b * base, n))
    return list(reversed(out))


def block_flops(P, pos0, n, Hq, d):
    """Algorithmic flops of one block: forward 4d(pairs), backward
    2d(3 prompt pairs + 5 response pairs), per query head."""
    pairs_p = n * P
    pairs_r = n * pos0 + n * (n + 1) // 2
    fwd = 4 * d * (pairs_p + pairs_r) * Hq
    bwd = 2 * d * (3 * pairs_p + 5 * pairs_r) * Hq
    dq_kernel = 2 * d * 3 * (pairs_p + pairs_r) * Hq
    return fwd, bwd, dq_kernel


def latent_step_flops(cfg, R):
    """Latent pages, per query head: forward 2(d_l + d_c) per visible pair;
    backward 2(2 d_l + d_c) per pair (S, dP, dq~) plus 2(d_l + d_c) per
    response pair (the key and value sides of the latent-row gradient)."""
    dl, dc = cfg.d_l, cfg.d_c
    tot = {"fwd": 0, "bwd": 0, "dq": 0}
    for pos0, n in block_list(R, cfg.blocks):
        pairs = n * cfg.P + n * pos0 + n * (n + 1) // 2
        pairs_r = n * pos0 + n * (n + 1) // 2
        tot["fwd"] += 2 * (dl + dc) * pairs * cfg.Hq
        tot["dq"] += 2 * (2 * dl + dc) * pairs * cfg.Hq
        tot["bwd"] += (2 * (2 * dl + dc) * pairs +
                       2 * (dl + dc) * pairs_r) * cfg.Hq
    return tot


def side_bytes(cfg, R):
    """Algorithmic bytes per launch of the bandwidth-bound kernels of one
    block (one block per step in the benchmarked workloads)."""
    Hkv, d, Hq, S1 = cfg.Hkv, cfg.d, cfg.Hq, cfg.shards + 1
    rows = R * Hq
    return {
        # read k, v and write both pages, per (token, kv head)
        "capture": 4 * cfg.P * Hkv * d * 2,
        "write_pages": 4 * R * Hkv * d * 2,
        # partials (m, l, O_s) read, O and lse written
        "lse_merge": rows * (S1 * (4 * d + 8) + 4 * d + 4),
        # O (fp32) and dO (bf16) read, D written
        "bwd_preprocess": rows * (6 * d + 4),
        # 2S+1 slices read (the dQ pass splits prompt shards in halves),
        # dQ read and written
        "dq_reduce": rows * d * 4 * (2 * cfg.shards + 1 + 2),
    }


def step_flops(cfg, R):
    tot = {"fwd": 0, "bwd": 0, "dq": 0}
    for pos0, n in block_list(R, cfg.blocks):
        f, b, q = block_flops(cfg.P, pos0, n, cfg.Hq, cfg.d)
        tot["fwd"] += f
        tot["bwd"] += b
        tot["dq"] += q
    return tot


# ------------------------------------------------------------------ peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16": d["bf16_tflops"],
                "bf16_sustained": d["bf16_tflops_sustained"],
                "hbm": d["hbm_gbs"], "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0,
            "source": "fallback"}


# Dense bf16 rate of one SM's tensor core: an M=128, N=256, K=16 tcgen05
# product every 128 cycles (measured by the issue-rate probe summarised in
# profiles/mma_rate.md).
TENSOR_FLOP_PER_CLK_SM = 8192
NOMINAL_DENSE_BF16_TFLOPS = 2250.0


def num_sms() -> int:
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(0).multi_processor_count
    return 152


def tensor_peaks(clocks):
    """The tensor core's dense bf16 rate (TFLOP/s) at the SM's maximum clock
    and at the median clock sampled during the timed region."""
    sms = num_sms()
    mx = (clocks or {}).get("sm_max_mhz") or 2070.0
    med = (clocks or {}).get("sm_mhz") or mx
    rate = TENSOR_FLOP_PER_CLK_SM * sms * 1e6 / 1e12
    return {"at_max_clock": rate * mx, "at_sampled_clock": rate * med,
            "sms": sms, "max_mhz": mx, "sampled_mhz": med}


def peak_pcts(value, peaks, clocks):
    """The step's rate as a percentage of each bf16 reference: the tensor
    core's own rate at the maximum and at the sampled clock, NVIDIA's nominal
    dense figure, and the cuBLAS matmul rates measured on this machine (a
    library rate: a good kernel can exceed it)."""
    tp = tensor_peaks(clocks)
    return {
        "pct_tensor_peak_max_clock": 100 * value / tp["at_max_clock"],
        "pct_tensor_peak_sampled_clock": 100 * value / tp["at_sampled_clock"],
        "pct_nominal_dense_bf16": 100 * value / NOMINAL_DENSE_BF16_TFLOPS,
        "pct_bf16_peak_burst": 100 * value / peaks["bf16"],
        "pct_bf16_peak_sustained": 100 * value / peaks["bf16_sustained"],
        "tensor_peak_tflops_max_clock": tp["at_max_clock"],
        "tensor_peak_tflops_sampled_clock": tp["at_sampled_clock"],
    }


def tensor_roofline(dom, achieved, peaks, clocks, traffic):
    """Roofline of a tensor-bound kernel: `peak`/`frac` against the measured
    sustained cuBLAS rate, `frac_at_clock` against the tensor core's rate at
    the sampled SM clock, `frac_max_clock` at the maximum clock."""
    tp = tensor_peaks(clocks)
    peak = peaks["bf16_sustained"]
    return {"bound": "tensor", "kernel": dom, "achieved": achieved,
            "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_kind": f"bf16 sustained cuBLAS rate ({peaks['source']})",
            "frac_at_clock": achieved / tp["at_sampled_clock"],
            "frac_max_clock": achieved / tp["at_max_clock"],
            "tensor_peak_at_clock": tp["at_sampled_clock"],
            "tensor_peak_max_clock": tp["at_max_clock"],
            "traffic": traffic}


L2_BYTES = 129 * 2 ** 20


def is_latent(cfg) -> bool:
    return isinstance(cfg, W.LatentConfig)


def l2_note(cfg) -> str:
    """How the timed region treats L2: every step streams the whole prompt
    K/V, so when that is larger than L2 no flush is needed."""
    kv = (cfg.P * cfg.d_l * 2 if is_latent(cfg)
          else 2 * cfg.P * cfg.Hkv * cfg.d * 2)
    if kv > L2_BYTES:
        return f"inputs larger than L2 ({kv / 1e9:.2f} GB prompt K/V); no flush"
    return (f"prompt K/V ({kv / 1e6:.1f} MB) fits in L2 and is not flushed: "
            "a warm-cache figure")


def traffic_record(kernel: str):
    """dram bytes per launch from a committed ncu summary, valid only while
    the kernel's source is unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for name in rec["sources"]:
        src = os.path.join(ROOT, "resident_prefix_attention_gb300", "csrc",
                           name)
        with open(src, "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec["source_sha256"]:
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader",
                 "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm = float(f[1].split()[0])
                mx = float(f[2].split()[0])
            except ValueError:
                continue
            sms.append(sm)
            maxs.append(mx)
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sms:
            return None
        loaded = [s for s in sms if s > 0.5 * max(sms)] or sms
        return {"sm_mhz": statistics.median(loaded),
                "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------ dist
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU leg
def cpu_sample(cfg, n_pos: int, seed: int = 0):
    """Time the oracle on one kv head's sampled query rows of the workload.

    Inputs of one kv head are drawn on the CPU with the workload's
    distributions (prompt keys with the 0.1% x8 outliers).  Returns
    (flops, seconds, description): flops are the rows' forward + dQ
    algorithmic flops, 10 d per visible key.
    """
    import numpy as np
    import oracle
    g = torch.Generator().manual_seed(seed)
    Hq, Hkv, d, P, R = cfg.Hq, cfg.Hkv, cfg.d, cfg.P, cfg.R
    G = Hq // Hkv
    kp = torch.randn(P, 1, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(P, 1, d, generator=g).to(torch.bfloat16)
    n_out = int(round(cfg.outlier_frac * P))
    if n_out:
        idx = torch.randperm(P, generator=g)[:n_out]
        kp[idx] = kp[idx] * 8
    kr = torch.randn(R, 1, d, generator=g).to(torch.bfloat16)
    vr = torch.randn(R, 1, d, generator=g).to(torch.bfloat16)
    pos = torch.randperm(R, generator=g)[:n_pos].tolist()
    q = torch.randn(R, G, d, generator=g).to(torch.bfloat16)
    dO = torch.randn(R, G, d, generator=g).to(torch.bfloat16)
    rows = [p for p in pos for _ in range(G)]
    heads = [h for _ in pos for h in range(G)]
    t0 = time.perf_counter()
    oracle.attention_rows(q, kp, vp, kr, vr, dO, rows, heads, 0, cfg.scale)
    dt = time.perf_counter() - t0
    keys = sum(P + p + 1 for p in rows)
    flops = 10 * d * keys
    desc = (f"{len(rows)} query rows ({n_pos} positions x {G} heads of one "
            f"kv head) against all {P} prompt keys + causal response keys; "
            f"forward + dQ")
    return flops, dt, desc


def latent_cpu_sample(cfg, n_pos: int, seed: int = 0):
    """Time the latent oracle on sampled query rows of the latent workload
    (all Hq heads of n_pos positions against every prompt latent row).
    Returns (flops, seconds, description), flops = forward + dq~ of those
    rows: 2(d_l + d_c) + 2(2 d_l + d_c) per visible key."""
    import oracle.latent as OL
    g = torch.Generator().manual_seed(seed)
    P, R, Hq, dl, dc = cfg.P, cfg.R, cfg.Hq, cfg.d_l, cfg.d_c
    lp = torch.randn(P, dl, generator=g).to(torch.bfloat16)
    n_out = int(round(cfg.outlier_frac * P))
    if n_out:
        idx = torch.randperm(P, generator=g)[:n_out]
        lp[idx, dc:] = lp[idx, dc:] * 8
    lr = torch.randn(R, dl, generator=g).to(torch.bfloat16)
    pos = torch.randperm(R, generator=g)[:n_pos].tolist()
    q = torch.randn(R, Hq, dl, generator=g).to(torch.bfloat16)
    dO = torch.randn(R, Hq, dc, generator=g).to(torch.bfloat16)
    rows = [p for p in pos for _ in range(Hq)]
    heads = [h for _ in pos for h in range(Hq)]
    t0 = time.perf_counter()
    OL.latent_rows(q, lp, lr, dO, rows, heads, 0, cfg.scale, dc)
    dt = time.perf_counter() - t0
    keys = sum(P + p + 1 for p in rows)
    flops = (2 * (dl + dc) + 2 * (2 * dl + dc)) * keys
    desc = (f"{len(rows)} query rows ({n_pos} positions x {Hq} heads) against "
            f"all {P} prompt latent rows + causal response rows; forward + "
            f"dq~")
    return flops, dt, desc


def reference_arm(args, cfg):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    n_pos = args.ref_positions
    cores = os.cpu_count()
    sample = latent_cpu_sample if is_latent(cfg) else cpu_sample
    for _ in range(args.warmup):
        sample(cfg, n_pos)
    tot_f, tot_t = 0, 0.0
    desc = ""
    for i in range(args.steps):
        f, t, desc = sample(cfg, n_pos, seed=i)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": metric_for(cfg), "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "P": cfg.P, "R": cfg.R,
                   "Hq": cfg.Hq, "Hkv": 1 if is_latent(cfg) else cfg.Hkv,
                   "head_dim": cfg.d_l if is_latent(cfg) else cfg.d,
                   "sample_positions": n_pos},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def gpu_arm(args, cfg):
    from resident_prefix_attention_gb300 import lsr
    from resident_prefix_attention_gb300.replay import ReplaySession
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.make_workload(cfg, seed=args.seed + rank, device=str(dev))
    resp = wl.responses[0]
    R = resp.q.shape[0]
    sess = ReplaySession(wl.page_table.numel(), cfg.Hkv, cfg.page_size, cfg.d,
                         wl.page_table, device=str(dev))
    # resident capture (A0): timed once, outside the metric
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record()
    sess.write(wl.k_prompt, wl.v_prompt, 0)
    c1.record()
    torch.cuda.synchronize()
    capture_ms = c0.elapsed_time(c1)
    del wl.k_prompt, wl.v_prompt
    q, dO, kr, vr = resp.q, resp.dO, resp.k, resp.v
    dq = torch.zeros(R, cfg.Hq, cfg.d, dtype=torch.float32, device=dev)
    dk, dv = sess.grad_pages(R)
    o = torch.empty(R, cfg.Hq, cfg.d, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.Hq, R, dtype=torch.float32, device=dev)
    nws = lsr.lsr_replay_workspace_size(cfg.shards, cfg.Hq, R, cfg.blocks,
                                        cfg.d)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        sess.write(kr, vr, cfg.P)
        sess.replay_response(q, dO, cfg.P, cfg.blocks, cfg.shards, cfg.scale,
                             dq, dk, dv, o=o, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert sess.device_status() == 0, "device status word set"
    fl = step_flops(cfg, R)
    total_flops = fl["fwd"] + fl["bwd"]

    # ---- device-resident timed region
    lsr.lsr_profile_set(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = ev0.elapsed_time(ev1) / args.steps
    kern = {}
    launches = 0
    for k in range(lsr.LSR_K_COUNT):
        n, t = lsr.lsr_profile_read(k)
        launches += n
        if n:
            kern[lsr.lsr_kernel_name(k)] = (n, t)
    lsr.lsr_profile_set(False)
    ms_max = max_over_ranks(ms, world)
    value = world * total_flops / (ms_max * 1e-3) / 1e12

    # ---- dominant kernel roofline (tensor-bound contraction)
    peaks = measured_peaks()
    n_dq, t_dq = kern["attn_bwd_dq"]
    n_fw, t_fw = kern["attn_fwd"]
    if t_dq >= t_fw:
        dom, n_dom, t_dom, fl_dom = "attn_bwd_dq", n_dq, t_dq, fl["dq"]
    else:
        dom, n_dom, t_dom, fl_dom = "attn_fwd", n_fw, t_fw, fl["fwd"]
    per_launch_flops = fl_dom / cfg.blocks
    achieved = per_launch_flops / (t_dom / n_dom * 1e-3) / 1e12
    clocks = clk.summary()
    roofline = tensor_roofline(dom, achieved, peaks, clocks,
                               traffic_record(dom))
    kernels_ms = {k: round(t / max(n, 1), 4) for k, (n, t) in kern.items()}
    per_step = {k: t / args.steps for k, (n, t) in kern.items()}
    phases = {
        "fwd_ms": per_step.get("attn_fwd", 0) + per_step.get("lse_merge", 0),
        "bwd_ms": sum(per_step.get(k, 0) for k in (
            "bwd_preprocess", "attn_bwd_dq", "dq_reduce", "attn_bwd_dkdv")),
        "capture_ms": capture_ms,
        "capture_gbs": side_bytes(cfg, R)["capture"] / (capture_ms * 1e-3)
        / 1e9,
    }
    side = {}
    for k, nbytes in side_bytes(cfg, R).items():
        if k in kern:
            n, t = kern[k]
            side[k] = {"ms": round(t / n, 4),
                       "gbs": round(nbytes / (t / n * 1e-3) / 1e9, 1)}

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        hdo = dO.cpu().pin_memory()
        hkr = kr.cpu().pin_memory()
        hvr = vr.cpu().pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        hdq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
        hdk = torch.empty(dk.shape, dtype=dk.dtype).pin_memory()
        hdv = torch.empty(dv.shape, dtype=dv.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hdo, hkr, hvr))
        d2h = sum(t.numel() * t.element_size()
                  for t in (ho, hlse, hdq, hdk, hdv))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            dO.copy_(hdo, non_blocking=True)
            kr.copy_(hkr, non_blocking=True)
            vr.copy_(hvr, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            hdq.copy_(dq, non_blocking=True)
            hdk.copy_(dk, non_blocking=True)
            hdv.copy_(dv, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ems = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world)
        e2e = {"value": world * total_flops / (ems * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems}
    assert sess.device_status() == 0, "device status word set"

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, t, desc = cpu_sample(cfg, args.cpu_positions)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
               "seconds": round(t, 2)}

    if rank == 0:
        line = {
            "metric": metric_for(cfg), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "P": cfg.P, "R": R,
                       "blocks": cfg.blocks, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                       "head_dim": cfg.d, "page_size": cfg.page_size,
                       "shards": cfg.shards, "flops_per_step": total_flops,
                       **peak_pcts(value, peaks, clocks),
                       "l2": l2_note(cfg),
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline, "kernel_ms_per_launch": kernels_ms,
            "phases": phases, "side_kernels": side,
            "gpu_launches": launches, "clocks": clocks,
            "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def gpu_latent_arm(args, cfg):
    """Latent-page replay: one resident prompt of latent rows, one response
    replayed in reverse blocks (response latent write + forward, merge and
    backward of every block per step)."""
    from resident_prefix_attention_gb300 import lsr
    from resident_prefix_attention_gb300.replay import LatentReplaySession
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.make_latent_workload(cfg, seed=args.seed + rank, device=str(dev))
    R = cfg.R
    sess = LatentReplaySession(wl.page_table.numel(), cfg.page_size,
                               wl.page_table, cfg.d_c, cfg.d_r,
                               device=str(dev))
    sess.write(wl.lat_prompt, 0)                      # resident capture
    torch.cuda.synchronize()
    del wl.lat_prompt
    q, dO, lr = wl.q, wl.dO, wl.lat_resp
    dq = torch.zeros(R, cfg.Hq, cfg.d_l, dtype=torch.float32, device=dev)
    dlat = sess.grad_pages(R)
    o = torch.empty(R, cfg.Hq, cfg.d_c, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.Hq, R, dtype=torch.float32, device=dev)
    nws = lsr.lsr_latent_replay_workspace_size(cfg.shards, cfg.Hq, R,
                                               cfg.blocks)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        sess.write(lr, cfg.P)
        sess.replay_response(q, dO, cfg.P, cfg.blocks, cfg.shards, cfg.scale,
                             dq, dlat, o=o, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert sess.device_status() == 0, "device status word set"
    fl = latent_step_flops(cfg, R)
    total_flops = fl["fwd"] + fl["bwd"]

    lsr.lsr_profile_set(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = ev0.elapsed_time(ev1) / args.steps
    kern = {}
    launches = 0
    for k in range(lsr.LSR_K_COUNT):
        n, t = lsr.lsr_profile_read(k)
        launches += n
        if n:
            kern[lsr.lsr_kernel_name(k)] = (n, t)
    lsr.lsr_profile_set(False)
    ms_max = max_over_ranks(ms, world)
    value = world * total_flops / (ms_max * 1e-3) / 1e12

    peaks = measured_peaks()
    n_dq, t_dq = kern["latent_bwd_dq"]
    n_fw, t_fw = kern["attn_fwd"]
    if t_dq >= t_fw:
        dom, n_dom, t_dom, fl_dom = "latent_bwd_dq", n_dq, t_dq, fl["dq"]
    else:
        dom, n_dom, t_dom, fl_dom = "attn_fwd", n_fw, t_fw, fl["fwd"]
    achieved = (fl_dom / cfg.blocks) / (t_dom / n_dom * 1e-3) / 1e12
    # DRAM bytes per launch are recorded for the 2M-position latent
    # workload only (key "<kernel>_latent" in profiles/ncu_traffic.json)
    traffic = traffic_record(dom + "_latent") if cfg.name == "latent" else None
    clocks = clk.summary()
    roofline = tensor_roofline(dom, achieved, peaks, clocks, traffic)
    kernels_ms = {k: round(t / max(n, 1), 4) for k, (n, t) in kern.items()}

    e2e = None
    if not args.no_e2e:
        hq, hdo, hlr = (t.cpu().pin_memory() for t in (q, dO, lr))
        outs = (o, lse, dq, dlat)
        hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory()
                for t in outs]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hdo, hlr))
        d2h = sum(t.numel() * t.element_size() for t in hout)

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            dO.copy_(hdo, non_blocking=True)
            lr.copy_(hlr, non_blocking=True)
            step()
            for h, t in zip(hout, outs):
                h.copy_(t, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ems = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world)
        e2e = {"value": world * total_flops / (ems * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems}
    assert sess.device_status() == 0, "device status word set"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, t, desc = latent_cpu_sample(cfg, args.latent_cpu_positions)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
               "seconds": round(t, 2)}

    if rank == 0:
        line = {
            "metric": metric_for(cfg), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "P": cfg.P, "R": R,
                       "blocks": cfg.blocks, "Hq": cfg.Hq,
                       "latent_dim": cfg.d_c, "rope_dim": cfg.d_r,
                       "page_size": cfg.page_size, "shards": cfg.shards,
                       "flops_per_step": total_flops,
                       **peak_pcts(value, peaks, clocks),
                       "l2": l2_note(cfg),
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline, "kernel_ms_per_launch": kernels_ms,
            "gpu_launches": launches, "clocks": clocks,
            "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def gpu_latent_group_arm(args, cfg):
    """The latent group workload: one resident prompt of latent rows and G
    responses, replayed serially (--concurrent 1, one response slot reused)
    or K at a time in one forward and one backward launch (--concurrent K,
    K response slots).  A step is one whole group; reports time per group
    and peak allocated bytes."""
    from resident_prefix_attention_gb300 import lsr
    from resident_prefix_attention_gb300.replay import LatentReplaySession
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    grp = W.make_latent_group(cfg, seed=args.seed + rank, device=str(dev))
    lengths = [r.q.shape[0] for r in grp.responses]
    Rmax = max(lengths)
    K = max(1, args.concurrent)
    ps = cfg.page_size
    slot = -(-Rmax // ps)
    table = grp.page_table
    if K > 1:
        extra = torch.arange(table.numel(), table.numel() + (K - 1) * slot,
                             dtype=torch.int32, device=dev)
        table = torch.cat([table, extra])
    sess = LatentReplaySession(table.numel(), ps, table, cfg.d_c, cfg.d_r,
                               device=str(dev))
    sess.write(grp.lat_prompt, 0)
    torch.cuda.synchronize()
    del grp.lat_prompt
    stream = torch.cuda.current_stream()
    if K == 1:
        dq = torch.zeros(Rmax, cfg.Hq, cfg.d_l, dtype=torch.float32,
                         device=dev)
        dlat = sess.grad_pages(Rmax)
        o = torch.empty(Rmax, cfg.Hq, cfg.d_c, dtype=torch.float32,
                        device=dev)
        lse = torch.empty(cfg.Hq * Rmax, dtype=torch.float32, device=dev)
        ws = torch.empty(lsr.lsr_latent_replay_workspace_size(
            cfg.shards, cfg.Hq, Rmax, 1), dtype=torch.uint8, device=dev)

        def group():
            for r in grp.responses:
                R = r.q.shape[0]
                sess.write(r.lat, cfg.P)
                sess.replay_response(r.q, r.dO, cfg.P, 1, cfg.shards,
                                     cfg.scale, dq[:R], dlat, o=o[:R],
                                     lse=lse[:cfg.Hq * R].view(cfg.Hq, R),
                                     workspace=ws)
    else:
        chunks = [list(range(i, min(i + K, cfg.G)))
                  for i in range(0, cfg.G, K)]
        page0 = [cfg.P // ps + j * slot for j in range(K)]

        def group():
            for ch in chunks:
                for j, k in enumerate(ch):
                    sess.write(grp.responses[k].lat, page0[j] * ps)
                sess.replay_group([grp.responses[k].q for k in ch],
                                  [grp.responses[k].dO for k in ch],
                                  page0[:len(ch)], cfg.P, cfg.shards,
                                  cfg.scale)

    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    for _ in range(args.warmup):
        group()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated()
    assert sess.device_status() == 0, "device status word set"
    flops = 0
    for R in lengths:
        fl = latent_step_flops(cfg, R)
        flops += fl["fwd"] + fl["bwd"]
    lsr.lsr_profile_set(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            group()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    launches = sum(lsr.lsr_profile_read(k)[0] for k in range(lsr.LSR_K_COUNT))
    lsr.lsr_profile_set(False)
    assert sess.device_status() == 0, "device status word set"
    value = world * flops / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    if rank == 0:
        clocks = clk.summary()
        print(json.dumps({
            "metric": metric_for(cfg), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "P": cfg.P, "G": cfg.G,
                       "concurrent": K, "lengths": lengths, "Hq": cfg.Hq,
                       "latent_dim": cfg.d_c, "rope_dim": cfg.d_r,
                       "flops_per_group": flops,
                       **peak_pcts(value, peaks, clocks),
                       "step": "one group", "l2": l2_note(cfg)},
            "time_per_group_ms": ms, "peak_allocated_bytes": peak,
            "gpu_launches": launches, "clocks": clocks,
        }), flush=True)


def gpu_group_arm(args, cfg):
    """The group workload: one resident prompt, G responses replayed
    serially, gradients accumulated in one window.  A step is one whole
    group.  Reports time per group and peak allocated bytes, and the peak
    growth from G=2 to G=8 (the explainer's "G is a schedule" measure)."""
    from resident_prefix_attention_gb300 import lsr
    from resident_prefix_attention_gb300.replay import ReplaySession
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.make_workload(cfg, seed=args.seed + rank, device=str(dev))
    lengths = [r.q.shape[0] for r in wl.responses]
    Rmax = max(lengths)
    K = max(1, args.concurrent)
    slot = -(-Rmax // cfg.page_size)               # pages per response slot
    table = wl.page_table
    if K > 1:                                      # K response-page slots
        extra = torch.arange(table.numel(), table.numel() + (K - 1) * slot,
                             dtype=torch.int32, device=dev)
        table = torch.cat([table, extra])
    sess = ReplaySession(table.numel(), cfg.Hkv, cfg.page_size, cfg.d, table,
                         device=str(dev))
    sess.write(wl.k_prompt, wl.v_prompt, 0)
    torch.cuda.synchronize()
    del wl.k_prompt, wl.v_prompt
    if K > 1:
        return group_concurrent(args, cfg, wl, sess, K, slot, lengths, world,
                                rank, local, dev)
    # accumulation window (update-boundary state) and replay temporaries,
    # sized once for the longest response
    dq = torch.zeros(Rmax, cfg.Hq, cfg.d, dtype=torch.float32, device=dev)
    dk, dv = sess.grad_pages(Rmax)
    o = torch.empty(Rmax, cfg.Hq, cfg.d, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.Hq * Rmax, dtype=torch.float32, device=dev)
    nws = lsr.lsr_replay_workspace_size(cfg.shards, cfg.Hq, Rmax, 1, cfg.d)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def group(G):
        for resp in wl.responses[:G]:
            R = resp.q.shape[0]
            sess.write(resp.k, resp.v, cfg.P)
            sess.replay_response(resp.q, resp.dO, cfg.P, 1, cfg.shards,
                                 cfg.scale, dq[:R], dk, dv, o=o[:R],
                                 lse=lse[:cfg.Hq * R].view(cfg.Hq, R),
                                 workspace=ws)

    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    group(2)
    torch.cuda.synchronize()
    peak2 = torch.cuda.max_memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    group(cfg.G)
    torch.cuda.synchronize()
    peak8 = torch.cuda.max_memory_allocated()
    for _ in range(max(0, args.warmup - 1)):
        group(cfg.G)
    assert sess.device_status() == 0, "device status word set"
    flops = 0
    for R in lengths:
        f = step_flops(cfg, R)
        flops += f["fwd"] + f["bwd"]
    lsr.lsr_profile_set(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            group(cfg.G)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    launches = sum(lsr.lsr_profile_read(k)[0] for k in range(lsr.LSR_K_COUNT))
    lsr.lsr_profile_set(False)
    assert sess.device_status() == 0, "device status word set"
    if rank == 0:
        peaks = measured_peaks()
        value = world * flops / (ms * 1e-3) / 1e12
        clocks = clk.summary()
        print(json.dumps({
            "metric": metric_for(cfg), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "P": cfg.P, "G": cfg.G,
                       "lengths": lengths, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                       "head_dim": cfg.d, "page_size": cfg.page_size,
                       "shards": cfg.shards, "flops_per_group": flops,
                       **peak_pcts(value, peaks, clocks),
                       "step": "one group of G serial replays",
                       "l2": l2_note(cfg)},
            "time_per_group_ms": ms,
            "peak_allocated_bytes_G2": peak2,
            "peak_allocated_bytes_G8": peak8,
            "peak_growth_G2_to_G8_bytes": peak8 - peak2,
            "gpu_launches": launches, "clocks": clocks,
        }), flush=True)


def group_concurrent(args, cfg, wl, sess, K, slot, lengths, world, rank,
                     local, dev):
    """The group workload with K responses per launch (lsr_replay_group):
    the responses of a batch occupy K response-page slots and K sets of
    live replay buffers, so peak memory grows with K."""
    from resident_prefix_attention_gb300 import lsr
    P0 = cfg.P // cfg.page_size
    batches = [list(range(i, min(i + K, cfg.G))) for i in range(0, cfg.G, K)]
    plans = []
    for b in batches:
        R = [lengths[i] for i in b]
        row0 = lsr.lsr_group_rows(cfg.Hq, cfg.Hkv, R)
        total = row0[-1]
        q = torch.zeros(total, cfg.Hq, cfg.d, dtype=torch.bfloat16, device=dev)
        dO = torch.zeros_like(q)
        for j, i in enumerate(b):
            q[row0[j]:row0[j] + R[j]] = wl.responses[i].q
            dO[row0[j]:row0[j] + R[j]] = wl.responses[i].dO
        npg = [-(-r // cfg.page_size) for r in R]
        plans.append(dict(b=b, R=R, q=q, dO=dO, total=total,
                          page0=[P0 + j * slot for j in range(len(b))],
                          gpage0=[sum(npg[:j]) for j in range(len(b))],
                          ngp=sum(npg)))
    tmax = max(pl["total"] for pl in plans)
    gmax = max(pl["ngp"] for pl in plans)
    o = torch.empty(tmax * cfg.Hq * cfg.d, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.Hq * tmax, dtype=torch.float32, device=dev)
    dq = torch.zeros(tmax * cfg.Hq * cfg.d, dtype=torch.float32, device=dev)
    gshape = (gmax, cfg.Hkv, cfg.page_size, cfg.d)
    dk = torch.zeros(gshape, dtype=torch.float32, device=dev)
    dv = torch.zeros(gshape, dtype=torch.float32, device=dev)
    ws = torch.empty(lsr.lsr_group_workspace_size(cfg.shards, cfg.Hq, tmax,
                                                  cfg.d),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def group():
        for pl in plans:
            for j, i in enumerate(pl["b"]):
                r = wl.responses[i]
                sess.write(r.k, r.v, pl["page0"][j] * cfg.page_size)
            t = pl["total"]
            lsr.lsr_replay_group(
                sess.pool, pl["R"], pl["page0"], pl["gpage0"], pl["q"],
                pl["dO"], cfg.P, sess.page_table, cfg.shards, cfg.scale,
                o[:t * cfg.Hq * cfg.d].view(t, cfg.Hq, cfg.d),
                lse[:cfg.Hq * t].view(cfg.Hq, t),
                dq[:t * cfg.Hq * cfg.d].view(t, cfg.Hq, cfg.d),
                dk[:pl["ngp"]], dv[:pl["ngp"]], ws)

    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    for _ in range(max(1, args.warmup)):
        group()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated()
    assert sess.device_status() == 0, "device status word set"
    flops = 0
    for R in lengths:
        f = step_flops(cfg, R)
        flops += f["fwd"] + f["bwd"]
    lsr.lsr_profile_set(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            group()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    launches = sum(lsr.lsr_profile_read(k)[0] for k in range(lsr.LSR_K_COUNT))
    lsr.lsr_profile_set(False)
    if rank == 0:
        peaks = measured_peaks()
        value = world * flops / (ms * 1e-3) / 1e12
        clocks = clk.summary()
        print(json.dumps({
            "metric": metric_for(cfg), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "P": cfg.P, "G": cfg.G,
                       "concurrent": K, "lengths": lengths,
                       "flops_per_group": flops,
                       **peak_pcts(value, peaks, clocks),
                       "step": f"one group, {len(plans)} launches of up to "
                               f"{K} responses",
                       "l2": l2_note(cfg)},
            "time_per_group_ms": ms, "peak_allocated_bytes": peak,
            "gpu_launches": launches, "clocks": clocks,
        }), flush=True)


def gpu_score_arm(args, cfg):
    """Graph-free scoring of the last `--score-rows` response positions
    against the resident prompt (forward + merge only; shard count chosen
    to fill the GPU).  With few rows the forward reads the prompt's K/V once
    and is bound by HBM bandwidth, reported as GB/s."""
    from resident_prefix_attention_gb300 import lsr
    from resident_prefix_attention_gb300.replay import (LatentReplaySession,
                                                        ReplaySession)
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    latent = is_latent(cfg)
    n = args.score_rows
    if latent:
        wl = W.make_latent_workload(cfg, seed=args.seed + rank,
                                    device=str(dev))
        R = cfg.R
        sess = LatentReplaySession(wl.page_table.numel(), cfg.page_size,
                                   wl.page_table, cfg.d_c, cfg.d_r,
                                   device=str(dev))
        sess.write(wl.lat_prompt, 0)
        sess.write(wl.lat_resp, cfg.P)
        del wl.lat_prompt
        q = wl.q[R - n:].contiguous()
        d_out, d_in, row_bytes = cfg.d_c, cfg.d_l, cfg.d_l * 2
    else:
        wl = W.make_workload(cfg, seed=args.seed + rank, device=str(dev))
        resp = wl.responses[0]
        R = resp.q.shape[0]
        sess = ReplaySession(wl.page_table.numel(), cfg.Hkv, cfg.page_size,
                             cfg.d, wl.page_table, device=str(dev))
        sess.write(wl.k_prompt, wl.v_prompt, 0)
        sess.write(resp.k, resp.v, cfg.P)
        del wl.k_prompt, wl.v_prompt
        q = resp.q[R - n:].contiguous()
        d_out, d_in, row_bytes = cfg.d, cfg.d, cfg.Hkv * cfg.d * 2 * 2
    shards = lsr.lsr_score_shards(sess.pool, cfg.Hq, n, cfg.P)
    ws = torch.empty(lsr.lsr_score_workspace_size(shards, cfg.Hq, n, d_out),
                     dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        sess.score(q, cfg.P, R - n, shards, cfg.scale, ws)
    torch.cuda.synchronize()
    lsr.lsr_profile_set(True)
    stream = torch.cuda.current_stream()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            sess.score(q, cfg.P, R - n, shards, cfg.scale, ws)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    nf, tf = lsr.lsr_profile_read(lsr.LSR_K_ATTN_FWD)
    launches = sum(lsr.lsr_profile_read(k)[0] for k in range(lsr.LSR_K_COUNT))
    lsr.lsr_profile_set(False)
    assert sess.device_status() == 0, "device status word set"
    # algorithmic bytes of the forward launch: prompt and visible response
    # K/V (or latent rows) once, q, and the partial statistics written
    kv = (cfg.P + R) * row_bytes
    part = (shards + 1) * n * cfg.Hq * (d_out + 2) * 4
    fwd_bytes = kv + n * cfg.Hq * d_in * 2 + part
    achieved = fwd_bytes / (tf / nf * 1e-3) / 1e9
    peaks = measured_peaks()
    if rank == 0:
        print(json.dumps({
            "metric": ("graph-free scoring of the last response rows against "
                       "the resident 2M prompt (HBM GB/s of the forward)"
                       + (", latent pages" if latent else "")),
            "value": world * fwd_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "score_rows": n,
                       "shards": shards, "P": cfg.P, "Hq": cfg.Hq,
                       "Hkv": 1 if latent else cfg.Hkv, "head_dim": d_in,
                       "l2": l2_note(cfg)},
            "roofline": {"bound": "hbm", "kernel": "attn_fwd",
                         "achieved": achieved, "peak": peaks["hbm"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm"],
                         "traffic": None},
            "gpu_launches": launches, "clocks": clk.summary(),
        }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="2M",
                    choices=sorted(W.CONFIGS) + sorted(W.LATENT_CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # CPU oracle sample sizes: about 10-30 s of host work on a GB300 host
    ap.add_argument("--cpu-positions", type=int, default=96)
    ap.add_argument("--latent-cpu-positions", type=int, default=8)
    ap.add_argument("--ref-positions", type=int, default=2)
    ap.add_argument("--concurrent", type=int, default=1,
                    help="group workload: responses replayed per launch")
    ap.add_argument("--score-rows", type=int, default=0,
                    help="time graph-free scoring of this many rows instead")
    args = ap.parse_args()
    cfg = W.CONFIGS.get(args.config) or W.LATENT_CONFIGS[args.config]
    if args.impl == "reference":
        reference_arm(args, cfg)
    elif args.score_rows > 0:
        gpu_score_arm(args, cfg)
    elif is_latent(cfg) and cfg.G > 1:
        gpu_latent_group_arm(args, cfg)
    elif is_latent(cfg):
        gpu_latent_arm(args, cfg)
    elif args.config == "group":
        gpu_group_arm(args, cfg)
    else:
        gpu_arm(args, cfg)


if __name__ == "__main__":
    main()
