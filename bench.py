#!/usr/bin/env python
"""Benchmark of the exact shared-prompt attention layer (forward + backward).

A step is one forward and one backward of one attention layer on the packed
P + N*R layout (all rows of the hot path: forward, D preprocess, dK/dV with
the prompt reduction, dQ), with inputs resident in HBM.  Default workload:
32 query / 8 KV heads, d = 128, P = 32768, N = 16, R = 2048 (packed 65,536
rows), bf16 N(0,1) inputs from the seeded generator.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own
independent replica of the layer (weak scaling, no data-path collective); the
timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from shared_prompt_exact_dualkv_gb300 import synthetic  # noqa: E402

METRIC = "DualKV fwd+bwd ms and useful TFLOP/s (% of GB300 bf16 peak) per attn layer"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def align256(x: int) -> int:
    return (x + 255) // 256 * 256


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def blas_threads():
    """Threads of the BLAS that numpy calls (the oracle's matrix products):
    threadpoolctl if installed, else the OpenBLAS thread query of the loaded
    library, else None."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except ImportError:
        pass
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ln.split()[-1].startswith("/")})
    except OSError:
        return None
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads", "scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        # raw samples go to $BENCH_CLOCKS_DIR (default: the system temp dir); the
        # JSON line carries their summary
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != self.gpu_index:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of `x` over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job useful TFLOP/s: the units all ranks processed over the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def recorded_traffic(kernel: str, workload: str, deterministic: bool):
    """DRAM bytes per launch (read + write) from the committed ncu capture of
    this kernel at this workload, or None if there is none or the kernel's
    sources changed since it was taken."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.md")
    if deterministic or not os.path.exists(path):
        return None
    text = open(path).read()
    m_bytes = re.search(r"^dram_bytes_per_launch: (\d+)$", text, re.M)
    m_hash = re.search(r"^sources_sha256: ([0-9a-f]+)$", text, re.M)
    m_src = re.search(r"^sources: (.+)$", text, re.M)
    if not (m_bytes and m_hash and m_src):
        return None
    h = hashlib.sha256()
    for f in m_src.group(1).split():
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        with open(fp, "rb") as fh:
            h.update(fh.read())
    return int(m_bytes.group(1)) if h.hexdigest() == m_hash.group(1) else None


def end_to_end(args, D, w, x, dev, q, lse, k, v, ws, stream, det, world):
    """Same step through the C ABI with host buffers: every step copies its
    inputs from pinned host memory and its results (out, lse, dq, dk, dv) back.
    A ring of `args.e2e_buffers` device buffer sets lets the host-to-device
    copies (copy-in stream) run up to that many steps minus one ahead of the
    kernels, and the device-to-host copies (copy-out stream) trail them.  Two
    sets suffice while every copy runs at link speed; a deeper ring keeps the
    kernels fed through the occasional single copy that stalls for about
    100 ms on these hosts after sustained load.  Returns (ms per step, h2d
    bytes, d2h bytes)."""
    nb = max(2, args.e2e_buffers)
    hin = [t.pin_memory() for t in (x.q, x.k, x.v, x.dout)]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    bufs = []
    for b in range(nb):
        ins = [torch.empty_like(t, device=dev) for t in (x.q, x.k, x.v, x.dout)]
        outs = [torch.empty_like(q), torch.empty_like(lse), torch.empty_like(q), torch.empty_like(k),
                torch.empty_like(v)]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        bws = torch.empty_like(ws)
        bufs.append((ins, outs, hout, bws))
    d2h = sum(t.numel() * t.element_size() for t in bufs[0][2])
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {name: [torch.cuda.Event() for _ in range(nb)] for name in ("in_ready", "comp_done", "out_done")}

    def e2e_step(i):
        b = i % nb
        ins, outs, hout, bws = bufs[b]
        (eq, ek, ev_, edo), (eo, el, edq, edk, edv) = ins, outs
        with torch.cuda.stream(cin):
            if i >= nb:
                cin.wait_event(ev["comp_done"][b])   # step i-nb finished reading this input set
            for dst, src in zip(ins, hin):
                dst.copy_(src, non_blocking=True)
            ev["in_ready"][b].record(cin)
        stream.wait_event(ev["in_ready"][b])
        if i >= nb:
            stream.wait_event(ev["out_done"][b])     # step i-nb's results have left this output set
        D.dualkv_fwd(eq, ek, ev_, w.P, w.R_lens, eo, el, w.scale, stream)
        D.dualkv_bwd(eq, ek, ev_, eo, edo, el, w.P, w.R_lens, w.scale, det, bws, edq, edk, edv, stream=stream)
        ev["comp_done"][b].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(ev["comp_done"][b])
            for dst, src in zip(hout, outs):
                dst.copy_(src, non_blocking=True)
            ev["out_done"][b].record(cout)

    for i in range(nb):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    for i in range(args.steps):
        e2e_step(i)
    cout.wait_stream(stream)
    cout.wait_stream(cin)
    e1.record(cout)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    del bufs

    return e2e_ms, h2d, d2h


def layer_flops(shape: dict, rows: int, pairs_per_head: int) -> dict:
    """Useful flops of one decoder layer, forward + backward: the GEMMs (2 per
    multiply-add, three times over for forward, dX and dW) and the attention
    (14*d per unmasked pair per q-head)."""
    H, I = shape["hidden"], shape["inter"]
    nq, nk = shape["Hq"] * shape["d"], shape["Hkv"] * shape["d"]
    gemm = 3 * 2 * rows * (H * (nq + 2 * nk) + nq * H + H * 2 * I + I * H)
    att = 14 * shape["d"] * shape["Hq"] * pairs_per_head
    return {"gemm": float(gemm), "attention": float(att)}


def layer_leg(D, w, dev, stream):
    """One Qwen3-8B-shaped decoder layer (random weights), forward + backward
    through dualkv_layer_fwd/bwd, on the packed rows of the workload and on its
    replicated N(P+R) rows (every sequence its own causal group)."""
    shape = synthetic.LAYER_SHAPES["qwen3_8b"]
    cfg = D.layer_config(**shape)
    out = {"shape": "qwen3_8b", **{k: shape[k] for k in ("hidden", "Hq", "Hkv", "d", "inter")}}
    gen = torch.Generator(device=dev).manual_seed(11)
    weights = {}
    for n, sh in D.layer_weight_shapes(cfg).items():
        r = torch.randn(sh, device=dev, generator=gen)
        weights[n] = (1.0 + 0.1 * r if n.startswith("ln") else r / math.sqrt(sh[1])).to(torch.bfloat16)
    layouts = {"packed": ([(w.P, tuple(w.R_lens))], w.T, w.pairs_per_head()),
               "replicated": ([(w.P + int(r), ()) for r in w.R_lens], w.T_replicated,
                              w.pairs_per_head_replicated())}
    # The replicated rows are gathered from the packed ones (sequence i =
    # [prompt ; response i]).  A prompt row's dy is split evenly over the N
    # sequences (exact for N a power of two); the shares add up to the packed
    # dy, and no sequence gets all-zero rows, which would lower the power
    # draw and flatter the replicated timing.
    x_p = torch.randn((w.T, shape["hidden"]), device=dev, generator=gen).to(torch.bfloat16)
    dy_p = torch.randn((w.T, shape["hidden"]), device=dev, generator=gen).to(torch.bfloat16)
    offs = w.offsets
    rep_idx = torch.cat([torch.cat([torch.arange(w.P), torch.arange(offs[i], offs[i] + int(r))])
                         for i, r in enumerate(w.R_lens)]).to(dev)
    results = {}
    for name, (groups, rows, pairs) in layouts.items():
        if name == "packed":
            x, dy = x_p, dy_p
        else:
            x, dy = x_p[rep_idx], dy_p[rep_idx]
            share = (dy_p[:w.P].float() / w.N).to(torch.bfloat16)
            start = 0
            for r in w.R_lens:
                dy[start:start + w.P] = share
                start += w.P + int(r)
        layer = D.PackedLayer(cfg, weights, groups)
        y = torch.empty_like(x)
        dx = torch.empty_like(x)
        grads = {n: torch.empty(t.shape, dtype=torch.float32, device=dev) for n, t in weights.items()}

        def fwd():
            D.dualkv_layer_fwd(cfg, weights, x, groups, y, layer.workspace, stream)

        def bwd():
            D.dualkv_layer_bwd(cfg, weights, x, dy, groups, dx, grads, layer.workspace, stream)

        with torch.cuda.stream(stream):
            for _ in range(2):
                fwd()
                bwd()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        f_ms = b_ms = 0.0
        steps = 3
        for i in range(steps):
            ev[0].record(stream)
            fwd()
            ev[1].record(stream)
            bwd()
            ev[2].record(stream)
            torch.cuda.synchronize()
            f_ms += ev[0].elapsed_time(ev[1]) / steps
            b_ms += ev[1].elapsed_time(ev[2]) / steps
        st, site = D.dualkv_last_device_error(stream)
        if st != 0:
            raise RuntimeError(f"device error {st} at wait site {site}")
        fl = layer_flops(shape, rows, pairs)
        nbytes = layer.workspace.numel() + 4 * x.numel() * 2
        out[name] = {"rows": rows, "fwd_ms": f_ms, "bwd_ms": b_ms, "ms": f_ms + b_ms,
                     "gemm_tflop": fl["gemm"] / 1e12, "attention_tflop": fl["attention"] / 1e12,
                     "tflops": (fl["gemm"] + fl["attention"]) / ((f_ms + b_ms) * 1e-3) / 1e12,
                     "device_bytes": nbytes}
        if name == "packed":
            results["packed"] = (y, dx, grads)
        else:
            # scatter the replicated results back to the packed rows
            y_r = torch.empty_like(x_p, dtype=torch.float32)
            dx_r = torch.zeros_like(x_p, dtype=torch.float32)
            start = 0
            for i, r in enumerate(w.R_lens):
                r = int(r)
                seq_y, seq_dx = y[start:start + w.P + r].float(), dx[start:start + w.P + r].float()
                y_r[offs[i]:offs[i] + r] = seq_y[w.P:]
                dx_r[offs[i]:offs[i] + r] = seq_dx[w.P:]
                if i == 0:
                    y_r[:w.P] = seq_y[:w.P]
                dx_r[:w.P] += seq_dx[:w.P]
                start += w.P + r
            py, pdx, pg = results["packed"]

            def rel(a, b):
                return float((a.float() - b.float()).norm() / b.float().norm())

            out["packed_vs_replicated_rel_l2"] = {
                "y": rel(py, y_r), "dx": rel(pdx, dx_r),
                "weight_grads_max": max(rel(pg[n], grads[n]) for n in pg)}
            del y_r, dx_r
        del layer, x, dy
        torch.cuda.empty_cache()
    out["speedup_packed"] = out["replicated"]["ms"] / out["packed"]["ms"]
    out["memory_reduction"] = 1.0 - out["packed"]["device_bytes"] / out["replicated"]["device_bytes"]
    out["rho_tokens"] = w.rho_tokens()
    return out


def gemm_leg(D, dev, stream, rows: int):
    """The layer's tensor-core GEMM (dualkv_gemm) against cuBLAS (torch.matmul,
    bf16 in, fp32 accumulation) on the same bf16 inputs, for one shape of each
    operand layout of a Qwen3-8B layer on `rows` packed rows: the QKV
    projection (X.W^T), the gate/up input gradient (dY.W) and the gate/up
    weight gradient (dY^T.X, fp32 out)."""
    H, I, nqkv = 4096, 12288, 6144
    gen = torch.Generator(device=dev).manual_seed(3)
    rnd = lambda *shape: torch.randn(shape, device=dev, generator=gen).to(torch.bfloat16)
    cases = {
        "qkv_fwd x.wT": (0, rnd(rows, H), rnd(nqkv, H), (rows, nqkv), torch.bfloat16),
        "gate_up_dx dy.w": (1, rnd(rows, 2 * I), rnd(2 * I, H), (rows, H), torch.bfloat16),
        "gate_up_dw dyT.x": (2, rnd(rows, 2 * I), rnd(rows, H), (2 * I, H), torch.float32),
    }
    out = {}
    for name, (kind, A, B, yshape, ydt) in cases.items():
        Y = torch.empty(yshape, dtype=ydt, device=dev)
        # cuBLAS arm: the same product in bf16 (for kind 2 with a bf16 result,
        # which it writes in half the bytes of the library's fp32 one)
        if kind == 0:
            M, K, N = A.shape[0], A.shape[1], B.shape[0]
            cublas = lambda: torch.matmul(A, B.T)
        elif kind == 1:
            M, K, N = A.shape[0], A.shape[1], B.shape[1]
            cublas = lambda: torch.matmul(A, B)
        else:
            K, M, N = A.shape[0], A.shape[1], B.shape[1]
            cublas = lambda: torch.matmul(A.T, B)
        ours = lambda: D.dualkv_gemm(kind, A, B, Y, stream=stream)
        flops = 2.0 * M * N * K
        res = {"M": M, "N": N, "K": K}
        for who, fn in (("library", ours), ("cublas", cublas)):
            with torch.cuda.stream(stream):
                for _ in range(2):
                    fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                for _ in range(5):
                    fn()
                b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / 5
            res[who] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
        res["library_over_cublas"] = res["library"]["tflops"] / res["cublas"]["tflops"]
        with torch.cuda.stream(stream):
            ours()
            check = cublas().float()
        torch.cuda.synchronize()
        res["rel_l2_vs_cublas"] = float((Y.float() - check).norm() / check.norm())
        del check
        out[name] = res
        del Y
    st, site = D.dualkv_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error {st} at wait site {site}")
    return out


def groups_leg(D, dev, stream):
    """Four prompt groups (Qwen3-8B shapes: 32/8 heads, d 128; each group a
    4096-token prompt and 8 responses of 4096 tokens) as one grouped forward +
    backward, against four single-group calls on the same rows."""
    Hq, Hkv, d, P, N, R = 32, 8, 128, 4096, 8, 4096
    groups = [(P, (R,) * N)] * 4
    T = synthetic.group_rows(groups)
    scale = d ** -0.5
    gen = torch.Generator(device=dev).manual_seed(5)
    q, do = (torch.randn((T, Hq, d), device=dev, generator=gen).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn((T, Hkv, d), device=dev, generator=gen).to(torch.bfloat16) for _ in range(2))
    out = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(D.dualkv_bwd_groups_workspace_bytes(groups, Hq, Hkv, d, False), dtype=torch.uint8,
                     device=dev)
    rows = P + N * R

    def grouped():
        D.dualkv_fwd_groups(q, k, v, groups, out, lse, scale, stream)
        D.dualkv_bwd_groups(q, k, v, out, do, lse, groups, scale, False, ws, dq, dk, dv, stream=stream)

    views = []
    for g in range(4):
        sl = slice(g * rows, (g + 1) * rows)
        views.append([t[sl] for t in (q, k, v, out, do, dq, dk, dv)] + [lse[:, sl].contiguous()])

    def separate():
        for qq, kk, vv, oo, dd, dqq, dkk, dvv, ll in views:
            D.dualkv_fwd(qq, kk, vv, P, (R,) * N, oo, ll, scale, stream)
            D.dualkv_bwd(qq, kk, vv, oo, dd, ll, P, (R,) * N, scale, False, ws, dqq, dkk, dvv, stream=stream)

    res = {"groups": 4, "P": P, "N": N, "R": R, "Hq": Hq, "Hkv": Hkv, "d": d, "T": T}
    flops = 4 * synthetic.make_workload("g", Hq, Hkv, d, P, (R,) * N).useful_flops()
    for name, fn in (("grouped", grouped), ("separate", separate)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(5):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / 5
        res[name] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
    st, site = D.dualkv_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error {st} at wait site {site}")
    return res


# --------------------------------------------------------------------------- CPU oracle timings

def _oracle_seq0_inputs(w: synthetic.Workload, seed: int):
    L = w.P + w.R_lens[0]
    g = torch.Generator("cpu").manual_seed(seed)
    return [torch.randn((L, 1, w.d), generator=g).to(torch.bfloat16).to(torch.float64).numpy() for _ in range(4)]


def oracle_sample_seconds(w: synthetic.Workload, seed: int = 0):
    """The fp64 oracle (as it stands) on one q-head and sequence 0 of the
    workload: replicated fwd + bwd of [prompt ; response_0].  Returns the
    seconds, the useful flops and (inputs, outputs) for sample_parity."""
    from oracle import attention as ora
    q, k, v, do = _oracle_seq0_inputs(w, seed)
    t0 = time.perf_counter()
    out, lse = ora.dualkv_forward(q, k, v, w.P, (w.R_lens[0],), w.scale)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, w.P, (w.R_lens[0],), w.scale)
    dt = time.perf_counter() - t0
    sub = synthetic.make_workload("s", 1, 1, w.d, w.P, (w.R_lens[0],))
    return dt, sub.useful_flops(), (q, k, v, do, out, lse, dq, dk, dv)


def sample_parity(D, w: synthetic.Workload, dev, stream, sample):
    """The library on the oracle sample's own inputs (one head, [prompt ;
    response_0] at the workload's P, R_0, d and scale), compared element by
    element with the oracle's outputs, outside the timed region."""
    q, k, v, do, ro, rl, rdq, rdk, rdv = sample
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(dev)   # exact: the inputs are bf16 values
    tq, tk, tv, tdo = (bf(a) for a in (q, k, v, do))
    R = (w.R_lens[0],)
    with torch.cuda.stream(stream):
        out, lse = D.forward(tq, tk, tv, w.P, R, w.scale, stream=stream)
        dq, dk, dv = D.backward(tq, tk, tv, out, tdo, lse, w.P, R, w.scale, stream=stream)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().double().numpy()
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    res = {"rows": int(q.shape[0]), "heads": 1,
           "out_max_abs": float(np.abs(f(out) - ro).max()), "out_rel_l2": rel(f(out), ro),
           "lse_max_abs": float(np.abs(f(lse) - rl).max()),
           "dq_rel_l2": rel(f(dq), rdq), "dk_rel_l2": rel(f(dk), rdk), "dv_rel_l2": rel(f(dv), rdv)}
    res["within_bounds"] = bool(res["out_max_abs"] <= 1e-2 and res["out_rel_l2"] <= 5e-3 and
                                res["lse_max_abs"] <= 1e-3 and
                                max(res["dq_rel_l2"], res["dk_rel_l2"], res["dv_rel_l2"]) <= 1e-2)
    return res


def oracle_rows_seconds(w: synthetic.Workload, rows: int, seed: int = 0):
    """The oracle's row-wise function on `rows` query rows of q-head 0 in
    sequence 0 (O, LSE and dQ of each row over its full visible key set).
    Credited work: 8*d flops per visible (query, key) pair (QK^T, PV, dO V^T,
    dS K)."""
    from oracle import attention as ora
    rng = np.random.default_rng(seed)
    q, k, v, do = _oracle_seq0_inputs(w, seed)
    L = q.shape[0]
    picks = np.sort(rng.choice(L, size=min(rows, L), replace=False))
    t0 = time.perf_counter()
    ora.rows_forward_backward(q, k, v, do, w.P, (w.R_lens[0],), w.scale, [0], picks.tolist())
    dt = time.perf_counter() - t0
    pairs = int(sum(int(t) + 1 for t in picks))
    return dt, 8.0 * w.d * pairs


# --------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The oracle timed on the host cores (rank 0 only), on the same workload."""
    if rank != 0:
        return
    w = synthetic.WORKLOADS[args.workload]
    # per-step sample sized so that warm-up + timed steps stay within ~2.5 minutes
    probe_dt, _ = oracle_rows_seconds(w, 16, seed=99)
    per_row = probe_dt / 16
    budget = 150.0 / max(1, args.steps + args.warmup)
    rows = int(max(8, min(4096, budget / max(per_row, 1e-6))))
    for i in range(args.warmup):
        oracle_rows_seconds(w, rows, seed=i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = oracle_rows_seconds(w, rows, seed=1000 + i)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "P": w.P, "N": w.N,
                   "R": list(w.R_lens[:1]) if len(set(w.R_lens)) == 1 else list(w.R_lens)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"per step: O, LSE and dQ of {rows} random query rows of q-head 0 in "
                                   f"sequence 0 (fp64 row-wise oracle), credited 8*d flops per visible pair"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="p32k", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--deterministic", action="store_true", help="time the deterministic backward (mode 1)")
    ap.add_argument("--mode", type=int, choices=[0, 1, 2], default=None,
                    help="backward mode: 0 atomic prompt dK/dV with a separate dQ kernel (default), "
                         "1 deterministic, 2 atomic with dQ fused into dK/dV")
    ap.add_argument("--quick", action="store_true", help="skip the other-mode, replicated and CPU oracle legs")
    ap.add_argument("--layer", action="store_true",
                    help="also time a Qwen3-8B-shaped decoder layer, packed against replicated")
    ap.add_argument("--gemm", action="store_true",
                    help="also time the layer's GEMM (one shape per operand layout) against cuBLAS on the "
                         "workload's packed rows")
    ap.add_argument("--groups", action="store_true",
                    help="also time four prompt groups in one call against four single-group calls")
    ap.add_argument("--e2e-buffers", type=int, default=3,
                    help="device buffer sets in the end-to-end leg's copy/compute ring (at least 2)")
    ap.add_argument("--kernels-only", action="store_true",
                    help="also skip the end-to-end leg (for profiling: one buffer set on the device)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        args.warmup = 3

    from shared_prompt_exact_dualkv_gb300 import dualkv as D

    w = synthetic.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    x = synthetic.make_inputs(w, seed=rank)
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.dout))
    out = torch.empty_like(q)
    lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    mode = args.mode if args.mode is not None else (1 if args.deterministic else 0)
    det = mode   # the backward mode, passed through to dualkv_bwd
    fused = mode == 2
    ws = torch.empty(D.dualkv_bwd_workspace_bytes(w.P, w.R_lens, w.Hq, w.Hkv, w.d, det), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step():
        D.dualkv_fwd(q, k, v, w.P, w.R_lens, out, lse, w.scale, stream)
        D.dualkv_bwd(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, det, ws, dq, dk, dv, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), world) / args.steps
    st, site = D.dualkv_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error {st} at wait site {site}")

    # per-kernel device time (events around each launch, same stream)
    D.dualkv_trace_enable(True)
    for _ in range(args.steps):
        step()
    tr = D.dualkv_trace_read()
    D.dualkv_trace_enable(False)
    # device time per step of each kernel (long work lists run as several launches)
    per_kernel = {name: tot / args.steps for name, (tot, cnt) in tr.items()}
    kernel_launches = {name: cnt // args.steps for name, (tot, cnt) in tr.items()}
    launches_per_step = sum(kernel_launches.values())

    e2e = None
    if not args.kernels_only:
        e2e = end_to_end(args, D, w, x, dev, q, lse, k, v, ws, stream, det, world)

    flops = w.useful_flops()
    value = weak_scaling_value(flops, ms, world)
    e2e_obj = None
    if e2e is not None:
        e2e_ms, h2d, d2h = e2e
        e2e_obj = {"value": weak_scaling_value(flops, e2e_ms, world), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "buffer_sets": max(2, args.e2e_buffers)}
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))

    # dominant kernel: dK/dV (products per unmasked pair: S^T, dP^T, dV, dK, and
    # dQ in the fused mode); per step, which is per launch whenever the work
    # list fits one launch
    dkdv_per_pair = 10 if fused else 8
    dkdv_ms = per_kernel.get("bwd_dkdv", 0.0)
    dkdv_flops = float(dkdv_per_pair) * w.d * w.Hq * w.pairs_per_head()
    dkdv_tf = dkdv_flops / (dkdv_ms * 1e-3) / 1e12 if dkdv_ms else None
    roofline = {"bound": "tensor", "kernel": "dkdv_kernel" + ("<fused dQ>" if fused else ""), "achieved": dkdv_tf,
                "peak": peak_sus, "unit": "TFLOP/s", "frac": (dkdv_tf / peak_sus) if dkdv_tf else None,
                "traffic": recorded_traffic("dkdv_kernel", w.name, det),
                "peak_source": f"{peak_src} bf16_tflops_sustained",
                "algorithmic": f"{dkdv_per_pair}*d flops per unmasked (query,key) pair per q-head",
                "launches_per_step": kernel_launches.get("bwd_dkdv", 0)}
    # The measured sustained rate was taken at the clock its own run settled
    # at; compare per MHz of sampled SM clock as well.
    peak_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    run_mhz = clock_info.get("sm_mhz")
    if dkdv_tf and peak_mhz and run_mhz:
        roofline["per_mhz"] = {"achieved_tflops_per_mhz": dkdv_tf / run_mhz, "run_sm_mhz": run_mhz,
                               "peak_tflops_per_mhz": peak_sus / peak_mhz, "peak_sm_mhz": peak_mhz,
                               "frac": (dkdv_tf / run_mhz) / (peak_sus / peak_mhz)}

    # every tensor-core kernel against the measured sustained bf16 rate; executed
    # flops per unmasked pair per q-head: forward 4d, dK/dV 8d (10d with dQ
    # fused), separate dQ 6d (S and dP recomputed)
    tensor_kernels = {}
    for name, per_pair in (("fwd", 4), ("bwd_dkdv", dkdv_per_pair)) + ((() if fused else (("bwd_dq", 6),))):
        kms = per_kernel.get(name, 0.0)
        fl = per_pair * w.d * w.Hq * w.pairs_per_head()
        tf = fl / (kms * 1e-3) / 1e12 if kms else None
        tensor_kernels[name] = {"tflop_per_step": fl / 1e12, "ms": kms, "achieved_tflops": tf,
                                "frac": (tf / peak_sus) if tf else None}

    # the two bandwidth-bound kernels of the backward, against the measured copy bandwidth
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    prompt_rows_bytes = w.P * w.Hkv * w.d * 4                      # one fp32 [P, Hkv, d] slice
    n_slices = 1
    if det == 1 and prompt_rows_bytes:
        acc_region = (ws.numel() - align256(w.T * w.Hq * 4)) // 2   # bytes of acc_k (= acc_v)
        n_slices = max(1, acc_region // prompt_rows_bytes)
    hbm_bytes = {
        # read O and dO, write D; zero the two fp32 accumulators in the atomic mode
        "bwd_preprocess": (2 * w.T * w.Hq * w.d * 2 + w.T * w.Hq * 4 + (0 if det == 1 else 2 * prompt_rows_bytes)
                           + (w.T * w.Hq * w.d * 4 if fused else 0)),
        # read every split slice of both accumulators, write bf16 prompt dK and dV
        "bwd_prompt_reduce": 2 * n_slices * prompt_rows_bytes + 2 * w.P * w.Hkv * w.d * 2,
    }
    if fused:
        # the dQ cast: read the fp32 accumulator, write bf16 dQ (trace slot of the dQ kernel)
        hbm_bytes["bwd_dq"] = w.T * w.Hq * w.d * (4 + 2)
    hbm_kernels = {}
    for name, nbytes in hbm_bytes.items():
        kms = per_kernel.get(name, 0.0)
        gbs = nbytes / (kms * 1e-3) / 1e9 if kms else None
        hbm_kernels[name] = {"bytes_per_launch": nbytes, "ms": kms, "achieved_gbs": gbs, "peak_gbs": hbm_peak,
                             "frac": (gbs / hbm_peak) if gbs else None,
                             "peak_source": f"{peak_src} hbm_gbs"}

    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "P": w.P, "N": w.N,
                   "R": list(w.R_lens[:1]) if len(set(w.R_lens)) == 1 else list(w.R_lens),
                   "T_packed": w.T, "T_replicated": w.T_replicated, "rho_tokens": round(w.rho_tokens(), 3),
                   "rho_pairs": round(w.rho_pairs(), 3), "useful_tflop_per_step": flops / 1e12,
                   "dkdv_mode": {0: "atomic, separate dQ", 1: "deterministic", 2: "atomic, dQ fused"}[mode],
                   "l2": "inputs larger than L2 (q alone %.0f MB > 129 MB)" % (q.numel() * 2 / 1e6),
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / peak_sus,
        "per_kernel_ms": per_kernel,
        "kernel_launches_per_step": kernel_launches,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock_info,
        "e2e": e2e_obj,
        "roofline": roofline,
        "tensor_kernels": tensor_kernels,
        "hbm_kernels": hbm_kernels,
    }

    if rank == 0 and not args.quick:
        # the other backward modes on the same inputs (backward alone)
        names = {0: "atomic", 1: "deterministic", 2: "atomic_fused_dq"}
        others = {}
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for m in (0, 1, 2):
            ws2 = torch.empty(D.dualkv_bwd_workspace_bytes(w.P, w.R_lens, w.Hq, w.Hkv, w.d, m), dtype=torch.uint8,
                              device=dev)
            for _ in range(2):
                D.dualkv_bwd(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, m, ws2, dq, dk, dv, stream=stream)
            a.record(stream)
            for _ in range(3):
                D.dualkv_bwd(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, m, ws2, dq, dk, dv, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            others[names[m]] = {"bwd_ms": a.elapsed_time(b) / 3, "workspace_bytes": ws2.numel()}
            del ws2
        result["bwd_modes"] = others
        # the same library on the replicated N(P+R) layout
        wr = w.replicated()
        gen = torch.Generator(device=dev).manual_seed(7)
        rq = torch.randn((wr.T, w.Hq, w.d), device=dev, generator=gen).to(torch.bfloat16)
        rk = torch.randn((wr.T, w.Hkv, w.d), device=dev, generator=gen).to(torch.bfloat16)
        rv = torch.randn((wr.T, w.Hkv, w.d), device=dev, generator=gen).to(torch.bfloat16)
        rdo = torch.randn((wr.T, w.Hq, w.d), device=dev, generator=gen).to(torch.bfloat16)
        rout, rlse = torch.empty_like(rq), torch.empty((w.Hq, wr.T), dtype=torch.float32, device=dev)
        rdq, rdk, rdv = torch.empty_like(rq), torch.empty_like(rk), torch.empty_like(rv)
        rws = torch.empty(max(1, D.dualkv_bwd_workspace_bytes(0, wr.R_lens, w.Hq, w.Hkv, w.d, False)),
                          dtype=torch.uint8, device=dev)

        def rstep():
            D.dualkv_fwd(rq, rk, rv, 0, wr.R_lens, rout, rlse, w.scale, stream)
            D.dualkv_bwd(rq, rk, rv, rout, rdo, rlse, 0, wr.R_lens, w.scale, False, rws, rdq, rdk, rdv, stream=stream)

        rstep()
        a.record(stream)
        for _ in range(2):
            rstep()
        b.record(stream)
        torch.cuda.synchronize()
        rms = a.elapsed_time(b) / 2
        # Device memory of one layer: the library allocates nothing, so this is
        # every caller-owned tensor of the call (inputs, outputs, workspace).
        def nbytes(ts):
            return sum(t.numel() * t.element_size() for t in ts)
        mem_packed = nbytes((q, k, v, do, out, lse, dq, dk, dv, ws))
        mem_rep = nbytes((rq, rk, rv, rdo, rout, rlse, rdq, rdk, rdv, rws))
        result["replicated_layout"] = {"ms_per_step": rms, "T": wr.T, "speedup_packed": rms / ms,
                                       "useful_tflop_replicated": wr.useful_flops() / 1e12}
        result["layer_memory_bytes"] = {"packed": mem_packed, "replicated": mem_rep,
                                        "reduction": 1.0 - mem_packed / mem_rep}
        del rq, rk, rv, rdo, rout, rlse, rdq, rdk, rdv, rws
        torch.cuda.empty_cache()
        if world == 1:
            dt, fl, sample = oracle_sample_seconds(w)
            result["parity_sample"] = sample_parity(D, w, dev, stream, sample)
            del sample
            # The replicated oracle's cost is linear in heads and, per sequence,
            # in its causal pairs: scale the one (head, sequence) sample to the
            # whole step.
            seq0_pairs = (w.P + w.R_lens[0]) * (w.P + w.R_lens[0] + 1) // 2
            full_s = dt * w.Hq * w.pairs_per_head_replicated() / seq0_pairs
            result["cpu_baseline"] = {
                "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                "blas_threads": blas_threads(), "seconds": dt,
                "sample": f"fp64 oracle fwd+bwd of q-head 0 on sequence 0 ([prompt; response_0], "
                          f"{w.P + w.R_lens[0]} rows); BLAS multithreaded, elementwise single-threaded",
                "extrapolated_step_seconds": full_s,
                "extrapolation": f"extrapolated, not measured: sample seconds x {w.Hq} q-heads x "
                                 f"(causal pairs of all {w.N} replicated sequences / pairs of sequence 0)"}
        st, site = D.dualkv_last_device_error(stream)
        if st != 0:
            raise RuntimeError(f"device error {st} at wait site {site}")

    if rank == 0 and args.groups:
        result["groups"] = groups_leg(D, dev, stream)

    if rank == 0 and args.gemm and not args.layer:
        result["gemm"] = gemm_leg(D, dev, stream, w.T)

    if rank == 0 and args.layer:
        del q, k, v, do, out, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
        result["layer"] = layer_leg(D, w, dev, stream)
        result["layer"]["gemm"] = gemm_leg(D, dev, stream, w.T)

    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
