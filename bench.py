"""Benchmark of one weight-absorbed MLA decode step on GB300, through libmla's C ABI.

A step is one pass of the whole hot path over one batch: append the step's new
tokens from hidden states (mla_append_cache), decode (mla_decode: query
absorption + RoPE, split planning, attention, LSE combine) and project the latent
outputs through the folded weights (mla_output_proj). The weight fold itself
(mla_absorb_weights) runs once at set-up, as at model load.

Default workload: DeepSeek-V2 shapes (128 heads, d_c 512, d_r 64, d_model 5120),
bf16, batch 32, every request 4096 cached tokens in shuffled 64-token pages.

Prints one JSON line. Under torchrun every rank runs its own replica of the
workload on its own GPU (requests are independent: no data-path collective) and
rank 0 prints the whole-job throughput (weak scaling).

`--impl reference` times the CPU oracle (fp64 numpy) on this host instead, one
request of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MLA decode tokens/s + latent-cache GB/s & TFLOP/s as % of GB300 roofline"
UNIT = "tokens/s"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- events

_CUDART = None


def event_ms(a, b) -> float:
    """Milliseconds between two recorded torch CUDA events. Read through the CUDA runtime
    directly, because some events are recorded inside libmla (torch does not see those)."""
    global _CUDART
    import ctypes
    if _CUDART is None:
        import mla_latent_kv_04_gb300 as M
        M.lib()
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                _CUDART = ctypes.CDLL(name)
                break
            except OSError:
                continue
        _CUDART.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                 ctypes.c_void_p]
    out = ctypes.c_float(0.0)
    rc = _CUDART.cudaEventElapsedTime(ctypes.byref(out), ctypes.c_void_p(a.cuda_event),
                                      ctypes.c_void_p(b.cuda_event))
    if rc != 0:
        raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
    return float(out.value)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- set-up

def setup(wl, dev, workers=0):
    """Seeded workload on the device: weights (folded once), the filled paged cache, the
    step's inputs. Uses only the library's calls; inputs are generated on the host.
    workers: decode workers (0: the library's default, one per CTA pair)."""
    import torch
    import mla_latent_kv_04_gb300 as M

    act = torch.float32 if wl.act == "f32" else torch.bfloat16
    scale = W.fp8_cache_scale(wl) if wl.cache == "fp8_e4m3" else 1.0
    cfg = M.make_config(wl.dims, wl.act, wl.cache, cache_scale=scale, rope_theta=wl.rope_theta)
    d = wl.dims
    H, D = d.num_heads, d.d_cache

    def up(x, dtype=act):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device=dev, dtype=dtype)

    wts = W.weights(wl)
    dw = {k: up(v) for k, v in wts.items()}
    bt, num_pages = W.page_table(wl)
    cdt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8,
           "fp8_e4m3_b128": torch.uint8}[wl.cache]
    row = W.cache_row_bytes(wl) // torch.tensor([], dtype=cdt).element_size()
    cache = torch.zeros(num_pages * d.page_size * row, dtype=cdt, device=dev)
    bt_d = up(bt, torch.int32)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    for b in range(wl.batch):
        n_lat, n_h = W.token_sources(wl, b)
        # every position, including the step's q_len new ones, is filled once so the cache is
        # complete; the timed step then re-appends the new tokens from h each iteration
        c, k = W.latent_rows(wl, b, wl.seq_lens[b])
        req, pos = W.append_batch(wl, b, 0, wl.seq_lens[b])
        M.mla_append_cache_latent(cfg, up(c), up(k), up(req, torch.int32), up(pos, torch.int32), bt_d,
                                  cache, rotate=True, dev_status=status)
    W_UK_abs = torch.empty(H * d.d_nope * d.d_latent, dtype=act, device=dev)
    W_comb = torch.empty(H * d.d_latent * d.d_model, dtype=act, device=dev)
    M.mla_absorb_weights(cfg, dw["W_UK"], dw["W_UV"], dw["W_O"], W_UK_abs, W_comb)
    assert M.mla_read_device_status(status) == M.MLA_OK
    B, q = wl.batch, wl.q_len
    qs = W.queries(wl)
    new_h = np.concatenate([W.hidden(wl, b, q) for b in range(B)])
    new_req = np.repeat(np.arange(B, dtype=np.int32), q)
    new_pos = np.concatenate([np.arange(wl.seq_lens[b] - q, wl.seq_lens[b], dtype=np.int32)
                              for b in range(B)])
    host = {"q_nope": qs["q_nope"], "q_pe": qs["q_pe"], "h": new_h,
            "seq_lens": np.array(wl.seq_lens, np.int32)}
    dev_in = {"q_nope": up(qs["q_nope"]), "q_pe": up(qs["q_pe"]), "h": up(new_h),
              "seq_lens": up(host["seq_lens"], torch.int32)}
    rows = B * q
    out_lat = torch.empty(rows * H * d.d_latent, dtype=act, device=dev)
    lse = torch.empty(rows * H, dtype=torch.float32, device=dev)
    out = torch.empty(rows * d.d_model, dtype=act, device=dev)
    ws = torch.zeros(M.mla_decode_workspace_size(cfg, B, q, num_workers=workers), dtype=torch.uint8,
                     device=dev)
    ws_o = torch.zeros(M.mla_output_proj_workspace_size(cfg, rows), dtype=torch.uint8, device=dev)
    ws_u = torch.zeros(M.mla_output_proj_unfolded_workspace_size(cfg, rows), dtype=torch.uint8,
                       device=dev)
    n_a = M.mla_append_cache_workspace_size(cfg, rows)
    ws_a = torch.zeros(n_a, dtype=torch.uint8, device=dev) if n_a else None
    # the query side from h (low-rank query compression), timed beside the step
    qdw = {k: up(v) for k, v in W.query_weights(wl).items()}
    query = {"w": qdw, "h": up(W.query_hidden(wl, rows)),
             "q_nope": torch.empty(rows * H * d.d_nope, dtype=act, device=dev),
             "q_pe": torch.empty(rows * H * d.d_rope, dtype=act, device=dev),
             "ws": torch.zeros(M.mla_query_workspace_size(cfg, d.d_q, rows), dtype=torch.uint8,
                               device=dev)}
    torch.cuda.synchronize()
    return {"cfg": cfg, "dw": dw, "cache": cache, "bt_d": bt_d, "W_UK_abs": W_UK_abs,
            "W_comb": W_comb, "host": host, "dev_in": dev_in,
            "new_req": up(new_req, torch.int32), "new_pos": up(new_pos, torch.int32),
            "out_lat": out_lat, "lse": lse, "out": out, "ws": ws, "ws_o": ws_o, "ws_u": ws_u,
            "ws_a": ws_a, "query": query, "workers": workers,
            "status": status}


def step(st, inp, ev=None):
    """One decode step through the C ABI on the current stream. ev: optional dict of event
    pairs ('append', 'decode', 'attn', 'oproj') recorded around each part."""
    import mla_latent_kv_04_gb300 as M
    cfg = st["cfg"]
    if ev:
        ev["append"][0].record()
    M.mla_append_cache(cfg, inp["h"], st["dw"]["W_DKV_KR"], st["new_req"], st["new_pos"], st["bt_d"],
                       st["cache"], dev_status=st["status"], workspace=st["ws_a"])
    if ev:
        ev["append"][1].record()
        ev["decode"][0].record()
    M.mla_decode(cfg, inp["q_nope"], inp["q_pe"], st["W_UK_abs"], st["cache"], st["bt_d"],
                 inp["seq_lens"], st["out_lat"], st["lse"], st["ws"], num_workers=st["workers"],
                 attn_events=ev["attn"] if ev else None)
    if ev:
        ev["decode"][1].record()
        ev["oproj"][0].record()
    M.mla_output_proj(cfg, st["out_lat"], st["W_comb"], st["out"], st["ws_o"])
    if ev:
        ev["oproj"][1].record()


L2_FLUSH_BYTES = 256 << 20      # twice the GB300's 129 MB L2
PART_REPS = 20


def graph_ms(fn, reps, mk):
    """Mean device time of fn(): `reps` calls captured back to back as one CUDA graph, the
    graph replayed 3 times after a warm-up replay, timed with CUDA events."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a, b = mk()
    a.record()
    for _ in range(3):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (3 * reps)


# ----------------------------------------------------------------------------- roofline

def kernel_work(wl):
    """Algorithmic bytes and FLOPs per launch of each timed part."""
    d = wl.dims
    H, B, q = d.num_heads, wl.batch, wl.q_len
    ea = W.elt_bytes(wl.act)
    dec_b = W.decode_bytes(wl)
    attn_bytes = dec_b["cache"] + dec_b["out_latent"] + dec_b["lse"] + dec_b["block_table"]
    attn_flops = W.decode_flops(wl) - 2.0 * B * q * H * d.d_nope * d.d_latent
    rows = B * q
    K = H * d.d_latent
    return {
        "attn": {"bytes": attn_bytes, "flops": attn_flops},
        "decode": {"bytes": sum(dec_b.values()), "flops": W.decode_flops(wl)},
        "oproj": {"bytes": K * d.d_model * ea + rows * K * ea + rows * d.d_model * ea,
                  "flops": 2.0 * rows * K * d.d_model},
        "append": {"bytes": rows * d.d_model * ea + d.d_model * d.d_cache * ea
                   + rows * W.cache_row_bytes(wl),
                   "flops": 2.0 * rows * d.d_model * d.d_cache},
        # the step's queries from h: W_DQ, W_UQ, W_QR, h in, q_nope and q_pe out (c_q, an
        # intermediate, is not counted)
        "query": {"bytes": (d.d_model * d.d_q + d.d_q * H * d.d_nope + d.d_model * H * d.d_rope) * ea
                  + rows * d.d_model * ea + rows * H * (d.d_nope + d.d_rope) * ea,
                  "flops": 2.0 * rows * (d.d_model * d.d_q + d.d_q * H * d.d_nope
                                         + d.d_model * H * d.d_rope)},
        # the unfolded output path: W_UV and W_O instead of W_comb (not part of the step)
        "oproj_unfolded": {"bytes": (d.d_latent * H * d.d_v + H * d.d_v * d.d_model) * ea
                           + rows * K * ea + rows * d.d_model * ea,
                           "flops": 2.0 * rows * (K * d.d_v + H * d.d_v * d.d_model)},
    }


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture
# of the kernel on one workload (summaries under profiles/), valid only for that workload and
# while the kernel's source file is the one captured: each entry carries the workload's name
# and that file's sha256, and reads as null otherwise.
NCU_TRAFFIC = {
    "attn": {"bytes": 155806464 + 234240, "workload": "v2_b32_s4096",
             "source": "mla_latent_kv_04_gb300/csrc/decode_tc.cu",
             "sha256": "10540466e20837f618c73b23ccf6f82a0b52171c2204ed073ccc1a2babc9de5a"},
    "oproj": {"bytes": 675325696 + 79872, "workload": "v2_b32_s4096",
              "source": "mla_latent_kv_04_gb300/csrc/gemm_tc.cu",
              "sha256": "3bacb2393e5669bca31a1706cfa0b4227f0e1cefa74c5e024b12fdd4e67b5c0e"},
    "append": {"bytes": 6258432 + 0, "workload": "v2_b32_s4096",
               "source": "mla_latent_kv_04_gb300/csrc/gemm_tc.cu",
               "sha256": "3bacb2393e5669bca31a1706cfa0b4227f0e1cefa74c5e024b12fdd4e67b5c0e"},
}


def ncu_traffic(part, workload="v2_b32_s4096"):
    import hashlib
    e = NCU_TRAFFIC.get(part)
    if not e or e["workload"] != workload:
        return None
    try:
        with open(os.path.join(ROOT, e["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return e["bytes"] if digest == e["sha256"] else None


def roofline_entry(work, ms, peaks, tensor_peak):
    sec = ms * 1e-3
    gbs = work["bytes"] / sec / 1e9
    tfs = work["flops"] / sec / 1e12
    t_hbm = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = work["flops"] / (tensor_peak * 1e12)
    if t_hbm >= t_tc:
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "tflops": round(tfs, 1),
                "tensor_frac": round(tfs / tensor_peak, 4)}
    return {"bound": "tensor", "achieved": round(tfs, 1), "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": round(tfs / tensor_peak, 4), "gbs": round(gbs, 1),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)}


# ----------------------------------------------------------------------------- CPU oracle

CPU_CHILD = r"""
import json, os, sys, time
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle, workloads as W
wl = W.WORKLOADS[sys.argv[2]]
budget = float(sys.argv[3]); max_requests = int(sys.argv[4]); warm = int(sys.argv[5])
wts = W.weights(wl)
A, C = oracle.absorb_weights(wts["W_UK"], wts["W_UV"], wts["W_O"], wl.dims.num_heads)
q = W.queries(wl)
scale = oracle.softmax_scale(wl.dims.d_nope, wl.dims.d_rope)
done = 0; tokens = 0; t_work = 0.0; b = 0; it = 0
while (t_work < budget or done == 0) and done < max_requests:
    S = wl.seq_lens[b]
    c, k = W.latent_rows(wl, b, S)
    h = W.hidden(wl, b, wl.q_len)
    t0 = time.perf_counter()
    cn, kr = oracle.project_latent(h, wts["W_DKV_KR"], wl.dims.d_latent)
    c = np.concatenate([c[:S - wl.q_len], cn]); k = np.concatenate([k[:S - wl.q_len], kr])
    k = oracle.rope(k, np.arange(S), wl.rope_theta)
    o, lse = oracle.decode_absorbed(c, k, q["q_nope"][b], q["q_pe"][b], A, scale, wl.rope_theta)
    out = oracle.output_projection(o.reshape(wl.q_len, -1), C)
    dt = time.perf_counter() - t0
    it += 1; b = (b + 1) % wl.batch
    if it <= warm:
        continue
    t_work += dt; done += 1; tokens += wl.q_len
print(json.dumps({"seconds": t_work, "requests": done, "tokens": tokens}))
"""


def cpu_oracle(wl, budget_s, max_requests=10 ** 9, warm=0):
    """Times the fp64 oracle's whole decode step (append projection, absorbed decode,
    folded output projection) on this host, request by request, in a child process whose
    BLAS may use every core. The first ``warm`` requests run untimed. Returns
    (tokens/s, threads, description, raw)."""
    threads = os.cpu_count() or 1
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    r = subprocess.run([sys.executable, "-c", CPU_CHILD, ROOT, wl.name, str(budget_s),
                        str(max_requests), str(warm)], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("cpu oracle failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    tps = res["tokens"] / res["seconds"]
    desc = (f"{res['requests']} of {wl.batch} requests ({res['tokens']} tokens, "
            f"{res['seconds']:.1f} s of fp64 numpy work: append projection, absorbed decode, "
            f"folded output projection)")
    return tps, threads, desc, res


# ----------------------------------------------------------------------------- ranks

def rank_env():
    """(world, rank, local_rank) from torchrun's environment; (1, 0, 0) without it."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the slowest replica sets the job's time). Needs the
    process group when world > 1."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step: int, world: int, ms: float) -> float:
    """Whole-job tokens/s: the tokens every replica processes in one step over the slowest
    replica's step time."""
    return tokens_per_rank_step * world / (ms * 1e-3)


def run_reference(args):
    """The reference arm: the CPU oracle on this host, one request of the workload per step:
    ``warmup`` untimed requests, then ``steps`` timed ones (fewer only if they would take more
    than --reference-budget seconds; the line's ``steps`` is the number actually timed).
    Under torchrun only rank 0 works and prints; the other ranks return at once."""
    _, rank, _ = rank_env()
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    tps, threads, desc, res = cpu_oracle(wl, args.reference_budget, max_requests=args.steps,
                                         warm=args.warmup)
    timed = int(res["requests"])
    ms = res["seconds"] / max(1, timed) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": round(tps, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": timed, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "seq_len": wl.seq_lens[0],
                       "q_len": wl.q_len,
                       "step_sample": "each step is 1 request of the batch (requests taken in "
                                      "turn), the oracle's whole step for it: append projection, "
                                      "absorbed decode, folded output projection"},
            "cpu_baseline": {"value": round(tps, 3), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(tps, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    if timed != args.steps:
        line["steps_requested"] = args.steps
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v2_b32_s4096", choices=list(W.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of fp64 oracle work for the cpu_baseline field")
    ap.add_argument("--reference-budget", type=float, default=180.0,
                    help="seconds of timed oracle work the reference arm may spend")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workers", type=int, default=0,
                    help="decode workers (0: the library's default, one per CTA pair)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import mla_latent_kv_04_gb300 as M

    world, rank, local = rank_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M.lib()
    wl = W.WORKLOADS[args.workload]
    st = setup(wl, dev, args.workers)
    inp = st["dev_in"]

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up
    for _ in range(args.warmup):
        step(st, inp)
    torch.cuda.synchronize()
    # The step as one CUDA graph: the library's calls captured once (their launches
    # and programmatic launch dependencies), then replayed; this removes the host launch
    # gaps between the step's kernels. The library counts launches when they are issued, so
    # the kernels of one step are counted at capture.
    graph = torch.cuda.CUDAGraph()
    n_cap = M.mla_kernel_launches()
    with torch.cuda.graph(graph):
        step(st, inp)
    launches_per_step = M.mla_kernel_launches() - n_cap
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # device-timed region: inputs resident in HBM
    K = args.steps
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa
    evs = [{k: mk() for k in ("append", "decode", "attn", "oproj")} for _ in range(K)]
    for e in evs:          # torch creates the CUDA event on first record; libmla records 'attn'
        for a, b2 in e.values():
            a.record()
            b2.record()
    torch.cuda.synchronize()
    t0, t1 = mk()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0.record()
    for i in range(K):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier()
    launches = launches_per_step * K
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / K
    # the same steps issued call by call on the stream (no graph), for comparison
    s0, s1 = mk()
    s0.record()
    for i in range(K):
        step(st, inp)
    s1.record()
    torch.cuda.synchronize()
    ms_stream = s0.elapsed_time(s1) / K
    # per-part breakdown. The attention kernel's own duration comes from the events libmla
    # records around it on its stream (a pass of its own: events between kernels chained by
    # programmatic dependent launch cost overlap). Each call of the step (append, decode,
    # output projection) is timed as a CUDA graph of L2 flush + call, minus a graph of the
    # flush alone, so that it starts from a cold L2 and without host launch gaps, as it does
    # inside the step; a stream pass with events between the calls would count the host's
    # launch time of the small calls instead.
    for i in range(K):
        step(st, inp, evs[i])
    torch.cuda.synchronize()
    parts = {"attn": sum(event_ms(e["attn"][0], e["attn"][1]) for e in evs) / K}
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    calls = {
        "append": lambda: M.mla_append_cache(st["cfg"], inp["h"], st["dw"]["W_DKV_KR"], st["new_req"],
                                             st["new_pos"], st["bt_d"], st["cache"],
                                             dev_status=st["status"], workspace=st["ws_a"]),
        "decode": lambda: M.mla_decode(st["cfg"], inp["q_nope"], inp["q_pe"], st["W_UK_abs"],
                                       st["cache"], st["bt_d"], inp["seq_lens"], st["out_lat"],
                                       st["lse"], st["ws"], num_workers=st["workers"]),
        "oproj": lambda: M.mla_output_proj(st["cfg"], st["out_lat"], st["W_comb"], st["out"],
                                           st["ws_o"]),
    }
    # the flush reads its buffer: clean lines, so no write-back of dirty ones lands on the call
    t_flush = graph_ms(lambda: flush.sum(), PART_REPS, mk)
    for k, f in calls.items():
        parts[k] = graph_ms(lambda: (flush.sum(), f()), PART_REPS, mk) - t_flush
    del flush
    # mla_decode alone, back to back with nothing recorded inside (its four kernels overlap
    # through programmatic dependent launch; the 151 MB cache is larger than L2)
    decode_alone_ms = graph_ms(calls["decode"], K, mk)
    # the unfolded output path (u_i = o_i W_i^UV, then u W_O), alone, back to back as a graph;
    # an alternative to the step's folded projection, not part of the step (its 185 MB of
    # weights are larger than L2)
    oproj_unfolded_ms = graph_ms(
        lambda: M.mla_output_proj_unfolded(st["cfg"], st["out_lat"], st["dw"]["W_UV"], st["dw"]["W_O"],
                                           st["out"], st["ws_u"]), K, mk)
    # the queries from h (c^Q = h W^DQ, q^C = c^Q W^UQ, q^R = h W^QR), alone, back to back
    # (150 MB of weights)
    qj = st["query"]
    query_ms = graph_ms(
        lambda: M.mla_query_from_hidden(st["cfg"], wl.dims.d_q, qj["h"], qj["w"]["W_DQ"], qj["w"]["W_UQ"],
                                        qj["w"]["W_QR"], qj["q_nope"], qj["q_pe"], qj["ws"]), K, mk)
    ms = max_over_ranks(ms, world)
    value = job_throughput(wl.batch * wl.q_len, world, ms)
    code = M.mla_read_device_status(st["status"])
    code2 = M.mla_read_device_status(st["ws"])
    assert code == M.MLA_OK and code2 == M.MLA_OK, (code, code2)

    # end-to-end: pinned host inputs copied in, result read back, every step. The inputs sit
    # in one pinned host buffer and one device buffer (views per tensor), and the step's two
    # results in one device buffer, so each step makes one copy each way.
    host = st["host"]
    act = inp["q_nope"].dtype
    srcs = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dtype=act if k != "seq_lens" else torch.int32)
            for k, v in host.items()}

    def packed(tensors, device, pin):
        """One byte buffer holding every tensor (256-byte aligned offsets) and views of it."""
        offs, total = {}, 0
        for k, v in tensors.items():
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        buf = torch.empty(total, dtype=torch.uint8, device=device, pin_memory=pin)
        views = {k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                 for k, v in tensors.items()}
        return buf, views

    pin_in, pinned = packed(srcs, "cpu", True)
    for k, v in srcs.items():
        pinned[k].copy_(v)
    dev_in_buf, dev2 = packed(srcs, dev, False)
    outs = {"out": st["out"], "lse": st["lse"]}
    dev_out_buf, dev_outs = packed(outs, dev, False)
    host_out_buf, _ = packed(outs, "cpu", True)
    st2 = dict(st, out=dev_outs["out"], lse=dev_outs["lse"])
    h2d = sum(v.numel() * v.element_size() for v in srcs.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    # the graph reads the step's inputs from the packed device buffer and writes its results
    # into the packed output buffer
    graph_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_e2e):
        step(st2, dev2)
    for _ in range(max(1, args.warmup)):
        dev_in_buf.copy_(pin_in, non_blocking=True)
        graph_e2e.replay()
        host_out_buf.copy_(dev_out_buf, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = mk()
    barrier()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(K):
        dev_in_buf.copy_(pin_in, non_blocking=True)
        graph_e2e.replay()
        host_out_buf.copy_(dev_out_buf, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1) / K
    ms_e2e = max_over_ranks(ms_e2e, world)

    if rank != 0:
        return
    peaks = _peaks()
    work = kernel_work(wl)
    tpk = peaks["bf16_tflops_sustained"]
    rl = {k: roofline_entry(work[k], parts[k], peaks, tpk) for k in parts}
    dom = max(("attn", "oproj", "append"), key=lambda k: parts[k])
    names = {"attn": "mla_decode attention kernel", "oproj": "mla_output_proj",
             "append": "mla_append_cache"}
    roof = dict(rl[dom])
    roof["kernel"] = names[dom]
    roof["traffic"] = ncu_traffic(dom, wl.name)
    cache_mb = wl.total_tokens * W.cache_row_bytes(wl) / 1e6
    wcomb_mb = wl.dims.num_heads * wl.dims.d_latent * wl.dims.d_model * W.elt_bytes(wl.act) / 1e6
    roof["peak_source"] = peaks["source"] + (" (sustained bf16)" if roof["bound"] == "tensor" else "")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.act, "data": "synthetic",
        "config": {"workload": wl.name, "description": wl.description, "batch": wl.batch,
                   "seq_len": wl.seq_lens[0], "q_len": wl.q_len, "heads": wl.dims.num_heads,
                   "cache_dtype": wl.cache, "page_size": wl.dims.page_size,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "decode_workers": args.workers if args.workers > 0 else "library default",
                   "launch": "the step captured once as a CUDA graph and replayed (its kernels "
                             "and programmatic launch dependencies); ms_per_step_stream "
                             "is the same step issued call by call",
                   "l2": f"inputs larger than L2: the step streams the {cache_mb:.0f} MB cache "
                         f"and the {wcomb_mb:.0f} MB folded W_comb"},
        "roofline": roof,
        "decode_roofline": dict(rl["attn"], kernel="mla_decode attention kernel",
                                traffic=ncu_traffic("attn", wl.name)),
        "parts_ms": {k: round(v, 4) for k, v in parts.items()},
        "parts_method": "append, decode, oproj: a CUDA graph of an L2 flush (a 256 MB read) and "
                        "the call, minus the flush alone (cold L2, no host launch gaps); attn: CUDA "
                        "events around the attention kernel on its stream",
        "decode_alone_ms": round(decode_alone_ms, 4),
        "ms_per_step_stream": round(ms_stream, 4),
        "query_from_hidden": dict(roofline_entry(work["query"], query_ms, peaks, tpk),
                                  ms=round(query_ms, 4),
                                  note="the step's queries from h: c^Q = h W^DQ, q^C = c^Q W^UQ, "
                                       "q^R = h W^QR (mla_query_from_hidden); timed alone, not "
                                       "part of the step, whose q_nope and q_pe are inputs"),
        "oproj_unfolded": dict(roofline_entry(work["oproj_unfolded"], oproj_unfolded_ms, peaks, tpk),
                               ms=round(oproj_unfolded_ms, 4),
                               note="alternative to the step's folded output projection: "
                                    "u_i = o_i W_i^UV then u W_O (W_UV + W_O instead of W_comb); "
                                    "not part of the step"),
        "parts_roofline": rl,
        "clocks": clk,
        "gpu_launches": int(launches),
        "e2e": {"value": round(job_throughput(wl.batch * wl.q_len, world, ms_e2e), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(ms_e2e, 4)},
    }
    if not args.no_cpu_baseline:
        tps, threads, desc, _ = cpu_oracle(wl, args.cpu_budget)
        line["cpu_baseline"] = {"value": round(tps, 3), "unit": UNIT, "cores": threads,
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
