"""GPU test harness: puts a seeded workload on the device through the library's own
calls, runs decode steps, and builds the oracle's expected values for the same inputs.

Device set-up uses only the Python binding of libmla (torch for memory). Expected
values come only from ``oracle`` (fp64, CPU) and the seeded draws in ``workloads``.
"""
from __future__ import annotations

import numpy as np
import torch

import mla_latent_kv_04_gb300 as M
import oracle
import workloads as W

SENTINEL = {"f32": 0x7FC0DEAD, "bf16": 0x7FC1, "fp8_e4m3": 0x7F, "fp8_e4m3_b128": 0x7F}   # NaN patterns


def torch_act(wl):
    return torch.float32 if wl.act == "f32" else torch.bfloat16


def to_dev(x: np.ndarray, dtype, dev):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=dev, dtype=dtype)


def config(wl, cache_scale=None):
    if wl.cache == "fp8_e4m3" and cache_scale is None:
        cache_scale = W.fp8_cache_scale(wl)
    return M.make_config(wl.dims, wl.act, wl.cache, cache_scale=cache_scale or 1.0,
                         rope_theta=wl.rope_theta)


def alloc_cache(wl, num_pages, dev, fill=True):
    D = wl.dims.d_cache
    n = num_pages * wl.dims.page_size * D
    if wl.cache == "fp8_e4m3_b128":
        t = torch.empty(num_pages * wl.dims.page_size * W.cache_row_bytes(wl), dtype=torch.uint8,
                        device=dev)
        if fill:
            t.fill_(SENTINEL["fp8_e4m3_b128"])
        return t
    if wl.cache == "f32":
        t = torch.empty(n, dtype=torch.int32, device=dev)
        if fill:
            t.fill_(SENTINEL["f32"])
        return t.view(torch.float32)
    if wl.cache == "bf16":
        t = torch.empty(n, dtype=torch.int16, device=dev)
        if fill:
            t.fill_(SENTINEL["bf16"])
        return t.view(torch.bfloat16)
    t = torch.empty(n, dtype=torch.uint8, device=dev)
    if fill:
        t.fill_(SENTINEL["fp8_e4m3"])
    return t


def build_state(wl, dev, cfg=None, chunk_tokens=1 << 16):
    """Weights and the filled paged cache for workload ``wl`` on device ``dev``."""
    cfg = cfg or config(wl)
    act = torch_act(wl)
    wts = W.weights(wl)
    dw = {k: to_dev(v, act, dev) for k, v in wts.items()}
    bt, num_pages = W.page_table(wl)
    cache = alloc_cache(wl, num_pages, dev)
    bt_d = to_dev(bt, torch.int32, dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    for b in range(wl.batch):
        n_lat, n_h = W.token_sources(wl, b)
        if n_lat:
            c, k = W.latent_rows(wl, b, n_lat)
            for s0 in range(0, n_lat, chunk_tokens):
                s1 = min(n_lat, s0 + chunk_tokens)
                req, pos = W.append_batch(wl, b, s0, s1 - s0)
                M.mla_append_cache_latent(cfg, to_dev(c[s0:s1], act, dev), to_dev(k[s0:s1], act, dev),
                                          to_dev(req, torch.int32, dev), to_dev(pos, torch.int32, dev),
                                          bt_d, cache, rotate=True, dev_status=status)
        if n_h:
            h = W.hidden(wl, b, n_h)
            req, pos = W.append_batch(wl, b, n_lat, n_h)
            aws = torch.empty(M.mla_append_cache_workspace_size(cfg, n_h), dtype=torch.uint8, device=dev)
            M.mla_append_cache(cfg, to_dev(h, act, dev), dw["W_DKV_KR"], to_dev(req, torch.int32, dev),
                               to_dev(pos, torch.int32, dev), bt_d, cache, dev_status=status,
                               workspace=aws if aws.numel() else None)
    H, d_c, d_n, d = wl.dims.num_heads, wl.dims.d_latent, wl.dims.d_nope, wl.dims.d_model
    W_UK_abs = torch.empty(H * d_n * d_c, dtype=act, device=dev)
    W_comb = torch.empty(H * d_c * d, dtype=act, device=dev)
    M.mla_absorb_weights(cfg, dw["W_UK"], dw["W_UV"], dw["W_O"], W_UK_abs, W_comb)
    code = M.mla_read_device_status(status)
    assert code == M.MLA_OK, f"append reported device status {code}"
    return {"cfg": cfg, "weights": wts, "dw": dw, "bt": bt, "bt_d": bt_d, "num_pages": num_pages,
            "cache": cache, "W_UK_abs": W_UK_abs, "W_comb": W_comb,
            "seq_lens_d": to_dev(np.array(wl.seq_lens, np.int32), torch.int32, dev)}


def run_decode(wl, st, dev, q=None, kernel=M.KERNEL_AUTO, num_workers=0):
    q = q or W.queries(wl)
    act = torch_act(wl)
    cfg = st["cfg"]
    B, qn, H, d_c = wl.batch, wl.q_len, wl.dims.num_heads, wl.dims.d_latent
    qn_d = to_dev(q["q_nope"], act, dev)
    qp_d = to_dev(q["q_pe"], act, dev)
    out = torch.empty(B * qn * H * d_c, dtype=act, device=dev)
    lse = torch.empty(B * qn * H, dtype=torch.float32, device=dev)
    nws = M.mla_decode_workspace_size(cfg, B, qn, num_workers=num_workers, kernel=kernel)
    ws = torch.zeros(nws, dtype=torch.uint8, device=dev)
    M.mla_decode(cfg, qn_d, qp_d, st["W_UK_abs"], st["cache"], st["bt_d"], st["seq_lens_d"], out, lse,
                 ws, num_workers=num_workers, kernel=kernel)
    code = M.mla_read_device_status(ws)
    torch.cuda.synchronize()
    return {"q": q, "out_latent": out.float().cpu().numpy().astype(np.float64).reshape(B, qn, H, d_c),
            "lse": lse.cpu().numpy().astype(np.float64).reshape(B, qn, H), "status": code,
            "out_latent_dev": out, "ws": ws}


# ----------------------------------------------------------------------------- expectations

def cached_rows(wl, b, weights, cache_scale=None):
    """The latent rows (c [S][d_c], k_rot [S][d_r], float64) of request b that the cache holds,
    computed by the oracle from the seeded draws, in the cache's storage format."""
    n_lat, n_h = W.token_sources(wl, b)
    d = wl.dims
    cs, ks = [], []
    if n_lat:
        c, k = W.latent_rows(wl, b, n_lat)
        cs.append(c.astype(np.float64))
        ks.append(oracle.rope(k.astype(np.float64), np.arange(n_lat), wl.rope_theta))
    if n_h:
        h = W.hidden(wl, b, n_h)
        c, kraw = oracle.project_latent(h, weights["W_DKV_KR"], d.d_latent)
        cs.append(c)
        ks.append(oracle.rope(kraw, np.arange(n_lat, n_lat + n_h), wl.rope_theta))
    c = np.concatenate(cs) if cs else np.zeros((0, d.d_latent))
    k = np.concatenate(ks) if ks else np.zeros((0, d.d_rope))
    if wl.cache == "bf16":
        c = W.round_bf16(c.astype(np.float32)).astype(np.float64) if n_h else c
        k = W.round_bf16(k.astype(np.float32)).astype(np.float64)
    elif wl.cache == "fp8_e4m3_b128":
        # the device quantises its fp32 rows directly (latent rows are bf16 values already)
        c = oracle.e4m3_block_dequantize(*oracle.e4m3_block_quantize(c.astype(np.float32), 128), 128)
        k = W.round_bf16(k.astype(np.float32)).astype(np.float64)
    elif wl.cache == "fp8_e4m3":
        s = np.float32(cache_scale)
        c = oracle.e4m3_decode(oracle.e4m3_encode(c.astype(np.float32) / s)) * float(s)
        k = oracle.e4m3_decode(oracle.e4m3_encode(k / float(s))) * float(s)
    return c, k


def expected_request(wl, b, weights, q, W_UK_abs64, heads=None, cache_scale=None):
    c, k = cached_rows(wl, b, weights, cache_scale)
    scale = oracle.softmax_scale(wl.dims.d_nope, wl.dims.d_rope)
    return oracle.decode_absorbed(c, k, q["q_nope"][b], q["q_pe"][b], W_UK_abs64, scale,
                                  wl.rope_theta, heads=heads)


def expected_request_decompressed(wl, b, weights, q, heads, cache_scale=None):
    c, k = cached_rows(wl, b, weights, cache_scale)
    scale = oracle.softmax_scale(wl.dims.d_nope, wl.dims.d_rope)
    return oracle.decode_decompressed(c, k, q["q_nope"][b], q["q_pe"][b], weights["W_UK"],
                                      weights["W_UV"], scale, wl.rope_theta, heads=heads)


def tolerance(wl, ref):
    """Per-tensor bound on max |err|: 1e-5 max|ref| for fp32, 1e-2 max|ref| + 1e-3 otherwise."""
    m = float(np.max(np.abs(ref[np.isfinite(ref)]))) if np.isfinite(ref).any() else 0.0
    return 1e-5 * m if wl.act == "f32" else 1e-2 * m + 1e-3


def max_err(got, ref):
    """max |got - ref| over finite reference entries; -inf entries must match exactly."""
    fin = np.isfinite(ref)
    if not np.array_equal(np.isneginf(got), np.isneginf(ref)):
        return float("inf")
    return float(np.max(np.abs(got[fin] - ref[fin]))) if fin.any() else 0.0


def run_full_step_tiny(wl, dev):
    """Smoke path: append every token from h, decode, project; returns device results and
    the oracle's (decompressed) expectations."""
    st = build_state(wl, dev)
    r = run_decode(wl, st, dev)
    cfg = st["cfg"]
    B, qn, H, d_c, d = wl.batch, wl.q_len, wl.dims.num_heads, wl.dims.d_latent, wl.dims.d_model
    act = torch_act(wl)
    out = torch.empty(B * qn * d, dtype=act, device=dev)
    ws = torch.zeros(M.mla_output_proj_workspace_size(cfg, B * qn), dtype=torch.uint8, device=dev)
    M.mla_output_proj(cfg, r["out_latent_dev"], st["W_comb"], out, ws)
    torch.cuda.synchronize()
    wts = st["weights"]
    exp_o, exp_l, exp_out = [], [], []
    for b in range(B):
        e = expected_request_decompressed(wl, b, wts, r["q"], list(range(H)))
        exp_o.append(e["o_lat"])
        exp_l.append(e["lse"])
        exp_out.append(oracle.mha_output(e["u"], wts["W_O"]))
    return {"out_latent": r["out_latent"], "lse": r["lse"],
            "out": out.float().cpu().numpy().astype(np.float64).reshape(B, qn, d),
            "expected": {"out_latent": np.stack(exp_o), "lse": np.stack(exp_l),
                         "out": np.stack(exp_out).reshape(B, qn, d)}}


def run_small_step_v2_bf16(dev):
    """Smoke path on the tensor cores: DeepSeek-V2 head shapes in bf16, two short requests
    whose last two tokens come from h (the cluster-GEMM append), a decode on the tcgen05
    kernel with split work, and the unfolded output projection of the two rows. Returns the
    device results and the fp64 oracle's expectations for the same inputs."""
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (70, 130), name="v2_smoke", new_from_h=2)
    st = build_state(wl, dev)
    r = run_decode(wl, st, dev, kernel=M.KERNEL_TC, num_workers=3)
    cfg = st["cfg"]
    B, H, d = wl.batch, wl.dims.num_heads, wl.dims.d_model
    wts = st["weights"]
    out = torch.empty(B * d, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(M.mla_output_proj_unfolded_workspace_size(cfg, B), dtype=torch.uint8, device=dev)
    M.mla_output_proj_unfolded(cfg, r["out_latent_dev"], st["dw"]["W_UV"], st["dw"]["W_O"], out, ws)
    torch.cuda.synchronize()
    W_UK_abs64 = np.stack([wts["W_UK"][:, i * 128:(i + 1) * 128].T.astype(np.float64) for i in range(H)])
    exp_o, exp_l = [], []
    for b in range(B):
        o, l = expected_request(wl, b, wts, r["q"], W_UK_abs64)
        exp_o.append(o)
        exp_l.append(l)
    exp_o = np.stack(exp_o)
    u = oracle.lift_latent(r["out_latent"].reshape(B, H * 512), wts["W_UV"], H)
    exp_out = oracle.mha_output(u, wts["W_O"])
    return {"wl": wl, "status": r["status"], "out_latent": r["out_latent"], "lse": r["lse"],
            "out": out.float().cpu().numpy().astype(np.float64).reshape(B, d),
            "expected": {"out_latent": exp_o, "lse": np.stack(exp_l), "out": exp_out}}
