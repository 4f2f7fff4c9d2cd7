"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same
seeded inputs. Tolerances: max|err| <= 1e-5 max|ref| for fp32, <= 1e-2 max|ref| + 1e-3
for bf16/fp8 (per tensor: latent output, LSE, projected output); cache placement is
bit-exact."""
import numpy as np
import pytest
import torch

import mla_latent_kv_04_gb300 as M
import oracle
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
KERNELS = [M.KERNEL_SIMT, M.KERNEL_TC]


def _kernel_id(k):
    return {M.KERNEL_SIMT: "simt", M.KERNEL_TC: "tcgen05"}[k]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    M.lib()


def _check(wl, got, ref, what):
    err = Hn.max_err(got, ref)
    tol = Hn.tolerance(wl, ref)
    assert err <= tol, f"{wl.name} {what}: max err {err:.3e} > tol {tol:.3e}"
    return err


def _check_all_requests(wl, st, r, requests=None, heads=None):
    W_UK_abs64 = oracle.absorb_weights(st["weights"]["W_UK"], st["weights"]["W_UV"],
                                       st["weights"]["W_O"], wl.dims.num_heads)[0]
    requests = range(wl.batch) if requests is None else requests
    hs = list(range(wl.dims.num_heads)) if heads is None else list(heads)
    got_o, got_l, exp_o, exp_l = [], [], [], []
    for b in requests:
        o, l = Hn.expected_request(wl, b, st["weights"], r["q"], W_UK_abs64, heads=hs,
                                   cache_scale=st["cfg"].cache_scale)
        exp_o.append(o)
        exp_l.append(l)
        got_o.append(r["out_latent"][b][:, hs])
        got_l.append(r["lse"][b][:, hs])
    e1 = _check(wl, np.stack(got_o), np.stack(exp_o), "out_latent")
    e2 = _check(wl, np.stack(got_l), np.stack(exp_l), "lse")
    return e1, e2


# ----------------------------------------------------------------------------- tiny fp32

def test_tiny_f32_full_path():
    wl = W.WORKLOADS["tiny_f32"]
    res = Hn.run_full_step_tiny(wl, DEV)
    for key in ("out_latent", "lse", "out"):
        _check(wl, res[key], res["expected"][key], key)


def test_tiny_f32_ragged_multi_request():
    wl = W.scaled(W.WORKLOADS["tiny_f32"], (1, 64, 65, 190, 0, 7), name="tiny_ragged", q_len=1)
    st = Hn.build_state(wl, DEV)
    r = Hn.run_decode(wl, st, DEV, kernel=M.KERNEL_SIMT, num_workers=5)
    assert r["status"] == M.MLA_OK
    _check_all_requests(wl, st, r)


# ----------------------------------------------------------------------------- V2 bf16, small

SMALL_Q1 = (1, 2, 63, 64, 65, 130, 700, 0)
SMALL_Q2 = (2, 3, 64, 65, 129, 0, 517)
# several causal query tokens per request (speculative decoding); q 64 is a chunk of a
# chunked prefill. Lengths include steps whose every token is new (seq_len == q_len).
SMALL_Q4 = (4, 5, 64, 67, 0, 300)
SMALL_Q8 = (8, 71, 128, 513)
CHUNK_Q64 = (64, 65, 190)


@pytest.mark.parametrize("kernel", KERNELS, ids=_kernel_id)
@pytest.mark.parametrize("q_len,lens", [(1, SMALL_Q1), (2, SMALL_Q2), (4, SMALL_Q4), (8, SMALL_Q8),
                                        (64, CHUNK_Q64)], ids=["q1", "q2", "q4", "q8", "q64"])
def test_v2_bf16_small_ragged(kernel, q_len, lens):
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], lens, name=f"v2_small_q{q_len}", q_len=q_len,
                  new_from_h=q_len)
    st = Hn.build_state(wl, DEV)
    r = Hn.run_decode(wl, st, DEV, kernel=kernel)
    assert r["status"] == M.MLA_OK
    _check_all_requests(wl, st, r)
    # empty request: zeros and -inf
    for b, s in enumerate(lens):
        if s == 0:
            assert not r["out_latent"][b].any() and np.isneginf(r["lse"][b]).all()


@pytest.mark.parametrize("kernel", KERNELS, ids=_kernel_id)
def test_split_count_invariance(kernel):
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (1000, 333, 64, 2049), name="v2_splits")
    st = Hn.build_state(wl, DEV)
    q = W.queries(wl)
    outs = []
    for nw in (1, 2, 7, 33, 200):
        r = Hn.run_decode(wl, st, DEV, q=q, kernel=kernel, num_workers=nw)
        assert r["status"] == M.MLA_OK
        _check_all_requests(wl, st, r)
        outs.append(r)
    for r in outs[1:]:
        d = np.max(np.abs(r["out_latent"] - outs[0]["out_latent"]))
        assert d <= 1e-2 * np.max(np.abs(outs[0]["out_latent"])) + 1e-3


@pytest.mark.parametrize("kernel", KERNELS, ids=_kernel_id)
@pytest.mark.parametrize("wl_name", ["v2_fp8_b128_s8192", "v2_fp8block_b128_s8192"],
                         ids=["per_tensor", "block128"])
def test_fp8_cache_small(kernel, wl_name):
    # partial pages, several pages, splits; e4m3 codes in the cache with one per-tensor scale,
    # or one scale per 128 latent elements of each token and k_pe in bf16
    wl = W.scaled(W.WORKLOADS[wl_name], (5, 64, 300, 1, 1000), name=wl_name + "_small")
    st = Hn.build_state(wl, DEV)
    for nw in (0, 3):
        r = Hn.run_decode(wl, st, DEV, kernel=kernel, num_workers=nw)
        assert r["status"] == M.MLA_OK
        _check_all_requests(wl, st, r)


def test_decompressed_oracle_agrees_on_gpu_inputs():
    # the explicit-decompression oracle (textbook MHA) on a few heads of the GPU run
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (77, 300), name="v2_decomp", q_len=2, new_from_h=2)
    st = Hn.build_state(wl, DEV)
    r = Hn.run_decode(wl, st, DEV)
    heads = [0, 1, 63, 127]
    for b in range(wl.batch):
        e = Hn.expected_request_decompressed(wl, b, st["weights"], r["q"], heads)
        _check(wl, r["out_latent"][b][:, heads], e["o_lat"], "out_latent (decompressed oracle)")
        _check(wl, r["lse"][b][:, heads], e["lse"], "lse (decompressed oracle)")


@pytest.mark.parametrize("rows", [3, 32, 512])
def test_output_projection_bf16(rows):
    # 32 rows: the batch-32 step; 512 rows: the ragged speculative step (256 x 2 tokens)
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (5, 9, 130), name="v2_oproj")
    st = Hn.build_state(wl, DEV)
    cfg = st["cfg"]
    rng = np.random.default_rng(5)
    o_lat = W.round_bf16((rng.standard_normal((rows, 128 * 512)) * 0.1).astype(np.float32))
    o_d = Hn.to_dev(o_lat, torch.bfloat16, DEV)
    out = torch.empty(rows * 5120, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(M.mla_output_proj_workspace_size(cfg, rows), dtype=torch.uint8, device=DEV)
    M.mla_output_proj(cfg, o_d, st["W_comb"], out, ws)
    torch.cuda.synchronize()
    _, W_comb64 = oracle.absorb_weights(st["weights"]["W_UK"], st["weights"]["W_UV"],
                                        st["weights"]["W_O"], 128)
    ref = oracle.output_projection(o_lat, W_comb64)
    got = out.float().cpu().numpy().reshape(rows, 5120)
    _check(wl, got, ref, "output projection")
    # the folded weights themselves (bf16-rounded fold of the same inputs)
    got_w = st["W_comb"].float().cpu().numpy().reshape(128 * 512, 5120)
    assert np.max(np.abs(got_w - W_comb64)) <= 1e-2 * np.max(np.abs(W_comb64)) + 1e-3
    got_a = st["W_UK_abs"].float().cpu().numpy().reshape(128, 128, 512)
    ref_a = oracle.absorb_weights(st["weights"]["W_UK"], st["weights"]["W_UV"], st["weights"]["W_O"],
                                  128)[0]
    assert np.array_equal(got_a, ref_a)           # a pure relayout: exact


def test_fold_every_element_at_v2_shapes():
    # mla_absorb_weights with bf16 weights at DeepSeek-V2 shapes (the tensor-core GEMM):
    # every element of W_comb = W_i^UV W_i^O (huny.dev §3-2) is the fp64 fold of the same
    # bf16 inputs rounded once to bf16 (|err| <= 2^-8 |ref|), up to the fp32 accumulation of
    # its 128 products (|err| <= 2^-16 sum_k |W_UV| |W_O|, far above the fp32 bound).
    wl = W.WORKLOADS["v2_b32_s4096"]
    H = wl.dims.num_heads
    wts = W.weights(wl)
    dw = {k: Hn.to_dev(v, torch.bfloat16, DEV) for k, v in wts.items() if k != "W_DKV_KR"}
    W_UK_abs = torch.empty(H * 128 * 512, dtype=torch.bfloat16, device=DEV)
    W_comb = torch.full((H * 512 * 5120,), float("nan"), dtype=torch.bfloat16, device=DEV)
    cfg = Hn.config(wl)
    M.mla_absorb_weights(cfg, dw["W_UK"], dw["W_UV"], dw["W_O"], W_UK_abs, W_comb)
    torch.cuda.synchronize()
    got = W_comb.float().cpu().numpy().astype(np.float64).reshape(H * 512, 5120)
    ref = oracle.absorb_weights(wts["W_UK"], wts["W_UV"], wts["W_O"], H)[1]
    mag = oracle.absorb_weights(np.abs(wts["W_UK"]), np.abs(wts["W_UV"]), np.abs(wts["W_O"]), H)[1]
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -16 * mag
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, f"{len(bad)} elements off, first {bad[0]}: got {got[tuple(bad[0])]}, " \
                          f"ref {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("wl_name,rows", [("v2_b32_s4096", 3), ("v2_b32_s4096", 40),
                                          ("tiny_f32", 5)])
def test_output_projection_unfolded(wl_name, rows):
    # huny.dev §3-2 read before the fold: u_i = o_i W_i^UV, out = sum_i u_i W_i^O; the bf16
    # path runs the tensor-core GEMMs (u rounded to bf16), the fp32 path the SIMT ones
    base = W.WORKLOADS[wl_name]
    wl = W.scaled(base, (5, 9) if wl_name != "tiny_f32" else (7,), name=wl_name + "_unfold")
    st = Hn.build_state(wl, DEV)
    cfg = st["cfg"]
    H, d_c, d = wl.dims.num_heads, wl.dims.d_latent, wl.dims.d_model
    act = Hn.torch_act(wl)
    rng = np.random.default_rng(6)
    o_lat = (rng.standard_normal((rows, H * d_c)) * 0.1).astype(np.float32)
    if wl.act != "f32":
        o_lat = W.round_bf16(o_lat)
    o_d = Hn.to_dev(o_lat, act, DEV)
    out = torch.empty(rows * d, dtype=act, device=DEV)
    ws = torch.zeros(M.mla_output_proj_unfolded_workspace_size(cfg, rows), dtype=torch.uint8,
                     device=DEV)
    M.mla_output_proj_unfolded(cfg, o_d, st["dw"]["W_UV"], st["dw"]["W_O"], out, ws)
    torch.cuda.synchronize()
    wts = st["weights"]
    ref = oracle.mha_output(oracle.lift_latent(o_lat, wts["W_UV"], H), wts["W_O"])
    got = out.float().cpu().numpy().astype(np.float64).reshape(rows, d)
    _check(wl, got, ref, "unfolded output projection")


# ----------------------------------------------------------------------------- query side

@pytest.mark.parametrize("wl_name,rows", [("v2_b32_s4096", 3), ("v2_b32_s4096", 40),
                                          ("tiny_f32", 5)], ids=["v2_3rows", "v2_40rows", "tiny_f32"])
def test_query_from_hidden(wl_name, rows):
    # c^Q = h W^DQ, q^C_i = c^Q W_i^UQ, un-rotated q^R_i = h W_i^QR against the oracle
    wl = W.WORKLOADS[wl_name]
    d = wl.dims
    H = d.num_heads
    cfg = Hn.config(wl)
    act = Hn.torch_act(wl)
    qw = W.query_weights(wl)
    h = W.query_hidden(wl, rows)
    dw = {k: Hn.to_dev(v, act, DEV) for k, v in qw.items()}
    q_nope = torch.empty(rows * H * d.d_nope, dtype=act, device=DEV)
    q_pe = torch.empty(rows * H * d.d_rope, dtype=act, device=DEV)
    ws = torch.zeros(M.mla_query_workspace_size(cfg, d.d_q, rows), dtype=torch.uint8, device=DEV)
    M.mla_query_from_hidden(cfg, d.d_q, Hn.to_dev(h, act, DEV), dw["W_DQ"], dw["W_UQ"], dw["W_QR"],
                            q_nope, q_pe, ws)
    torch.cuda.synchronize()
    ref_n, ref_p, _ = oracle.compress_query(h, qw["W_DQ"], qw["W_UQ"], qw["W_QR"], H)
    got_n = q_nope.float().cpu().numpy().astype(np.float64).reshape(rows, H, d.d_nope)
    got_p = q_pe.float().cpu().numpy().astype(np.float64).reshape(rows, H, d.d_rope)
    _check(wl, got_n, ref_n, "q_nope from h")
    _check(wl, got_p, ref_p, "q_pe from h")


# ----------------------------------------------------------------------------- placement

@pytest.mark.parametrize("wl_name", ["tiny_f32", "v2_b32_s4096", "v2_fp8_b128_s8192",
                                     "v2_fp8block_b128_s8192"])
def test_append_placement_is_bit_exact(wl_name):
    base = W.WORKLOADS[wl_name]
    wl = W.scaled(base, (70, 1, 128, 200), name=wl_name + "_place")
    cfg = Hn.config(wl, cache_scale=0.0173 if wl.cache == "fp8_e4m3" else None)
    bt, num_pages = W.page_table(wl)
    cache = Hn.alloc_cache(wl, num_pages, DEV)
    bt_d = Hn.to_dev(bt, torch.int32, DEV)
    act = Hn.torch_act(wl)
    rows_c, rows_k, reqs, poss = [], [], [], []
    rng = np.random.default_rng(11)
    for b, S in enumerate(wl.seq_lens):
        c, k = W.latent_rows(wl, b, S)
        req, pos = W.append_batch(wl, b, 0, S)
        keep = rng.random(S) < 0.7          # leave holes: unwritten slots keep the sentinel
        rows_c.append(c[keep]); rows_k.append(k[keep]); reqs.append(req[keep]); poss.append(pos[keep])
    c = np.concatenate(rows_c); k = np.concatenate(rows_k)
    req = np.concatenate(reqs); pos = np.concatenate(poss)
    perm = rng.permutation(len(req))                # arbitrary row order
    c, k, req, pos = c[perm], k[perm], req[perm], pos[perm]
    M.mla_append_cache_latent(cfg, Hn.to_dev(c, act, DEV), Hn.to_dev(k, act, DEV),
                              Hn.to_dev(req, torch.int32, DEV), Hn.to_dev(pos, torch.int32, DEV), bt_d,
                              cache, rotate=False)
    torch.cuda.synchronize()
    rows = np.concatenate([c, k], axis=1)
    D = wl.dims.d_cache
    if wl.cache == "fp8_e4m3_b128":
        # [codes | fp32 block scales | bf16 k_pe] bytes, the oracle's quantiser on the same values
        codes, scales = oracle.e4m3_block_quantize(c.astype(np.float32), 128)
        kb = (k.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        enc = np.concatenate([codes, scales.astype(np.float32).view(np.uint8),
                              kb.view(np.uint8)], axis=1)
        got = cache.cpu().numpy()
        fill = np.uint8(Hn.SENTINEL["fp8_e4m3_b128"])
        D = W.cache_row_bytes(wl)
    elif wl.cache == "f32":
        enc = rows.astype(np.float32).view(np.uint32)
        got = cache.view(torch.int32).cpu().numpy().view(np.uint32)
        fill = np.uint32(Hn.SENTINEL["f32"])
    elif wl.cache == "bf16":
        enc = (rows.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        got = cache.view(torch.int16).cpu().numpy().view(np.uint16)
        fill = np.uint16(Hn.SENTINEL["bf16"])
    else:
        s = np.float32(cfg.cache_scale)
        enc = oracle.e4m3_encode(rows.astype(np.float32) / s)
        got = cache.cpu().numpy()
        fill = np.uint8(Hn.SENTINEL["fp8_e4m3"])
    exp = oracle.cache_image(num_pages, wl.dims.page_size, enc, req, pos, bt, fill)
    assert np.array_equal(got.reshape(num_pages, wl.dims.page_size, D), exp)


def test_append_from_h_values():
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (3, 66), name="v2_append_h", fill="h")
    st = Hn.build_state(wl, DEV)
    got = st["cache"].float().cpu().numpy().reshape(st["num_pages"], 64, 576)
    for b, S in enumerate(wl.seq_lens):
        c, k = Hn.cached_rows(wl, b, st["weights"])
        rows = np.concatenate([c, k], axis=1)
        for p in range(S):
            g = got[st["bt"][b, p // 64], p % 64]
            assert np.max(np.abs(g - rows[p])) <= 1e-2 * np.max(np.abs(rows)) + 1e-3


def _nearest_e4m3_ok(codes, v, slack):
    """Each e4m3 code is a nearest code (saturating at 448) to some value within ``slack`` of
    the exact value v, all in code units: the device rounds its fp32 result, which differs
    from v by at most the slack, so where v lies that close to the midpoint of two codes
    either one is accepted. The sign must match unless the code is zero."""
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))     # increasing
    a = np.minimum(np.abs(v), 448.0)
    i = np.searchsorted(table, a)
    best = np.minimum(np.abs(table[np.minimum(i, len(table) - 1)] - a),
                      np.abs(table[np.maximum(i - 1, 0)] - a))
    got = oracle.e4m3_decode(codes)
    ok_sign = (got == 0) | (np.sign(got) == np.sign(v))
    return ok_sign & (np.abs(np.abs(got) - a) <= best + 2.0 * slack)


@pytest.mark.parametrize("cache_kind", ["bf16", "fp8_e4m3", "fp8_e4m3_b128"])
def test_append_prefill_chunks_from_h(cache_kind):
    # Chunked prefill: every position of three requests comes from h through the append
    # projection, in two calls of 1500 and 501 rows whose rows mix the requests in random
    # order. The projection GEMM spans several 256-token tiles and a ragged tail.
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (700, 1, 1300), name="v2_prefill_" + cache_kind,
                  fill="h", cache=cache_kind)
    fp8 = cache_kind == "fp8_e4m3"
    cfg = Hn.config(wl, cache_scale=6.0 / 448.0 if fp8 else None)
    act = Hn.torch_act(wl)
    wts = W.weights(wl)
    W_d = Hn.to_dev(wts["W_DKV_KR"], act, DEV)
    bt, num_pages = W.page_table(wl)
    cache = Hn.alloc_cache(wl, num_pages, DEV)
    bt_d = Hn.to_dev(bt, torch.int32, DEV)
    hs, reqs, poss = [], [], []
    for b, S in enumerate(wl.seq_lens):
        hs.append(W.hidden(wl, b, S))
        r_, p_ = W.append_batch(wl, b, 0, S)
        reqs.append(r_)
        poss.append(p_)
    h, req, pos = np.concatenate(hs), np.concatenate(reqs), np.concatenate(poss)
    perm = np.random.default_rng(12).permutation(len(req))
    h, req, pos = h[perm], req[perm], pos[perm]
    status = torch.zeros(4, dtype=torch.int32, device=DEV)
    for lo, hi in ((0, 1500), (1500, len(req))):
        ws = torch.empty(M.mla_append_cache_workspace_size(cfg, hi - lo), dtype=torch.uint8, device=DEV)
        M.mla_append_cache(cfg, Hn.to_dev(h[lo:hi], act, DEV), W_d,
                           Hn.to_dev(req[lo:hi], torch.int32, DEV), Hn.to_dev(pos[lo:hi], torch.int32, DEV),
                           bt_d, cache, dev_status=status, workspace=ws)
    assert M.mla_read_device_status(status) == M.MLA_OK
    D, P = wl.dims.d_cache, wl.dims.page_size
    d_c = wl.dims.d_latent
    if cache_kind == "fp8_e4m3_b128":
        raw = cache.cpu().numpy().reshape(num_pages, P, W.cache_row_bytes(wl))
        fill = np.uint8(Hn.SENTINEL["fp8_e4m3_b128"])
    elif fp8:
        raw = cache.cpu().numpy().reshape(num_pages, P, D)
        fill = np.uint8(Hn.SENTINEL["fp8_e4m3"])
    else:
        raw = cache.view(torch.int16).cpu().numpy().view(np.uint16).reshape(num_pages, P, D)
        fill = np.uint16(Hn.SENTINEL["bf16"])
    written = np.zeros((num_pages, P), bool)
    for b, S in enumerate(wl.seq_lens):
        c, kraw = oracle.project_latent(W.hidden(wl, b, S).astype(np.float64), wts["W_DKV_KR"],
                                        wl.dims.d_latent)
        ref = np.concatenate([c, oracle.rope(kraw, np.arange(S), wl.rope_theta)], axis=1)
        pg, sl = bt[b, np.arange(S) // P], np.arange(S) % P
        written[pg, sl] = True
        if cache_kind == "fp8_e4m3_b128":
            rows_b = raw[pg, sl]
            scales = np.ascontiguousarray(rows_b[:, d_c:d_c + d_c // 32]).view(np.float32).astype(np.float64)
            hb = np.abs(W.hidden(wl, b, S)).astype(np.float64) @ np.abs(wts["W_DKV_KR"]).astype(np.float64)
            # each block's scale is the device's fp32 amax / 448: within the fp32 error of the
            # largest element's dot product of the exact one
            amax = np.abs(ref[:, :d_c]).reshape(S, -1, 128).max(axis=2)
            bound = hb[:, :d_c].reshape(S, -1, 128).max(axis=2)
            assert (np.abs(scales * 448.0 - amax) <= 1e-6 * bound + 1e-6 * amax).all()
            v = ref[:, :d_c] / np.repeat(scales, 128, axis=1)
            slack = 1e-6 * hb[:, :d_c] / np.repeat(scales, 128, axis=1) + 1e-5 * np.abs(v)
            ok = _nearest_e4m3_ok(rows_b[:, :d_c], v, slack)
            assert ok.all(), f"request {b}: {int((~ok).sum())} codes are not a nearest e4m3 code"
            kbits = np.ascontiguousarray(rows_b[:, d_c + d_c // 32:]).view(np.uint16).astype(np.uint32) << 16
            _check(wl, kbits.view(np.float32).astype(np.float64), ref[:, d_c:], f"k_pe rows of request {b}")
        elif fp8:
            # fp32 error of the device's dot products: a small multiple of the unit roundoff
            # times sum_k |h_k W_kj| (the rotation adds the bounds of a pair), plus the
            # rotation's own relative error
            hb = np.abs(W.hidden(wl, b, S)).astype(np.float64) @ np.abs(wts["W_DKV_KR"]).astype(np.float64)
            kb = np.repeat(hb[:, wl.dims.d_latent::2] + hb[:, wl.dims.d_latent + 1::2], 2, axis=1)
            v = ref / cfg.cache_scale
            slack = 1e-6 * np.concatenate([hb[:, :wl.dims.d_latent], kb], axis=1) / cfg.cache_scale
            ok = _nearest_e4m3_ok(raw[pg, sl], v, slack + 1e-5 * np.abs(v))
            assert ok.all(), f"request {b}: {int((~ok).sum())} codes are not a nearest e4m3 code"
        else:
            got = raw[pg, sl].astype(np.uint32) << 16
            got = got.view(np.float32).astype(np.float64)
            _check(wl, got, ref, f"cache rows of request {b}")
    assert (raw[~written] == fill).all(), "a slot no append wrote lost its sentinel"


# ----------------------------------------------------------------------------- guards

def test_device_guard_skips_bad_pages_and_lengths():
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (100, 70, 64), name="v2_guard")
    st = Hn.build_state(wl, DEV)
    bad_bt = st["bt"].copy()
    bad_bt[1, 1] = st["num_pages"] + 5          # request 1: a page id past the cache
    st2 = dict(st)
    st2["bt_d"] = Hn.to_dev(bad_bt, torch.int32, DEV)
    sl = np.array(wl.seq_lens, np.int32)
    sl[2] = 64 * bad_bt.shape[1] + 1            # request 2: longer than its block-table row
    st2["seq_lens_d"] = Hn.to_dev(sl, torch.int32, DEV)
    r = Hn.run_decode(wl, st2, DEV)
    assert r["status"] == M.MLA_ERR_DEVICE_GUARD
    _check_all_requests(wl, st, r, requests=[0])         # the clean request is untouched
    assert not r["out_latent"][2].any() and np.isneginf(r["lse"][2]).all()
    # append with a bad request id: the row is skipped and flagged, nothing else changes
    status = torch.zeros(4, dtype=torch.int32, device=DEV)
    before = st["cache"].clone()
    c = torch.zeros(512, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    M.mla_append_cache_latent(st["cfg"], c, k, torch.tensor([7], dtype=torch.int32, device=DEV),
                              torch.tensor([0], dtype=torch.int32, device=DEV), st["bt_d"], st["cache"],
                              dev_status=status)
    assert M.mla_read_device_status(status) == M.MLA_ERR_DEVICE_GUARD
    assert torch.equal(before.view(torch.int16), st["cache"].view(torch.int16))


# ----------------------------------------------------------------------------- full sizes

FULL = ["v2_b32_s4096", "v2_long_splitkv", "v2_ragged_spec", "v2_fp8_b128_s8192", "v2_spec_q4",
        "v2_fp8block_b128_s8192"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_request_and_head(name):
    # each workload at its full size, in the launch configuration bench.py times (default
    # kernel, default split plan), every request, query token and head against the absorbed
    # fp64 oracle (itself pinned to the decompressed route)
    wl = W.WORKLOADS[name]
    st = Hn.build_state(wl, DEV)
    r = Hn.run_decode(wl, st, DEV)
    assert r["status"] == M.MLA_OK
    _check_all_requests(wl, st, r)
    del st
    torch.cuda.empty_cache()


def test_prologue_fallback_for_thousands_of_requests():
    # 2100 single-token requests: a split plan too large for the query-absorption GEMM
    # block's shared memory (above 1981 groups at 76 workers), so the planner and the q_pe
    # rotation run in their own kernel ahead of the GEMM
    lens = np.random.default_rng(31).integers(1, 257, size=2100)
    lens[::97] = 0                                   # a few empty requests among them
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], tuple(int(x) for x in lens), name="v2_many",
                  spare_pages=3)
    st = Hn.build_state(wl, DEV)
    for nw in (0, 40):
        r = Hn.run_decode(wl, st, DEV, num_workers=nw)
        assert r["status"] == M.MLA_OK
        _check_all_requests(wl, st, r)
        empty = np.nonzero(lens == 0)[0]
        assert not r["out_latent"][empty].any() and np.isneginf(r["lse"][empty]).all()
