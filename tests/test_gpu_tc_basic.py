"""The tcgen05 decode kernel on small cases, from one page upwards, against the oracle and
against the SIMT kernel (same inputs, same plan)."""
import numpy as np
import pytest
import torch

import mla_latent_kv_04_gb300 as M
import oracle
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(lens, q_len=1, workers=1, new_from_h=0):
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], lens, name="tc_basic", q_len=q_len,
                  new_from_h=new_from_h)
    st = Hn.build_state(wl, DEV)
    q = W.queries(wl)
    r_tc = Hn.run_decode(wl, st, DEV, q=q, kernel=M.KERNEL_TC, num_workers=workers)
    assert r_tc["status"] == M.MLA_OK, r_tc["status"]
    W_UK_abs64 = oracle.absorb_weights(st["weights"]["W_UK"], st["weights"]["W_UV"],
                                       st["weights"]["W_O"], 128)[0]
    for b in range(wl.batch):
        o, l = Hn.expected_request(wl, b, st["weights"], q, W_UK_abs64)
        for got, ref, what in ((r_tc["out_latent"][b], o, "out_latent"), (r_tc["lse"][b], l, "lse")):
            err = Hn.max_err(got, ref)
            tol = Hn.tolerance(wl, ref)
            assert err <= tol, f"request {b} {what}: max err {err:.3e} > {tol:.3e}"
    return wl, st, q, r_tc


def test_tc_one_full_page():
    _run((64,))


def test_tc_one_partial_page():
    _run((5,))


def test_tc_several_pages_one_worker():
    _run((200,))


def test_tc_several_requests_and_splits():
    _run((300, 1000, 64, 1), workers=3)


def test_tc_matches_simt():
    wl, st, q, r_tc = _run((700, 129, 2048), workers=4)
    r_s = Hn.run_decode(wl, st, DEV, q=q, kernel=M.KERNEL_SIMT, num_workers=4)
    d = np.max(np.abs(r_tc["out_latent"] - r_s["out_latent"]))
    assert d <= 1e-2 * np.max(np.abs(r_s["out_latent"])) + 1e-3
    assert np.max(np.abs(r_tc["lse"] - r_s["lse"])) <= 1e-2 * np.max(np.abs(r_s["lse"])) + 1e-3


def _rescale_counts(s_log2, page):
    """Head-pages on which the running row maximum (started at each item's first page) grows
    by more than 2^8 in log2 units, the kernel's lazy rescale rule, for one item's scores."""
    pm = np.stack([s_log2[:, i:i + page].max(1) for i in range(0, s_log2.shape[1], page)], 1)
    m, n = pm[:, 0].copy(), 0
    for j in range(1, pm.shape[1]):
        up = pm[:, j] > m + 8.0
        n += int(up.sum())
        m = np.where(up, pm[:, j], m)
    return n


@pytest.mark.parametrize("workers", [1, 3])
def test_tc_rescale_on_growing_scores(workers):
    """Latent rows whose magnitude grows along the sequence (up to 7x) make the running row
    maximum rise by more than 2^8 many times inside one work item, so the kernel rescales O
    on those pages (the count is checked from the oracle's own scores); the output must
    still match the oracle, with and without split items."""
    lens = (1500, 700)
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], lens, name="tc_rescale")
    cfg = Hn.config(wl)
    act = torch.bfloat16
    wts = W.weights(wl)
    dw = {k: Hn.to_dev(v, act, DEV) for k, v in wts.items()}
    bt, num_pages = W.page_table(wl)
    cache = Hn.alloc_cache(wl, num_pages, DEV)
    bt_d = Hn.to_dev(bt, torch.int32, DEV)
    status = torch.zeros(4, dtype=torch.int32, device=DEV)
    rows = []
    for b, S in enumerate(wl.seq_lens):
        c, k = W.latent_rows(wl, b, S)
        ramp = (1.0 + 6.0 * np.arange(S) / S)[:, None]
        c = W.round_bf16((c * ramp).astype(np.float32))
        req, pos = W.append_batch(wl, b, 0, S)
        M.mla_append_cache_latent(cfg, Hn.to_dev(c, act, DEV), Hn.to_dev(k, act, DEV),
                                  Hn.to_dev(req, torch.int32, DEV), Hn.to_dev(pos, torch.int32, DEV),
                                  bt_d, cache, rotate=True, dev_status=status)
        k_rot = oracle.rope(k.astype(np.float64), np.arange(S), wl.rope_theta)
        rows.append((c.astype(np.float64), W.round_bf16(k_rot.astype(np.float32)).astype(np.float64)))
    assert M.mla_read_device_status(status) == M.MLA_OK
    H, d_c, d_n, d = wl.dims.num_heads, wl.dims.d_latent, wl.dims.d_nope, wl.dims.d_model
    W_UK_abs = torch.empty(H * d_n * d_c, dtype=act, device=DEV)
    W_comb = torch.empty(H * d_c * d, dtype=act, device=DEV)
    M.mla_absorb_weights(cfg, dw["W_UK"], dw["W_UV"], dw["W_O"], W_UK_abs, W_comb)
    st = {"cfg": cfg, "cache": cache, "bt_d": bt_d, "W_UK_abs": W_UK_abs,
          "seq_lens_d": Hn.to_dev(np.array(wl.seq_lens, np.int32), torch.int32, DEV)}
    q = W.queries(wl)
    r = Hn.run_decode(wl, st, DEV, q=q, kernel=M.KERNEL_TC, num_workers=workers)
    assert r["status"] == M.MLA_OK, r["status"]
    W_UK_abs64 = oracle.absorb_weights(wts["W_UK"], wts["W_UV"], wts["W_O"], H)[0]
    scale = oracle.softmax_scale(d_n, wl.dims.d_rope)
    rescales = 0
    for b, S in enumerate(wl.seq_lens):
        c, k_rot = rows[b]
        o, l = oracle.decode_absorbed(c, k_rot, q["q_nope"][b], q["q_pe"][b], W_UK_abs64, scale,
                                      wl.rope_theta)
        qh = oracle.absorbed_query(q["q_nope"][b], W_UK_abs64)[0]
        qr = oracle.rope(q["q_pe"][b][0], S - 1, wl.rope_theta)
        rescales += _rescale_counts((qh @ c.T + qr @ k_rot.T) * scale * np.log2(np.e), 64)
        for got, ref, what in ((r["out_latent"][b], o, "out_latent"), (r["lse"][b], l, "lse")):
            err = Hn.max_err(got, ref)
            tol = Hn.tolerance(wl, ref)
            assert err <= tol, f"request {b} {what}: max err {err:.3e} > {tol:.3e}"
    assert rescales > 100, rescales


@pytest.mark.parametrize("cache", ["bf16", "fp8_e4m3"])
def test_tc_wait_limit_reports_timeout_and_recovers(cache):
    # The kernel's failure path, exercised without any fault: worker 0's first page is never
    # loaded (a testing hook of mla_decode_opts), so one of its barrier waits runs out after
    # the 200 us limit. The kernel records MLA_ERR_TIMEOUT, every role leaves its loop, the
    # tensor memory is released and the CTA pair meets at its final barrier; the call's status
    # reads the timeout. The next call in the same process, without the hook, must match the
    # oracle (a leaked tensor-memory allocation or a stuck CTA would stall or break it).
    base = W.WORKLOADS["v2_b32_s4096"] if cache == "bf16" else W.WORKLOADS["v2_fp8_b128_s8192"]
    wl = W.scaled(base, (200, 130, 64), name="tc_timeout_" + cache)
    st = Hn.build_state(wl, DEV)
    q = W.queries(wl)
    act = torch.bfloat16
    B, H, d_c = wl.batch, 128, 512
    out = torch.empty(B * H * d_c, dtype=act, device=DEV)
    lse = torch.empty(B * H, dtype=torch.float32, device=DEV)
    ws = torch.zeros(M.mla_decode_workspace_size(st["cfg"], B, 1, num_workers=3, kernel=M.KERNEL_TC),
                     dtype=torch.uint8, device=DEV)
    M.mla_decode(st["cfg"], Hn.to_dev(q["q_nope"], act, DEV), Hn.to_dev(q["q_pe"], act, DEV),
                 st["W_UK_abs"], st["cache"], st["bt_d"], st["seq_lens_d"], out, lse, ws,
                 num_workers=3, kernel=M.KERNEL_TC, wait_limit_us=200, withhold_page=1)
    assert M.mla_read_device_status(ws) == M.MLA_ERR_TIMEOUT
    # the same process, the same buffers, no hook: a clean call that matches the oracle
    r = Hn.run_decode(wl, st, DEV, q=q, kernel=M.KERNEL_TC, num_workers=3)
    assert r["status"] == M.MLA_OK
    W_UK_abs64 = oracle.absorb_weights(st["weights"]["W_UK"], st["weights"]["W_UV"],
                                       st["weights"]["W_O"], 128)[0]
    for b in range(wl.batch):
        o, l = Hn.expected_request(wl, b, st["weights"], q, W_UK_abs64,
                                   cache_scale=st["cfg"].cache_scale)
        for got, ref, what in ((r["out_latent"][b], o, "out_latent"), (r["lse"][b], l, "lse")):
            err = Hn.max_err(got, ref)
            tol = Hn.tolerance(wl, ref)
            assert err <= tol, f"request {b} {what}: max err {err:.3e} > {tol:.3e}"
