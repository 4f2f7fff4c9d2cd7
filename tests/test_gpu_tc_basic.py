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
