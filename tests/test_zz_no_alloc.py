"""mla_decode_noalloc, the decode call that uses the library's own fixed device scratch
array instead of a workspace the caller allocates (for callers that cannot call
cudaMalloc when they decode: a plugin inside a runtime that owns every device
allocation, a serving loop whose memory footprint is frozen after warm-up). Kept in its
own file, collected last, so that a run that stops at the first failure has already run
every other test.

Through the C ABI: two calls in a row, after a call on another batch has left its own
contents in the array, give bit for bit the latent output and LSE of mla_decode with a
caller workspace, and both match the fp64 oracle within the bf16 tolerance of the other
tests (1e-2 max|ref| + 1e-3); the device status of each call reads back through
mla_decode_noalloc_status; an oversized batch is refused."""
import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_04_gb300 as M
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _noalloc(st, wl, q, act):
    B, qn, H, d_c = wl.batch, wl.q_len, 128, 512
    out = torch.full((B * qn * H * d_c,), float("nan"), dtype=act, device=DEV)
    lse = torch.full((B * qn * H,), float("nan"), dtype=torch.float32, device=DEV)
    M.mla_decode_noalloc(st["cfg"], Hn.to_dev(q["q_nope"], act, DEV), Hn.to_dev(q["q_pe"], act, DEV),
                         st["W_UK_abs"], st["cache"], st["bt_d"], st["seq_lens_d"], out, lse)
    code = M.mla_decode_noalloc_status()
    return out, lse, code


def test_noalloc_matches_workspace_decode_and_oracle_twice():
    act = torch.bfloat16
    # another batch first, so the array holds a different plan, query and partials
    other = W.scaled(W.WORKLOADS["v2_b32_s4096"], (3000, 5, 1, 640), name="noalloc_other")
    st_o = Hn.build_state(other, DEV)
    _, _, code = _noalloc(st_o, other, W.queries(other), act)
    assert code == M.MLA_OK
    del st_o

    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (700, 64, 2, 2000, 0), name="noalloc", q_len=2,
                  new_from_h=2)
    st = Hn.build_state(wl, DEV)
    q = W.queries(wl)
    ref = Hn.run_decode(wl, st, DEV, q=q)        # mla_decode, caller-provided workspace
    assert ref["status"] == M.MLA_OK
    B, qn, H, d_c = wl.batch, wl.q_len, 128, 512
    W_UK_abs64 = np.stack([st["weights"]["W_UK"][:, i * 128:(i + 1) * 128].T.astype(np.float64)
                           for i in range(H)])
    exp = [Hn.expected_request(wl, b, st["weights"], q, W_UK_abs64) for b in range(B)]
    exp_o = np.stack([e[0] for e in exp])
    exp_l = np.stack([e[1] for e in exp])
    for call in range(2):
        out, lse, code = _noalloc(st, wl, q, act)
        assert code == M.MLA_OK, f"call {call}: device status {code}"
        # same kernels, same plan, same inputs: the same bits as the workspace decode
        assert torch.equal(out.view(torch.int16), ref["out_latent_dev"].view(torch.int16)), \
            f"call {call}: latent output differs from mla_decode's"
        got_o = out.float().cpu().numpy().astype(np.float64).reshape(B, qn, H, d_c)
        got_l = lse.cpu().numpy().astype(np.float64).reshape(B, qn, H)
        assert np.array_equal(got_l, ref["lse"], equal_nan=False)
        for got, e, what in ((got_o, exp_o, "out_latent"), (got_l, exp_l, "lse")):
            err = Hn.max_err(got, e)
            tol = Hn.tolerance(wl, e)
            assert err <= tol, f"call {call} {what} vs oracle: max err {err:.3e} > {tol:.3e}"


def test_noalloc_status_reports_device_guards():
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (100, 70), name="noalloc_guard")
    st = Hn.build_state(wl, DEV)
    bad = st["bt"].copy()
    bad[1, 1] = st["num_pages"] + 5               # request 1: a page id past the cache
    st2 = dict(st)
    st2["bt_d"] = Hn.to_dev(bad, torch.int32, DEV)
    _, _, code = _noalloc(st2, wl, W.queries(wl), torch.bfloat16)
    assert code == M.MLA_ERR_DEVICE_GUARD
    assert M.mla_decode_noalloc_status() == M.MLA_OK     # read once, then cleared


def test_noalloc_refuses_batches_beyond_its_array():
    cfg = M.make_config(W.V2, "bf16", "bf16")
    need = M.mla_decode_workspace_size(cfg, 4096, 2)
    assert need > 64 << 20
    fake = ctypes.c_void_p(256)       # never dereferenced: the size check comes first
    st = M.lib().mla_decode_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, 1, fake, 1, fake,
                                    4096, 2, fake, fake, None)
    assert st == M.MLA_ERR_WORKSPACE
    assert "64" in M.mla_last_error() or "scratch" in M.mla_last_error()
