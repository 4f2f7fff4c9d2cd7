"""mla_decode_noalloc, the decode call that uses the library's own fixed device scratch
array instead of a workspace the caller allocates (for callers that cannot call
cudaMalloc when they decode). Kept in its own file, collected last, so that a run that
stops at the first failure has already run every other test.

Checks, through the C ABI, that two calls in a row give the same latent output and LSE
as mla_decode with a caller workspace, within the bf16 parity tolerance of the other
tests (1e-2 max|ref| + 1e-3), and that an oversized batch is refused."""
import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_04_gb300 as M
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_noalloc_matches_workspace_decode_twice():
    wl = W.scaled(W.WORKLOADS["v2_b32_s4096"], (700, 64, 2, 2000, 0), name="noalloc", q_len=2,
                  new_from_h=2)
    st = Hn.build_state(wl, DEV)
    q = W.queries(wl)
    ref = Hn.run_decode(wl, st, DEV, q=q)        # mla_decode, caller-provided workspace
    assert ref["status"] == M.MLA_OK
    act = Hn.torch_act(wl)
    B, qn, H, d_c = wl.batch, wl.q_len, 128, 512
    qn_d = Hn.to_dev(q["q_nope"], act, DEV)
    qp_d = Hn.to_dev(q["q_pe"], act, DEV)
    for call in range(2):
        out = torch.full((B * qn * H * d_c,), float("nan"), dtype=act, device=DEV)
        lse = torch.full((B * qn * H,), float("nan"), dtype=torch.float32, device=DEV)
        M.mla_decode_noalloc(st["cfg"], qn_d, qp_d, st["W_UK_abs"], st["cache"], st["bt_d"],
                             st["seq_lens_d"], out, lse)
        torch.cuda.synchronize()
        got_o = out.float().cpu().numpy().astype(np.float64).reshape(B, qn, H, d_c)
        got_l = lse.cpu().numpy().astype(np.float64).reshape(B, qn, H)
        for got, exp, what in ((got_o, ref["out_latent"], "out_latent"), (got_l, ref["lse"], "lse")):
            err = Hn.max_err(got, exp)
            tol = Hn.tolerance(wl, exp)
            assert err <= tol, f"call {call} {what}: max err {err:.3e} > {tol:.3e}"


def test_noalloc_refuses_batches_beyond_its_array():
    cfg = M.make_config(W.V2, "bf16", "bf16")
    need = M.mla_decode_workspace_size(cfg, 4096, 2)
    assert need > 64 << 20
    fake = ctypes.c_void_p(256)       # never dereferenced: the size check comes first
    st = M.lib().mla_decode_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, 1, fake, 1, fake,
                                    4096, 2, fake, fake, None)
    assert st == M.MLA_ERR_WORKSPACE
    assert "64" in M.mla_last_error() or "scratch" in M.mla_last_error()
