"""The seeded input module: bf16 encoding, page tables and workload shapes."""
import numpy as np
import pytest

import workloads as W


def test_round_bf16_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000) * 3, rng.standard_normal(1000) * 1e-30,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8], np.float32)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(W.round_bf16(x), ref)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_page_table_is_a_partition(name):
    wl = W.WORKLOADS[name]
    bt, num_pages = W.page_table(wl)
    used = []
    for b in range(wl.batch):
        n = wl.pages_of(b)
        assert (bt[b, :n] >= 0).all() and (bt[b, n:] == -1).all()
        used.extend(bt[b, :n].tolist())
    assert len(set(used)) == len(used) == num_pages - wl.spare_pages
    assert max(used) < num_pages


def test_draws_are_deterministic_and_representable():
    wl = W.WORKLOADS["v2_b32_s4096"]
    a = W.latent_rows(wl, 3, 10)[0]
    b = W.latent_rows(wl, 3, 10)[0]
    assert np.array_equal(a, b)
    assert np.array_equal(W.round_bf16(a), a)
    c = W.latent_rows(wl, 4, 10)[0]
    assert not np.array_equal(a, c)


def test_ragged_lengths():
    wl = W.WORKLOADS["v2_ragged_spec"]
    s = np.array(wl.seq_lens)
    assert wl.batch == 256 and s.min() >= 512 and s.max() <= 8192
    assert 1500 < np.median(s) < 2800


def test_decode_work_counts():
    wl = W.WORKLOADS["v2_b32_s4096"]
    by = W.decode_bytes(wl)
    assert by["cache"] == 32 * 4096 * 576 * 2
    assert by["W_UK_abs"] == 128 * 128 * 512 * 2
    f = W.decode_flops(wl)
    assert f == 32 * (2 * 128 * 4096 * (576 + 512) + 2 * 128 * 128 * 512)
