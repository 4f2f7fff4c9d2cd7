"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print (tests/golden), closed forms, special cases that reduce to a
library routine (scipy, complex arithmetic, torch's fp8 cast), or an
independent route to the same quantity (the decompressed and absorbed forms of
the pages' simulation Cases 3-5 in huny.dev "DeepSeek MLA 해부" §5).
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------- cache sizes

def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


@pytest.mark.parametrize("row", _read_table("cache_sizes.txt"), ids=lambda r: r[0])
def test_cache_sizes_match_pages(row):
    name, kind, layers, seq, bpe, dims, expected, unit, cite = row
    kw = {k: int(v) for k, v in (p.split("=") for p in dims.split(","))}
    got = oracle.cache_bytes(kind, int(layers), int(seq), int(bpe), **kw)
    div = {"B": 1, "KiB": 2 ** 10, "MiB": 2 ** 20, "GiB": 2 ** 30}[unit]
    val = got / div
    if expected.startswith("~"):
        exp = float(expected[1:])
        decimals = len(expected.split(".")[1]) if "." in expected else 0
        # an approximate figure ("about 8.5 GB") is within one unit of its last printed
        # digit of the exact value (8.4375 GiB here)
        assert abs(val - exp) <= 10 ** (-decimals), (name, val, exp, cite)
    else:
        assert val == float(expected), (name, val, expected, cite)


@pytest.mark.parametrize("row", _read_table("ratios.txt"), ids=lambda r: r[0])
def test_ratios_match_pages(row):
    name, num, den, expected, tol, cite = row
    num, den, exp, tol = float(num), float(den), float(expected), float(tol)
    if name.endswith("_pct"):
        val = 100.0 * (1.0 - num / den)
    else:
        val = num / den
    assert abs(val - exp) <= tol, (name, val, exp, cite)


def test_mla_row_is_576_elements():
    # donmain.dev "위치 정보와 압축의 충돌": the cache holds c_t (512) and k_t^R (64), 576 total;
    # the same page calls it GQA-2.25, i.e. 2.25 KV heads of 2*128 elements.
    assert oracle.cache_elems_per_token("mla", d_latent=512, d_rope=64) == 576
    assert oracle.cache_elems_per_token("mla", d_latent=512, d_rope=64) == 2.25 * 2 * 128
    assert oracle.cache_elems_per_token("mha", num_heads=128, head_dim=128) == 32768
    assert W.V2.d_cache == 576


# ----------------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = _rng(0).standard_normal((5, 16))
    assert np.array_equal(oracle.rope(x, np.zeros(5, int)), x)


def test_rope_matches_complex_rotation():
    # pair (x_2k, x_2k+1) as the complex number x_2k + i x_2k+1, multiplied by
    # exp(i * pos * theta^(-2k/d)): an independent formulation of the same rotation.
    rng = _rng(1)
    d = 64
    x = rng.standard_normal((7, d))
    pos = np.array([0, 1, 2, 63, 4095, 65536, 131071])
    z = x[:, 0::2] + 1j * x[:, 1::2]
    k = np.arange(d // 2)
    rot = np.exp(1j * pos[:, None] * np.power(10000.0, -2.0 * k / d))
    zr = z * rot
    y = oracle.rope(x, pos)
    assert np.allclose(y[:, 0::2], zr.real, rtol=0, atol=1e-12)
    assert np.allclose(y[:, 1::2], zr.imag, rtol=0, atol=1e-12)


def test_rope_first_pair_turns_one_radian_per_position():
    x = np.zeros(8)
    x[0] = 1.0
    y = oracle.rope(x, 1)
    assert y[0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[1] == pytest.approx(math.sin(1.0), abs=1e-15)
    # last pair of d=8: frequency 10000^(-6/8)
    x = np.zeros(8)
    x[6] = 1.0
    y = oracle.rope(x, 1000)
    a = 1000 * 10000.0 ** (-0.75)
    assert y[6] == pytest.approx(math.cos(a), abs=1e-14)
    assert y[7] == pytest.approx(math.sin(a), abs=1e-14)


def test_rope_preserves_norm_and_is_relative():
    # donmain.dev "위치 정보와 압축의 충돌": RoPE makes q.k depend on the relative position.
    rng = _rng(2)
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    for m, n in [(5, 3), (1000, 998), (70000, 69998)]:
        assert np.linalg.norm(oracle.rope(q, m)) == pytest.approx(np.linalg.norm(q), rel=1e-13)
        a = oracle.rope(q, m) @ oracle.rope(k, n)
        b = oracle.rope(q, m - n) @ k
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)


# ----------------------------------------------------------------------------- projections

def test_project_latent_splits_columns():
    # W = identity: c_t = h_t W^DKV picks the first d_c features, the rotary key the rest.
    rng = _rng(3)
    h = rng.standard_normal((4, 20))
    c, k = oracle.project_latent(h, np.eye(20), 16)
    assert np.array_equal(c, h[:, :16]) and np.array_equal(k, h[:, 16:])


def test_compress_query_by_brute_force():
    # huny.dev "DeepSeek MLA 해부" §2-2 (c^Q = h W^DQ, q^C_i = c^Q W_i^UQ) and §2-3 (the
    # rotary query h W_i^QR), evaluated with plain Python sums over the definitions.
    rng = _rng(41)
    T, d, d_q, H, d_n, d_r = 3, 7, 5, 3, 4, 2
    h = rng.standard_normal((T, d))
    W_DQ = rng.standard_normal((d, d_q))
    W_UQ = rng.standard_normal((d_q, H * d_n))
    W_QR = rng.standard_normal((d, H * d_r))
    q_nope, q_pe, c_q = oracle.compress_query(h, W_DQ, W_UQ, W_QR, H)
    assert q_nope.shape == (T, H, d_n) and q_pe.shape == (T, H, d_r) and c_q.shape == (T, d_q)
    for t in range(T):
        for i in range(H):
            for n in range(d_n):
                ref = 0.0
                for r in range(d_q):
                    cq = 0.0
                    for k in range(d):
                        cq += h[t, k] * W_DQ[k, r]
                    ref += cq * W_UQ[r, i * d_n + n]
                assert q_nope[t, i, n] == pytest.approx(ref, rel=1e-12, abs=1e-12)
            for r in range(d_r):
                ref = sum(h[t, k] * W_QR[k, i * d_r + r] for k in range(d))
                assert q_pe[t, i, r] == pytest.approx(ref, rel=1e-12, abs=1e-12)


def test_compress_query_identity_weights_pick_head_blocks():
    # W^DQ = I and W^UQ = I: head i's content query is c^Q's i-th block of d_n features;
    # W^QR = I: head i's rotary query is h's i-th block of d_r features.
    rng = _rng(42)
    H, d_n = 3, 4
    h = rng.standard_normal((2, H * d_n))
    q_nope, q_pe, c_q = oracle.compress_query(h, np.eye(H * d_n), np.eye(H * d_n),
                                              np.eye(H * d_n), H)
    assert np.array_equal(c_q, h)
    for i in range(H):
        assert np.array_equal(q_nope[:, i], h[:, i * d_n:(i + 1) * d_n])
        assert np.array_equal(q_pe[:, i], h[:, i * d_n:(i + 1) * d_n])


def test_merged_query_weights_equal_two_steps():
    # thakicloud "어텐션은 무엇을 캐시하는가": the latent-query and latent-key weights multiply
    # into one. (c^Q W_i^UQ) (W_i^UK)^T = c^Q (W_i^UQ (W_i^UK)^T) by associativity.
    rng = _rng(43)
    T, d, d_q, H, d_n, d_r, d_c = 4, 12, 6, 3, 5, 2, 7
    h = rng.standard_normal((T, d))
    W_DQ = rng.standard_normal((d, d_q))
    W_UQ = rng.standard_normal((d_q, H * d_n))
    W_QR = rng.standard_normal((d, H * d_r))
    W_UK = rng.standard_normal((d_c, H * d_n))
    q_nope, _, c_q = oracle.compress_query(h, W_DQ, W_UQ, W_QR, H)
    W_UK_abs, _ = oracle.absorb_weights(W_UK, W_UK, np.zeros((H * d_n, 1)), H)
    two_step = oracle.absorbed_query(q_nope, W_UK_abs)
    W_UQK = oracle.merge_query_weights(W_UQ, W_UK, H)
    assert W_UQK.shape == (H, d_q, d_c)
    one_step = oracle.merged_query(c_q, W_UQK)
    assert np.max(np.abs(one_step - two_step)) <= 1e-12 * np.max(np.abs(two_step))
    # and element by element from the definition q_hat_i = q^C_i . W_i^UK rows
    for t, i, c in ((0, 0, 0), (3, 2, 6), (1, 1, 3)):
        ref = sum(q_nope[t, i, n] * W_UK[c, i * d_n + n] for n in range(d_n))
        assert one_step[t, i, c] == pytest.approx(ref, rel=1e-12)


def test_decompress_uses_head_column_blocks():
    rng = _rng(4)
    d_c, H, d_n = 8, 3, 4
    c = rng.standard_normal((5, d_c))
    W_UK = np.zeros((d_c, H * d_n))
    W_UK[:d_n, 1 * d_n:2 * d_n] = np.eye(d_n)         # only head 1, identity on c[:d_n]
    W_UV = np.zeros((d_c, H * d_n))
    W_UV[d_c - d_n:, 2 * d_n:3 * d_n] = 2 * np.eye(d_n)  # only head 2, 2x on c[-d_n:]
    kC, vC = oracle.decompress(c, W_UK, W_UV, H)
    assert np.array_equal(kC[:, 1], c[:, :d_n])
    assert not kC[:, 0].any() and not kC[:, 2].any()
    assert np.array_equal(vC[:, 2], 2 * c[:, d_c - d_n:])
    assert not vC[:, :2].any()


def _tiny_case(seed=5, S=37, q=1, H=4, d_c=16, d_r=8, d_n=6, d_v=5, d=12):
    rng = _rng(seed)
    c = rng.standard_normal((S, d_c))
    k_rot = oracle.rope(rng.standard_normal((S, d_r)), np.arange(S))
    q_nope = rng.standard_normal((q, H, d_n))
    q_pe = rng.standard_normal((q, H, d_r))
    W_UK = rng.standard_normal((d_c, H * d_n)) / math.sqrt(d_c)
    W_UV = rng.standard_normal((d_c, H * d_v)) / math.sqrt(d_c)
    W_O = rng.standard_normal((H * d_v, d)) / math.sqrt(H * d_v)
    scale = oracle.softmax_scale(d_n, d_r)
    return dict(c=c, k_rot=k_rot, q_nope=q_nope, q_pe=q_pe, W_UK=W_UK, W_UV=W_UV, W_O=W_O,
                scale=scale, H=H)


def test_score_is_content_plus_rotary_by_brute_force():
    # huny.dev §5 Case 3 / §2-3 score split, evaluated with plain Python loops from the
    # definitions: k^C = c W_i^UK, q^R = RoPE(q_pe) at p = S-1.
    T = _tiny_case(seed=6, S=9)
    r = oracle.decode_decompressed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], T["W_UK"],
                                   T["W_UV"], T["scale"])
    S, d_c = T["c"].shape
    d_n = T["q_nope"].shape[2]
    d_r = T["q_pe"].shape[2]
    for i in (0, 3):
        qr = oracle.rope(T["q_pe"][0, i], S - 1)
        for j in (0, 4, 8):
            content = 0.0
            for n in range(d_n):
                kc = sum(T["c"][j, cc] * T["W_UK"][cc, i * d_n + n] for cc in range(d_c))
                content += T["q_nope"][0, i, n] * kc
            rot = sum(qr[m] * T["k_rot"][j, m] for m in range(d_r))
            s = (content + rot) * T["scale"]
            s_oracle = r["lse"][0, i] + math.log(r["A"][0][i][j])
            assert s_oracle == pytest.approx(s, rel=1e-11, abs=1e-12)


def test_softmax_rows_and_lse():
    T = _tiny_case(seed=7, S=50)
    r = oracle.decode_decompressed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], T["W_UK"],
                                   T["W_UV"], T["scale"])
    for i in range(T["H"]):
        A = r["A"][0][i]
        assert A.min() >= 0.0
        assert A.sum() == pytest.approx(1.0, abs=1e-14)
        s = r["lse"][0, i] + np.log(A)
        assert scipy.special.logsumexp(s) == pytest.approx(r["lse"][0, i], abs=1e-12)
        assert np.allclose(scipy.special.softmax(s), A, atol=1e-15)


@pytest.mark.parametrize("q", [1, 2])
def test_absorbed_equals_decompressed(q):
    # huny.dev §3-1 (W^UK absorbed into the query) and §5 Case 4.
    T = _tiny_case(seed=8, S=41, q=q)
    r = oracle.decode_decompressed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], T["W_UK"],
                                   T["W_UV"], T["scale"])
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    o, lse = oracle.decode_absorbed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], W_UK_abs,
                                    T["scale"])
    assert np.max(np.abs(o - r["o_lat"])) <= 1e-12 * np.max(np.abs(o))
    assert np.max(np.abs(lse - r["lse"])) <= 1e-12 * np.max(np.abs(lse))


def test_latent_output_lifts_to_value_output():
    # huny.dev §3-2, first equation: sum_j A_j (c_j W_i^UV) = (sum_j A_j c_j) W_i^UV.
    T = _tiny_case(seed=9, S=30, q=2)
    r = oracle.decode_decompressed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], T["W_UK"],
                                   T["W_UV"], T["scale"])
    d_v = T["W_UV"].shape[1] // T["H"]
    for i in range(T["H"]):
        lifted = r["o_lat"][:, i] @ T["W_UV"][:, i * d_v:(i + 1) * d_v]
        assert np.allclose(lifted, r["u"][:, i], rtol=0, atol=1e-13)


def test_folded_output_projection_is_lossless():
    # huny.dev §3-2 second equation and §5 Case 5: sum_i u_i W_i^O == o_lat . W_comb.
    T = _tiny_case(seed=10, S=25, q=2)
    r = oracle.decode_decompressed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], T["W_UK"],
                                   T["W_UV"], T["scale"])
    _, W_comb = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    a = oracle.mha_output(r["u"], T["W_O"])
    b = oracle.output_projection(r["o_lat"].reshape(r["o_lat"].shape[0], -1), W_comb)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


def test_lift_latent_equals_decompressed_value_output():
    # huny.dev §3-2, first equation: the decompressed route's value output u (values
    # c_j W_i^UV averaged by the attention weights) is the latent output lifted by W_i^UV.
    T = _tiny_case(seed=13, S=27, q=2)
    r = oracle.decode_decompressed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], T["W_UK"],
                                   T["W_UV"], T["scale"])
    u = oracle.lift_latent(r["o_lat"], T["W_UV"], T["H"])
    assert u.shape == r["u"].shape
    assert np.max(np.abs(u - r["u"])) <= 1e-13 * max(1.0, np.max(np.abs(r["u"])))
    # a head-block weight that is the identity on head 1 only copies that head's first dims
    d_c, H = T["c"].shape[1], T["H"]
    d_v = T["W_UV"].shape[1] // H
    W = np.zeros((d_c, H * d_v))
    W[:d_v, d_v:2 * d_v] = np.eye(d_v)
    u1 = oracle.lift_latent(r["o_lat"], W, H)
    assert np.array_equal(u1[:, 1], r["o_lat"][:, 1, :d_v])
    assert not u1[:, 0].any() and not u1[:, 2:].any()


def test_unfolded_output_path_equals_folded():
    # huny.dev §3-2 second equation, both sides: sum_i (o_i W_i^UV) W_i^O == o . W_comb.
    T = _tiny_case(seed=14, S=19, q=2)
    rng = np.random.default_rng(14)
    H, d_c = T["H"], T["c"].shape[1]
    o = rng.standard_normal((3, H * d_c))
    _, W_comb = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], H)
    a = oracle.mha_output(oracle.lift_latent(o, T["W_UV"], H), T["W_O"])
    b = oracle.output_projection(o, W_comb)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


def test_seq_len_one_returns_the_only_latent():
    T = _tiny_case(seed=11, S=1)
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    o, lse = oracle.decode_absorbed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], W_UK_abs,
                                    T["scale"])
    assert np.array_equal(o[0], np.broadcast_to(T["c"][0], o[0].shape))
    # the LSE of a single key is its score; rotation at position 0 is the identity
    d_n = T["q_nope"].shape[2]
    for i in range(T["H"]):
        kc = T["c"][0] @ T["W_UK"][:, i * d_n:(i + 1) * d_n]
        s = (T["q_nope"][0, i] @ kc + T["q_pe"][0, i] @ T["k_rot"][0]) * T["scale"]
        assert lse[0, i] == pytest.approx(s, abs=1e-13)


def test_zero_query_gives_uniform_average():
    T = _tiny_case(seed=12, S=33, q=2)
    zq = np.zeros_like(T["q_nope"])
    zp = np.zeros_like(T["q_pe"])
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    o, lse = oracle.decode_absorbed(T["c"], T["k_rot"], zq, zp, W_UK_abs, T["scale"])
    S = T["c"].shape[0]
    for t in range(2):
        n = S - 2 + t + 1
        assert np.allclose(o[t], T["c"][:n].mean(axis=0), atol=1e-14)
        assert np.allclose(lse[t], math.log(n), atol=1e-14)


def test_identical_keys():
    T = _tiny_case(seed=13, S=20)
    c = np.broadcast_to(T["c"][3], T["c"].shape).copy()
    kr = np.broadcast_to(T["k_rot"][3], T["k_rot"].shape).copy()
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    o, lse = oracle.decode_absorbed(c, kr, T["q_nope"], T["q_pe"], W_UK_abs, T["scale"])
    one, lse1 = oracle.decode_absorbed(c[:1], kr[:1], T["q_nope"], np.zeros_like(T["q_pe"]),
                                       W_UK_abs, T["scale"])
    assert np.allclose(o[0], c[0], atol=1e-14)
    # S equal keys: LSE = score + ln S (the rotary part differs only through q's position)
    qr = oracle.rope(T["q_pe"][0], 19)
    d_n = T["q_nope"].shape[2]
    for i in range(T["H"]):
        s = (T["q_nope"][0, i] @ (c[0] @ T["W_UK"][:, i * d_n:(i + 1) * d_n]) + qr[i] @ kr[0]) \
            * T["scale"]
        assert lse[0, i] == pytest.approx(s + math.log(20), abs=1e-12)


def test_dominant_key_wins():
    # a huge rotary score on key 5 makes the softmax one-hot there: o_lat -> c_5
    T = _tiny_case(seed=14, S=16)
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    qr = oracle.rope(T["q_pe"][0], 15)                     # [H][d_r], query at p = 15
    kr = T["k_rot"].copy()
    kr[5] = 1e3 * qr.sum(axis=0) / np.linalg.norm(qr.sum(axis=0))
    o, lse = oracle.decode_absorbed(T["c"], kr, T["q_nope"], T["q_pe"], W_UK_abs, T["scale"])
    hit = 0
    for i in range(T["H"]):
        if (qr[i] @ kr[5]) * T["scale"] > 200:
            hit += 1
            assert np.allclose(o[0, i], T["c"][5], atol=1e-12)
    assert hit >= 1


@pytest.mark.parametrize("S,q", [(29, 2), (29, 5), (40, 8), (8, 8)])
def test_causal_token_equals_shorter_request(S, q):
    # Speculative decoding (secrett2633.cloud "[vLLM] Multi-head Latent Attention", the
    # reshape_query_for_spec_decode step) with the causal reading: query token t of a q-token
    # step sees exactly the keys a 1-token step of length S - q + t + 1 sees. (8, 8) is a step
    # whose every token is new: its first token sees only key 0.
    T = _tiny_case(seed=15, S=S, q=q)
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    oq, lq = oracle.decode_absorbed(T["c"], T["k_rot"], T["q_nope"], T["q_pe"], W_UK_abs,
                                    T["scale"])
    for t in range(q):
        n = S - q + t + 1
        o1, l1 = oracle.decode_absorbed(T["c"][:n], T["k_rot"][:n], T["q_nope"][t:t + 1],
                                        T["q_pe"][t:t + 1], W_UK_abs, T["scale"])
        assert np.array_equal(oq[t], o1[0]) and np.array_equal(lq[t], l1[0])
    if S == q:
        assert np.array_equal(oq[0], np.broadcast_to(T["c"][0], oq[0].shape))


def test_empty_request():
    T = _tiny_case(seed=16, S=5)
    W_UK_abs, _ = oracle.absorb_weights(T["W_UK"], T["W_UV"], T["W_O"], T["H"])
    o, lse = oracle.decode_absorbed(T["c"][:0], T["k_rot"][:0], T["q_nope"], T["q_pe"],
                                    W_UK_abs, T["scale"])
    assert not o.any() and np.all(np.isneginf(lse))


def test_combine_partials_matches_full_softmax():
    rng = _rng(17)
    s = rng.standard_normal(300) * 3
    V = rng.standard_normal((300, 7))
    cuts = [0, 64, 65, 200, 300]
    o_parts, l_parts = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o_parts.append(scipy.special.softmax(s[a:b]) @ V[a:b])
        l_parts.append(scipy.special.logsumexp(s[a:b]))
    o, L = oracle.combine_partials(np.array(o_parts), np.array(l_parts))
    assert np.allclose(o, scipy.special.softmax(s) @ V, atol=1e-13)
    assert L == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


def test_absorb_weights_layout():
    rng = _rng(18)
    H, d_c, d_n, d_v, d = 3, 5, 4, 2, 6
    W_UK = rng.standard_normal((d_c, H * d_n))
    W_UV = rng.standard_normal((d_c, H * d_v))
    W_O = rng.standard_normal((H * d_v, d))
    A, C = oracle.absorb_weights(W_UK, W_UV, W_O, H)
    assert A.shape == (H, d_n, d_c) and C.shape == (H * d_c, d)
    for i in range(H):
        for n in range(d_n):
            for cc in range(d_c):
                assert A[i, n, cc] == W_UK[cc, i * d_n + n]
        for cc in range(d_c):
            for x in range(d):
                ref = sum(W_UV[cc, i * d_v + v] * W_O[i * d_v + v, x] for v in range(d_v))
                assert C[i * d_c + cc, x] == pytest.approx(ref, abs=1e-13)


# ----------------------------------------------------------------------------- fp8 e4m3

def test_e4m3_known_codes():
    # OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits, max finite 448, no inf.
    dec = oracle.e4m3_decode
    assert dec(0x38) == 1.0 and dec(0xB8) == -1.0 and dec(0x30) == 0.5
    assert dec(0x7E) == 448.0 and dec(0x08) == 2.0 ** -6 and dec(0x01) == 2.0 ** -9
    assert dec(0x07) == 7 * 2.0 ** -9 and dec(0x3F) == 1.875
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    enc = oracle.e4m3_encode
    assert enc(1.0) == 0x38 and enc(-448.0) == 0xFE and enc(1e6) == 0x7E and enc(-1e6) == 0xFE
    assert enc(1.0 + 1 / 16) == 0x38          # tie between 1.0 and 1.125 -> even mantissa
    assert enc(1.0 + 3 / 16) == 0x3A          # tie between 1.125 and 1.25 -> even mantissa
    assert enc(1.0 + 1 / 16 + 1e-9) == 0x39
    assert enc(2.0 ** -10) == 0x00            # half the smallest subnormal -> even (zero)
    assert enc(3 * 2.0 ** -10) == 0x02        # tie between 1 and 2 subnormal steps -> even
    assert enc(464.0) == 0x7E                 # beyond 448 saturates
    assert enc(-1e-9) == 0x80 and enc(-0.0) == 0x80   # sign kept when rounding to zero


def test_e4m3_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = _rng(19)
    x = np.concatenate([rng.standard_normal(200000) * 40, rng.standard_normal(20000) * 1e-2,
                        np.linspace(-448, 448, 30001)]).astype(np.float32)
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_round_trip_is_exact_on_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(vals)
    assert np.array_equal(back, codes)


# ----------------------------------------------------------------------------- paged cache

def test_block_quantize_round_trips_codes_times_a_power_of_two():
    # huny.dev §6 (fp8 latent with per-block dynamic scales): rows built as e4m3 code values
    # times a power-of-two scale, each block holding a +-448 code, come back bit for bit.
    rng = _rng(51)
    n, d, block = 6, 512, 128
    codes = rng.integers(0, 0x7F, size=(n, d), dtype=np.uint8) | (rng.integers(0, 2, (n, d)) << 7).astype(np.uint8)
    codes[:, ::block] = 0x7E                           # 448 in every block
    s = 2.0 ** rng.integers(-12, 4, size=(n, d // block))
    x = oracle.e4m3_decode(codes).reshape(n, d // block, block) * s[..., None]
    got_c, got_s = oracle.e4m3_block_quantize(x.reshape(n, d), block)
    assert np.array_equal(got_s, s.astype(np.float32))
    # -0 and +0 both decode to 0: compare values
    assert np.array_equal(oracle.e4m3_decode(got_c), oracle.e4m3_decode(codes))


def test_block_quantize_error_bound_and_amax():
    rng = _rng(52)
    x = rng.standard_normal((40, 512)) * np.exp(rng.standard_normal((40, 1)) * 3)
    codes, scales = oracle.e4m3_block_quantize(x, 128)
    deq = oracle.e4m3_block_dequantize(codes, scales, 128)
    xb = np.abs(x.astype(np.float32)).reshape(40, 4, 128)
    # the largest magnitude of every block lands on the largest code
    big = np.argmax(xb, axis=2)
    cb = codes.reshape(40, 4, 128)
    assert ((np.take_along_axis(cb, big[..., None], 2)[..., 0] & 0x7F) == 0x7E).all()
    # half a unit in the last place of e4m3 (3 mantissa bits), relative to the element's
    # binade, or half the subnormal step 2^-9, in units of the block's scale
    q = np.abs(x.astype(np.float32)).reshape(40, 4, 128) / scales[..., None].astype(np.float64)
    e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    half_ulp = 0.5 * 2.0 ** (e - 3)
    err = np.abs(deq - x.astype(np.float32)).reshape(40, 4, 128) / scales[..., None]
    assert (err <= half_ulp * (1 + 1e-6) + 1e-12).all()


def test_block_quantize_blocks_are_independent_and_zero_blocks_stay_zero():
    rng = _rng(53)
    x = rng.standard_normal((3, 256))
    x[1, 128:] = 0.0
    c0, s0 = oracle.e4m3_block_quantize(x, 128)
    assert s0[1, 1] == 0 and not c0[1, 128:].any()
    assert not oracle.e4m3_block_dequantize(c0, s0, 128)[1, 128:].any()
    y = x.copy()
    y[0, :128] *= 2.0 ** 5                              # only block (0, 0) changes
    c1, s1 = oracle.e4m3_block_quantize(y, 128)
    assert s1[0, 0] == s0[0, 0] * 2.0 ** 5
    assert np.array_equal(c1, c0)
    assert np.array_equal(np.delete(s1.ravel(), 0), np.delete(s0.ravel(), 0))


def test_cache_image_hand_example():
    # page size 4 for a hand-checkable case: request 0 owns pages [2, 0], request 1 owns [1].
    bt = np.array([[2, 0], [1, -1]], dtype=np.int32)
    rows = np.arange(4 * 3, dtype=np.int16).reshape(4, 3) + 1
    req = np.array([0, 0, 1, 0])
    pos = np.array([0, 5, 3, 4])
    img = oracle.cache_image(4, 4, rows, req, pos, bt, fill=-7)
    assert (img[2, 0] == rows[0]).all()      # (0, 0): page bt[0][0] = 2, slot 0
    assert (img[0, 1] == rows[1]).all()      # (0, 5): page bt[0][1] = 0, slot 1
    assert (img[1, 3] == rows[2]).all()      # (1, 3): page bt[1][0] = 1, slot 3
    assert (img[0, 0] == rows[3]).all()      # (0, 4): page 0, slot 0
    written = {(2, 0), (0, 1), (1, 3), (0, 0)}
    for p in range(4):
        for s in range(4):
            if (p, s) not in written:
                assert (img[p, s] == -7).all()
