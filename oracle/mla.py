"""Plain float64 CPU oracle of weight-absorbed MLA decode. TEST INFRASTRUCTURE ONLY.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py``; it never imports the CUDA path, and the CUDA path never imports
it. Inputs are the values the GPU consumes, promoted to float64.

Pages cited (title, site):
  [P1] "DeepSeek Multi-Head Latent Attention(MLA) 해부: 저차원 KV 압축과 Decoupled RoPE를
       통한 VRAM 98% 절감 및 행렬 흡수(Matrix Absorption) 추론 가속 원리" (blog.huny.dev)
  [P2] "KV Cache를 10분의 1로 줄인 MLA의 트릭" (donmain.dev)
  [P3] "[vLLM] Multi-head Latent Attention: KV 캐시를 압축하는 DeepSeek의 어텐션"
       (blog.secrett2633.cloud)
  [P4] thakicloud.com tech blog, "transformer-attention-kv-cache-math"

Readings taken where the pages are silent (each also listed in the design notes):
  * softmax scale = 1/sqrt(d_nope + d_rope), the width of the un-absorbed q.k of
    [P1] §2-3 (concatenated query/key equation);
  * RoPE rotates interleaved pairs (2k, 2k+1) by pos * theta^(-2k/d_r), theta =
    10000, positions 0-based; [P1] §2-3 only says "orthogonal rotation";
  * k_pe is rotated once, when appended; q_pe is rotated at the query position
    p_t = seq_len - q_len + t;
  * query token t of a request attends to key positions 0..p_t (causal);
  * fp8 cache: e4m3, one per-tensor scale, round-to-nearest-even, saturating to
    +-448; the dequantised value is code * scale;
  * an empty request (seq_len 0) has latent output 0 and LSE -inf.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, the pages' printed numbers, library routines or an
independent route to the same quantity.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "softmax_scale", "rope", "project_latent", "decompress", "decode_decompressed",
    "absorb_weights", "absorbed_query", "decode_absorbed", "output_projection",
    "lift_latent", "mha_output", "compress_query", "merge_query_weights", "merged_query",
    "e4m3_encode", "e4m3_decode", "e4m3_block_quantize", "e4m3_block_dequantize",
    "cache_image", "cache_elems_per_token", "cache_bytes", "combine_partials",
]


def softmax_scale(d_nope: int, d_rope: int) -> float:
    """1/sqrt(d_n + d_r): the score of [P1] §2-3 is a dot product of the concatenated
    [q^C ; q^R] and [k^C ; k^R], whose width is d_n + d_r."""
    return 1.0 / math.sqrt(d_nope + d_rope)


def rope(x, pos, theta: float = 10000.0):
    """Rotary position embedding of the decoupled key/query ([P1] §2-3, k^R = RoPE(h W^KR)
    and q^R = RoPE(h W^QR); [P2] "위치 정보와 압축의 충돌").

    x: [..., d_r]; pos: integer array broadcastable to x.shape[:-1].
    Pair k = (x[2k], x[2k+1]) is rotated counter-clockwise by angle pos * theta^(-2k/d_r).
    """
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    k = np.arange(d_r // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * k / d_r)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


def project_latent(h, W_DKV_KR, d_latent: int):
    """c_t = h_t W^DKV ([P1] §2-1 eq.) and the raw decoupled key h_t W^KR ([P1] §2-3).

    W_DKV_KR is [d_model][d_c + d_r] = [W^DKV | W^KR]. Returns (c [n][d_c], k_raw [n][d_r]).
    """
    P = np.asarray(h, np.float64) @ np.asarray(W_DKV_KR, np.float64)
    return P[:, :d_latent], P[:, d_latent:]


def compress_query(h, W_DQ, W_UQ, W_QR, num_heads: int):
    """The query side: c^Q_t = h_t W^DQ and q^C_{t,i} = c^Q_t W_i^UQ ([P1] §2-2, low-rank
    query compression), and head i's rotary query before its rotation, h_t W_i^QR ([P1] §2-3;
    the decode rotates it at the query position).

    W_DQ [d_model][d_q]; W_UQ [d_q][H*d_n], head i owning columns i*d_n..(i+1)*d_n-1; W_QR
    [d_model][H*d_r] likewise. Returns q_nope [T][H][d_n], q_pe [T][H][d_r] (not rotated) and
    c_q [T][d_q].
    """
    h = np.asarray(h, np.float64)
    c_q = h @ np.asarray(W_DQ, np.float64)
    q_nope = (c_q @ np.asarray(W_UQ, np.float64)).reshape(h.shape[0], num_heads, -1)
    q_pe = (h @ np.asarray(W_QR, np.float64)).reshape(h.shape[0], num_heads, -1)
    return q_nope, q_pe, c_q


def merge_query_weights(W_UQ, W_UK, num_heads: int):
    """The latent-query weight multiplied into the latent-key weight ([P4] "어텐션은 무엇을
    캐시하는가": the two merge into one): W^UQK_i = W_i^UQ (W_i^UK)^T, so that head i's
    absorbed query is c^Q W^UQK_i without forming q^C.

    W_UQ [d_q][H*d_n], W_UK [d_c][H*d_n] -> [H][d_q][d_c].
    """
    W_UQ = np.asarray(W_UQ, np.float64)
    W_UK = np.asarray(W_UK, np.float64)
    d_n = W_UQ.shape[1] // num_heads
    return np.stack([W_UQ[:, i * d_n:(i + 1) * d_n] @ W_UK[:, i * d_n:(i + 1) * d_n].T
                     for i in range(num_heads)])


def merged_query(c_q, W_UQK):
    """q_hat_i = c^Q W^UQK_i. c_q [T][d_q], W_UQK [H][d_q][d_c] -> [T][H][d_c]."""
    return np.einsum("tq,hqc->thc", np.asarray(c_q, np.float64), np.asarray(W_UQK, np.float64))


def decompress(c, W_UK, W_UV, num_heads: int):
    """Explicit up-projection k^C_{j,i} = c_j W_i^UK, v^C_{j,i} = c_j W_i^UV ([P1] §2-1,
    second equation). W_UK is [d_c][H*d_n] with head i in columns i*d_n..(i+1)*d_n-1;
    W_UV likewise. Returns k_C [S][H][d_n], v_C [S][H][d_v]."""
    c = np.asarray(c, np.float64)
    S = c.shape[0]
    kC = (c @ np.asarray(W_UK, np.float64)).reshape(S, num_heads, -1)
    vC = (c @ np.asarray(W_UV, np.float64)).reshape(S, num_heads, -1)
    return kC, vC


def decode_decompressed(c, k_rot, q_nope, q_pe, W_UK, W_UV, scale: float, theta: float = 10000.0,
                        heads=None):
    """Textbook multi-head attention over explicitly decompressed keys and values.

    One request. c [S][d_c] and k_rot [S][d_r] are the cached latent and the already
    rotated decoupled key of positions 0..S-1. q_nope [q][H][d_n], q_pe [q][H][d_r] are
    the step's queries (q_pe not yet rotated). Query token t sits at p_t = S - q + t and
    sees keys 0..p_t.

    Per head i ([P1] §2-3 concatenation and score split; [P1] §3-2 first equation):
      q = [q^C ; RoPE(q_pe, p_t)],  k_j = [c_j W_i^UK ; k^R_j],
      s_j = (q . k_j) * scale,  A = softmax(s),  LSE = log sum_j exp(s_j),
      u = sum_j A_j v^C_j  (v^C_j = c_j W_i^UV),  o_lat = sum_j A_j c_j.
    Returns dict of u [q][h][d_v], o_lat [q][h][d_c], lse [q][h], A (list per t of [h][p_t+1]).
    """
    c = np.asarray(c, np.float64)
    k_rot = np.asarray(k_rot, np.float64)
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    S = c.shape[0]
    q, H = q_nope.shape[0], q_nope.shape[1]
    heads = list(range(H)) if heads is None else list(heads)
    kC, vC = decompress(c, W_UK, W_UV, H)
    d_c = c.shape[1]
    u = np.zeros((q, len(heads), vC.shape[2]))
    o = np.zeros((q, len(heads), d_c))
    lse = np.full((q, len(heads)), -np.inf)
    probs = []
    for t in range(q):
        p_t = S - q + t
        At = []
        for hi, i in enumerate(heads):
            if S == 0 or p_t < 0:
                At.append(np.zeros(0))
                continue
            qr = rope(q_pe[t, i], p_t, theta)
            qv = np.concatenate([q_nope[t, i], qr])
            K = np.concatenate([kC[:p_t + 1, i, :], k_rot[:p_t + 1]], axis=1)
            s = (K @ qv) * scale
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            A = e / l
            lse[t, hi] = m + math.log(l)
            u[t, hi] = A @ vC[:p_t + 1, i, :]
            o[t, hi] = A @ c[:p_t + 1]
            At.append(A)
        probs.append(At)
    return {"u": u, "o_lat": o, "lse": lse, "A": probs}


def absorb_weights(W_UK, W_UV, W_O, num_heads: int):
    """Weight absorption done once at model load ([P2] "위치 정보와 압축의 충돌": absorb
    W^UK into the query side and W^UV into W^O; [P1] §3-1 and §3-2).

    Returns W_UK_abs [H][d_n][d_c] with W_UK_abs[i] = (W_i^UK)^T, and
    W_comb [H*d_c][d_model] whose block i is W_i^UV W_i^O ([P1] §3-2, W_i^combined).
    """
    W_UK = np.asarray(W_UK, np.float64)
    W_UV = np.asarray(W_UV, np.float64)
    W_O = np.asarray(W_O, np.float64)
    d_c = W_UK.shape[0]
    d_n = W_UK.shape[1] // num_heads
    d_v = W_UV.shape[1] // num_heads
    W_UK_abs = np.stack([W_UK[:, i * d_n:(i + 1) * d_n].T for i in range(num_heads)])
    W_comb = np.concatenate(
        [W_UV[:, i * d_v:(i + 1) * d_v] @ W_O[i * d_v:(i + 1) * d_v, :] for i in range(num_heads)],
        axis=0)
    assert W_comb.shape[0] == num_heads * d_c
    return W_UK_abs, W_comb


def absorbed_query(q_nope, W_UK_abs):
    """q_hat_i = q^C_i (W_i^UK)^T ([P1] §3-1 equation, the under-braced term).
    q_nope [..., H, d_n], W_UK_abs [H][d_n][d_c] -> [..., H, d_c]."""
    return np.einsum("...hn,hnc->...hc", np.asarray(q_nope, np.float64),
                     np.asarray(W_UK_abs, np.float64))


def decode_absorbed(c, k_rot, q_nope, q_pe, W_UK_abs, scale: float, theta: float = 10000.0,
                    heads=None):
    """Weight-absorbed decode of one request, all heads ([P1] §3-1 and §3-2; [P2]
    "위치 정보와 압축의 충돌": score = q_hat . c_s + q^R . k^R_s).

    The MQA form of [P3] "MLA의 MQA 디코딩 경로": every head attends over the one
    shared latent row [c_j ; k^R_j]. Same positions and causal rule as
    decode_decompressed. ``heads`` optionally restricts the computation to a list of
    head indices (the outputs then follow that order). Returns o_lat [q][h][d_c]
    (= sum_j A_j c_j) and lse [q][h].
    """
    c = np.asarray(c, np.float64)
    k_rot = np.asarray(k_rot, np.float64)
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    if heads is not None:
        heads = list(heads)
        q_nope, q_pe = q_nope[:, heads], q_pe[:, heads]
        W_UK_abs = np.asarray(W_UK_abs)[heads]
    S, d_c = c.shape
    q, H = q_nope.shape[0], q_nope.shape[1]
    o = np.zeros((q, H, d_c))
    lse = np.full((q, H), -np.inf)
    if S == 0:
        return o, lse
    q_hat = absorbed_query(q_nope, W_UK_abs)                      # [q][H][d_c]
    for t in range(q):
        p_t = S - q + t
        if p_t < 0:
            continue
        qr = rope(q_pe[t], p_t, theta)                            # [H][d_r]
        s = (q_hat[t] @ c[:p_t + 1].T + qr @ k_rot[:p_t + 1].T) * scale   # [H][p_t+1]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        o[t] = (e / l) @ c[:p_t + 1]
        lse[t] = (m + np.log(l))[:, 0]
    return o, lse


def output_projection(o_lat, W_comb):
    """Output_t = sum_i o_lat_i W_i^combined ([P1] §3-2, second equation).
    o_lat [rows][H*d_c] (head-major), W_comb [H*d_c][d_model]."""
    return np.asarray(o_lat, np.float64) @ np.asarray(W_comb, np.float64)


def lift_latent(o_lat, W_UV, num_heads: int):
    """u_i = o_lat_i W_i^UV, each head's latent output lifted to its value width ([P1] §3-2,
    first equation: sum_j A_j (c_j W_i^UV) = (sum_j A_j c_j) W_i^UV).
    o_lat [rows][H][d_c] (or [rows][H*d_c]), W_UV [d_c][H*d_v] (head i owns columns
    i*d_v..) -> u [rows][H][d_v]."""
    o = np.asarray(o_lat, np.float64)
    o = o.reshape(o.shape[0], num_heads, -1)
    W = np.asarray(W_UV, np.float64)
    d_v = W.shape[1] // num_heads
    return np.einsum("rhc,chv->rhv", o, W.reshape(W.shape[0], num_heads, d_v))


def mha_output(u, W_O):
    """Output_t = sum_i u_i W_i^O, the un-folded form ([P1] §3-2, left side).
    u [rows][H][d_v], W_O [H*d_v][d_model]."""
    u = np.asarray(u, np.float64)
    return u.reshape(u.shape[0], -1) @ np.asarray(W_O, np.float64)


def combine_partials(o_parts, lse_parts):
    """Merge attention results computed over disjoint key ranges of the same query:
    L = log sum_s exp(lse_s), o = sum_s exp(lse_s - L) o_s. Exact for softmax, since
    each o_s is normalised by its own sum exp(lse_s) ([P3] "FP8 MLA 지원": num_splits
    and the decode LSE return of "FlashMLAImpl")."""
    lse_parts = np.asarray(lse_parts, np.float64)
    o_parts = np.asarray(o_parts, np.float64)
    m = lse_parts.max(axis=0)
    w = np.exp(lse_parts - m)
    L = m + np.log(w.sum(axis=0))
    o = (np.exp(lse_parts - L)[..., None] * o_parts).sum(axis=0)
    return o, L


# ----------------------------------------------------------------------------- fp8 e4m3
# The fp8 KV-cache of [P1] §6 (FP8 E4M3) and [P3] "FP8 MLA 지원" (cache dtype
# "fp8_e4m3"). E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
# bits, no infinities, largest finite 448, smallest subnormal 2^-9.

def e4m3_decode(codes):
    """Value of each e4m3 byte (NaN codes 0x7F/0xFF map to NaN)."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return sign * val


_E4M3_POS = None


def _e4m3_table():
    global _E4M3_POS
    if _E4M3_POS is None:
        codes = np.arange(0x7F, dtype=np.uint8)          # 0x00..0x7E: all non-negative finite
        _E4M3_POS = e4m3_decode(codes)                   # increasing
    return _E4M3_POS


def e4m3_encode(x):
    """Encode float values to e4m3 bytes: round to the nearest representable value,
    ties to the code with an even mantissa, magnitudes beyond 448 saturate to 448, the
    sign is kept (so a negative value that rounds to zero gives -0). Exact on the given
    values (no intermediate rounding)."""
    x = np.asarray(x, dtype=np.float64)
    vals = _e4m3_table()
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == vals[hi], hi, code)
    out = code.astype(np.uint8)
    # the sign bit is kept even when the magnitude rounds to zero (-0 is 0x80)
    return np.where(np.signbit(x), out | 0x80, out).astype(np.uint8)


def e4m3_block_quantize(x, block: int = 128):
    """Block-wise dynamic e4m3 quantisation of latent rows, the fp8 cache [P1] §6 describes
    for DeepSeek-V3: the latent vector in fp8 with a scale per block, computed from the
    values when they are written (the decoupled rotary key stays in bf16 and is not passed
    here). The pages give no block size; a block is `block` consecutive elements of one
    token's row.

    Per block: scale = fp32(amax |x|) / 448 rounded once to fp32; codes = e4m3_encode of the
    fp32 quotient fp32(x) / scale (each quotient rounded once to fp32, then encoded exactly).
    A block of zeros has scale 0 and codes 0. x [n][d], d a multiple of block -> (codes uint8
    [n][d], scales float32 [n][d / block]).
    """
    x32 = np.asarray(x, dtype=np.float32)
    n, d = x32.shape
    assert d % block == 0
    xb = x32.reshape(n, d // block, block)
    amax = np.max(np.abs(xb), axis=2).astype(np.float32)
    scales = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(scales > 0, scales, np.float32(1.0)).astype(np.float32)
    quot = (xb / safe[..., None]).astype(np.float32)
    codes = e4m3_encode(quot)
    codes = np.where((scales > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(n, d), scales


def e4m3_block_dequantize(codes, scales, block: int = 128):
    """Value of block-quantised rows: code value times its block's scale (float64)."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, d = codes.shape
    v = e4m3_decode(codes).reshape(n, d // block, block)
    return (v * np.asarray(scales, np.float64)[..., None]).reshape(n, d)


# ----------------------------------------------------------------------------- paged cache

def cache_image(num_pages: int, page_size: int, rows, req_ids, positions, block_table, fill):
    """Expected paged cache after appends: the combined latent row of token (b, pos) sits at
    cache[block_table[b][pos // page_size]][pos % page_size][:] ([P3] "FlashMLABackend":
    block size 64; "FlashMLAImpl": one combined kv_c_and_k_pe_cache). ``rows`` [T][D] are
    the encoded rows (any dtype); every slot not written keeps ``fill``."""
    rows = np.asarray(rows)
    D = rows.shape[1]
    img = np.empty((num_pages, page_size, D), dtype=rows.dtype)
    img[...] = fill
    bt = np.asarray(block_table)
    for r in range(rows.shape[0]):
        b, p = int(req_ids[r]), int(positions[r])
        img[bt[b, p // page_size], p % page_size] = rows[r]
    return img


def cache_elems_per_token(kind: str, *, num_heads=0, head_dim=0, kv_heads=0, d_latent=0,
                          d_rope=0) -> int:
    """Cached elements per token per layer ([P1] §1 memory equation and §4 table; [P2]
    "MLA, 압축이라는 다른 길" and "위치 정보와 압축의 충돌"):
      MHA: 2 * n_h * d_h;  GQA: 2 * n_kv * d_h;  MLA: d_c + d_h^R."""
    if kind == "mha":
        return 2 * num_heads * head_dim
    if kind == "gqa":
        return 2 * kv_heads * head_dim
    if kind == "mla":
        return d_latent + d_rope
    raise ValueError(kind)


def cache_bytes(kind: str, layers: int, seq: int, bytes_per_elem: int, **dims) -> int:
    """Per-request cache bytes = elements/token/layer * layers * seq * bytes ([P1] §1)."""
    return cache_elems_per_token(kind, **dims) * layers * seq * bytes_per_elem
