"""Seeded synthetic inputs for weight-absorbed MLA decode.

This module holds shapes, seeds and random draws only. It contains none of the
attention arithmetic, so both sides of every parity check (the CUDA library and
the CPU oracle) can consume bit-identical inputs without sharing any code of
the method itself.

Workload shapes follow the DeepSeek-V2 dimensions the pages give
(huny.dev "DeepSeek MLA 해부" §2-1: d_c = 512, 128 heads x 128; donmain.dev
"KV Cache를 10분의 1로 줄인 MLA의 트릭", section "MLA, 압축이라는 다른 길":
d_model = 5120, d_c = 512, and section "위치 정보와 압축의 충돌": d_h^R = 64),
and the 64-token page of the vLLM FlashMLA backend (secrett2633.cloud
"[vLLM] Multi-head Latent Attention", section "FlashMLABackend").

Floating-point draws are returned as float32 arrays whose values are exactly
representable in the workload's activation dtype (bf16 values are rounded to
nearest-even here, once), so converting them to a device bf16 tensor and
promoting them to fp64 are both exact.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import numpy as np

PAGE = 64


@dataclass(frozen=True)
class Dims:
    num_heads: int
    d_model: int
    d_latent: int
    d_rope: int
    d_nope: int
    d_v: int
    page_size: int = PAGE
    d_q: int = 0            # query compression rank (c^Q width)

    @property
    def d_cache(self) -> int:
        return self.d_latent + self.d_rope


# d_q: the pages write c^Q = h W^DQ without its width; 1536 is DeepSeek-V2's, 48 = 3 d_c / 4
# keeps the tiny shape's proportion between the query and latent ranks.
V2 = Dims(num_heads=128, d_model=5120, d_latent=512, d_rope=64, d_nope=128, d_v=128, d_q=1536)
TINY = Dims(num_heads=16, d_model=256, d_latent=64, d_rope=16, d_nope=32, d_v=32, d_q=48)


@dataclass(frozen=True)
class Workload:
    """One decode workload: shapes, lengths, dtypes and the seed of every draw.

    seq_lens count cached tokens *including* the q_len tokens of this step.
    ``fill`` says how the cache is produced: 'h' = every cached token comes from
    a hidden state through the append projection; 'latent' = c_kv and the raw
    (un-rotated) k_pe are drawn directly, and the last ``new_from_h`` tokens of
    each request come from hidden states.
    """

    name: str
    dims: Dims
    act: str            # 'f32' | 'bf16'
    cache: str          # 'f32' | 'bf16' | 'fp8_e4m3'
    seq_lens: tuple
    q_len: int
    seed: int
    fill: str           # 'h' | 'latent'
    new_from_h: int = 0
    spare_pages: int = 3
    rope_theta: float = 10000.0
    description: str = ""

    @property
    def batch(self) -> int:
        return len(self.seq_lens)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))

    def pages_of(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.dims.page_size)


def _lognormal_lengths(seed: int, n: int, median: float, sigma: float, lo: int, hi: int) -> tuple:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x5E9])))
    z = rng.standard_normal(n)
    s = np.clip(np.rint(np.exp(math.log(median) + sigma * z)), lo, hi).astype(np.int64)
    return tuple(int(v) for v in s)


WORKLOADS = {
    "tiny_f32": Workload(
        name="tiny_f32", dims=TINY, act="f32", cache="f32", seq_lens=(128,), q_len=1, seed=0,
        fill="h",
        description="tiny MLA decode, fp32: batch 1, 16 heads, d_model 256, d_c 64, rope 16, "
                    "head dim 32, context 128, page 64"),
    "v2_b32_s4096": Workload(
        name="v2_b32_s4096", dims=V2, act="bf16", cache="bf16", seq_lens=(4096,) * 32, q_len=1,
        seed=1, fill="latent",
        description="DeepSeek-V2-shaped decode, bf16: 128 heads, d_c 512, k_pe 64, batch 32, "
                    "seq_len 4096, shuffled 64-token pages"),
    "v2_long_splitkv": Workload(
        name="v2_long_splitkv", dims=V2, act="bf16", cache="bf16",
        seq_lens=(32768, 65536, 98304, 131072), q_len=1, seed=2, fill="latent",
        description="long-context split-KV decode, bf16: batch 4, seq_lens 32K..128K"),
    "v2_ragged_spec": Workload(
        name="v2_ragged_spec", dims=V2, act="bf16", cache="bf16",
        seq_lens=_lognormal_lengths(3, 256, 2048.0, math.log(4.0) / 2.0, 512, 8192), q_len=2,
        seed=3, fill="latent", new_from_h=2,
        description="ragged large-batch speculative decode, bf16: batch 256, lognormal lengths "
                    "(median 2048, clipped 512..8192), 2 query tokens, 2 tokens appended from h"),
    "v2_spec_q4": Workload(
        name="v2_spec_q4", dims=V2, act="bf16", cache="bf16", seq_lens=(4096,) * 64, q_len=4,
        seed=5, fill="latent", new_from_h=4,
        description="multi-token speculative decode, bf16: batch 64, seq_len 4096, 4 causal "
                    "query tokens per request, the 4 new tokens appended from h"),
    "v2_fp8_b128_s8192": Workload(
        name="v2_fp8_b128_s8192", dims=V2, act="bf16", cache="fp8_e4m3", seq_lens=(8192,) * 128,
        q_len=1, seed=4, fill="latent",
        description="fp8 e4m3 latent cache with one per-tensor scale, bf16 q/out: batch 128, "
                    "seq_len 8192"),
    "v2_fp8block_b128_s8192": Workload(
        name="v2_fp8block_b128_s8192", dims=V2, act="bf16", cache="fp8_e4m3_b128",
        seq_lens=(8192,) * 128, q_len=1, seed=6, fill="latent",
        description="block-scaled fp8 latent cache (e4m3 with one scale per 128 latent elements "
                    "of each token, k_pe in bf16), bf16 q/out: batch 128, seq_len 8192"),
}


def scaled(wl: Workload, seq_lens, name=None, **kw) -> Workload:
    """Same workload family (dims, dtypes, seed) with other lengths: for small parity cases."""
    d = dict(wl.__dict__)
    d.update(kw)
    d["seq_lens"] = tuple(int(s) for s in seq_lens)
    d["name"] = name or (wl.name + "_scaled")
    return Workload(**d)


# ----------------------------------------------------------------------------- draws

def _stream(seed: int, *key) -> np.random.Generator:
    words = [int(seed)]
    for k in key:
        words.append(zlib.crc32(str(k).encode()) if not isinstance(k, (int, np.integer)) else int(k))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32.

    This is input encoding (the workload's storage format), not method
    arithmetic. NaN/Inf never occur in the draws.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def _as_act(x: np.ndarray, act: str) -> np.ndarray:
    x = x.astype(np.float32)
    return round_bf16(x) if act == "bf16" else x


def normal(wl: Workload, key, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) draw for stream ``key`` of the workload, in the activation dtype."""
    g = _stream(wl.seed, *(key if isinstance(key, tuple) else (key,)))
    return _as_act(g.standard_normal(shape, dtype=np.float64) * std, wl.act)


def weights(wl: Workload) -> dict:
    """All projection weights, each N(0, 1/fan_in), in the activation dtype.

    Layouts (row-major): W_DKV_KR [d_model][d_c + d_r] = [W^DKV | W^KR];
    W_UK [d_c][H*d_n]; W_UV [d_c][H*d_v]; W_O [H*d_v][d_model].
    """
    d = wl.dims
    H = d.num_heads
    return {
        "W_DKV_KR": normal(wl, "W_DKV_KR", (d.d_model, d.d_cache), 1.0 / math.sqrt(d.d_model)),
        "W_UK": normal(wl, "W_UK", (d.d_latent, H * d.d_nope), 1.0 / math.sqrt(d.d_latent)),
        "W_UV": normal(wl, "W_UV", (d.d_latent, H * d.d_v), 1.0 / math.sqrt(d.d_latent)),
        "W_O": normal(wl, "W_O", (H * d.d_v, d.d_model), 1.0 / math.sqrt(H * d.d_v)),
    }


def query_weights(wl: Workload) -> dict:
    """Query-side weights, each N(0, 1/fan_in), in the activation dtype: W_DQ [d_model][d_q],
    W_UQ [d_q][H*d_n] and W_QR [d_model][H*d_r] (head i owns columns i*d_n.. / i*d_r..)."""
    d = wl.dims
    H = d.num_heads
    return {
        "W_DQ": normal(wl, "W_DQ", (d.d_model, d.d_q), 1.0 / math.sqrt(d.d_model)),
        "W_UQ": normal(wl, "W_UQ", (d.d_q, H * d.d_nope), 1.0 / math.sqrt(d.d_q)),
        "W_QR": normal(wl, "W_QR", (d.d_model, H * d.d_rope), 1.0 / math.sqrt(d.d_model)),
    }


def query_hidden(wl: Workload, rows: int) -> np.ndarray:
    """Hidden states [rows][d_model] ~ N(0,1) of the step's query tokens."""
    return normal(wl, "h_q", (rows, wl.dims.d_model))


def queries(wl: Workload) -> dict:
    """q_nope [B][q][H][d_n] and un-rotated q_pe [B][q][H][d_r], N(0,1)."""
    d = wl.dims
    B, q, H = wl.batch, wl.q_len, d.num_heads
    return {
        "q_nope": normal(wl, "q_nope", (B, q, H, d.d_nope)),
        "q_pe": normal(wl, "q_pe", (B, q, H, d.d_rope)),
    }


def hidden(wl: Workload, b: int, n: int) -> np.ndarray:
    """Hidden states h [n][d_model] ~ N(0,1) for the tokens of request b that come from h."""
    return normal(wl, ("h", b), (n, wl.dims.d_model))


def latent_rows(wl: Workload, b: int, n: int):
    """c_kv [n][d_c] and raw k_pe [n][d_r] ~ N(0,1) for positions 0..n-1 of request b."""
    d = wl.dims
    return (normal(wl, ("c_kv", b), (n, d.d_latent)),
            normal(wl, ("k_pe", b), (n, d.d_rope)))


def token_sources(wl: Workload, b: int):
    """(n_latent, n_from_h): the first n_latent positions are drawn as latents, the rest from h."""
    S = int(wl.seq_lens[b])
    if wl.fill == "h":
        return 0, S
    n_h = min(wl.new_from_h, S)
    return S - n_h, n_h


def page_table(wl: Workload):
    """Shuffled block table.

    Returns (block_table int32 [B][max_pages], num_pages). Request b owns
    ceil(seq_len_b / 64) pages taken in order from one random permutation of
    all page ids; unused entries are -1; ``spare_pages`` ids are never used so
    their contents must stay untouched by appends.
    """
    B = wl.batch
    need = [wl.pages_of(b) for b in range(B)]
    max_pages = max(1, max(need) if need else 1)
    num_pages = int(sum(need)) + wl.spare_pages
    perm = _stream(wl.seed, "block_table").permutation(num_pages).astype(np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :need[b]] = perm[off:off + need[b]]
        off += need[b]
    return bt, num_pages


def fp8_cache_scale(wl: Workload) -> float:
    """Per-tensor e4m3 scale of the latent-filled cache: amax over every drawn c_kv and raw
    k_pe value, divided by 448 (the largest finite e4m3 magnitude). Computed on the drawn
    (bf16) values in float32."""
    amax = 0.0
    for b in range(wl.batch):
        n_lat, _ = token_sources(wl, b)
        if n_lat == 0:
            continue
        c, k = latent_rows(wl, b, n_lat)
        amax = max(amax, float(np.abs(c).max()), float(np.abs(k).max()))
    return float(np.float32(amax) / np.float32(448.0))


def append_batch(wl: Workload, b: int, start: int, n: int):
    """req_ids and positions (int32) for appending positions start..start+n-1 of request b."""
    return (np.full(n, b, dtype=np.int32), np.arange(start, start + n, dtype=np.int32))


def decode_flops(wl: Workload) -> float:
    """Algorithmic FLOPs of one decode call: absorption + scores + latent output."""
    d = wl.dims
    H = d.num_heads
    f = 0.0
    for b in range(wl.batch):
        S = int(wl.seq_lens[b])
        for t in range(wl.q_len):
            kv = S - wl.q_len + t + 1 if S > 0 else 0
            f += 2.0 * H * kv * (d.d_cache + d.d_latent)
        f += 2.0 * wl.q_len * H * d.d_nope * d.d_latent
    return f


def elt_bytes(dtype: str) -> int:
    return {"f32": 4, "bf16": 2, "fp8_e4m3": 1, "fp8_e4m3_b128": 1}[dtype]


def cache_row_bytes(wl: Workload) -> int:
    """Bytes of one token's cache row: (d_c + d_r) elements, or for the block-scaled fp8
    cache d_c codes, one fp32 scale per 128 latent elements and d_r bf16 values."""
    d = wl.dims
    if wl.cache == "fp8_e4m3_b128":
        return d.d_latent + 4 * (d.d_latent // 128) + 2 * d.d_rope
    return d.d_cache * elt_bytes(wl.cache)


def decode_bytes(wl: Workload) -> dict:
    """Algorithmic HBM bytes of one decode call, by tensor (each read or written once)."""
    d = wl.dims
    H, B, q = d.num_heads, wl.batch, wl.q_len
    ea = elt_bytes(wl.act)
    kv_tokens = sum(int(s) for s in wl.seq_lens)
    return {
        "cache": kv_tokens * cache_row_bytes(wl),
        "W_UK_abs": H * d.d_nope * d.d_latent * ea,
        "q": B * q * H * (d.d_nope + d.d_rope) * ea,
        "out_latent": B * q * H * d.d_latent * ea,
        "lse": B * q * H * 4,
        "block_table": sum(wl.pages_of(b) for b in range(B)) * 4 + B * 4,
    }
