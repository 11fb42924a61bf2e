"""fp64 CPU oracle for the DSA attention step (index-K store -> lightning
indexer -> top-2048 -> sparse MLA).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module; only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` do.  It shares no code, constant or helper with the
CUDA library: every constant below is restated from the pages on its own.

Sources (the four web pages collected for dsa_sparse_attention_indexer):

* "vLLM 推理链路概览：以 GLM-5.2 为例", section "DSA Indexer": the indexer score
  s_ij = sum_m w_im ReLU(<q_im, k_j>) and I_i = TopK_{j,2048}(s_ij); section
  "Sparse MLA Attention": alpha = softmax_{j in I, j <= i}(q k^T / sqrt(256)),
  o = sum alpha v.
* "GLM-5.3 推理全链路(十一)", section "索引器缓存里存的是什么": index key = k_norm
  (LayerNorm) -> RoPE on the first 64 dims -> FP8 with one 4-byte ue8m0 scale
  per 128 dims, 132 B/token, 64-token pages of 8448 B; section "主 KV 缓存里存的
  是什么": latent row = 512 FP8 + four 4-byte scales (+ 64 RoPE dims), 656 B.
  Section "优化二: 短上下文直接跳过打分": context <= 2048 selects [0..L-1, -1...].
  Section "配置里的 78 个字符": the indexer_types list and the freq/offset rule.
* "GLM-5.3 推理全链路(一)", section 4.5: indexer_rope_interleave=True, and the
  full layers 0, 1, 2, 6, 10, ..., 74 (21 full, 57 shared).
* "GLM-5.3 推理全链路(十一)", sections "优化三: MTP 迭代内复用 topk" and "优化四":
  the draft steps of one MTP iteration reuse the first step's top-k (only with
  one draft candidate per step), a carried seed row of index_topk +
  index_kpool - 1 int32 is a plain copy of a selected top-k row.
* "GLM-5.3 推理全链路(十一)", section "两个框架的对照": the indexer cache may be
  stored as MXFP4, 128/2 packed bytes + 128/32 ue8m0 scales = 68 B per token.

Readings where the pages are silent (each also listed in the design notes):
LayerNorm eps 1e-6 with optional affine; interleaved RoPE pairs (2i, 2i+1),
angle = pos * base^(-2i/64), base 10000; the ue8m0 scale rounds UP (smallest
power of two with amax <= 448 * scale, amax == 0 -> scale 1) and is stored as an
fp32 power of two; an index-K page stores the 64 payload rows first and then the
64 fp32 scales; a latent row is [512 FP8 | 4 x fp32 scale | 64 bf16 RoPE];
ties in the top-k go to the lower position, -0.0 equals +0.0, and the selected
positions are listed in ascending order followed by -1 padding.

Parity pins: every function here is pinned by tests under ``-m "not gpu"``
(codec vs the format definition and torch's float8 casts, the E4M3 spacing used
by the one-ulp bar against the value set torch decodes, the score magnitude D_j
against the score without cancellation and a term-by-term sum with it, layout
constants the pages print, the 21/57 schedule, brute-force top-k, sparse == dense attention
when the context fits in the top-k, closed forms, the MTP seed width and
draft-step read counts the pages print, brute-force top-k per draft position,
the 68-byte MXFP4 token, the E2M1 codec against its value table and rounding
rule, the MX scale property amax / 2**e in [4, 8), the MXFP4 key of a token
within the format's bound of torch's LayerNorm and a complex rotation, and a
whole request's MXFP4 top-k against brute force, the context-parallel merges of
top-k candidates and of attention parts against brute force and dense attention).
The MTP reading where the pages are silent: a draft step with a context of at
most 2048 publishes its all-positions row like any other step.  The LayerNorm
eps, RoPE base and RoPE pairing are NOT fixed by the pages: "parity unpinned" for those three
parameters - the tests check only self-consistency (moments, pair norms, the
rotation group law) for them.
"""

from __future__ import annotations

import math
import numpy as np

# ----------------------------------------------------------------------------
# Constants restated from the pages ("GLM-5.3 推理全链路(十一)", index cache and
# main KV cache sections; "vLLM 推理链路概览", DSA Indexer / Sparse MLA).
# ----------------------------------------------------------------------------
PAGE_TOKENS = 64                   # page_size == 64 (asserted on the CUDA path)
INDEX_HEAD_DIM = 128               # index_head_dim == 128
INDEX_HEADS = 32                   # 32 indexer query heads
INDEX_TOKEN_BYTES = 128 + 4        # FP8 key + one 4-byte scale per 128 dims
INDEX_PAGE_BYTES = PAGE_TOKENS * INDEX_TOKEN_BYTES   # 8448
LATENT_DIM = 512                   # kv_lora_rank
ROPE_DIM = 64                      # qk_rope_head_dim
LATENT_TOKEN_BYTES = 512 + 4 * 4 + 64 * 2            # 656
LATENT_PAGE_BYTES = PAGE_TOKENS * LATENT_TOKEN_BYTES  # 41984
MLA_HEADS = 64
TOPK = 2048                        # index_topk
SOFTMAX_SCALE = 1.0 / math.sqrt(256.0)
E4M3_MAX = 448.0


# ----------------------------------------------------------------------------
# FP8 E4M3 codec written from the OCP FP8 format definition: 1 sign bit, 4
# exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN.
# ----------------------------------------------------------------------------
def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 codes, in fp64 (NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            out[code] = np.nan
        elif exp == 0:
            out[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)      # subnormal
        else:
            out[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return out


_E4M3_TABLE = e4m3_decode_table()
# Non-negative finite codes 0x00..0x7E in increasing value order.
_E4M3_POS_CODES = np.arange(0x7F, dtype=np.int64)
_E4M3_POS_VALS = _E4M3_TABLE[:0x7F]


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8).astype(np.int64)]


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round each |x| <= 448 to the nearest E4M3 value, ties to the even code.

    The caller guarantees |x| <= 448 (the scale rule below ensures it), so no
    saturation rule is needed.  A value that rounds to zero keeps its sign.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    if np.any(ax > E4M3_MAX) or np.any(~np.isfinite(ax)):
        raise ValueError("e4m3_encode: input outside [-448, 448]")
    hi = np.searchsorted(_E4M3_POS_VALS, ax, side="left")       # first value >= ax
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS_VALS[hi] - ax
    d_lo = ax - _E4M3_POS_VALS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((lo & 1) == 0))
    code = np.where(pick_lo, lo, hi)
    code = np.where(ax == _E4M3_POS_VALS[hi], hi, code)          # exact hits
    sign = np.signbit(x).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def e4m3_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of E4M3 values around |v| (the step used for the 1-ulp bar)."""
    av = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(av, 2.0 ** -6)))
    return 2.0 ** (e - 3)


# ----------------------------------------------------------------------------
# ue8m0 block scale: a pure power of two, one per 128 values.
# ----------------------------------------------------------------------------
def ue8m0_exponent(amax):
    """Smallest integer e with amax <= 448 * 2**e; amax == 0 gives e = 0.

    Works elementwise.  The logarithm only gives a starting guess; the result
    is settled by exact comparisons against powers of two (ldexp is exact in
    fp64).
    """
    a = np.asarray(amax, dtype=np.float64)
    e = np.zeros(a.shape, dtype=np.int64)
    nz = a > 0
    e[nz] = np.floor(np.log2(a[nz] / E4M3_MAX)).astype(np.int64)
    for _ in range(4):
        up = nz & (a > np.ldexp(E4M3_MAX, e))
        e[up] += 1
        down = nz & (a <= np.ldexp(E4M3_MAX, e - 1))
        e[down] -= 1
    assert np.all(a[nz] <= np.ldexp(E4M3_MAX, e[nz]))
    assert np.all(a[nz] > np.ldexp(E4M3_MAX, e[nz] - 1))
    return e if e.ndim else int(e)


def quantize_blocks_128(x: np.ndarray):
    """Quantise each run of 128 values: returns (E4M3 codes, fp64 scales 2**e)."""
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] == 128
    e = np.asarray(ue8m0_exponent(np.max(np.abs(x), axis=-1)))
    scales = np.ldexp(1.0, e)
    codes = e4m3_encode(x / scales[..., None])
    return codes, scales


# ----------------------------------------------------------------------------
# Index-key preparation: k_norm (LayerNorm) -> RoPE on dims 0..63 -> FP8.
# ----------------------------------------------------------------------------
def layer_norm(x: np.ndarray, gamma=None, beta=None, eps: float = 1e-6) -> np.ndarray:
    """LayerNorm over the last axis with biased variance."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    y = (x - mu) / np.sqrt(var + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    if beta is not None:
        y = y + np.asarray(beta, dtype=np.float64)
    return y


def rope_interleaved(x: np.ndarray, pos: np.ndarray, base: float = 10000.0,
                     rope_dims: int = 64) -> np.ndarray:
    """Rotate the pairs (x[2i], x[2i+1]), i < rope_dims/2, by pos * base**(-2i/rope_dims).

    Dims >= rope_dims pass through unchanged.
    """
    x = np.array(x, dtype=np.float64, copy=True)
    pos = np.asarray(pos, dtype=np.float64).reshape(-1, 1)
    i = np.arange(rope_dims // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / rope_dims)
    ang = pos * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x0 = x[..., 0:rope_dims:2].copy()
    x1 = x[..., 1:rope_dims:2].copy()
    x[..., 0:rope_dims:2] = x0 * c - x1 * s
    x[..., 1:rope_dims:2] = x0 * s + x1 * c
    return x


def index_k_prepare(k: np.ndarray, pos: np.ndarray, gamma=None, beta=None,
                    eps: float = 1e-6, rope_base: float = 10000.0):
    """The index key of each token before caching: (E4M3 codes [n,128], scale [n])."""
    y = layer_norm(k, gamma, beta, eps)
    y = rope_interleaved(y, pos, rope_base, 64)
    return quantize_blocks_128(y)


# ----------------------------------------------------------------------------
# Paged cache byte layouts.
# ----------------------------------------------------------------------------
def index_cache_write(cache: np.ndarray, slot: np.ndarray, codes: np.ndarray,
                      scales: np.ndarray) -> None:
    """Write tokens into an index-K cache [num_pages, 8448] (uint8).

    Within a page: bytes [0, 8192) hold the 64 FP8 rows of 128 B, bytes
    [8192, 8448) hold the 64 scales as little-endian fp32.  slot < 0 is skipped.
    """
    assert cache.dtype == np.uint8 and cache.shape[1] == INDEX_PAGE_BYTES
    slot = np.asarray(slot, dtype=np.int64)
    keep = slot >= 0
    page, row = np.divmod(slot[keep], PAGE_TOKENS)
    cache[page[:, None], row[:, None] * 128 + np.arange(128)] = np.asarray(codes)[keep]
    sbytes = np.asarray(scales, dtype="<f4")[keep].view(np.uint8).reshape(-1, 4)
    cache[page[:, None], PAGE_TOKENS * 128 + 4 * row[:, None] + np.arange(4)] = sbytes


def index_cache_read(cache: np.ndarray, page_table_row: np.ndarray, n_tokens: int):
    """Read logical tokens 0..n-1 of one request: (codes [n,128], scales fp64 [n])."""
    j = np.arange(n_tokens, dtype=np.int64)
    page = np.asarray(page_table_row, dtype=np.int64)[j // PAGE_TOKENS]
    row = j % PAGE_TOKENS
    codes = cache[page[:, None], row[:, None] * 128 + np.arange(128)]
    sb = cache[page[:, None], PAGE_TOKENS * 128 + 4 * row[:, None] + np.arange(4)]
    scales = np.ascontiguousarray(sb).view("<f4").reshape(-1).astype(np.float64)
    return codes, scales


def latent_quantize(c: np.ndarray):
    """Latent c [n,512] -> (codes [n,512], scales [n,4]) with one scale per 128 dims."""
    c = np.asarray(c, dtype=np.float64)
    codes, scales = quantize_blocks_128(c.reshape(c.shape[0], 4, 128))
    return codes.reshape(c.shape[0], 512), scales


def latent_cache_write(cache: np.ndarray, slot: np.ndarray, codes: np.ndarray,
                       scales: np.ndarray, rope_bf16_bits: np.ndarray) -> None:
    """Write tokens into a latent cache [num_pages, 41984] (uint8).

    Token row of 656 B at 656 * (slot % 64): [0,512) FP8 latent, [512,528) four
    little-endian fp32 scales, [528,656) 64 RoPE values as raw bf16 bits.
    """
    assert cache.dtype == np.uint8 and cache.shape[1] == LATENT_PAGE_BYTES
    slot = np.asarray(slot, dtype=np.int64)
    keep = slot >= 0
    page, row = np.divmod(slot[keep], PAGE_TOKENS)
    base = row[:, None] * LATENT_TOKEN_BYTES
    cache[page[:, None], base + np.arange(512)] = np.asarray(codes)[keep]
    sb = np.asarray(scales, dtype="<f4")[keep].view(np.uint8).reshape(-1, 16)
    cache[page[:, None], base + 512 + np.arange(16)] = sb
    rb = np.ascontiguousarray(np.asarray(rope_bf16_bits, dtype="<u2")[keep]).view(np.uint8)
    cache[page[:, None], base + 528 + np.arange(128)] = rb.reshape(-1, 128)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def latent_cache_read_rows(cache: np.ndarray, page_table_row: np.ndarray,
                           positions: np.ndarray) -> np.ndarray:
    """Dequantised 576-d rows [len(positions), 576]: (c * scale | rope)."""
    j = np.asarray(positions, dtype=np.int64)
    page = np.asarray(page_table_row, dtype=np.int64)[j // PAGE_TOKENS]
    base = (j % PAGE_TOKENS)[:, None] * LATENT_TOKEN_BYTES
    rows = cache[page[:, None], base + np.arange(LATENT_TOKEN_BYTES)]
    out = np.empty((len(j), LATENT_DIM + ROPE_DIM), dtype=np.float64)
    sc = np.ascontiguousarray(rows[:, 512:528]).view("<f4").astype(np.float64)   # [n,4]
    out[:, :512] = e4m3_decode(rows[:, :512]) * np.repeat(sc, 128, axis=1)
    out[:, 512:] = bf16_bits_to_f64(np.ascontiguousarray(rows[:, 528:656]).view("<u2"))
    return out


# ----------------------------------------------------------------------------
# Lightning indexer ("vLLM 推理链路概览", DSA Indexer).
# ----------------------------------------------------------------------------
def index_q_quantize(q: np.ndarray):
    """Indexer query [T,32,128] -> (E4M3 codes, per-head scales [T,32])."""
    return quantize_blocks_128(q)


def indexer_scores(q_codes, q_scales, w, k_codes, k_scales) -> np.ndarray:
    """s_j = sum_m w_m * ReLU(<q_m, k_j>) on the dequantised FP8 values.

    q_codes [32,128], q_scales [32], w [32], k_codes [L,128], k_scales [L];
    returns fp64 [L].
    """
    q = e4m3_decode(q_codes) * np.asarray(q_scales, np.float64)[:, None]
    k = e4m3_decode(k_codes) * np.asarray(k_scales, np.float64)[:, None]
    dots = k @ q.T                                   # [L, 32]
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


def score_magnitude(q_codes, q_scales, w, k_codes, k_scales) -> np.ndarray:
    """D_j = sum_m |w_m| * |<q_m, k_j>|: the scale against which a score's
    relative error is measured (>= |s_j|, equal to it without cancellation)."""
    q = e4m3_decode(q_codes) * np.asarray(q_scales, np.float64)[:, None]
    k = e4m3_decode(k_codes) * np.asarray(k_scales, np.float64)[:, None]
    dots = k @ q.T
    return np.abs(dots) @ np.abs(np.asarray(w, dtype=np.float64))


def topk_positions(scores: np.ndarray, n_valid: int, k: int = TOPK) -> np.ndarray:
    """Top-k positions among scores[0:n_valid] as int32 [k], ascending, -1 padded.

    n_valid <= k selects every valid position ("优化二").  Otherwise the order is
    descending score, ties to the lower position; -0.0 and +0.0 are equal.
    """
    out = np.full(k, -1, dtype=np.int32)
    if n_valid <= k:
        out[:n_valid] = np.arange(n_valid, dtype=np.int32)
        return out
    s = np.asarray(scores[:n_valid], dtype=np.float64) + 0.0    # -0.0 -> +0.0
    order = np.lexsort((np.arange(n_valid), -s))
    out[:] = np.sort(order[:k]).astype(np.int32)
    return out


# ----------------------------------------------------------------------------
# Sparse MLA in absorbed (MQA) form ("vLLM 推理链路概览", Sparse MLA Attention).
# ----------------------------------------------------------------------------
def sparse_mla(q: np.ndarray, positions: np.ndarray, kv_rows: np.ndarray,
               query_pos: int, scale: float = SOFTMAX_SCALE):
    """One query token: q [64,576], positions [k] (-1 = empty), kv_rows [k,576]
    dequantised rows for those positions.  Returns (out [64,512], lse [64]).

    Only positions j with 0 <= j <= query_pos take part (the causal mask).
    """
    positions = np.asarray(positions)
    keep = (positions >= 0) & (positions <= query_pos)
    kv = np.asarray(kv_rows, dtype=np.float64)[keep]
    q = np.asarray(q, dtype=np.float64)
    if kv.shape[0] == 0:
        return np.zeros((q.shape[0], LATENT_DIM)), np.full(q.shape[0], -np.inf)
    s = (q @ kv.T) * scale                           # [64, n]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ kv[:, :LATENT_DIM]) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


# ----------------------------------------------------------------------------
# Context-parallel split of one long request over G ranks ("GLM-5.3 推理全链路
# (十一)", 两个框架的对照: with prefill context parallelism the indexer's reads
# are spread over the ranks; "Accelerating GLM-5.3-Flash on H200", prefill 的
# 重点是少搬一次、少等一次: CP4 on the prefill side).  Each rank holds a disjoint
# slice of the request's positions, scores it, and keeps its own top-k; the
# top-k of the whole context is the top-k of the union of those lists, because
# every globally selected position is also selected within its own slice.
# Attention over the selected positions splits the same way: a rank attends
# over the selected positions it holds, and the parts are combined by their
# log-sum-exp.
# ----------------------------------------------------------------------------
def cp_merge_topk(cand_pos_list, cand_score_list, k: int = TOPK) -> np.ndarray:
    """Top-k of the union of per-rank candidate lists.

    cand_pos_list[g]: global positions (-1 = no candidate); cand_score_list[g]:
    their scores.  Order: descending score, ties to the lower position, -0.0
    equal to +0.0.  Returns int32 [k]: the selected positions ascending, -1
    padded.
    """
    pos = np.concatenate([np.asarray(p, dtype=np.int64).ravel() for p in cand_pos_list])
    sc = np.concatenate([np.asarray(s, dtype=np.float64).ravel() for s in cand_score_list])
    keep = pos >= 0
    pos, sc = pos[keep], sc[keep] + 0.0
    order = np.lexsort((pos, -sc))[:k]
    out = np.full(k, -1, dtype=np.int32)
    sel = np.sort(pos[order])
    out[:sel.size] = sel
    return out


def lse_merge(outs, lses):
    """Softmax attention over a disjoint union of key sets, from the parts.

    outs[g] [H, D]: attention normalised within part g; lses[g] [H]: the
    natural-log sum of exp(score) over part g (-inf for an empty part).  With
    M = max_g lse_g and w_g = exp(lse_g - M):
        out = sum_g w_g out_g / sum_g w_g,   lse = M + log(sum_g w_g).
    Returns (out [H, D], lse [H]); a head empty in every part gives 0 and -inf.
    """
    lses = np.stack([np.asarray(x, dtype=np.float64) for x in lses])    # [G, H]
    outs = np.stack([np.asarray(x, dtype=np.float64) for x in outs])    # [G, H, D]
    M = np.max(lses, axis=0)                                            # [H]
    finite = np.isfinite(M)
    w = np.where(np.isfinite(lses), np.exp(lses - np.where(finite, M, 0.0)), 0.0)
    den = w.sum(axis=0)
    out = np.where(finite[:, None], (w[:, :, None] * outs).sum(axis=0) / np.where(finite, den, 1.0)[:, None], 0.0)
    lse = np.where(finite, M + np.log(np.where(finite, den, 1.0)), -np.inf)
    return out, lse


# ----------------------------------------------------------------------------
# Full / shared layer schedule ("配置里的 78 个字符").
# ----------------------------------------------------------------------------
def parse_indexer_types(types) -> list:
    """True for a full layer (runs the indexer), False for a shared layer."""
    out = []
    for t in types:
        if t == "full":
            out.append(True)
        elif t == "shared":
            out.append(False)
        else:
            raise ValueError(f"unknown indexer type {t!r}")
    return out


def layer_skips_topk(layer_id: int, freq: int, offset: int) -> bool:
    """The parameterised form: skip (shared) iff max(l - offset + 1, 0) % freq != 0."""
    return max(layer_id - offset + 1, 0) % freq != 0


def layer_skips_topk_config(layer_id: int, indexer_types=None, cli_factor: int = 1, index_topk_pattern=None,
                            index_topk_freq: int = 1, index_skip_topk_offset=None) -> bool:
    """Whether a layer reuses the previous top-k, from whichever schedule fields
    a config carries, in the order the pages give ("配置里的 78 个字符"): the
    explicit indexer_types list; else cli_factor > 1 (a fresh top-k every
    cli_factor layers); else index_topk_pattern ('S' marks a shared layer);
    else the index_topk_freq rule with index_skip_topk_offset, whose default 2
    gives max(layer_id - 1, 0) % freq != 0 (layers 0 and 1 full, 2 shared).
    Layers past the end of a list or pattern are full."""
    if indexer_types is not None:
        return 0 <= layer_id < len(indexer_types) and indexer_types[layer_id] == "shared"
    if cli_factor > 1:
        return layer_id % cli_factor != 0
    if index_topk_pattern is not None:
        return layer_id < len(index_topk_pattern) and index_topk_pattern[layer_id] == "S"
    off = 2 if index_skip_topk_offset is None else index_skip_topk_offset
    return layer_skips_topk(layer_id, index_topk_freq, off)


# ----------------------------------------------------------------------------
# One request through the whole step, for the tests and the CPU baseline.
# ----------------------------------------------------------------------------
def request_topk(q_idx, w, idx_cache, page_table_row, seq_len, q_len):
    """Indexer + top-k for one request's query tokens.

    q_idx [q_len,32,128] fp64, w [q_len,32].  Query token t sits at position
    p = seq_len - q_len + t and sees the L_t = p + 1 positions 0..p.  Returns
    (topk int32 [q_len, 2048], scores list of fp64 [L_t] or None when L_t <= 2048).
    """
    k_codes, k_scales = index_cache_read(idx_cache, page_table_row, seq_len)
    out = np.empty((q_len, TOPK), dtype=np.int32)
    all_scores = []
    for t in range(q_len):
        n_valid = seq_len - q_len + t + 1
        if n_valid <= TOPK:
            out[t] = topk_positions(None, n_valid)
            all_scores.append(None)
            continue
        qc, qs = index_q_quantize(q_idx[t])
        s = indexer_scores(qc, qs, w[t], k_codes[:n_valid], k_scales[:n_valid])
        out[t] = topk_positions(s, n_valid)
        all_scores.append(s)
    return out, all_scores


# ----------------------------------------------------------------------------
# Top-k reuse across the draft steps of one MTP iteration ("GLM-5.3 推理全链路
# (十一)", sections 优化三: MTP 迭代内复用 topk, 优化四: PD 分离下的 seed 传输,
# 乘法二: 投机草稿步数 × full 层数, and 误解四).
# ----------------------------------------------------------------------------
def mtp_topk_width(index_topk: int = TOPK, index_kpool: int = 1) -> int:
    """Width of a seed row: index_topk + index_kpool - 1 (2048 for GLM-5.3,
    whose index_kpool is 1; the extra kpool - 1 slots are tail slots)."""
    if index_topk < 1 or index_kpool < 1:
        raise ValueError("index_topk and index_kpool must be >= 1")
    return index_topk + index_kpool - 1


def mtp_seed_write(topk: np.ndarray, src_rows: np.ndarray, width: int) -> np.ndarray:
    """Seed buffer [n, width] int32: row r is a plain copy of the selected
    top-k row topk[src_rows[r]] (2048 int32), the tail slots are -1.  A source
    row outside topk gives a row of -1."""
    topk = np.asarray(topk, dtype=np.int32)
    src_rows = np.asarray(src_rows, dtype=np.int64)
    if width < TOPK:
        raise ValueError("seed width below index_topk")
    seed = np.full((len(src_rows), width), -1, dtype=np.int32)
    for r, s in enumerate(src_rows):
        if 0 <= s < topk.shape[0]:
            seed[r, :TOPK] = topk[s]
    return seed


class MtpShareState:
    """The shared top-k state across the draft steps of one MTP iteration.

    begin(): reuse is on only when it is enabled AND the draft keeps one
    candidate per step (eagle topk == 1: with more, the draft's rows are
    reordered and a carried row no longer matches its request).  With reuse on,
    a carried seed is kept when keep_carry_seed is set and one is given;
    otherwise the state starts empty.  While reuse is on, the first step that
    has no indices runs the indexer and publishes; every later step takes the
    published indices.  end() forgets everything.  With reuse off every draft
    step runs its own indexer.
    """

    def __init__(self):
        self.reuse = False
        self.indices = None

    def begin(self, enabled: bool, eagle_topk: int, keep_carry_seed: bool = False, seed=None) -> bool:
        self.reuse = bool(enabled) and eagle_topk == 1
        self.indices = None
        if self.reuse and keep_carry_seed and seed is not None:
            self.indices = np.asarray(seed, dtype=np.int32)
        return self.reuse

    def needs_scoring(self) -> bool:
        return not (self.reuse and self.indices is not None)

    def publish(self, topk: np.ndarray):
        self.indices = np.asarray(topk, dtype=np.int32)

    def end(self):
        self.reuse = False
        self.indices = None


def mtp_draft_topk(q_idx, w, idx_cache, page_table_row, seq_len0, n_steps, state: MtpShareState):
    """The indices every draft step of one request attends with.

    Draft step k (k = 0 .. n_steps-1) holds seq_len0 + k tokens and queries the
    last one, at position seq_len0 - 1 + k, with q_idx[k] [32,128] and w[k] [32].
    A step that needs scoring runs the indexer + top-2048 on its whole visible
    context and publishes; the others reuse the published row as it is.
    Returns (topk int32 [n_steps, 2048], index-cache tokens read), the read
    count being 0 for a reused step, and the context for a scored one (a
    context <= 2048 takes every position without scores and reads nothing)."""
    out = np.empty((n_steps, TOPK), dtype=np.int32)
    read = 0
    for k in range(n_steps):
        L = seq_len0 + k
        if state.needs_scoring():
            row, _ = request_topk(q_idx[k:k + 1], w[k:k + 1], idx_cache, page_table_row, L, 1)
            if state.reuse:
                state.publish(row[0])
            out[k] = row[0]
            read += L if L > TOPK else 0
        else:
            out[k] = state.indices
    return out, read


# ----------------------------------------------------------------------------
# MXFP4 index-K cache ("GLM-5.3 推理全链路(十一)", section 两个框架的对照: the same
# indexer cache stored as MXFP4, head_dim/2 bytes of packed values plus
# head_dim/block ue8m0 scales, 128/2 + 128/32 = 68 B per token).
#
# Readings where the pages are silent: MXFP4 as the OCP Microscaling format
# defines it - blocks of 32 values share one E8M0 scale 2**e with
# e = floor(log2(amax)) - 2 (2 is the exponent of E2M1's largest value, 6), the
# elements are E2M1 rounded to nearest with ties to even and saturated at +-6;
# amax == 0 gives e = 0.  Two values per byte, the even element in the low
# nibble.  A page holds the 64 packed rows of 64 B, then the 64 tokens' 4 scale
# bytes (e + 127), 4352 B in all.  The query side is unchanged (FP8, one scale
# per head) and scores are formed on the dequantised values.
# ----------------------------------------------------------------------------
MXFP4_BLOCK = 32
MXFP4_TOKEN_BYTES = INDEX_HEAD_DIM // 2 + INDEX_HEAD_DIM // MXFP4_BLOCK     # 68
MXFP4_PAGE_BYTES = PAGE_TOKENS * MXFP4_TOKEN_BYTES                          # 4352
E2M1_EMAX = 2                      # 6 = 1.5 * 2**2


def e2m1_decode_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes: sign bit 3, exponent bits 2..1 with
    bias 1, mantissa bit 0; exponent 0 is subnormal (m * 0.5)."""
    out = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 8 else 1.0
        exp = (code >> 1) & 3
        man = code & 1
        out[code] = sign * (man * 0.5 if exp == 0 else (1.0 + man / 2.0) * 2.0 ** (exp - 1))
    return out


_E2M1_TABLE = e2m1_decode_table()
_E2M1_POS_VALS = _E2M1_TABLE[:8]


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    return _E2M1_TABLE[np.asarray(codes, dtype=np.int64) & 15]


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E2M1 value of each x (|x| > 6 saturates to 6), ties to the even
    code; the sign bit follows x (a value that rounds to zero keeps it)."""
    x = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(x)):
        raise ValueError("e2m1_encode: non-finite input")
    ax = np.minimum(np.abs(x), _E2M1_POS_VALS[7])
    hi = np.minimum(np.searchsorted(_E2M1_POS_VALS, ax, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E2M1_POS_VALS[hi] - ax
    d_lo = ax - _E2M1_POS_VALS[lo]
    code = np.where((d_lo < d_hi) | ((d_lo == d_hi) & ((lo & 1) == 0)), lo, hi)
    code = np.where(ax == _E2M1_POS_VALS[hi], hi, code)
    return (code | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)


def mxfp4_exponent(amax):
    """Shared block exponent floor(log2(amax)) - 2, clamped to [-127, 127];
    amax == 0 gives 0.  frexp gives floor(log2) exactly."""
    a = np.asarray(amax, dtype=np.float64)
    _, k = np.frexp(a)                                  # a = m * 2**k, m in [0.5, 1)
    e = np.where(a > 0, k.astype(np.int64) - 1 - E2M1_EMAX, 0)
    e = np.clip(e, -127, 127)
    return e if e.ndim else int(e)


def quantize_mxfp4(x: np.ndarray):
    """[..., 128] -> (E2M1 codes [..., 128] in 0..15, block exponents [..., 4])."""
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] == INDEX_HEAD_DIM
    xb = x.reshape(x.shape[:-1] + (INDEX_HEAD_DIM // MXFP4_BLOCK, MXFP4_BLOCK))
    e = np.asarray(mxfp4_exponent(np.max(np.abs(xb), axis=-1)))
    codes = e2m1_encode(xb / np.ldexp(1.0, e)[..., None])
    return codes.reshape(x.shape), e


def mxfp4_dequant(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    c = e2m1_decode(codes)
    cb = c.reshape(c.shape[:-1] + (INDEX_HEAD_DIM // MXFP4_BLOCK, MXFP4_BLOCK))
    return (cb * np.ldexp(1.0, np.asarray(exps))[..., None]).reshape(c.shape)


def index_k_prepare_mxfp4(k: np.ndarray, pos: np.ndarray, gamma=None, beta=None,
                          eps: float = 1e-6, rope_base: float = 10000.0):
    """The index key of each token as MXFP4: (codes [n,128], exponents [n,4])."""
    y = layer_norm(k, gamma, beta, eps)
    y = rope_interleaved(y, pos, rope_base, 64)
    return quantize_mxfp4(y)


def mxfp4_cache_write(cache: np.ndarray, slot: np.ndarray, codes: np.ndarray, exps: np.ndarray) -> None:
    """Write tokens into an MXFP4 index-K cache [num_pages, 4352] (uint8).

    Within a page: bytes [0, 4096) hold the 64 rows of 64 packed bytes (byte j
    = code 2j | code 2j+1 << 4), bytes [4096, 4352) the 64 tokens' 4 scale
    bytes e + 127.  slot < 0 is skipped."""
    assert cache.dtype == np.uint8 and cache.shape[1] == MXFP4_PAGE_BYTES
    slot = np.asarray(slot, dtype=np.int64)
    keep = slot >= 0
    page, row = np.divmod(slot[keep], PAGE_TOKENS)
    c = np.asarray(codes, dtype=np.uint8)[keep]
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    cache[page[:, None], row[:, None] * 64 + np.arange(64)] = packed
    eb = (np.asarray(exps, dtype=np.int64)[keep] + 127).astype(np.uint8)
    cache[page[:, None], PAGE_TOKENS * 64 + 4 * row[:, None] + np.arange(4)] = eb


def mxfp4_cache_read(cache: np.ndarray, page_table_row: np.ndarray, n_tokens: int):
    """Logical tokens 0..n-1 of one request: (codes [n,128], exponents [n,4])."""
    j = np.arange(n_tokens, dtype=np.int64)
    page = np.asarray(page_table_row, dtype=np.int64)[j // PAGE_TOKENS]
    row = j % PAGE_TOKENS
    packed = cache[page[:, None], row[:, None] * 64 + np.arange(64)]
    codes = np.empty((n_tokens, INDEX_HEAD_DIM), dtype=np.uint8)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    exps = cache[page[:, None], PAGE_TOKENS * 64 + 4 * row[:, None] + np.arange(4)].astype(np.int64) - 127
    return codes, exps


def indexer_scores_mxfp4(q_codes, q_scales, w, k_codes, k_exps) -> np.ndarray:
    """s_j = sum_m w_m * ReLU(<q_m, k_j>) with FP8 queries and MXFP4 keys."""
    q = e4m3_decode(q_codes) * np.asarray(q_scales, np.float64)[:, None]
    k = mxfp4_dequant(k_codes, k_exps)
    return np.maximum(k @ q.T, 0.0) @ np.asarray(w, dtype=np.float64)


def score_magnitude_mxfp4(q_codes, q_scales, w, k_codes, k_exps) -> np.ndarray:
    q = e4m3_decode(q_codes) * np.asarray(q_scales, np.float64)[:, None]
    k = mxfp4_dequant(k_codes, k_exps)
    return np.abs(k @ q.T) @ np.abs(np.asarray(w, dtype=np.float64))


def request_topk_mxfp4(q_idx, w, cache, page_table_row, seq_len, q_len):
    """request_topk over an MXFP4 index-K cache."""
    k_codes, k_exps = mxfp4_cache_read(cache, page_table_row, seq_len)
    out = np.empty((q_len, TOPK), dtype=np.int32)
    all_scores = []
    for t in range(q_len):
        n_valid = seq_len - q_len + t + 1
        if n_valid <= TOPK:
            out[t] = topk_positions(None, n_valid)
            all_scores.append(None)
            continue
        qc, qs = index_q_quantize(q_idx[t])
        s = indexer_scores_mxfp4(qc, qs, w[t], k_codes[:n_valid], k_exps[:n_valid])
        out[t] = topk_positions(s, n_valid)
        all_scores.append(s)
    return out, all_scores


# ----------------------------------------------------------------------------
# The latent row written upstream of sparse MLA, from the A-projection outputs
# ("GLM-5.3 推理全链路(一)", section 4.3 两个 RMSNorm 与 RoPE: kv_a_layernorm over
# the 512-d kv_c, RoPE on the 64-d k_pe only, and the fused kernel writes the
# result into the KV pool - and, on a layer with an indexer, the index key too).
# Readings where the pages are silent: RMSNorm y = x / sqrt(mean(x^2) + eps)
# times an optional gamma, eps 1e-6; the k_pe rotation uses the index key's
# convention (interleaved pairs, base 10000, all 64 dims); the rotated values
# are stored as bf16 rounded to nearest even (through torch's fp64 -> bf16
# cast, a library step).
# ----------------------------------------------------------------------------
def rms_norm(x: np.ndarray, gamma=None, eps: float = 1e-6) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    return y


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float64))).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def latent_prepare(kv_c: np.ndarray, k_pe: np.ndarray, pos: np.ndarray, gamma=None, eps: float = 1e-6,
                   rope_base: float = 10000.0):
    """One latent row per token from the raw kv_c [n,512] and k_pe [n,64]:
    (FP8 codes [n,512], scales [n,4], RoPE bf16 bits [n,64])."""
    c = rms_norm(kv_c, gamma, eps)
    r = rope_interleaved(np.asarray(k_pe, dtype=np.float64), pos, rope_base, ROPE_DIM)
    codes, scales = latent_quantize(c)
    return codes, scales, f64_to_bf16_bits(r)
