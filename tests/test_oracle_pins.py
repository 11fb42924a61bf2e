"""Pins for the fp64 oracle, independent of the oracle's own formulas.

Each test checks the oracle against something other than itself: the format
definition through torch's float8 casts (a library routine), numbers the pages
print (tests/golden/pages_constants.json), closed forms, invariants, brute force
on tiny inputs, and textbook special cases (sparse attention over the whole
context equals dense attention computed by torch's SDPA).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))


def g(name):
    return GOLDEN[name]["value"]


# ------------------------------------------------------------------ FP8 codec
def test_e4m3_decode_matches_torch_for_all_256_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert np.array_equal(ref[~nan], mine[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9      # max normal, min subnormal


def test_e4m3_encode_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(1)
    mags = np.exp2(rng.uniform(-12, np.log2(448.0), 200000))
    x = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x.astype(np.float64)), ref)


def test_e4m3_encode_ties_to_even_at_every_midpoint():
    vals = O.e4m3_decode_table()[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2.0                   # exactly representable in fp32
    ref = torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = O.e4m3_encode(mids)
    assert np.array_equal(mine, ref)
    assert np.all(mine % 2 == 0)                          # the even neighbour wins


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)


# ------------------------------------------------------------------ ue8m0 scale
@pytest.mark.parametrize("amax,e", [(448.0, 0), (448.0001, 1), (1.0, -8), (0.875, -9),
                                    (0.0, 0), (3.5, -7), (3.5000001, -6), (896.0, 1)])
def test_ue8m0_hand_values(amax, e):
    assert O.ue8m0_exponent(amax) == e


def test_ue8m0_defining_property_and_e8m0_representable():
    rng = np.random.default_rng(2)
    a = np.exp2(rng.uniform(-60, 60, 10000))
    e = O.ue8m0_exponent(a)
    assert np.all(a <= 448.0 * np.exp2(e)) and np.all(a > 448.0 * np.exp2(e - 1))
    s = torch.from_numpy(np.exp2(e).astype(np.float32))
    back = s.to(torch.float8_e8m0fnu).to(torch.float32)       # a power of two survives e8m0
    assert torch.equal(back, s)


def test_quantised_block_within_half_ulp_and_no_saturation():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((500, 128)) * np.exp2(rng.uniform(-20, 20, (500, 1)))
    codes, scales = O.quantize_blocks_128(x)
    deq = O.e4m3_decode(codes) * scales[:, None]
    assert np.all(np.abs(deq / scales[:, None]) <= 448.0)
    err = np.abs(deq - x) / scales[:, None]
    assert np.all(err <= O.e4m3_ulp(x / scales[:, None]) / 2 + 1e-300)


def _torch_e4m3_values():
    """Finite non-negative E4M3 values in code order, decoded by torch's cast."""
    v = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.all(np.diff(v) > 0)
    return v


def test_e4m3_ulp_is_the_gap_to_the_next_value_of_the_format():
    # The one-ulp store bar rests on this spacing, so it is pinned to the value
    # set torch decodes, not to the oracle's own table: at every finite
    # non-negative code the spacing is the distance to the next code's value
    # (the largest code, 448, keeps the spacing of its binade), and strictly
    # between two neighbouring codes it is the gap between them.
    v = _torch_e4m3_values()
    gaps = np.append(np.diff(v), v[-1] - v[-2])
    assert np.array_equal(O.e4m3_ulp(v), gaps)
    assert np.array_equal(O.e4m3_ulp(-v), gaps)                    # sign-blind
    rng = np.random.default_rng(31)
    t = rng.uniform(0.0, 1.0, v.size - 1)
    inner = v[:-1] + t * (v[1:] - v[:-1])
    inner = inner[(inner > v[:-1]) & (inner < v[1:])]
    lo = np.searchsorted(v, inner, side="right") - 1
    assert np.array_equal(O.e4m3_ulp(inner), v[lo + 1] - v[lo])
    # a doubled or halved spacing would move these hand values
    assert O.e4m3_ulp(1.0) == 0.125 and O.e4m3_ulp(448.0) == 32.0 and O.e4m3_ulp(2.0 ** -9) == 2.0 ** -9


# ------------------------------------------------------------------ LayerNorm / RoPE
def test_layer_norm_matches_torch_and_moments():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 128)) * 3 + 1
    gm, bt = rng.standard_normal(128), rng.standard_normal(128)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), torch.from_numpy(gm),
                                         torch.from_numpy(bt), eps=1e-6).numpy()
    assert np.allclose(O.layer_norm(x, gm, bt, 1e-6), ref, rtol=1e-12, atol=1e-12)
    y = O.layer_norm(x)
    assert np.allclose(y.mean(-1), 0, atol=1e-12) and np.allclose(y.var(-1), 1, atol=1e-5)


def test_rope_equals_complex_rotation_and_keeps_pair_norms():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((10, 128))
    pos = rng.integers(0, 2 ** 20, 10)
    y = O.rope_interleaved(x, pos, 10000.0, 64)
    z = x[:, 0:64:2] + 1j * x[:, 1:64:2]
    theta = 10000.0 ** (-np.arange(32) * 2 / 64)
    zr = z * np.exp(1j * pos[:, None] * theta[None, :])
    assert np.allclose(y[:, 0:64:2], zr.real, atol=1e-9) and np.allclose(y[:, 1:64:2], zr.imag, atol=1e-9)
    assert np.array_equal(y[:, 64:], x[:, 64:])                     # dims 64..127 untouched
    assert np.allclose(np.abs(z), np.hypot(y[:, 0:64:2], y[:, 1:64:2]))
    assert np.allclose(O.rope_interleaved(x, np.zeros(10), 10000.0), x)   # position 0 = identity
    a, b = 1234, 98765                                              # R(a) R(b) = R(a + b)
    ab = O.rope_interleaved(O.rope_interleaved(x, np.full(10, a)), np.full(10, b))
    assert np.allclose(ab, O.rope_interleaved(x, np.full(10, a + b)), atol=1e-9)


# ------------------------------------------------------------------ layouts
def test_layout_constants_match_the_pages():
    assert O.INDEX_TOKEN_BYTES == g("index_k_token_bytes")
    assert O.INDEX_PAGE_BYTES == g("index_k_page_bytes")
    assert O.PAGE_TOKENS == g("page_size")
    assert O.INDEX_HEAD_DIM == g("index_head_dim")
    assert O.LATENT_TOKEN_BYTES == g("latent_token_bytes")
    assert O.LATENT_DIM + O.ROPE_DIM == g("latent_dims")
    assert O.LATENT_PAGE_BYTES == 64 * 656 == 41984
    assert O.TOPK == g("index_topk") and O.INDEX_HEADS == g("indexer_heads")
    assert O.MLA_HEADS == g("mla_heads")
    assert O.SOFTMAX_SCALE == 1.0 / math.sqrt(g("softmax_denominator_sqrt")) == 1.0 / 16
    assert O.TOPK * 4 == g("topk_row_bytes")


def test_byte_accounting_printed_on_the_pages():
    assert O.INDEX_TOKEN_BYTES * 10 ** 5 == g("read_bytes_per_layer_L1e5")
    assert abs(21 * O.INDEX_TOKEN_BYTES * 10 ** 5 - g("read_bytes_21_layers_L1e5")) < 0.01 * 277e6
    assert O.INDEX_TOKEN_BYTES * 10 ** 6 == g("read_bytes_per_layer_L1e6")
    flops = 2 * O.MLA_HEADS * O.LATENT_DIM * O.TOPK
    assert abs(flops - g("sparse_mla_flops_per_layer")) < 0.01 * flops


def test_index_cache_roundtrip_and_page_layout():
    rng = np.random.default_rng(6)
    cache = np.zeros((5, O.INDEX_PAGE_BYTES), dtype=np.uint8)
    pt = np.array([3, 0, 4], dtype=np.int32)
    n = 150
    codes = rng.integers(0, 256, (n, 128)).astype(np.uint8)
    scales = np.exp2(rng.integers(-10, 3, n)).astype(np.float64)
    slots = pt[np.arange(n) // 64] * 64 + np.arange(n) % 64
    slots[7] = -1                                                 # skipped
    O.index_cache_write(cache, slots, codes, scales)
    c2, s2 = O.index_cache_read(cache, pt, n)
    keep = np.arange(n) != 7
    assert np.array_equal(c2[keep], codes[keep]) and np.array_equal(s2[keep], scales[keep])
    # token 65 is logical page 1 -> physical page 0, row 1
    assert np.array_equal(cache[0, 128:256], codes[65])
    assert np.frombuffer(cache[0, 8192 + 4:8192 + 8].tobytes(), "<f4")[0] == scales[65]
    assert not cache[3, 7 * 128:8 * 128].any()                    # the skipped slot


def test_latent_cache_roundtrip_dequantises_exactly():
    rng = np.random.default_rng(7)
    n = 70
    c = rng.standard_normal((n, 512))
    rope = torch.randn(n, 64, dtype=torch.float32).to(torch.bfloat16)
    codes, scales = O.latent_quantize(c)
    cache = np.zeros((2, O.LATENT_PAGE_BYTES), dtype=np.uint8)
    pt = np.array([1, 0], dtype=np.int32)
    slots = pt[np.arange(n) // 64] * 64 + np.arange(n) % 64
    O.latent_cache_write(cache, slots, codes, scales, rope.view(torch.int16).numpy().view(np.uint16))
    rows = O.latent_cache_read_rows(cache, pt, np.arange(n))
    assert np.array_equal(rows[:, :512], O.e4m3_decode(codes) * np.repeat(scales, 128, axis=1))
    assert np.array_equal(rows[:, 512:], rope.to(torch.float64).numpy())
    assert np.max(np.abs(rows[:, :512] - c) / np.repeat(scales, 128, axis=1)) <= 16.0  # half an ulp at 448


# ------------------------------------------------------------------ schedule
def test_schedule_matches_the_printed_full_layers():
    full = g("full_layers")
    types = ["full" if l in full else "shared" for l in range(g("num_layers"))]
    is_full = O.parse_indexer_types(types)
    assert sum(is_full) == g("n_full") and len(is_full) - sum(is_full) == g("n_shared")
    assert types[:7] == g("indexer_types_prefix")
    freq, off = g("index_topk_freq"), g("index_skip_topk_offset")
    assert [not O.layer_skips_topk(l, freq, off) for l in range(78)] == is_full
    with pytest.raises(ValueError):
        O.parse_indexer_types(["full", "dense"])


# ------------------------------------------------------------------ indexer scores
def _brute_scores(qd, w, kd):
    L = kd.shape[0]
    out = np.zeros(L)
    for j in range(L):
        tot = 0.0
        for m in range(qd.shape[0]):
            dot = 0.0
            for d in range(qd.shape[1]):
                dot += qd[m, d] * kd[j, d]
            tot += w[m] * (dot if dot > 0 else 0.0)
        out[j] = tot
    return out


def test_indexer_scores_brute_force():
    rng = np.random.default_rng(8)
    L = 9
    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((L, 128))
    w = rng.standard_normal(32) / math.sqrt(32)
    qc, qs = O.index_q_quantize(q)
    kc, ks = O.quantize_blocks_128(k)
    s = O.indexer_scores(qc, qs, w, kc, ks)
    ref = _brute_scores(O.e4m3_decode(qc) * qs[:, None], w, O.e4m3_decode(kc) * ks[:, None])
    assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)
    # a positive rescale of the head weights rescales every score exactly
    assert np.array_equal(O.indexer_scores(qc, qs, 4.0 * w, kc, ks), 4.0 * s)
    D = O.score_magnitude(qc, qs, w, kc, ks)
    assert np.all(D >= np.abs(s) - 1e-12)


def test_score_magnitude_equals_the_score_without_cancellation_and_brute_force_with_it():
    # D_j scales the 1e-3 score bar, so an over-estimate would loosen every
    # score check.  Without cancellation (every w_m > 0 and every dot >= 0)
    # D_j is |s_j| exactly; with cancellation it is the plain sum of
    # |w_m| |<q_m, k_j>| written out term by term.
    rng = np.random.default_rng(32)
    L = 11
    q = np.abs(rng.standard_normal((32, 128)))
    k = np.abs(rng.standard_normal((L, 128)))
    w = np.abs(rng.standard_normal(32)) + 0.01
    qc, qs = O.index_q_quantize(q)
    kc, ks = O.quantize_blocks_128(k)
    s = O.indexer_scores(qc, qs, w, kc, ks)
    assert np.all(s > 0)
    assert np.array_equal(O.score_magnitude(qc, qs, w, kc, ks), s)

    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((L, 128))
    w = rng.standard_normal(32) / math.sqrt(32)
    qc, qs = O.index_q_quantize(q)
    kc, ks = O.quantize_blocks_128(k)
    dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    qd = dec(qc) * qs[:, None]
    kd = dec(kc) * ks[:, None]
    ref = np.zeros(L)
    for j in range(L):
        for m in range(32):
            dot = 0.0
            for d in range(128):
                dot += qd[m, d] * kd[j, d]
            ref[j] += abs(w[m]) * abs(dot)
    D = O.score_magnitude(qc, qs, w, kc, ks)
    assert np.allclose(D, ref, rtol=1e-12, atol=0.0)
    s = O.indexer_scores(qc, qs, w, kc, ks)
    assert np.any(D > np.abs(s) * 1.5)                  # this case does cancel


# ------------------------------------------------------------------ top-k
def _brute_topk(s, k):
    """Repeated extraction of the best remaining (score desc, position asc)."""
    s = list(s)
    taken = set()
    for _ in range(k):
        best = None
        for j, v in enumerate(s):
            if j in taken:
                continue
            if best is None or v > s[best]:
                best = j
        taken.add(best)
    return sorted(taken)


@pytest.mark.parametrize("L", [2049, 2100, 2600])
def test_topk_brute_force_with_heavy_ties(L):
    rng = np.random.default_rng(L)
    s = rng.integers(-3, 4, L).astype(np.float64)         # only 7 distinct values
    s[rng.integers(0, L, 50)] = -0.0
    got = O.topk_positions(s, L)
    assert got.dtype == np.int32 and np.all(got >= 0)
    assert got.tolist() == _brute_topk([v + 0.0 for v in s], 2048)


def test_topk_brute_force_small_k_distinct_and_signed_zero():
    s = np.array([0.0, -0.0, 1.0, -0.0, 0.0, 2.0, -1.0])
    assert O.topk_positions(s, 7, k=4).tolist() == [0, 1, 2, 5]      # -0 ties +0: lower positions win
    assert O.topk_positions(s, 7, k=3).tolist() == [0, 2, 5]


@pytest.mark.parametrize("L", [0, 1, 63, 64, 2047, 2048])
def test_short_context_selects_everything(L):
    out = O.topk_positions(None, L)
    assert out.tolist() == list(range(L)) + [-1] * (2048 - L)


def test_request_topk_short_context_rule_and_causality():
    rng = np.random.default_rng(9)
    L, q_len = 2051, 6                      # query tokens at positions 2045..2050
    cache = np.zeros((33, O.INDEX_PAGE_BYTES), np.uint8)
    pt = rng.permutation(33).astype(np.int32)
    kc, ks = O.index_k_prepare(rng.standard_normal((L, 128)), np.arange(L))
    O.index_cache_write(cache, pt[np.arange(L) // 64] * 64 + np.arange(L) % 64, kc, ks)
    qi = rng.standard_normal((q_len, 32, 128))
    w = rng.standard_normal((q_len, 32))
    topk, scores = O.request_topk(qi, w, cache, pt, L, q_len)
    for t in range(q_len):
        n = L - q_len + t + 1
        if n <= 2048:
            assert topk[t].tolist() == list(range(n)) + [-1] * (2048 - n)
            assert scores[t] is None
        else:
            assert topk[t].max() <= n - 1 and len(set(topk[t].tolist())) == 2048
            assert len(scores[t]) == n


def test_request_topk_invariant_under_page_permutation_and_linear_in_the_key_scale():
    rng = np.random.default_rng(12)
    L, q_len = 4200, 2
    kc, ks = O.index_k_prepare(rng.standard_normal((L, 128)), np.arange(L))
    qi = rng.standard_normal((q_len, 32, 128))
    w = rng.standard_normal((q_len, 32)) / math.sqrt(32)
    pages = (L + 63) // 64
    outs = []
    for seed, pool in ((1, pages), (2, pages + 9)):     # two physical layouts of the same request
        pt = np.random.default_rng(seed).permutation(pool)[:pages].astype(np.int32)
        cache = np.zeros((pool, O.INDEX_PAGE_BYTES), np.uint8)
        O.index_cache_write(cache, pt[np.arange(L) // 64] * 64 + np.arange(L) % 64, kc, ks)
        outs.append(O.request_topk(qi, w, cache, pt, L, q_len))
    assert np.array_equal(outs[0][0], outs[1][0])
    for a, b in zip(outs[0][1], outs[1][1]):
        assert np.array_equal(a, b)
    # a power-of-two boost of some keys' scales (the x4 tokens of the 32K workload)
    # multiplies exactly their scores by 4 and leaves every other score unchanged
    qc, qs = O.index_q_quantize(qi[1])
    boost = np.zeros(L, bool)
    boost[::97] = True
    s0 = O.indexer_scores(qc, qs, w[1], kc, ks)
    s1 = O.indexer_scores(qc, qs, w[1], kc, np.where(boost, 4.0 * ks, ks))
    assert np.array_equal(s1[boost], 4.0 * s0[boost]) and np.array_equal(s1[~boost], s0[~boost])
    top0 = set(O.topk_positions(s0, L).tolist())
    top1 = set(O.topk_positions(s1, L).tolist())
    # a boosted key already selected with a positive score stays selected
    assert all(j in top1 for j in np.flatnonzero(boost) if j in top0 and s0[j] > 0)


# ------------------------------------------------------------------ sparse MLA
def test_sparse_mla_equals_dense_sdpa_when_context_fits():
    rng = np.random.default_rng(10)
    L = 300
    q = rng.standard_normal((64, 576))
    kv = rng.standard_normal((L, 576))
    idx = np.full(2048, -1)
    idx[:L] = rng.permutation(L)              # any order of the full set
    p = L - 1
    out, lse = O.sparse_mla(q, idx, kv[np.maximum(idx, 0)], p)
    Q = torch.from_numpy(q)[None, :, None, :].transpose(1, 2)         # [1,1,64,576]
    K = torch.from_numpy(kv)[None, None]                              # [1,1,L,576]
    V = torch.from_numpy(kv[:, :512])[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=1.0 / 16)[0, 0].numpy()
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)
    ref_lse = torch.logsumexp(torch.from_numpy(q @ kv.T / 16.0), dim=1).numpy()
    assert np.allclose(lse, ref_lse, rtol=1e-12)


def test_sparse_mla_special_cases():
    rng = np.random.default_rng(11)
    kv = rng.standard_normal((5, 576))
    q = rng.standard_normal((64, 576))
    idx = np.array([3] + [-1] * 2047)
    out, _ = O.sparse_mla(q, idx, kv[np.maximum(idx, 0)], 10)
    assert np.allclose(out, np.broadcast_to(kv[3, :512], (64, 512)))       # one key: o = v
    idx = np.array([0, 1, 2, 3, 4] + [-1] * 2043)
    out, lse = O.sparse_mla(np.zeros((64, 576)), idx, kv[np.maximum(idx, 0)], 10)
    assert np.allclose(out, np.broadcast_to(kv[:, :512].mean(0), (64, 512)))  # q = 0: mean of V
    assert np.allclose(lse, np.log(5.0))
    out, _ = O.sparse_mla(q, idx, kv[np.maximum(idx, 0)], 2)               # causal: j <= 2 only
    ref, _ = O.sparse_mla(q, np.array([0, 1, 2]), kv[:3], 2)
    assert np.allclose(out, ref)


# ------------------------------------------------------------------ MTP top-k reuse
def _mtp_request(rng, L0, n_steps):
    """Index cache of one request that grows to L0 + n_steps - 1 tokens, and
    the indexer query of each draft step."""
    L = L0 + n_steps - 1
    pages = (L + 63) // 64
    cache = np.zeros((pages + 2, O.INDEX_PAGE_BYTES), np.uint8)
    pt = rng.permutation(pages + 2)[:pages].astype(np.int32)
    kc, ks = O.index_k_prepare(rng.standard_normal((L, 128)), np.arange(L))
    O.index_cache_write(cache, pt[np.arange(L) // 64] * 64 + np.arange(L) % 64, kc, ks)
    qi = rng.standard_normal((n_steps, 32, 128))
    w = rng.standard_normal((n_steps, 32)) / math.sqrt(32)
    return cache, pt, kc, ks, qi, w


def test_mtp_seed_width_and_draft_reads_printed_on_the_pages():
    assert O.mtp_topk_width() == g("mtp_seed_width") == g("index_topk")
    assert O.mtp_topk_width(2048, 3) == 2050                      # kpool - 1 tail slots
    assert O.mtp_topk_width() * 4 == g("mtp_seed_bytes_per_request")
    # the oracle's read count at a small context: one scored step with reuse,
    # every step without
    rng = np.random.default_rng(21)
    n = g("mtp_draft_steps")
    L0 = 2100
    cache, pt, _, _, qi, w = _mtp_request(rng, L0, n)
    st = O.MtpShareState()
    assert st.begin(True, 1)
    _, read_reuse = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    st.end()
    assert not st.begin(False, 1)
    _, read_plain = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    assert read_reuse == L0 and read_plain == sum(L0 + k for k in range(n))
    # the same counts at a 1M context give the byte figures the pages print
    L = 10 ** 6
    assert abs(O.INDEX_TOKEN_BYTES * L - g("mtp_draft_reads_reuse_L1e6")) <= 0.01 * 132e6
    assert abs(O.INDEX_TOKEN_BYTES * sum(L + k for k in range(n)) - g("mtp_draft_reads_no_reuse_L1e6")) <= 0.01 * 660e6


def test_mtp_steps_without_reuse_match_brute_force_per_position():
    rng = np.random.default_rng(22)
    n, L0 = 3, 2050
    cache, pt, kc, ks, qi, w = _mtp_request(rng, L0, n)
    st = O.MtpShareState()
    assert not st.begin(True, eagle_topk=4)                       # several draft candidates: reuse off
    topk, read = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    assert read == sum(L0 + k for k in range(n))
    kd = O.e4m3_decode(kc) * ks[:, None]
    for k in range(n):
        L = L0 + k                                                # step k queries position L0 - 1 + k
        qc, qs = O.index_q_quantize(qi[k])
        qd = O.e4m3_decode(qc) * qs[:, None]
        s = np.maximum(kd[:L] @ qd.T, 0.0) @ w[k]
        best = np.lexsort((np.arange(L), -s))[:2048]              # score desc, then position asc
        assert topk[k].tolist() == sorted(best.tolist())


def test_mtp_reuse_carries_the_first_step_and_keep_carry_seed():
    rng = np.random.default_rng(23)
    n, L0 = 4, 2060
    cache, pt, kc, ks, qi, w = _mtp_request(rng, L0, n)
    st = O.MtpShareState()
    st.begin(False, 1)
    plain, _ = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    st.end()
    assert st.begin(True, 1) and st.needs_scoring()
    reuse, read = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    assert not st.needs_scoring()
    assert read == L0 and all(np.array_equal(reuse[k], plain[0]) for k in range(n))
    assert any(not np.array_equal(plain[k], plain[0]) for k in range(1, n))   # reuse is an approximation
    st.end()
    assert st.needs_scoring() and st.indices is None
    # a carried seed is used from the first draft step on, and nothing is read
    seed = O.mtp_seed_write(plain, np.array([2]), O.mtp_topk_width())
    assert st.begin(True, 1, keep_carry_seed=True, seed=seed[0])
    got, read = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    assert read == 0 and all(np.array_equal(got[k], plain[2]) for k in range(n))
    st.end()
    # without keep_carry_seed the seed is dropped and the first step scores
    assert st.begin(True, 1, keep_carry_seed=False, seed=seed[0]) and st.needs_scoring()
    st.end()


def test_mtp_short_context_step_publishes_every_position():
    rng = np.random.default_rng(24)
    n, L0 = 3, 2047                                               # steps at contexts 2047, 2048, 2049
    cache, pt, _, _, qi, w = _mtp_request(rng, L0, n)
    st = O.MtpShareState()
    st.begin(True, 1)
    got, read = O.mtp_draft_topk(qi, w, cache, pt, L0, n, st)
    assert read == 0
    assert all(got[k].tolist() == list(range(L0)) + [-1] for k in range(n))


def test_mtp_seed_write_copies_rows_and_pads_the_tail():
    topk = np.arange(3 * 2048, dtype=np.int32).reshape(3, 2048)
    seed = O.mtp_seed_write(topk, np.array([2, 0, 5, -1]), 2050)
    assert seed.shape == (4, 2050)
    assert np.array_equal(seed[0, :2048], topk[2]) and np.array_equal(seed[1, :2048], topk[0])
    assert (seed[:, 2048:] == -1).all() and (seed[2] == -1).all() and (seed[3] == -1).all()
    with pytest.raises(ValueError):
        O.mtp_seed_write(topk, np.array([0]), 2047)


# ------------------------------------------------------------------ MXFP4 index-K cache
def test_mxfp4_layout_constants_printed_on_the_pages():
    assert O.MXFP4_TOKEN_BYTES == g("mxfp4_token_bytes") == 128 // 2 + 128 // g("mxfp4_block")
    assert O.MXFP4_PAGE_BYTES == 64 * 68
    assert O.MXFP4_TOKEN_BYTES / O.INDEX_TOKEN_BYTES < 0.52          # "the read volume halves"


def test_e2m1_table_is_the_format_value_set():
    t = O.e2m1_decode_table()
    # sign-magnitude with magnitudes 2**(e-1) * (1 + m/2) for e > 0 and m/2 for e = 0
    assert t[:8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(t[8:], -t[:8]) and np.signbit(t[8])
    for c in range(16):                                           # every code round-trips
        assert O.e2m1_encode(np.array([t[c]]))[0] == c


def test_e2m1_encode_nearest_ties_to_even_and_saturates():
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.uniform(-8, 8, 4000), np.arange(-7.0, 7.01, 0.25)])
    codes = O.e2m1_encode(x)
    v = O.e2m1_decode(codes)
    vals = O.e2m1_decode_table()[:8]
    for xi, vi, ci in zip(x, v, codes):                            # brute-force nearest
        ax = min(abs(xi), 6.0)
        d = np.abs(vals - ax)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert (ci & 7) == want and (xi < 0) == bool(ci & 8)
    # the ties, by hand
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0, 100.0: 6.0}
    for a, b in ties.items():
        assert O.e2m1_decode(O.e2m1_encode(np.array([a])))[0] == b


@pytest.mark.parametrize("amax,e", [(6.0, 0), (7.99, 0), (8.0, 1), (4.0, 0), (3.99, -1), (1.0, -2), (0.0, 0),
                                    (2.0 ** -140, -127), (2.0 ** 140, 127)])
def test_mx_shared_exponent_hand_values(amax, e):
    assert O.mxfp4_exponent(amax) == e


def test_mxfp4_block_scale_property_and_error_bound():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((300, 128)) * np.exp2(rng.integers(-12, 12, (300, 1)))
    codes, exps = O.quantize_mxfp4(x)
    assert exps.shape == (300, 4)
    xb = x.reshape(300, 4, 32)
    amax = np.abs(xb).max(axis=-1)
    r = amax / np.exp2(exps)
    assert np.all((r >= 4.0) & (r < 8.0))                          # OCP: floor(log2 amax) - emax
    deq = O.mxfp4_dequant(codes, exps).reshape(300, 4, 32)
    step = np.exp2(exps)[..., None]
    sat = np.abs(xb) > 6.0 * step
    err = np.abs(deq - xb)
    assert np.all(err[~sat] <= 1.0 * np.broadcast_to(step, xb.shape)[~sat] + 1e-300)   # half the widest gap (4 -> 6)
    assert np.all(err[sat] <= 2.0 * np.broadcast_to(step, xb.shape)[sat])              # saturation: |x| < 8 * 2**e


def test_mxfp4_cache_roundtrip_and_nibble_order():
    rng = np.random.default_rng(33)
    cache = np.zeros((4, O.MXFP4_PAGE_BYTES), dtype=np.uint8)
    pt = np.array([2, 0, 3], dtype=np.int32)
    n = 140
    codes = rng.integers(0, 16, (n, 128)).astype(np.uint8)
    exps = rng.integers(-20, 20, (n, 4))
    slots = pt[np.arange(n) // 64] * 64 + np.arange(n) % 64
    O.mxfp4_cache_write(cache, slots, codes, exps)
    c2, e2 = O.mxfp4_cache_read(cache, pt, n)
    assert np.array_equal(c2, codes) and np.array_equal(e2, exps)
    # token 65: logical page 1 -> physical page 0, row 1; element 0 in the low nibble
    assert cache[0, 64] == (codes[65, 0] | (codes[65, 1] << 4))
    assert cache[0, 4096 + 4 + 2] == exps[65, 2] + 127


def test_mxfp4_scores_brute_force():
    rng = np.random.default_rng(34)
    L = 7
    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((L, 128))
    w = rng.standard_normal(32) / math.sqrt(32)
    qc, qs = O.index_q_quantize(q)
    kc, ke = O.quantize_mxfp4(k)
    s = O.indexer_scores_mxfp4(qc, qs, w, kc, ke)
    kd = O.mxfp4_dequant(kc, ke)
    ref = _brute_scores(O.e4m3_decode(qc) * qs[:, None], w, kd)
    assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)
    assert np.all(O.score_magnitude_mxfp4(qc, qs, w, kc, ke) >= np.abs(s) - 1e-12)


def _e2m1_value(code):
    # OCP MX E2M1: bit 3 sign, then magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
    mag = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}[int(code) & 7]
    return -mag if int(code) & 8 else mag


def _mx_values(codes, exps):
    v = np.vectorize(_e2m1_value)(codes).reshape(codes.shape[:-1] + (4, 32))
    return (v * np.exp2(exps)[..., None]).reshape(codes.shape)


def test_index_k_prepare_mxfp4_within_the_format_bound_of_norm_then_rotation():
    # independent of the oracle's own LayerNorm and RoPE: torch's LayerNorm and
    # a complex rotation of the interleaved pairs, then the MX rounding bound
    rng = np.random.default_rng(35)
    n = 64
    k = rng.standard_normal((n, 128)) * np.exp2(rng.integers(-8, 8, (n, 1))) + rng.standard_normal((n, 1))
    pos = rng.integers(0, 1 << 20, n)
    pos[0] = 0
    k[5] = 3.25                                           # a constant row: LayerNorm gives 0
    codes, exps = O.index_k_prepare_mxfp4(k, pos)
    y = torch.nn.functional.layer_norm(torch.from_numpy(k), (128,), eps=1e-6)
    i = torch.arange(32, dtype=torch.float64)
    ang = torch.from_numpy(pos.astype(np.float64))[:, None] * 10000.0 ** (-2.0 * i / 64)
    z = torch.complex(y[:, 0:64:2], y[:, 1:64:2]) * torch.polar(torch.ones_like(ang), ang)
    ref = y.clone()
    ref[:, 0:64:2], ref[:, 1:64:2] = z.real, z.imag
    ref = ref.numpy()
    got = _mx_values(codes, exps)
    step = np.repeat(np.exp2(exps), 32, axis=1)
    sat = np.abs(ref) > 6.0 * step
    err = np.abs(got - ref)
    assert np.all(err[~sat] <= step[~sat] * (1 + 1e-9))   # at most half of the widest code gap (4 -> 6)
    assert np.all(err[sat] <= 2.0 * step[sat] * (1 + 1e-9))
    blk = np.abs(ref).reshape(n, 4, 32).max(axis=-1)
    live = blk > 1e-9
    r = blk[live] / np.exp2(exps[live])
    assert np.all((r >= 4.0 * (1 - 1e-9)) & (r < 8.0 * (1 + 1e-9)))   # shared exponent floor(log2 amax) - 2
    assert not np.any(got[5]) and np.all(exps[5] == 0)    # constant row
    assert np.allclose(got[0], _mx_values(*O.quantize_mxfp4(y.numpy()[:1]))[0])   # position 0: no rotation


def test_request_topk_mxfp4_brute_force_and_short_context_rule():
    rng = np.random.default_rng(36)
    L, q_len = 2053, 6                                    # query tokens at positions 2047..2052
    npg = 33
    cache = np.zeros((npg, O.MXFP4_PAGE_BYTES), np.uint8)
    pt = rng.permutation(npg).astype(np.int32)
    codes, exps = O.index_k_prepare_mxfp4(rng.standard_normal((L, 128)), np.arange(L))
    O.mxfp4_cache_write(cache, pt[np.arange(L) // 64] * 64 + np.arange(L) % 64, codes, exps)
    qi = rng.standard_normal((q_len, 32, 128))
    w = rng.standard_normal((q_len, 32))
    topk, scores = O.request_topk_mxfp4(qi, w, cache, pt, L, q_len)
    kd = _mx_values(codes, exps)                          # from the codes as written, not read back
    for t in range(q_len):
        n = L - q_len + t + 1
        if n <= 2048:
            assert topk[t].tolist() == list(range(n)) + [-1] * (2048 - n)
            assert scores[t] is None
            continue
        qc, qs = O.index_q_quantize(qi[t])
        qd = O.e4m3_decode(qc) * qs[:, None]
        # scores by a matrix route (not the pins' loop helper): sum_m w_m relu(q_m . k_j)
        ref = np.maximum(kd[:n] @ qd.T, 0.0) @ w[t]
        assert np.allclose(scores[t], ref, rtol=1e-10, atol=1e-10)
        order = sorted(range(n), key=lambda j: (-ref[j], j))   # key desc, ties to the lower position
        kth = ref[order[2047]]
        want, got = set(order[:2048]), set(topk[t].tolist())
        assert len(got) == 2048 and max(got) <= n - 1
        assert all(abs(ref[j] - kth) <= 1e-9 * max(1.0, abs(kth)) for j in want ^ got)


# ------------------------------------------------------------------ schedule fallbacks
def test_schedule_fallback_chain_follows_the_pages():
    n = g("num_layers")
    full = set(g("full_layers"))
    types = ["full" if l in full else "shared" for l in range(n)]
    # the explicit list wins over every other field
    assert [not O.layer_skips_topk_config(l, indexer_types=types, cli_factor=3, index_topk_freq=2)
            for l in range(n)] == [l in full for l in range(n)]
    # GLM-5.3's parameterised fields give the same 21 / 57 split as its list
    fr = [not O.layer_skips_topk_config(l, index_topk_freq=g("index_topk_freq"),
                                        index_skip_topk_offset=g("index_skip_topk_offset")) for l in range(n)]
    assert fr == [l in full for l in range(n)] and sum(fr) == g("n_full")
    # the default offset: layers 0 and 1 full, layer 2 shared, then one full layer in every 4
    d = [not O.layer_skips_topk_config(l, index_topk_freq=4) for l in range(12)]
    assert d == [True, True, False, False, False, True, False, False, False, True, False, False]
    # cli_factor: a fresh top-k every cli_factor layers, ahead of the pattern and the freq rule
    assert [not O.layer_skips_topk_config(l, cli_factor=3, index_topk_pattern="SSSS", index_topk_freq=5)
            for l in range(7)] == [True, False, False, True, False, False, True]
    # pattern: 'S' is shared, anything else and anything past its end is full
    assert [O.layer_skips_topk_config(l, index_topk_pattern="FSSFS") for l in range(7)] == \
        [False, True, True, False, True, False, False]
    # a list shorter than the model: layers past its end are full
    assert not O.layer_skips_topk_config(5, indexer_types=["full", "shared"])


# ------------------------------------------------------------------ fused latent store
def test_rms_norm_against_torch_and_its_defining_property():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((50, 512)) * np.exp2(rng.integers(-5, 5, (50, 1)))
    gam = rng.uniform(0.5, 1.5, 512)
    y = O.rms_norm(x, None, 1e-6)
    assert np.allclose((y * y).mean(axis=-1), 1.0 / (1.0 + 1e-6 / (x * x).mean(axis=-1)), rtol=1e-12)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (512,), torch.from_numpy(gam), eps=1e-6).numpy()
    assert np.allclose(O.rms_norm(x, gam, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_latent_prepare_rotates_only_the_rope_dims_and_rounds_to_bf16():
    rng = np.random.default_rng(42)
    n = 40
    kv = rng.standard_normal((n, 512))
    pe = rng.standard_normal((n, 64))
    pos = rng.integers(0, 1 << 20, n)
    codes, scales, rbits = O.latent_prepare(kv, pe, pos)
    # the latent part is the plain quantisation of the RMS-normalised kv_c
    c2, s2 = O.latent_quantize(O.rms_norm(kv))
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)
    # the RoPE part keeps each pair's norm up to bf16 rounding, and position 0 is the identity
    r = O.bf16_bits_to_f64(rbits)
    assert np.allclose(np.hypot(r[:, 0::2], r[:, 1::2]), np.hypot(pe[:, 0::2], pe[:, 1::2]), rtol=2 ** -7)
    _, _, r0 = O.latent_prepare(kv[:1], pe[:1], np.array([0]))
    assert np.array_equal(O.bf16_bits_to_f64(r0), O.bf16_bits_to_f64(O.f64_to_bf16_bits(pe[:1])))
    # nearest bf16: within half a bf16 ulp of the exact rotation
    exact = O.rope_interleaved(pe, pos, 10000.0, 64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(r - exact) <= 0.5 * ulp * (1 + 1e-9))


# ------------------------------------------------------------------ context-parallel merges
@pytest.mark.parametrize("cuts", [(1000,), (700, 1900), (5, 2100, 2200)])
def test_cp_merge_topk_of_slice_topks_is_the_whole_topk(cuts):
    # Scores with heavy ties and signed zeros over L positions, cut into
    # disjoint slices; each slice keeps its own top-k by brute force; the merge
    # of those lists must be the brute-force top-k of the whole row.
    rng = np.random.default_rng(41 + len(cuts))
    L, k = 2400, 64
    s = rng.integers(-40, 40, L).astype(np.float64) / 8.0
    s[rng.integers(0, L, 50)] = -0.0
    edges = [0, *cuts, L]
    cand_pos, cand_sc = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        loc = _brute_topk(s[a:b], min(k, b - a))
        cand_pos.append(np.array(loc) + a)
        cand_sc.append(s[a:b][loc])
    got = O.cp_merge_topk(cand_pos, cand_sc, k=k)
    assert got.tolist() == _brute_topk(s, k)
    # at the full width, against an independent argsort of (score desc, position asc)
    L2 = 9000
    s2 = np.round(rng.standard_normal(L2) * 4) / 4
    order = sorted(range(L2), key=lambda j: (-(s2[j] + 0.0), j))[:2048]
    pos, sc = [], []
    for a, b in ((0, 3000), (3000, 3001), (3001, L2)):
        loc = sorted(range(a, b), key=lambda j: (-(s2[j] + 0.0), j))[:2048]
        pos.append(np.array(loc + [-1] * (2048 - len(loc))))
        sc.append(np.array([s2[j] for j in loc] + [0.0] * (2048 - len(loc))))
    assert O.cp_merge_topk(pos, sc).tolist() == sorted(order)


def test_lse_merge_of_attention_parts_equals_dense_attention():
    # Attention over a key set split into parts, each normalised on its own with
    # its log-sum-exp, merges to dense softmax attention over all keys (torch SDPA
    # in fp64), including an empty part.
    rng = np.random.default_rng(43)
    H, D, n = 4, 16, 37
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((n, D)) * 2.0
    v = rng.standard_normal((n, D))
    parts = [np.arange(0, 11), np.arange(11, 11), np.arange(11, 30), np.arange(30, n)]
    outs, lses = [], []
    for idx in parts:
        if idx.size == 0:
            outs.append(np.zeros((H, D)))
            lses.append(np.full(H, -np.inf))
            continue
        sc = q @ k[idx].T
        m = sc.max(axis=1, keepdims=True)
        p = np.exp(sc - m)
        outs.append(p @ v[idx] / p.sum(axis=1, keepdims=True))
        lses.append(m[:, 0] + np.log(p.sum(axis=1)))
    out, lse = O.lse_merge(outs, lses)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(k)[None, None].expand(1, H, n, D),
        torch.from_numpy(v)[None, None].expand(1, H, n, D), scale=1.0)[0, :, 0, :].numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    ref_lse = np.log(np.exp(q @ k.T).sum(axis=1))
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    out0, lse0 = O.lse_merge([np.zeros((H, D))] * 2, [np.full(H, -np.inf)] * 2)
    assert not out0.any() and np.all(np.isneginf(lse0))
