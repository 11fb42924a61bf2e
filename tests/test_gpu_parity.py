"""GPU parity on small seeded cases: every CUDA call against the fp64 oracle.

Sizes span several tiles / pages and ragged tails; edge cases include empty
and short contexts (<= 2048 selects everything), exact multiples of the page
and of the top-k, -1 padding, causal limits of multi-token rows, ties and
signed zeros in the top-k, skipped and out-of-range cache slots.
"""

import math

import numpy as np
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
from oracle import dsa_oracle as O
from synth import Workload, page_table, batch_meta
from tests.oracle_side import (bf16_bits, check_attention, check_scores, check_topk_row, f64,
                               oracle_index_cache, oracle_latent_cache, round_bf16)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gen(seed):
    return torch.Generator().manual_seed(seed)


# ------------------------------------------------------------------ stores
def _decode_index_cache(cache_u8: np.ndarray, slots: np.ndarray):
    page, row = np.divmod(slots, 64)
    codes = cache_u8[page[:, None], row[:, None] * 128 + np.arange(128)]
    sc = np.ascontiguousarray(cache_u8[page[:, None], 8192 + 4 * row[:, None] + np.arange(4)]).view("<f4")
    return codes, sc.reshape(-1).astype(np.float64)


@pytest.mark.parametrize("affine", [False, True])
def test_index_k_store_matches_oracle(affine):
    g = _gen(11)
    n, num_pages = 3000, 60
    mag = torch.exp2(torch.randint(-6, 7, (n, 1), generator=g).float())
    k = (torch.randn(n, 128, generator=g) * mag + torch.randn(n, 1, generator=g)).to(torch.bfloat16)
    k[5] = 0.0                                          # constant row: LayerNorm output 0, scale 1
    k[6] = 3.0
    pos = torch.randint(0, 1 << 20, (n,), generator=g, dtype=torch.int32)
    slots = torch.randperm(num_pages * 64, generator=g)[:n].to(torch.int64)
    slots[::50] = -1                                    # padded rows: write skipped
    gamma = (torch.rand(128, generator=g) + 0.5) if affine else None
    beta = (torch.randn(128, generator=g) * 0.1) if affine else None
    cache = torch.zeros(num_pages * 8448, dtype=torch.uint8, device=DEV)
    st = D.new_device_status(DEV)
    D.dsa_index_k_store(k.to(DEV), pos.to(DEV), slots.to(DEV), cache,
                        gamma=None if gamma is None else gamma.to(DEV),
                        beta=None if beta is None else beta.to(DEV), dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    gcache = cache.cpu().numpy().reshape(num_pages, 8448)
    kf = f64(k)
    y = O.rope_interleaved(O.layer_norm(kf, None if gamma is None else f64(gamma),
                                        None if beta is None else f64(beta), 1e-6), pos.numpy(), 10000.0)
    ocodes, oscales = O.quantize_blocks_128(y)
    s = slots.numpy()
    keep = s >= 0
    gcodes, gscales = _decode_index_cache(gcache, s[keep])
    oc, os_ = ocodes[keep], oscales[keep]
    amax = np.max(np.abs(y[keep]), axis=1)
    smis = gscales != os_
    # scale differences only where amax / 448 sits on a power of two
    if smis.any():
        ratio = amax[smis] / 448.0
        assert np.all(np.abs(ratio / np.exp2(np.round(np.log2(ratio))) - 1) < 1e-5)
    assert smis.mean() < 1e-3
    gd = O.e4m3_decode(gcodes) * gscales[:, None]
    od = O.e4m3_decode(oc) * os_[:, None]
    ulp = np.maximum(O.e4m3_ulp(od / os_[:, None]) * os_[:, None], O.e4m3_ulp(gd / gscales[:, None]) * gscales[:, None])
    assert np.all(np.abs(gd - od) <= ulp * (1 + 1e-12))
    assert (np.abs(gd - od) > 0).mean() < 1e-3
    # untouched slots stay zero
    written = np.zeros(num_pages * 64, bool)
    written[s[keep]] = True
    unw = np.nonzero(~written)[0]
    c2, s2 = _decode_index_cache(gcache, unw)
    assert not c2.any() and not s2.any()


def test_latent_store_matches_oracle():
    g = _gen(12)
    n, num_pages = 700, 15
    c = (torch.randn(n, 512, generator=g) * torch.exp2(torch.randint(-4, 5, (n, 4), generator=g).float())
         .repeat_interleave(128, dim=1)).to(torch.bfloat16)
    rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    slots = torch.randperm(num_pages * 64, generator=g)[:n].to(torch.int64)
    slots[3] = -1
    cache = torch.zeros(num_pages * 41984, dtype=torch.uint8, device=DEV)
    D.dsa_latent_kv_store(c.to(DEV), rope.to(DEV), slots.to(DEV), cache)
    gcache = cache.cpu().numpy().reshape(num_pages, 41984)
    s = slots.numpy()
    keep = s >= 0
    ocache = np.zeros_like(gcache)
    codes, scales = O.latent_quantize(f64(c))
    O.latent_cache_write(ocache, s, codes, scales, bf16_bits(rope))
    grows = O.latent_cache_read_rows(gcache, np.arange(num_pages), s[keep])
    orows = O.latent_cache_read_rows(ocache, np.arange(num_pages), s[keep])
    assert np.array_equal(grows[:, 512:], orows[:, 512:])             # RoPE copied bit-exactly
    sc = np.repeat(scales[keep], 128, axis=1)
    assert np.all(np.abs(grows[:, :512] - orows[:, :512]) <= O.e4m3_ulp(orows[:, :512] / sc) * sc)
    written = np.zeros(num_pages * 64, bool)
    written[s[keep]] = True
    for sl in np.nonzero(~written)[0][:50]:                        # untouched rows stay zero
        assert not gcache[sl // 64, (sl % 64) * 656:(sl % 64 + 1) * 656].any()


def test_store_records_out_of_range_slot_without_fault():
    cache = torch.zeros(2 * 8448, dtype=torch.uint8, device=DEV)
    k = torch.randn(3, 128).to(torch.bfloat16).to(DEV)
    pos = torch.zeros(3, dtype=torch.int32, device=DEV)
    slots = torch.tensor([0, 128, 5], dtype=torch.int64, device=DEV)      # 128 >= 2 pages * 64
    st = D.new_device_status(DEV)
    D.dsa_index_k_store(k, pos, slots, cache, dev_status=st)
    out = D.dsa_device_status_read(st)
    assert out[0] & D.DEVERR_SLOT_RANGE and out[1] == 1 and out[2] == 128
    assert cache.view(2, 8448)[0, 5 * 128:6 * 128].any()                 # the good rows were written


# ------------------------------------------------------------------ top-k from scores
def _score_rows(g):
    rows = []
    for n in [1, 63, 64, 65, 2047, 2048, 2049, 2050, 4097, 10000, 70001]:
        rows.append(torch.randn(n, generator=g))
    ties = torch.randint(-3, 4, (9000,), generator=g).float()
    ties[torch.randint(0, 9000, (300,), generator=g)] = -0.0
    rows.append(ties)
    z = torch.zeros(5000)
    z[::2] = -0.0                                      # only signed zeros: lowest positions win
    rows.append(z)
    w = torch.randn(3000, generator=g)
    w[::3] = -math.inf
    rows.append(w)
    rows.append(torch.full((2500,), 7.0))              # all equal
    return rows


def test_topk_from_scores_bit_exact():
    g = _gen(13)
    rows = _score_rows(g)
    ld = max(r.numel() for r in rows) + 3
    S = torch.full((len(rows), ld), float("nan"))
    for i, r in enumerate(rows):
        S[i, :r.numel()] = r
    vl = torch.tensor([r.numel() for r in rows], dtype=torch.int32)
    topk = D.dsa_topk_from_scores(S.to(DEV), vl.to(DEV), max_len=ld).cpu().numpy()
    for i, r in enumerate(rows):
        ref = O.topk_positions(r.double().numpy(), r.numel())
        assert np.array_equal(topk[i], ref), f"row {i} (n={r.numel()})"


def test_topk_from_scores_fallback_paths():
    # a boundary bin larger than the shared-memory buffer (40000 equal keys), a
    # row longer than the position bitmap (sorted instead), and rows that are not
    # 16-byte aligned (ld odd: scalar loads)
    g = _gen(17)
    rows = [torch.full((40000,), 3.0), torch.randn(1_100_000, generator=g), torch.randn(9001, generator=g)]
    eq = torch.randn(30000, generator=g)
    eq[5000:25000] = 0.25                               # 20000 equal keys around the cut
    rows.append(eq)
    ld = max(r.numel() for r in rows) + 1               # odd: rows 1.. start off 16-byte alignment
    S = torch.full((len(rows), ld), float("nan"))
    for i, r in enumerate(rows):
        S[i, :r.numel()] = r
    vl = torch.tensor([r.numel() for r in rows], dtype=torch.int32)
    topk = D.dsa_topk_from_scores(S.to(DEV), vl.to(DEV), max_len=ld).cpu().numpy()
    for i, r in enumerate(rows):
        ref = O.topk_positions(r.double().numpy(), r.numel())
        assert np.array_equal(topk[i], ref), f"row {i} (n={r.numel()})"


# ------------------------------------------------------------------ indexer
def _small_workload(seq_len, q_len, seed):
    return Workload("small", seed, list(seq_len), list(q_len), ["full"])


SMALL_SEQ = [1, 63, 64, 65, 2047, 2048, 2049, 2100, 4097, 6000, 3000, 2051]
SMALL_Q = [1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 6, 6]


def _build_indexer_case(seq, qlen, seed, boost_req=None):
    w = _small_workload(seq, qlen, seed)
    g = _gen(seed)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    raw, pos, slots = [], [], []
    for r, L in enumerate(w.seq_len):
        raw.append(torch.randn(L, 128, generator=g).to(torch.bfloat16))
        p = np.arange(L)
        pos.append(p)
        slots.append(pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64)
    boost = [np.zeros(L, bool) for L in w.seq_len]
    if boost_req is not None:
        boost[boost_req][::97] = True                   # a few boosted keys
    ocache = oracle_index_cache(w.num_pages, [f64(x) for x in raw], pos, slots, boost)
    q = torch.randn(w.total_q, 32, 128, generator=g).to(torch.bfloat16)
    wt = torch.randn(w.total_q, 32, generator=g) / math.sqrt(32)
    # oracle: scores, magnitudes and top-k per row
    rows = []
    qs = meta["q_start"].numpy()
    for r, L in enumerate(w.seq_len):
        kc, ks = O.index_cache_read(ocache, pt[r].numpy(), L)
        for t in range(w.q_len[r]):
            i = qs[r] + t
            n = L - w.q_len[r] + t + 1
            qc, qsc = O.index_q_quantize(f64(q[i]))
            s = O.indexer_scores(qc, qsc, f64(wt[i]), kc[:n], ks[:n])
            m = O.score_magnitude(qc, qsc, f64(wt[i]), kc[:n], ks[:n])
            rows.append(dict(r=r, i=i, n=n, s=s, mag=m, topk=O.topk_positions(s, n)))
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=w.max_q_len, total_q=w.total_q)
    return dict(w=w, cache=torch.from_numpy(ocache.reshape(-1)).to(DEV), q=q.to(DEV), wt=wt.to(DEV),
                batch=batch, rows=rows)


@pytest.fixture(scope="module")
def indexer_case():
    return _build_indexer_case(SMALL_SEQ, SMALL_Q, 777, boost_req=9)


# Decode batches (one query row per request) take the fused tensor-core path.
DECODE_SEQ = [2049, 1, 100, 2048, 4097, 6000, 2100, 33000, 10000, 70000, 128 * 40, 128 * 40 + 1, 8191,
              300000]                                   # past 2^18 positions: ranked by a sort, not a bitmap


@pytest.fixture(scope="module")
def decode_case():
    return _build_indexer_case(DECODE_SEQ, [1] * len(DECODE_SEQ), 991, boost_req=7)


@pytest.fixture(scope="module")
def decode_many_case():
    rng = np.random.default_rng(5)
    seq = rng.integers(1, 9000, 300).tolist()           # more requests than CTAs, many short ones
    return _build_indexer_case(seq, [1] * len(seq), 992)


def _check_indexer_topk(c, max_diff):
    T = c["w"].total_q
    sc = torch.empty(T, 2048, device=DEV)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"], topk_scores=sc, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    topk, sc = topk.cpu().numpy(), sc.cpu().numpy()
    ndiff = 0
    for row in c["rows"]:
        i = row["i"]
        ndiff += check_topk_row(topk[i], row["topk"], row["s"], row["mag"], row["n"], what=f"row {i}")
        if row["n"] > 2048:
            check_scores(sc[i], row["s"][topk[i]], row["mag"][topk[i]], what=f"selected scores row {i}")
        else:
            assert not sc[i].any()
    assert ndiff <= max_diff


def test_indexer_topk_decode_tensor_core_path(decode_case):
    _check_indexer_topk(decode_case, 2)


def test_indexer_topk_decode_many_requests(decode_many_case):
    _check_indexer_topk(decode_many_case, 4)


def test_indexer_topk_decode_more_rows_than_sms_up_to_the_small_merge_bitmap():
    """More decode rows than SMs select with the two-blocks-per-SM merge, whose
    position bitmap holds 2^18 positions: contexts up to exactly that size."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    seq = [250000, 262144, 100000] + [2100] * (sms + 1)
    c = _build_indexer_case(seq, [1] * len(seq), 1212, boost_req=1)
    _check_indexer_topk(c, 4)


@pytest.mark.parametrize("fill", [0x00, 0xAB, 0xFF])
def test_indexer_topk_decode_dirty_workspace(decode_case, fill):
    """The workspace content on entry must not matter (it is caller memory)."""
    c = decode_case
    nbytes = D.dsa_indexer_topk_workspace_size(c["batch"])
    ws = torch.full((nbytes,), fill, dtype=torch.uint8, device=DEV)
    st = D.new_device_status(DEV)
    got = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"], ws=ws, dev_status=st).cpu().numpy()
    assert D.dsa_device_status_read(st)[0] == 0
    for row in c["rows"]:
        check_topk_row(got[row["i"]], row["topk"], row["s"], row["mag"], row["n"], what=f"row {row['i']}")


def test_indexer_topk_decode_repeatable(decode_case):
    c = decode_case
    a = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"])
    b = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"])
    assert torch.equal(a, b)


def test_indexer_scores_match_oracle(indexer_case):
    c = indexer_case
    st = D.new_device_status(DEV)
    S = D.dsa_indexer_scores(c["q"], c["wt"], c["cache"], c["batch"], dev_status=st).cpu().numpy()
    assert D.dsa_device_status_read(st)[0] == 0
    for row in c["rows"]:
        i, n = row["i"], row["n"]
        check_scores(S[i, :n], row["s"], row["mag"], what=f"row {i}")
        assert np.all(np.isneginf(S[i, n:c["w"].seq_len[row["r"]]]))     # causal: j > p masked


def test_indexer_topk_matches_oracle(indexer_case):
    _check_indexer_topk(indexer_case, 2)


def test_indexer_scores_cuda_core_match_oracle_and_the_tensor_core_rows(decode_case):
    """The CUDA-core scorer kept for comparison: same scores within the bar,
    on a decode batch (a 300K-token request included)."""
    c = decode_case
    st = D.new_device_status(DEV)
    S = D.dsa_indexer_scores_cuda_core(c["q"], c["wt"], c["cache"], c["batch"], dev_status=st).cpu().numpy()
    assert D.dsa_device_status_read(st)[0] == 0
    T = D.dsa_indexer_scores(c["q"], c["wt"], c["cache"], c["batch"]).cpu().numpy()
    for row in c["rows"]:
        i, n = row["i"], row["n"]
        check_scores(S[i, :n], row["s"], row["mag"], what=f"row {i}")
        check_scores(S[i, :n], T[i, :n].astype(np.float64), 2 * row["mag"], what=f"row {i} vs tensor cores")


def test_indexer_scores_cuda_core_refuses_multi_token_rows(indexer_case):
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_scores_cuda_core(indexer_case["q"], indexer_case["wt"], indexer_case["cache"],
                                       indexer_case["batch"])
    assert e.value.name == "DSA_ERR_UNSUPPORTED"


def test_indexer_topk_fed_oracle_fp32_scores_is_bit_exact(indexer_case):
    c = indexer_case
    rows = [r for r in c["rows"] if r["n"] > 0]
    ld = max(r["n"] for r in rows)
    S = torch.full((len(rows), ld), -math.inf)
    for k, r in enumerate(rows):
        S[k, :r["n"]] = torch.from_numpy(r["s"].astype(np.float32))
    vl = torch.tensor([r["n"] for r in rows], dtype=torch.int32)
    topk = D.dsa_topk_from_scores(S.to(DEV), vl.to(DEV)).cpu().numpy()
    for k, r in enumerate(rows):
        ref = O.topk_positions(r["s"].astype(np.float32).astype(np.float64), r["n"])
        assert np.array_equal(topk[k], ref)


@pytest.mark.parametrize("case", ["indexer_case", "decode_case"])
def test_indexer_records_bad_page_without_fault(case, request):
    c = request.getfixturevalue(case)
    b = c["batch"]
    pt = b.page_table.clone()
    pt[9, 3] = c["w"].num_pages + 5                        # request 9, logical page 3: out of range
    bad = D.Batch(b.seq_len, b.q_start, pt, c["w"].num_pages, max_seq_len=b.c.max_seq_len,
                  max_q_len=b.c.max_q_len, total_q=b.total_q)
    st = D.new_device_status(DEV)
    D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], bad, dev_status=st)
    out = D.dsa_device_status_read(st)
    assert out[0] & D.DEVERR_PAGE_RANGE and out[2] == c["w"].num_pages + 5


# ------------------------------------------------------------------ sparse MLA
MLA_SEQ = [1, 100, 2048, 3000, 5000, 2500]
MLA_Q = [1, 1, 1, 6, 2, 1]


@pytest.fixture(scope="module")
def mla_case():
    w = _small_workload(MLA_SEQ, MLA_Q, 4242)
    g = _gen(31)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    cs, rs, slots = [], [], []
    for r, L in enumerate(w.seq_len):
        cs.append(f64(torch.randn(L, 512, generator=g).to(torch.bfloat16)))
        rs.append(torch.randn(L, 64, generator=g).to(torch.bfloat16))
        p = np.arange(L)
        slots.append(pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64)
    ocache = oracle_latent_cache(w.num_pages, cs, [bf16_bits(x) for x in rs], slots)
    q = torch.randn(w.total_q, 64, 576, generator=g).to(torch.bfloat16)
    qs = meta["q_start"].numpy()
    topk = np.full((w.total_q, 2048), -1, np.int32)
    for r, L in enumerate(w.seq_len):
        for t in range(w.q_len[r]):
            i = qs[r] + t
            p = L - w.q_len[r] + t
            if p + 1 <= 2048:
                topk[i] = O.topk_positions(None, p + 1)
            else:
                sel = np.sort(np.random.default_rng(i).choice(p + 1, 2048, replace=False))
                topk[i] = sel
    topk[0, 5] = -1                                     # stray -1 inside a short row's list
    topk[3][100:110] = -1                               # holes in a full row
    # row 4 (request 3, t = 0 of 6) gets a few entries beyond its own position (causal mask)
    p4 = MLA_SEQ[3] - 6
    topk[4][-3:] = [p4 + 1, p4 + 2, p4 + 3]
    topk[4] = np.sort(topk[4])
    ref_out, ref_lse = [], []
    for r, L in enumerate(w.seq_len):
        for t in range(w.q_len[r]):
            i = qs[r] + t
            p = L - w.q_len[r] + t
            idx = topk[i]
            rows = O.latent_cache_read_rows(ocache, pt[r].numpy(), np.maximum(idx, 0))
            o, lse = O.sparse_mla(f64(q[i]), idx, rows, p)
            ref_out.append(o)
            ref_lse.append(lse)
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=w.max_q_len, total_q=w.total_q)
    return dict(w=w, cache=torch.from_numpy(ocache.reshape(-1)).to(DEV), q=q.to(DEV),
                topk=torch.from_numpy(topk).to(DEV), batch=batch, out=np.stack(ref_out), lse=np.stack(ref_lse))


def _mla_decode_rows_case(T, seed):
    """T decode requests (one row each) of 2200.. tokens with 2048 random selected
    positions (a few holes), built and evaluated as in mla_case."""
    seq = [2200 + 37 * r for r in range(T)]
    w = _small_workload(seq, [1] * T, seed)
    g = _gen(seed)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    cs, rs, slots = [], [], []
    for r, L in enumerate(w.seq_len):
        cs.append(f64(torch.randn(L, 512, generator=g).to(torch.bfloat16)))
        rs.append(torch.randn(L, 64, generator=g).to(torch.bfloat16))
        pp = np.arange(L)
        slots.append(pt[r, pp // 64].numpy().astype(np.int64) * 64 + pp % 64)
    ocache = oracle_latent_cache(w.num_pages, cs, [bf16_bits(x) for x in rs], slots)
    q = torch.randn(T, 64, 576, generator=g).to(torch.bfloat16)
    topk = np.stack([np.sort(np.random.default_rng(seed * 1000 + i).choice(L, 2048, replace=False))
                     for i, L in enumerate(w.seq_len)]).astype(np.int32)
    topk[::7, 300:305] = -1                              # holes
    ref_out, ref_lse = [], []
    for i, L in enumerate(w.seq_len):
        rows = O.latent_cache_read_rows(ocache, pt[i].numpy(), np.maximum(topk[i], 0))
        o, lse = O.sparse_mla(f64(q[i]), topk[i], rows, L - 1)
        ref_out.append(o)
        ref_lse.append(lse)
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=1, total_q=T)
    return dict(cache=torch.from_numpy(ocache.reshape(-1)).to(DEV), q=q.to(DEV), topk=torch.from_numpy(topk).to(DEV),
                batch=batch, out=np.stack(ref_out), lse=np.stack(ref_lse))


# With 152 SMs: 24 rows run as clusters of 4 CTAs per row, 48 as clusters of 2,
# 100 as one CTA per row (the 12-row case above takes global partials).
@pytest.mark.parametrize("T", [24, 48, 100])
def test_sparse_mla_row_splits_match_oracle(T):
    c = _mla_decode_rows_case(T, 500 + T)
    lse = torch.empty(T, 64, device=DEV)
    st = D.new_device_status(DEV)
    out = D.dsa_sparse_mla_decode(c["q"], c["topk"], c["cache"], c["batch"], out_dtype=D.DTYPE_F32, lse=lse,
                                  dev_status=st)
    outb = D.dsa_sparse_mla_decode(c["q"], c["topk"], c["cache"], c["batch"], out_dtype=D.DTYPE_BF16)
    assert D.dsa_device_status_read(st)[0] == 0
    out, outb = out.cpu().numpy(), outb.float().cpu().numpy()
    for i in range(T):
        check_attention(out[i], c["out"][i], what=f"T={T} row {i}")
        check_attention(outb[i], round_bf16(c["out"][i]), what=f"T={T} bf16 row {i}")
    assert np.allclose(lse.cpu().numpy(), c["lse"], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("entry", ["decode", "prefill"])
def test_sparse_mla_fp32_matches_oracle(mla_case, entry):
    c = mla_case
    fn = D.dsa_sparse_mla_decode if entry == "decode" else D.dsa_sparse_mla_prefill
    lse = torch.empty(c["w"].total_q, 64, device=DEV)
    st = D.new_device_status(DEV)
    out = fn(c["q"], c["topk"], c["cache"], c["batch"], out_dtype=D.DTYPE_F32, lse=lse, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    out = out.cpu().numpy()
    for i in range(c["w"].total_q):
        check_attention(out[i], c["out"][i], what=f"{entry} row {i}")
    assert np.allclose(lse.cpu().numpy(), c["lse"], rtol=1e-5, atol=1e-4)


def test_sparse_mla_bf16_matches_oracle_rounded(mla_case):
    c = mla_case
    out = D.dsa_sparse_mla_decode(c["q"], c["topk"], c["cache"], c["batch"], out_dtype=D.DTYPE_BF16)
    out = out.float().cpu().numpy()
    for i in range(c["w"].total_q):
        check_attention(out[i], round_bf16(c["out"][i]), what=f"bf16 row {i}")


def test_sparse_mla_empty_row_and_shared_layer_handle(mla_case):
    c = mla_case
    topk = c["topk"].clone()
    topk[1] = -1                                       # nothing selected
    share = D.TopkShare()
    with pytest.raises(D.DsaError) as e:
        D.dsa_sparse_mla_decode(c["q"], None, c["cache"], c["batch"], share=share)
    assert e.value.code == 5                           # no full layer published yet
    share.publish(0, topk)
    lse = torch.empty(c["w"].total_q, 64, device=DEV)
    a = D.dsa_sparse_mla_decode(c["q"], None, c["cache"], c["batch"], share=share, out_dtype=D.DTYPE_F32, lse=lse)
    b = D.dsa_sparse_mla_decode(c["q"], topk, c["cache"], c["batch"], out_dtype=D.DTYPE_F32)
    assert torch.equal(a, b)
    assert not a[1].any() and torch.isneginf(lse[1]).all()


def test_sparse_mla_records_bad_page_without_fault(mla_case):
    c = mla_case
    b = c["batch"]
    pt = b.page_table.clone()
    pt[4, 10] = -7                                     # request 4: logical page 10 corrupted
    bad = D.Batch(b.seq_len, b.q_start, pt, c["w"].num_pages, max_seq_len=b.c.max_seq_len,
                  max_q_len=b.c.max_q_len, total_q=b.total_q)
    st = D.new_device_status(DEV)
    out = D.dsa_sparse_mla_decode(c["q"], c["topk"], c["cache"], bad, out_dtype=D.DTYPE_F32, dev_status=st)
    res = D.dsa_device_status_read(st)
    assert res[0] & D.DEVERR_PAGE_RANGE and res[2] == -7
    assert torch.isfinite(out).all()


def test_sparse_mla_query_rows_of_any_magnitude_and_rope_overflow(mla_case):
    # The kernel computes in fp16; every query row is first scaled by a power of
    # two, so rows far outside fp16's range (x 2^20) or deep in its subnormals
    # (x 2^-20) still match the oracle.  A key RoPE value of 2^16 or more does
    # not fit fp16: it is recorded, and the output stays finite.
    c = mla_case
    w = c["w"]
    ocache = c["cache"].cpu().numpy().reshape(w.num_pages, -1)
    pt = c["batch"].page_table.cpu().numpy()
    qs = c["batch"].q_start.cpu().numpy()
    q = c["q"].clone()
    rows = {3: 2.0 ** 20, 5: 2.0 ** -20, 11: 2.0 ** 16}
    for i, f in rows.items():
        q[i] = (q[i].double() * f).to(torch.bfloat16)      # exact: a power of two
    assert q[3].float().abs().max() > 65504.0
    st = D.new_device_status(DEV)
    lse = torch.empty(w.total_q, 64, device=DEV)
    out = D.dsa_sparse_mla_decode(q, c["topk"], c["cache"], c["batch"], out_dtype=D.DTYPE_F32, lse=lse,
                                  dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    topk = c["topk"].cpu().numpy()
    for i in range(w.total_q):
        r = int(np.searchsorted(qs, i, side="right") - 1)
        p = w.seq_len[r] - w.q_len[r] + (i - qs[r])
        if i in rows:
            krows = O.latent_cache_read_rows(ocache, pt[r], np.maximum(topk[i], 0))
            ref, ref_lse = O.sparse_mla(f64(q[i]), topk[i], krows, p)
        else:
            ref, ref_lse = c["out"][i], c["lse"][i]
        check_attention(out[i], ref, what=f"scaled q row {i}")
        assert np.allclose(lse[i], ref_lse, rtol=1e-5, atol=1e-4)
    # one selected token of row 3 gets a RoPE value beyond fp16's range
    j = int(topk[3][topk[3] >= 0][7])
    bad_cache = ocache.copy()
    r3 = int(np.searchsorted(qs, 3, side="right") - 1)
    page, slot = pt[r3][j // 64], j % 64
    off = slot * O.LATENT_TOKEN_BYTES + 512 + 16 + 2 * 5
    big = torch.tensor([70000.0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
    bad_cache[page, off:off + 2] = big
    st = D.new_device_status(DEV)
    out = D.dsa_sparse_mla_decode(c["q"], c["topk"], torch.from_numpy(bad_cache.reshape(-1)).to(DEV), c["batch"],
                                  out_dtype=D.DTYPE_F32, dev_status=st)
    res = D.dsa_device_status_read(st)
    assert res[0] & D.DEVERR_FP16_RANGE
    assert torch.isfinite(out).all()


# ------------------------------------------------------------------ fused latent store
@pytest.mark.parametrize("with_index", [False, True])
def test_latent_store_fused_matches_oracle(with_index):
    g = _gen(61)
    n, num_pages = 1500, 30
    kv = (torch.randn(n, 512, generator=g) * torch.exp2(torch.randint(-4, 5, (n, 1), generator=g).float())
          ).to(torch.bfloat16)
    pe = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, 1 << 20, (n,), generator=g, dtype=torch.int32)
    slots = torch.randperm(num_pages * 64, generator=g)[:n].to(torch.int64)
    slots[::37] = -1
    gam = torch.rand(512, generator=g) + 0.5
    idx_k = torch.randn(n, 128, generator=g).to(torch.bfloat16) if with_index else None
    kvc = torch.zeros(num_pages * O.LATENT_PAGE_BYTES, dtype=torch.uint8, device=DEV)
    ikc = torch.zeros(num_pages * O.INDEX_PAGE_BYTES, dtype=torch.uint8, device=DEV) if with_index else None
    st = D.new_device_status(DEV)
    D.dsa_latent_kv_store_fused(kv.to(DEV), pe.to(DEV), pos.to(DEV), slots.to(DEV), kvc, kv_gamma=gam.to(DEV),
                                idx_k=None if idx_k is None else idx_k.to(DEV), idxk_cache=ikc, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    codes, scales, rbits = O.latent_prepare(f64(kv), f64(pe), pos.numpy(), f64(gam))
    s = slots.numpy()
    keep = s >= 0
    cache = kvc.cpu().numpy().reshape(num_pages, O.LATENT_PAGE_BYTES)
    page, row = np.divmod(s[keep], 64)
    rows = cache[page[:, None], row[:, None] * 656 + np.arange(656)]
    gcodes = rows[:, :512]
    gsc = np.ascontiguousarray(rows[:, 512:528]).view("<f4").astype(np.float64)
    grope = O.bf16_bits_to_f64(np.ascontiguousarray(rows[:, 528:656]).view("<u2"))
    # latent: scales equal except at power-of-two amax, values within one FP8 ulp
    smis = gsc != scales[keep]
    assert smis.mean() < 2e-3
    gd = O.e4m3_decode(gcodes).reshape(-1, 4, 128) * gsc[..., None]
    od = O.e4m3_decode(codes[keep]).reshape(-1, 4, 128) * scales[keep][..., None]
    ulp = np.maximum(O.e4m3_ulp(od / scales[keep][..., None]) * scales[keep][..., None],
                     O.e4m3_ulp(gd / gsc[..., None]) * gsc[..., None])
    assert np.all(np.abs(gd - od) <= ulp * (1 + 1e-12))
    # RoPE dims: within one bf16 ulp of the oracle's nearest bf16
    orope = O.bf16_bits_to_f64(rbits[keep])
    bulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(orope), 1e-30))) - 7)
    assert np.all(np.abs(grope - orope) <= bulp * (1 + 1e-9))
    assert (grope != orope).mean() < 2e-2
    if with_index:                                      # the same bytes as the plain index-K store
        ref = torch.zeros_like(ikc)
        D.dsa_index_k_store(idx_k.to(DEV), pos.to(DEV), slots.to(DEV), ref)
        assert torch.equal(ikc, ref)



def test_indexer_topk_decode_all_keys_equal():
    """Rows whose every cached key is the same stored bytes: every score ties, so
    the top-2048 is positions 0..2047 exactly.  The boundary bin then holds far
    more than 2048 candidates (the radix selection, in shared memory and in
    place)."""
    seq = [3000, 20000, 2049]
    w = _small_workload(seq, [1] * len(seq), 4444)
    g = _gen(4444)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    one_codes, one_scales = O.index_k_prepare(f64(torch.randn(1, 128, generator=g).to(torch.bfloat16)), np.array([5]))
    cache = np.zeros((w.num_pages, O.INDEX_PAGE_BYTES), np.uint8)
    for r, L in enumerate(seq):
        p = np.arange(L)
        O.index_cache_write(cache, pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64,
                            np.repeat(one_codes, L, axis=0), np.repeat(one_scales, L))
    q = torch.randn(len(seq), 32, 128, generator=g).to(torch.bfloat16)
    wt = torch.randn(len(seq), 32, generator=g).abs() / math.sqrt(32)
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=1, total_q=len(seq))
    sc = torch.empty(len(seq), 2048, device=DEV)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk(q.to(DEV), wt.to(DEV), torch.from_numpy(cache.reshape(-1)).to(DEV), batch,
                              topk_scores=sc, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    topk, sc = topk.cpu().numpy(), sc.cpu().numpy()
    for r, L in enumerate(seq):
        assert topk[r].tolist() == list(range(2048)), f"row {r}"
        kc, ks = O.index_cache_read(cache, pt[r].numpy(), 1)
        qc, qs = O.index_q_quantize(f64(q[r]))
        s1 = O.indexer_scores(qc, qs, f64(wt[r]), kc, ks)[0]
        m1 = O.score_magnitude(qc, qs, f64(wt[r]), kc, ks)[0]
        check_scores(sc[r], np.full(2048, s1), np.full(2048, m1), what=f"row {r} scores")
        assert np.all(sc[r] == sc[r][0])


# ------------------------------------------------------------------ multi-row top-k without score rows
# Batches with several query rows per request stream each row's candidates into
# workspace slots, compacting a slot to its exact top-2048 when it fills.  These
# contexts are long enough that a row block is cut into several CTA pieces and
# slots fill several times.
LONG_SEQ = [40000, 25000, 9000, 2100]
LONG_Q = [6, 8, 3, 5]


@pytest.fixture(scope="module")
def multirow_long_case():
    return _build_indexer_case(LONG_SEQ, LONG_Q, 4321, boost_req=1)


def test_indexer_topk_multirow_streaming_matches_oracle(multirow_long_case):
    _check_indexer_topk(multirow_long_case, 4)


@pytest.mark.parametrize("fill", [0x00, 0xFF])
def test_indexer_topk_multirow_dirty_workspace_and_repeat(multirow_long_case, fill):
    c = multirow_long_case
    nbytes = D.dsa_indexer_topk_workspace_size(c["batch"])
    ws = torch.full((nbytes,), fill, dtype=torch.uint8, device=DEV)
    st = D.new_device_status(DEV)
    a = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"], ws=ws, dev_status=st)
    b = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"], ws=ws, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    assert torch.equal(a, b)
    got = a.cpu().numpy()
    for row in c["rows"]:
        check_topk_row(got[row["i"]], row["topk"], row["s"], row["mag"], row["n"], what=f"row {row['i']}")


# Requests with one or two rows in a multi-row batch leave some epilogue groups
# without rows (a group takes a third of a block's rows); requests with more
# than 8 rows span several row blocks, the last one ragged.
MIXED_SEQ = [30000, 12000, 5000, 20000, 2200]
MIXED_Q = [1, 2, 9, 17, 10]


@pytest.fixture(scope="module")
def multirow_mixed_case():
    return _build_indexer_case(MIXED_SEQ, MIXED_Q, 2468, boost_req=3)


def test_indexer_topk_multirow_groups_without_rows_and_several_row_blocks(multirow_mixed_case):
    _check_indexer_topk(multirow_mixed_case, 4)


def test_indexer_scores_multirow_groups_without_rows_and_several_row_blocks(multirow_mixed_case):
    c = multirow_mixed_case
    st = D.new_device_status(DEV)
    sc = D.dsa_indexer_scores(c["q"], c["wt"], c["cache"], c["batch"], dev_status=st).cpu().numpy()
    assert D.dsa_device_status_read(st)[0] == 0
    for row in c["rows"]:
        i, n = row["i"], row["n"]
        check_scores(sc[i, :n], row["s"], row["mag"], what=f"row {i}")
        assert np.all(np.isneginf(sc[i, n:c["w"].seq_len[row["r"]]]))     # causal: j > p masked


@pytest.fixture(scope="module")
def multirow_many_case():
    # more query rows than SMs: the merge runs two blocks per SM
    rng = np.random.default_rng(13)
    seq = rng.integers(2100, 9000, 40).tolist()
    ql = rng.integers(2, 8, 40).tolist()
    return _build_indexer_case(seq, ql, 1357, boost_req=5)


def test_indexer_topk_multirow_more_rows_than_sms(multirow_many_case):
    assert multirow_many_case["w"].total_q > torch.cuda.get_device_properties(0).multi_processor_count
    _check_indexer_topk(multirow_many_case, 8)


@pytest.mark.parametrize("seq,ql", [([5, 2048, 100, 1], [1, 1, 1, 1]),       # decode, nothing to score
                                     ([2000, 700, 2048], [6, 3, 8]),         # several rows per request
                                     ([1, 2048, 40], [1, 5, 1])])
def test_indexer_topk_when_no_row_sees_more_than_2048_positions(seq, ql):
    """Every row selects all its positions: 0..n-1 ascending, then -1; the plan
    holds no tile, and the score and merge kernels must cope with that."""
    c = _build_indexer_case(seq, ql, 4242)
    _check_indexer_topk(c, 0)
    got = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"]).cpu().numpy()
    for row in c["rows"]:
        n = row["n"]
        assert np.array_equal(got[row["i"], :n], np.arange(n)) and np.all(got[row["i"], n:] == -1)


def test_indexer_topk_multirow_slots_published_above_the_decode_buffer_size():
    """One request with 2 rows on a 730,000-token context: 5,704 tiles over the
    SMs give each CTA a piece of about 37 tiles, whose rows publish about 4,736
    candidates each (more than the decode kernel's 4608-entry buffer) without a
    compaction.  The merge filter must take every one of them."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = 730000
    assert 36 * 128 * sms < L < 48 * 128 * sms          # pieces longer than 36 tiles, shorter than the first check
    c = _build_indexer_case([L], [2], 8642)
    _check_indexer_topk(c, 2)


def test_indexer_topk_multirow_workspace_has_no_score_rows():
    # the workspace holds candidate slots, not T x context score rows: for 8192
    # rows on a 131072-token context it stays far below the 4.29 GB of fp32 rows
    seq, ql = [131072], [8192]
    w = _small_workload(seq, ql, 1)
    meta = batch_meta(w, "cpu")
    pt = torch.zeros((1, 131072 // 64), dtype=torch.int32)
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), 2048, max_seq_len=131072,
                    max_q_len=8192, total_q=8192)
    nbytes = D.dsa_indexer_topk_workspace_size(batch)
    assert nbytes < 8192 * 131072 * 4 // 4


@pytest.mark.parametrize("seq,ql", [([20000, 5000], [4, 7]),
                                     # more rows than SMs (the two-blocks-per-SM merge): each row's
                                     # ~6000 tied candidates overflow its 4096-entry boundary buffer
                                     ([6000] * 40, [5] * 40)])
def test_indexer_topk_multirow_all_keys_equal(seq, ql):
    """Multi-row batches whose every cached key is the same: every score ties,
    so each row with more than 2048 visible positions selects 0..2047 exactly,
    through compactions of slots made entirely of ties."""
    w = _small_workload(seq, ql, 4545)
    g = _gen(4545)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    one_codes, one_scales = O.index_k_prepare(f64(torch.randn(1, 128, generator=g).to(torch.bfloat16)), np.array([5]))
    cache = np.zeros((w.num_pages, O.INDEX_PAGE_BYTES), np.uint8)
    for r, L in enumerate(seq):
        p = np.arange(L)
        O.index_cache_write(cache, pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64,
                            np.repeat(one_codes, L, axis=0), np.repeat(one_scales, L))
    T = sum(ql)
    q = torch.randn(T, 32, 128, generator=g).to(torch.bfloat16)
    wt = torch.randn(T, 32, generator=g).abs() / math.sqrt(32)
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=max(ql), total_q=T)
    sc = torch.empty(T, 2048, device=DEV)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk(q.to(DEV), wt.to(DEV), torch.from_numpy(cache.reshape(-1)).to(DEV), batch,
                              topk_scores=sc, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    topk, sc = topk.cpu().numpy(), sc.cpu().numpy()
    qs = meta["q_start"].numpy()
    for r, L in enumerate(seq):
        for t in range(ql[r]):
            i = qs[r] + t
            assert topk[i].tolist() == list(range(2048)), f"row {i}"
            assert np.all(sc[i] == sc[i][0])
