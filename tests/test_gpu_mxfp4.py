"""GPU parity of the MXFP4 index-K variant ("GLM-5.3 推理全链路(十一)", 两个框架的对照:
128/2 packed bytes + 128/32 ue8m0 scales = 68 B per token) against the fp64
oracle: the store (LayerNorm -> RoPE -> MX block scale -> E2M1) and the decode
indexer + top-2048 over an MXFP4 cache.
"""

import math

import numpy as np
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
from oracle import dsa_oracle as O
from synth import Workload, batch_meta, page_table
from tests.oracle_side import check_scores, check_topk_row, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
PB = O.MXFP4_PAGE_BYTES


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _decode_mx_cache(cache: np.ndarray, slots: np.ndarray):
    page, row = np.divmod(slots, 64)
    packed = cache[page[:, None], row[:, None] * 64 + np.arange(64)]
    codes = np.empty((len(slots), 128), np.uint8)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    exps = cache[page[:, None], 4096 + row[:, None] * 4 + np.arange(4)].astype(np.int64) - 127
    return codes, exps


@pytest.mark.parametrize("affine", [False, True])
def test_index_k_store_mxfp4_matches_oracle(affine):
    g = _gen(21)
    n, num_pages = 3000, 60
    mag = torch.exp2(torch.randint(-6, 7, (n, 1), generator=g).float())
    k = (torch.randn(n, 128, generator=g) * mag + torch.randn(n, 1, generator=g)).to(torch.bfloat16)
    k[5] = 0.0                                          # constant row: every block 0, exponent 0
    pos = torch.randint(0, 1 << 20, (n,), generator=g, dtype=torch.int32)
    slots = torch.randperm(num_pages * 64, generator=g)[:n].to(torch.int64)
    slots[::50] = -1
    gamma = (torch.rand(128, generator=g) + 0.5) if affine else None
    beta = (torch.randn(128, generator=g) * 0.1) if affine else None
    cache = torch.zeros(num_pages * PB, dtype=torch.uint8, device=DEV)
    st = D.new_device_status(DEV)
    D.dsa_index_k_store_mxfp4(k.to(DEV), pos.to(DEV), slots.to(DEV), cache,
                              gamma=None if gamma is None else gamma.to(DEV),
                              beta=None if beta is None else beta.to(DEV), dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    gcache = cache.cpu().numpy().reshape(num_pages, PB)
    y = O.rope_interleaved(O.layer_norm(f64(k), None if gamma is None else f64(gamma),
                                        None if beta is None else f64(beta), 1e-6), pos.numpy(), 10000.0)
    ocodes, oexps = O.quantize_mxfp4(y)
    s = slots.numpy()
    keep = s >= 0
    gcodes, gexps = _decode_mx_cache(gcache, s[keep])
    oc, oe = ocodes[keep], oexps[keep]
    yk = y[keep].reshape(-1, 4, 32)
    amax = np.abs(yk).max(axis=-1)
    emis = gexps != oe
    if emis.any():                                      # only where amax sits on a power of two
        r = amax[emis]
        assert np.all(np.abs(r / np.exp2(np.round(np.log2(r))) - 1) < 1e-5)
    assert emis.mean() < 1e-3
    gd = O.mxfp4_dequant(gcodes, gexps).reshape(-1, 4, 32)
    od = O.mxfp4_dequant(oc, oe).reshape(-1, 4, 32)
    step = np.maximum(np.exp2(gexps), np.exp2(oe))[..., None]
    assert np.all(np.abs(gd - od) <= 2.0 * step)        # at most one step of the coarsest grid spacing
    assert (gcodes != oc).mean() < 2e-3
    if s[5] >= 0:                                       # the constant row: signed zeros, exponent 0
        j = int(np.flatnonzero(s[keep] == s[5])[0])
        assert np.array_equal(gcodes[j], oc[j]) and np.array_equal(gexps[j], oe[j])
        if not affine:                                  # LayerNorm of a constant is 0 (beta shifts it)
            assert np.all(gexps[j] == 0) and not np.any(O.e2m1_decode(gcodes[j]))
    written = np.zeros(num_pages * 64, bool)
    written[s[keep]] = True
    c2, e2 = _decode_mx_cache(gcache, np.nonzero(~written)[0])
    assert not c2.any() and np.all(e2 == -127)          # untouched bytes stay zero


def test_index_k_store_mxfp4_records_out_of_range_slot():
    cache = torch.zeros(2 * PB, dtype=torch.uint8, device=DEV)
    k = torch.randn(3, 128).to(torch.bfloat16).to(DEV)
    st = D.new_device_status(DEV)
    D.dsa_index_k_store_mxfp4(k, torch.zeros(3, dtype=torch.int32, device=DEV),
                              torch.tensor([0, 500, 1], dtype=torch.int64, device=DEV), cache, dev_status=st)
    hs = D.dsa_device_status_read(st)
    assert hs[0] == D.DEVERR_SLOT_RANGE and hs[1] == 1


MX_SEQ = [2049, 1, 100, 2048, 4097, 6000, 2100, 33000, 10000, 128 * 40, 128 * 40 + 1, 8191]


@pytest.fixture(scope="module")
def mx_case():
    seq = MX_SEQ
    w = Workload("mx", 5151, list(seq), [1] * len(seq), ["full"])
    g = _gen(5151)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    cache = np.zeros((w.num_pages, PB), np.uint8)
    for r, L in enumerate(seq):
        raw = f64(torch.randn(L, 128, generator=g).to(torch.bfloat16))
        p = np.arange(L)
        codes, exps = O.index_k_prepare_mxfp4(raw, p)
        boost = np.zeros(L, bool)
        boost[::97] = r == 7                            # a few x4 keys in one request
        O.mxfp4_cache_write(cache, pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64, codes,
                            exps + 2 * boost[:, None])
    q = torch.randn(w.total_q, 32, 128, generator=g).to(torch.bfloat16)
    wt = torch.randn(w.total_q, 32, generator=g) / math.sqrt(32)
    rows = []
    for r, L in enumerate(seq):
        kc, ke = O.mxfp4_cache_read(cache, pt[r].numpy(), L)
        qc, qs = O.index_q_quantize(f64(q[r]))
        s = O.indexer_scores_mxfp4(qc, qs, f64(wt[r]), kc, ke)
        m = O.score_magnitude_mxfp4(qc, qs, f64(wt[r]), kc, ke)
        rows.append(dict(i=r, n=L, s=s, mag=m, topk=O.topk_positions(s, L)))
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=1, total_q=w.total_q)
    return dict(w=w, cache=torch.from_numpy(cache.reshape(-1)).to(DEV), q=q.to(DEV), wt=wt.to(DEV), batch=batch,
                rows=rows, pt=pt)


def test_indexer_topk_mxfp4_matches_oracle(mx_case):
    c = mx_case
    T = c["w"].total_q
    sc = torch.empty(T, 2048, device=DEV)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk_mxfp4(c["q"], c["wt"], c["cache"], c["batch"], topk_scores=sc, dev_status=st)
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
    assert ndiff <= 2
    again = D.dsa_indexer_topk_mxfp4(c["q"], c["wt"], c["cache"], c["batch"]).cpu().numpy()
    assert np.array_equal(again, topk)                  # repeatable


def test_indexer_topk_mxfp4_records_bad_page_without_fault(mx_case):
    c = mx_case
    pt = c["pt"].clone()
    pt[4, 3] = c["w"].num_pages + 7                     # request 4 (4097 tokens): one page id out of range
    meta = batch_meta(c["w"], "cpu")
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), c["w"].num_pages,
                    max_seq_len=c["w"].max_seq_len, max_q_len=1, total_q=c["w"].total_q)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk_mxfp4(c["q"], c["wt"], c["cache"], batch, dev_status=st).cpu().numpy()
    hs = D.dsa_device_status_read(st)
    assert hs[0] & D.DEVERR_PAGE_RANGE
    assert not np.any((topk[4] >= 3 * 64) & (topk[4] < 4 * 64))   # the skipped page contributes nothing


# Several query rows per request (speculative verify, prefill chunks): row t of
# a request sees positions 0 .. L - q_len + t; rows of 2047 and 2048 visible
# positions take the short-context rule.
MXR_SEQ = [9000, 2050, 40000, 3000]
MXR_Q = [4, 4, 3, 5]


def _mx_keys(seq, seed):
    g = _gen(seed)
    return g, [f64(torch.randn(L, 128, generator=g).to(torch.bfloat16)) for L in seq]


@pytest.fixture(scope="module")
def mx_rows_case():
    w = Workload("mxr", 6161, list(MXR_SEQ), list(MXR_Q), ["full"])
    g, raws = _mx_keys(MXR_SEQ, 6161)
    pt = page_table(w, "cpu")
    meta = batch_meta(w, "cpu")
    mx = np.zeros((w.num_pages, PB), np.uint8)
    fp8 = np.zeros((w.num_pages, O.INDEX_PAGE_BYTES), np.uint8)
    for r, L in enumerate(MXR_SEQ):
        p = np.arange(L)
        slots = pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64
        codes, exps = O.index_k_prepare_mxfp4(raws[r], p)
        O.mxfp4_cache_write(mx, slots, codes, exps)
        c8, s8 = O.index_k_prepare(raws[r], p)
        O.index_cache_write(fp8, slots, c8, s8)
    q = torch.randn(w.total_q, 32, 128, generator=g).to(torch.bfloat16)
    wt = torch.randn(w.total_q, 32, generator=g) / math.sqrt(32)
    qs = meta["q_start"].numpy()
    rows = []
    for r, L in enumerate(MXR_SEQ):
        ql = MXR_Q[r]
        topk, scores = O.request_topk_mxfp4(f64(q[qs[r]:qs[r] + ql]), f64(wt[qs[r]:qs[r] + ql]), mx, pt[r].numpy(),
                                            L, ql)
        kc, ke = O.mxfp4_cache_read(mx, pt[r].numpy(), L)
        k8, s8 = O.index_cache_read(fp8, pt[r].numpy(), L)
        for t in range(ql):
            i = qs[r] + t
            n = L - ql + t + 1
            row = dict(i=i, n=n, topk=topk[t], s=scores[t])
            if n > 2048:
                qc, qsc = O.index_q_quantize(f64(q[i]))
                row["mag"] = O.score_magnitude_mxfp4(qc, qsc, f64(wt[i]), kc[:n], ke[:n])
                s_fp8 = O.indexer_scores(qc, qsc, f64(wt[i]), k8[:n], s8[:n])
                row["overlap"] = len(set(O.topk_positions(s_fp8, n).tolist()) & set(topk[t].tolist())) / 2048
            rows.append(row)
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), pt.to(DEV), w.num_pages,
                    max_seq_len=w.max_seq_len, max_q_len=max(MXR_Q), total_q=w.total_q)
    return dict(w=w, mx=torch.from_numpy(mx.reshape(-1)).to(DEV), fp8=torch.from_numpy(fp8.reshape(-1)).to(DEV),
                q=q.to(DEV), wt=wt.to(DEV), batch=batch, rows=rows)


def test_indexer_topk_mxfp4_multi_token_rows_match_oracle(mx_rows_case):
    c = mx_rows_case
    T = c["w"].total_q
    sc = torch.empty(T, 2048, device=DEV)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk_mxfp4(c["q"], c["wt"], c["mx"], c["batch"], topk_scores=sc, dev_status=st)
    assert D.dsa_device_status_read(st)[0] == 0
    topk, sc = topk.cpu().numpy(), sc.cpu().numpy()
    ndiff = 0
    for row in c["rows"]:
        i = row["i"]
        if row["n"] <= 2048:
            assert np.array_equal(topk[i], row["topk"]), f"short row {i}"
            continue
        ndiff += check_topk_row(topk[i], row["topk"], row["s"], row["mag"], row["n"], what=f"row {i}")
        check_scores(sc[i], row["s"][topk[i]], row["mag"][topk[i]], what=f"selected scores row {i}")
    assert ndiff <= 4
    nbytes = D.dsa_indexer_topk_workspace_size(c["batch"])
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)   # a dirty workspace changes nothing
    again = D.dsa_indexer_topk_mxfp4(c["q"], c["wt"], c["mx"], c["batch"], ws=ws).cpu().numpy()
    assert np.array_equal(again, topk)


# The MXFP4 keys change the selection itself ("GLM-5.3 推理全链路(十一)", 两个框架的
# 对照): on these Gaussian keys the oracle's MXFP4 and FP8 top-2048 share 0.88 to
# 0.93 of their positions.  The library's two selections must share as much (up to
# the positions the parity rule lets differ) and never fall below 0.85.
OVERLAP_FLOOR = 0.85


def test_indexer_topk_mxfp4_vs_fp8_selection_overlap(mx_rows_case):
    c = mx_rows_case
    t4 = D.dsa_indexer_topk_mxfp4(c["q"], c["wt"], c["mx"], c["batch"]).cpu().numpy()
    t8 = D.dsa_indexer_topk(c["q"], c["wt"], c["fp8"], c["batch"]).cpu().numpy()
    seen = []
    for row in c["rows"]:
        i = row["i"]
        if row["n"] <= 2048:
            assert np.array_equal(t4[i], t8[i])
            continue
        ov = len(set(t4[i].tolist()) & set(t8[i].tolist())) / 2048
        seen.append(ov)
        assert ov >= OVERLAP_FLOOR, f"row {i}: overlap {ov:.3f}"
        assert abs(ov - row["overlap"]) <= 0.01, f"row {i}: overlap {ov:.3f}, oracle {row['overlap']:.3f}"
    assert len(seen) >= 10


def test_indexer_topk_mxfp4_refuses_too_many_rows():
    w = Workload("mx2", 1, [70000], [65536], ["full"])
    meta = batch_meta(w, "cpu")
    batch = D.Batch(meta["seq_len"].to(DEV), meta["q_start"].to(DEV), page_table(w, DEV), w.num_pages,
                    max_seq_len=70000, max_q_len=65536, total_q=65536)
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_topk_mxfp4(torch.zeros(65536, 32, 128, dtype=torch.bfloat16, device=DEV),
                                 torch.zeros(65536, 32, device=DEV), torch.zeros(w.num_pages * PB, dtype=torch.uint8,
                                                                                 device=DEV), batch,
                                 ws=torch.empty(4096, dtype=torch.uint8, device=DEV))
    assert e.value.name == "DSA_ERR_UNSUPPORTED"
