"""Parity at the full benchmark sizes (GPU), on sampled query rows.

Each workload runs exactly the calls the benchmark times, on its full
synthetic batch: dsa_indexer_topk for the full layer, published through a
share handle, then sparse MLA for the full layer and, for decode32k, for a
shared layer that reuses the same indices with its own latent cache.  For a few
sampled query rows the fp64 oracle recomputes everything those rows depend on:

- the scores of every visible position and the oracle top-2048, from the
  index-K pages the GPU wrote (the stores have their own parity tests);
- sparse MLA over the GPU-selected positions, from the GPU-written latent rows.

The bars are those of the small parity tests: scores within 1e-3 D_j, selected
sets differing only within that tolerance of the 2048th score, and attention
within rel-L2 1e-3 / max-abs 1e-2 of the oracle rounded to bf16.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
import synth
from oracle import dsa_oracle as O
from oracle_side import check_attention, check_scores, check_topk_row, f64, round_bf16

pytestmark = pytest.mark.gpu

CHUNK = 1 << 16                      # positions per oracle scoring chunk (bounds host memory)


def _pages(cache, page_row, n_tokens, page_bytes):
    """The request's first ceil(n / 64) pages as a compact host array, and the
    identity page table that reads them."""
    npg = (n_tokens + 63) // 64
    ids = page_row[:npg].to(torch.int64)
    pages = cache.view(-1, page_bytes).index_select(0, ids).cpu().numpy()
    return pages, np.arange(npg, dtype=np.int64)


def _oracle_row_scores(idx_pages, ident, q, wt, n):
    """Oracle scores and magnitudes of positions 0..n-1 for one query row."""
    qc, qs = O.index_q_quantize(q)
    kc, ks = O.index_cache_read(idx_pages, ident, n)
    s = np.empty(n)
    m = np.empty(n)
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        s[a:b] = O.indexer_scores(qc, qs, wt, kc[a:b], ks[a:b])
        m[a:b] = O.score_magnitude(qc, qs, wt, kc[a:b], ks[a:b])
    return s, m


CASES = {
    # workload: sampled rows (indices into the batch's query rows)
    "tiny": [0],
    "decode32k": [0, 17, 63],
    "decode1m": [2],
    "verify64k": [0, 5, 6 * 77 + 3, 767],
    "prefill128k": [0, 4097, 8191],
}


@pytest.mark.parametrize("name", list(CASES))
def test_full_size_sampled_rows(name):
    from synth.gpu import GpuWorkload
    w = synth.workload(name)
    layers = [0, 1] if len(w.layers) > 1 else [0]
    gw = GpuWorkload(w, "cuda", layers=layers)
    st = D.new_device_status("cuda")
    share = D.TopkShare()
    T = w.total_q
    topk = torch.empty((T, D.TOPK), dtype=torch.int32, device="cuda")
    sel = torch.empty((T, D.TOPK), dtype=torch.float32, device="cuda")
    D.dsa_indexer_topk(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, topk=topk, topk_scores=sel, share=share,
                       layer_id=0, dev_status=st)
    mla = D.dsa_sparse_mla_decode if w.max_q_len == 1 else D.dsa_sparse_mla_prefill
    outs = {l: mla(gw.q_mla[l], None, gw.kv_cache[l], gw.batch, share=share, dev_status=st) for l in layers}
    torch.cuda.synchronize()
    assert D.dsa_device_status_read(st)[0] == 0

    q_start = gw.q_start.cpu().numpy()
    seq = gw.seq_len.cpu().numpy()
    for i in CASES[name]:
        r = int(np.searchsorted(q_start, i, side="right") - 1)
        qn = int(q_start[r + 1] - q_start[r])
        p = int(seq[r]) - qn + (i - int(q_start[r]))
        n = p + 1
        row_topk = topk[i].cpu().numpy()
        idx_pages, ident = _pages(gw.idx_cache, gw.pt[r], n, D.IDXK_PAGE_BYTES)
        s, mag = _oracle_row_scores(idx_pages, ident, f64(gw.q_idx[i]), f64(gw.w_idx[i]), n)
        check_topk_row(row_topk, O.topk_positions(s, n), s, mag, n, what=f"{name} row {i}")
        if n > D.TOPK:
            check_scores(sel[i].cpu().numpy(), s[row_topk], mag[row_topk], what=f"{name} row {i} selected")
        valid = row_topk[row_topk >= 0]
        for l in layers:
            kv_pages, kident = _pages(gw.kv_cache[l], gw.pt[r], n, D.KV_PAGE_BYTES)
            rows = O.latent_cache_read_rows(kv_pages, kident, valid)
            ref, _ = O.sparse_mla(f64(gw.q_mla[l][i]), valid, rows, p)
            check_attention(outs[l][i].float().cpu().numpy(), round_bf16(ref), what=f"{name} layer {l} row {i}")


def test_full_size_mxfp4_decode1m_sampled_row():
    """decode1m over an MXFP4 index-K cache: one sampled row rescored by the oracle
    at all 1,048,576 positions, from the MXFP4 pages the GPU wrote."""
    from synth.gpu import GpuWorkload
    w = synth.workload("decode1m")
    w.index_format = "mxfp4"
    gw = GpuWorkload(w, "cuda", layers=[])
    st = D.new_device_status("cuda")
    T = w.total_q
    sel = torch.empty((T, D.TOPK), dtype=torch.float32, device="cuda")
    topk = D.dsa_indexer_topk_mxfp4(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, topk_scores=sel, dev_status=st)
    torch.cuda.synchronize()
    assert D.dsa_device_status_read(st)[0] == 0
    i = 1
    n = int(gw.seq_len[i])
    pages, ident = _pages(gw.idx_cache, gw.pt[i], n, D.IDXK_MXFP4_PAGE_BYTES)
    qc, qs = O.index_q_quantize(f64(gw.q_idx[i]))
    kc, ke = O.mxfp4_cache_read(pages, ident, n)
    wt = f64(gw.w_idx[i])
    s = np.empty(n)
    m = np.empty(n)
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        s[a:b] = O.indexer_scores_mxfp4(qc, qs, wt, kc[a:b], ke[a:b])
        m[a:b] = O.score_magnitude_mxfp4(qc, qs, wt, kc[a:b], ke[a:b])
    row = topk[i].cpu().numpy()
    check_topk_row(row, O.topk_positions(s, n), s, m, n, what="mxfp4 decode1m")
    check_scores(sel[i].cpu().numpy(), s[row], m[row], what="mxfp4 decode1m selected")


def test_full_size_mtp_iteration_sampled_request():
    """One MTP iteration at full size (4 requests, 5 draft steps from a
    1,048,576-token context): the first step's top-2048 against the oracle, the
    later steps carrying that row bit for bit, every step's attention against the
    oracle from the GPU-written latent rows."""
    from synth.gpu import GpuWorkload
    w = synth.workload("mtp5_1m")
    gw = GpuWorkload(w, "cuda", layers=[0])
    nd, B = w.draft_steps, w.batch
    st = D.new_device_status("cuda")

    def rows(t, k):
        return t.view(B, nd, *t.shape[1:])[:, k].contiguous()

    q0 = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    share = D.TopkShare()
    topk = torch.empty((B, D.TOPK), dtype=torch.int32, device="cuda")
    sel = torch.empty((B, D.TOPK), dtype=torch.float32, device="cuda")
    outs, carried, scored = [], [], []
    with share.mtp_iteration(True, 1) as reuse:
        assert reuse
        for k in range(nd):
            seq = (gw.seq_len - (nd - 1 - k)).contiguous()
            bk = D.Batch(seq, q0, gw.pt, w.num_pages, max_seq_len=w.max_seq_len - (nd - 1 - k), max_q_len=1, total_q=B)
            scored.append(share.needs_scoring())
            if scored[-1]:
                D.dsa_indexer_topk(rows(gw.q_idx, k), rows(gw.w_idx, k), gw.idx_cache, bk, topk=topk, topk_scores=sel,
                                   share=share, layer_id=0, dev_status=st)
            carried.append(topk.clone())
            outs.append(D.dsa_sparse_mla_decode(rows(gw.q_mla[0], k), None, gw.kv_cache[0], bk, share=share,
                                                dev_status=st))
    torch.cuda.synchronize()
    assert D.dsa_device_status_read(st)[0] == 0
    assert scored == [True] + [False] * (nd - 1)
    assert all(torch.equal(c, carried[0]) for c in carried)
    r = 2
    L0 = int(gw.seq_len[r]) - (nd - 1)                   # the first draft step's context
    i0 = r * nd                                          # request r's first draft row in the workload's rows
    idx_pages, ident = _pages(gw.idx_cache, gw.pt[r], L0, D.IDXK_PAGE_BYTES)
    s, mag = _oracle_row_scores(idx_pages, ident, f64(gw.q_idx[i0]), f64(gw.w_idx[i0]), L0)
    row = carried[0][r].cpu().numpy()
    check_topk_row(row, O.topk_positions(s, L0), s, mag, L0, what="mtp step 0")
    check_scores(sel[r].cpu().numpy(), s[row], mag[row], what="mtp step 0 selected")
    valid = row[row >= 0]
    kv_pages, kident = _pages(gw.kv_cache[0], gw.pt[r], L0 + nd - 1, D.KV_PAGE_BYTES)
    lat = O.latent_cache_read_rows(kv_pages, kident, valid)
    for k in range(nd):
        ref, _ = O.sparse_mla(f64(gw.q_mla[0][i0 + k]), valid, lat, L0 - 1 + k)
        check_attention(outs[k][r].float().cpu().numpy(), round_bf16(ref), what=f"mtp step {k}")
