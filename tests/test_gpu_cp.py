"""The context-parallel split through the C ABI on one GPU (GPU).

G ranks are emulated one after another on the same device: each holds a
page-aligned slice of every request, described to the library as requests of
seq_len = slice length over its own page-table rows (the physical caches are
shared, so no data moves).  The per-slice top-2048 lists merged by
dsa_cp_topk_merge must equal the single-rank top-2048 of the whole context bit
for bit (same scores, same tie rule); the per-slice attention parts merged by
dsa_cp_attention_merge must match the single-rank attention and the oracle.
No collective runs here: the exchanges are the stacks of the emulated ranks'
outputs.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
import synth
from oracle import dsa_oracle as O
from tests.oracle_side import check_attention, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _workload():
    from synth.gpu import GpuWorkload
    w = synth.workload("decode32k", batch=6, ctx=14000)
    return GpuWorkload(w, DEV, layers=[0])


@pytest.fixture(scope="module")
def gw():
    return _workload()


def _slices(gw, G, seed):
    """Per rank: its slice [start, start + len) of every request, page-aligned,
    each longer than 2048 tokens."""
    rng = np.random.default_rng(seed)
    seq = gw.seq_len.cpu().numpy()
    starts = np.zeros((G, seq.size), np.int64)
    lens = np.zeros((G, seq.size), np.int64)
    for r, L in enumerate(seq):
        pages = (L + 63) // 64
        cuts, lo = [], 33                              # every slice at least 33 pages (2112 tokens)
        for g in range(G - 1):
            hi = pages - 34 * (G - 1 - g)
            cuts.append(int(rng.integers(lo, hi + 1)))
            lo = cuts[-1] + 33
        edges = [0, *(c * 64 for c in cuts), int(L)]
        for g in range(G):
            starts[g, r], lens[g, r] = edges[g], edges[g + 1] - edges[g]
        assert lens[:, r].min() > 2048
    return starts, lens


def _rank_batch(gw, start, length):
    pt = gw.pt.clone()
    for r in range(pt.shape[0]):
        p0 = int(start[r]) // 64
        npg = (int(length[r]) + 63) // 64
        row = torch.full_like(pt[r], -1)
        row[:npg] = gw.pt[r, p0:p0 + npg]
        pt[r] = row
    seq = torch.as_tensor(length, dtype=torch.int32, device=DEV)
    return D.Batch(seq, gw.q_start, pt, gw.w.num_pages, max_seq_len=int(length.max()), max_q_len=1,
                   total_q=gw.batch.total_q)


@pytest.mark.parametrize("G", [2, 3])
def test_context_parallel_merges_equal_the_whole_request(gw, G):
    T = gw.batch.total_q
    starts, lens = _slices(gw, G, 900 + G)
    st = D.new_device_status(DEV)
    # the whole context on one rank
    ref = torch.empty((T, D.TOPK), dtype=torch.int32, device=DEV)
    ref_sc = torch.empty((T, D.TOPK), dtype=torch.float32, device=DEV)
    D.dsa_indexer_topk(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, topk=ref, topk_scores=ref_sc, dev_status=st)
    ref_lse = torch.empty((T, 64), device=DEV)
    ref_out = D.dsa_sparse_mla_decode(gw.q_mla[0], ref, gw.kv_cache[0], gw.batch, out_dtype=D.DTYPE_F32,
                                      lse=ref_lse, dev_status=st)
    # every rank's slice: local top-2048 with scores
    batches = [_rank_batch(gw, starts[g], lens[g]) for g in range(G)]
    cand_pos = torch.empty((G, T, D.TOPK), dtype=torch.int32, device=DEV)
    cand_sc = torch.empty((G, T, D.TOPK), dtype=torch.float32, device=DEV)
    for g in range(G):
        D.dsa_indexer_topk(gw.q_idx, gw.w_idx, gw.idx_cache, batches[g], topk=cand_pos[g], topk_scores=cand_sc[g],
                           dev_status=st)
    offs = torch.as_tensor(starts, dtype=torch.int64, device=DEV)
    merged_sc = torch.empty((T, D.TOPK), dtype=torch.float32, device=DEV)
    merged = D.dsa_cp_topk_merge(cand_pos, cand_sc, offs, topk_scores=merged_sc, dev_status=st)
    torch.cuda.synchronize()
    assert D.dsa_device_status_read(st)[0] == 0
    assert torch.equal(merged, ref)
    assert torch.equal(merged_sc, ref_sc)
    # every rank attends over the selected positions it holds; the parts merge
    o_parts = torch.empty((G, T, 64, 512), dtype=torch.float32, device=DEV)
    l_parts = torch.empty((G, T, 64), dtype=torch.float32, device=DEV)
    for g in range(G):
        loc = D.dsa_cp_topk_localize(merged, torch.as_tensor(starts[g], device=DEV),
                                     torch.as_tensor(lens[g], device=DEV))
        D.dsa_sparse_mla_decode(gw.q_mla[0], loc, gw.kv_cache[0], batches[g], out=o_parts[g], out_dtype=D.DTYPE_F32,
                                lse=l_parts[g], dev_status=st)
    lse = torch.empty((T, 64), device=DEV)
    out = D.dsa_cp_attention_merge(o_parts, l_parts, out_dtype=D.DTYPE_F32, lse=lse)
    outb = D.dsa_cp_attention_merge(o_parts, l_parts, out_dtype=D.DTYPE_BF16)
    torch.cuda.synchronize()
    assert D.dsa_device_status_read(st)[0] == 0
    for i in range(T):
        check_attention(out[i].cpu().numpy(), f64(ref_out[i]), what=f"G={G} row {i} vs single rank")
    torch.testing.assert_close(lse, ref_lse, rtol=1e-5, atol=1e-4)
    torch.testing.assert_close(outb.float(), out.to(torch.bfloat16).float(), rtol=0, atol=0)
    # and one row against the fp64 oracle on the same cache bytes
    r = 1
    ocache = gw.kv_cache[0].cpu().numpy().reshape(gw.w.num_pages, -1)
    idx = ref[r].cpu().numpy()
    rows = O.latent_cache_read_rows(ocache, gw.pt[r].cpu().numpy(), np.maximum(idx, 0))
    o_ref, _ = O.sparse_mla(f64(gw.q_mla[0][r]), idx, rows, int(gw.seq_len[r]) - 1)
    check_attention(out[r].cpu().numpy(), o_ref, what="merged vs oracle")


def test_localize_keeps_only_the_slice_in_order():
    rng = np.random.default_rng(5)
    T = 3
    glob = np.full((T, 2048), -1, np.int32)
    for t in range(T):
        n = [2048, 1500, 0][t]
        glob[t, :n] = np.sort(rng.choice(50000, n, replace=False))
    start = np.array([10000, 0, 5], np.int64)
    length = np.array([20000, 25000, 100], np.int64)
    loc = D.dsa_cp_topk_localize(torch.from_numpy(glob).to(DEV), torch.from_numpy(start).to(DEV),
                                 torch.from_numpy(length).to(DEV)).cpu().numpy()
    for t in range(T):
        row = glob[t]
        want = row[(row >= start[t]) & (row < start[t] + length[t])] - start[t]
        assert np.array_equal(loc[t, :want.size], want) and np.all(loc[t, want.size:] == -1)
