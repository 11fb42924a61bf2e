"""The context-parallel split on CPU ranks (gloo, world size 2).

Two processes each hold one slice of a long decode request, cut at a position
that is not a page boundary, in caches of their own.  The binding's
ContextParallel drives the two exchanges over the gloo process group; the
per-rank steps (indexer + top-k with scores, the merges, sparse MLA with its
log-sum-exp) are done here by the fp64 oracle, since a CPU rank has no GPU.
The merged top-2048 must equal the oracle's top-2048 of the whole context, and
the merged attention must equal the oracle's attention over it.
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

L_CTX = 5000
CUT = 2601            # rank 0 holds positions [0, 2601), rank 1 [2601, 5000)


def _request(seed=77):
    """The whole request's raw inputs (seeded), shared by both ranks and the check."""
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(L_CTX, 128, generator=g).to(torch.bfloat16).double().numpy()
    c = torch.randn(L_CTX, 512, generator=g).to(torch.bfloat16).double().numpy()
    r = torch.randn(L_CTX, 64, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 32, 128, generator=g).to(torch.bfloat16).double().numpy()
    w = (torch.randn(1, 32, generator=g) / 32 ** 0.5).double().numpy()
    qm = torch.randn(1, 64, 576, generator=g).to(torch.bfloat16).double().numpy()
    return k, c, r.contiguous().view(torch.int16).numpy().view(np.uint16), q, w, qm


class _Slice:
    """A rank's slice [a, b) of the request in caches of its own (local positions)."""

    def __init__(self, a, b):
        from oracle import dsa_oracle as O
        k, c, rbits, _, _, _ = _request()
        n = b - a
        npg = (n + 63) // 64
        self.n = n
        self.pt = np.arange(npg, dtype=np.int32)[::-1].copy()            # any page layout
        slots = self.pt[np.arange(n) // 64].astype(np.int64) * 64 + np.arange(n) % 64
        self.idx = np.zeros((npg, O.INDEX_PAGE_BYTES), np.uint8)
        codes, scales = O.index_k_prepare(k[a:b], np.arange(a, b))      # RoPE at the global positions
        O.index_cache_write(self.idx, slots, codes, scales)
        self.kv = np.zeros((npg, O.LATENT_PAGE_BYTES), np.uint8)
        lc, lsc = O.latent_quantize(c[a:b])
        O.latent_cache_write(self.kv, slots, lc, lsc, rbits[a:b])


class OracleOps:
    """The per-rank steps, by the fp64 oracle (host tensors in, host tensors out)."""

    def indexer_topk(self, q, w, idxk_cache, batch, ws=None, dev_status=None, stream=None):
        from oracle import dsa_oracle as O
        sl = batch
        kc, ks = O.index_cache_read(sl.idx, sl.pt, sl.n)
        qc, qs = O.index_q_quantize(q.numpy()[0])
        s = O.indexer_scores(qc, qs, w.numpy()[0], kc, ks)
        top = O.topk_positions(s, sl.n)
        sc = np.where(top >= 0, s[np.maximum(top, 0)], 0.0)
        return torch.from_numpy(top[None].copy()), torch.from_numpy(sc[None].astype(np.float32))

    def topk_merge(self, cand_pos, cand_scores, pos_offset, dev_status=None, stream=None):
        from oracle import dsa_oracle as O
        G, T = cand_pos.shape[:2]
        out = np.empty((T, 2048), np.int32)
        for t in range(T):
            pos = [np.where(cand_pos[g, t].numpy() >= 0, cand_pos[g, t].numpy() + int(pos_offset[g, t]), -1)
                   for g in range(G)]
            out[t] = O.cp_merge_topk(pos, [cand_scores[g, t].numpy() for g in range(G)])
        return torch.from_numpy(out)

    def topk_localize(self, topk, slice_start, slice_len, stream=None):
        out = np.full(topk.shape, -1, np.int32)
        for t in range(topk.shape[0]):
            a, n = int(slice_start[t]), int(slice_len[t])
            row = topk[t].numpy()
            mine = row[(row >= a) & (row < a + n)] - a
            out[t, :mine.size] = mine
        return torch.from_numpy(out)

    def sparse_mla(self, q, local_topk, kv_cache, batch, softmax_scale, ws=None, dev_status=None, stream=None):
        from oracle import dsa_oracle as O
        sl = batch
        idx = local_topk[0].numpy()
        rows = O.latent_cache_read_rows(sl.kv, sl.pt, np.maximum(idx, 0))
        o, lse = O.sparse_mla(q[0].numpy(), idx, rows, sl.n - 1, scale=softmax_scale)
        return torch.from_numpy(o[None]), torch.from_numpy(lse[None])

    def attention_merge(self, o_parts, lse_parts, out_dtype, stream=None):
        from oracle import dsa_oracle as O
        o, lse = O.lse_merge([o_parts[g, 0].numpy() for g in range(o_parts.shape[0])],
                             [lse_parts[g, 0].numpy() for g in range(lse_parts.shape[0])])
        return torch.from_numpy(o[None]), torch.from_numpy(lse[None])


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import dsa_sparse_attention_indexer_gb300 as D
    a, b = (0, CUT) if rank == 0 else (CUT, L_CTX)
    sl = _Slice(a, b)
    _, _, _, q, w, qm = _request()
    cp = D.ContextParallel(ops=OracleOps())
    start = torch.tensor([a], dtype=torch.int64)
    length = torch.tensor([b - a], dtype=torch.int64)
    topk = cp.indexer_topk(torch.from_numpy(q), torch.from_numpy(w), None, sl, start)
    o, lse = cp.sparse_mla(torch.from_numpy(qm), topk, None, sl, start, length)
    out[rank] = (topk.numpy(), o.numpy(), lse.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_context_parallel_two_gloo_ranks_match_the_whole_request():
    from oracle import dsa_oracle as O
    world = 2
    port = 29700 + os.getpid() % 1000
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    # the whole request on one rank, by the oracle
    whole = _Slice(0, L_CTX)
    _, _, _, q, w, qm = _request()
    ref_topk, _ = O.request_topk(q, w, whole.idx, whole.pt, L_CTX, 1)
    rows = O.latent_cache_read_rows(whole.kv, whole.pt, np.maximum(ref_topk[0], 0))
    ref_o, ref_lse = O.sparse_mla(qm[0], ref_topk[0], rows, L_CTX - 1)
    for rank in range(world):
        topk, o, lse = out[rank]
        assert np.array_equal(topk[0], ref_topk[0]), f"rank {rank}: merged top-k differs"
        assert np.allclose(o[0], ref_o, rtol=1e-9, atol=1e-12)
        assert np.allclose(lse[0], ref_lse, rtol=1e-12, atol=1e-12)
    # both slices contributed selected positions
    assert (ref_topk[0] < CUT).sum() > 100 and (ref_topk[0] >= CUT).sum() > 100
