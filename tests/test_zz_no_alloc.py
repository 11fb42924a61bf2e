"""dsa_indexer_topk_noalloc against dsa_indexer_topk (GPU).

The file name sorts last so that it also runs after every other test; it
passes on its own as well.  Both entry points run the same kernels on the
same inputs, one with a caller workspace and one with the library's fixed
scratch, so the indices must agree exactly and the scores within 1e-6
relative; the no-alloc call is made twice in a row.
"""
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
import synth

pytestmark = pytest.mark.gpu


def _workload(batch, ctx):
    from synth.gpu import GpuWorkload
    w = synth.workload("decode32k", batch=batch, ctx=ctx)
    return GpuWorkload(w, "cuda", layers=[0])


def test_noalloc_matches_workspace_entry_point_twice():
    gw = _workload(batch=24, ctx=12000)
    T = gw.batch.total_q
    ref = torch.empty((T, D.TOPK), dtype=torch.int32, device="cuda")
    ref_sc = torch.empty((T, D.TOPK), dtype=torch.float32, device="cuda")
    D.dsa_indexer_topk(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, topk=ref, topk_scores=ref_sc)
    for _ in range(2):
        st = D.new_device_status("cuda")
        topk = torch.full((T, D.TOPK), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((T, D.TOPK), float("nan"), dtype=torch.float32, device="cuda")
        D.dsa_indexer_topk_noalloc(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, topk=topk, topk_scores=sc,
                                   dev_status=st)
        torch.cuda.synchronize()
        assert D.dsa_device_status_read(st)[0] == 0
        assert torch.equal(topk, ref)
        torch.testing.assert_close(sc, ref_sc, rtol=1e-6, atol=0.0)


def test_noalloc_rejects_batches_beyond_the_scratch():
    # 400 decode rows need more than the 16 MiB scratch on any GPU
    w = synth.workload("decode32k", ctx=3000)
    w.seq_len = (list(w.seq_len) * 7)[:400]
    w.q_len = [1] * 400
    from synth.gpu import GpuWorkload
    big = GpuWorkload(w, "cuda", layers=[])
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_topk_noalloc(big.q_idx, big.w_idx, big.idx_cache, big.batch)
    assert e.value.name == "DSA_ERR_SCRATCH_LIMIT"


def test_noalloc_rejects_non_decode_batches():
    from synth.gpu import GpuWorkload
    w = synth.workload("verify64k", batch=2, ctx=4000)
    gw = GpuWorkload(w, "cuda", layers=[])
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_topk_noalloc(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch)
    assert e.value.name == "DSA_ERR_UNSUPPORTED"
