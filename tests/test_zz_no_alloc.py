"""dsa_indexer_topk_noalloc against dsa_indexer_topk (GPU).

The file name sorts last so that it also runs after every other test; it
passes on its own as well.  Both entry points run the same kernels on the
same inputs, one with a caller workspace and one with the library's fixed
scratch, so the indices must agree exactly and the scores within 1e-6
relative; the no-alloc call is made twice in a row.
"""
import os
import re

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


def _scratch_need(B, S):
    """Bytes the header gives for a decode batch of B rows on S SMs (before
    the up to 768 bytes of alignment it allows)."""
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dsa.h")).read()
    per_seg = int(re.search(r"\(S \+ B\) \* (\d+)", text).group(1))
    return (4224 * B + 255) // 256 * 256 + 16384 * B + (S + B) * per_seg + 12 * (B + 1) + 8 * S


def test_noalloc_at_the_largest_batch_that_fits_and_one_row_more():
    # The end of the scratch, where the plan's candidate arrays sit, is used
    # only by the largest batches: run the largest batch that the header's
    # formula says fits on this GPU, compare it with the workspace entry point,
    # and check that one row more is refused before any launch.
    from synth.gpu import GpuWorkload
    S = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    cap = D.NOALLOC_SCRATCH_BYTES
    fit = max(B for B in range(1, 1024) if _scratch_need(B, S) + 768 <= cap)
    nofit = min(B for B in range(1, 1024) if _scratch_need(B, S) > cap)
    assert nofit == fit + 1

    def batch_of(rows):
        w = synth.workload("decode32k", ctx=4096)
        w.seq_len = (list(w.seq_len) * (rows // len(w.seq_len) + 1))[:rows]
        w.q_len = [1] * rows
        return GpuWorkload(w, "cuda", layers=[])

    gw = batch_of(fit)
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
    del gw
    big = batch_of(nofit)
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_topk_noalloc(big.q_idx, big.w_idx, big.idx_cache, big.batch)
    assert e.value.name == "DSA_ERR_SCRATCH_LIMIT"
