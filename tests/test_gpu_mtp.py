"""GPU parity of top-k reuse across the draft steps of one MTP iteration
("GLM-5.3 推理全链路(十一)", 优化三 and 优化四) against the fp64 oracle.

One MTP layer, B requests, five draft steps: step k holds L0 + k tokens and
queries position L0 - 1 + k.  With reuse on, only the first step runs the
indexer and every step attends with its indices; with reuse off (several draft
candidates per step) every step scores; with a carried seed no step scores.
The caches are built by the oracle for the whole iteration up front.
"""

import math

import numpy as np
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
from oracle import dsa_oracle as O
from synth import Workload, page_table
from tests.oracle_side import (bf16_bits, check_attention, check_topk_row, f64, oracle_index_cache,
                               oracle_latent_cache)

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_STEPS = 5
L0S = [2046, 2100, 3000, 5000]          # the first request crosses the 2048 short-context limit


def _gen(seed):
    return torch.Generator().manual_seed(seed)


@pytest.fixture(scope="module")
def mtp_case():
    B = len(L0S)
    full = [L + N_STEPS - 1 for L in L0S]
    w = Workload("mtp", 8080, full, [N_STEPS] * B, ["full"])
    g = _gen(8080)
    pt = page_table(w, "cpu")
    raw, cs, rs, pos, slots = [], [], [], [], []
    for r, L in enumerate(full):
        raw.append(f64(torch.randn(L, 128, generator=g).to(torch.bfloat16)))
        cs.append(f64(torch.randn(L, 512, generator=g).to(torch.bfloat16)))
        rs.append(torch.randn(L, 64, generator=g).to(torch.bfloat16))
        p = np.arange(L)
        pos.append(p)
        slots.append(pt[r, p // 64].numpy().astype(np.int64) * 64 + p % 64)
    icache = oracle_index_cache(w.num_pages, raw, pos, slots)
    kvcache = oracle_latent_cache(w.num_pages, cs, [bf16_bits(x) for x in rs], slots)
    q_idx = torch.randn(N_STEPS, B, 32, 128, generator=g).to(torch.bfloat16)
    w_idx = torch.randn(N_STEPS, B, 32, generator=g) / math.sqrt(32)
    q_mla = torch.randn(N_STEPS, B, 64, 576, generator=g).to(torch.bfloat16)
    batches = []
    for k in range(N_STEPS):
        seq = torch.tensor([L + k for L in L0S], dtype=torch.int32)
        batches.append(D.Batch(seq.to(DEV), torch.arange(B + 1, dtype=torch.int32).to(DEV), pt.to(DEV), w.num_pages,
                               max_seq_len=max(L0S) + k, max_q_len=1, total_q=B))
    return dict(B=B, pt=pt.numpy(), icache=icache, kvcache=kvcache, q_idx=q_idx, w_idx=w_idx, q_mla=q_mla,
                d_icache=torch.from_numpy(icache.reshape(-1)).to(DEV),
                d_kvcache=torch.from_numpy(kvcache.reshape(-1)).to(DEV),
                d_q_idx=q_idx.to(DEV), d_w_idx=w_idx.to(DEV), d_q_mla=q_mla.to(DEV), batches=batches)


def _oracle_iteration(c, enabled, eagle_topk, seed=None):
    """Per request: the oracle's top-k of every draft step, its scores and
    magnitudes when the step scored, and the attention output of every step."""
    res = []
    for r, L0 in enumerate(L0S):
        st = O.MtpShareState()
        st.begin(enabled, eagle_topk, keep_carry_seed=seed is not None, seed=None if seed is None else seed[r])
        qi, wi = f64(c["q_idx"][:, r]), f64(c["w_idx"][:, r])
        kc, ks = O.index_cache_read(c["icache"], c["pt"][r], L0 + N_STEPS - 1)
        steps = []
        for k in range(N_STEPS):
            L = L0 + k
            scored = st.needs_scoring()
            row, _ = O.mtp_draft_topk(qi[k:k + 1], wi[k:k + 1], c["icache"], c["pt"][r], L, 1, st)
            s = mag = None
            if scored and L > 2048:
                qc, qs = O.index_q_quantize(qi[k])
                s = O.indexer_scores(qc, qs, wi[k], kc[:L], ks[:L])
                mag = O.score_magnitude(qc, qs, wi[k], kc[:L], ks[:L])
            idx = row[0]
            rows = O.latent_cache_read_rows(c["kvcache"], c["pt"][r], np.maximum(idx, 0))
            out, _ = O.sparse_mla(f64(c["q_mla"][k, r]), idx, rows, L - 1)
            steps.append(dict(topk=idx, scored=scored, s=s, mag=mag, n=L, out=out))
        st.end()
        res.append(steps)
    return res


def _gpu_iteration(c, enabled, eagle_topk, seed=None):
    share = D.TopkShare()
    topk = torch.empty(c["B"], 2048, dtype=torch.int32, device=DEV)
    st = D.new_device_status(DEV)
    tk, outs, scored = [], [], []
    with share.mtp_iteration(enabled, eagle_topk, keep_carry_seed=seed is not None, seed=seed) as reuse:
        for k in range(N_STEPS):
            need = share.needs_scoring()
            if need:
                D.dsa_indexer_topk(c["d_q_idx"][k], c["d_w_idx"][k], c["d_icache"], c["batches"][k], topk=topk,
                                   share=share, layer_id=78, dev_status=st)
            scored.append(need)
            p, rows, _ = share.get() if reuse else (topk.data_ptr(), c["B"], 78)
            used = topk if p == topk.data_ptr() else seed
            tk.append(used.clone())
            outs.append(D.dsa_sparse_mla_decode(c["d_q_mla"][k], None if reuse else topk, c["d_kvcache"],
                                                c["batches"][k], share=share if reuse else None,
                                                out_dtype=D.DTYPE_F32, dev_status=st))
    assert D.dsa_device_status_read(st)[0] == 0
    with pytest.raises(D.DsaError):                      # the iteration's indices are gone
        share.get()
    return reuse, scored, [t.cpu().numpy() for t in tk], [o.cpu().numpy() for o in outs]


def _compare(c, ora, gpu_topk, gpu_out, max_diff):
    """Scored rows against the oracle's selection rule (at most max_diff
    positions in all may differ, each within the score tolerance of the cut);
    a reused row is the scored row it carries, so only its attention is
    compared, where that row matched.  Attention everywhere the rows agree."""
    ndiff = 0
    for r in range(c["B"]):
        for k in range(N_STEPS):
            o = ora[r][k]
            if o["s"] is not None:
                d = check_topk_row(gpu_topk[k][r], o["topk"], o["s"], o["mag"], o["n"], what=f"req {r} step {k}")
                ndiff += d
            else:
                d = int(not np.array_equal(gpu_topk[k][r], o["topk"]))
                assert not (o["scored"] and d), f"req {r} step {k}: short-context row differs"
            if d == 0:
                check_attention(gpu_out[k][r], o["out"], what=f"req {r} step {k}")
    assert ndiff <= max_diff


def test_mtp_reuse_scores_once_and_matches_oracle(mtp_case):
    c = mtp_case
    ora = _oracle_iteration(c, True, 1)
    reuse, scored, tk, out = _gpu_iteration(c, True, 1)
    assert reuse and scored == [True] + [False] * (N_STEPS - 1)
    assert [s["scored"] for s in ora[0]] == scored
    for k in range(1, N_STEPS):                          # the carried row, bit for bit
        assert np.array_equal(tk[k], tk[0])
    _compare(c, ora, tk, out, max_diff=2)


def test_mtp_without_reuse_scores_every_step(mtp_case):
    c = mtp_case
    ora = _oracle_iteration(c, True, 3)                  # three draft candidates per step: reuse off
    reuse, scored, tk, out = _gpu_iteration(c, True, 3)
    assert not reuse and scored == [True] * N_STEPS
    _compare(c, ora, tk, out, max_diff=2)


def test_mtp_seed_write_is_a_plain_row_copy():
    g = _gen(17)
    T = 9
    topk = torch.randint(-1, 1 << 20, (T, 2048), generator=g, dtype=torch.int32)
    src = torch.tensor([4, 0, 8, -1, 9, 3], dtype=torch.int32)
    for width in (2048, 2050, 2052):
        st = D.new_device_status(DEV)
        seed = D.dsa_mtp_seed_write(topk.to(DEV), src_row=src.to(DEV), width=width, dev_status=st)
        hs = D.dsa_device_status_read(st)
        assert hs[0] == 4 and hs[1] == 2                   # rows -1 and 9 are out of range
        assert np.array_equal(seed.cpu().numpy(), O.mtp_seed_write(topk.numpy(), src.numpy(), width))
    seed = D.dsa_mtp_seed_write(topk.to(DEV))           # identity rows, default width
    assert torch.equal(seed.cpu(), topk)


def test_mtp_carried_seed_skips_every_indexer(mtp_case):
    c = mtp_case
    seeds = []
    for r, L0 in enumerate(L0S):                          # seeded selections inside each request's first context
        n = L0 - 1
        sel = np.sort(np.random.default_rng(900 + r).choice(n, min(n, 2048), replace=False)).astype(np.int32)
        seeds.append(np.concatenate([sel, np.full(2048 - len(sel), -1, np.int32)]))
    seeds = np.stack(seeds)
    d_seed = D.dsa_mtp_seed_write(torch.from_numpy(seeds).to(DEV))
    ora = _oracle_iteration(c, True, 1, seed=seeds)
    reuse, scored, tk, out = _gpu_iteration(c, True, 1, seed=d_seed)
    assert reuse and scored == [False] * N_STEPS
    assert all(np.array_equal(t, seeds) for t in tk)
    _compare(c, ora, tk, out, max_diff=0)
