"""Device-side set-up of a synthetic workload.

Draws the raw inputs with ``synth`` on the GPU and fills the paged caches of the
cached prefix through the library's own store calls (the caches are the step's
resident state).  Returns everything one step of the DSA path needs.
"""

from __future__ import annotations

import torch

import dsa_sparse_attention_indexer_gb300 as D

from . import (PAGE, Workload, batch_meta, boost_mask, index_keys, indexer_query, latent, mla_query,
               page_table, token_positions_and_slots)


class GpuWorkload:
    """Caches, batch descriptor and per-step inputs of one workload on `device`.

    store_new=True also writes the new query tokens into the caches (so the
    caches are complete without running a step); the step writes them again.
    """

    def __init__(self, w: Workload, device="cuda", *, store_new: bool = True, layers=None,
                 chunk_tokens: int = 1 << 22):
        self.w = w
        self.device = device
        self._D = D
        self.layers = list(range(len(w.layers))) if layers is None else list(layers)
        self.pt = page_table(w, device)
        meta = batch_meta(w, device)
        self.seq_len, self.q_start = meta["seq_len"], meta["q_start"]
        self.tok_start = meta["tok_start"]
        self.batch = D.Batch(self.seq_len, self.q_start, self.pt, w.num_pages, max_seq_len=w.max_seq_len,
                             max_q_len=w.max_q_len, total_q=w.total_q)
        self.dev_status = D.new_device_status(device)
        self.mx = w.index_format == "mxfp4"
        self.idx_page_bytes = D.IDXK_MXFP4_PAGE_BYTES if self.mx else D.IDXK_PAGE_BYTES
        self.idx_cache = torch.zeros(w.num_pages * self.idx_page_bytes, dtype=torch.uint8, device=device)
        self.index_k_store = D.dsa_index_k_store_mxfp4 if self.mx else D.dsa_index_k_store
        self.indexer_topk = D.dsa_indexer_topk_mxfp4 if self.mx else D.dsa_indexer_topk
        self.kv_cache = {l: torch.zeros(w.num_pages * D.KV_PAGE_BYTES, dtype=torch.uint8, device=device)
                         for l in self.layers}
        which = "all" if store_new else "prefix"
        req, pos, slot = token_positions_and_slots(w, self.pt, device, which="all")
        keep = torch.ones_like(pos, dtype=torch.bool)
        if not store_new:
            keep = pos < (self.seq_len.to(torch.int64)[req] - torch.tensor(w.q_len, device=device)[req])
        self.all_pos, self.all_slot = pos, slot
        n = pos.numel()
        k_all = index_keys(w, n, device)
        for a in range(0, n, chunk_tokens):
            b_ = min(n, a + chunk_tokens)
            sl = torch.where(keep[a:b_], slot[a:b_], torch.full_like(slot[a:b_], -1))
            self.index_k_store(k_all[a:b_], pos[a:b_].contiguous(), sl.contiguous(), self.idx_cache,
                                dev_status=self.dev_status)
        del k_all
        if w.boost_frac > 0:
            bm = boost_mask(w, device)
            bs = slot[bm]
            if self.mx:                                    # x4: every block exponent + 2
                sv = self.idx_cache.view(-1, self.idx_page_bytes)[:, 64 * 64:].view(-1, PAGE, 4)
                sv[bs // PAGE, bs % PAGE] += 2
            else:
                sv = D.index_cache_scale_view(self.idx_cache)
                sv[bs // PAGE, bs % PAGE] *= 4.0
        for l in self.layers:
            c_all, r_all = latent(w, l, n, device)
            for a in range(0, n, chunk_tokens):
                b_ = min(n, a + chunk_tokens)
                sl = torch.where(keep[a:b_], slot[a:b_], torch.full_like(slot[a:b_], -1))
                D.dsa_latent_kv_store(c_all[a:b_], r_all[a:b_], sl.contiguous(), self.kv_cache[l],
                                      dev_status=self.dev_status)
            del c_all, r_all
        # per-step inputs: the new tokens' raw keys / latents and the queries
        nreq, npos, nslot = token_positions_and_slots(w, self.pt, device, which="new")
        self.new_pos, self.new_slot = npos.contiguous(), nslot.contiguous()
        new_rows = (self.tok_start.to(device)[nreq] + npos.to(torch.int64))
        self.new_rows = new_rows
        self.new_k = index_keys(w, n, device)[new_rows].contiguous()
        self.new_c, self.new_r = {}, {}
        for l in self.layers:
            c_all, r_all = latent(w, l, n, device)
            self.new_c[l] = c_all[new_rows].contiguous()
            self.new_r[l] = r_all[new_rows].contiguous()
            del c_all, r_all
        self.q_idx, self.w_idx = indexer_query(w, device)
        self.q_mla = {l: mla_query(w, l, device) for l in self.layers}
        torch.cuda.synchronize()
        st = D.dsa_device_status_read(self.dev_status)
        if st[0] != 0:
            raise RuntimeError(f"device errors while filling caches: {st}")

    def other_index_cache(self, chunk_tokens: int = 1 << 22) -> torch.Tensor:
        """The index-K cache of the same keys (and boosts) in the other format
        (MXFP4 for an FP8 workload, FP8 for an MXFP4 one), through the
        library's own store."""
        D, w = self._D, self.w
        mx = not self.mx
        pb = D.IDXK_MXFP4_PAGE_BYTES if mx else D.IDXK_PAGE_BYTES
        cache = torch.zeros(w.num_pages * pb, dtype=torch.uint8, device=self.device)
        store = D.dsa_index_k_store_mxfp4 if mx else D.dsa_index_k_store
        n = self.all_pos.numel()
        k_all = index_keys(w, n, self.device)
        for a in range(0, n, chunk_tokens):
            b_ = min(n, a + chunk_tokens)
            store(k_all[a:b_], self.all_pos[a:b_].contiguous(), self.all_slot[a:b_].contiguous(), cache,
                  dev_status=self.dev_status)
        del k_all
        if w.boost_frac > 0:
            bs = self.all_slot[boost_mask(w, self.device)]
            if mx:
                sv = cache.view(-1, pb)[:, 64 * 64:].view(-1, PAGE, 4)
                sv[bs // PAGE, bs % PAGE] += 2
            else:
                sv = D.index_cache_scale_view(cache)
                sv[bs // PAGE, bs % PAGE] *= 4.0
        torch.cuda.synchronize()
        return cache

    # raw host copies for the oracle ------------------------------------------
    def request_rows(self, r: int):
        a, b = int(self.tok_start[r]), int(self.tok_start[r + 1])
        return a, b

    def raw_index_keys(self, r: int) -> torch.Tensor:
        a, b = self.request_rows(r)
        return index_keys(self.w, self.all_pos.numel(), self.device)[a:b].cpu()

    def raw_latent(self, l: int, r: int, positions=None):
        a, b = self.request_rows(r)
        c_all, r_all = latent(self.w, l, self.all_pos.numel(), self.device)
        if positions is None:
            return c_all[a:b].cpu(), r_all[a:b].cpu()
        idx = torch.as_tensor(positions, dtype=torch.int64, device=self.device) + a
        return c_all[idx].cpu(), r_all[idx].cpu()

    def boosted(self, r: int) -> torch.Tensor:
        a, b = self.request_rows(r)
        return boost_mask(self.w, "cpu")[a:b]
