#!/usr/bin/env python
"""Benchmark of the DSA attention step (index-K store -> indexer + top-2048 ->
sparse MLA per layer of a full/shared group) through libdsa.

One step = one pass of the whole path over one batch of synthetic decode
input.  Default workload: 64 requests x 1 decode token, context 32768 +-25 %,
layer group [full, shared, shared, shared].  Metric: query tokens per second
through the group (and us per layer); the roofline is reported for the
dominant call against the measured HBM copy bandwidth.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
requests are independent; no collective on the data path) and rank 0 prints
one JSON line with the whole-job throughput.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "DSA query-tokens/s at 32K-1M ctx; achieved HBM GB/s vs ~8 TB/s peak"
L2_BYTES = 129 * 1024 * 1024

# DRAM traffic per launch from an ncu capture, keyed by (workload, call), with the
# kernel source it was taken on; valid only while that source is unchanged
# (sha256 prefix over the .cu file and every local header it includes).
# All three are full-size captures of dram__bytes_read.sum + dram__bytes_write.sum
# (one pass): the sparse-MLA kernel of decode32k, the score kernel of the decode1m
# and of the verify64k indexer call.
NCU_TRAFFIC = {
    ("decode32k", "sparse_mla_decode"): (105.3e6, "dsa_sparse_attention_indexer_gb300/csrc/mla_tc.cu",
                                         "9fc76894adc7ad04"),
    ("decode1m", "indexer_topk"): (555.7e6, "dsa_sparse_attention_indexer_gb300/csrc/indexer_tc.cu",
                                   "91076d6c62feda2a"),
    ("verify64k", "indexer_topk"): (1405.1e6, "dsa_sparse_attention_indexer_gb300/csrc/indexer_mt.cu",
                                    "0ec2a1c459694845"),
}
FP8_OVER_BF16 = 2.0          # nominal dense tensor rate ratio (4.5 / 2.25 PFLOP/s), used only if the
                             # FP8 GEMM measurement below cannot run


def measure_fp8_tflops(device, n=8192, reps=10):
    """Dense FP8 (E4M3 x E4M3 -> bf16) tensor throughput of this GPU: the
    library GEMM (torch._scaled_mm) on n^3, best of `reps`, CUDA events.  The
    denominator for the indexer's FP8 contraction; None if unavailable."""
    try:
        a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn).t()     # column-major second operand
        one = torch.ones((), device=device)
        for _ in range(3):
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.synchronize()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def file_sha(path):
    """sha256 prefix of a CUDA source and the local headers it includes
    (csrc/ and include/), each once, in first-include order."""
    dirs = [os.path.dirname(os.path.join(ROOT, path)), os.path.join(ROOT, "include")]
    seen, order = set(), []

    def visit(full):
        if full in seen:
            return
        seen.add(full)
        order.append(full)
        with open(full, "rb") as f:
            for line in f.read().decode("utf-8", "replace").splitlines():
                m = re.match(r'\s*#\s*include\s+"([^"]+)"', line)
                if m:
                    for d in dirs:
                        cand = os.path.join(d, m.group(1))
                        if os.path.exists(cand):
                            visit(cand)
                            break

    visit(os.path.join(ROOT, path))
    h = hashlib.sha256()
    for full in order:
        with open(full, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        top = max(sm)
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
def workload_bytes(w, mtp_reuse=True):
    """Algorithmic bytes of one step: index-K read once per request per full
    layer, plus 656 B per selected token per query row per layer.  An MTP
    draft iteration reads index-K in its first step only when the steps reuse
    the top-k, in every step otherwise.  An MXFP4 index cache holds 68 B per
    token instead of 132."""
    tb = 68 if w.index_format == "mxfp4" else 132
    n_full = sum(1 for t in w.layers if t == "full")
    idx = 0
    kv = 0
    for L, q in zip(w.seq_len, w.q_len):
        if w.draft_steps and not mtp_reuse:
            idx += sum(tb * (L - q + t + 1) for t in range(q))
        else:
            idx += tb * (L - q + 1 if w.draft_steps else L)
        for t in range(q):
            kv += 656 * min(2048, L - q + t + 1)
    return n_full * idx, kv * len(w.layers), idx, kv


def _timer(timers, stream, external=False):
    """t(name, fn): runs fn on `stream`, bracketed by timing events kept in
    timers[name] when timers is given.  external=True makes the events
    recordable inside a CUDA graph capture, so a captured step carries its own
    per-call timestamps."""

    def t(name, fn):
        if timers is None:
            fn()
            return
        kw = {"enable_timing": True}
        if external:
            kw["external"] = True
        e0, e1 = torch.cuda.Event(**kw), torch.cuda.Event(**kw)
        e0.record(stream)
        fn()
        e1.record(stream)
        timers.setdefault(name, []).append((e0, e1))
    return t


class Step:
    """All device buffers of one step and the calls that make it up."""

    def __init__(self, gw, D, fused_store=False):
        self.gw = gw
        self.D = D
        self.fused_store = fused_store    # one fused latent (+ index-K) store per layer from raw kv_c / k_pe
        w = gw.w
        dev = gw.device
        self.share = D.TopkShare()
        self.topk = torch.empty((w.total_q, 2048), dtype=torch.int32, device=dev)
        self.idx_ws = D.workspace(D.dsa_indexer_topk_workspace_size(gw.batch), dev)
        self.mla_ws = D.workspace(D.dsa_sparse_mla_workspace_size(gw.batch), dev)
        self.out = {l: torch.empty((w.total_q, 64, 512), dtype=torch.bfloat16, device=dev) for l in gw.layers}
        self.full = [t == "full" for t in w.layers]
        self.launches_per_step = 0

    def run(self, stream, timers=None, before_layer=None, after_layer=None, external=False, before_mla=None):
        """One step on `stream`.  before_layer(l) / before_mla(l) / after_layer(l),
        when given, run just before layer l's first call, just before its sparse
        MLA and just after it (the e2e graph hangs its copies there)."""
        D, gw = self.D, self.gw
        t = _timer(timers, stream, external)

        first_full = True
        for li, l in enumerate(gw.layers):
            if before_layer is not None:
                before_layer(l)
            if self.fused_store:
                t("latent_kv_store", lambda: self._fused(l, self.full[li], stream))
            else:
                if self.full[li]:
                    t("index_k_store", lambda: gw.index_k_store(gw.new_k, gw.new_pos, gw.new_slot, gw.idx_cache,
                                                                     dev_status=gw.dev_status, stream=stream))
                t("latent_kv_store", lambda: D.dsa_latent_kv_store(gw.new_c[l], gw.new_r[l], gw.new_slot,
                                                                     gw.kv_cache[l], dev_status=gw.dev_status,
                                                                     stream=stream))
            if self.full[li]:
                t("indexer_topk", lambda: gw.indexer_topk(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch,
                                                             topk=self.topk, share=self.share, layer_id=l,
                                                             ws=self.idx_ws, dev_status=gw.dev_status,
                                                             stream=stream))
                first_full = False
            if before_mla is not None:
                before_mla(l)
            t("sparse_mla_decode", lambda: D.dsa_sparse_mla_decode(
                gw.q_mla[l], None, gw.kv_cache[l], gw.batch, share=self.share, out=self.out[l], ws=self.mla_ws,
                dev_status=gw.dev_status, stream=stream))
            if after_layer is not None:
                after_layer(l)
        return first_full

    def _fused(self, l, full, stream):
        gw = self.gw
        self.D.dsa_latent_kv_store_fused(gw.new_c[l], gw.new_r[l], gw.new_pos, gw.new_slot, gw.kv_cache[l],
                                         idx_k=gw.new_k if full else None, idxk_cache=gw.idx_cache if full else None,
                                         dev_status=gw.dev_status, stream=stream)

    def e2e_io(self):
        """(inputs needed first, a layer's other inputs, a layer's sparse-MLA
        queries, a layer's output) of the e2e step."""
        gw = self.gw
        first = {"q_idx": gw.q_idx, "w_idx": gw.w_idx, "new_k": gw.new_k, "new_pos": gw.new_pos,
                 "new_slot": gw.new_slot}
        per = {l: {f"c{l}": gw.new_c[l], f"r{l}": gw.new_r[l]} for l in gw.layers}
        mla_q = {l: {f"q{l}": gw.q_mla[l]} for l in gw.layers}
        return first, per, mla_q, self.out

    def calls(self):
        """(name, fn) for every call of one step, in order (for per-call timing)."""
        out = []

        D, gw = self.D, self.gw
        stream = torch.cuda.current_stream()
        for li, l in enumerate(gw.layers):
            if self.fused_store:
                out.append(("latent_kv_store", (lambda l=l, f=self.full[li]: self._fused(l, f, stream))))
            if self.full[li] and not self.fused_store:
                out.append(("index_k_store", lambda: gw.index_k_store(
                    gw.new_k, gw.new_pos, gw.new_slot, gw.idx_cache, dev_status=gw.dev_status, stream=stream)))
            if not self.fused_store:
                out.append(("latent_kv_store", (lambda l=l: D.dsa_latent_kv_store(
                    gw.new_c[l], gw.new_r[l], gw.new_slot, gw.kv_cache[l], dev_status=gw.dev_status,
                    stream=stream))))
            if self.full[li]:
                out.append(("indexer_topk", (lambda l=l: gw.indexer_topk(
                    gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, topk=self.topk, share=self.share, layer_id=l,
                    ws=self.idx_ws, dev_status=gw.dev_status, stream=stream))))
            out.append(("sparse_mla_decode", (lambda l=l: D.dsa_sparse_mla_decode(
                gw.q_mla[l], None, gw.kv_cache[l], gw.batch, share=self.share, out=self.out[l], ws=self.mla_ws,
                dev_status=gw.dev_status, stream=stream))))
        return out


class MtpStep:
    """One MTP draft iteration: the MTP layer runs `draft_steps` times, step k
    on a batch whose requests hold k more tokens than at step 0.  Every step
    stores its draft token's index key and latent row; with reuse on only the
    first step runs the indexer and every step attends with its top-k (the
    share handle's MTP iteration), with reuse off every step scores."""

    def __init__(self, gw, D, reuse=True):
        self.gw = gw
        self.D = D
        self.reuse = reuse
        w = gw.w
        dev = gw.device
        n, B = w.draft_steps, w.batch
        self.n = n
        self.share = D.TopkShare()
        self.topk = torch.empty((B, 2048), dtype=torch.int32, device=dev)
        q0 = torch.arange(B + 1, dtype=torch.int32, device=dev)
        self.batches = []
        for k in range(n):
            seq = gw.seq_len - (n - 1 - k)
            self.batches.append(D.Batch(seq.contiguous(), q0, gw.pt, w.num_pages, max_seq_len=w.max_seq_len - (n - 1 - k),
                                        max_q_len=1, total_q=B))
        self.idx_ws = D.workspace(max(D.dsa_indexer_topk_workspace_size(b) for b in self.batches), dev)
        self.mla_ws = D.workspace(max(D.dsa_sparse_mla_workspace_size(b) for b in self.batches), dev)

        def rows(t, k):                      # draft token k of every request (request-major rows)
            return t.view(B, n, *t.shape[1:])[:, k].contiguous()

        l0 = gw.layers[0]
        self.inp = [{"q_idx": rows(gw.q_idx, k), "w_idx": rows(gw.w_idx, k), "new_k": rows(gw.new_k, k),
                     "new_pos": rows(gw.new_pos, k), "new_slot": rows(gw.new_slot, k), "c": rows(gw.new_c[l0], k),
                     "r": rows(gw.new_r[l0], k), "q_mla": rows(gw.q_mla[l0], k)} for k in range(n)]
        self.kv = gw.kv_cache[l0]
        self.out = {k: torch.empty((B, 64, 512), dtype=torch.bfloat16, device=dev) for k in range(n)}
        self.launches_per_step = 0

    def _store_k(self, k, stream):
        x = self.inp[k]
        self.gw.index_k_store(x["new_k"], x["new_pos"], x["new_slot"], self.gw.idx_cache,
                                 dev_status=self.gw.dev_status, stream=stream)

    def _store_c(self, k, stream):
        x = self.inp[k]
        self.D.dsa_latent_kv_store(x["c"], x["r"], x["new_slot"], self.kv, dev_status=self.gw.dev_status,
                                   stream=stream)

    def _indexer(self, k, stream):
        x = self.inp[k]
        self.gw.indexer_topk(x["q_idx"], x["w_idx"], self.gw.idx_cache, self.batches[k], topk=self.topk,
                                share=self.share, layer_id=0, ws=self.idx_ws, dev_status=self.gw.dev_status,
                                stream=stream)

    def _mla(self, k, stream, topk=None):
        x = self.inp[k]
        self.D.dsa_sparse_mla_decode(x["q_mla"], topk, self.kv, self.batches[k],
                                     share=None if topk is not None else self.share, out=self.out[k],
                                     ws=self.mla_ws, dev_status=self.gw.dev_status, stream=stream)

    def run(self, stream, timers=None, before_layer=None, after_layer=None, external=False, before_mla=None):
        t = _timer(timers, stream, external)

        with self.share.mtp_iteration(enabled=self.reuse, eagle_topk=1):
            for k in range(self.n):
                if before_layer is not None:
                    before_layer(k)
                t("index_k_store", lambda: self._store_k(k, stream))
                t("latent_kv_store", lambda: self._store_c(k, stream))
                if self.share.needs_scoring():
                    t("indexer_topk", lambda: self._indexer(k, stream))
                if before_mla is not None:
                    before_mla(k)
                t("sparse_mla_decode", lambda: self._mla(k, stream))
                if after_layer is not None:
                    after_layer(k)

    def e2e_io(self):
        per = {k: {f"{name}{k}": v for name, v in self.inp[k].items() if name != "q_mla"} for k in range(self.n)}
        mla_q = {k: {f"q_mla{k}": self.inp[k]["q_mla"]} for k in range(self.n)}
        return {}, per, mla_q, self.out

    def calls(self):
        stream = torch.cuda.current_stream()
        out = []
        for k in range(self.n):
            out.append(("index_k_store", (lambda k=k: self._store_k(k, stream))))
            out.append(("latent_kv_store", (lambda k=k: self._store_c(k, stream))))
            if k == 0 or not self.reuse:
                out.append(("indexer_topk", (lambda k=k: self._indexer(k, stream))))
            out.append(("sparse_mla_decode", (lambda k=k: self._mla(k, stream, topk=self.topk))))
        return out


# our kernels per call (the sparse-MLA call also issues one memset of its row counters)
KERNELS_PER_CALL = {"index_k_store": 1, "latent_kv_store": 1, "indexer_topk": 4, "sparse_mla_decode": 1}


def kernels_per_call(name, rows, sms, multi_row=False):
    """Kernels one call launches.  The indexer launches four for a decode batch
    (prep, score, merge filter, merge) and five for a batch with several rows
    per request (FP8: quantisation, plan, score rows, merge filter, merge;
    MXFP4: the virtual decode batch, then the four).  Sparse MLA launches one kernel when its rows are cut into
    clusters of 2 or 4 CTAs or taken whole, and a second, the log-sum-exp
    combine, when CTAs leave partials: the library's split rule, restated."""
    if name == "indexer_topk" and multi_row:
        return 5
    if name != "sparse_mla_decode":
        return KERNELS_PER_CALL[name]
    if rows < sms:
        per = sms // rows
        c = min(per, 22) if per >= 8 else 4 if per >= 4 else 2 if per >= 2 else 1
        ctas = rows * c
    else:
        ctas = sms
    if rows <= ctas:
        c, extra = divmod(ctas, rows)
        return 1 if extra == 0 and c in (1, 2, 4) else 2
    return 2 if rows < 8 * ctas else 1


def call_flops(name, w):
    """Tensor-core FLOPs of one launch of a call: the indexer's FP8 scoring
    (32 heads x 128 dims x 2 per visible token and query row) and sparse MLA's
    fp16 S and P.V (64 heads x (576 + 512) x 2 per selected token and row)."""
    f = 0
    for L, q in zip(w.seq_len, w.q_len):
        for t in range(1 if w.draft_steps else q):          # a draft step's launch has one row per request
            n = L - q + t + 1
            if name == "indexer_topk" and n > 2048:
                f += n * 32 * 128 * 2
            elif name == "sparse_mla_decode":
                f += min(2048, n) * 64 * (576 + 512) * 2
    return f


def call_bytes(name, w):
    """Algorithmic bytes of one launch of a call (a draft step's launch covers
    one of the draft_steps rows of every request)."""
    _, _, idx, kv = workload_bytes(w)
    per = w.draft_steps or 1
    if name == "indexer_topk":
        return idx
    if name == "sparse_mla_decode":
        return kv / per
    if name == "index_k_store":
        return w.total_q * (256 + (68 if w.index_format == "mxfp4" else 132)) / per
    if name == "latent_kv_store":
        return w.total_q * (1152 + 656) / per
    return 0


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over every rank of the job."""
    t_ = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t_, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t_.tolist()]


def job_throughput(rows_per_rank, world, ms):
    """Query rows per second of the whole job: every rank runs its own replica
    of the workload, and the step takes as long as the slowest rank."""
    return rows_per_rank * world / (ms / 1000.0)


# ----------------------------------------------------------------------------
def selection_overlap(gw, D):
    """How much the MXFP4 index-K cache changes the selection: for every query
    row with more than 2048 visible positions, the share of its FP8 top-2048
    that the MXFP4 top-2048 also holds (same keys, queries and weights; the
    other format's cache is stored outside the timed region)."""
    other = gw.other_index_cache()
    fp8, mx = (other, gw.idx_cache) if gw.mx else (gw.idx_cache, other)
    t8 = D.dsa_indexer_topk(gw.q_idx, gw.w_idx, fp8, gw.batch)
    t4 = D.dsa_indexer_topk_mxfp4(gw.q_idx, gw.w_idx, mx, gw.batch)
    w = gw.w
    n_vis = torch.tensor([L - ql + t + 1 for L, ql in zip(w.seq_len, w.q_len) for t in range(ql)],
                         device=t8.device)
    both = torch.sort(torch.cat([t8, t4], 1), 1).values
    common = ((both[:, 1:] == both[:, :-1]) & (both[:, 1:] >= 0)).sum(1).double() / 2048.0
    common = common[n_vis > 2048]
    del other, t8, t4, both
    torch.cuda.empty_cache()
    if common.numel() == 0:
        return {"rows": 0}
    return {"mean": round(float(common.mean()), 4), "min": round(float(common.min()), 4),
            "rows": int(common.numel())}


def scorer_comparison(gw, D, reps=5):
    """Decode batches: device time of the score rows from the tensor-core
    kernel (dsa_indexer_scores) and from the CUDA-core kernel kept to measure
    it against (dsa_indexer_scores_cuda_core), CUDA events, mean of `reps`
    after one warm-up; outside the timed region."""
    w = gw.w
    if max(w.q_len) > 1 or w.draft_steps or gw.mx:
        return None
    out = {}
    sc = torch.empty((w.total_q, w.max_seq_len), dtype=torch.float32, device=gw.device)
    for name, fn in (("tensor_cores", D.dsa_indexer_scores), ("cuda_cores", D.dsa_indexer_scores_cuda_core)):
        fn(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, scores=sc)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn(gw.q_idx, gw.w_idx, gw.idx_cache, gw.batch, scores=sc)
        e1.record()
        torch.cuda.synchronize()
        out[name] = round(e0.elapsed_time(e1) * 1000.0 / reps, 1)
    del sc
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, workload=None, with_e2e=True):
    import dsa_sparse_attention_indexer_gb300 as D
    import synth
    from synth.gpu import GpuWorkload

    dev = f"cuda:{torch.cuda.current_device()}"
    w = synth.workload(workload or args.workload, batch=args.batch, ctx=args.ctx)
    w.index_format = args.index_cache
    gw = GpuWorkload(w, dev)
    step = MtpStep(gw, D, reuse=not args.no_mtp_reuse) if w.draft_steps else Step(gw, D, args.fused_store)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()                      # graphs are captured on a non-default stream
    torch.cuda.set_stream(stream)
    total_bytes = sum(workload_bytes(w, not args.no_mtp_reuse)[:2])
    flush = total_bytes < 4 * L2_BYTES
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None

    # Capture one step (and, separately, each call) into CUDA graphs: decode
    # steps are replayed as graphs, which keeps host launch overhead out of
    # the device timeline.  Two eager runs first do the one-time set-up.
    for _ in range(2):
        step.run(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step.run(stream)
    call_graphs = {}
    for name, fn in step.calls():
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            fn()
        call_graphs.setdefault(name, []).append(g_)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    st = D.dsa_device_status_read(gw.dev_status)
    if st[0] != 0:
        raise RuntimeError(f"device errors during warm-up: {st}")

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    gpu_id = str(getattr(props, "uuid", "0"))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) >= 32:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    if world > 1:
        torch.distributed.barrier()
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if flush:
        tot = 0.0
        for _ in range(args.steps):
            flush_buf.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
        ms = tot / args.steps
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    # Per-call device time, two ways.
    # (a) inside the step: a second capture of the whole step carries timing
    #     events between its calls, so every call is timed where it runs, with
    #     the caches as the step leaves them; averaged over replays.
    # (b) alone and cold: each call's own graph, one replay after a 256 MB
    #     write that evicts L2, averaged over replays.
    reps = max(3, min(args.steps, 20))
    per_call, per_launch, counts = {}, {}, {}
    in_step_ok = True
    try:
        inst_timers = {}
        inst = torch.cuda.CUDAGraph()
        with torch.cuda.graph(inst, stream=stream):
            step.run(stream, timers=inst_timers, external=True)
        torch.cuda.synchronize()
        acc = {k: 0.0 for k in inst_timers}
        for _ in range(reps):
            inst.replay()
            torch.cuda.synchronize()
            for k, evs in inst_timers.items():
                acc[k] += sum(e0.elapsed_time(e1) for e0, e1 in evs)
        for k, evs in inst_timers.items():
            per_call[k] = acc[k] * 1000.0 / reps
            per_launch[k] = per_call[k] / len(evs)
            counts[k] = len(evs)
        del inst
    except Exception:                                  # events not capturable here: time an eager step
        in_step_ok = False
        acc, counts = {}, {}
        for _ in range(reps):
            tm = {}
            step.run(stream, timers=tm)
            torch.cuda.synchronize()
            for k, evs in tm.items():
                acc[k] = acc.get(k, 0.0) + sum(e0.elapsed_time(e1) for e0, e1 in evs)
                counts[k] = len(evs)
        for k in acc:
            per_call[k] = acc[k] * 1000.0 / reps
            per_launch[k] = per_call[k] / counts[k]
    cold_call, cold_launch = {}, {}
    cold_flush = flush_buf if flush_buf is not None else torch.empty(256 * 1024 * 1024, dtype=torch.uint8,
                                                                       device=dev)
    for name, graphs in call_graphs.items():
        tot = 0.0
        for g_ in graphs:
            for _ in range(reps):
                cold_flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g_.replay()
                e1.record(stream)
                e1.synchronize()
                tot += e0.elapsed_time(e1) / reps
        cold_call[name] = tot * 1000.0
        cold_launch[name] = tot * 1000.0 / len(graphs)
    if flush_buf is None:
        del cold_flush
    timers = {k: [None] * len(v) for k, v in call_graphs.items()}
    overlap = selection_overlap(gw, D)
    scorers = scorer_comparison(gw, D)
    if not with_e2e:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        return dict(w=w, ms=ms, per_call=per_call, per_launch=per_launch, cold_call=cold_call,
                    cold_launch=cold_launch, in_step=in_step_ok, clocks=clocks, flush=flush, overlap=overlap,
                    scorers=scorers)

    # ---- end to end: host buffers in, host buffers out, through the same calls
    first_in, layer_in, mla_in, outs = step.e2e_io()
    dev_of = dict(first_in)
    for l in layer_in:
        dev_of.update(layer_in[l])
        dev_of.update(mla_in[l])
    pinned_in = {k: v.cpu().pin_memory() for k, v in dev_of.items()}
    pinned_out = {l: torch.empty(outs[l].shape, dtype=outs[l].dtype).pin_memory() for l in outs}
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pinned_out.values())
    # One e2e step = every input copied in from pinned memory, the step, every
    # layer's output read back, and a host wait for the result.  A copy-in
    # stream brings, in order: the inputs needed first and the first layer's
    # other inputs, then its sparse-MLA queries, then every later layer's
    # inputs.  The compute stream waits for each group just before its first
    # use (the first layer's start, its sparse MLA, the second layer's start):
    # three waits, since every wait between two kernels costs their overlap.
    # A copy-out stream reads each layer's output as soon as its sparse MLA is
    # done.  Captured as one graph like the device-timed step.  First-layer
    # queries larger than L2 are copied after that layer's indexer instead:
    # streamed in during the indexer, they evict the index-K cache that a
    # prefill's row blocks re-read from L2.
    cs_in, cs_out = torch.cuda.Stream(), torch.cuda.Stream()
    layer_ids = list(layer_in)
    groups = [list(first_in) + list(layer_in[layer_ids[0]]), list(mla_in[layer_ids[0]]),
              [k for l in layer_ids[1:] for k in list(layer_in[l]) + list(mla_in[l])]]
    late_q = sum(dev_of[k].numel() * dev_of[k].element_size() for k in groups[1]) > L2_BYTES

    def e2e_step():
        fork = torch.cuda.Event()
        fork.record(stream)
        cs_in.wait_event(fork)
        cs_out.wait_event(fork)
        ready = [torch.cuda.Event() for _ in groups]

        def copy_group(g):
            for k in groups[g]:
                dev_of[k].copy_(pinned_in[k], non_blocking=True)
            ready[g].record(cs_in)

        with torch.cuda.stream(cs_in):
            for g in range(len(groups)):
                if not (late_q and g == 1):
                    copy_group(g)

        def before(l):
            if l == layer_ids[0]:
                stream.wait_event(ready[0])
            elif len(layer_ids) > 1 and l == layer_ids[1]:
                stream.wait_event(ready[2])

        def before_mla(l):
            if l == layer_ids[0]:
                if late_q:                                  # after the first layer's indexer
                    after_idx = torch.cuda.Event()
                    after_idx.record(stream)
                    cs_in.wait_event(after_idx)
                    with torch.cuda.stream(cs_in):
                        copy_group(1)
                stream.wait_event(ready[1])

        def after(l):
            done = torch.cuda.Event()
            done.record(stream)
            cs_out.wait_event(done)
            with torch.cuda.stream(cs_out):
                pinned_out[l].copy_(outs[l], non_blocking=True)

        step.run(stream, before_layer=before, after_layer=after, before_mla=before_mla)
        if len(layer_ids) == 1:
            stream.wait_event(ready[2])                    # (no later layer: nothing left to copy)
        join = torch.cuda.Event()
        join.record(cs_out)
        stream.wait_event(join)

    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_step()
    torch.cuda.synchronize()
    for _ in range(2):
        e2e_graph.replay()
        stream.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_graph.replay()
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1000.0 / e2e_steps

    if world > 1:
        ms, e2e_ms = max_over_ranks([ms, e2e_ms], dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mla_rows = len(w.seq_len) if w.draft_steps else w.total_q     # a draft step's launch: one row per request
    return dict(w=w, ms=ms, e2e_ms=e2e_ms, per_call=per_call, per_launch=per_launch, cold_call=cold_call,
                cold_launch=cold_launch, in_step=in_step_ok, clocks=clocks, flush=flush, h2d=h2d, d2h=d2h,
                overlap=overlap, scorers=scorers,
                launches=sum(kernels_per_call(k, mla_rows, sms, multi_row=max(w.q_len) > 1 and not w.draft_steps)
                             * len(v) for k, v in timers.items()))


# ----------------------------------------------------------------------------
def oracle_sample(w, budget_s: float, max_requests: int = 64, mtp_reuse: bool = True):
    """Time the fp64 oracle on whole requests of the workload until ~budget_s.

    Per request, the inputs are drawn with the same distributions (request-
    scoped seeds); the index cache is built outside the timing (it is resident
    state), and so are the latent rows of the positions the step selects.
    Timed: index-Q quantisation, scoring of every visible position, top-2048,
    and sparse MLA for every layer of the group.  Returns (requests, seconds).
    """
    import synth
    from oracle import dsa_oracle as O

    done, spent = 0, 0.0
    for r in range(min(w.batch, max_requests)):
        L, qn = w.seq_len[r], w.q_len[r]
        npg = (L + 63) // 64
        g = torch.Generator().manual_seed(w.seed * 7919 + r)
        pt = torch.randperm(npg, generator=g).numpy().astype(np.int32)
        pos = np.arange(L)
        slots = pt[pos // 64].astype(np.int64) * 64 + pos % 64
        k = synth.normal_bf16(w, f"idx_k/req{r}", (L, 128), "cpu")
        mx = w.index_format == "mxfp4"
        if mx:
            idx_cache = np.zeros((npg, O.MXFP4_PAGE_BYTES), np.uint8)
            codes, exps = O.index_k_prepare_mxfp4(k.double().numpy(), pos)
            O.mxfp4_cache_write(idx_cache, slots, codes, exps)
        else:
            idx_cache = np.zeros((npg, O.INDEX_PAGE_BYTES), np.uint8)
            codes, scales = O.index_k_prepare(k.double().numpy(), pos)
            O.index_cache_write(idx_cache, slots, codes, scales)
        q_rows = synth.normal_bf16(w, f"idx_q/req{r}", (qn, 32, 128), "cpu").double().numpy()
        wr = (torch.randn((qn, 32), generator=g) / math.sqrt(32.0)).double().numpy()
        t0 = time.perf_counter()
        if w.draft_steps:                                   # one MTP iteration: the draft steps in turn
            st = O.MtpShareState()
            st.begin(mtp_reuse, 1)
            topk, _ = O.mtp_draft_topk(q_rows, wr, idx_cache, pt, L - qn + 1, qn, st)
            st.end()
        elif mx:
            topk, _ = O.request_topk_mxfp4(q_rows, wr, idx_cache, pt, L, qn)
        else:
            topk, _ = O.request_topk(q_rows, wr, idx_cache, pt, L, qn)
        spent += time.perf_counter() - t0
        sel = np.unique(topk[topk >= 0])
        for l in range(len(w.layers)):
            c = synth.normal_bf16(w, f"lat_c/{l}/req{r}", (L, 512), "cpu")[sel].double().numpy()
            rp = synth.normal_bf16(w, f"lat_r/{l}/req{r}", (L, 64), "cpu")[sel].contiguous()
            lc, ls = O.latent_quantize(c)
            cache = np.zeros((npg, O.LATENT_PAGE_BYTES), np.uint8)
            O.latent_cache_write(cache, slots[sel], lc, ls, rp.view(torch.int16).numpy().view(np.uint16))
            qm = synth.normal_bf16(w, f"mla_q/{l}/req{r}", (qn, 64, 576), "cpu").double().numpy()
            t0 = time.perf_counter()
            for t in range(qn):
                rows = O.latent_cache_read_rows(cache, pt, np.maximum(topk[t], 0))
                O.sparse_mla(qm[t], topk[t], rows, L - qn + t)
            spent += time.perf_counter() - t0
        done += 1
        if spent >= budget_s:
            break
    return done, spent


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, on the host cores, on a bounded
    sample of the same workload."""
    import synth
    w = synth.workload(args.workload, batch=args.batch, ctx=args.ctx)
    w.index_format = args.index_cache
    total_q = 0
    t_all = 0.0
    steps_done = 0
    # The NumPy oracle has nothing to warm (no compilation, no device caches), so
    # --warmup adds no passes; at most 3 timed passes keep any --steps within minutes.
    for _ in range(max(1, args.steps if args.steps <= 3 else 3)):
        n, sec = oracle_sample(w, args.ref_budget, mtp_reuse=not args.no_mtp_reuse)
        total_q += sum(w.q_len[:n])
        t_all += sec
        steps_done += 1
    return dict(w=w, value=total_q / t_all, sample=f"{total_q} query rows ({total_q // steps_done} per pass) "
                f"of {w.name}, full indexer + top-k + {len(w.layers)} sparse-MLA layers each", seconds=t_all)


# ----------------------------------------------------------------------------
def roofline(res, pk):
    """The roofline record of a run's dominant call: its algorithmic bytes (or
    tensor FLOPs, when those take longer at the measured peak) per launch over
    the launch's in-step event time, against the measured HBM copy bandwidth
    (or the measured tensor peak of the call's operand type)."""
    w = res["w"]
    dom = max(res["per_call"], key=lambda k: res["per_call"][k])
    dom_us = res["per_launch"][dom]
    dom_bytes = call_bytes(dom, w)
    dom_flops = call_flops(dom, w)
    fp8 = dom == "indexer_topk"
    tensor_peak = pk["fp8_tflops"] if fp8 else pk["bf16_tflops"]
    tensor_bound = dom_flops / (tensor_peak * 1e12) > dom_bytes / (pk["hbm_gbs"] * 1e9)
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": dom_flops / (dom_us * 1e-6) / 1e12, "peak": tensor_peak,
                "unit": "TFLOP/s", "peak_note": ("FP8: " + pk["fp8_source"]) if fp8 else "fp16: measured bf16 burst"}
    else:
        roof = {"bound": "hbm", "achieved": dom_bytes / (dom_us * 1e-6) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    traffic = None
    rec = NCU_TRAFFIC.get((w.name + ("+mxfp4" if w.index_format == "mxfp4" else ""), dom))
    if rec and file_sha(rec[1]) == rec[2]:
        traffic = rec[0]
    cold = res["cold_launch"].get(dom)
    return {"kernel": dom, **roof, "traffic": traffic, "peak_source": pk["source"],
            "algorithmic_bytes_per_launch": dom_bytes, "algorithmic_flops_per_launch": dom_flops,
            "us_per_launch": dom_us, "us_per_launch_alone_l2_flushed": cold,
            "frac_alone_l2_flushed": (roof["frac"] * dom_us / cold) if cold else None}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode32k",
                    choices=["tiny", "decode32k", "decode1m", "verify64k", "prefill128k", "mtp5_1m"])
    ap.add_argument("--batch", type=int, default=None, help="shrink the workload to its first N requests (profiling)")
    ap.add_argument("--ctx", type=int, default=None, help="shrink every context proportionally (profiling)")
    ap.add_argument("--ref-budget", type=float, default=15.0, help="seconds of oracle work per reference pass")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--index-cache", default="fp8", choices=["fp8", "mxfp4"],
                    help="index-K cache format")
    ap.add_argument("--fused-store", action="store_true",
                    help="store each layer's latent row (and, on full layers, the index key) with the fused "
                         "RMSNorm / RoPE call from raw kv_c and k_pe")
    ap.add_argument("--no-mtp-reuse", action="store_true",
                    help="MTP workloads: every draft step runs its own indexer (the comparison point)")
    ap.add_argument("--secondary", default="decode1m",
                    choices=["none", "tiny", "decode32k", "decode1m", "verify64k", "prefill128k", "mtp5_1m"],
                    help="a second workload measured after the headline one and reported in its line's "
                         "'secondary' block (device time and roofline only)")
    args = ap.parse_args()
    if args.index_cache == "mxfp4" and args.workload == "mtp5_1m":
        ap.error("--index-cache mxfp4 covers every workload but mtp5_1m (its draft steps share FP8 selections)")
    if args.fused_store and (args.index_cache == "mxfp4" or args.workload == "mtp5_1m"):
        ap.error("--fused-store writes FP8 index keys in the layer-group step")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, rank, world)
        w = res["w"]
        line = {
            "impl": "reference", "metric": METRIC, "value": res["value"], "unit": "query_tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "batch": w.batch, "q_len": w.q_len[0], "layers": w.layers,
                       "mean_ctx": float(np.mean(w.seq_len))},
            "cpu_baseline": {"value": res["value"], "unit": "query_tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": res["sample"]},
            "e2e": {"value": res["value"], "unit": "query_tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = f"cuda:{torch.cuda.current_device()}"
    pk = peaks()
    fp8_meas = measure_fp8_tflops(dev)
    if fp8_meas is not None:
        pk["fp8_tflops"], pk["fp8_source"] = fp8_meas, "measured (torch._scaled_mm E4M3 8192^3, best of 10)"
    else:
        pk["fp8_tflops"], pk["fp8_source"] = pk["bf16_tflops"] * FP8_OVER_BF16, "measured bf16 x nominal 2"
    res = run_ours(args, rank, world)
    w = res["w"]
    ms = res["ms"]
    idx_b, kv_b, _, _ = workload_bytes(w, not args.no_mtp_reuse)
    step_bytes = idx_b + kv_b
    value = job_throughput(w.total_q, world, ms)
    roof = roofline(res, pk)
    line = {
        "metric": METRIC, "value": value, "unit": "query_tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8-e4m3 cache, fp32/fp16 compute", "data": "synthetic (seeded)",
        "config": {
            "workload": w.name, "description": w.description, "batch": w.batch, "q_len": w.q_len[0],
            "mean_ctx": float(np.mean(w.seq_len)), "layers": w.layers,
            "us_per_layer": ms * 1000.0 / len(w.layers),
            "l2": ("flushed (256 MB write) between timed steps" if res["flush"] else
                   f"inputs larger than L2 ({step_bytes / 1e6:.0f} MB algorithmic bytes per step), no flush"),
            "algorithmic_bytes_per_step": step_bytes,
            "step_hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
            "step_frac_of_measured_hbm": step_bytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "step_frac_of_8tbs": step_bytes / (ms * 1e-3) / 1e9 / 8000.0,
            "us_per_call": {k: round(v, 2) for k, v in res["per_call"].items()},
            "us_per_call_timing": ("events between the calls inside the captured step" if res["in_step"]
                                   else "events between the calls of an eager step"),
            "us_per_launch_alone_l2_flushed": {k: round(v, 2) for k, v in res["cold_launch"].items()},
            **({"draft_steps": w.draft_steps, "mtp_reuse": not args.no_mtp_reuse} if w.draft_steps else {}),
            "index_cache": w.index_format,
            "store": "fused" if args.fused_store else "separate",
            "mxfp4_vs_fp8_topk_overlap": res["overlap"],
            "indexer_score_rows_us": res["scorers"],
        },
        "roofline": roof,
        "peaks": {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"], "source": pk["source"],
                  "fp8_tflops": pk["fp8_tflops"], "fp8_source": pk["fp8_source"]},
        "clocks": res["clocks"],
        "e2e": {"value": job_throughput(w.total_q, world, res["e2e_ms"]), "unit": "query_tokens/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"], "ms_per_step": res["e2e_ms"]},
        "gpu_launches": res["launches"] * args.steps,
    }
    if args.secondary != "none" and args.secondary != w.name:
        del res
        torch.cuda.empty_cache()
        r2 = run_ours(args, rank, world, workload=args.secondary, with_e2e=False)
        w2 = r2["w"]
        b2 = sum(workload_bytes(w2)[:2])
        line["secondary"] = {
            "workload": w2.name, "description": w2.description,
            "value": job_throughput(w2.total_q, world, r2["ms"]), "unit": "query_tokens/s",
            "ms_per_step": r2["ms"], "algorithmic_bytes_per_step": b2,
            "step_hbm_gbs": b2 / (r2["ms"] * 1e-3) / 1e9,
            "step_frac_of_measured_hbm": b2 / (r2["ms"] * 1e-3) / 1e9 / pk["hbm_gbs"],
            "us_per_call": {k: round(v, 2) for k, v in r2["per_call"].items()},
            "us_per_launch_alone_l2_flushed": {k: round(v, 2) for k, v in r2["cold_launch"].items()},
            "roofline": roofline(r2, pk), "clocks": r2["clocks"],
            "mxfp4_vs_fp8_topk_overlap": r2["overlap"],
            "indexer_score_rows_us": r2["scorers"],
        }
    if rank == 0 and not args.no_cpu_baseline:
        n, sec = oracle_sample(w, args.ref_budget, mtp_reuse=not args.no_mtp_reuse)
        qrows = sum(w.q_len[:n])
        line["cpu_baseline"] = {"value": qrows / sec, "unit": "query_tokens/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{n} of {w.batch} requests ({qrows} query rows): indexer over the full "
                                          f"context + top-2048 + {len(w.layers)} sparse-MLA layers, fp64 numpy"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
