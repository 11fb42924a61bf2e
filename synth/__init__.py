"""Seeded synthetic inputs for the DSA attention step.

Shared by the tests and ``bench.py``; it holds none of the method's arithmetic
(no normalisation, rotation, quantisation, scoring or attention): it only draws
the raw tensors a model layer would hand to the step, and lays out the page
tables.  Every tensor comes from ``torch.Generator`` streams seeded from
(workload seed, tensor name), so a workload is reproducible on one device type;
the GPU tests copy what the oracle needs back to the host.

Workloads (sizes and distributions of the DSA decode / verify / prefill shapes):

* ``tiny``      - 1 request, 1 decode token, context 8192, one full layer.
* ``decode32k`` - 64 requests, 1 decode token each, context 32768 +-25 % (uniform),
                  layer group [full, shared, shared, shared]; 1 % of each request's
                  tokens carry an index key boosted x4 after caching.
* ``decode1m``  - 4 requests, 1 decode token each, context 1,048,576, one full layer.
* ``verify64k`` - 128 requests x 6 query tokens (1 + 5 draft), context 65536.
* ``prefill128k`` - 1 request, 8192 new tokens on a 122,880-token prefix.
* ``mtp5_1m``   - one MTP draft iteration: 4 requests, one MTP layer, 5 draft
                  steps; step k holds 1,048,576 + k tokens and queries the last.
                  The 5 draft tokens of a request are its 5 "new" tokens.

Distributions: indexer q ~ N(0,1) bf16 [T,32,128]; head weights ~ N(0,1)/sqrt(32)
fp32 [T,32]; raw index keys ~ N(0,1) bf16 [n,128]; absorbed MLA q ~ N(0,1) bf16
[T,64,576]; latent c ~ N(0,1) bf16 [n,512]; latent RoPE part ~ N(0,1) bf16 [n,64].
Page tables map each request's logical pages onto a seeded random permutation
of the page pool.
"""

from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch

SEED_BASE = 20261202
PAGE = 64


@dataclass
class Workload:
    name: str
    seed: int
    seq_len: list            # tokens per request, including the new query tokens
    q_len: list              # new query tokens per request
    layers: list             # "full" / "shared" per layer of the group
    boost_frac: float = 0.0  # fraction of each request's tokens with a x4 index key
    description: str = ""
    draft_steps: int = 0     # > 0: the new tokens are the draft steps of one MTP iteration
    index_format: str = "fp8"  # index-K cache: "fp8" (132 B/token) or "mxfp4" (68 B/token)

    @property
    def batch(self) -> int:
        return len(self.seq_len)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_len))

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_len))

    @property
    def pages_per_request(self) -> list:
        return [(L + PAGE - 1) // PAGE for L in self.seq_len]

    @property
    def num_pages(self) -> int:
        return int(sum(self.pages_per_request))

    @property
    def max_pages(self) -> int:
        return int(max(self.pages_per_request))

    @property
    def max_seq_len(self) -> int:
        return int(max(self.seq_len))

    @property
    def max_q_len(self) -> int:
        return int(max(self.q_len))


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1000003 + zlib.crc32(name.encode())) % (2 ** 63))
    return g


def workload(name: str, *, batch: int | None = None, ctx: int | None = None) -> Workload:
    """The named workload, optionally shrunk (batch / context) for fast tests."""
    if name == "tiny":
        w = Workload(name, SEED_BASE + 0, [8192], [1], ["full"],
                     description="1 request, 1 decode token, context 8192, one full layer")
    elif name == "decode32k":
        g = _gen(SEED_BASE + 1, "seq_len", "cpu")
        B = 64
        lens = torch.randint(24576, 40960 + 1, (B,), generator=g).tolist()
        w = Workload(name, SEED_BASE + 1, lens, [1] * B,
                     ["full", "shared", "shared", "shared"], boost_frac=0.01,
                     description="64 requests x 1 decode token, context 32768 +-25%, "
                                 "group [full, shared, shared, shared]")
    elif name == "decode1m":
        w = Workload(name, SEED_BASE + 2, [1048576] * 4, [1] * 4, ["full"],
                     description="4 requests x 1 decode token, context 1,048,576, one full layer")
    elif name == "verify64k":
        w = Workload(name, SEED_BASE + 3, [65536] * 128, [6] * 128, ["full"],
                     description="128 requests x 6 verify tokens, context 65536, one full layer")
    elif name == "mtp5_1m":
        n = 5
        w = Workload(name, SEED_BASE + 5, [1048576 + n - 1] * 4, [n] * 4, ["full"], draft_steps=n,
                     description="one MTP iteration: 4 requests x 5 draft steps from a 1,048,576-token context, "
                                 "one MTP layer")
    elif name == "prefill128k":
        w = Workload(name, SEED_BASE + 4, [131072], [8192], ["full"],
                     description="1 request, 8192 new tokens on a 122,880-token prefix")
    else:
        raise KeyError(name)
    if batch is not None:
        w.seq_len = w.seq_len[:batch]
        w.q_len = w.q_len[:batch]
    if ctx is not None:
        # shrink every context proportionally, keeping the ragged mix
        top = max(w.seq_len)
        w.seq_len = [max(q, int(round(L * ctx / top))) for L, q in zip(w.seq_len, w.q_len)]
    return w


def page_table(w: Workload, device) -> torch.Tensor:
    """int32 [B, max_pages]: request r's logical page k -> physical page.

    The pool holds exactly num_pages pages; their order is a seeded random
    permutation.  Unused entries are -1.
    """
    g = _gen(w.seed, "page_perm", "cpu")
    perm = torch.randperm(w.num_pages, generator=g).to(torch.int32)
    pt = torch.full((w.batch, w.max_pages), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(w.pages_per_request):
        pt[r, :n] = perm[off:off + n]
        off += n
    return pt.to(device)


def batch_meta(w: Workload, device) -> dict:
    """seq_len [B], q_start [B+1] (cu-seqlens of query tokens), tok_start [B+1]."""
    seq = torch.tensor(w.seq_len, dtype=torch.int32)
    ql = torch.tensor(w.q_len, dtype=torch.int32)
    q_start = torch.zeros(w.batch + 1, dtype=torch.int32)
    q_start[1:] = torch.cumsum(ql, 0)
    tok_start = torch.zeros(w.batch + 1, dtype=torch.int64)
    tok_start[1:] = torch.cumsum(seq.to(torch.int64), 0)
    return {"seq_len": seq.to(device), "q_start": q_start.to(device), "tok_start": tok_start}


def token_positions_and_slots(w: Workload, pt: torch.Tensor, device, *, which: str = "all"):
    """Positions and cache slots of every cached token, request-major.

    which = "all" | "prefix" (tokens before the new query tokens) | "new".
    Returns (request index [n] int64, position [n] int32, slot [n] int64).
    """
    reqs, poss = [], []
    for r, (L, q) in enumerate(zip(w.seq_len, w.q_len)):
        lo, hi = {"all": (0, L), "prefix": (0, L - q), "new": (L - q, L)}[which]
        poss.append(torch.arange(lo, hi, dtype=torch.int64))
        reqs.append(torch.full((hi - lo,), r, dtype=torch.int64))
    req = torch.cat(reqs)
    pos = torch.cat(poss)
    ptc = pt.to("cpu").to(torch.int64)
    slot = ptc[req, pos // PAGE] * PAGE + pos % PAGE
    return req.to(device), pos.to(torch.int32).to(device), slot.to(device)


def normal_bf16(w: Workload, name: str, shape, device, std: float = 1.0) -> torch.Tensor:
    g = _gen(w.seed, name, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def index_keys(w: Workload, n: int, device, tag: str = "all") -> torch.Tensor:
    """Raw (pre-LayerNorm) index keys, bf16 [n, 128]."""
    return normal_bf16(w, f"idx_k/{tag}", (n, 128), device)


def indexer_query(w: Workload, device):
    """(q bf16 [T,32,128], head weights fp32 [T,32] ~ N(0,1)/sqrt(32))."""
    q = normal_bf16(w, "idx_q", (w.total_q, 32, 128), device)
    g = _gen(w.seed, "idx_w", device)
    wt = torch.randn((w.total_q, 32), generator=g, device=device) / math.sqrt(32.0)
    return q, wt


def latent(w: Workload, layer: int, n: int, device, tag: str = "all"):
    """(c bf16 [n,512], rope bf16 [n,64]) of one layer."""
    return (normal_bf16(w, f"lat_c/{layer}/{tag}", (n, 512), device),
            normal_bf16(w, f"lat_r/{layer}/{tag}", (n, 64), device))


def mla_query(w: Workload, layer: int, device) -> torch.Tensor:
    """Absorbed MLA query bf16 [T, 64, 576]."""
    return normal_bf16(w, f"mla_q/{layer}", (w.total_q, 64, 576), device)


def boost_mask(w: Workload, device) -> torch.Tensor:
    """bool [total_tokens]: the boost_frac of each request's tokens whose cached
    index key is scaled x4 (exactly: its power-of-two scale times 4)."""
    out = torch.zeros(w.total_tokens, dtype=torch.bool)
    if w.boost_frac <= 0:
        return out.to(device)
    g = _gen(w.seed, "boost", "cpu")
    off = 0
    for L in w.seq_len:
        k = max(1, int(round(L * w.boost_frac)))
        idx = torch.randperm(L, generator=g)[:k]
        out[off + idx] = True
        off += L
    return out.to(device)
