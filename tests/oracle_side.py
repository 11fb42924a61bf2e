"""Oracle-side helpers for the parity tests: build caches and expected values
with the fp64 oracle only (no CUDA path involved), and the comparison rules.

Tolerances (the bars of the method's statement):
* store: dequantised values within one FP8 ulp; scales equal except where
  amax sits on a power-of-two boundary (fp32 vs fp64 LayerNorm/RoPE rounding);
* top-k fed with the oracle's fp32 scores: bit-exact;
* indexer scores: |s_gpu - s| <= 1e-3 * D_j with D_j = sum_m |w_m| |<q_m,k_j>|
  (>= |s_j|); selected sets may differ only at positions whose oracle score is
  within that tolerance of the 2048th score;
* sparse MLA: relative L2 <= 1e-3 and max abs <= 1e-2 against fp64 (fp32
  output), and the same against the oracle rounded to bf16 for bf16 output.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import dsa_oracle as O

SCORE_RTOL = 1e-3
ATTN_REL_L2 = 1e-3
ATTN_MAX_ABS = 1e-2


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_index_cache(num_pages, per_request_raw, positions, slots, boost=None, eps=1e-6, base=10000.0):
    """uint8 [num_pages, 8448] built by the oracle from raw keys.

    per_request_raw: list of fp64 arrays [n_r, 128]; positions / slots: lists of
    int arrays; boost: optional list of bool arrays (x4 on the stored scale).
    """
    cache = np.zeros((num_pages, O.INDEX_PAGE_BYTES), dtype=np.uint8)
    for r, raw in enumerate(per_request_raw):
        codes, scales = O.index_k_prepare(raw, positions[r], eps=eps, rope_base=base)
        if boost is not None:
            scales = np.where(boost[r], scales * 4.0, scales)
        O.index_cache_write(cache, slots[r], codes, scales)
    return cache


def oracle_latent_cache(num_pages, per_request_c, per_request_rope_bits, slots):
    cache = np.zeros((num_pages, O.LATENT_PAGE_BYTES), dtype=np.uint8)
    for r, c in enumerate(per_request_c):
        codes, scales = O.latent_quantize(c)
        O.latent_cache_write(cache, slots[r], codes, scales, per_request_rope_bits[r])
    return cache


def check_scores(gpu: np.ndarray, ref: np.ndarray, mag: np.ndarray, what=""):
    err = np.abs(gpu.astype(np.float64) - ref)
    bad = err > SCORE_RTOL * mag + 1e-30
    assert not bad.any(), (f"{what}: {bad.sum()} scores off; worst rel "
                           f"{np.max(err / np.maximum(mag, 1e-30)):.3e}")


def check_topk_row(gpu_row, ora_row, s_ora, mag, n_valid, what=""):
    gpu_row = np.asarray(gpu_row)
    ora_row = np.asarray(ora_row)
    if n_valid <= O.TOPK:
        assert np.array_equal(gpu_row, ora_row), f"{what}: short-context row differs"
        return 0
    assert np.all(gpu_row >= 0) and np.all(gpu_row < n_valid), f"{what}: index out of range"
    assert np.all(np.diff(gpu_row) > 0), f"{what}: not strictly ascending"
    g, o = set(gpu_row.tolist()), set(ora_row.tolist())
    theta = s_ora[ora_row].min()
    diff = g ^ o
    for j in diff:
        tol = SCORE_RTOL * max(mag[j], mag[ora_row[np.argmin(s_ora[ora_row])]])
        assert abs(s_ora[j] - theta) <= tol, (f"{what}: position {j} (score {s_ora[j]:.6g}) differs but is "
                                             f"not within tolerance of the 2048th score {theta:.6g}")
    return len(diff)


def check_attention(gpu: np.ndarray, ref: np.ndarray, what=""):
    gpu = gpu.astype(np.float64)
    num = np.linalg.norm(gpu - ref)
    den = max(np.linalg.norm(ref), 1e-30)
    mx = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    assert num / den <= ATTN_REL_L2 and mx <= ATTN_MAX_ABS, f"{what}: rel L2 {num / den:.3e}, max abs {mx:.3e}"
    return num / den, mx


def round_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()
