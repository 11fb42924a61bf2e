"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/dsa.h declares, and
reject bad arguments on the host before anything is launched.  Fake device
addresses are never dereferenced on these paths.
"""

import ctypes
import json
import os
import re
import subprocess

import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_constants.json")))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(D.LIB_PATH):
        from dsa_sparse_attention_indexer_gb300 import build
        build.build()
    return D.lib()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**\s*(dsa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", D.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_constants_match_header_and_pages(L):
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    consts = dict(re.findall(r"#define\s+(DSA_\w+)\s+(\d+)", text))
    assert int(consts["DSA_IDXK_TOKEN_BYTES"]) == GOLDEN["index_k_token_bytes"]["value"] == D.IDXK_TOKEN_BYTES
    assert int(consts["DSA_IDXK_PAGE_BYTES"]) == GOLDEN["index_k_page_bytes"]["value"] == D.IDXK_PAGE_BYTES
    assert int(consts["DSA_KV_TOKEN_BYTES"]) == GOLDEN["latent_token_bytes"]["value"] == D.KV_TOKEN_BYTES
    assert int(consts["DSA_PAGE_TOKENS"]) == 64 and int(consts["DSA_TOPK"]) == 2048
    assert int(consts["DSA_KV_PAGE_BYTES"]) == 64 * 656
    assert L.dsa_abi_version() == 1


def test_status_strings(L):
    for code in range(0, 8):
        assert len(D.status_string(code)) > 0
    assert D.status_string(99) == "unknown status"


def _fake_batch(B=2, T=2, max_seq=4096, max_q=1, pages=128):
    fake = 0x10000000
    return D.DsaBatch(B, (max_seq + 63) // 64, max_seq, max_q, T, pages, fake, fake + 256, fake + 512)


def test_store_argument_errors(L):
    s = None
    fk = ctypes.c_void_p(0x20000000)
    assert L.dsa_index_k_store(None, fk, fk, 1, None, None, 1e-6, 1e4, fk, 1, None, s) == 1
    assert L.dsa_index_k_store(fk, fk, fk, -1, None, None, 1e-6, 1e4, fk, 1, None, s) == 1
    assert L.dsa_index_k_store(fk, fk, fk, 0, None, None, 1e-6, 1e4, fk, 1, None, s) == 0   # nothing to do
    odd = ctypes.c_void_p(0x20000001)
    assert L.dsa_index_k_store(odd, fk, fk, 1, None, None, 1e-6, 1e4, fk, 1, None, s) == 2
    assert L.dsa_index_k_store(fk, fk, fk, 1, None, None, 1e-6, -1.0, fk, 1, None, s) == 1
    assert L.dsa_latent_kv_store(fk, None, fk, 1, fk, 1, None, s) == 1
    assert L.dsa_latent_kv_store(fk, fk, fk, 1, odd, 1, None, s) == 2


def test_batch_validation_and_workspace_sizes(L):
    n = ctypes.c_size_t(0)
    b = _fake_batch()
    assert L.dsa_indexer_topk_workspace_size(ctypes.byref(b), ctypes.byref(n)) == 0 and n.value > 0
    assert L.dsa_sparse_mla_workspace_size(ctypes.byref(b), ctypes.byref(n)) == 0
    assert L.dsa_indexer_scores_workspace_size(ctypes.byref(b), ctypes.byref(n)) == 0
    assert n.value >= 2 * (4096 + 128) and n.value % 256 == 0      # quantised q + the row-block plan
    assert L.dsa_indexer_topk_workspace_size(None, ctypes.byref(n)) == 1
    bad = _fake_batch()
    bad.max_pages = 1                                   # 64 tokens cannot hold max_seq_len
    assert L.dsa_indexer_topk_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1
    bad = _fake_batch(T=5, max_q=1)                     # T > B * max_q_len
    assert L.dsa_indexer_topk_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1
    bad = _fake_batch()
    bad.seq_len = None
    assert L.dsa_indexer_topk_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1


def test_indexer_and_mla_argument_errors(L):
    fk = ctypes.c_void_p(0x30000000)
    odd = ctypes.c_void_p(0x30000004)
    b = _fake_batch()
    ws = ctypes.c_void_p(0x40000000)
    # null query / unaligned cache / missing workspace
    assert L.dsa_indexer_topk(None, fk, fk, ctypes.byref(b), fk, None, None, 0, ws, 1 << 30, None, None) == 1
    assert L.dsa_indexer_topk(fk, fk, odd, ctypes.byref(b), fk, None, None, 0, ws, 1 << 30, None, None) == 2
    assert L.dsa_indexer_topk(fk, fk, fk, ctypes.byref(b), fk, None, None, 0, ws, 16, None, None) == 4
    # sparse MLA: bad dtype, bad scale, shared layer without a published top-k
    assert L.dsa_sparse_mla_decode(fk, fk, None, fk, ctypes.byref(b), 0.0625, fk, 7, None, ws, 1 << 30, None, None) == 1
    assert L.dsa_sparse_mla_decode(fk, fk, None, fk, ctypes.byref(b), -1.0, fk, 0, None, ws, 1 << 30, None, None) == 1
    share = ctypes.c_void_p()
    assert L.dsa_topk_share_create(ctypes.byref(share)) == 0
    assert L.dsa_sparse_mla_decode(fk, None, share, fk, ctypes.byref(b), 0.0625, fk, 0, None, ws, 1 << 30,
                                   None, None) == 5
    assert L.dsa_sparse_mla_prefill(fk, None, None, fk, ctypes.byref(b), 0.0625, fk, 0, None, ws, 1 << 30,
                                    None, None) == 1
    assert L.dsa_topk_share_destroy(share) == 0
    # top-k from scores: ld < max_len
    assert L.dsa_topk_from_scores(fk, 10, fk, 1, 20, fk, None, 0, None) == 1
    assert L.dsa_topk_from_scores(fk, 10, fk, 0, 10, fk, None, 0, None) == 0      # zero rows: no launch


def test_calls_over_zero_rows_launch_nothing(L):
    """A batch whose requests bring no query rows: every call returns DSA_OK
    with NULL buffers, and an indexer call still publishes its empty top-k to
    a share handle (a shared layer before any full layer is still an error)."""
    b = ctypes.byref(_fake_batch(B=2, T=0))
    N = None
    assert L.dsa_indexer_topk(N, N, N, b, N, N, N, 0, N, 0, N, N) == 0
    assert L.dsa_indexer_topk_mxfp4(N, N, N, b, N, N, N, 0, N, 0, N, N) == 0
    assert L.dsa_indexer_topk_noalloc(N, N, N, b, N, N, N, 0, N, N) == 0
    assert L.dsa_indexer_scores(N, N, N, b, N, 0, N, 0, N, N) == 0
    assert L.dsa_indexer_scores_cuda_core(N, N, N, b, N, 0, N, 0, N, N) == 0
    share = ctypes.c_void_p()
    assert L.dsa_topk_share_create(ctypes.byref(share)) == 0
    assert L.dsa_sparse_mla_decode(N, N, share, N, b, 0.0625, N, 0, N, N, 0, N, N) == 5   # no full layer yet
    assert L.dsa_indexer_topk(N, N, N, b, N, N, share, 0, N, 0, N, N) == 0               # publishes 0 rows
    assert L.dsa_sparse_mla_decode(N, N, share, N, b, 0.0625, N, 0, N, N, 0, N, N) == 0
    assert L.dsa_sparse_mla_prefill(N, N, share, N, b, 0.0625, N, 1, N, N, 0, N, N) == 0
    assert L.dsa_topk_share_destroy(share) == 0
    # zero tokens or rows in the calls that take a count
    assert L.dsa_index_k_store(N, N, N, 0, N, N, 1e-6, 1e4, N, 1, N, N) == 0
    assert L.dsa_latent_kv_store(N, N, N, 0, N, 1, N, N) == 0
    assert L.dsa_topk_from_scores(N, 0, N, 0, 0, N, N, 0, N) == 0


def test_cuda_core_scorer_and_mxfp4_rows_argument_errors(L):
    fk = ctypes.c_void_p(0x30000000)
    ws = ctypes.c_void_p(0x40000000)
    b = _fake_batch()
    assert L.dsa_indexer_scores_cuda_core(None, fk, fk, ctypes.byref(b), fk, 4096, ws, 1 << 20, None, None) == 1
    assert L.dsa_indexer_scores_cuda_core(fk, fk, fk, ctypes.byref(b), fk, 100, ws, 1 << 20, None, None) == 1   # ld
    assert L.dsa_indexer_scores_cuda_core(fk, fk, fk, ctypes.byref(b), fk, 4096, ws, 16, None, None) == 4
    multi = _fake_batch(B=2, T=4, max_q=2)
    assert L.dsa_indexer_scores_cuda_core(fk, fk, fk, ctypes.byref(multi), fk, 4096, ws, 1 << 20, None, None) == 3
    # MXFP4 with several rows per request: at most 65535 rows (each becomes a one-row request)
    big = _fake_batch(B=1, T=70000, max_q=70000, max_seq=80000, pages=2000)
    assert L.dsa_indexer_topk_mxfp4(fk, fk, fk, ctypes.byref(big), fk, None, None, 0, ws, 1 << 40, None, None) == 3
    assert L.dsa_debug_set_wait_limit_ns(2_000_000_000) == 0


def test_context_parallel_argument_errors(L):
    fk = ctypes.c_void_p(0x30000000)
    odd = ctypes.c_void_p(0x30000004)
    # merge: rank count outside 1..8, null inputs, unaligned lists; zero rows launch nothing
    assert L.dsa_cp_topk_merge(fk, fk, fk, 0, 4, fk, None, None, None) == 1
    assert L.dsa_cp_topk_merge(fk, fk, fk, 9, 4, fk, None, None, None) == 1
    assert L.dsa_cp_topk_merge(None, fk, fk, 2, 4, fk, None, None, None) == 1
    assert L.dsa_cp_topk_merge(odd, fk, fk, 2, 4, fk, None, None, None) == 2
    assert L.dsa_cp_topk_merge(fk, fk, fk, 2, 0, fk, None, None, None) == 0
    # localize: in place is refused; negative rows
    assert L.dsa_cp_topk_localize(fk, 4, fk, fk, fk, None) == 1
    assert L.dsa_cp_topk_localize(fk, -1, fk, fk, ctypes.c_void_p(0x31000000), None) == 1
    assert L.dsa_cp_topk_localize(fk, 0, fk, fk, ctypes.c_void_p(0x31000000), None) == 0
    # attention merge: bad dtype, null parts, unaligned output
    assert L.dsa_cp_attention_merge(fk, fk, 2, 4, fk, 7, None, None) == 1
    assert L.dsa_cp_attention_merge(None, fk, 2, 4, fk, 0, None, None) == 1
    assert L.dsa_cp_attention_merge(fk, fk, 2, 4, odd, 0, None, None) == 2
    assert L.dsa_cp_attention_merge(fk, fk, 2, 0, fk, 0, None, None) == 0


def test_schedule_parser_and_freq_rule(L):
    full = GOLDEN["full_layers"]["value"]
    types = ["full" if l in full else "shared" for l in range(78)]
    is_full = D.dsa_parse_indexer_types(types)
    assert sum(is_full) == 21 and len(is_full) - sum(is_full) == 57
    assert [l for l in range(78) if is_full[l]] == full
    assert D.dsa_schedule_from_freq(78, 4, 3) == is_full
    # the vLLM default offset 2 differs at layers 2 and 3 (full/shared swap)
    v = D.dsa_schedule_from_freq(78, 4, 2)
    assert v[:4] == [True, True, False, False] or v[:4] == [True, True, False, True]
    with pytest.raises(D.DsaError):
        D.dsa_parse_indexer_types(["full", "sparse"])


def test_schedule_resolve_matches_the_oracle_chain(L):
    from oracle import dsa_oracle as O
    import random
    rng = random.Random(5)
    for trial in range(300):
        n = rng.randint(0, 90)
        kw = {}
        if rng.random() < 0.3:
            kw["indexer_types"] = [rng.choice(["full", "shared"]) for _ in range(rng.randint(0, 90))]
        if rng.random() < 0.4:
            kw["cli_factor"] = rng.randint(0, 5)
        if rng.random() < 0.4:
            kw["index_topk_pattern"] = "".join(rng.choice("FS") for _ in range(rng.randint(0, 90)))
        kw["index_topk_freq"] = rng.randint(1, 6)
        if rng.random() < 0.6:
            kw["index_skip_topk_offset"] = rng.randint(0, 5)
        got = D.dsa_schedule_resolve(n, **kw)
        want = [not O.layer_skips_topk_config(l, **kw) for l in range(n)]
        assert got == want, (trial, kw)
    with pytest.raises(D.DsaError):
        D.dsa_schedule_resolve(4, indexer_types=["full", "fuII"])
    with pytest.raises(D.DsaError):
        D.dsa_schedule_resolve(4, index_topk_freq=0)


def test_share_handle_lifecycle(L):
    s = D.TopkShare()
    with pytest.raises(D.DsaError) as e:
        s.get()
    assert e.value.code == 5
    # the handle only records the pointer: publish a fake one through the C call
    assert L.dsa_topk_share_publish(s.handle, 6, ctypes.c_void_p(0x50000000), 7) == 0
    assert s.get() == (0x50000000, 7, 6)
    s.reset()
    with pytest.raises(D.DsaError):
        s.get()


def test_mtp_share_state_follows_the_iteration_rules(L):
    """The host-only MTP calls take the same decisions as the oracle's share
    state, step by step (no device memory is touched)."""
    from oracle import dsa_oracle as O
    h = ctypes.c_void_p()
    assert L.dsa_topk_share_create(ctypes.byref(h)) == 0
    fake_topk, fake_seed = ctypes.c_void_p(0x50000000), ctypes.c_void_p(0x60000000)
    on, needs = ctypes.c_int32(), ctypes.c_int32()
    p, rows, lid = ctypes.c_void_p(), ctypes.c_int64(), ctypes.c_int32()

    def needs_scoring():
        assert L.dsa_topk_share_needs_scoring(h, ctypes.byref(needs)) == 0
        return bool(needs.value)

    cases = [(1, 1, 0, None), (1, 3, 0, None), (0, 1, 0, None), (1, 1, 1, fake_seed), (1, 1, 0, fake_seed),
             (1, 2, 1, fake_seed)]
    for enabled, etk, keep, seed in cases:
        ora = O.MtpShareState()
        ora_on = ora.begin(bool(enabled), etk, bool(keep), None if seed is None else [7])
        assert L.dsa_topk_share_mtp_begin(h, enabled, etk, keep, seed, 3, 2048, ctypes.byref(on)) == 0
        assert bool(on.value) == ora_on
        for step in range(3):
            assert needs_scoring() == ora.needs_scoring()
            if ora.needs_scoring():                # the step runs the indexer, which publishes
                if ora.reuse:
                    ora.publish([step])
                assert L.dsa_topk_share_publish(h, 78, fake_topk, 3) == 0
            else:
                assert L.dsa_topk_share_get(h, ctypes.byref(p), ctypes.byref(rows), ctypes.byref(lid)) == 0
                assert p.value == (fake_seed.value if keep and seed is not None else fake_topk.value)
        assert L.dsa_topk_share_mtp_end(h) == 0
        ora.end()
        assert needs_scoring() and L.dsa_topk_share_get(h, ctypes.byref(p), None, None) == 5
    # argument errors
    assert L.dsa_topk_share_mtp_begin(h, 1, 0, 0, None, 0, 0, None) == 1           # eagle topk < 1
    assert L.dsa_topk_share_mtp_begin(h, 1, 1, 1, fake_seed, 3, 2051, None) == 3   # kpool tail not consumable
    assert L.dsa_topk_share_mtp_begin(h, 1, 5, 1, fake_seed, 3, 2051, ctypes.byref(on)) == 0 and on.value == 0
    assert L.dsa_topk_share_needs_scoring(h, None) == 1
    assert L.dsa_topk_share_destroy(h) == 0
    w = ctypes.c_int32()
    assert L.dsa_mtp_topk_width(2048, 1, ctypes.byref(w)) == 0 and w.value == GOLDEN["mtp_seed_width"]["value"]
    assert L.dsa_mtp_topk_width(2048, 4, ctypes.byref(w)) == 0 and w.value == 2051
    assert L.dsa_mtp_topk_width(0, 1, ctypes.byref(w)) == 1
    fk = ctypes.c_void_p(0x70000000)
    assert L.dsa_mtp_seed_write(fk, 4, None, 4, fk, 2047, None, None) == 1          # width below 2048
    assert L.dsa_mtp_seed_write(fk, 4, None, -1, fk, 2048, None, None) == 1
    assert L.dsa_mtp_seed_write(fk, 4, None, 0, fk, 2048, None, None) == 0          # nothing to do
    assert L.dsa_mtp_seed_write(ctypes.c_void_p(0x70000004), 4, None, 4, fk, 2048, None, None) == 2


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(D, "_lib", None)
    monkeypatch.setattr(D, "LIB_PATH", "/nonexistent/libdsa.so")
    with pytest.raises(D.DsaLibraryMissing):
        D.lib()


def test_binding_rejects_host_tensors_and_wrong_dtypes():
    # the library reads and writes through raw device pointers: a host tensor or
    # a wrong element type is refused in the binding, before any call into it
    bf = torch.zeros(4, 128, dtype=torch.bfloat16)
    i32 = torch.zeros(4, dtype=torch.int32)
    i64 = torch.zeros(4, dtype=torch.int64)
    u8 = torch.zeros(8448, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        D.dsa_index_k_store(bf, i32, i64, u8)
    with pytest.raises(TypeError, match="torch.bfloat16"):
        D.dsa_index_k_store(bf.float(), i32, i64, u8)
    with pytest.raises(ValueError, match="contiguous"):
        D.dsa_index_k_store(bf.t(), i32, i64, u8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        D.Batch(i32, torch.zeros(5, dtype=torch.int32), torch.zeros(4, 2, dtype=torch.int32), 8,
                max_seq_len=128, max_q_len=1, total_q=4)
    with pytest.raises(ValueError, match="CUDA tensor"):
        D.dsa_topk_from_scores(torch.zeros(2, 4096), torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        D.dsa_device_status_read(torch.zeros(4, dtype=torch.int32))


def test_decode_workspace_follows_the_header_formula(L):
    # dsa.h gives the decode indexer's scratch for T = B rows on S SMs as
    #   round_up(4224 T, 256) + 16384 T + (S + B) * 36884 + 12 (B + 1) + 8 S
    # plus at most 768 bytes of alignment; the workspace call sizes it for
    # S = 1024, so its answer must fall in that window
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dsa.h")).read()
    per_seg = int(re.search(r"\(S \+ B\) \* (\d+)", text).group(1))
    n = ctypes.c_size_t(0)
    for B in (1, 4, 64, 151, 300, 1000):
        b = _fake_batch(B=B, T=B, max_q=1)
        assert L.dsa_indexer_topk_workspace_size(ctypes.byref(b), ctypes.byref(n)) == 0
        S = 1024
        base = (4224 * B + 255) // 256 * 256 + 16384 * B + (S + B) * per_seg + 12 * (B + 1) + 8 * S
        assert base <= n.value <= base + 768, (B, n.value - base)
    # and the row limit the header states for 152 SMs follows from it, alignment included
    fit, nofit = (int(x) for x in re.search(r"\((\d+) rows fit at S = 152, (\d+) do", text).groups())
    need = lambda B: (4224 * B + 255) // 256 * 256 + 16384 * B + (152 + B) * per_seg + 12 * (B + 1) + 8 * 152
    assert nofit == fit + 1
    assert need(fit) + 768 <= 16 << 20 < need(nofit)
