"""Failure detection on the GPU without a fault: every pipeline wait of the
decode indexer's score kernel is time-bounded and records DSA_DEVERR_TIMEOUT
when it gives up.  With the limit forced to 0 the waits give up at once; the
kernel lets its copies and MMAs in flight land, releases its tensor memory and
returns, the context stays usable, and the next call with the normal limit
matches the oracle.
"""

import numpy as np
import pytest
import torch

import dsa_sparse_attention_indexer_gb300 as D
from tests.oracle_side import check_topk_row
from tests.test_gpu_parity import _build_indexer_case

pytestmark = pytest.mark.gpu
DEV = "cuda"
NORMAL_NS = 2_000_000_000

SEQ = [9000, 3000, 20000, 5000, 2100, 12000]


@pytest.fixture(scope="module")
def case():
    return _build_indexer_case(SEQ, [1] * len(SEQ), 8181)


def test_forced_timeout_is_recorded_without_a_fault_and_the_next_call_is_exact(case):
    c = case
    try:
        D.dsa_debug_set_wait_limit_ns(0)
        for _ in range(3):
            st = D.new_device_status(DEV)
            D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"], dev_status=st)
            torch.cuda.synchronize()                    # raises if the context were lost
            hs = D.dsa_device_status_read(st)
            assert hs[0] & D.DEVERR_TIMEOUT, f"no timeout recorded: {hs}"
    finally:
        D.dsa_debug_set_wait_limit_ns(NORMAL_NS)
    st = D.new_device_status(DEV)
    topk = D.dsa_indexer_topk(c["q"], c["wt"], c["cache"], c["batch"], dev_status=st).cpu().numpy()
    assert D.dsa_device_status_read(st)[0] == 0
    ndiff = 0
    for row in c["rows"]:
        ndiff += check_topk_row(topk[row["i"]], row["topk"], row["s"], row["mag"], row["n"], what=f"row {row['i']}")
    assert ndiff <= 2
