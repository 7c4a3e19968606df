"""Failure detection without a GPU fault: the decode kernels' bounded waits.

Every wait inside the decode kernel gives up after a limit, records PGQA_ETIMEOUT in
dev_status and lets the kernel end, so a stalled producer or a lost arrival never
hangs the GPU. Here the limit is set to 1 ns (pgqa_set_decode_wait_limit_ns): the
consumer warps' first waits for pages still in flight from HBM run out. The call
must report PGQA_ETIMEOUT and the context must stay usable: with the default limit
back and the workspace zero-filled again, the next call matches the oracle."""
import pytest
import torch

import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import DecodeRun, assert_attention_close, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [workloads.llama3_8b_decode,
                                  lambda: workloads.llama70b_decode(cache_dtype="e4m3")])
def test_decode_wait_runs_out_and_reports_timeout(make):
    inp = make()
    run = DecodeRun(inp)
    try:
        pgqa.set_decode_wait_limit_ns(1)
        run.decode()
        torch.cuda.synchronize()
        assert int(run.status.item()) == pgqa.ETIMEOUT
    finally:
        pgqa.set_decode_wait_limit_ns(0)
    # the GPU and the context are fine: a full call on a fresh workspace is correct
    run.status.zero_()
    run.ws.zero_()
    run.decode()
    assert run.status_code() == 0
    ref_out, ref_lse = oracle_decode(inp)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, inp.name + " after a timeout")


def test_default_limit_completes_without_timeout():
    """The same call with the default limit (2 s) never reports a timeout."""
    inp = workloads.llama3_8b_decode()
    run = DecodeRun(inp)
    pgqa.set_decode_wait_limit_ns(0)
    for _ in range(3):
        run.decode()
    assert run.status_code() == 0
