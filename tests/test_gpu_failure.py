"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every kernel of the library waits on mbarriers with a wait that gives up after
about a second, writes DSA_ERR_TIMEOUT to the caller's status word and returns.
dsa_bounded_wait_selftest runs that wait on a barrier that gets no arrival (a
flag that nothing sets); the test checks that the status reaches the host, that
the stream and context stay usable, and that the next call of the real path on
the same status word's stream still gives the oracle's answer.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_ratio_gb300 import _binding as B
from deepseek_v4_sparse_ratio_gb300 import inputs
from deepseek_v4_sparse_ratio_gb300.runner import DeviceWorkload

from parity import attention_reference, bf16_to_f64, check_attention, check_selection

pytestmark = pytest.mark.gpu


def test_wait_with_arrival_completes_at_once(dsa):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_bounded_wait_selftest(True, status)
    torch.cuda.synchronize()
    assert status.item() == B.DSA_OK


def test_wait_without_arrival_times_out_and_context_survives(dsa):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    B.dsa_bounded_wait_selftest(False, status)
    torch.cuda.synchronize()                    # the kernel ends on its own
    dt = time.perf_counter() - t0
    assert status.item() == B.DSA_ERR_TIMEOUT
    assert 0.2 < dt < 30.0, dt
    # the first error is kept: a second expiry does not overwrite it
    B.dsa_bounded_wait_selftest(True, status)
    torch.cuda.synchronize()
    assert status.item() == B.DSA_ERR_TIMEOUT

    # the context is still usable: one small chunk of the real path (24 pooled
    # rows > k, so the full score + top-k path), checked against the oracle
    wl = inputs.draw(inputs.small(77, [96], index_topk=8))
    dw = DeviceWorkload(wl, tile_rows=64)
    dw.run_chunk(0)
    torch.cuda.synchronize()
    dw.check_status()
    T = 96
    ref_state = oracle.PoolState(4)
    res = oracle.prefill_chunk(ref_state, wl.t["raw_ik"], wl.t["raw_kv"], 0,
                               wl.t["q_idx"], wl.t["w"].numpy(), wl.t["q"], wl.t["raw_kv"], 0,
                               np.arange(T), wl.index_topk, wl.window, 1.0 / math.sqrt(512))
    check_selection(dw.sel[:T].cpu().numpy(), res["sel"], res["pos"], res["n"], wl.index_topk,
                    res["scores"], res["mag"])
    gsel = dw.sel[:T].cpu().numpy()
    ref = attention_reference(res, gsel, wl.t["q"], wl.t["raw_kv"], 0, ref_state.pooled_kv,
                              wl.window, 1.0 / math.sqrt(512))
    check_attention(bf16_to_f64(dw.out[:T]), ref)
