"""Failure detection without a GPU fault: a device-side wait on an mbarrier
that nothing arrives at runs out after a short cycle limit (the same bounded
wait the tensor-core kernels use), the kernel reports through the device error
word and returns, and the CUDA context stays usable for the next call."""
import numpy as np
import pytest
import torch

import kda_synth as ks
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import assert_o_close, gpu_chain_outputs, oracle_chains, prefill_device_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    st, code = kda.kda_device_error()   # start from a clear word
    assert st == 0 and code == 0, (st, code)
    kda.kda_check_wait_timeout(1_000_000)   # about 0.5 ms of SM clocks
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    assert kda.STATUS[st] == "KDA_ERR_DEVICE_TIMEOUT" and code == 2, (st, code)
    st, code = kda.kda_device_error()   # reading clears it
    assert st == 0 and code == 0, (st, code)


def test_context_usable_after_a_reported_timeout():
    kda.kda_check_wait_timeout(200_000)
    torch.cuda.synchronize()
    assert kda.kda_device_error()[0] == 4
    w = ks.PrefillWorkload("after_timeout", "bf16", 1, 130, 2, 128, 128, seed=5, s0_std=0.05)
    t = prefill_device_inputs(w, "cuda")
    o, sf = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"])
    torch.cuda.synchronize()
    assert kda.kda_device_error() == (0, 0)
    pairs = [(0, h) for h in range(w.H)]
    o_ref, _ = oracle_chains(w, pairs, None)
    assert_o_close(gpu_chain_outputs(w, o, pairs, None), o_ref, w.dtype)
    assert np.isfinite(sf.cpu().numpy()).all()
