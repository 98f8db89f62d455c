"""The allocation-free prefill entry point, kda_chunk_fwd_noalloc.

It serves callers that cannot call cudaMalloc (for example a serving engine
that reserved nearly all device memory up front): the scratch space lives in a
fixed array inside the library instead of a caller-provided workspace.  These
tests call it through the C ABI and check it against kda_chunk_fwd, the
entry point with a caller-provided workspace, on two calls in a row with
different problems: the results must be bit-identical (the same kernels run
on the same inputs), so the second call cannot depend on what the first left
in the shared array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import kda_synth as ks
import linear_attention_recurrence_chunk_gb300 as kda


def _fn(lib):
    f = lib.kda_chunk_fwd_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, ctypes.c_int, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def test_noalloc_rejects_problems_larger_than_its_scratch():
    """A problem needing more than the fixed scratch size is refused on the
    host, before any device work (so this runs without a GPU)."""
    lib = kda.load_library()
    f = _fn(lib)
    fake = 1 << 40
    st = f(fake, fake + (1 << 33), fake + (2 << 33), fake + (3 << 33), fake + (4 << 33), None, None, 1, 1, 1 << 20,
           32, 128, 128, 1, fake + (5 << 33), None, None)
    assert st == 1
    assert lib.kda_chunk_fwd_workspace_size(1, 1 << 20, 32, 128, 128, 1, 1) > 64 * 1024 * 1024


def test_noalloc_status_order_matches_chunk_fwd():
    """Invalid and unsupported shapes get the status kda_chunk_fwd gives them
    (an invalid dtype or shape is KDA_ERR_INVALID_ARG before an unsupported
    head size is KDA_ERR_UNSUPPORTED); host-side checks only, nothing runs."""
    lib = kda.load_library()
    f = _fn(lib)
    g = lib.kda_chunk_fwd
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    g.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, ctypes.c_int, vp, vp, vp, ctypes.c_size_t,
                  vp]
    g.restype = ctypes.c_int
    fake = 1 << 40
    ptrs = [fake, fake + (1 << 33), fake + (2 << 33), fake + (3 << 33), fake + (4 << 33), None, None]
    cases = [  # (num_seqs, B, T, H, d_k, d_v, dtype)
        (1, 1, 64, 2, 96, 128, 7),      # invalid dtype and unsupported d_k
        (1, 1, 64, 2, 128, 128, 7),     # invalid dtype
        (2, 1, 64, 2, 96, 128, 1),      # num_seqs != B without cu_seqlens, unsupported d_k
        (1, 1, -1, 2, 128, 128, 1),     # negative T
        (1, 1, 64, 2, 96, 128, 1),      # unsupported d_k only
        (1, 1, 64, 0, 128, 128, 1),     # H = 0
    ]
    for ns, B, T, H, dk, dv, dt in cases:
        a = f(*ptrs, ns, B, T, H, dk, dv, dt, fake + (5 << 33), None, None)
        b = g(*ptrs, ns, B, T, H, dk, dv, dt, fake + (5 << 33), None, fake + (6 << 33), 1 << 30, None)
        assert a == b and a in (1, 2), (ns, B, T, H, dk, dv, dt, a, b)


@pytest.mark.gpu
def test_noalloc_matches_chunk_fwd_two_calls_in_a_row():
    import torch

    from kda_synth.torchio import prefill_inputs

    lib = kda.load_library()
    f = _fn(lib)
    cases = [
        ks.PrefillWorkload("noalloc_a", "bf16", 2, 300, 4, 128, 128, seed=501, s0_std=0.05),
        ks.PrefillWorkload("noalloc_b", "bf16", 1, 450, 3, 128, 128, seed=502, s0_std=0.05,
                           seq_lens=np.array([200, 0, 129, 121])),
    ]
    for w in cases:
        t = prefill_inputs(w, "cuda")
        o_ref, s_ref = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"],
                                         cu_seqlens=t["cu"])
        o = torch.full_like(t["v"], 5.0)
        sf = torch.full_like(s_ref, 5.0)
        stream = torch.cuda.current_stream()
        st = f(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["g"].data_ptr(), t["beta"].data_ptr(),
               t["s0"].data_ptr(), None if t["cu"] is None else t["cu"].data_ptr(), w.num_seqs, w.B, w.T, w.H,
               w.d_k, w.d_v, 1, o.data_ptr(), sf.data_ptr(), stream.cuda_stream)
        assert st == 0, kda.STATUS.get(st, st)
        torch.cuda.synchronize()
        status, code = kda.kda_device_error()
        assert status == 0 and code == 0
        # the same kernels on the same inputs: bit-identical results, whatever the
        # previous call (of another size) left in the shared array
        assert torch.equal(o, o_ref)
        assert torch.equal(sf, s_ref)
