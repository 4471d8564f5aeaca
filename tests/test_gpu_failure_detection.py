"""Failure detection without a GPU fault.

Every wait inside the kernels (TMA stages, accumulator hand-offs, draining
the tensor cores) is bounded: when its limit passes, the kernel records a code
in a device status word and returns normally instead of hanging.  Here a
diagnostic kernel waits, with the same wait code, on a barrier that nothing
ever completes, with a 1 ms limit; the host must then read the self-test code,
and the context must still compute correct results afterwards.  Nothing in
this file faults, traps or hangs the GPU.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from lm_head_selected_gb300 import _lib, build
    build.build()
    return _lib.load()


def _status(lib):
    code = ctypes.c_uint(0)
    st = lib.linear_logp_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                       ctypes.byref(code))
    return st, code.value


def test_bounded_wait_reports_instead_of_hanging(lib):
    from lm_head_selected_gb300 import _lib
    assert _status(lib) == (0, 0)  # clean before
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.linear_logp_selftest_wait_timeout(1_000_000, stream) == 0
    st, code = _status(lib)
    assert st == _lib.LLP_ERR_DEVICE_TIMEOUT
    assert code == _lib.DEVICE_SELFTEST_CODE
    assert _status(lib) == (0, 0)  # reading clears the word

    # the context is still usable: a forward on the tiny workload matches the oracle
    import lm_head_selected_gb300 as llp
    inp = workloads.tiny()
    logp, lse = llp.linear_logp_fwd(inp.hidden.cuda(), inp.weight.cuda(), inp.targets.cuda(), inp.bias.cuda())
    ref, _ = oracle.forward(inp.hidden.double().numpy(), inp.weight.double().numpy(), inp.bias.double().numpy(),
                            inp.targets.numpy(), None)
    assert np.max(np.abs(logp.double().cpu().numpy() - ref)) < 5e-3
    assert _status(lib) == (0, 0)
