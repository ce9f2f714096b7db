"""Failure detection without a GPU fault: a bounded wait that runs out.

A one-warp kernel waits on a barrier that nothing arrives on, through the
same bounded-wait helper every kernel of the library uses.  The wait must give
up after its limit and report through the device error word, the stream must
stay usable, and the word must be clear again after it is read."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_attention_94_gb300 import _lib, ops
from tests.parity import assert_o

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_reports():
    lib = ops.lib()
    assert ops.device_error() == 0
    t0 = time.perf_counter()
    st = lib.fa_selftest_wait_timeout(50.0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.FA_OK
    code = ctypes.c_uint(0)
    st = lib.fa_device_error(ctypes.byref(code))
    elapsed = time.perf_counter() - t0
    assert st == _lib.FA_ERR_TIMEOUT
    assert code.value == _lib.FA_DEVERR_SELFTEST_CODE
    assert elapsed < 5.0                      # bounded: 50 ms limit, not a hang
    assert ops.device_error() == 0            # reading the word cleared it


def test_context_usable_after_timeout():
    lib = ops.lib()
    lib.fa_selftest_wait_timeout(20.0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert lib.fa_device_error(None) == _lib.FA_ERR_TIMEOUT
    x = synth.make_dense(1, 2, 300, 64, seed=3, with_do=False)
    o, lse = ops.fwd(*(x[n].cuda() for n in ("q", "k", "v")), causal=True)
    o_ref, _ = oracle.forward(*(synth.to_f64(x[n]) for n in ("q", "k", "v")), 1 / np.sqrt(64), True)
    assert_o(synth.to_f64(o), o_ref, "forward after a timed-out wait")
    assert ops.device_error() == 0


def test_selftest_argument_checks():
    lib = ops.lib()
    assert lib.fa_selftest_wait_timeout(0.0, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(1e9, None) == _lib.FA_ERR_INVALID_ARG
