"""The hardware fact the GEMM's design rests on, pinned against the
toolkit: this CUDA toolkit's ptxas rejects the integer form of the
5th-generation tensor-core MMA (tcgen05.mma kind::i8) for sm_103a, B300's
architecture, and accepts it for sm_100a; it accepts the bf16/fp16 form
(kind::f16) for sm_103a.  So exact INT8 x INT8 -> INT32 products on B300's
tcgen05 tensor cores are made from integer codes carried as bf16 values,
which is what the library does.  Assembles a one-instruction PTX kernel;
needs no GPU."""
import pytest

from w8a8_int8_linear_act_b300 import peaks


def _ptxas(target, kind):
    ok, msg, ver = peaks.ptxas_accepts_tcgen05(target, kind)
    if ok is None:
        pytest.skip(msg)
    return ok, msg


def test_tcgen05_integer_mma_rejected_for_sm_103a():
    ok, msg = _ptxas("sm_103a", "i8")
    assert not ok and "kind::i8" in msg and "sm_103a" in msg


def test_tcgen05_integer_mma_accepted_for_sm_100a():
    ok, msg = _ptxas("sm_100a", "i8")
    assert ok, msg


def test_tcgen05_bf16_mma_accepted_for_sm_103a():
    ok, msg = _ptxas("sm_103a", "f16")
    assert ok, msg
