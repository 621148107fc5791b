"""Failure detection on the GPU without a GPU fault: a bounded mbarrier wait
that nothing satisfies gives up after its time limit, the kernel returns, the
library's device status word reports GBATTN_EDEVICE_TIMEOUT once (then reads
clear), and the context stays usable for the next call (the consumer waiting
for a producer commit that never comes, M4.6 "FlashAttention-3/4 Hardware
Pipelines" 0x03)."""
import math

import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import attn_fwd, gbattn_device_status, gbattn_selftest_bounded_wait
from exact_tiled_attention_gb300.binding import GBATTN_EDEVICE_TIMEOUT
from exact_tiled_attention_gb300.inputs import make_prefill
from tests.parity_util import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu


def test_satisfied_wait_reports_nothing():
    gbattn_device_status()  # clear whatever an earlier call left
    gbattn_selftest_bounded_wait(True)
    assert gbattn_device_status() == 0


def test_unsatisfied_wait_gives_up_and_the_context_survives():
    gbattn_device_status()
    gbattn_selftest_bounded_wait(False)
    assert gbattn_device_status() == GBATTN_EDEVICE_TIMEOUT
    assert gbattn_device_status() == 0  # read and cleared
    q, k, v = make_prefill(1, 2, 2, 130, 130, 64, torch.bfloat16, 3, device="cuda")
    o, lse = attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), 1.0 / math.sqrt(64), True)
    assert_attn_close(o, lse, o_ref, lse_ref, "forward after a timed-out wait")
