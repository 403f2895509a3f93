"""GPU test of the decode kernels' device-side failure path, without a GPU
fault.

Every wait of the decode kernel for staged payload data is bounded.  Here the
host asks the next launch (ndq_test_withhold_copy) to withhold the staging
copy of one tile, as if the copy had been lost: nothing ever completes that
stage, so the decode warps waiting for it give up after a short limit (1 ms),
set their bit in the device fault word and stop; the CTA's producer, which
then finds its ring never released, gives up as well, waits for every copy it
did issue, and stops.  Nothing faults or hangs: the call returns, the fault
word reports what happened, and the next launch decodes bit-exactly again.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_bit_exact

pytestmark = pytest.mark.gpu

import quantized_weight_block_gb300 as ndq  # noqa: E402

CONSUMER_GAVE_UP = 2  # bit 1 of the fault word
PRODUCER_GAVE_UP = 1  # bit 0


def _decode(fmt, shape, x, y):
    rc = ndq.ndq_dequantize_packed(ndq.format_id(fmt), shape, ndq.NDQ_BFLOAT16, x.data_ptr(), x.numel(),
                                   y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ndq.ndq_status_string(rc)


def _bits(y):
    return y.cpu().view(torch.uint16).numpy()


@pytest.fixture(autouse=True)
def _clean_fault_word():
    ndq.get_device_fault()  # start from a clear word
    yield
    ndq.ndq_test_withhold_copy(-1, 1)


def test_withheld_copy_expires_and_the_next_launch_is_exact(orc):
    # 7168 tiles over a persistent grid: every CTA stages many tiles, so the
    # CTA that loses tile 0 has later copies in flight when its decode warps
    # stop, and its producer then waits on a stage nobody releases
    fmt, shape = "gguf:q4_k", (14336, 4096)
    xn = synth.payload(fmt, shape, seed=3)
    x = torch.from_numpy(xn).cuda()
    y = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    assert ndq.ndq_test_withhold_copy(0, 1000) == 0
    _decode(fmt, shape, x, y)
    torch.cuda.synchronize()
    f = ndq.get_device_fault()
    assert f & CONSUMER_GAVE_UP and f & PRODUCER_GAVE_UP, f
    # the request was consumed: the next launch is complete and exact
    y.fill_(float("nan"))
    _decode(fmt, shape, x, y)
    torch.cuda.synchronize()
    assert ndq.get_device_fault() == 0
    assert_bit_exact(_bits(y), orc.decode_parallel(fmt, shape, xn, "bfloat16"), "bfloat16", "after expiry")


def test_withheld_copy_of_a_cta_with_one_tile(orc):
    # fewer tiles than resident CTAs: the affected CTA's only tile is lost;
    # its producer has nothing else to stage, only its decode warps give up
    fmt, shape = "gguf:q6_k", (64, 8192)
    xn = synth.payload(fmt, shape, seed=4)
    x = torch.from_numpy(xn).cuda()
    y = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    assert ndq.ndq_test_withhold_copy(5, 1000) == 0
    _decode(fmt, shape, x, y)
    torch.cuda.synchronize()
    assert ndq.get_device_fault() == CONSUMER_GAVE_UP
    # every tile but the withheld one (elements 5*8192 .. 6*8192) was decoded
    want = orc.decode(fmt, shape, xn, "bfloat16").reshape(-1)
    got = _bits(y).reshape(-1)
    keep = np.ones(got.size, bool)
    keep[5 * 8192:6 * 8192] = False
    assert_bit_exact(got[keep], want[keep], "bfloat16", "other tiles")
    _decode(fmt, shape, x, y)
    torch.cuda.synchronize()
    assert ndq.get_device_fault() == 0
    assert_bit_exact(_bits(y), want, "bfloat16", "after expiry")


def test_withheld_copy_in_a_batched_launch(orc):
    # the whole-model kernel (q8_0 / q4_k / q6_k batch), a tile in the middle
    specs = [("gguf:q4_k", (1024, 4096), 1), ("gguf:q6_k", (2048, 4096), 2), ("gguf:q8_0", (4096, 4096), 3)]
    xs = [synth.payload(f, s, seed=k) for f, s, k in specs]
    items = [(f, s, torch.from_numpy(x).cuda(), torch.empty(s, dtype=torch.bfloat16, device="cuda"))
             for (f, s, _), x in zip(specs, xs)]
    assert ndq.ndq_test_withhold_copy(700, 1000) == 0
    ws = ndq.dequantize_packed_batched(items)
    torch.cuda.synchronize()
    assert ndq.get_device_fault() & CONSUMER_GAVE_UP
    ws = ndq.dequantize_packed_batched(items)
    torch.cuda.synchronize()
    del ws
    assert ndq.get_device_fault() == 0
    for (f, s, _), x, it in zip(specs, xs, items):
        assert_bit_exact(_bits(it[3]), orc.decode(f, s, x, "bfloat16"), "bfloat16", f"after expiry {f}")
