"""Failure detection on the GPU without a fault.

Every wait inside the forward kernel (on a TMA copy, an MMA, a hand-off
between warps) gives up after one second, sets the library's device status
word and lets the kernel shut down cleanly.  Here a test hook leaves one K tile
unloaded, so one wait must run out: the host must then read FA_ERR_TIMEOUT,
and the same context must go on computing correct results.
"""
import math
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_28_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_28_gb300 import build, ops as _ops
    build.build()
    _ops.load_library()
    return _ops


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


# d = 64 covers the ring whose K and V tiles of a key step share one barrier
@pytest.mark.parametrize("item,causal,d", [(0, False, 128), (5, True, 128), (3, True, 64)])
def test_missing_tile_times_out_and_the_context_stays_usable(ops, item, causal, d):
    B, H, Nq, Nk = 1, 4, 1024, 1024
    scale = float(np.float32(1 / math.sqrt(d)))
    q, k, v = inputs.custom_inputs(61, B, H, Nq, Nk, d)
    Q, K, V = to_dev(q), to_dev(k), to_dev(v)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert item < len(ops.schedule(B, H, Nq, Nk, d, int(causal), num_sms=sms))
    ops.check_device_status()                       # nothing pending from earlier tests
    t0 = time.monotonic()
    assert ops.fa_fwd_test_missing_load(Q, K, V, item=item, scale=scale, causal=causal) == ops.FA_OK
    with pytest.raises(ops.FAError) as e:
        ops.check_device_status()
    assert e.value.status == ops.FA_ERR_TIMEOUT
    assert time.monotonic() - t0 < 30                # bounded: about a second per expired wait
    # the status word was read and cleared, and the context still computes
    ops.check_device_status()
    o, lse = ops.fa_fwd(Q, K, V, scale=scale, causal=causal)
    ops.check_device_status()
    rows = np.arange(0, B * H * Nq, 37, dtype=np.int64)
    O_ref, L_ref = oracle.attention_rows(q, k, v, scale, causal, rows=rows)
    sel = torch.from_numpy(rows).cuda()
    err = np.abs(o.reshape(-1, d)[sel].float().cpu().numpy() - O_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.abs(lse.reshape(-1)[sel].cpu().numpy() - L_ref).max() <= 1e-3


def test_missing_load_rejects_a_negative_item(ops):
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    assert ops.fa_fwd_test_missing_load(q, q, q, item=-1) == ops.FA_ERR_INVALID_ARG
