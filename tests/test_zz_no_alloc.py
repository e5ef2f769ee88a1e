"""The no-allocation split-key entry point, fa_fwd_splitkv_noalloc.

Some callers cannot allocate device memory at the moment they run attention:
serving loops whose latency budget rules out the allocator (cudaMalloc may
synchronise the device), frameworks whose allocator owns all memory up front,
or plugins that an inference runtime hands only the tensors they read and
write and forbids to allocate while they execute.  This entry point serves
them: its partial results live in a fixed 16 MiB scratch array inside the
library rather than in a workspace the caller allocates.

Its results must match those of the workspace-based entry point,
fa_fwd_splitkv, call after call, even though every call reuses -- and leaves
behind -- the same scratch contents.  This file is named so that pytest
collects it last.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from exact_attention_28_gb300 import build, inputs, ops  # noqa: E402

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3   # the tolerances of the parity tests


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", [
    (2, 8, 20, 3000, 128, False, 4),
    (1, 6, 300, 1500, 64, True, 3),
    (1, 32, 1, 32768, 128, False, 0),     # a decode shape; the library picks the slice count
])
def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(lib, B, H, Nq, Nk, d, causal, splits):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    scale = float(np.float32(1 / math.sqrt(d)))
    for seed in (101, 202):                  # two calls in a row, different inputs
        q, k, v = inputs.custom_inputs(seed, B, H, Nq, Nk, d)
        Q, K, V = to_dev(q), to_dev(k), to_dev(v)
        O = torch.empty_like(Q)
        LSE = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
        st = lib.fa_fwd_splitkv_noalloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                                        B, H, Nq, Nk, d, scale, int(causal), splits, None)
        assert st == ops.FA_OK, ops.status_string(st)
        torch.cuda.synchronize()
        assert lib.fa_check_device_status(None) == ops.FA_OK
        O_ref, LSE_ref = ops.fa_fwd_splitkv(Q, K, V, scale=scale, causal=causal, num_splits=splits)
        torch.cuda.synchronize()
        err = (O.float() - O_ref.float()).abs()
        assert err.max().item() <= O_MAX and err.mean().item() <= O_MEAN
        assert (LSE - LSE_ref).abs().max().item() <= LSE_MAX
        assert torch.isfinite(O.float()).all() and torch.isfinite(LSE).all()


def test_noalloc_rejects_work_beyond_the_scratch_area(lib):
    # 4 slices x 4096 heads x 1024 rows x 129 floats is far beyond 16 MiB:
    # refused before anything is enqueued (so this needs no GPU).
    p = 1 << 20
    st = lib.fa_fwd_splitkv_noalloc(p, p, p, p, p, 64, 64, 1024, 4096, 128, 0.088, 0, 4, None)
    assert st == ops.FA_ERR_TOO_LARGE
    assert "16 MiB" in ops.status_string(st)
