"""The no-allocation split-key entry point, fa_fwd_splitkv_noalloc.

Some callers cannot allocate device memory at the moment they run attention:
serving loops whose latency budget rules out the allocator (cudaMalloc may
synchronise the device), frameworks whose allocator owns all memory up front,
or plugins that an inference runtime hands only the tensors they read and
write and forbids to allocate while they execute.  This entry point serves
them: its partial results live in a fixed 16 MiB scratch array inside the
library rather than in a workspace the caller allocates.

Its results must equal those of the workspace-based entry point,
fa_fwd_splitkv, bit for bit (the same kernels run with the same number of
key slices), and match the fp64 oracle within the parity tolerances, call
after call, even though every call reuses -- and leaves behind -- the same
scratch contents.  A large call that fills most of the array runs first, then
smaller ones, among them a causal call whose early query tiles have empty key
slices (their partials are skipped, so stale values left by the earlier call
must not leak in).  This file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from exact_attention_28_gb300 import build, inputs, ops  # noqa: E402

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3   # the tolerances of the parity tests
SCRATCH = 16 << 20                           # bytes of the library's scratch array


def scratch_bytes(splits, BH, Nq, d):
    """Bytes of partials a call needs: fp32 O rounded up to 256 bytes, then fp32 LSE."""
    o = splits * BH * Nq * d * 4
    return (o + 255) // 256 * 256 + splits * BH * Nq * 4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def check_against_oracle(q, k, v, scale, causal, O, LSE):
    import oracle
    B, H, Nq, d = q.shape
    rows = np.arange(B * H * Nq)
    if rows.size > 2048:   # large calls: a fixed sample of rows across heads and tiles
        rows = np.unique(np.concatenate([rows[:256], rows[-256:],
                                         np.random.default_rng(0).integers(0, rows.size, 1536)]))
    O_ref, L_ref = oracle.attention_rows(q, k, v, scale, causal, rows=rows)
    o = O.reshape(-1, d)[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    l = LSE.reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    err = np.abs(o - O_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(l - L_ref).max() <= LSE_MAX


# (B, H, Nq, Nk, d, causal, num_splits, seed); the first fills 12.7 of the 16 MiB
CALLS = [
    (1, 16, 256, 3000, 128, False, 6, 101),
    (1, 3, 300, 1500, 64, True, 8, 202),       # early query tiles: 6 of 8 key slices empty
    (1, 3, 300, 1500, 64, True, 8, 303),       # the same shape again, other inputs
    (1, 32, 1, 32768, 128, False, 0, 404),     # a decode shape; the library picks the slice count
    (2, 4, 200, 600, 64, True, 1, 606),         # one slice: no partials, the scratch area is not used
]


@pytest.mark.gpu
def test_noalloc_equals_workspace_entry_and_oracle_call_after_call(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    for i, (B, H, Nq, Nk, d, causal, splits, seed) in enumerate(CALLS):
        q, k, v = inputs.custom_inputs(seed, B, H, Nq, Nk, d)
        scale = float(np.float32(1 / math.sqrt(d)))
        Q, K, V = to_dev(q), to_dev(k), to_dev(v)
        O = torch.empty_like(Q)
        LSE = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
        if i == 1:   # once through the Python binding, which checks o and lse
            ops.fa_fwd_splitkv_noalloc(Q, K, V, O, LSE, scale=scale, causal=causal, num_splits=splits)
        else:
            st = lib.fa_fwd_splitkv_noalloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                                            B, H, Nq, Nk, d, scale, int(causal), splits, None)
            assert st == ops.FA_OK, ops.status_string(st)
        torch.cuda.synchronize()
        assert lib.fa_check_device_status(None) == ops.FA_OK
        O_ws, LSE_ws = ops.fa_fwd_splitkv(Q, K, V, scale=scale, causal=causal, num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(O, O_ws) and torch.equal(LSE, LSE_ws), f"call {i}: differs from the workspace path"
        check_against_oracle(q, k, v, scale, causal, O, LSE)


@pytest.mark.gpu
def test_noalloc_largest_call_that_fits(lib):
    # 13 slices x 41 heads x 61 rows x (128 + 1) floats: 16,776,708 bytes of the 16,777,216
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H, Nq, Nk, d, splits = 1, 41, 61, 13 * 128, 128, 13
    assert scratch_bytes(splits, B * H, Nq, d) <= SCRATCH < scratch_bytes(splits, B * H, Nq + 1, d)
    q, k, v = inputs.custom_inputs(505, B, H, Nq, Nk, d)
    scale = float(np.float32(1 / math.sqrt(d)))
    Q, K, V = to_dev(q), to_dev(k), to_dev(v)
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ops.fa_fwd_splitkv_noalloc(Q, K, V, O, LSE, scale=scale, num_splits=splits)
    ops.check_device_status()
    O_ws, LSE_ws = ops.fa_fwd_splitkv(Q, K, V, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(O, O_ws) and torch.equal(LSE, LSE_ws)
    check_against_oracle(q, k, v, scale, False, O, LSE)


def test_noalloc_rejects_work_beyond_the_scratch_area(lib):
    # refused before anything is enqueued, so these fake (aligned) pointers are
    # never touched and the test needs no GPU
    p = 1 << 20
    st = lib.fa_fwd_splitkv_noalloc(p, p, p, p, p, 64, 64, 1024, 4096, 128, 0.088, 0, 4, None)
    assert st == ops.FA_ERR_TOO_LARGE
    assert "16 MiB" in ops.status_string(st)
    # one step past the limit: 2 slices x 3 heads x 5419 rows x 129 floats = 16 MiB + 8 bytes
    assert scratch_bytes(2, 3, 5419, 128) == SCRATCH + 8
    assert lib.fa_fwd_splitkv_noalloc(p, p, p, p, p, 1, 3, 5419, 4096, 128, 0.088, 0, 2, None) == ops.FA_ERR_TOO_LARGE


def test_noalloc_accepts_the_largest_call_that_fits_without_a_gpu(lib):
    # without a device the fitting call gets past the size check and fails
    # at the first CUDA call (never with FA_ERR_TOO_LARGE)
    if torch.cuda.is_available():
        pytest.skip("covered with real buffers by test_noalloc_largest_call_that_fits")
    p = 1 << 20
    st = lib.fa_fwd_splitkv_noalloc(p, p, p, p, p, 1, 41, 61, 13 * 128, 128, 0.088, 0, 13, None)
    assert st == ops.FA_ERR_CUDA
