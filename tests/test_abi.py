"""The C-ABI library: it loads, exports what include/fa.h declares, and
rejects bad arguments on the host before touching the GPU."""
import ctypes
import math
import os
import re

import pytest

import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
from exact_attention_28_gb300 import build, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"fa_fwd", "fa_fwd_host", "fa_check_device_status", "fa_status_string"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_binding_matches_header_arity(lib):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER, encoding="utf-8").read(), flags=re.S)
    for name in declared_functions():
        m = re.search(rf"\b{name}\s*\(([^)]*)\)", text)
        nparams = 0 if m.group(1).strip() in ("", "void") else m.group(1).count(",") + 1
        assert len(getattr(lib, name).argtypes) == nparams, name


def test_status_strings(lib):
    for s in range(7):
        assert ops.status_string(s)
    assert "unknown" in ops.status_string(99)


def test_status_mapping_to_python_errors(lib):
    """Each status code has its own name in the header's enum order, and the
    binding turns every non-OK status into an FAError carrying that code."""
    names = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED", "FA_ERR_CUDA",
             "FA_ERR_TIMEOUT", "FA_ERR_TOO_LARGE"]
    assert [getattr(ops, n) for n in names] == list(range(7))
    for code, name in enumerate(names):
        assert ops.status_string(code).startswith(name)
        if code == ops.FA_OK:
            ops._check(code)   # no exception
            continue
        with pytest.raises(ops.FAError) as err:
            ops._check(code)
        assert err.value.status == code and name in str(err.value)
    assert "wait expired" in ops.status_string(ops.FA_ERR_TIMEOUT)


def test_device_status_check_without_a_gpu_is_an_error(lib):
    # the status word lives on the device: without one the check cannot
    # report FA_OK (it would hide a failure), it reports FA_ERR_CUDA
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.fa_check_device_status(None) == ops.FA_ERR_CUDA
    with pytest.raises(ops.FAError) as err:
        ops.check_device_status(0)
    assert err.value.status == ops.FA_ERR_CUDA


GOOD = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000,
            B=1, H=1, Nq=4, Nk=4, d=64, scale=0.125, causal=0)


def call(**kw):
    a = dict(GOOD, **kw)
    return ops.raw_fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"],
                          a["d"], a["scale"], a["causal"])


@pytest.mark.parametrize("kw,expected", [
    (dict(q=0), ops.FA_ERR_INVALID_ARG),
    (dict(k=0), ops.FA_ERR_INVALID_ARG),
    (dict(v=0), ops.FA_ERR_INVALID_ARG),
    (dict(o=0), ops.FA_ERR_INVALID_ARG),
    (dict(lse=0), ops.FA_ERR_INVALID_ARG),
    (dict(B=0), ops.FA_ERR_INVALID_ARG),
    (dict(H=-1), ops.FA_ERR_INVALID_ARG),
    (dict(Nq=0), ops.FA_ERR_INVALID_ARG),
    (dict(Nk=0), ops.FA_ERR_INVALID_ARG),
    (dict(scale=math.nan), ops.FA_ERR_INVALID_ARG),
    (dict(scale=math.inf), ops.FA_ERR_INVALID_ARG),
    (dict(d=96), ops.FA_ERR_UNSUPPORTED),
    (dict(d=32), ops.FA_ERR_UNSUPPORTED),     # the smallest test shape on the Triton page
    (dict(d=256), ops.FA_ERR_UNSUPPORTED),
    (dict(q=0x10008), ops.FA_ERR_MISALIGNED),
    (dict(o=0x40002), ops.FA_ERR_MISALIGNED),
    (dict(lse=0x50002), ops.FA_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 16), ops.FA_ERR_INVALID_ARG),   # B*H overflow
])
def test_argument_errors_before_any_launch(lib, kw, expected):
    assert call(**kw) == expected


@pytest.mark.parametrize("splits,ws,nbytes,expected", [
    (0, 0x100000, 1 << 30, ops.FA_ERR_INVALID_ARG),      # num_splits < 1
    (257, 0x100000, 1 << 30, ops.FA_ERR_INVALID_ARG),    # num_splits > 256
    (2, 0, 1 << 30, ops.FA_ERR_INVALID_ARG),             # NULL workspace
    (2, 0x100010, 1 << 30, ops.FA_ERR_MISALIGNED),       # not 256-byte aligned
    (2, 0x100000, 64, ops.FA_ERR_INVALID_ARG),           # too small
])
def test_splitkv_argument_errors(lib, splits, ws, nbytes, expected):
    a = GOOD
    st = lib.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                            a["scale"], a["causal"], splits, ws, nbytes, None)
    assert st == expected


def test_host_entry_rejects_null_host_buffers(lib):
    vp = ctypes.c_void_p
    st = lib.fa_fwd_host(None, vp(1 << 16), vp(1 << 16), vp(1 << 16), vp(1 << 16),
                         vp(1 << 16), vp(1 << 16), vp(1 << 16), vp(1 << 16), vp(1 << 16),
                         1, 1, 4, 4, 64, 0.125, 0, None)
    assert st == ops.FA_ERR_INVALID_ARG


def test_no_gpu_means_cuda_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # Valid arguments on a machine without a GPU: the call must fail loudly.
    assert call() == ops.FA_ERR_CUDA


PAGED = dict(q=0x10000, kc=0x20000, vc=0x30000, table=0x60000, seq=0x70000, o=0x40000, lse=0x50000,
             B=1, H=1, Nq=4, max_blocks=2, num_blocks=2, bs=64, d=64, scale=0.125, causal=0)


@pytest.mark.parametrize("kw,expected", [
    (dict(table=0), ops.FA_ERR_INVALID_ARG),
    (dict(seq=0), ops.FA_ERR_INVALID_ARG),
    (dict(max_blocks=0), ops.FA_ERR_INVALID_ARG),
    (dict(num_blocks=0), ops.FA_ERR_INVALID_ARG),
    (dict(bs=48), ops.FA_ERR_UNSUPPORTED),
    (dict(bs=8), ops.FA_ERR_UNSUPPORTED),
    (dict(bs=512), ops.FA_ERR_UNSUPPORTED),
    (dict(table=0x60002), ops.FA_ERR_MISALIGNED),
    (dict(seq=0x70001), ops.FA_ERR_MISALIGNED),
    (dict(d=96), ops.FA_ERR_UNSUPPORTED),
])
@pytest.mark.parametrize("split", [False, True])
def test_paged_argument_errors(lib, kw, expected, split):
    a = dict(PAGED, **kw)
    args = (a["q"], a["kc"], a["vc"], a["table"], a["seq"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
            a["max_blocks"], a["num_blocks"], a["bs"], a["d"], a["scale"], a["causal"])
    if split:
        st = lib.fa_fwd_paged_splitkv(*args, 2, 0x100000, 1 << 30, None)
    else:
        st = lib.fa_fwd_paged(*args, None)
    assert st == expected


@pytest.mark.parametrize("splits,ws,nbytes,expected", [
    (0, 0x100000, 1 << 30, ops.FA_ERR_INVALID_ARG),
    (2, 0, 1 << 30, ops.FA_ERR_INVALID_ARG),
    (2, 0x100010, 1 << 30, ops.FA_ERR_MISALIGNED),
    (2, 0x100000, 64, ops.FA_ERR_INVALID_ARG),
])
def test_paged_splitkv_workspace_errors(lib, splits, ws, nbytes, expected):
    a = PAGED
    st = lib.fa_fwd_paged_splitkv(a["q"], a["kc"], a["vc"], a["table"], a["seq"], a["o"], a["lse"], a["B"], a["H"],
                                  a["Nq"], a["max_blocks"], a["num_blocks"], a["bs"], a["d"], a["scale"],
                                  a["causal"], splits, ws, nbytes, None)
    assert st == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(d=64), ops.FA_ERR_UNSUPPORTED),
    (dict(dq=0), ops.FA_ERR_INVALID_ARG),
    (dict(dv=0), ops.FA_ERR_INVALID_ARG),
    (dict(dk=0x80002), ops.FA_ERR_MISALIGNED),
    (dict(q=0x10008), ops.FA_ERR_MISALIGNED),
    (dict(Nk=0), ops.FA_ERR_INVALID_ARG),
])
def test_fp8_forward_argument_errors(lib, kw, expected):
    a = dict(q=0x10000, k=0x20000, v=0x30000, dq=0x80000, dk=0x80100, dv=0x80200, o=0x40000, lse=0x50000,
             B=1, H=1, Nq=4, Nk=4, d=128, scale=0.125, causal=0)
    a.update(kw)
    st = lib.fa_fwd_fp8(a["q"], a["k"], a["v"], a["dq"], a["dk"], a["dv"], a["o"], a["lse"], a["B"], a["H"],
                        a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], None)
    assert st == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(x=0), ops.FA_ERR_INVALID_ARG),
    (dict(descale=0), ops.FA_ERR_INVALID_ARG),
    (dict(N=0), ops.FA_ERR_INVALID_ARG),
    (dict(N=65535 * 64 + 1), ops.FA_ERR_INVALID_ARG),
    (dict(d=96), ops.FA_ERR_UNSUPPORTED),
    (dict(x=0x10002), ops.FA_ERR_MISALIGNED),
    (dict(x8=0x20004), ops.FA_ERR_MISALIGNED),
    (dict(signs=0x30002), ops.FA_ERR_MISALIGNED),
])
def test_quantize_argument_errors(lib, kw, expected):
    a = dict(x=0x10000, x8=0x20000, descale=0x40000, B=1, H=1, N=4, d=128, signs=0, transpose=0)
    a.update(kw)
    st = lib.fa_quantize_fp8(a["x"], a["x8"], a["descale"], a["B"], a["H"], a["N"], a["d"], a["signs"] or None,
                             a["transpose"], None)
    assert st == expected


def test_host_groups_rule(lib):
    # small calls are not pipelined; a group keeps >= 8 MiB of inputs; at most
    # 8 groups and one head per group
    assert ops.host_groups(1, 1, 256, 256, 64, 152) == 1
    assert ops.host_groups(1, 4, 1024, 1024, 128, 152) == 1      # 3 MiB of inputs
    assert ops.host_groups(1, 16, 1024, 1024, 128, 152) == 1     # 12 MiB: one group of 8 MiB
    assert ops.host_groups(1, 16, 1024, 2048, 128, 152) == 2     # 20 MiB
    assert ops.host_groups(2, 16, 4096, 4096, 128, 152) == 8     # 96 MiB, capped at 8
    assert ops.host_groups(3, 17, 2048, 2048, 128, 152) == 8
    assert ops.host_groups(1, 2, 65536, 65536, 128, 1) == 2      # capped at one head per group
    assert ops.host_groups(8, 32, 128, 8192, 128, 152) == 8
    for bad in [(0, 1, 1, 1, 64, 1), (1, 1, 1, 1, 96, 1), (1, 1, 1, 1, 64, 0)]:
        assert ops.host_groups(*bad) == 0
