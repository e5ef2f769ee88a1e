"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output):
  O:   max |err| <= 2e-2 and mean |err| <= 2e-3
  LSE: max |err| <= 1e-3
Small shapes are compared on every element; the full-size workloads on rows
sampled across heads, tile boundaries and the ragged tail, which the oracle
computes one by one.  All full-size rows are additionally checked against an
fp32 PyTorch evaluation of the same definition.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_28_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


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


def run_gpu(ops, q, k, v, scale, causal, stream=None):
    o, lse = ops.fa_fwd(to_dev(q), to_dev(k), to_dev(v), scale=scale, causal=causal, stream=stream)
    ops.check_device_status(stream)
    return o, lse


def errors(o_gpu, lse_gpu, O_ref, L_ref):
    o = o_gpu.float().cpu().numpy().astype(np.float64).reshape(O_ref.shape)
    l = lse_gpu.cpu().numpy().astype(np.float64).reshape(L_ref.shape)
    eo = np.abs(o - O_ref)
    el = np.abs(l - L_ref)
    return eo.max(), eo.mean(), el.max()


def assert_close(o_gpu, lse_gpu, O_ref, L_ref, tag=""):
    emax, emean, elmax = errors(o_gpu, lse_gpu, O_ref, L_ref)
    assert np.isfinite(emax) and np.isfinite(elmax), tag
    assert emax <= O_MAX, f"{tag} max|dO| = {emax:.3e}"
    assert emean <= O_MEAN, f"{tag} mean|dO| = {emean:.3e}"
    assert elmax <= LSE_MAX, f"{tag} max|dLSE| = {elmax:.3e}"


def full_case(ops, q, k, v, scale, causal, tag=""):
    o, lse = run_gpu(ops, q, k, v, scale, causal)
    O_ref, L_ref = oracle.attention(q, k, v, scale, causal)
    assert_close(o, lse, O_ref, L_ref, tag)
    return o, lse


def sample_rows(B, H, Nq, n_random=1024, seed=0):
    """Rows across first/last/random heads at tile edges, plus random rows."""
    rng = np.random.default_rng(seed)
    BH = B * H
    heads = sorted({0, BH - 1, *rng.integers(0, BH, 6).tolist()})
    edge = sorted({i for t in range(0, Nq, 128) for i in (t, t + 1, t + 63, t + 127, t + 128, t + 255)
                   if i < Nq} | {Nq - 1})
    rows = {h * Nq + i for h in heads for i in edge}
    rows |= set(rng.integers(0, BH * Nq, n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def torch_reference(q, k, v, scale, causal):
    """fp32 evaluation of the definition on the GPU, one head at a time."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    qf, kf, vf = q.float().reshape(B * H, Nq, d), k.float().reshape(B * H, Nk, d), v.float().reshape(B * H, Nk, d)
    O = torch.empty((B * H, Nq, d), dtype=torch.float32, device=q.device)
    L = torch.empty((B * H, Nq), dtype=torch.float32, device=q.device)
    mask = None
    if causal:
        mask = torch.arange(Nk, device=q.device)[None, :] > torch.arange(Nq, device=q.device)[:, None]
    for h in range(B * H):
        s = (qf[h] @ kf[h].T) * scale
        if mask is not None:
            s = s.masked_fill(mask, -math.inf)
        L[h] = torch.logsumexp(s, dim=-1)
        O[h] = torch.softmax(s, dim=-1) @ vf[h]
    return O.reshape(B, H, Nq, d), L.reshape(B, H, Nq)


# ----------------------------------------------------------------- workloads

SMALL = ["single_head_n256_d64", "causal_b4_h16_n1024_d64"]
LARGE = ["b2_h16_n4096_d128", "causal_h32_n16384_d128_sigma2",
         "b8_h32_q128_kv8192_d128", "b8_h32_q128_kv8229_d128"]


@pytest.mark.parametrize("name", SMALL)
def test_small_workloads_every_element(ops, name):
    w = inputs.WORKLOADS[name]
    q, k, v, scale = inputs.make_inputs(w)
    full_case(ops, q, k, v, scale, w.causal, name)


@pytest.mark.parametrize("name", LARGE)
def test_full_size_workloads_sampled_rows(ops, name):
    w = inputs.WORKLOADS[name]
    q, k, v, scale = inputs.make_inputs(w)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o, lse = ops.fa_fwd(qd, kd, vd, scale=scale, causal=w.causal)
    ops.check_device_status()
    rows = sample_rows(w.B, w.H, w.Nq, seed=w.index)
    O_ref, L_ref = oracle.attention_rows(q, k, v, scale, w.causal, rows=rows)
    o_rows = o.reshape(-1, w.d)[torch.from_numpy(rows).cuda()]
    l_rows = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    assert_close(o_rows, l_rows, O_ref, L_ref, name)
    # every row, against fp32 PyTorch on the GPU (a property check at full size)
    O_t, L_t = torch_reference(qd, kd, vd, scale, w.causal)
    eo = (o.float() - O_t).abs()
    assert eo.max().item() <= O_MAX and eo.mean().item() <= O_MEAN, name
    assert (lse - L_t).abs().max().item() <= LSE_MAX, name
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [
    (1, 1), (1, 37), (37, 1), (100, 100), (128, 128), (129, 129), (255, 257), (257, 255),
    (300, 1000), (1000, 300), (384, 384), (640, 129),
])
def test_ragged_shapes(ops, d, causal, Nq, Nk):
    q, k, v = inputs.custom_inputs(7000 + Nq * 3 + Nk, 1, 2, Nq, Nk, d)
    full_case(ops, q, k, v, float(np.float32(1 / math.sqrt(d))), causal, f"{Nq}x{Nk}x{d} causal={causal}")


@pytest.mark.parametrize("shape", [(256, 256, 64), (128, 256, 64)])
def test_triton_page_test_shapes(ops, shape):
    # the test cases of the Triton FlashAttention exercise page (seqlen_q,
    # seqlen_k, head_dim), here in bf16 against the fp64 oracle
    Nq, Nk, d = shape
    q, k, v = inputs.custom_inputs(42, 1, 1, Nq, Nk, d)
    full_case(ops, q, k, v, float(np.float32(1 / math.sqrt(d))), False, str(shape))


def test_many_heads_small_sequences(ops):
    # far more work items than SMs: every item of the persistent schedule runs
    q, k, v = inputs.custom_inputs(123, 8, 64, 200, 160, 64)
    full_case(ops, q, k, v, 0.125, True, "many heads")


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_closed_form(ops, causal):
    # Q = 0: O_i = mean of the visible V rows, LSE_i = ln |J_i|
    B, H, Nq, Nk, d = 1, 3, 300, 260, 128
    _, k, v = inputs.custom_inputs(99, B, H, Nq, Nk, d)
    q = np.zeros((B, H, Nq, d), dtype=np.uint16)
    o, lse = run_gpu(ops, q, k, v, 0.0883883, causal)
    vf = oracle.bf16_bits_to_f64(v)
    n = np.minimum(np.arange(Nq) + 1, Nk) if causal else np.full(Nq, Nk)
    O_ref = np.stack([vf[:, :, :c].mean(axis=2) for c in n], axis=2)
    L_ref = np.broadcast_to(np.log(n), (B, H, Nq))
    assert_close(o, lse, O_ref, L_ref, "Q = 0")


def test_dominant_logit_selects_its_value_row(ops):
    B, H, Nq, Nk, d = 1, 2, 256, 384, 64
    jstar = 301
    kf = np.zeros((B, H, Nk, d), dtype=np.float32)
    kf[:, :, jstar, 0] = 16.0
    qf = np.zeros((B, H, Nq, d), dtype=np.float32)
    qf[:, :, :, 0] = 8.0          # score 16 * 8 * scale(=0.5) = 64 >= 40 over every other key
    _, _, v = inputs.custom_inputs(5, B, H, Nq, Nk, d)
    q, k = inputs.fp32_to_bf16_bits(qf), inputs.fp32_to_bf16_bits(kf)
    o, lse = run_gpu(ops, q, k, v, 0.5, False)
    vstar = oracle.bf16_bits_to_f64(v)[:, :, jstar]
    assert np.abs(o.float().cpu().numpy() - vstar[:, :, None, :]).max() <= 2 ** -8 * np.abs(vstar).max() + 1e-6
    assert np.abs(lse.cpu().numpy() - 64.0).max() <= 1e-3


def test_large_logits_rescaling(ops):
    # scores of std ~ 16: the running maximum moves often and far
    q, k, v = inputs.custom_inputs(31337, 1, 4, 512, 1536, 128, sigma=(4.0, 4.0, 1.0))
    full_case(ops, q, k, v, float(np.float32(1 / math.sqrt(128))), True, "large logits")


@pytest.mark.parametrize("scale", [-0.125, 0.0, 1e-3, 2.0])
def test_unusual_scales(ops, scale):
    q, k, v = inputs.custom_inputs(4242, 1, 2, 200, 300, 64)
    full_case(ops, q, k, v, scale, False, f"scale={scale}")
    full_case(ops, q, k, v, scale, True, f"scale={scale} causal")


def test_permutation_invariance_noncausal(ops):
    q, k, v = inputs.custom_inputs(777, 1, 2, 256, 512, 128)
    perm = np.random.default_rng(0).permutation(512)
    o1, l1 = run_gpu(ops, q, k, v, 0.088, False)
    o2, l2 = run_gpu(ops, q, np.ascontiguousarray(k[:, :, perm]), np.ascontiguousarray(v[:, :, perm]), 0.088, False)
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * 2 ** -8
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_repeatable_and_stream_safe(ops):
    q, k, v = inputs.custom_inputs(2024, 2, 4, 640, 640, 128)
    o1, l1 = run_gpu(ops, q, k, v, 0.088, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = run_gpu(ops, q, k, v, 0.088, True, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_host_buffer_entry_point(ops):
    B, H, Nq, Nk, d = 1, 4, 384, 512, 128
    q, k, v = inputs.custom_inputs(55, B, H, Nq, Nk, d)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = pin(q), pin(k), pin(v)
    ho = torch.empty((B, H, Nq, d), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (hq, hk, hv))
    do = torch.empty_like(ho, device="cuda")
    dl = torch.empty_like(hl, device="cuda")
    ops.fa_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, 0.088, causal=False)
    ops.check_device_status()
    O_ref, L_ref = oracle.attention(q, k, v, 0.088, False)
    assert_close(ho, hl, O_ref, L_ref, "host entry")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,N", [(128, 2048), (64, 4096)])
def test_host_buffer_entry_point_pipelined_groups(ops, causal, d, N):
    # 51 heads: fa_fwd_host pipelines them in ragged groups of heads (8 groups
    # of 6 or 7); each group runs the same kernel on its heads, so the result
    # is bit-identical to one fa_fwd over the device buffers.
    B, H, Nq, Nk = 3, 17, N, N
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = ops.host_groups(B, H, Nq, Nk, d, sms)
    assert groups >= 2
    scale = float(np.float32(1 / math.sqrt(d)))
    q, k, v = inputs.custom_inputs(77, B, H, Nq, Nk, d)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = pin(q), pin(k), pin(v)
    ho = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16).pin_memory()
    hl = torch.full((B, H, Nq), float("nan"), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (hq, hk, hv))
    do = torch.empty_like(ho, device="cuda")
    dl = torch.empty_like(hl, device="cuda")
    stream = torch.cuda.Stream()
    ops.fa_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, scale, causal=causal, stream=stream)
    stream.synchronize()
    ops.check_device_status()
    o_ref, l_ref = run_gpu(ops, q, k, v, scale, causal)
    assert torch.equal(ho, o_ref.cpu()) and torch.equal(hl, l_ref.cpu())
    rows = sample_rows(B, H, Nq, n_random=256, seed=5)
    Or, Lr = oracle.attention_rows(q, k, v, scale, causal, rows=rows)
    sel = torch.from_numpy(rows)
    assert_close(ho.reshape(-1, d)[sel], hl.reshape(-1)[sel], Or, Lr, "pipelined host entry")


def test_host_entry_point_orders_after_earlier_work_and_serves_two_threads(ops):
    # The pipelined path forks from the caller's stream after the work already
    # on it: here the host inputs are only written by a copy enqueued just
    # before the call.  Two host threads calling at once on their own streams
    # both get their own, correct results.
    import threading
    B, H, Nq, Nk, d = 2, 16, 1024, 1024, 128
    assert ops.host_groups(B, H, Nq, Nk, d, 152) >= 2
    scale = float(np.float32(1 / math.sqrt(d)))

    def one_call(seed, results, slot):
        q, k, v = inputs.custom_inputs(seed, B, H, Nq, Nk, d)
        src = [to_dev(a) for a in (q, k, v)]
        host = [torch.zeros(t.shape, dtype=torch.bfloat16).pin_memory() for t in src]
        ho = torch.empty((B, H, Nq, d), dtype=torch.bfloat16).pin_memory()
        hl = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
        dev = [torch.empty_like(t) for t in src]
        do = torch.empty_like(dev[0])
        dl = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for h, t in zip(host, src):
                h.copy_(t, non_blocking=True)       # the inputs reach host memory on `stream` only
        ops.fa_fwd_host(*host, ho, hl, *dev, do, dl, scale, causal=True, stream=stream)
        stream.synchronize()
        o_ref, l_ref = ops.fa_fwd(*src, scale=scale, causal=True)
        torch.cuda.synchronize()
        results[slot] = torch.equal(ho, o_ref.cpu()) and torch.equal(hl, l_ref.cpu())

    results = [None, None]
    one_call(301, results, 0)
    assert results[0]
    threads = [threading.Thread(target=one_call, args=(400 + i, results, i)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    ops.check_device_status()
    assert results == [True, True]


# ------------------------------------------------------------- split keys

def run_split(ops, q, k, v, scale, causal, splits):
    o, lse = ops.fa_fwd_splitkv(to_dev(q), to_dev(k), to_dev(v), scale=scale, causal=causal, num_splits=splits)
    ops.check_device_status()
    return o, lse


@pytest.mark.parametrize("name", ["b8_h32_q128_kv8192_d128", "b8_h32_q128_kv8229_d128", "decode_b1_h32_q1_kv32768_d128"])
def test_split_keys_short_query_long_key_workloads(ops, name):
    w = inputs.WORKLOADS[name]
    q, k, v, scale = inputs.make_inputs(w)
    o, lse = run_split(ops, q, k, v, scale, w.causal, 0)
    rows = sample_rows(w.B, w.H, w.Nq, seed=w.index)
    O_ref, L_ref = oracle.attention_rows(q, k, v, scale, w.causal, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    assert_close(o.reshape(-1, w.d)[idx], lse.reshape(-1)[idx], O_ref, L_ref, name)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk,d", [(1, 4096, 128), (16, 1000, 64), (300, 1500, 128), (640, 129, 64), (1, 1, 128)])
def test_split_keys_against_oracle(ops, splits, causal, Nq, Nk, d):
    q, k, v = inputs.custom_inputs(9000 + Nq + Nk, 2, 3, Nq, Nk, d)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = run_split(ops, q, k, v, scale, causal, splits)
    O_ref, L_ref = oracle.attention(q, k, v, scale, causal)
    assert_close(o, lse, O_ref, L_ref, f"splits={splits} {Nq}x{Nk}x{d} causal={causal}")


def test_split_keys_decode_shape_auto(ops):
    # one query per head against a long cache: 32 work items without splitting
    B, H, Nq, Nk, d = 1, 32, 1, 32768, 128
    q, k, v = inputs.custom_inputs(31, B, H, Nq, Nk, d)
    ns, _ = ops.splitkv_workspace(B, H, Nq, Nk, d, False, 0)
    assert ns > 1
    o, lse = run_split(ops, q, k, v, 0.088, False, 0)
    O_ref, L_ref = oracle.attention(q, k, v, 0.088, False)
    assert_close(o, lse, O_ref, L_ref, "decode")
