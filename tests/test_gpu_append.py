"""kv_append_quant on the GPU must match the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, require_gpu

pytestmark = pytest.mark.gpu


def _all_fp16(include_nonfinite=False):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    if not include_nonfinite:
        x = x[np.isfinite(x)]
    pad = (-len(x)) % 128
    return np.concatenate([x, np.zeros(pad, np.float16)])


def _run(kv_dtype, kvals, vvals, H, ks, vs, slots, num_pages, fill=0x5A, k_stride=None):
    pq = require_gpu()
    T = len(slots)
    k = torch.from_numpy(kvals.reshape(T, H, 128)).cuda()
    v = torch.from_numpy(vvals.reshape(T, H, 128)).cuda()
    if k_stride is not None:   # place k / v as column slices of a wider buffer
        big = torch.zeros((T, k_stride), dtype=torch.float16, device="cuda")
        big[:, 128:128 + H * 128] = k.reshape(T, -1)
        k = big[:, 128:128 + H * 128].view(T, H, 128)
        big2 = torch.zeros((T, k_stride), dtype=torch.float16, device="cuda")
        big2[:, 64 * 8:64 * 8 + H * 128] = v.reshape(T, -1)
        v = big2[:, 64 * 8:64 * 8 + H * 128].view(T, H, 128)
    pages = pq.new_pages(num_pages, H, kv_dtype, "cuda",
                         fill=(fill if kv_dtype != W.FP16 else 0.0))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ks_t = torch.tensor(np.atleast_1d(ks), dtype=torch.float32, device="cuda")
    vs_t = torch.tensor(np.atleast_1d(vs), dtype=torch.float32, device="cuda")
    sl = torch.from_numpy(np.asarray(slots, dtype=np.int64)).cuda()
    pq.kv_append_quant(k, v, sl, kv_dtype, ks_t, vs_t, pages, status=status)
    got = pages.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if kv_dtype == W.FP16 else got.numpy()
    pool = oracle.new_pool(num_pages, H, 128, kv_dtype, fill=(fill if kv_dtype != W.FP16 else 0))
    ref = oracle.kv_append_quant(kvals.reshape(T, H, 128), vvals.reshape(T, H, 128), slots,
                                 kv_dtype, ks, vs, pool)
    return got, ref, int(status.item())


# Scales: powers of two (every quotient exact, so E4M3 midpoints and INT8
# half-integers are hit exactly), calibrated amax / 448 and amax / 127 scales
# (quotients that fall within an ulp of those boundaries), plain values, and
# scales outside [2^-125, 2^125] where the encode takes the division.
SCALES = [1.0, 86.625 / 448.0, 2.0 ** -7, 3.0, 1000.0, 0.3,
          W.scale_from_amax(86.5, 448.0), W.scale_from_amax(86.5, 127.0),
          W.scale_from_amax(7.0, 448.0), 2.0 ** -126, 2.0 ** 126, 1.5e-38]


@pytest.mark.parametrize("kv_dtype", [W.FP8_E4M3, W.INT8])
@pytest.mark.parametrize("scale", SCALES)
def test_every_fp16_value_bit_exact(kv_dtype, scale):
    x = _all_fp16()
    T = len(x) // 128
    rng = np.random.default_rng(1)
    slots = rng.permutation(T + 40)[:T]                 # scattered slots in a larger pool
    got, ref, st = _run(kv_dtype, x, x[::-1].copy(), 1, scale, scale * 0.5, slots, (T + 40) // 16 + 1)
    assert st == 0
    assert np.array_equal(got, ref)


def test_fp16_pool_is_a_bit_copy():
    x = _all_fp16()
    T = len(x) // 128
    got, ref, st = _run(W.FP16, x, x, 1, 1.0, 1.0, np.arange(T), T // 16 + 1)
    assert st == 0 and np.array_equal(got, ref)


@pytest.mark.parametrize("kv_dtype", [W.FP8_E4M3, W.INT8])
def test_nonfinite_inputs_follow_saturating_reading(kv_dtype):
    # reading (parity unpinned by the pages): E4M3 NaN->0x7F, Inf->+-448;
    # INT8 NaN->0, Inf->+-127
    x = _all_fp16(include_nonfinite=True)
    T = len(x) // 128
    got, ref, st = _run(kv_dtype, x, x, 1, 0.75, 0.75, np.arange(T), T // 16 + 1)
    assert np.array_equal(got, ref)


def test_per_head_scales_and_strided_inputs_int8():
    rng = np.random.default_rng(2)
    H, T = 8, 300
    k = (rng.normal(0, 1, (T, H, 128)) * np.where(rng.random((T, H, 128)) < 0.01, 20, 1)).astype(np.float16)
    v = rng.normal(0, 3, (T, H, 128)).astype(np.float16)
    ks = (np.abs(k).reshape(T, H, -1).max(axis=(0, 2)) / 127).astype(np.float32)
    vs = (np.abs(v).reshape(T, H, -1).max(axis=(0, 2)) / 127).astype(np.float32)
    slots = rng.permutation(40 * 16)[:T]
    got, ref, st = _run(W.INT8, k.ravel(), v.ravel(), H, ks, vs, slots, 40, k_stride=(H + 4) * 128)
    assert st == 0 and np.array_equal(got, ref)


def test_untouched_slots_negative_and_out_of_pool():
    rng = np.random.default_rng(3)
    H, T = 2, 64
    x = rng.normal(0, 1, (T, H, 128)).astype(np.float16)
    slots = np.arange(T) * 3
    slots[5] = -1
    slots[9] = -7
    got, ref, st = _run(W.FP8_E4M3, x.ravel(), x.ravel(), H, 0.01, 0.02, slots, 13)
    assert st == 0 and np.array_equal(got, ref)
    # a slot past the pool is skipped and reported
    pq = require_gpu()
    pages = pq.new_pages(2, 1, W.FP8_E4M3, "cuda", fill=7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kk = torch.ones((2, 1, 128), dtype=torch.float16, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    pq.kv_append_quant(kk, kk, torch.tensor([3, 32], dtype=torch.int64, device="cuda"),
                       W.FP8_E4M3, one, one, pages, status=status)
    assert pq.status_bits(status) == ["slot beyond the pool"]
    p = pages.cpu().numpy()
    assert (p[0, 0, :, 3] == 0x38).all()
    p[0, 0, :, 3] = 7
    assert (p == 7).all()


def test_bad_scale_reported_and_skipped():
    pq = require_gpu()
    pages = pq.new_pages(1, 1, W.INT8, "cuda", fill=9)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kk = torch.ones((1, 1, 128), dtype=torch.float16, device="cuda")
    bad = torch.tensor([0.0], dtype=torch.float32, device="cuda")
    pq.kv_append_quant(kk, kk, torch.tensor([0], dtype=torch.int64, device="cuda"), W.INT8,
                       bad, bad, pages, status=status)
    assert "bad scale" in pq.status_bits(status)
    assert (pages.cpu().numpy() == 9).all()


@pytest.mark.parametrize("name", ["int8_decode_append_262k", "e4m3_verify_512k_stress"])
def test_workload_pools_bit_exact(name):
    w = W.workload(name, scale=0.004)
    c = Case(w)
    assert np.array_equal(c.gpu_pool_bytes(), c.pool_o)


def test_fragmented_8192_token_chunk_bit_exact():
    # the long-context stress workload's append: 8192 tokens starting at offset
    # 7 inside a page of a fragmented pool
    pq = require_gpu()
    w = W.workload("e4m3_verify_512k_stress", scale=0.004)
    w.append_tokens = 8192
    plan = W.plan_pool(w)
    ks, vs = W.calibrated_scales(w, "cuda")
    k, v = W.append_chunk(w, "cuda")
    pages = pq.new_pages(plan.num_pages, w.num_kv_heads, w.kv_dtype, "cuda", fill=0x11)
    pq.kv_append_quant(k, v, torch.from_numpy(plan.append_slots).cuda(), w.kv_dtype, ks, vs, pages)
    pool = oracle.new_pool(plan.num_pages, w.num_kv_heads, 128, w.kv_dtype, fill=0x11)
    ref = oracle.kv_append_quant(k.cpu().numpy(), v.cpu().numpy(), plan.append_slots, w.kv_dtype,
                                 ks.cpu().numpy(), vs.cpu().numpy(), pool)
    assert np.array_equal(pages.cpu().numpy(), ref)


def test_generator_is_identical_on_cpu_and_gpu():
    require_gpu()
    a = W.draw_values(5, W.KIND_K, 2, 100, 4196, 8, 128, True, "cuda").cpu()
    b = W.draw_values(5, W.KIND_K, 2, 100, 4196, 8, 128, True, "cpu")
    assert torch.equal(a, b)
