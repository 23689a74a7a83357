"""GPU parity of the int4 cold-tier codec (bit-exact against the oracle) on
block shapes that take both kernel variants (values kept in registers, and
two passes for blocks of more than 16384 values) and both pool types."""
import numpy as np
import pytest
import torch

from oracle import formats as ofmt
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


@pytest.mark.parametrize("fmt,bs,hkv,d", [("f16", 16, 4, 256), ("f16", 32, 4, 256),
                                          ("f32", 16, 2, 64), ("f16", 16, 1, 64),
                                          ("f32", 32, 8, 128)])
def test_int4_round_trip_bit_exact(mt, fmt, bs, hkv, d):
    rng = np.random.default_rng(80 + bs + hkv + d)
    n_phys = 24
    rb = ofmt.row_bytes(fmt, hkv, d)
    vals = (rng.standard_normal((n_phys * bs, hkv * d)) * rng.uniform(0.1, 10)).astype(np.float32)
    vals[3 * bs:4 * bs] = 0.0  # an all-zero block: scale 0, nibbles 8
    pool = ofmt.encode_rows(fmt, vals, hkv, d)
    src = np.array([3, 7, 0, 23, 11], dtype=np.int32)
    dst = np.array([1, 2, 5, 9, 12], dtype=np.int32)
    n_el = bs * hkv * d
    dev = to_dev(pool)
    scales = torch.empty(len(src), dtype=torch.float32, device="cuda")
    nib = torch.empty(len(src), n_el // 2, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.mt_kv_quant_int4(fmt, dev, bs, hkv, d, n_phys, to_dev(src), scales, nib, status=status)
    mt.mt_kv_dequant_int4(fmt, dev, bs, hkv, d, n_phys, to_dev(dst), scales, nib, status=status)
    assert mt.mt_check_device_status(status) == 0
    g_s, g_n = scales.cpu().numpy(), nib.cpu().numpy()
    host = pool.copy()
    ty = np.float16 if fmt == "f16" else np.float32
    for i, (a, b) in enumerate(zip(src, dst)):
        s, n = ofmt.int4_quantize_block(pool[a * bs:(a + 1) * bs].view(ty))
        assert g_s[i].view(np.uint32) == np.float32(s).view(np.uint32)
        assert np.array_equal(g_n[i], n)
        host[b * bs:(b + 1) * bs] = ofmt.int4_dequantize_block(s, n, n_el, fmt).view(np.uint8).reshape(bs, rb)
    assert np.array_equal(dev.cpu().numpy(), host)
    # an out-of-range id is skipped and flagged
    bad = to_dev(np.array([n_phys + 3], dtype=np.int32))
    mt.mt_kv_quant_int4(fmt, dev, bs, hkv, d, n_phys, bad, scales, nib, status=status)
    assert mt.mt_check_device_status(status) == mt.MT_ERR_DEVICE_CHECK


def test_int4_codes_at_ties_and_tiny_scales(mt):
    # values placed exactly on and next to half-integer multiples of the
    # scale, plus a block whose amax is subnormal in f32
    fmt, bs, hkv, d = "f32", 16, 1, 32
    n_el = bs * hkv * d
    rng = np.random.default_rng(90)
    scale = np.float32(0.3)
    k = rng.integers(-7, 7, n_el).astype(np.float32)
    vals = ((k + 0.5) * scale).astype(np.float32)
    vals[::3] = np.nextafter(vals[::3], np.float32(np.inf))
    vals[1::3] = np.nextafter(vals[1::3], np.float32(-np.inf))
    vals[0] = 7 * scale
    blocks = [vals, (vals * np.float32(1e-38)).astype(np.float32),
              rng.standard_normal(n_el).astype(np.float32)]
    pool = np.concatenate([b.reshape(bs, hkv * d) for b in blocks]).astype(np.float32)
    pool_b = pool.view(np.uint8).reshape(3 * bs, -1).copy()
    src = np.array([0, 1, 2], dtype=np.int32)
    dev = to_dev(pool_b)
    scales = torch.empty(3, dtype=torch.float32, device="cuda")
    nib = torch.empty(3, n_el // 2, dtype=torch.uint8, device="cuda")
    mt.mt_kv_quant_int4(fmt, dev, bs, hkv, d, 3, to_dev(src), scales, nib)
    g_n = nib.cpu().numpy()
    for i in range(3):
        s, n = ofmt.int4_quantize_block(pool[i * bs:(i + 1) * bs])
        assert scales.cpu().numpy()[i].view(np.uint32) == np.float32(s).view(np.uint32)
        assert np.array_equal(g_n[i], n), i
