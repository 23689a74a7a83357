"""Decode without allocation: mt_paged_attn_decode_static.

Callers that cannot allocate device memory when they decode (a fixed memory
budget that must not grow, an embedder without an allocator, a thread that
must stay out of the CUDA allocator) use this entry point: it keeps its
split-K scratch in an array built into the library instead of a caller's
workspace. These checks call it through the C ABI twice in a row, on two
different workloads, and compare each result with the workspace entry point
on the same inputs, within the parity tolerances; compare a call made right
after a larger one (whose partial results are still in the shared array)
directly with the CPU oracle; and check that a call too large for the
built-in array is refused. This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, assert_lse, oracle_decode, oracle_pools, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def _args(mt, w, k_dev, v_dev):
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda")
    spans = None if w.spans is None else to_dev(w.spans)
    return mt.paged_attn_args(w.fmt, q, k_dev, v_dev, to_dev(w.block_table),
                              to_dev(w.context_lens), out, n_kv_heads=w.n_kv_heads,
                              block_size=w.block_size, n_phys_blocks=w.n_phys_blocks,
                              scale=w.scale, spans=spans, lse=lse)


def _both(mt, w):
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    ref = _args(mt, w, k_dev, v_dev)
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(ref), dtype=torch.uint8, device="cuda")
    assert 0 < ws.numel() <= mt.MT_STATIC_SCRATCH_BYTES
    mt.mt_paged_attn_decode(ref, ws)
    got = _args(mt, w, k_dev, v_dev)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.mt_paged_attn_decode_static(got, status=status)
    assert mt.mt_check_device_status(status) == 0
    assert mt.mt_check_device_status(ws) == 0
    o_ref, o_got = ref._tensors[5].cpu().numpy(), got._tensors[5].cpu().numpy()
    l_ref, l_got = ref._tensors[7].cpu().numpy(), got._tensors[7].cpu().numpy()
    return o_ref, o_got, l_ref, l_got


def test_static_scratch_matches_workspace_on_two_calls_in_a_row(mt):
    # first call: Llama-3-shaped f16; second call: q8_0 with windows, other
    # shapes, so stale scratch from the first call cannot pass for a result
    cases = [workloads.llama3_f16(seed=61, n_seqs=7, ctx_lo=30, ctx_hi=900),
             workloads.llama3_q8_prefix(seed=62, n_seqs=4, prefix=96, suffix_lo=5,
                                        suffix_hi=70)]
    for w in cases:
        o_ref, o_got, l_ref, l_got = _both(mt, w)
        tol = TOL[w.fmt]
        assert np.isfinite(o_got).all()
        assert np.abs(o_got - o_ref).max() <= tol, w.name
        fin = np.isfinite(l_ref)
        assert (np.isfinite(l_got) == fin).all()
        assert np.abs(l_got[fin] - l_ref[fin]).max() <= tol, w.name


def test_static_scratch_matches_oracle_after_a_larger_call(mt):
    # a larger call with other shapes leaves its partials in the shared
    # array; the next call must not read any of them
    big = workloads.llama3_f16(seed=64, n_seqs=24, ctx_lo=200, ctx_hi=3000)
    kp, vp = oracle_pools(big)
    a = _args(mt, big, to_dev(kp), to_dev(vp))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.mt_paged_attn_decode_static(a, status=status)
    assert mt.mt_check_device_status(status) == 0
    for w in (workloads.smollm2_f32(seed=65, n_seqs=3, ctx_lo=40, ctx_hi=300),
              workloads.llama3_q8_prefix(seed=66, n_seqs=5, prefix=64, suffix_lo=3,
                                         suffix_hi=90)):
        kp, vp = oracle_pools(w)
        a = _args(mt, w, to_dev(kp), to_dev(vp))
        mt.mt_paged_attn_decode_static(a, status=status)
        assert mt.mt_check_device_status(status) == 0
        want, want_lse = oracle_decode(w, kp, vp)
        got, got_lse = a._tensors[5].cpu().numpy(), a._tensors[7].cpu().numpy()
        assert_close(got, want, TOL[w.fmt], f"{w.name} static")
        assert_lse(got_lse, want_lse, TOL[w.fmt], f"{w.name} static")


def test_static_scratch_refuses_calls_that_do_not_fit(mt):
    w = workloads.llama3_f16(seed=63, n_seqs=3, ctx_lo=20, ctx_hi=60)
    kp, vp = oracle_pools(w)
    a = _args(mt, w, to_dev(kp), to_dev(vp))
    a.n_seqs = 40000  # scratch grows with the sequence count; nothing is launched
    assert mt.mt_paged_attn_workspace_bytes(a) > mt.MT_STATIC_SCRATCH_BYTES
    with pytest.raises(mt.MtError) as e:
        mt.mt_paged_attn_decode_static(a)
    assert e.value.status == mt.MT_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
