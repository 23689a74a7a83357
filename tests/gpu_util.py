"""Helpers shared by the GPU parity tests: build the oracle's pools from the
seeded inputs, move arrays to the device, and run the oracle on a workload."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oatt
from oracle import formats as ofmt

TOL = {"f32": 1e-4, "f16": 2e-3, "q8_0": 2e-3}


def dev():
    return torch.device("cuda:0")


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(dev())


def oracle_pools(w):
    """Pool bytes as the oracle stores the workload's history rows."""
    kp = ofmt.encode_rows(w.fmt, w.k_hist, w.n_kv_heads, w.head_dim)
    vp = ofmt.encode_rows(w.fmt, w.v_hist, w.n_kv_heads, w.head_dim)
    return kp, vp


def oracle_decode(w, kp, vp, table=None, seqs=None, heads=None):
    table = w.block_table if table is None else table
    return oatt.paged_attn_decode(w.fmt, w.q, kp, vp, table, w.context_lens, w.spans,
                                  w.n_heads, w.n_kv_heads, w.head_dim, w.block_size, w.scale,
                                  seqs=seqs, heads=heads)


def gpu_decode(mt, w, k_pool, v_pool, table=None, n_ctas=0, context_lens=None, spans="w"):
    table = w.block_table if table is None else table
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device=dev())
    sp = None
    if isinstance(spans, str):
        sp = None if w.spans is None else to_dev(w.spans)
    elif spans is not None:
        sp = to_dev(spans)
    ctx = to_dev(w.context_lens if context_lens is None else context_lens)
    args = mt.paged_attn_args(w.fmt, q, k_pool, v_pool, to_dev(table), ctx, out,
                              n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                              n_phys_blocks=w.n_phys_blocks, scale=w.scale, spans=sp, lse=lse,
                              n_ctas=n_ctas)
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args), dtype=torch.uint8, device=dev())
    mt.mt_paged_attn_decode(args, ws)
    st = mt.mt_check_device_status(ws)
    return out.cpu().numpy(), lse.cpu().numpy(), st


def assert_close(got, want, tol, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got.astype(np.float64) - want).max() if got.size else 0.0
    assert err <= tol, f"{what}: max |err| {err:.3g} > {tol}"
    return err


def assert_lse(got, want, tol, what=""):
    inf = np.isinf(want)
    assert (np.isinf(got) == inf).all(), f"{what}: -inf pattern differs"
    assert (got[inf] < 0).all()
    if (~inf).any():
        err = np.abs(got[~inf] - want[~inf]).max()
        assert err <= tol, f"{what}: lse max |err| {err:.3g} > {tol}"
