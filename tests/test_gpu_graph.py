"""CUDA-graph capture of a decode step through the C ABI.

The library's compute calls launch asynchronously on the caller's stream and
never synchronise, allocate or copy from the host, so a multi-layer step
(fused store + decode per layer, a cascade decode, a prefill) can be
captured once and replayed. A replay must reproduce the eager results
exactly: the kernels are deterministic and the graph holds the same
launches with the same arguments.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import oracle_pools, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def test_captured_step_replays_eager_results(mt):
    w = workloads.llama3_f16(seed=71, n_seqs=6, ctx_lo=40, ctx_hi=400)
    n_layers = 3
    kp, vp = oracle_pools(w)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    layers = []
    for _ in range(n_layers):
        k_dev, v_dev = to_dev(kp), to_dev(vp)
        q = torch.randn(w.n_seqs, w.n_heads, w.head_dim, generator=g, device="cuda")
        out = torch.zeros_like(q)
        kn = torch.randn(w.n_seqs, w.n_kv_heads * w.head_dim, generator=g, device="cuda")
        vn = torch.randn_like(kn)
        args = mt.paged_attn_args("f16", q, k_dev, v_dev, to_dev(w.block_table),
                                  to_dev(w.context_lens), out, n_kv_heads=w.n_kv_heads,
                                  block_size=w.block_size, n_phys_blocks=w.n_phys_blocks,
                                  scale=w.scale)
        layers.append((k_dev, v_dev, q, out, kn, vn, args))
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(layers[0][6]), dtype=torch.uint8,
                     device="cuda")
    # a cascade over the first 3 sequences (sharing the first block) and a
    # prefill of the last 4 positions of every sequence, in the same step
    table_c = w.block_table.copy()
    table_c[1:3, 0] = table_c[0, 0]
    qc = torch.randn(w.n_seqs, w.n_heads, w.head_dim, generator=g, device="cuda")
    oc = torch.zeros_like(qc)
    kc, vc = to_dev(kp), to_dev(vp)
    args_c = mt.paged_attn_args("f16", qc, kc, vc, to_dev(table_c), to_dev(w.context_lens), oc,
                                n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                                n_phys_blocks=w.n_phys_blocks, scale=w.scale)
    groups = [(0, 3, 1)]
    ws_c = torch.zeros(mt.mt_paged_attn_cascade_workspace_bytes(args_c, groups),
                       dtype=torch.uint8, device="cuda")
    q_start = torch.arange(0, 4 * w.n_seqs + 1, 4, dtype=torch.int32, device="cuda")
    qp = torch.randn(4 * w.n_seqs, w.n_heads, w.head_dim, generator=g, device="cuda")
    op = torch.zeros_like(qp)
    args_p = mt.prefill_args("f16", qp, kc, vc, to_dev(w.block_table), to_dev(w.context_lens),
                             q_start, op, n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                             n_phys_blocks=w.n_phys_blocks, scale=w.scale)
    ws_p = torch.zeros(mt.mt_paged_prefill_workspace_bytes(args_p), dtype=torch.uint8,
                       device="cuda")
    pools0 = [(k.clone(), v.clone()) for (k, v, *_r) in layers]

    def step():
        for (k_dev, v_dev, q, out, kn, vn, args) in layers:
            mt.mt_paged_attn_decode_append(args, kn, vn, ws)
        mt.mt_paged_attn_decode_cascade(args_c, groups, ws_c)
        mt.mt_paged_attn_prefill(args_p, ws_p)

    step()  # eager (also configures every kernel before capture)
    torch.cuda.synchronize()
    eager = [l[3].clone() for l in layers] + [oc.clone(), op.clone()]
    pools1 = [(l[0].clone(), l[1].clone()) for l in layers]
    assert any(not torch.equal(a[0], b[0]) for a, b in zip(pools0, pools1))  # rows stored

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in [l[3] for l in layers] + [oc, op]:
        t.zero_()
    for (k_dev, v_dev, *_r), (k0, v0) in zip(layers, pools0):
        k_dev.copy_(k0)
        v_dev.copy_(v0)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    got = [l[3] for l in layers] + [oc, op]
    for a, b in zip(got, eager):
        assert torch.equal(a, b)
    for (k_dev, v_dev, *_r), (k1, v1) in zip(layers, pools1):
        assert torch.equal(k_dev, k1) and torch.equal(v_dev, v1)
    for wsx in (ws, ws_c, ws_p):
        assert mt.mt_check_device_status(wsx) == 0
