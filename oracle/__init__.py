"""CPU oracle for the paged GQA decode path — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement, in numpy, of what the path
computes: attention in float64 over each sequence's valid positions gathered
into a dense array, and the storage formats, cold-tier codec, ordered row
mover and grow-on-demand re-layout written out from their definitions.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg
(and its `--impl reference` arm) may import or run anything in this package.
The product path (the CUDA library and its Python binding) never imports it,
and this package imports nothing from the product path; the two share only
the seeded input generators of `paged_kv_cache_gqa_gb300.workloads`, which
hold none of the method's arithmetic.

Sources (web pages, cited by title and section):
  * "KV Cache Design — cells, format, sessions" (minfer): cells vs
    positions and the attn_span window (section 1); verbatim row moves and
    order_moves (section 2); KvFormat {f32, f16, q8_0}, the Q8_0 cell width
    and the store quantiser (section 3).
  * "Tiered KV cache — architecture" (llama.cpp memory tier): the
    paged-attention block model and kInvalidBlockId holes, kernel dispatch
    (-INFINITY logits for holes), the per-block int4-with-scale cold codec
    (section "The three-tier model").
  * "KV cache" (sipllm): grow-on-demand capacity doubling and the verbatim
    re-layout (section "Design").

Every function is pinned by `tests/test_oracle_*.py` against values fixed by
the pages or by mathematics (library routines, closed forms, invariants,
brute force); none is "parity unpinned".
"""
