"""CPU oracle for the paged decode-attention path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or run anything in this package.  The product path
(the C-ABI library and its Python binding) never calls it, and this package
imports nothing from the product: the two share no code.  Inputs reach both
sides from the seeded generator in ``paged_kv_cache_73_gb300.workloads``,
which holds none of the method's arithmetic.

Sources (three web pages on vLLM / PagedAttention, SOSP 2023):

* [note]    "vLLM / PagedAttention -- 把 LLM 服务的瓶颈从显存碎片里救出来"
            (awesome.papernotes.org, era5_genai_explosion/2023_vllm)
* [lecture] "vLLM" lecture notes (formulaic.cloudchewie.com,
            docs/large-language-models/llm-inference/5-vllm)
* [guide]   "vLLM / PagedAttention (SOSP 2023)" (upskillscore.com,
            guides/system-design/genai-vllm-pagedattention)

Modules:

* ``attention``     -- single-query attention over a paged K/V pool, fp64.
* ``cache_ops``     -- the slot-mapping scatter of new K/V and the block copy.
* ``block_manager`` -- block tables, free list, reference counts, copy-on-write.
* ``sizes``         -- K/V bytes per token.

Every function is pinned by a ``-m "not gpu"`` test against facts fixed
outside it (the pages' worked examples, a library attention routine, closed
forms, invariants); none is "parity unpinned".
"""
