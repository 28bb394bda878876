"""Oracle: a plain, slow, float64 CPU restatement of paged KV-cache decode.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.  The
product path (the CUDA library and its Python binding) never imports, calls or
links anything here, and nothing here imports the product.  The two share only
the seeded input generators in ``pkv_workloads`` (which hold none of the
method's arithmetic).

Every function cites the web page and section it restates.  The pages are five
articles about the KV cache; their titles, as used in the citations, are:

* "What a KV cache is and why it is the crux of LLM inference"
  (a practitioner essay; sections 1-5, e.g. 2.2 "three design consensuses",
  3.1 memory layout, 3.2 life cycle, 3.3 quantisation, 4.2 a minimal cache).
* "KV Cache, the memory notepad of LLM inference"
  (an explainer; sections 一..十: 二 the attention formula, 三 prefill/decode,
  四 a NumPy toy, 五 a memory formula, 六 GQA/MQA/paging/quantisation).
* "Series 03: why the KV cache eats memory, and how PagedAttention pages it"
  (sections 1.2 the size formula, 2.3 shared prefixes, 3.1 block tables,
  3.2 on-demand allocation, 3.3 copy-on-write, 4.2 a memory budget).
* "KV cache capacity planning, from the budget to task-level regression"
  (sections 1 the size formula, 2 a budget calculator and length buckets,
  3 paging does not change precision, 4 FP8 KV cache, 5 FP8 roll-out).
* "KV Cache: principle and memory share (kp-013)"
  (sections 公式与模型 the byte formula and derivations, 图示 the decode
  diagram, 自测题 the self-test).

Modules
-------
kv_bytes     closed-form KV byte counts and the budget calculator.
block_pool   the physical block pool, refcounts and per-sequence block tables.
slots        slot mapping: logical position -> physical slot.
append       writing new K/V rows into their slots (a bit copy).
e4m3         the OCP FP8 E4M3 code table, encoder and decoder.
e5m2         the OCP FP8 E5M2 code table, encoder and decoder.
int8         INT8 codes with per-block min-max scaling (encode, decode, re-quantising append).
attention    paged decode attention and the contiguous (no-cache) comparator.
prefill      paged prefill / extend attention (causal over the cached context).
toy_model    a tiny projection model that recomputes K/V from scratch.
numerics     exact decoding of stored fp16 / bf16 bit patterns to float64.

Parity: every function is pinned by the tests in ``tests/test_oracle_*.py``
against closed forms, invariants or brute force; none is "parity unpinned".
"""
