"""CPU oracle for the MiniMax-M3 NVFP4 lightning indexer.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
NumPy (float64) statement of what the indexer computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  It shares no code with the CUDA library in
``sparse_attention_block_nvfp4_gb300`` and never imports it; the only module
both sides use is ``workloads`` (seeded inputs, no indexer arithmetic).

What it follows (page: vllm.models.minimax_m3.nvidia.indexer_nvfp4):
  * the module description: the index-K side cache holds packed NVFP4 pages
    ``[num_blocks, 128, 72]`` (E2M1 codes, then E4M3 block scales, no global
    scale); index-Q is E4M3; the indexer writes 15 score-ranked history pages
    plus the query's local page last (init_blocks=0, local_blocks=1) as
    logical block ids;
  * ``MiniMaxM3IndexerNvfp4Impl.__init__``: top-k 16, 128-token blocks,
    head dim 128, "max" scoring;
  * ``_build_prefill_chunks``: only pages before the last query's local page
    are scored (history pages = (seq_len - 1) // 128);
  * page vllm.models.minimax_m3.nvidia.indexer_flashinfer, builder ``build``:
    per-token valid pages = position // 128 + 1; ``forward``: scores are
    unscaled, tokens are right-aligned to the sequence end; top-k output is
    -1 tail-padded.

Readings the pages leave open are listed in each function's docstring.

Modules:
  formats  - E2M1 / E4M3 value tables, decoding and round-to-nearest-even.
  nvfp4    - NVFP4 page-row decoding and the quantise-insert.
  mxfp4    - MXFP4 page decoding and the OCP MX quantise-insert (page
             vllm.models.minimax_m3.amd.indexer_mxfp4: the same scores and
             top-k over [pages, 8704] e2m1 / e8m0 pages).
  norm_rope - qk-norm (RMSNorm) and RoPE of the index key before the NVFP4
             insert: the float64 definition, its bf16 rounding, the error
             bound of an fp32 evaluation and the row check built on it.
  indexer  - positions, page scores, selection; decode and prefill oracles.
  attend   - block-sparse attention over the selected pages of a bf16 main
             KV cache (the consumer of the [T, H, 16] id buffer), float64,
             with the error bound of an fp32 evaluation.
  brute    - scalar pure-Python brute force for tiny inputs (a pin).
  checker  - parity checker (ids modulo score ties within tolerance).

Parity pins (see tests/test_oracle_*.py): hand-worked byte examples under
tests/golden/, exhaustive format tables against torch / ml_dtypes casts,
scalar brute force, closed-form special cases, invariants, and planted
mistakes that each pin must catch.  No function here is "parity unpinned".
"""
from . import formats, nvfp4, norm_rope, indexer, checker, brute, attend  # noqa: F401
