"""Float64 CPU oracle for ring-order attention, the zigzag partition, the LSE
merge and the context-parallel KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library; both sides receive the same seeded inputs from
``context_long_sequence_ring_gb300.inputs``.

Everything here is written from the pages' definitions, in their order and
notation, with numpy float64 and plain loops (a matmul is the only library
primitive).  Sources, by page title and section:

* "Parallelism-CP" diagram (scholia-log training-infra notes): Q/K/V are cut
  along the sequence across cards; K/V rotate around a ring; each card
  computes its own Q against all K; after wrapping around every Q block has
  seen every K/V block.
* guijiagi.com tag page "Ring Attention", article on the distributed
  challenge of long contexts, section "ring topology": step t, rank i works on
  the K/V block of rank (i - t) mod N and forwards what it holds to i + 1.
* same page, article on the attention memory wall, "key insight": the
  blockwise decomposition softmax(QK^T)V = sum_j e^{s_j} V_j / sum_j e^{s_j}
  with a running max and running sum updated per block.
* vLLM-Ascend developer guide "Context Parallel (CP)": section "Block table"
  (virtual blocks and the interleaved slot mapping, with the rule
  block_size % cp_kv_cache_interleave_size == 0), section "Prefill context
  parallel (PCP)" / head-tail token partition (pad, split into 2*pcp parts,
  pair part i with part 2*pcp-1-i, restore index), and the decode sections
  (partial outputs and LSEs merged by a cp_lse_ag_out_rs-style update).
* guijiagi.com tag page "Ring Attention", article on the evolution of
  long-context techniques, section 1.2 "RoPE": the rotary position embedding
  of query and key rows.

Parity status of every function is recorded in its docstring; all are pinned
by the ``-m "not gpu"`` tests (closed forms, hand-worked golden values,
invariants and brute force on tiny inputs).
"""

from .attention import (full_attention, attention_rows, attention_block, segmented_attention,
                        ring_attention, ring_partials, ring_step, lse_merge, rank_chunks,
                        causal_pairs_per_rank, causal_tiles_per_rank)
from .partition import zigzag_partition, gather_rows
from .rope import rope_theta, rope_cos_sin, rotate_half, apply_rope, rope_gather
from .kvcache import (cp_slot_mapping, cp_token_location, cp_kv_scatter, cp_kv_gather,
                      cp_decode, cp_decode_partials, cp_lse_ag_out_rs, decode_reference)

__all__ = [
    "full_attention", "attention_rows", "attention_block", "segmented_attention",
    "ring_attention", "ring_partials", "ring_step",
    "lse_merge", "rank_chunks", "causal_pairs_per_rank", "causal_tiles_per_rank",
    "zigzag_partition", "gather_rows", "cp_slot_mapping", "cp_token_location",
    "cp_kv_scatter", "cp_kv_gather", "cp_decode", "cp_decode_partials", "cp_lse_ag_out_rs",
    "decode_reference",
    "rope_theta", "rope_cos_sin", "rotate_half", "apply_rope", "rope_gather",
]
