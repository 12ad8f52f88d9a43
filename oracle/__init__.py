"""Plain, slow CPU oracle of the Flash-dLLM per-layer denoising-step hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import or call it. It shares no
code with the CUDA library and never reads anything the CUDA library wrote.

Everything is computed in float64 from the exactly-widened inputs. Where a
stored tensor has a storage dtype (bf16 or fp32), the oracle rounds its
float64 result to that dtype at the same point the pages' data flow stores it
(the KV cache and the query buffer); decisions (commit, accept, top-k) are
taken on float64 values.

Every function cites the passage it follows. Pages cited:
  [FD]  "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding for Fast,
        Memory-Efficient Diffusion LLMs" (paper digest): sections "Background",
        "Core method", "Method steps in detail" (Algorithm 2 steps 1-4,
        Eq. (2)), "Reproduction" (hyper-parameters).
  [FA]  "What is Flash-dLLM? ..." article: section "How does Flash-Verify let
        the model draft and verify itself?".
  [FAST] Fast-dLLM news piece: sections "Confidence-aware parallel decoding"
        and the key-value cache for block-wise decoding (PrefixCache,
        DualCache; oracle/refresh.py).
  [FREE] FlashDLM note: key design 1, FreeCache (oracle/refresh.py).

Readings of silent or conflicting points (RoPE convention, view-visibility
rule, acceptance order, tie-breaks, ...) are listed in the repository's
design notes; each function states the reading it uses.

Parity status: every function below is pinned by tests/test_oracle_pins.py
(closed forms, hand-worked golden fixtures, invariants, brute force), and the
refresh policies of oracle/refresh.py by tests/test_refresh_pins.py. The
accuracy effect of the selective refresh itself is out of scope and not
modelled.
"""
from .flash_dllm import (  # noqa: F401
    KIND_NORMAL, KIND_WINDOW, store_round, slot_of, slot_map, work_list,
    project_qkv, rope, qkv_rope_cache_write, visible_positions, visible_keys,
    sched_attn, track_topk, row_confidence, unmask, verify, tv_point_mass,
    lm_head_logits, lm_head_unmask, lm_head_verify,
)
