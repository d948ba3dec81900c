"""CPU oracle for the EAGLE-3 training-time-test (TTT) draft-step core.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously
correct statement of what the GPU path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product path (the C-ABI library and
its Python binding) never imports, calls or links anything here, and this
package imports nothing from the product.

Everything is NumPy float64 on the host.  Each function cites the passage of
the source page it follows; the page is the xllm-io review of
"SpecForge: A Flexible and Efficient Open-Source Training Framework for
Speculative Decoding" (cited below as "SpecForge review").

Modules
-------
mask       the BlockMask predicate M (SpecForge review, §三 "BlockMask
           构造算法" and §四 "BlockMask 构造"), element by element.
attention  masked softmax attention over the concatenated TTT KV blocks,
           forward and backward, written from the definition.
soft_ce    the masked soft-target softmax cross-entropy and its in-place
           gradient (SpecForge review, §三 "内存高效梯度计算", §四
           "掩码 Softmax 损失" / "原地反向传播"), per-row or per-element g.
lm_head    the draft's LM head z = h W^T followed by the soft-CE: loss and
           the gradients of h and W.
verify     speculative-decoding verification by rejection sampling (the
           "FlashSpec" practice page, §3.4 "验证器的具体实现").

Readings of the page where it is silent:
  * kv indexes the concatenation of k+1 blocks, each Q_LEN long; block 0 is
    the causal block (implied by the ``mod Q_LEN`` terms of the mask).
  * Query head h uses KV head h // (H / H_kv).
  * lse is the natural-log logsumexp of the scaled scores; the scale is an
    argument (1/sqrt(D) in every workload).
  * A row with no unmasked key (only when T = 0) has O = 0, lse = -inf and
    contributes no gradient.            -> convention, parity unpinned
  * Per-call gradients are overwritten, not accumulated.  -> convention
  * The soft-CE loss returned is L = sum_r g_r * l_r; the per-row loss
    reported for a row with g_r = 0 is 0 (the row is masked out of the
    loss).                                -> convention, parity unpinned
"""

from . import mask, attention, soft_ce, lm_head, verify  # noqa: F401

__all__ = ["mask", "attention", "soft_ce", "lm_head", "verify"]
