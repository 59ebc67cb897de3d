"""Oracle for the splash-attention hot path: plain, slow, fp64, CPU only.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or
run anything in this package.  The CUDA library never imports it, and this
package imports nothing from the CUDA library: the two share no code.  The
only module both sides use is ``workloads`` (seeded random inputs, no
arithmetic of the method).

What it computes, and the passage each piece follows:

* ``masks``      -- the element-wise masks named on "Splash Attention: When
  the Mask Stops Being Arithmetic and Becomes the Loop", section "What is
  MaskInfo in splash attention?" (CausalMask, LocalMask, ChunkedCausalMask,
  a dense array).
* ``mask_info``  -- the block classifier (same page, "What is splash
  attention and how is it different from flash attention?" and "Does
  splash attention make every sparse mask faster?"), the MaskInfo arrays
  block_mask / data_next / mask_next / partial_mask_blocks / q_sequence and
  their integer downcast ("What is MaskInfo in splash attention?"), and the
  grid-shrink pass ("What does grid shrinking do in splash attention?").
* ``attention``  -- dense masked softmax attention and its analytic
  gradients, with the saved residuals and the rowsum(dO*O) term of "Flash
  Attention on a TPU, Line by Line", sections "What does the TPU flash
  attention kernel save for the backward pass?" and "Why does the TPU flash
  attention backward pass run two kernels instead of one?".
  Optional soft cap and attention sinks follow the ``logits_soft_cap`` and
  ``softmax_aux`` arguments of the EasyDeL ``blocksparse_attention``
  operator page.
* ``shards``     -- attention over one shard of the key axis (unnormalised
  accumulator, maximum, normaliser) and the merge of shards with the
  flash rescaling and one final divide (Splash page, "What does ring
  attention add on top of the splash kernel?").

Every function is pinned by ``tests/test_oracle_*.py`` against what the
pages print (block counts, grid widths, partial-block bytes), closed forms,
library routines on special cases, autograd and finite differences.
Parity pins: none unpinned (the values MaskInfo stores at empty, full and
padding cells are fixed by this library's own contract, stated in the
docstrings; the pages leave them open).
"""
from . import masks, mask_info, attention  # noqa: F401
