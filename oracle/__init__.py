"""Plain fp64 CPU oracle for packed variable-length context-parallel attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run this package.
The library under ``context_attention_cpattn_gb300`` never imports it, and it
imports nothing from the library: the two share no code.  The only common
dependency is the seeded input module ``inputs``, which holds no arithmetic of
the method.

Contents and the passages each follows:

* ``attention`` - softmax attention inside each packed sequence, written out
  from its definition (THD packing with cu_seqlens: "Speeding up
  Variable-Length Training with Dynamic Context Parallelism and NVIDIA
  Megatron Core", section on dynamic rescheduling and packing, Fig. 1; the
  result must not depend on how the sequence is split: "Scaling video
  training with parallelism", opening section).  Also the attention of a
  query-row set over a key-row set (one ring step's block, "Scaling video
  training with parallelism", section 2, Ring Attention).
* ``attention_bwd`` - fp64 gradients dQ, dK, dV of the packed attention from
  the chain rule, and one ring step's backward block using the final O and
  LSE (the pages train with blockwise ring attention: "Scaling video training
  with parallelism", section 2).
* ``merge`` - the exact log-sum-exp merge of block partials.  The pages name
  blockwise attention with a KV ring but not the merge; the merge written
  here is the plain identity that recombines softmax partials exactly.
* ``plan`` - zigzag, 2-D h x w and contiguous context-parallel splits and the
  ring schedule (LongVILA news article, Fig. 5 / Table 2 ZIGZAG-RINGATTN;
  LongCat-Video context-parallel article, tensor split strategy and its FAQ;
  "Scaling video training with parallelism", section 3, Fig. 2).
* ``loss`` - per-token loss normalisation over valid tokens (Dynamic-CP
  article, section "Loss computation and FLOPS statistics").
* ``flops`` - THD-aware FLOP count from real sequence lengths (same section).
* ``teacher_forcing`` - LongLive-2.0's clean/noisy pairs: the teacher-forcing
  mask, dense masked attention, the paired plan ("Scaling video training with
  parallelism", section 4).  The mask is a reading of a truncated page:
  parity partly unpinned.
* ``dcp`` - the Dynamic-CP scheduler: Eq. 1-3 quotas, per-sample CP size,
  packing into micro-batches and the micro-batch count sweep (Dynamic-CP
  article, data-scheduling and runtime sections).

Every function here is pinned by ``tests/test_oracle_*.py`` against brute
force, closed forms, library routines and invariants.  Two are partial:
``dcp.schedule`` follows a prose heuristic and ``teacher_forcing.allowed`` a
mask the page does not finish stating, so past their pins their parity is
unpinned.
"""

from . import attention, attention_bwd, dcp, flops, loss, merge, plan, teacher_forcing  # noqa: F401
