"""CPU oracle for one wavefront round of Wave Forcing's chunk-wise causal DiT.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` do.

It is plain, slow, obviously-correct fp64 numpy written from the paper
"Wave Forcing: Towards Speed-of-Light Streaming Video Generation"
(arXiv 2611.00859):

* ``schedule``  -- rounds, active set, store, anchor/history/eviction and the
  ordered context of each task (Sec. 2 Eq. 2; Sec. 3.1 Eq. 3-5; App. B.3
  "Round schedule and cache semantics"; App. B.4 Eq. 16; App. B.8).
* ``rope``      -- 3D rotary position embedding in fp64 (the pages only say
  "QKV projection and RoPE", Sec. 4.2; the axis split and pair convention are
  this project's reading, so RoPE parity is *internal*: parity unpinned
  against the paper for the convention, pinned by rotation invariants).
* ``attention`` -- dense softmax attention with a materialised boolean mask.
* ``round``     -- the whole round: token universe, mask M_WF(s, j) = 1[j >= s]
  (Sec. 3.1 Eq. 4) materialised token x token, and a sequential replay over
  the ordered contexts of Eq. 5 (App. B.6, Proposition 1).

It shares no code with the CUDA path; the only module both sides use is
``wf_synth`` (seeded random inputs, no method arithmetic).
"""
