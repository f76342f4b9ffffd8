"""Plain CPU oracle of the ZeRO-DP partitioned mixed-precision AdamW step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the library's product path never
does.  It shares no code with the CUDA path.

* ``oracle/zero_oracle.c`` — per-element arithmetic in plain C (16-bit decode
  and round-to-nearest-even encode, the gradient reduction, 128-element chunk
  sums of squares, AdamW), one binary32 rounding per operation;
* ``oracle/layout.py`` — flat layout, shards, buckets, ZeRO-3 units, memory
  and communication accounting (plain Python integers and Fractions);
* ``oracle/step.py`` — the DDP reference (the plain definition) and the literal
  ZeRO-1/2/3 simulation, plus a sampled per-element form for full-size buffers.

Pins (tests marked ``not gpu``): the pages' memory tables and worked values,
the exact communication-volume forms, brute-force layout checks, library
round-to-nearest-even casts, exact rational sums, the closed form of AdamW
under a constant gradient, ``torch.optim.AdamW`` at N_d = 1, the closed-form
norm of a constant gradient, the fp16 overflow skip, and ZeRO-k == DDP; for
gradient accumulation, exact rational bounds for both summation orders and
M = 1 == the plain step; the sampled form (``SampledElements``,
``FullSumsq``) reproduces the whole-buffer simulation bit for bit; and
planted mistakes (bias correction, decay, betas, eps, coupled decay, a dropped
rank, the divisor) each fail one of the pins.
"""
