"""CPU oracle for paged GQA attention: test infrastructure, not product code.

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  The CUDA path never calls it, and it
shares no code with the CUDA path: no kernels, headers, helpers or tables.

Everything here is plain NumPy in float64 (the e4m3 encoder decides its code
from a float32 quotient, the precision the write kernel uses).  Sources, by
page title and section:

* TensorFold PR #1373 ("paged batches take the tensor-core tiles"), "What
  changes": paged and contiguous (slab) streams read the same bytes, addressed
  by cache position through the page table or the slab.
* TensorFold PR #2011 ("pages by default; page looked up once;
  hpattn_p256_kernel"), review section "Is paged output the same as windowed
  output?": the page address ``PT[k0/256]*PS + (hk*256 + k0%256)*D`` and that
  masked keys contribute nothing.
* TensorFold Issue #1344 ("a batch takes the partial-only attention path"),
  "Mechanism": attention as split partials (running max, sum, unnormalised
  output) followed by a merge.
* The attention formula itself, the GQA head mapping, the causal rule and the
  e4m3 format are not stated on the pages; the readings taken are written in
  each module's docstring.

Modules:
  e4m3       OCP FP8 E4M3 ("fn") decode table and round-to-nearest-even,
             saturating encoder.
  kvcache    the physical cache (page pool or slab) and the KV row write.
  attention  one-pass softmax attention per (row, head), split partials and
             their log-sum-exp merge.

Parity status: every function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``; none is "parity unpinned".
"""

from . import e4m3, kvcache, attention  # noqa: F401
