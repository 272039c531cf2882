"""Block-sparse attention decode over an NVFP4 KV cache, native on GB300 (sm_103a).

The decode path -- NVFP4 quantise-and-insert, FP8 indexer scan with top-16 +
recent block selection, split-context sparse GQA attention over the selected
blocks and the log-sum-exp merge -- runs in the CUDA kernels of ``libmsa.so``
behind the C ABI of ``include/msa.h``.  ``ops`` is the thin ctypes binding,
``workloads`` the seeded synthetic inputs, ``harness`` the device-side cache
fill used by tests and benchmarks.
"""

from . import ops, workloads  # noqa: F401
