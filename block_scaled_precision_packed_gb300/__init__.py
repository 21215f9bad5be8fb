"""bsq: block-scaled packed-precision matrix products for one GB300 (sm_103a).

The compute path is the C-ABI library ``libbsq.so`` (hand-written CUDA, built
by ``build``); ``bsq`` is its thin Python binding.  ``synthetic`` draws the
seeded workloads the tests and the benchmark share.
"""
