"""CPU baselines that bench.py reports beside the GPU numbers.

``allcore`` is an all-core C implementation (pthreads) of the row scan and of
the 1-D exclusive scan. It is a measurement baseline only: it is neither the
oracle (``oracle/``, single-threaded and fp64, which checks the GPU path) nor
a fallback, and the product package never imports it.
"""
