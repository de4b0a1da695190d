"""Oracle for paged KV-cache decode: plain, slow, obviously correct CPU code.

TEST INFRASTRUCTURE ONLY.  ``reference`` is a numpy/float64 restatement;
``native`` loads the C/float64 twin (``pa_oracle.c``, OpenMP).  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It shares no code with the CUDA library.
"""
