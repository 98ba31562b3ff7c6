"""CPU fp64 oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product (the CUDA library and its binding) never touches it, and it shares no
code with the product: no kernels, headers, helpers or constants.

Contents
--------
``attn_fp64.c``   the materialising definition (forward and analytic backward),
                  plain C with OpenMP over rows; built into ``_build/liborattn.so``.
``reference.py``  ctypes wrapper of the C oracle (``attn_fwd``, ``attn_bwd``).
``brute.py``      pure-Python triple loops for tiny shapes (second, independent
                  transcription of the same definition).
``online.py``     a separate CPU online-softmax forward (tile by tile, running
                  max and sum, rescale when the max grows), used to pin the
                  exactness claim of the tiled method.
``fp8.py``        attention on FP8 (e4m3) operands: block or per-tensor scaling and
                  the incoherent-processing rotation, for the FP8 variant.

Every function cites the passage of the pages it follows.  Pins (tests that
check the oracle against something other than itself) live in
``tests/test_oracle_pins.py``.
"""
