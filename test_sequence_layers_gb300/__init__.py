"""GB300-native forward pass of the Test-Time-Training (TTT) layer.

The compute path is the CUDA library ``libttt.so`` (C ABI in ``include/ttt.h``);
``abi`` is its Python binding and ``synth`` the seeded synthetic-input generator.
"""
from .abi import (TTTError, ttt_launch_count, ttt_linear_fwd, ttt_mlp_fwd,  # noqa: F401
                  ttt_sync_status)
