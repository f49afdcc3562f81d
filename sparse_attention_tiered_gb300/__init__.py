"""GB300-native (sm_103a) SPIN sparse-decode data path.

The compute path is the CUDA library libspin.so (C ABI in include/spin.h);
this package only builds it, loads it and marshals arguments.
"""
from ._binding import (EXPORTS, SpinError, load, spin_append_kv, spin_create, spin_set_buffer, spin_debug_export, spin_debug_read_page,  # noqa: F401
                       spin_debug_summaries, spin_decode_step, spin_decode_step_host, spin_destroy,
                       spin_index_offload, spin_last_error, spin_measure_host_read, spin_select_noalloc, spin_stats)
from .context import SpinContext  # noqa: F401
