"""GB300-native Sparse Delta Memory (SDM) hot path.

The chunked write/read op and the single-token decode step run as hand-written
sm_103a CUDA kernels in libsdm_gb300.so behind the C ABI of include/sdm.h.  This
package is the thin Python binding: ``sdm_write_read``, ``sdm_decode_step`` and the
training pair ``sdm_write_read_train`` / ``sdm_write_read_backward`` and the layer forward
``sdm_layer_forward`` take torch CUDA tensors and pass their pointers through.  Importing it loads the library
and fails loudly if it has not been built (``python gated_delta_rule_factor_gb300/build.py``).
"""

from . import _abi
from ._abi import SdmError, SdmShape
from .ops import (backward_workspace_size, decode_workspace_size, last_device_error, launch_count,
                  layer_backward_workspace_size, layer_workspace_size, make_shape, profile_begin, profile_end,
                  sdm_decode_step, sdm_layer_backward, sdm_layer_forward, sdm_layer_forward_train,
                  sdm_write_read,
                  sdm_write_read_backward, sdm_write_read_static, sdm_write_read_train,
                  snapshot_bytes, test_factor_scores, test_force_simt_scorer, test_force_write_read_layout,
                  test_stall_decode_copy, write_read_workspace_size)

lib = _abi.load()

__all__ = [
    "SdmError", "SdmShape", "backward_workspace_size", "decode_workspace_size", "last_device_error",
    "launch_count", "layer_backward_workspace_size", "layer_workspace_size", "make_shape", "profile_begin", "profile_end", "sdm_decode_step", "sdm_layer_backward", "sdm_layer_forward",
    "sdm_layer_forward_train",
    "sdm_write_read", "sdm_write_read_backward", "sdm_write_read_static", "sdm_write_read_train", "snapshot_bytes",
    "test_factor_scores", "test_force_simt_scorer", "test_force_write_read_layout", "test_stall_decode_copy",
    "write_read_workspace_size", "lib",
]
