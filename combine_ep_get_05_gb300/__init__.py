"""GB300 (sm_103a) expert-parallel dispatch / combine.

The single-GPU data-parallel hot path of MoE expert-parallel dispatch and
combine, with R virtual EP ranks held as slabs of one GPU's HBM:

  ep_get_layout      counts, is_token_in_rank / node, stable slots (one kernel)
  ep_dispatch        destination-major permute of bf16 rows or fused 1x128 E4M3
  ep_restripe_prob   prob [T][nodes][P] -> [nodes][max_tokens][P]
  ep_dispatch_nodes  node-level dense / sparse (run-length) dispatch
  ep_combine         fp32 ascending-rank gather-reduce back to token order
  ep_combine_fp8     the same from FP8 rows (E4M3 codes + 1x128 scales)
  ep_combine_weights the received top-k weight rows summed back to token order
  ep_get_expert_layout / ep_dispatch_permuted / ep_permute_received /
  ep_combine_permuted  the expert-major (dispatch + permute) path, fused or split
  ep_dispatch_permuted_ll  the same for a decode-sized batch in one launch
  ep_combine_send    send phase of a split combine (expert-major rows -> rank slabs);
                     ep_combine is its receive phase
  ep_combine_permuted_ll   the expert-major combine shaped for decode-sized batches

The C ABI is include/ep.h (libep_gb300.so, built in-tree by build.py); the
functions here with the same names are its ctypes binding, and api.py
allocates buffers and chains the calls.
"""
from ._lib import (  # noqa: F401
    ABI_VERSION, DTYPE_BF16, DTYPE_E4M3, EP_ERR_CUDA, EP_ERR_INVALID, EP_ERR_SCRATCH, EP_OK,
    LAYOUT_NOALLOC_SCRATCH_BYTES, EXPORTS, FLAG_BAD_EXPERT,
    FLAG_CAPACITY, FLAG_TIMEOUT, FLAG_WORKSPACE, NODES_DENSE, NODES_SPARSE, EpError, ep_combine, ep_dispatch,
    ep_dispatch_nodes, ep_get_layout, ep_get_layout_noalloc, ep_layout_workspace_size, ep_restripe_prob, lib,
    ep_combine_permuted, ep_dispatch_permuted, ep_expert_layout_workspace_size, ep_get_expert_layout,
    ep_permute_received, ep_combine_fp8, ep_combine_weights, ep_dispatch_permuted_ll, ep_combine_send,
    ep_combine_permuted_ll,
)
from .api import (  # noqa: F401
    Dispatched, Layout, alloc_dispatch, alloc_layout, combine, combine_fp8, combine_weights, dispatch, get_layout,
    read_flags,
)
from .build import LIB_PATH, build as build_library  # noqa: F401
