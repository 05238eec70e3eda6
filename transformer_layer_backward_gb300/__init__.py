"""GB300 (sm_103a) LoRA transformer layer backward.

The computation lives in the CUDA library ``lib/libtlb.so`` (C ABI declared in
``include/tlb.h``); this package loads it and marshals torch tensors into it.
Importing the package does not touch the GPU; ``load()`` fails loudly when the
library has not been built.
"""
from . import _abi
from ._abi import TlbError, load
from .api import (act_backward, adamw, adamw_cfg, adamw_cfg_of, attn_backward, debug_skip_barrier_arrival, ffn_backward, layer_acts,
                  layer_backward, layer_cfg, layer_cfg_of, layer_weights, launch_count, launch_names, linear_backward, linear_workspace, lora,
                  lora_grad_adamw, lora_grad_adamw_noalloc, profile_events,
                  rmsnorm_backward, rope_backward, softmax_backward, stack_backward, stack_workspace,
                  workspace, workspace_bytes, workspace_status)

__all__ = ["TlbError", "load", "act_backward", "adamw", "adamw_cfg", "adamw_cfg_of", "attn_backward", "debug_skip_barrier_arrival",
           "ffn_backward", "layer_acts", "layer_backward", "layer_cfg", "layer_cfg_of", "layer_weights", "launch_count", "launch_names", "linear_backward", "linear_workspace", "lora",
           "lora_grad_adamw", "lora_grad_adamw_noalloc", "profile_events", "rmsnorm_backward", "rope_backward", "softmax_backward",
           "stack_backward", "stack_workspace", "workspace", "workspace_bytes", "workspace_status", "_abi"]
