"""SimSD speculative verification for diffusion LLMs on GB300 (sm_103a).

The hot path -- RoPE-copy + paged KV append, split-KV attention under the
token-level temporal causal mask, split merge, and rejection-sampling
acceptance along the temporal order -- runs in the CUDA kernels of
libsimsd.so behind the C ABI in include/simsd.h.  ``binding`` marshals torch
tensors into that ABI; ``staging`` moves host arrays into the device layouts
the ABI expects.  There is no CPU fallback.
"""
from .binding import (SimsdError, accept, accept_workspace_size, layout, lib,
                      prompt_append, read_status, status_string, verify_attn,
                      verify_workspace_size)

__all__ = ["SimsdError", "accept", "accept_workspace_size", "layout", "lib",
           "prompt_append", "read_status", "status_string", "verify_attn",
           "verify_workspace_size"]
