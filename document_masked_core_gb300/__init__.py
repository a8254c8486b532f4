"""Document-masked core attention for GB300 (sm_103a).

Core attention softmax(Q K^T / sqrt(d)) V run as one launch over a rebatched
pool of CA-tasks (query shards of packed documents with their causal KV
context), forward, backward and the LSE merge of split-KV partial results.
The kernels live in libca.so (C ABI, include/ca.h); this package binds it with
ctypes and uses torch only for device memory and streams.
"""
from .capi import (CA_DTYPE_BF16, CA_DTYPE_FP32, CAError, Plan, dry_run, dry_run_workload, load,  # noqa: F401
                   merge, version)

__all__ = ["Plan", "merge", "dry_run", "dry_run_workload", "load", "version", "CAError", "CA_DTYPE_BF16", "CA_DTYPE_FP32",
           "alloc_forward", "alloc_backward", "workspace"]


def workspace(plan, device="cuda"):
    """Device workspace for ``plan`` (uint8, at least 16 bytes)."""
    import torch
    return torch.empty(max(16, plan.info()["workspace_bytes"]), dtype=torch.uint8, device=device)


def alloc_forward(plan, device="cuda"):
    """Uninitialised O and LSE buffers for ``plan``."""
    import torch
    info = plan.info()
    odt = torch.float32 if plan.o_dtype == CA_DTYPE_FP32 else torch.bfloat16
    o = torch.empty((info["total_q"], plan.num_q_heads, plan.head_dim), dtype=odt, device=device)
    lse = torch.empty((info["total_q"], plan.num_q_heads), dtype=torch.float32, device=device)
    return o, lse


def alloc_backward(plan, device="cuda"):
    """Uninitialised dQ, dK, dV buffers (bf16) for ``plan``."""
    import torch
    info = plan.info()
    dq = torch.empty((info["total_q"], plan.num_q_heads, plan.head_dim), dtype=torch.bfloat16, device=device)
    dk = torch.empty((info["total_kv"], plan.num_kv_heads, plan.head_dim), dtype=torch.bfloat16, device=device)
    dv = torch.empty_like(dk)
    return dq, dk, dv
