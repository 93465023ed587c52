"""Tensor-level convenience over gqa_forward: derives the dims from torch
tensor shapes, keeps a reusable workspace, and raises on a non-OK status.
Marshalling only; the CUDA library does the work."""
from __future__ import annotations

from typing import Optional

import torch

from . import _binding as B

_DT = {torch.float16: B.GQA_DTYPE_FP16, torch.bfloat16: B.GQA_DTYPE_BF16}


class Workspace:
    """A grow-only device scratch buffer for gqa_forward.  It also remembers
    the dims struct and scratch size of the shapes it has served, so that a
    decode loop pays for them once."""

    def __init__(self, device=None):
        self.device = device
        self.buf: Optional[torch.Tensor] = None
        self.plans = {}

    def get(self, nbytes: int, device) -> Optional[torch.Tensor]:
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != torch.device(device):
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf


def dims_for(query, key, k_buf, num_heads, kv_num_heads, cos_cache=None, attention_bias=None,
             rotary_interleaved=0, past_seq_len=0, kv_eviction=0):
    """The dims struct of a call.  key None means packed QKV: query holds
    (num_heads + 2 kv_num_heads) heads per token."""
    Bsz, S, width = query.shape
    D = width // (num_heads if key is not None else num_heads + 2 * kv_num_heads)
    M = k_buf.shape[2]
    bb, bh = (attention_bias.shape[0], attention_bias.shape[1]) if attention_bias is not None else (1, 1)
    rows = cos_cache.shape[0] if cos_cache is not None else 0
    return B.make_dims(Bsz, S, num_heads, kv_num_heads, D, M, _DT[query.dtype], rotary_interleaved, rows, bb, bh,
                       past_seq_len, kv_eviction)


def _plan(workspace, host, query, key, k_buf, num_heads, kv_num_heads, cos_cache, attention_bias,
          rotary_interleaved, total_sequence_length, local_window_size, past_seq_len=0, kv_eviction=0):
    key_ = (host, past_seq_len, kv_eviction, key is None, tuple(query.shape), query.dtype, tuple(k_buf.shape),
            num_heads, kv_num_heads,
            None if cos_cache is None else cos_cache.shape[0],
            None if attention_bias is None else tuple(attention_bias.shape[:2]), rotary_interleaved,
            int(total_sequence_length), int(local_window_size))
    plan = workspace.plans.get(key_)
    if plan is None:
        dims = dims_for(query, key, k_buf, num_heads, kv_num_heads, cos_cache, attention_bias, rotary_interleaved,
                        past_seq_len, kv_eviction)
        size = B.gqa_workspace_size_host if host else B.gqa_workspace_size
        plan = (dims, size(dims, total_sequence_length, local_window_size))
        if len(workspace.plans) > 64:
            workspace.plans.clear()
        workspace.plans[key_] = plan
    return plan


def forward(query, key, value, k_buf, v_buf, seqlens_k, total_sequence_length, num_heads, kv_num_heads,
            cos_cache=None, sin_cache=None, scale=0.0, local_window_size=0, attention_bias=None,
            output=None, workspace: Optional[Workspace] = None, stream=None, rotary_interleaved=0,
            past_key=None, past_value=None, kv_eviction=0):
    """One GroupQueryAttention step.  k_buf/v_buf are updated in place: with
    past_key/past_value None they are the shared past/present buffers;
    otherwise they are the present buffers, which become past + new, and
    past_key/past_value [B, Hkv, Mp, D] are read only.  key and value None:
    packed QKV in query.  kv_eviction=1: sliding-window cache that keeps the
    most recent max_seq_len tokens contiguously.  Returns the output tensor
    [B, S, H*D]."""
    workspace = workspace or Workspace()
    mp = 0 if past_key is None else past_key.shape[2]
    dims, nbytes = _plan(workspace, False, query, key, k_buf, num_heads, kv_num_heads, cos_cache, attention_bias,
                         rotary_interleaved, total_sequence_length, local_window_size, mp, kv_eviction)
    ws = workspace.get(nbytes, query.device)
    if output is None:
        output = query.new_empty(query.shape[:2] + (num_heads * dims.head_size,))
    if stream is None:
        stream = torch.cuda.current_stream(query.device)
    pk = k_buf if past_key is None else past_key
    pv = v_buf if past_value is None else past_value
    st = B.gqa_forward(dims, query, key, value, pk, pv, k_buf, v_buf, seqlens_k, total_sequence_length,
                       cos_cache, sin_cache, scale, local_window_size, attention_bias, output, ws,
                       0 if ws is None else ws.numel(), stream)
    if st != B.GQA_OK:
        raise B.GqaError(st)
    return output


def forward_host(query, key, value, k_buf, v_buf, seqlens_k, total_sequence_length, num_heads, kv_num_heads,
                 cos_cache=None, sin_cache=None, scale=0.0, local_window_size=0, attention_bias=None,
                 output=None, workspace: Optional[Workspace] = None, stream=None, rotary_interleaved=0,
                 past_key=None, past_value=None, kv_eviction=0):
    """forward() with query/key/value/seqlens_k and the output as pinned CPU
    tensors (gqa_forward_host); k_buf, v_buf (and past_key/past_value in the
    non-shared binding), the caches and the bias stay on the device.  The
    returned output is valid once `stream` has reached the end of the step
    (synchronise it before reading)."""
    workspace = workspace or Workspace()
    dev = k_buf.device
    mp = 0 if past_key is None else past_key.shape[2]
    dims, nbytes = _plan(workspace, True, query, key, k_buf, num_heads, kv_num_heads, cos_cache, attention_bias,
                         rotary_interleaved, total_sequence_length, local_window_size, mp, kv_eviction)
    ws = workspace.get(nbytes, dev)
    if output is None:
        output = torch.empty(query.shape[:2] + (num_heads * dims.head_size,), dtype=query.dtype, pin_memory=True)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    pk = k_buf if past_key is None else past_key
    pv = v_buf if past_value is None else past_value
    st = B.gqa_forward_host(dims, query, key, value, pk, pv, k_buf, v_buf, seqlens_k, total_sequence_length,
                            cos_cache, sin_cache, scale, local_window_size, attention_bias, output, ws,
                            0 if ws is None else ws.numel(), stream)
    if st != B.GQA_OK:
        raise B.GqaError(st, "gqa_forward_host")
    return output
