"""Seeded synthetic inputs for GroupQueryAttention over a shared KV buffer.

This module only draws numbers and lays them out in the operator's input
layouts; it holds none of the operator's arithmetic.  It is the one module the
CUDA path's tests, the oracle's tests and the benchmark share.

Layouts (all row-major, element type T = fp16 or bf16):
  query            [B, S, H*D]
  key, value       [B, S, Hkv*D]          (the new tokens)
  k_buf, v_buf     [B, Hkv, M, D]         (shared past/present buffer, BNSH)
  seqlens_k        [B] int32              (past length of each sequence)
  cos, sin         [rows, D/2]            (rotary caches, an operator input)
  attention_bias   [Bb, Hb, S, total]     (optional)

The workloads follow the operator's description on the onnxruntime discussion
"Clarification about GroupQueryAttention behavior" (shared BNSH buffer of
max_sequence_length, attention_bias shape) and the rocMLIR "KV Cache" example
(a 32-token prompt with head size 8, then a decode step of 33 in a buffer of
max_seq_len), at the batch/head/length mixes listed in ``CONFIGS``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}

# A quiet NaN in each element type, used to fill buffer slots that no valid
# key may read (any unmasked read then poisons the output).
SENTINEL_BITS = {"fp16": 0x7E00, "bf16": 0x7FC0}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str              # "fp16" | "bf16"
    batch: int
    seq_len: int            # S: new tokens per sequence
    num_heads: int          # H
    kv_num_heads: int       # Hkv
    head_size: int          # D
    max_seq_len: int        # M
    past_lo: int            # past lengths drawn uniformly from [past_lo, past_hi]
    past_hi: int
    bias_shape: Optional[tuple] = None   # (Bb, Hb) or None; the last two dims are (S, total)
    bias_std: float = 0.5
    local_window_size: int = 0          # <= 0: full causal
    total_sequence_length: Optional[int] = None   # None: max_b(past_b) + S
    rotary: bool = True
    seed: int = 0
    kv_eviction: bool = False       # sliding-window cache: keep the max_seq_len most recent tokens
    packed: bool = False            # new rows as one packed query tensor [B, S, (H + 2 Hkv) * D]

    @property
    def group(self) -> int:
        return self.num_heads // self.kv_num_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny prefill+decode pair, batched decode, long prefill,
# chunked prefill with bias, long-context decode with and without a window.
CONFIGS = {
    "tiny_prefill": Workload("tiny_prefill", "fp16", 1, 32, 4, 2, 8, 64, 0, 0, seed=0),
    "tiny_decode": Workload("tiny_decode", "fp16", 1, 1, 4, 2, 8, 64, 32, 32, seed=0),
    "decode_b16": Workload("decode_b16", "bf16", 16, 1, 32, 8, 128, 4096, 1, 4095, seed=1),
    "prefill_2k": Workload("prefill_2k", "fp16", 4, 2048, 32, 8, 128, 4096, 0, 0, seed=2),
    "chunked_prefill": Workload("chunked_prefill", "fp16", 8, 128, 32, 8, 128, 4096, 0, 3968,
                                bias_shape=(1, 1), total_sequence_length=4096, seed=3),
    "chunked_overflow": Workload("chunked_overflow", "fp16", 1, 128, 32, 8, 128, 4096, 4000, 4000,
                                 bias_shape=(1, 1), total_sequence_length=4096, seed=103),
    "long_decode": Workload("long_decode", "bf16", 8, 1, 64, 8, 128, 32768, 16384, 32767, seed=4),
    "long_decode_w4096": Workload("long_decode_w4096", "bf16", 8, 1, 64, 8, 128, 32768, 16384, 32767,
                                  local_window_size=4096, seed=4),
    # the batched decode with its new rows in the packed QKV form
    "decode_b16_packed": Workload("decode_b16_packed", "bf16", 16, 1, 32, 8, 128, 4096, 1, 4095, seed=1,
                                  packed=True),
    # the batched decode on a full sliding-window cache (window = capacity =
    # 4096 slots): every step evicts the oldest token of every sequence
    "swa_decode_b16": Workload("swa_decode_b16", "bf16", 16, 1, 32, 8, 128, 4096, 4096, 8191,
                               local_window_size=4096, seed=5, kv_eviction=True),
}


def rotary_cache(rows: int, head_size: int, dtype: str, base: float = 10000.0):
    """cos/sin caches [rows, D/2]: entry (p, j) = cos/sin(p * base^(-2j/D)),
    evaluated in float64 and rounded to T.  The operator takes these caches as
    inputs; both the CUDA path and the oracle receive the same bits."""
    half = head_size // 2
    inv = base ** (-(torch.arange(half, dtype=torch.float64) * 2.0) / head_size)
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * inv[None, :]
    t = DTYPES[dtype]
    return torch.cos(ang).to(t).contiguous(), torch.sin(ang).to(t).contiguous()


def draw_past(w: Workload, gen: torch.Generator) -> torch.Tensor:
    if w.past_lo == w.past_hi:
        return torch.full((w.batch,), w.past_lo, dtype=torch.int32)
    return torch.randint(w.past_lo, w.past_hi + 1, (w.batch,), generator=gen, dtype=torch.int64).to(torch.int32)


def make_inputs(w: Workload, seed: Optional[int] = None, sentinel: bool = True,
                fill_past: bool = True, device: str = "cpu") -> dict:
    """Draw one batch of inputs for workload ``w``.

    Q/K/V and the past region of the buffer are N(0, 1); the bias is
    N(0, bias_std).  Buffer slots at or beyond each sequence's past length hold
    the NaN sentinel when ``sentinel`` is set, zeros otherwise.  The past
    lengths always come from a CPU generator; with ``device`` other than
    "cpu" the bulk tensors are drawn there (same distributions, other
    values), which is much faster for the large buffers."""
    seed = w.seed if seed is None else seed
    gen = torch.Generator().manual_seed(seed)
    dgen = gen if device == "cpu" else torch.Generator(device).manual_seed(seed)
    t = DTYPES[w.dtype]
    B, S, H, Hkv, D, M = w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len
    past = draw_past(w, gen)
    total = w.total_sequence_length if w.total_sequence_length is not None else int(past.max()) + S

    def randn(*shape):
        return torch.randn(*shape, generator=dgen, device=device)

    q = randn(B, S, H * D).to(t)
    k = randn(B, S, Hkv * D).to(t)
    v = randn(B, S, Hkv * D).to(t)

    bufs = []
    for _ in range(2):
        if sentinel:
            buf = torch.full((B, Hkv, M, D), SENTINEL_BITS[w.dtype], dtype=torch.int16, device=device).view(t)
        else:
            buf = torch.zeros(B, Hkv, M, D, dtype=t, device=device)
        if fill_past:
            for b in range(B):
                n = min(int(past[b]), M)    # an evicting cache holds at most M rows
                if n > 0:
                    buf[b, :, :n, :] = randn(Hkv, n, D).to(t)
        bufs.append(buf)

    rows = max(total, M)
    cos, sin = rotary_cache(rows, D, w.dtype) if w.rotary else (None, None)
    if cos is not None and device != "cpu":
        cos, sin = cos.to(device), sin.to(device)

    bias = None
    if w.bias_shape is not None:
        Bb, Hb = w.bias_shape
        bias = (randn(Bb, Hb, S, total) * w.bias_std).to(t)

    return {
        "workload": w, "query": q, "key": k, "value": v,
        "k_buf": bufs[0], "v_buf": bufs[1], "seqlens_k": past.to(device),
        "total_sequence_length": int(total), "cos": cos, "sin": sin,
        "attention_bias": bias, "scale": 1.0 / math.sqrt(D),
        "local_window_size": w.local_window_size,
    }


def bits(t: torch.Tensor):
    """Raw 16-bit patterns of a fp16/bf16 tensor as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def decode_bytes(w: Workload, past: torch.Tensor) -> int:
    """Algorithmic bytes of one decode call: the visible K and V rows of every
    (sequence, KV head), the query and the output, and the appended K/V row.
    On an evicting cache see evict_decode_bytes."""
    if w.kv_eviction:
        return evict_decode_bytes(w, past)
    e = 2
    L = past.to(torch.int64) + w.seq_len
    if w.local_window_size > 0:
        L = torch.clamp(L, max=w.local_window_size)
    kv = int(L.sum()) * w.kv_num_heads * w.head_size * e * 2
    qo = 2 * w.batch * w.seq_len * w.num_heads * w.head_size * e
    app = 2 * w.batch * w.seq_len * w.kv_num_heads * w.head_size * e
    return kv + qo + app


def evict_decode_bytes(w: Workload, past: torch.Tensor) -> int:
    """Algorithmic bytes of one decode call on the evicting cache: per
    (sequence, KV head), every cached K and V row that the step must read at
    least once -- those its token sees and those that move down -- read once,
    the moved rows written once, plus the query and output and the new row
    (read from the input, written to its slot)."""
    e, D, M, W = 2, w.head_size, w.max_seq_len, w.local_window_size
    row = D * e * 2                                 # one K row and one V row
    total = 0
    for pb in past.tolist():
        n_old = min(pb, M)
        n_keep = min(pb + 1, M)
        moved = n_keep - 1 if n_old + 1 > n_keep else 0
        seen = n_old if W <= 0 else min(n_old, W - 1)   # cached rows inside the window
        total += w.kv_num_heads * (max(moved, seen) * row + moved * row)
    total += 2 * w.batch * w.num_heads * D * e      # query in, output out
    total += 2 * w.batch * w.kv_num_heads * D * e   # new K and V rows written
    return total


def prefill_flops(w: Workload, past: torch.Tensor) -> int:
    """Algorithmic FLOPs of one prefill call: 4*D per visible (query, key) pair
    per query head (2 for Q.K^T, 2 for P.V); masked pairs are not counted."""
    S, W = w.seq_len, w.local_window_size
    pairs = 0
    for pb in past.tolist():
        for i in range(S):
            p = pb + i
            n = p + 1
            if W > 0:
                n = min(n, W)
            pairs += n
    return 4 * w.head_size * w.num_heads * pairs
