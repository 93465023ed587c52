"""Plain, slow CPU oracle for GroupQueryAttention over a shared BNSH KV buffer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg
use it.  It shares no code with the CUDA path.

Sources (page title, then the passage):
  [ORT]  "Clarification about GroupQueryAttention behavior" (onnxruntime
         discussion 29659): the shared past/present buffer of
         max_sequence_length (the quoted operator text), the failure when the
         buffer has no room (tianleiwu's reply), the attention_bias shape and
         the sliding-window cache that keeps only the min(total, capacity)
         most recent tokens contiguously (ZackyLake's SWA follow-up).
  [MLIR] "[TorchOnnxToTorch] Add pad+scatter KV cache and mask to GQA"
         (torch-mlir PR 4471), the PR description: position ids = arange plus
         the past length from seqlens_k, key rotary on kv_num_heads, seqlens_k
         is 0 for an empty past, scatter of the new K/V at seqlens_k, causal
         mask k_pos <= past_len + q_pos.
  [ROC]  "KV Cache" (rocMLIR discussion 1617), "Example": gemm0 = Q x K,
         softmax, gemm1 = QK x V over the grown sequence.

Precision.  Attention is computed in float64 from the T-rounded (fp16/bf16)
operands.  The rotary step ends in a rounding to T whose result is stored in
the buffer and must match bit for bit; that rounding decision is taken in
fp32 with a fixed operation order (no fused multiply-add), the precision the
GPU kernels use.

Every array of element type T is passed as its raw 16-bit patterns
(numpy uint16); ``dtype`` is "fp16" or "bf16".
"""
from __future__ import annotations

import numpy as np

STATUS_OK = 0
STATUS_INVALID_ARGUMENT = 1
STATUS_KV_OVERFLOW = 2


# ---------------------------------------------------------------------------
# IEEE 754 binary16 and bfloat16 <-> binary32.
# ---------------------------------------------------------------------------
def t_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of T bit patterns to float32."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    raise ValueError(dtype)


def f32_to_t(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> T bit patterns, round to nearest, ties to even."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "fp16":
        with np.errstate(over="ignore"):   # beyond 65504 -> inf, as IEEE says
            return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        # keep the upper 16 bits; add half an ulp of the kept part, plus one
        # when the kept part is odd, so that exact halves go to the even side
        keep_odd = (u >> np.uint64(16)) & np.uint64(1)
        r = ((u + np.uint64(0x7FFF) + keep_odd) >> np.uint64(16)).astype(np.uint16)
        nan = np.isnan(x)
        if nan.any():
            sign = ((u >> np.uint64(16)) & np.uint64(0x8000)).astype(np.uint16)
            r = np.where(nan, sign | np.uint16(0x7FC0), r)
        return r
    raise ValueError(dtype)


def t_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    return t_to_f32(bits, dtype).astype(np.float64)


# ---------------------------------------------------------------------------
# Step 1: positions and rotary embedding ([MLIR] PR description).
# ---------------------------------------------------------------------------
def positions(seqlens_k: np.ndarray, seq_len: int) -> np.ndarray:
    """Position of new token i of sequence b: past length plus i ([MLIR]:
    arange plus the past_seqlens offset; seqlens_k is 0 for an empty past)."""
    past = np.asarray(seqlens_k, dtype=np.int64)
    return past[:, None] + np.arange(seq_len, dtype=np.int64)[None, :]


def rotary(x_bits: np.ndarray, pos: np.ndarray, cos_bits: np.ndarray, sin_bits: np.ndarray,
           dtype: str, interleaved: bool = False) -> np.ndarray:
    """Rotary embedding of x [B, S, heads, D] at positions pos [B, S].  Pair j
    (j < D/2) is (x[j], x[j + D/2]) in the non-interleaved layout and
    (x[2j], x[2j + 1]) in the interleaved one; it is rotated by the angle
    whose cosine and sine are cos/sin[pos, j]:
        y1 = x1 * c - x2 * s
        y2 = x2 * c + x1 * s
    in fp32, products first, no fused multiply-add, then rounded to T."""
    D = x_bits.shape[-1]
    half = D // 2
    x = t_to_f32(x_bits, dtype)
    c = t_to_f32(cos_bits, dtype)[pos][:, :, None, :]   # [B, S, 1, D/2]
    s = t_to_f32(sin_bits, dtype)[pos][:, :, None, :]
    if interleaved:
        x1 = x[..., 0::2]
        x2 = x[..., 1::2]
    else:
        x1 = x[..., :half]
        x2 = x[..., half:]
    t1 = np.multiply(x1, c, dtype=np.float32)
    t2 = np.multiply(x2, s, dtype=np.float32)
    y1 = np.subtract(t1, t2, dtype=np.float32)
    t3 = np.multiply(x2, c, dtype=np.float32)
    t4 = np.multiply(x1, s, dtype=np.float32)
    y2 = np.add(t3, t4, dtype=np.float32)
    if interleaved:
        y = np.empty_like(x)
        y[..., 0::2] = y1
        y[..., 1::2] = y2
        return f32_to_t(y, dtype)
    return f32_to_t(np.concatenate([y1, y2], axis=-1), dtype)


# ---------------------------------------------------------------------------
# Step 0, non-shared binding only: the present state starts as the past
# ([ORT], ZackyLake's summary 2b: when past and present are different tensors,
# present is past + new; [MLIR] pad+scatter: the past rows come first and the
# new rows are scattered after them at seqlens_k).
# ---------------------------------------------------------------------------
def present_from_past(present_bits: np.ndarray, past_bits: np.ndarray, seqlens_k: np.ndarray) -> np.ndarray:
    """Return a copy of present [B, Hkv, M, D] whose slots [0, seqlens_k[b])
    of every KV head hold the same slots of past [B, Hkv, Mp, D].  Every
    other slot keeps its bits (the new rows land after the past ones in
    step 2)."""
    out = present_bits.copy()
    for b in range(present_bits.shape[0]):
        n = int(seqlens_k[b])
        out[b, :, :n, :] = past_bits[b, :, :n, :]
    return out


# ---------------------------------------------------------------------------
# Step 2: scatter-append into the shared buffer ([MLIR]; [ORT] quoted text).
# ---------------------------------------------------------------------------
def scatter_append(buf_bits: np.ndarray, new_bits: np.ndarray, seqlens_k: np.ndarray) -> np.ndarray:
    """Return a copy of buf [B, Hkv, M, D] with new token i of sequence b
    (new [B, S, Hkv, D]) written at slot seqlens_k[b] + i of every KV head.
    Every other slot keeps its bits."""
    out = buf_bits.copy()
    B, S = new_bits.shape[:2]
    for b in range(B):
        for i in range(S):
            out[b, :, int(seqlens_k[b]) + i, :] = new_bits[b, i]
    return out


# ---------------------------------------------------------------------------
# Step 3: masked attention ([ROC] Example; [MLIR] causal mask; [ORT] bias and
# sliding window).
# ---------------------------------------------------------------------------
def visible(past: int, seq_len: int, window: int) -> np.ndarray:
    """Boolean [S, past+S]: key j is visible to new token i iff
    j <= past + i ([MLIR] causal mask) and, with a window W > 0, j is one of
    the W most recent positions up to and including past + i ([ORT])."""
    p = past + np.arange(seq_len)[:, None]
    j = np.arange(past + seq_len)[None, :]
    vis = j <= p
    if window > 0:
        vis &= j > p - window
    return vis


def attention(q_bits, k_buf, v_buf, seqlens_k, num_heads, kv_num_heads, scale, window,
              bias_bits, dtype, batches=None, heads=None, return_probs=False):
    """Output [B, S, H, D] float64 (NaN where not computed).

    Query head h reads KV head h // (H / Hkv).  For token i of sequence b the
    scores over keys j < past_b + S are scale * q . k_j plus
    bias[b or 0, h or 0, i, j] (bias indexed by the absolute key position),
    masked keys are dropped, and the softmax weights average the value rows.
    q_bits is [B, S, H, D]; k_buf/v_buf are [B, Hkv, M, D]."""
    B, S, H, D = q_bits.shape
    G = num_heads // kv_num_heads
    q = t_to_f64(q_bits, dtype)
    out = np.full((B, S, H, D), np.nan)
    probs = {}
    bias = None if bias_bits is None else t_to_f64(bias_bits, dtype)
    for b in (range(B) if batches is None else batches):
        past = int(seqlens_k[b])
        L = past + S
        vis = visible(past, S, window)
        K_all = t_to_f64(k_buf[b, :, :L, :], dtype)
        V_all = t_to_f64(v_buf[b, :, :L, :], dtype)
        for h in (range(H) if heads is None else heads):
            kh = h // G
            z = (q[b, :, h, :] @ K_all[kh].T) * scale
            if bias is not None:
                bb = b if bias.shape[0] > 1 else 0
                hb = h if bias.shape[1] > 1 else 0
                z = z + bias[bb, hb, :, :L]
            z = np.where(vis, z, -np.inf)
            zmax = z.max(axis=1, keepdims=True)
            e = np.exp(z - zmax)
            P = e / e.sum(axis=1, keepdims=True)
            out[b, :, h, :] = P @ V_all[kh]
            if return_probs:
                probs[(b, h)] = P
    return (out, probs) if return_probs else out


# ---------------------------------------------------------------------------
# Packed QKV input: one tensor holding every token's query, key and value
# heads.
# ---------------------------------------------------------------------------
def unpack_qkv(packed_bits: np.ndarray, num_heads: int, kv_num_heads: int):
    """query [B, S, (H + 2 Hkv) * D] in the packed form -> (query [B, S, H*D],
    key [B, S, Hkv*D], value [B, S, Hkv*D]).  Each token's row is read as
    [heads, head_size] with the head index outer ([MLIR] PR description: the
    [batch, seq, hidden] input is reshaped to [batch, seq, heads, head_size]):
    heads [0, H) are the query heads, [H, H + Hkv) the key heads and
    [H + Hkv, H + 2 Hkv) the value heads."""
    B, S, width = packed_bits.shape
    n = num_heads + 2 * kv_num_heads
    D = width // n
    x = packed_bits.reshape(B, S, n, D)
    q = x[:, :, :num_heads].reshape(B, S, num_heads * D)
    k = x[:, :, num_heads:num_heads + kv_num_heads].reshape(B, S, kv_num_heads * D)
    v = x[:, :, num_heads + kv_num_heads:].reshape(B, S, kv_num_heads * D)
    return q.copy(), k.copy(), v.copy()


# ---------------------------------------------------------------------------
# Sliding-window cache with contiguous eviction ([ORT], ZackyLake's SWA
# follow-up: the op keeps only the min(total_sequence_length, cache_capacity)
# most recent tokens, contiguously).  Here the capacity is the buffer's
# max_seq_len slots M, and seqlens_k[b] = P_b counts every token of the
# sequence before the call (its absolute position), which may exceed M: the
# buffer then holds the n_old = min(P_b, M) most recent of them, slot s
# holding position P_b - n_old + s.
# ---------------------------------------------------------------------------
def cached_count(past: int, max_seq_len: int) -> int:
    """Tokens of a sequence held in the buffer on entry: min(P_b, M)."""
    return min(int(past), max_seq_len)


def evict_keep_recent(buf_bits: np.ndarray, new_bits: np.ndarray, seqlens_k: np.ndarray) -> np.ndarray:
    """Return a copy of buf [B, Hkv, M, D] in which, per sequence, the cached
    tokens followed by the S new ones (new [B, S, Hkv, D]) are cut to their
    n_keep = min(P_b + S, M) most recent, stored contiguously from slot 0.
    Slots [n_keep, M) keep their bits."""
    out = buf_bits.copy()
    B, Hkv, M, D = buf_bits.shape
    for b in range(B):
        n_old = cached_count(seqlens_k[b], M)
        seq = np.concatenate([buf_bits[b, :, :n_old, :], new_bits[b].transpose(1, 0, 2)], axis=1)
        n_keep = min(int(seqlens_k[b]) + new_bits.shape[1], M)
        out[b, :, :n_keep, :] = seq[:, seq.shape[1] - n_keep:, :]
    return out


def attention_evicting(q_bits, k_buf, v_buf, k_new, v_new, seqlens_k, num_heads, kv_num_heads, scale, window,
                       bias_bits, dtype):
    """Output [B, S, H, D] float64 of a call in the evicting mode: token i of
    sequence b (position p = P_b + i) attends over the keys that exist for
    the call -- the n_old cached tokens (positions P_b - n_old ...) and the S
    new ones -- that are causal (j <= p) and, with W > 0, among the W most
    recent (j > p - W).  The bias is read at the absolute key position j.
    k_buf/v_buf [B, Hkv, M, D] are the buffers on entry; k_new/v_new
    [B, S, Hkv, D] the new rows (keys rotated)."""
    B, S, H, D = q_bits.shape
    M = k_buf.shape[2]
    G = num_heads // kv_num_heads
    q = t_to_f64(q_bits, dtype)
    bias = None if bias_bits is None else t_to_f64(bias_bits, dtype)
    out = np.full((B, S, H, D), np.nan)
    for b in range(B):
        past = int(seqlens_k[b])
        n_old = cached_count(past, M)
        K = t_to_f64(np.concatenate([k_buf[b, :, :n_old], k_new[b].transpose(1, 0, 2)], axis=1), dtype)
        V = t_to_f64(np.concatenate([v_buf[b, :, :n_old], v_new[b].transpose(1, 0, 2)], axis=1), dtype)
        kpos = past - n_old + np.arange(n_old + S)
        p = past + np.arange(S)[:, None]
        vis = kpos[None, :] <= p
        if window > 0:
            vis &= kpos[None, :] > p - window
        for h in range(H):
            kh = h // G
            z = (q[b, :, h, :] @ K[kh].T) * scale
            if bias is not None:
                z = z + bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0][:, kpos]
            z = np.where(vis, z, -np.inf)
            e = np.exp(z - z.max(axis=1, keepdims=True))
            out[b, :, h, :] = (e / e.sum(axis=1, keepdims=True)) @ V[kh]
    return out


# ---------------------------------------------------------------------------
# The whole operator.
# ---------------------------------------------------------------------------
def check_lengths(seqlens_k, seq_len, max_seq_len, total_sequence_length, evict=False) -> int:
    """Step 4: the operator fails when the buffer has no room for the new
    tokens ([ORT], tianleiwu's reply).  A sequence whose past plus new tokens
    exceeds total_sequence_length (the last dimension of attention_bias) is an
    invalid argument.  In the evicting mode the buffer always has room (the
    oldest tokens make way), so only the invalid-argument checks remain."""
    if total_sequence_length > max_seq_len and not evict:
        return STATUS_KV_OVERFLOW
    status = STATUS_OK
    for pb in np.asarray(seqlens_k, dtype=np.int64):
        if pb + seq_len > max_seq_len and not evict:
            return STATUS_KV_OVERFLOW
        if pb < 0 or pb + seq_len > total_sequence_length:
            status = STATUS_INVALID_ARGUMENT
    return status


def gqa_forward(query, key, value, k_buf, v_buf, seqlens_k, total_sequence_length,
                cos_cache, sin_cache, num_heads, kv_num_heads, scale, local_window_size,
                attention_bias, dtype, batches=None, heads=None, interleaved=False,
                past_key=None, past_value=None, evict=False):
    """Returns (status, out, k_buf_new, v_buf_new).

    Packed QKV: key and value None, query [B, S, (H + 2 Hkv) * D] (see
    unpack_qkv).  evict=True selects the sliding-window cache with
    contiguous eviction (shared binding only; see evict_keep_recent and
    attention_evicting); batches/heads are ignored there.

    Shared binding (past_key/past_value None): k_buf/v_buf are the one
    past/present buffer.  Non-shared binding: past_key/past_value
    [B, Hkv, Mp, D] hold the past, k_buf/v_buf are the present buffers as
    they are on entry, and the present comes back as past + new (step 0); a
    past length beyond Mp is an invalid argument.

    query [B, S, H*D], key/value [B, S, Hkv*D], k_buf/v_buf [B, Hkv, M, D],
    cos/sin [rows, D/2] or None (no rotary), attention_bias [Bb, Hb, S, total]
    or None; ``interleaved`` selects the rotary pairing.  ``out`` is float64
    [B, S, H*D] (unrounded); on an error the
    buffers come back unchanged and ``out`` is None.  scale <= 0 means
    1/sqrt(D); the scale is taken as a float32 value, as the operator's
    attribute is."""
    if key is None and value is None:
        query, key, value = unpack_qkv(query, num_heads, kv_num_heads)
    if evict and past_key is not None:
        raise ValueError("the evicting cache is defined for the shared binding only")
    B, S = query.shape[:2]
    Hkv, M, D = k_buf.shape[1:]
    H = num_heads
    status = check_lengths(seqlens_k, S, M, total_sequence_length, evict)
    if status == STATUS_OK and past_key is not None and np.any(np.asarray(seqlens_k) > past_key.shape[2]):
        status = STATUS_INVALID_ARGUMENT
    if status != STATUS_OK:
        return status, None, k_buf.copy(), v_buf.copy()
    if past_key is not None:
        k_buf = present_from_past(k_buf, past_key, seqlens_k)
        v_buf = present_from_past(v_buf, past_value, seqlens_k)
    scale = float(np.float32(scale)) if scale > 0 else float(np.float32(1.0 / np.sqrt(D)))
    q = query.reshape(B, S, H, D)
    k = key.reshape(B, S, Hkv, D)
    v = value.reshape(B, S, Hkv, D)
    if cos_cache is not None:
        pos = positions(seqlens_k, S)
        q = rotary(q, pos, cos_cache, sin_cache, dtype, interleaved)
        k = rotary(k, pos, cos_cache, sin_cache, dtype, interleaved)
    if evict:
        out = attention_evicting(q, k_buf, v_buf, k, v, seqlens_k, H, Hkv, scale, local_window_size,
                                 attention_bias, dtype)
        kb = evict_keep_recent(k_buf, k, seqlens_k)
        vb = evict_keep_recent(v_buf, v, seqlens_k)
        return STATUS_OK, out.reshape(B, S, H * D), kb, vb
    kb = scatter_append(k_buf, k, seqlens_k)
    vb = scatter_append(v_buf, v, seqlens_k)
    out = attention(q, kb, vb, seqlens_k, H, Hkv, scale, local_window_size, attention_bias,
                    dtype, batches=batches, heads=heads)
    return STATUS_OK, out.reshape(B, S, H * D), kb, vb
