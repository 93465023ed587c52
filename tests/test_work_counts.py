"""The bench's numerators: algorithmic bytes of a decode call and algorithmic
FLOPs of a prefill call, counted independently from the oracle's visibility
mask and from closed forms."""
import numpy as np
import torch

import oracle
from shared_kv_cache_gb300 import workloads as W


def _visible_keys(past, S, window):
    return sum(int(oracle.visible(int(pb), S, window).sum()) for pb in past)


def test_decode_bytes_counts_visible_rows():
    for name in ("decode_b16", "long_decode", "long_decode_w4096"):
        w = W.CONFIGS[name]
        past = W.make_inputs(w, sentinel=False)["seqlens_k"] if name == "decode_b16" else \
            torch.tensor(np.random.default_rng(3).integers(w.past_lo, w.past_hi + 1, w.batch), dtype=torch.int32)
        keys = _visible_keys(past.tolist(), 1, w.local_window_size)
        e = 2
        want = (keys * w.kv_num_heads * w.head_size * e * 2            # visible K and V rows
                + 2 * w.batch * w.num_heads * w.head_size * e          # query in, output out
                + 2 * w.batch * w.kv_num_heads * w.head_size * e)      # appended K and V rows
        assert W.decode_bytes(w, past) == want, name


def test_decode_bytes_of_the_headline_draw():
    w = W.CONFIGS["decode_b16"]
    assert W.decode_bytes(w, W.make_inputs(w, sentinel=False)["seqlens_k"]) == 103_755_776


def test_window_caps_every_sequence_at_w_keys():
    w = W.CONFIGS["long_decode_w4096"]
    past = torch.full((w.batch,), 20000, dtype=torch.int32)
    e = 2
    assert W.decode_bytes(w, past) == (w.batch * 4096 * w.kv_num_heads * w.head_size * e * 2
                                       + 2 * w.batch * w.num_heads * w.head_size * e
                                       + 2 * w.batch * w.kv_num_heads * w.head_size * e)


def test_prefill_flops_counts_visible_pairs():
    w = W.CONFIGS["chunked_prefill"].with_(seq_len=16, batch=3)
    past = [0, 7, 40]
    for window in (0, 9):
        ww = w.with_(local_window_size=window)
        pairs = _visible_keys(past, ww.seq_len, window)
        assert W.prefill_flops(ww, torch.tensor(past)) == 4 * w.head_size * w.num_heads * pairs


def test_prefill_flops_closed_form_for_an_empty_past():
    w = W.CONFIGS["prefill_2k"]
    S = w.seq_len
    want = 4 * w.head_size * w.num_heads * w.batch * S * (S + 1) // 2
    assert W.prefill_flops(w, torch.zeros(w.batch, dtype=torch.int32)) == want
    assert abs(want - 1.375e11) / 1.375e11 < 1e-3


def test_evicting_decode_bytes_from_the_oracle():
    """On the evicting cache a step reads every cached row that its token
    sees or that moves (the union, once), writes the moved rows, and writes
    the new row.  The moved rows are counted from the oracle's eviction with
    position-coded rows, the seen ones from the window on absolute positions."""
    w = W.CONFIGS["swa_decode_b16"].with_(batch=4, max_seq_len=16, local_window_size=6, head_size=8,
                                          num_heads=4, kv_num_heads=2)
    past = [3, 15, 16, 40]
    M, D, e = w.max_seq_len, w.head_size, 2
    rows_read = rows_moved = 0
    for pb in past:
        n_old = oracle.cached_count(pb, M)
        first = pb - n_old
        buf = np.zeros((1, 1, M, 1), dtype=np.uint16)
        buf[0, 0, :n_old, 0] = np.arange(first, pb) + 1         # row = its position + 1
        new = np.full((1, 1, 1, 1), pb + 1, dtype=np.uint16)
        out = oracle.evict_keep_recent(buf, new, np.array([pb]))
        n_keep = min(pb + 1, M)
        kept_old = set(int(x) - 1 for x in out[0, 0, :n_keep, 0]) - {pb}
        # a row moves when it stays but changes slot
        moved = {p for p in kept_old if (p - first) != (p - (pb + 1 - n_keep))}
        seen = {p for p in range(first, pb) if p > pb - w.local_window_size}
        rows_read += len(moved | seen)
        rows_moved += len(moved)
    want = (w.kv_num_heads * (rows_read + rows_moved) * D * e * 2
            + 2 * w.batch * w.num_heads * D * e + 2 * w.batch * w.kv_num_heads * D * e)
    assert W.decode_bytes(w, torch.tensor(past)) == want
