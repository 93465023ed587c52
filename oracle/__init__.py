"""CPU oracle for GroupQueryAttention over a shared KV buffer.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the product path never does."""
from .gqa_oracle import *  # noqa: F401,F403
from .gqa_oracle import (STATUS_OK, STATUS_INVALID_ARGUMENT, STATUS_KV_OVERFLOW,  # noqa: F401
                         t_to_f32, f32_to_t, t_to_f64, positions, rotary, present_from_past, scatter_append,
                         visible, attention, check_lengths, gqa_forward, unpack_qkv, cached_count,
                         evict_keep_recent, attention_evicting)
